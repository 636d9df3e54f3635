"""GPU parity of the SEPARATE layout (grouped-query attention over separate
key and value caches, optional head sink and q/k RMSNorm) through the C ABI
against the oracle: the full-size grouped-query decode batch and variants
over decode and prefill tokens. The reading of the op's SEPARATE mode is the
one stated in include/pa_latent.h."""
import numpy as np
import pytest
import torch

from paged_latent_attention_cache_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


def _check(w):
    got = Hn.run_gpu_separate(w)
    ref = Hn.run_oracle_separate(w)
    assert got["flags"] == 0, hex(got["flags"])
    Hn.check_separate_caches(w, got, ref)
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO {w.name}: max abs err {err:.3e}, {ratio:.3f} of the scale-aware bound")


def test_gqa_decode_parity():
    """32 query heads over 8 kv heads, head size 128 with full RoPE, q/k
    RMSNorm and sink logits, batch 32, contexts U[1024, 8192]."""
    _check(W.gqa_decode())


VARIANTS = {
    "gqa": dict(num_heads=8, kv_num_heads=2, head_size=128),
    "mha": dict(num_heads=4, kv_num_heads=4, head_size=128),
    "mqa_128_heads": dict(num_heads=128, kv_num_heads=1, head_size=64),
    "sink_only": dict(num_heads=8, kv_num_heads=2, head_size=128, head_sink=True),
    "norm_only": dict(num_heads=8, kv_num_heads=2, head_size=128, qk_norm=True),
    "softcap_window": dict(num_heads=8, kv_num_heads=4, head_size=128, softcap=2.5,
                           local_window_size=7, head_sink=True),
    "fp16": dict(num_heads=8, kv_num_heads=2, head_size=128, dtype=torch.float16,
                 head_sink=True, qk_norm=True),
    "vhs_64": dict(num_heads=8, kv_num_heads=2, head_size=128, v_head_size=64),
    "hs_256": dict(num_heads=16, kv_num_heads=2, head_size=256, rotary_dim=64),
    "hs_64_partial_rope": dict(num_heads=12, kv_num_heads=3, head_size=64, rotary_dim=32,
                               rotary_offset=16),
    "interleaved": dict(num_heads=8, kv_num_heads=2, head_size=128, rotary_interleaved=1),
    "no_rotary": dict(num_heads=8, kv_num_heads=2, head_size=128, rotary_dim=0, qk_norm=True),
    "bs_16": dict(num_heads=8, kv_num_heads=2, head_size=128, block_size=16, head_sink=True),
    "bs_128": dict(num_heads=8, kv_num_heads=2, head_size=128, block_size=128, qk_norm=True),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_separate_variants(name):
    kw = dict(block_size=64, seed=51, drop_slots=2)
    kw.update(VARIANTS[name])
    w = W.make_separate_workload(f"sep_{name}", q_lens=[1, 1, 9, 0, 40],
                                 past_lens=[3000, 0, 70, 5, 3], **kw)
    _check(w)
