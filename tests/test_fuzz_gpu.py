"""Seeded random configurations through the C ABI against the oracle.

Each case draws a geometry (latent width 64..256 in steps of 16, 576/512, or
now and then 320/512/1024 for the portable kernels; any value width up to
it; 1..128 heads), a rotary placement (half-split or
interleaved, or none), a block size, a window and softcap, the cache format
(16-bit or FP8 where the tensor-core kernels read it) and a small ragged
batch of decode sequences followed by prefill chunks, some slots -1. The
outputs meet the scale-aware bound and the cache rows the write rules; on
the geometries the tensor-core kernels cover, both read phases run there;
a second run gives the same bits.
The SEPARATE layout gets the same treatment (kv heads, group sizes, widths,
sink logits and q/k RMSNorm drawn at random).
"""
import random

import numpy as np
import pytest
import torch

from paged_latent_attention_cache_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu

CASES = 32


def _draw(seed: int):
    rng = random.Random(1000 + seed)  # (the same draws on every machine)
    pair = rng.random() < 0.2
    wide = not pair and rng.random() < 0.12  # a latent wider than 256: the portable kernels
    if pair:
        hs, vhs, H = 576, 512, rng.choice([16, 64, 128])
        ro, rd = rng.choice([(512, 64), (512, 64), (0, 64), (0, 0), (256, 64)])
    elif wide:
        hs = rng.choice([320, 512, 1024])
        vhs = rng.randint(1, hs)
        H = rng.choice([1, 4, 16])
        rd = 64
        ro = hs - 64
    else:
        hs = rng.randint(4, 16) * 16
        vhs = rng.randint(1, hs)
        H = rng.choice([1, 3, 4, 8, 16, 32, 64, 100, 128])
        rd = rng.choice([0, 16, 32, 64]) if hs >= 64 else 0
        rd = min(rd, hs - hs % 16)
        ro = rng.randint(0, (hs - rd) // 8) * 8 if rd else 0
    inter = int(rd > 0 and rng.random() < 0.3)
    bs = rng.choice([16, 32, 64, 128])
    fp8 = rng.random() < 0.25
    dtype = torch.float16 if rng.random() < 0.35 else torch.bfloat16
    window = rng.choice([-1, -1, 0, 7, 100])
    softcap = rng.choice([0.0, 0.0, 2.0, 30.0])
    nd, npf = rng.randint(0, 3), rng.randint(0, 2)
    if nd + npf == 0:
        nd = 1
    q_lens = [1] * nd + [rng.randint(2, 23) for _ in range(npf)]
    long_ctx = rng.random() < 0.3  # decode contexts of thousands of keys: many key splits
    past = [rng.randint(1000, 5000) if long_ctx and q == 1 else rng.randint(0, 299)
            for q in q_lens]
    default_scale = vhs == hs and rng.random() < 0.5
    kw = dict(dtype=dtype, num_heads=H, head_size=hs, v_head_size=vhs, rotary_offset=ro,
              rotary_dim=rd, rotary_interleaved=inter, block_size=bs,
              local_window_size=window, softcap=softcap, seed=seed,
              drop_slots=rng.randint(0, 1),
              scale=None if default_scale else rng.uniform(0.03, 0.2))
    if fp8:
        kw.update(cache_dtype="e4m3", k_scale=rng.choice([1 / 64, 0.0123]))
    tensor_core = H <= 128 and (64 <= hs <= 256 or (pair and (rd == 0 or ro >= 320 or
                                                               ro + rd <= 256)))
    return q_lens, past, kw, default_scale, tensor_core


@pytest.mark.parametrize("seed", range(CASES))
def test_random_configuration(seed):
    q_lens, past, kw, default_scale, tensor_core = _draw(seed)
    if kw.get("cache_dtype") == "e4m3" and not tensor_core:
        kw.pop("cache_dtype"), kw.pop("k_scale")   # FP8 reads are built on the tensor cores
    w = W.make_workload(f"fuzz{seed}", q_lens=q_lens, past_lens=past, **kw)
    desc = {k: v for k, v in kw.items() if k != "seed"} | dict(q_lens=q_lens, past=past)
    got = Hn.run_gpu(w, scale=0.0 if default_scale else None)
    assert got["flags"] == 0, (hex(got["flags"]), desc)
    if tensor_core:
        assert (got["op"].kernel_family(0), got["op"].kernel_family(1)) == (1, 1), desc
    again = Hn.run_gpu(w, scale=0.0 if default_scale else None)  # deterministic: same bits
    assert np.array_equal(got["out"], again["out"]), desc
    ref = Hn.run_oracle(w)
    Hn.check_cache(w, got["cache"], ref["cache"])
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO fuzz{seed}: {ratio:.3f} of the scale-aware bound ({desc})")


SEPARATE_CASES = 16


def _draw_separate(seed: int):
    rng = random.Random(5000 + seed)
    kvh = rng.choice([1, 2, 3, 4, 8])
    grp = rng.choice([1, 2, 3, 4, 8, 16]) if kvh > 1 else rng.choice([1, 4, 32, 128])
    hs = rng.randint(4, 16) * 16
    vhs = rng.randint(8, hs // 8) * 8
    rd = rng.choice([0, 16, 32, 64, hs - hs % 32])
    rd = min(rd, hs)
    ro = rng.randint(0, (hs - rd) // 8) * 8 if rd else 0
    nd, npf = rng.randint(0, 3), rng.randint(0, 2)
    if nd + npf == 0:
        npf = 1
    q_lens = [1] * nd + [rng.randint(2, 23) for _ in range(npf)]
    past = [rng.randint(0, 299) for _ in q_lens]
    kw = dict(dtype=torch.float16 if rng.random() < 0.35 else torch.bfloat16,
              num_heads=kvh * grp, kv_num_heads=kvh, head_size=hs, v_head_size=vhs,
              rotary_offset=ro, rotary_dim=rd, rotary_interleaved=int(rd > 0 and rng.random() < 0.3),
              block_size=rng.choice([16, 32, 64, 128]),
              local_window_size=rng.choice([-1, -1, 0, 7, 100]),
              softcap=rng.choice([0.0, 0.0, 2.0, 30.0]), head_sink=rng.random() < 0.5,
              qk_norm=rng.random() < 0.5, seed=seed, drop_slots=rng.randint(0, 1),
              scale=rng.uniform(0.03, 0.2))
    return q_lens, past, kw


@pytest.mark.parametrize("seed", range(SEPARATE_CASES))
def test_random_separate_configuration(seed):
    """SEPARATE layout (grouped-query heads over separate key and value
    caches, optional sink logit and q/k RMSNorm): random geometries within
    the tensor-core kernels' range (widths 64..256, value width a multiple
    of 8, up to 128 query heads per kv head), options and ragged batches."""
    q_lens, past, kw = _draw_separate(seed)
    w = W.make_separate_workload(f"sepfuzz{seed}", q_lens=q_lens, past_lens=past, **kw)
    desc = {k: v for k, v in kw.items() if k != "seed"} | dict(q_lens=q_lens, past=past)
    got = Hn.run_gpu_separate(w)
    assert got["flags"] == 0, (hex(got["flags"]), desc)
    ref = Hn.run_oracle_separate(w)
    Hn.check_separate_caches(w, got, ref)
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO sepfuzz{seed}: {ratio:.3f} of the scale-aware bound ({desc})")
