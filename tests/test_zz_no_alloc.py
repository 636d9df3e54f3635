"""The allocation-free decode entry point (pa_latent_decode_noalloc) against
the workspace-based one.

pa_latent_decode_noalloc serves callers that cannot allocate device memory
(a host framework that owns every allocation, a serving loop that must not
touch the allocator while running): it runs the same decode with the
library's static scratch instead of a caller workspace. This file is
collected last so that a stop-at-first-failure run has already run every
other test; it passes on its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from oracle import pa_oracle as O
from paged_latent_attention_cache_gb300 import binding as B
from paged_latent_attention_cache_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["glm_decode", "dsv3_decode"])
def test_noalloc_decode_matches_workspace_decode(name):
    w = Hn.workload(name)
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    cache = d.key_cache.clone()
    op.write(d.key, d.cos_cache, d.sin_cache, d.slot_mapping, d.cumseq, d.past, cache)
    shape = (w.num_tokens, w.num_heads * w.v_head_size)
    ref = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
    op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table, ref,
              0, w.num_decode_seqs)
    torch.cuda.synchronize()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    tol = Hn.TOL[w.dtype]
    ref_f = O.bits_to_f64(W.to_bits(ref), W.dtype_tag(w.dtype))
    assert np.isfinite(ref_f).all()
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        out = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
        B.pa_latent_decode_noalloc(op.params, d.query, cache, d.cos_cache, d.sin_cache, d.cumseq,
                                   d.past, d.block_table, out, 0, w.num_decode_seqs,
                                   err_flags=flags)
        torch.cuda.synchronize()
        got = O.bits_to_f64(W.to_bits(out), W.dtype_tag(w.dtype))
        assert np.isfinite(got).all()
        assert np.max(np.abs(got - ref_f)) <= tol
    assert int(flags.item()) == 0


def test_noalloc_rejects_calls_beyond_the_scratch():
    w = Hn.workload("glm_decode")
    p = B.make_params(**dict(W.oracle_params(w), dtype=w.dtype))
    huge = 1 << 20  # sequences: far more partials than 32 MiB holds
    assert B.pa_latent_workspace_size(p, huge, huge) > (32 << 20)
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.PaError) as e:
        B.pa_latent_decode_noalloc(p, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                   0, huge, num_tokens=huge, num_seqs=huge)
    assert e.value.status == B.PA_ERR_WORKSPACE
    assert "static scratch" in str(e.value)
