"""The allocation-free decode entry point (pa_latent_decode_noalloc) against
the workspace-based one.

pa_latent_decode_noalloc serves callers that cannot allocate device memory
(a host framework that owns every allocation, a serving loop that must not
touch the allocator while running): it runs the same decode with the
library's static scratch instead of a caller workspace. Both run the same
kernels with the same split plan, so their outputs are bit-equal. This file
is collected last so that a stop-at-first-failure run has already run every
other test; it passes on its own in a fresh process as well.
"""
import pytest
import torch

from paged_latent_attention_cache_gb300 import binding as B
from paged_latent_attention_cache_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu

SCRATCH = 32 << 20


def _prepared(w):
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    cache = d.key_cache.clone()
    op.write(d.key, d.cos_cache, d.sin_cache, d.slot_mapping, d.cumseq, d.past, cache)
    return d, op, cache


def _noalloc(w, d, op, cache, lo, hi, flags):
    out = torch.full((w.num_tokens, w.num_heads * w.v_head_size), float("nan"), dtype=w.dtype,
                     device="cuda")
    B.pa_latent_decode_noalloc(op.params, d.query, cache, d.cos_cache, d.sin_cache, d.cumseq,
                               d.past, d.block_table, out, lo, hi, err_flags=flags)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", ["glm_decode", "dsv3_decode"])
def test_noalloc_decode_matches_workspace_decode(name):
    w = Hn.workload(name)
    d, op, cache = _prepared(w)
    shape = (w.num_tokens, w.num_heads * w.v_head_size)
    ref = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
    op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table, ref,
              0, w.num_decode_seqs)
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        out = _noalloc(w, d, op, cache, 0, w.num_decode_seqs, flags)
        assert torch.equal(out, ref)
    assert int(flags.item()) == 0


def test_noalloc_limit_per_geometry():
    """The scratch holds a 576/512 decode of 127 sequences but not 128, and a
    192/128 decode of 504 but not 505 (workspace size of the call's range)."""
    for geo, fits in ((W.DSV3, 127), (W.GLM, 504)):
        p = B.make_params(dtype=torch.bfloat16, num_heads=128 if geo is W.DSV3 else 64,
                          block_size=64, num_blocks=1 << 16, max_blocks_per_seq=64,
                          cos_rows=4096, scale=W.DSV3_SCALE, **geo)
        assert B.pa_latent_workspace_size(p, fits, fits) <= SCRATCH
        assert B.pa_latent_workspace_size(p, fits + 1, fits + 1) > SCRATCH


def test_noalloc_decodes_a_range_of_a_larger_batch():
    """A 576/512 batch of 200 sequences needs more than the scratch as a
    whole; ranges of it that fit are decoded, bit-equal to the workspace
    decode of the same range, and the whole batch is rejected."""
    B_ = 200
    w = W.make_workload("noalloc_big", q_lens=[1] * B_, past_lens=[150 + 7 * i for i in range(B_)],
                        num_heads=128, **W.DSV3, block_size=64, scale=W.DSV3_SCALE, seed=41)
    p = B.make_params(**dict(W.oracle_params(w), dtype=w.dtype))
    assert B.pa_latent_workspace_size(p, B_, B_) > SCRATCH
    d, op, cache = _prepared(w)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    for lo, hi in ((0, 64), (64, 191), (191, 200)):
        ref = torch.full((w.num_tokens, w.num_heads * w.v_head_size), float("nan"),
                         dtype=w.dtype, device="cuda")
        op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table,
                  ref, lo, hi)
        out = _noalloc(w, d, op, cache, lo, hi, flags)
        assert torch.equal(out[lo:hi], ref[lo:hi]), (lo, hi)
        assert torch.isnan(out[:lo].float()).all() and torch.isnan(out[hi:].float()).all()
    assert int(flags.item()) == 0
    with pytest.raises(B.PaError) as e:
        _noalloc(w, d, op, cache, 0, B_, flags)
    assert e.value.status == B.PA_ERR_WORKSPACE


def test_noalloc_rejects_calls_beyond_the_scratch():
    w = Hn.workload("glm_decode")
    p = B.make_params(**dict(W.oracle_params(w), dtype=w.dtype))
    huge = 1 << 20  # sequences: far more partials than 32 MiB holds
    assert B.pa_latent_workspace_size(p, huge, huge) > SCRATCH
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.PaError) as e:
        B.pa_latent_decode_noalloc(p, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                   0, huge, num_tokens=huge, num_seqs=huge)
    assert e.value.status == B.PA_ERR_WORKSPACE
    assert "static scratch" in str(e.value)
