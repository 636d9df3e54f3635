"""Shared helpers of the GPU tests: run a workload through the C ABI, run
the oracle on the same seeded inputs, and compare.

Tolerances: cache rows written through RoPE within 1 ulp of the dtype
(non-rotary channels and untouched rows bit-exact); attention outputs within
max-abs 2e-3 (fp16) / 1.5e-2 (bf16) of the oracle's float64 result.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

from oracle import pa_oracle as O
from paged_latent_attention_cache_gb300 import workloads as W

TOL = {torch.float16: 2e-3, torch.bfloat16: 1.5e-2}


def run_gpu(w: W.Workload, portable=False, device="cuda", scale=None):
    """``scale=0.0`` passes the library's "default scale" value instead of
    the workload's explicit one (the oracle keeps the explicit value)."""
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    d = w.to(device)
    op = PagedLatentAttention.from_workload(w, device=device, portable=portable)
    if scale is not None:
        op.params.scale = float(scale)
    cache = d.key_cache.clone()
    out = torch.full((w.num_tokens, w.num_heads * w.v_head_size), float("nan"),
                     dtype=w.dtype, device=device)
    op.forward(d.query, d.key, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past,
               d.block_table, d.slot_mapping, w.num_decode_seqs, out=out)
    torch.cuda.synchronize()
    return dict(cache=W.to_bits(cache), out=W.to_bits(out), flags=op.error_flags(), op=op)


def run_oracle(w: W.Workload, tokens=None):
    p = W.oracle_params(w)
    cache, out_bits, out = O.run_operator_bits(
        W.to_bits(w.query), W.to_bits(w.key), W.to_bits(w.key_cache), W.to_bits(w.cos_cache),
        W.to_bits(w.sin_cache), w.cumseq.numpy(), w.past.numpy(), w.block_table.numpy(),
        w.slot_mapping.numpy(), p, tokens)
    return dict(cache=cache, out_bits=out_bits, out=out)


@functools.lru_cache(maxsize=8)
def workload(name: str):
    return W.WORKLOADS[name]()


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def check_cache(w: W.Workload, got: np.ndarray, ref: np.ndarray):
    """Rows no token wrote are bit-exact; written rows are bit-exact outside
    the rotary channels and within 1 ulp inside them. Returns the number of
    rotary values that differ by that ulp."""
    hs = w.head_size
    g = got.reshape(-1, hs)
    r = ref.reshape(-1, hs)
    written = np.zeros(g.shape[0], dtype=bool)
    sl = w.slot_mapping.numpy()
    written[sl[sl >= 0]] = True
    same = (g[~written] == r[~written]).all(axis=1)
    assert same.all(), f"{(~same).sum()} unwritten cache rows changed"
    ro, rd = w.rotary_offset, w.rotary_dim
    rot = np.zeros(hs, dtype=bool)
    rot[ro:ro + rd] = True
    gw, rw = g[written], r[written]
    exact = gw[:, ~rot] == rw[:, ~rot]
    assert exact.all(), f"{(~exact).sum()} non-rotary cache values differ"
    if not rd:
        return 0
    d = np.abs(_ordered(gw[:, rot]) - _ordered(rw[:, rot]))
    assert d.max(initial=0) <= 1, f"rotary cache channels differ by {d.max()} ulp"
    return int((d > 0).sum())


def check_out(w: W.Workload, got_bits: np.ndarray, ref_f64: np.ndarray, tokens=None):
    dt = W.dtype_tag(w.dtype)
    g = got_bits if tokens is None else got_bits[np.asarray(tokens)]
    gf = O.bits_to_f64(g, dt)
    assert np.isfinite(gf).all(), "non-finite output"
    err = np.abs(gf - ref_f64.reshape(gf.shape))
    tol = TOL[w.dtype]
    assert err.max() <= tol, f"max abs error {err.max():.3e} > {tol}"
    return float(err.max())


def sample_tokens(w: W.Workload, per_seq: int = 24, seed: int = 0):
    """First/last token of each sequence, tokens next to block boundaries
    and a seeded random draw."""
    rng = np.random.default_rng(seed)
    cs = w.cumseq.tolist()
    out = set()
    for b in range(w.num_seqs):
        lo, hi = cs[b], cs[b + 1]
        if hi <= lo:
            continue
        out.update({lo, hi - 1})
        past = w.past_lens[b]
        for t in range(lo, hi):
            pos = past + t - lo
            if pos % w.block_size in (0, w.block_size - 1) and rng.random() < 0.05:
                out.add(t)
        out.update(int(x) for x in rng.integers(lo, hi, size=min(per_seq, hi - lo)))
    return sorted(out)
