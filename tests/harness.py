"""Shared helpers of the GPU tests: run a workload through the C ABI, run
the oracle on the same seeded inputs, and compare.

Tolerances: cache rows written through RoPE within 1 ulp of the dtype
(non-rotary channels and untouched rows bit-exact). Attention outputs meet
two bounds against the oracle's float64 result:

* the fixed bound max |err| <= 2e-3 (fp16) / 1.5e-2 (bf16), stated for
  inputs with the configurations' spread (N(0, 0.5^2) queries); on the
  peaked variants (queries scaled by 8 up to 2^17, logits of tens to
  10^5) the 16-bit query operand alone moves scores by more than that bound
  allows for O(1) outputs, and only the scale-aware bound applies;
* per element, |err| <= K_REL * u * (|ref| + n_p + n_q + n_d), u the unit
  roundoff of the dtype (2^-8 bf16, 2^-11 fp16) and n_* the oracle's
  ``error_scales``: the output's sensitivity to rounding the probabilities
  and the query operand to 16 bits, the two roundings a tensor-core kernel
  adds to the operator's arithmetic, plus the rounding of the output itself.
  With independent roundings of at most u the error's standard deviation is
  about u / sqrt(3) times the sum of the scales; K_REL = 6 leaves room for the
  largest of some 10^7 elements (about 5.5 standard deviations). Unlike the
  fixed bound it scales with the output, so it rejects a 1.2x softmax scale
  or a missing query rotation on the full-size decode batches, whose
  near-uniform softmax makes every output small.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

from oracle import pa_oracle as O
from paged_latent_attention_cache_gb300 import workloads as W

TOL = {torch.float16: 2e-3, torch.bfloat16: 1.5e-2}
UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}
K_REL = 6.0


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
    cache, out_bits, out, scales = O.run_operator_bits(
        W.to_bits(w.query), W.to_bits(w.key), W.to_bits(w.key_cache), W.to_bits(w.cos_cache),
        W.to_bits(w.sin_cache), w.cumseq.numpy(), w.past.numpy(), w.block_table.numpy(),
        w.slot_mapping.numpy(), p, tokens, stats=True)
    return dict(cache=cache, out_bits=out_bits, out=out, scales=scales)


@functools.lru_cache(maxsize=8)
def workload(name: str):
    return W.WORKLOADS[name]()


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def _ordered8(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes (sign-magnitude) mapped to integers in value order."""
    c = codes.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c)


def check_cache(w: W.Workload, got: np.ndarray, ref: np.ndarray):
    """Rows no token wrote are bit-exact; written rows are bit-exact outside
    the rotary channels and within 1 ulp (FP8 cache: 1 code) inside them.
    Returns the number of rotary values that differ by that ulp."""
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
    order = _ordered8 if w.cache_dtype == "e4m3" else _ordered
    d = np.abs(order(gw[:, rot]) - order(rw[:, rot]))
    assert d.max(initial=0) <= 1, f"rotary cache channels differ by {d.max()} ulp"
    return int((d > 0).sum())


def output_bound(dtype, ref_f64: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Per-element bound K_REL * u * (|ref| + n_p + n_q + n_d) (see above);
    ``scales`` is the oracle's ``[tokens, 3, H*vhs]`` array."""
    ref = ref_f64.reshape(scales.shape[0], -1)
    return K_REL * UNIT_ROUNDOFF[dtype] * (np.abs(ref) + scales.sum(axis=1))


def check_out(w: W.Workload, got_bits: np.ndarray, ref_f64: np.ndarray, tokens=None,
              scales=None, fixed_bound=None):
    """Both bounds of the module docstring (the scale-aware one when the
    oracle's ``scales`` are given; the fixed one unless the workload's query
    was scaled, or ``fixed_bound`` says otherwise). Returns (max abs error,
    largest ratio of an element's error to its scale-aware bound, or None)."""
    dt = W.dtype_tag(w.dtype)
    g = got_bits if tokens is None else got_bits[np.asarray(tokens)]
    gf = O.bits_to_f64(g, dt)
    assert np.isfinite(gf).all(), "non-finite output"
    err = np.abs(gf - ref_f64.reshape(gf.shape))
    tol = TOL[w.dtype]
    if fixed_bound is None:
        fixed_bound = w.meta.get("query_gain", 1.0) == 1.0
    if fixed_bound:
        assert err.max() <= tol, f"max abs error {err.max():.3e} > {tol}"
    else:
        assert scales is not None, "a peaked workload needs the scale-aware bound"
    ratio = None
    if scales is not None:
        bound = output_bound(w.dtype, ref_f64, scales).reshape(err.shape)
        over = err > bound
        ratio = float(np.max(err / np.maximum(bound, 1e-300)))
        if over.any():
            i = np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)
            raise AssertionError(
                f"{int(over.sum())} of {err.size} outputs exceed the scale-aware bound; worst "
                f"at {tuple(int(x) for x in i)}: |err| {err[i]:.3e} > {bound[i]:.3e} "
                f"(ratio {ratio:.2f})")
    return float(err.max()), ratio


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


# ---------------------------------------------------------------------------
# SEPARATE layout
# ---------------------------------------------------------------------------

def run_gpu_separate(w, device="cuda"):
    from paged_latent_attention_cache_gb300.api import SeparateAttention
    d = w.to(device)
    op = SeparateAttention.from_workload(w, device=device)
    kc, vc = d.key_cache.clone(), d.value_cache.clone()
    out = torch.full((w.num_tokens, w.num_heads * w.v_head_size), float("nan"), dtype=w.dtype,
                     device=device)
    op.forward(d.query, d.key, d.value, kc, vc, d.cos_cache, d.sin_cache, d.cumseq, d.past,
               d.block_table, d.slot_mapping, w.num_decode_seqs, head_sink=d.head_sink,
               q_norm_weight=d.q_norm_weight, k_norm_weight=d.k_norm_weight, out=out)
    torch.cuda.synchronize()
    return dict(kcache=W.to_bits(kc), vcache=W.to_bits(vc), out=W.to_bits(out),
                flags=op.error_flags(), op=op)


def run_oracle_separate(w, tokens=None):
    tb = W.to_bits
    opt = lambda t: None if t is None else tb(t)
    kb, vb, ob, out, sc = O.run_separate_bits(
        tb(w.query), tb(w.key), tb(w.value), tb(w.key_cache), tb(w.value_cache),
        tb(w.cos_cache), tb(w.sin_cache), w.cumseq.numpy(), w.past.numpy(),
        w.block_table.numpy(), w.slot_mapping.numpy(), W.separate_oracle_params(w),
        opt(w.head_sink), opt(w.q_norm_weight), opt(w.k_norm_weight), tokens, stats=True)
    return dict(kcache=kb, vcache=vb, out_bits=ob, out=out, scales=sc)


def check_separate_caches(w, got, ref):
    """Value rows are copies: bit-exact. Key rows: unwritten rows bit-exact;
    written rows bit-exact where neither RMSNorm nor RoPE touches a channel,
    within 1 ulp elsewhere (f32 against the oracle's float64)."""
    vg, vr = got["vcache"], ref["vcache"]
    assert np.array_equal(vg, vr), f"{(vg != vr).sum()} value-cache values differ"
    hs = w.head_size
    g = got["kcache"].reshape(-1, hs)
    r = ref["kcache"].reshape(-1, hs)
    kvh = w.kv_num_heads
    written = np.zeros(g.shape[0] // kvh, dtype=bool)
    sl = w.slot_mapping.numpy()
    written[sl[sl >= 0]] = True
    written = np.repeat(written, kvh)
    assert (g[~written] == r[~written]).all(), "unwritten key-cache rows changed"
    touched = np.zeros(hs, dtype=bool)
    if w.k_norm_weight is not None:
        touched[:] = True
    touched[w.rotary_offset:w.rotary_offset + w.rotary_dim] = True
    gw, rw = g[written], r[written]
    assert (gw[:, ~touched] == rw[:, ~touched]).all(), "untouched key channels differ"
    d = np.abs(_ordered(gw[:, touched]) - _ordered(rw[:, touched]))
    assert d.max(initial=0) <= 1, f"key channels differ by {d.max()} ulp"
