"""CPU oracle for the paged LATENT (absorbed-MLA) attention operator.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow, obviously-correct restatement of what the operator
computes, in float64 numpy, sharing no code with the CUDA path. Sources (the
onnx-runtime-ep-cuda ``paged_attention.rs`` page and the PR pages around it):

* token -> (sequence, absolute position): ``paged_attention.rs`` device
  helper ``locate_token`` (first sequence whose cumulative end exceeds the
  token; position = past + offset inside the sequence).
* partial RoPE on channels ``[rotary_offset, rotary_offset + rotary_dim)``:
  ``paged_attention.rs`` helper ``rope_channel`` (non-interleaved: the first
  half rotates with -sin against the partner half channels away, the second
  half with +sin; interleaved: even/odd neighbours).
* write phase: ``paged_attention.rs`` ``write_impl`` and the module doc
  "Write phase" (post-RoPE row rounded to the cache dtype and stored at
  ``key_cache[slot]``; slot -1 skips).
* read phase: ``paged_attention.rs`` ``attn_impl`` and the module doc "Read
  phase" (causal keys 0..=pos, window skip when pos-j > window, score =
  scale * q.k then softcap*tanh(s/softcap), softmax, V = leading
  v_head_size channels of the same latent row, output rounded to dtype,
  zero when no key is visible).
* softmax form: PR #1978 review ("online-softmax ... algebraically identical
  to the oracle's two-pass"); this oracle is the two-pass form.

Precision: every value is converted exactly to float64; RoPE, dot products,
softmax and the weighted sum are evaluated in float64 and only the stored
results (cache rows, outputs) are rounded, round-to-nearest-even, to the
operator dtype. The pages' own oracle accumulates in f32; float64 only
tightens the reference.

Pins (tests/test_oracle_pins.py): the rounding routine against torch and
numpy casts, RoPE against complex multiplication and the relative-position
identity, the attention against a naive contiguous dense attention, against
decomposed multi-head latent attention, placement invariance under a
permuted block table, untouched cache rows for slot -1, and closed-form
special cases. ``error_scales`` (a tolerance helper for the parity tests,
not part of the operator) is pinned by its closed forms on one key and on
equal probabilities, by a Monte Carlo run of independently perturbed
probabilities and scores, and by a finite-difference derivative in one
query channel.
"""
from __future__ import annotations

import numpy as np

BF16 = "bf16"
F16 = "f16"


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of bf16/f16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


_FMT = {
    # mantissa bits, minimum normal exponent, largest finite value
    BF16: (7, -126, float.fromhex("0x1.fep127")),
    F16: (10, -14, 65504.0),
}


def round_f64_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest bf16/f16 value, ties to even,
    overflowing to +-inf, and return the bit patterns (uint16).

    The rounding is done directly from float64 (no intermediate float32):
    with e = max(floor(log2|x|), emin) the representable spacing is
    2^(e - mantissa_bits); x / spacing is an exact float64 and
    ``np.rint`` rounds it half-to-even."""
    mant, emin, maxv = _FMT[dtype]
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, ex = np.frexp(ax)           # ax = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, emin)
    spacing = np.ldexp(1.0, (e - mant).astype(np.int64))
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(x / spacing) * spacing
    r = np.where(np.isfinite(x), r, x)
    r = np.where(np.abs(r) > maxv, np.copysign(np.inf, x), r)
    if dtype == BF16:
        return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return r.astype(np.float16).view(np.uint16)


def round_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the dtype and widen back to float64."""
    return bits_to_f64(round_f64_to_bits(x, dtype), dtype)


# FP8 cache format: OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits with bias
# 7, 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; codes
# 0x7F and 0xFF are NaN (there are no infinities), so the largest finite
# value is 1.75 * 2^8 = 448.
E4M3 = "e4m3"
E4M3_MAX = 448.0


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact values of E4M3 codes (uint8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of float64 values: round to nearest, ties to even,
    saturating to +-448 (values of magnitude 448 or more give the largest
    finite code); a value that rounds to zero keeps its sign (0x80 for a
    negative one)."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.minimum(np.abs(x), E4M3_MAX)
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(ax)                       # ax = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)    # unbiased exponent, subnormals at -6
    spacing = np.ldexp(1.0, e - 3)
    r = np.minimum(np.rint(ax / spacing) * spacing, E4M3_MAX)
    # code of the rounded magnitude r
    with np.errstate(divide="ignore"):
        _, er = np.frexp(r)
    er = er.astype(np.int64) - 1
    normal = r >= 2.0 ** -6
    ef = np.where(normal, er + 7, 0)
    mf = np.where(normal, np.rint((r / np.ldexp(1.0, er) - 1.0) * 8.0), np.rint(r / 2.0 ** -9))
    code = (ef << 3) | mf.astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    return code.astype(np.uint8)


def quantize_e4m3(row: np.ndarray, k_scale: float) -> np.ndarray:
    """E4M3 codes of a cache row: each channel's value rounded to float32,
    divided by k_scale in float32 (IEEE division), then rounded to E4M3."""
    v32 = np.asarray(row, dtype=np.float64).astype(np.float32)
    q32 = v32 / np.float32(k_scale)
    return round_to_e4m3(q32.astype(np.float64))


# ---------------------------------------------------------------------------
# Token location and RoPE
# ---------------------------------------------------------------------------

def locate_token(t: int, cumseq: np.ndarray, past: np.ndarray):
    """(sequence b, absolute position) of global token t: b is the first
    sequence whose cumulative end cumseq[b+1] exceeds t; the position is
    past[b] plus t's offset inside that sequence. Tokens outside
    [0, cumseq[B]) are rejected (the pages fall back to sequence 0; the
    operator contract requires cumseq[B] == T)."""
    B = len(past)
    for b in range(B):
        if t < int(cumseq[b + 1]):
            if t < int(cumseq[b]):
                raise ValueError("cumulative_sequence_length is not monotone")
            return b, int(past[b]) + (t - int(cumseq[b]))
    raise ValueError(f"token {t} lies beyond cumulative_sequence_length[B]")


def rope_row(x: np.ndarray, pos: int, rotary_offset: int, rotary_dim: int,
             cos_tab: np.ndarray, sin_tab: np.ndarray, interleaved: bool) -> np.ndarray:
    """Partial RoPE of one head row (float64) at absolute position ``pos``.

    Channels outside [ro, ro+rd) are returned unchanged. Inside, with
    half = rd/2 and c_i, s_i = cos_tab[pos, i], sin_tab[pos, i]:

    * non-interleaved: channel ro+i (i < half) pairs with ro+i+half,
      out[ro+i] = x[ro+i] c_i - x[ro+i+half] s_i and
      out[ro+i+half] = x[ro+i+half] c_i + x[ro+i] s_i;
    * interleaved: channel ro+2i pairs with ro+2i+1,
      out[ro+2i] = x[ro+2i] c_i - x[ro+2i+1] s_i and
      out[ro+2i+1] = x[ro+2i+1] c_i + x[ro+2i] s_i.
    """
    out = np.array(x, dtype=np.float64, copy=True)
    if rotary_dim == 0:
        return out
    half = rotary_dim // 2
    c = cos_tab[pos, :half]
    s = sin_tab[pos, :half]
    seg = out[rotary_offset:rotary_offset + rotary_dim]
    if interleaved:
        a = seg[0::2].copy()
        b = seg[1::2].copy()
        seg[0::2] = a * c - b * s
        seg[1::2] = b * c + a * s
    else:
        a = seg[:half].copy()
        b = seg[half:].copy()
        seg[:half] = a * c - b * s
        seg[half:] = b * c + a * s
    return out


# ---------------------------------------------------------------------------
# The paged cache: one latent row per slot (slot = block * bs + offset)
# ---------------------------------------------------------------------------

class F64Cache:
    """Cache rows held exactly in float64 (no rounding on store)."""

    def __init__(self, rows: np.ndarray):
        self.rows = np.array(rows, dtype=np.float64, copy=True)

    @property
    def num_rows(self) -> int:
        return self.rows.shape[0]

    def get(self, idx) -> np.ndarray:
        return self.rows[idx]

    def put(self, slot: int, row: np.ndarray):
        self.rows[slot] = row


class E4M3Cache:
    """Cache rows held as E4M3 codes with one scale for the whole cache: a
    store quantizes the float64 row (``quantize_e4m3``), a load returns the
    code's value times k_scale (exact in float64)."""

    def __init__(self, codes: np.ndarray, k_scale: float):
        self.codes = np.array(codes, dtype=np.uint8, copy=True)
        self.k_scale = float(k_scale)

    @property
    def num_rows(self) -> int:
        return self.codes.shape[0]

    def get(self, idx) -> np.ndarray:
        return e4m3_to_f64(self.codes[idx]) * self.k_scale

    def put(self, slot: int, row: np.ndarray):
        self.codes[slot] = quantize_e4m3(row, self.k_scale)


class BitsCache:
    """Cache rows held as bf16/f16 bit patterns; a store rounds the float64
    row to the dtype, a load widens exactly."""

    def __init__(self, bits: np.ndarray, dtype: str):
        self.bits = np.array(bits, dtype=np.uint16, copy=True)
        self.dtype = dtype

    @property
    def num_rows(self) -> int:
        return self.bits.shape[0]

    def get(self, idx) -> np.ndarray:
        return bits_to_f64(self.bits[idx], self.dtype)

    def put(self, slot: int, row: np.ndarray):
        self.bits[slot] = round_f64_to_bits(row, self.dtype)


# ---------------------------------------------------------------------------
# The operator: write phase, then read phase
# ---------------------------------------------------------------------------

def _check_geometry(p: dict):
    hs, vhs = p["head_size"], p["v_head_size"] or p["head_size"]
    assert 1 <= vhs <= hs
    assert p["rotary_offset"] + p["rotary_dim"] <= hs
    return hs, vhs


def latent_write(key, cos_tab: np.ndarray, sin_tab: np.ndarray, slot_mapping: np.ndarray,
                 cumseq: np.ndarray, past: np.ndarray, cache, p: dict):
    """Write phase. ``key`` maps a token index to its float64 latent row
    (an array ``[T, hs]`` or a callable); ``cache`` is an F64Cache or
    BitsCache and is updated in place.

    For every token t, in order: skip when slot_mapping[t] < 0; otherwise
    apply partial RoPE to key[t] at the token's absolute position and store
    the row (rounded to the cache dtype by the cache) at row
    slot_mapping[t]."""
    _check_geometry(p)
    get_key = key if callable(key) else (lambda t: key[t])
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        if slot >= cache.num_rows:
            raise ValueError(f"slot {slot} outside the cache")
        _, pos = locate_token(t, cumseq, past)
        cache.put(slot, rope_row(get_key(t), pos, p["rotary_offset"], p["rotary_dim"],
                                 cos_tab, sin_tab, bool(p["rotary_interleaved"])))
    return cache


def visible_keys(pos: int, window: int):
    """Causal keys 0..=pos, minus those with pos - j > window when the
    window is enabled (window >= 0)."""
    lo = 0 if window < 0 else max(0, pos - window)
    return range(lo, pos + 1)


def cache_row_index(b: int, j: int, block_table: np.ndarray, block_size: int,
                    num_blocks: int) -> int:
    """Row of logical key j of sequence b: block_table[b, j // bs] is the
    physical block, j % bs the offset inside it."""
    phys = int(block_table[b, j // block_size])
    if not 0 <= phys < num_blocks:
        raise ValueError(f"block_table[{b}, {j // block_size}] = {phys} is not a block")
    return phys * block_size + j % block_size


def latent_attend_token(t: int, q_row: np.ndarray, cache, cos_tab: np.ndarray,
                        sin_tab: np.ndarray, cumseq: np.ndarray, past: np.ndarray,
                        block_table: np.ndarray, p: dict, stats: bool = False):
    """Read phase for token t, all heads: returns float64 ``[H, vhs]``.
    ``q_row`` is the token's float64 query row ``[H*hs]``.

    q_h = RoPE(q_row[h*hs:(h+1)*hs]) (kept in float64), K_j the cache row of
    visible key j, s_hj = scale * q_h . K_j, then
    s_hj = softcap * tanh(s_hj / softcap) when softcap > 0, a two-pass
    softmax over j, and out_h = sum_j p_hj K_j[:vhs] / sum_j p_hj; zero
    when no key is visible.

    With ``stats=True`` it returns ``(out, scales)``, ``scales`` being the
    ``error_scales`` of this token (a test-tolerance helper; the operator's
    result is ``out`` alone)."""
    hs, vhs = _check_geometry(p)
    H = p["num_heads"]
    bs = p["block_size"]
    num_blocks = cache.num_rows // bs
    b, pos = locate_token(t, cumseq, past)
    q = np.stack([rope_row(q_row[h * hs:(h + 1) * hs], pos, p["rotary_offset"],
                           p["rotary_dim"], cos_tab, sin_tab,
                           bool(p["rotary_interleaved"])) for h in range(H)])
    keys = list(visible_keys(pos, p["local_window_size"]))
    if not keys:
        zero = np.zeros((H, vhs))
        return (zero, np.zeros((3, H, vhs))) if stats else zero
    rows = [cache_row_index(b, j, block_table, bs, num_blocks) for j in keys]
    K = cache.get(rows)                               # [n, hs]
    s = (q @ K.T) * p["scale"]                        # [H, n]
    if p["softcap"] > 0.0:
        s = p["softcap"] * np.tanh(s / p["softcap"])
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    den = w.sum(axis=1, keepdims=True)
    out = (w @ K[:, :vhs]) / den
    if not stats:
        return out
    return out, error_scales(q, K, w / den, out, p["scale"], vhs)


def error_scales(q: np.ndarray, K: np.ndarray, prob: np.ndarray, out: np.ndarray,
                 scale: float, vhs: int) -> np.ndarray:
    """How strongly one token's attention output reacts to rounding inside
    a kernel, per output element. TEST-TOLERANCE HELPER: the operator does
    not compute this; the parity tests scale their per-element bound by it.

    ``q`` [H, hs] rotated queries, ``K`` [n, hs] visible key rows (V_j =
    K_j[:vhs]), ``prob`` [H, n] the softmax probabilities, ``out`` [H, vhs].
    Returns float64 ``[3, H, vhs]``:

    * ``[0]`` n_p = sqrt(sum_j p_j^2 V_jc^2): the standard deviation of the
      output when every probability is multiplied by an independent
      (1 + e_j), per unit standard deviation of e_j (rounding P to 16 bits
      before the product with V).
    * ``[1]`` n_q = sqrt(sum_j p_j^2 g_j^2 (V_jc - out_c)^2) with
      g_j = scale * sqrt(sum_d q_d^2 K_jd^2): the same for independent score
      perturbations of standard deviation g_j per unit (rounding the query
      operand to 16 bits perturbs score j by about that much, first order:
      d out_c / d s_j = p_j (V_jc - out_c)).
    * ``[2]`` n_d = scale * |q_c| * sum_j p_j (V_jc - out_c)^2: the size of
      d out_c / d log q_c, which is coherent over the keys because query
      channel c multiplies value channel c (K_jc = V_jc) in every score.
    """
    V = K[:, :vhs]
    V2 = V * V
    n_p = np.sqrt(np.maximum((prob * prob) @ V2, 0.0))
    g2 = (scale * scale) * ((q * q) @ (K * K).T)                 # [H, n]
    a = prob * prob * g2
    var_a = (a @ V2) - 2.0 * out * (a @ V) + out * out * a.sum(axis=1, keepdims=True)
    n_q = np.sqrt(np.maximum(var_a, 0.0))
    var_p = (prob @ V2) - out * out
    n_d = scale * np.abs(q[:, :vhs]) * np.maximum(var_p, 0.0)
    return np.stack([n_p, n_q, n_d])


def latent_attend(query, cache, cos_tab, sin_tab, cumseq, past, block_table, p,
                  tokens=None, stats: bool = False):
    """Read phase for the listed tokens (default: all). ``query`` maps a
    token index to its float64 row (an array ``[T, H*hs]`` or a callable).
    Returns float64 ``[len(tokens), H, vhs]`` (with ``stats``: and the
    ``error_scales`` stacked as ``[len(tokens), 3, H, vhs]``)."""
    get_q = query if callable(query) else (lambda t: query[t])
    tokens = range(int(cumseq[-1])) if tokens is None else tokens
    res = [latent_attend_token(int(t), get_q(int(t)), cache, cos_tab, sin_tab,
                               cumseq, past, block_table, p, stats) for t in tokens]
    if not stats:
        return np.stack(res)
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res])


# ---------------------------------------------------------------------------
# Bit-level entry point (operator dtype in, operator dtype out)
# ---------------------------------------------------------------------------

def run_operator_bits(query_bits, key_bits, cache_bits, cos_bits, sin_bits, cumseq, past,
                      block_table, slot_mapping, p: dict, tokens=None, stats: bool = False):
    """Write then read, on uint16 bit arrays of the operator dtype.

    Shapes: query ``[T, H*hs]``, key ``[T, hs]``, cache
    ``[num_blocks, bs, 1, hs]`` (any shape with hs last), cos/sin
    ``[rows, rd/2]``. The read phase sees the cache after the write. With
    ``p["cache_dtype"] == "e4m3"`` the cache holds uint8 E4M3 codes scaled
    by ``p["k_scale"]`` (returned as codes).
    Returns (new cache bits in the input's shape, output bits
    ``[len(tokens), H*vhs]``, output float64 before rounding); with
    ``stats`` a fourth item, the ``error_scales`` ``[len(tokens), 3, H*vhs]``."""
    dt = p["dtype"]
    hs, _ = _check_geometry(p)
    shape = cache_bits.shape
    if p.get("cache_dtype") == E4M3:
        cache = E4M3Cache(np.asarray(cache_bits).reshape(-1, hs), p["k_scale"])
    else:
        cache = BitsCache(np.asarray(cache_bits).reshape(-1, hs), dt)
    cos_tab = bits_to_f64(cos_bits, dt)
    sin_tab = bits_to_f64(sin_bits, dt)
    latent_write(lambda t: bits_to_f64(key_bits[t], dt), cos_tab, sin_tab,
                 np.asarray(slot_mapping), cumseq, past, cache, p)
    res = latent_attend(lambda t: bits_to_f64(query_bits[t], dt), cache, cos_tab, sin_tab,
                        cumseq, past, block_table, p, tokens, stats)
    out = res[0] if stats else res
    out = out.reshape(out.shape[0], -1)
    stored = cache.codes if isinstance(cache, E4M3Cache) else cache.bits
    if not stats:
        return stored.reshape(shape), round_f64_to_bits(out, dt), out
    sc = res[1].reshape(out.shape[0], 3, -1)
    return stored.reshape(shape), round_f64_to_bits(out, dt), out, sc


# ---------------------------------------------------------------------------
# SEPARATE layout: grouped-query attention over separate key and value caches
# ---------------------------------------------------------------------------
# The second dense mode of the op (PR #1940 page: the oracle covers
# "SEPARATE (GQA, RoPE, softcap, local window, head_sink, q/k RMSNorm)";
# "num_heads % kv_num_heads == 0"; the ORT v1.29 input list on the PR #1978
# page: value(2), value_cache(4), head_sink(11), q_norm_weight(12),
# k_norm_weight(13)). Readings where the pages are silent: key_cache is
# [num_blocks, bs, kv_num_heads, hs] and value_cache [num_blocks, bs,
# kv_num_heads, vhs] (slot-major like the LATENT cache); query head h reads kv
# head h // (num_heads / kv_num_heads); RMSNorm y = x / sqrt(mean(x^2) + eps) * w
# over a head's hs channels with one weight vector for all heads, applied
# before RoPE; the sink is one raw logit per query head (no scale, no
# softcap) that joins the softmax denominator only; values get neither norm
# nor rotation.

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def separate_write(key, value, cos_tab, sin_tab, slot_mapping, cumseq, past, kcache, vcache,
                   p: dict, k_norm=None):
    """Write phase, SEPARATE layout. ``key(t)`` -> float64 [kvH, hs] and
    ``value(t)`` -> [kvH, vhs] (arrays or callables). For every token with
    slot >= 0 and every kv head g: k = RoPE(RMSNorm(key[t, g]) if k_norm
    else key[t, g]) is stored at cache row slot * kvH + g, and value[t, g]
    unchanged at the same row of the value cache (both rounded by the
    caches)."""
    kvh = p["kv_num_heads"]
    get_k = key if callable(key) else (lambda t: key[t])
    get_v = value if callable(value) else (lambda t: value[t])
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:  # slot -1: this token's rows are not written
            continue
        if (slot + 1) * kvh > kcache.num_rows:
            raise ValueError(f"slot {slot} outside the cache")
        _, pos = locate_token(t, cumseq, past)
        k, v = get_k(t), get_v(t)
        for g in range(kvh):
            kg = rms_norm(k[g], k_norm, p["rms_eps"]) if k_norm is not None else k[g]
            kcache.put(slot * kvh + g, rope_row(kg, pos, p["rotary_offset"], p["rotary_dim"],
                                                cos_tab, sin_tab, bool(p["rotary_interleaved"])))
            vcache.put(slot * kvh + g, v[g])
    return kcache, vcache


def separate_attend_token(t: int, q_row: np.ndarray, kcache, vcache, cos_tab, sin_tab, cumseq,
                          past, block_table, p: dict, head_sink=None, q_norm=None,
                          stats: bool = False):
    """Read phase, SEPARATE layout, token t, all query heads: float64
    [H, vhs]. q_h = RoPE(RMSNorm(q_row[h]) if q_norm else q_row[h]); keys
    and values of the visible positions j are rows (block_table[b, j // bs]
    * bs + j % bs) * kvH + g of the caches, g = h // (H / kvH); s_hj = scale
    * q_h . K_j, softcap as in the LATENT mode; with a sink logit z_h the
    softmax is exp(s_hj - m) / (sum_j exp(s_hj - m) + exp(z_h - m)), m =
    max(max_j s_hj, z_h); out_h = sum_j p_hj V_j (zero when no key is
    visible). ``stats``: also the ``error_scales`` [3, H, vhs]."""
    H, kvh = p["num_heads"], p["kv_num_heads"]
    hs = p["head_size"]
    vhs = p["v_head_size"] or hs
    grp = H // kvh
    bs = p["block_size"]
    num_blocks = kcache.num_rows // (bs * kvh)
    b, pos = locate_token(t, cumseq, past)
    keys = list(visible_keys(pos, p["local_window_size"]))
    out = np.zeros((H, vhs))
    scales = np.zeros((3, H, vhs))
    slots = [cache_row_index(b, j, block_table, bs, num_blocks) for j in keys]
    for h in range(H):
        g = h // grp
        qh = q_row[h * hs:(h + 1) * hs]
        if q_norm is not None:
            qh = rms_norm(qh, q_norm, p["rms_eps"])
        qh = rope_row(qh, pos, p["rotary_offset"], p["rotary_dim"], cos_tab, sin_tab,
                      bool(p["rotary_interleaved"]))
        if not keys:
            continue
        K = kcache.get([s * kvh + g for s in slots])
        V = vcache.get([s * kvh + g for s in slots])
        s = (K @ qh) * p["scale"]
        cap = p["softcap"]
        if cap > 0.0:
            s = cap * np.tanh(s / cap)
        m = s.max()
        extra = 0.0
        if head_sink is not None:
            m = max(m, float(head_sink[h]))
            extra = np.exp(float(head_sink[h]) - m)
        w = np.exp(s - m)
        den = w.sum() + extra
        out[h] = (w @ V) / den
        if stats:
            # the probability, query-rounding and diagonal terms, with V a
            # separate matrix (the diagonal term needs K_jc = V_jc, which only
            # holds when the value rows are the key rows; it is omitted here)
            prob = (w / den)[None, :]
            sc = error_scales_kv(qh[None, :], K, V, prob, out[h][None, :], p["scale"])
            scales[:, h, :] = sc[:, 0, :]
    return (out, scales) if stats else out


def error_scales_kv(q: np.ndarray, K: np.ndarray, V: np.ndarray, prob: np.ndarray,
                    out: np.ndarray, scale: float) -> np.ndarray:
    """``error_scales`` for separate key and value rows (TEST-TOLERANCE
    HELPER): n_p = sqrt(sum_j p_j^2 V_jc^2), n_q = sqrt(sum_j p_j^2 g_j^2
    (V_jc - out_c)^2) with g_j = scale * sqrt(sum_d q_d^2 K_jd^2), and n_d =
    0 (no query channel meets a value channel in every score). [3, H, vhs]."""
    V2 = V * V
    n_p = np.sqrt(np.maximum(np.square(prob) @ V2, 0.0))
    g2 = (scale * scale) * ((q * q) @ (K * K).T)
    a = prob * prob * g2
    var_a = (a @ V2) - 2.0 * (a @ V) * out + out * out * a.sum(axis=1, keepdims=True)
    n_q = np.sqrt(np.maximum(var_a, 0.0))
    return np.stack([n_p, n_q, np.zeros_like(n_p)])


def run_separate_bits(query_bits, key_bits, value_bits, kcache_bits, vcache_bits, cos_bits,
                      sin_bits, cumseq, past, block_table, slot_mapping, p: dict,
                      head_sink_bits=None, q_norm_bits=None, k_norm_bits=None, tokens=None,
                      stats: bool = False):
    """SEPARATE write then read on uint16 bit arrays of the operator dtype:
    query [T, H*hs], key [T, kvH*hs], value [T, kvH*vhs], caches
    [num_blocks, bs, kvH, hs|vhs], head_sink [H], norm weights [hs]. Returns
    (key cache bits, value cache bits, output bits [len(tokens), H*vhs],
    output float64[, error scales [len(tokens), 3, H*vhs]])."""
    dt = p["dtype"]
    hs, kvh = p["head_size"], p["kv_num_heads"]
    vhs = p["v_head_size"] or hs
    kc = BitsCache(np.asarray(kcache_bits).reshape(-1, hs), dt)
    vc = BitsCache(np.asarray(vcache_bits).reshape(-1, vhs), dt)
    cos_t, sin_t = bits_to_f64(cos_bits, dt), bits_to_f64(sin_bits, dt)
    kn = None if k_norm_bits is None else bits_to_f64(k_norm_bits, dt)
    qn = None if q_norm_bits is None else bits_to_f64(q_norm_bits, dt)
    sink = None if head_sink_bits is None else bits_to_f64(head_sink_bits, dt)
    separate_write(lambda t: bits_to_f64(key_bits[t], dt).reshape(kvh, hs),
                   lambda t: bits_to_f64(value_bits[t], dt).reshape(kvh, vhs), cos_t, sin_t,
                   np.asarray(slot_mapping), cumseq, past, kc, vc, p, kn)
    tokens = range(int(cumseq[-1])) if tokens is None else tokens
    res = [separate_attend_token(int(t), bits_to_f64(query_bits[int(t)], dt), kc, vc, cos_t,
                                 sin_t, cumseq, past, block_table, p, sink, qn, stats)
           for t in tokens]
    if stats:
        out = np.stack([r[0] for r in res]).reshape(len(res), -1)
        sc = np.stack([r[1] for r in res]).reshape(len(res), 3, -1)
    else:
        out = np.stack(res).reshape(len(res), -1)
    shp_k, shp_v = np.asarray(kcache_bits).shape, np.asarray(vcache_bits).shape
    ret = (kc.bits.reshape(shp_k), vc.bits.reshape(shp_v), round_f64_to_bits(out, dt), out)
    return ret + (sc,) if stats else ret
