"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test fixes one part of the oracle against something independent of it:
a library cast, complex multiplication, a trigonometric identity, a naive
contiguous attention written from the textbook definition, decomposed
multi-head latent attention, or a closed form. Sources: the
onnx-runtime-ep-cuda ``paged_attention.rs`` page (module doc "Write phase" /
"Read phase", ``rope_channel``, ``attn_impl``) and PR #1940's test list
("oracle == naive contiguous dense", "placement-invariance across a
permuted block table", "slot_mapping=-1 write suppression", "absorbed LATENT
== decomposed multi-head latent attention at tiny and 576/512/64 dims").
"""
import cmath
import math

import numpy as np
import pytest
import torch

from oracle import pa_oracle as O
from paged_latent_attention_cache_gb300 import workloads as W


def _params(**kw):
    p = dict(dtype="bf16", num_heads=2, head_size=32, v_head_size=16, rotary_offset=16,
             rotary_dim=16, rotary_interleaved=0, cos_rows=64, block_size=16,
             num_blocks=8, max_blocks_per_seq=4, scale=0.2, softcap=0.0,
             local_window_size=-1)
    p.update(kw)
    return p


def _exact_tables(rows, rd, theta=10000.0):
    """float64 cos/sin tables (not rounded to any dtype)."""
    half = rd // 2
    ang = np.arange(rows)[:, None] * theta ** (-2.0 * np.arange(half)[None, :] / rd)
    return np.cos(ang), np.sin(ang), ang


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch_cast():
    """float32 inputs (exact in float64): the oracle's direct rounding must
    equal torch's float32 -> bfloat16 round-to-nearest-even cast, including
    exact ties, subnormals and overflow."""
    rng = np.random.default_rng(0)
    with np.errstate(over="ignore"):
        big = (rng.standard_normal(5000) * 3e38).astype(np.float32)   # near/over max
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),    # subnormal range
        big,
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.40e38], dtype=np.float32),
    ])
    # exact ties: a bf16 value plus half a bf16 spacing
    base = rng.standard_normal(4000).astype(np.float32)
    bb = (base.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = np.concatenate([x, bb.view(np.float32)])
    ours = O.round_f64_to_bits(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_f16_matches_numpy_cast():
    """float64 inputs: numpy's float64 -> float16 cast rounds directly from
    double (ties to even); the oracle must agree bit for bit."""
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000),
        rng.standard_normal(5000) * 1e-6,         # f16 subnormals
        rng.standard_normal(5000) * 7e4,          # overflow region
        np.array([65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 0.0]),
    ])
    ours = O.round_f64_to_bits(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("interleaved", [0, 1])
def test_rope_is_complex_rotation(interleaved):
    """Each rotary pair (a, b) maps to the complex product
    (a + ib) * exp(i * pos * theta^(-2k/rd)): real part to a's channel,
    imaginary part to b's channel. Channels outside the suffix are
    unchanged."""
    rng = np.random.default_rng(2)
    hs, ro, rd = 48, 16, 32
    cos_t, sin_t, ang = _exact_tables(100, rd)
    for pos in (0, 1, 7, 99):
        x = rng.standard_normal(hs)
        y = O.rope_row(x, pos, ro, rd, cos_t, sin_t, bool(interleaved))
        assert np.array_equal(y[:ro], x[:ro]) and np.array_equal(y[ro + rd:], x[ro + rd:])
        for k in range(rd // 2):
            ia, ib = (ro + 2 * k, ro + 2 * k + 1) if interleaved else (ro + k, ro + k + rd // 2)
            z = complex(x[ia], x[ib]) * cmath.exp(1j * ang[pos, k])
            assert abs(y[ia] - z.real) < 1e-12 and abs(y[ib] - z.imag) < 1e-12


@pytest.mark.parametrize("interleaved", [0, 1])
def test_rope_relative_position(interleaved):
    """<R(m) q, R(n) k> = <R(m-n) q, k>: the rotary score depends only on the
    relative position (requires exact angle tables and consistent pairing)."""
    rng = np.random.default_rng(3)
    hs, ro, rd = 32, 0, 32
    cos_t, sin_t, _ = _exact_tables(200, rd)
    q, k = rng.standard_normal(hs), rng.standard_normal(hs)
    for m, n in [(5, 2), (150, 3), (77, 77), (199, 0)]:
        lhs = O.rope_row(q, m, ro, rd, cos_t, sin_t, bool(interleaved)) @ \
            O.rope_row(k, n, ro, rd, cos_t, sin_t, bool(interleaved))
        rhs = O.rope_row(q, m - n, ro, rd, cos_t, sin_t, bool(interleaved)) @ k
        assert abs(lhs - rhs) < 1e-10


def test_rope_identity_cases():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(64)
    cos_t, sin_t, _ = _exact_tables(10, 16)
    assert np.array_equal(O.rope_row(x, 3, 8, 0, cos_t, sin_t, False), x)     # rd = 0
    assert np.array_equal(O.rope_row(x, 0, 8, 16, cos_t, sin_t, False), x)    # pos 0
    y = O.rope_row(x, 9, 8, 16, cos_t, sin_t, False)
    # pair norms are preserved
    a, b = x[8:16], x[16:24]
    ya, yb = y[8:16], y[16:24]
    assert np.allclose(a * a + b * b, ya * ya + yb * yb, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Attention against a naive contiguous dense attention
# ---------------------------------------------------------------------------

def _paged_from_contiguous(rng, past_lens, q_lens, p, drop=()):
    """Build a paged problem from per-sequence contiguous past rows: the
    test itself scatters rows into a randomly permuted pool."""
    hs, H, bs = p["head_size"], p["num_heads"], p["block_size"]
    B = len(past_lens)
    ctx = [a + b for a, b in zip(past_lens, q_lens)]
    nblk = [(c + bs - 1) // bs for c in ctx]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb)
    bt = -np.ones((B, max(nblk)), dtype=np.int64)
    off = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += nblk[b]
    pool = rng.standard_normal((nb * bs, hs))         # garbage everywhere
    past_rows = [rng.standard_normal((n, hs)) for n in past_lens]
    for b in range(B):
        for j in range(past_lens[b]):
            pool[bt[b, j // bs] * bs + j % bs] = past_rows[b][j]
    T = sum(q_lens)
    cumseq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
    past = np.array(past_lens)
    slots, t = np.zeros(T, dtype=np.int64), 0
    for b in range(B):
        for i in range(q_lens[b]):
            pos = past_lens[b] + i
            slots[t] = bt[b, pos // bs] * bs + pos % bs
            t += 1
    for t in drop:
        slots[t] = -1
    key = rng.standard_normal((T, hs))
    query = rng.standard_normal((T, H * hs))
    p = dict(p, num_blocks=nb, max_blocks_per_seq=bt.shape[1])
    return dict(pool=pool, bt=bt, cumseq=cumseq, past=past, slots=slots, key=key,
                query=query, past_rows=past_rows, p=p)


def _naive_rope(x, pos, ro, rd, ang):
    """RoPE through complex multiplication (non-interleaved pairing)."""
    y = list(x)
    for k in range(rd // 2):
        z = complex(x[ro + k], x[ro + k + rd // 2]) * cmath.exp(1j * ang[pos, k])
        y[ro + k], y[ro + k + rd // 2] = z.real, z.imag
    return y


def _naive_dense(prob, ang):
    """Textbook causal attention per sequence over a contiguous [ctx, hs]
    key matrix (past rows followed by the rotated new rows), with a full
    masked score matrix and pure-Python exp/sum."""
    p = prob["p"]
    hs, vhs, H = p["head_size"], p["v_head_size"], p["num_heads"]
    ro, rd, win = p["rotary_offset"], p["rotary_dim"], p["local_window_size"]
    outs = []
    t = 0
    for b, P in enumerate(prob["past"]):
        L = int(prob["cumseq"][b + 1] - prob["cumseq"][b])
        K = [list(r) for r in prob["past_rows"][b]]
        for i in range(L):
            K.append(_naive_rope(prob["key"][t + i], P + i, ro, rd, ang))
        for i in range(L):
            pos = P + i
            o = np.zeros((H, vhs))
            for h in range(H):
                q = _naive_rope(prob["query"][t + i][h * hs:(h + 1) * hs], pos, ro, rd, ang)
                mask = [j <= pos and (win < 0 or pos - j <= win) for j in range(len(K))]
                sc = [sum(q[d] * K[j][d] for d in range(hs)) * p["scale"] if mask[j] else None
                      for j in range(len(K))]
                if p["softcap"] > 0:
                    sc = [None if s is None else p["softcap"] * math.tanh(s / p["softcap"])
                          for s in sc]
                mx = max(s for s in sc if s is not None)
                e = [0.0 if s is None else math.exp(s - mx) for s in sc]
                den = sum(e)
                for d in range(vhs):
                    o[h, d] = sum(e[j] * K[j][d] for j in range(len(K))) / den
            outs.append(o)
        t += L
    return np.stack(outs)


@pytest.mark.parametrize("softcap,window", [(0.0, -1), (1.5, -1), (0.0, 3), (2.0, 0)])
def test_attention_matches_naive_contiguous(softcap, window):
    rng = np.random.default_rng(5)
    p = _params(softcap=softcap, local_window_size=window, num_heads=3, head_size=32,
                v_head_size=24, rotary_offset=16, rotary_dim=16, block_size=4)
    prob = _paged_from_contiguous(rng, past_lens=[5, 0, 9], q_lens=[3, 4, 1], p=p)
    cos_t, sin_t, ang = _exact_tables(64, p["rotary_dim"])
    cache = O.latent_write(prob["key"], cos_t, sin_t, prob["slots"], prob["cumseq"],
                           prob["past"], O.F64Cache(prob["pool"]), prob["p"])
    ours = O.latent_attend(prob["query"], cache, cos_t, sin_t, prob["cumseq"],
                           prob["past"], prob["bt"], prob["p"])
    ref = _naive_dense(prob, ang)
    assert np.max(np.abs(ours - ref)) < 1e-12


# ---------------------------------------------------------------------------
# Absorbed latent attention == decomposed multi-head latent attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("c,dn,dv,dr,H", [(128, 32, 32, 64, 3), (512, 128, 128, 64, 4)])
def test_absorbed_equals_decomposed_mla(c, dn, dv, dr, H):
    """Per head h: k_hj = W_UK[h] c_j, v_hj = W_UV[h] c_j and
    score = q_nope . k_hj + rope(q_pe) . rope(k_pe_j). Feeding the oracle the
    absorbed query [W_UK[h]^T q_nope ; q_pe] and latent key [c_j ; k_pe_j]
    (rotary suffix at offset c) must give W_UV[h] o_lat = o_h."""
    rng = np.random.default_rng(6)
    past_lens, q_lens = [6, 2], [2, 3]
    B, T = 2, 5
    hs = c + dr
    scale = 1.0 / math.sqrt(dn + dr)
    W_UK = rng.standard_normal((H, dn, c)) / math.sqrt(c)
    W_UV = rng.standard_normal((H, dv, c)) / math.sqrt(c)
    _, _, ang = _exact_tables(32, dr)
    cos_t, sin_t, _ = _exact_tables(32, dr)
    ctx = [a + b for a, b in zip(past_lens, q_lens)]
    lat = [rng.standard_normal((n, c)) for n in ctx]      # c_j per sequence
    kpe = [rng.standard_normal((n, dr)) for n in ctx]     # k_pe_j before RoPE
    q_nope = rng.standard_normal((T, H, dn))
    q_pe = rng.standard_normal((T, H, dr))

    def crope(x, pos):
        y = np.array(x, dtype=np.float64)
        h = dr // 2
        z = (x[:h] + 1j * x[h:]) * np.exp(1j * ang[pos, :h])
        y[:h], y[h:] = z.real, z.imag
        return y

    # decomposed reference
    ref = np.zeros((T, H, dv))
    t = 0
    for b in range(B):
        for i in range(q_lens[b]):
            pos = past_lens[b] + i
            for h in range(H):
                s = np.array([q_nope[t, h] @ (W_UK[h] @ lat[b][j]) +
                              crope(q_pe[t, h], pos) @ crope(kpe[b][j], j)
                              for j in range(pos + 1)]) * scale
                w = np.exp(s - s.max())
                w /= w.sum()
                ref[t, h] = sum(w[j] * (W_UV[h] @ lat[b][j]) for j in range(pos + 1))
            t += 1

    # absorbed problem through the oracle: past rows pre-rotated in the
    # cache (they were written by earlier steps), new rows written now.
    bs = 4
    nblk = [(n + bs - 1) // bs for n in ctx]
    bt = np.full((B, max(nblk)), -1)
    perm = rng.permutation(sum(nblk))
    bt[0, :nblk[0]] = perm[:nblk[0]]
    bt[1, :nblk[1]] = perm[nblk[0]:]
    pool = np.zeros((sum(nblk) * bs, hs))
    keys, queries, slots = np.zeros((T, hs)), np.zeros((T, H * hs)), np.zeros(T, dtype=int)
    t = 0
    for b in range(B):
        for j in range(past_lens[b]):
            pool[bt[b, j // bs] * bs + j % bs] = np.concatenate([lat[b][j], crope(kpe[b][j], j)])
        for i in range(q_lens[b]):
            j = past_lens[b] + i
            keys[t] = np.concatenate([lat[b][j], kpe[b][j]])
            slots[t] = bt[b, j // bs] * bs + j % bs
            for h in range(H):
                queries[t, h * hs:(h + 1) * hs] = np.concatenate([W_UK[h].T @ q_nope[t, h],
                                                                  q_pe[t, h]])
            t += 1
    cumseq = np.array([0, q_lens[0], T])
    p = _params(num_heads=H, head_size=hs, v_head_size=c, rotary_offset=c, rotary_dim=dr,
                block_size=bs, num_blocks=sum(nblk), max_blocks_per_seq=bt.shape[1],
                scale=scale, cos_rows=32)
    cache = O.latent_write(keys, cos_t, sin_t, slots, cumseq, np.array(past_lens),
                           O.F64Cache(pool), p)
    o_lat = O.latent_attend(queries, cache, cos_t, sin_t, cumseq, np.array(past_lens), bt, p)
    got = np.einsum("hvc,thc->thv", W_UV, o_lat)
    assert np.max(np.abs(got - ref)) < 1e-10


# ---------------------------------------------------------------------------
# Paging invariants on the bit-level operator
# ---------------------------------------------------------------------------

def _bits_problem(w):
    p = W.oracle_params(w)
    return dict(q=W.to_bits(w.query), k=W.to_bits(w.key), cache=W.to_bits(w.key_cache),
                cos=W.to_bits(w.cos_cache), sin=W.to_bits(w.sin_cache),
                cumseq=w.cumseq.numpy(), past=w.past.numpy(), bt=w.block_table.numpy(),
                slots=w.slot_mapping.numpy(), p=p)


def _run(b, tokens=None):
    return O.run_operator_bits(b["q"], b["k"], b["cache"], b["cos"], b["sin"], b["cumseq"],
                               b["past"], b["bt"], b["slots"], b["p"], tokens)


def _small(seed=7, dtype=torch.bfloat16, **kw):
    args = dict(q_lens=[1, 5, 3], past_lens=[17, 0, 30], dtype=dtype, num_heads=2,
                head_size=64, v_head_size=32, rotary_offset=32, rotary_dim=32,
                block_size=16, num_blocks=12, seed=seed, drop_slots=2)
    args.update(kw)
    return W.make_workload("small", **args)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_placement_invariance(dtype):
    """Moving every physical block to another place in the pool, with
    block_table and slot_mapping remapped, leaves the output bits unchanged."""
    w = _small(dtype=dtype)
    a = _bits_problem(w)
    rng = np.random.default_rng(8)
    nb, bs = w.num_blocks, w.block_size
    perm = rng.permutation(nb)                  # old block i -> new block perm[i]
    b = dict(a)
    cache = a["cache"].copy()
    cache[perm] = a["cache"]
    b["cache"] = cache
    bt = a["bt"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    b["bt"] = bt
    sl = a["slots"].copy()
    m = sl >= 0
    sl[m] = perm[sl[m] // bs] * bs + sl[m] % bs
    b["slots"] = sl
    ca, oa, _ = _run(a)
    cb, ob, _ = _run(b)
    assert np.array_equal(oa, ob)
    # new block perm[i] holds what old block i held
    assert np.array_equal(cb[perm], ca)


def test_slot_minus_one_leaves_cache_untouched():
    """Only rows named by a non-negative slot change; rows of dropped
    tokens keep their old bits."""
    w = _small()
    a = _bits_problem(w)
    new_cache, _, _ = _run(a)
    hs = w.head_size
    old = a["cache"].reshape(-1, hs)
    new = new_cache.reshape(-1, hs)
    written = set(int(s) for s in a["slots"] if s >= 0)
    changed = set(np.nonzero(np.any(old != new, axis=1))[0].tolist())
    assert changed <= written
    # the dropped tokens' home rows are untouched
    dropped = [t for t in range(len(a["slots"])) if a["slots"][t] < 0]
    assert dropped
    for t in dropped:
        b = int(np.searchsorted(a["cumseq"], t, side="right") - 1)
        pos = int(a["past"][b]) + t - int(a["cumseq"][b])
        row = int(a["bt"][b, pos // w.block_size]) * w.block_size + pos % w.block_size
        assert np.array_equal(old[row], new[row])


def test_no_rotary_write_is_a_byte_copy():
    w = _small(rotary_dim=0, rotary_offset=0)
    a = _bits_problem(w)
    new_cache, _, _ = _run(a)
    new = new_cache.reshape(-1, w.head_size)
    for t, s in enumerate(a["slots"]):
        if s >= 0:
            assert np.array_equal(new[s], a["k"][t])


def test_non_rotary_channels_copied_exactly():
    w = _small()
    a = _bits_problem(w)
    new = _run(a)[0].reshape(-1, w.head_size)
    ro, rd = w.rotary_offset, w.rotary_dim
    for t, s in enumerate(a["slots"]):
        if s >= 0:
            assert np.array_equal(new[s, :ro], a["k"][t, :ro])
            assert np.array_equal(new[s, ro + rd:], a["k"][t, ro + rd:])


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_single_visible_key_returns_its_value_row():
    """window = 0 (and any token at position 0) sees only its own key: the
    output is that cache row's leading v_head_size channels, exactly."""
    w = _small(local_window_size=0)
    a = _bits_problem(w)
    cache, out, _ = _run(a)
    cache = cache.reshape(-1, w.head_size)
    H, vhs = w.num_heads, w.v_head_size
    for t in range(w.num_tokens):
        b = int(np.searchsorted(a["cumseq"], t, side="right") - 1)
        pos = int(a["past"][b]) + t - int(a["cumseq"][b])
        row = int(a["bt"][b, pos // w.block_size]) * w.block_size + pos % w.block_size
        for h in range(H):
            assert np.array_equal(out[t, h * vhs:(h + 1) * vhs], cache[row, :vhs])


def test_equal_keys_give_that_value():
    w = _small(rotary_dim=0, rotary_offset=0)
    a = _bits_problem(w)
    row = a["cache"].reshape(-1, w.head_size)[0].copy()
    a["cache"] = np.broadcast_to(row, a["cache"].reshape(-1, w.head_size).shape).copy() \
        .reshape(a["cache"].shape)
    a["k"] = np.broadcast_to(row, a["k"].shape).copy()
    _, out, _ = _run(a)
    for h in range(w.num_heads):
        assert np.all(out[:, h * w.v_head_size:(h + 1) * w.v_head_size] ==
                      row[:w.v_head_size][None, :])


def test_window_covering_context_is_no_window():
    a = _bits_problem(_small(local_window_size=-1))
    b = _bits_problem(_small(local_window_size=10 ** 6))
    assert np.array_equal(_run(a)[1], _run(b)[1])


def test_huge_softcap_is_no_softcap():
    a = _bits_problem(_small())
    b = _bits_problem(_small(softcap=1e9))
    fa, fb = _run(a)[2], _run(b)[2]
    assert np.max(np.abs(fa - fb)) < 1e-9


def test_two_key_softcap_closed_form():
    """One head, no RoPE, query e0*4, scale 1/4: the scores are the keys'
    channel 0. Keys (1, 1) and (3, -1) under softcap 2 give weights
    1/(1+e^{d}) and e^{d}/(1+e^{d}) with d = 2tanh(3/2) - 2tanh(1/2)."""
    hs = 16
    q = np.zeros((1, hs)); q[0, 0] = 4.0
    pool = np.zeros((16, hs)); pool[5, 0], pool[5, 1] = 1.0, 1.0   # key 0 at slot 5
    key = np.zeros((1, hs)); key[0, 0], key[0, 1] = 3.0, -1.0       # key 1, new
    p = _params(num_heads=1, head_size=hs, v_head_size=hs, rotary_offset=0, rotary_dim=0,
                block_size=16, num_blocks=1, max_blocks_per_seq=1, scale=0.25, softcap=2.0)
    # slot = 0*16 + 1 for position 1; the past row sits at position 0 -> slot 0
    pool[0] = pool[5]
    cache = O.latent_write(key, None, None, np.array([1]), np.array([0, 1]),
                           np.array([1]), O.F64Cache(pool), p)
    out = O.latent_attend(q, cache, None, None, np.array([0, 1]), np.array([1]),
                          np.array([[0]]), p)[0, 0]
    d = 2 * math.tanh(1.5) - 2 * math.tanh(0.5)
    w1 = math.exp(d) / (1 + math.exp(d))
    w0 = 1 - w1
    assert abs(out[0] - (w0 * 1 + w1 * 3)) < 1e-14
    assert abs(out[1] - (w0 * 1 - w1 * 1)) < 1e-14
    assert np.all(out[2:] == 0)


# ---------------------------------------------------------------------------
# error_scales: the tolerance helper of the parity tests (not the operator)
# ---------------------------------------------------------------------------

def _textbook_attention(q, K, scale, vhs, s_extra=None):
    """softmax(scale * q K^T (+ s_extra)) @ K[:, :vhs], normalised; written
    from the definition, independent of the oracle."""
    s = scale * (q @ K.T)
    if s_extra is not None:
        s = s + s_extra
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w @ K[:, :vhs]) / w.sum(axis=1, keepdims=True), w / w.sum(axis=1, keepdims=True)


def _scales_case(seed=0, H=3, n=40, hs=32, vhs=16, scale=0.3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((H, hs))
    K = rng.standard_normal((n, hs))
    out, prob = _textbook_attention(q, K, scale, vhs)
    return q, K, prob, out, scale, vhs


def test_error_scales_single_key():
    """One key: the output is that key's value row; only the probability
    term is left, equal to |V|."""
    rng = np.random.default_rng(3)
    q, K = rng.standard_normal((2, 24)), rng.standard_normal((1, 24))
    prob = np.ones((2, 1))
    out = np.repeat(K[:, :8], 2, axis=0)
    sc = O.error_scales(q, K, prob, out, 0.4, 8)
    assert np.allclose(sc[0], np.abs(out), rtol=0, atol=1e-15)
    # (the square roots of cancelling sums: zero to about sqrt(eps))
    assert np.allclose(sc[1], 0.0, atol=1e-6) and np.allclose(sc[2], 0.0, atol=1e-12)


def test_error_scales_equal_probabilities():
    """q = 0 gives equal probabilities 1/n; with |V_jc| = a the probability
    term is a / sqrt(n), and nothing depends on the scores."""
    rng = np.random.default_rng(4)
    n, a = 50, 0.75
    K = a * np.sign(rng.standard_normal((n, 16)))
    q = np.zeros((2, 16))
    out, prob = _textbook_attention(q, K, 0.5, 8)
    sc = O.error_scales(q, K, prob, out, 0.5, 8)
    assert np.allclose(sc[0], a / math.sqrt(n), rtol=1e-12)
    assert np.allclose(sc[1], 0.0) and np.allclose(sc[2], 0.0)


def test_error_scales_probability_term_monte_carlo():
    """Multiplying each probability by an independent (1 + sigma e_j),
    e ~ N(0, 1), moves the output by sigma * n_p in standard deviation."""
    q, K, prob, out, scale, vhs = _scales_case(5)
    sc = O.error_scales(q, K, prob, out, scale, vhs)
    rng = np.random.default_rng(6)
    trials, sigma = 4000, 1e-3
    e = rng.standard_normal((trials,) + prob.shape)
    d = np.einsum("thj,jc->thc", prob[None] * sigma * e, K[:, :vhs]) / sigma
    assert np.allclose(d.std(axis=0), sc[0], rtol=0.06)


def test_error_scales_score_term_monte_carlo():
    """Perturbing score j by an independent sigma * g_j * e_j, with
    g_j = scale * sqrt(sum_d q_d^2 K_jd^2), moves the softmax output by
    sigma * n_q in standard deviation (first order)."""
    q, K, prob, out, scale, vhs = _scales_case(7)
    sc = O.error_scales(q, K, prob, out, scale, vhs)
    g = scale * np.sqrt((q * q) @ (K * K).T)
    rng = np.random.default_rng(8)
    trials, sigma = 3000, 1e-5
    d = np.stack([(_textbook_attention(q, K, scale, vhs,
                                       sigma * g * rng.standard_normal(g.shape))[0] - out)
                  / sigma for _ in range(trials)])
    assert np.allclose(d.std(axis=0), sc[1], rtol=0.06)


def test_error_scales_diagonal_term_is_a_derivative():
    """Scaling query channel c by (1 + eps) moves output channel c by
    eps * n_d (query channel c meets value channel c in every score)."""
    q, K, prob, out, scale, vhs = _scales_case(9)
    sc = O.error_scales(q, K, prob, out, scale, vhs)
    eps = 1e-6
    for h in range(q.shape[0]):
        for c in range(vhs):
            qp, qm = q.copy(), q.copy()
            qp[h, c] *= 1 + eps
            qm[h, c] *= 1 - eps
            d = (_textbook_attention(qp, K, scale, vhs)[0][h, c] -
                 _textbook_attention(qm, K, scale, vhs)[0][h, c]) / (2 * eps)
            assert abs(abs(d) - sc[2, h, c]) <= 1e-6 * max(1.0, sc[2, h, c])


def test_stats_leave_the_result_unchanged():
    """The statistics variant returns the same output as the plain read."""
    w = W.tiny()
    p = W.oracle_params(w)
    dt = p["dtype"]
    cache = O.BitsCache(W.to_bits(w.key_cache).reshape(-1, w.head_size), dt)
    cos_t, sin_t = O.bits_to_f64(W.to_bits(w.cos_cache), dt), O.bits_to_f64(W.to_bits(w.sin_cache), dt)
    q = O.bits_to_f64(W.to_bits(w.query), dt)
    args = (cache, cos_t, sin_t, w.cumseq.numpy(), w.past.numpy(), w.block_table.numpy(), p)
    plain = O.latent_attend(q, *args)
    out, sc = O.latent_attend(q, *args, stats=True)
    assert np.array_equal(plain, out)
    assert sc.shape == (w.num_tokens, 3, w.num_heads, w.v_head_size) and (sc >= 0).all()


# ---------------------------------------------------------------------------
# FP8 (E4M3) latent cache
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch():
    """All 256 codes decode to torch's float8_e4m3fn values (NaN codes too)."""
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_rounding_matches_torch_cast_in_range():
    """float32 inputs up to the saturation point: the codes equal torch's
    float32 -> float8_e4m3fn cast (round to nearest, ties to even),
    including exact ties and subnormals."""
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000) * 20, rng.standard_normal(5000) * 1e-2,
                        rng.uniform(-464, 464, 5000)])
    vals = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    vals = np.sort(vals[np.isfinite(vals)])
    mids = (vals[1:] + vals[:-1]) / 2                     # exact ties
    x = np.concatenate([x, mids, -mids, [0.0, -0.0, 464.0, -464.0]]).astype(np.float32)
    ours = O.round_to_e4m3(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_rounding_is_nearest_by_brute_force():
    """Each code is the finite E4M3 value nearest to x (ties: even mantissa),
    found by comparing against all 254 finite values."""
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(3000) * 30, rng.standard_normal(1000) * 0.01])
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_to_f64(codes)
    fin = np.isfinite(vals)
    got = O.round_to_e4m3(x)
    for xi, ci in zip(x, got):
        d = np.abs(vals[fin] - xi)
        best = codes[fin][d == d.min()]
        if len(best) > 1:   # a tie: the even mantissa wins; the sign follows x
            best = best[(best & 1) == 0]
        best = best[np.signbit(O.e4m3_to_f64(best)) == np.signbit(xi)] if len(best) > 1 else best
        assert O.e4m3_to_f64(np.array([ci]))[0] == O.e4m3_to_f64(best[:1])[0], (xi, ci, best)


def test_e4m3_saturates_to_448():
    """Magnitudes at or beyond 448 give the largest finite code, 0x7E (448)
    or 0xFE (-448); nothing becomes NaN."""
    x = np.array([448.0, 460.0, 464.0, 465.0, 1e6, 3e38, -465.0, -1e30])
    codes = O.round_to_e4m3(x)
    assert codes.tolist() == [0x7E] * 6 + [0xFE] * 2


def test_fp8_write_is_exact_for_representable_rows():
    """Without rotation, a key row whose values are k_scale times E4M3
    values is stored as exactly those codes."""
    rng = np.random.default_rng(13)
    k_scale = 2.0 ** -6
    codes = rng.integers(0, 256, size=(3, 32)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11                      # no NaN codes
    rows = O.e4m3_to_f64(codes) * k_scale
    p = _params(rotary_dim=0, rotary_offset=0, cache_dtype=O.E4M3, k_scale=k_scale)
    cache = O.E4M3Cache(np.zeros((8 * 16, 32), np.uint8), k_scale)
    cumseq, past = np.array([0, 3]), np.array([0])
    O.latent_write(rows, None, None, np.array([5, 17, 40]), cumseq, past, cache, p)
    assert np.array_equal(cache.codes[[5, 17, 40]], codes)


def test_fp8_read_equals_plain_read_of_dequantized_cache():
    """The FP8 operator equals the plain operator run on a cache holding the
    dequantized values (exact in bf16 for k_scale = 2^-6): dequantization is
    code * k_scale and nothing else changes in the read phase."""
    rng = np.random.default_rng(14)
    k_scale = 2.0 ** -6
    codes = (rng.integers(0, 2, (8 * 16, 32)) << 7 | rng.integers(8, 14, (8 * 16, 32)) << 3 |
             rng.integers(0, 8, (8 * 16, 32))).astype(np.uint8)
    T, H = 5, 2
    q = rng.standard_normal((T, H * 32)) * 0.5
    cumseq, past = np.array([0, 2, 5]), np.array([17, 30])
    bt = rng.permutation(8).reshape(2, 4)
    cos_t, sin_t, _ = _exact_tables(64, 16)
    p8 = _params(cache_dtype=O.E4M3, k_scale=k_scale)
    pb = _params()
    fp8 = O.latent_attend(q, O.E4M3Cache(codes, k_scale), cos_t, sin_t, cumseq, past, bt, p8)
    plain = O.latent_attend(q, O.F64Cache(O.e4m3_to_f64(codes) * k_scale), cos_t, sin_t, cumseq,
                            past, bt, pb)
    assert np.array_equal(fp8, plain)
    # and the dequantized values are bf16 values (a bf16 cache would hold them exactly)
    vals = O.e4m3_to_f64(codes) * k_scale
    assert np.array_equal(O.round_f64(vals, "bf16"), vals)


def test_fp8_quantization_divides_by_k_scale_in_float32():
    """The stored code of value v is round_to_e4m3(f32(f32(v) / f32(k_scale)))."""
    rng = np.random.default_rng(15)
    v = rng.standard_normal(4000) * 0.5
    k = 0.0123
    got = O.quantize_e4m3(v, k)
    q = (v.astype(np.float32) / np.float32(k)).astype(np.float64)
    vals = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    # the decoded code is within half a spacing of f32(v)/k (nearest value)
    dec = O.e4m3_to_f64(got)
    spacing = np.ldexp(1.0, (np.maximum(np.floor(np.log2(np.abs(q) + 1e-300)), -6) - 3)
                       .astype(np.int64))
    assert np.all(np.abs(dec - q) <= spacing / 2 + 1e-12)
    assert np.isfinite(vals[got]).all()


# ---------------------------------------------------------------------------
# SEPARATE layout (grouped-query attention, head sink, q/k RMSNorm)
# ---------------------------------------------------------------------------

def _sep_params(**kw):
    p = dict(dtype="bf16", num_heads=4, kv_num_heads=2, head_size=32, v_head_size=32,
             rotary_offset=0, rotary_dim=16, rotary_interleaved=0, cos_rows=64, block_size=16,
             num_blocks=8, max_blocks_per_seq=4, scale=0.2, softcap=0.0, local_window_size=-1,
             rms_eps=1e-6)
    p.update(kw)
    return p


def _complex_rope(x, pos, rd, theta=10000.0):
    """Half-split RoPE of x's first rd channels as a complex rotation (float64)."""
    half = rd // 2
    ang = pos * theta ** (-2.0 * np.arange(half) / rd)
    z = (x[:half] + 1j * x[half:rd]) * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag, x[rd:]])


def _sep_case(seed, **kw):
    from paged_latent_attention_cache_gb300 import workloads as W
    w = W.make_separate_workload("pin", q_lens=[1, 6, 3], past_lens=[21, 4, 30], block_size=16,
                                 seed=seed, cos_rows=64, **kw)
    p = W.separate_oracle_params(w)
    return w, p


def _naive_separate(w, p):
    """Per sequence: contiguous keys/values (cached rows below the sequence's
    past, new rows from the inputs: RMSNorm by torch, RoPE as a complex
    rotation with exact angles, rounded to bf16 by torch), then per query
    head a softmax over the visible keys and the sink logit."""
    from paged_latent_attention_cache_gb300 import workloads as W
    dt = torch.bfloat16
    f = lambda t: t.to(torch.float64).numpy()
    H, kvh, hs, vhs, bs = w.num_heads, w.kv_num_heads, w.head_size, w.v_head_size, w.block_size
    grp = H // kvh
    kc = f(w.key_cache).reshape(-1, kvh, hs)
    vc = f(w.value_cache).reshape(-1, kvh, vhs)
    out = []
    cs = w.cumseq.tolist()
    for b in range(w.num_seqs):
        P, q = w.past_lens[b], w.q_lens[b]
        ctx = P + q
        Ks, Vs = np.zeros((ctx, kvh, hs)), np.zeros((ctx, kvh, vhs))
        for j in range(P):
            row = int(w.block_table[b, j // bs]) * bs + j % bs
            Ks[j], Vs[j] = kc[row], vc[row]
        for i in range(q):
            t = cs[b] + i
            kt = w.key[t].view(kvh, hs).to(torch.float32)
            if w.k_norm_weight is not None:
                kt = torch.nn.functional.rms_norm(kt.double(), (hs,), w.k_norm_weight.double(),
                                                  eps=w.rms_eps)
            kt = kt.double().numpy()
            for g in range(kvh):
                r = _complex_rope(kt[g], P + i, w.rotary_dim)
                Ks[P + i, g] = torch.from_numpy(r).to(dt).double().numpy()
            Vs[P + i] = f(w.value[t].view(kvh, vhs))
        for i in range(q):
            t, pos = cs[b] + i, P + i
            lo = 0 if w.local_window_size < 0 else max(0, pos - w.local_window_size)
            o = np.zeros((H, vhs))
            for h in range(H):
                qh = w.query[t, h * hs:(h + 1) * hs].double()
                if w.q_norm_weight is not None:
                    qh = torch.nn.functional.rms_norm(qh, (hs,), w.q_norm_weight.double(),
                                                      eps=w.rms_eps)
                qh = _complex_rope(qh.numpy(), pos, w.rotary_dim)
                K, V = Ks[lo:pos + 1, h // grp], Vs[lo:pos + 1, h // grp]
                s = w.scale * (K @ qh)
                if w.softcap > 0:
                    s = w.softcap * np.tanh(s / w.softcap)
                z = [] if w.head_sink is None else [float(w.head_sink[h])]
                m = max([s.max()] + z)
                e = np.exp(s - m)
                o[h] = (e @ V) / (e.sum() + sum(np.exp(zz - m) for zz in z))
            out.append(o.reshape(-1))
    return np.stack(out)


def _sep_oracle(w, p, tokens=None, stats=False):
    from paged_latent_attention_cache_gb300 import workloads as W
    tb = W.to_bits
    return O.run_separate_bits(
        tb(w.query), tb(w.key), tb(w.value), tb(w.key_cache), tb(w.value_cache),
        _exact_bits(w.cos_cache), _exact_bits(w.sin_cache), w.cumseq.numpy(), w.past.numpy(),
        w.block_table.numpy(), w.slot_mapping.numpy(), p,
        None if w.head_sink is None else tb(w.head_sink),
        None if w.q_norm_weight is None else tb(w.q_norm_weight),
        None if w.k_norm_weight is None else tb(w.k_norm_weight), tokens, stats)


def _exact_bits(t):
    from paged_latent_attention_cache_gb300 import workloads as W
    return W.to_bits(t)


@pytest.mark.parametrize("kw", [
    dict(num_heads=4, kv_num_heads=2, head_size=32, rotary_dim=16),
    dict(num_heads=4, kv_num_heads=4, head_size=32, rotary_dim=32, head_sink=True),
    dict(num_heads=6, kv_num_heads=1, head_size=48, rotary_dim=32, qk_norm=True),
    dict(num_heads=8, kv_num_heads=2, head_size=64, rotary_dim=64, head_sink=True, qk_norm=True,
         softcap=2.0, local_window_size=5),
], ids=["gqa", "mha_sink", "mqa_norm", "all_options"])
def test_separate_matches_naive_dense(kw):
    """The SEPARATE oracle equals a naive per-sequence contiguous attention
    written from the definitions (torch RMSNorm, complex RoPE with exact
    angles: the tolerance covers the cos/sin tables' bf16 rounding)."""
    w, p = _sep_case(41, **kw)
    # exact angles in the naive form; the oracle reads the bf16 tables
    got = _sep_oracle(w, p)[3]
    ref = _naive_separate(w, p)
    assert np.abs(got - ref).max() < 2e-2 * max(1.0, np.abs(ref).max())
    # with exact float64 tables the two agree to rounding of the stored keys
    p64 = dict(p)
    w64 = w
    cos, sin, _ = _exact_tables(w.cos_rows, w.rotary_dim)
    kc, vc = (O.BitsCache(W_bits(w.key_cache).reshape(-1, w.head_size), "bf16"),
              O.BitsCache(W_bits(w.value_cache).reshape(-1, w.v_head_size), "bf16"))
    f = lambda t: O.bits_to_f64(W_bits(t), "bf16")
    kn = None if w.k_norm_weight is None else f(w.k_norm_weight)
    qn = None if w.q_norm_weight is None else f(w.q_norm_weight)
    sink = None if w.head_sink is None else f(w.head_sink)
    O.separate_write(lambda t: f(w.key)[t].reshape(w.kv_num_heads, -1),
                     lambda t: f(w.value)[t].reshape(w.kv_num_heads, -1), cos, sin,
                     w.slot_mapping.numpy(), w.cumseq.numpy(), w.past.numpy(), kc, vc, p64, kn)
    q = f(w.query)
    exact = np.stack([O.separate_attend_token(t, q[t], kc, vc, cos, sin, w.cumseq.numpy(),
                                              w.past.numpy(), w.block_table.numpy(), p64, sink,
                                              qn).reshape(-1) for t in range(w.num_tokens)])
    assert np.abs(exact - ref).max() < 1e-9 + 4e-3 * np.abs(ref).max()


def W_bits(t):
    from paged_latent_attention_cache_gb300 import workloads as W
    return W.to_bits(t)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((7, 64)) * 3
    w = rng.standard_normal(64)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w),
                                       eps=1e-6).numpy()
    assert np.allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_head_sink_closed_forms():
    """One visible key with score s and sink z: out = V * e^s / (e^s + e^z);
    a sink of -inf-like size changes nothing; a huge sink sends the output
    to zero."""
    p = _sep_params(num_heads=2, kv_num_heads=1, rotary_dim=0, head_size=16, v_head_size=16,
                    block_size=16, num_blocks=1, max_blocks_per_seq=1, scale=0.5)
    rng = np.random.default_rng(43)
    K = rng.standard_normal((16, 16))
    V = rng.standard_normal((16, 16))
    kc, vc = O.F64Cache(K), O.F64Cache(V)
    q = rng.standard_normal(32)
    args = (kc, vc, None, None, np.array([0, 1]), np.array([0]), np.array([[0]]), p)
    for z in (-0.7, 1.3):
        out = O.separate_attend_token(0, q, *args, head_sink=np.array([z, z]))
        for h in range(2):
            s = 0.5 * q[h * 16:(h + 1) * 16] @ K[0]
            assert np.allclose(out[h], V[0] * np.exp(s) / (np.exp(s) + np.exp(z)), rtol=1e-12)
    plain = O.separate_attend_token(0, q, *args)
    assert np.allclose(O.separate_attend_token(0, q, *args, head_sink=np.array([-1e4, -1e4])),
                       plain, rtol=1e-12)
    assert np.abs(O.separate_attend_token(0, q, *args, head_sink=np.array([1e4, 1e4]))).max() == 0


def test_separate_reduces_to_latent():
    """One kv head, values equal to the keys, no rotation, no norm, no sink:
    the SEPARATE read equals the LATENT read with v_head_size == head_size."""
    rng = np.random.default_rng(44)
    rows = rng.standard_normal((8 * 16, 32))
    q = rng.standard_normal((5, 4 * 32))
    cumseq, past, bt = np.array([0, 2, 5]), np.array([17, 30]), rng.permutation(8).reshape(2, 4)
    ps = _sep_params(kv_num_heads=1, rotary_dim=0)
    pl = _params(rotary_dim=0, rotary_offset=0, v_head_size=32, num_heads=4)
    sep = np.stack([O.separate_attend_token(t, q[t], O.F64Cache(rows), O.F64Cache(rows), None,
                                            None, cumseq, past, bt, ps) for t in range(5)])
    lat = O.latent_attend(q, O.F64Cache(rows), None, None, cumseq, past, bt, pl)
    assert np.allclose(sep, lat, rtol=1e-12, atol=1e-14)


def test_separate_placement_invariance_and_slot_minus_one():
    """Permuting the physical blocks (block table and slots remapped) leaves
    the outputs bit-identical; slot -1 tokens leave both caches untouched."""
    w, p = _sep_case(45, num_heads=4, kv_num_heads=2, head_size=32, rotary_dim=16,
                     head_sink=True, qk_norm=True, drop_slots=2)
    kb, vb, ob, _ = _sep_oracle(w, p)
    nb, bs = w.num_blocks, w.block_size
    perm = np.random.default_rng(46).permutation(nb)
    inv = np.argsort(perm)
    w2 = copy_sep(w)
    w2.key_cache = w.key_cache[inv]
    w2.value_cache = w.value_cache[inv]
    bt = w.block_table.numpy().copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    w2.block_table = torch.from_numpy(bt)
    sl = w.slot_mapping.numpy().copy()
    ok = sl >= 0
    sl[ok] = perm[sl[ok] // bs] * bs + sl[ok] % bs
    w2.slot_mapping = torch.from_numpy(sl)
    kb2, vb2, ob2, _ = _sep_oracle(w2, p)
    assert np.array_equal(ob, ob2)
    skipped = w.slot_mapping.numpy()
    untouched = np.ones(nb * bs, bool)
    untouched[skipped[skipped >= 0]] = False
    kv = w.kv_num_heads
    assert np.array_equal(kb.reshape(nb * bs, -1)[untouched],
                          W_bits(w.key_cache).reshape(nb * bs, -1)[untouched])
    assert np.array_equal(vb.reshape(nb * bs, -1)[untouched],
                          W_bits(w.value_cache).reshape(nb * bs, -1)[untouched])


def copy_sep(w):
    from paged_latent_attention_cache_gb300 import workloads as W
    return W.SeparateWorkload(**{k: getattr(w, k) for k in w.__dataclass_fields__})
