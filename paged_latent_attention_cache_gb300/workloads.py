"""Seeded synthetic inputs for the paged LATENT attention operator.

This module only draws inputs: random latent rows, a pre-filled paged cache
pool, block tables, slot mappings, sequence offsets and the RoPE cos/sin
tables the operator takes as inputs. It performs none of the operator's own
arithmetic (no RoPE application, no scatter, no attention), so the CPU oracle
and the GPU path can both consume the same draw without sharing any of the
method's code.

Tensor layouts follow the operator schema of `com.microsoft::PagedAttention`
v1 in LATENT mode as the onnx-runtime-ep-cuda `paged_attention.rs` page
states it (schema input list in the PR #1978 review, "ORT v1.29 schema"):

* ``query``        ``[T, H*hs]``            f16/bf16
* ``key``          ``[T, hs]``              latent rows, same dtype
* ``key_cache``    ``[num_blocks, bs, 1, hs]`` paged latent cache, in the
  query dtype, or uint8 E4M3 codes with one ``k_scale`` for an FP8 cache
* ``cumseq``       int32 ``[B+1]``           ``cumulative_sequence_length``
* ``past``         int32 ``[B]``             ``past_seqlens`` (context - q_len)
* ``block_table``  int32 ``[B, max_blocks]`` physical block per logical block,
  padded with -1
* ``cos_cache``/``sin_cache`` ``[cos_rows, rd/2]`` in the query dtype
* ``slot_mapping`` int32 ``[T]``             ``block*bs + offset``, -1 = skip

Sequences are ordered decode-first: the first ``num_decode_seqs`` sequences
have exactly one new token each, so one ``decode`` call covers
``[0, num_decode_seqs)`` and one ``prefill`` call covers the rest.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import torch

ROPE_THETA = 10000.0


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_heads: int
    head_size: int
    v_head_size: int
    rotary_offset: int
    rotary_dim: int
    rotary_interleaved: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    cos_rows: int
    scale: float
    softcap: float
    local_window_size: int
    q_lens: List[int]
    past_lens: List[int]
    num_decode_seqs: int
    query: torch.Tensor
    key: torch.Tensor
    key_cache: torch.Tensor
    cos_cache: torch.Tensor
    sin_cache: torch.Tensor
    cumseq: torch.Tensor
    past: torch.Tensor
    block_table: torch.Tensor
    slot_mapping: torch.Tensor
    meta: Dict[str, object] = field(default_factory=dict)
    cache_dtype: Optional[str] = None   # None: the query dtype; "e4m3": FP8 codes
    k_scale: float = 1.0                # FP8 cache: value = code * k_scale

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    def params(self) -> Dict[str, object]:
        return dict(
            dtype=self.dtype, num_heads=self.num_heads, head_size=self.head_size,
            v_head_size=self.v_head_size, rotary_offset=self.rotary_offset,
            rotary_dim=self.rotary_dim, rotary_interleaved=self.rotary_interleaved,
            cos_rows=self.cos_rows, block_size=self.block_size,
            num_blocks=self.num_blocks, max_blocks_per_seq=self.max_blocks_per_seq,
            scale=self.scale, softcap=self.softcap,
            local_window_size=self.local_window_size, cache_dtype=self.cache_dtype,
            k_scale=self.k_scale)

    def to(self, device) -> "Workload":
        out = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("query", "key", "key_cache", "cos_cache", "sin_cache", "cumseq",
                  "past", "block_table", "slot_mapping"):
            setattr(out, k, getattr(self, k).to(device))
        out.meta = dict(self.meta)
        return out


def _normal(shape, gen: torch.Generator, std: float, dtype: torch.dtype,
            chunk: int = 1 << 26) -> torch.Tensor:
    """N(0, std^2) draw rounded to ``dtype``, generated in chunks so a
    multi-GB bf16 tensor never needs a same-size f32 intermediate."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=dtype)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = (torch.randn(hi - lo, generator=gen) * std).to(dtype)
    return out.view(*shape)


def _e4m3_codes(shape, gen: torch.Generator) -> torch.Tensor:
    """Seeded E4M3 cache contents (uint8 codes, drawn directly as bit
    fields): random sign, exponent field uniform in 8..13 (magnitudes 2 to
    120, about what N(0, 0.5^2) rows divided by k_scale = 1/64 span) and a
    random 3-bit mantissa. No code is NaN."""
    n = 1
    for s in shape:
        n *= int(s)
    sign = torch.randint(0, 2, (n,), generator=gen, dtype=torch.int32) << 7
    exp = torch.randint(8, 14, (n,), generator=gen, dtype=torch.int32) << 3
    man = torch.randint(0, 8, (n,), generator=gen, dtype=torch.int32)
    return (sign | exp | man).to(torch.uint8).view(*shape)


def rope_tables(cos_rows: int, rotary_dim: int, dtype: torch.dtype,
                theta: float = ROPE_THETA):
    """cos/sin input tables ``[cos_rows, rotary_dim/2]``: angle(p, i) =
    p * theta^(-2i/rotary_dim), evaluated in f64 and rounded to ``dtype``."""
    half = rotary_dim // 2
    if half == 0:
        z = torch.zeros(max(cos_rows, 1), 1, dtype=dtype)
        return z, z.clone()
    p = torch.arange(cos_rows, dtype=torch.float64)[:, None]
    i = torch.arange(half, dtype=torch.float64)[None, :]
    ang = p * torch.pow(torch.tensor(theta, dtype=torch.float64), -2.0 * i / rotary_dim)
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


def make_workload(name: str, q_lens: Sequence[int], past_lens: Sequence[int], *,
                  dtype=torch.bfloat16, num_heads: int, head_size: int,
                  v_head_size: int, rotary_offset: int, rotary_dim: int,
                  rotary_interleaved: int = 0, block_size: int,
                  num_blocks: Optional[int] = None,
                  max_blocks_per_seq: Optional[int] = None,
                  cos_rows: Optional[int] = None, scale: Optional[float] = None,
                  softcap: float = 0.0, local_window_size: int = -1,
                  seed: int = 0, std: float = 0.5, query_gain: float = 1.0,
                  drop_slots: int = 0, drop_frac: float = 0.0,
                  num_decode_seqs: Optional[int] = None,
                  block_table_shape: Optional[Sequence[int]] = None,
                  cache_dtype: Optional[str] = None, k_scale: float = 1.0 / 64) -> Workload:
    """Draw one seeded batch.

    ``drop_slots`` / ``drop_frac`` set that many (or that fraction of) seeded
    slot_mapping entries to -1. ``query_gain`` multiplies the drawn query
    (a power of two keeps the scaling exact) so that the logits spread over
    tens or hundreds and the softmax is peaked instead of near-uniform.
    ``block_table_shape`` lets a caller ask for a block table that is
    literally a permutation of the whole pool reshaped (the tiny
    configuration's wording). ``cache_dtype="e4m3"`` makes the cache an FP8
    one: the pool holds seeded E4M3 codes (``_e4m3_codes``) with one
    ``k_scale``; the keys stay in the query dtype (the write phase quantizes
    them)."""
    assert len(q_lens) == len(past_lens)
    gen = torch.Generator().manual_seed(seed)
    B = len(q_lens)
    ctx = [int(p) + int(q) for p, q in zip(past_lens, q_lens)]
    nblk = [(c + block_size - 1) // block_size for c in ctx]
    need = sum(nblk)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(nblk) if nblk else 1)
    if num_blocks is None:
        num_blocks = max(need, 1)
    assert num_blocks >= need, (num_blocks, need)
    T = sum(int(q) for q in q_lens)
    if cos_rows is None:
        cos_rows = max(max(ctx) if ctx else 1, 1)
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)

    # Physical placement: a seeded permutation of the pool, dealt to the
    # sequences in order.
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    block_table = torch.full((B, max_blocks_per_seq), -1, dtype=torch.int32)
    if block_table_shape is not None:
        bt = perm.view(*block_table_shape)
        assert bt.shape == block_table.shape
        block_table = bt.clone()
    else:
        off = 0
        for b in range(B):
            block_table[b, :nblk[b]] = perm[off:off + nblk[b]]
            off += nblk[b]

    cumseq = torch.zeros(B + 1, dtype=torch.int32)
    for b in range(B):
        cumseq[b + 1] = cumseq[b] + int(q_lens[b])
    past = torch.tensor([int(p) for p in past_lens], dtype=torch.int32)

    slot = torch.empty(T, dtype=torch.int32)
    t = 0
    for b in range(B):
        for i in range(int(q_lens[b])):
            pos = int(past_lens[b]) + i
            phys = int(block_table[b, pos // block_size])
            slot[t] = phys * block_size + pos % block_size
            t += 1
    n_drop = drop_slots + int(round(drop_frac * T))
    if n_drop > 0 and T > 0:
        idx = torch.randperm(T, generator=gen)[:min(n_drop, T)]
        slot[idx] = -1

    query = _normal((T, num_heads * head_size), gen, std, dtype)
    if query_gain != 1.0:
        query = (query.float() * query_gain).to(dtype)
    key = _normal((T, head_size), gen, std, dtype)
    if cache_dtype == "e4m3":
        key_cache = _e4m3_codes((num_blocks, block_size, 1, head_size), gen)
    else:
        assert cache_dtype is None, cache_dtype
        key_cache = _normal((num_blocks, block_size, 1, head_size), gen, std, dtype)
    cos, sin = rope_tables(cos_rows, rotary_dim, dtype)
    if num_decode_seqs is None:
        num_decode_seqs = 0
        for q in q_lens:
            if int(q) != 1:
                break
            num_decode_seqs += 1
    return Workload(name=name, dtype=dtype, num_heads=num_heads, head_size=head_size,
                    v_head_size=v_head_size, rotary_offset=rotary_offset,
                    rotary_dim=rotary_dim, rotary_interleaved=rotary_interleaved,
                    block_size=block_size, num_blocks=num_blocks,
                    max_blocks_per_seq=max_blocks_per_seq, cos_rows=cos_rows,
                    scale=float(scale), softcap=float(softcap),
                    local_window_size=int(local_window_size),
                    q_lens=[int(q) for q in q_lens], past_lens=[int(p) for p in past_lens],
                    num_decode_seqs=int(num_decode_seqs), query=query, key=key,
                    key_cache=key_cache, cos_cache=cos, sin_cache=sin, cumseq=cumseq,
                    past=past, block_table=block_table, slot_mapping=slot,
                    meta=dict(seed=seed, std=std, query_gain=query_gain),
                    cache_dtype=cache_dtype,
                    k_scale=float(k_scale) if cache_dtype is not None else 1.0)


# ---------------------------------------------------------------------------
# The five named workloads. Dimensions: GLM-style latent 192 / value 128 /
# rotary 64 at offset 128; DeepSeek-V3-style latent 576 / value 512 / rotary
# 64 at offset 512 with scale 1/sqrt(128+64).
# ---------------------------------------------------------------------------

GLM = dict(head_size=192, v_head_size=128, rotary_offset=128, rotary_dim=64)
DSV3 = dict(head_size=576, v_head_size=512, rotary_offset=512, rotary_dim=64)
DSV3_SCALE = 1.0 / math.sqrt(192.0)


def tiny(seed: int = 1, dtype=torch.bfloat16) -> Workload:
    """Tiny prefill+decode: 4 heads, GLM dims, bs=16, pasts {5,20} with
    {7,1} new tokens, a block table that is a permutation of 8 blocks and
    one slot set to -1. Sequences are stored decode-first: seq 0 is the
    (past 20, 1 new) decode, seq 1 the (past 5, 7 new) prefill."""
    return make_workload("tiny", q_lens=[1, 7], past_lens=[20, 5], dtype=dtype,
                         num_heads=4, **GLM, block_size=16, num_blocks=8,
                         max_blocks_per_seq=4, cos_rows=256,
                         scale=1.0 / math.sqrt(192.0), seed=seed, drop_slots=1,
                         block_table_shape=(2, 4))


def glm_decode(seed: int = 2, batch: int = 32, dtype=torch.bfloat16) -> Workload:
    """GLM-style dense MLA decode: H=64, batch 32, one new token per sequence,
    contexts uniform in [1024, 8192], bs=64, blocks dealt from a shuffled
    pool of 8192."""
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    ctx = torch.randint(1024, 8193, (batch,), generator=g).tolist()
    return make_workload("glm_decode", q_lens=[1] * batch, past_lens=[c - 1 for c in ctx],
                         dtype=dtype, num_heads=64, **GLM, block_size=64,
                         num_blocks=8192, max_blocks_per_seq=128, cos_rows=8192,
                         scale=1.0 / math.sqrt(192.0), seed=seed)


def dsv3_decode(seed: int = 3, batch: int = 64, context: int = 4096,
                dtype=torch.bfloat16) -> Workload:
    """DeepSeek-V3-style absorbed MLA decode: H=128, 576/512, batch 64,
    context 4096 each, bs=64, permuted block table."""
    nb = batch * ((context + 63) // 64)
    return make_workload("dsv3_decode", q_lens=[1] * batch,
                         past_lens=[context - 1] * batch, dtype=dtype, num_heads=128,
                         **DSV3, block_size=64, num_blocks=nb,
                         max_blocks_per_seq=(context + 63) // 64, cos_rows=context,
                         scale=DSV3_SCALE, seed=seed)


def dsv3_prefill(seed: int = 4, new_tokens: int = 4096,
                 pasts=(0, 0, 2048, 2048), dtype=torch.bfloat16) -> Workload:
    """DeepSeek-V3-style chunked prefill: H=128, 4 sequences of 4096 new
    tokens on top of pasts {0,0,2048,2048}, causal, bs=128."""
    ctx = [p + new_tokens for p in pasts]
    nb = sum((c + 127) // 128 for c in ctx)
    return make_workload("dsv3_prefill", q_lens=[new_tokens] * len(pasts),
                         past_lens=list(pasts), dtype=dtype, num_heads=128, **DSV3,
                         block_size=128, num_blocks=nb,
                         max_blocks_per_seq=max((c + 127) // 128 for c in ctx),
                         cos_rows=max(ctx), scale=DSV3_SCALE, seed=seed)


def mixed_serving(seed: int = 5, n_decode: int = 48, n_prefill: int = 4,
                  chunk: int = 512, dtype=torch.float16) -> Workload:
    """Mixed serving batch, fp16, GLM dims, H=64, bs=16: 48 decode sequences
    with contexts log-uniform in [128, 32768] and 4 prefill chunks of 512
    tokens with no past; window 4096, softcap 50, 5% of slots set to -1."""
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    u = torch.rand(n_decode, generator=g, dtype=torch.float64)
    ctx = torch.round(torch.exp(math.log(128) + u * (math.log(32768) - math.log(128))))
    ctx = ctx.to(torch.int64).tolist()
    q_lens = [1] * n_decode + [chunk] * n_prefill
    past = [c - 1 for c in ctx] + [0] * n_prefill
    need = sum((p + q + 15) // 16 for p, q in zip(past, q_lens))
    return make_workload("mixed_serving", q_lens=q_lens, past_lens=past, dtype=dtype,
                         num_heads=64, **GLM, block_size=16,
                         num_blocks=need + need // 8, max_blocks_per_seq=32768 // 16,
                         cos_rows=32768, scale=1.0 / math.sqrt(192.0), softcap=50.0,
                         local_window_size=4096, seed=seed, drop_frac=0.05,
                         num_decode_seqs=n_decode)


def peaked(w: Workload, gain: float) -> Workload:
    """A copy of ``w`` whose query is multiplied by ``gain`` (exact for a
    power of two in range): the logits spread over tens to thousands of
    units, so the softmax is peaked rather than near-uniform."""
    out = Workload(**{k: getattr(w, k) for k in w.__dataclass_fields__})
    out.query = (w.query.float() * gain).to(w.dtype)
    out.name = f"{w.name}_q{gain:g}"
    out.meta = dict(w.meta, query_gain=gain)
    return out


def dsv3_prefill_small(seed: int = 6, dtype=torch.bfloat16) -> Workload:
    """A quarter-size DeepSeek-V3-style chunked prefill (4 x 1024 new tokens
    on pasts {0,0,512,512}, bs=128): the same kernel as dsv3_prefill with
    about 1.2 GB on the device, small enough for a many-pass profiler
    capture."""
    w = dsv3_prefill(seed=seed, new_tokens=1024, pasts=(0, 0, 512, 512), dtype=dtype)
    w.name = "dsv3_prefill_small"
    return w


def glm_decode_fp8(seed: int = 7, batch: int = 32) -> Workload:
    """glm_decode's shape (contexts uniform in [1024, 8192]) with an FP8
    (E4M3) latent cache, k_scale = 1/64."""
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    ctx = torch.randint(1024, 8193, (batch,), generator=g).tolist()
    return make_workload("glm_decode_fp8", q_lens=[1] * batch, past_lens=[c - 1 for c in ctx],
                         num_heads=64, **GLM, block_size=64, num_blocks=8192,
                         max_blocks_per_seq=128, cos_rows=8192, scale=1.0 / math.sqrt(192.0),
                         seed=seed, cache_dtype="e4m3")


def dsv3_decode_fp8(seed: int = 8, batch: int = 64, context: int = 4096) -> Workload:
    """dsv3_decode's shape with an FP8 (E4M3) latent cache, k_scale = 1/64."""
    nb = batch * ((context + 63) // 64)
    return make_workload("dsv3_decode_fp8", q_lens=[1] * batch,
                         past_lens=[context - 1] * batch, num_heads=128, **DSV3,
                         block_size=64, num_blocks=nb, max_blocks_per_seq=(context + 63) // 64,
                         cos_rows=context, scale=DSV3_SCALE, seed=seed, cache_dtype="e4m3")


WORKLOADS = {
    "tiny": tiny,
    "glm_decode": glm_decode,
    "dsv3_decode": dsv3_decode,
    "dsv3_prefill": dsv3_prefill,
    "mixed_serving": mixed_serving,
    "dsv3_prefill_small": dsv3_prefill_small,
    "glm_decode_fp8": glm_decode_fp8,
    "dsv3_decode_fp8": dsv3_decode_fp8,
}


def to_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16/f16 tensor's bit patterns, or the uint8
    codes of an FP8 cache (a copy on the host when the tensor lives on a
    device)."""
    import numpy as np
    if t.dtype == torch.uint8:
        return t.detach().contiguous().cpu().numpy()
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def dtype_tag(dtype: torch.dtype) -> str:
    return {torch.bfloat16: "bf16", torch.float16: "f16"}[dtype]


def oracle_params(w: "Workload") -> Dict[str, object]:
    """The workload's operator parameters with the dtype as a tag string."""
    p = w.params()
    p["dtype"] = dtype_tag(w.dtype)
    if w.cache_dtype is None:
        p.pop("k_scale")
    return p


# ---------------------------------------------------------------------------
# SEPARATE layout (grouped-query attention over separate key / value caches)
# ---------------------------------------------------------------------------

@dataclass
class SeparateWorkload:
    """Inputs of the op's SEPARATE mode: query [T, H*hs], key [T, kvH*hs],
    value [T, kvH*vhs], key_cache [num_blocks, bs, kvH, hs], value_cache
    [num_blocks, bs, kvH, vhs], optional head_sink [H] (a sink logit per
    query head) and q/k RMSNorm weights [hs]; the index tensors as in
    ``Workload``."""
    name: str
    dtype: torch.dtype
    num_heads: int
    kv_num_heads: int
    head_size: int
    v_head_size: int
    rotary_offset: int
    rotary_dim: int
    rotary_interleaved: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    cos_rows: int
    scale: float
    softcap: float
    local_window_size: int
    rms_eps: float
    q_lens: List[int]
    past_lens: List[int]
    num_decode_seqs: int
    query: torch.Tensor
    key: torch.Tensor
    value: torch.Tensor
    key_cache: torch.Tensor
    value_cache: torch.Tensor
    cos_cache: torch.Tensor
    sin_cache: torch.Tensor
    cumseq: torch.Tensor
    past: torch.Tensor
    block_table: torch.Tensor
    slot_mapping: torch.Tensor
    head_sink: Optional[torch.Tensor] = None
    q_norm_weight: Optional[torch.Tensor] = None
    k_norm_weight: Optional[torch.Tensor] = None
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    def params(self) -> Dict[str, object]:
        return dict(dtype=self.dtype, num_heads=self.num_heads, kv_num_heads=self.kv_num_heads,
                    head_size=self.head_size, v_head_size=self.v_head_size,
                    rotary_offset=self.rotary_offset, rotary_dim=self.rotary_dim,
                    rotary_interleaved=self.rotary_interleaved, cos_rows=self.cos_rows,
                    block_size=self.block_size, num_blocks=self.num_blocks,
                    max_blocks_per_seq=self.max_blocks_per_seq, scale=self.scale,
                    softcap=self.softcap, local_window_size=self.local_window_size,
                    rms_eps=self.rms_eps)

    def to(self, device) -> "SeparateWorkload":
        out = SeparateWorkload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("query", "key", "value", "key_cache", "value_cache", "cos_cache", "sin_cache",
                  "cumseq", "past", "block_table", "slot_mapping", "head_sink", "q_norm_weight",
                  "k_norm_weight"):
            v = getattr(self, k)
            setattr(out, k, None if v is None else v.to(device))
        out.meta = dict(self.meta)
        return out


def make_separate_workload(name: str, q_lens: Sequence[int], past_lens: Sequence[int], *,
                           dtype=torch.bfloat16, num_heads: int, kv_num_heads: int,
                           head_size: int, v_head_size: Optional[int] = None,
                           rotary_offset: int = 0, rotary_dim: Optional[int] = None,
                           rotary_interleaved: int = 0, block_size: int,
                           num_blocks: Optional[int] = None,
                           max_blocks_per_seq: Optional[int] = None,
                           cos_rows: Optional[int] = None, scale: Optional[float] = None,
                           softcap: float = 0.0, local_window_size: int = -1,
                           rms_eps: float = 1e-6, head_sink: bool = False,
                           qk_norm: bool = False, seed: int = 0, std: float = 0.5,
                           drop_slots: int = 0, drop_frac: float = 0.0) -> SeparateWorkload:
    """Draw one seeded SEPARATE-layout batch: the block placement, offsets
    and slots as ``make_workload`` draws them; query/key/value and both
    cache pools N(0, std^2); sink logits N(0, 1) per query head; RMSNorm
    weights N(1, 0.2^2). Sequences with one new token come first."""
    base = make_workload(name, q_lens, past_lens, dtype=dtype, num_heads=num_heads,
                         head_size=head_size, v_head_size=v_head_size or head_size,
                         rotary_offset=rotary_offset,
                         rotary_dim=head_size if rotary_dim is None else rotary_dim,
                         rotary_interleaved=rotary_interleaved, block_size=block_size,
                         num_blocks=num_blocks, max_blocks_per_seq=max_blocks_per_seq,
                         cos_rows=cos_rows, scale=scale, softcap=softcap,
                         local_window_size=local_window_size, seed=seed, std=std,
                         drop_slots=drop_slots, drop_frac=drop_frac)
    assert num_heads % kv_num_heads == 0
    vhs = base.v_head_size
    gen = torch.Generator().manual_seed(seed + 7777)
    T = base.num_tokens
    key = _normal((T, kv_num_heads * head_size), gen, std, dtype)
    value = _normal((T, kv_num_heads * vhs), gen, std, dtype)
    kc = _normal((base.num_blocks, block_size, kv_num_heads, head_size), gen, std, dtype)
    vc = _normal((base.num_blocks, block_size, kv_num_heads, vhs), gen, std, dtype)
    sink = (torch.randn(num_heads, generator=gen)).to(dtype) if head_sink else None
    qn = (1.0 + 0.2 * torch.randn(head_size, generator=gen)).to(dtype) if qk_norm else None
    kn = (1.0 + 0.2 * torch.randn(head_size, generator=gen)).to(dtype) if qk_norm else None
    return SeparateWorkload(
        name=name, dtype=dtype, num_heads=num_heads, kv_num_heads=kv_num_heads,
        head_size=head_size, v_head_size=vhs, rotary_offset=base.rotary_offset,
        rotary_dim=base.rotary_dim, rotary_interleaved=rotary_interleaved,
        block_size=block_size, num_blocks=base.num_blocks,
        max_blocks_per_seq=base.max_blocks_per_seq, cos_rows=base.cos_rows, scale=base.scale,
        softcap=softcap, local_window_size=local_window_size, rms_eps=rms_eps,
        q_lens=base.q_lens, past_lens=base.past_lens, num_decode_seqs=base.num_decode_seqs,
        query=base.query, key=key, value=value, key_cache=kc, value_cache=vc,
        cos_cache=base.cos_cache, sin_cache=base.sin_cache, cumseq=base.cumseq, past=base.past,
        block_table=base.block_table, slot_mapping=base.slot_mapping, head_sink=sink,
        q_norm_weight=qn, k_norm_weight=kn, meta=dict(seed=seed, std=std))


def gqa_decode(seed: int = 9, batch: int = 32) -> SeparateWorkload:
    """Grouped-query decode: 32 query heads over 8 kv heads, head size 128
    with full RoPE, batch 32 x one new token, contexts uniform in
    [1024, 8192], bs = 64, q/k RMSNorm and a sink logit per head."""
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    ctx = torch.randint(1024, 8193, (batch,), generator=g).tolist()
    return make_separate_workload("gqa_decode", q_lens=[1] * batch,
                                  past_lens=[c - 1 for c in ctx], num_heads=32, kv_num_heads=8,
                                  head_size=128, block_size=64, cos_rows=8192, seed=seed,
                                  head_sink=True, qk_norm=True)


def separate_oracle_params(w: SeparateWorkload) -> Dict[str, object]:
    p = w.params()
    p["dtype"] = dtype_tag(w.dtype)
    return p


WORKLOADS["gqa_decode"] = gqa_decode
