"""GPU edge cases: option variants, odd geometries, empty and ragged
batches, device error flags, determinism and CUDA-graph capture/replay."""
import numpy as np
import pytest
import torch

from paged_latent_attention_cache_gb300 import binding as B
from paged_latent_attention_cache_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


def _check(w, portable=False, tokens=None, default_scale=False, family=None):
    """Runs w through the C ABI and checks it against the oracle; ``family``
    (when given) is the kernel family both read phases must use (1 =
    tcgen05 tensor cores, 0 = portable CUDA cores)."""
    got = Hn.run_gpu(w, portable=portable, scale=0.0 if default_scale else None)
    if family is not None:
        assert (got["op"].kernel_family(0), got["op"].kernel_family(1)) == (family, family)
    ref = Hn.run_oracle(w, tokens)
    assert got["flags"] == 0, hex(got["flags"])
    Hn.check_cache(w, got["cache"], ref["cache"])
    err, ratio = Hn.check_out(w, got["out"], ref["out"], tokens, ref["scales"])
    print(f"RATIO {w.name}: max abs err {err:.3e}, {ratio:.3f} of the scale-aware bound")
    return got


VARIANTS = {
    "interleaved": dict(rotary_interleaved=1),
    "no_rotary": dict(rotary_dim=0, rotary_offset=0),
    "vhs_eq_hs_default_scale": dict(v_head_size=192, scale=0.0),
    "odd_vhs": dict(v_head_size=40),
    "heads_6": dict(num_heads=6),
    "bs_32": dict(block_size=32),
    "bs_256": dict(block_size=256),
    "window_0": dict(local_window_size=0),
    "window_5": dict(local_window_size=5),
    "window_huge": dict(local_window_size=1 << 20),
    "softcap_3": dict(softcap=3.0),
    "softcap_tight": dict(softcap=0.5, scale=0.3),
    "fp16": dict(dtype=torch.float16),
    "fp16_no_rotary": dict(dtype=torch.float16, rotary_dim=0, rotary_offset=0),
    "rotary_at_0": dict(rotary_offset=0, rotary_dim=32),
}


@pytest.mark.parametrize("portable", [False, True], ids=["default", "portable"])
@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_variant(name, portable):
    kw = dict(num_heads=4, **W.GLM, block_size=16, seed=21, drop_slots=2)
    kw.update(VARIANTS[name])
    default_scale = kw.pop("scale", None) == 0.0
    w = W.make_workload(name, q_lens=[1, 1, 9, 0, 33], past_lens=[70, 0, 40, 5, 3], **kw)
    _check(w, portable, default_scale=default_scale, family=0 if portable else 1)


FP8_VARIANTS = {
    "plain": {},
    "bs_16": dict(block_size=16),
    "bs_128": dict(block_size=128),
    "softcap": dict(softcap=3.0),
    "window_5": dict(local_window_size=5),
    "fp16_query": dict(dtype=torch.float16),
    "interleaved": dict(rotary_interleaved=1),
    "no_rotary": dict(rotary_dim=0, rotary_offset=0),
    "heads_128": dict(num_heads=128),
    "hs_256_vhs_256": dict(head_size=256, v_head_size=256, rotary_offset=192),
    "hs_80_vhs_48": dict(head_size=80, v_head_size=48, rotary_offset=16),
    # wide latents with narrow values: 64-key tiles (two E4M3 stages do not
    # fit beside 128-key ones)
    "hs_224_vhs_106": dict(head_size=224, v_head_size=106, rotary_offset=160),
    "hs_256_vhs_128_heads_128": dict(head_size=256, v_head_size=128, rotary_offset=192,
                                     num_heads=128),
    "k_scale_odd": dict(k_scale=0.0123),
    "saturating_keys": dict(k_scale=2.0 ** -10),
}


@pytest.mark.parametrize("name", sorted(FP8_VARIANTS))
def test_fp8_cache_variants(name):
    """FP8 (E4M3) latent cache on the tensor-core kernels: decode and
    prefill tokens (split decode over a long context, prefill chunks with
    ragged tails), option variants and geometries. saturating_keys uses a
    k_scale small enough that many written values exceed 448 and saturate."""
    kw = dict(num_heads=4, **W.GLM, block_size=64, seed=29, drop_slots=2, cache_dtype="e4m3")
    kw.update(FP8_VARIANTS[name])
    w = W.make_workload(f"fp8_{name}", q_lens=[1, 1, 9, 0, 33], past_lens=[3000, 0, 40, 5, 3],
                        **kw)
    _check(w, family=1)


def test_fp8_query_beyond_fp16_range_is_flagged():
    """A bf16 query value beyond 65504 cannot enter the fp16 operands of the
    FP8-cache read: it is saturated and PA_DEVERR_RANGE is raised."""
    w = W.make_workload("fp8_range", q_lens=[1, 3], past_lens=[50, 7], num_heads=4, **W.GLM,
                        block_size=16, seed=30, cache_dtype="e4m3")
    w.query[0, 5] = 3.0e5
    got = Hn.run_gpu(w)
    assert got["flags"] & B.PA_DEVERR_RANGE
    from oracle import pa_oracle as O
    assert np.isfinite(O.bits_to_f64(got["out"], "bf16")).all()


def test_fp8_cache_not_built_paths_say_so():
    """FP8 on the portable kernels is not built: the read calls return
    PA_ERR_NOT_IMPLEMENTED before any launch."""
    w = W.make_workload("fp8_nyi", q_lens=[1], past_lens=[10], block_size=16, seed=31,
                        cache_dtype="e4m3", num_heads=4, **W.GLM)
    with pytest.raises(B.PaError) as e:
        Hn.run_gpu(w, portable=True)
    assert e.value.status == B.PA_ERR_NOT_IMPLEMENTED


@pytest.mark.parametrize("kw", [dict(block_size=64), dict(block_size=16),
                                dict(block_size=64, dtype=torch.float16),
                                dict(block_size=64, k_scale=0.0123, softcap=4.0),
                                dict(block_size=128, local_window_size=100)],
                         ids=["bs64", "bs16", "fp16", "odd_scale_softcap", "bs128_window"])
def test_fp8_cache_pair_kernel(kw):
    """FP8 (E4M3) cache on the 576/512 CTA-pair kernel (two converter warps,
    two fp16 and two E4M3 stages): decode and prefill tokens with several
    key tiles and ragged tails."""
    w = W.make_workload("fp8_pair", q_lens=[1, 1, 70, 1], past_lens=[300, 1, 200, 129],
                        num_heads=128, **W.DSV3, seed=32, scale=W.DSV3_SCALE, drop_slots=1,
                        cache_dtype="e4m3", **kw)
    _check(w, family=1)


@pytest.mark.parametrize("hs,vhs,ro,rd,H,family", [
    (64, 64, 0, 0, 2, 1), (576, 512, 512, 64, 16, 1), (256, 200, 128, 128, 3, 1),
    (1024, 512, 960, 64, 2, 0), (128, 128, 64, 64, 100, 1), (80, 48, 16, 64, 5, 1),
    (256, 256, 0, 64, 128, 1), (160, 1, 96, 64, 7, 1), (208, 136, 0, 0, 64, 1)])
def test_geometries(hs, vhs, ro, rd, H, family):
    """Latent widths up to 256 (multiples of 16; a last 64-channel slab may be
    partial) and any value width up to the latent width run on the
    tensor-core kernels, as does 576/512; wider latents use the portable
    kernels. Decode and prefill tokens, heads up to 128."""
    w = W.make_workload("geo", q_lens=[1, 17], past_lens=[100, 30], num_heads=H, head_size=hs,
                        v_head_size=vhs, rotary_offset=ro, rotary_dim=rd, block_size=16,
                        seed=22, scale=0.08)
    _check(w, family=family)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("hs", [64, 128, 192, 256])
def test_vhs_equal_hs_default_scale(hs, dtype):
    """v_head_size == head_size with the default scale 1/sqrt(head_size)
    (the rule of paged_attention.rs execute: an explicit scale is required
    only when v_head_size != head_size), on the tensor-core kernels, over a
    long decode (several key splits) and a prefill chunk."""
    w = W.make_workload("vhs_eq_hs", q_lens=[1, 1, 40], past_lens=[3000, 64, 100], num_heads=16,
                        head_size=hs, v_head_size=hs, rotary_offset=hs - 64, rotary_dim=64,
                        block_size=64, seed=27, dtype=dtype)
    _check(w, default_scale=True, family=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("bs", [16, 64])
def test_pair_kernel_dtypes_and_boxes(dtype, bs):
    """The CTA-pair kernel (576/512 latent) with bf16 and fp16 inputs, one
    box per key tile (64-row blocks) and four (16-row blocks), over decode
    and prefill tokens with several key tiles and ragged tails."""
    w = W.make_workload("pair", q_lens=[1, 1, 70, 1], past_lens=[300, 1, 200, 129],
                        num_heads=128, **W.DSV3, block_size=bs, seed=31, dtype=dtype,
                        drop_slots=1)
    _check(w)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_pair_kernel_large_logits(dtype):
    """The CTA pair splits each score into two partial dot products that it
    exchanges between its SMs. With the query scaled by 128 the partial
    logits reach hundreds of log2 units; the outputs meet the scale-aware
    bound (the fixed bound is for unscaled queries)."""
    w = W.make_workload("pair_peaked", q_lens=[1, 1, 40], past_lens=[300, 77, 150],
                        num_heads=128, **W.DSV3, block_size=64, seed=33, dtype=dtype,
                        query_gain=128, scale=W.DSV3_SCALE)
    w.name = f"pair_peaked_x128_{W.dtype_tag(dtype)}"
    assert Hn.run_gpu(w)["op"].kernel_family(0) == 1
    _check(w)


def _one_hot_rows_valid(w, got_bits, ref):
    """At logits of 10^5 the softmax is one-hot: the output is the value row
    of the top-scoring key. Rounding the query operand to 16 bits moves a
    score by up to scale * u * sum_d |q_d K_jd|, so where two keys' scores lie
    that close, either key is a correct result. Rows that miss the
    scale-aware bound must be the value row of such a near-tied key, and
    there must be few of them."""
    from oracle import pa_oracle as O
    dt = W.dtype_tag(w.dtype)
    u = Hn.UNIT_ROUNDOFF[w.dtype]
    T, H, hs, vhs, bs = w.num_tokens, w.num_heads, w.head_size, w.v_head_size, w.block_size
    got = O.bits_to_f64(got_bits, dt).reshape(T, H, vhs)
    assert np.isfinite(got).all()
    refo = ref["out"].reshape(T, H, vhs)
    bound = Hn.output_bound(w.dtype, ref["out"], ref["scales"]).reshape(T, H, vhs)
    bad = np.argwhere((np.abs(got - refo) > bound).any(axis=2))
    assert len(bad) <= 0.01 * T * H, len(bad)
    cache = O.bits_to_f64(ref["cache"].reshape(-1, hs), dt)
    cos_t, sin_t = O.bits_to_f64(W.to_bits(w.cos_cache), dt), O.bits_to_f64(W.to_bits(w.sin_cache), dt)
    q = O.bits_to_f64(W.to_bits(w.query), dt)
    cs, past, bt = w.cumseq.numpy(), w.past.numpy(), w.block_table.numpy()
    for t, h in bad:
        b, pos = O.locate_token(int(t), cs, past)
        qh = O.rope_row(q[t, h * hs:(h + 1) * hs], pos, w.rotary_offset, w.rotary_dim, cos_t,
                        sin_t, False)
        K = cache[[O.cache_row_index(b, j, bt, bs, w.num_blocks) for j in range(pos + 1)]]
        s = w.scale * (K @ qh)
        slack = w.scale * u * (np.abs(K) @ np.abs(qh))
        top = int(np.argmax(s))
        near = np.where(s + slack >= s[top] - slack[top])[0]
        assert any(np.array_equal(got[t, h], K[j, :vhs]) for j in near), (int(t), int(h))
    return len(bad)


@pytest.mark.parametrize("dtype,gain", [(torch.bfloat16, 2 ** 17), (torch.float16, 2 ** 13)],
                         ids=["bf16-x2^17", "fp16-x2^13"])
def test_pair_kernel_logits_beyond_fp16_range(dtype, gain):
    """Partial logits beyond 6e4 (past the fp16 range): no overflow, no NaN,
    and every output row is the value row of a top-scoring key (up to the
    query operand's rounding, see _one_hot_rows_valid)."""
    w = W.make_workload("pair_huge", q_lens=[1, 1, 40], past_lens=[300, 77, 150],
                        num_heads=128, **W.DSV3, block_size=64, seed=33, dtype=dtype,
                        query_gain=gain, scale=W.DSV3_SCALE)
    got = Hn.run_gpu(w)
    assert got["flags"] == 0 and got["op"].kernel_family(0) == 1
    ref = Hn.run_oracle(w)
    Hn.check_cache(w, got["cache"], ref["cache"])
    ties = _one_hot_rows_valid(w, got["out"], ref)
    print(f"RATIO pair_huge x{gain} {W.dtype_tag(dtype)}: {ties} near-tied rows")


def _graph_kernel_nodes(fn):
    """Kernel launches of fn() captured in a CUDA graph (driver API count)."""
    import ctypes
    g = torch.cuda.CUDAGraph(keep_graph=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        fn()
    g.instantiate()
    cu = ctypes.CDLL("libcuda.so.1")
    h = ctypes.c_void_p(g.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(h, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) == 0
    cnt = 0
    for nd in nodes:
        t = ctypes.c_int(-1)
        cu.cuGraphNodeGetType(ctypes.c_void_p(nd), ctypes.byref(t))
        cnt += t.value == 0
    return cnt


@pytest.mark.parametrize("name", ["mixed_serving", "tiny"])
def test_mixed_batch_in_one_grid(name):
    """A batch of decode and prefill sequences read by one pa_latent_mixed
    call: one attention grid (write + attention + combine = 3 launches,
    against 4 for a decode call and a prefill call), and both forms meet the
    bounds against the oracle."""
    w = Hn.workload(name)
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    base = d.key_cache.clone()
    ref = Hn.run_oracle(w)
    shape = (w.num_tokens, w.num_heads * w.v_head_size)
    for one_call, launches in ((True, 3), (False, 4)):
        cache = base.clone()
        out = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
        fn = lambda: op.forward(d.query, d.key, cache, d.cos_cache, d.sin_cache, d.cumseq,
                                d.past, d.block_table, d.slot_mapping, w.num_decode_seqs,
                                out=out, one_call=one_call)
        assert _graph_kernel_nodes(fn) == launches
        cache.copy_(base)
        fn()
        torch.cuda.synchronize()
        assert op.error_flags() == 0
        Hn.check_cache(w, W.to_bits(cache), ref["cache"])
        err, ratio = Hn.check_out(w, W.to_bits(out), ref["out"], scales=ref["scales"])
        print(f"RATIO {name} one_call={one_call}: max abs err {err:.3e}, {ratio:.3f} of bound")


def test_long_decode_splits():
    """Long contexts (many key splits merged by the combine step)."""
    w = W.make_workload("long", q_lens=[1, 1, 1], past_lens=[20000, 3, 777], num_heads=16,
                        **W.GLM, block_size=64, seed=23)
    _check(w)
    _check(w, portable=True)


def test_empty_batch_is_a_no_op():
    w = W.make_workload("empty", q_lens=[0, 0], past_lens=[3, 4], num_heads=2, **W.GLM,
                        block_size=16, seed=24)
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    cache = d.key_cache.clone()
    out = torch.empty(0, 2 * 128, dtype=w.dtype, device="cuda")
    op.forward(d.query, d.key, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past,
               d.block_table, d.slot_mapping, 0, out=out)
    torch.cuda.synchronize()
    assert torch.equal(cache, d.key_cache) and op.error_flags() == 0


def test_deterministic_and_graph_replay_bit_equal():
    """Capture write + decode + prefill in one CUDA graph; 3 replays are bit
    equal to the eager result (the pages' capture + 3 replays gate)."""
    w = W.tiny()
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    base = d.key_cache.clone()
    cache = base.clone()
    out = torch.empty(w.num_tokens, w.num_heads * w.v_head_size, dtype=w.dtype, device="cuda")
    args = (d.query, d.key, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table,
            d.slot_mapping, w.num_decode_seqs)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        op.forward(*args, out=out)
    torch.cuda.current_stream().wait_stream(s)
    eager_out, eager_cache = out.clone(), cache.clone()
    cache.copy_(base)
    op.forward(*args, out=out)
    assert torch.equal(out, eager_out) and torch.equal(cache, eager_cache)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        op.forward(*args, out=out)
    for _ in range(3):
        cache.copy_(base)
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager_out) and torch.equal(cache, eager_cache)
    assert op.error_flags() == 0


@pytest.mark.parametrize("own_slots", [False, True], ids=["after_write", "own_slots"])
@pytest.mark.parametrize("name", ["glm_decode", "mixed_serving", "dsv3_decode", "tiny"])
def test_after_write_flag_bit_equal(name, own_slots):
    """The first read call after the write phase may start early
    (PA_FLAG_AFTER_WRITE, and with PA_FLAG_OWN_SLOTS load the rows below
    each sequence's new tokens before the write completes); its output is
    bit-equal to the same calls made without the flags, eagerly and inside a
    CUDA graph."""
    w = Hn.workload(name)
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w, own_slots=own_slots)
    base = d.key_cache.clone()
    shape = (w.num_tokens, w.num_heads * w.v_head_size)
    nd = w.num_decode_seqs

    def step(cache, out, flag):
        op.write(d.key, d.cos_cache, d.sin_cache, d.slot_mapping, d.cumseq, d.past, cache)
        if nd > 0:
            op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table,
                      out, 0, nd, after_write=flag)
        if nd < w.num_seqs:
            op.prefill(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past,
                       d.block_table, out, nd, w.num_seqs, after_write=flag and nd == 0)

    res = {}
    for flag in (False, True):
        cache = base.clone()
        out = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
        step(cache, out, flag)
        torch.cuda.synchronize()
        res[flag] = (out.clone(), cache.clone())
    assert torch.equal(res[False][0], res[True][0]) and torch.equal(res[False][1], res[True][1])
    cache = base.clone()
    out = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(cache, out, True)   # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        step(cache, out, True)
    for _ in range(2):
        cache.copy_(base)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, res[False][0]) and torch.equal(cache, res[False][1])
    assert op.error_flags() == 0


@pytest.mark.parametrize("name", ["glm_decode", "dsv3_decode"])
def test_workspace_reuse_across_batch_sizes(name):
    """Decode splits publish their partials and the per-sequence plan in
    the workspace, and the combine kernel merges them. One workspace serves
    calls over different sequence ranges in a row: a repeated full call is
    bit-equal to the first, and a call over a sub-range (a different split
    plan, so different rounding) agrees with it within the output tolerance.
    A plan or partial left behind by an earlier call and read by a later
    one would show up as a mismatch."""
    w = Hn.workload(name)
    d = w.to("cuda")
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    op = PagedLatentAttention.from_workload(w)
    cache = d.key_cache.clone()
    op.write(d.key, d.cos_cache, d.sin_cache, d.slot_mapping, d.cumseq, d.past, cache)
    shape = (w.num_tokens, w.num_heads * w.v_head_size)
    nd = w.num_decode_seqs

    def run(lo, hi):
        out = torch.full(shape, float("nan"), dtype=w.dtype, device="cuda")
        op.decode(d.query, cache, d.cos_cache, d.sin_cache, d.cumseq, d.past, d.block_table,
                  out, lo, hi)
        torch.cuda.synchronize()
        return out

    ref = run(0, nd)
    assert torch.isfinite(ref.float()).all()
    tol = Hn.TOL[w.dtype]
    for lo, hi in [(0, nd // 2), (nd // 2, nd), (1, 2), (0, nd), (3, nd - 5), (0, nd)]:
        got = run(lo, hi)
        rows = slice(lo, hi)  # decode-first: sequence b's token is row b
        if (lo, hi) == (0, nd):
            assert torch.equal(got, ref), (lo, hi)
        else:
            g, r = got[rows].float(), ref[rows].float()
            assert torch.isfinite(g).all(), (lo, hi)
            assert (g - r).abs().max().item() <= tol, (lo, hi)
    assert op.error_flags() == 0


def _flag_case(mutate, expect_bit, phase="both"):
    w = W.make_workload("flags", q_lens=[1, 4], past_lens=[30, 10], num_heads=4, **W.GLM,
                        block_size=16, seed=25, cos_rows=64)
    mutate(w)
    got = Hn.run_gpu(w)
    assert got["flags"] & expect_bit, hex(got["flags"])
    return w, got


def test_flag_slot_out_of_range():
    def m(w):
        w.slot_mapping[2] = w.num_blocks * w.block_size + 5
    w, got = _flag_case(m, B.PA_DEVERR_SLOT)


def test_flag_bad_block_zeroes_rows():
    def m(w):
        w.block_table[1, 0] = -1           # a block the prefill sequence reads
    w, got = _flag_case(m, B.PA_DEVERR_BLOCK)
    vals = got["out"][1:5]
    assert np.all(vals == 0)               # rows of the affected sequence are zero


def test_flag_position_beyond_cos_cache():
    def m(w):
        w.past[0] = 100                    # cos_rows is 64
    _flag_case(m, B.PA_DEVERR_POSITION)


def test_flag_decode_qlen():
    w = W.make_workload("flags", q_lens=[2, 4], past_lens=[30, 10], num_heads=4, **W.GLM,
                        block_size=16, seed=26)
    w.num_decode_seqs = 1                  # sequence 0 has 2 tokens: not a decode
    got = Hn.run_gpu(w)
    assert got["flags"] & B.PA_DEVERR_DECODE_QLEN
    rows = got["out"]
    from oracle import pa_oracle as O
    f = O.bits_to_f64(rows, "bf16")
    assert np.isnan(f[0:2]).all()          # rows of the rejected sequence untouched
    assert np.isfinite(f[2:]).all()        # the prefill sequence still ran


def test_flag_cumseq_short():
    def m(w):
        w.cumseq[-1] = w.cumseq[-1] - 1    # last token lies beyond cumseq[B]
    _flag_case(m, B.PA_DEVERR_CUMSEQ)


def test_flag_context_beyond_block_table():
    def m(w):
        w.past[1] = w.max_blocks_per_seq * w.block_size   # cos_rows too small as well
    w, got = _flag_case(m, B.PA_DEVERR_CONTEXT | B.PA_DEVERR_POSITION)


def test_gather_probe_reads_the_batch():
    """The paged streaming probe (a measurement aid that reads every visible
    cache row through the block table with the decode kernels' TMA boxes)
    runs over ragged contexts, block sizes 16 and 64 and every sweep shape
    without a device error, and reports a block-table entry outside the
    pool as the read phase does."""
    from paged_latent_attention_cache_gb300.api import PagedLatentAttention
    for bs in (16, 64):
        w = W.make_workload("probe", q_lens=[1] * 5, past_lens=[0, 63, 64, 200, 1000],
                            num_heads=4, **W.GLM, block_size=bs, seed=40, scale=0.07)
        d = w.to("cuda")
        p = PagedLatentAttention.from_workload(w, device="cuda").params
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for tile_keys, stages, ctas in [(64, 2, 1), (128, 4, 1), (64, 4, 2), (32, 3, 4)]:
            B.pa_latent_gather_probe(p, d.key_cache, d.past, d.block_table, tile_keys, stages,
                                     ctas, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        bt = d.block_table.clone()
        bt[4, 2] = w.key_cache.shape[0] + 5
        B.pa_latent_gather_probe(p, d.key_cache, d.past, bt, 64, 2, 1, err)
        torch.cuda.synchronize()
        assert int(err.item()) == B.PA_DEVERR_BLOCK


def _pair_units_workload(**kw):
    """DeepSeek dims, H=128, two prefill sequences of 90 tokens: 180 token
    units over one wave of 76 CTA pairs, so every pair attends two or three
    tokens in turn (token 179 - u is unit u; pair p takes u = p, p+76, p+152)."""
    base = dict(q_lens=[90, 90], past_lens=[100, 60], num_heads=128, **W.DSV3, block_size=64,
                seed=33, scale=W.DSV3_SCALE)
    base.update(kw)
    return W.make_workload("pair_units", **base)


def _positions(w):
    cs, past = w.cumseq.tolist(), w.past.tolist()
    return [past[b] + t - cs[b] for b in range(w.num_seqs) for t in range(cs[b], cs[b + 1])]


def test_pair_prefill_invalid_positions_in_later_units():
    """On the persistent CTA-pair prefill, tokens whose position lies past the
    cos/sin rows (sequence 0's last 40 tokens, units 90-129: a pair's second
    token) are flagged and their rows zeroed; every other token matches the
    oracle. (The invalid tokens write no cache row.)"""
    w = _pair_units_workload(cos_rows=150)
    pos = _positions(w)
    bad = [t for t, p in enumerate(pos) if p >= 150]
    good = [t for t, p in enumerate(pos) if p < 150]
    assert len(bad) == 40
    w.slot_mapping[bad] = -1
    got = Hn.run_gpu(w)
    assert got["flags"] == B.PA_DEVERR_POSITION, hex(got["flags"])
    assert np.all(got["out"][bad] == 0)
    ref = Hn.run_oracle(w, good)
    Hn.check_out(w, got["out"], ref["out"], good, ref["scales"])


def test_pair_prefill_bad_block_stays_with_its_tokens():
    """A block-table entry outside the pool in sequence 1 (read by all its
    tokens, which the pairs attend first) zeroes exactly sequence 1's rows:
    the tokens of sequence 0 that the same pairs attend afterwards match the
    oracle (the per-token error bit is cleared between tokens)."""
    w = _pair_units_workload()
    w.block_table[1, 0] = w.num_blocks + 3
    got = Hn.run_gpu(w)
    assert got["flags"] == B.PA_DEVERR_BLOCK, hex(got["flags"])
    from oracle import pa_oracle as O
    assert np.all(O.bits_to_f64(got["out"][90:], "bf16") == 0)  # (+0 or -0: O times 0)
    good = list(range(90))
    ref = Hn.run_oracle(w, good)
    Hn.check_out(w, got["out"], ref["out"], good, ref["scales"])


def _prefill_units_workload(**kw):
    """GLM dims, H=64 (two tokens per unit of the single-CTA kernel),
    prefill sequences of 1200 and 700 tokens on pasts 0 and 300: 950 units,
    three waves and more of the two-CTAs-per-SM prefill shape."""
    base = dict(q_lens=[1200, 700], past_lens=[0, 300], num_heads=64, **W.GLM, block_size=16,
                seed=41, scale=0.07)
    base.update(kw)
    return W.make_workload("prefill_units", **base)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_prefill_many_units(dtype):
    """A long chunked prefill on the half-SM prefill shape (units of two
    tokens, contexts up to 1000 keys): every token against the oracle, and a
    second run gives the same bits."""
    w = _prefill_units_workload(dtype=dtype)
    got = _check(w, family=1)
    again = Hn.run_gpu(w)
    assert np.array_equal(got["out"], again["out"])


def test_mixed_many_units():
    """A mixed batch in one grid: 40 decode sequences (long contexts,
    several key splits each) ahead of 1500 prefill tokens, with a window and
    a softcap."""
    q_lens = [1] * 40 + [900, 600]
    past = [2000 + 37 * i for i in range(40)] + [0, 450]
    w = W.make_workload("mixed_units", q_lens=q_lens, past_lens=past, num_heads=64, **W.GLM,
                        block_size=16, seed=42, scale=0.07, dtype=torch.float16,
                        local_window_size=700, softcap=30.0, num_decode_seqs=40, drop_frac=0.05)
    _check(w, family=1)


def test_prefill_invalid_positions_among_valid_units():
    """Tokens past the cos/sin rows (sequence 0's last 200) are flagged and
    their rows zeroed; every other token matches the oracle."""
    w = _prefill_units_workload(cos_rows=1000)
    pos = _positions(w)
    bad = [t for t, p in enumerate(pos) if p >= 1000]
    good = [t for t, p in enumerate(pos) if p < 1000]
    assert len(bad) == 200
    w.slot_mapping[bad] = -1
    got = Hn.run_gpu(w)
    assert got["flags"] == B.PA_DEVERR_POSITION, hex(got["flags"])
    assert np.all(got["out"][bad] == 0)
    ref = Hn.run_oracle(w, good)
    Hn.check_out(w, got["out"], ref["out"], good, ref["scales"])


def test_prefill_bad_block_stays_with_its_units():
    """A block-table entry outside the pool at sequence 0's keys 640-655
    zeroes exactly the rows of the units that read it (sequence 0's tokens
    at positions 640 and later; a unit's two tokens share their tiles); every
    other unit matches the oracle."""
    w = _prefill_units_workload()
    w.block_table[0, 40] = w.num_blocks + 3
    got = Hn.run_gpu(w)
    assert got["flags"] == B.PA_DEVERR_BLOCK, hex(got["flags"])
    from oracle import pa_oracle as O
    pos = _positions(w)
    bad = [t for t in range(1200) if pos[t] >= 640]
    bad_set = set(bad)
    good = [t for t in range(w.num_tokens) if t not in bad_set]
    assert np.all(O.bits_to_f64(got["out"][bad], "bf16") == 0)  # (+0 or -0: O times 0)
    ref = Hn.run_oracle(w, good)
    Hn.check_out(w, got["out"], ref["out"], good, ref["scales"])
