"""The C-ABI library loads, exports every entry point include/pa_latent.h
declares, and rejects invalid arguments on the host before any launch.
No test here touches a GPU: every call below returns from host-side checks.
"""
import ctypes
import os
import re

import pytest

from paged_latent_attention_cache_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    build.build()
    from paged_latent_attention_cache_gb300 import binding
    return binding


def _declared():
    src = open(os.path.join(ROOT, "include", "pa_latent.h")).read()
    return sorted(set(re.findall(r"\b(pa_(?:latent|separate)_\w+)\s*\(", src)))


def test_header_declares_the_three_calls():
    d = _declared()
    for name in ("pa_latent_write", "pa_latent_decode", "pa_latent_prefill"):
        assert name in d


def test_library_exports_every_declared_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(B.EXPORTED) == _declared()


def _sep(B, **kw):
    base = dict(dtype=B.PA_DTYPE_BF16, num_heads=8, kv_num_heads=2, head_size=128,
                rotary_dim=128, cos_rows=256, block_size=16, num_blocks=8, max_blocks_per_seq=4)
    base.update(kw)
    return B.make_separate_params(**base)


def test_separate_params_checked(B):
    """SEPARATE layout: kv_num_heads must divide num_heads; the default scale
    is allowed for any value width; rms_eps must be finite and >= 0; the
    portable flag is not a path this layout has."""
    assert B.pa_separate_validate(_sep(B)) == B.PA_OK
    assert B.pa_separate_validate(_sep(B, v_head_size=64)) == B.PA_OK
    assert B.pa_separate_validate(_sep(B, kv_num_heads=3)) == B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_separate_validate(_sep(B, kv_num_heads=0)) == B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_separate_validate(_sep(B, rms_eps=-1.0)) == B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_separate_validate(_sep(B, rms_eps=float("nan"))) == B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_separate_validate(_sep(B, block_size=24)) == B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_separate_validate(_sep(B, flags=B.PA_FLAG_PORTABLE)) == B.PA_ERR_NOT_IMPLEMENTED
    assert B.pa_separate_workspace_size(_sep(B), 32, 32) > 0
    assert B.pa_separate_workspace_size(_sep(B, kv_num_heads=3), 32, 32) == 0


def test_fp8_params_checked(B):
    """An FP8 cache needs a finite k_scale > 0; unknown cache formats are
    rejected."""
    assert B.pa_latent_validate(_good(B, cache_dtype="e4m3", k_scale=0.02)) == B.PA_OK
    assert B.pa_latent_validate(_good(B, cache_dtype="e4m3", k_scale=0.0)) == \
        B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_latent_validate(_good(B, cache_dtype="e4m3", k_scale=float("inf"))) == \
        B.PA_ERR_INVALID_ARGUMENT
    assert B.pa_latent_validate(_good(B, cache_dtype=7)) == B.PA_ERR_INVALID_ARGUMENT


def _good(B, **kw):
    base = dict(dtype=B.PA_DTYPE_BF16, num_heads=4, head_size=192, v_head_size=128,
                rotary_offset=128, rotary_dim=64, cos_rows=256, block_size=16, num_blocks=8,
                max_blocks_per_seq=4, scale=0.07)
    base.update(kw)
    return B.make_params(**base)


def test_valid_params_accepted(B):
    assert B.pa_latent_validate(_good(B)) == B.PA_OK
    # vhs == hs may use the default scale
    assert B.pa_latent_validate(_good(B, v_head_size=0, scale=0.0)) == B.PA_OK
    assert B.pa_latent_validate(_good(B, rotary_dim=0, rotary_offset=0)) == B.PA_OK
    assert B.pa_latent_validate(_good(B, rotary_interleaved=1)) == B.PA_OK


@pytest.mark.parametrize("kw,status,needle", [
    (dict(dtype=7), 2, "float16"),
    (dict(num_heads=0), 1, "num_heads"),
    (dict(head_size=200), 1, "multiple of 16"),
    (dict(head_size=2048, v_head_size=128), 2, "maximum"),
    (dict(v_head_size=193), 1, "v_head_size"),
    (dict(scale=0.0), 1, "explicit scale"),
    (dict(scale=-1.0), 1, "scale"),
    (dict(scale=float("nan")), 1, "scale"),
    (dict(block_size=24), 1, "power of two"),
    (dict(block_size=8), 1, "power of two"),
    (dict(rotary_dim=8), 1, "multiple of 16"),
    (dict(rotary_offset=132), 1, "multiple of 8"),
    (dict(rotary_offset=144), 1, "exceeds head_size"),
    (dict(cos_rows=0), 1, "cos_rows"),
    (dict(rotary_interleaved=2), 1, "rotary_interleaved"),
    (dict(num_blocks=0), 1, "num_blocks"),
    (dict(max_blocks_per_seq=0), 1, "max_blocks_per_seq"),
    (dict(softcap=float("inf")), 1, "softcap"),
    (dict(flags=0x10), 1, "flag"),
])
def test_invalid_params_rejected(B, kw, status, needle):
    p = _good(B, **kw)
    assert B.pa_latent_validate(p) == status
    assert needle in B.last_error()


def _call(Bm, fn, p, **over):
    """Calls a read entry point with fake but aligned non-null pointers; only
    host-side checks can run because each case is rejected before launch."""
    a = dict(q=0x10000, T=8, cache=0x20000, cos=0x30000, sin=0x40000, cumseq=0x50000,
             past=0x60000, bt=0x70000, B=2, sb=0, se=2, ws=None, wsb=0, out=0x80000,
             err=0x90000)
    a.update(over)
    vp = ctypes.c_void_p
    return fn(ctypes.byref(p), vp(a["q"]), a["T"], vp(a["cache"]), vp(a["cos"]), vp(a["sin"]),
              vp(a["cumseq"]), vp(a["past"]), vp(a["bt"]), a["B"], a["sb"], a["se"],
              vp(a["ws"]) if a["ws"] else None, ctypes.c_size_t(a["wsb"]), vp(a["out"]),
              vp(a["err"]), None)


@pytest.mark.parametrize("over,needle", [
    (dict(q=0), "NULL"),
    (dict(bt=0), "NULL"),
    (dict(q=0x10008), "16-byte"),
    (dict(out=0x80004), "16-byte"),
    (dict(cumseq=0x50002), "4-byte"),
    (dict(sb=1, se=3), "sequence range"),
    (dict(sb=-1), "sequence range"),
    (dict(T=-1), "num_tokens"),
    (dict(T=2 ** 31), "num_tokens"),
])
def test_read_phase_host_rejections(B, over, needle):
    p = _good(B)
    for fn in (B.lib.pa_latent_decode, B.lib.pa_latent_prefill):
        s = _call(B, fn, p, **over)
        assert s == B.PA_ERR_INVALID_ARGUMENT, (over, B.last_error())
        assert needle in B.last_error()


def test_decode_needs_a_token_per_sequence(B):
    s = _call(B, B.lib.pa_latent_decode, _good(B), T=1, se=2)
    assert s == B.PA_ERR_INVALID_ARGUMENT and "tokens" in B.last_error()


def test_empty_calls_are_no_ops(B):
    assert _call(B, B.lib.pa_latent_decode, _good(B), T=0) == B.PA_OK
    assert _call(B, B.lib.pa_latent_prefill, _good(B), sb=1, se=1) == B.PA_OK


def test_write_host_rejections(B):
    p = _good(B)
    vp = ctypes.c_void_p
    args = [vp(0x10000), 4, vp(0x30000), vp(0x40000), vp(0x50000), vp(0x60000), vp(0x70000), 2,
            vp(0x80000), vp(0x90000), None]
    bad = list(args); bad[0] = None
    assert B.lib.pa_latent_write(ctypes.byref(p), *bad) == B.PA_ERR_INVALID_ARGUMENT
    bad = list(args); bad[8] = vp(0x80008)
    assert B.lib.pa_latent_write(ctypes.byref(p), *bad) == B.PA_ERR_INVALID_ARGUMENT
    bad = list(args); bad[2] = None
    assert B.lib.pa_latent_write(ctypes.byref(p), *bad) == B.PA_ERR_INVALID_ARGUMENT
    assert "cos_cache" in B.last_error()
    bad = list(args); bad[1] = 0
    assert B.lib.pa_latent_write(ctypes.byref(p), *bad) == B.PA_OK   # nothing to do
    bad = list(args); bad[7] = 0
    assert B.lib.pa_latent_write(ctypes.byref(p), *bad) == B.PA_ERR_INVALID_ARGUMENT


def test_gather_probe_host_rejections(B):
    """The paged streaming probe checks its sweep parameters, pointers and
    shared-memory budget on the host (no call here reaches a launch)."""
    p = _good(B)
    vp = ctypes.c_void_p
    good = [vp(0x10000), vp(0x20000), vp(0x30000), 2, 64, 4, 1, vp(0x40000), None]

    def call(params=p, **over):
        a = list(good)
        for i, v in over.items():
            a[int(i[1:])] = v
        return B.lib.pa_latent_gather_probe(ctypes.byref(params), *a)
    for over, needle in [(dict(a4=48), "tile_keys"), (dict(a5=0), "stages"),
                         (dict(a5=9), "stages"), (dict(a6=5), "ctas_per_sm"),
                         (dict(a3=0), "num_seqs"), (dict(a3=5000), "num_seqs"),
                         (dict(a0=None), "NULL"), (dict(a7=None), "NULL"),
                         (dict(a0=vp(0x10008)), "aligned"), (dict(a1=vp(0x20002)), "aligned")]:
        assert call(**over) == B.PA_ERR_INVALID_ARGUMENT, (over, B.last_error())
        assert needle in B.last_error(), (over, B.last_error())
    big = _good(B, head_size=576, v_head_size=512, rotary_offset=512)
    assert call(params=big, a4=128, a5=8) == B.PA_ERR_INVALID_ARGUMENT
    assert "shared memory" in B.last_error()
    assert call(params=_good(B, cache_dtype="e4m3", k_scale=0.02)) == B.PA_ERR_NOT_IMPLEMENTED


def test_status_strings(B):
    for s, name in [(0, "PA_OK"), (1, "PA_ERR_INVALID_ARGUMENT"), (2, "PA_ERR_NOT_IMPLEMENTED"),
                    (3, "PA_ERR_CUDA"), (4, "PA_ERR_WORKSPACE")]:
        assert B.status_string(s) == name


def test_kernel_family_query(B):
    assert B.pa_latent_kernel_family(_good(B, num_heads=0), 0) == -1
    assert B.pa_latent_kernel_family(_good(B, flags=B.PA_FLAG_PORTABLE), 0) == 0
    assert B.pa_latent_kernel_family(_good(B), 5) == -1
