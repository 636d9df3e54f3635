"""ctypes binding of libpa_latent.so (include/pa_latent.h).

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels. The functions carry the C names and take torch tensors (device
memory) where the C ABI takes device pointers; the current torch CUDA stream
is passed unless one is given. A non-OK status raises PaError with the
library's message. Importing this module without the built library raises:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_latent.so")

PA_OK = 0
PA_ERR_INVALID_ARGUMENT = 1
PA_ERR_NOT_IMPLEMENTED = 2
PA_ERR_CUDA = 3
PA_ERR_WORKSPACE = 4

PA_DTYPE_F16 = 0
PA_DTYPE_BF16 = 1

PA_CACHE_DEFAULT = 0
PA_CACHE_FP8_E4M3 = 1

PA_DEVERR_SLOT = 0x01
PA_DEVERR_BLOCK = 0x02
PA_DEVERR_POSITION = 0x04
PA_DEVERR_CUMSEQ = 0x08
PA_DEVERR_DECODE_QLEN = 0x10
PA_DEVERR_CONTEXT = 0x20
PA_DEVERR_TIMEOUT = 0x40
PA_DEVERR_RANGE = 0x80

PA_FLAG_PORTABLE = 0x1
PA_FLAG_AFTER_WRITE = 0x2
PA_FLAG_OWN_SLOTS = 0x4

EXPORTED = ("pa_latent_validate", "pa_latent_write", "pa_latent_decode", "pa_latent_prefill",
            "pa_latent_mixed", "pa_latent_gather_probe",
            "pa_latent_decode_noalloc", "pa_latent_workspace_size", "pa_latent_kernel_family",
            "pa_latent_status_string", "pa_latent_last_error", "pa_separate_validate",
            "pa_separate_write", "pa_separate_decode", "pa_separate_prefill",
            "pa_separate_workspace_size")


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class pa_latent_params(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("v_head_size", ctypes.c_int32),
        ("rotary_offset", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rotary_interleaved", ctypes.c_int32),
        ("cos_rows", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("local_window_size", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("cache_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
    ]


class pa_separate_params(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("kv_num_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("v_head_size", ctypes.c_int32),
        ("rotary_offset", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rotary_interleaved", ctypes.c_int32),
        ("cos_rows", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("local_window_size", ctypes.c_int32),
        ("rms_eps", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run "
                          "`python -m paged_latent_attention_cache_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER(pa_latent_params)
    lib.pa_latent_validate.argtypes = [P]
    lib.pa_latent_validate.restype = ctypes.c_int
    lib.pa_latent_write.argtypes = [P, vp, i64, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    lib.pa_latent_write.restype = ctypes.c_int
    read = [P, vp, i64, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp, vp, vp]
    lib.pa_latent_decode.argtypes = read
    lib.pa_latent_decode.restype = ctypes.c_int
    lib.pa_latent_prefill.argtypes = read
    lib.pa_latent_prefill.restype = ctypes.c_int
    lib.pa_latent_mixed.argtypes = [P, vp, i64, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, vp, vp,
                                    vp]
    lib.pa_latent_mixed.restype = ctypes.c_int
    lib.pa_latent_decode_noalloc.argtypes = [P, vp, i64, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                             vp, vp, vp]
    lib.pa_latent_decode_noalloc.restype = ctypes.c_int
    lib.pa_latent_gather_probe.argtypes = [P, vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.pa_latent_gather_probe.restype = ctypes.c_int
    lib.pa_latent_workspace_size.argtypes = [P, i32, i64]
    lib.pa_latent_workspace_size.restype = sz
    lib.pa_latent_kernel_family.argtypes = [P, i32]
    lib.pa_latent_kernel_family.restype = i32
    lib.pa_latent_status_string.argtypes = [ctypes.c_int]
    lib.pa_latent_status_string.restype = ctypes.c_char_p
    lib.pa_latent_last_error.argtypes = []
    lib.pa_latent_last_error.restype = ctypes.c_char_p
    S = ctypes.POINTER(pa_separate_params)
    lib.pa_separate_validate.argtypes = [S]
    lib.pa_separate_validate.restype = ctypes.c_int
    lib.pa_separate_write.argtypes = [S, vp, vp, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.pa_separate_write.restype = ctypes.c_int
    sread = [S, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp, vp, vp]
    lib.pa_separate_decode.argtypes = sread
    lib.pa_separate_decode.restype = ctypes.c_int
    lib.pa_separate_prefill.argtypes = sread
    lib.pa_separate_prefill.restype = ctypes.c_int
    lib.pa_separate_workspace_size.argtypes = [S, i32, i64]
    lib.pa_separate_workspace_size.restype = sz
    return lib


lib = _load()


def status_string(s: int) -> str:
    return lib.pa_latent_status_string(int(s)).decode()


def last_error() -> str:
    return lib.pa_latent_last_error().decode()


def _check(s: int):
    if s != PA_OK:
        raise PaError(s, last_error())


def make_params(*, dtype, num_heads, head_size, v_head_size=0, rotary_offset=0, rotary_dim=0,
                rotary_interleaved=0, cos_rows=1, block_size, num_blocks, max_blocks_per_seq,
                scale=0.0, softcap=0.0, local_window_size=-1, flags=0, cache_dtype=None,
                k_scale=1.0) -> pa_latent_params:
    """``cache_dtype``: None / PA_CACHE_DEFAULT (the dtype), or "e4m3" /
    PA_CACHE_FP8_E4M3 with the FP8 cache's ``k_scale``."""
    if isinstance(dtype, torch.dtype):
        dtype = {torch.float16: PA_DTYPE_F16, torch.bfloat16: PA_DTYPE_BF16}.get(dtype, -1)
    if cache_dtype is None:
        cache_dtype = PA_CACHE_DEFAULT
    elif isinstance(cache_dtype, str):
        cache_dtype = {"e4m3": PA_CACHE_FP8_E4M3}.get(cache_dtype, -1)
    return pa_latent_params(int(dtype), int(num_heads), int(head_size), int(v_head_size),
                            int(rotary_offset), int(rotary_dim), int(rotary_interleaved),
                            int(cos_rows), int(block_size), int(num_blocks),
                            int(max_blocks_per_seq), float(scale), float(softcap),
                            int(local_window_size), int(flags), int(cache_dtype),
                            float(k_scale))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def pa_latent_validate(p: pa_latent_params) -> int:
    return lib.pa_latent_validate(ctypes.byref(p))


def pa_latent_workspace_size(p: pa_latent_params, num_seqs: int, num_tokens: int) -> int:
    return int(lib.pa_latent_workspace_size(ctypes.byref(p), int(num_seqs), int(num_tokens)))


def pa_latent_kernel_family(p: pa_latent_params, phase: int) -> int:
    return int(lib.pa_latent_kernel_family(ctypes.byref(p), int(phase)))


def pa_latent_write(p: pa_latent_params, key, cos_cache, sin_cache, slot_mapping, cumseq, past,
                    key_cache, err_flags=None, stream=None, num_tokens=None, num_seqs=None):
    T = key.shape[0] if num_tokens is None else num_tokens
    B = past.shape[0] if num_seqs is None else num_seqs
    _check(lib.pa_latent_write(ctypes.byref(p), _ptr(key), int(T), _ptr(cos_cache),
                               _ptr(sin_cache), _ptr(slot_mapping), _ptr(cumseq), _ptr(past),
                               int(B), _ptr(key_cache), _ptr(err_flags), _stream(stream)))


def pa_latent_gather_probe(p: pa_latent_params, key_cache, past, block_table, tile_keys: int,
                           stages: int, ctas_per_sm: int, err_flags, stream=None, num_seqs=None):
    """The paged streaming probe (measurement aid): reads every visible
    cache row of the batch through the block table, computes nothing."""
    B = past.shape[0] if num_seqs is None else num_seqs
    _check(lib.pa_latent_gather_probe(ctypes.byref(p), _ptr(key_cache), _ptr(past),
                                      _ptr(block_table), int(B), int(tile_keys), int(stages),
                                      int(ctas_per_sm), _ptr(err_flags), _stream(stream)))


def _read(fn, p, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
          seq_begin, seq_end, workspace, err_flags, stream, num_tokens, num_seqs):
    T = query.shape[0] if num_tokens is None else num_tokens
    B = past.shape[0] if num_seqs is None else num_seqs
    se = B if seq_end is None else seq_end
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(fn(ctypes.byref(p), _ptr(query), int(T), _ptr(key_cache), _ptr(cos_cache),
              _ptr(sin_cache), _ptr(cumseq), _ptr(past), _ptr(block_table), int(B),
              int(seq_begin), int(se), _ptr(workspace), ctypes.c_size_t(ws_bytes), _ptr(out),
              _ptr(err_flags), _stream(stream)))


def pa_latent_decode(p, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                     seq_begin=0, seq_end=None, workspace=None, err_flags=None, stream=None,
                     num_tokens=None, num_seqs=None):
    _read(lib.pa_latent_decode, p, query, key_cache, cos_cache, sin_cache, cumseq, past,
          block_table, out, seq_begin, seq_end, workspace, err_flags, stream, num_tokens, num_seqs)


def pa_latent_prefill(p, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                      seq_begin=0, seq_end=None, workspace=None, err_flags=None, stream=None,
                      num_tokens=None, num_seqs=None):
    _read(lib.pa_latent_prefill, p, query, key_cache, cos_cache, sin_cache, cumseq, past,
          block_table, out, seq_begin, seq_end, workspace, err_flags, stream, num_tokens, num_seqs)


def pa_latent_mixed(p, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                    num_decode_seqs, workspace=None, err_flags=None, stream=None):
    """Decodes [0, num_decode_seqs) and prefills the rest of the batch in one
    call (one grid where the single-CTA tensor-core kernel runs)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pa_latent_mixed(ctypes.byref(p), _ptr(query), int(query.shape[0]),
                               _ptr(key_cache), _ptr(cos_cache), _ptr(sin_cache), _ptr(cumseq),
                               _ptr(past), _ptr(block_table), int(past.shape[0]),
                               int(num_decode_seqs), _ptr(workspace), ctypes.c_size_t(ws_bytes),
                               _ptr(out), _ptr(err_flags), _stream(stream)))


def pa_latent_decode_noalloc(p, query, key_cache, cos_cache, sin_cache, cumseq, past,
                             block_table, out, seq_begin=0, seq_end=None, err_flags=None,
                             stream=None, num_tokens=None, num_seqs=None):
    """Decode using the library's static scratch instead of a workspace (for
    callers that cannot allocate device memory)."""
    T = query.shape[0] if num_tokens is None else num_tokens
    B = past.shape[0] if num_seqs is None else num_seqs
    se = B if seq_end is None else seq_end
    _check(lib.pa_latent_decode_noalloc(
        ctypes.byref(p), _ptr(query), int(T), _ptr(key_cache), _ptr(cos_cache), _ptr(sin_cache),
        _ptr(cumseq), _ptr(past), _ptr(block_table), int(B), int(seq_begin), int(se), _ptr(out),
        _ptr(err_flags), _stream(stream)))


def alloc_workspace(p: pa_latent_params, num_seqs: int, num_tokens: int,
                    device="cuda") -> Optional[torch.Tensor]:
    """A workspace tensor of the size the library asks for (None if 0)."""
    n = pa_latent_workspace_size(p, num_seqs, num_tokens)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)


def make_separate_params(*, dtype, num_heads, kv_num_heads, head_size, v_head_size=0,
                         rotary_offset=0, rotary_dim=0, rotary_interleaved=0, cos_rows=1,
                         block_size, num_blocks, max_blocks_per_seq, scale=0.0, softcap=0.0,
                         local_window_size=-1, rms_eps=1e-6, flags=0) -> pa_separate_params:
    if isinstance(dtype, torch.dtype):
        dtype = {torch.float16: PA_DTYPE_F16, torch.bfloat16: PA_DTYPE_BF16}.get(dtype, -1)
    return pa_separate_params(int(dtype), int(num_heads), int(kv_num_heads), int(head_size),
                              int(v_head_size), int(rotary_offset), int(rotary_dim),
                              int(rotary_interleaved), int(cos_rows), int(block_size),
                              int(num_blocks), int(max_blocks_per_seq), float(scale),
                              float(softcap), int(local_window_size), float(rms_eps), int(flags))


def pa_separate_validate(p: pa_separate_params) -> int:
    return int(lib.pa_separate_validate(ctypes.byref(p)))


def pa_separate_workspace_size(p: pa_separate_params, num_seqs: int, num_tokens: int) -> int:
    return int(lib.pa_separate_workspace_size(ctypes.byref(p), int(num_seqs), int(num_tokens)))


def pa_separate_write(p, key, value, cos_cache, sin_cache, k_norm_weight, slot_mapping, cumseq,
                      past, key_cache, value_cache, err_flags=None, stream=None):
    _check(lib.pa_separate_write(
        ctypes.byref(p), _ptr(key), _ptr(value), int(key.shape[0]), _ptr(cos_cache),
        _ptr(sin_cache), _ptr(k_norm_weight), _ptr(slot_mapping), _ptr(cumseq), _ptr(past),
        int(past.shape[0]), _ptr(key_cache), _ptr(value_cache), _ptr(err_flags),
        _stream(stream)))


def _sread(fn, p, query, key_cache, value_cache, cos_cache, sin_cache, q_norm_weight, head_sink,
           cumseq, past, block_table, out, seq_begin, seq_end, workspace, err_flags, stream):
    B = past.shape[0]
    se = B if seq_end is None else seq_end
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(fn(ctypes.byref(p), _ptr(query), int(query.shape[0]), _ptr(key_cache),
              _ptr(value_cache), _ptr(cos_cache), _ptr(sin_cache), _ptr(q_norm_weight),
              _ptr(head_sink), _ptr(cumseq), _ptr(past), _ptr(block_table), int(B),
              int(seq_begin), int(se), _ptr(workspace), ctypes.c_size_t(ws_bytes), _ptr(out),
              _ptr(err_flags), _stream(stream)))


def pa_separate_decode(p, query, key_cache, value_cache, cos_cache, sin_cache, q_norm_weight,
                       head_sink, cumseq, past, block_table, out, seq_begin=0, seq_end=None,
                       workspace=None, err_flags=None, stream=None):
    _sread(lib.pa_separate_decode, p, query, key_cache, value_cache, cos_cache, sin_cache,
           q_norm_weight, head_sink, cumseq, past, block_table, out, seq_begin, seq_end,
           workspace, err_flags, stream)


def pa_separate_prefill(p, query, key_cache, value_cache, cos_cache, sin_cache, q_norm_weight,
                        head_sink, cumseq, past, block_table, out, seq_begin=0, seq_end=None,
                        workspace=None, err_flags=None, stream=None):
    _sread(lib.pa_separate_prefill, p, query, key_cache, value_cache, cos_cache, sin_cache,
           q_norm_weight, head_sink, cumseq, past, block_table, out, seq_begin, seq_end,
           workspace, err_flags, stream)


def default_scale(head_size: int) -> float:
    return 1.0 / math.sqrt(head_size)
