"""User-facing operator object over the C ABI.

``PagedLatentAttention`` holds the operator parameters, the split-KV
workspace and the device error word, all allocated once at construction;
``forward`` then only enqueues the library's kernels (write phase, decode
phase for the decode-first sequences, prefill phase for the rest) and is
safe to record into a CUDA graph after one eager call.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class PagedLatentAttention:
    def __init__(self, *, dtype: torch.dtype, num_heads: int, head_size: int,
                 v_head_size: int = 0, rotary_offset: int = 0, rotary_dim: int = 0,
                 rotary_interleaved: int = 0, cos_rows: int = 1, block_size: int,
                 num_blocks: int, max_blocks_per_seq: int, scale: float = 0.0,
                 softcap: float = 0.0, local_window_size: int = -1, max_seqs: int,
                 max_tokens: int, device="cuda", portable: bool = False,
                 own_slots: bool = False, cache_dtype=None, k_scale: float = 1.0):
        self.dtype = dtype
        self.num_heads = num_heads
        self.head_size = head_size
        self.v_head_size = v_head_size or head_size
        self.params = B.make_params(
            dtype=dtype, num_heads=num_heads, head_size=head_size, v_head_size=v_head_size,
            rotary_offset=rotary_offset, rotary_dim=rotary_dim,
            rotary_interleaved=rotary_interleaved, cos_rows=cos_rows, block_size=block_size,
            num_blocks=num_blocks, max_blocks_per_seq=max_blocks_per_seq, scale=scale,
            softcap=softcap, local_window_size=local_window_size,
            flags=B.PA_FLAG_PORTABLE if portable else 0, cache_dtype=cache_dtype,
            k_scale=k_scale)
        s = B.pa_latent_validate(self.params)
        if s != B.PA_OK:
            raise B.PaError(s, B.last_error())
        # the same parameters for the first read call after the write phase
        # (own_slots: every slot is its token's own position, see
        # PA_FLAG_OWN_SLOTS)
        self.params_after_write = B.pa_latent_params.from_buffer_copy(self.params)
        self.params_after_write.flags |= B.PA_FLAG_AFTER_WRITE | (
            B.PA_FLAG_OWN_SLOTS if own_slots else 0)
        self.device = torch.device(device)
        self.max_seqs, self.max_tokens = max_seqs, max_tokens
        self.workspace = B.alloc_workspace(self.params, max_seqs, max_tokens, self.device)
        self.err_flags = torch.zeros(1, dtype=torch.int32, device=self.device)

    @classmethod
    def from_workload(cls, w, device="cuda", portable=False,
                      own_slots=True) -> "PagedLatentAttention":
        """Operator for a generated workload; its slot mappings point every
        token at its own position (see ``workloads.make_workload``)."""
        return cls(dtype=w.dtype, num_heads=w.num_heads, head_size=w.head_size,
                   v_head_size=w.v_head_size, rotary_offset=w.rotary_offset,
                   rotary_dim=w.rotary_dim, rotary_interleaved=w.rotary_interleaved,
                   cos_rows=w.cos_rows, block_size=w.block_size, num_blocks=w.num_blocks,
                   max_blocks_per_seq=w.max_blocks_per_seq, scale=w.scale, softcap=w.softcap,
                   local_window_size=w.local_window_size, max_seqs=w.num_seqs,
                   max_tokens=max(w.num_tokens, 1), device=device, portable=portable,
                   own_slots=own_slots, cache_dtype=w.cache_dtype, k_scale=w.k_scale)

    def kernel_family(self, phase: int) -> int:
        return B.pa_latent_kernel_family(self.params, phase)

    def write(self, key, cos_cache, sin_cache, slot_mapping, cumseq, past, key_cache,
              stream=None):
        B.pa_latent_write(self.params, key, cos_cache, sin_cache, slot_mapping, cumseq, past,
                          key_cache, self.err_flags, stream)

    def _read_params(self, after_write: bool):
        return self.params_after_write if after_write else self.params

    def decode(self, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
               seq_begin=0, seq_end=None, stream=None, after_write: bool = False):
        """Decode phase over sequences [seq_begin, seq_end). ``after_write``:
        this call directly follows ``write`` on the same stream (see
        PA_FLAG_AFTER_WRITE)."""
        B.pa_latent_decode(self._read_params(after_write), query, key_cache, cos_cache, sin_cache, cumseq, past,
                           block_table, out, seq_begin, seq_end, self.workspace,
                           self.err_flags, stream)

    def prefill(self, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                seq_begin=0, seq_end=None, stream=None, after_write: bool = False):
        B.pa_latent_prefill(self._read_params(after_write), query, key_cache, cos_cache, sin_cache, cumseq, past,
                            block_table, out, seq_begin, seq_end, self.workspace,
                            self.err_flags, stream)

    def mixed(self, query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
              num_decode_seqs: int, stream=None, after_write: bool = False):
        """Read phase of the whole batch in one call: decode over
        [0, num_decode_seqs), prefill over the rest (see pa_latent_mixed)."""
        B.pa_latent_mixed(self._read_params(after_write), query, key_cache, cos_cache, sin_cache,
                          cumseq, past, block_table, out, num_decode_seqs, self.workspace,
                          self.err_flags, stream)

    def forward(self, query, key, key_cache, cos_cache, sin_cache, cumseq, past, block_table,
                slot_mapping, num_decode_seqs: int, out: Optional[torch.Tensor] = None,
                stream=None, one_call: bool = True) -> torch.Tensor:
        """Write phase over all tokens, then decode over sequences
        [0, num_decode_seqs) and prefill over the rest; returns ``out``. A
        batch with both kinds of sequences is read by one pa_latent_mixed
        call (``one_call=False``: a decode call and a prefill call)."""
        T = query.shape[0]
        nseq = past.shape[0]
        if out is None:
            out = torch.empty(T, self.num_heads * self.v_head_size, dtype=self.dtype,
                              device=query.device)
        self.write(key, cos_cache, sin_cache, slot_mapping, cumseq, past, key_cache, stream)
        if one_call and 0 < num_decode_seqs < nseq:
            self.mixed(query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                       num_decode_seqs, stream, after_write=True)
            return out
        if num_decode_seqs > 0:
            self.decode(query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                        0, num_decode_seqs, stream, after_write=True)
        if num_decode_seqs < nseq:
            self.prefill(query, key_cache, cos_cache, sin_cache, cumseq, past, block_table, out,
                         num_decode_seqs, nseq, stream, after_write=num_decode_seqs == 0)
        return out

    def error_flags(self) -> int:
        """Reads the device error word (synchronises with the device)."""
        return int(self.err_flags.item())

    def reset_error_flags(self):
        self.err_flags.zero_()


class SeparateAttention:
    """The op's SEPARATE mode (grouped-query attention over separate key and
    value caches, optional head sink and q/k RMSNorm) over the C ABI: holds
    the parameters, the decode workspace and the error word; ``forward``
    issues write -> decode -> prefill like ``PagedLatentAttention``."""

    def __init__(self, *, dtype: torch.dtype, num_heads: int, kv_num_heads: int, head_size: int,
                 v_head_size: int = 0, rotary_offset: int = 0, rotary_dim: int = 0,
                 rotary_interleaved: int = 0, cos_rows: int = 1, block_size: int,
                 num_blocks: int, max_blocks_per_seq: int, scale: float = 0.0,
                 softcap: float = 0.0, local_window_size: int = -1, rms_eps: float = 1e-6,
                 max_seqs: int, max_tokens: int, device="cuda", own_slots: bool = False):
        self.dtype = dtype
        self.num_heads = num_heads
        self.v_head_size = v_head_size or head_size
        self.params = B.make_separate_params(
            dtype=dtype, num_heads=num_heads, kv_num_heads=kv_num_heads, head_size=head_size,
            v_head_size=v_head_size, rotary_offset=rotary_offset, rotary_dim=rotary_dim,
            rotary_interleaved=rotary_interleaved, cos_rows=cos_rows, block_size=block_size,
            num_blocks=num_blocks, max_blocks_per_seq=max_blocks_per_seq, scale=scale,
            softcap=softcap, local_window_size=local_window_size, rms_eps=rms_eps)
        s = B.pa_separate_validate(self.params)
        if s != B.PA_OK:
            raise B.PaError(s, B.last_error())
        self.params_after_write = B.pa_separate_params.from_buffer_copy(self.params)
        self.params_after_write.flags |= B.PA_FLAG_AFTER_WRITE | (
            B.PA_FLAG_OWN_SLOTS if own_slots else 0)
        self.device = torch.device(device)
        n = B.pa_separate_workspace_size(self.params, max_seqs, max_tokens)
        self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device) if n else None
        self.err_flags = torch.zeros(1, dtype=torch.int32, device=self.device)

    @classmethod
    def from_workload(cls, w, device="cuda", own_slots=True) -> "SeparateAttention":
        return cls(dtype=w.dtype, num_heads=w.num_heads, kv_num_heads=w.kv_num_heads,
                   head_size=w.head_size, v_head_size=w.v_head_size,
                   rotary_offset=w.rotary_offset, rotary_dim=w.rotary_dim,
                   rotary_interleaved=w.rotary_interleaved, cos_rows=w.cos_rows,
                   block_size=w.block_size, num_blocks=w.num_blocks,
                   max_blocks_per_seq=w.max_blocks_per_seq, scale=w.scale, softcap=w.softcap,
                   local_window_size=w.local_window_size, rms_eps=w.rms_eps,
                   max_seqs=w.num_seqs, max_tokens=max(w.num_tokens, 1), device=device,
                   own_slots=own_slots)

    def forward(self, query, key, value, key_cache, value_cache, cos_cache, sin_cache, cumseq,
                past, block_table, slot_mapping, num_decode_seqs: int, head_sink=None,
                q_norm_weight=None, k_norm_weight=None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        T, nseq = query.shape[0], past.shape[0]
        if out is None:
            out = torch.empty(T, self.num_heads * self.v_head_size, dtype=self.dtype,
                              device=query.device)
        B.pa_separate_write(self.params, key, value, cos_cache, sin_cache, k_norm_weight,
                            slot_mapping, cumseq, past, key_cache, value_cache, self.err_flags,
                            stream)
        if num_decode_seqs > 0:
            B.pa_separate_decode(self.params_after_write, query, key_cache, value_cache,
                                 cos_cache, sin_cache, q_norm_weight, head_sink, cumseq, past,
                                 block_table, out, 0, num_decode_seqs, self.workspace,
                                 self.err_flags, stream)
        if num_decode_seqs < nseq:
            p = self.params_after_write if num_decode_seqs == 0 else self.params
            B.pa_separate_prefill(p, query, key_cache, value_cache, cos_cache, sin_cache,
                                  q_norm_weight, head_sink, cumseq, past, block_table, out,
                                  num_decode_seqs, nseq, self.workspace, self.err_flags, stream)
        return out

    def error_flags(self) -> int:
        return int(self.err_flags.item())
