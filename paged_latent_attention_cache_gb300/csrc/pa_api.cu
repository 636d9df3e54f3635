// C-ABI entry points: host-side validation, defaulting and dispatch.
//
// The checks follow paged_attention.rs execute() (geometry cross-checks,
// "explicit 'scale' attribute is required when v_head_size != head_size",
// block_size "must be a power of two >= 16", v_head_size "in 1..=head_size",
// rotary_offset + rotary_dim <= head_size) and the rotary-cache rules of the
// PR #1940 validator (head_size % 16 == 0, rotary_dim = 2 * cos dims[1] with
// dims[1] a multiple of 8, i.e. rotary_dim % 16 == 0) and the PR #1955 review
// (rotary_offset % 8 == 0). Everything here is host arithmetic on scalars:
// no device memory is touched and nothing is allocated, so the entry points
// can be recorded into CUDA graphs.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <string>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

thread_local std::string g_last_error;
thread_local const char* g_launch_step = nullptr;

pa_status fail(pa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pa_status fail(pa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-device SM count, looked up once per device (atomic: several host
// threads may make their first call at once).
int sm_count(int device) {
  static std::atomic<int> cache[64];
  if (device >= 0 && device < 64) {
    const int c = cache[device].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
    n = 148;
  if (device >= 0 && device < 64) cache[device].store(n, std::memory_order_relaxed);
  return n;
}

pa_status resolve(const pa_latent_params* p, Geometry* g) {
  if (!p) return fail(PA_ERR_INVALID_ARGUMENT, "params is NULL");
  if (p->dtype != PA_DTYPE_F16 && p->dtype != PA_DTYPE_BF16)
    return fail(PA_ERR_NOT_IMPLEMENTED, "dtype %d: only float16 and bfloat16 are implemented",
                p->dtype);
  if (p->num_heads < 1) return fail(PA_ERR_INVALID_ARGUMENT, "num_heads must be >= 1");
  const int hs = p->head_size;
  if (hs < 16 || hs % 16 != 0)
    return fail(PA_ERR_INVALID_ARGUMENT, "head_size %d must be a positive multiple of 16", hs);
  if (hs > kMaxHeadSize)
    return fail(PA_ERR_NOT_IMPLEMENTED, "head_size %d exceeds the supported maximum %d", hs,
                kMaxHeadSize);
  const int vhs = p->v_head_size == 0 ? hs : p->v_head_size;
  if (vhs < 1 || vhs > hs)
    return fail(PA_ERR_INVALID_ARGUMENT, "v_head_size %d must be in 1..=head_size %d", vhs, hs);
  if (p->rotary_dim < 0 || p->rotary_offset < 0)
    return fail(PA_ERR_INVALID_ARGUMENT, "rotary_offset/rotary_dim must be >= 0");
  if (p->rotary_dim > 0) {
    if (p->rotary_dim % 16 != 0)
      return fail(PA_ERR_INVALID_ARGUMENT,
                  "rotary_dim %d must be a multiple of 16 (cos_cache dims[1] a multiple of 8)",
                  p->rotary_dim);
    if (p->rotary_offset % 8 != 0)
      return fail(PA_ERR_INVALID_ARGUMENT, "rotary_offset %d must be a multiple of 8",
                  p->rotary_offset);
    if (p->rotary_offset + p->rotary_dim > hs)
      return fail(PA_ERR_INVALID_ARGUMENT, "rotary_offset %d + rotary_dim %d exceeds head_size %d",
                  p->rotary_offset, p->rotary_dim, hs);
    if (p->cos_rows < 1)
      return fail(PA_ERR_INVALID_ARGUMENT, "cos_rows must be >= 1 when rotary_dim > 0");
  }
  if (p->rotary_interleaved != 0 && p->rotary_interleaved != 1)
    return fail(PA_ERR_INVALID_ARGUMENT, "rotary_interleaved must be 0 or 1");
  const int bs = p->block_size;
  if (bs < 16 || (bs & (bs - 1)) != 0)
    return fail(PA_ERR_INVALID_ARGUMENT, "block_size %d must be a power of two >= 16", bs);
  if (p->num_blocks < 1) return fail(PA_ERR_INVALID_ARGUMENT, "num_blocks must be >= 1");
  if ((int64_t)p->num_blocks * bs > INT32_MAX)
    return fail(PA_ERR_INVALID_ARGUMENT, "num_blocks * block_size exceeds the int32 slot range");
  if (p->max_blocks_per_seq < 1)
    return fail(PA_ERR_INVALID_ARGUMENT, "max_blocks_per_seq must be >= 1");
  if ((int64_t)p->max_blocks_per_seq * bs > INT32_MAX)
    return fail(PA_ERR_INVALID_ARGUMENT, "max_blocks_per_seq * block_size exceeds int32");
  float scale = p->scale;
  if (!(isfinite(scale)) || scale < 0.f)
    return fail(PA_ERR_INVALID_ARGUMENT, "scale must be finite and >= 0");
  if (scale == 0.f) {
    if (vhs != hs)
      return fail(PA_ERR_INVALID_ARGUMENT,
                  "an explicit scale is required when v_head_size (%d) != head_size (%d)", vhs,
                  hs);
    scale = 1.0f / sqrtf((float)hs);
  }
  if (!isfinite(p->softcap)) return fail(PA_ERR_INVALID_ARGUMENT, "softcap must be finite");
  if (p->flags & ~(PA_FLAG_PORTABLE | PA_FLAG_AFTER_WRITE | PA_FLAG_OWN_SLOTS))
    return fail(PA_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", p->flags);
  if (p->cache_dtype != PA_CACHE_DEFAULT && p->cache_dtype != PA_CACHE_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARGUMENT, "cache_dtype %d is not a pa_cache_dtype", p->cache_dtype);
  const bool fp8 = p->cache_dtype == PA_CACHE_FP8_E4M3;
  if (fp8 && !(isfinite(p->k_scale) && p->k_scale > 0.f))
    return fail(PA_ERR_INVALID_ARGUMENT, "an FP8 cache needs a finite k_scale > 0");

  g->dtype = p->dtype;
  g->H = p->num_heads;
  g->hs = hs;
  g->vhs = vhs;
  g->rd = p->rotary_dim;
  g->ro = p->rotary_dim > 0 ? p->rotary_offset : 0;
  g->interleaved = p->rotary_interleaved;
  g->cos_rows = p->cos_rows;
  g->bs = bs;
  g->num_blocks = p->num_blocks;
  g->max_blocks = p->max_blocks_per_seq;
  g->scale = scale;
  g->softcap = p->softcap > 0.f ? p->softcap : 0.f;
  g->window = p->local_window_size < 0 ? -1 : p->local_window_size;
  g->fp8 = fp8 ? 1 : 0;
  g->k_scale = fp8 ? p->k_scale : 1.f;
  g->kvh = 1;
  g->rms_eps = 0.f;
  g->flags = p->flags;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  g->device = dev;
  g->num_sms = sm_count(dev);
  return PA_OK;
}

pa_status check_tokens(int64_t num_tokens, int32_t num_seqs, const Geometry& g) {
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARGUMENT, "num_tokens must be >= 0");
  if (num_seqs < 0) return fail(PA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0");
  if (num_tokens > INT32_MAX)
    return fail(PA_ERR_INVALID_ARGUMENT, "num_tokens must fit in int32");
  if (num_tokens * (int64_t)g.H >= ((int64_t)1 << 31))
    return fail(PA_ERR_INVALID_ARGUMENT, "num_tokens * num_heads must be < 2^31");
  return PA_OK;
}

pa_status cuda_status(cudaError_t e, const char* what) {
  const char* step = g_launch_step;
  g_launch_step = nullptr;
  if (e == cudaSuccess) return PA_OK;
  if (step) return fail(PA_ERR_CUDA, "%s (%s): %s", what, step, cudaGetErrorString(e));
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool use_tc(const Geometry& g, Phase ph) {
  return !(g.flags & PA_FLAG_PORTABLE) && tc_supported(g, ph);
}

// Workspace one read call needs: decode over sequences [seq_begin, seq_end),
// prefill over num_tokens tokens.
size_t call_workspace(const Geometry& g, Phase ph, int32_t seq_begin, int32_t seq_end,
                      int64_t num_tokens) {
  if (use_tc(g, ph)) return tc_call_workspace(g, ph, seq_begin, seq_end);
  const int64_t nq = ph == Phase::kDecode ? (int64_t)(seq_end - seq_begin) : num_tokens;
  return portable_call_workspace(g, ph, nq);
}

pa_status read_phase(Phase ph, const pa_latent_params* p, const void* query, int64_t num_tokens,
                     const void* key_cache, const void* cos_cache, const void* sin_cache,
                     const int32_t* cumseq, const int32_t* past, const int32_t* block_table,
                     int32_t num_seqs, int32_t seq_begin, int32_t seq_end, void* workspace,
                     size_t workspace_bytes, void* out, int32_t* err_flags, void* stream) {
  Geometry g;
  pa_status s = resolve(p, &g);
  if (s != PA_OK) return s;
  if ((s = check_tokens(num_tokens, num_seqs, g)) != PA_OK) return s;
  if (seq_begin < 0 || seq_end < seq_begin || seq_end > num_seqs)
    return fail(PA_ERR_INVALID_ARGUMENT, "sequence range [%d, %d) outside [0, %d)", seq_begin,
                seq_end, num_seqs);
  if (num_tokens == 0 || seq_end == seq_begin) return PA_OK;
  if (ph == Phase::kDecode && (int64_t)(seq_end - seq_begin) > num_tokens)
    return fail(PA_ERR_INVALID_ARGUMENT,
                "decode over %d sequences needs at least that many tokens (have %lld)",
                seq_end - seq_begin, (long long)num_tokens);
  if (!query || !key_cache || !cumseq || !past || !block_table || !out)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (g.rd > 0 && (!cos_cache || !sin_cache))
    return fail(PA_ERR_INVALID_ARGUMENT, "cos_cache/sin_cache are required when rotary_dim > 0");
  if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(out, 16) ||
      (g.rd > 0 && (!aligned(cos_cache, 16) || !aligned(sin_cache, 16))))
    return fail(PA_ERR_INVALID_ARGUMENT, "half-precision tensors must be 16-byte aligned");
  if (!aligned(cumseq, 4) || !aligned(past, 4) || !aligned(block_table, 4) ||
      !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  if (workspace && !aligned(workspace, 256))
    return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");

  ReadArgs a{query,     num_tokens, key_cache,   nullptr,   nullptr,     nullptr,
             cos_cache, sin_cache,  cumseq,      past,      block_table, num_seqs,
             seq_begin, seq_end,    seq_begin,   seq_end,   workspace,   workspace_bytes,
             out,       err_flags,  reinterpret_cast<cudaStream_t>(stream)};
  const bool tc = use_tc(g, ph);
  if (g.fp8 && !tc)
    return fail(PA_ERR_NOT_IMPLEMENTED,
                "an FP8 cache is read by the tensor-core kernels only (latent widths 64..256 "
                "on one SM; not with PA_FLAG_PORTABLE)");
  const size_t need = call_workspace(g, ph, seq_begin, seq_end, num_tokens);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace ? workspace_bytes : (size_t)0, need);
  cudaError_t e = tc ? launch_tc(g, ph, a) : launch_portable(g, ph, a);
  return cuda_status(e, tc ? "tensor-core attention launch" : "portable attention launch");
}

}  // namespace

// SEPARATE layout: the LATENT checks that apply (dtype, block size, rotary,
// window, softcap, flags) plus kv_num_heads dividing num_heads and the
// RMSNorm epsilon; scale 0 selects 1/sqrt(head_size).
pa_status resolve_separate(const pa_separate_params* p, Geometry* g) {
  if (!p) return fail(PA_ERR_INVALID_ARGUMENT, "params is NULL");
  if (p->kv_num_heads < 1 || p->num_heads < 1 || p->num_heads % p->kv_num_heads != 0)
    return fail(PA_ERR_INVALID_ARGUMENT,
                "num_heads %d must be a positive multiple of kv_num_heads %d", p->num_heads,
                p->kv_num_heads);
  if (!(isfinite(p->rms_eps) && p->rms_eps >= 0.f))
    return fail(PA_ERR_INVALID_ARGUMENT, "rms_eps must be finite and >= 0");
  pa_latent_params q = {};
  q.dtype = p->dtype;
  q.num_heads = p->num_heads;
  q.head_size = p->head_size;
  q.v_head_size = p->v_head_size;
  q.rotary_offset = p->rotary_offset;
  q.rotary_dim = p->rotary_dim;
  q.rotary_interleaved = p->rotary_interleaved;
  q.cos_rows = p->cos_rows;
  q.block_size = p->block_size;
  q.num_blocks = p->num_blocks;
  q.max_blocks_per_seq = p->max_blocks_per_seq;
  q.softcap = p->softcap;
  q.local_window_size = p->local_window_size;
  q.flags = p->flags;
  // the default scale is allowed for any value width here
  q.scale = p->scale;
  const int hs = p->head_size;
  if (p->scale == 0.f && hs >= 16 && hs % 16 == 0) q.scale = 1.0f / sqrtf((float)hs);
  if (q.v_head_size > hs && hs > 0)
    return fail(PA_ERR_INVALID_ARGUMENT, "v_head_size %d must be in 1..=head_size %d",
                q.v_head_size, hs);
  const pa_status s = resolve(&q, g);
  if (s != PA_OK) return s;
  if (p->flags & PA_FLAG_PORTABLE)
    return fail(PA_ERR_NOT_IMPLEMENTED, "the SEPARATE layout runs on the tensor-core kernels only");
  g->kvh = p->kv_num_heads;
  g->rms_eps = p->rms_eps;
  return PA_OK;
}

pa_status separate_read(Phase ph, const pa_separate_params* p, const void* query,
                        int64_t num_tokens, const void* key_cache, const void* value_cache,
                        const void* cos_cache, const void* sin_cache, const void* q_norm,
                        const void* head_sink, const int32_t* cumseq, const int32_t* past,
                        const int32_t* block_table, int32_t num_seqs, int32_t seq_begin,
                        int32_t seq_end, void* workspace, size_t workspace_bytes, void* out,
                        int32_t* err_flags, void* stream) {
  Geometry g;
  pa_status s = resolve_separate(p, &g);
  if (s != PA_OK) return s;
  if ((s = check_tokens(num_tokens, num_seqs, g)) != PA_OK) return s;
  if (seq_begin < 0 || seq_end < seq_begin || seq_end > num_seqs)
    return fail(PA_ERR_INVALID_ARGUMENT, "sequence range [%d, %d) outside [0, %d)", seq_begin,
                seq_end, num_seqs);
  if (num_tokens == 0 || seq_end == seq_begin) return PA_OK;
  if (ph == Phase::kDecode && (int64_t)(seq_end - seq_begin) > num_tokens)
    return fail(PA_ERR_INVALID_ARGUMENT,
                "decode over %d sequences needs at least that many tokens (have %lld)",
                seq_end - seq_begin, (long long)num_tokens);
  if (!query || !key_cache || !value_cache || !cumseq || !past || !block_table || !out)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (g.rd > 0 && (!cos_cache || !sin_cache))
    return fail(PA_ERR_INVALID_ARGUMENT, "cos_cache/sin_cache are required when rotary_dim > 0");
  if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(out, 16) || (g.rd > 0 && (!aligned(cos_cache, 16) || !aligned(sin_cache, 16))) ||
      (q_norm && !aligned(q_norm, 16)) || (head_sink && !aligned(head_sink, 2)))
    return fail(PA_ERR_INVALID_ARGUMENT,
                "half-precision tensors must be 16-byte aligned (head_sink 2-byte)");
  if (!aligned(cumseq, 4) || !aligned(past, 4) || !aligned(block_table, 4) ||
      !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  if (workspace && !aligned(workspace, 256))
    return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (!separate_supported(g, ph))
    return fail(PA_ERR_NOT_IMPLEMENTED,
                "SEPARATE layout: head_size and v_head_size in 64..256 and at most 128 query "
                "heads per kv head run on the tensor-core kernels; this geometry does not");
  const size_t need = separate_call_workspace(g, ph, seq_begin, seq_end);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace ? workspace_bytes : (size_t)0, need);
  ReadArgs a{query,     num_tokens, key_cache,   value_cache, head_sink,   q_norm,
             cos_cache, sin_cache,  cumseq,      past,        block_table, num_seqs,
             seq_begin, seq_end,    seq_begin,   seq_end,     workspace,   workspace_bytes,
             out,       err_flags,  reinterpret_cast<cudaStream_t>(stream)};
  return cuda_status(launch_separate_read(g, ph, a), "SEPARATE attention launch");
}

// One read call over a whole batch: decode splits for sequences [0, nd)
// and prefill units for [nd, num_seqs) in one attention launch where the
// single-CTA tensor-core kernels run; otherwise a decode call and a prefill
// call in that order.
pa_status mixed_read(const pa_latent_params* p, const void* query, int64_t num_tokens,
                     const void* key_cache, const void* cos_cache, const void* sin_cache,
                     const int32_t* cumseq, const int32_t* past, const int32_t* block_table,
                     int32_t num_seqs, int32_t nd, void* workspace, size_t workspace_bytes,
                     void* out, int32_t* err_flags, void* stream) {
  Geometry g;
  pa_status s = resolve(p, &g);
  if (s != PA_OK) return s;
  if (nd < 0 || nd > num_seqs)
    return fail(PA_ERR_INVALID_ARGUMENT, "num_decode_seqs %d outside [0, %d]", nd, num_seqs);
  const bool one_grid = nd > 0 && nd < num_seqs && use_tc(g, Phase::kMixed);
  if (!one_grid) {
    if (nd > 0) {
      s = read_phase(Phase::kDecode, p, query, num_tokens, key_cache, cos_cache, sin_cache,
                     cumseq, past, block_table, num_seqs, 0, nd, workspace, workspace_bytes, out,
                     err_flags, stream);
      if (s != PA_OK) return s;
    }
    if (nd == num_seqs) return PA_OK;
    // a prefill call that follows the decode call reads no earlier write
    pa_latent_params q = *p;
    if (nd > 0) q.flags &= ~(PA_FLAG_AFTER_WRITE | PA_FLAG_OWN_SLOTS);
    return read_phase(Phase::kPrefill, &q, query, num_tokens, key_cache, cos_cache, sin_cache,
                      cumseq, past, block_table, num_seqs, nd, num_seqs, workspace,
                      workspace_bytes, out, err_flags, stream);
  }
  if ((s = check_tokens(num_tokens, num_seqs, g)) != PA_OK) return s;
  if ((int64_t)nd > num_tokens)
    return fail(PA_ERR_INVALID_ARGUMENT,
                "decode over %d sequences needs at least that many tokens (have %lld)", nd,
                (long long)num_tokens);
  if (!query || !key_cache || !cumseq || !past || !block_table || !out)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (g.rd > 0 && (!cos_cache || !sin_cache))
    return fail(PA_ERR_INVALID_ARGUMENT, "cos_cache/sin_cache are required when rotary_dim > 0");
  if (!aligned(query, 16) || !aligned(key_cache, 16) || !aligned(out, 16) ||
      (g.rd > 0 && (!aligned(cos_cache, 16) || !aligned(sin_cache, 16))))
    return fail(PA_ERR_INVALID_ARGUMENT, "half-precision tensors must be 16-byte aligned");
  if (!aligned(cumseq, 4) || !aligned(past, 4) || !aligned(block_table, 4) ||
      !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  if (workspace && !aligned(workspace, 256))
    return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  const size_t need = tc_call_workspace(g, Phase::kMixed, 0, nd);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace ? workspace_bytes : (size_t)0, need);
  ReadArgs a{query,     num_tokens, key_cache, nullptr, nullptr,     nullptr,
             cos_cache, sin_cache,  cumseq,    past,    block_table, num_seqs,
             0,         nd,         nd,        num_seqs, workspace,  workspace_bytes,
             out,       err_flags,  reinterpret_cast<cudaStream_t>(stream)};
  return cuda_status(launch_tc(g, Phase::kMixed, a), "tensor-core attention launch (mixed)");
}

pa_status record_error(pa_status s, const char* msg) { return fail(s, "%s", msg); }

void set_launch_step(const char* step) { g_launch_step = step; }

pa_status decode_call_workspace(const pa_latent_params* p, int32_t seq_begin, int32_t seq_end,
                                size_t* need) {
  Geometry g;
  const pa_status s = resolve(p, &g);
  if (s != PA_OK) return s;
  *need = seq_end > seq_begin && seq_begin >= 0
              ? call_workspace(g, Phase::kDecode, seq_begin, seq_end, seq_end - seq_begin)
              : 0;
  return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_latent_validate(const pa_latent_params* p) {
  Geometry g;
  return resolve(p, &g);
}

pa_status pa_latent_write(const pa_latent_params* p, const void* key, int64_t num_tokens,
                          const void* cos_cache, const void* sin_cache,
                          const int32_t* slot_mapping, const int32_t* cumseq,
                          const int32_t* past, int32_t num_seqs, void* key_cache,
                          int32_t* err_flags, void* stream) {
  Geometry g;
  pa_status s = resolve(p, &g);
  if (s != PA_OK) return s;
  if ((s = check_tokens(num_tokens, num_seqs, g)) != PA_OK) return s;
  if (num_tokens == 0) return PA_OK;
  if (num_seqs < 1) return fail(PA_ERR_INVALID_ARGUMENT, "tokens given but num_seqs is 0");
  if (!key || !slot_mapping || !cumseq || !past || !key_cache)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (g.rd > 0 && (!cos_cache || !sin_cache))
    return fail(PA_ERR_INVALID_ARGUMENT, "cos_cache/sin_cache are required when rotary_dim > 0");
  if (!aligned(key, 16) || !aligned(key_cache, 16) ||
      (g.rd > 0 && (!aligned(cos_cache, 16) || !aligned(sin_cache, 16))))
    return fail(PA_ERR_INVALID_ARGUMENT, "half-precision tensors must be 16-byte aligned");
  if (!aligned(slot_mapping, 4) || !aligned(cumseq, 4) || !aligned(past, 4) ||
      !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  return cuda_status(launch_write(g, key, num_tokens, cos_cache, sin_cache, slot_mapping, cumseq,
                                  past, num_seqs, key_cache, err_flags,
                                  reinterpret_cast<cudaStream_t>(stream)),
                     "write launch");
}

pa_status pa_latent_decode(const pa_latent_params* p, const void* query, int64_t num_tokens,
                           const void* key_cache, const void* cos_cache,
                           const void* sin_cache, const int32_t* cumseq,
                           const int32_t* past, const int32_t* block_table,
                           int32_t num_seqs, int32_t seq_begin, int32_t seq_end,
                           void* workspace, size_t workspace_bytes, void* out,
                           int32_t* err_flags, void* stream) {
  return read_phase(Phase::kDecode, p, query, num_tokens, key_cache, cos_cache, sin_cache, cumseq,
                    past, block_table, num_seqs, seq_begin, seq_end, workspace, workspace_bytes,
                    out, err_flags, stream);
}

pa_status pa_latent_prefill(const pa_latent_params* p, const void* query, int64_t num_tokens,
                            const void* key_cache, const void* cos_cache,
                            const void* sin_cache, const int32_t* cumseq,
                            const int32_t* past, const int32_t* block_table,
                            int32_t num_seqs, int32_t seq_begin, int32_t seq_end,
                            void* workspace, size_t workspace_bytes, void* out,
                            int32_t* err_flags, void* stream) {
  return read_phase(Phase::kPrefill, p, query, num_tokens, key_cache, cos_cache, sin_cache,
                    cumseq, past, block_table, num_seqs, seq_begin, seq_end, workspace,
                    workspace_bytes, out, err_flags, stream);
}

pa_status pa_latent_mixed(const pa_latent_params* p, const void* query, int64_t num_tokens,
                          const void* key_cache, const void* cos_cache, const void* sin_cache,
                          const int32_t* cumseq, const int32_t* past,
                          const int32_t* block_table, int32_t num_seqs,
                          int32_t num_decode_seqs, void* workspace, size_t workspace_bytes,
                          void* out, int32_t* err_flags, void* stream) {
  return mixed_read(p, query, num_tokens, key_cache, cos_cache, sin_cache, cumseq, past,
                    block_table, num_seqs, num_decode_seqs, workspace, workspace_bytes, out,
                    err_flags, stream);
}

pa_status pa_latent_gather_probe(const pa_latent_params* p, const void* key_cache,
                                 const int32_t* past, const int32_t* block_table,
                                 int32_t num_seqs, int32_t tile_keys, int32_t stages,
                                 int32_t ctas_per_sm, int32_t* err_flags, void* stream) {
  Geometry g;
  pa_status s = resolve(p, &g);
  if (s != PA_OK) return s;
  if (g.fp8) return fail(PA_ERR_NOT_IMPLEMENTED, "the gather probe reads 16-bit caches only");
  if (num_seqs < 1 || num_seqs > 4096)
    return fail(PA_ERR_INVALID_ARGUMENT, "num_seqs must be in 1..4096");
  if (tile_keys != 32 && tile_keys != 64 && tile_keys != 128)
    return fail(PA_ERR_INVALID_ARGUMENT, "tile_keys must be 32, 64 or 128");
  if (stages < 1 || stages > 8) return fail(PA_ERR_INVALID_ARGUMENT, "stages must be in 1..8");
  if (ctas_per_sm < 1 || ctas_per_sm > 4)
    return fail(PA_ERR_INVALID_ARGUMENT, "ctas_per_sm must be in 1..4");
  if (gather_probe_smem(g, tile_keys, stages, num_seqs) > kMaxProbeSmem)
    return fail(PA_ERR_INVALID_ARGUMENT, "stages x tile exceed the probe's shared memory");
  if (!key_cache || !past || !block_table || !err_flags)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (!aligned(key_cache, 16))
    return fail(PA_ERR_INVALID_ARGUMENT, "key_cache must be 16-byte aligned");
  if (!aligned(past, 4) || !aligned(block_table, 4) || !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  return cuda_status(launch_gather_probe(g, key_cache, past, block_table, num_seqs, tile_keys,
                                         stages, ctas_per_sm, err_flags,
                                         reinterpret_cast<cudaStream_t>(stream)),
                     "gather probe launch");
}

size_t pa_latent_workspace_size(const pa_latent_params* p, int32_t num_seqs,
                                int64_t num_tokens) {
  Geometry g;
  if (resolve(p, &g) != PA_OK) return 0;
  if (num_seqs <= 0 || num_tokens <= 0) return 0;
  size_t need = 0;
  for (Phase ph : {Phase::kDecode, Phase::kPrefill}) {
    size_t n = use_tc(g, ph) ? tc_workspace_bytes(g, ph, num_seqs, num_tokens)
                             : portable_workspace_bytes(g, ph, num_seqs, num_tokens);
    if (n > need) need = n;
  }
  return need;
}

int32_t pa_latent_kernel_family(const pa_latent_params* p, int32_t phase) {
  Geometry g;
  if (resolve(p, &g) != PA_OK || (phase != 0 && phase != 1)) return -1;
  return use_tc(g, phase == 0 ? Phase::kDecode : Phase::kPrefill) ? 1 : 0;
}

const char* pa_latent_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARGUMENT: return "PA_ERR_INVALID_ARGUMENT";
    case PA_ERR_NOT_IMPLEMENTED: return "PA_ERR_NOT_IMPLEMENTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_latent_last_error(void) { return g_last_error.c_str(); }

pa_status pa_separate_validate(const pa_separate_params* p) {
  Geometry g;
  return resolve_separate(p, &g);
}

pa_status pa_separate_write(const pa_separate_params* p, const void* key, const void* value,
                            int64_t num_tokens, const void* cos_cache, const void* sin_cache,
                            const void* k_norm_weight, const int32_t* slot_mapping,
                            const int32_t* cumseq, const int32_t* past, int32_t num_seqs,
                            void* key_cache, void* value_cache, int32_t* err_flags,
                            void* stream) {
  Geometry g;
  pa_status s = resolve_separate(p, &g);
  if (s != PA_OK) return s;
  if ((s = check_tokens(num_tokens, num_seqs, g)) != PA_OK) return s;
  if (num_tokens == 0) return PA_OK;
  if (num_seqs < 1) return fail(PA_ERR_INVALID_ARGUMENT, "tokens given but num_seqs is 0");
  if (g.hs > 256 || g.vhs % 8 != 0 || g.vhs > 256)
    return fail(PA_ERR_NOT_IMPLEMENTED,
                "SEPARATE write: head_size <= 256 and v_head_size a multiple of 8 <= 256");
  if (!key || !value || !slot_mapping || !cumseq || !past || !key_cache || !value_cache)
    return fail(PA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (g.rd > 0 && (!cos_cache || !sin_cache))
    return fail(PA_ERR_INVALID_ARGUMENT, "cos_cache/sin_cache are required when rotary_dim > 0");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || (k_norm_weight && !aligned(k_norm_weight, 16)) ||
      (g.rd > 0 && (!aligned(cos_cache, 16) || !aligned(sin_cache, 16))))
    return fail(PA_ERR_INVALID_ARGUMENT, "half-precision tensors must be 16-byte aligned");
  if (!aligned(slot_mapping, 4) || !aligned(cumseq, 4) || !aligned(past, 4) ||
      !aligned(err_flags, 4))
    return fail(PA_ERR_INVALID_ARGUMENT, "int32 tensors must be 4-byte aligned");
  SeparateWriteArgs a{key,    value,       num_tokens, cos_cache, sin_cache, k_norm_weight,
                      slot_mapping, cumseq, past, num_seqs, key_cache, value_cache, err_flags,
                      reinterpret_cast<cudaStream_t>(stream)};
  return cuda_status(launch_separate_write(g, a), "SEPARATE write launch");
}

pa_status pa_separate_decode(const pa_separate_params* p, const void* query, int64_t num_tokens,
                             const void* key_cache, const void* value_cache,
                             const void* cos_cache, const void* sin_cache,
                             const void* q_norm_weight, const void* head_sink,
                             const int32_t* cumseq, const int32_t* past,
                             const int32_t* block_table, int32_t num_seqs, int32_t seq_begin,
                             int32_t seq_end, void* workspace, size_t workspace_bytes, void* out,
                             int32_t* err_flags, void* stream) {
  return separate_read(Phase::kDecode, p, query, num_tokens, key_cache, value_cache, cos_cache,
                       sin_cache, q_norm_weight, head_sink, cumseq, past, block_table, num_seqs,
                       seq_begin, seq_end, workspace, workspace_bytes, out, err_flags, stream);
}

pa_status pa_separate_prefill(const pa_separate_params* p, const void* query,
                              int64_t num_tokens, const void* key_cache, const void* value_cache,
                              const void* cos_cache, const void* sin_cache,
                              const void* q_norm_weight, const void* head_sink,
                              const int32_t* cumseq, const int32_t* past,
                              const int32_t* block_table, int32_t num_seqs, int32_t seq_begin,
                              int32_t seq_end, void* workspace, size_t workspace_bytes,
                              void* out, int32_t* err_flags, void* stream) {
  return separate_read(Phase::kPrefill, p, query, num_tokens, key_cache, value_cache, cos_cache,
                       sin_cache, q_norm_weight, head_sink, cumseq, past, block_table, num_seqs,
                       seq_begin, seq_end, workspace, workspace_bytes, out, err_flags, stream);
}

size_t pa_separate_workspace_size(const pa_separate_params* p, int32_t num_seqs,
                                  int64_t num_tokens) {
  Geometry g;
  if (resolve_separate(p, &g) != PA_OK || num_seqs <= 0 || num_tokens <= 0) return 0;
  return separate_call_workspace(g, Phase::kDecode, 0, num_seqs);
}

}  // extern "C"
