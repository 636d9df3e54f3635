// Write phase: partial RoPE on each new latent key row, scattered into the
// paged cache (paged_attention.rs, module doc "Write phase" / write_impl).
//
// One thread per (token, 8-channel group): a 16-byte load of the group, a
// 16-byte load of its rotary partner group when the group is rotary, and a
// 16-byte store into the cache row. Rows are 16-byte aligned (hs % 16 == 0)
// so every access is a full vector; a warp covers 32 consecutive groups,
// i.e. whole rows, so loads and stores are coalesced. HBM traffic is the
// algorithmic minimum: each key row read once (plus its 128-byte rotary
// partner slice, which hits L1), each written row stored once.
#include <cuda_fp8.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// Largest batch whose cumulative offsets are staged in shared memory (the
// token -> sequence search then runs on chip instead of as a chain of
// dependent global loads).
constexpr int kStagedSeqs = 8191;

// FP8 = the cache holds E4M3 codes: each channel's (rotated) value v is
// stored as e4m3(v / k_scale), the division an IEEE f32 one, the conversion
// rounding to nearest even and saturating at +-448.
template <typename T, bool FP8>
__global__ void __launch_bounds__(256)
latent_write_kernel(const T* __restrict__ key, const T* __restrict__ cos_cache,
                    const T* __restrict__ sin_cache, const int32_t* __restrict__ slot_mapping,
                    const int32_t* __restrict__ cumseq, const int32_t* __restrict__ past,
                    int32_t num_seqs, void* __restrict__ key_cache, int64_t num_tokens, int hs,
                    int ro, int rd, int interleaved, int cos_rows, int64_t num_slots,
                    float k_scale, int32_t* err_flags) {
  // A kernel launched after this one with programmatic dependent launch may
  // start its prologue now; it waits (griddepcontrol.wait) for this grid to
  // complete before it reads the cache.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ int32_t s_cum[];  // cumseq[0..num_seqs] when staged
  const bool staged = num_seqs <= kStagedSeqs;
  if (staged) {
    for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) s_cum[i] = cumseq[i];
    __syncthreads();
  }
  const int32_t* cum = staged ? s_cum : cumseq;
  const int groups = hs >> 3;
  const int64_t total = num_tokens * groups;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / groups;
    const int g = (int)(i - t * groups);
    const int d0 = g << 3;
    const T* row = key + t * hs;
    // loads that depend on nothing else go out first
    const int32_t slot = slot_mapping[t];
    uint4 v = *reinterpret_cast<const uint4*>(row + d0);
    const bool rot = rd > 0 && d0 >= ro && d0 < ro + rd;
    uint4 vp = v;
    if (rot && !interleaved) {
      const int half = rd >> 1;
      const int dp = (d0 - ro < half) ? d0 + half : d0 - half;
      vp = *reinterpret_cast<const uint4*>(row + dp);
    }
    if (slot < 0) {
      if (slot < -1 && g == 0) raise_flag(err_flags, PA_DEVERR_SLOT);
      continue;
    }
    if ((int64_t)slot >= num_slots) {
      if (g == 0) raise_flag(err_flags, PA_DEVERR_SLOT);
      continue;
    }
    int32_t b;
    int64_t pos;
    if (!locate_token(t, cum, past, num_seqs, g == 0 ? err_flags : nullptr, &b, &pos))
      continue;
    if (rd > 0 && (pos < 0 || pos >= cos_rows)) {  // whole row skipped
      if (g == 0) raise_flag(err_flags, pos < 0 ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
      continue;
    }
    if (FP8) {
      float x[8];
      unpack8<T>(v, x);
      if (rot) {
        float xp[8];
        unpack8<T>(vp, xp);
        rope8<T>(x, xp, d0, ro, rd, interleaved, cos_cache + pos * (rd >> 1),
                 sin_cache + pos * (rd >> 1));
      }
      uint32_t w[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * k], k_scale), __fdiv_rn(x[4 * k + 1], k_scale)),
            __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * k + 2], k_scale), __fdiv_rn(x[4 * k + 3], k_scale)),
            __NV_SATFINITE, __NV_E4M3);
        w[k] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(key_cache) + (int64_t)slot * hs + d0) =
          make_uint2(w[0], w[1]);
      continue;
    }
    if (rot) {
      float x[8], xp[8];
      unpack8<T>(v, x);
      unpack8<T>(vp, xp);
      const T* crow = cos_cache + pos * (rd >> 1);
      const T* srow = sin_cache + pos * (rd >> 1);
      rope8<T>(x, xp, d0, ro, rd, interleaved, crow, srow);
      v = pack8<T>(x);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<T*>(key_cache) + (int64_t)slot * hs + d0) = v;
  }
}

cudaError_t launch_write(const Geometry& g, const void* key, int64_t num_tokens,
                         const void* cos_cache, const void* sin_cache,
                         const int32_t* slot_mapping, const int32_t* cumseq, const int32_t* past,
                         int32_t num_seqs, void* key_cache, int32_t* err_flags,
                         cudaStream_t stream) {
  const int64_t total = num_tokens * (g.hs >> 3);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)g.num_sms * 16;
  if (blocks > cap) blocks = cap;
  const int64_t num_slots = (int64_t)g.num_blocks * g.bs;
  const size_t smem = num_seqs <= kStagedSeqs ? (size_t)(num_seqs + 1) * sizeof(int32_t) : 0;
  auto go = [&](auto kern, auto* typed) {
    using TP = std::remove_pointer_t<decltype(typed)>;
    kern<<<(unsigned)blocks, threads, smem, stream>>>(
        (const TP*)key, (const TP*)cos_cache, (const TP*)sin_cache, slot_mapping, cumseq, past,
        num_seqs, key_cache, num_tokens, g.hs, g.ro, g.rd, g.interleaved, g.cos_rows, num_slots,
        g.k_scale, err_flags);
  };
  if (g.dtype == PA_DTYPE_BF16) {
    if (g.fp8) go(latent_write_kernel<__nv_bfloat16, true>, (__nv_bfloat16*)nullptr);
    else go(latent_write_kernel<__nv_bfloat16, false>, (__nv_bfloat16*)nullptr);
  } else {
    if (g.fp8) go(latent_write_kernel<__half, true>, (__half*)nullptr);
    else go(latent_write_kernel<__half, false>, (__half*)nullptr);
  }
  return cudaGetLastError();
}

}  // namespace pa

