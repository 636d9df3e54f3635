// Device helpers shared by the paged LATENT attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_latent.h"

namespace pa {

// Largest latent width the kernels accept (register and shared-memory budget
// of the portable kernel).
constexpr int kMaxHeadSize = 1024;

// ---------------------------------------------------------------------------
// Half-precision element traits
// ---------------------------------------------------------------------------
template <typename T> struct Half;
template <> struct Half<__half> {
  static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};
template <> struct Half<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// 8 half-precision values moved as one 16-byte vector.
template <typename T>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const T* h = reinterpret_cast<const T*>(&v);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = Half<T>::to_f32(h[i]);
}
template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  T* h = reinterpret_cast<T*>(&v);
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = Half<T>::from_f32(f[i]);
  return v;
}

__device__ __forceinline__ void raise_flag(int32_t* flags, int32_t bit) {
  if (flags) atomicOr(flags, bit);
}

// ---------------------------------------------------------------------------
// Token -> (sequence, absolute position). The sequence is the b with
// cumseq[b] <= t < cumseq[b+1] (the first b whose end exceeds t), found by
// binary search over the monotone offsets; the position is past[b] + t -
// cumseq[b]. Returns false (and flags the error) when t is not inside
// [cumseq[0], cumseq[B]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool locate_token(int64_t t, const int32_t* __restrict__ cumseq,
                                             const int32_t* __restrict__ past, int32_t num_seqs,
                                             int32_t* flags, int32_t* b_out, int64_t* pos_out) {
  if (num_seqs <= 0 || t < cumseq[0] || t >= cumseq[num_seqs]) {
    raise_flag(flags, PA_DEVERR_CUMSEQ);
    return false;
  }
  int lo = 0, hi = num_seqs - 1;  // answer in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (t < cumseq[mid + 1]) hi = mid; else lo = mid + 1;
  }
  if (t < cumseq[lo]) {  // offsets not monotone
    raise_flag(flags, PA_DEVERR_CUMSEQ);
    return false;
  }
  *b_out = lo;
  *pos_out = (int64_t)past[lo] + (t - cumseq[lo]);
  return true;
}

// Rotates 8 consecutive channels [d0, d0+8) of a row held in `x` (f32) with
// their partner channels `xp` (f32). Channels inside [ro, ro+rd) only; the
// caller guarantees the 8-channel group lies entirely inside or outside the
// rotary range (ro % 8 == 0, rd % 16 == 0).
//   non-interleaved: i = d - ro; first half  out = x c_i - x[d+rd/2] s_i,
//                               second half out = x c_{i-rd/2} + x[d-rd/2] s_{i-rd/2}
//   interleaved:     i = (d - ro)/2; even out = x c_i - x[d+1] s_i,
//                                    odd  out = x c_i + x[d-1] s_i
// The partner values for interleaved rows come from x itself.
template <typename T>
__device__ __forceinline__ void rope8(float (&x)[8], const float (&xp)[8], int d0, int ro, int rd,
                                      int interleaved, const T* __restrict__ cos_row,
                                      const T* __restrict__ sin_row) {
  const int r = d0 - ro;
  const int half = rd >> 1;
  if (!interleaved) {
    const int i0 = r < half ? r : r - half;
    const float sign = r < half ? -1.f : 1.f;
    float c[8], s[8];
    unpack8<T>(*reinterpret_cast<const uint4*>(cos_row + i0), c);
    unpack8<T>(*reinterpret_cast<const uint4*>(sin_row + i0), s);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = fmaf(x[k], c[k], sign * xp[k] * s[k]);
  } else {
    const int i0 = r >> 1;  // 4 angle entries for 8 channels
    float y[8];
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const float c = Half<T>::to_f32(cos_row[i0 + (k >> 1)]);
      const float s = Half<T>::to_f32(sin_row[i0 + (k >> 1)]);
      y[k] = fmaf(x[k], c, -x[k + 1] * s);
      y[k + 1] = fmaf(x[k + 1], c, x[k] * s);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = y[k];
  }
}

}  // namespace pa
