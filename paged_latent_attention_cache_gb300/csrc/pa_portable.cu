// Portable read phase on CUDA cores: correct for every geometry the
// validator accepts (any head count, hs a multiple of 16 up to 1024, any
// v_head_size), used where no tensor-core kernel is specialised and as a
// cross-check of the tensor-core kernels.
//
// Operator (paged_attention.rs, module doc "Read phase" / attn_impl): for
// each query token t (sequence b, position pos) and head h,
//   q = RoPE(query[t, h]) kept in f32,
//   s_j = scale * q . K_j for keys j in [max(0, pos - window), pos]
//         (K_j the cache row block_table[b, j/bs]*bs + j%bs),
//   s_j = softcap * tanh(s_j / softcap) if softcap > 0,
//   out = sum_j softmax(s)_j K_j[:vhs].
// The softmax is evaluated online (running max m, denominator l and
// accumulator rescaled by exp(m_old - m_new)), the form the pages' kernel
// uses and which equals the two-pass definition algebraically.
//
// Shape of the kernel: one CTA of 4 warps per (query, group of 4 heads,
// key split); each warp owns one head. Keys stream through shared memory in
// tiles of 32 rows gathered through the block table with 16-byte loads;
// in a tile, lane r scores key r (a full-row dot product against the
// broadcast query), the warp reduces max/sum with shuffles, and each lane
// accumulates 8 value channels per 256 for all 32 keys. With more than one
// key split the CTA writes (m, l, unnormalised accumulator) to the
// workspace and a combine kernel merges the splits by log-sum-exp.
#include <math.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 4;    // heads per CTA
constexpr int kTile = 32;    // keys per shared-memory tile

struct PortableParams {
  const void* query;
  const void* key_cache;
  const void* cos_cache;
  const void* sin_cache;
  const int32_t* cumseq;
  const int32_t* past;
  const int32_t* block_table;
  void* out;
  float* ws_acc;    // [Q][S][H][vhs]
  float* ws_ml;     // [Q][S][H][2]
  int32_t* err_flags;
  int64_t num_tokens;
  int num_seqs, seq_begin, seq_end;
  int H, hs, vhs, ro, rd, interleaved, cos_rows, bs, num_blocks, max_blocks;
  float scale, softcap;
  int window;
  int splits;
  int decode;       // 1: query slot x is sequence seq_begin + x (q_len must be 1)
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Resolves the query slot of this CTA to (token, sequence, position).
// Returns false when the CTA has nothing to do.
__device__ __forceinline__ bool resolve_query(const PortableParams& P, int64_t x, int64_t* t,
                                              int32_t* b, int64_t* pos, bool report) {
  if (P.decode) {
    const int32_t bb = P.seq_begin + (int32_t)x;
    const int32_t q0 = P.cumseq[bb], q1 = P.cumseq[bb + 1];
    if (q1 - q0 != 1) {
      if (report) raise_flag(P.err_flags, PA_DEVERR_DECODE_QLEN);
      return false;
    }
    if (q0 < 0 || q0 >= P.num_tokens) {
      if (report) raise_flag(P.err_flags, PA_DEVERR_CUMSEQ);
      return false;
    }
    *t = q0;
    *b = bb;
    *pos = (int64_t)P.past[bb];
    return true;
  }
  if (!locate_token(x, P.cumseq, P.past, P.num_seqs, report ? P.err_flags : nullptr, b, pos))
    return false;
  if (*b < P.seq_begin || *b >= P.seq_end) return false;
  *t = x;
  return true;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kWarps * 32)
portable_attn_kernel(PortableParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int hs = P.hs, vhs = P.vhs;
  const int kstride = hs + 8;                      // padded row (bank-conflict free)
  float* q_s = reinterpret_cast<float*>(smem_raw);                  // [kWarps][hs]
  T* k_s = reinterpret_cast<T*>(q_s + kWarps * hs);                 // [kTile][kstride]
  int64_t* rowoff = reinterpret_cast<int64_t*>(k_s + kTile * kstride);  // [kTile]
  __shared__ int bad_block;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWarps + warp;
  const int split = blockIdx.z;
  const bool report = (threadIdx.x == 0 && blockIdx.y == 0 && split == 0);

  int64_t t, pos;
  int32_t b;
  if (!resolve_query(P, blockIdx.x, &t, &b, &pos, report)) return;
  const int64_t ctx_cap = (int64_t)P.max_blocks * P.bs;
  const bool bad_ctx = P.past[b] < 0 || pos >= ctx_cap;
  const bool bad_pos = P.rd > 0 && pos >= P.cos_rows;
  const int64_t q_index = P.decode ? (int64_t)blockIdx.x : 0;
  T* out_row = reinterpret_cast<T*>(P.out) + t * (int64_t)P.H * vhs;

  if (bad_ctx || bad_pos) {
    if (report) raise_flag(P.err_flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
    if (split == 0 && h < P.H)
      for (int c = lane; c < vhs; c += 32) out_row[h * vhs + c] = Half<T>::from_f32(0.f);
    return;
  }

  // Key range of this split.
  const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
  const int64_t n = pos + 1 - lo;
  const int64_t chunk = (n + P.splits - 1) / P.splits;
  const int64_t k_begin = lo + (int64_t)split * chunk;
  const int64_t k_end = min(pos + 1, k_begin + chunk);

  // Post-RoPE query rows in f32.
  if (h < P.H) {
    const T* qrow = reinterpret_cast<const T*>(P.query) + t * (int64_t)P.H * hs + (int64_t)h * hs;
    const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * (P.rd >> 1);
    const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * (P.rd >> 1);
    for (int d0 = lane * 8; d0 < hs; d0 += 256) {
      float x[8], xp[8];
      unpack8<T>(*reinterpret_cast<const uint4*>(qrow + d0), x);
      if (P.rd > 0 && d0 >= P.ro && d0 < P.ro + P.rd) {
        if (!P.interleaved) {
          const int half = P.rd >> 1;
          const int dp = (d0 - P.ro < half) ? d0 + half : d0 - half;
          unpack8<T>(*reinterpret_cast<const uint4*>(qrow + dp), xp);
        }
        rope8<T>(x, xp, d0, P.ro, P.rd, P.interleaved, crow, srow);
      }
      float4* dst = reinterpret_cast<float4*>(q_s + warp * hs + d0);
      dst[0] = make_float4(x[0], x[1], x[2], x[3]);
      dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  if (threadIdx.x == 0) bad_block = 0;

  float m = -INFINITY, l = 0.f;
  float acc[NV][8];
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;

  const T* cache = reinterpret_cast<const T*>(P.key_cache);
  const int vec_per_row = hs >> 3;
  for (int64_t j0 = k_begin; j0 < k_end; j0 += kTile) {
    __syncthreads();  // previous tile consumed (and q_s / bad_block visible)
    if (threadIdx.x < kTile) {
      const int64_t j = j0 + threadIdx.x;
      int64_t off = -1;
      if (j < k_end) {
        const int32_t phys = P.block_table[(int64_t)b * P.max_blocks + j / P.bs];
        if (phys >= 0 && phys < P.num_blocks) {
          off = ((int64_t)phys * P.bs + j % P.bs) * hs;
        } else {
          bad_block = 1;
          raise_flag(P.err_flags, PA_DEVERR_BLOCK);
        }
      }
      rowoff[threadIdx.x] = off;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < kTile * vec_per_row; v += kWarps * 32) {
      const int r = v / vec_per_row, c = v - r * vec_per_row;
      const int64_t off = rowoff[r];
      uint4 val = make_uint4(0, 0, 0, 0);
      if (off >= 0) val = *reinterpret_cast<const uint4*>(cache + off + c * 8);
      *reinterpret_cast<uint4*>(k_s + r * kstride + c * 8) = val;
    }
    __syncthreads();
    if (h >= P.H) continue;

    // Scores: lane r <-> key j0 + r.
    float s = -INFINITY;
    if (rowoff[lane] >= 0) {
      const T* kr = k_s + lane * kstride;
      const float* qr = q_s + warp * hs;
      float dot = 0.f;
      for (int d0 = 0; d0 < hs; d0 += 8) {
        float kx[8];
        unpack8<T>(*reinterpret_cast<const uint4*>(kr + d0), kx);
        const float4 qa = *reinterpret_cast<const float4*>(qr + d0);
        const float4 qb = *reinterpret_cast<const float4*>(qr + d0 + 4);
        dot = fmaf(qa.x, kx[0], dot); dot = fmaf(qa.y, kx[1], dot);
        dot = fmaf(qa.z, kx[2], dot); dot = fmaf(qa.w, kx[3], dot);
        dot = fmaf(qb.x, kx[4], dot); dot = fmaf(qb.y, kx[5], dot);
        dot = fmaf(qb.z, kx[6], dot); dot = fmaf(qb.w, kx[7], dot);
      }
      s = dot * P.scale;
      if (P.softcap > 0.f) s = P.softcap * tanhf(s / P.softcap);
    }
    const float m_new = fmaxf(m, warp_max(s));
    const float corr = (m == -INFINITY) ? 0.f : __expf(m - m_new);
    const float p = (s == -INFINITY) ? 0.f : __expf(s - m_new);
    l = l * corr + warp_sum(p);
    m = m_new;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[k][e] *= corr;
    for (int r = 0; r < kTile; ++r) {
      const float pr = __shfl_sync(0xffffffffu, p, r);
      if (pr == 0.f) continue;  // warp-uniform
      const T* vr = k_s + r * kstride;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int c0 = lane * 8 + k * 256;
        if (c0 < vhs) {
          float vx[8];
          unpack8<T>(*reinterpret_cast<const uint4*>(vr + c0), vx);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[k][e] = fmaf(pr, vx[e], acc[k][e]);
        }
      }
    }
  }
  __syncthreads();
  if (h >= P.H) return;
  const bool zero = bad_block != 0;

  if (P.splits == 1) {
    const float inv = (l > 0.f && !zero) ? 1.f / l : 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int c0 = lane * 8 + k * 256;
      if (c0 >= vhs) continue;
      T* dst = out_row + h * vhs + c0;
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = acc[k][e] * inv;
      if ((vhs & 7) == 0) {
        *reinterpret_cast<uint4*>(dst) = pack8<T>(o);
      } else {
        for (int e = 0; e < 8 && c0 + e < vhs; ++e) dst[e] = Half<T>::from_f32(o[e]);
      }
    }
    return;
  }
  // Split partial: (m, l, unnormalised accumulator).
  const int64_t base = (q_index * P.splits + split) * P.H + h;
  float* wacc = P.ws_acc + base * vhs;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int c0 = lane * 8 + k * 256;
    for (int e = 0; e < 8 && c0 + e < vhs; ++e) wacc[c0 + e] = zero ? 0.f : acc[k][e];
  }
  if (lane == 0) {  // a NaN max marks a split that read an invalid block
    P.ws_ml[base * 2 + 0] = zero ? __int_as_float(0x7fc00000) : m;
    P.ws_ml[base * 2 + 1] = zero ? 0.f : l;
  }
}

// Merges the key splits of one (query, head): with M = max over splits of
// m_s, out = sum_s e^{m_s - M} acc_s / sum_s e^{m_s - M} l_s (0 when the
// denominator is 0, or when any split read an invalid block).
template <typename T>
__global__ void __launch_bounds__(128)
portable_combine_kernel(PortableParams P) {
  const int64_t x = blockIdx.x;
  const int h = blockIdx.y;
  int64_t t, pos;
  int32_t b;
  if (!resolve_query(P, x, &t, &b, &pos, false)) return;
  const int64_t ctx_cap = (int64_t)P.max_blocks * P.bs;
  if (P.past[b] < 0 || pos >= ctx_cap || (P.rd > 0 && pos >= P.cos_rows)) return;
  const int S = P.splits;
  float M = -INFINITY;
  bool bad = false;
  for (int s = 0; s < S; ++s) {
    const float ms = P.ws_ml[((x * S + s) * P.H + h) * 2];
    bad |= isnan(ms);
    M = fmaxf(M, ms);  // fmaxf ignores a NaN operand
  }
  float L = 0.f;
  for (int s = 0; s < S && !bad; ++s) {
    const float* ml = P.ws_ml + ((x * S + s) * P.H + h) * 2;
    if (ml[1] > 0.f) L += __expf(ml[0] - M) * ml[1];
  }
  T* dst = reinterpret_cast<T*>(P.out) + t * (int64_t)P.H * P.vhs + (int64_t)h * P.vhs;
  for (int c = threadIdx.x; c < P.vhs; c += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < S && !bad; ++s) {
      const int64_t base = (x * S + s) * P.H + h;
      const float* ml = P.ws_ml + base * 2;
      if (ml[1] > 0.f) o += __expf(ml[0] - M) * P.ws_acc[base * P.vhs + c];
    }
    dst[c] = Half<T>::from_f32(L > 0.f && !bad ? o / L : 0.f);
  }
}

int portable_splits(const Geometry& g, Phase ph, int32_t num_queries) {
  if (ph == Phase::kPrefill || num_queries <= 0) return 1;
  const int64_t groups = (g.H + kWarps - 1) / kWarps;
  const int64_t ctas = (int64_t)num_queries * groups;
  const int64_t target = 4LL * g.num_sms;
  int64_t s = (target + ctas - 1) / ctas;
  const int64_t max_ctx = (int64_t)g.max_blocks * g.bs;
  const int64_t by_len = (max_ctx + 255) / 256;
  if (s > by_len) s = by_len;
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  return (int)s;
}

size_t smem_bytes(const Geometry& g) {
  return (size_t)kWarps * g.hs * sizeof(float) + (size_t)kTile * (g.hs + 8) * 2 +
         (size_t)kTile * sizeof(int64_t);
}

template <typename T, int NV>
cudaError_t launch_typed(const Geometry& g, Phase ph, const ReadArgs& a, PortableParams& P,
                         int64_t nq) {
  const size_t smem = smem_bytes(g);
  static std::atomic<bool> configured[64];
  cudaError_t e = once_per_device(configured, g.device, [] {
    return cudaFuncSetAttribute(portable_attn_kernel<T, NV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kWarps * pa::kMaxHeadSize * 4 +
                                      kTile * (pa::kMaxHeadSize + 8) * 2 + kTile * 8));
  });
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)nq, (unsigned)((g.H + kWarps - 1) / kWarps), (unsigned)P.splits);
  portable_attn_kernel<T, NV><<<grid, kWarps * 32, smem, a.stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess || P.splits == 1) return e;
  portable_combine_kernel<T><<<dim3((unsigned)nq, (unsigned)g.H), 128, 0, a.stream>>>(P);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_nv(const Geometry& g, Phase ph, const ReadArgs& a, PortableParams& P,
                      int64_t nq) {
  switch ((g.vhs + 255) / 256) {
    case 1: return launch_typed<T, 1>(g, ph, a, P, nq);
    case 2: return launch_typed<T, 2>(g, ph, a, P, nq);
    case 3: return launch_typed<T, 3>(g, ph, a, P, nq);
    default: return launch_typed<T, 4>(g, ph, a, P, nq);
  }
}

}  // namespace

// Workspace of one call that merges `units` (query, split) pairs.
size_t partial_bytes(const Geometry& g, int64_t units) {
  const size_t per = (size_t)units * g.H;
  const size_t acc = ((per * g.vhs * sizeof(float)) + 255) & ~(size_t)255;
  return acc + per * 2 * sizeof(float);
}

size_t portable_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs,
                                int64_t num_tokens) {
  (void)num_tokens;
  if (ph == Phase::kPrefill || num_seqs <= 0) return 0;
  // S(nq) does not grow with nq, so S(1) is the most splits any call gets.
  const int64_t s1 = portable_splits(g, ph, 1);
  if (s1 <= 1) return 0;
  // A call over nq <= num_seqs queries merges nq * S(nq) partials, and
  // nq * S(nq) <= nq * (target/(nq*groups) + 1) <= target/groups + num_seqs.
  const int64_t groups = (g.H + kWarps - 1) / kWarps;
  const int64_t target = 4LL * g.num_sms;
  int64_t units = (target + groups - 1) / groups + num_seqs;
  if (units > s1 * num_seqs) units = s1 * num_seqs;
  return partial_bytes(g, units);
}

size_t portable_call_workspace(const Geometry& g, Phase ph, int64_t nq) {
  const int S = portable_splits(g, ph, (int32_t)nq);
  return S > 1 ? partial_bytes(g, nq * S) : 0;
}

cudaError_t launch_portable(const Geometry& g, Phase ph, const ReadArgs& a) {
  const int64_t nq = ph == Phase::kDecode ? (int64_t)(a.seq_end - a.seq_begin) : a.num_tokens;
  if (nq <= 0) return cudaSuccess;
  PortableParams P;
  P.query = a.query; P.key_cache = a.key_cache;
  P.cos_cache = a.cos_cache; P.sin_cache = a.sin_cache;
  P.cumseq = a.cumseq; P.past = a.past; P.block_table = a.block_table;
  P.out = a.out; P.err_flags = a.err_flags;
  P.num_tokens = a.num_tokens; P.num_seqs = a.num_seqs;
  P.seq_begin = a.seq_begin; P.seq_end = a.seq_end;
  P.H = g.H; P.hs = g.hs; P.vhs = g.vhs; P.ro = g.ro; P.rd = g.rd;
  P.interleaved = g.interleaved; P.cos_rows = g.cos_rows; P.bs = g.bs;
  P.num_blocks = g.num_blocks; P.max_blocks = g.max_blocks;
  P.scale = g.scale; P.softcap = g.softcap; P.window = g.window;
  P.decode = ph == Phase::kDecode ? 1 : 0;
  // Split count is sized for the call's own query count, which never
  // exceeds num_seqs (the workspace bound).
  P.splits = portable_splits(g, ph, (int32_t)nq);
  if (P.splits > 1) {
    if (a.workspace == nullptr || a.workspace_bytes < partial_bytes(g, nq * P.splits))
      return cudaErrorInvalidValue;  // checked by the caller first
    const size_t per = (size_t)nq * P.splits * g.H;
    const size_t acc = ((per * g.vhs * sizeof(float)) + 255) & ~(size_t)255;
    P.ws_acc = reinterpret_cast<float*>(a.workspace);
    P.ws_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(a.workspace) + acc);
  } else {
    P.ws_acc = nullptr;
    P.ws_ml = nullptr;
  }
  if (g.dtype == PA_DTYPE_BF16) return launch_nv<__nv_bfloat16>(g, ph, a, P, nq);
  return launch_nv<__half>(g, ph, a, P, nq);
}

}  // namespace pa
