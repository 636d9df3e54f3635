// Tensor-core read phase for sm_103a: tcgen05 MMAs with TMEM accumulators,
// paged key tiles gathered by TMA through the block table.
//
// Operator (paged_attention.rs, module doc "Read phase" / attn_impl): for a
// query token at position pos and every head h,
//   S[h, j] = scale * RoPE(q_h) . K_j      (K_j: cache row of key j)
//   S = softcap * tanh(S / softcap)        (softcap > 0)
//   out[h] = softmax_j(S[h, :]) @ K[:, :vhs],  keys j in [lo, pos].
// Every head of a token shares the same latent rows, so both products are
// dense contractions with the heads as the M dimension:
//   QK^T : M = 128 rows (heads, zero-padded), N = key tile, K = head_size
//   PV   : M = 128 rows, N = a group of value channels, K = key tile,
// and the key tile staged once in shared memory is the B operand of both
// (K-major for QK^T; its leading value channels read MN-major for PV).
//
// CTA = one query token x one group of value channels (2 groups of 256 when
// vhs = 512: a 128 x 512 f32 accumulator alone fills the 512 TMEM columns, so
// the two groups live on two SMs and each recomputes S), optionally one
// split of the token's keys (decode: splits are merged by a log-sum-exp
// combine kernel). Warp roles:
//   warps 0-3  softmax + epilogue; thread i owns row i (TMEM lane i): loads Q
//              with RoPE into swizzled shared memory, reads S from TMEM,
//              masks/softcaps, runs the online softmax with lazy rescaling
//              (the reference max only moves when it grows by > 2^8), writes
//              P (16-bit) to TMEM, finally normalises O and stores it.
//   warp 4     TMA producer: per key tile, one 2-D box (64 channels x rows of
//              one cache block) per 64-channel slab, 128-byte swizzle.
//   warp 5     TMEM allocation and the single MMA-issuing thread.
// Pipelines: K tiles in a STAGES-deep ring (full/empty mbarriers), S and P
// double-buffered in TMEM. Every mbarrier wait is bounded: on expiry the
// CTA sets PA_DEVERR_TIMEOUT in the error word, drains what it issued and
// exits without trapping.
#include <cuda.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace tc {

constexpr int kThreads = 192;
constexpr int kRows = 128;               // MMA M: TMEM lanes
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;     // lazy-rescale threshold (factor 256)

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// 16 consecutive 32-bit TMEM columns of this thread's lane; the wait is in
// the same statement so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format):
// start address, leading / stride byte offsets (>> 4), version 1, layout 2.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: f32 accumulator, A/B both bf16 or
// both f16, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Parameters
// ---------------------------------------------------------------------------
struct Params {
  const void* query;
  void* out;
  float* ws_o;      // [units][G][128][VG]   (key-split partials, decode)
  float* ws_ml;     // [units][G][128][2]    (log2-domain max, denominator)
  const void* cos_cache;
  const void* sin_cache;
  const int32_t* cumseq;
  const int32_t* past;
  const int32_t* block_table;
  int32_t* err_flags;
  int64_t num_tokens;
  int64_t num_slots;
  int num_seqs, seq_begin, seq_end;
  int H, vhs, ro, rd, interleaved, cos_rows, bs, num_blocks, max_blocks;
  float scale_log2;  // scale * log2(e)
  float cap_in;      // scale / softcap   (softcap > 0)
  float cap_out;     // softcap * log2(e)
  int softcap_on;
  int window;
  int splits;        // key splits per decode token (1: write the output directly)
  int decode;
  int box_rows;      // rows per TMA box: min(N, bs)
};

template <int HS, int VG, int G, int N, int STAGES>
struct Cfg {
  static constexpr int kBoxes = HS / 64;                  // 64-channel slabs
  static constexpr int kQBytes = kRows * HS * 2;
  static constexpr int kQBox = kRows * 128;                // bytes per Q slab
  static constexpr int kKBox = N * 128;                    // bytes per K slab
  static constexpr int kStageBytes = N * HS * 2;
  static constexpr int kSmemData = kQBytes + STAGES * kStageBytes;
  // TMEM columns: O | S0 | S1 | P0 | P1
  static constexpr int kColO = 0;
  static constexpr int kColS = VG;
  static constexpr int kColP = VG + 2 * N;
  static constexpr int kCols = VG + 2 * N + N;  // P is 16-bit: N/2 columns x 2 buffers
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                   : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM budget");
  static_assert(HS % 64 == 0 && VG % 64 == 0 && VG <= 256 && N % 32 == 0 && N <= 256, "shape");
};

struct Barriers {
  uint64_t full[8], empty[8];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t q_full;
  uint64_t drain;
  uint32_t tmem_base;
  int bad;
  int abort;
};

// Bounded wait on an mbarrier phase: non-blocking polls, then polls with a
// short sleep; about a second in total before giving up. Returns false (and
// marks the CTA aborted) on expiry or when another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* err) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
    if (i >= 4096u) __nanosleep(32);
  }
  *abort = 1;
  raise_flag(err, PA_DEVERR_TIMEOUT);
  return false;
}

// Bounded wait used while tearing down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* err) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_test_wait(bar, parity)) return;
    if (i >= 4096u) __nanosleep(32);
  }
  raise_flag(err, PA_DEVERR_TIMEOUT);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// The attention kernel
// ---------------------------------------------------------------------------
template <typename T, int HS, int VG, int G, int N, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
tc_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ Params P) {
  using C = Cfg<HS, VG, G, N, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + C::kQBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kSmemData);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % G;            // value-channel group
  const int64_t unit = blockIdx.x / G;

  // ---- resolve the query token, its sequence and key range (uniform) ----
  int64_t t, pos;
  int32_t b;
  int split = 0;
  int64_t x = unit;
  if (P.decode) {
    x = unit / P.splits;
    split = (int)(unit % P.splits);
    b = P.seq_begin + (int32_t)x;
    const int32_t q0 = P.cumseq[b], q1 = P.cumseq[b + 1];
    if (q1 - q0 != 1) {
      if (tid == 0 && g == 0 && split == 0) raise_flag(P.err_flags, PA_DEVERR_DECODE_QLEN);
      return;
    }
    if (q0 < 0 || q0 >= P.num_tokens) {
      if (tid == 0 && g == 0 && split == 0) raise_flag(P.err_flags, PA_DEVERR_CUMSEQ);
      return;
    }
    t = q0;
    pos = P.past[b];
  } else {
    if (!locate_token(unit, P.cumseq, P.past, P.num_seqs,
                      (tid == 0 && g == 0) ? P.err_flags : nullptr, &b, &pos))
      return;
    if (b < P.seq_begin || b >= P.seq_end) return;
    t = unit;
  }
  const int vhs = P.vhs;
  T* out_row = reinterpret_cast<T*>(P.out) + t * (int64_t)P.H * vhs;
  const bool bad_ctx = P.past[b] < 0 || pos >= (int64_t)P.max_blocks * P.bs;
  const bool bad_pos = P.rd > 0 && pos >= P.cos_rows;
  if (bad_ctx || bad_pos) {
    if (tid == 0 && g == 0 && split == 0)
      raise_flag(P.err_flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
    if (split == 0)
      for (int i = tid; i < P.H * VG; i += kThreads) {
        const int h = i / VG, c = i % VG;
        out_row[(int64_t)h * vhs + g * VG + c] = Half<T>::from_f32(0.f);
      }
    return;
  }
  const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
  const int64_t tile_first = lo / N, tile_last = pos / N;
  const int64_t ntiles_all = tile_last - tile_first + 1;
  const int64_t per = (ntiles_all + P.splits - 1) / P.splits;
  const int64_t t_begin = tile_first + (int64_t)split * per;
  const int64_t t_end = min(tile_last + 1, t_begin + per);
  const int n = (int)max((int64_t)0, t_end - t_begin);
  const int64_t part = (x * P.splits + split) * G + g;  // partial slot (decode splits)

  if (n == 0) {  // an empty key split contributes nothing
    if (P.splits > 1)
      for (int r = tid; r < kRows; r += kThreads) {
        P.ws_ml[(part * kRows + r) * 2 + 0] = -INFINITY;
        P.ws_ml[(part * kRows + r) * 2 + 1] = 0.f;
      }
    return;
  }

  // ---- setup: barriers, TMEM ----
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->s_free[i]), kRows);
      mbar_init(smem_u32(&bars->p_full[i]), kRows);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_full), kRows);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->bad = 0;
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) prefetch_tmap(&kmap);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;

  if (warp < 4) {
    // =================== softmax / epilogue warps ===================
    const int row = tid;  // TMEM lane == head
    // Q with RoPE into the 128B-swizzled K-major layout: slab s holds
    // channels [64s, 64s+64); row r's 16-byte chunk c sits at chunk c ^ (r&7).
    {
      const T* q = reinterpret_cast<const T*>(P.query) + t * (int64_t)P.H * HS;
      const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * (P.rd >> 1);
      const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * (P.rd >> 1);
      constexpr int kChunks = HS / 8;
      for (int i = tid; i < kRows * kChunks; i += 128) {
        const int r = i / kChunks, c = i - r * kChunks;
        const int d0 = c * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < P.H) {
          const T* qr = q + (int64_t)r * HS;
          v = *reinterpret_cast<const uint4*>(qr + d0);
          if (P.rd > 0 && d0 >= P.ro && d0 < P.ro + P.rd) {
            float xv[8], xp[8];
            unpack8<T>(v, xv);
            if (!P.interleaved) {
              const int half = P.rd >> 1;
              const int dp = (d0 - P.ro < half) ? d0 + half : d0 - half;
              unpack8<T>(*reinterpret_cast<const uint4*>(qr + dp), xp);
            }
            rope8<T>(xv, xp, d0, P.ro, P.rd, P.interleaved, crow, srow);
            v = pack8<T>(xv);
          }
        }
        const int slab = d0 >> 6, ch = (d0 >> 3) & 7;
        *reinterpret_cast<uint4*>(q_s + slab * C::kQBox + r * 128 + ((ch ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async();
      mbar_arrive(smem_u32(&bars->q_full));
    }

    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int k = 0; k < n && ok; ++k) {
      const int sb = k & 1;
      const int64_t j0 = (t_begin + k) * N;
      ok = __all_sync(0xffffffffu,
                      wait_bar(smem_u32(&bars->s_full[sb]), (k >> 1) & 1, abort, P.err_flags));
      if (!ok) break;
      tc_fence_after();
      float s[N];
#pragma unroll
      for (int c = 0; c < N; c += 16) {
        uint32_t r[16];
        tmem_ld16(lane_addr + C::kColS + sb * N + c, r);
#pragma unroll
        for (int e = 0; e < 16; ++e) s[c + e] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->s_free[sb]));

      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < N; ++c) {
        const int64_t j = j0 + c;
        float v = P.softcap_on ? P.cap_out * tanhf(s[c] * P.cap_in) : s[c] * P.scale_log2;
        v = (j >= lo && j <= pos) ? v : -INFINITY;
        s[c] = v;
        mt = fmaxf(mt, v);
      }
      float factor = 1.f;
      bool rescale = false;
      if (k == 0) {
        m_used = mt;
      } else if (mt > m_used + kRescaleLog2) {
        factor = ex2(m_used - mt);
        m_used = mt;
        l *= factor;
        rescale = true;
      }
      uint32_t pk[N / 2];
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < N; c += 2) {
        const float p0 = ex2(s[c] - m_used), p1 = ex2(s[c + 1] - m_used);
        lsum += p0 + p1;
        pk[c / 2] = pack2<T>(p0, p1);
      }
      l += lsum;

      // Keys outside [lo, pos] in a boundary tile: zero their value rows so
      // stale or unwritten cache slots cannot reach the PV product.
      if (j0 < lo || j0 + N - 1 > pos) {
        uint8_t* kst = k_s + (k % STAGES) * C::kStageBytes;
        constexpr int kVSlabs = VG / 64;
        for (int i = tid; i < N * kVSlabs * 8; i += 128) {
          const int rr = i / (kVSlabs * 8);
          const int rem = i - rr * (kVSlabs * 8);
          const int slab = g * kVSlabs + rem / 8, ch = rem & 7;
          const int64_t j = j0 + rr;
          if (j < lo || j > pos)
            *reinterpret_cast<uint4*>(kst + slab * C::kKBox + rr * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }

      // P buffer sb is free once PV(k-2) has completed.
      if (k >= 2) {
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[sb]), ((k - 2) >> 1) & 1,
                                              abort, P.err_flags));
        if (!ok) break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < N / 2; c += 16) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = pk[c + e];
        tmem_st16(lane_addr + C::kColP + sb * (N / 2) + c, r);
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O may only be touched once PV(k-1) has completed.
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[sb ^ 1]),
                                              ((k - 1) >> 1) & 1, abort, P.err_flags));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < VG; c += 16) {
          uint32_t r[16];
          tmem_ld16(lane_addr + C::kColO + c, r);
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
          tmem_st16(lane_addr + C::kColO + c, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[sb]));
    }

    // ---- epilogue ----
    named_sync(2, 160);  // the producer has finished issuing (bad-block flag final)
    ok = __all_sync(0xffffffffu, ok && !*abort);
    if (ok)
      ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[(n - 1) & 1]),
                                            ((n - 1) >> 1) & 1, abort, P.err_flags));
    if (ok) {
      tc_fence_after();
      const bool bad = bars->bad != 0;
      if (P.splits == 1) {
        const float inv = (l > 0.f && !bad) ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < VG; c += 16) {
          uint32_t r[16];
          tmem_ld16(lane_addr + C::kColO + c, r);
          if (row < P.H) {
            uint4 o[2];
            uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              ow[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(out_row + (int64_t)row * vhs + g * VG + c);
            dst[0] = o[0];
            dst[1] = o[1];
          }
        }
      } else {
        float* wo = P.ws_o + (part * kRows + row) * VG;
#pragma unroll 1
        for (int c = 0; c < VG; c += 16) {
          uint32_t r[16];
          tmem_ld16(lane_addr + C::kColO + c, r);
          float4* dst = reinterpret_cast<float4*>(wo + c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                 __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
        }
        // a NaN max marks a split that read an invalid block
        P.ws_ml[(part * kRows + row) * 2 + 0] = bad ? __int_as_float(0x7fc00000) : m_used;
        P.ws_ml[(part * kRows + row) * 2 + 1] = bad ? 0.f : l;
      }
    }
  } else if (warp == 4) {
    // =================== TMA producer ===================
    const int nsub = N / P.box_rows;
    const int32_t* bt = P.block_table + (int64_t)b * P.max_blocks;
    int issued = 0;
    for (int k = 0; k < n; ++k) {
      const int stage = k % STAGES;
      if (k >= STAGES) {
        bool okw = true;
        if (lane == 0)
          okw = wait_bar(smem_u32(&bars->empty[stage]), ((k / STAGES) & 1) ^ 1, abort,
                         P.err_flags);
        if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
      }
      const int64_t j0 = (t_begin + k) * N;
      // coordinates of the nsub boxes of rows (one cache block each)
      int y = (int)P.num_slots;  // out of range: TMA fills zeros
      if (lane < nsub) {
        const int64_t key0 = j0 + (int64_t)lane * P.box_rows;
        if (key0 <= pos && key0 + P.box_rows - 1 >= lo) {
          const int32_t phys = bt[key0 / P.bs];
          if (phys >= 0 && phys < P.num_blocks) {
            y = (int)((int64_t)phys * P.bs + key0 % P.bs);
          } else {
            bars->bad = 1;
            raise_flag(P.err_flags, PA_DEVERR_BLOCK);
          }
        }
      }
      // broadcast the coordinates, then lane 0 issues every box
      int ysub[8];
#pragma unroll
      for (int sb = 0; sb < 8; ++sb) ysub[sb] = __shfl_sync(0xffffffffu, y, sb < nsub ? sb : 0);
      if (lane == 0) {
        const uint32_t full = smem_u32(&bars->full[stage]);
        mbar_expect_tx(full, C::kStageBytes);
        const uint32_t dst0 = smem_u32(k_s + stage * C::kStageBytes);
#pragma unroll 1
        for (int slab = 0; slab < C::kBoxes; ++slab)
#pragma unroll 1
          for (int sb = 0; sb < nsub; ++sb)
            tma_load_2d(dst0 + slab * C::kKBox + sb * P.box_rows * 128, &kmap, slab * 64,
                        ysub[sb], full);
      }
      issued = k + 1;
      __syncwarp();
    }
    if (*abort && lane == 0) {
      // copies still in flight must land before the CTA exits
      for (int st = 0; st < STAGES && st < issued; ++st) {
        const int kl = issued - 1 - ((issued - 1 - st) % STAGES);
        drain_wait(smem_u32(&bars->full[st]), (kl / STAGES) & 1, P.err_flags);
      }
    }
    __syncwarp();
    named_arrive(2, 160);
  } else {
    // =================== MMA issuer (warp 5) ===================
    if (lane == 0) {
      constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
      constexpr uint32_t kIdQK = idesc_f16(kBf16, kRows, N, false);
      constexpr uint32_t kIdPV = idesc_f16(kBf16, kRows, VG, true);
      const uint32_t q_base = smem_u32(q_s);
      const uint32_t k_base = smem_u32(k_s);
      bool ok = wait_bar(smem_u32(&bars->q_full), 0, abort, P.err_flags);
      int issued_pv = -1;
      auto issue_qk = [&](int k) -> bool {
        const int stage = k % STAGES, sb = k & 1;
        if (!wait_bar(smem_u32(&bars->full[stage]), (k / STAGES) & 1, abort, P.err_flags))
          return false;
        if (k >= 2 &&
            !wait_bar(smem_u32(&bars->s_free[sb]), ((k - 2) >> 1) & 1, abort, P.err_flags))
          return false;
        tc_fence_after();
        const uint32_t kb = k_base + stage * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < HS / 16; ++kk) {
          const int slab = kk >> 2, w = (kk & 3) * 32;
          const uint64_t a = sdesc(q_base + slab * C::kQBox + w, 16, 1024);
          const uint64_t bdesc = sdesc(kb + slab * C::kKBox + w, 16, 1024);
          mma_ss(tmem + C::kColS + sb * N, a, bdesc, kIdQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&bars->s_full[sb]));
        return true;
      };
      auto issue_pv = [&](int k) -> bool {
        const int stage = k % STAGES, sb = k & 1;
        if (!wait_bar(smem_u32(&bars->p_full[sb]), (k >> 1) & 1, abort, P.err_flags))
          return false;
        tc_fence_after();
        const uint32_t vb = k_base + stage * C::kStageBytes + (g * (VG / 64)) * C::kKBox;
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk) {
          // B = V[keys 16kk.., channels]: MN-major, 64-channel slabs kKBox apart
          // (leading offset), 8-key groups 1024 bytes apart (stride offset).
          const uint64_t bdesc = sdesc(vb + kk * 16 * 128, C::kKBox, 1024);
          mma_ts(tmem + C::kColO, tmem + C::kColP + sb * (N / 2) + kk * 8, bdesc, kIdPV,
                 (k > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&bars->pv_done[sb]));
        tc_commit(smem_u32(&bars->empty[stage]));
        issued_pv = k;
        return true;
      };
      if (ok) {
        tc_fence_after();
        ok = issue_qk(0);
        for (int k = 0; k < n && ok; ++k) {
          if (k + 1 < n) ok = issue_qk(k + 1);
          if (ok) ok = issue_pv(k);
        }
      }
      (void)issued_pv;
      // every MMA issued above completes before TMEM is released
      tc_commit(smem_u32(&bars->drain));
      drain_wait(smem_u32(&bars->drain), 0, P.err_flags);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merges key splits: M = max_s m_s, out = sum_s 2^(m_s-M) O_s / sum_s 2^(m_s-M) l_s.
template <typename T, int VG, int G>
__global__ void __launch_bounds__(128) tc_combine_kernel(const __grid_constant__ Params P) {
  const int64_t x = blockIdx.x;
  const int h = blockIdx.y;
  const int32_t b = P.seq_begin + (int32_t)x;
  const int32_t q0 = P.cumseq[b], q1 = P.cumseq[b + 1];
  if (q1 - q0 != 1 || q0 < 0 || q0 >= P.num_tokens) return;
  const int64_t pos = P.past[b];
  if (P.past[b] < 0 || pos >= (int64_t)P.max_blocks * P.bs || (P.rd > 0 && pos >= P.cos_rows))
    return;
  const int S = P.splits;
  T* dst = reinterpret_cast<T*>(P.out) + (int64_t)q0 * P.H * P.vhs + (int64_t)h * P.vhs;
  for (int c = threadIdx.x; c < G * VG; c += blockDim.x) {
    const int g = c / VG, cc = c - g * VG;
    float M = -INFINITY;
    bool bad = false;
    for (int s = 0; s < S; ++s) {
      const float m = P.ws_ml[((((x * S + s) * G + g) * kRows) + h) * 2];
      bad |= isnan(m);
      M = fmaxf(M, m);
    }
    float L = 0.f, o = 0.f;
    for (int s = 0; s < S && !bad; ++s) {
      const int64_t slot = ((x * S + s) * G + g) * kRows + h;
      const float l = P.ws_ml[slot * 2 + 1];
      if (l > 0.f) {
        const float w = ex2(P.ws_ml[slot * 2] - M);
        L += w * l;
        o += w * P.ws_o[slot * VG + cc];
      }
    }
    dst[c] = Half<T>::from_f32(L > 0.f && !bad ? o / L : 0.f);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

struct Shape {
  int hs, vg, groups, n, stages;
};

bool pick(const Geometry& g, Shape* s) {
  if (g.H > kRows) return false;
  if (g.hs == 192 && g.vhs == 128) {
    *s = {192, 128, 1, 64, 4};
    return true;
  }
  if (g.hs == 576 && g.vhs == 512) {
    *s = {576, 256, 2, 32, 2};
    return true;
  }
  return false;
}

int splits_for(const Geometry& g, const Shape& s, Phase ph, int64_t nq) {
  if (ph == Phase::kPrefill || nq <= 0) return 1;
  int64_t sp = g.num_sms / (nq * s.groups);
  const int64_t max_tiles = ((int64_t)g.max_blocks * g.bs + s.n - 1) / s.n;
  const int64_t cap = max_tiles / 4 > 1 ? max_tiles / 4 : 1;
  if (sp > cap) sp = cap;
  if (sp > 32) sp = 32;
  if (sp < 1) sp = 1;
  return (int)sp;
}

size_t partial_bytes(const Shape& s, int64_t units) {
  const size_t per = (size_t)units * s.groups * kRows;
  const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
  return o + per * 2 * sizeof(float);
}

template <typename T, int HS, int VG, int G, int N, int STAGES>
cudaError_t launch_shape(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq) {
  using C = Cfg<HS, VG, G, N, STAGES>;
  const size_t smem = C::kSmemData + sizeof(Barriers) + 1024;
  static bool configured[64] = {false};
  if (g.device >= 0 && g.device < 64 && !configured[g.device]) {
    cudaError_t e = cudaFuncSetAttribute(tc_attn_kernel<T, HS, VG, G, N, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[g.device] = true;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)HS, (cuuint64_t)g.num_blocks * g.bs};
  const cuuint64_t strides[1] = {(cuuint64_t)HS * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)P.box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map,
                   std::is_same<T, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, const_cast<void*>(a.key_cache), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int64_t units = ph == Phase::kDecode ? nq * P.splits : nq;
  tc_attn_kernel<T, HS, VG, G, N, STAGES>
      <<<(unsigned)(units * G), kThreads, smem, a.stream>>>(map, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || P.splits == 1) return e;
  tc_combine_kernel<T, VG, G><<<dim3((unsigned)nq, (unsigned)g.H), 128, 0, a.stream>>>(P);
  return cudaGetLastError();
}

}  // namespace tc

bool tc_supported(const Geometry& g, Phase ph) {
  (void)ph;
  tc::Shape s;
  return tc::pick(g, &s);
}

size_t tc_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs, int64_t num_tokens) {
  (void)num_tokens;
  tc::Shape s;
  if (ph == Phase::kPrefill || num_seqs <= 0 || !tc::pick(g, &s)) return 0;
  // nq * S(nq) <= max(nq, num_sms / groups) for S(nq) = max(1, num_sms/(nq*groups)).
  int64_t units = num_seqs > g.num_sms ? num_seqs : g.num_sms;
  if (tc::splits_for(g, s, ph, 1) <= 1) return 0;
  return tc::partial_bytes(s, units);
}

size_t tc_call_workspace(const Geometry& g, Phase ph, const ReadArgs& a) {
  tc::Shape s;
  if (!tc::pick(g, &s)) return 0;
  const int64_t nq = ph == Phase::kDecode ? (int64_t)(a.seq_end - a.seq_begin) : a.num_tokens;
  const int sp = tc::splits_for(g, s, ph, nq);
  return sp > 1 ? tc::partial_bytes(s, nq * sp) : 0;
}

cudaError_t launch_tc(const Geometry& g, Phase ph, const ReadArgs& a) {
  tc::Shape s;
  if (!tc::pick(g, &s)) return cudaErrorNotSupported;
  const int64_t nq = ph == Phase::kDecode ? (int64_t)(a.seq_end - a.seq_begin) : a.num_tokens;
  if (nq <= 0) return cudaSuccess;
  tc::Params P;
  P.query = a.query;
  P.out = a.out;
  P.cos_cache = a.cos_cache;
  P.sin_cache = a.sin_cache;
  P.cumseq = a.cumseq;
  P.past = a.past;
  P.block_table = a.block_table;
  P.err_flags = a.err_flags;
  P.num_tokens = a.num_tokens;
  P.num_slots = (int64_t)g.num_blocks * g.bs;
  P.num_seqs = a.num_seqs;
  P.seq_begin = a.seq_begin;
  P.seq_end = a.seq_end;
  P.H = g.H;
  P.vhs = g.vhs;
  P.ro = g.ro;
  P.rd = g.rd;
  P.interleaved = g.interleaved;
  P.cos_rows = g.cos_rows;
  P.bs = g.bs;
  P.num_blocks = g.num_blocks;
  P.max_blocks = g.max_blocks;
  P.scale_log2 = g.scale * tc::kLog2e;
  P.softcap_on = g.softcap > 0.f ? 1 : 0;
  P.cap_in = g.softcap > 0.f ? g.scale / g.softcap : 0.f;
  P.cap_out = g.softcap * tc::kLog2e;
  P.window = g.window;
  P.decode = ph == Phase::kDecode ? 1 : 0;
  P.splits = tc::splits_for(g, s, ph, nq);
  P.box_rows = s.n < g.bs ? s.n : g.bs;
  P.ws_o = nullptr;
  P.ws_ml = nullptr;
  if (P.splits > 1) {
    const size_t per = (size_t)nq * P.splits * s.groups * tc::kRows;
    const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
    if (a.workspace == nullptr || a.workspace_bytes < o + per * 2 * sizeof(float))
      return cudaErrorInvalidValue;
    P.ws_o = reinterpret_cast<float*>(a.workspace);
    P.ws_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(a.workspace) + o);
  }
  const bool bf16 = g.dtype == PA_DTYPE_BF16;
  if (s.hs == 192) {
    return bf16 ? tc::launch_shape<__nv_bfloat16, 192, 128, 1, 64, 4>(g, ph, a, P, nq)
                : tc::launch_shape<__half, 192, 128, 1, 64, 4>(g, ph, a, P, nq);
  }
  return bf16 ? tc::launch_shape<__nv_bfloat16, 576, 256, 2, 32, 2>(g, ph, a, P, nq)
              : tc::launch_shape<__half, 576, 256, 2, 32, 2>(g, ph, a, P, nq);
}

}  // namespace pa
