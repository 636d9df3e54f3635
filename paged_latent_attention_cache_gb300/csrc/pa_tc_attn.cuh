// Tensor-core read phase for sm_103a (single-CTA kernel, shared by pa_tc.cu and
// pa_tc_glm.cu): tcgen05 MMAs with TMEM accumulators,
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
// CTA = one work unit: one query token (prefill with H <= 64: 128/H
// consecutive tokens of one sequence, every row with its own position), or
// in decode one split of a token's keys (splits are merged by a log-sum-exp
// combine kernel). Any latent width up to 256 (a multiple of 16) and any
// value width up to it run here: the width is cut into 64-channel slabs
// (channels beyond hs of the last slab are loaded as zeros by TMA), the O
// accumulator holds vg = 64 * ceil(vhs / 64) channels and only the first vhs
// are stored. The 576/512 geometry runs on a CTA pair (pa_tc_pair.cu).
// Warp roles:
//   warps 0-3  softmax + epilogue; thread i owns row i (TMEM lane i): loads Q
//              with RoPE into swizzled shared memory, reads S from TMEM,
//              masks/softcaps, runs the online softmax with lazy rescaling
//              (the reference max only moves when it grows by > 2^8), writes
//              P (16-bit) to TMEM, finally normalises O and stores it.
//   warp 4     TMA producer: per key tile, one 2-D box (64 channels x rows of
//              one cache block) per 64-channel slab, 128-byte swizzle.
//   warp 5     TMEM allocation and the single MMA-issuing thread.
//   (With 64 query rows the producer and MMA warps are 6 and 7, on other
//   scheduler partitions than the two softmax warps that hold rows.)
// Pipelines: K tiles in a STAGES-deep ring (full/empty mbarriers), S and P
// in two TMEM buffers each (where two CTAs share an SM, each tile's P is
// written over its own S columns instead: POS). Every
// mbarrier wait is bounded: on expiry the
// CTA sets PA_DEVERR_TIMEOUT in the error word, drains what it issued and
// exits without trapping.
#pragma once

#include <cuda_fp8.h>

#include <cfloat>
#include <cmath>
#include <type_traits>

#include "pa_tc_common.cuh"

namespace pa {
namespace tc {

// TMEM columns allocated for `used` columns: a power of two >= 32.
constexpr int fixed_tmem_cols(int used) {
  return used <= 32 ? 32 : used <= 64 ? 64 : used <= 128 ? 128 : used <= 256 ? 256 : 512;
}


// FP8 cache with a bf16 query: one query row, in place in its swizzled
// slabs (16-byte chunk c of row r at c ^ (r & 7)), from bf16 to fp16 (the
// MMA operands of that path), its rotary channels rotated in f32 first. A
// value beyond the fp16 range is saturated and flags PA_DEVERR_RANGE.
template <typename T, int QBOX>
__device__ __noinline__ void q_row_to_f16(uint8_t* q_s, int row, int hs, const Params& P,
                                          int64_t pos) {
  auto at = [&](int d0) -> uint4* {
    const int slab = d0 >> 6, ch = (d0 >> 3) & 7;
    return reinterpret_cast<uint4*>(q_s + slab * QBOX + row * 128 + ((ch ^ (row & 7)) << 4));
  };
  const int ro = P.rd > 0 ? P.ro : hs, rd = P.rd, half = rd >> 1;
  const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * half;
  const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * half;
  bool big = false;
  for (int d0 = 0; d0 < hs; d0 += 8) {
    const bool rot = d0 >= ro && d0 < ro + rd;
    float a[8];
    unpack8<T>(*at(d0), a);
    if (rot && !P.interleaved) {
      if (d0 >= ro + half) continue;  // rotated with its partner below
      float bb[8], na[8], nb[8];
      unpack8<T>(*at(d0 + half), bb);
#pragma unroll
      for (int e = 0; e < 8; ++e) { na[e] = a[e]; nb[e] = bb[e]; }
      rope8<T>(na, bb, d0, ro, rd, 0, crow, srow);
      rope8<T>(nb, a, d0 + half, ro, rd, 0, crow, srow);
      *at(d0) = pack8_f16_sat(na, &big);
      *at(d0 + half) = pack8_f16_sat(nb, &big);
      continue;
    }
    if (rot) {
      float dummy[8];
      rope8<T>(a, dummy, d0, ro, rd, 1, crow, srow);
    }
    *at(d0) = pack8_f16_sat(a, &big);
  }
  if (big) raise_flag(P.err_flags, PA_DEVERR_RANGE);
}


// ---------------------------------------------------------------------------
// MMA issue sequences. Not inlined: the MMA warp runs each once on scratch
// operands during the prologue (see the MMA issuer), which brings these
// instructions into the instruction cache and starts the tensor pipe
// before the first key tile lands, while the memory system is still idle.
// ---------------------------------------------------------------------------
// S(d) = Q K^T over nk 16-channel K-steps: K-steps of 16 (32 bytes) within
// each 128-byte slab; the descriptors' address fields (bytes / 16) advance.
// NKF > 0 fixes the step count at compile time (the loop is then unrolled).
template <int QBOX, int KBOX, int NKF>
__device__ __noinline__ void issue_qk(uint32_t d, uint64_t a0, uint64_t b0, int nk, uint32_t id) {
  if (NKF) nk = NKF;
#pragma unroll
  for (int kk = 0; kk < (NKF ? NKF : nk); ++kk) {
    const uint32_t col = (uint32_t)(kk & 3) * 2;  // 32 bytes / 16
    const uint32_t slab = (uint32_t)(kk >> 2);
    mma_ss(d, a0 + (slab * (QBOX >> 4) + col), b0 + (slab * (KBOX >> 4) + col), id,
           kk > 0 ? 1u : 0u);
  }
}
// O(d) (+)= P(a) V over N keys: K-steps of 16 keys (8 TMEM columns of
// packed 16-bit P; 2048 bytes of MN-major V, 128 in the address field).
template <int N>
__device__ __noinline__ void issue_pv(uint32_t d, uint32_t a, uint64_t b0, uint32_t acc0,
                                      uint32_t id) {
#pragma unroll
  for (int kk = 0; kk < N / 16; ++kk)
    mma_ts(d, a + kk * 8, b0 + (uint64_t)(kk * 128), id, (acc0 || kk > 0) ? 1u : 0u);
}

// ---------------------------------------------------------------------------
// The attention kernel
// ---------------------------------------------------------------------------
// HSF, VGF, STF > 0 fix the latent width, the value accumulator width and
// the stage count at compile time (the shapes measured and tuned for the
// 192/128 geometry); 0 takes them from the launch's Params (any other
// width). Fixed values keep every CTA's one-time code short: its
// instructions are fetched cold on every launch.
// FP8: the cache holds E4M3 codes; the MMAs then take fp16 operands (the
// query rounded to fp16 once, the key tiles converted exactly, P in fp16).
template <typename T, int N, int QR, int NB, bool CAP, int HSF, int VGF, int STF, bool FP8,
          bool POS>
__global__ void __launch_bounds__(Tile<N, QR, NB, FP8>::kThreads, 1)
tc_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ Params P) {
  using C = Tile<N, QR, NB, FP8>;
  using TM = typename std::conditional<FP8, __half, T>::type;  // MMA operand type
  constexpr int kSlabsF = (HSF + 63) / 64;
  constexpr int kTmemColsF = fixed_tmem_cols(VGF + NB * N + (POS ? 0 : NB * N / 2));
  // P (16-bit, N/2 columns per tile) has buffers of its own after the S
  // buffers, or (POS) is written over its own tile's S columns
  const int hs = HSF ? HSF : P.hs;
  const int slabs = HSF ? kSlabsF : P.slabs;
  const int vg = VGF ? VGF : P.vg;
  const int stages = STF ? STF : P.stages;
  const int stage_bytes = HSF ? N * kSlabsF * 128 : P.stage_bytes;
  const int q_bytes = HSF ? QR * kSlabsF * 128 : P.q_bytes;
  const int col_s = VGF ? VGF : P.col_s;          // TMEM: O | S x NB | P x NB
  const int col_p = POS ? col_s : VGF ? VGF + NB * N : P.col_p;
  constexpr int kPStride = POS ? N : N / 2;  // TMEM columns from one P buffer to the next
  const uint32_t tmem_cols = VGF ? (uint32_t)kTmemColsF : (uint32_t)P.tmem_cols;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Work work;
  __shared__ Barriers bars_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* q_s = smem;             // slabs query slabs of QR rows
  uint8_t* k_s = smem + q_bytes;   // stages key stages of N rows x slabs slabs
  uint8_t* k8_s = k_s + stages * stage_bytes;  // FP8: stages8 E4M3 tiles of N rows x hs bytes
  Barriers* bars = &bars_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x;
  const int vhs = P.vhs;

  // ---- prologue: warp 0 resolves the work while warps 1/5 set up ----
  // With programmatic dependent launch this CTA may start while the previous
  // kernel on the stream is still running: nothing reads inputs or writes
  // outputs before griddepcontrol.wait returns, except when P.early says that
  // the previous kernel is this library's write phase; then only the cache
  // rows it writes are off limits, and the producer waits before its first
  // cache load. Dependents (the split combine) are released only when this
  // CTA reaches its epilogue, so their waiting CTAs do not share the SM with
  // the main loop.
  if (warp == 0) {
    if (!P.early) grid_dep_wait();
    Work w;
    if (P.mixed ? unit < P.units : P.decode != 0) {
      // the query region is free until the query load that follows the plan
      w = decode_plan_warp<N>(P, unit, reinterpret_cast<int*>(q_s), q_bytes / 4);
      fence_proxy_async();  // the scratch is overwritten by the query TMA later
      if (w.status == 0) {
        const int32_t q0 = P.cumseq[w.b], q1 = P.cumseq[w.b + 1];
        if (lane == 0 && w.split == 0) P.ws_plan[w.b - P.seq_begin] = make_int2(w.first, w.splits);
        if (q1 - q0 != 1) {
          if (lane == 0) raise_flag(P.err_flags, PA_DEVERR_DECODE_QLEN);
          w.status = 2;
        } else if (q0 < 0 || q0 >= P.num_tokens) {
          if (lane == 0) raise_flag(P.err_flags, PA_DEVERR_CUMSEQ);
          w.status = 2;
        } else {
          w.t = q0;
          w.past = P.past[w.b];
          w.pos = w.past;
          w.ntok = 1;
        }
      }
    } else if (P.tpc > 1 || P.mixed) {
      w = prefill_group_warp(P, P.mixed ? unit - P.units : unit, P.tpc);
      if (w.status == 0) {
        const int64_t lo_key = P.window >= 0 ? max((int64_t)0, w.pos - P.window) : 0;
        w.t_begin = lo_key / N;
        w.t_end = (w.pos + w.ntok - 1) / N + 1;
      }
    } else {
      int32_t b;
      int64_t pos;
      w.status = 1;
      w.splits = 1;
      w.decode = 0;
      // CTA `unit` takes token T - 1 - unit: the tokens with the most keys
      // (the last of each sequence) start first, short ones fill in behind
      const int64_t tok = P.num_tokens - 1 - unit;
      if (locate_token(tok, P.cumseq, P.past, P.num_seqs,
                       lane == 0 ? P.err_flags : nullptr, &b, &pos) &&
          b >= P.seq_begin && b < P.seq_end) {
        w.status = 0;
        w.b = b;
        w.t = tok;
        w.pos = pos;
        w.past = P.past[b];
        w.ntok = 1;
        const int64_t lo_key = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
        w.t_begin = lo_key / N;
        w.t_end = pos / N + 1;
      }
    }
    if (w.status == 0) {
      const int64_t pos_hi = w.pos + w.ntok - 1;  // the unit's last token
      const bool bad_ctx = w.past < 0 || pos_hi >= (int64_t)P.max_blocks * P.bs ||
                           w.t + w.ntok > P.num_tokens;
      const bool bad_pos = P.rd > 0 && pos_hi >= P.cos_rows;
      if (bad_ctx || bad_pos) {
        if (lane == 0)
          raise_flag(P.err_flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
        T* out_row = reinterpret_cast<T*>(P.out) + w.t * (int64_t)P.H * vhs;
        const int rows = min((int64_t)w.ntok, P.num_tokens - w.t) * P.H;
        for (int i = lane; i < rows * vhs; i += 32) out_row[i] = Half<T>::from_f32(0.f);
        w.status = 2;
      }
    }
    if (lane == 0) work = w;
    fence_proxy_async();  // scratch stores before the query load reuses the region
  } else if (warp == 1 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      // (FP8: the key tile is complete when every converter thread has
      // written its part; otherwise when the TMA bytes have landed)
      mbar_init(smem_u32(&bars->full[s]), FP8 ? 128 : 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    if (FP8) {
      for (int s = 0; s < P.stages8; ++s) {
        mbar_init(smem_u32(&bars->full8[s]), 1);
        mbar_init(smem_u32(&bars->empty8[s]), 128);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->s_free[i]), kRows);
      mbar_init(smem_u32(&bars->p_full[i]), kRows);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_tma), 1);
    mbar_init(smem_u32(&bars->q_full), kRows);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->bad = 0;
    bars->abort = 0;
    fence_barrier_init();
  } else if (warp == C::kProdWarp && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
  } else if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), tmem_cols);
    tmem_relinquish();
  }
  if (warp != 0 && !P.early) grid_dep_wait();  // every thread is ordered after the previous grid
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  const Work W = work;

  if (W.status == 0) {
    // The unit's rows are ntok consecutive tokens' heads (row r: token t +
    // r / H at position pos + r / H). Keys any row sees lie in [lo, pos_hi];
    // every row sees at least [lo_hi, pos].
    const int64_t t = W.t, pos = W.pos, t_begin = W.t_begin;
    const int32_t b = W.b;
    const int splits = W.splits, ntok = W.ntok, rows = W.ntok * P.H;
    const int64_t pos_hi = pos + ntok - 1;
    const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
    const int64_t lo_hi = P.window >= 0 ? max((int64_t)0, pos_hi - P.window) : 0;
    const int n = (int)max((int64_t)0, W.t_end - t_begin);
    const int64_t part = unit;  // partial slot (decode splits)
    T* out_row = reinterpret_cast<T*>(P.out) + t * (int64_t)P.H * vhs;

    if (warp < 4) {
      // =================== softmax / epilogue warps ===================
      const int row = tid;                 // TMEM lane == query row
      const bool live = warp * 32 < rows;  // warp holds at least one real row
      // this row's token position and first visible key (rows past the unit:
      // nothing visible)
      const int64_t pos_r = row < rows ? pos + row / P.H : -1;
      const int64_t lo_r = P.window >= 0 ? max((int64_t)0, pos_r - P.window) : 0;
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      // Pass k = -1 runs the tile code once with every wait, arrive, shared
      // memory write and state update switched off, on whatever TMEM holds:
      // it brings the loop's instructions into the instruction cache while
      // the query and the first key tile are still in flight, instead of on
      // the first tile's critical path. (The opaque start keeps the compiler
      // from peeling it into a copy of its own.)
      int k_first = -1;
      asm volatile("" : "+r"(k_first));
      for (int k = k_first; k < n && ok; ++k) {
        const bool dry = k < 0;
        if (k == 0) {  // every work item has n >= 1 tiles
          // Q arrives by TMA in the 128B-swizzled K-major layout (slab s holds
          // channels [64s, 64s+64); row r's 16-byte chunk c sits at c ^ (r&7));
          // each thread then rotates its own row's rotary channels in place.
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->q_tma), 0, abort, P.err_flags));
          if (FP8 && !std::is_same<T, __half>::value) {
            // bf16 query, fp16 MMA operands: the whole row is rounded to fp16
            // in place (its rotary channels rotated first, in f32)
            if (ok && row < rows) q_row_to_f16<T, C::kQBox>(q_s, row, hs, P, pos_r);
          } else if (ok && P.rd > 0 && row < rows) {
            const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos_r * (P.rd >> 1);
            const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos_r * (P.rd >> 1);
            auto at = [&](int d0) -> uint4* {
              const int slab = d0 >> 6, ch = (d0 >> 3) & 7;
              return reinterpret_cast<uint4*>(q_s + slab * C::kQBox + row * 128 +
                                              ((ch ^ (row & 7)) << 4));
            };
            if (!P.interleaved) {
              const int half = P.rd >> 1;
              for (int d0 = P.ro; d0 < P.ro + half; d0 += 8) {
                float a[8], bb[8], na[8], nb[8];
                unpack8<T>(*at(d0), a);
                unpack8<T>(*at(d0 + half), bb);
#pragma unroll
                for (int e = 0; e < 8; ++e) { na[e] = a[e]; nb[e] = bb[e]; }
                rope8<T>(na, bb, d0, P.ro, P.rd, 0, crow, srow);
                rope8<T>(nb, a, d0 + half, P.ro, P.rd, 0, crow, srow);
                *at(d0) = pack8<T>(na);
                *at(d0 + half) = pack8<T>(nb);
              }
            } else {
              for (int d0 = P.ro; d0 < P.ro + P.rd; d0 += 8) {
                float a[8], dummy[8];
                unpack8<T>(*at(d0), a);
                rope8<T>(a, dummy, d0, P.ro, P.rd, 1, crow, srow);
                *at(d0) = pack8<T>(a);
              }
            }
          }
          fence_proxy_async();
          mbar_arrive(smem_u32(&bars->q_full));
          if (!ok) break;
        }
        const int sb = NB == 2 ? (k & 1) : 0;
        const int64_t j0 = (t_begin + k) * N;
        // a tile with keys that some row must not see (uniform across the CTA)
        const bool edge = !dry && (j0 < lo_hi || j0 + N - 1 > pos);
        if (!dry) {
          ok = __all_sync(0xffffffffu,
                          wait_bar(smem_u32(&bars->s_full[sb]), (k / NB) & 1, abort, P.err_flags));
          if (!ok) break;
        }
        // The tile is handled in 32-column chunks read from TMEM twice (row
        // maximum of the raw scores, then probabilities), which keeps the
        // loop body short: the first tile then does not wait long for its
        // instructions. The softcap c*tanh(x/c) is increasing, so the
        // maximum of the capped scores is the cap of the raw maximum and
        // only pass 2 applies it, per element.
        float factor = 1.f;
        bool rescale = false;
        // Scores in the log2 domain: v * sl (sl = scale*log2e) without
        // softcap, cap_out * tanh(v * cap_in) with it.
        const float sl = CAP ? 1.f : P.scale_log2;
        const uint32_t s_addr = lane_addr + col_s + sb * N;
        // this row's visible columns [clo, chi] of the tile
        int clo = 0, chi = N - 1;
        if (edge) {
          clo = (int)min((int64_t)N, max((int64_t)0, lo_r - j0));
          chi = (int)max((int64_t)-1, min((int64_t)(N - 1), pos_r - j0));
        }
        int mode = 2;  // softcap in pass 2: 1 series, 2 tanh_ex2
        if (live) {
          tc_fence_after();
          float vmax = -INFINITY, vmin = INFINITY;  // over the visible raw scores
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
            if (c >= clo && c + 31 <= chi) {
              if (CAP) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  vmax = fmaxf(vmax, __uint_as_float(r[e]));
                  vmin = fminf(vmin, __uint_as_float(r[e]));
                }
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) vmax = fmaxf(vmax, __uint_as_float(r[e]));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                if (c + e >= clo && c + e <= chi) {
                  vmax = fmaxf(vmax, __uint_as_float(r[e]));
                  vmin = fminf(vmin, __uint_as_float(r[e]));
                }
              }
            }
          }
          float mt;  // the tile's row maximum in the log2 domain
          if (CAP) {
            mt = vmax == -INFINITY ? -INFINITY : P.cap_out * tanh_ex2(vmax * P.cap_in);
            // the series serves the whole warp's tile when every real row's
            // scores are small (the dry pass takes it to warm its code)
            const bool small = row >= rows || fmaxf(vmax, -vmin) <= P.cap_vlim;
            mode = (P.cap_poly && __all_sync(0xffffffffu, small || dry)) ? 1 : 2;
          } else {
            mt = vmax * sl;
          }
          if (dry) {
          } else if (k == 0) {
            m_used = mt;
          } else if (mt > m_used + kRescaleLog2) {  // (also when no key was visible before)
            factor = ex2(m_used - mt);
            m_used = mt;
            l *= factor;
            rescale = true;
          }
        }

        // Keys no row sees (outside [lo, pos_hi]) in a boundary tile: zero
        // their value rows so stale or unwritten cache slots cannot reach
        // the PV product (rows that mask a key seen by another row give it
        // probability 0, and its value row is a written, finite row).
        if (edge) {
          uint8_t* kst = k_s + (k % stages) * stage_bytes;
          const int vslabs = vg / 64;
          for (int i = tid; i < N * vslabs * 8; i += 128) {
            const int rr = i / (vslabs * 8);
            const int rem = i - rr * (vslabs * 8);
            const int slab = rem / 8, ch = rem & 7;
            const int64_t j = j0 + rr;
            if (j < lo || j > pos_hi)
              *reinterpret_cast<uint4*>(kst + slab * C::kKBox + rr * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }

        // P buffer sb is free once PV(k-NB) has completed. (POS: P goes over
        // S(k), which QK^T(k) wrote only after PV(k-NB) had completed.)
        if (!POS && k >= NB) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[sb]),
                                                ((k - NB) / NB) & 1, abort, P.err_flags));
          if (!ok) break;
        }
        if (live) {
          tc_fence_after();
          float lsum = 0.f;
          // a row that has seen no key yet (several tokens per unit, window)
          // has every score at -inf: its probabilities are 0, not NaN
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          const ExpArgs A{sl, mu, P.cap_in, P.cap_out, P.cap_a[0], P.cap_a[1], P.cap_a[2],
                          P.cap_a[3], P.cap_a[4]};
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32], pk[16];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
            if (!(c >= clo && c + 31 <= chi)) {  // masked keys: v = -inf
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c + e < clo || c + e > chi) r[e] = __float_as_uint(-INFINITY);
            }
            if (!CAP) lsum += exp_chunk<TM, 0>(r, pk, A);
            else if (mode == 1) lsum += exp_chunk<TM, 1>(r, pk, A);
            else lsum += exp_chunk<TM, 2>(r, pk, A);
            tmem_st16(lane_addr + col_p + sb * kPStride + c / 2, pk);
          }
          if (!dry) l += lsum;
          if (__any_sync(0xffffffffu, rescale)) {
            // O may only be touched once PV(k-1) has completed.
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[(k - 1) % NB]),
                                                  ((k - 1) / NB) & 1, abort, P.err_flags));
            if (ok) {
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < vg; c += 16) {
                uint32_t r[16];
                tmem_ld16(lane_addr + c, r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
                tmem_st16(lane_addr + c, r);
              }
            }
          }
          tmem_wait_st();
        }
        if (!ok) break;
        tc_fence_before();
        if (dry) continue;
        mbar_arrive(smem_u32(&bars->s_free[sb]));
        mbar_arrive(smem_u32(&bars->p_full[sb]));
      }

      // ---- epilogue ----
      grid_dep_launch();
      named_sync(2, 160);  // the producer has finished issuing (bad-block flag final)
      ok = __all_sync(0xffffffffu, ok && !*abort);
      if (ok)
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[(n - 1) % NB]),
                                              ((n - 1) / NB) & 1, abort, P.err_flags));
      if (ok && live) {
        tc_fence_after();
        const bool bad = bars->bad != 0;
        if (splits == 1) {
          const float inv = (l > 0.f && !bad) ? P.out_scale / l : 0.f;
          const bool vec = vhs % 8 == 0;  // 16-byte aligned output rows
#pragma unroll 1
          for (int c = 0; c < vg && c < vhs; c += 16) {
            uint32_t r[16];
            tmem_ld16(lane_addr + c, r);
            if (row < rows) {
              T* dst = out_row + (int64_t)row * vhs + c;
              if (vec && c + 16 <= vhs) {
                uint4 o[2];
                uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  ow[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv,
                                   __uint_as_float(r[2 * e + 1]) * inv);
                reinterpret_cast<uint4*>(dst)[0] = o[0];
                reinterpret_cast<uint4*>(dst)[1] = o[1];
              } else {  // the ragged last channels of the row
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (c + e < vhs) dst[e] = Half<T>::from_f32(__uint_as_float(r[e]) * inv);
              }
            }
          }
        } else {
          float* wo = P.ws_o + (part * kRows + row) * vg;
#pragma unroll 1
          for (int c = 0; c < vg; c += 16) {
            uint32_t r[16];
            tmem_ld16(lane_addr + c, r);
            if (row < rows) {
              float4* dst = reinterpret_cast<float4*>(wo + c);
              const float os = P.out_scale;
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_float4(__uint_as_float(r[4 * e]) * os,
                                     __uint_as_float(r[4 * e + 1]) * os,
                                     __uint_as_float(r[4 * e + 2]) * os,
                                     __uint_as_float(r[4 * e + 3]) * os);
            }
          }
          if (row < rows) {
            // a NaN max marks a split that read an invalid block
            P.ws_ml[(part * kRows + row) * 2 + 0] = bad ? __int_as_float(0x7fc00000) : m_used;
            P.ws_ml[(part * kRows + row) * 2 + 1] = bad ? 0.f : l;
          }
        }
      }
    } else if (warp == C::kProdWarp) {
      // =================== TMA producer ===================
      if (lane == 0) {  // Q: one box of QR rows (this token's heads) per 64-channel slab
        const uint32_t qb = smem_u32(&bars->q_tma);
        mbar_expect_tx(qb, (uint32_t)q_bytes);
        for (int slab = 0; slab < slabs; ++slab)
          tma_load_2d(smem_u32(q_s) + slab * C::kQBox, &qmap, slab * 64, (int)(t * P.H), qb);
      }
      // With P.early the write grid may still run: cache rows are read only
      // after griddepcontrol.wait, except (P.own_slots) the tiles below the
      // sequence's first new position, which the write does not touch.
      int dirty_from = 0;
      if (P.early && P.own_slots) dirty_from = (int)max((int64_t)0, W.past / N - t_begin);
      bool waited = !P.early;
      const int nsub = N / P.box_rows;
      // (Block ids are looked up tile by tile here: fetching them ahead, as
      // the CTA-pair kernel does, issues the first stages of every CTA at
      // once, and the first tiles then arrive later behind that burst.)
      const int32_t* bt = P.block_table + (int64_t)b * P.max_blocks;
      // the ring the copies land in: key tiles, or (FP8) the E4M3 tiles the
      // converter warps read
      const int pst = FP8 ? P.stages8 : stages;
      uint64_t* pfull = FP8 ? bars->full8 : bars->full;
      uint64_t* pempty = FP8 ? bars->empty8 : bars->empty;
      const int pbytes = FP8 ? P.stage8_bytes : stage_bytes;
      uint8_t* pbase = FP8 ? k8_s : k_s;
      int issued = 0;
      for (int k = 0; k < n; ++k) {
        const int stage = k % pst;
        if (!waited && k >= dirty_from) {
          grid_dep_wait();  // the write phase's cache rows are complete and visible
          waited = true;
        }
        // coordinates of the nsub boxes of rows (one cache block each), worked
        // out (block id loaded) before the wait for the stage, so that the
        // copies go out as soon as the stage is free
        int y = (int)P.num_slots;  // out of range: TMA fills zeros
        if (lane < nsub) {
          const int64_t key0 = (t_begin + k) * N + (int64_t)lane * P.box_rows;
          if (key0 <= pos_hi && key0 + P.box_rows - 1 >= lo) {
            const int32_t phys = bt[key0 / P.bs];
            if (phys >= 0 && phys < P.num_blocks) {
              y = (int)((int64_t)phys * P.bs + (key0 & (int64_t)(P.bs - 1)));
            } else {
              bars->bad = 1;
              raise_flag(P.err_flags, PA_DEVERR_BLOCK);
            }
          }
        }
        if (k >= pst) {
          bool okw = true;
          if (lane == 0)
            okw = wait_bar(smem_u32(&pempty[stage]), ((k / pst) & 1) ^ 1, abort, P.err_flags);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
        } else if (W.decode && k == 2 && nsub <= 2) {
          // Decode: every CTA starts at once, and with few copies per tile
          // their first stages would all be in flight together; the first
          // tile then lands only behind most of that burst. The first two
          // tiles go out now, the later stages once tile 0 has landed (GLM
          // decode: 35.6 -> 33.7 us per step).
          bool okw = true;
          if (lane == 0) okw = wait_bar(smem_u32(&pfull[0]), 0, abort, P.err_flags);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
        }
        if (lane == 0) mbar_expect_tx(smem_u32(&pfull[stage]), (uint32_t)pbytes);
        __syncwarp();
        if (lane < nsub) {  // lane sb issues the boxes of rows sb (every slab)
          const uint32_t full = smem_u32(&pfull[stage]);
          if (FP8) {  // one box of box_rows whole E4M3 rows (hs bytes each)
            tma_load_2d(smem_u32(pbase + stage * pbytes) + lane * P.box_rows * hs, &kmap, 0, y,
                        full);
          } else {
            const uint32_t dst0 = smem_u32(pbase + stage * pbytes) + lane * P.box_rows * 128;
#pragma unroll 1
            for (int slab = 0; slab < slabs; ++slab)
              tma_load_2d(dst0 + slab * C::kKBox, &kmap, slab * 64, y, full);
          }
        }
        issued = k + 1;
        __syncwarp();
      }
      if (!waited) grid_dep_wait();  // the grid completes after the write grid
      if (*abort && lane == 0) {
        // copies still in flight must land before the CTA exits
        drain_wait(smem_u32(&bars->q_tma), 0, P.err_flags);
        for (int st = 0; st < pst && st < issued; ++st) {
          const int kl = issued - 1 - ((issued - 1 - st) % pst);
          drain_wait(smem_u32(&pfull[st]), (kl / pst) & 1, P.err_flags);
        }
      }
      __syncwarp();
      named_arrive(2, 160);
    } else if (warp == C::kMmaWarp) {
      // =================== MMA issuer ===================
      if (lane == 0) {
        constexpr bool kBf16 = std::is_same<TM, __nv_bfloat16>::value;
        constexpr uint32_t kIdQK = idesc_f16(kBf16, kRows, N, false);
        const uint32_t id_pv = idesc_f16(kBf16, kRows, vg, true);
        const int nk = hs / 16;  // QK^T K-steps
        const uint32_t q_base = smem_u32(q_s);
        const uint32_t k_base = smem_u32(k_s);
        // Warm-up: one QK^T into S buffer NB-1 and one PV into O, on whatever
        // shared memory and TMEM hold. Both are overwritten before they are
        // read (QK^T(NB-1) and PV(0) start without accumulation; the
        // softmax's dry pass reads S buffer NB-1 as scratch), and every later
        // commit also tracks them.
        issue_qk<C::kQBox, C::kKBox, HSF / 16>(tmem + col_s + (NB - 1) * N, sdesc(q_base, 16, 1024),
                                     sdesc(k_base, 16, 1024), nk, kIdQK);
        issue_pv<N>(tmem, tmem + col_p + (NB - 1) * kPStride, sdesc(k_base, C::kKBox, 1024), 0u,
                    id_pv);
        bool ok = wait_bar(smem_u32(&bars->q_full), 0, abort, P.err_flags);
        if (ok) {
          tc_fence_after();
          // Event loop: QK^T(k) needs its key tile (full) and a free S buffer
          // (s_free of k-NB); PV(k) needs P(k) (p_full). Issue whichever is
          // ready, QK^T first, so neither waits behind the other's inputs.
          int kq = 0, kp = 0;
          const uint64_t t0 = globaltimer();
          uint32_t spins = 0;
          while (kp < n) {
            bool progressed = false;
            // PV first: it is short and releases the key stage to the producer.
            if (kp < kq) {
              const int stage = kp % stages, sb = kp % NB;
              if (mbar_test_wait(smem_u32(&bars->p_full[sb]), (kp / NB) & 1)) {
                tc_fence_after();
                // B = V[keys, channels]: MN-major, 64-channel slabs kKBox apart
                // (leading offset), 8-key groups 1024 bytes apart (stride).
                issue_pv<N>(tmem, tmem + col_p + sb * kPStride,
                            sdesc(k_base + stage * stage_bytes, C::kKBox, 1024),
                            kp > 0 ? 1u : 0u, id_pv);
                tc_commit(smem_u32(&bars->pv_done[sb]));
                tc_commit(smem_u32(&bars->empty[stage]));
                ++kp;
                progressed = true;
              }
            }
            // QK^T(kq): needs its key tile and a free S buffer. (POS: P(kq-NB)
            // lies in that buffer, so PV(kq-NB) must have completed; before
            // the first reuse, the warm-up PV that read buffer NB-1 has
            // completed with QK^T(0), whose commit tracks it.)
            if (kq < n && kq < kp + NB) {
              const int stage = kq % stages, sb = kq % NB;
              if (mbar_test_wait(smem_u32(&bars->full[stage]), (kq / stages) & 1) &&
                  (kq < NB ? (!POS || kq == 0 || mbar_test_wait(smem_u32(&bars->s_full[0]), 0))
                           : (mbar_test_wait(smem_u32(&bars->s_free[sb]), ((kq - NB) / NB) & 1) &&
                              (!POS || mbar_test_wait(smem_u32(&bars->pv_done[sb]),
                                                      ((kq - NB) / NB) & 1))))) {
                tc_fence_after();
                issue_qk<C::kQBox, C::kKBox, HSF / 16>(tmem + col_s + sb * N, sdesc(q_base, 16, 1024),
                                             sdesc(k_base + stage * stage_bytes, 16, 1024), nk,
                                             kIdQK);
                tc_commit(smem_u32(&bars->s_full[sb]));
                ++kq;
                progressed = true;
              }
            }
            if (progressed) {
              spins = 0;
              continue;
            }
            if ((++spins & 15u) == 0) {
              if (*abort) { ok = false; break; }
              if (globaltimer() - t0 > kWaitLimitNs * 4) {
                *abort = 1;
                raise_flag(P.err_flags, PA_DEVERR_TIMEOUT);
                ok = false;
                break;
              }
            }
          }
        }
        // every MMA issued above completes before TMEM is released
        tc_commit(smem_u32(&bars->drain));
        drain_wait(smem_u32(&bars->drain), 0, P.err_flags);
      }
      __syncwarp();
    } else if (FP8 && warp >= C::kConvWarp) {
      // =============== E4M3 -> fp16 key tiles (FP8 cache) ===============
      // Per tile: wait for its E4M3 rows (full8) and a free fp16 stage
      // (empty, committed after PV of the tile that used it before), convert
      // (every E4M3 value is an fp16 normal, so exactly) into the 128-byte-
      // swizzled K-major layout the MMAs read (16-byte chunk c of row r at
      // c ^ (r & 7) in its 64-channel slab), then release both. The tile's
      // N rows x hs/16 chunks are dealt to the 128 threads chunk by chunk,
      // so consecutive threads read consecutive chunks of a row (no bank
      // conflicts on the E4M3 reads).
      const int ct = tid - C::kConvWarp * 32;
      const int hs16 = hs / 16;
      const int dr = 128 / hs16, dj = 128 - dr * hs16;  // (row, chunk) step of 128 chunks
      const int st8 = P.stages8;
      for (int k = 0; k < n; ++k) {
        const int s8 = k % st8, s16 = k % stages;
        bool okc = wait_bar(smem_u32(&bars->full8[s8]), (k / st8) & 1, abort, P.err_flags);
        if (okc && k >= stages)
          okc = wait_bar(smem_u32(&bars->empty[s16]), ((k / stages) & 1) ^ 1, abort,
                         P.err_flags);
        if (!__all_sync(0xffffffffu, okc)) break;
        const uint8_t* src8 = k8_s + s8 * P.stage8_bytes;
        int r = ct / hs16, j = ct - r * hs16;
#pragma unroll 2
        for (; r < N; r += dr, j += dj) {
          if (j >= hs16) {
            j -= hs16;
            ++r;
            if (r >= N) break;
          }
          uint8_t* dst = k_s + s16 * stage_bytes + r * 128;
          const uint4 v = *reinterpret_cast<const uint4*>(src8 + r * hs + j * 16);
          const uint4 lo = make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                                      e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2(v.z & 0xffffu), e4m3x2_to_f16x2(v.z >> 16),
                                      e4m3x2_to_f16x2(v.w & 0xffffu), e4m3x2_to_f16x2(v.w >> 16));
          const int c0 = j * 16, ch = (c0 >> 3) & 7;
          uint8_t* d = dst + (c0 >> 6) * C::kKBox;
          *reinterpret_cast<uint4*>(d + ((ch ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(d + (((ch + 1) ^ (r & 7)) << 4)) = hi;
        }
        fence_proxy_async();  // the generic-proxy stores, before the MMAs read them
        mbar_arrive(smem_u32(&bars->full[s16]));
        mbar_arrive(smem_u32(&bars->empty8[s8]));
      }
    }
  }

  if (W.status != 0) grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Shared-memory budgets: one CTA per SM (the opt-in maximum less a margin
// for the static Work/Barriers block and the 1024-byte alignment pad), and
// half an SM for the two-CTAs-per-SM prefill shape.
constexpr int kSmemBudget = 227 * 1024 - 1024;
constexpr int kHalfSmemBudget = 113 * 1024 - 1024;

inline int q_bytes(const Shape& s) { return s.qr * ((s.hs + 63) / 64) * 128; }
inline int stage_bytes(const Shape& s) { return s.n * ((s.hs + 63) / 64) * 128; }
inline int stage8_bytes(const Shape& s) { return s.n * s.hs; }
inline int smem_bytes(const Shape& s) {
  return q_bytes(s) + s.stages * stage_bytes(s) + s.stages8 * stage8_bytes(s) + 1024;
}
inline int tmem_cols_used(const Shape& s) {
  return s.vg + s.nb * s.n + (s.pos ? 0 : s.nb * s.n / 2);
}
inline int tmem_alloc_cols(int used) {
  int c = 32;
  while (c < used) c <<= 1;
  return c;
}

template <typename T, int N, int QR, int NB, int HSF, int VGF, int STF, bool FP8 = false,
          bool POS = false>
cudaError_t launch_shape(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                         const Shape& s) {
  using C = Tile<N, QR, NB, FP8>;
  P.hs = g.hs;
  P.slabs = (g.hs + 63) / 64;
  P.stages = s.stages;
  P.stage_bytes = stage_bytes(s);
  P.q_bytes = q_bytes(s);
  P.col_s = s.vg;
  P.col_p = POS ? s.vg : s.vg + NB * N;
  P.tmem_cols = tmem_alloc_cols(tmem_cols_used(s));
  P.stages8 = s.stages8;
  P.stage8_bytes = stage8_bytes(s);
  const size_t smem = (size_t)smem_bytes(s);
  // the softcap code is compiled only into the kernels that use it; the
  // dynamic shared-memory limit is raised once per device to the opt-in
  // maximum less the kernel's static shared memory
  static std::atomic<bool> configured[2][64];
  const int cap = P.softcap_on ? 1 : 0;
  auto kern = cap ? tc_attn_kernel<T, N, QR, NB, true, HSF, VGF, STF, FP8, POS>
                  : tc_attn_kernel<T, N, QR, NB, false, HSF, VGF, STF, FP8, POS>;
  cudaError_t e = once_per_device(configured[cap], g.device, [&] {
    int optin = 0;
    cudaFuncAttributes fa;
    cudaError_t r = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                           g.device);
    if (r == cudaSuccess) r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - (int)fa.sharedSizeBytes);
  });
  if (e != cudaSuccess) {
    set_launch_step("kernel shared-memory attribute");
    return e;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_launch_step("driver tensor-map encoder lookup");
    return cudaErrorNotSupported;
  }
  const CUtensorMapDataType dt = std::is_same<T, __nv_bfloat16>::value
                                     ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // Cache rows [num_blocks*bs, hs]: boxes of 64 channels x box_rows rows (a
  // box that reaches past channel hs reads zeros there); FP8: boxes of whole
  // E4M3 rows (hs bytes) x box_rows rows, unswizzled.
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)g.hs, (cuuint64_t)g.num_blocks * g.bs};
  const cuuint64_t strides[1] = {(cuuint64_t)g.hs * 2};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r;
  if (FP8) {
    const cuuint64_t strides8[1] = {(cuuint64_t)g.hs};
    const cuuint32_t box8[2] = {(cuuint32_t)g.hs, (cuuint32_t)P.box_rows};
    r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.key_cache), dims,
            strides8, box8, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint32_t box[2] = {64, (cuuint32_t)P.box_rows};
    r = enc(&map, dt, 2, const_cast<void*>(a.key_cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    set_launch_step("cache tensor map");
    return cudaErrorInvalidValue;
  }
  // Query rows [T*H, hs]: one QR-row box per 64-channel slab loads a token's heads.
  CUtensorMap qmap;
  const cuuint64_t qdims[2] = {(cuuint64_t)g.hs, (cuuint64_t)a.num_tokens * g.H};
  const cuuint32_t qbox[2] = {64, (cuuint32_t)QR};
  r = enc(&qmap, dt, 2, const_cast<void*>(a.query), qdims, strides, qbox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_launch_step("query tensor map");
    return cudaErrorInvalidValue;
  }
  // grid: the decode units, the prefill units, or (mixed) both
  const int64_t units = ph == Phase::kDecode  ? (int64_t)P.units
                        : ph == Phase::kMixed ? (int64_t)P.units + nq
                                              : nq;
  e = launch_pdl(kern, dim3((unsigned)units), dim3(C::kThreads), smem, a.stream, map, qmap, P);
  if (e != cudaSuccess) {
    set_launch_step("attention kernel launch");
    return e;
  }
  if (ph == Phase::kPrefill) return e;
  e = launch_combine<T>(P, g.H, (int64_t)(P.seq_end - P.seq_begin), a.stream);
  if (e != cudaSuccess) set_launch_step("combine kernel launch");
  return e;
}

// FP8-cache decode at 192/128 with H <= 64: fp16 key stages and E4M3 stages
// (GLM-style decode: 37.2 us per decode call with 3 + 2, 39.2 us with 2 + 4;
// a tile holds its fp16 stage from conversion through PV).
constexpr int kFp8Stages16 = 3, kFp8Stages8 = 2;

// The 192/128 shapes compiled with their geometry fixed (pa_tc_glm.cu).
inline bool fixed_shape(const Shape& s) {
  if (s.hs != 192 || s.vg != 128 || s.pair) return false;
  if (s.stages8)
    return s.n == 128 && s.qr == 64 && s.nb == 2 && s.stages == kFp8Stages16 &&
           s.stages8 == kFp8Stages8;
  if (s.pos) return s.n == 64 && s.qr == 128 && s.nb == 2 && s.stages == 2;
  return (s.n == 128 && s.qr == 64 && s.nb == 2 && s.stages == 4) ||
         (s.n == 128 && s.qr == 128 && s.nb == 2 && s.stages == 3);
}
template <typename T>
cudaError_t launch_fixed(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                         const Shape& s);
// FP8-cache shapes (pa_tc_fp8.cu).
template <typename T>
cudaError_t launch_fp8(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                       const Shape& s);

}  // namespace tc
}  // namespace pa
