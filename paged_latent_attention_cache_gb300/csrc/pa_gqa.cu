// SEPARATE layout: grouped-query paged attention over separate key and value
// caches, with an optional sink logit per query head and optional RMSNorm of
// the query and key heads (the op's second dense mode; PR #1940 page, oracle
// of "SEPARATE (GQA, RoPE, softcap, local window, head_sink, q/k RMSNorm)";
// input order value(2), value_cache(4), head_sink(11), q_norm_weight(12),
// k_norm_weight(13) on the PR #1978 page).
//
//   write: k = RoPE(RMSNorm(key[t, g]) * w_k) -> key_cache[slot, g]
//          value[t, g]                      -> value_cache[slot, g]
//   read:  q = RoPE(RMSNorm(query[t, h]) * w_q), g = h / (H / kvH),
//          s_j = scale * q . K_j[g] (softcap as in LATENT), m = max(s, z_h),
//          out[t, h] = sum_j e^(s_j - m) V_j[g] / (sum_j e^(s_j - m) + e^(z_h - m))
//
// The read kernel has the single-CTA LATENT kernel's structure (warp roles,
// pipelines, bounded waits, split-KV decode with a device-side plan): a work
// unit is tpc tokens x grp query heads of one kv head (decode: grp rows), the
// query rows arrive by a 3-D TMA box (tokens x heads of the group), and each
// key tile's stage holds the key rows (QK^T's B operand) followed by the
// value rows (PV's B operand), both gathered by 3-D boxes (channels, kv head,
// cache rows) through the block table.
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "pa_tc_common.cuh"

namespace pa {

// ===========================================================================
// Write phase: one warp per (token, kv head); lane l holds channels
// [8l, 8l + 8) of the key row (hs <= 256) and of the value row (vhs <= 256).
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(256)
separate_write_kernel(const T* __restrict__ key, const T* __restrict__ value,
                      const T* __restrict__ cos_cache, const T* __restrict__ sin_cache,
                      const T* __restrict__ k_norm, const int32_t* __restrict__ slot_mapping,
                      const int32_t* __restrict__ cumseq, const int32_t* __restrict__ past,
                      int32_t num_seqs, T* __restrict__ key_cache, T* __restrict__ value_cache,
                      int64_t num_tokens, int kvh, int hs, int vhs, int ro, int rd,
                      int interleaved, int cos_rows, int64_t num_slots, float eps,
                      int32_t* err_flags) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int ng = hs >> 3, nvg = vhs >> 3;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < num_tokens * kvh; row += warps) {
    const int64_t t = row / kvh;
    const int g = (int)(row - t * kvh);
    const int32_t slot = slot_mapping[t];
    float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (lane < ng) unpack8<T>(*reinterpret_cast<const uint4*>(key + row * hs + lane * 8), x);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (lane < nvg) v = *reinterpret_cast<const uint4*>(value + row * vhs + lane * 8);
    if (slot < 0) {
      if (slot < -1 && g == 0 && lane == 0) raise_flag(err_flags, PA_DEVERR_SLOT);
      continue;
    }
    if ((int64_t)slot >= num_slots) {
      if (g == 0 && lane == 0) raise_flag(err_flags, PA_DEVERR_SLOT);
      continue;
    }
    int32_t b;
    int64_t pos;
    if (!locate_token(t, cumseq, past, num_seqs, (g == 0 && lane == 0) ? err_flags : nullptr, &b,
                      &pos))
      continue;
    if (rd > 0 && (pos < 0 || pos >= cos_rows)) {
      if (g == 0 && lane == 0)
        raise_flag(err_flags, pos < 0 ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
      continue;
    }
    if (k_norm) {  // RMSNorm over the head's hs channels, in f32
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float r = 1.0f / sqrtf(ss / (float)hs + eps);
      if (lane < ng) {
        float w[8];
        unpack8<T>(*reinterpret_cast<const uint4*>(k_norm + lane * 8), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = x[e] * r * w[e];
      }
    }
    const int d0 = lane * 8;
    const bool rot = rd > 0 && d0 >= ro && d0 < ro + rd;
    // the rotary partner group of a half-split rotation lives in another lane
    const int half = rd >> 1;
    const int src = rot && !interleaved ? ((d0 - ro < half) ? lane + (half >> 3)
                                                            : lane - (half >> 3))
                                        : lane;
    float xp[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) xp[e] = __shfl_sync(0xffffffffu, x[e], src & 31);
    if (rot) rope8<T>(x, xp, d0, ro, rd, interleaved, cos_cache + pos * half, sin_cache + pos * half);
    const int64_t crow = (int64_t)slot * kvh + g;
    if (lane < ng) *reinterpret_cast<uint4*>(key_cache + crow * hs + d0) = pack8<T>(x);
    if (lane < nvg) *reinterpret_cast<uint4*>(value_cache + crow * vhs + d0) = v;
  }
}

cudaError_t launch_separate_write(const Geometry& g, const SeparateWriteArgs& a) {
  const int64_t rows = a.num_tokens * g.kvh;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)g.num_sms * 16;
  if (blocks > cap) blocks = cap;
  const int64_t num_slots = (int64_t)g.num_blocks * g.bs;
  auto go = [&](auto* typed) {
    using TP = std::remove_pointer_t<decltype(typed)>;
    separate_write_kernel<TP><<<(unsigned)blocks, threads, 0, a.stream>>>(
        (const TP*)a.key, (const TP*)a.value, (const TP*)a.cos_cache, (const TP*)a.sin_cache,
        (const TP*)a.k_norm, a.slot_mapping, a.cumseq, a.past, a.num_seqs, (TP*)a.key_cache,
        (TP*)a.value_cache, a.num_tokens, g.kvh, g.hs, g.vhs, g.ro, g.rd, g.interleaved,
        g.cos_rows, num_slots, g.rms_eps, a.err_flags);
  };
  if (g.dtype == PA_DTYPE_BF16) go((__nv_bfloat16*)nullptr);
  else go((__half*)nullptr);
  return cudaGetLastError();
}

namespace tc {

// ===========================================================================
// Read phase
// ===========================================================================

// One query row (thread = row) in place in its swizzled slabs (16-byte chunk
// c of row r at c ^ (r & 7)): RMSNorm with the weight (when given), then the
// rotation of its rotary channels, both in f32, rounded to T once.
template <typename T, int QBOX>
__device__ __noinline__ void gqa_q_row(uint8_t* q_s, int row, int hs, const Params& P,
                                       int64_t pos) {
  auto at = [&](int d0) -> uint4* {
    const int slab = d0 >> 6, ch = (d0 >> 3) & 7;
    return reinterpret_cast<uint4*>(q_s + slab * QBOX + row * 128 + ((ch ^ (row & 7)) << 4));
  };
  float r = 1.f;
  const T* w = reinterpret_cast<const T*>(P.q_norm);
  if (w) {
    float ss = 0.f;
    for (int d0 = 0; d0 < hs; d0 += 8) {
      float a[8];
      unpack8<T>(*at(d0), a);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(a[e], a[e], ss);
    }
    r = 1.0f / sqrtf(ss / (float)hs + P.rms_eps);
  }
  auto load = [&](int d0, float (&a)[8]) {
    unpack8<T>(*at(d0), a);
    if (w) {
      float wv[8];
      unpack8<T>(*reinterpret_cast<const uint4*>(w + d0), wv);
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = a[e] * r * wv[e];
    }
  };
  const int ro = P.rd > 0 ? P.ro : hs, rd = P.rd, half = rd >> 1;
  const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * half;
  const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * half;
  for (int d0 = 0; d0 < hs; d0 += 8) {
    const bool rot = d0 >= ro && d0 < ro + rd;
    if (!rot && !w) continue;  // nothing to change
    if (rot && !P.interleaved) {
      if (d0 >= ro + half) continue;  // rotated with its partner below
      float a[8], bb[8], na[8], nb[8];
      load(d0, a);
      load(d0 + half, bb);
#pragma unroll
      for (int e = 0; e < 8; ++e) { na[e] = a[e]; nb[e] = bb[e]; }
      rope8<T>(na, bb, d0, ro, rd, 0, crow, srow);
      rope8<T>(nb, a, d0 + half, ro, rd, 0, crow, srow);
      *at(d0) = pack8<T>(na);
      *at(d0 + half) = pack8<T>(nb);
      continue;
    }
    float a[8];
    load(d0, a);
    if (rot) {
      float dummy[8];
      rope8<T>(a, dummy, d0, ro, rd, 1, crow, srow);
    }
    *at(d0) = pack8<T>(a);
  }
}

template <int N>
__device__ __noinline__ void gqa_issue_qk(uint32_t d, uint64_t a0, uint64_t b0, int nk, uint32_t id,
                                          uint32_t qbox16, uint32_t kbox16) {
  for (int kk = 0; kk < nk; ++kk) {
    const uint32_t col = (uint32_t)(kk & 3) * 2, slab = (uint32_t)(kk >> 2);
    mma_ss(d, a0 + (slab * qbox16 + col), b0 + (slab * kbox16 + col), id, kk > 0 ? 1u : 0u);
  }
}
template <int N>
__device__ __noinline__ void gqa_issue_pv(uint32_t d, uint32_t a, uint64_t b0, uint32_t acc0,
                                          uint32_t id) {
#pragma unroll
  for (int kk = 0; kk < N / 16; ++kk)
    mma_ts(d, a + kk * 8, b0 + (uint64_t)(kk * 128), id, (acc0 || kk > 0) ? 1u : 0u);
}

template <typename T, int N, int QR, bool CAP>
__global__ void __launch_bounds__(Tile<N, QR, 2>::kThreads, 1)
tc_gqa_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const __grid_constant__ CUtensorMap qmap, const __grid_constant__ Params P) {
  using C = Tile<N, QR, 2>;
  constexpr int NB = 2;
  const int hs = P.hs, slabs = P.slabs, vg = P.vg, stages = P.stages;
  const int stage_bytes = P.stage_bytes, q_bytes = P.q_bytes;
  const int col_s = P.col_s, col_p = P.col_p;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Work work;
  __shared__ Barriers bars_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + q_bytes;  // stage: key slabs, then value slabs, N rows each
  Barriers* bars = &bars_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = P.kvh, grp = P.grp, H = P.H;
  const int unit = blockIdx.x / kvh;
  const int gk = blockIdx.x - unit * kvh;  // this CTA's kv head
  const int vhs = P.vhs;

  if (warp == 0) {
    if (!P.early) grid_dep_wait();
    Work w;
    if (P.decode) {
      w = decode_plan_warp<N>(P, unit, reinterpret_cast<int*>(q_s), q_bytes / 4);
      fence_proxy_async();  // the scratch is overwritten by the query TMA later
      if (w.status == 0) {
        const int32_t q0 = P.cumseq[w.b], q1 = P.cumseq[w.b + 1];
        if (lane == 0 && w.split == 0 && gk == 0)
          P.ws_plan[w.b - P.seq_begin] = make_int2(w.first, w.splits);
        if (q1 - q0 != 1) {
          if (lane == 0 && gk == 0) raise_flag(P.err_flags, PA_DEVERR_DECODE_QLEN);
          w.status = 2;
        } else if (q0 < 0 || q0 >= P.num_tokens) {
          if (lane == 0 && gk == 0) raise_flag(P.err_flags, PA_DEVERR_CUMSEQ);
          w.status = 2;
        } else {
          w.t = q0;
          w.past = P.past[w.b];
          w.pos = w.past;
          w.ntok = 1;
        }
      }
    } else {
      w = prefill_group_warp(P, unit, P.tpc);
      if (w.status == 0) {
        const int64_t lo_key = P.window >= 0 ? max((int64_t)0, w.pos - P.window) : 0;
        w.t_begin = lo_key / N;
        w.t_end = (w.pos + w.ntok - 1) / N + 1;
      }
    }
    if (w.status == 0) {
      const int64_t pos_hi = w.pos + w.ntok - 1;
      const bool bad_ctx = w.past < 0 || pos_hi >= (int64_t)P.max_blocks * P.bs ||
                           w.t + w.ntok > P.num_tokens;
      const bool bad_pos = P.rd > 0 && pos_hi >= P.cos_rows;
      if (bad_ctx || bad_pos) {
        if (lane == 0 && gk == 0)
          raise_flag(P.err_flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
        const int nt = (int)min((int64_t)w.ntok, P.num_tokens - w.t);
        for (int i = lane; i < nt * grp * vhs; i += 32) {
          const int tt = i / (grp * vhs), rem = i - tt * grp * vhs;
          const int hh = gk * grp + rem / vhs, c = rem % vhs;
          reinterpret_cast<T*>(P.out)[((w.t + tt) * H + hh) * (int64_t)vhs + c] =
              Half<T>::from_f32(0.f);
        }
        w.status = 2;
      }
    }
    if (lane == 0) work = w;
    fence_proxy_async();
  } else if (warp == 1 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
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
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
  } else if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), (uint32_t)P.tmem_cols);
    tmem_relinquish();
  }
  if (warp != 0 && !P.early) grid_dep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  const Work W = work;

  if (W.status == 0) {
    const int64_t t = W.t, pos = W.pos, t_begin = W.t_begin;
    const int32_t b = W.b;
    const int splits = W.splits, ntok = W.ntok, rows = W.ntok * grp;
    const int64_t pos_hi = pos + ntok - 1;
    const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
    const int64_t lo_hi = P.window >= 0 ? max((int64_t)0, pos_hi - P.window) : 0;
    const int n = (int)max((int64_t)0, W.t_end - t_begin);
    const int64_t part = blockIdx.x;  // partial slot of a decode split: unit * kvh + gk

    if (warp < 4) {
      // =================== softmax / epilogue ===================
      const int row = tid;  // row = token offset * grp + head in the group
      const bool live = warp * 32 < rows;
      const int64_t pos_r = row < rows ? pos + row / grp : -1;
      const int64_t lo_r = P.window >= 0 ? max((int64_t)0, pos_r - P.window) : 0;
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int k = 0; k < n && ok; ++k) {
        if (k == 0) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->q_tma), 0, abort, P.err_flags));
          if (ok && row < rows && (P.rd > 0 || P.q_norm)) gqa_q_row<T, C::kQBox>(q_s, row, hs, P, pos_r);
          fence_proxy_async();
          mbar_arrive(smem_u32(&bars->q_full));
          if (!ok) break;
        }
        const int sb = k & 1;
        const int64_t j0 = (t_begin + k) * N;
        const bool edge = j0 < lo_hi || j0 + N - 1 > pos;
        ok = __all_sync(0xffffffffu,
                        wait_bar(smem_u32(&bars->s_full[sb]), (k / NB) & 1, abort, P.err_flags));
        if (!ok) break;
        float factor = 1.f;
        bool rescale = false;
        const float sl = CAP ? 1.f : P.scale_log2;
        const uint32_t s_addr = lane_addr + col_s + sb * N;
        int clo = 0, chi = N - 1;
        if (edge) {
          clo = (int)min((int64_t)N, max((int64_t)0, lo_r - j0));
          chi = (int)max((int64_t)-1, min((int64_t)(N - 1), pos_r - j0));
        }
        int mode = 2;
        if (live) {
          tc_fence_after();
          float vmax = -INFINITY, vmin = INFINITY;
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (c + e >= clo && c + e <= chi) {
                vmax = fmaxf(vmax, __uint_as_float(r[e]));
                vmin = fminf(vmin, __uint_as_float(r[e]));
              }
            }
          }
          float mt;
          if (CAP) {
            mt = vmax == -INFINITY ? -INFINITY : P.cap_out * tanh_ex2(vmax * P.cap_in);
            const bool small = row >= rows || fmaxf(vmax, -vmin) <= P.cap_vlim;
            mode = (P.cap_poly && __all_sync(0xffffffffu, small)) ? 1 : 2;
          } else {
            mt = vmax * sl;
          }
          if (k == 0) {
            m_used = mt;
          } else if (mt > m_used + kRescaleLog2) {
            factor = ex2(m_used - mt);
            m_used = mt;
            l *= factor;
            rescale = true;
          }
        }
        if (edge) {  // zero the value rows of keys no row of the unit sees
          uint8_t* vst = k_s + (k % stages) * stage_bytes + P.k_bytes;
          const int vslabs = vg / 64;
          for (int i = tid; i < N * vslabs * 8; i += 128) {
            const int rr = i / (vslabs * 8);
            const int rem = i - rr * (vslabs * 8);
            const int slab = rem / 8, ch = rem & 7;
            const int64_t j = j0 + rr;
            if (j < lo || j > pos_hi)
              *reinterpret_cast<uint4*>(vst + slab * C::kKBox + rr * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        if (k >= NB) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[sb]),
                                                ((k - NB) / NB) & 1, abort, P.err_flags));
          if (!ok) break;
        }
        if (live) {
          tc_fence_after();
          float lsum = 0.f;
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          const ExpArgs A{sl, mu, P.cap_in, P.cap_out, P.cap_a[0], P.cap_a[1], P.cap_a[2],
                          P.cap_a[3], P.cap_a[4]};
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32], pk[16];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
            if (!(c >= clo && c + 31 <= chi)) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c + e < clo || c + e > chi) r[e] = __float_as_uint(-INFINITY);
            }
            if (!CAP) lsum += exp_chunk<T, 0>(r, pk, A);
            else if (mode == 1) lsum += exp_chunk<T, 1>(r, pk, A);
            else lsum += exp_chunk<T, 2>(r, pk, A);
            tmem_st16(lane_addr + col_p + sb * (N / 2) + c / 2, pk);
          }
          l += lsum;
          if (__any_sync(0xffffffffu, rescale)) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[(k - 1) & 1]),
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
        mbar_arrive(smem_u32(&bars->s_free[sb]));
        mbar_arrive(smem_u32(&bars->p_full[sb]));
      }

      // ---- epilogue ----
      grid_dep_launch();
      named_sync(2, 160);
      ok = __all_sync(0xffffffffu, ok && !*abort);
      if (ok)
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[(n - 1) & 1]),
                                              ((n - 1) / NB) & 1, abort, P.err_flags));
      if (ok && live) {
        tc_fence_after();
        const bool bad = bars->bad != 0;
        const int hh = gk * grp + row % grp;  // this row's query head
        if (splits == 1) {
          // the sink logit z joins the denominator: with M = max(m, z),
          // out = O 2^(m-M) / (l 2^(m-M) + 2^(z-M)) (log2 domain)
          float f = 1.f, lz = l;
          if (P.head_sink && row < rows) {
            const float z = Half<T>::to_f32(reinterpret_cast<const T*>(P.head_sink)[hh]) * kLog2e;
            const float M = fmaxf(m_used, z);
            f = m_used == -INFINITY ? 0.f : ex2(m_used - M);
            lz = l * f + ex2(z - M);
          }
          const float inv = (lz > 0.f && !bad) ? f / lz : 0.f;
          T* dst = reinterpret_cast<T*>(P.out) + ((t + row / grp) * H + hh) * (int64_t)vhs;
          const bool vec = vhs % 8 == 0;
#pragma unroll 1
          for (int c = 0; c < vg && c < vhs; c += 16) {
            uint32_t r[16];
            tmem_ld16(lane_addr + c, r);
            if (row < rows) {
              if (vec && c + 16 <= vhs) {
                uint4 o[2];
                uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  ow[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv,
                                   __uint_as_float(r[2 * e + 1]) * inv);
                reinterpret_cast<uint4*>(dst + c)[0] = o[0];
                reinterpret_cast<uint4*>(dst + c)[1] = o[1];
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (c + e < vhs) dst[c + e] = Half<T>::from_f32(__uint_as_float(r[e]) * inv);
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
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                     __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
            }
          }
          if (row < rows) {
            P.ws_ml[(part * kRows + row) * 2 + 0] = bad ? __int_as_float(0x7fc00000) : m_used;
            P.ws_ml[(part * kRows + row) * 2 + 1] = bad ? 0.f : l;
          }
        }
      }
    } else if (warp == C::kProdWarp) {
      // =================== TMA producer ===================
      if (lane == 0) {  // Q: one 3-D box (64 channels x grp heads x tpc tokens) per slab
        const uint32_t qb = smem_u32(&bars->q_tma);
        const int qrows = grp * (P.decode ? 1 : P.tpc);
        mbar_expect_tx(qb, (uint32_t)(slabs * qrows * 128));
        for (int slab = 0; slab < slabs; ++slab)
          tma_load_3d(smem_u32(q_s) + slab * C::kQBox, &qmap, slab * 64, gk * grp, (int)t, qb);
      }
      int dirty_from = 0;
      if (P.early && P.own_slots) dirty_from = (int)max((int64_t)0, W.past / N - t_begin);
      bool waited = !P.early;
      const int nsub = N / P.box_rows;
      const int32_t* bt = P.block_table + (int64_t)b * P.max_blocks;
      int issued = 0;
      for (int k = 0; k < n; ++k) {
        const int stage = k % stages;
        if (!waited && k >= dirty_from) {
          grid_dep_wait();
          waited = true;
        }
        // the boxes' rows (block ids loaded) before the wait for the stage,
        // so that the copies go out as soon as the stage is free
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
        if (k >= stages) {
          bool okw = true;
          if (lane == 0)
            okw = wait_bar(smem_u32(&bars->empty[stage]), ((k / stages) & 1) ^ 1, abort,
                           P.err_flags);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
        }
        if (lane == 0) mbar_expect_tx(smem_u32(&bars->full[stage]), (uint32_t)stage_bytes);
        __syncwarp();
        if (lane < nsub) {  // lane sb issues the boxes of rows sb: key slabs, then value slabs
          const uint32_t full = smem_u32(&bars->full[stage]);
          const uint32_t dst0 = smem_u32(k_s + stage * stage_bytes) + lane * P.box_rows * 128;
#pragma unroll 1
          for (int slab = 0; slab < slabs; ++slab)
            tma_load_3d(dst0 + slab * C::kKBox, &kmap, slab * 64, gk, y, full);
#pragma unroll 1
          for (int slab = 0; slab < P.vslabs; ++slab)
            tma_load_3d(dst0 + P.k_bytes + slab * C::kKBox, &vmap, slab * 64, gk, y, full);
        }
        issued = k + 1;
        __syncwarp();
      }
      if (!waited) grid_dep_wait();
      if (*abort && lane == 0) {
        drain_wait(smem_u32(&bars->q_tma), 0, P.err_flags);
        for (int st = 0; st < stages && st < issued; ++st) {
          const int kl = issued - 1 - ((issued - 1 - st) % stages);
          drain_wait(smem_u32(&bars->full[st]), (kl / stages) & 1, P.err_flags);
        }
      }
      __syncwarp();
      named_arrive(2, 160);
    } else if (warp == C::kMmaWarp) {
      // =================== MMA issuer ===================
      if (lane == 0) {
        constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
        constexpr uint32_t kIdQK = idesc_f16(kBf16, kRows, N, false);
        const uint32_t id_pv = idesc_f16(kBf16, kRows, vg, true);
        const int nk = hs / 16;
        const uint32_t q_base = smem_u32(q_s);
        const uint32_t k_base = smem_u32(k_s);
        bool ok = wait_bar(smem_u32(&bars->q_full), 0, abort, P.err_flags);
        if (ok) {
          tc_fence_after();
          int kq = 0, kp = 0;
          const uint64_t t0 = globaltimer();
          uint32_t spins = 0;
          while (kp < n) {
            bool progressed = false;
            if (kp < kq) {
              const int stage = kp % stages, sb = kp & 1;
              if (mbar_test_wait(smem_u32(&bars->p_full[sb]), (kp / NB) & 1)) {
                tc_fence_after();
                gqa_issue_pv<N>(tmem, tmem + col_p + sb * (N / 2),
                                sdesc(k_base + stage * stage_bytes + P.k_bytes, C::kKBox, 1024),
                                kp > 0 ? 1u : 0u, id_pv);
                tc_commit(smem_u32(&bars->pv_done[sb]));
                tc_commit(smem_u32(&bars->empty[stage]));
                ++kp;
                progressed = true;
              }
            }
            if (kq < n && kq < kp + NB) {
              const int stage = kq % stages, sb = kq & 1;
              if (mbar_test_wait(smem_u32(&bars->full[stage]), (kq / stages) & 1) &&
                  (kq < NB ||
                   mbar_test_wait(smem_u32(&bars->s_free[sb]), ((kq - NB) / NB) & 1))) {
                tc_fence_after();
                gqa_issue_qk<N>(tmem + col_s + sb * N, sdesc(q_base, 16, 1024),
                                sdesc(k_base + stage * stage_bytes, 16, 1024), nk, kIdQK,
                                C::kQBox >> 4, C::kKBox >> 4);
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
        tc_commit(smem_u32(&bars->drain));
        drain_wait(smem_u32(&bars->drain), 0, P.err_flags);
      }
      __syncwarp();
    }
  }

  if (W.status != 0) grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)P.tmem_cols);
  }
}

// Split merge for grouped-query decode, with the sink logit: for query head
// h of sequence x, the partials of kv head g = h / grp, row h % grp of each
// split are folded as in tc_combine_kernel, then the sink joins the sum.
// Thread = 4 consecutive value channels of one head.
template <typename T>
__global__ void __launch_bounds__(256) gqa_combine_kernel(const __grid_constant__ Params P) {
  grid_dep_wait();
  constexpr int CPT = 4;
  const int vg = P.vg;
  const int tph = vg / CPT, hpb = 256 / tph;
  const int hl = (int)threadIdx.x / tph;
  if (hl >= hpb) return;
  const int x = blockIdx.x;
  const int h = blockIdx.y * hpb + hl;
  const int c0 = ((int)threadIdx.x % tph) * CPT;
  const int2 plan = P.ws_plan[x];
  const int32_t q0 = P.cumseq[P.seq_begin + x];
  const int S = plan.y;
  if (S > 1 && h < P.H && c0 < P.vhs) {
    const int g = h / P.grp, r = h % P.grp;
    float M = -INFINITY, L = 0.f, o[CPT] = {0.f, 0.f, 0.f, 0.f};
    bool bad = false;
    for (int s = 0; s < S; ++s) {
      const int64_t slot = ((int64_t)(plan.x + s) * P.kvh + g) * kRows + r;
      const float2 ml = reinterpret_cast<const float2*>(P.ws_ml)[slot];
      const float4 ov = *reinterpret_cast<const float4*>(P.ws_o + slot * vg + c0);
      bad |= isnan(ml.x);
      if (ml.y > 0.f && !isnan(ml.x)) {
        if (ml.x > M) {
          const float f = ex2(M - ml.x);
          L *= f;
#pragma unroll
          for (int e = 0; e < CPT; ++e) o[e] *= f;
          M = ml.x;
        }
        const float w = ex2(ml.x - M);
        L += w * ml.y;
        o[0] += w * ov.x; o[1] += w * ov.y; o[2] += w * ov.z; o[3] += w * ov.w;
      }
    }
    float f = 1.f;
    if (P.head_sink) {
      const float z = Half<T>::to_f32(reinterpret_cast<const T*>(P.head_sink)[h]) * kLog2e;
      const float Mz = fmaxf(M, z);
      f = M == -INFINITY ? 0.f : ex2(M - Mz);
      L = L * f + ex2(z - Mz);
    }
    const float inv = (L > 0.f && !bad) ? f / L : 0.f;
    T* dst = reinterpret_cast<T*>(P.out) + ((int64_t)q0 * P.H + h) * P.vhs + c0;
#pragma unroll
    for (int e = 0; e < CPT; ++e)
      if (c0 + e < P.vhs) dst[e] = Half<T>::from_f32(o[e] * inv);
  }
}

// ===========================================================================
// Host side
// ===========================================================================
namespace {

constexpr int kSmemBudget = 227 * 1024 - 1024;

struct GShape {
  int n, qr, stages, slabs, vslabs, vg;
};

bool gqa_pick(const Geometry& g, Phase ph, GShape* s) {
  const int grp = g.H / g.kvh;
  if (g.hs < 64 || g.hs > 256 || g.vhs < 64 || g.vhs > 256 || grp > kRows) return false;
  GShape t;
  t.slabs = (g.hs + 63) / 64;
  t.vslabs = (g.vhs + 63) / 64;
  t.vg = 64 * t.vslabs;
  t.n = t.vg > 128 ? 64 : 128;
  t.qr = (ph == Phase::kDecode && grp <= 64) ? 64 : 128;
  const int q = t.qr * t.slabs * 128, st = t.n * (t.slabs + t.vslabs) * 128;
  t.stages = (kSmemBudget - 1024 - q) / st;
  if (t.stages > 8) t.stages = 8;
  if (t.stages < 2) return false;
  *s = t;
  return true;
}

inline int64_t gqa_decode_units(const Geometry& g, int64_t nseq) {
  // one wave of CTAs over the (sequence split, kv head) pairs, at least one
  // unit per sequence
  const int64_t wave = (g.num_sms + g.kvh - 1) / g.kvh;
  return nseq > wave ? nseq : wave;
}

inline size_t gqa_ws_bytes(const GShape& s, int64_t units, int kvh, int64_t nseq) {
  const size_t per = (size_t)units * kvh * kRows;
  const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
  const size_t ml = ((per * 2 * sizeof(float)) + 255) & ~(size_t)255;
  return o + ml + (size_t)nseq * sizeof(int2);
}

template <typename T, int N, int QR>
cudaError_t gqa_launch(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                       const GShape& s) {
  using C = Tile<N, QR, 2>;
  const int grp = g.H / g.kvh;
  P.hs = g.hs;
  P.slabs = s.slabs;
  P.vslabs = s.vslabs;
  P.vg = s.vg;
  P.groups = 1;
  P.stages = s.stages;
  P.k_bytes = N * s.slabs * 128;
  P.stage_bytes = N * (s.slabs + s.vslabs) * 128;
  P.q_bytes = QR * s.slabs * 128;
  P.col_s = s.vg;
  P.col_p = s.vg + 2 * N;
  {
    const int used = s.vg + 3 * N;
    int c = 32;
    while (c < used) c <<= 1;
    P.tmem_cols = c;
  }
  const size_t smem = (size_t)P.q_bytes + (size_t)s.stages * P.stage_bytes + 1024;
  static std::atomic<bool> configured[2][64];
  const int cap = P.softcap_on ? 1 : 0;
  auto kern = cap ? tc_gqa_kernel<T, N, QR, true> : tc_gqa_kernel<T, N, QR, false>;
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
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint64_t nslots = (cuuint64_t)g.num_blocks * g.bs;
  // caches viewed as [slots][kv heads][channels]: boxes of 64 channels x one
  // kv head x box_rows cache rows
  CUtensorMap kmap, vmap, qmap;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)g.hs, (cuuint64_t)g.kvh, nslots};
    const cuuint64_t str[2] = {(cuuint64_t)g.hs * 2, (cuuint64_t)g.kvh * g.hs * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)P.box_rows};
    if (enc(&kmap, dt, 3, const_cast<void*>(a.key_cache), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      set_launch_step("key cache tensor map");
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)g.vhs, (cuuint64_t)g.kvh, nslots};
    const cuuint64_t str[2] = {(cuuint64_t)g.vhs * 2, (cuuint64_t)g.kvh * g.vhs * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)P.box_rows};
    if (enc(&vmap, dt, 3, const_cast<void*>(a.value_cache), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      set_launch_step("value cache tensor map");
      return cudaErrorInvalidValue;
    }
  }
  {
    // query [T][H][hs]: boxes of 64 channels x grp heads x tpc tokens
    const cuuint64_t dims[3] = {(cuuint64_t)g.hs, (cuuint64_t)g.H, (cuuint64_t)a.num_tokens};
    const cuuint64_t str[2] = {(cuuint64_t)g.hs * 2, (cuuint64_t)g.H * g.hs * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)grp, (cuuint32_t)(P.decode ? 1 : P.tpc)};
    if (enc(&qmap, dt, 3, const_cast<void*>(a.query), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      set_launch_step("query tensor map");
      return cudaErrorInvalidValue;
    }
  }
  const int64_t units = ph == Phase::kDecode ? (int64_t)P.units : nq;
  e = launch_pdl(kern, dim3((unsigned)(units * g.kvh)), dim3(C::kThreads), smem, a.stream, kmap,
                 vmap, qmap, P);
  if (e != cudaSuccess) {
    set_launch_step("attention kernel launch");
    return e;
  }
  if (ph != Phase::kDecode) return e;
  const int hpb = 256 / (s.vg / 4);
  e = launch_pdl(gqa_combine_kernel<T>, dim3((unsigned)nq, (unsigned)((g.H + hpb - 1) / hpb)),
                 dim3(256), 0, a.stream, P);
  if (e != cudaSuccess) set_launch_step("combine kernel launch");
  return e;
}

}  // namespace
}  // namespace tc

bool separate_supported(const Geometry& g, Phase ph) {
  tc::GShape s;
  return tc::gqa_pick(g, ph, &s);
}

size_t separate_call_workspace(const Geometry& g, Phase ph, int32_t seq_begin, int32_t seq_end) {
  tc::GShape s;
  if (ph == Phase::kPrefill || seq_end <= seq_begin || !tc::gqa_pick(g, ph, &s)) return 0;
  const int64_t nq = (int64_t)(seq_end - seq_begin);
  return tc::gqa_ws_bytes(s, tc::gqa_decode_units(g, nq), g.kvh, nq);
}

cudaError_t launch_separate_read(const Geometry& g, Phase ph, const ReadArgs& a) {
  tc::GShape s;
  if (!tc::gqa_pick(g, ph, &s)) return cudaErrorNotSupported;
  const int grp = g.H / g.kvh;
  const int tpc = ph == Phase::kPrefill ? (s.qr / grp > 0 ? s.qr / grp : 1) : 1;
  const int64_t nseq = (int64_t)(a.seq_end - a.seq_begin);
  const int64_t nq = ph == Phase::kDecode ? nseq : (a.num_tokens + tpc - 1) / tpc + nseq;
  if (nq <= 0 || (ph == Phase::kPrefill && a.num_tokens <= 0)) return cudaSuccess;
  tc::Params P{};
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
  P.out_scale = 1.f;
  P.scale_log2 = g.scale * tc::kLog2e;
  P.softcap_on = g.softcap > 0.f ? 1 : 0;
  P.cap_in = g.softcap > 0.f ? g.scale / g.softcap : 0.f;
  P.cap_out = g.softcap * tc::kLog2e;
  P.cap_poly = 0;
  P.cap_vlim = 0.f;
  if (g.softcap > 0.f) {
    const double ci = (double)g.scale / (double)g.softcap;
    const double co = (double)g.softcap * 1.4426950408889634;
    const double t[5] = {1.0, -1.0 / 3.0, 2.0 / 15.0, -17.0 / 315.0, 62.0 / 2835.0};
    bool normal = true;
    double pw = ci;
    for (int i = 0; i < 5; ++i) {
      const double c = co * t[i] * pw;
      normal = normal && std::isfinite(c) && std::fabs(c) >= (double)FLT_MIN &&
               std::fabs(c) <= (double)FLT_MAX;
      P.cap_a[i] = (float)c;
      pw *= ci * ci;
    }
    const double vlim = 0.25 / ci;
    P.cap_poly = normal && vlim <= (double)FLT_MAX ? 1 : 0;
    P.cap_vlim = P.cap_poly ? (float)vlim : 0.f;
  }
  P.window = g.window;
  P.decode = ph == Phase::kDecode ? 1 : 0;
  P.box_rows = s.n < g.bs ? s.n : g.bs;
  P.early = (g.flags & PA_FLAG_AFTER_WRITE) ? 1 : 0;
  P.own_slots = (g.flags & PA_FLAG_OWN_SLOTS) ? 1 : 0;
  P.tpc = tpc;
  P.mixed = 0;
  P.pf_begin = a.seq_begin;
  P.pf_end = a.seq_end;
  P.kvh = g.kvh;
  P.grp = grp;
  P.head_sink = a.head_sink;
  P.q_norm = a.q_norm;
  P.rms_eps = g.rms_eps;
  if (ph == Phase::kDecode) {
    const int64_t units = tc::gqa_decode_units(g, nq);
    P.units = (int)units;
    const size_t per = (size_t)units * g.kvh * tc::kRows;
    const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
    const size_t ml = ((per * 2 * sizeof(float)) + 255) & ~(size_t)255;
    if (a.workspace == nullptr || a.workspace_bytes < tc::gqa_ws_bytes(s, units, g.kvh, nq)) {
      set_launch_step("decode workspace");
      return cudaErrorInvalidValue;
    }
    char* w = reinterpret_cast<char*>(a.workspace);
    P.ws_o = reinterpret_cast<float*>(w);
    P.ws_ml = reinterpret_cast<float*>(w + o);
    P.ws_plan = reinterpret_cast<int2*>(w + o + ml);
  }
  const bool bf16 = g.dtype == PA_DTYPE_BF16;
  auto go = [&](auto* typed) -> cudaError_t {
    using TP = std::remove_pointer_t<decltype(typed)>;
    if (s.n == 128 && s.qr == 64) return tc::gqa_launch<TP, 128, 64>(g, ph, a, P, nq, s);
    if (s.n == 128) return tc::gqa_launch<TP, 128, 128>(g, ph, a, P, nq, s);
    if (s.qr == 64) return tc::gqa_launch<TP, 64, 64>(g, ph, a, P, nq, s);
    return tc::gqa_launch<TP, 64, 128>(g, ph, a, P, nq, s);
  };
  return bf16 ? go((__nv_bfloat16*)nullptr) : go((__half*)nullptr);
}

}  // namespace pa
