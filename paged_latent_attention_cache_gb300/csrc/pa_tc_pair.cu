// Tensor-core read phase for the 576/512 latent geometry on a CTA pair.
//
// Operator (paged_attention.rs, module doc "Read phase" / attn_impl):
//   out[h] = softmax_j(scale * RoPE(q_h) . K_j) @ K_j[:512],  j in [lo, pos].
// A 128-head output accumulator of 512 f32 columns fills a whole SM's TMEM
// and a 128 x 576 query tile most of its shared memory, so one token is
// handled by a cluster of two CTAs on two SMs that split the latent channels:
//
//   CTA c in {0,1} holds the query channels [288c, 288c+288) (four 64-channel
//   slabs and a 32-channel half slab) and loads five 64-channel slabs of
//   every key tile. Its QK^T covers 18 of the 36 16-channel K steps, so
//   S = S_0 + S_1 with S_c its partial. CTA c accumulates O[:, 256c : 256c+256]
//   = P @ V with V = four of its key slabs: each output half on one SM and no
//   product computed twice.
//
// The partial scores are exchanged by four dedicated warps (6-9, one per
// TMEM lane quadrant): per tile they read S_c from TMEM, send it to the peer
// through distributed shared memory (st.async, completing on the peer's
// mbarrier), add the peer's rows (the f32 sum S_0 + S_1 is the same in both
// CTAs, so both hold bit-identical S, P, m and l) and write the sum back for
// the softmax warps; the exchange of tile k+1 overlaps the softmax of tile
// k. The partials travel as f32 (32 KB per tile, one tile in flight), so the
// exchange adds no rounding and no range limit to the scores.
// Three S buffers: O 256 + 3 x 64 + P 2 x 32 = 512 TMEM columns.
//
// Roles: warps 0-3 softmax/epilogue (thread = head row = TMEM lane), warp 4
// TMA producer, warp 5 TMEM allocation + the MMA-issuing thread, warps 6-9
// score exchange (FP8 cache: warps 10-11 convert E4M3 tiles to fp16). Key
// tiles of 64 keys in 3 stages (FP8 cache: 2 fp16 stages fed from 2 E4M3
// stages); every wait is bounded.
//
// Work units: decode runs one pair per unit of the device plan (a sequence's
// key split). Prefill is persistent: at most one wave of pairs, each looping
// over tokens T-1-p, T-1-p-npairs, ... (the longest first). Every role
// resolves the units itself and counts key tiles across them, so the key
// ring, the S/P buffers and the exchange carry on from one token to the next;
// a token's query is loaded once QK^T of the previous token's last tile has
// completed, and its first PV starts the O accumulator afresh.
#include "pa_tc_cluster.cuh"

namespace pa {
namespace tc {

// FP8 cache with a bf16 query: one query row of this CTA's slabs (four full
// 128-byte-swizzled slabs from global slab q_full0, and a 32-channel half
// slab) from bf16 to fp16 in place. Rotary channels (inside the full slabs)
// are rotated in f32 and rounded once; every other 16-byte chunk of the row
// is converted where it lies (an element-wise conversion needs no
// unswizzling). A value beyond 65504 is saturated and flags PA_DEVERR_RANGE.
template <typename T, int QBOX, int QHALF>
__device__ __noinline__ void pair_q_row_to_f16(uint8_t* q_s, int row, int q_full0, int q_full_off,
                                               int q_half_off, const Params& P, int64_t pos) {
  const int c_lo = q_full0 * 64, c_hi = c_lo + 4 * 64;
  const bool rope = P.rd > 0 && P.ro >= c_lo && P.ro + P.rd <= c_hi;
  const int ro = P.ro, rd = P.rd, half = rd >> 1;
  bool big = false;
  auto at = [&](int d0) -> uint4* {
    const int slab = (d0 >> 6) - q_full0, ch = (d0 >> 3) & 7;
    return reinterpret_cast<uint4*>(q_s + q_full_off + slab * QBOX + row * 128 +
                                    ((ch ^ (row & 7)) << 4));
  };
  if (rope) {
    const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * half;
    const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * half;
    if (!P.interleaved) {
      for (int d0 = ro; d0 < ro + half; d0 += 8) {
        float a[8], bb[8], na[8], nb[8];
        unpack8<T>(*at(d0), a);
        unpack8<T>(*at(d0 + half), bb);
#pragma unroll
        for (int e = 0; e < 8; ++e) { na[e] = a[e]; nb[e] = bb[e]; }
        rope8<T>(na, bb, d0, ro, rd, 0, crow, srow);
        rope8<T>(nb, a, d0 + half, ro, rd, 0, crow, srow);
        *at(d0) = pack8_f16_sat(na, &big);
        *at(d0 + half) = pack8_f16_sat(nb, &big);
      }
    } else {
      for (int d0 = ro; d0 < ro + rd; d0 += 8) {
        float a[8], dummy[8];
        unpack8<T>(*at(d0), a);
        rope8<T>(a, dummy, d0, ro, rd, 1, crow, srow);
        *at(d0) = pack8_f16_sat(a, &big);
      }
    }
  }
  for (int s = 0; s < 4; ++s) {
    uint4* base = reinterpret_cast<uint4*>(q_s + q_full_off + s * QBOX + row * 128);
    for (int pc = 0; pc < 8; ++pc) {
      const int d0 = (q_full0 + s) * 64 + ((pc ^ (row & 7)) << 3);
      if (rope && d0 >= ro && d0 < ro + rd) continue;  // already fp16
      float a[8];
      unpack8<T>(base[pc], a);
      base[pc] = pack8_f16_sat(a, &big);
    }
  }
  uint4* hb = reinterpret_cast<uint4*>(q_s + q_half_off + row * 64);
  for (int pc = 0; pc < 4; ++pc) {
    float a[8];
    unpack8<T>(hb[pc], a);
    hb[pc] = pack8_f16_sat(a, &big);
  }
  if (big) raise_flag(P.err_flags, PA_DEVERR_RANGE);
}

// Work of prefill unit u: token T - 1 - u (the tokens with the most keys,
// the last of each sequence, come first), with its key-tile range. status
// 0: attend; 1: no work here (a token outside [seq_begin, seq_end), or one
// that cannot be located); 2: an invalid context or position (reported,
// output rows to be zeroed). Errors are raised into `flags` when non-null.
template <int N>
__device__ Work pair_prefill_work(const Params& P, int64_t u, int32_t* flags) {
  Work w;
  w.status = 1;
  w.splits = 1;
  int32_t b;
  int64_t pos;
  const int64_t tok = P.num_tokens - 1 - u;
  if (locate_token(tok, P.cumseq, P.past, P.num_seqs, flags, &b, &pos) && b >= P.seq_begin &&
      b < P.seq_end) {
    w.status = 0;
    w.b = b;
    w.t = tok;
    w.pos = pos;
    w.past = P.past[b];
    const int64_t lo_key = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
    w.t_begin = lo_key / N;
    w.t_end = pos / N + 1;
    const bool bad_ctx = w.past < 0 || w.pos >= (int64_t)P.max_blocks * P.bs;
    const bool bad_pos = P.rd > 0 && w.pos >= P.cos_rows;
    if (bad_ctx || bad_pos) {
      raise_flag(flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
      w.status = 2;
    }
  }
  return w;
}

// The i-th work unit of a CTA pair. Decode: the one unit of the device plan
// (`first`, i == 0). Prefill: the grid is at most one wave of pairs, and
// pair p takes units p, p + npairs, p + 2 npairs, ... of the P.units tokens
// (`first` is unit p, resolved in the prologue). False past the last unit.
template <int N>
__device__ __forceinline__ bool pair_unit(const Params& P, const Work& first, int i, int pair,
                                          int npairs, int32_t* flags, Work* w) {
  if (i == 0) {
    *w = first;
    return P.decode || pair < P.units;
  }
  if (P.decode) return false;
  const int64_t u = pair + (int64_t)i * npairs;
  if (u >= P.units) return false;
  *w = pair_prefill_work<N>(P, u, flags);
  return true;
}

template <int N, int STAGES, bool FP8 = false>
struct PairCfg {
  // warps 0-3, 4, 5, 6-9 (see above); FP8: converter warps 10-11
  static constexpr int kThreads = FP8 ? 384 : 320;
  static constexpr int kSlabs = 5;                  // 64-channel slabs per CTA (of 9)
  static constexpr int kSteps = 18;                 // 16-channel QK^T K-steps per CTA
  static constexpr int kQBox = kRows * 128;         // bytes per full query slab (SW128)
  static constexpr int kQHalf = kRows * 64;         // the 32 channels of slab 4 (SW64)
  static constexpr int kQBytes = 4 * kQBox + kQHalf;
  static constexpr int kKBox = N * 128;             // bytes per key slab of a stage
  static constexpr int kStageBytes = kSlabs * kKBox;
  static constexpr int kXBytes = kRows * N * 4;     // incoming partial-S rows
  // FP8 cache: two E4M3 stages of N rows x this CTA's 320 channels (a box
  // of 256 channels and one of 64: a TMA box is at most 256 elements wide)
  static constexpr int kStages8 = FP8 ? 2 : 0;
  static constexpr int kStage8Bytes = N * kSlabs * 64;
  static constexpr int kSmemData =
      kQBytes + STAGES * kStageBytes + kXBytes + kStages8 * kStage8Bytes;
  static constexpr int kVG = 256;                   // output channels per CTA
  static constexpr int kSBufs = 3;                  // S buffers in TMEM
  static constexpr int kColO = 0;
  static constexpr int kColS = kVG;
  static constexpr int kColP = kVG + kSBufs * N;
  static constexpr int kTmemCols = 512;
  static_assert(kVG + kSBufs * N + N <= 512, "TMEM budget");
  static_assert(N % 32 == 0 && N <= 128, "key tile");
};

struct PairBarriers {
  uint64_t full[4], empty[4];
  uint64_t full8[2], empty8[2];  // FP8 cache: E4M3 ring (TMA -> converter warps)
  uint64_t s_part[3];  // QK^T(k) has written this CTA's partial S (tcgen05.commit)
  uint64_t s_sum[3];   // the exchange warps have written S_0 + S_1 back (128 arrivals)
  uint64_t s_free[3];  // the softmax warps are done with the S buffer (128 arrivals)
  uint64_t p_full[2], pv_done[2];
  uint64_t q_tma, q_full;
  uint64_t x_in[1];   // x_s holds the peer's partial rows (local expect_tx + the
                       // peer's st.async complete_tx bytes)
  uint64_t x_out[1];  // the peer has read the rows this CTA sent into its x_s
  uint64_t drain;
  uint32_t tmem_base;
  int bad_mask;  // bit (a & 31): attended unit a read a block id outside the pool
  int abort;
  int xfail;  // an exchange warp's wait failed: all four leave after the tile's barrier
};

// FP8: the cache holds E4M3 codes; two converter warps turn each E4M3 tile
// into the fp16 tile the MMAs read, the query is rounded to fp16 once, and
// P is fp16 (every E4M3 value is an fp16 normal, so the keys are exact).
template <typename T, int N, int STAGES, bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<N, STAGES, FP8>::kThreads, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap qmap64, const __grid_constant__ CUtensorMap kmap8b,
               const __grid_constant__ Params P) {
  using C = PairCfg<N, STAGES, FP8>;
  using TM = typename std::conditional<FP8, __half, T>::type;  // MMA operand type
  constexpr int G = 2, VG = C::kVG, NS = C::kSBufs;
  // Score exchange: f32 partials, one 32 KB tile in x_s at a time. (A 16-bit
  // format would hold two tiles, but it rounds a partial logit L by |L| *
  // 2^-11, several times P's own rounding once |L| reaches tens, and it
  // overflows beyond 65504.)
  constexpr int kXTile = kRows * N * 4;  // bytes per tile
  static_assert(kXTile <= C::kXBytes, "exchange buffer");
  extern __shared__ uint8_t smem_raw[];
  __shared__ Work work;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + C::kQBytes;
  float* x_s = reinterpret_cast<float*>(smem + C::kQBytes + STAGES * C::kStageBytes);
  uint8_t* k8_s = smem + C::kQBytes + STAGES * C::kStageBytes + C::kXBytes;  // FP8 ring
  PairBarriers* bars = reinterpret_cast<PairBarriers*>(smem + C::kSmemData);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t g = cluster_rank();         // channel half == value group
  const uint32_t peer = g ^ 1u;
  const int unit = blockIdx.x / G;
  const int vhs = P.vhs;

  // ---- prologue (same plan in both CTAs of the pair) ----
  // As in the single-CTA kernel: inputs are read only after griddepcontrol.wait,
  // except with P.early (the previous kernel is the write phase), where the
  // producer waits before its first cache load.
  if (warp == 0) {
    if (!P.early) grid_dep_wait();
    Work w;
    if (P.decode) {
      // the query region is free until the query load after the plan
      w = decode_plan_warp<N>(P, unit, reinterpret_cast<int*>(q_s), C::kQBytes / 4);
      fence_proxy_async();  // the scratch is overwritten by the query TMA later
      if (w.status == 0) {
        const int32_t q0 = P.cumseq[w.b], q1 = P.cumseq[w.b + 1];
        if (lane == 0 && w.split == 0 && g == 0)
          P.ws_plan[w.b - P.seq_begin] = make_int2(w.first, w.splits);
        if (q1 - q0 != 1) {
          if (lane == 0 && g == 0) raise_flag(P.err_flags, PA_DEVERR_DECODE_QLEN);
          w.status = 2;
        } else if (q0 < 0 || q0 >= P.num_tokens) {
          if (lane == 0 && g == 0) raise_flag(P.err_flags, PA_DEVERR_CUMSEQ);
          w.status = 2;
        } else {
          w.t = q0;
          w.past = P.past[w.b];
          w.pos = w.past;
        }
      }
    } else {
      // this pair's first unit (later ones are resolved as the roles reach them)
      w = pair_prefill_work<N>(P, unit, (lane == 0 && g == 0) ? P.err_flags : nullptr);
      if (w.status == 2) {  // invalid context or position: the token's output rows are zero
        T* out_row = reinterpret_cast<T*>(P.out) + w.t * (int64_t)P.H * vhs;
        for (int i = lane; i < P.H * VG; i += 32) {
          const int h = i / VG, c = i % VG;
          out_row[(int64_t)h * vhs + g * VG + c] = Half<T>::from_f32(0.f);
        }
      }
    }
    if (P.decode && w.status == 0) {
      const bool bad_ctx = w.past < 0 || w.pos >= (int64_t)P.max_blocks * P.bs;
      const bool bad_pos = P.rd > 0 && w.pos >= P.cos_rows;
      if (bad_ctx || bad_pos) {
        if (lane == 0 && g == 0)
          raise_flag(P.err_flags, bad_ctx ? PA_DEVERR_CONTEXT : PA_DEVERR_POSITION);
        T* out_row = reinterpret_cast<T*>(P.out) + w.t * (int64_t)P.H * vhs;
        for (int i = lane; i < P.H * VG; i += 32) {
          const int h = i / VG, c = i % VG;
          out_row[(int64_t)h * vhs + g * VG + c] = Half<T>::from_f32(0.f);
        }
        w.status = 2;
      }
    }
    if (lane == 0) work = w;
  } else if (warp == 1 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // (FP8: complete when both converter warps have written their rows)
      mbar_init(smem_u32(&bars->full[s]), FP8 ? 64 : 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int s = 0; s < C::kStages8; ++s) {
      mbar_init(smem_u32(&bars->full8[s]), 1);
      mbar_init(smem_u32(&bars->empty8[s]), 64);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bars->s_part[i]), 1);
      mbar_init(smem_u32(&bars->s_sum[i]), kRows);
      mbar_init(smem_u32(&bars->s_free[i]), kRows);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->p_full[i]), kRows);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->q_tma), 1);
    mbar_init(smem_u32(&bars->q_full), kRows);
    mbar_init(smem_u32(&bars->x_in[0]), 1);
    mbar_init(smem_u32(&bars->x_out[0]), 1);
    // armed for tile 0
    mbar_expect_tx(smem_u32(&bars->x_in[0]), kXTile);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->bad_mask = 0;
    bars->abort = 0;
    bars->xfail = 0;
    fence_barrier_init();
  } else if (warp == 4 && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
    prefetch_tmap(&qmap64);
    if (FP8) prefetch_tmap(&kmap8b);
  } else if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp != 0 && !P.early) grid_dep_wait();
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  const Work W = work;

  {
    // Every role walks the pair's units (pair_unit) on its own and counts key
    // tiles globally across them, so the ring stages, S/P buffers, exchange
    // buffer and their barrier phases simply continue from one unit to the
    // next; the query region, q_tma and q_full turn over once per attended
    // unit (a: the number of units attended so far).
    const int npairs = (int)(gridDim.x / G);
    const int pair = unit;
    const int slab0 = 4 * (int)g;  // global slab of local key slab 0
    // Query layout in shared memory: CTA 0 holds full slabs 0-3 (SW128) then
    // channels 256-287 as a 64-byte-swizzled half slab; CTA 1 holds channels
    // 288-319 as the half slab, then full slabs 5-8.
    const int q_full0 = g ? 5 : 0;                         // global slab of full slab 0
    const int q_full_off = g ? C::kQHalf : 0;              // byte offset of full slab 0
    const int q_half_off = g ? 0 : 4 * C::kQBox;           // byte offset of the half slab

    if (warp < 4) {
      // =================== softmax / epilogue ===================
      const int row = tid;
      const bool live = warp * 32 < P.H;
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
      int32_t* rflags = (tid == 0 && g == 0) ? P.err_flags : nullptr;  // (units after the first)
      bool ok = true;
      int kbase = 0;  // global index of the unit's first key tile
      int au = 0;     // units attended so far
      for (int iu = 0; ok; ++iu) {
        Work w;
        if (!pair_unit<N>(P, W, iu, pair, npairs, iu == 0 ? nullptr : rflags, &w)) break;
        if (w.status == 2 && iu > 0 && row < P.H) {  // invalid context or position: zero rows
          T* zrow = reinterpret_cast<T*>(P.out) + w.t * (int64_t)P.H * vhs + (int64_t)row * vhs +
                    g * VG;
          for (int c = 0; c < VG; ++c) zrow[c] = Half<T>::from_f32(0.f);
        }
        if (w.status != 0) continue;
        const int64_t t = w.t, pos = w.pos, t_begin = w.t_begin;
        const int splits = w.splits;
        const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
        const int n = (int)max((int64_t)0, w.t_end - t_begin);
        const int64_t part = (int64_t)pair * G + g;
        T* out_row = reinterpret_cast<T*>(P.out) + t * (int64_t)P.H * vhs;
        float m_used = -INFINITY, l = 0.f;
        // Pass kk = -1 (first attended unit only) runs the tile code once with
        // every wait, arrive, shared memory write and state update switched
        // off, on whatever TMEM holds: it brings the loop's instructions into
        // the instruction cache while the query and the first key tile are
        // still in flight. (The opaque start keeps the compiler from peeling
        // it into a copy of its own.)
        int k_first = au == 0 ? -1 : 0;
        asm volatile("" : "+r"(k_first));
        for (int kk = k_first; kk < n && ok; ++kk) {
        const bool dry = kk < 0;
        const int k = dry ? -1 : kbase + kk;  // global tile index (stages, buffers, phases)
        if (kk == 0) {  // every attended unit has n >= 1 tiles: its query
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->q_tma), au & 1, abort, P.err_flags));
          // RoPE in place on this CTA's slabs (the pair kernel only runs when
          // the rotary channels and their partners lie inside one CTA's slabs).
          if (FP8 && !std::is_same<T, __half>::value) {
            // bf16 query, fp16 MMA operands: this CTA's query channels of the
            // row become fp16 in place (rotary channels rotated in f32 first)
            if (ok && row < P.H)
              pair_q_row_to_f16<T, C::kQBox, C::kQHalf>(q_s, row, q_full0, q_full_off,
                                                        q_half_off, P, pos);
          } else if (ok && P.rd > 0 && row < P.H) {
            const int c_lo = q_full0 * 64, c_hi = c_lo + 4 * 64;  // full query slabs only
            if (P.ro >= c_lo && P.ro + P.rd <= c_hi) {
              const T* crow = reinterpret_cast<const T*>(P.cos_cache) + pos * (P.rd >> 1);
              const T* srow = reinterpret_cast<const T*>(P.sin_cache) + pos * (P.rd >> 1);
              auto at = [&](int d0) -> uint4* {
                const int slab = (d0 >> 6) - q_full0, ch = (d0 >> 3) & 7;
                return reinterpret_cast<uint4*>(q_s + q_full_off + slab * C::kQBox + row * 128 +
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
          }
          fence_proxy_async();
          mbar_arrive(smem_u32(&bars->q_full));
          if (!ok) break;
        }
        const int sb = dry ? 0 : k % NS;   // S buffer
        const int pb = dry ? 1 : k & 1;    // P buffer
        const int64_t j0 = (t_begin + kk) * N;
        const bool edge = !dry && (j0 < lo || j0 + N - 1 > pos);
        if (!dry) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_sum[sb]), (k / NS) & 1, abort,
                                                P.err_flags));
          if (!ok) break;
        }
        // The tile is handled in 32-column chunks read from TMEM twice (row
        // maximum, then exponentials), which keeps the loop body short.
        float factor = 1.f;
        bool rescale = false;
        const float sl = P.softcap_on ? 1.f : P.scale_log2;
        const uint32_t s_addr = lane_addr + C::kColS + sb * N;
        if (live) {
          tc_fence_after();
          float mt = -INFINITY;
          const bool rewrite = P.softcap_on || edge;
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
            if (rewrite) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                float v = __uint_as_float(r[e]);
                if (P.softcap_on) v = P.cap_out * tanhf(v * P.cap_in);
                const int64_t j = j0 + c + e;
                if (edge && (j < lo || j > pos)) v = -INFINITY;
                r[e] = __float_as_uint(v);
              }
              tmem_st32(s_addr + c, r);
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) mt = fmaxf(mt, __uint_as_float(r[e]));
          }
          if (rewrite) tmem_wait_st();
          mt *= sl;
          if (dry) {
          } else if (kk == 0) {
            m_used = mt;
          } else if (mt > m_used + kRescaleLog2) {
            factor = ex2(m_used - mt);
            m_used = mt;
            l *= factor;
            rescale = true;
          }
        }
        if (edge) {  // zero value rows of masked keys (stale cache slots)
          uint8_t* kst = k_s + (k % STAGES) * C::kStageBytes;
          for (int i = tid; i < N * 4 * 8; i += 128) {
            const int rr = i / 32, rem = i - rr * 32;
            const int slab = rem / 8, ch = rem & 7;
            const int64_t j = j0 + rr;
            if (j < lo || j > pos)
              *reinterpret_cast<uint4*>(kst + slab * C::kKBox + rr * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        if (k >= 2) {  // P buffer pb is free once PV(k-2) has completed
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[pb]),
                                                ((k - 2) >> 1) & 1, abort, P.err_flags));
          if (!ok) break;
        }
        if (live) {
          tc_fence_after();
          float lsum = 0.f;
#pragma unroll 1
          for (int c = 0; c < N; c += 32) {
            uint32_t r[32], pk[16];
            tmem_ld32_nowait(s_addr + c, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ex2(fmaf(__uint_as_float(r[2 * e]), sl, -m_used));
              const float p1 = ex2(fmaf(__uint_as_float(r[2 * e + 1]), sl, -m_used));
              lsum += p0 + p1;
              pk[e] = pack2<TM>(p0, p1);
            }
            tmem_st16(lane_addr + C::kColP + pb * (N / 2) + c / 2, pk);
          }
          if (!dry) l += lsum;
          if (__any_sync(0xffffffffu, rescale)) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[pb ^ 1]),
                                                  ((k - 1) >> 1) & 1, abort, P.err_flags));
            if (ok) {
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < VG; c += 16) {
                uint32_t r[16];
                tmem_ld16(lane_addr + C::kColO + c, r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
                tmem_st16(lane_addr + C::kColO + c, r);
              }
            }
          }
          tmem_wait_st();
        }
        if (!ok) break;
        tc_fence_before();
        if (dry) continue;
        mbar_arrive(smem_u32(&bars->s_free[sb]));
        mbar_arrive(smem_u32(&bars->p_full[pb]));
      }

        // ---- epilogue of the unit ----
        if (!ok) break;
        ok = __all_sync(0xffffffffu, *abort == 0);
        const int kl = kbase + n - 1;  // the unit's last tile
        if (ok)
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[kl & 1]), (kl >> 1) & 1,
                                                abort, P.err_flags));
        if (ok && live) {
        tc_fence_after();
        // The producer set the unit's bit (if any) before it issued the
        // unit's tiles; every tile of the unit has been through QK^T, the
        // exchange and PV since, all ordered behind that issue by barrier
        // waits. (Adding an explicit acquire here measured 1-3 % slower.)
        const bool bad = ((*reinterpret_cast<volatile int*>(&bars->bad_mask) >> (au & 31)) & 1) != 0;
        if (splits == 1) {
          const float inv = (l > 0.f && !bad) ? P.out_scale / l : 0.f;
#pragma unroll 1
          for (int c = 0; c < VG; c += 16) {
            uint32_t r[16];
            tmem_ld16(lane_addr + C::kColO + c, r);
            if (row < P.H) {
              uint4 o[2];
              uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                ow[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv,
                                 __uint_as_float(r[2 * e + 1]) * inv);
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
            if (row < P.H) {
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
          if (row < P.H) {
            P.ws_ml[(part * kRows + row) * 2 + 0] = bad ? __int_as_float(0x7fc00000) : m_used;
            P.ws_ml[(part * kRows + row) * 2 + 1] = bad ? 0.f : l;
          }
        }
        }
        kbase += n;
        ++au;
      }
      grid_dep_launch();
      named_sync(2, 160);
    } else if (warp >= 6 && warp < 10) {  // (FP8: warps 10-11 convert, below)
      // =================== partial-score exchange ===================
      // Warp w handles TMEM lanes 32*(w%4)..+31 (the quadrant its SM
      // sub-partition may access). Per tile: read this CTA's partial S rows,
      // send them to the peer's x_s with st.async (the bytes complete on the
      // peer's x_in), wait for the peer's rows, form S_0 + S_1 (f32 addition
      // is commutative, so both CTAs get the same bits) and write the sum
      // back into the S buffer for the softmax warps. x_s is chunk-major:
      // 16-byte chunk q of row r at [q][r], so a warp's store of one chunk
      // for its 32 rows is 512 contiguous bytes.
      constexpr int kChunks = N / 4;  // 16-byte chunks per row and tile
      const int xq = warp & 3, xrow = xq * 32 + lane, xt = tid - 192;  // xt: 0..127
      const uint32_t lane_addr = tmem + ((uint32_t)(xq * 32) << 16);
      const uint32_t x_row = smem_u32(x_s) + xrow * 16;  // chunk 0 of this row
      const uint32_t x_peer = map_peer(x_row, peer);
      const uint32_t x_in_peer = map_peer(smem_u32(&bars->x_in[0]), peer);
      const uint32_t x_out_peer = map_peer(smem_u32(&bars->x_out[0]), peer);
      volatile int* xfail = &bars->xfail;
      bool ok = true;
      int k = 0;  // global tile index
      for (int iu = 0; ok && *xfail == 0; ++iu) {
        Work w;
        if (!pair_unit<N>(P, W, iu, pair, npairs, nullptr, &w)) break;
        if (w.status != 0) continue;
        const int n = (int)max((int64_t)0, w.t_end - w.t_begin);
        for (int kk = 0; kk < n; ++kk, ++k) {
        const int sb = k % NS;
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_part[sb]), (k / NS) & 1, abort,
                                              P.err_flags));
        uint32_t r[N / 32][32];
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < N / 32; ++c)
            tmem_ld32_nowait(lane_addr + C::kColS + sb * N + c * 32, r[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < N / 32; ++c) reg_fence(r[c]);
          if (k >= 1)  // the peer has read tile k - 1 from x_s
            ok = __all_sync(0xffffffffu, wait_bar_cluster(smem_u32(&bars->x_out[0]),
                                                          (k - 1) & 1, abort, P.err_flags));
        }
        if (ok) {
#pragma unroll
          for (int q = 0; q < kChunks; ++q)
            st_async_b32x4(x_peer + q * kRows * 16, r[q / 8][(4 * q) & 31],
                           r[q / 8][(4 * q + 1) & 31], r[q / 8][(4 * q + 2) & 31],
                           r[q / 8][(4 * q + 3) & 31], x_in_peer);
          ok = __all_sync(0xffffffffu, wait_bar_cluster(smem_u32(&bars->x_in[0]), k & 1, abort,
                                                        P.err_flags));
        }
        if (ok) {
          const uint8_t* src = reinterpret_cast<const uint8_t*>(x_s) + xrow * 16;
#pragma unroll
          for (int q = 0; q < kChunks; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + q * kRows * 16);
            uint32_t* d = &r[q / 8][(4 * q) & 31];
            d[0] = __float_as_uint(__uint_as_float(d[0]) + __uint_as_float(v.x));
            d[1] = __float_as_uint(__uint_as_float(d[1]) + __uint_as_float(v.y));
            d[2] = __float_as_uint(__uint_as_float(d[2]) + __uint_as_float(v.z));
            d[3] = __float_as_uint(__uint_as_float(d[3]) + __uint_as_float(v.w));
          }
        } else if (lane == 0) {
          *xfail = 1;
        }
        // x_s is released to the peer once every row of it has been read (the
        // named barrier); the peer's next tile waits for that, so the release
        // comes before the sum goes back to TMEM. All four exchange warps pass
        // every tile's barrier, a failed tile's included, and leave the loop
        // together after it.
        named_sync(3, 128);
        if (*xfail != 0) break;
        if (xt == 0) {
          // armed for the next tile (after the last one it is never used)
          mbar_expect_tx(smem_u32(&bars->x_in[0]), kXTile);
          arrive_peer_relaxed(x_out_peer);
        }
#pragma unroll
        for (int c = 0; c < N / 32; ++c)
          tmem_st32(lane_addr + C::kColS + sb * N + c * 32, r[c]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->s_sum[sb]));
        }
      }
    } else if (warp == 4) {
      // =================== TMA producer ===================
      // With P.early the write grid may still run: cache rows are read only
      // after griddepcontrol.wait, except (P.own_slots) the first unit's tiles
      // below its sequence's first new position, which the write does not touch.
      bool waited = !P.early;
      const int nsub = N / P.box_rows;
      // the ring the copies land in: key stages, or (FP8) the E4M3 stages
      constexpr int PST = FP8 ? C::kStages8 : STAGES;
      uint64_t* pfull = FP8 ? bars->full8 : bars->full;
      uint64_t* pempty = FP8 ? bars->empty8 : bars->empty;
      int k = 0;        // global tile index
      int au = 0;       // units attended so far (query loads issued)
      int last_k = -1;  // the previous attended unit's last tile
      bool okp = true;
      for (int iu = 0; okp; ++iu) {
        Work w;
        if (!pair_unit<N>(P, W, iu, pair, npairs, nullptr, &w)) break;
        if (w.status != 0) continue;
        const int64_t t = w.t, pos = w.pos, t_begin = w.t_begin;
        const int32_t b = w.b;
        const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
        const int n = (int)max((int64_t)0, w.t_end - t_begin);
        // (the unit's first block ids are requested before anything else)
        BlockIds ids{P.block_table + (int64_t)b * P.max_blocks, t_begin * N, lo, pos,
                     P.box_rows, P.bs, n * nsub};
        ids.start(lane);
        int dirty_from = 0;
        if (P.early && P.own_slots) dirty_from = (int)max((int64_t)0, w.past / N - t_begin);
        // the query region is free once QK^T of the previous unit's last tile
        // has completed
        if (last_k >= 0) {
          bool okw = true;
          if (lane == 0)
            okw = wait_bar(smem_u32(&bars->s_part[last_k % NS]), (last_k / NS) & 1, abort,
                           P.err_flags);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
        }
        if (lane == 0) {  // this CTA's five query slabs (QR = 128 rows: the token's heads)
          atomicAnd(&bars->bad_mask, ~(1 << (au & 31)));
          const uint32_t qb = smem_u32(&bars->q_tma);
          mbar_expect_tx(qb, C::kQBytes);
          for (int j = 0; j < 4; ++j)
            tma_load_2d(smem_u32(q_s) + q_full_off + j * C::kQBox, &qmap, (q_full0 + j) * 64,
                        (int)(t * P.H), qb);
          tma_load_2d(smem_u32(q_s) + q_half_off, &qmap64, g ? 288 : 256, (int)(t * P.H), qb);
        }
        for (int kk = 0; kk < n; ++kk, ++k) {
          const int stage = k % PST;
          if (!waited && kk >= dirty_from) {
            grid_dep_wait();  // the write phase's cache rows are complete and visible
            waited = true;
          }
          // The boxes' rows are worked out before the wait for the stage, so
          // that the copies go out as soon as the stage is free (block size: a
          // power of two).
          int y = (int)P.num_slots;  // out of range: TMA fills zeros
          const int phys = ids.get(kk * nsub, lane & (nsub - 1), lane);
          if (lane < nsub && ids.visible(kk * nsub + lane)) {
            if (phys >= 0 && phys < P.num_blocks) {
              const int64_t key0 = (t_begin + kk) * N + (int64_t)lane * P.box_rows;
              y = (int)((int64_t)phys * P.bs + (key0 & (int64_t)(P.bs - 1)));
            } else {
              atomicOr(&bars->bad_mask, 1 << (au & 31));
              raise_flag(P.err_flags, PA_DEVERR_BLOCK);
            }
          }
          if (k >= PST) {
            bool okw = true;
            if (lane == 0)
              okw = wait_bar(smem_u32(&pempty[stage]), ((k / PST) & 1) ^ 1, abort, P.err_flags);
            if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) {
              okp = false;
              break;
            }
          }
          if (lane == 0)
            mbar_expect_tx(smem_u32(&pfull[stage]), FP8 ? C::kStage8Bytes : C::kStageBytes);
          __syncwarp();
          if (lane < nsub) {
            const uint32_t full = smem_u32(&pfull[stage]);
            if (FP8) {
              // this CTA's 320 E4M3 channels of box_rows rows: 256 into the
              // stage's first part (256-byte rows), 64 into its second part
              const uint32_t d8 = smem_u32(k8_s + stage * C::kStage8Bytes);
              tma_load_2d(d8 + lane * P.box_rows * 256, &kmap, slab0 * 64, y, full);
              tma_load_2d(d8 + N * 256 + lane * P.box_rows * 64, &kmap8b, slab0 * 64 + 256, y,
                          full);
            } else {
              const uint32_t dst0 =
                  smem_u32(k_s + stage * C::kStageBytes) + lane * P.box_rows * 128;
#pragma unroll 1
              for (int j = 0; j < C::kSlabs; ++j)
                tma_load_2d(dst0 + j * C::kKBox, &kmap, (slab0 + j) * 64, y, full);
            }
          }
          __syncwarp();
        }
        ++au;
        last_k = k - 1;
      }
      if (!waited) grid_dep_wait();  // the grid completes after the write grid
      if (*abort && lane == 0) {
        // copies still in flight land before the CTA leaves
        if (au > 0) drain_wait(smem_u32(&bars->q_tma), (au - 1) & 1, P.err_flags);
        for (int st = 0; st < PST && st < k; ++st) {
          const int kl = k - 1 - ((k - 1 - st) % PST);
          drain_wait(smem_u32(&pfull[st]), (kl / PST) & 1, P.err_flags);
        }
      }
      __syncwarp();
      named_arrive(2, 160);
    } else if (warp == 5) {
      // =================== MMA issuer ===================
      if (lane == 0) {
        constexpr bool kBf16 = std::is_same<TM, __nv_bfloat16>::value;
        constexpr uint32_t kIdQK = idesc_f16(kBf16, kRows, N, false);
        constexpr uint32_t kIdPV = idesc_f16(kBf16, kRows, VG, true);
        const uint32_t q_base = smem_u32(q_s);
        const uint32_t k_base = smem_u32(k_s);
        // Two cursors over the attended units: the one QK^T is in and the one
        // PV is in (global first tile, tile count, attended index).
        struct Cursor {
          int iu, first, n, a;
        };
        auto advance = [&](Cursor& c) -> bool {
          for (;;) {
            Work w;
            if (!pair_unit<N>(P, W, ++c.iu, pair, npairs, nullptr, &w)) return false;
            if (w.status != 0) continue;
            c.first += c.n;
            c.n = (int)max((int64_t)0, w.t_end - w.t_begin);
            ++c.a;
            return true;
          }
        };
        Cursor cq{-1, 0, 0, -1}, cp{-1, 0, 0, -1};
        bool more_q = advance(cq), more_p = advance(cp);
        bool ok = true;
        int kq = 0, kp = 0;  // global tiles whose QK^T / PV have been issued
        uint64_t t0 = globaltimer();
        uint32_t spins = 0;
        while (more_p) {
          bool progressed = false;
          if (kp < kq) {
            const int stage = kp % STAGES, pb = kp & 1;
            if (mbar_test_wait(smem_u32(&bars->p_full[pb]), (kp >> 1) & 1)) {
              tc_fence_after();
              const uint32_t vb = k_base + stage * C::kStageBytes;  // V = local slabs 0-3
              // descriptor address field (bytes / 16) advances 2048 / 16 per 16 keys
              const uint64_t b0 = sdesc(vb, C::kKBox, 1024);
              const bool fresh = kp == cp.first;  // the unit's first tile: O starts over
#pragma unroll
              for (int kk = 0; kk < N / 16; ++kk)
                mma_ts(tmem + C::kColO, tmem + C::kColP + pb * (N / 2) + kk * 8,
                       b0 + (uint64_t)(kk * 128), kIdPV, (!fresh || kk > 0) ? 1u : 0u);
              tc_commit(smem_u32(&bars->pv_done[pb]));
              tc_commit(smem_u32(&bars->empty[stage]));
              ++kp;
              if (kp == cp.first + cp.n) more_p = advance(cp);
              progressed = true;
            }
          }
          // QK^T(kq): needs its key tile, a free S buffer (s_free of kq-NS)
          // and, for a unit's first tile, the unit's rotated query (q_full)
          // (at most two tiles ahead of PV: a PV queued behind more QK^T in
          // the in-order tensor pipe would hold its key stage longer)
          if (more_q && kq < kp + 2) {
            const int stage = kq % STAGES, sb = kq % NS;
            if ((kq != cq.first || mbar_test_wait(smem_u32(&bars->q_full), cq.a & 1)) &&
                mbar_test_wait(smem_u32(&bars->full[stage]), (kq / STAGES) & 1) &&
                (kq < NS ||
                 mbar_test_wait(smem_u32(&bars->s_free[sb]), ((kq - NS) / NS) & 1))) {
              tc_fence_after();
              const uint32_t kb = k_base + stage * C::kStageBytes;
              // Descriptors built once; per step only the address field
              // (bytes / 16) moves.
              const uint64_t b0 = sdesc(kb, 16, 1024);
              const uint64_t af0 = sdesc(q_base + q_full_off, 16, 1024);
              const uint64_t ah0 = sdesc64(q_base + q_half_off);
#pragma unroll
              for (int i = 0; i < C::kSteps; ++i) {
                // CTA g covers K steps [18g, 18g+18) = channels [288g, 288g+288):
                // the key operand is local slab e>>2, step e&3 (e = i + 2g); the
                // query operand is a full slab, or the 32-channel half slab.
                const int e = i + 2 * (int)g;
                const uint32_t kslab = (uint32_t)(e >> 2), w = (uint32_t)(e & 3) * 2;
                const bool half = g ? (i < 2) : (i >= 16);
                uint64_t a;
                if (half) {
                  a = ah0 + (uint64_t)((g ? i : i - 16) * 2);
                } else {
                  const uint32_t j = (uint32_t)(g ? (i - 2) >> 2 : i >> 2);
                  const uint32_t wq = (uint32_t)(g ? (i - 2) & 3 : i & 3) * 2;
                  a = af0 + (j * (C::kQBox >> 4) + wq);
                }
                mma_ss(tmem + C::kColS + sb * N, a, b0 + (kslab * (C::kKBox >> 4) + w), kIdQK,
                       i > 0 ? 1u : 0u);
              }
              tc_commit(smem_u32(&bars->s_part[sb]));
              ++kq;
              if (kq == cq.first + cq.n) more_q = advance(cq);
              progressed = true;
            }
          }
          if (progressed) {
            spins = 0;
            t0 = globaltimer();
            continue;
          }
          if ((++spins & 15u) == 0) {
            if (*abort) { ok = false; break; }
            if (globaltimer() - t0 > kWaitLimitNs * 4) {  // no progress for that long
              *abort = 1;
              raise_flag(P.err_flags, PA_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        (void)ok;
        tc_commit(smem_u32(&bars->drain));
        drain_wait(smem_u32(&bars->drain), 0, P.err_flags);
      }
      __syncwarp();
    } else if (FP8 && warp >= 10) {
      // =============== E4M3 -> fp16 key tiles (FP8 cache) ===============
      // The tile's 64 rows x 20 chunks of 16 channels are dealt to the 64
      // threads chunk by chunk (consecutive threads read consecutive 16-byte
      // chunks of a row, so the E4M3 reads do not collide in the shared-
      // memory banks): from the two parts of the E4M3 stage into the five
      // swizzled fp16 slabs (16-byte chunk c of row r at c ^ (r & 7)), once
      // the fp16 stage is free (PV of the tile that used it before is done).
      const int ct = tid - 320;  // 0..63
      constexpr int kS8 = C::kStages8 > 0 ? C::kStages8 : 1;  // (non-FP8 builds never run this)
      int k = 0;  // global tile index
      bool okc = true;
      for (int iu = 0; okc; ++iu) {
        Work w;
        if (!pair_unit<N>(P, W, iu, pair, npairs, nullptr, &w)) break;
        if (w.status != 0) continue;
        const int n = (int)max((int64_t)0, w.t_end - w.t_begin);
        for (int kk = 0; kk < n; ++kk, ++k) {
        const int s8 = k % kS8, s16 = k % STAGES;
        okc = wait_bar(smem_u32(&bars->full8[s8]), (k / kS8) & 1, abort, P.err_flags);
        if (okc && k >= STAGES)
          okc = wait_bar(smem_u32(&bars->empty[s16]), ((k / STAGES) & 1) ^ 1, abort,
                         P.err_flags);
        okc = __all_sync(0xffffffffu, okc);
        if (!okc) break;
        const uint8_t* s8p = k8_s + s8 * C::kStage8Bytes;
#pragma unroll 4
        for (int i = ct; i < N * 20; i += 64) {  // chunk j of row r
          const int r = i / 20, j = i - r * 20;
          uint8_t* dst = k_s + s16 * C::kStageBytes + r * 128;
          const uint4 v = *reinterpret_cast<const uint4*>(
              j < 16 ? s8p + r * 256 + j * 16 : s8p + N * 256 + r * 64 + (j - 16) * 16);
          const uint4 lo = make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                                      e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2(v.z & 0xffffu), e4m3x2_to_f16x2(v.z >> 16),
                                      e4m3x2_to_f16x2(v.w & 0xffffu), e4m3x2_to_f16x2(v.w >> 16));
          const int ch = (j & 3) * 2;  // first 16-byte chunk of the pair in its slab
          uint8_t* d = dst + (j >> 2) * C::kKBox;
          *reinterpret_cast<uint4*>(d + ((ch ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(d + (((ch + 1) ^ (r & 7)) << 4)) = hi;
        }
        fence_proxy_async();
        mbar_arrive(smem_u32(&bars->full[s16]));
        mbar_arrive(smem_u32(&bars->empty8[s8]));
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync_all();  // the peer no longer writes into this CTA's shared memory
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <typename T, bool FP8>
cudaError_t launch_pair_impl(const Geometry& g, Phase ph, const ReadArgs& a, Params& P,
                             int64_t nq) {
  // bf16/fp16 cache: three key stages; FP8 cache: two fp16 key stages fed
  // by the converter warps from two E4M3 stages (the same shared memory)
  constexpr int N = 64, STAGES = FP8 ? 2 : 3;
  using C = PairCfg<N, STAGES, FP8>;
  const size_t smem = C::kSmemData + sizeof(PairBarriers) + 1024;
  static std::atomic<bool> configured[64];
  auto kern = tc_pair_kernel<T, N, STAGES, FP8>;
  cudaError_t e = once_per_device(configured, g.device, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  CUtensorMap map, qmap, map8b;
  const cuuint64_t dims[2] = {576, (cuuint64_t)g.num_blocks * g.bs};
  const cuuint64_t strides[1] = {576 * 2};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r;
  if (FP8) {
    // E4M3 rows of 576 bytes: boxes of 256 and of 64 channels x box_rows rows
    const cuuint64_t strides8[1] = {576};
    const cuuint32_t box_a[2] = {256, (cuuint32_t)P.box_rows};
    const cuuint32_t box_b[2] = {64, (cuuint32_t)P.box_rows};
    r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.key_cache), dims,
            strides8, box_a, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
      r = enc(&map8b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.key_cache), dims,
              strides8, box_b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint32_t box[2] = {64, (cuuint32_t)P.box_rows};
    r = enc(&map, dt, 2, const_cast<void*>(a.key_cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    map8b = map;  // (unused)
  }
  if (r != CUDA_SUCCESS) {
    set_launch_step("cache tensor map");
    return cudaErrorInvalidValue;
  }
  const cuuint64_t qdims[2] = {576, (cuuint64_t)a.num_tokens * g.H};
  const cuuint32_t qbox[2] = {64, (cuuint32_t)kRows};
  r = enc(&qmap, dt, 2, const_cast<void*>(a.query), qdims, strides, qbox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  // 32-channel boxes (64-byte rows, 64-byte swizzle) for the half query slab
  CUtensorMap qmap64;
  const cuuint32_t qbox64[2] = {32, (cuuint32_t)kRows};
  if (r == CUDA_SUCCESS)
    r = enc(&qmap64, dt, 2, const_cast<void*>(a.query), qdims, strides, qbox64, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_launch_step("query tensor map");
    return cudaErrorInvalidValue;
  }
  // decode: one pair per unit of the plan; prefill: at most one wave of
  // pairs, each looping over its share of the nq token units
  int64_t pairs = P.units;
  if (ph != Phase::kDecode) {
    P.units = (int)nq;
    pairs = nq < g.num_sms / 2 ? nq : g.num_sms / 2;
  }
  e = launch_pdl(kern, dim3((unsigned)(pairs * 2)), dim3(C::kThreads), smem, a.stream, map, qmap,
                 qmap64, map8b, P);
  if (e != cudaSuccess) {
    set_launch_step("attention kernel launch");
    return e;
  }
  if (ph != Phase::kDecode) return e;
  e = launch_combine<T>(P, g.H, nq, a.stream);
  if (e != cudaSuccess) set_launch_step("combine kernel launch");
  return e;
}

template <typename T>
cudaError_t launch_pair(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq) {
  return g.fp8 ? launch_pair_impl<T, true>(g, ph, a, P, nq)
               : launch_pair_impl<T, false>(g, ph, a, P, nq);
}

template cudaError_t launch_pair<__nv_bfloat16>(const Geometry&, Phase, const ReadArgs&, Params&,
                                                int64_t);
template cudaError_t launch_pair<__half>(const Geometry&, Phase, const ReadArgs&, Params&,
                                         int64_t);

}  // namespace tc
}  // namespace pa


