// Shared pieces of the tensor-core (tcgen05 / TMEM / TMA) read-phase
// kernels: PTX wrappers, descriptors, bounded mbarrier waits, parameters,
// the device-side decode work plan, the split combine kernel and host-side
// tensor-map / launch helpers. Included by pa_tc.cu and pa_tc_pair.cu.
#pragma once

#include <cuda.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace tc {

constexpr int kThreads = 192;
constexpr int kRows = 128;               // MMA M: TMEM lanes
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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
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
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
      "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
      "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 consecutive columns without waiting; pair with tmem_wait_ld() and
// reg_fence() before the registers are read.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Orders later uses of r after the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]),
                 "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7]));
}
// Programmatic dependent launch controls (no-ops for an ordinary launch).
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh from its definition, tanh(y) = 1 - 2 / (1 + e^(2y)), with one
// ex2.approx and one rcp.approx: absolute error about 1e-7 (the final
// subtraction's rounding), so a softcapped score c*tanh(s/c) is off by
// about c * 1e-7. Saturates to +-1 (e^(2y) -> inf gives 1 - 0, -> 0 gives -1).
__device__ __forceinline__ float tanh_ex2(float y) {
  const float e = ex2(y * (2.f * kLog2e));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return fmaf(-2.f, r, 1.f);
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
  int2* ws_plan;    // [nseq] (first unit, number of key splits) per decode sequence
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
  // Softcap by its odd series in the raw score v: cap_out * tanh(v * cap_in)
  // = v * (cap_a[0] + v^2 (cap_a[1] + ... + v^2 cap_a[4])), used where
  // |v| <= cap_vlim (|v * cap_in| <= 1/4) when cap_poly (coefficients
  // representable as normal floats).
  float cap_a[5];
  float cap_vlim;
  int cap_poly;
  int window;
  int units;         // decode: CTA units (per value group) the grid provides
  int decode;
  int box_rows;      // rows per TMA box: min(N, bs)
  int early;         // the previous kernel is the write phase: inputs other than
                     // the cache may be read before griddepcontrol.wait
  int tpc;           // prefill: consecutive tokens per work unit (rows = tpc * H <= 128)
  int own_slots;     // with early: the write touches no row below a sequence's past
  // One grid for a mixed batch: units [0, units) are the decode splits of
  // sequences [seq_begin, seq_end), the units after them prefill units of
  // sequences [pf_begin, pf_end) (a prefill-only launch has pf_* = seq_*).
  int mixed;
  int pf_begin, pf_end;
  // Accumulator layout: `groups` CTAs (or CTAs of a pair) each hold `vg`
  // value channels of a head (vg a multiple of 64, groups * vg >= vhs).
  int vg, groups;
  // Single-CTA kernel geometry (pa_tc.cu), fixed per launch on the host:
  int hs;            // latent width (channels hs..slabs*64 of the last slab read as zeros)
  int slabs;         // 64-channel slabs per row: ceil(hs / 64)
  int stages;        // key stages in the shared-memory ring (<= 8)
  int stage_bytes;   // N * slabs * 128
  int q_bytes;       // query rows * slabs * 128
  int col_s, col_p;  // TMEM columns of the S and P buffers (O starts at column 0)
  int tmem_cols;     // TMEM columns allocated (a power of two >= 32)
  // FP8 cache (E4M3 codes, value = code * k_scale): the E4M3 tiles land in a
  // ring of their own (stages8 stages of N rows x hs bytes) and are
  // converted to fp16 tiles; k_scale is folded into scale_log2 / the softcap
  // factors and into out_scale, which multiplies the output (1 otherwise).
  int stages8, stage8_bytes;
  float out_scale;
  // SEPARATE layout (grouped-query attention, pa_gqa.cu): a work unit holds
  // tpc tokens x grp query heads of one kv head; keys and values come from
  // their own caches into the two parts of a stage.
  int kvh, grp;            // kv heads; query heads per kv head
  const void* head_sink;   // [H] sink logits (query dtype), or null
  const void* q_norm;      // [hs] RMSNorm weight of the query (query dtype), or null
  float rms_eps;
  int vslabs;              // 64-channel value slabs of a stage
  int k_bytes;             // bytes of a stage's key part (the value part follows)
};

// Compile-time part of a single-CTA kernel configuration: N keys per tile,
// QR query rows kept in shared memory (128, or 64 when H <= 64: the M=128
// MMA then reads rows 64-127 from the next slab, rows that are never
// stored), NB S/P buffers in TMEM. The latent width, value channels and
// stage count are per-launch values in Params.
template <int N, int QR, int NB, bool FP8 = false>
struct Tile {
  static constexpr int kQBox = QR * 128;  // bytes per query slab
  static constexpr int kKBox = N * 128;   // bytes per key slab of a stage
  static_assert(N % 32 == 0 && N <= 128, "key tile");
  static_assert(QR == 64 || QR == 128, "query rows");
  static_assert(NB == 1 || NB == 2, "S/P buffers");
  // Warp roles: 0-3 softmax; producer and MMA issuer on warps 4 and 5, or,
  // with 64 query rows (only softmax warps 0 and 1 hold rows), on warps 6
  // and 7, which share no scheduler partition (warp % 4) with a live
  // softmax warp; warps 4 and 5 then have no role.
  static constexpr int kProdWarp = QR == 64 ? 6 : 4;
  static constexpr int kMmaWarp = kProdWarp + 1;
  // FP8 cache: four converter warps (one per scheduler partition) after the
  // MMA warp turn E4M3 key tiles into fp16 tiles.
  static constexpr int kConvWarp = kMmaWarp + 1;
  static constexpr int kThreads = 32 * (kMmaWarp + 1 + (FP8 ? 4 : 0));
};

struct Barriers {
  uint64_t full[8], empty[8];
  uint64_t full8[8], empty8[8];  // FP8 cache: E4M3 tile ring (TMA -> converters)
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t q_tma, q_full;
  uint64_t drain;
  uint32_t tmem_base;
  int bad;
  int abort;
};

// Resolved work of one CTA (written by warp 0 during the prologue).
struct Work {
  int64_t t, pos, t_begin, t_end;  // t, pos: the unit's first token and its position
  int64_t past;                    // past_seqlens[b]: the sequence's first new position
  int b, splits, first, split;
  int ntok;    // consecutive tokens of sequence b in the unit (rows = ntok * H)
  int status;  // 0 = run, 1 = idle, 2 = error already reported (write nothing more)
  int decode;  // the unit is a decode split
};

// Block ids of the key boxes a producer warp copies, requested 32 boxes at
// a time ahead of use. Box i of the CTA's key range starts at key
// key0 + i * box_rows and lies in one cache block; lane l holds the id of
// box 32 * j + l of the batch j in use, and batch j + 1 is requested as soon
// as batch j comes into use, so the block-table load is normally complete
// before a tile's copies are issued instead of on every tile's path.
// Boxes with no visible key (outside [lo, hi]) or past the range are not
// looked up.
struct BlockIds {
  const int32_t* bt;  // the sequence's block-table row
  int64_t key0, lo, hi;
  int box_rows, bs, nbox;
  int cur, nxt, batch;
  __device__ __forceinline__ bool visible(int i) const {
    const int64_t key = key0 + (int64_t)i * box_rows;
    return i < nbox && key <= hi && key + box_rows - 1 >= lo;
  }
  __device__ __forceinline__ int fetch(int i) const {
    // (block size: a power of two)
    return visible(i) ? bt[(key0 + (int64_t)i * box_rows) >> (__ffs(bs) - 1)] : 0;
  }
  __device__ __forceinline__ void start(int lane) {
    batch = 0;
    cur = fetch(lane);
    nxt = fetch(32 + lane);
  }
  // Id of box `first + sub` (first: a multiple of the boxes per tile, which
  // divides 32; sub < boxes per tile). Called by the whole warp with
  // boxes in increasing order.
  __device__ __forceinline__ int get(int first, int sub, int lane) {
    const int j = first >> 5;
    if (j != batch) {  // the next batch (uniform across the warp)
      batch = j;
      cur = nxt;
      nxt = fetch(32 * (j + 1) + lane);
    }
    return __shfl_sync(0xffffffffu, cur, (first & 31) + sub);
  }
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
// Non-blocking probe (used where one thread polls several barriers).
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

// Bounded wait on an mbarrier phase. try_wait lets the hardware suspend the
// thread while the phase is pending (no issue slots burnt); the wait gives
// up after about a second of %globaltimer time, or as soon as another role
// of the CTA has aborted, and then returns false.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort = 1;
  raise_flag(err, PA_DEVERR_TIMEOUT);
  return false;
}

// Bounded wait used while tearing down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 15u) == 15u && globaltimer() - t0 > kWaitLimitNs) break;
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

// Two E4M3 codes (low byte first) as an fp16x2 word (low half first).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Eight f32 values as fp16, saturated to +-65504; records in *big whether one
// was beyond that range (NaN stays NaN).
__device__ __forceinline__ uint4 pack8_f16_sat(const float (&f)[8], bool* big) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = f[2 * i], b = f[2 * i + 1];
    *big |= fabsf(a) > 65504.f || fabsf(b) > 65504.f;
    a = fminf(fmaxf(a, -65504.f), 65504.f);
    b = fminf(fmaxf(b, -65504.f), 65504.f);
    w[i] = pack2<__half>(a, b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Probabilities of one 32-column chunk of a row's scores (softmax pass 2):
// p = 2^(s - mu) with s the log2-domain score of the raw product v, packed
// to 16 bits in pk; returns their sum. A masked key arrives as v = -inf and
// gets p = 0 in every mode. MODE 0: no softcap, s = v * sl. MODE 1:
// softcap by the Maclaurin series of tanh truncated after the ninth power,
// s = v * (a1 + v^2 (a3 + v^2 (a5 + v^2 (a7 + v^2 a9)))); for
// |v * cap_in| <= 1/4 the series alternates with decreasing terms, so the
// truncation error is below its next term, 1382/155925 * 4^-11 < 3e-9
// (relative to softcap), under the rounding of the evaluation; v = -inf
// gives q = +inf (a9 > 0) and s = -inf. MODE 2: softcap through tanh_ex2
// (any score), with v = -inf mapped to s = -inf explicitly.
struct ExpArgs {
  float sl, mu, cap_in, cap_out, a1, a3, a5, a7, a9;
};
template <typename T, int MODE>
__device__ __forceinline__ float exp_chunk(const uint32_t (&r)[32], uint32_t (&pk)[16],
                                           const ExpArgs& A) {
  float lsum = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float p[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = __uint_as_float(r[2 * e + h]);
      float x;
      if (MODE == 0) {
        x = fmaf(v, A.sl, -A.mu);
      } else if (MODE == 1) {
        const float v2 = v * v;
        const float q = fmaf(fmaf(fmaf(fmaf(A.a9, v2, A.a7), v2, A.a5), v2, A.a3), v2, A.a1);
        x = fmaf(v, q, -A.mu);
      } else {
        x = fmaf(A.cap_out, tanh_ex2(v * A.cap_in), -A.mu);
        if (v == -INFINITY) x = -INFINITY;
      }
      p[h] = ex2(x);
    }
    lsum += p[0] + p[1];
    pk[e] = pack2<T>(p[0], p[1]);
  }
  return lsum;
}

// ---------------------------------------------------------------------------
// Decode work plan. Each valid decode sequence has n_b key tiles; it is cut
// into c_b(T) = ceil(n_b / T) splits of at most T tiles, T being the smallest
// split length for which all splits fit in the grid's units. Invalid
// sequences (q_len != 1, out-of-range position) get one unit, which only
// reports the error. Every CTA derives the same plan from past_seqlens with
// one warp (lane-strided sequences, shuffle reductions), so no host round
// trip or separate planning launch is needed.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t decode_tiles(const Params& P, int b, int n_tile) {
  // (the three loads are issued together: b is a valid sequence index)
  const int32_t q0 = P.cumseq[b], q1 = P.cumseq[b + 1];
  const int64_t pos = P.past[b];
  if (q1 - q0 != 1 || q0 < 0 || q0 >= P.num_tokens) return 0;
  if (pos < 0 || pos >= (int64_t)P.max_blocks * P.bs || (P.rd > 0 && pos >= P.cos_rows)) return 0;
  const int64_t lo = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
  return pos / n_tile - lo / n_tile + 1;
}

// Splits of a sequence with `tiles` key tiles at split length T (a
// sequence without tiles still takes one unit, which reports its error).
__device__ __forceinline__ int ceil_div32(int a, int b) {
  return (int)(((uint32_t)a + (uint32_t)b - 1u) / (uint32_t)b);
}
__device__ __forceinline__ int splits32(int tiles, int T) {
  return tiles <= 0 ? 1 : ceil_div32(tiles, T);
}

// Tile count of sequence i >= 32 (lane-strided beyond the first 32): from
// the shared-memory scratch the plan filled, or reloaded past its capacity.
template <int N>
__device__ __forceinline__ int far_tiles(const Params& P, int i, int seq_begin, const int* more,
                                         int cap) {
  return i - 32 < cap ? more[i - 32] : (int)decode_tiles(P, seq_begin + i, N);
}

// Sum over the warp of the splits of every sequence at split length T.
// Lane l holds sequences l, l+32, ...; `own` is the tile count of sequence
// l. Batches of up to 32 sequences are summed from registers alone.
template <int N>
__device__ __forceinline__ int warp_splits(const Params& P, int own, int T, int nseq,
                                           int seq_begin, const int* more, int cap) {
  const int lane = threadIdx.x & 31;
  int cnt = lane < nseq ? splits32(own, T) : 0;
  if (nseq > 32) {
    for (int i = lane + 32; i < nseq; i += 32)
      cnt += splits32(far_tiles<N>(P, i, seq_begin, more, cap), T);
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt;
}

// Run by one full warp; returns the unit's plan in every lane. Units are
// numbered lane by lane (lane 0's sequences first, each sequence's splits
// consecutive), the same in every CTA. The code runs once per CTA, so it is
// kept short: its instructions are fetched cold on every launch. `more` is
// shared-memory scratch for the tile counts of sequences 32.. (up to `cap`
// of them), which later passes read instead of reloading them.
template <int N>
__device__ Work decode_plan_warp(const Params& P, int unit, int* more, int cap) {
  const int lane = threadIdx.x & 31;
  const int seq_begin = P.seq_begin, nseq = P.seq_end - seq_begin, units = P.units;
  const int own = lane < nseq ? (int)decode_tiles(P, seq_begin + lane, N) : 0;
  // Smallest T with sum_b ceil(n_b / T) <= units. Since n_b / T <=
  // ceil(n_b / T) <= n_b / T + 1, it lies in [ceil(total / units),
  // ceil(total / (units - nseq))] (total = sum_b n_b; units >= nseq), and
  // T = the longest sequence (one split each) always fits, so a bisection
  // over [ceil(total / units), min(that bound, longest)] takes a few steps.
  int total = lane < nseq ? max(own, 0) : 0, longest = total;
  for (int i = lane + 32; i < nseq; i += 32) {
    const int t = (int)decode_tiles(P, seq_begin + i, N);
    if (i - 32 < cap) more[i - 32] = t;
    total += max(t, 0);
    longest = max(longest, t);
  }
  __syncwarp();
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    total += __shfl_xor_sync(0xffffffffu, total, o);
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
  }
  int lo = max(1, ceil_div32(total, units));
  int hi = units > nseq ? min(ceil_div32(total, units - nseq), longest) : longest;
  hi = max(lo, hi);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (warp_splits<N>(P, own, mid, nseq, seq_begin, more, cap) <= units) hi = mid; else lo = mid + 1;
  }
  const int T = lo;
  // this lane's units, then an exclusive scan over the lanes
  int mine = 0;
  for (int i = lane; i < nseq; i += 32)
    mine += splits32(i == lane ? own : far_tiles<N>(P, i, seq_begin, more, cap), T);
  int incl = mine;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - mine;
  Work w;
  w.status = 1;
  w.b = -1;
  w.decode = 1;
  w.t_begin = w.t_end = 0;
  int hit = 0, tiles_hit = 0;
  for (int i = lane; i < nseq; i += 32) {
    const int tiles = i == lane ? own : far_tiles<N>(P, i, seq_begin, more, cap);
    const int c = splits32(tiles, T);
    if (unit >= run && unit < run + c) {
      hit = 1;
      tiles_hit = tiles;
      w.b = seq_begin + i;
      w.split = unit - run;
      w.splits = c;
      w.first = run;
    }
    run += c;
  }
  const unsigned who = __ballot_sync(0xffffffffu, hit);
  if (who == 0) return w;  // idle unit
  const int src = __ffs(who) - 1;
  w.b = __shfl_sync(0xffffffffu, w.b, src);
  w.split = __shfl_sync(0xffffffffu, w.split, src);
  w.splits = __shfl_sync(0xffffffffu, w.splits, src);
  w.first = __shfl_sync(0xffffffffu, w.first, src);
  tiles_hit = __shfl_sync(0xffffffffu, tiles_hit, src);
  if (tiles_hit > 0) {
    const int64_t pos = P.past[w.b];
    const int64_t lo_key = P.window >= 0 ? max((int64_t)0, pos - P.window) : 0;
    w.t_begin = lo_key / N + (int64_t)w.split * T;
    w.t_end = min(pos / N + 1, w.t_begin + T);
  }
  w.status = 0;
  return w;
}

// Merges the key splits of each decode sequence (plan written by the
// attention kernel): M = max_s m_s, out = sum_s 2^(m_s-M) O_s / sum_s
// 2^(m_s-M) l_s; zero when a split read an invalid block.
// Prefill work unit `unit` with up to `tpc` consecutive tokens of one
// sequence per unit (the query tile then holds tpc tokens' heads, which share
// every key tile). Sequences of [seq_begin, seq_end) get ceil(q_b / tpc)
// units each, numbered in sequence order; CTA `unit` takes number
// total - 1 - unit, so the units with the most keys (the last tokens) start
// first and short ones fill in behind them. Run by one full warp.
__device__ __forceinline__ Work prefill_group_warp(const Params& P, int unit, int tpc) {
  const int lane = threadIdx.x & 31;
  const int seq_begin = P.pf_begin, nseq = P.pf_end - seq_begin;
  Work w;
  w.status = 1;
  w.splits = 1;
  w.ntok = 0;
  w.decode = 0;
  int total = 0;
  for (int i = lane; i < nseq; i += 32) {
    const int q = P.cumseq[seq_begin + i + 1] - P.cumseq[seq_begin + i];
    total += q > 0 ? ceil_div32(q, tpc) : 0;
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  if (unit >= total) return w;  // idle unit
  unit = total - 1 - unit;
  int run = 0;
  for (int base = 0; base < nseq; base += 32) {
    const int i = base + lane;
    int cnt = 0, q0 = 0, q = 0;
    if (i < nseq) {
      q0 = P.cumseq[seq_begin + i];
      q = P.cumseq[seq_begin + i + 1] - q0;
      cnt = q > 0 ? ceil_div32(q, tpc) : 0;
    }
    int incl = cnt;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int start = run + incl - cnt;
    const unsigned who = __ballot_sync(0xffffffffu, cnt > 0 && unit >= start && unit < start + cnt);
    if (who) {
      const int src = __ffs(who) - 1;
      const int grp = __shfl_sync(0xffffffffu, unit - start, src);
      const int first = __shfl_sync(0xffffffffu, q0, src);
      const int len = __shfl_sync(0xffffffffu, q, src);
      w.b = seq_begin + base + src;
      w.t = first + (int64_t)grp * tpc;
      w.ntok = min(tpc, len - grp * tpc);
      w.past = P.past[w.b];
      w.pos = w.past + grp * tpc;
      w.status = 0;
      return w;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return w;  // idle unit
}

// Log-sum-exp merge of a decode sequence's key splits:
//   O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s
// (log2-domain maxima, unnormalised partial outputs). A NaN partial maximum
// marks a split that read an invalid block: the row becomes zeros, as does a
// row that saw no key (sum = 0). Thread = CPT consecutive accumulator
// channels of one head (groups * vg channels, of which the first vhs are
// stored); each thread issues the loads of a round of splits together and
// folds them with a running maximum, so the merge costs the plan load plus
// one round trip per round of splits. VGF, GF > 0 fix vg and groups at
// compile time (the 192/128 and 576/512 shapes), 0 takes them from Params.
template <typename T, int CPT, int VGF, int GF>
__global__ void __launch_bounds__(256) tc_combine_kernel(const __grid_constant__ Params P) {
  grid_dep_wait();  // the attention kernel's partials are complete and visible
  constexpr int kRound = CPT >= 16 ? 4 : 8;  // splits whose loads are in flight together
  static_assert(CPT % 4 == 0, "combine shape");
  const int vg = VGF ? VGF : P.vg, groups = GF ? GF : P.groups;
  const int tph = groups * vg / CPT;         // threads per head
  const int hpb = 256 / tph;                 // heads per CTA
  const int hl = (int)threadIdx.x / tph;
  if (hl >= hpb) return;
  const int x = blockIdx.x;
  const int h = blockIdx.y * hpb + hl;
  const int c0 = ((int)threadIdx.x % tph) * CPT;  // channel in [0, groups*vg)
  const int g = c0 / vg, cc = c0 - g * vg;
  const int2 plan = P.ws_plan[x];
  const int32_t q0 = P.cumseq[P.seq_begin + x];
  const int S = plan.y;
  if (S > 1 && h < P.H && c0 < P.vhs) {  // (one split: the attention kernel wrote the output)
    float M = -INFINITY, L = 0.f, o[CPT];
#pragma unroll
    for (int e = 0; e < CPT; ++e) o[e] = 0.f;
    bool bad = false;
    for (int s0 = 0; s0 < S; s0 += kRound) {
      float2 ml[kRound];
      float4 ov[kRound][CPT / 4];
#pragma unroll
      for (int i = 0; i < kRound; ++i) {
        if (s0 + i < S) {
          const int64_t slot = ((int64_t)(plan.x + s0 + i) * groups + g) * kRows + h;
          ml[i] = reinterpret_cast<const float2*>(P.ws_ml)[slot];
          const float4* src = reinterpret_cast<const float4*>(P.ws_o + slot * vg + cc);
#pragma unroll
          for (int q = 0; q < CPT / 4; ++q) ov[i][q] = src[q];
        }
      }
#pragma unroll
      for (int i = 0; i < kRound; ++i) {
        if (s0 + i < S) {
          const float m = ml[i].x, l = ml[i].y;
          bad |= isnan(m);
          if (l > 0.f && !isnan(m)) {
            if (m > M) {  // new running maximum: rescale what is folded so far
              const float f = ex2(M - m);
              L *= f;
#pragma unroll
              for (int e = 0; e < CPT; ++e) o[e] *= f;
              M = m;
            }
            const float w = ex2(m - M);
            L += w * l;
#pragma unroll
            for (int q = 0; q < CPT / 4; ++q) {
              o[4 * q] += w * ov[i][q].x; o[4 * q + 1] += w * ov[i][q].y;
              o[4 * q + 2] += w * ov[i][q].z; o[4 * q + 3] += w * ov[i][q].w;
            }
          }
        }
      }
    }
    const float inv = (L > 0.f && !bad) ? 1.f / L : 0.f;
    T* dst = reinterpret_cast<T*>(P.out) + ((int64_t)q0 * P.H + h) * P.vhs + c0;
    if (c0 + CPT <= P.vhs && P.vhs % 8 == 0) {  // whole, aligned vectors
      uint32_t pk[CPT / 2];
#pragma unroll
      for (int e = 0; e < CPT / 2; ++e) pk[e] = pack2<T>(o[2 * e] * inv, o[2 * e + 1] * inv);
      if (CPT == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
      } else {
#pragma unroll
        for (int q = 0; q < CPT / 8; ++q)
          reinterpret_cast<uint4*>(dst)[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                                                        pk[4 * q + 3]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < CPT; ++e)
        if (c0 + e < P.vhs) dst[e] = Half<T>::from_f32(o[e] * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// Host-side helpers
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static:
// its initialisation is thread-safe).
inline EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// A read-phase configuration chosen on the host: value channels per CTA
// (vg) and CTAs per head group (groups), the key tile (n), stage count,
// query rows kept (qr), S/P buffers (nb); pair = the 576/512 CTA-pair kernel.
struct Shape {
  int hs, vg, groups, n, stages, qr, nb;
  bool pair;
  int stages8 = 0;  // FP8 cache: E4M3 stages (0: the cache is in the query dtype)
  bool pos = false;  // P written over its tile's S columns (no TMEM of its own)
};

// Decode grid: one wave of CTAs (one per SM), at least one unit per sequence.
inline int64_t decode_units(const Geometry& g, const Shape& s, int64_t nseq) {
  const int64_t wave = g.num_sms / s.groups;
  return nseq > wave ? nseq : wave;
}

inline size_t decode_ws_bytes(const Shape& s, int64_t units, int64_t nseq) {
  const size_t per = (size_t)units * s.groups * kRows;
  const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
  const size_t ml = ((per * 2 * sizeof(float)) + 255) & ~(size_t)255;
  return o + ml + (size_t)nseq * sizeof(int2);
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) (void)cudaGetLastError();  // not left behind for a later call
  return e;
}

// Split combine of a decode call over nq sequences, launched after the
// attention kernel with programmatic dependent launch.
template <typename T>
cudaError_t launch_combine(const Params& P, int H, int64_t nq, cudaStream_t st) {
  const int cpt = P.groups * P.vg >= 512 ? 16 : 4;
  const int hpb = 256 / (P.groups * P.vg / cpt);
  const dim3 grid((unsigned)nq, (unsigned)((H + hpb - 1) / hpb));
  if (P.vg == 128 && P.groups == 1)
    return launch_pdl(tc_combine_kernel<T, 4, 128, 1>, grid, dim3(256), 0, st, P);
  if (P.vg == 256 && P.groups == 2)
    return launch_pdl(tc_combine_kernel<T, 16, 256, 2>, grid, dim3(256), 0, st, P);
  return cpt == 16 ? launch_pdl(tc_combine_kernel<T, 16, 0, 0>, grid, dim3(256), 0, st, P)
                   : launch_pdl(tc_combine_kernel<T, 4, 0, 0>, grid, dim3(256), 0, st, P);
}

// CTA-pair kernel for the 576/512 geometry (pa_tc_pair.cu).
template <typename T>
cudaError_t launch_pair(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq);

}  // namespace tc
}  // namespace pa
