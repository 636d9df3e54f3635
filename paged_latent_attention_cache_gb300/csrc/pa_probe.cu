// Paged streaming probe: the cache traffic of the read phase alone.
//
// Every visible latent row of a decode batch (positions 0..past[b] of each
// sequence b) is gathered through the block table by the 2-D TMA boxes the
// tensor-core kernels use (64 channels x box_rows rows, 128-byte swizzle)
// into a ring of shared-memory stages, and each stage is refilled as soon as
// its previous tile has landed: there is no arithmetic and no consumer, so
// the achieved rate is the ceiling of paged TMA streaming for the chosen
// tile size, stage count and CTAs per SM. Tiles are dealt round-robin over
// the CTAs of one wave, so every SM streams the same share.
#include "pa_tc_common.cuh"

namespace pa {
using namespace tc;
namespace {

constexpr int kMaxProbeSeqs = 4096;  // prefix sums staged in shared memory

struct ProbeArgs {
  const int32_t* past;
  const int32_t* block_table;
  int32_t* err_flags;
  int64_t num_slots;
  int num_seqs, max_blocks, bs, box_rows, tile_keys, slabs, stages, num_blocks;
  uint32_t stage_bytes;
};

__global__ void __launch_bounds__(32) gather_probe_kernel(const __grid_constant__ CUtensorMap kmap,
                                                          const __grid_constant__ ProbeArgs A) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)A.stages * A.stage_bytes);
  int* first_tile = reinterpret_cast<int*>(full + A.stages);  // [num_seqs + 1]
  const int lane = threadIdx.x;

  // first_tile[b] = tiles of sequences < b (tiles = ceil(context / tile_keys))
  int run = 0;
  for (int b0 = 0; b0 < A.num_seqs; b0 += 32) {
    const int b = b0 + lane;
    const int ctx = b < A.num_seqs ? max(A.past[b] + 1, 0) : 0;
    int v = (ctx + A.tile_keys - 1) / A.tile_keys;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (b < A.num_seqs) first_tile[b + 1] = run + v;
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) {
    first_tile[0] = 0;
    abort_flag = 0;
    for (int s = 0; s < A.stages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (lane != 0) return;
  const int total = first_tile[A.num_seqs];
  const int sub = A.tile_keys / A.box_rows;
  const uint32_t slab_bytes = (uint32_t)A.tile_keys * 128;
  int k = 0;
  for (int t = blockIdx.x; t < total; t += gridDim.x, ++k) {
    const int s = k % A.stages;
    if (k >= A.stages &&
        !wait_bar(smem_u32(&full[s]), ((k / A.stages) - 1) & 1, &abort_flag, A.err_flags))
      break;
    // sequence of tile t: the last b with first_tile[b] <= t
    int lo = 0, hi = A.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (first_tile[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t key0 = (int64_t)(t - first_tile[b]) * A.tile_keys;
    const int64_t last = A.past[b];
    mbar_expect_tx(smem_u32(&full[s]), A.stage_bytes);
    const uint32_t dst = smem_u32(smem + (size_t)s * A.stage_bytes);
    for (int q = 0; q < sub; ++q) {
      const int64_t key = key0 + (int64_t)q * A.box_rows;
      int y = (int)A.num_slots;  // past the context: the box is filled with zeros
      if (key <= last && key / A.bs >= A.max_blocks) {
        raise_flag(A.err_flags, PA_DEVERR_CONTEXT);  // past the block table's row
      } else if (key <= last) {
        const int phys = A.block_table[(int64_t)b * A.max_blocks + key / A.bs];
        if (phys >= 0 && phys < A.num_blocks) {
          y = (int)((int64_t)phys * A.bs + key % A.bs);
        } else {
          raise_flag(A.err_flags, PA_DEVERR_BLOCK);
        }
      }
      for (int j = 0; j < A.slabs; ++j)
        tma_load_2d(dst + j * slab_bytes + q * A.box_rows * 128, &kmap, j * 64, y,
                    smem_u32(&full[s]));
    }
  }
  // every copy still in flight has landed before the CTA exits
  for (int s = 0; s < A.stages && s < k; ++s) {
    const int uses = (k - s + A.stages - 1) / A.stages;
    drain_wait(smem_u32(&full[s]), (uses - 1) & 1, A.err_flags);
  }
}

}  // namespace

// Dynamic shared memory a probe CTA may use: the 227 KB per-block limit less
// room for the kernel's static shared memory.
const size_t kMaxProbeSmem = 226 * 1024;

size_t gather_probe_smem(const Geometry& g, int tile_keys, int stages, int num_seqs) {
  const size_t stage_bytes = (size_t)((g.hs + 63) / 64) * tile_keys * 128;
  return stages * stage_bytes + stages * sizeof(uint64_t) + (num_seqs + 1) * sizeof(int) + 1024;
}

cudaError_t launch_gather_probe(const Geometry& g, const void* key_cache, const int32_t* past,
                                const int32_t* block_table, int num_seqs, int tile_keys,
                                int stages, int ctas_per_sm, int32_t* err_flags,
                                cudaStream_t stream) {
  if (num_seqs > kMaxProbeSeqs) return cudaErrorInvalidValue;
  const size_t smem = gather_probe_smem(g, tile_keys, stages, num_seqs);
  static std::atomic<bool> configured[64];
  cudaError_t e = once_per_device(configured, g.device, [&] {
    return cudaFuncSetAttribute(gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kMaxProbeSmem);
  });
  if (e != cudaSuccess) return e;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = g.dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  ProbeArgs A;
  A.past = past;
  A.block_table = block_table;
  A.err_flags = err_flags;
  A.num_slots = (int64_t)g.num_blocks * g.bs;
  A.num_seqs = num_seqs;
  A.max_blocks = g.max_blocks;
  A.bs = g.bs;
  A.box_rows = g.bs < tile_keys ? g.bs : tile_keys;
  A.tile_keys = tile_keys;
  A.slabs = (g.hs + 63) / 64;
  A.stages = stages;
  A.num_blocks = g.num_blocks;
  A.stage_bytes = (uint32_t)(A.slabs * tile_keys * 128);
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)g.hs, (cuuint64_t)A.num_slots};
  const cuuint64_t strides[1] = {(cuuint64_t)g.hs * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)A.box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, dt, 2, const_cast<void*>(key_cache), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  gather_probe_kernel<<<(unsigned)(g.num_sms * ctas_per_sm), 32, smem, stream>>>(map, A);
  return cudaGetLastError();
}

}  // namespace pa
