// Allocation-free decode entry point.
//
// pa_latent_decode needs a caller-provided workspace for the split-KV
// partials. Some callers cannot provide one: an execution provider whose
// host framework owns every device allocation, a serving loop that must not
// touch the allocator once it is running, or plain C code with no device
// allocator of its own. For them pa_latent_decode_noalloc runs the same
// decode with the library's own scratch: a fixed-size array in device global
// memory, created when the library is loaded on a GPU and held until the
// process exits. Nothing is allocated per call.
#include <stdio.h>

#include <mutex>

#include "pa_internal.h"

namespace {

// Scratch for the split-KV partials and the per-sequence plan of one decode
// call: 32 MiB. A tensor-core decode call needs about 264 KB per sequence
// with the 576/512 geometry (two SMs x 128 rows x (256 + 2) f32) and 67 KB
// with 192/128, for at least as many sequences as the grid's work units (one
// per SM, or per SM pair), so calls of up to 127 sequences (576/512) or 504
// sequences (192/128) fit; larger calls are rejected.
constexpr size_t kScratchBytes = 32ull << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_scratch on the current device. In host code the
// symbol is only a stand-in; the real address comes from the runtime, once
// per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

pa_status pa_latent_decode_noalloc(const pa_latent_params* p, const void* query,
                                   int64_t num_tokens, const void* key_cache,
                                   const void* cos_cache, const void* sin_cache,
                                   const int32_t* cumseq, const int32_t* past,
                                   const int32_t* block_table, int32_t num_seqs,
                                   int32_t seq_begin, int32_t seq_end, void* out,
                                   int32_t* err_flags, void* stream) {
  size_t need = 0;
  const pa_status s = pa::decode_call_workspace(p, seq_begin, seq_end, &need);
  if (s != PA_OK) return s;
  if (need > kScratchBytes) {
    char msg[192];
    snprintf(msg, sizeof msg,
             "this decode call needs %zu bytes of scratch; the library's static scratch holds "
             "%zu bytes (use pa_latent_decode with a caller workspace)",
             need, kScratchBytes);
    return pa::record_error(PA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    char msg[192];
    snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch: %s",
             cudaGetErrorString(e));
    return pa::record_error(PA_ERR_CUDA, msg);
  }
  return pa_latent_decode(p, query, num_tokens, key_cache, cos_cache, sin_cache, cumseq, past,
                          block_table, num_seqs, seq_begin, seq_end, scratch, kScratchBytes, out,
                          err_flags, stream);
}

}  // extern "C"
