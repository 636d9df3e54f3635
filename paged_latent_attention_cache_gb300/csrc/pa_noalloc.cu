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
// call. 32 MiB covers the decode calls of every geometry with a tensor-core
// kernel up to a few hundred sequences (a 576/512 batch of 64 sequences uses
// about 20 MiB); larger calls are rejected.
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
  pa_status s = pa_latent_validate(p);
  if (s != PA_OK) return s;
  const size_t need = pa_latent_workspace_size(p, num_seqs, num_tokens);
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
