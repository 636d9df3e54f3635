// Internal interface between the C-ABI entry points and the kernel
// launchers. Not installed; the public interface is include/pa_latent.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "pa_latent.h"

namespace pa {

// Validated operator geometry with defaults resolved.
struct Geometry {
  int dtype;        // pa_dtype
  int H;            // query heads
  int hs;           // latent width
  int vhs;          // value width (v_head_size, 0 resolved to hs)
  int ro, rd;       // rotary offset / dim
  int interleaved;  // 0 / 1
  int cos_rows;
  int bs;           // block size
  int num_blocks;
  int max_blocks;   // block_table columns
  float scale;      // resolved (never 0)
  float softcap;    // <= 0: off
  int window;       // < 0: off
  int fp8;          // key_cache holds E4M3 codes (PA_CACHE_FP8_E4M3)
  float k_scale;    // FP8 cache: value = code * k_scale (1 otherwise)
  int kvh;          // kv heads (1 in the LATENT layout)
  float rms_eps;    // SEPARATE layout: RMSNorm epsilon
  int flags;
  int num_sms;      // SM count of the current device
  int device;       // current device ordinal
};

// Paged streaming probe (pa_probe.cu): shared memory per CTA, and the launch.
extern const size_t kMaxProbeSmem;
size_t gather_probe_smem(const Geometry& g, int tile_keys, int stages, int num_seqs);
cudaError_t launch_gather_probe(const Geometry& g, const void* key_cache, const int32_t* past,
                                const int32_t* block_table, int num_seqs, int tile_keys,
                                int stages, int ctas_per_sm, int32_t* err_flags,
                                cudaStream_t stream);

// kMixed: one launch over a batch whose first sequences are decodes (one
// new token each) and the rest prefills.
enum class Phase { kDecode = 0, kPrefill = 1, kMixed = 2 };

// Runs an idempotent per-device set-up action (a kernel attribute) once per
// device ordinal < 64. Safe when several host threads make their first call
// at the same time: the flags are atomic, and two threads that both see a
// flag unset both run the action, which is harmless.
template <typename F>
cudaError_t once_per_device(std::atomic<bool> (&done)[64], int device, F&& action) {
  if (device < 0 || device >= 64) return action();
  if (done[device].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = action();
  if (e == cudaSuccess) done[device].store(true, std::memory_order_release);
  return e;
}

// Records msg as the calling thread's pa_latent_last_error() text and
// returns s.
pa_status record_error(pa_status s, const char* msg);

// Names the step of a launch that failed (a static string); the entry
// point adds it to the error text of a failed launch. Cleared per call.
void set_launch_step(const char* step);

// ---- write phase (pa_write.cu)
cudaError_t launch_write(const Geometry& g, const void* key, int64_t num_tokens,
                         const void* cos_cache, const void* sin_cache,
                         const int32_t* slot_mapping, const int32_t* cumseq, const int32_t* past,
                         int32_t num_seqs, void* key_cache, int32_t* err_flags,
                         cudaStream_t stream);

// Arguments of one read-phase call.
struct ReadArgs {
  const void* query;
  int64_t num_tokens;
  const void* key_cache;
  const void* value_cache;  // SEPARATE layout only (null otherwise)
  const void* head_sink;    // SEPARATE layout, optional
  const void* q_norm;       // SEPARATE layout, optional
  const void* cos_cache;
  const void* sin_cache;
  const int32_t* cumseq;
  const int32_t* past;
  const int32_t* block_table;
  int32_t num_seqs, seq_begin, seq_end;
  int32_t pf_begin, pf_end;  // kMixed: the prefill sequences (decode: [seq_begin, seq_end))
  void* workspace;
  size_t workspace_bytes;
  void* out;
  int32_t* err_flags;
  cudaStream_t stream;
};

// ---- portable CUDA-core attention (pa_portable.cu)
size_t portable_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs,
                                int64_t num_tokens);
// Workspace a call over nq queries (decode: sequences, prefill: tokens) needs.
size_t portable_call_workspace(const Geometry& g, Phase ph, int64_t nq);
cudaError_t launch_portable(const Geometry& g, Phase ph, const ReadArgs& a);

// ---- tcgen05 / TMA attention (pa_tc.cu)
bool tc_supported(const Geometry& g, Phase ph);
size_t tc_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs, int64_t num_tokens);
// Workspace one read call over sequences [seq_begin, seq_end) needs.
size_t tc_call_workspace(const Geometry& g, Phase ph, int32_t seq_begin, int32_t seq_end);
cudaError_t launch_tc(const Geometry& g, Phase ph, const ReadArgs& a);

// ---- SEPARATE layout (pa_gqa.cu)
struct SeparateWriteArgs {
  const void* key;
  const void* value;
  int64_t num_tokens;
  const void* cos_cache;
  const void* sin_cache;
  const void* k_norm;  // optional
  const int32_t* slot_mapping;
  const int32_t* cumseq;
  const int32_t* past;
  int32_t num_seqs;
  void* key_cache;
  void* value_cache;
  int32_t* err_flags;
  cudaStream_t stream;
};
cudaError_t launch_separate_write(const Geometry& g, const SeparateWriteArgs& a);
bool separate_supported(const Geometry& g, Phase ph);
size_t separate_call_workspace(const Geometry& g, Phase ph, int32_t seq_begin, int32_t seq_end);
cudaError_t launch_separate_read(const Geometry& g, Phase ph, const ReadArgs& a);

// ---- shared by the entry points (pa_api.cu)
// Workspace bytes a decode call over sequences [seq_begin, seq_end) of these
// parameters needs on the current device, or an error status for invalid
// parameters. Host-only.
pa_status decode_call_workspace(const pa_latent_params* p, int32_t seq_begin, int32_t seq_end,
                                size_t* need);

}  // namespace pa
