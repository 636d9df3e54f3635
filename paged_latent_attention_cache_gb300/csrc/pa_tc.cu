// Tensor-core (tcgen05 / TMEM / TMA) read phase. Specialisations are added
// per geometry; geometries without one run the portable kernels.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

bool tc_supported(const Geometry& g, Phase ph) {
  (void)g;
  (void)ph;
  return false;
}

size_t tc_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs, int64_t num_tokens) {
  (void)g; (void)ph; (void)num_seqs; (void)num_tokens;
  return 0;
}

size_t tc_call_workspace(const Geometry& g, Phase ph, const ReadArgs& a) {
  (void)g; (void)ph; (void)a;
  return 0;
}

cudaError_t launch_tc(const Geometry& g, Phase ph, const ReadArgs& a) {
  (void)g; (void)ph; (void)a;
  return cudaErrorNotSupported;
}

}  // namespace pa
