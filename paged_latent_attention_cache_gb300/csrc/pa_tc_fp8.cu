// The single-CTA tensor-core kernel's FP8-cache shapes: E4M3 key tiles
// copied by TMA, converted to fp16 in shared memory by four converter warps,
// and multiplied with fp16 operands (the latent width and stage counts come
// from the launch's Params).
#include "pa_tc_attn.cuh"

namespace pa {
namespace tc {

template <typename T>
cudaError_t launch_fp8(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                       const Shape& s) {
  if (s.n == 128 && s.qr == 64) return launch_shape<T, 128, 64, 2, 0, 0, 0, true>(g, ph, a, P, nq, s);
  if (s.n == 128) return launch_shape<T, 128, 128, 2, 0, 0, 0, true>(g, ph, a, P, nq, s);
  if (s.qr == 64) return launch_shape<T, 64, 64, 2, 0, 0, 0, true>(g, ph, a, P, nq, s);
  return launch_shape<T, 64, 128, 2, 0, 0, 0, true>(g, ph, a, P, nq, s);
}

template cudaError_t launch_fp8<__nv_bfloat16>(const Geometry&, Phase, const ReadArgs&, Params&,
                                               int64_t, const Shape&);
template cudaError_t launch_fp8<__half>(const Geometry&, Phase, const ReadArgs&, Params&, int64_t,
                                        const Shape&);

}  // namespace tc
}  // namespace pa
