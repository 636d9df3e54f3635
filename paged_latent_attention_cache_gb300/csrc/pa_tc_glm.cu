// The single-CTA tensor-core kernel's 192/128 shapes (GLM-style latent 192,
// value 128), compiled with the latent width, value width and stage count
// fixed: decode with a 64-row query tile and four 128-key stages, prefill at
// two CTAs per SM (64-key tiles, two stages, two S buffers with P written
// over its S), the 128-row
// query tile with three 128-key stages, and FP8-cache decode (fp16 key
// stages fed by converter warps from E4M3 stages).
#include "pa_tc_attn.cuh"

namespace pa {
namespace tc {

template <typename T>
cudaError_t launch_fixed(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                         const Shape& s) {
  if (s.stages8)  // FP8-cache decode
    return launch_shape<T, 128, 64, 2, 192, 128, kFp8Stages16, true>(g, ph, a, P, nq, s);
  if (s.n == 128 && s.qr == 64) return launch_shape<T, 128, 64, 2, 192, 128, 4>(g, ph, a, P, nq, s);
  if (s.pos) return launch_shape<T, 64, 128, 2, 192, 128, 2, false, true>(g, ph, a, P, nq, s);
  return launch_shape<T, 128, 128, 2, 192, 128, 3>(g, ph, a, P, nq, s);
}

template cudaError_t launch_fixed<__nv_bfloat16>(const Geometry&, Phase, const ReadArgs&, Params&,
                                                 int64_t, const Shape&);
template cudaError_t launch_fixed<__half>(const Geometry&, Phase, const ReadArgs&, Params&, int64_t,
                                          const Shape&);

}  // namespace tc
}  // namespace pa
