// Tensor-core read phase: kernel shape selection and launch (host side).
// The single-CTA kernel is in pa_tc_attn.cuh (instantiated here for any
// latent width up to 256, and in pa_tc_glm.cu for the 192/128 shapes with
// their geometry fixed at compile time); the 576/512 CTA-pair kernel is in
// pa_tc_pair.cu.
#include "pa_tc_attn.cuh"

namespace pa {
namespace tc {

bool pick(const Geometry& g, Phase ph, Shape* s) {
  if (g.H > kRows) return false;
  // a mixed batch runs in one grid on the single-CTA kernel, in its prefill
  // shape (the decode splits then use that shape too)
  if (ph == Phase::kMixed) {
    if (g.hs == 576 && g.vhs == 512) return false;
    ph = Phase::kPrefill;
  }
  if (g.hs == 576 && g.vhs == 512) {
    // CTA-pair kernel (pa_tc_pair.cu): each CTA rotates the query channels it
    // holds, so the rotary channels must lie in one CTA's range. It reads a
    // cache in the query dtype, or (FP8) two fp16 stages and two E4M3 stages.
    if (!(g.rd == 0 || g.ro >= 320 || g.ro + g.rd <= 256)) return false;
    *s = Shape{576, 256, 2, 64, g.fp8 ? 2 : 3, 128, 2, true, g.fp8 ? 2 : 0};
    return true;
  }
  // (a latent narrower than one 64-channel TMA box runs on the portable kernels)
  if (g.hs > 256 || g.hs < 64) return false;
  const int vg = 64 * ((g.vhs + 63) / 64);
  if (g.fp8) {
    // FP8 cache: two fp16 key stages (the converted tiles the MMAs read) and
    // as many E4M3 stages as the rest of shared memory holds (they carry
    // the copies in flight from HBM). 128-key tiles where two E4M3 stages
    // fit beside them (not for value widths above 128, for the TMEM budget),
    // else 64-key tiles.
    auto fp8_shape = [&](int n) {
      Shape t{g.hs, vg, 1, n, 2, (ph == Phase::kDecode && g.H <= 64) ? 64 : 128, 2, false};
      const bool glm = g.hs == 192 && vg == 128 && t.qr == 64 && n == 128;
      if (glm) t.stages = kFp8Stages16;
      t.stages8 = (kSmemBudget - 1024 - q_bytes(t) - t.stages * stage_bytes(t)) / stage8_bytes(t);
      if (t.stages8 > 8) t.stages8 = 8;
      if (glm && t.stages8 > kFp8Stages8) t.stages8 = kFp8Stages8;
      return t;
    };
    Shape t = fp8_shape(vg > 128 ? 64 : 128);
    if (t.stages8 < 2 && t.n == 128) t = fp8_shape(64);
    if (t.stages8 < 2 || tmem_cols_used(t) > 512) return false;
    *s = t;
    return true;
  }
  // Prefill with H <= 64 (units of 128 / H tokens, each a short chain of a
  // few key tiles) runs two CTAs per SM where they fit in half an SM: 64-key
  // tiles, two stages and two S buffers, each tile's P written over its own
  // S so that QK^T of the next tile runs during the softmax of this one (97
  // KB of shared memory and 256 TMEM columns at 192/128).
  if (ph == Phase::kPrefill && g.H <= 64) {
    const Shape u{g.hs, vg, 1, 64, 2, 128, 2, false, 0, true};
    if (smem_bytes(u) <= kHalfSmemBudget && tmem_alloc_cols(tmem_cols_used(u)) <= 256) {
      *s = u;
      return true;
    }
  }
  // Otherwise one CTA per SM: 128-key tiles (64 when the value accumulator
  // is wider than 128 channels, for the TMEM budget vg + 2 * 1.5 N <= 512),
  // a 64-row query tile for decode with H <= 64, and as many key stages as
  // shared memory holds (four at 192/128 decode, three with 128 query rows).
  Shape t{g.hs, vg, 1, vg > 128 ? 64 : 128, 0, (ph == Phase::kDecode && g.H <= 64) ? 64 : 128,
          2, false};
  t.stages = (kSmemBudget - 1024 - q_bytes(t)) / stage_bytes(t);
  if (t.stages > 8) t.stages = 8;
  if (t.stages < 2 || tmem_cols_used(t) > 512) return false;
  *s = t;
  return true;
}

// Any other single-CTA shape runs with its geometry taken from Params.
template <typename T>
cudaError_t launch_single(const Geometry& g, Phase ph, const ReadArgs& a, Params& P, int64_t nq,
                          const Shape& s) {
  if (fixed_shape(s)) return launch_fixed<T>(g, ph, a, P, nq, s);
  if (s.stages8) return launch_fp8<T>(g, ph, a, P, nq, s);
  if (s.n == 128 && s.qr == 64) return launch_shape<T, 128, 64, 2, 0, 0, 0>(g, ph, a, P, nq, s);
  if (s.n == 128) return launch_shape<T, 128, 128, 2, 0, 0, 0>(g, ph, a, P, nq, s);
  if (s.pos) return launch_shape<T, 64, 128, 2, 0, 0, 0, false, true>(g, ph, a, P, nq, s);
  if (s.qr == 64) return launch_shape<T, 64, 64, 2, 0, 0, 0>(g, ph, a, P, nq, s);
  return launch_shape<T, 64, 128, 2, 0, 0, 0>(g, ph, a, P, nq, s);
}

}  // namespace tc

bool tc_supported(const Geometry& g, Phase ph) {
  tc::Shape s;
  return tc::pick(g, ph, &s);
}

size_t tc_workspace_bytes(const Geometry& g, Phase ph, int32_t num_seqs, int64_t num_tokens) {
  (void)num_tokens;
  tc::Shape s;
  if (ph == Phase::kPrefill || num_seqs <= 0 || !tc::pick(g, ph, &s)) return 0;
  return tc::decode_ws_bytes(s, tc::decode_units(g, s, num_seqs), num_seqs);
}

size_t tc_call_workspace(const Geometry& g, Phase ph, int32_t seq_begin, int32_t seq_end) {
  tc::Shape s;
  if (ph == Phase::kPrefill || seq_end <= seq_begin || !tc::pick(g, ph, &s)) return 0;
  const int64_t nq = (int64_t)(seq_end - seq_begin);
  return tc::decode_ws_bytes(s, tc::decode_units(g, s, nq), nq);
}

cudaError_t launch_tc(const Geometry& g, Phase ph, const ReadArgs& a) {
  tc::Shape s;
  if (!tc::pick(g, ph, &s)) return cudaErrorNotSupported;
  // prefill units: 128 / H consecutive tokens of one sequence (one token on
  // the CTA pair); at most ceil(T / tpc) + nseq units are needed. A mixed
  // launch has the decode splits of [seq_begin, seq_end) first, then the
  // prefill units of [pf_begin, pf_end).
  const int tpc = (ph != Phase::kDecode && s.groups == 1) ? tc::kRows / g.H : 1;
  const int64_t nseq = (int64_t)(a.seq_end - a.seq_begin);
  const int64_t npf = ph == Phase::kMixed ? (int64_t)(a.pf_end - a.pf_begin) : nseq;
  const int64_t nq = ph == Phase::kDecode ? nseq
                     : tpc > 1 || ph == Phase::kMixed ? (a.num_tokens + tpc - 1) / tpc + npf
                                                      : a.num_tokens;
  if (nq <= 0 || (ph != Phase::kDecode && a.num_tokens <= 0)) return cudaSuccess;
  tc::Params P;
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
  // An FP8 cache's keys are code * k_scale: the kernels multiply the codes,
  // so k_scale joins the score scale (and the softcap factors) and the
  // output scale.
  const float eff = g.scale * g.k_scale;
  P.out_scale = g.k_scale;
  P.scale_log2 = eff * tc::kLog2e;
  P.softcap_on = g.softcap > 0.f ? 1 : 0;
  P.cap_in = g.softcap > 0.f ? eff / g.softcap : 0.f;
  P.cap_out = g.softcap * tc::kLog2e;
  // Series coefficients a_(2i+1) = softcap * log2(e) * t_(2i+1) * (scale /
  // softcap)^(2i+1), t = 1, -1/3, 2/15, -17/315, 62/2835 (the Maclaurin
  // coefficients of tanh); the series is used only when all are normal floats.
  P.cap_poly = 0;
  P.cap_vlim = 0.f;
  for (int i = 0; i < 5; ++i) P.cap_a[i] = 0.f;
  if (g.softcap > 0.f) {
    const double ci = (double)eff / (double)g.softcap;
    const double co = (double)g.softcap * 1.4426950408889634;
    const double t[5] = {1.0, -1.0 / 3.0, 2.0 / 15.0, -17.0 / 315.0, 62.0 / 2835.0};
    bool normal = true;
    double pw = ci;
    for (int i = 0; i < 5; ++i) {
      const double a = co * t[i] * pw;
      normal = normal && std::isfinite(a) && std::fabs(a) >= (double)FLT_MIN &&
               std::fabs(a) <= (double)FLT_MAX;
      P.cap_a[i] = (float)a;
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
  P.tpc = tpc;
  P.own_slots = (g.flags & PA_FLAG_OWN_SLOTS) ? 1 : 0;
  P.mixed = ph == Phase::kMixed ? 1 : 0;
  P.pf_begin = a.pf_begin;
  P.pf_end = a.pf_end;
  P.ws_o = nullptr;
  P.ws_ml = nullptr;
  P.ws_plan = nullptr;
  P.units = 0;
  if (ph != Phase::kPrefill) {
    const int64_t units = tc::decode_units(g, s, nseq);
    P.units = (int)units;
    const size_t per = (size_t)units * s.groups * tc::kRows;
    const size_t o = ((per * s.vg * sizeof(float)) + 255) & ~(size_t)255;
    const size_t ml = ((per * 2 * sizeof(float)) + 255) & ~(size_t)255;
    if (a.workspace == nullptr || a.workspace_bytes < tc::decode_ws_bytes(s, units, nseq)) {
      set_launch_step("decode workspace");
      return cudaErrorInvalidValue;
    }
    char* w = reinterpret_cast<char*>(a.workspace);
    P.ws_o = reinterpret_cast<float*>(w);
    P.ws_ml = reinterpret_cast<float*>(w + o);
    P.ws_plan = reinterpret_cast<int2*>(w + o + ml);
  }
  P.vg = s.vg;
  P.groups = s.groups;
  const bool bf16 = g.dtype == PA_DTYPE_BF16;
  if (s.pair)
    return bf16 ? tc::launch_pair<__nv_bfloat16>(g, ph, a, P, nq)
                : tc::launch_pair<__half>(g, ph, a, P, nq);
  return bf16 ? tc::launch_single<__nv_bfloat16>(g, ph, a, P, nq, s)
              : tc::launch_single<__half>(g, ph, a, P, nq, s);
}

}  // namespace pa

