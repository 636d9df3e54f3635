// Helpers of the CTA-pair kernel (pa_tc_pair.cu):
// cluster rank and barrier, distributed-shared-memory addressing, remote
// stores that complete on the peer's mbarrier, and bounded cluster-scope waits.
#pragma once
#include "pa_tc_common.cuh"

namespace pa {
namespace tc {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(peer));
  return r;
}
// Relaxed remote arrive: used where the ordering it announces (loads that
// have already returned their values) needs no release fence, so the thread
// does not wait for its own in-flight remote stores.
__device__ __forceinline__ void arrive_peer_relaxed(uint32_t raddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr)
               : "memory");
}
// Shared-memory descriptor for a K-major operand with 64-byte rows in the
// 64-byte swizzle layout (8-row atoms of 512 bytes): layout type 4.
__device__ __forceinline__ uint64_t sdesc64(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}
// Remote 16-byte store of four 32-bit words (bit patterns, no conversion)
// whose arrival completes tx bytes on the peer's mbarrier.
__device__ __forceinline__ void st_async_b32x4(uint32_t raddr, uint32_t a, uint32_t b,
                                               uint32_t c, uint32_t d, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(raddr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (for arrivals made by the peer).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity,
                                                 volatile int* abort, int32_t* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort = 1;
  raise_flag(err, PA_DEVERR_TIMEOUT);
  return false;
}

}  // namespace tc
}  // namespace pa
