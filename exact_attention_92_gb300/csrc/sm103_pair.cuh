// CTA-pair primitives for the sm_103a kernels that run two CTAs on
// neighbouring SMs as one (tcgen05.mma.cta_group::2, clusters of 2): the
// pair's rank, addresses in the leader CTA (rank 0), cluster barriers,
// arrivals on and bounded waits for the leader's barriers, tile copies that
// complete on a leader barrier, and the pair MMAs and commits.
#pragma once

#include "sm103_primitives.cuh"

namespace fa {
namespace dev {

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of `p` (this CTA's shared memory) in the leader CTA's shared
// memory window, for cluster-scope operations.
__device__ __forceinline__ uint32_t at_leader(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// One arrival of the whole warp on a leader barrier.  What these arrivals
// hand over is tensor memory (read or written by this warp, completed by
// tcgen05.wait and ordered by tcgen05.fence::before_thread_sync), not
// generic memory, so the arrive keeps its default CTA-scope release: with a
// cluster-scope release (and acquire on the waiting side) the backward ran
// 29-36% slower.
__device__ __forceinline__ void arrive_leader_warp(uint32_t bar_cl) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0)
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}
// Bounded wait on a barrier the other CTA arrives on (same give-up rules
// as mbar_wait).
__device__ __forceinline__ bool try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_cl(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
  const uint32_t b = smem_u32(bar);
  if (try_wait_cl(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (try_wait_cl(b, parity)) return true;
    if (*reinterpret_cast<volatile unsigned int*>(ctl.status) != 0u) return false;
    if (globaltimer_ns() - t0 > ctl.timeout_ns) {
      atomicCAS(ctl.status, 0u, (unsigned int)FA_ERR_TIMEOUT | (where << 8));
      return false;
    }
  }
}
// 3-D tiled load into this CTA's shared memory whose completion counts on a
// barrier of the leader CTA.
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cl, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cl), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Pair MMAs (M = 256), issued by the leader for both CTAs; warp-wide, one
// elected lane issues.
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %3};\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` in both CTAs once every pair MMA issued so far completes.
__device__ __forceinline__ void commit2(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "h"((unsigned short)3)
      : "memory");
}

// Round r of the persistent schedule of a grid of CTA pairs hands pair
// units [r G, (r + 1) G) to the G pairs, in reverse pair order on odd
// rounds (as snake_unit does for single CTAs).  Both CTAs of a pair walk
// the same units.
__device__ __forceinline__ int pair_unit(int r) {
  const int G = (int)gridDim.x >> 1, c = (int)blockIdx.x >> 1;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

}  // namespace dev
}  // namespace fa
