// PTX helpers for kernels that run on CTA pairs (clusters of two CTAs on
// two SMs, tcgen05 cta_group::2).
#pragma once
#include "common.cuh"
#include "gemm_core.cuh"  // TileCoord

namespace mok {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` once this thread's
// earlier tcgen05 operations have completed.
__device__ __forceinline__ void commit2(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// TMA 2D load into this CTA's shared memory, completing on an mbarrier that
// may live in the peer CTA (leader_bar is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, int32_t x, int32_t y,
                                                 uint32_t leader_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(leader_bar)
      : "memory");
}
// The same with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* m, int32_t x, int32_t y,
                                                      uint32_t leader_bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(leader_bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// tcgen05.cp of one 128-row block of 32-bit words (512 B, word 4 l + c holds
// row 32 c + l) into 4 TMEM columns of every lane quarter: lane 32 q + l,
// column c receives word 4 l + c.  With cta_group::2 each CTA of the pair
// copies from its own shared memory (same offset) into its own TMEM.  The
// source is a no-swizzle K-major operand of 16-byte rows (8-row core matrices
// 128 B apart).
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}
__device__ __forceinline__ void tmem_cp_block2(uint32_t taddr, uint32_t saddr) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc_rows16(saddr))
               : "memory");
}

// Named barrier id for n threads (a multiple of 32; every thread of each
// participating warp calls it).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// AND of p over the n threads of named barrier id (all of them must call it).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t n, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void st_shared_b32(void* p, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// N of a tile whose routed rows are the MMA's N dimension: the tile's rows
// (at most 256) rounded up to 16.
__device__ __forceinline__ int t_ncols(const TileCoord& c) {
  const int n = min(c.rows - c.mt * 256, 256);
  return (n + 15) & ~15;
}

}  // namespace mok
