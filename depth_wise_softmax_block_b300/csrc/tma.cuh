// Bulk-tensor (TMA) copies and mbarrier waits for sm_103a, as inline PTX.
//
// Every wait on an mbarrier is bounded in time (the GPU's nanosecond clock %globaltimer): a wait
// of the pipeline (a stage whose copy or whose consumers are late) gives up after
// kWaitLimitNs, a drain (a CTA waiting for its own copies in flight before it exits) after
// kDrainLimitNs.  A wait that gives up counts the event in the device word `g_wait_timeouts`
// (read and cleared through attnres_poll_device_errors) and returns false, so a kernel whose
// copies never land ends in well under a second instead of spinning forever.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

// Count of bounded waits that gave up (one copy per translation unit that includes this file),
// and the value the last read-and-clear took from it.
static __device__ unsigned int g_wait_timeouts = 0;
static __device__ unsigned int g_wait_taken = 0;

// A legitimate wait lasts microseconds (a copy landing, a stage being consumed).
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;    // 200 ms
constexpr uint64_t kDrainLimitNs = 2000ull * 1000 * 1000;  // 2 s

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Reads and clears this translation unit's timeout word in one atomic exchange on the device,
// after every kernel of the device (on every stream) has finished.  Host only; synchronous.
// 0xffffffff if a CUDA call failed.
static __global__ void take_wait_timeouts_kernel() {
  g_wait_taken = atomicExch(&g_wait_timeouts, 0u);
}
static inline unsigned int take_wait_timeouts() {
  if (cudaDeviceSynchronize() != cudaSuccess) return 0xffffffffu;
  take_wait_timeouts_kernel<<<1, 1>>>();
  if (cudaGetLastError() != cudaSuccess) return 0xffffffffu;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wait_taken, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes the initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Polls until the phase with the given parity has completed (true), or until `limit_ns` have
// passed since the first failed poll (false, and the event is counted).  kCluster: acquire at
// cluster scope (arrivals from other CTAs of the cluster).
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_for(uint32_t a, uint32_t parity, uint64_t limit_ns) {
  auto poll = [&]() {
    return kCluster ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (poll()) return true;
    if (global_ns() - t0 > limit_ns) break;
  }
  atomicAdd(&g_wait_timeouts, 1u);
  return false;
}

// A wait of the pipeline; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for<false>(smem_addr(bar), parity, kWaitLimitNs);
}

// A CTA waiting for its own copies (or MMAs) in flight before it exits; false after kDrainLimitNs.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for<false>(smem_addr(bar), parity, kDrainLimitNs);
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Tiled loads global -> shared; completion is signalled on `bar` as transaction bytes.
// The innermost coordinate x must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Tensor store of a shared-memory tile (written by this CTA's threads, made visible with
// fence_proxy_async first) into the box at (x, y, z); tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most N of this thread's committed bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Every bulk group of this thread complete (its global writes done).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Four 8x8 b16 matrices stored transposed: register k of thread i holds row i / 4, columns
// 2 (i % 4) and 2 (i % 4) + 1 of matrix k; thread i gives the shared-memory address of row
// i % 8 of matrix i / 8 of the stored (transposed) matrices, 16 bytes each.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t row_addr, uint32_t r0, uint32_t r1,
                                                  uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(
                   row_addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// ---- thread-block clusters: distributed shared memory --------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Arrive (release at cluster scope) on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

// mbar_wait with acquire at cluster scope (the arrivals come from other CTAs); bounded.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for<true>(smem_addr(bar), parity, kWaitLimitNs);
}

// All threads of all CTAs of the cluster (every thread must execute it, convergently).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Barrier over the first `n` threads of the CTA (named barrier `id`, id > 0).
__device__ __forceinline__ void named_barrier(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile written by a 128-byte-swizzled
// tensor copy (rows of 128 bytes, tile base aligned to 1024 bytes).
__device__ __forceinline__ int sw128(int row, int chunk) {
  return (row << 7) + (((chunk ^ row) & 7) << 4);
}

}  // namespace attnres
