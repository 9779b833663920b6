// Inline-PTX wrappers for the tensor-core kernels (sm_103a): mbarriers with
// bounded waits, TMA tile loads, tcgen05 fences, shared-memory matrix
// descriptors, commits and TMEM loads; plus the host helpers that build TMA
// descriptors. Internal to libmoe.so.
#pragma once

#include "moe_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace moe {

// Host helpers (defined in k_ffn_tc.cu).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64 cols], 128B swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// 2-D bf16 or fp32 tensor [rows, cols] (cols % 8 == 0, 16-byte-aligned base), box
// [32 rows, 32 columns], 64-byte (bf16) or 128-byte (fp32) swizzle: a GEMM's
// output for stage_store_bf16 / stage_store_f32. False if it cannot be made.
bool make_rows_map(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, bool f32);
// The same for fp32 with a [32 rows, 16 columns] box (64-byte rows, 64-byte
// swizzle), for stage_store_f32x16.
bool make_rows_map16(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols);
int sm_count();
// Limit of every bounded mbarrier wait, in ns: MOE_WAIT_LIMIT_NS if set (read
// at each launch, so a test can shorten it to force the timeout path), else 2 s.
unsigned long long wait_limit_ns();

namespace {

constexpr unsigned long long kDrainLimitNs = 2000000000ull;  // 2 s per drain wait

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait. Returns false if this CTA is aborting (limit reached here or
// elsewhere in the CTA); the first thread to run out records the error.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          DeviceStatus *st, int where,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 >= limit_ns) {
      *abort_flag = 1;
      record_error(st, MOE_ERR_TIMEOUT, (long long)where);
      return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
  }
}

// try_wait with acquire at cluster scope: for barriers that another CTA of the
// cluster arrives on (release.cluster) after writing this CTA's shared memory.
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (see mbar_wait).
__device__ __forceinline__ bool mbar_wait_cl(uint64_t *bar, uint32_t parity,
                                             volatile int *abort_flag, DeviceStatus *st,
                                             int where, unsigned long long limit_ns) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 >= limit_ns) {
      *abort_flag = 1;
      record_error(st, MOE_ERR_TIMEOUT, (long long)where);
      return false;
    }
    if (mbar_try_wait_cl(bar, parity)) return true;
  }
}

// Wait used while draining after an abort: bounded, no abort check.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kDrainLimitNs) return;
  }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// TMA stores of a shared-memory tile, and the bulk-group bookkeeping around
// them (each store group is committed by the thread that issued it).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x,
                                             int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   (uint64_t)map),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          (uint64_t)map),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The thread's committed store groups have read their shared memory: all of
// them, or all but the most recent one.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_but1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// The thread's committed store groups are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Generic-proxy writes to shared memory, visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Three 16-column TMEM loads (lanes of this warp's quadrant) and one wait:
// r[0..15] from a0, r[16..31] from a1, r[32..47] from a2.
__device__ __forceinline__ void tmem_ld16x3(uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t (&r)[48]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, "
      "%8, %9, %10, %11, %12, %13, %14, %15}, [%48];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, "
      "%24, %25, %26, %27, %28, %29, %30, %31}, [%49];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, "
      "%40, %41, %42, %43, %44, %45, %46, %47}, [%50];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(a0), "r"(a1), "r"(a2)
      : "memory");
}

// One warp's 32 output rows x 32 columns of a GEMM epilogue (lane l holds row
// l), staged in shared memory and sent by one TMA store at column n, row r0
// (tmO: the output [rows, N], box [32 rows, 32 columns]; bf16 in the 64-byte
// swizzle, fp32 in the 128-byte swizzle). Per-lane row stores send 32 rows'
// 16-byte pieces per instruction; a TMA store writes whole row segments. buf
// (4 KB, 1024-byte aligned) is one of the warp's two staging tiles, used in
// turn: before it is written, the store that last read it (two chunks back)
// must have read it.
__device__ __forceinline__ void stage_store_bf16(const CUtensorMap *tmO, float *buf,
                                                 const uint32_t (&packed)[16], int n, int r0) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_read_but1();
  __syncwarp();
  uint4 *row = reinterpret_cast<uint4 *>(buf) + lane * 4;  // 64-byte rows
  const int x = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    row[q ^ x] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmO, buf, n, r0);
    bulk_commit();
  }
}
__device__ __forceinline__ void stage_store_f32(const CUtensorMap *tmO, float *buf,
                                                const float (&f)[32], int n, int r0) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_read_but1();
  __syncwarp();
  float4 *row = reinterpret_cast<float4 *>(buf) + lane * 8;  // 128-byte rows
#pragma unroll
  for (int q = 0; q < 8; ++q)
    row[q ^ (lane & 7)] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmO, buf, n, r0);
    bulk_commit();
  }
}

// The same for 16 fp32 columns (64-byte rows in the 64-byte swizzle, the
// [32 x 16] box of make_rows_map16): f points at this lane's 16 values.
__device__ __forceinline__ void stage_store_f32x16(const CUtensorMap *tmO, float *buf,
                                                   const float *f, int n, int r0) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_read_but1();
  __syncwarp();
  float4 *row = reinterpret_cast<float4 *>(buf) + lane * 4;  // 64-byte rows
  const int x = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    row[q ^ x] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmO, buf, n, r0);
    bulk_commit();
  }
}

// ----------------------------------------------------------------------------- CTA pairs
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Arrive on a barrier of any CTA of the cluster with the default semantics
// (release at CTA scope): for barriers that only order tcgen05 accesses, which
// the tcgen05 fences around the barrier order, with no shared data to publish
// (a cluster-scope release would wait for every earlier store of the thread).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// 32-bit store to a shared-memory word of any CTA of the cluster (an address
// from mapa, or this CTA's own).
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(bar_cluster_addr), "r"(x), "r"(y)
      : "memory");
}
// Arrives on the barrier at this offset in every CTA of `mask` (bit = cluster rank).
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask = 0x3) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

}  // namespace
}  // namespace moe
