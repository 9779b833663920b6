// Stage 4 experts on the 5th-generation tensor cores ("Switch Transformer",
// step 6: each expert owns its W1 [d, d_ff] and W2 [d_ff, d]; "Outrageously
// Large", the expert networks E_i). Grouped GEMM over the packed rows:
//   layer 1: hbuf[r] = ReLU(xbuf[r] W1[e] + b1[e])            (bf16 out)
//   layer 2: zbuf[r] = row_gate[r] * (hbuf[r] W2[e] + b2[e])  (fp32 out)
//
// Design (one persistent CTA per SM, 6 warps):
//   warp 0     TMA producer: A tile [128 rows x 64 K] (K-major, 128B swizzle)
//              and B tile [64 K x 256 N] as four [64 x 64] boxes (N-major,
//              i.e. the weights' own row-major layout, 128B swizzle) into a
//              4-stage shared-memory ring, completion on mbarriers.
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//              and one lane issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32)
//              M=128 N=256 K=16, four per stage; tcgen05.commit frees the
//              stage and, after a tile's last stage, hands the accumulator to
//              the epilogue.
//   warps 2-5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, bias,
//              ReLU or gate scale, stores; frees the accumulator so the MMA
//              warp can start the tile after next while this one drains.
// Tiles run over (expert, n block, m block) with m fastest, so CTAs working at
// the same time share the same weight columns in L2. Every wait is bounded:
// past the limit the CTA records MOE_ERR_TIMEOUT, stops issuing, waits
// (bounded) for its copies and MMAs in flight, frees TMEM and returns.
#include "moe_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace moe {
namespace {

constexpr int BM = kTcBM;  // 128 rows (TMEM lanes)
constexpr int BN = 256;    // accumulator columns per tile
constexpr int BK = 64;     // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int kThreads = 192;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BK * BN * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;     // two accumulators
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

struct Params {
  int K, N, E, n_blocks;
  const int32_t *offset;  // [E+1] packed-row offsets
  const float *row_gate;  // layer 2 only
  const __nv_bfloat16 *bias;  // [E, N] or null
  void *out;              // layer 1: bf16 [rows, N]; layer 2: fp32 [rows, N]
  DeviceStatus *st;
};

// ----------------------------------------------------------------------------- PTX wrappers
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
                                          DeviceStatus *st, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        record_error(st, MOE_ERR_TIMEOUT, (long long)where);
        return false;
      }
    }
  }
}

// Wait used while draining after an abort: bounded, no abort check.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
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

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B MN-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
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

// ----------------------------------------------------------------------------- tile map
struct TileMap {
  int *start;  // shared [E+1]: first tile of each expert
  int E, n_blocks;
  const int32_t *offset;
  __device__ void locate(int tile, int &e, int &m_blk, int &n_blk, int &row0, int &rows) const {
    int lo = 0, hi = E;  // largest e with start[e] <= tile
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    e = lo;
    row0 = offset[e];
    rows = offset[e + 1] - row0;
    const int mt = (rows + BM - 1) / BM;
    const int local = tile - start[e];
    n_blk = local / mt;
    m_blk = local % mt;
  }
};

template <int LAYER>
__global__ void __launch_bounds__(kThreads, 1)
k_ffn_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
         const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128B-swizzle atoms.
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  uint64_t *full = bars, *empty = bars + STAGES;
  uint64_t *acc_full = bars + 2 * STAGES, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *tile_start = reinterpret_cast<int *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Tile prefix over experts: ceil(rows_e / BM) * n_blocks tiles each (warp 2).
  if (warp == 2) {
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      int e = e0 + lane;
      int t = 0;
      if (e < p.E) {
        int rows = p.offset[e + 1] - p.offset[e];
        t = (rows + BM - 1) / BM * p.n_blocks;
      }
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < p.E) tile_start[e] = carry + incl - t;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[p.E] = carry;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[p.E];
  TileMap map{tile_start, p.E, p.n_blocks, p.offset};
  const int num_kb = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- producer
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, mb, nb, row0, rows;
        map.locate(tile, e, mb, nb, row0, rows);
        const int arow = row0 + mb * BM;
        const int n0 = nb * BN;
        const int brow = e * p.K;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * BK, arow);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sB + s * B_BYTES + j * (BK * 128), &tmB, &full[s], n0 + j * 64,
                        brow + kb * BK);
        }
      }
      // Copies in flight complete before the CTA leaves (bounded).
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)STAGES ? issued - STAGES : 0; q < issued; ++q)
        mbar_drain(&full[q % STAGES], (q / STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA issuer
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 2)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(b0 + kk * 2048, BK * 128, 1024);
            umma(tmem_d, ad, bd, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      // MMAs in flight complete before TMEM is freed (bounded).
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int r_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
      int e, mb, nb, row0, rows;
      map.locate(tile, e, mb, nb, row0, rows);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      // Warp-uniform decision before the warp-collective TMEM loads.
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 4));
      if (!ready) break;
      tc_fence_after();
      const int m = mb * BM + r_in_tile;
      const bool valid = m < rows;
      const size_t r = (size_t)row0 + m;
      const float g = (LAYER == 2 && valid) ? p.row_gate[r] : 1.f;
      bool bad = false;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int n = nb * BN + c * 32;
        uint32_t v[32];
        const uint32_t taddr =
            tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + c * 32);
        tmem_ld32(taddr, v);  // warp-collective: every lane loads
        if (!valid || n >= p.N) continue;
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          f[j] = __uint_as_float(v[j]);
          if (p.bias) f[j] += __bfloat162float(p.bias[(size_t)e * p.N + n + j]);
        }
        if (LAYER == 1) {
          __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + r * p.N + n;
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(fmaxf(f[2 * j], 0.f), fmaxf(f[2 * j + 1], 0.f));
            packed[j] = *reinterpret_cast<uint32_t *>(&h2);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            reinterpret_cast<uint4 *>(o)[q] =
                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        } else {
          float *o = static_cast<float *>(p.out) + r * p.N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            f[j] *= g;
            bad |= !isfinite(f[j]);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4 *>(o)[q] =
                make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
        }
      }
      if (bad) record_error(p.st, MOE_ERR_NONFINITE, (long long)r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64 cols], 128B swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

constexpr size_t smem_bytes(int E) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + (2 * STAGES + 5) * 8 + 8 + (size_t)(E + 1) * 4;
}

template <int LAYER>
cudaError_t launch_layer(const CUtensorMap &a, const CUtensorMap &b, const Params &p,
                         cudaStream_t s) {
  const size_t smem = smem_bytes(p.E);
  cudaError_t err = cudaFuncSetAttribute(k_ffn_tc<LAYER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  k_ffn_tc<LAYER><<<sm_count(), kThreads, smem, s>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

bool ffn_tc_supported(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0 &&
         smem_bytes(c.E) <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const moe_config &c, int C, const void *xbuf, const int32_t *offset,
                          const int32_t *mtiles, const float *row_gate, const void *W1,
                          const void *b1, const void *W2, const void *b2, void *hbuf, float *zbuf,
                          DeviceStatus *st, cudaStream_t s) {
  (void)C;
  (void)mtiles;
  const uint64_t A = (uint64_t)c.T * c.k;
  CUtensorMap ta1, tb1, ta2, tb2;
  if (!make_map(&ta1, xbuf, A, c.d, BM) || !make_map(&tb1, W1, (uint64_t)c.E * c.d, c.d_ff, BK) ||
      !make_map(&ta2, hbuf, A, c.d_ff, BM) || !make_map(&tb2, W2, (uint64_t)c.E * c.d_ff, c.d, BK))
    return cudaErrorInvalidValue;
  Params p1{c.d, c.d_ff, c.E, (c.d_ff + BN - 1) / BN, offset, row_gate,
            static_cast<const __nv_bfloat16 *>(b1), hbuf, st};
  cudaError_t err = launch_layer<1>(ta1, tb1, p1, s);
  if (err != cudaSuccess) return err;
  Params p2{c.d_ff, c.d, c.E, (c.d + BN - 1) / BN, offset, row_gate,
            static_cast<const __nv_bfloat16 *>(b2), zbuf, st};
  return launch_layer<2>(ta2, tb2, p2, s);
}

}  // namespace moe
