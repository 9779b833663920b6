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
#include "tc_ptx.cuh"

#include <stdlib.h>

#include <mutex>

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
// One-CTA kernel's epilogue staging: per epilogue warp two 2 KB tiles, each
// [32 rows x 32 columns] of bf16 output or [32 x 16] of fp32 (64-byte rows,
// 64-byte swizzle).
constexpr int STG_TILE = 32 * 32 / 2;  // 2 KB, counted in floats
constexpr int STG_BYTES = 4 * 2 * STG_TILE * 4;

struct Params {
  int K, N, E, n_blocks;
  uint32_t *sched;        // [2] the CTA-pair kernel's tile counter and done count (zero at launch)
  int dynamic;            // CTA-pair kernel: tiles from the counter (else round robin)
  int half_tiles;         // CTA-pair kernel: short last row tiles at M = 128
  const int32_t *offset;  // [E+1] packed-row offsets
  const float *row_gate;  // layer 2 only
  const __nv_bfloat16 *bias;  // [E, N] or null
  void *out;              // layer 1: bf16 [rows, N]; layer 2: fp32 (or bf16) [rows, N]
  DeviceStatus *st;
  unsigned long long wait_ns;  // bounded-wait limit
  int z_bf16;                  // layer 2 writes Z in bf16
  int tma_out;                 // whole 32-row groups of the output leave by TMA store
  int snake;                   // CTA-pair kernel: 1 = odd waves of tiles run K backwards,
                               // 2 = every tile does (0 = none)
};

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

// tmO: the output [rows, N] when p.tma_out is set: bf16 with a [32 rows, 32
// columns] box, or fp32 (layer 2's Z) with a [32 rows, 16 columns] box, both
// in the 64-byte swizzle.
template <int LAYER>
__global__ void __launch_bounds__(kThreads, 1)
k_ffn_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
         const __grid_constant__ CUtensorMap tmO, const Params p) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128B-swizzle atoms.
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  float *stg_all = reinterpret_cast<float *>(sB + STAGES * B_BYTES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES + STG_BYTES);
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
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 1, p.wait_ns)) {
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
    pdl_trigger();  // all loads issued: the next kernel may be scheduled
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA issuer
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 2, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 3, p.wait_ns)) {
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
    pdl_trigger();
  } else {
    // ----------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int r_in_tile = quad * 32 + lane;
    float *stg = stg_all + (size_t)(warp - 2) * 2 * STG_TILE;  // this warp's two tiles
    uint32_t stg_cnt = 0;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
      int e, mb, nb, row0, rows;
      map.locate(tile, e, mb, nb, row0, rows);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      // Warp-uniform decision before the warp-collective TMEM loads.
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 4, p.wait_ns));
      if (!ready) break;
      tc_fence_after();
      const int m = mb * BM + r_in_tile;
      const bool valid = m < rows;
      const size_t r = (size_t)row0 + m;
      const float g = (LAYER == 2 && valid) ? p.row_gate[r] : 1.f;
      // The output of a warp whose 32 rows all belong to this expert leaves by
      // TMA store (a partial group would spill into the next expert's rows).
      const bool tma_rows = p.tma_out && m - lane + 32 <= rows;
      const int r0 = row0 + m - lane;
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
        float *sbuf = stg + (stg_cnt & 1u) * STG_TILE;
        if (LAYER == 1) {
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(fmaxf(f[2 * j], 0.f), fmaxf(f[2 * j + 1], 0.f));
            packed[j] = *reinterpret_cast<uint32_t *>(&h2);
          }
          if (tma_rows) {
            stage_store_bf16(&tmO, sbuf, packed, n, r0);
            ++stg_cnt;
          } else {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + r * p.N + n;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<uint4 *>(o)[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                           packed[4 * q + 2], packed[4 * q + 3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            f[j] *= g;
            bad |= !isfinite(f[j]);
          }
          if (p.z_bf16) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
              packed[j] = *reinterpret_cast<uint32_t *>(&h2);
            }
            if (tma_rows) {
              stage_store_bf16(&tmO, sbuf, packed, n, r0);
              ++stg_cnt;
            } else {
              __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + r * p.N + n;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                reinterpret_cast<uint4 *>(o)[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                             packed[4 * q + 2], packed[4 * q + 3]);
            }
          } else if (tma_rows) {
            // fp32: the chunk's two 16-column halves, one staging tile each
            stage_store_f32x16(&tmO, sbuf, f, n, r0);
            ++stg_cnt;
            stage_store_f32x16(&tmO, stg + (stg_cnt & 1u) * STG_TILE, f + 16, n + 16, r0);
            ++stg_cnt;
          } else {
            float *o = static_cast<float *>(p.out) + r * p.N + n;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4 *>(o)[q] =
                  make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
          }
        }
      }
      if (bad) record_error(p.st, MOE_ERR_NONFINITE, (long long)r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores are complete
    pdl_trigger();
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

// ----------------------------------------------------------------------------- CTA-pair variant
// Same GEMM with tcgen05.mma.cta_group::2: a cluster of two CTAs on two SMs
// computes a 256-row x 256-column tile. Each CTA loads its own 128 rows of A
// and half (128 columns) of the B tile, so each SM takes in 32 KB per K step
// instead of 48 KB for the same MMA work; the even CTA of the pair issues the
// MMAs, which read B from both CTAs' shared memory and write each CTA's rows
// to that CTA's TMEM. The odd CTA's TMA completions are counted on the even
// CTA's "full" barriers; the MMA commits arrive (multicast) on both CTAs'
// "empty" and "accumulator full" barriers; both CTAs' epilogues arrive on the
// even CTA's "accumulator empty" barriers.
constexpr int P_STAGES = 6;
// Tile indices handed from the even CTA's producer to the kernel's other
// roles, in flight at once (the producer runs at most a tile ahead of the MMA,
// which runs at most two ahead of the epilogue).
constexpr int kRing = 8;
// Arrivals that free a ring slot: the even CTA's MMA issuer and four epilogue
// warps, the odd CTA's producer and four epilogue warps.
constexpr int kRingConsumers = 10;
constexpr int P_BN_HALF = BN / 2;               // B columns held per CTA
constexpr int P_A_BYTES = BM * BK * 2;          // 16 KB
constexpr int P_B_BYTES = BK * P_BN_HALF * 2;   // 16 KB
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
// Epilogue staging of the CTA-pair kernel: per epilogue warp two 4 KB tiles,
// each [32 rows x 32 columns] of the output (fp32 in the 128-byte swizzle,
// bf16 in the 64-byte swizzle).
constexpr int P_STG_TILE = 32 * 32;  // floats
constexpr int P_STG_BYTES = 4 * 2 * P_STG_TILE * 4;

// kind::f16, fp32 accumulate, bf16 A/B, A K-major, B MN-major, M = 256, N = 256.
constexpr uint32_t kIdescPair = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                                ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
// The same with M = 128 (64 rows per CTA), for an expert's last row tile
// when it holds at most 128 rows: half the MMA work of a 256-row tile. Its
// accumulator in each CTA: TMEM lanes 0-63 hold the CTA's 64 rows for
// columns 0-127 of the tile, lanes 64-127 the same rows for columns 128-255,
// both at accumulator columns 0-127.
constexpr uint32_t kIdescPairHalf = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) |
                                    (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
                                    ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void umma_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
template <int LAYER>
__global__ void __launch_bounds__(kThreads, 1)
k_ffn_tc_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmO, const Params p) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + P_STAGES * P_A_BYTES;
  float *stg_all = reinterpret_cast<float *>(sB + P_STAGES * P_B_BYTES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + P_STAGES * P_B_BYTES + P_STG_BYTES);
  uint64_t *full = bars, *empty = bars + P_STAGES;
  uint64_t *acc_full = bars + 2 * P_STAGES, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint64_t *tfull = drain + 1, *tempty = tfull + kRing;  // the tile ring's barriers
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + kRing);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *ring = reinterpret_cast<volatile int *>(tmem_slot + 2);  // [kRing] tile indices
  int *tile_start = const_cast<int *>(ring + kRing);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's expect_tx arrival
      mbar_init(&empty[s], 1);  // one multicast commit per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // four epilogue warps in each CTA
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&tfull[r], 1);                // the even CTA's producer publishes
      mbar_init(&tempty[r], kRingConsumers);  // used in the even CTA only
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {  // expert tile prefix: ceil(rows_e / 256) * n_blocks tiles each
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < p.E) {
        const int rows = p.offset[e + 1] - p.offset[e];
        t = (rows + 2 * BM - 1) / (2 * BM) * p.n_blocks;
      }
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < p.E) tile_start[e] = carry + incl - t;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[p.E] = carry;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[p.E];
  const int num_kb = p.K / BK;

  // half: the expert's last row tile holds at most 128 rows and runs as an
  // M = 128 tile (kIdescPairHalf), each CTA taking 64 of them.
  auto locate = [&](int tile, int &e, int &pm, int &nb, int &row0, int &rows, bool &half) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    e = lo;
    row0 = p.offset[e];
    rows = p.offset[e + 1] - row0;
    const int mt = (rows + 2 * BM - 1) / (2 * BM);
    const int local = tile - tile_start[e];
    nb = local / mt;
    pm = local % mt;
    half = p.half_tiles && pm == mt - 1 && rows - pm * 2 * BM <= BM;
  };

  if (warp == 0) {
    if (lane == 0) {
      // --------------------------------------------------------- producer (both CTAs)
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      // Tiles: each pair's first is its index; the even CTA's producer takes
      // every later one from the counter when it needs it, so pairs that run
      // ahead take more tiles, and publishes it (or total_tiles: the end)
      // through the ring to the other roles of both CTAs.
      // The take for the next tile is issued a few k-blocks before this
      // tile's last load, so its round trip overlaps the loads in flight.
      uint32_t it = 0;
      bool ok = true;
      long long taken = -1;  // the next tile's take, once issued
      int tile_rr = pair;    // round-robin order (p.dynamic == 0)
      for (int j = 0; ok; ++j) {
        const int slot = j % kRing;
        const uint32_t rph = (uint32_t)(j / kRing) & 1u;
        int tile;
        if (leader) {
          if (j == 0) {
            tile = pair;
          } else if (p.dynamic) {
            if (taken < 0) taken = atomicAdd(p.sched, 1u);
            tile = (int)min(taken + n_pairs, (long long)total_tiles);
            taken = -1;
          } else {
            tile_rr += n_pairs;
            tile = min(tile_rr, total_tiles);
          }
          if (!mbar_wait_cl(&tempty[slot], rph ^ 1u, abort_flag, p.st, 15, p.wait_ns)) {
            ok = false;
            break;
          }
          ring[slot] = tile;
          st_cluster_u32(mapa(smem_u32((const void *)&ring[slot]), 1), (uint32_t)tile);
          mbar_arrive_cluster(smem_u32(&tfull[slot]));
          mbar_arrive_cluster(mapa(smem_u32(&tfull[slot]), 1));
        } else {
          if (!mbar_wait_cl(&tfull[slot], rph, abort_flag, p.st, 16, p.wait_ns)) {
            ok = false;
            break;
          }
          tile = ring[slot];
          mbar_arrive_cluster(mapa(smem_u32(&tempty[slot]), 0));
        }
        if (tile >= total_tiles) break;
        int e, pm, nb, row0, rows;
        bool half;
        locate(tile, e, pm, nb, row0, rows, half);
        // A half tile's CTA uses the first 64 of the 128 rows its box brings.
        const int arow = row0 + pm * 2 * BM + (int)rank * (half ? BM / 2 : BM);
        const int ncol = nb * BN + (int)rank * P_BN_HALF;
        const int brow = e * p.K;
        const int take_at = num_kb > 4 ? num_kb - 4 : 0;
        // Tiles of odd waves (tile / pairs) walk K from the end: their first
        // K blocks are the ones the wave before read last, so the operand
        // rows and stripes the two waves share are still in L2. The sum's
        // order is fixed by the tile, so results do not depend on which
        // pair takes it.
        const bool rev = p.snake == 2 || (p.snake == 1 && ((tile / n_pairs) & 1));
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          if (leader && p.dynamic && kb == take_at) taken = atomicAdd(p.sched, 1u);
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 11, p.wait_ns)) {
            ok = false;
            break;
          }
          const int kx = (rev ? num_kb - 1 - kb : kb) * BK;
          const uint32_t full_leader = mapa(smem_u32(&full[s]), 0);
          if (leader) mbar_expect_tx(&full[s], 2 * P_STAGE_BYTES);
          tma_load_2d_pair(sA + s * P_A_BYTES, &tmA, full_leader, kx, arow);
#pragma unroll
          for (int q = 0; q < P_BN_HALF / 64; ++q)
            tma_load_2d_pair(sB + s * P_B_BYTES + q * (BK * 128), &tmB, full_leader,
                             ncol + q * 64, brow + kx);
        }
      }
      // This CTA's copies have landed once the MMAs that read them are done.
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)P_STAGES ? issued - P_STAGES : 0; q < issued; ++q)
        mbar_drain(&empty[q % P_STAGES], (q / P_STAGES) & 1u);
      if (leader && p.dynamic) {
        // The last pair to finish resets the counter for the next launch
        // (every pair's last take precedes its count).
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == (uint32_t)n_pairs - 1) {
          atomicExch(p.sched, 0u);
          atomicExch(p.sched + 1, 0u);
        }
      }
    }
    __syncwarp();
    pdl_trigger();  // all loads issued: the next kernel may be scheduled
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // --------------------------------------------------------- MMA issuer (even CTA)
      uint32_t it = 0;
      bool ok = true;
      for (int local = 0; ok; ++local) {
        const int slot = local % kRing;
        if (!mbar_wait_cl(&tfull[slot], (uint32_t)(local / kRing) & 1u, abort_flag, p.st, 17,
                          p.wait_ns))
          break;
        const int tile = ring[slot];
        mbar_arrive_cluster(smem_u32(&tempty[slot]));
        if (tile >= total_tiles) break;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        int e, pm, nb, row0, rows;
        bool half;
        locate(tile, e, pm, nb, row0, rows, half);
        const uint32_t idesc = half ? kIdescPairHalf : kIdescPair;
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 12, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 13, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * P_A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * P_B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(b0 + kk * 2048, BK * 128, 1024);
            umma_pair(tmem_d, ad, bd, idesc, (kb | kk) ? 1u : 0u);
          }
          umma_commit_pair(&empty[s]);
        }
        if (ok) umma_commit_pair(&acc_full[buf]);
      }
      umma_commit_pair(drain, 0x1);
      mbar_drain(drain, 0);
    }
    __syncwarp();
    pdl_trigger();
  } else {
    // ------------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    const int r_in_tile = quad * 32 + lane;
    const uint32_t acc_empty_leader0 = mapa(smem_u32(&acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa(smem_u32(&acc_empty[1]), 0);
    float *stg = stg_all + (size_t)(warp - 2) * 2 * P_STG_TILE;  // this warp's two tiles
    uint32_t stg_cnt = 0;                                         // chunks staged so far
    for (int local = 0;; ++local) {
      const int slot = local % kRing;
      int tile = total_tiles;
      bool got = false;
      if (lane == 0) {
        got = mbar_wait_cl(&tfull[slot], (uint32_t)(local / kRing) & 1u, abort_flag, p.st, 18,
                           p.wait_ns);
        if (got) {
          tile = ring[slot];
          mbar_arrive_cluster(mapa(smem_u32(&tempty[slot]), 0));
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (!got || tile >= total_tiles) break;
      int e, pm, nb, row0, rows;
      bool half;
      locate(tile, e, pm, nb, row0, rows, half);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 14, p.wait_ns));
      if (!ready) break;
      tc_fence_after();
      // Full tile: lane quadrant q holds rows 32q.. of this CTA's 128, all
      // 256 columns. Half tile: quadrants 0-1 hold the CTA's 64 rows for
      // columns 0-127, quadrants 2-3 the same rows for columns 128-255.
      const int m = half ? pm * 2 * BM + (int)rank * (BM / 2) + (quad & 1) * 32 + lane
                         : pm * 2 * BM + (int)rank * BM + r_in_tile;
      const int ncol0 = nb * BN + (half ? (quad >> 1) * (BN / 2) : 0);
      const int nchunks = half ? BN / 64 : BN / 32;
      const bool valid = m < rows;
      const size_t r = (size_t)row0 + m;
      const float g = (LAYER == 2 && valid) ? p.row_gate[r] : 1.f;
      // The warp's 32 rows all belong to this expert: they leave by TMA store
      // (a partial group would spill into the next expert's rows).
      const bool tma_rows = p.tma_out && m - lane + 32 <= rows;
      const int r0 = row0 + m - lane;
      bool bad = false;
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        const int n = ncol0 + c * 32;
        uint32_t v[32];
        const uint32_t taddr =
            tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + c * 32);
        tmem_ld32(taddr, v);
        if (!valid || n >= p.N) continue;
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          f[j] = __uint_as_float(v[j]);
          if (p.bias) f[j] += __bfloat162float(p.bias[(size_t)e * p.N + n + j]);
        }
        float *sbuf = stg + (stg_cnt & 1u) * P_STG_TILE;
        if (LAYER == 1) {
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 h2 =
                __floats2bfloat162_rn(fmaxf(f[2 * j], 0.f), fmaxf(f[2 * j + 1], 0.f));
            packed[j] = *reinterpret_cast<uint32_t *>(&h2);
          }
          if (tma_rows) {
            stage_store_bf16(&tmO, sbuf, packed, n, r0);
            ++stg_cnt;
          } else {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + r * p.N + n;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<uint4 *>(o)[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                           packed[4 * q + 2], packed[4 * q + 3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            f[j] *= g;
            bad |= !isfinite(f[j]);
          }
          if (p.z_bf16) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
              packed[j] = *reinterpret_cast<uint32_t *>(&h2);
            }
            if (tma_rows) {
              stage_store_bf16(&tmO, sbuf, packed, n, r0);
              ++stg_cnt;
            } else {
              __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) + r * p.N + n;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                reinterpret_cast<uint4 *>(o)[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                             packed[4 * q + 2], packed[4 * q + 3]);
            }
          } else if (tma_rows) {
            stage_store_f32(&tmO, sbuf, f, n, r0);
            ++stg_cnt;
          } else {
            float *o = static_cast<float *>(p.out) + r * p.N + n;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4 *>(o)[q] =
                  make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
          }
        }
      }
      if (bad) record_error(p.st, MOE_ERR_NONFINITE, (long long)r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(buf ? acc_empty_leader1 : acc_empty_leader0);
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores are complete
    pdl_trigger();
  }
  tc_fence_before();
  cluster_sync_all();  // every MMA reading either CTA's memory and every TMEM read are done
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

// ----------------------------------------------------------------------------- host side
// Looked up once; a function-local static with an initializer is thread-safe.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
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

// 2-D tensor [rows, cols] (cols % 8 == 0, 16-byte-aligned base) of bf16 or
// fp32: an expert GEMM's output, box [32 rows, 32 columns] in the 64-byte
// (bf16) or 128-byte (fp32) swizzle, for the CTA-pair kernel's TMA stores.
bool make_rows_map(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, bool f32) {
  auto fn = encode_fn();
  if (!fn || (uintptr_t)base % 16 != 0 || cols % 8 != 0) return false;
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_rows_map16(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn || (uintptr_t)base % 16 != 0 || cols % 8 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long wait_limit_ns() {
  const char *v = getenv("MOE_WAIT_LIMIT_NS");
  if (v && *v) return strtoull(v, nullptr, 10);
  return 2000000000ull;
}

int sm_count() {
  static const int n = [] {
    int dev = 0, m = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev);
    return m > 0 ? m : 1;
  }();
  return n;
}

namespace {

constexpr size_t smem_bytes(int E) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + STG_BYTES + (2 * STAGES + 5) * 8 + 8 +
         (size_t)(E + 1) * 4;
}

template <int LAYER>
cudaError_t launch_layer(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                         const Params &p, cudaStream_t s) {
  const size_t smem = smem_bytes(p.E);
  cudaError_t err = cudaFuncSetAttribute(k_ffn_tc<LAYER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  launch_pdl_c(kPdlGemm, k_ffn_tc<LAYER>, sm_count(), kThreads, smem, s, a, b, o, p);
  return cudaGetLastError();
}

constexpr size_t smem_bytes_pair(int E) {
  return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_STG_BYTES +
         (2 * P_STAGES + 5 + 2 * kRing) * 8 + 8 + (size_t)kRing * 4 + (size_t)(E + 1) * 4;
}

cudaLaunchAttribute pair_cluster_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Clusters of two that can be resident at once (0 if the device cannot host one).
// The answer depends on the shared-memory size (it grows with E), so it is kept
// per size, under a lock, in a small table; a full table means no caching.
std::mutex g_pair_mu;

int pair_clusters(size_t smem) {
  constexpr int kSlots = 16;
  static size_t keys[kSlots];
  static int vals[kSlots];
  static int used = 0;
  std::lock_guard<std::mutex> lock(g_pair_mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == smem) return vals[i];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count() / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1] = {pair_cluster_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(k_ffn_tc_pair<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k_ffn_tc_pair<1>, &cfg) != cudaSuccess)
    n = 0;
  if (used < kSlots) {
    keys[used] = smem;
    vals[used] = n;
    ++used;
  }
  return n;
}

template <int LAYER>
cudaError_t launch_layer_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                              const Params &p, int clusters, cudaStream_t s) {
  const size_t smem = smem_bytes_pair(p.E);
  cudaError_t err = cudaFuncSetAttribute(
      k_ffn_tc_pair<LAYER>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2] = {pair_cluster_attr(), {}};
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled(kPdlGemm) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_ffn_tc_pair<LAYER>, a, b, o, p);
}

// MOE_FFN_SCHED=static makes the CTA-pair kernel take its tiles round robin
// instead of from the counter (read at each call; for comparisons).
int ffn_dynamic() {
  const char *v = getenv("MOE_FFN_SCHED");
  return v && v[0] == 's' ? 0 : 1;
}

// MOE_FFN_SNAKE=0 keeps every CTA-pair tile's K order forward, =all runs
// every tile backwards (read at each call; for comparisons and tests);
// otherwise odd waves run backwards.
int ffn_snake() {
  const char *v = getenv("MOE_FFN_SNAKE");
  if (!v || !*v) return 1;
  return v[0] == '0' ? 0 : (v[0] == 'a' ? 2 : 1);
}

// MOE_FFN_TC_VARIANT=single or =pair forces one kernel (read at each call);
// otherwise the rule in launch_ffn_tc picks per layer.
int ffn_variant() {
  const char *v = getenv("MOE_FFN_TC_VARIANT");
  if (!v || !*v) return 0;
  return v[0] == 's' ? 1 : (v[0] == 'p' ? 2 : 0);
}

// Clusters available to the CTA-pair kernel, or 0 when the one-CTA kernel must
// run (forced, or a device without room).
int pair_clusters_for(int E) {
  if (ffn_variant() == 1 || smem_bytes_pair(E) > 227 * 1024) return 0;
  return pair_clusters(smem_bytes_pair(E));
}

}  // namespace

bool ffn_tc_supported(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0 &&
         smem_bytes(c.E) <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const moe_config &c, int C, const void *xbuf, const int32_t *offset,
                          const int32_t *mtiles, const float *row_gate, const void *W1,
                          const void *b1, const void *W2, const void *b2, void *hbuf, void *zbuf,
                          bool z_bf16, DeviceStatus *st, cudaStream_t s) {
  (void)mtiles;
  const uint64_t A = (uint64_t)c.T * c.k;
  CUtensorMap ta1, tb1, ta2, tb2;
  if (!make_map(&ta1, xbuf, A, c.d, BM) || !make_map(&tb1, W1, (uint64_t)c.E * c.d, c.d_ff, BK) ||
      !make_map(&ta2, hbuf, A, c.d_ff, BM) || !make_map(&tb2, W2, (uint64_t)c.E * c.d_ff, c.d, BK))
    return cudaErrorInvalidValue;
  uint32_t *sched = &st->gemm_next;  // gemm_next, gemm_done: adjacent words
  const int dyn = ffn_dynamic();
  // MOE_FFN_HALF=0 runs every row tile at M = 256 (read at each call; for comparisons).
  const char *hv = getenv("MOE_FFN_HALF");
  const int half = hv && hv[0] == '0' ? 0 : 1;
  Params p1{c.d, c.d_ff, c.E, (c.d_ff + BN - 1) / BN, sched, dyn, half, offset, row_gate,
            static_cast<const __nv_bfloat16 *>(b1), hbuf, st, wait_limit_ns()};
  Params p2{c.d_ff, c.d, c.E, (c.d + BN - 1) / BN, sched, dyn, half, offset, row_gate,
            static_cast<const __nv_bfloat16 *>(b2), zbuf, st, wait_limit_ns(), z_bf16 ? 1 : 0};
  // Per layer: the CTA pair pays off for long K and enough 256-row tiles to
  // fill several waves; otherwise the one-CTA kernel's finer tiles win.
  const long rows = (long)c.T * c.k < (long)c.E * C ? (long)c.T * c.k : (long)c.E * C;
  const int clusters = pair_clusters_for(c.E);
  const bool force_pair = ffn_variant() == 2;
  auto pair_for = [&](int K, int N) {
    return clusters > 0 &&
           (force_pair || (K >= 2048 && (rows / 256) * ((N + BN - 1) / BN) >= 4L * clusters));
  };
  // The CTA-pair kernel's output maps (H, then Z): box [32 rows, 32 columns].
  // The one-CTA kernel stores fp32 Z in 16-column boxes (its staging tiles
  // are 2 KB).
  CUtensorMap to1, to2, to2s;
  p1.tma_out = make_rows_map(&to1, hbuf, A, c.d_ff, false) ? 1 : 0;
  p2.tma_out = make_rows_map(&to2, zbuf, A, c.d, !z_bf16) ? 1 : 0;
  if (!p1.tma_out) to1 = ta1;  // unused
  if (!p2.tma_out) to2 = ta2;
  p1.snake = p2.snake = ffn_snake();
  Params p2s = p2;
  if (z_bf16) {
    to2s = to2;
  } else {
    p2s.tma_out = make_rows_map16(&to2s, zbuf, A, c.d) ? 1 : 0;
    if (!p2s.tma_out) to2s = ta2;
  }
  cudaError_t err = pair_for(c.d, c.d_ff) ? launch_layer_pair<1>(ta1, tb1, to1, p1, clusters, s)
                                          : launch_layer<1>(ta1, tb1, to1, p1, s);
  if (err != cudaSuccess) return err;
  return pair_for(c.d_ff, c.d) ? launch_layer_pair<2>(ta2, tb2, to2, p2, clusters, s)
                               : launch_layer<2>(ta2, tb2, to2s, p2s, s);
}

}  // namespace moe
