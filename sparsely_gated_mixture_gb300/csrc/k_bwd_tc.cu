// Backward of the expert networks on the 5th-generation tensor cores
// ("Outrageously Large Neural Networks", section 3.4: the experts and the
// gate are trained by plain back-propagation; "Switch Transformer", step 6:
// each expert owns W1 [d, d_ff] and W2 [d_ff, d]). One grouped-GEMM kernel in
// three modes over the rows each expert received in the forward:
//
//   dgrad through W2 (mode 0):  D = dY_rows W2[e]^T           [rows, d_ff]
//       epilogue: dgate partial <D_r, h_r> per 256-column block, and
//       dpre_r = g_r * D_r * [h_r > 0] in bf16 (pad rows written as zero)
//   dgrad through W1 (mode 1):  dX_rows = dpre_rows W1[e]^T   [rows, d]   (fp32)
//   weight gradient  (mode 2):  dW[e] = A_rows^T B_rows       [M, N]      (fp32)
//       dW2: A = h rows, B = g * dY rows;  dW1: A = x rows, B = dpre rows
//
// The backward's own row buffers (dY, g*dY, dpre, dX) give each expert a
// block of rows padded to a multiple of 64 (at least 64), pad rows zero, at
// the offsets poff[e]. The weight-gradient mode runs its K loop over those
// padded rows: the pad rows of B are zero, so whatever A holds there (the
// next expert's rows, or rows the caller zeroed past the last one) adds
// nothing, and no K tail needs masking.
//
// Operand layouts (bf16, 128-byte swizzle, as the forward kernel):
//   modes 0, 1: A K-major [128 rows x 64 K]; B K-major [256 rows x 64 K]: the
//               weight's own rows (W2[e] is [d_ff, d]: row f holds K = d
//               contiguous values; W1[e] is [d, d_ff]: row i holds d_ff).
//   mode 2:     A MN-major (M contiguous) as two [64 K x 64 M] boxes, B
//               MN-major as four [64 K x 64 N] boxes; the instruction
//               descriptor's transpose bits select MN-major for both.
// Warp roles, the 4-stage ring, two TMEM accumulators and the bounded waits
// are those of the forward kernel: warp 0 TMA producer, warp 1 TMEM owner and
// MMA issuer, warps 2-5 epilogue.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

#include <stdlib.h>

#include <mutex>

namespace moe {
namespace {

constexpr int BM = kTcBM;  // 128 rows (TMEM lanes)
constexpr int BN = 256;    // accumulator columns per tile
constexpr int BK = 64;     // K per stage
constexpr int STAGES = 4;
constexpr int kThreads = 192;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BK * BN * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;

struct BParams {
  int mode;
  int K;          // modes 0, 1: reduction length
  int N;          // output columns
  int M;          // mode 2: output rows per expert
  int E, n_blocks, m_blocks;
  const int32_t *offset;  // [E+1] the forward's packed row offsets
  const int32_t *poff;    // [E+1] padded row offsets
  const float *row_gate;  // mode 0: [packed rows]
  const __nv_bfloat16 *hbuf;  // mode 0: [packed rows, N]
  void *out;      // mode 0: bf16 [padded rows, N]; mode 1: fp32 [padded rows, N];
                  // mode 2: fp32 [E, M, N]
  float *dgpart;  // mode 0: [padded rows, n_blocks]
  DeviceStatus *st;
  unsigned long long wait_ns;
  uint32_t *sched;  // [2] the CTA-pair kernel's tile counter and done count (zero at launch)
  int dynamic;      // CTA-pair kernel: tiles from the counter (else round robin)
  int tma_out;      // CTA-pair kernel, modes 0 and 1: 32-row groups leave by TMA store
  int snake;        // CTA-pair kernel: 1 = odd waves of tiles run K backwards, 2 = all do
};

// The CTA-pair kernel's tile ring, as in the forward expert GEMM: tile
// indices from the even CTA's producer to the MMA issuer, both CTAs'
// epilogue warps and the odd CTA's producer (ten arrivals free a slot).
constexpr int kRing = 8;
constexpr int kRingConsumers = 10;

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M = 128,
// N = 256; bits 15 / 16 select MN-major A / B.
template <int MODE>
__host__ __device__ constexpr uint32_t bwd_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((MODE == 2 ? 1u : 0u) << 15) |
         ((MODE == 2 ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

template <int MODE>
__device__ __forceinline__ void umma_b(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(bwd_idesc<MODE>()), "r"(acc)
      : "memory");
}

// Tile -> (expert, m block, n block), the expert's first padded row, its
// padded and real row counts, and the number of K blocks.
struct BTile {
  int e, mb, nb, prow0, prows, rows, num_kb;
};

// Weight-gradient tiles of one expert: the blocks of the operand with fewer
// of them run fastest, so the CTAs working at the same time share the larger
// operand's block and the expert's smaller operand stays whole in L2 (dW2:
// 56 blocks of h columns and 16 of dU at the large-expert widths).
__device__ __forceinline__ void wgrad_order(int local, int m_blocks, int n_blocks, int &mb,
                                            int &nb) {
  if (m_blocks <= n_blocks) {
    nb = local / m_blocks;
    mb = local - nb * m_blocks;
  } else {
    mb = local / n_blocks;
    nb = local - mb * n_blocks;
  }
}

template <int MODE>
__device__ __forceinline__ BTile locate(const BParams &p, const int *start, int tile) {
  BTile t;
  if (MODE == 2) {
    const int per = p.m_blocks * p.n_blocks;
    t.e = tile / per;
    const int local = tile - t.e * per;
    wgrad_order(local, p.m_blocks, p.n_blocks, t.mb, t.nb);
  } else {
    int lo = 0, hi = p.E;  // largest e with start[e] <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    t.e = lo;
  }
  t.prow0 = p.poff[t.e];
  t.prows = p.poff[t.e + 1] - t.prow0;
  t.rows = p.offset[t.e + 1] - p.offset[t.e];
  if (MODE != 2) {
    const int mt = (t.prows + BM - 1) / BM;
    const int local = tile - start[t.e];
    t.nb = local / mt;
    t.mb = local - t.nb * mt;
    t.num_kb = p.K / BK;
  } else {
    t.num_kb = t.prows / BK;
  }
  return t;
}

// One lane's row m of a finished tile: 32 accumulator columns at a time from
// TMEM (lane_addr: this warp's lanes, this accumulator), stored as the mode
// asks. Warp-collective (every lane loads). Modes 0 and 1 in the CTA-pair
// kernel pass stg (the warp's two staging tiles), tmO (the output [padded
// rows, N]) and cnt: the warp's 32 rows, inside the expert's padded block
// (its size is a multiple of 64), then leave by TMA store, mode 1's pad rows
// included (zero, as dpre's pad rows are).
template <int MODE>
__device__ __forceinline__ void epilogue_rows(const BParams &p, const BTile &t, int m,
                                              uint32_t lane_addr, float *stg = nullptr,
                                              const CUtensorMap *tmO = nullptr,
                                              uint32_t *cnt = nullptr) {
  const int m0 = m - (int)(threadIdx.x & 31);  // the warp's first row
  const bool tma = MODE != 2 && stg != nullptr && m0 + 32 <= t.prows;
  // Rows this lane writes: mode 0 every padded row of the expert (pad rows
  // as zero), mode 1 the real rows (every padded row through TMA), mode 2 the
  // output rows m < M.
  const bool valid = MODE == 0 ? m < t.prows
                     : MODE == 1 ? (tma || m < t.rows)
                                 : m < p.M;
  const bool real = m < t.rows;
  const size_t pr = (size_t)t.prow0 + m;
  const size_t q = (size_t)p.offset[t.e] + m;
  const float g = (MODE == 0 && valid && real) ? p.row_gate[q] : 0.f;
  float part = 0.f;
  bool bad = false;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int n = t.nb * BN + c * 32;
    uint32_t v[32];
    tmem_ld32(lane_addr + (uint32_t)(c * 32), v);  // warp-collective
    if (!valid || n >= p.N) continue;
    if (MODE == 0) {
      float h[32];
      if (real) {
        const uint4 *hp = reinterpret_cast<const uint4 *>(p.hbuf + q * p.N + n);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 u = hp[w];
          const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&uu[j]);
            h[8 * w + 2 * j] = __low2float(b2);
            h[8 * w + 2 * j + 1] = __high2float(b2);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = 0.f;
      }
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float d0 = __uint_as_float(v[2 * j]), d1 = __uint_as_float(v[2 * j + 1]);
        part = fmaf(d0, h[2 * j], part);
        part = fmaf(d1, h[2 * j + 1], part);
        const float p0 = h[2 * j] > 0.f ? g * d0 : 0.f;
        const float p1 = h[2 * j + 1] > 0.f ? g * d1 : 0.f;
        bad |= !isfinite(p0) || !isfinite(p1);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        packed[j] = *reinterpret_cast<uint32_t *>(&b2);
      }
      if (tma) {
        stage_store_bf16(tmO, stg + (*cnt & 1u) * 1024, packed, n, t.prow0 + m0);
        ++*cnt;
      } else {
        uint4 *o =
            reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + pr * p.N + n);
#pragma unroll
        for (int w = 0; w < 4; ++w)
          o[w] = make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2],
                            packed[4 * w + 3]);
      }
    } else {
      float f[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        f[j] = __uint_as_float(v[j]);
        bad |= !isfinite(f[j]);
      }
      if (tma) {
        stage_store_f32(tmO, stg + (*cnt & 1u) * 1024, f, n, t.prow0 + m0);
        ++*cnt;
      } else {
        float *o = MODE == 1
                       ? static_cast<float *>(p.out) + pr * p.N + n
                       : static_cast<float *>(p.out) + ((size_t)t.e * p.M + m) * p.N + n;
#pragma unroll
        for (int w = 0; w < 8; ++w)
          reinterpret_cast<float4 *>(o)[w] =
              make_float4(f[4 * w], f[4 * w + 1], f[4 * w + 2], f[4 * w + 3]);
      }
    }
  }
  if (MODE == 0 && valid) p.dgpart[pr * p.n_blocks + t.nb] = part;
  if (bad) record_error(p.st, MOE_ERR_NONFINITE, (long long)(MODE == 2 ? m : (long long)pr));
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
         const BParams p) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
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
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Dgrad modes: tile prefix over experts, ceil(padded rows / BM) * n_blocks each.
  if (MODE != 2 && warp == 2) {
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < p.E) t = (p.poff[e + 1] - p.poff[e] + BM - 1) / BM * p.n_blocks;
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
  const int total_tiles = MODE == 2 ? p.E * p.m_blocks * p.n_blocks : tile_start[p.E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- producer
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const BTile t = locate<MODE>(p, tile_start, tile);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 31, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], STAGE_BYTES);
          if (MODE != 2) {
            tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * BK, t.prow0 + t.mb * BM);
            tma_load_2d(sB + s * B_BYTES, &tmB, &full[s], kb * BK, t.e * p.N + t.nb * BN);
          } else {
            const int arow = p.offset[t.e] + kb * BK, brow = t.prow0 + kb * BK;
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_2d(sA + s * A_BYTES + j * (BK * 128), &tmA, &full[s], t.mb * BM + j * 64,
                          arow);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sB + s * B_BYTES + j * (BK * 128), &tmB, &full[s], t.nb * BN + j * 64,
                          brow);
          }
        }
      }
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)STAGES ? issued - STAGES : 0; q < issued; ++q)
        mbar_drain(&full[q % STAGES], (q / STAGES) & 1u);
    }
    __syncwarp();
    pdl_trigger();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA issuer
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++local) {
        const BTile t = locate<MODE>(p, tile_start, tile);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 32, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 33, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            uint64_t ad, bd;
            if (MODE != 2) {
              ad = sdesc(a0 + kk * 32, 16, 1024);
              bd = sdesc(b0 + kk * 32, 16, 1024);
            } else {
              ad = sdesc(a0 + kk * 2048, BK * 128, 1024);
              bd = sdesc(b0 + kk * 2048, BK * 128, 1024);
            }
            umma_b<MODE>(tmem_d, ad, bd, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
    pdl_trigger();
  } else {
    // ----------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int r_in_tile = quad * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
      const BTile t = locate<MODE>(p, tile_start, tile);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 34, p.wait_ns));
      if (!ready) break;
      tc_fence_after();
      const int m = t.mb * BM + r_in_tile;
      epilogue_rows<MODE>(p, t, m, tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)(buf * BN));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
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
// The same three modes with tcgen05.mma.cta_group::2: a cluster of two CTAs
// on two SMs computes a 256-row x 256-column tile; each CTA loads its own 128
// rows of A and 128 of the tile's 256 B columns (rows of the K-major weight
// in the dgrad modes, 64-column boxes of the MN-major rows in the weight
// gradient), so each SM takes in 32 KB per K step instead of 48 KB. The even
// CTA issues the MMAs; the odd CTA's copies complete on the even CTA's "full"
// barriers, commits arrive on both CTAs' barriers, and both CTAs' epilogues
// arrive on the even CTA's "accumulator empty" barriers (the forward's pair
// kernel, same protocol).
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = BM * BK * 2;          // 16 KB
constexpr int P_B_BYTES = BK * (BN / 2) * 2;    // 16 KB
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
// Weight-gradient epilogue staging: per epilogue warp two [32 rows x 32
// columns] fp32 tiles (4 KB each) in the 128-byte swizzle.
constexpr int P_STG_TILE = 32 * 32;  // floats
constexpr int P_STG_BYTES = 4 * 2 * P_STG_TILE * 4;

template <int MODE>
__host__ __device__ constexpr uint32_t bwd_idesc_pair() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((MODE == 2 ? 1u : 0u) << 15) |
         ((MODE == 2 ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(256 >> 4) << 24);
}

template <int MODE>
__device__ __forceinline__ void umma_b_pair(uint32_t tmem_d, uint64_t a, uint64_t b,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(bwd_idesc_pair<MODE>()), "r"(acc)
      : "memory");
}

// Pair tiles: dgrad modes over (expert, 256-row block, n block) with
// ceil(padded rows / 256) row blocks per expert; weight gradient over (expert,
// n block, 256-row block of the output) with ceil(M / 256) row blocks.
template <int MODE>
__device__ __forceinline__ BTile locate_pair(const BParams &p, const int *start, int tile) {
  BTile t;
  const int mb2 = (p.M + 2 * BM - 1) / (2 * BM);
  if (MODE == 2) {
    const int per = mb2 * p.n_blocks;
    t.e = tile / per;
    const int local = tile - t.e * per;
    wgrad_order(local, mb2, p.n_blocks, t.mb, t.nb);
  } else {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    t.e = lo;
  }
  t.prow0 = p.poff[t.e];
  t.prows = p.poff[t.e + 1] - t.prow0;
  t.rows = p.offset[t.e + 1] - p.offset[t.e];
  if (MODE != 2) {
    const int mt = (t.prows + 2 * BM - 1) / (2 * BM);
    const int local = tile - start[t.e];
    t.nb = local / mt;
    t.mb = local - t.nb * mt;
    t.num_kb = p.K / BK;
  } else {
    t.num_kb = t.prows / BK;
  }
  return t;
}

// The weight-gradient epilogue of the CTA-pair kernel: this warp's 32 rows
// m0 .. m0+31 of expert e's dW tile, 32 columns at a time from TMEM into one
// of the warp's two staging tiles, then out by a TMA store into dW viewed as
// [E, M, N] (tmO), which drops rows past M and columns past N. The per-lane
// row stores of the other modes send 32 rows' 16-byte pieces per instruction;
// here each store writes whole 128-byte row segments, and the fp32 output
// (4 bytes per product of a K = rows-per-expert reduction) no longer holds
// the tensor pipe back. cnt counts this warp's staged chunks (buffer parity).
__device__ __forceinline__ void epilogue_wgrad_tma(const BParams &p, const BTile &t, int m0,
                                                   uint32_t lane_addr, float *stg,
                                                   const CUtensorMap *tmO, uint32_t &cnt) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int n = t.nb * BN + c * 32;
    uint32_t v[32];
    tmem_ld32(lane_addr + (uint32_t)(c * 32), v);  // warp-collective
    if (n >= p.N) continue;
    float *buf = stg + (cnt & 1u) * P_STG_TILE;
    if (lane == 0) bulk_wait_read_but1();  // this buffer's previous store has read it
    __syncwarp();
    float4 *row = reinterpret_cast<float4 *>(buf + lane * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      bad |= !isfinite(f.x) || !isfinite(f.y) || !isfinite(f.z) || !isfinite(f.w);
      row[q ^ (lane & 7)] = f;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmO, buf, n, m0, t.e);
      bulk_commit();
    }
    ++cnt;
  }
  if (bad && m0 + lane < p.M) record_error(p.st, MOE_ERR_NONFINITE, (long long)(m0 + lane));
}

// tmO: mode 2's output dW as [E, M, N] fp32, box [1, 32, 32], 128-byte
// swizzle; modes 0 and 1: the output [padded rows, N] (bf16 / fp32), box [32,
// 32], when p.tma_out is set.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_bwd_tc_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmO, const BParams p) {
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
  uint64_t *tfull = drain + 1, *tempty = tfull + kRing;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + kRing);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *ring = reinterpret_cast<volatile int *>(tmem_slot + 2);
  int *tile_start = const_cast<int *>(ring + kRing);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&tfull[r], 1);
      mbar_init(&tempty[r], kRingConsumers);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (MODE != 2 && warp == 2) {  // ceil(padded rows / 256) * n_blocks tiles per expert
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int t = 0;
      if (e < p.E) t = (p.poff[e + 1] - p.poff[e] + 2 * BM - 1) / (2 * BM) * p.n_blocks;
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
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int mb2 = (p.M + 2 * BM - 1) / (2 * BM);
  const int total_tiles = MODE == 2 ? p.E * mb2 * p.n_blocks : tile_start[p.E];

  if (warp == 0) {
    if (lane == 0) {
      // --------------------------------------------------------- producer (both CTAs)
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      // Tiles: each pair's first is its index, every later one taken from the
      // counter by the even CTA's producer (the take issued a few k-blocks
      // before the current tile's last load) and published through the ring.
      uint32_t it = 0;
      bool ok = true;
      long long taken = -1;
      int tile_rr = pair;
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
          if (!mbar_wait_cl(&tempty[slot], rph ^ 1u, abort_flag, p.st, 45, p.wait_ns)) {
            ok = false;
            break;
          }
          ring[slot] = tile;
          st_cluster_u32(mapa(smem_u32((const void *)&ring[slot]), 1), (uint32_t)tile);
          mbar_arrive_cluster(smem_u32(&tfull[slot]));
          mbar_arrive_cluster(mapa(smem_u32(&tfull[slot]), 1));
        } else {
          if (!mbar_wait_cl(&tfull[slot], rph, abort_flag, p.st, 46, p.wait_ns)) {
            ok = false;
            break;
          }
          tile = ring[slot];
          mbar_arrive_cluster(mapa(smem_u32(&tempty[slot]), 0));
        }
        if (tile >= total_tiles) break;
        const BTile t = locate_pair<MODE>(p, tile_start, tile);
        const int take_at = t.num_kb > 4 ? t.num_kb - 4 : 0;
        // Odd waves of tiles walk K from the end, starting on the blocks the
        // wave before read last (still in L2); the order is fixed per tile.
        const bool rev = p.snake == 2 || (p.snake == 1 && ((tile / n_pairs) & 1));
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          if (leader && p.dynamic && kb == take_at) taken = atomicAdd(p.sched, 1u);
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 41, p.wait_ns)) {
            ok = false;
            break;
          }
          const int kx = (rev ? t.num_kb - 1 - kb : kb) * BK;
          const uint32_t full_leader = mapa(smem_u32(&full[s]), 0);
          if (leader) mbar_expect_tx(&full[s], 2 * P_STAGE_BYTES);
          if (MODE != 2) {
            tma_load_2d_pair(sA + s * P_A_BYTES, &tmA, full_leader, kx,
                             t.prow0 + t.mb * 2 * BM + (int)rank * BM);
            tma_load_2d_pair(sB + s * P_B_BYTES, &tmB, full_leader, kx,
                             t.e * p.N + t.nb * BN + (int)rank * (BN / 2));
          } else {
            const int arow = p.offset[t.e] + kx, brow = t.prow0 + kx;
            const int mcol = t.mb * 2 * BM + (int)rank * BM;
            const int ncol = t.nb * BN + (int)rank * (BN / 2);
#pragma unroll
            for (int q = 0; q < BM / 64; ++q)
              tma_load_2d_pair(sA + s * P_A_BYTES + q * (BK * 128), &tmA, full_leader,
                               mcol + q * 64, arow);
#pragma unroll
            for (int q = 0; q < (BN / 2) / 64; ++q)
              tma_load_2d_pair(sB + s * P_B_BYTES + q * (BK * 128), &tmB, full_leader,
                               ncol + q * 64, brow);
          }
        }
      }
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)P_STAGES ? issued - P_STAGES : 0; q < issued; ++q)
        mbar_drain(&empty[q % P_STAGES], (q / P_STAGES) & 1u);
      if (leader && p.dynamic) {
        // The last pair to finish resets the counter for the next launch.
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == (uint32_t)n_pairs - 1) {
          atomicExch(p.sched, 0u);
          atomicExch(p.sched + 1, 0u);
        }
      }
    }
    __syncwarp();
    pdl_trigger();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // --------------------------------------------------------- MMA issuer (even CTA)
      uint32_t it = 0;
      bool ok = true;
      for (int local = 0; ok; ++local) {
        const int slot = local % kRing;
        if (!mbar_wait_cl(&tfull[slot], (uint32_t)(local / kRing) & 1u, abort_flag, p.st, 47,
                          p.wait_ns))
          break;
        const int tile = ring[slot];
        mbar_arrive_cluster(smem_u32(&tempty[slot]));
        if (tile >= total_tiles) break;
        const BTile t = locate_pair<MODE>(p, tile_start, tile);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 42, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % P_STAGES;
          const uint32_t ph = (it / P_STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 43, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * P_A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * P_B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            uint64_t ad, bd;
            if (MODE != 2) {
              ad = sdesc(a0 + kk * 32, 16, 1024);
              bd = sdesc(b0 + kk * 32, 16, 1024);
            } else {
              ad = sdesc(a0 + kk * 2048, BK * 128, 1024);
              bd = sdesc(b0 + kk * 2048, BK * 128, 1024);
            }
            umma_b_pair<MODE>(tmem_d, ad, bd, (kb | kk) ? 1u : 0u);
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
    uint32_t stg_cnt = 0;
    for (int local = 0;; ++local) {
      const int slot = local % kRing;
      int tile = total_tiles;
      bool got = false;
      if (lane == 0) {
        got = mbar_wait_cl(&tfull[slot], (uint32_t)(local / kRing) & 1u, abort_flag, p.st, 48,
                           p.wait_ns);
        if (got) {
          tile = ring[slot];
          mbar_arrive_cluster(mapa(smem_u32(&tempty[slot]), 0));
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (!got || tile >= total_tiles) break;
      const BTile t = locate_pair<MODE>(p, tile_start, tile);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 44, p.wait_ns));
      if (!ready) break;
      tc_fence_after();
      const int m = t.mb * 2 * BM + (int)rank * BM + r_in_tile;
      const uint32_t lane_addr =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN);
      if constexpr (MODE == 2)
        epilogue_wgrad_tma(p, t, m - lane, lane_addr, stg, &tmO, stg_cnt);
      else
        epilogue_rows<MODE>(p, t, m, lane_addr, p.tma_out ? stg : nullptr, &tmO, &stg_cnt);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(buf ? acc_empty_leader1 : acc_empty_leader0);
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores are complete
    pdl_trigger();
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

constexpr size_t bwd_smem_bytes_pair(int E, int mode) {
  (void)mode;
  return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_STG_BYTES +
         (2 * P_STAGES + 5 + 2 * kRing) * 8 + 8 + (size_t)kRing * 4 + (size_t)(E + 1) * 4;
}

constexpr size_t bwd_smem_bytes(int E) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + (2 * STAGES + 5) * 8 + 8 + (size_t)(E + 1) * 4;
}

cudaLaunchAttribute cluster2_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Clusters of two the pair kernel of this mode can keep resident (0 if none),
// for the shared-memory size of this E; looked up once per (mode, size).
template <int MODE>
int pair_clusters_bwd(size_t smem) {
  constexpr int kSlots = 8;
  static std::mutex mu;
  static size_t keys[kSlots];
  static int vals[kSlots];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == smem) return vals[i];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count() / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1] = {cluster2_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(k_bwd_tc_pair<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k_bwd_tc_pair<MODE>, &cfg) != cudaSuccess) {
    n = 0;
    cudaGetLastError();
  }
  if (used < kSlots) {
    keys[used] = smem;
    vals[used] = n;
    ++used;
  }
  return n;
}

template <int MODE>
cudaError_t launch_mode_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                             const BParams &p, int clusters, cudaStream_t s) {
  const size_t smem = bwd_smem_bytes_pair(p.E, MODE);
  cudaError_t err = cudaFuncSetAttribute(
      k_bwd_tc_pair<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2] = {cluster2_attr(), {}};
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled(kPdlGemm) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_bwd_tc_pair<MODE>, a, b, o, p);
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap &a, const CUtensorMap &b, const BParams &p,
                        cudaStream_t s) {
  const size_t smem = bwd_smem_bytes(p.E);
  cudaError_t err = cudaFuncSetAttribute(k_bwd_tc<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  launch_pdl_c(kPdlGemm, k_bwd_tc<MODE>, sm_count(), kThreads, smem, s, a, b, p);
  return cudaGetLastError();
}

// 3-D fp32 tensor [E, M, N] (N % 4 == 0): the weight gradient, box [1, 32
// rows, 32 columns] in the 128-byte swizzle, for the CTA-pair kernel's TMA
// stores (rows past M and columns past N of a box are not written).
bool make_out_map3(CUtensorMap *m, float *base, int E, int M, int N) {
  auto fn = encode_fn();
  if (!fn || N % 4 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)M * N * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace

bool bwd_tc_supported(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0 &&
         bwd_smem_bytes(c.E) <= 227 * 1024 && encode_fn() != nullptr;
}

// MOE_BWD_TC_VARIANT=single or =pair forces one kernel (read at each call);
// otherwise the CTA pair runs where its reduction is long (K >= 1024; for the
// weight gradient, the rows per expert, bounded by the capacity) and it has
// at least four waves of 256 x 256 tiles.
static int bwd_variant() {
  const char *v = getenv("MOE_BWD_TC_VARIANT");
  if (!v || !*v) return 0;
  return v[0] == 's' ? 1 : (v[0] == 'p' ? 2 : 0);
}

template <int MODE>
static int pick_pair(const BwdGemm &g, long long k_len, long long tiles) {
  const int force = bwd_variant();
  if (force == 1 || bwd_smem_bytes_pair(g.E, MODE) > 227 * 1024) return 0;
  const int clusters = pair_clusters_bwd<MODE>(bwd_smem_bytes_pair(g.E, MODE));
  if (clusters <= 0) return 0;
  if (force == 2) return clusters;
  return (k_len >= 1024 && tiles >= 4LL * clusters) ? clusters : 0;
}

cudaError_t launch_bwd_gemm(const BwdGemm &g, DeviceStatus *st, cudaStream_t s) {
  CUtensorMap ta, tb;
  BParams p{};
  p.mode = g.mode;
  p.K = g.K;
  p.N = g.N;
  p.M = g.M;
  p.E = g.E;
  p.n_blocks = (g.N + BN - 1) / BN;
  p.m_blocks = (g.M + BM - 1) / BM;
  p.offset = g.offset;
  p.poff = g.poff;
  p.row_gate = g.row_gate;
  p.hbuf = static_cast<const __nv_bfloat16 *>(g.hbuf);
  p.out = g.out;
  p.dgpart = g.dgpart;
  p.st = st;
  p.wait_ns = wait_limit_ns();
  p.sched = &st->gemm_next;  // gemm_next, gemm_done: adjacent words
  {
    const char *v = getenv("MOE_FFN_SCHED");  // =static: round robin (for comparisons)
    p.dynamic = v && v[0] == 's' ? 0 : 1;
    // =0: every tile's K forward, =all: every tile's backwards (comparisons, tests)
    const char *sv = getenv("MOE_FFN_SNAKE");
    p.snake = !sv || !*sv ? 1 : (sv[0] == '0' ? 0 : (sv[0] == 'a' ? 2 : 1));
  }
  const long long nb = (g.N + BN - 1) / BN;
  if (g.mode == 2) {
    // A: the forward's packed rows [a_rows, M]; B: padded rows [b_rows, N].
    if (!make_map(&ta, g.A, (uint64_t)g.a_rows, (uint64_t)g.M, 64) ||
        !make_map(&tb, g.B, (uint64_t)g.b_rows, (uint64_t)g.N, 64))
      return cudaErrorInvalidValue;
    const int cl = pick_pair<2>(g, g.k_len, (long long)g.E * ((g.M + 255) / 256) * nb);
    CUtensorMap to;
    if (cl > 0 && (uintptr_t)g.out % 16 == 0 &&
        make_out_map3(&to, static_cast<float *>(g.out), g.E, g.M, g.N))
      return launch_mode_pair<2>(ta, tb, to, p, cl, s);
    return launch_mode<2>(ta, tb, p, s);
  }
  // A: padded rows [a_rows, K]; B: the weight as [E*N rows, K] (the pair
  // kernel loads half of a tile's 256 B rows per CTA).
  const long long tiles = (g.a_rows + 255) / 256 * nb;
  const int cl = g.mode == 0 ? pick_pair<0>(g, g.K, tiles) : pick_pair<1>(g, g.K, tiles);
  if (!make_map(&ta, g.A, (uint64_t)g.a_rows, (uint64_t)g.K, BM) ||
      !make_map(&tb, g.B, (uint64_t)g.E * g.N, (uint64_t)g.K, cl > 0 ? BN / 2 : BN))
    return cudaErrorInvalidValue;
  if (cl > 0) {
    CUtensorMap to = ta;  // unused unless p.tma_out
    p.tma_out = make_rows_map(&to, g.out, (uint64_t)g.a_rows, (uint64_t)g.N, g.mode == 1) ? 1 : 0;
    return g.mode == 0 ? launch_mode_pair<0>(ta, tb, to, p, cl, s)
                       : launch_mode_pair<1>(ta, tb, to, p, cl, s);
  }
  return g.mode == 0 ? launch_mode<0>(ta, tb, p, s) : launch_mode<1>(ta, tb, p, s);
}

}  // namespace moe
