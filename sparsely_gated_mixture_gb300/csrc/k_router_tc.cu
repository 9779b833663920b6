// Stage 1 router on the tensor cores ("Outrageously Large", Noisy Top-K
// Gating step 1, Eq. 4; "Switch Transformer", step 1: the router is fp32).
//
// x is bf16, so every product x_i * W[i,e] is exact once W is written as the
// sum of three bf16 pieces: hi = bf16(W), mid = bf16(W - hi), lo = bf16(W -
// hi - mid), with W = hi + mid + lo exactly (each piece carries 8 of fp32's
// 24 significand bits; the differences are exact in fp32). The router is then
// three bf16 GEMMs, x * hi + x * mid + x * lo, accumulated in fp32 in TMEM:
// the fp32 router's arithmetic at the tensor cores' rate.
//
// k_router_split builds the pieces, transposed so that each B row is one
// output column (K contiguous): columns 2e and 2e+1 are expert e's clean and
// noise logits (noisy gate) or column e is expert e (no noise); each block of
// BNR columns holds its hi, mid and lo rows back to back, and the columns are
// padded with zero rows to a whole number of blocks.
// k_router_tc is one persistent CTA per SM: a TMA warp loads x [128 tokens x
// 64 K] and the [3*BNR rows x 64 K] B box (the three pieces) per stage
// (BNR <= 64), one lane issues 4 tcgen05.mma (M=128, N=3*BNR, K=16, both
// operands K-major, 128B swizzle) into one of two TMEM accumulators, whose
// three BNR-wide sections are summed per column, and eight epilogue
// warps (two per TMEM lane quadrant) turn each token's columns into
// c = acc + b, sigma = Softplus(z) and H = c + noise * sigma, 16 accumulator
// columns at a time: 8 experts with the noise term (clean/noise pairs), whose
// [32 tokens x 8 experts] fp32 tiles of c, sigma and H go to shared memory
// (32-byte swizzle) and out with one TMA store each; 16 experts without it,
// where only H is written ([32 x 16], 64-byte swizzle; c = H, sigma = 0). Rows
// of E floats that are not 16-byte multiples (E % 4 != 0) take a staged store
// per row segment, on one warp per quadrant.
#include "gate_math.cuh"
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

#include <stdlib.h>

namespace moe {
namespace {

constexpr int RBM = 128, RBK = 64;
constexpr int kREpiWarps = 8;  // two per TMEM lane quadrant, taking 16-column units in turn
constexpr int kRThreads = 64 + 32 * kREpiWarps;

struct RParams {
  int T, d, E, noisy, NC, NCP, n_blocks, tma_out;
  const float *noise, *bias;
  float *c_out, *s_out, *H_out;
  DeviceStatus *st;
  unsigned long long wait_ns;  // bounded-wait limit
  // Fused selection (one column block, one tile per CTA): k, gate mode and
  // the selection outputs; partials may be null (no balancing sums).
  int fused, k, mode;
  int32_t *idx;
  float *gate, *thr, *rowstat, *partials;
};

// Softplus(z) = max(z, 0) + log1p(t), t = exp(-|z|) in (0, 1]. log1p(t) is
// 2 atanh(s) with s = t / (2 + t) in [0, 1/3], summed as the odd series
// 2 s (1 + s^2/3 + s^4/5 + ... + s^12/13): the truncation is below 2^-26
// relative, and in fp32 the result matches log1pf(expf(-|z|)) to within a few
// ulps (max 3.4 vs 3.0 ulps of Softplus against the exact value).
__device__ __forceinline__ float softplus_r(float z) {
  const float t = expf(-fabsf(z));
  const float sv = __fdividef(t, 2.f + t);
  const float s2 = sv * sv;
  float q = 1.f / 13.f;
  q = fmaf(s2, q, 1.f / 11.f);
  q = fmaf(s2, q, 1.f / 9.f);
  q = fmaf(s2, q, 1.f / 7.f);
  q = fmaf(s2, q, 1.f / 5.f);
  q = fmaf(s2, q, 1.f / 3.f);
  q = fmaf(s2, q, 1.f);
  return fmaxf(z, 0.0f) + 2.f * sv * q;
}

// Row l of a [32 x 8] fp32 tile in the 32-byte swizzle of the TMA store:
// 16-byte chunk q of row l sits at chunk q ^ ((l >> 2) & 1).
__device__ __forceinline__ void tile_row_store8(float *tile, int l, const float *v) {
  float4 *row = reinterpret_cast<float4 *>(tile + l * 8);
  const int x = (l >> 2) & 1;
  row[x] = make_float4(v[0], v[1], v[2], v[3]);
  row[1 ^ x] = make_float4(v[4], v[5], v[6], v[7]);
}

// Row l of a [32 x 16] fp32 tile in the 64-byte swizzle of the TMA store:
// 16-byte chunk q of row l sits at chunk q ^ ((l >> 1) & 3).
__device__ __forceinline__ void tile_row_store(float *tile, int l, const float *v) {
  float4 *row = reinterpret_cast<float4 *>(tile + l * 16);
  const int x = (l >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    row[q ^ x] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// grid (ceil(d/32), ceil(NCP/32)), block (32, 8): a 32 x 32 transpose tile.
// Output rows are grouped per column block of BNR: block b holds hi rows,
// then mid rows, then lo rows of its BNR columns, so one TMA box of 3*BNR rows
// brings all three pieces of a block.
// It runs first in the gate, so it also clears the status word (after its
// dependent-launch wait, before any later kernel can record an error).
__global__ void k_router_split(int d, int E, int noisy, int NC, int NCP, int BNR,
                               const float *__restrict__ Wg, const float *__restrict__ Wn,
                               __nv_bfloat16 *__restrict__ B, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) {
    st->code = 0;
    st->aux_ticket = 0;
    st->detail = 0;
    st->slot_ticket = 0;
    st->reserved = 0;
    st->gemm_next = 0;
    st->gemm_done = 0;
  }
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int k = k0 + r, n = n0 + threadIdx.x;
    float w = 0.f;
    if (k < d && n < NC) {
      const int e = noisy ? n >> 1 : n;
      const float *src = (noisy && (n & 1)) ? Wn : Wg;
      w = src[(size_t)k * E + e];
    }
    tile[r][threadIdx.x] = w;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int n = n0 + r, k = k0 + threadIdx.x;
    if (n >= NCP || k >= d) continue;
    const float w = tile[threadIdx.x][r];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    const size_t row0 = (size_t)(n / BNR) * 3 * BNR + (n % BNR);
    B[(row0 + 0 * (size_t)BNR) * d + k] = hi;
    B[(row0 + 1 * (size_t)BNR) * d + k] = mid;
    B[(row0 + 2 * (size_t)BNR) * d + k] = lo;
  }
}

// Epilogue staging, 24 KB (kept small so that more pipeline stages fit:
// the mainloop is bound by how many bytes are in flight). TMA-store path: per
// epilogue warp 3 KB, three [32 x 8] fp32 tiles (c, sigma, H) or one [32 x 16]
// H tile. Row-segment path: per warp of the first of each quadrant, 6 KB,
// three [32 rows x 16 experts] tiles with columns XOR-swizzled by row.
constexpr int kEpiTile = 32 * 16;
constexpr int kEpiWarpFloats = 3 * 32 * 8;  // TMA-store path, per warp
constexpr int EPI_BYTES = 4 * 3 * kEpiTile * 4;
static_assert(kREpiWarps * kEpiWarpFloats * 4 <= EPI_BYTES, "staging");

template <int BNR>
struct RCfg {
  static constexpr int A_BYTES = RBM * RBK * 2;  // 16 KB
  static constexpr int NB = 3 * BNR;              // MMA N: the three pieces side by side
  static constexpr int B_BYTES = NB * RBK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int FIT = (227 * 1024 - 1024 - EPI_BYTES - 256) / STAGE;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int TMEM_COLS = 2 * NB <= 64 ? 64 : (2 * NB <= 128 ? 128 : (2 * NB <= 256 ? 256 : 512));
  // kind::f16: fp32 accumulate, bf16 A and B, both K-major, M = 128, N = 3*BNR.
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                                    ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(RBM >> 4) << 24);
  static constexpr size_t SMEM =
      1024 + (size_t)STAGES * STAGE + EPI_BYTES + (2 * STAGES + 5) * 8 + 8;
  static_assert(STAGES >= 2, "router tile too wide for two pipeline stages");
};

template <int BNR>
__device__ __forceinline__ void umma_r(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(RCfg<BNR>::IDESC), "r"(acc)
      : "memory");
}

// Epilogue for up to 16 experts e0 .. e0+ne-1 of the warp's 32 tokens t0 ..
// t0+31. Lane l holds token t0+l's clean logits cv[], noise logits zv[] and
// noise draws nz[] (noisy gate) in registers; c, sigma and H go through the
// warp's staging tiles so that each store instruction writes two tokens'
// 16-expert row segments.
__device__ __forceinline__ int swz(int row, int col) { return row * 16 + (col ^ (row & 15)); }

__device__ __forceinline__ void router_rows(const RParams &p, int t0, int e0, int ne,
                                            const float *cv, const float *zv, const float *nz,
                                            float *stg) {
  const int lane = threadIdx.x & 31;
  float *sc = stg, *ss = stg + kEpiTile, *sh = stg + 2 * kEpiTile;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float c = cv[j];
    if (p.bias && j < ne) c += p.bias[e0 + j];
    float sg = 0.f, h = c;
    if (p.noisy && j < 8) {
      sg = softplus_r(zv[j]);
      h = fmaf(nz[j], sg, c);
    }
    sc[swz(lane, j)] = c;
    ss[swz(lane, j)] = sg;
    sh[swz(lane, j)] = h;
  }
  __syncwarp();
  const int half = lane >> 4, col = lane & 15;
  bool bad = false;
#pragma unroll 4
  for (int r = 0; r < 32; r += 2) {
    const int row = r + half, t = t0 + row;
    if (t < p.T && col < ne) {
      const size_t o = (size_t)t * p.E + e0 + col;
      const float h = sh[swz(row, col)];
      p.c_out[o] = sc[swz(row, col)];
      p.s_out[o] = ss[swz(row, col)];
      p.H_out[o] = h;
      bad |= !isfinite(h);
    }
  }
  if (bad) record_error(p.st, MOE_ERR_NONFINITE, (long long)t0);
  __syncwarp();
}

// Token t's noise draws for experts e0 .. e0+7 (zero past E or T).
__device__ __forceinline__ void load_noise8(const RParams &p, int t, int e0, float *nz) {
  if (t < p.T && (p.E & 3) == 0 && e0 + 8 <= p.E) {
    const float4 *src = reinterpret_cast<const float4 *>(p.noise + (size_t)t * p.E + e0);
    const float4 a = src[0], b = src[1];
    nz[0] = a.x; nz[1] = a.y; nz[2] = a.z; nz[3] = a.w;
    nz[4] = b.x; nz[5] = b.y; nz[6] = b.z; nz[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      nz[j] = (t < p.T && e0 + j < p.E) ? p.noise[(size_t)t * p.E + e0 + j] : 0.f;
  }
}

// The biases of experts e0 .. e0+n-1 (n <= 16; zero past E, past n or
// without a bias) for an epilogue unit; every lane loads the same values.
__device__ __forceinline__ void load_bias_n(const RParams &p, int e0, int n, float (&b)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) b[j] = (p.bias && j < n && e0 + j < p.E) ? p.bias[e0 + j] : 0.f;
}

// One unit of the TMA-store epilogue with the noise term: experts e0 .. e0+7
// of tokens t0 .. t0+31 (lane l = token t0 + l). cv holds the clean logits and
// zv the noise logits on entry, bu the unit's biases; c, sigma and H are
// computed in registers, then (once this warp's previous stores have read its
// staging tiles) written as three [32 x 8] tiles and stored by TMA.
// With fused selection, row points at this lane's token row in the shared
// row buffers (c, sigma and H planes, plane stride ps floats); else null.
__device__ __forceinline__ void router_unit_noisy(const RParams &p, const CUtensorMap *mc,
                                                  const CUtensorMap *ms, const CUtensorMap *mh,
                                                  int t0, int e0, float *cv, float *zv,
                                                  const float *nz, const float *bu, float *stg,
                                                  float *row, int ps) {
  const int lane = threadIdx.x & 31;
  float *sc = stg, *ss = stg + 256, *sh = stg + 512;
  float h[8];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (p.bias) cv[j] += bu[j];
    zv[j] = softplus_r(zv[j]);
    h[j] = fmaf(nz[j], zv[j], cv[j]);
    bad |= e0 + j < p.E && !isfinite(h[j]);
  }
  if (row) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (e0 + j < p.E) {
        row[e0 + j] = h[j];
        row[ps + e0 + j] = cv[j];
        row[2 * ps + e0 + j] = zv[j];
      }
  }
  if (bad && t0 + lane < p.T) record_error(p.st, MOE_ERR_NONFINITE, (long long)(t0 + lane));
  if (lane == 0) bulk_wait_read_all();  // the last unit's stores have read the tiles
  __syncwarp();
  tile_row_store8(sc, lane, cv);
  tile_row_store8(ss, lane, zv);
  tile_row_store8(sh, lane, h);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(mh, sh, e0, t0);
    tma_store_2d(mc, sc, e0, t0);
    tma_store_2d(ms, ss, e0, t0);
    bulk_commit();
  }
}

// One unit without the noise term: H = c for experts e0 .. e0+15, one
// [32 x 16] tile.
__device__ __forceinline__ void router_unit_clean(const RParams &p, const CUtensorMap *mh, int t0,
                                                  int e0, float *cv, const float *bu, float *stg,
                                                  float *row) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (p.bias) cv[j] += bu[j];
    bad |= e0 + j < p.E && !isfinite(cv[j]);
  }
  if (row) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (e0 + j < p.E) row[e0 + j] = cv[j];
  }
  if (bad && t0 + lane < p.T) record_error(p.st, MOE_ERR_NONFINITE, (long long)(t0 + lane));
  if (lane == 0) bulk_wait_read_all();  // the last unit's stores have read the tile
  __syncwarp();
  tile_row_store(stg, lane, cv);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(mh, stg, e0, t0);
    bulk_commit();
  }
}

// The 16 accumulator columns u*16 .. of a tile for this lane's token: column
// j is hi[j] + (mid[j] + lo[j]) from the three BNR-wide sections.
template <int BNR>
__device__ __forceinline__ void unit_columns(uint32_t lane_addr, int u, float (&v)[16]) {
  uint32_t r[48];
  tmem_ld16x3(lane_addr + (uint32_t)(u * 16), lane_addr + (uint32_t)(BNR + u * 16),
              lane_addr + (uint32_t)(2 * BNR + u * 16), r);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = __uint_as_float(r[j]) + (__uint_as_float(r[16 + j]) + __uint_as_float(r[32 + j]));
}

// ----------------------------------------------------------------------------- fused selection
// When one column block holds every expert of a token (one tile per row
// block) and each CTA takes one tile, the epilogue also selects
// ("Outrageously Large", Eq. 5 and the load estimator of Appendix A;
// "Switch Transformer", step 2): the units leave the tile's c, sigma and H
// rows in shared memory (the pipeline stages, free once the CTA's only
// accumulator is full), a thread per token keeps its k + 1 largest H in
// registers (value descending, lower index first on ties; a NaN never
// enters) and writes the picks, gates, thresholds and row statistics, and a
// thread per (16-token group, expert) adds the group's balancing terms in
// token order into the partial row of those 16 tokens.
constexpr int kFuseMaxK = 8;

struct FuseSmem {
  float *h, *c, *s;  // [RBM][E + 1] planes (c and s with the noise term only)
  int ps;            // plane stride in floats
  float4 *sc;        // [RBM] k-th and (k+1)-th largest H, row max, 1 / sum of exp
  int *ci;           // [RBM][kFuseMaxK] chosen experts
  float *cg;         // [RBM][kFuseMaxK] their gates
  float *se;         // [RBM] sum of exp(H - max)
  float *run;        // [runs][groups x E][4] balancing sums of token runs (256 x 4 at most)
};

__host__ __device__ constexpr size_t fuse_bytes(int E, int noisy) {
  return (size_t)(noisy ? 3 : 1) * RBM * (E + 1) * 4 + 16 + (size_t)RBM * 16 +
         (size_t)RBM * kFuseMaxK * 8 + (size_t)RBM * 4 + 32 * kREpiWarps * 16;
}

__device__ __forceinline__ FuseSmem fuse_smem(uint8_t *base, int E, int noisy) {
  FuseSmem f;
  f.ps = RBM * (E + 1);
  f.h = reinterpret_cast<float *>(base);
  f.c = noisy ? f.h + f.ps : nullptr;
  f.s = noisy ? f.h + 2 * f.ps : nullptr;
  const uintptr_t end = reinterpret_cast<uintptr_t>(f.h + (size_t)(noisy ? 3 : 1) * f.ps);
  f.sc = reinterpret_cast<float4 *>((end + 15) & ~uintptr_t(15));
  f.ci = reinterpret_cast<int *>(f.sc + RBM);
  f.cg = reinterpret_cast<float *>(f.ci + RBM * kFuseMaxK);
  f.se = f.cg + RBM * kFuseMaxK;
  f.run = f.se + RBM;
  return f;
}

// Barrier 1 over the epilogue warps only (the TMA and MMA warps never join it).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kREpiWarps) : "memory");
}
// The same barrier, returning whether v held on every epilogue thread.
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, a;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred a, 1, %2, q;\n"
      " selp.u32 %0, 1, 0, a;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(32 * kREpiWarps)
      : "memory");
  return r != 0;
}

// et = epilogue thread 0..255; mb = the tile's row block. Every epilogue
// thread calls this (it holds the barriers). Threads 0..127 keep the picks of
// token et, threads 128..255 sum exp(H - max) of token et - 128 meanwhile;
// the balancing sums of a (16-token group, expert) are split into S runs of
// 16/S tokens so that every thread takes part, each run's terms unrolled so
// that their exponentials overlap, and the runs added in order.
template <int KM>  // KM >= k
__device__ __forceinline__ void fused_select(const RParams &p, const FuseSmem &f, int mb, int et) {
  const int E = p.E, rs = E + 1, k = p.k;
  const int ntok = min(RBM, p.T - mb * RBM);
  epi_sync();  // every unit's rows are in shared memory
  float lv[KM + 1];
  int li[KM + 1];
  if (et < ntok) {
    const float *h = f.h + et * rs;
#pragma unroll
    for (int j = 0; j <= KM; ++j) {
      lv[j] = -INFINITY;
      li[j] = E;
    }
    for (int e = 0; e < E; ++e) {
      float v = h[e];
      int i = e;
#pragma unroll
      for (int j = 0; j <= KM; ++j) {
        // Slots 0..k ordered by (value descending, index ascending); an
        // empty slot is (-inf, E). The entry carried down (the new one, or
        // one it displaced) goes before any equal value of higher index. A
        // NaN compares false and never enters.
        const bool take = j <= k && (v > lv[j] || (v == lv[j] && i < li[j]));
        const float tv = lv[j];
        const int ti = li[j];
        lv[j] = take ? v : tv;
        li[j] = take ? i : ti;
        v = take ? tv : v;
        i = take ? ti : i;
      }
    }
  } else if (et >= RBM && et - RBM < ntok) {
    const float *h = f.h + (et - RBM) * rs;
    float mx = -INFINITY;  // fmaxf drops NaN, as the picks do: mx = the first pick
    for (int e = 0; e < E; ++e) mx = fmaxf(mx, h[e]);
    float se = 0.f;
#pragma unroll 2
    for (int e = 0; e < E; ++e) se += expf(h[e] - mx);
    f.se[et - RBM] = se;
  }
  epi_sync();  // the sums of exponentials are in shared memory
  if (et < ntok) {
    const size_t t = (size_t)mb * RBM + et;
    const float mx = lv[0], se = f.se[et];
    float g[KM];
    if (p.mode == MOE_GATE_SWITCH) {
      g[0] = expf(lv[0] - mx) / se;
#pragma unroll
      for (int j = 1; j < KM; ++j) g[j] = 0.f;
    } else {
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        g[j] = j < k ? expf(lv[j] - lv[0]) : 0.f;
        z += g[j];  // in pick order; the terms past k are zero
      }
      const float iz = 1.f / z;
#pragma unroll
      for (int j = 0; j < KM; ++j) g[j] *= iz;
    }
    float th0 = lv[0], th1 = lv[1];
#pragma unroll
    for (int j = 1; j <= KM; ++j) {
      if (j == k - 1) th0 = lv[j];
      if (j == k) th1 = lv[j];
    }
    if (k >= E) th1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) {
        p.idx[t * k + j] = li[j];
        p.gate[t * k + j] = g[j];
        f.ci[et * kFuseMaxK + j] = li[j];
        f.cg[et * kFuseMaxK + j] = g[j];
      }
    p.thr[2 * t] = th0;
    p.thr[2 * t + 1] = th1;
    p.rowstat[2 * t] = mx;
    p.rowstat[2 * t + 1] = se;
    f.sc[et] = make_float4(th0, th1, mx, 1.f / se);
  }
  epi_sync();  // the token scalars are in shared memory
  if (!p.partials) return;
  const int ngroups = (ntok + 15) / 16;
  const int owners = ngroups * E;
  int S = 1;  // runs per (group, expert), the same for every tile of the launch
  while (S < 8 && 8 * E * S * 2 <= 32 * kREpiWarps) S *= 2;
  const int L = 16 / S;
  for (int i = et; i < owners * S; i += 32 * kREpiWarps) {
    const int sl = i / owners, o = i - sl * owners;  // consecutive threads: consecutive experts
    const int gi = o / E, e = o - gi * E;
    const int t0 = gi * 16 + sl * L;
    const int n = min(L, ntok - t0);
    float imp = 0.f, ld = 0.f, fc = 0.f, pb = 0.f;
#pragma unroll 2
    for (int u = 0; u < 16; ++u) {
      if (u >= n) break;
      const int tt = t0 + u;
      const float4 sc = f.sc[tt];
      const int *ci = f.ci + tt * kFuseMaxK;
      const float *cg = f.cg + tt * kFuseMaxK;
      bool in = false;
      float gv = 0.f;
#pragma unroll
      for (int j = 0; j < KM; ++j)
        if (j < k && ci[j] == e) {
          in = true;
          gv = cg[j];
        }
      imp += gv;
      const float sv = f.s ? f.s[tt * rs + e] : 0.f;
      float pr;
      if (k == E) {
        pr = 1.f;
      } else if (sv == 0.f) {
        pr = in ? 1.f : 0.f;
      } else {
        pr = normal_cdf(__fdividef(f.c[tt * rs + e] - (in ? sc.y : sc.x), sv));
      }
      ld += pr;
      if (ci[0] == e) fc += 1.f;
      pb += expf(f.h[tt * rs + e] - sc.z) * sc.w;
    }
    if (S == 1) {
      float *out = p.partials + ((size_t)mb * (RBM / 16) + gi) * 4 * E + e;
      out[0] = imp;
      out[E] = ld;
      out[2 * E] = fc;
      out[3 * E] = pb;
    } else {
      float *r = f.run + ((size_t)sl * owners + o) * 4;
      r[0] = imp;
      r[1] = ld;
      r[2] = fc;
      r[3] = pb;
    }
  }
  if (S == 1) return;
  epi_sync();  // every run's sums are in shared memory
  for (int o = et; o < owners; o += 32 * kREpiWarps) {
    const int gi = o / E, e = o - gi * E;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < S; ++sl) {
      const float *r = f.run + ((size_t)sl * owners + o) * 4;
      acc.x += r[0];
      acc.y += r[1];
      acc.z += r[2];
      acc.w += r[3];
    }
    float *out = p.partials + ((size_t)mb * (RBM / 16) + gi) * 4 * E + e;
    out[0] = acc.x;
    out[E] = acc.y;
    out[2 * E] = acc.z;
    out[3 * E] = acc.w;
  }
}

// KMF = 0: no fused selection; else the pick list length of fused_select.
template <int BNR, int KMF>
__global__ void __launch_bounds__(kRThreads, 1)
k_router_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
            const __grid_constant__ CUtensorMap tmH, const RParams p) {
  using C = RCfg<BNR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float *staging = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE + EPI_BYTES);
  uint64_t *full = bars, *empty = bars + C::STAGES;
  uint64_t *acc_full = bars + 2 * C::STAGES, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kREpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // barriers and TMEM are set up; now the inputs may be read
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int m_blocks = (p.T + RBM - 1) / RBM;
  const int total = m_blocks * p.n_blocks;
  const int num_kb = (p.d + RBK - 1) / RBK;

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 21, p.wait_ns)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + s * C::STAGE;
          mbar_expect_tx(&full[s], C::STAGE);
          tma_load_2d(st, &tmA, &full[s], kb * RBK, mb * RBM);
          tma_load_2d(st + C::A_BYTES, &tmB, &full[s], kb * RBK, nb * C::NB);
        }
      }
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)C::STAGES ? issued - C::STAGES : 0; q < issued; ++q)
        mbar_drain(&full[q % C::STAGES], (q / C::STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 22, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * C::NB);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 23, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * C::STAGE);
#pragma unroll
          for (int kk = 0; kk < RBK / 16; ++kk) {
            const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(a0 + C::A_BYTES + kk * 32, 16, 1024);
            umma_r<BNR>(tmem_d, ad, bd, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;          // TMEM lanes 32*quad .. 32*quad+31
    const int sub = (warp - 2) >> 2;    // this warp's units: sub, sub+2, ...
    int local = 0;
    float nz_next[8];   // noise of this warp's next unit
    int nz_tile = -1;   // the tile whose first unit nz_next already holds
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                     p.st, 24, p.wait_ns));
      if (KMF > 0) ready = epi_all(ready);  // the fused phase's barriers need all warps
      if (!ready) break;
      tc_fence_after();
      const int t0 = mb * RBM + quad * 32;
      const uint32_t lane_addr =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * C::NB);
      const int t = t0 + lane;
      const int ncols = min(p.NC - nb * BNR, BNR);
      if (p.tma_out) {
        // Units of 16 accumulator columns (8 experts with the noise term, 16
        // without), dealt to the quadrant's two warps in turn. The next
        // unit's noise is loaded while this one is computed; after this
        // warp's last unit of the tile, its first unit of the CTA's next tile,
        // so the load overlaps the wait for the next accumulator.
        float *stg = staging + (size_t)(warp - 2) * kEpiWarpFloats;
        const int nunits = (ncols + 15) / 16;
        float *row = nullptr;  // this lane's token row in the fused-selection buffers
        FuseSmem fs{};
        if (KMF > 0) {
          fence_proxy_async_smem();  // the stages' last MMA reads are complete (acc_full)
          fs = fuse_smem(smem, p.E, p.noisy);
          row = fs.h + (quad * 32 + lane) * (p.E + 1);
        }
        const int epu = p.noisy ? 8 : 16;  // experts per unit
        const int eb = p.noisy ? (nb * BNR) >> 1 : nb * BNR;  // first expert of the block
        if (p.noisy && sub < nunits && nz_tile != tile) load_noise8(p, t, eb + sub * 8, nz_next);
#pragma unroll 1
        for (int u = sub; u < nunits; u += 2) {
          float nz[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) nz[j] = nz_next[j];
          if (p.noisy) {
            if (u + 2 < nunits) {
              load_noise8(p, t, eb + (u + 2) * 8, nz_next);
            } else if (tile + (int)gridDim.x < total) {
              const int nt = tile + gridDim.x;
              const int nmb = nt / p.n_blocks, nnb = nt % p.n_blocks;
              const int nncols = min(p.NC - nnb * BNR, BNR);
              if (sub < (nncols + 15) / 16) {
                load_noise8(p, nmb * RBM + quad * 32 + lane, ((nnb * BNR) >> 1) + sub * 8,
                            nz_next);
                nz_tile = nt;
              }
            }
          }
          float bu[16];  // issued before the TMEM loads, so their latencies overlap
          load_bias_n(p, eb + u * epu, epu, bu);
          float v[16];
          unit_columns<BNR>(lane_addr, u, v);
          if (p.noisy) {
            float cv[8], zv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              cv[j] = v[2 * j];
              zv[j] = v[2 * j + 1];
            }
            router_unit_noisy(p, &tmC, &tmS, &tmH, t0, eb + u * epu, cv, zv, nz, bu, stg, row,
                              fs.ps);
          } else {
            router_unit_clean(p, &tmH, t0, eb + u * epu, v, bu, stg, row);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        if constexpr (KMF > 0) fused_select<KMF>(p, fs, mb, threadIdx.x - 64);
        continue;
      }
      // Row-segment path: the first warp of each quadrant, 16 columns at a
      // time.
      float *stg = staging + (size_t)(warp - 2) * 3 * kEpiTile;
      const int nchunks = sub == 0 ? (ncols + 15) / 16 : 0;
      // 16 columns at a time: 8 experts (noisy, clean/noise pairs) or 16.
      // The next chunk's noise is loaded while this one is computed.
      if (p.noisy && nchunks > 0) load_noise8(p, t, (nb * BNR) >> 1, nz_next);
#pragma unroll 1
      for (int c16 = 0; c16 < nchunks; ++c16) {
        const int n = nb * BNR + c16 * 16;
        float nz[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) nz[j] = nz_next[j];
        if (p.noisy && c16 + 1 < nchunks) load_noise8(p, t, (n + 16) >> 1, nz_next);
        // Column j of the block is hi[j] + (mid[j] + lo[j]), from the three
        // BNR-wide sections of the accumulator.
        uint32_t vh[16], vm[16], vl[16];
        tmem_ld16(lane_addr + (uint32_t)(c16 * 16), vh);
        tmem_ld16(lane_addr + (uint32_t)(BNR + c16 * 16), vm);
        tmem_ld16(lane_addr + (uint32_t)(2 * BNR + c16 * 16), vl);
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = __uint_as_float(vh[j]) + (__uint_as_float(vm[j]) + __uint_as_float(vl[j]));
        float cv[16], zv[16];
        int e0, ne;
        if (p.noisy) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            cv[j] = v[2 * j];
            zv[j] = v[2 * j + 1];
          }
#pragma unroll
          for (int j = 8; j < 16; ++j) cv[j] = zv[j] = 0.f;
          e0 = n >> 1;
          ne = p.E - e0 < 8 ? p.E - e0 : 8;
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            cv[j] = v[j];
            zv[j] = 0.f;
          }
          e0 = n;
          ne = p.E - e0 < 16 ? p.E - e0 : 16;
        }
        router_rows(p, t0, e0, ne, cv, zv, nz, stg);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  if (warp >= 2 && lane == 0) bulk_wait_all();  // this warp's TMA stores are complete
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------------------- CTA-pair form
// The unfused router with tcgen05.mma.cta_group::2, for many column blocks
// (large E). A cluster of two CTAs on two SMs computes a 256-token x
// BNR-column tile: each CTA loads its own 128 token rows of x and half of the
// three pieces' 3*BNR B rows (the even CTA rows 0 .. 3*BNR/2 - 1 of the
// block, the odd CTA the rest), 28 KB per 64-deep K step instead of the
// one-CTA form's 40 KB for the same work per SM. The even CTA issues the MMAs
// (M = 256, N = 3*BNR); each CTA's token rows land in its own TMEM with the
// one-CTA form's column layout (hi, mid, lo sections), and each CTA's eight
// epilogue warps run the TMA-store epilogue on its rows. The odd CTA's TMA
// completions are counted on the even CTA's "full" barriers, the MMA commits
// arrive (multicast) on both CTAs' "empty" and "accumulator full" barriers,
// and both CTAs' epilogue warps arrive on the even CTA's "accumulator empty"
// barriers. Tiles go round robin over the pairs.
//
// The noise draws of a tile (this CTA's 128 tokens x BNR/2 experts, fp32)
// come into shared memory by TMA, issued by the producer after the tile's
// operand loads, into one of two buffers: the epilogue reads them from there
// instead of loading them from HBM a unit ahead, a latency it could not hide.
template <int BNR>
struct RPCfg {
  static constexpr int NB = 3 * BNR;
  static constexpr int B_ROWS = NB / 2;                  // B rows held per CTA
  static constexpr int A_BYTES = RBM * RBK * 2;          // 16 KB
  static constexpr int B_BYTES = B_ROWS * RBK * 2;       // 12 KB at BNR = 64
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NZ_COLS = BNR / 2;                // experts per tile (noise term)
  static constexpr int NZ_BYTES = RBM * NZ_COLS * 4;     // 16 KB at BNR = 64
  static constexpr int FIT = (227 * 1024 - 1024 - 2 * NZ_BYTES - EPI_BYTES - 512) / STAGE;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int TMEM_COLS = RCfg<BNR>::TMEM_COLS;
  // kind::f16: fp32 accumulate, bf16 A and B, both K-major, M = 256, N = 3*BNR.
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                                    ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + 2 * NZ_BYTES + EPI_BYTES +
                                 (2 * STAGES + 9) * 8 + 8;
  static_assert(NZ_COLS * 4 == 128, "one 128-byte swizzled row of noise per token");
  static_assert(B_ROWS % 8 == 0 && STAGE % 1024 == 0, "swizzle atoms");
  static_assert(STAGES >= 4, "pipeline depth");
};

__device__ __forceinline__ void umma_rp(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Noise draws of token row r (0..127) of a tile, experts u*8 .. u*8+7 of the
// tile's 32, from a [128 x 32] fp32 buffer in the 128-byte swizzle (16-byte
// chunk q of row r at chunk q ^ (r & 7)).
__device__ __forceinline__ void noise_from_smem(const float *buf, int r, int u, float *nz) {
  const float4 *row = reinterpret_cast<const float4 *>(buf + r * 32);
  const float4 a = row[(2 * u) ^ (r & 7)], b = row[(2 * u + 1) ^ (r & 7)];
  nz[0] = a.x; nz[1] = a.y; nz[2] = a.z; nz[3] = a.w;
  nz[4] = b.x; nz[5] = b.y; nz[6] = b.z; nz[7] = b.w;
}

// tmB's box is RPCfg::B_ROWS rows; tmN the noise [T, E] fp32, box [128 tokens
// x BNR/2 experts], 128-byte swizzle (unused without the noise term); tmC,
// tmS, tmH as for k_router_tc (the TMA-store epilogue only).
template <int BNR>
__global__ void __launch_bounds__(kRThreads, 1)
k_router_tc_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmN, const __grid_constant__ CUtensorMap tmC,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmH,
                 const RParams p) {
  using C = RPCfg<BNR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float *nzbuf = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE);  // [2][128][32]
  float *staging = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE + 2 * C::NZ_BYTES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE + 2 * C::NZ_BYTES +
                                                EPI_BYTES);
  uint64_t *full = bars, *empty = bars + C::STAGES;
  uint64_t *acc_full = bars + 2 * C::STAGES, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint64_t *nz_full = drain + 1, *nz_empty = nz_full + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(nz_empty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's expect_tx arrival
      mbar_init(&empty[s], 1);  // one multicast commit per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kREpiWarps);  // both CTAs' epilogue warps
      mbar_init(&nz_full[b], 1);                 // this CTA's expect_tx arrival
      mbar_init(&nz_empty[b], kREpiWarps);       // this CTA's epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  pdl_wait();  // the split weights come from the kernel before
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int m_blocks = (p.T + 2 * RBM - 1) / (2 * RBM);
  const int total = m_blocks * p.n_blocks;
  const int num_kb = (p.d + RBK - 1) / RBK;

  if (warp == 0) {
    if (lane == 0) {
      // ----------------------------------------------------------- producer (both CTAs)
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      if (p.noisy) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmN) : "memory");
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total; tile += n_pairs, ++local) {
        const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
        const int arow = mb * 2 * RBM + (int)rank * RBM;
        const int brow = nb * C::NB + (int)rank * C::B_ROWS;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 25, p.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = mapa(smem_u32(&full[s]), 0);
          if (leader) mbar_expect_tx(&full[s], 2 * C::STAGE);
          uint8_t *st = smem + s * C::STAGE;
          tma_load_2d_pair(st, &tmA, full_leader, kb * RBK, arow);
          tma_load_2d_pair(st + C::A_BYTES, &tmB, full_leader, kb * RBK, brow);
        }
        if (ok && p.noisy) {
          // The tile's noise, once the epilogue is done with this buffer's
          // previous tile (two tiles back).
          const int nbuf = local & 1;
          const uint32_t use = (uint32_t)(local >> 1);
          if (!mbar_wait(&nz_empty[nbuf], (use & 1u) ^ 1u, abort_flag, p.st, 29, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&nz_full[nbuf], C::NZ_BYTES);
          tma_load_2d(nzbuf + nbuf * (C::NZ_BYTES / 4), &tmN, &nz_full[nbuf], nb * C::NZ_COLS,
                      arow);
        }
      }
      // This CTA's copies have landed once the MMAs that read them are done,
      // and its noise once the epilogue has read it.
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)C::STAGES ? issued - C::STAGES : 0; q < issued; ++q)
        mbar_drain(&empty[q % C::STAGES], (q / C::STAGES) & 1u);
      if (p.noisy)
        for (int q = local > 2 ? local - 2 : 0; q < local; ++q)
          mbar_drain(&nz_full[q & 1], (uint32_t)(q >> 1) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ----------------------------------------------------------- MMA issuer (even CTA)
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total; tile += n_pairs, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 26, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * C::NB);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 27, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * C::STAGE);
#pragma unroll
          for (int kk = 0; kk < RBK / 16; ++kk) {
            const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(a0 + C::A_BYTES + kk * 32, 16, 1024);
            umma_rp(tmem_d, ad, bd, C::IDESC, (kb | kk) ? 1u : 0u);
          }
          umma_commit_pair(&empty[s]);
        }
        if (ok) umma_commit_pair(&acc_full[buf]);
      }
      umma_commit_pair(drain, 0x1);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;        // TMEM lanes 32*quad .. 32*quad+31
    const int sub = (warp - 2) >> 2;  // this warp's units: sub, sub+2, ...
    const uint32_t acc_empty_leader0 = mapa(smem_u32(&acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = mapa(smem_u32(&acc_empty[1]), 0);
    float *stg = staging + (size_t)(warp - 2) * kEpiWarpFloats;
    const int epu = p.noisy ? 8 : 16;  // experts per unit
    const int r = quad * 32 + lane;    // this lane's token row in the tile
    int local = 0;
    for (int tile = pair; tile < total; tile += n_pairs, ++local) {
      const int mb = tile / p.n_blocks, nb = tile % p.n_blocks;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      bool ready = mbar_wait(&acc_full[buf], use & 1u, abort_flag, p.st, 28, p.wait_ns);
      if (p.noisy) ready = ready && mbar_wait(&nz_full[buf], use & 1u, abort_flag, p.st, 30,
                                              p.wait_ns);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      const int t0 = mb * 2 * RBM + (int)rank * RBM + quad * 32;
      const uint32_t lane_addr =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * C::NB);
      const int ncols = min(p.NC - nb * BNR, BNR);
      const int nunits = (ncols + 15) / 16;
      const int eb = p.noisy ? (nb * BNR) >> 1 : nb * BNR;  // first expert of the block
      const float *nzt = nzbuf + buf * (C::NZ_BYTES / 4);
#pragma unroll 1
      for (int u = sub; u < nunits; u += 2) {
        float bu[16];  // issued before the TMEM loads, so their latencies overlap
        load_bias_n(p, eb + u * epu, epu, bu);
        float nz[8];
        if (p.noisy) noise_from_smem(nzt, r, u, nz);
        float v[16];
        unit_columns<BNR>(lane_addr, u, v);
        if (p.noisy) {
          float cv[8], zv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            cv[j] = v[2 * j];
            zv[j] = v[2 * j + 1];
          }
          router_unit_noisy(p, &tmC, &tmS, &tmH, t0, eb + u * epu, cv, zv, nz, bu, stg, nullptr,
                            0);
        } else {
          router_unit_clean(p, &tmH, t0, eb + u * epu, v, bu, stg, nullptr);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_remote(buf ? acc_empty_leader1 : acc_empty_leader0);
        if (p.noisy) mbar_arrive(&nz_empty[buf]);
      }
    }
  }
  if (warp >= 2 && lane == 0) bulk_wait_all();  // this warp's TMA stores are complete
  tc_fence_before();
  cluster_sync_all();  // every MMA reading either CTA's memory and every TMEM read are done
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ----------------------------------------------------------------------------- grouped form
// The hierarchical layer's secondary gates, only where they are used: the
// (token, primary pick) pairs come packed by group (xg: group i's tokens in
// rows goff[i] .. goff[i+1]-1, as the slot pass and gather lay them out), and
// group i's rows meet only group i's weight columns (n-blocks i*nbg ..
// i*nbg+nbg-1 of the split weights). A tile is (group, 128-row block,
// n-block). Outputs c, sigma, H [rows][b] are written at padded row offsets
// poff[i] = sum over earlier groups of their row blocks * 128, so a ragged
// tail's rows land in its own group's padding (never read), not in the next
// group's rows. A row's noise is noise[t][i*b + j] with t its packed token.
struct GParams {
  int a, nbg, kp, noise_stride;
  const int32_t *goff;    // [a+1] exact packed-row offsets of the groups
  const int32_t *grow;    // [rows] packed row -> t * kp + q
  int32_t *poff_out;      // [a+1] padded output offsets (written by block 0)
};

__device__ __forceinline__ void load_noise8_g(const RParams &p, int t, size_t e0, float *nz) {
  if (t < 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) nz[j] = 0.f;
    return;
  }
  const float4 *src = reinterpret_cast<const float4 *>(p.noise + (size_t)t * p.d + e0);
  const float4 u = src[0], v = src[1];
  nz[0] = u.x; nz[1] = u.y; nz[2] = u.z; nz[3] = u.w;
  nz[4] = v.x; nz[5] = v.y; nz[6] = v.z; nz[7] = v.w;
}

// p: T = output rows (padded), E = b, d = the noise row stride (a*b; the K
// width is in gd), noise / noisy as usual, no bias, tma_out set.
template <int BNR>
__global__ void __launch_bounds__(kRThreads, 1)
k_router_grp(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
             const __grid_constant__ CUtensorMap tmH, const RParams p, const GParams g, int gd) {
  using C = RCfg<BNR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float *staging = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE + EPI_BYTES);
  uint64_t *full = bars, *empty = bars + C::STAGES;
  uint64_t *acc_full = bars + 2 * C::STAGES, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *gtile = const_cast<int *>(reinterpret_cast<volatile int *>(abort_flag + 1));  // [a+1]
  int *gpoff = gtile + g.a + 1;                                                      // [a+1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kREpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the group offsets come from the slot pass
  pdl_trigger();
  if (threadIdx.x == 0) {  // tile and padded-row prefixes over the groups
    int tiles = 0, rows = 0;
    for (int i = 0; i < g.a; ++i) {
      gtile[i] = tiles;
      gpoff[i] = rows;
      const int mt = (g.goff[i + 1] - g.goff[i] + RBM - 1) / RBM;
      tiles += mt * g.nbg;
      rows += mt * RBM;
    }
    gtile[g.a] = tiles;
    gpoff[g.a] = rows;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= g.a; i += blockDim.x) g.poff_out[i] = gpoff[i];
  const uint32_t tmem_base = *tmem_slot;
  const int total = gtile[g.a];
  const int num_kb = (gd + RBK - 1) / RBK;
  // tile -> (group, row block, n-block in the group)
  auto locate = [&](int tile, int &gi, int &mb, int &nb) {
    int lo = 0, hi = g.a - 1;
    while (lo < hi) {  // the last group whose first tile is <= tile
      const int mid = (lo + hi + 1) >> 1;
      if (gtile[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    gi = lo;
    const int local = tile - gtile[lo];
    mb = local / g.nbg;
    nb = local - mb * g.nbg;
  };

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int gi, mb, nb;
        locate(tile, gi, mb, nb);
        const int row0 = g.goff[gi] + mb * RBM, n_abs = gi * g.nbg + nb;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.st, 31, p.wait_ns)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + s * C::STAGE;
          mbar_expect_tx(&full[s], C::STAGE);
          tma_load_2d(st, &tmA, &full[s], kb * RBK, row0);
          tma_load_2d(st + C::A_BYTES, &tmB, &full[s], kb * RBK, n_abs * C::NB);
        }
      }
      const uint32_t issued = it;
      for (uint32_t q = issued > (uint32_t)C::STAGES ? issued - C::STAGES : 0; q < issued; ++q)
        mbar_drain(&full[q % C::STAGES], (q / C::STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.st, 32, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * C::NB);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, p.st, 33, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * C::STAGE);
#pragma unroll
          for (int kk = 0; kk < RBK / 16; ++kk) {
            const uint64_t ad = sdesc(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(a0 + C::A_BYTES + kk * 32, 16, 1024);
            umma_r<BNR>(tmem_d, ad, bd, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&acc_full[buf]);
      }
      umma_commit(drain);
      mbar_drain(drain, 0);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int sub = (warp - 2) >> 2;
    int local = 0;
    float *stg = staging + (size_t)(warp - 2) * kEpiWarpFloats;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      int gi, mb, nb;
      locate(tile, gi, mb, nb);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const bool ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag,
                                                           p.st, 34, p.wait_ns));
      if (!ready) break;
      tc_fence_after();
      const int cnt = g.goff[gi + 1] - g.goff[gi];
      const int lrow = mb * RBM + quad * 32 + lane;  // row within the group
      int t = -1;                                     // this lane's token, if a real row
      if (lrow < cnt) t = g.grow[g.goff[gi] + lrow] / g.kp;
      const int t0 = gpoff[gi] + mb * RBM + quad * 32;  // output row of lane 0
      const uint32_t lane_addr =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * C::NB);
      const int nunits = BNR / 16;  // the group's blocks are whole (checked on the host)
      const int epu = p.noisy ? 8 : 16;
      const int eb = p.noisy ? (nb * BNR) >> 1 : nb * BNR;  // first in-group expert
#pragma unroll 1
      for (int u = sub; u < nunits; u += 2) {
        float nz[8];
        if (p.noisy) load_noise8_g(p, t, (size_t)gi * p.E + eb + u * 8, nz);
        const float bu[16] = {};  // no router bias in the grouped form
        float v[16];
        unit_columns<BNR>(lane_addr, u, v);
        if (p.noisy) {
          float cv[8], zv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            cv[j] = v[2 * j];
            zv[j] = v[2 * j + 1];
          }
          router_unit_noisy(p, &tmC, &tmS, &tmH, t0, eb + u * epu, cv, zv, nz, bu, stg, nullptr,
                            0);
        } else {
          router_unit_clean(p, &tmH, t0, eb + u * epu, v, bu, stg, nullptr);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  if (warp >= 2 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::TMEM_COLS)
                 : "memory");
  }
}

int tile_cols(int NC) { return NC <= 16 ? 16 : NC <= 32 ? 32 : 64; }

// 2-D fp32 tensor [T, E] (E contiguous, E % 4 == 0): the router's output
// tiles, box [32 tokens, 8 experts] in the 32-byte swizzle (noise term) or
// [32 tokens, 16 experts] in the 64-byte swizzle (without).
bool make_out_map(CUtensorMap *m, float *base, int T, int E, bool noisy) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)E * 4};
  cuuint32_t box[2] = {noisy ? 8u : 16u, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            noisy ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MOE_ROUTER_PAIR=0 keeps the one-CTA form, =1 takes the CTA-pair form
// wherever it applies (read at each call; for comparisons and tests);
// otherwise the pair form runs where there are at least four 128-row tiles per
// SM over two or more column blocks.
bool use_pair(int tiles, int n_blocks) {
  const char *v = getenv("MOE_ROUTER_PAIR");
  if (v && v[0] == '0') return false;
  if (n_blocks < 2) return false;
  if (v && v[0] == '1') return true;
  return tiles >= 4 * sm_count();
}

cudaLaunchAttribute router_cluster_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Clusters of two that can be resident at once for the CTA-pair form (0 if
// none); one shared-memory size, so looked up once.
int pair_router_clusters() {
  static const int n = [] {
    const size_t smem = RPCfg<64>::SMEM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1] = {router_cluster_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int m = 0;
    if (cudaFuncSetAttribute(k_router_tc_pair<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&m, k_router_tc_pair<64>, &cfg) != cudaSuccess)
      m = 0;
    return m;
  }();
  return n;
}

// 2-D fp32 tensor [T, E] (E % 4 == 0): the noise draws, box [128 tokens, 32
// experts] in the 128-byte swizzle, for the CTA-pair form's epilogue.
bool make_noise_map(CUtensorMap *m, const float *base, int T, int E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)E * 4};
  cuuint32_t box[2] = {32u, (cuuint32_t)RBM};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BNR>
cudaError_t launch_router_pair(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tn,
                               const CUtensorMap &tc, const CUtensorMap &ts, const CUtensorMap &th,
                               const RParams &p, int clusters, cudaStream_t s) {
  const size_t smem = RPCfg<BNR>::SMEM;
  cudaError_t err = cudaFuncSetAttribute(k_router_tc_pair<BNR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2] = {router_cluster_attr(), {}};
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_router_tc_pair<BNR>, ta, tb, tn, tc, ts, th, p);
}

template <int BNR>
cudaError_t run(const moe_config &c, const void *x, const float *Wg, const float *Wn,
                const float *noise, const float *bias, float *cc, float *sg, float *H,
                void *bsplit, DeviceStatus *st, cudaStream_t s, const RouterSelect *sel,
                bool *selected) {
  const int noisy = Wn != nullptr;
  const int NC = noisy ? 2 * c.E : c.E;
  const int n_blocks = (NC + BNR - 1) / BNR;
  const int NCP = n_blocks * BNR;
  dim3 sg_grid((c.d + 31) / 32, (NCP + 31) / 32);
  launch_pdl(k_router_split, sg_grid, dim3(32, 8), 0, s, c.d, c.E, noisy, NC, NCP, BNR, Wg, Wn,
      static_cast<__nv_bfloat16 *>(bsplit), st);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tb, tc, ts, th;
  if (!make_map(&ta, x, (uint64_t)c.T, (uint64_t)c.d, RBM) ||
      !make_map(&tb, bsplit, (uint64_t)3 * NCP, (uint64_t)c.d, 3 * BNR))
    return cudaErrorInvalidValue;
  // The TMA-store epilogue needs 16-byte rows and 16-byte-aligned outputs.
  const bool tma_out = c.E % 4 == 0 && (uintptr_t)cc % 16 == 0 && (uintptr_t)sg % 16 == 0 &&
                       (uintptr_t)H % 16 == 0 && make_out_map(&tc, cc, c.T, c.E, noisy) &&
                       make_out_map(&ts, sg, c.T, c.E, noisy) &&
                       make_out_map(&th, H, c.T, c.E, noisy);
  if (!tma_out) th = ts = tc = ta;  // unused
  // Fused selection: one column block, the TMA-store epilogue, k <= 8, and
  // one tile per CTA (its pipeline stages then hold the selection buffers).
  // MOE_ROUTER_SELECT=separate keeps the selection kernels instead.
  static const bool separate = [] {
    const char *v = getenv("MOE_ROUTER_SELECT");
    return v && v[0] == 's';
  }();
  const bool fuse = !separate && sel != nullptr && tma_out && n_blocks == 1 && c.k <= kFuseMaxK &&
                    fuse_bytes(c.E, noisy) <= (size_t)RCfg<BNR>::STAGES * RCfg<BNR>::STAGE;
  RParams p{c.T, c.d, c.E, noisy, NC, NCP, n_blocks, tma_out ? 1 : 0, noise, bias, cc, sg, H, st,
            wait_limit_ns(), fuse ? 1 : 0, c.k, c.gate_mode,
            fuse ? sel->idx : nullptr, fuse ? sel->gate : nullptr, fuse ? sel->thr : nullptr,
            fuse ? sel->rowstat : nullptr, fuse ? sel->partials : nullptr};
  const int tiles = ((c.T + RBM - 1) / RBM) * n_blocks;
  if constexpr (BNR == 64) {
    if (!fuse && tma_out && use_pair(tiles, n_blocks)) {
      const int clusters = pair_router_clusters();
      CUtensorMap tbp, tn = ta;  // tn: unused without the noise term
      if (clusters > 0 &&
          make_map(&tbp, bsplit, (uint64_t)3 * NCP, (uint64_t)c.d, RPCfg<BNR>::B_ROWS) &&
          (!noisy || ((uintptr_t)noise % 16 == 0 && make_noise_map(&tn, noise, c.T, c.E)))) {
        const int pair_tiles = ((c.T + 2 * RBM - 1) / (2 * RBM)) * n_blocks;
        const int n = pair_tiles < clusters ? pair_tiles : clusters;
        err = launch_router_pair<BNR>(ta, tbp, tn, tc, ts, th, p, n, s);
        if (err == cudaSuccess && selected) *selected = false;
        return err;
      }
    }
  }
  const size_t smem = RCfg<BNR>::SMEM;
  const int grid = fuse || tiles < sm_count() ? tiles : sm_count();
  const int kmf = !fuse ? 0 : c.k <= 2 ? 2 : c.k <= 4 ? 4 : kFuseMaxK;
  auto kernel = kmf == 0 ? k_router_tc<BNR, 0>
              : kmf == 2 ? k_router_tc<BNR, 2>
              : kmf == 4 ? k_router_tc<BNR, 4>
                         : k_router_tc<BNR, kFuseMaxK>;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  launch_pdl(kernel, grid, kRThreads, smem, s, ta, tb, tc, ts, th, p);
  err = cudaGetLastError();
  if (err == cudaSuccess && selected) *selected = fuse;
  return err;
}

template <int BNR>
cudaError_t run_grp(const GroupedRouter &r, DeviceStatus *st, cudaStream_t s) {
  const int noisy = r.Wn != nullptr;
  const int ncg = (noisy ? 2 : 1) * r.b;  // a group's output columns
  const int NC = r.a * ncg, n_blocks = NC / BNR;
  dim3 sg_grid((r.d + 31) / 32, (NC + 31) / 32);
  launch_pdl(k_router_split, sg_grid, dim3(32, 8), 0, s, r.d, r.a * r.b, noisy, NC, NC, BNR, r.Wg,
      r.Wn, static_cast<__nv_bfloat16 *>(r.bsplit), st);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tb, tc, ts, th;
  const int rows_pad = r.T * r.kp + r.a * RBM;
  if (!make_map(&ta, r.xg, (uint64_t)r.T * r.kp, (uint64_t)r.d, RBM) ||
      !make_map(&tb, r.bsplit, (uint64_t)3 * NC, (uint64_t)r.d, 3 * BNR) ||
      !make_out_map(&th, r.H, rows_pad, r.b, noisy))
    return cudaErrorInvalidValue;
  if (noisy) {
    if (!make_out_map(&tc, r.c, rows_pad, r.b, true) ||
        !make_out_map(&ts, r.sigma, rows_pad, r.b, true))
      return cudaErrorInvalidValue;
  } else {
    tc = ts = th;
  }
  RParams p{rows_pad, r.a * r.b, r.b, noisy, NC, NC, n_blocks, 1, r.noise, nullptr, r.c, r.sigma,
            r.H, st, wait_limit_ns(), 0, 0, 0, nullptr, nullptr, nullptr, nullptr, nullptr};
  GParams g{r.a, ncg / BNR, r.kp, r.a * r.b, r.goff, r.grow, r.poff};
  const size_t smem = RCfg<BNR>::SMEM + (size_t)8 * (r.a + 1);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  err = cudaFuncSetAttribute(k_router_grp<BNR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (err != cudaSuccess) return err;
  const long max_tiles = ((long)r.T * r.kp / RBM + r.a) * (ncg / BNR);
  const int grid = max_tiles < sm_count() ? (int)max_tiles : sm_count();
  launch_pdl(k_router_grp<BNR>, grid, kRThreads, smem, s, ta, tb, tc, ts, th, p, g, r.d);
  return cudaGetLastError();
}

}  // namespace

bool router_grouped_supported(int d, int b, bool noisy, bool bf16) {
  const int ncg = (noisy ? 2 : 1) * b;
  return bf16 && d % 8 == 0 && b % 4 == 0 && (ncg == 16 || ncg == 32 || ncg % 64 == 0) &&
         encode_fn() != nullptr;
}

cudaError_t launch_router_grouped(const GroupedRouter &r, DeviceStatus *st, cudaStream_t s) {
  const int ncg = (r.Wn ? 2 : 1) * r.b;
  if (ncg == 16) return run_grp<16>(r, st, s);
  if (ncg == 32) return run_grp<32>(r, st, s);
  return run_grp<64>(r, st, s);
}

bool router_tc_supported(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && c.d % 8 == 0 && encode_fn() != nullptr;
}

size_t router_tc_split_bytes(const moe_config &c) {
  const int NC = 2 * c.E;  // the noisy layout is the larger one
  const int BNR = tile_cols(NC);
  const size_t NCP = (size_t)((NC + BNR - 1) / BNR) * BNR;
  return 3 * NCP * (size_t)c.d * 2;
}

cudaError_t launch_router_tc(const moe_config &c, const void *x, const float *Wg, const float *Wn,
                             const float *noise, const float *bias, float *cc, float *sg, float *H,
                             void *bsplit, DeviceStatus *st, cudaStream_t s,
                             const RouterSelect *sel, bool *selected) {
  switch (tile_cols(Wn ? 2 * c.E : c.E)) {
    case 16: return run<16>(c, x, Wg, Wn, noise, bias, cc, sg, H, bsplit, st, s, sel, selected);
    case 32: return run<32>(c, x, Wg, Wn, noise, bias, cc, sg, H, bsplit, st, s, sel, selected);
    default: return run<64>(c, x, Wg, Wn, noise, bias, cc, sg, H, bsplit, st, s, sel, selected);
  }
}

}  // namespace moe
