// Backward of the layer, CUDA-core kernels: padded row offsets, the dy
// gather, the gate gradient of each kept choice, the gradients of the
// balancing losses and of the gate softmax, the router weight gradients, the
// bias gradients and the input gradient ("Outrageously Large Neural
// Networks", section 3.4 "Training the gating network": gradients reach W_g
// through the selected softmax gates and W_noise through the smooth load
// estimator; "Switch Transformer", step 8: f is built from integer decisions
// and carries no gradient, P and the selected gate do).
//
// With the forward's choices fixed (top-k set, capacity drops, ReLU pattern),
//   dL/dgate[t,j] = <dy_t, U_e(x_t)> (kept) + dImportance_e
//   U_e(x) = h W2[e] + b2[e],  <dy_t, h W2> = <dy_t W2^T, h> (the GEMM epilogue)
//   top-k gates: dH_S = G (dG - <G, dG>); Switch: the full softmax at the argmax
//   load: P = Phi((c - thr) / sigma): phi/sigma to c, -phi u/sigma to sigma,
//         -phi/sigma to the expert whose noisy logit is thr
//   H = c + n sigma, sigma = Softplus(z): dz = dsigma * sigmoid(z), and
//   sigmoid(z) = 1 - exp(-sigma) exactly, so z need not be kept.
// All sums run in a fixed order: results are identical from run to run.
#include "moe_internal.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kRowPad = kBwdRowPad;  // padded rows per expert are a multiple of 64 (at least 64)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Largest e with a[e] <= v over a[0..n] (a ascending, a[0] <= v < a[n]).
__device__ __forceinline__ int find_block(const int32_t *__restrict__ a, int n, int v) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[j]);
    f[2 * j] = __low2float(b);
    f[2 * j + 1] = __high2float(b);
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t *>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ----------------------------------------------------------------------------- padded offsets
// poff[e] = sum over e' < e of max(64, roundup(rows_e', 64)); one block of 1024.
__global__ void __launch_bounds__(1024) k_bwd_offsets(int E, const int32_t *__restrict__ offset,
                                                      int32_t *__restrict__ poff) {
  pdl_wait();
  __shared__ int wsum[32];
  const int e = threadIdx.x, lane = e & 31, w = e >> 5;
  int v = 0;
  if (e < E) {
    const int rows = offset[e + 1] - offset[e];
    v = rows <= kRowPad ? kRowPad : (rows + kRowPad - 1) / kRowPad * kRowPad;
  }
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    wsum[lane] = s;  // inclusive prefix of the warp totals
  }
  __syncthreads();
  const int before = (w > 0 ? wsum[w - 1] : 0) + incl - v;
  if (e < E) poff[e] = before;
  if (e == E - 1) poff[E] = before + v;
  pdl_trigger();
}

// Rows [A_acc, A_acc + 64) of the forward's packed x and h rows are read by
// the weight-gradient GEMM as the K tail of the last experts (against zero
// pad rows): they are zeroed so that they hold finite values.
__global__ void k_bwd_tail_zero(const int32_t *__restrict__ offset, int E, long long A_rows,
                                int d, int d_ff, __nv_bfloat16 *__restrict__ xbuf,
                                __nv_bfloat16 *__restrict__ hbuf) {
  pdl_wait();
  const long long a0 = offset[E];
  const long long r1 = a0 + kRowPad < A_rows ? a0 + kRowPad : A_rows;
  const long long nx = (r1 - a0) * (d / 8), nh = (r1 - a0) * (d_ff / 8);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nx + nh;
       i += (long long)gridDim.x * blockDim.x) {
    if (i < nx)
      reinterpret_cast<uint4 *>(xbuf + a0 * d)[i] = z;
    else
      reinterpret_cast<uint4 *>(hbuf + a0 * d_ff)[i - nx] = z;
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- dy gather
// One warp per padded row: a real row gets dy of its token (dY) and
// g * dy (dU), both bf16; a pad row gets zeros.
__global__ void __launch_bounds__(256)
k_bwd_gather(long long P_max, int E, int k, int d, const int32_t *__restrict__ offset,
             const int32_t *__restrict__ poff, const int32_t *__restrict__ row_token,
             const float *__restrict__ row_gate, const __nv_bfloat16 *__restrict__ dy,
             __nv_bfloat16 *__restrict__ dY, __nv_bfloat16 *__restrict__ dU) {
  pdl_wait();
  const long long pr = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (pr >= P_max || pr >= poff[E]) {
    pdl_trigger();
    return;
  }
  const int e = find_block(poff, E, (int)pr);
  const int m = (int)(pr - poff[e]);
  const int rows = offset[e + 1] - offset[e];
  const int nv = d / 8;
  uint4 *oy = reinterpret_cast<uint4 *>(dY + pr * d);
  uint4 *ou = reinterpret_cast<uint4 *>(dU + pr * d);
  if (m < rows) {
    const int q = offset[e] + m;
    const int t = row_token[q] / k;
    const float g = row_gate[q];
    const uint4 *src = reinterpret_cast<const uint4 *>(dy + (size_t)t * d);
    for (int v = lane; v < nv; v += 32) {
      const uint4 u = src[v];
      oy[v] = u;
      float f[8];
      bf16x8_to_f32(u, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] *= g;
      ou[v] = f32_to_bf16x8(f);
    }
  } else {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = lane; v < nv; v += 32) {
      oy[v] = z;
      ou[v] = z;
    }
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- gate gradient per kept choice
// dg[a] = sum over the dgrad GEMM's column blocks of <D_r, h_r> + <dy_t, b2_e>,
// for the assignment a = t*k + j of packed row q (one warp per row).
__global__ void __launch_bounds__(256)
k_bwd_dg(int E, int k, int d, int n_blocks, const int32_t *__restrict__ offset,
         const int32_t *__restrict__ poff, const int32_t *__restrict__ row_token,
         const float *__restrict__ dgpart, const __nv_bfloat16 *__restrict__ dy,
         const __nv_bfloat16 *__restrict__ b2, float *__restrict__ dg) {
  pdl_wait();
  const long long q = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (q >= offset[E]) {
    pdl_trigger();
    return;
  }
  const int e = find_block(offset, E, (int)q);
  const long long pr = poff[e] + (q - offset[e]);
  const int a = row_token[q];
  float s = 0.f;
  for (int nb = lane; nb < n_blocks; nb += 32) s += dgpart[pr * n_blocks + nb];
  if (b2) {
    const int t = a / k;
    const uint4 *yv = reinterpret_cast<const uint4 *>(dy + (size_t)t * d);
    const uint4 *bv = reinterpret_cast<const uint4 *>(b2 + (size_t)e * d);
    for (int v = lane; v < d / 8; v += 32) {
      float fy[8], fb[8];
      bf16x8_to_f32(yv[v], fy);
      bf16x8_to_f32(bv[v], fb);
#pragma unroll
      for (int j = 0; j < 8; ++j) s = fmaf(fy[j], fb[j], s);
    }
  }
  s = warp_sum(s);
  if (lane == 0) dg[a] = s;
  pdl_trigger();
}

// ----------------------------------------------------------------------------- loss coefficients
// coef[0][e] = w_imp  * d CV(Importance)^2 / d Importance_e
// coef[1][e] = w_load * d CV(Load)^2 / d Load_e
//     d (var / m^2) / d v_e = 2 (v_e - m) / (E m^2) - 2 var / (E m^3)
// coef[2][e] = w_aux * 0.01 * E * f_e / T   (dL/dp_{t,e} of the Switch loss)
// from the forward's balancing totals aux [4][E] (double-float pairs:
// importance, load, f, Pbar); fp64, one block, fixed order. A term whose
// weight is 0 is 0 without reading its totals (they may never have been
// formed).
__global__ void __launch_bounds__(256)
k_bwd_coef(int T, int E, const float2 *__restrict__ aux, float w_imp, float w_load, float w_aux,
           float *__restrict__ coef) {
  pdl_wait();
  __shared__ double stat[4];
  const float wq[2] = {w_imp, w_load};
  if (threadIdx.x < 2 && wq[threadIdx.x] != 0.f) {
    const int q = threadIdx.x;
    double m = 0.0;
    for (int e = 0; e < E; ++e) m += (double)aux[q * E + e].x + (double)aux[q * E + e].y;
    m /= E;
    double var = 0.0;
    for (int e = 0; e < E; ++e) {
      const double v = (double)aux[q * E + e].x + (double)aux[q * E + e].y - m;
      var += v * v;
    }
    stat[2 * q] = m;
    stat[2 * q + 1] = var / E;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float out = 0.f;
      if (wq[q] != 0.f) {
        const double m = stat[2 * q], var = stat[2 * q + 1];
        const double v = (double)aux[q * E + e].x + (double)aux[q * E + e].y;
        if (m > 0.0)
          out = (float)((double)wq[q] *
                        (2.0 * (v - m) / (E * m * m) - 2.0 * var / (E * m * m * m)));
      }
      coef[q * E + e] = out;
    }
    float fo = 0.f;
    if (w_aux != 0.f) {
      const double f = (double)aux[2 * E + e].x + (double)aux[2 * E + e].y;
      fo = (float)((double)w_aux * 0.01 * E * f / T);
    }
    coef[2 * E + e] = fo;
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- gate backward
struct GateBwd {
  int T, E, k, mode, noisy, load_on, aux_on, dg_total;
  const float *H, *c, *sigma, *noise, *rowstat, *thr, *gate;
  const int32_t *idx;
  const uint8_t *keep;
  const float *dg;    // dg_total: dL/dgate [T,k]; else the kept choices' <dy, U> by assignment
  const float *coef;  // [3][E]
  float *dgate_out;   // [T,k] or null
  float *dc, *dz;     // [T,E]
};

// One warp per token. Pass 1: the softmax inner product, the load terms'
// sums per threshold owner and the (k+1)-th pick; pass 2: dH, dc and dz.
__global__ void __launch_bounds__(256) k_bwd_gate(const GateBwd p) {
  pdl_wait();
  const int t = (int)((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= p.T) {
    pdl_trigger();
    return;
  }
  const int E = p.E, k = p.k;
  const size_t row = (size_t)t * E;
  int ch[16];
  float tk[16];
  float mydg = 0.f, myg = 0.f;
  int myi = -1;
  if (lane < k) {
    myi = p.idx[(size_t)t * k + lane];
    myg = p.gate[(size_t)t * k + lane];
    if (p.dg_total) {
      mydg = p.dg[(size_t)t * k + lane];
    } else {
      mydg = (p.keep[(size_t)t * k + lane] ? p.dg[(size_t)t * k + lane] : 0.f) + p.coef[myi];
    }
    if (p.dgate_out) p.dgate_out[(size_t)t * k + lane] = mydg;
  }
  const float s = warp_sum(lane < k ? myg * mydg : 0.f);
  const float mytk = lane < k ? myg * (mydg - s) : 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    ch[j] = __shfl_sync(0xffffffffu, myi, j);
    tk[j] = __shfl_sync(0xffffffffu, mytk, j);
  }
  const bool sw = p.mode == MOE_GATE_SWITCH;
  const bool soft = sw || p.aux_on;
  const float dG0 = __shfl_sync(0xffffffffu, mydg, 0);
  const float mx = p.rowstat[2 * (size_t)t], inv_se = 1.f / p.rowstat[2 * (size_t)t + 1];
  const float hk = p.thr[2 * (size_t)t], hk1 = p.thr[2 * (size_t)t + 1];
  const float *cc = p.noisy ? p.c : p.H;
  const float inv_sqrt_2pi = 0.3989422804014327f;
  // Pass 1.
  float pd = 0.f, sA = 0.f, sB = 0.f;
  float bestv = -INFINITY;
  int besti = 0x7fffffff;
  for (int e = lane; e < E; e += 32) {
    bool chosen = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) chosen |= j < k && ch[j] == e;
    const float h = p.H[row + e];
    if (soft) {
      const float pe = expf(h - mx) * inv_se;
      const float dp = p.coef[2 * E + e] + (sw && e == ch[0] ? dG0 : 0.f);
      pd = fmaf(pe, dp, pd);
    }
    if (p.load_on) {
      if (!chosen && (h > bestv || (h == bestv && e < besti))) {
        bestv = h;
        besti = e;
      }
      const float sg = p.sigma[row + e];
      if (sg > 0.f) {
        const float u = (cc[row + e] - (chosen ? hk1 : hk)) / sg;
        const float gl = p.coef[E + e] * (expf(-0.5f * u * u) * inv_sqrt_2pi) / sg;
        if (chosen) sA += gl;
        else sB += gl;
      }
    }
  }
  pd = warp_sum(pd);
  sA = warp_sum(sA);
  sB = warp_sum(sB);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bestv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
    if (ov > bestv || (ov == bestv && oi < besti)) {
      bestv = ov;
      besti = oi;
    }
  }
  int kth = -1;  // the k-th pick: the threshold owner for experts not chosen
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j == k - 1) kth = ch[j];
  // Pass 2.
  for (int e = lane; e < E; e += 32) {
    bool chosen = false;
    float dH = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < k && ch[j] == e) {
        chosen = true;
        if (!sw) dH += tk[j];
      }
    const float h = p.H[row + e];
    if (soft) {
      const float pe = expf(h - mx) * inv_se;
      const float dp = p.coef[2 * E + e] + (sw && e == ch[0] ? dG0 : 0.f);
      dH = fmaf(pe, dp - pd, dH);
    }
    float dcl = 0.f, dsl = 0.f;
    if (p.load_on) {
      if (e == besti) dH -= sA;
      if (e == kth) dH -= sB;
      const float sg = p.sigma[row + e];
      if (sg > 0.f) {
        const float u = (cc[row + e] - (chosen ? hk1 : hk)) / sg;
        const float gl = p.coef[E + e] * (expf(-0.5f * u * u) * inv_sqrt_2pi) / sg;
        dcl = gl;
        dsl = -gl * u;
      }
    }
    p.dc[row + e] = dH + dcl;
    if (p.noisy) {
      const float sg = p.sigma[row + e];
      const float dsg = fmaf(p.noise[row + e], dH, dsl);
      p.dz[row + e] = dsg * -expm1f(-sg);  // sigmoid(z) = 1 - exp(-Softplus(z))
    }
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- router weight gradients
// dW[i][col] = sum_t x[t][i] * D[t][col] over the columns D = [dc | dz]
// (dWg then dW_noise), split over token chunks into partials [S][d][NC];
// the blocks of the first i tile also sum the columns of D (the bias).
constexpr int kXtdTI = 64, kXtdTC = 32, kXtdTT = 32;

__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }

template <typename XT>
__global__ void __launch_bounds__(256)
k_bwd_xtd(int T, int d, int E, int NC, int tpc, const XT *__restrict__ x,
          const float *__restrict__ dc, const float *__restrict__ dz, float *__restrict__ part,
          float *__restrict__ bpart) {
  pdl_wait();
  __shared__ float xs[kXtdTT][kXtdTI];
  __shared__ float ds[kXtdTT][kXtdTC + 1];
  const int i0 = blockIdx.x * kXtdTI, c0 = blockIdx.y * kXtdTC, sidx = blockIdx.z;
  const int t_begin = sidx * tpc, t_end = min(T, t_begin + tpc);
  const int ti = threadIdx.x & 63, cg = threadIdx.x >> 6;  // 4 groups of 8 columns
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float bsum = 0.f;  // thread < kXtdTC of the first i tile: column sum
  for (int tb = t_begin; tb < t_end; tb += kXtdTT) {
    for (int u = threadIdx.x; u < kXtdTT * kXtdTI; u += 256) {
      const int tt = u / kXtdTI, ii = u % kXtdTI;
      const int t = tb + tt, i = i0 + ii;
      xs[tt][ii] = (t < t_end && i < d) ? to_f(x[(size_t)t * d + i]) : 0.f;
    }
    for (int u = threadIdx.x; u < kXtdTT * kXtdTC; u += 256) {
      const int tt = u / kXtdTC, cc = u % kXtdTC;
      const int t = tb + tt, col = c0 + cc;
      float v = 0.f;
      if (t < t_end && col < NC)
        v = col < E ? dc[(size_t)t * E + col] : dz[(size_t)t * E + (col - E)];
      ds[tt][cc] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int tt = 0; tt < kXtdTT; ++tt) {
      const float xv = xs[tt][ti];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(xv, ds[tt][cg * 8 + j], acc[j]);
    }
    if (blockIdx.x == 0 && threadIdx.x < kXtdTC)
      for (int tt = 0; tt < kXtdTT; ++tt) bsum += ds[tt][threadIdx.x];
    __syncthreads();
  }
  const int i = i0 + ti;
  if (i < d)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = c0 + cg * 8 + j;
      if (col < NC) part[((size_t)sidx * d + i) * NC + col] = acc[j];
    }
  if (blockIdx.x == 0 && threadIdx.x < kXtdTC && c0 + threadIdx.x < NC)
    bpart[(size_t)sidx * NC + c0 + threadIdx.x] = bsum;
  pdl_trigger();
}

// The same partials for a narrow router (NC = E or 2E columns, NC <= 32, E a
// multiple of 4, bf16 x), together with the router's share of dx, in one
// pass. Thread i of block (256-feature tile, token chunk) owns feature i: per
// step of TT tokens it loads its x[t][i] for all TT tokens at once (the
// block's loads of a token are 512 contiguous bytes, and TT of them are in
// flight per thread), the block stages the TT rows of D in shared memory, and
// the thread adds x[t][i] D[t][col] to its NC sums and (with dxr) stores
// dxr[t][i] = sum_col D[t][col] W'[col][i] from W' values held in registers.
// The tiled kernels above take 64 x 32 output tiles with K = the tokens;
// at NC = 16 half their threads computed zero columns, and dxr went through
// a second pass over D.
constexpr int kNarrowNC = 32;
constexpr int kNarrowFeat = 256;  // features per block

template <int NCM, int TT>  // NCM >= NC, a multiple of 4; TT tokens per step
__global__ void __launch_bounds__(256)
k_bwd_router_narrow(int T, int d, int E, int NC, int tpc, const __nv_bfloat16 *__restrict__ x,
                    const float *__restrict__ dc, const float *__restrict__ dz,
                    const float *__restrict__ Wg, const float *__restrict__ Wn,
                    float *__restrict__ part, float *__restrict__ bpart,
                    float *__restrict__ dxr) {
  pdl_wait();
  __shared__ __align__(16) float Ds[TT][NCM];
  const int i = blockIdx.x * kNarrowFeat + threadIdx.x, sidx = blockIdx.y;
  const int t_begin = sidx * tpc, t_end = min(T, t_begin + tpc);
  const bool feat = i < d;
  float w[NCM], acc[NCM];
#pragma unroll
  for (int c = 0; c < NCM; ++c) {
    acc[c] = 0.f;
    w[c] = 0.f;
    if (dxr && feat && c < NC) w[c] = c < E ? Wg[(size_t)i * E + c] : Wn[(size_t)i * E + c - E];
  }
  const bool bcol = blockIdx.x == 0 && (int)threadIdx.x < NC;  // the bias column sums
  float bsum = 0.f;
  for (int tb = t_begin; tb < t_end; tb += TT) {
    const int nt = min(TT, t_end - tb);
    float xv[TT];
#pragma unroll
    for (int u = 0; u < TT; ++u)
      xv[u] = (feat && u < nt) ? __bfloat162float(x[(size_t)(tb + u) * d + i]) : 0.f;
    __syncthreads();  // the previous step's rows of D are no longer read
    for (int q = threadIdx.x; q < TT * NCM; q += blockDim.x) {
      const int u = q / NCM, c = q - u * NCM;
      float v = 0.f;
      if (u < nt && c < NC)
        v = c < E ? dc[(size_t)(tb + u) * E + c] : dz[(size_t)(tb + u) * E + c - E];
      Ds[u][c] = v;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < TT; ++u) {
      float D[NCM];
#pragma unroll
      for (int q = 0; q < NCM / 4; ++q) {
        const float4 v = reinterpret_cast<const float4 *>(Ds[u])[q];
        D[4 * q] = v.x;
        D[4 * q + 1] = v.y;
        D[4 * q + 2] = v.z;
        D[4 * q + 3] = v.w;
      }
      float r = 0.f;
#pragma unroll
      for (int c = 0; c < NCM; ++c) {
        acc[c] = fmaf(xv[u], D[c], acc[c]);
        r = fmaf(D[c], w[c], r);
      }
      if (dxr && feat && u < nt) dxr[(size_t)(tb + u) * d + i] = r;
      if (bcol) bsum += Ds[u][threadIdx.x];
    }
  }
  if (feat)
#pragma unroll
    for (int c = 0; c < NCM; ++c)
      if (c < NC) part[((size_t)sidx * d + i) * NC + c] = acc[c];
  if (bcol) bpart[(size_t)sidx * NC + threadIdx.x] = bsum;
  pdl_trigger();
}

// Sum the partials over the token chunks in order: dWg [d,E], dWn [d,E], dbias [E].
__global__ void k_bwd_xtd_reduce(int d, int E, int NC, int S, const float *__restrict__ part,
                                 const float *__restrict__ bpart, float *__restrict__ dWg,
                                 float *__restrict__ dWn, float *__restrict__ dbias) {
  pdl_wait();
  const long long n = (long long)d * NC;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n + NC;
       u += (long long)gridDim.x * blockDim.x) {
    if (u < n) {
      float s = 0.f;
      for (int q = 0; q < S; ++q) s += part[(size_t)q * n + u];
      const int i = (int)(u / NC), col = (int)(u % NC);
      if (col < E) dWg[(size_t)i * E + col] = s;
      else dWn[(size_t)i * E + col - E] = s;
    } else {
      const int col = (int)(u - n);
      if (col < E && dbias) {
        float s = 0.f;
        for (int q = 0; q < S; ++q) s += bpart[(size_t)q * NC + col];
        dbias[col] = s;
      }
    }
  }
  pdl_trigger();
}

// dxr[t][i] = sum_col D[t][col] W'[col][i], W' = [W_g^T ; W_noise^T]: the
// router's share of dx. 64 tokens x 64 features per block, 4 x 4 per thread.
constexpr int kDxrT = 64, kDxrI = 64, kDxrC = 16;

__global__ void __launch_bounds__(256)
k_bwd_dxr(int T, int d, int E, int NC, const float *__restrict__ dc, const float *__restrict__ dz,
          const float *__restrict__ Wg, const float *__restrict__ Wn, float *__restrict__ dxr) {
  pdl_wait();
  __shared__ float Ds[kDxrC][kDxrT + 1];
  __shared__ float Ws[kDxrC][kDxrI + 1];
  const int t0 = blockIdx.y * kDxrT, i0 = blockIdx.x * kDxrI;
  const int tq = threadIdx.x >> 4, iq = threadIdx.x & 15;
  float acc[4][4] = {};
  for (int c0 = 0; c0 < NC; c0 += kDxrC) {
    for (int u = threadIdx.x; u < kDxrT * kDxrC; u += 256) {
      const int tt = u / kDxrC, cc = u % kDxrC;
      const int t = t0 + tt, col = c0 + cc;
      float v = 0.f;
      if (t < T && col < NC) v = col < E ? dc[(size_t)t * E + col] : dz[(size_t)t * E + col - E];
      Ds[cc][tt] = v;
    }
    for (int u = threadIdx.x; u < kDxrI * kDxrC; u += 256) {
      const int ii = u / kDxrC, cc = u % kDxrC;
      const int i = i0 + ii, col = c0 + cc;
      float v = 0.f;
      if (i < d && col < NC) v = col < E ? Wg[(size_t)i * E + col] : Wn[(size_t)i * E + col - E];
      Ws[cc][ii] = v;
    }
    __syncthreads();
#pragma unroll
    for (int cc = 0; cc < kDxrC; ++cc) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = Ds[cc][tq * 4 + r];
        b[r] = Ws[cc][iq + 16 * r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(a[r], b[q], acc[r][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = t0 + tq * 4 + r;
    if (t >= T) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + iq + 16 * q;
      if (i < d) dxr[(size_t)t * d + i] = acc[r][q];
    }
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- expert bias gradients
// out[e][c] = sum over the expert's real rows m of s_m * src[poff[e] + m][c]
// (s_m = row_gate of the packed row when given, else 1): partial sums over
// chunks of 128 rows, then the chunks in order.
constexpr int kColRows = 128;

template <typename S>
__global__ void __launch_bounds__(256)
k_bwd_colsum(int E, int cols, int chunks, const int32_t *__restrict__ offset,
             const int32_t *__restrict__ poff, const float *__restrict__ row_gate,
             const S *__restrict__ src, float *__restrict__ part) {
  pdl_wait();
  const int c = blockIdx.x * 256 + threadIdx.x, e = blockIdx.y, ch = blockIdx.z;
  if (c < cols) {
    const int rows = offset[e + 1] - offset[e];
    const int m0 = ch * kColRows, m1 = min(rows, m0 + kColRows);
    float s = 0.f;
    for (int m = m0; m < m1; ++m) {
      const float v = to_f(src[((size_t)poff[e] + m) * cols + c]);
      s = row_gate ? fmaf(row_gate[offset[e] + m], v, s) : s + v;
    }
    part[((size_t)ch * E + e) * cols + c] = s;
  }
  pdl_trigger();
}

__global__ void k_bwd_colsum_reduce(int E, int cols, int chunks, const float *__restrict__ part,
                                    float *__restrict__ out) {
  pdl_wait();
  const long long n = (long long)E * cols;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n;
       u += (long long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < chunks; ++q) s += part[(size_t)q * n + u];
    out[u] = s;
  }
  pdl_trigger();
}

// ----------------------------------------------------------------------------- input gradient
// dx_t = dy_t + dxr_t + sum over kept choices j (in order) of dX[poff[e_j] + pos_j]
// (one warp per token, 8 features per lane step; fp32 sums, bf16 out).
__global__ void __launch_bounds__(256)
k_bwd_dx(int T, int d, int k, const int32_t *__restrict__ idx, const int32_t *__restrict__ pos,
         const uint8_t *__restrict__ keep, const int32_t *__restrict__ poff,
         const float *__restrict__ dX, const float *__restrict__ dxr,
         const __nv_bfloat16 *__restrict__ dy, __nv_bfloat16 *__restrict__ dx) {
  pdl_wait();
  const long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) {
    pdl_trigger();
    return;
  }
  long long rows[16];
  int nk = 0;
  for (int j = 0; j < k; ++j)
    if (keep[t * k + j]) rows[nk++] = (long long)poff[idx[t * k + j]] + pos[t * k + j];
  const uint4 *yv = reinterpret_cast<const uint4 *>(dy + t * d);
  uint4 *ov = reinterpret_cast<uint4 *>(dx + t * d);
  for (int v = lane; v < d / 8; v += 32) {
    float f[8];
    bf16x8_to_f32(yv[v], f);
    if (dxr) {
      const float4 *r = reinterpret_cast<const float4 *>(dxr + t * d + 8 * v);
      const float4 a = r[0], b = r[1];
      f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w;
      f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
    }
    for (int j = 0; j < nk; ++j) {
      const float4 *r = reinterpret_cast<const float4 *>(dX + rows[j] * d + 8 * v);
      const float4 a = r[0], b = r[1];
      f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w;
      f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
    }
    ov[v] = f32_to_bf16x8(f);
  }
  pdl_trigger();
}

int grid_for(long long work, int per_block) {
  long long b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > 0x7fffffffLL) b = 0x7fffffffLL;
  return (int)b;
}

}  // namespace

// Token chunks of the router's weight-gradient partials: about four blocks
// per SM for whichever kernel runs (the narrow one for NC <= 32 columns, one
// block per 256 features; the tiled one per 64 x 32 tile).
int xtd_splits(int T, int d, int NC) {
  const long long tiles =
      NC <= kNarrowNC
          ? (long long)((d + kNarrowFeat - 1) / kNarrowFeat)
          : (long long)((d + kXtdTI - 1) / kXtdTI) * ((NC + kXtdTC - 1) / kXtdTC);
  long long S = (4LL * sm_count() + tiles - 1) / tiles;
  const long long maxS = (T + kXtdTT - 1) / kXtdTT;
  if (S > maxS) S = maxS;
  if (S < 1) S = 1;
  return (int)S;
}

int colsum_chunks(int C) { return (C + kColRows - 1) / kColRows; }

cudaError_t launch_bwd_offsets(int E, const int32_t *offset, int32_t *poff, cudaStream_t s) {
  return launch_pdl(k_bwd_offsets, 1, 1024, 0, s, E, offset, poff);
}

cudaError_t launch_bwd_tail_zero(const moe_config &c, const int32_t *offset, void *xbuf,
                                 void *hbuf, cudaStream_t s) {
  const long long n = (long long)kRowPad * (c.d + c.d_ff) / 8;
  return launch_pdl(k_bwd_tail_zero, grid_for(n, 256), 256, 0, s, offset, c.E,
                    (long long)c.T * c.k, c.d, c.d_ff, static_cast<__nv_bfloat16 *>(xbuf),
                    static_cast<__nv_bfloat16 *>(hbuf));
}

cudaError_t launch_bwd_gather(const moe_config &c, long long P_max, const int32_t *offset,
                              const int32_t *poff, const int32_t *row_token,
                              const float *row_gate, const void *dy, void *dY, void *dU,
                              cudaStream_t s) {
  return launch_pdl(k_bwd_gather, grid_for(P_max, 8), 256, 0, s, P_max, c.E, c.k, c.d, offset,
                    poff, row_token, row_gate, static_cast<const __nv_bfloat16 *>(dy),
                    static_cast<__nv_bfloat16 *>(dY), static_cast<__nv_bfloat16 *>(dU));
}

cudaError_t launch_bwd_dg(const moe_config &c, int n_blocks, const int32_t *offset,
                          const int32_t *poff, const int32_t *row_token, const float *dgpart,
                          const void *dy, const void *b2, float *dg, cudaStream_t s) {
  return launch_pdl(k_bwd_dg, grid_for((long long)c.T * c.k, 8), 256, 0, s, c.E, c.k, c.d,
                    n_blocks, offset, poff, row_token, dgpart,
                    static_cast<const __nv_bfloat16 *>(dy), static_cast<const __nv_bfloat16 *>(b2),
                    dg);
}

cudaError_t launch_bwd_coef(const moe_config &c, const float2 *aux_vec, float w_imp,
                            float w_load, float w_aux, float *coef, cudaStream_t s) {
  return launch_pdl(k_bwd_coef, 1, 256, 0, s, c.T, c.E, aux_vec, w_imp, w_load, w_aux, coef);
}

cudaError_t launch_bwd_gate(const moe_config &c, bool noisy, bool load_on, bool aux_on,
                            bool dg_total, const float *H, const float *cc, const float *sigma,
                            const float *noise, const float *rowstat, const float *thr,
                            const int32_t *idx, const float *gate, const uint8_t *keep,
                            const float *dg, const float *coef, float *dgate_out, float *dc,
                            float *dz, cudaStream_t s) {
  GateBwd p{c.T, c.E, c.k, c.gate_mode, noisy ? 1 : 0, load_on ? 1 : 0, aux_on ? 1 : 0,
            dg_total ? 1 : 0, H, cc, sigma, noise, rowstat, thr, gate, idx, keep, dg, coef,
            dgate_out, dc, dz};
  return launch_pdl(k_bwd_gate, grid_for(c.T, 8), 256, 0, s, p);
}

cudaError_t launch_bwd_router(const moe_config &c, bool noisy, const void *x, const float *Wg,
                              const float *Wn, const float *dc, const float *dz, float *part,
                              float *bpart, float *dWg, float *dWn, float *dbias, float *dxr,
                              cudaStream_t s) {
  const int NC = noisy ? 2 * c.E : c.E;
  const int S = xtd_splits(c.T, c.d, NC);  // part holds S * d * NC, bpart S * NC floats
  const int tpc = ((c.T + S - 1) / S + kXtdTT - 1) / kXtdTT * kXtdTT;
  if (c.act_dtype == MOE_BF16 && NC <= kNarrowNC && c.E % 4 == 0) {
    // One pass for the weight gradients' partials and the share of dx.
    const dim3 gn((c.d + kNarrowFeat - 1) / kNarrowFeat, S);
    cudaError_t err =
        NC <= 16 ? launch_pdl(k_bwd_router_narrow<16, 32>, gn, 256, 0, s, c.T, c.d, c.E, NC, tpc,
                              static_cast<const __nv_bfloat16 *>(x), dc, dz, Wg, Wn, part, bpart,
                              dxr)
                 : launch_pdl(k_bwd_router_narrow<kNarrowNC, 16>, gn, 256, 0, s, c.T, c.d, c.E,
                              NC, tpc, static_cast<const __nv_bfloat16 *>(x), dc, dz, Wg, Wn,
                              part, bpart, dxr);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_bwd_xtd_reduce, grid_for((long long)c.d * NC + NC, 256), 256, 0, s, c.d,
                      c.E, NC, S, (const float *)part, (const float *)bpart, dWg, dWn, dbias);
  }
  const dim3 g1((c.d + kXtdTI - 1) / kXtdTI, (NC + kXtdTC - 1) / kXtdTC, S);
  cudaError_t err =
      c.act_dtype == MOE_BF16
          ? launch_pdl(k_bwd_xtd<__nv_bfloat16>, g1, 256, 0, s, c.T, c.d, c.E, NC, tpc,
                       static_cast<const __nv_bfloat16 *>(x), dc, dz, part, bpart)
          : launch_pdl(k_bwd_xtd<float>, g1, 256, 0, s, c.T, c.d, c.E, NC, tpc,
                       static_cast<const float *>(x), dc, dz, part, bpart);
  if (err != cudaSuccess) return err;
  err = launch_pdl(k_bwd_xtd_reduce, grid_for((long long)c.d * NC + NC, 256), 256, 0, s, c.d,
                   c.E, NC, S, (const float *)part, (const float *)bpart, dWg, dWn, dbias);
  if (err != cudaSuccess) return err;
  if (!dxr) return cudaSuccess;
  const dim3 g2((c.d + kDxrI - 1) / kDxrI, (c.T + kDxrT - 1) / kDxrT);
  return launch_pdl(k_bwd_dxr, g2, 256, 0, s, c.T, c.d, c.E, NC, dc, dz, Wg, Wn, dxr);
}

cudaError_t launch_bwd_colsum(const moe_config &c, int cols, int chunks, const int32_t *offset,
                              const int32_t *poff, const float *row_gate, const void *src,
                              bool src_f32, float *part, float *out, cudaStream_t s) {
  const dim3 g((cols + 255) / 256, c.E, chunks);
  cudaError_t err =
      src_f32 ? launch_pdl(k_bwd_colsum<float>, g, 256, 0, s, c.E, cols, chunks, offset, poff,
                           row_gate, static_cast<const float *>(src), part)
              : launch_pdl(k_bwd_colsum<__nv_bfloat16>, g, 256, 0, s, c.E, cols, chunks, offset,
                           poff, row_gate, static_cast<const __nv_bfloat16 *>(src), part);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_bwd_colsum_reduce, grid_for((long long)c.E * cols, 256), 256, 0, s, c.E,
                    cols, chunks, (const float *)part, out);
}

// Launched in plain stream order (no programmatic dependent launch): it
// follows a join with the side stream, whose results (the router's share of
// dx) it reads.
cudaError_t launch_bwd_dx(const moe_config &c, const int32_t *idx, const int32_t *pos,
                          const uint8_t *keep, const int32_t *poff, const float *dX,
                          const float *dxr, const void *dy, void *dx, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(c.T, 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, k_bwd_dx, c.T, c.d, c.k, idx, pos, keep, poff, dX, dxr,
                            static_cast<const __nv_bfloat16 *>(dy),
                            static_cast<__nv_bfloat16 *>(dx));
}

}  // namespace moe
