// Stages 1-2 and the balancing sums of stage 5.
//
// Router ("Outrageously Large Neural Networks", section 3.4, Noisy Top-K Gating
// step 1, Eq. 4; "Switch Transformer", step 1: the router runs in fp32):
//   c = x Wg + b,  sigma = Softplus(x Wnoise),  H = c + noise * sigma.
// Selection (Eq. 5 / Switch step 2): the k largest H in (value desc, index asc)
// order, gates = softmax over them (TOPK) or the full-softmax probability of
// the argmax (SWITCH).
// Balancing sums (Eqs. 6-10; Switch step 8): per-block partial sums in token
// order, finished in fp64 by one block, so results are run-to-run identical.
#include "moe_internal.cuh"

#include <math.h>
#include <stdlib.h>

namespace moe {
namespace {

constexpr int kRtTok = 32;     // tokens per router block (one per lane)
constexpr int kRtWarps = 8;    // warps per router block; each takes a slice of each K chunk
constexpr int kRtKC = 256;     // K chunk staged in shared memory
constexpr int kRtXPitch = kRtKC + 1;
constexpr int kMaxK = 16;      // largest k the selection kernel keeps in registers

__device__ __forceinline__ float load_act(const void *p, int dtype, size_t i) {
  if (dtype == MOE_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  return static_cast<const float *>(p)[i];
}

__device__ __forceinline__ float softplus_f(float z) {
  // log(1 + e^z) without overflow: max(z, 0) + log1p(exp(-|z|)).
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}

// One block: kRtTok tokens x BE experts. Lane = token; warp w accumulates the
// w-th slice of every staged K chunk; the slices are added in warp order.
template <int BE, bool NOISY>
__global__ void __launch_bounds__(kRtWarps * 32)
k_router(int T, int d, int E, const void *__restrict__ x, int xdtype, const float *__restrict__ Wg,
         const float *__restrict__ Wn, const float *__restrict__ noise,
         const float *__restrict__ bias, float *__restrict__ c_out, float *__restrict__ s_out,
         float *__restrict__ H_out, DeviceStatus *st) {
  extern __shared__ float4 smem4[];
  float *smem = reinterpret_cast<float *>(smem4);
  float *xs = smem;                                  // [kRtTok][kRtXPitch]
  float *wgs = xs + kRtTok * kRtXPitch;              // [kRtKC][BE]
  float *wns = wgs + kRtKC * BE;                     // [kRtKC][BE] (NOISY)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTok;
  const int e0 = blockIdx.y * BE;

  float accc[BE], accz[NOISY ? BE : 1];
#pragma unroll
  for (int e = 0; e < BE; ++e) accc[e] = 0.f;
#pragma unroll
  for (int e = 0; e < (NOISY ? BE : 1); ++e) accz[e] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kRtKC) {
    __syncthreads();
    for (int i = tid; i < kRtTok * kRtKC; i += blockDim.x) {
      int r = i / kRtKC, kk = i % kRtKC;
      int t = t0 + r, k = k0 + kk;
      xs[r * kRtXPitch + kk] = (t < T && k < d) ? load_act(x, xdtype, (size_t)t * d + k) : 0.f;
    }
    for (int i = tid; i < kRtKC * BE; i += blockDim.x) {
      int kk = i / BE, e = i % BE;
      int k = k0 + kk, ee = e0 + e;
      bool ok = k < d && ee < E;
      wgs[i] = ok ? Wg[(size_t)k * E + ee] : 0.f;
      if (NOISY) wns[i] = ok ? Wn[(size_t)k * E + ee] : 0.f;
    }
    __syncthreads();
    constexpr int kSlice = kRtKC / kRtWarps;
    const float *xrow = xs + lane * kRtXPitch + warp * kSlice;
    const float *wg = wgs + warp * kSlice * BE;
    const float *wn = wns + warp * kSlice * BE;
#pragma unroll 4
    for (int kk = 0; kk < kSlice; ++kk) {
      float xv = xrow[kk];
#pragma unroll
      for (int e = 0; e < BE; ++e) accc[e] = fmaf(xv, wg[kk * BE + e], accc[e]);
      if (NOISY) {
#pragma unroll
        for (int e = 0; e < BE; ++e) accz[e] = fmaf(xv, wn[kk * BE + e], accz[e]);
      }
    }
  }
  __syncthreads();
  // Cross-warp sum in warp order through shared memory (reuses the staging area).
  constexpr int kVals = NOISY ? 2 * BE : BE;
  float *red = smem;  // [kRtWarps][kRtTok][kVals]
#pragma unroll
  for (int e = 0; e < BE; ++e) red[(warp * kRtTok + lane) * kVals + e] = accc[e];
  if (NOISY) {
#pragma unroll
    for (int e = 0; e < BE; ++e) red[(warp * kRtTok + lane) * kVals + BE + e] = accz[e];
  }
  __syncthreads();
  for (int i = tid; i < kRtTok * BE; i += blockDim.x) {
    int r = i / BE, e = i % BE;
    int t = t0 + r, ee = e0 + e;
    if (t >= T || ee >= E) continue;
    float cv = 0.f, zv = 0.f;
    for (int w = 0; w < kRtWarps; ++w) {
      cv += red[(w * kRtTok + r) * kVals + e];
      if (NOISY) zv += red[(w * kRtTok + r) * kVals + BE + e];
    }
    if (bias) cv += bias[ee];
    float sg = 0.f, h = cv;
    if (NOISY) {
      sg = softplus_f(zv);
      h = fmaf(noise[(size_t)t * E + ee], sg, cv);
    }
    size_t o = (size_t)t * E + ee;
    c_out[o] = cv;
    s_out[o] = sg;
    H_out[o] = h;
    if (!isfinite(h)) record_error(st, MOE_ERR_NONFINITE, (long long)o);
  }
}

template <int BE, bool NOISY>
cudaError_t run_router(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                       const float *noise, const float *bias, float *c, float *s, float *H,
                       DeviceStatus *st, cudaStream_t stream) {
  size_t xs = (size_t)kRtTok * kRtXPitch * 4;
  size_t ws = (size_t)kRtKC * BE * 4 * (NOISY ? 2 : 1);
  size_t red = (size_t)kRtWarps * kRtTok * (NOISY ? 2 : 1) * BE * 4;
  size_t smem = xs + ws > red ? xs + ws : red;
  auto kern = k_router<BE, NOISY>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((cfg.T + kRtTok - 1) / kRtTok, (cfg.E + BE - 1) / BE);
  kern<<<grid, kRtWarps * 32, smem, stream>>>(cfg.T, cfg.d, cfg.E, x, cfg.act_dtype, Wg, Wn, noise,
                                               bias, c, s, H, st);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- router, vector path
// The same arithmetic as k_router, laid out for streaming: each warp owns TPW
// tokens over the whole K range and its lanes split K (lane l takes
// k = l, l+32, ... of each 256-wide chunk); x rows (16-byte cp.async) and the
// W chunk (cp.async) are double-buffered in shared memory, so loads of chunk
// c+1 overlap the FMAs of chunk c. The lanes' partial sums are combined by a
// fixed xor-butterfly, so results are run-to-run identical.
constexpr int kRvWarps = 8;
constexpr int kRvKC = 256;

__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename XT, int BE, bool NOISY, int TPW>
__global__ void __launch_bounds__(kRvWarps * 32)
k_router_vec(int T, int d, int E, int w16, const XT *__restrict__ x, const float *__restrict__ Wg,
             const float *__restrict__ Wn, const float *__restrict__ noise,
             const float *__restrict__ bias, float *__restrict__ c_out, float *__restrict__ s_out,
             float *__restrict__ H_out, DeviceStatus *st) {
  constexpr int NC = NOISY ? 2 * BE : BE;  // columns: BE clean, then BE noise
  constexpr int WP = NC + 4;               // padded W row: conflict-free float4 reads
  constexpr int VEC = 16 / (int)sizeof(XT);
  constexpr int TOK = kRvWarps * TPW;
  extern __shared__ float4 smem4[];
  float *Ws = reinterpret_cast<float *>(smem4);                  // [2][KC][WP]
  XT *Xs = reinterpret_cast<XT *>(Ws + 2 * kRvKC * WP);          // [2][warps][TPW][KC]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TOK + warp * TPW;
  const int e0 = blockIdx.y * BE;
  const int nchunks = (d + kRvKC - 1) / kRvKC;

  auto stage = [&](int chunk, int buf) {
    const int k0 = chunk * kRvKC;
    float *wdst = Ws + (size_t)buf * kRvKC * WP;
    if (w16) {  // E % 4 == 0: 16-byte pieces of each W row segment
      constexpr int NV = NC / 4;
      for (int i = threadIdx.x; i < kRvKC * NV; i += blockDim.x) {
        const int kk = i / NV, cv = (i % NV) * 4;
        const int k = k0 + kk, col = cv < BE ? cv : cv - BE, e = e0 + col;
        const float *src = cv < BE ? Wg : Wn;
        const bool ok = k < d && e < E;
        cp_async16(wdst + kk * WP + cv, ok ? src + (size_t)k * E + e : src, ok ? 16 : 0);
      }
    } else {
      for (int i = threadIdx.x; i < kRvKC * NC; i += blockDim.x) {
        const int kk = i / NC, cv = i % NC;
        const int k = k0 + kk, col = cv < BE ? cv : cv - BE, e = e0 + col;
        const float *src = cv < BE ? Wg : Wn;
        const bool ok = k < d && e < E;
        cp_async4(wdst + kk * WP + cv, ok ? src + (size_t)k * E + e : src, ok ? 4 : 0);
      }
    }
    XT *xdst = Xs + ((size_t)(buf * kRvWarps + warp) * TPW) * kRvKC;
    constexpr int NVX = TPW * kRvKC / VEC;
    for (int v = lane; v < NVX; v += 32) {
      const int tl = v / (kRvKC / VEC), kv = (v % (kRvKC / VEC)) * VEC;
      const int t = t0 + tl, k = k0 + kv;
      const bool ok = t < T && k < d;
      cp_async16(xdst + tl * kRvKC + kv, ok ? x + (size_t)t * d + k : x, ok ? 16 : 0);
    }
    cp_async_commit();
  };

  float acc[TPW][NC];
#pragma unroll
  for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
    for (int j = 0; j < NC; ++j) acc[tl][j] = 0.f;

  stage(0, 0);
  if (nchunks > 1) stage(1, 1);
  else cp_async_commit();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int buf = ch & 1;
    cp_async_wait<1>();
    __syncthreads();
    const float *w = Ws + (size_t)buf * kRvKC * WP;
    const XT *xw = Xs + ((size_t)(buf * kRvWarps + warp) * TPW) * kRvKC;
#pragma unroll 2
    for (int j = 0; j < kRvKC / 32; ++j) {
      const int kk = lane + 32 * j;
      float xv[TPW];
#pragma unroll
      for (int tl = 0; tl < TPW; ++tl) xv[tl] = to_f(xw[tl * kRvKC + kk]);
      const float4 *wr = reinterpret_cast<const float4 *>(w + kk * WP);
#pragma unroll
      for (int c4 = 0; c4 < NC / 4; ++c4) {
        const float4 wv = wr[c4];
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
          acc[tl][4 * c4 + 0] = fmaf(xv[tl], wv.x, acc[tl][4 * c4 + 0]);
          acc[tl][4 * c4 + 1] = fmaf(xv[tl], wv.y, acc[tl][4 * c4 + 1]);
          acc[tl][4 * c4 + 2] = fmaf(xv[tl], wv.z, acc[tl][4 * c4 + 2]);
          acc[tl][4 * c4 + 3] = fmaf(xv[tl], wv.w, acc[tl][4 * c4 + 3]);
        }
      }
    }
    __syncthreads();
    if (ch + 2 < nchunks) stage(ch + 2, buf);
    else cp_async_commit();  // keep one group per iteration
  }
  cp_async_wait<0>();
  // Fixed butterfly: every lane ends with the full sums.
#pragma unroll
  for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
    for (int j = 0; j < NC; ++j)
#pragma unroll
      for (int o = 16; o; o >>= 1) acc[tl][j] += __shfl_xor_sync(0xffffffffu, acc[tl][j], o);
#pragma unroll
  for (int tl = 0; tl < TPW; ++tl) {
#pragma unroll
    for (int el = 0; el < BE; ++el) {
      if (((tl * BE + el) & 31) != lane) continue;
      const int t = t0 + tl, e = e0 + el;
      if (t >= T || e >= E) continue;
      float cv = acc[tl][el];
      if (bias) cv += bias[e];
      float sg = 0.f, h = cv;
      if (NOISY) {
        sg = softplus_f(acc[tl][BE + el]);
        h = fmaf(noise[(size_t)t * E + e], sg, cv);
      }
      const size_t o = (size_t)t * E + e;
      c_out[o] = cv;
      s_out[o] = sg;
      H_out[o] = h;
      if (!isfinite(h)) record_error(st, MOE_ERR_NONFINITE, (long long)o);
    }
  }
}

template <typename XT, int BE, bool NOISY, int TPW>
cudaError_t run_router_vec(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                           const float *noise, const float *bias, float *c, float *s, float *H,
                           DeviceStatus *st, cudaStream_t stream) {
  constexpr int NC = NOISY ? 2 * BE : BE;
  const size_t smem = (size_t)2 * kRvKC * (NC + 4) * 4 +
                      (size_t)2 * kRvWarps * TPW * kRvKC * sizeof(XT);
  auto kern = k_router_vec<XT, BE, NOISY, TPW>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((cfg.T + kRvWarps * TPW - 1) / (kRvWarps * TPW), (cfg.E + BE - 1) / BE);
  kern<<<grid, kRvWarps * 32, smem, stream>>>(cfg.T, cfg.d, cfg.E, cfg.E % 4 == 0 ? 1 : 0,
                                               static_cast<const XT *>(x), Wg, Wn, noise, bias, c,
                                               s, H, st);
  return cudaGetLastError();
}

template <typename XT, bool NOISY>
cudaError_t router_vec_dispatch(const moe_config &cfg, const void *x, const float *Wg,
                                const float *Wn, const float *noise, const float *bias, float *c,
                                float *s, float *H, DeviceStatus *st, cudaStream_t stream) {
  if (cfg.E <= 8)
    return run_router_vec<XT, 8, NOISY, 4>(cfg, x, Wg, Wn, noise, bias, c, s, H, st, stream);
  if (cfg.E <= 16 || NOISY)
    return run_router_vec<XT, 16, NOISY, NOISY ? 2 : 4>(cfg, x, Wg, Wn, noise, bias, c, s, H, st,
                                                          stream);
  return run_router_vec<XT, 32, NOISY, 2>(cfg, x, Wg, Wn, noise, bias, c, s, H, st, stream);
}

// ----------------------------------------------------------------------------- selection
// One warp per token; expert e lives in lane e % 32, slot e / 32. On return
// every lane holds the same results: topv/topi = the k+1 (k if k == E) largest
// values in (value desc, index asc) order, mx = max, se = sum of exp(v - mx).
// A NaN never wins; if only NaNs remain a round yields E (out of range),
// which the consumers reject. The router has already flagged the NaN.
template <int VPL>
__device__ __forceinline__ void warp_topk(const float (&v)[VPL], int E, int k, int lane,
                                          float *topv, int *topi, float &mx, float &se) {
  mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) mx = fmaxf(mx, v[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  se = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) se += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  uint32_t taken = 0;
  const int rounds = k < E ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int bi = E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      const bool ok = e < E && !((taken >> i) & 1u);
      if (ok && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    topv[r] = bv;
    topi[r] = bi;
  }
}

// The gate of choice j (TOPK: softmax over the kept k; SWITCH: the full
// softmax at the argmax).
__device__ __forceinline__ float gate_of(int j, int k, int mode, const float *topv, float mx,
                                         float se) {
  if (mode == MOE_GATE_SWITCH) return expf(topv[0] - mx) / se;
  float z = 0.f;
  for (int q = 0; q < k; ++q) z += expf(topv[q] - topv[0]);
  return expf(topv[j] - topv[0]) / z;
}

template <int VPL>
__global__ void __launch_bounds__(256)
k_select(int T, int E, int k, int mode, const float *__restrict__ H, int32_t *__restrict__ idx,
         float *__restrict__ gate, float *__restrict__ thr, float *__restrict__ rowstat) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float *h = H + (size_t)t * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? h[e] : -INFINITY;
  }
  float topv[kMaxK + 1], mx, se;
  int topi[kMaxK + 1];
  warp_topk<VPL>(v, E, k, lane, topv, topi, mx, se);
  if (lane == 0) {
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = topi[j];
      gate[(size_t)t * k + j] = gate_of(j, k, mode, topv, mx, se);
    }
    thr[2 * (size_t)t] = topv[k - 1];
    thr[2 * (size_t)t + 1] = k < E ? topv[k] : -INFINITY;
    rowstat[2 * (size_t)t] = mx;
    rowstat[2 * (size_t)t + 1] = se;
  }
}

// ----------------------------------------------------------------------------- balancing partials
// Block (token block b, expert chunk): warp w walks tokens t0+w, t0+w+8, ...
// of the block in order; lane l owns experts chunk0 + l + 32 i. The eight
// warps' sums are added in warp order, so every partial is run-to-run
// identical. partials layout: [block][4][E] = importance, load, first-choice
// count, sum of Softmax(H).
constexpr int kAuxWarps = 8;
constexpr int kAuxMaxK = 16;

template <int VPL>
__global__ void __launch_bounds__(kAuxWarps * 32)
k_aux_partials(int T, int E, int k, int tb, int noisy, const float *__restrict__ c,
               const float *__restrict__ sg, const float *__restrict__ H,
               const float *__restrict__ rowstat, const int32_t *__restrict__ idx,
               const float *__restrict__ gate, const float *__restrict__ thr,
               float *__restrict__ partials) {
  constexpr int CH = 32 * VPL;
  __shared__ float red[kAuxWarps][4][CH];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x, e0 = blockIdx.y * CH;
  const int t0 = b * tb, t1 = min(T, t0 + tb);
  float acc[4][VPL];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[q][i] = 0.f;
  for (int t = t0 + warp; t < t1; t += kAuxWarps) {
    // All of this token's loads first, so they are in flight together.
    const float th0 = thr[2 * (size_t)t], th1 = thr[2 * (size_t)t + 1];
    const float mx = rowstat[2 * (size_t)t], inv_se = 1.f / rowstat[2 * (size_t)t + 1];
    int chosen_e[kAuxMaxK];
    float chosen_g[kAuxMaxK];
#pragma unroll
    for (int j = 0; j < kAuxMaxK; ++j) {
      chosen_e[j] = j < k ? idx[(size_t)t * k + j] : -1;
      chosen_g[j] = j < k ? gate[(size_t)t * k + j] : 0.f;
    }
    float cv[VPL], sv[VPL], hv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = e0 + lane + 32 * i;
      const size_t o = (size_t)t * E + (e < E ? e : 0);
      hv[i] = H[o];
      cv[i] = noisy ? c[o] : 0.f;
      sv[i] = noisy ? sg[o] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = e0 + lane + 32 * i;
      if (e >= E) continue;
      float g = 0.f;
      bool in = false;
#pragma unroll
      for (int j = 0; j < kAuxMaxK; ++j)
        if (chosen_e[j] == e) {
          in = true;
          g = chosen_g[j];
        }
      acc[0][i] += g;
      float p;
      if (k == E) {
        p = 1.f;
      } else if (sv[i] == 0.f) {
        p = in ? 1.f : 0.f;
      } else {
        const float u = (cv[i] - (in ? th1 : th0)) / sv[i];
        p = 0.5f * erfcf(-u * 0.70710678118654752f);
      }
      acc[1][i] += p;
      if (chosen_e[0] == e) acc[2][i] += 1.f;
      acc[3][i] += expf(hv[i] - mx) * inv_se;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < VPL; ++i) red[warp][q][lane + 32 * i] = acc[q][i];
  __syncthreads();
  for (int v = threadIdx.x; v < 4 * CH; v += blockDim.x) {
    const int q = v / CH, el = v % CH, e = e0 + el;
    if (e >= E) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kAuxWarps; ++w) sum += red[w][q][el];
    partials[((size_t)b * 4 + q) * E + e] = sum;
  }
}

// Selection and balancing partials in one pass, for E <= 256: the warp that
// selects token t's experts goes on to add t's contributions to the expert
// sums its lanes own, so H, the chosen experts and the gates are read once.
// Token order, warp order and the block sums are those of k_aux_partials, so
// the partials are bit-identical to the two-kernel path.
template <int VPL>
__global__ void __launch_bounds__(kAuxWarps * 32)
k_select_aux(int T, int E, int k, int mode, int tb, int noisy, const float *__restrict__ c,
             const float *__restrict__ sg, const float *__restrict__ H,
             int32_t *__restrict__ idx, float *__restrict__ gate, float *__restrict__ thr,
             float *__restrict__ rowstat, float *__restrict__ partials) {
  constexpr int CH = 32 * VPL;
  __shared__ float red[kAuxWarps][4][CH];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int t0 = b * tb, t1 = min(T, t0 + tb);
  float acc[4][VPL];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[q][i] = 0.f;
  for (int t = t0 + warp; t < t1; t += kAuxWarps) {
    float v[VPL], cv[VPL], sv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      const size_t o = (size_t)t * E + (e < E ? e : 0);
      v[i] = e < E ? H[o] : -INFINITY;
      cv[i] = noisy ? c[o] : 0.f;
      sv[i] = noisy ? sg[o] : 0.f;
    }
    float topv[kMaxK + 1], mx, se;
    int topi[kMaxK + 1];
    warp_topk<VPL>(v, E, k, lane, topv, topi, mx, se);
    float g[kMaxK];
    for (int j = 0; j < k; ++j) g[j] = gate_of(j, k, mode, topv, mx, se);
    const float th0 = topv[k - 1], th1 = k < E ? topv[k] : -INFINITY;
    if (lane == 0) {
      for (int j = 0; j < k; ++j) {
        idx[(size_t)t * k + j] = topi[j];
        gate[(size_t)t * k + j] = g[j];
      }
      thr[2 * (size_t)t] = th0;
      thr[2 * (size_t)t + 1] = th1;
      rowstat[2 * (size_t)t] = mx;
      rowstat[2 * (size_t)t + 1] = se;
    }
    const float inv_se = 1.f / se;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) continue;
      float gi = 0.f;
      bool in = false;
      for (int j = 0; j < k; ++j)
        if (topi[j] == e) {
          in = true;
          gi = g[j];
        }
      acc[0][i] += gi;
      float p;
      if (k == E) {
        p = 1.f;
      } else if (sv[i] == 0.f) {
        p = in ? 1.f : 0.f;
      } else {
        const float u = (cv[i] - (in ? th1 : th0)) / sv[i];
        p = 0.5f * erfcf(-u * 0.70710678118654752f);
      }
      acc[1][i] += p;
      if (topi[0] == e) acc[2][i] += 1.f;
      acc[3][i] += expf(v[i] - mx) * inv_se;
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < VPL; ++i) red[warp][q][lane + 32 * i] = acc[q][i];
  __syncthreads();
  for (int vv = threadIdx.x; vv < 4 * CH; vv += blockDim.x) {
    const int q = vv / CH, e = vv % CH;
    if (e >= E) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kAuxWarps; ++w) sum += red[w][q][e];
    partials[((size_t)b * 4 + q) * E + e] = sum;
  }
}

// Finalize, one launch. A block (E <= 256) or a warp sums each expert's
// partials over the token blocks (thread j takes blocks j, j+G, ... in order;
// fp64; then a fixed butterfly), writing aux_vec [4][E] = importance, load,
// f, Pbar. The block that
// finishes last (a ticket in the status word, reset by that block) then
// computes CV^2 of importance and load (population variance) and the Switch
// loss 0.01 * E * sum(f * Pbar) in a fixed order.
constexpr int kFinThreads = 256;

// Sum over the block in a fixed order (xor butterfly in each warp, then the
// warp totals in warp order): identical on every run.
__device__ double block_sum_fixed(double v, double *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double r = 0;
#pragma unroll
  for (int w = 0; w < kFinThreads / 32; ++w) r += sh[w];
  __syncthreads();
  return r;
}

// G threads sum one expert's partials: the whole block (G = 256, few experts)
// or one warp (G = 32, eight experts per block).
template <int G>
__global__ void __launch_bounds__(kFinThreads)
k_aux_finalize(int T, int E, int nb, const float *__restrict__ partials,
               double *__restrict__ aux_vec, float *__restrict__ importance,
               float *__restrict__ load, float *__restrict__ out3, DeviceStatus *st) {
  __shared__ double sh[kFinThreads];
  __shared__ int last;
  constexpr int PER = kFinThreads / G;  // experts per block
  const int e = blockIdx.x * PER + threadIdx.x / G;
  const int j = threadIdx.x % G;
  double v[4] = {0, 0, 0, 0};
  if (e < E) {
    for (int b = j; b < nb; b += G) {
      const float *q = partials + (size_t)b * 4 * E + e;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] += q[(size_t)i * E];
    }
  }
  double tot[4];
  if (G == kFinThreads) {
#pragma unroll
    for (int i = 0; i < 4; ++i) tot[i] = block_sum_fixed(v[i], sh);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int o = 16; o; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
      tot[i] = v[i];
    }
  }
  if (j == 0 && e < E) {
    aux_vec[e] = tot[0];
    aux_vec[E + e] = tot[1];
    aux_vec[2 * E + e] = tot[2] / T;
    aux_vec[3 * E + e] = tot[3] / T;
    if (importance) importance[e] = (float)tot[0];
    if (load) load[e] = (float)tot[1];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned ticket = atomicAdd(reinterpret_cast<unsigned *>(&st->aux_ticket), 1u);
    last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const volatile double *av = aux_vec;
  double s_imp = 0, s_ld = 0, s_fp = 0;
  for (int i = threadIdx.x; i < E; i += kFinThreads) {
    s_imp += av[i];
    s_ld += av[E + i];
    s_fp += av[2 * E + i] * av[3 * E + i];
  }
  const double m_imp = block_sum_fixed(s_imp, sh) / E;
  const double m_ld = block_sum_fixed(s_ld, sh) / E;
  const double fp = block_sum_fixed(s_fp, sh);
  double v_imp = 0, v_ld = 0;
  for (int i = threadIdx.x; i < E; i += kFinThreads) {
    const double a = av[i] - m_imp, l = av[E + i] - m_ld;
    v_imp += a * a;
    v_ld += l * l;
  }
  v_imp = block_sum_fixed(v_imp, sh) / E;
  v_ld = block_sum_fixed(v_ld, sh) / E;
  if (threadIdx.x == 0) {
    out3[0] = (float)(v_imp / (m_imp * m_imp));
    out3[1] = (float)(v_ld / (m_ld * m_ld));
    out3[2] = (float)(0.01 * E * fp);
    st->aux_ticket = 0;  // ready for the next call
  }
}

}  // namespace

cudaError_t launch_router(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                          const float *noise, const float *bias, float *c, float *sigma, float *H,
                          void *bsplit, DeviceStatus *st, cudaStream_t s) {
  const bool noisy = Wn != nullptr;
  // bf16 tokens: the tensor-core router (MOE_ROUTER=simt selects the CUDA-core kernels).
  static int force_simt = -1;
  if (force_simt < 0) {
    const char *v = getenv("MOE_ROUTER");
    force_simt = (v && v[0] == 's') ? 1 : 0;
  }
  if (!force_simt && router_tc_supported(cfg))
    return launch_router_tc(cfg, x, Wg, Wn, noise, bias, c, sigma, H, bsplit, st, s);
  // Vector path: whole 16-byte pieces of every x row, and a small expert count
  // (beyond it the per-block W traffic of this layout grows with E).
  const bool vec = cfg.E <= 64 &&
                   (cfg.act_dtype == MOE_BF16 ? cfg.d % 8 == 0 : cfg.d % 4 == 0);
  if (vec) {
    if (cfg.act_dtype == MOE_BF16)
      return noisy ? router_vec_dispatch<__nv_bfloat16, true>(cfg, x, Wg, Wn, noise, bias, c,
                                                              sigma, H, st, s)
                   : router_vec_dispatch<__nv_bfloat16, false>(cfg, x, Wg, Wn, noise, bias, c,
                                                               sigma, H, st, s);
    return noisy ? router_vec_dispatch<float, true>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s)
                 : router_vec_dispatch<float, false>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st,
                                                     s);
  }
  if (cfg.E <= 8)
    return noisy ? run_router<8, true>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s)
                 : run_router<8, false>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s);
  if (cfg.E <= 16)
    return noisy ? run_router<16, true>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s)
                 : run_router<16, false>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s);
  return noisy ? run_router<32, true>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s)
               : run_router<32, false>(cfg, x, Wg, Wn, noise, bias, c, sigma, H, st, s);
}

cudaError_t launch_select(const moe_config &cfg, const float *H, int32_t *idx, float *gate,
                          float *thr, float *rowstat, DeviceStatus *st, cudaStream_t s) {
  (void)st;
  const int warps = 8;
  dim3 grid((cfg.T + warps - 1) / warps);
  int vpl = (cfg.E + 31) / 32;
#define MOE_SEL(V)                                                                          \
  k_select<V><<<grid, warps * 32, 0, s>>>(cfg.T, cfg.E, cfg.k, cfg.gate_mode, H, idx, gate, \
                                          thr, rowstat)
  if (vpl <= 1) MOE_SEL(1);
  else if (vpl <= 2) MOE_SEL(2);
  else if (vpl <= 4) MOE_SEL(4);
  else if (vpl <= 8) MOE_SEL(8);
  else if (vpl <= 16) MOE_SEL(16);
  else MOE_SEL(32);
#undef MOE_SEL
  return cudaGetLastError();
}

// Tokens per partial-sum block: small blocks (two tokens per warp) where the
// fused selection kernel runs (two tokens per warp), so it has enough CTAs;
// larger ones for E > 256.
int aux_token_block(int E) { return E <= 256 ? 16 : 256; }

cudaError_t launch_aux_partials(const moe_config &cfg, bool noisy, const float *c,
                                const float *sigma, const float *H, const float *rowstat,
                                const int32_t *idx, const float *gate, const float *thr,
                                float *partials, int n_blocks, cudaStream_t s) {
  const int tb = aux_token_block(cfg.E);
  const int vpl = cfg.E <= 32 ? 1 : (cfg.E <= 64 ? 2 : (cfg.E <= 128 ? 4 : 8));
  dim3 grid(n_blocks, (cfg.E + 32 * vpl - 1) / (32 * vpl));
#define MOE_AUXP(V)                                                                           \
  k_aux_partials<V><<<grid, kAuxWarps * 32, 0, s>>>(cfg.T, cfg.E, cfg.k, tb, noisy ? 1 : 0, c, \
                                                     sigma, H, rowstat, idx, gate, thr, partials)
  if (vpl == 1) MOE_AUXP(1);
  else if (vpl == 2) MOE_AUXP(2);
  else if (vpl == 4) MOE_AUXP(4);
  else MOE_AUXP(8);
#undef MOE_AUXP
  return cudaGetLastError();
}

cudaError_t launch_select_aux(const moe_config &cfg, bool noisy, const float *c, const float *sigma,
                              const float *H, int32_t *idx, float *gate, float *thr,
                              float *rowstat, float *partials, int n_blocks, cudaStream_t s) {
  const int tb = aux_token_block(cfg.E);
  const int vpl = cfg.E <= 32 ? 1 : (cfg.E <= 64 ? 2 : (cfg.E <= 128 ? 4 : 8));
#define MOE_SELAUX(V)                                                                           \
  k_select_aux<V><<<n_blocks, kAuxWarps * 32, 0, s>>>(cfg.T, cfg.E, cfg.k, cfg.gate_mode, tb,   \
                                                       noisy ? 1 : 0, c, sigma, H, idx, gate, thr, \
                                                       rowstat, partials)
  if (vpl == 1) MOE_SELAUX(1);
  else if (vpl == 2) MOE_SELAUX(2);
  else if (vpl == 4) MOE_SELAUX(4);
  else MOE_SELAUX(8);
#undef MOE_SELAUX
  return cudaGetLastError();
}

cudaError_t launch_aux_finalize(const moe_config &cfg, const float *partials, int n_blocks,
                                float *out3, float *importance, float *load, double *aux_vec,
                                DeviceStatus *st, cudaStream_t s) {
  // Many partial rows (16-token blocks, E <= 256): a block per expert; few
  // (256-token blocks): a warp per expert.
  if (cfg.E <= 256)
    k_aux_finalize<kFinThreads><<<cfg.E, kFinThreads, 0, s>>>(cfg.T, cfg.E, n_blocks, partials,
                                                              aux_vec, importance, load, out3, st);
  else
    k_aux_finalize<32><<<(cfg.E + 7) / 8, kFinThreads, 0, s>>>(cfg.T, cfg.E, n_blocks, partials,
                                                               aux_vec, importance, load, out3, st);
  return cudaGetLastError();
}

}  // namespace moe
