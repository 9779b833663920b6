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
#include "gate_math.cuh"

#include <math.h>
#include <stdlib.h>

#include <type_traits>

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
  pdl_wait();
  pdl_trigger();
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
  launch_pdl(kern, grid, kRtWarps * 32, smem, stream, cfg.T, cfg.d, cfg.E, x, cfg.act_dtype, Wg, Wn,
      noise, bias, c, s, H, st);
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
  pdl_wait();
  pdl_trigger();
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
  launch_pdl(kern, grid, kRvWarps * 32, smem, stream, cfg.T, cfg.d, cfg.E, cfg.E % 4 == 0 ? 1 : 0,
      static_cast<const XT *>(x), Wg, Wn, noise, bias, c, s, H, st);
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
// lane r (r < k+1, or k if k == E) holds the r-th pick (myv, myi) of the k+1
// largest values in (value desc, index asc) order, and every lane holds
// mx = max and se = sum of exp(v - mx). Results stay in registers: a pick is
// read from its lane with a shuffle. A NaN never wins; if only NaNs remain a
// round yields E (out of range), which the consumers reject. The router has
// already flagged the NaN.
template <int VPL>
__device__ __forceinline__ void warp_topk(const float (&v)[VPL], int E, int k, int lane,
                                          float &myv, int &myi, float &mx, float &se) {
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
    if (lane == r) {
      myv = bv;
      myi = bi;
    }
  }
}

// The same results as warp_topk, for wide rows (VPL >= 16), by a threshold:
// tau = the R-th largest of the 32 lanes' maxima (R = rounds). R distinct
// values are >= tau, so the R-th largest value overall is >= tau and every
// member of the top R is a candidate (value >= tau). The candidates (rarely
// more than a handful) are packed into the warp's 32-entry scratch, one per
// lane, and R rounds of a warp arg-max pick them in (value desc, index asc)
// order. Returns false, having written nothing, when tau is -inf or there are
// more than 32 candidates (heavy ties); the caller then runs warp_topk. se is
// summed with the fast exponential here (relative error ~1e-6).
template <int VPL>
__device__ __forceinline__ bool warp_topk_thresh(const float (&v)[VPL], int E, int k, int lane,
                                                 float2 *scratch, float &myv, int &myi,
                                                 float &mx, float &se) {
  float m = -INFINITY;  // fmaxf drops NaN
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) m = fmaxf(m, v[i]);
  mx = m;
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int rounds = k < E ? k + 1 : k;
  float cur = m, tau = -INFINITY;
  for (int r = 0; r < rounds; ++r) {
    float w = cur;
#pragma unroll
    for (int o = 16; o; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
    tau = w;
    const unsigned hit = __ballot_sync(0xffffffffu, cur == w);
    if (lane == __ffs(hit) - 1) cur = -INFINITY;
  }
  if (tau == -INFINITY) return false;
  int n = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) n += (lane + 32 * i < E && v[i] >= tau) ? 1 : 0;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total > 32) return false;
  se = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) se += __expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  int o = incl - n;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E && v[i] >= tau) scratch[o++] = make_float2(v[i], __int_as_float(e));
  }
  __syncwarp();
  float cv = -INFINITY;
  int ci = E;
  if (lane < total) {
    const float2 q = scratch[lane];
    cv = q.x;
    ci = __float_as_int(q.y);
  }
  __syncwarp();  // scratch is free for the warp's next token
  for (int r = 0; r < rounds; ++r) {
    float bv = cv;
    int bi = ci;
#pragma unroll
    for (int o2 = 16; o2; o2 >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o2);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o2);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == r) {
      myv = bv;
      myi = bi;
    }
    if (ci == bi) {
      cv = -INFINITY;
      ci = E;
    }
  }
  return true;
}

// The gate held by lane j < k (TOPK: softmax over the kept k, the
// normaliser summed in pick order; SWITCH: the full-softmax probability of the
// argmax). Every lane takes part; lanes >= k get 0.
__device__ __forceinline__ float warp_gate(float myv, int k, int mode, float mx, float se,
                                           int lane) {
  const float v0 = __shfl_sync(0xffffffffu, myv, 0);
  if (mode == MOE_GATE_SWITCH) return lane == 0 ? expf(v0 - mx) / se : 0.f;
  const float ej = lane < k ? expf(myv - v0) : 0.f;
  float z = 0.f;
  for (int q = 0; q < k; ++q) z += __shfl_sync(0xffffffffu, ej, q);
  return lane < k ? ej / z : 0.f;
}

// Token t's selection outputs: the k picks and gates from lanes 0..k-1, the
// thresholds (k-th and (k+1)-th values) and the row statistics from lane 0.
__device__ __forceinline__ void store_selection(size_t t, int E, int k, int lane, float myv,
                                                int myi, float g, float th0, float th1, float mx,
                                                float se, int32_t *__restrict__ idx,
                                                float *__restrict__ gate, float *__restrict__ thr,
                                                float *__restrict__ rowstat) {
  if (lane < k) {
    idx[t * k + lane] = myi;
    gate[t * k + lane] = g;
  }
  if (lane == 0) {
    thr[2 * t] = th0;
    thr[2 * t + 1] = th1;
    rowstat[2 * t] = mx;
    rowstat[2 * t + 1] = se;
  }
}

template <int VPL>
__global__ void __launch_bounds__(256)
k_select(int T, int E, int k, int mode, const float *__restrict__ H, int32_t *__restrict__ idx,
         float *__restrict__ gate, float *__restrict__ thr, float *__restrict__ rowstat) {
  pdl_wait();
  pdl_trigger();
  __shared__ float2 scratch[8][32];
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
  float myv = -INFINITY, mx, se;
  int myi = E;
  if (VPL < 16 ||
      !warp_topk_thresh<VPL>(v, E, k, lane, scratch[threadIdx.x >> 5], myv, myi, mx, se))
    warp_topk<VPL>(v, E, k, lane, myv, myi, mx, se);
  const float g = warp_gate(myv, k, mode, mx, se, lane);
  const float th0 = __shfl_sync(0xffffffffu, myv, k - 1);
  const float thk = __shfl_sync(0xffffffffu, myv, k & 31);
  store_selection(t, E, k, lane, myv, myi, g, th0, k < E ? thk : -INFINITY, mx, se, idx, gate, thr,
                  rowstat);
}

// ----------------------------------------------------------------------------- balancing partials
// Partials layout: [token block][4][E] = importance, load, first-choice count,
// sum of Softmax(H), each a sum over the block's tokens.
constexpr int kAuxWarps = 8;

// E > 256: the column form. Partial row b covers the contiguous tokens
// [b T / P, (b+1) T / P), P = aux_rows(T, E): at most kColRows, one wave of
// four blocks on each of 152 SMs, so every block has an equal share. Thread j
// owns V consecutive experts (e0 = chunk start + V j) and walks its block's
// tokens in order, so each sum runs in one thread in token order (identical on
// every run). The per-token scalars (thresholds, row max, 1 / sum of
// exponentials, chosen experts and gates) are staged in shared memory kColTB
// tokens at a time; the c, sigma and H loads are coalesced across the block
// (V = 4: one 16-byte load each).
constexpr int kColThreads = 256;
constexpr int kColTB = 64;
constexpr int kColU = 2;  // tokens whose loads are in flight together
constexpr int kColRows = 4 * 152;

template <int V, int KM>  // KM >= k
__global__ void __launch_bounds__(kColThreads, 4)
k_aux_cols(int T, int E, int k, int noisy, int P, const float *__restrict__ c,
           const float *__restrict__ sg, const float *__restrict__ H,
           const float *__restrict__ rowstat, const int32_t *__restrict__ idx,
           const float *__restrict__ gate, const float *__restrict__ thr,
           float *__restrict__ partials) {
  pdl_wait();
  pdl_trigger();
  using VT = typename std::conditional<V == 4, float4, float>::type;
  __shared__ float4 s_tok[kColTB];  // th0, th1, mx, 1/se
  __shared__ int s_idx[kColTB][KM];
  __shared__ float s_g[kColTB][KM];
  const int b = blockIdx.x;
  const int tb0 = (int)((long long)b * T / P), tb1 = (int)((long long)(b + 1) * T / P);
  const int e0 = blockIdx.y * (kColThreads * V) + threadIdx.x * V;
  const bool active = e0 < E;
  float imp[V], ld[V], fc[V], ps[V];
#pragma unroll
  for (int q = 0; q < V; ++q) imp[q] = ld[q] = fc[q] = ps[q] = 0.f;
  for (int t0 = tb0; t0 < tb1; t0 += kColTB) {
    const int nt = min(kColTB, tb1 - t0);
    __syncthreads();  // the previous chunk's scalars are no longer read
    for (int i = threadIdx.x; i < nt; i += kColThreads) {
      const size_t t = (size_t)t0 + i;
      s_tok[i] = make_float4(thr[2 * t], thr[2 * t + 1], rowstat[2 * t], 1.f / rowstat[2 * t + 1]);
    }
    for (int i = threadIdx.x; i < nt * k; i += kColThreads) {
      s_idx[i / k][i % k] = idx[(size_t)t0 * k + i];
      s_g[i / k][i % k] = gate[(size_t)t0 * k + i];
    }
    __syncthreads();
    if (!active) continue;
    for (int tt0 = 0; tt0 < nt; tt0 += kColU) {
      VT hv[kColU], cv[kColU], sv[kColU];
#pragma unroll
      for (int u = 0; u < kColU; ++u) {
        const int tt = min(tt0 + u, nt - 1);  // a repeated row past the end is loaded, not used
        const size_t o = ((size_t)t0 + tt) * E + e0;
        hv[u] = *reinterpret_cast<const VT *>(H + o);
        if (noisy) {
          cv[u] = *reinterpret_cast<const VT *>(c + o);
          sv[u] = *reinterpret_cast<const VT *>(sg + o);
        }
      }
#pragma unroll
      for (int u = 0; u < kColU; ++u) {
        const int tt = tt0 + u;
        if (tt >= nt) break;
        const float4 sc = s_tok[tt];
        unsigned in = 0;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (j >= k) break;
          const unsigned rel = (unsigned)(s_idx[tt][j] - e0);
          if (rel < (unsigned)V) {
            in |= 1u << rel;
            const float g = s_g[tt][j];
#pragma unroll
            for (int q = 0; q < V; ++q)
              if (rel == (unsigned)q) {
                imp[q] += g;
                if (j == 0) fc[q] += 1.f;
              }
          }
        }
        const float *h = reinterpret_cast<const float *>(&hv[u]);
        const float *cc = reinterpret_cast<const float *>(&cv[u]);
        const float *ss = reinterpret_cast<const float *>(&sv[u]);
#pragma unroll
        for (int q = 0; q < V; ++q) {
          const bool isin = (in >> q) & 1u;
          float p;
          if (k == E) {
            p = 1.f;
          } else if (!noisy || ss[q] == 0.f) {
            p = isin ? 1.f : 0.f;
          } else {
            p = normal_cdf(__fdividef(cc[q] - (isin ? sc.y : sc.x), ss[q]));
          }
          ld[q] += p;
          ps[q] += __expf(h[q] - sc.z) * sc.w;
        }
      }
    }
  }
  if (!active) return;
  float *out = partials + (size_t)b * 4 * E + e0;
  const float *acc[4] = {imp, ld, fc, ps};
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    VT r;
    float *rp = reinterpret_cast<float *>(&r);
#pragma unroll
    for (int q = 0; q < V; ++q) rp[q] = acc[a][q];
    *reinterpret_cast<VT *>(out + (size_t)a * E) = r;
  }
}

// Selection and balancing partials in one pass, for E <= 256: the warp that
// selects token t's experts goes on to add t's contributions to the expert
// sums its lanes own, so H, the chosen experts and the gates are read once.
// Block b covers tokens [16 b, 16 b + 16); warp w takes tokens t0+w, t0+w+8
// in order and the eight warps' sums are added in warp order, so every
// partial is run-to-run identical.
template <int VPL, int KM>  // KM >= k: the chosen list kept in registers
__global__ void __launch_bounds__(kAuxWarps * 32)
k_select_aux(int T, int E, int k, int mode, int tb, int noisy, const float *__restrict__ c,
             const float *__restrict__ sg, const float *__restrict__ H,
             int32_t *__restrict__ idx, float *__restrict__ gate, float *__restrict__ thr,
             float *__restrict__ rowstat, float *__restrict__ partials) {
  pdl_wait();
  pdl_trigger();
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
    float myv = -INFINITY, mx, se;
    int myi = E;
    warp_topk<VPL>(v, E, k, lane, myv, myi, mx, se);
    const float g = warp_gate(myv, k, mode, mx, se, lane);
    const float th0 = __shfl_sync(0xffffffffu, myv, k - 1);
    const float thk = __shfl_sync(0xffffffffu, myv, k & 31);
    const float th1 = k < E ? thk : -INFINITY;
    store_selection(t, E, k, lane, myv, myi, g, th0, th1, mx, se, idx, gate, thr, rowstat);
    int ce[KM];
    float cg[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      ce[j] = __shfl_sync(0xffffffffu, myi, j);
      cg[j] = __shfl_sync(0xffffffffu, g, j);
      if (j >= k) ce[j] = -1;
    }
    const float inv_se = 1.f / se;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= E) continue;
      float gi = 0.f;
      bool in = false;
#pragma unroll
      for (int j = 0; j < KM; ++j)
        if (ce[j] == e) {
          in = true;
          gi = cg[j];
        }
      acc[0][i] += gi;
      float p;
      if (k == E) {
        p = 1.f;
      } else if (sv[i] == 0.f) {
        p = in ? 1.f : 0.f;
      } else {
        p = normal_cdf(__fdividef(cv[i] - (in ? th1 : th0), sv[i]));
      }
      acc[1][i] += p;
      if (ce[0] == e) acc[2][i] += 1.f;
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

// Finalize, one launch: each expert's partials are summed over the partial
// rows in a fixed order (fp64), writing aux_vec [4][E] = importance, load, f,
// Pbar; the last block to finish then forms the three losses (finish_aux).
constexpr int kFinThreads = 256;

// Sum over the block in a fixed order (xor butterfly in each warp, then the
// warp totals in warp order): identical on every run.
// Double-float ("ff") arithmetic: a value is hi + lo with |lo| <= ulp(hi)/2,
// about 44 significant bits from fp32 operations alone (the fp64 pipe of this
// part is narrow). Sums use Knuth's TwoSum, products Dekker's TwoProduct via
// FMA (Knuth, TAOCP vol. 2, 4.2.2; Dekker 1971); for a fixed order of
// operations every result is run-to-run identical.
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const float s = a.hi + b.hi;
  const float v = s - a.hi;
  const float e = (a.hi - (s - v)) + (b.hi - v);  // a.hi + b.hi = s + e exactly
  const float t = e + (a.lo + b.lo);
  const float hi = s + t;
  return {hi, t - (hi - s)};
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = a.hi * b.hi;
  const float e = fmaf(a.hi, b.hi, -p);  // a.hi * b.hi = p + e exactly
  const float t = e + (a.hi * b.lo + a.lo * b.hi);
  const float hi = p + t;
  return {hi, t - (hi - p)};
}
__device__ __forceinline__ double ff_to_d(ff a) { return (double)a.hi + (double)a.lo; }
__device__ __forceinline__ ff d_to_ff(double x) {
  const float h = (float)x;
  return {h, (float)(x - (double)h)};
}
__device__ __forceinline__ ff ff_ld(const float2 *p) {
  const float2 v = __ldcg(p);  // written by other blocks of this launch: read at L2
  return {v.x, v.y};
}

// N sums over the block at once: a fixed xor butterfly in each warp, then the
// warp totals in warp order by N threads, shared back. sh holds >= 33 N.
template <int N>
__device__ void block_sum_ff(ff (&v)[N], ff *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int o = 16; o; o >>= 1)
      v[i] = ff_add(v[i], ff{__shfl_xor_sync(0xffffffffu, v[i].hi, o),
                             __shfl_xor_sync(0xffffffffu, v[i].lo, o)});
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) sh[warp * N + i] = v[i];
  __syncthreads();
  if (threadIdx.x < N) {
    ff r{0.f, 0.f};
    for (int w = 0; w < nw; ++w) r = ff_add(r, sh[w * N + threadIdx.x]);
    sh[32 * N + threadIdx.x] = r;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = sh[32 * N + i];
  __syncthreads();
}

// Expert e's totals (importance, load, f, Pbar) into aux [4][E] as ff, and the
// optional fp32 copies of importance and load.
__device__ __forceinline__ void store_expert_totals(int T, int E, int e, int q, ff tot,
                                                    float2 *__restrict__ aux,
                                                    float *__restrict__ importance,
                                                    float *__restrict__ load,
                                                    float *__restrict__ raw) {
  const ff v = q >= 2 ? d_to_ff(ff_to_d(tot) / T) : tot;
  aux[(size_t)q * E + e] = make_float2(v.hi, v.lo);
  const float f32 = (float)ff_to_d(tot);
  if (q == 0 && importance) importance[e] = f32;
  if (q == 1 && load) load[e] = f32;
  if (raw) raw[(size_t)q * E + e] = f32;
}

// Run by every block of a finalize launch once its aux entries are written:
// the block that finishes last (a ticket in the status word, reset by that
// block) computes CV^2 of importance and load (population variance, two
// passes) and the Switch loss 0.01 * E * sum(f * Pbar), in ff with a fixed
// order, the last few scalar steps in fp64.
__device__ void finish_aux(int E, const float2 *__restrict__ aux, float *__restrict__ out3,
                           DeviceStatus *st, ff *sh) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned ticket = atomicAdd(reinterpret_cast<unsigned *>(&st->aux_ticket), 1u);
    last = ticket == gridDim.x * gridDim.y - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  ff s3[3] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    s3[0] = ff_add(s3[0], ff_ld(aux + i));
    s3[1] = ff_add(s3[1], ff_ld(aux + E + i));
    s3[2] = ff_add(s3[2], ff_mul(ff_ld(aux + 2 * E + i), ff_ld(aux + 3 * E + i)));
  }
  block_sum_ff<3>(s3, sh);
  const double m_imp = ff_to_d(s3[0]) / E, m_ld = ff_to_d(s3[1]) / E;
  const ff nm_imp = d_to_ff(-m_imp), nm_ld = d_to_ff(-m_ld);
  ff v2[2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const ff a = ff_add(ff_ld(aux + i), nm_imp), l = ff_add(ff_ld(aux + E + i), nm_ld);
    v2[0] = ff_add(v2[0], ff_mul(a, a));
    v2[1] = ff_add(v2[1], ff_mul(l, l));
  }
  block_sum_ff<2>(v2, sh);
  if (threadIdx.x == 0) {
    const double v_imp = ff_to_d(v2[0]) / E, v_ld = ff_to_d(v2[1]) / E;
    out3[0] = (float)(v_imp / (m_imp * m_imp));
    out3[1] = (float)(v_ld / (m_ld * m_ld));
    out3[2] = (float)(0.01 * E * ff_to_d(s3[2]));
    st->aux_ticket = 0;  // ready for the next call
  }
}

// E <= 256: a block per expert; thread j takes rows j, j+256, ... in order,
// then a fixed butterfly.
__global__ void __launch_bounds__(kFinThreads)
k_aux_finalize(int T, int E, int nb, const float *__restrict__ partials, float2 *__restrict__ aux,
               float *__restrict__ importance, float *__restrict__ load,
               float *__restrict__ out3, DeviceStatus *st, float *__restrict__ raw) {
  pdl_wait();
  pdl_trigger();
  __shared__ ff sh[kFinThreads];
  const int e = blockIdx.x;
  ff tot[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int b = threadIdx.x; b < nb; b += kFinThreads) {
    const float *q = partials + (size_t)b * 4 * E + e;
#pragma unroll
    for (int i = 0; i < 4; ++i) tot[i] = ff_add(tot[i], ff{q[(size_t)i * E], 0.f});
  }
  block_sum_ff<4>(tot, sh);
  if (threadIdx.x < 4) store_expert_totals(T, E, e, threadIdx.x, tot[threadIdx.x], aux,
                                           importance, load, raw);
  finish_aux(E, aux, out3, st, sh);
}

// E > 256: block (32-expert group, quantity q). Lane l takes expert
// 32 group + l and warp w the partial rows w, w+16, ... in order, so the row
// reads are coalesced and kFinBatch of them are in flight at once; the
// sixteen warp sums are added in warp order.
constexpr int kFinColThreads = 512;
constexpr int kFinBatch = 16;

__global__ void __launch_bounds__(kFinColThreads)
k_aux_finalize_cols(int T, int E, int nb, const float *__restrict__ partials,
                    float2 *__restrict__ aux, float *__restrict__ importance,
                    float *__restrict__ load, float *__restrict__ out3, DeviceStatus *st,
                    float *__restrict__ raw) {
  pdl_wait();
  pdl_trigger();
  __shared__ ff sh[kFinColThreads];
  constexpr int NW = kFinColThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane, q = blockIdx.y;
  ff v{0.f, 0.f};
  if (e < E) {
    const float *p = partials + (size_t)q * E + e;
    for (int b0 = warp; b0 < nb; b0 += NW * kFinBatch) {
      float r[kFinBatch];
#pragma unroll
      for (int u = 0; u < kFinBatch; ++u) {
        const int b = b0 + u * NW;
        r[u] = b < nb ? p[(size_t)b * 4 * E] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kFinBatch; ++u) v = ff_add(v, ff{r[u], 0.f});
    }
  }
  sh[threadIdx.x] = v;
  __syncthreads();
  if (warp == 0 && e < E) {
    ff tot{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < NW; ++w) tot = ff_add(tot, sh[w * 32 + lane]);
    store_expert_totals(T, E, e, q, tot, aux, importance, load, raw);
  }
  __syncthreads();
  finish_aux(E, aux, out3, st, sh);
}

// ----------------------------------------------------------------------------- hierarchical gate
// "Outrageously Large", Hierarchical Mixture-of-Experts: a groups of b
// experts (flat expert i*b + j). The primary gate (the flat gate over a
// groups) has picked groups idx_p [T,kp] with gates g_p [T,kp]; here each
// picked group's secondary gate takes the top ks of its b secondary noisy
// logits (warp_topk: value descending, lower index first) with a softmax over
// them, and token t's choice q*ks + r is expert i*b + j_r with gate
// g_p[t,q] * G_i(x_t)_{j_r}.
//
// Balancing partials, one row per block of kHierTok tokens, for the finalize:
// [0] Importance_H (sum of the product gates), [1] the in-group smooth load
// Load_i(X^(i))_j (P_i(x, j) = Phi((c - kth_excluding) / sigma) inside the
// group, summed over the tokens that picked group i; the pick indicator
// without noise; 1 when ks == b), [2] |X^(i)| at j = 0 of each group (0
// elsewhere), [3] 0. A warp takes whole groups and its lanes the group's
// experts, walking the block's tokens in order, so every sum has one fixed
// order and the loads of a token's group row are coalesced.
constexpr int kHierTokMax = 64;  // tokens per block and per partial row (64, or 32: hier_tokens)
constexpr int kHierWarps = 8;
constexpr int kHierMaxKp = 8;    // largest primary k

// Tokens per block: 64, or 32 when the block's P buffer ([tokens][kp][b]
// floats, kp*b <= a*b <= 1024) would pass 128 KB at 64.
__host__ __device__ inline int hier_tokens(int kp, int b) { return kp * b <= 512 ? 64 : 32; }

template <int VPL, int KMS>  // b <= 32 * VPL, ks <= KMS
__global__ void __launch_bounds__(kHierWarps * 32)
k_hier_select(int T, int a, int b, int kp, int ks, int noisy, const int32_t *__restrict__ idx_p,
              const float *__restrict__ g_p, const float *__restrict__ cs,
              const float *__restrict__ ss, const float *__restrict__ Hs,
              const int32_t *__restrict__ poff, const int32_t *__restrict__ pos_p,
              int32_t *__restrict__ idx, float *__restrict__ gate, float *__restrict__ partials,
              DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_grp[kHierTokMax][kHierMaxKp];        // picked group, or -1
  __shared__ float s_gp[kHierTokMax][kHierMaxKp];       // its primary gate
  __shared__ int s_pick[kHierTokMax][kHierMaxKp][KMS];  // in-group picks
  __shared__ float s_gate[kHierTokMax][kHierMaxKp][KMS];  // their product gates
  extern __shared__ float s_P[];                        // [tokens][kp][b]: P_i(x_t, j)
  const int E = a * b, k = kp * ks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int TB = hier_tokens(kp, b);
  const int t0 = blockIdx.x * TB, nt = min(TB, T - t0);
  const bool sums = partials != nullptr;
  for (int u = threadIdx.x; u < nt * kp; u += blockDim.x) {  // the block's primary picks
    const int i = idx_p[(size_t)t0 * kp + u];
    s_grp[u / kp][u % kp] = (i >= 0 && i < a) ? i : -1;
    s_gp[u / kp][u % kp] = g_p[(size_t)t0 * kp + u];
  }
  __syncthreads();
  for (int pr = warp; pr < nt * kp; pr += kHierWarps) {
    const int tt = pr / kp, q = pr - tt * kp;
    const size_t t = (size_t)t0 + tt;
    const int i = s_grp[tt][q];
    if (i < 0) {  // the primary gate flagged a NaN row, or a bad index
      if (lane == 0) record_error(st, MOE_ERR_BOUNDS, (long long)t);
      if (lane < ks) {
        idx[t * k + q * ks + lane] = E;  // out of range: the slot pass rejects it
        gate[t * k + q * ks + lane] = 0.f;
      }
      continue;
    }
    // The group's row of H, c and sigma, loaded together (one trip): in the
    // dense [T][a*b] layout, or the grouped router's compact row.
    const size_t o = poff ? ((size_t)poff[i] + pos_p[t * kp + q]) * b : t * E + (size_t)i * b;
    float v[VPL], cv[VPL], sv[VPL];
#pragma unroll
    for (int m = 0; m < VPL; ++m) {
      const int j = lane + 32 * m;
      v[m] = j < b ? Hs[o + j] : -INFINITY;
      cv[m] = (sums && noisy && j < b) ? cs[o + j] : 0.f;
      sv[m] = (sums && noisy && j < b) ? ss[o + j] : 0.f;
    }
    float myv = -INFINITY, mx, se;
    int myi = b;
    warp_topk<VPL>(v, b, ks, lane, myv, myi, mx, se);
    const float gs = warp_gate(myv, ks, MOE_GATE_TOPK_SOFTMAX, mx, se, lane);
    const float th0 = __shfl_sync(0xffffffffu, myv, ks - 1);
    const float thk = __shfl_sync(0xffffffffu, myv, ks & 31);
    const float th1 = ks < b ? thk : -INFINITY;
    const float gp = s_gp[tt][q];
    if (lane < ks) {
      const float g = gp * gs;
      idx[t * k + q * ks + lane] = myi < b ? i * b + myi : E;
      gate[t * k + q * ks + lane] = g;
      s_pick[tt][q][lane] = myi;
      s_gate[tt][q][lane] = g;
    }
    if (!sums) continue;
    // P_i(x_t, j) for the group's experts: Phi((c - kth_excluding) / sigma),
    // kth_excluding = the (ks+1)-th in-group logit for a pick, else the ks-th.
    int pk[KMS];
#pragma unroll
    for (int r = 0; r < KMS; ++r) pk[r] = __shfl_sync(0xffffffffu, myi, r);
    float *P = s_P + ((size_t)tt * kp + q) * b;
#pragma unroll
    for (int m = 0; m < VPL; ++m) {
      const int j = lane + 32 * m;
      if (j >= b) break;
      bool in = false;
#pragma unroll
      for (int r = 0; r < KMS; ++r) in |= r < ks && pk[r] == j;
      float p;
      if (ks == b) p = 1.f;
      else if (sv[m] == 0.f) p = in ? 1.f : 0.f;
      else p = normal_cdf(__fdividef(cv[m] - (in ? th1 : th0), sv[m]));
      P[j] = p;
    }
  }
  if (!sums) return;
  __syncthreads();
  // Per group (a warp) and expert (a lane): the block's tokens in order.
  float *row = partials + (size_t)blockIdx.x * 4 * E;
  for (int i = warp; i < a; i += kHierWarps) {
    float imp[VPL], ld[VPL];
#pragma unroll
    for (int m = 0; m < VPL; ++m) imp[m] = ld[m] = 0.f;
    float cnt = 0.f;
    for (int tt = 0; tt < nt; ++tt) {
      for (int q = 0; q < kp; ++q) {
        if (s_grp[tt][q] != i) continue;
        cnt += 1.f;
        const float *P = s_P + ((size_t)tt * kp + q) * b;
#pragma unroll
        for (int m = 0; m < VPL; ++m) {
          const int j = lane + 32 * m;
          if (j >= b) break;
          float gv = 0.f;
#pragma unroll
          for (int r = 0; r < KMS; ++r)
            if (r < ks && s_pick[tt][q][r] == j) gv = s_gate[tt][q][r];
          imp[m] += gv;
          ld[m] += P[j];
        }
      }
    }
#pragma unroll
    for (int m = 0; m < VPL; ++m) {
      const int j = lane + 32 * m;
      if (j >= b) break;
      const int e = i * b + j;
      row[e] = imp[m];
      row[E + e] = ld[m];
      row[2 * E + e] = j == 0 ? cnt : 0.f;
      row[3 * E + e] = 0.f;
    }
  }
}

// The hierarchical losses from the two finalizes' sums (one block, a thread
// per flat expert): Load_H[i*b+j] = Load_p[i] * Load_i(X^(i))_j / |X^(i)|,
// 0 where |X^(i)| = 0 (in fp32, about 1e-7 relative); out2 =
// [CV(Importance_H)^2, CV(Load_H)^2] with the population variance, the means
// and squared deviations summed in double-float in a fixed order (as the flat
// finalize does). |X^(i)| comes back from the finalize as a mean over T and
// is restored to the integer count. Also carries an error the primary gate
// recorded in its own status word over to the layer's status word.
constexpr int kHierTailThreads = 1024;

__global__ void __launch_bounds__(kHierTailThreads)
k_hier_tail(int T, int a, int b, const float2 *__restrict__ aux_s, const float2 *__restrict__ aux_p,
            float *__restrict__ out2, DeviceStatus *st, const DeviceStatus *st_p) {
  pdl_wait();
  pdl_trigger();
  __shared__ ff sh[32 * 2 + 2];
  const int E = a * b, e = threadIdx.x;
  if (threadIdx.x == 0 && st->code == 0 && st_p->code != 0) {
    st->detail = st_p->detail;
    st->code = st_p->code;
  }
  if (!out2) return;
  ff imp{0.f, 0.f}, lh{0.f, 0.f};
  if (e < E) {
    const int i = e / b;
    imp = ff_ld(aux_s + e);
    const float2 al = aux_s[E + e], ac = aux_s[2 * E + i * b], ap = aux_p[a + i];
    const float cnt = (float)rint(((double)ac.x + (double)ac.y) * T);
    lh.hi = cnt > 0.f ? (ap.x + ap.y) * (al.x + al.y) / cnt : 0.f;
  }
  ff m2[2] = {imp, lh};
  block_sum_ff<2>(m2, sh);
  const double m_imp = ff_to_d(m2[0]) / E, m_ld = ff_to_d(m2[1]) / E;
  ff v2[2] = {{0.f, 0.f}, {0.f, 0.f}};
  if (e < E) {
    const ff di = ff_add(imp, d_to_ff(-m_imp)), dl = ff_add(lh, d_to_ff(-m_ld));
    v2[0] = ff_mul(di, di);
    v2[1] = ff_mul(dl, dl);
  }
  block_sum_ff<2>(v2, sh);
  if (threadIdx.x == 0) {
    const double v_imp = ff_to_d(v2[0]) / E, v_ld = ff_to_d(v2[1]) / E;
    out2[0] = (float)(v_imp / (m_imp * m_imp));
    out2[1] = (float)(v_ld / (m_ld * m_ld));
  }
}

}  // namespace

cudaError_t launch_router(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                          const float *noise, const float *bias, float *c, float *sigma, float *H,
                          void *bsplit, DeviceStatus *st, cudaStream_t s,
                          const RouterSelect *sel, bool *selected) {
  const bool noisy = Wn != nullptr;
  if (selected) *selected = false;
  // bf16 tokens: the tensor-core router (MOE_ROUTER=simt selects the CUDA-core kernels).
  static const bool force_simt = [] {
    const char *v = getenv("MOE_ROUTER");
    return v && v[0] == 's';
  }();
  // The tensor-core router's first kernel clears the status word; the
  // CUDA-core routers start from a cleared one.
  if (!force_simt && router_tc_supported(cfg))
    return launch_router_tc(cfg, x, Wg, Wn, noise, bias, c, sigma, H, bsplit, st, s, sel,
                            selected);
  {
    const cudaError_t err = cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s);
    if (err != cudaSuccess) return err;
  }
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
  launch_pdl(k_select<V>, grid, warps * 32, 0, s, cfg.T, cfg.E, cfg.k, cfg.gate_mode, H, idx,      \
      gate, thr, rowstat)
  if (vpl <= 1) MOE_SEL(1);
  else if (vpl <= 2) MOE_SEL(2);
  else if (vpl <= 4) MOE_SEL(4);
  else if (vpl <= 8) MOE_SEL(8);
  else if (vpl <= 16) MOE_SEL(16);
  else MOE_SEL(32);
#undef MOE_SEL
  return cudaGetLastError();
}

// Partial rows of the balancing sums: one per 16 tokens (two per warp) where
// the fused selection kernel runs (E <= 256), so it has enough CTAs; for the
// column kernel the same, capped at one wave of its blocks.
int aux_rows(int T, int E) {
  const int r = (T + 15) / 16;
  return E <= 256 ? r : (r < kColRows ? r : kColRows);
}

cudaError_t launch_aux_partials(const moe_config &cfg, bool noisy, const float *c,
                                const float *sigma, const float *H, const float *rowstat,
                                const int32_t *idx, const float *gate, const float *thr,
                                float *partials, int n_blocks, cudaStream_t s) {
  const bool v4 = cfg.E % 4 == 0;
  const int per = kColThreads * (v4 ? 4 : 1);
  dim3 grid(n_blocks, (cfg.E + per - 1) / per);
#define MOE_COLS(V, KM)                                                                       \
  launch_pdl(k_aux_cols<V, KM>, grid, kColThreads, 0, s, cfg.T, cfg.E, cfg.k, noisy ? 1 : 0,       \
      n_blocks, c, sigma, H, rowstat, idx, gate, thr, partials)
  if (v4) {
    if (cfg.k <= 4) MOE_COLS(4, 4);
    else MOE_COLS(4, kMaxK);
  } else {
    if (cfg.k <= 4) MOE_COLS(1, 4);
    else MOE_COLS(1, kMaxK);
  }
#undef MOE_COLS
  return cudaGetLastError();
}

cudaError_t launch_select_aux(const moe_config &cfg, bool noisy, const float *c, const float *sigma,
                              const float *H, int32_t *idx, float *gate, float *thr,
                              float *rowstat, float *partials, int n_blocks, cudaStream_t s) {
  const int tb = 16;  // tokens per partial row (aux_rows)
  const int vpl = cfg.E <= 32 ? 1 : (cfg.E <= 64 ? 2 : (cfg.E <= 128 ? 4 : 8));
#define MOE_SELAUX_K(V, KM)                                                                   \
  launch_pdl(k_select_aux<V, KM>, n_blocks, kAuxWarps * 32, 0, s, cfg.T, cfg.E, cfg.k,             \
      cfg.gate_mode, tb, noisy ? 1 : 0, c, sigma, H, idx, gate, thr, rowstat, partials)
#define MOE_SELAUX(V)                 \
  do {                                \
    if (cfg.k <= 2)                   \
      MOE_SELAUX_K(V, 2);             \
    else if (cfg.k <= 4)              \
      MOE_SELAUX_K(V, 4);             \
    else                              \
      MOE_SELAUX_K(V, kMaxK);         \
  } while (0)
  if (vpl == 1) MOE_SELAUX(1);
  else if (vpl == 2) MOE_SELAUX(2);
  else if (vpl == 4) MOE_SELAUX(4);
  else MOE_SELAUX(8);
#undef MOE_SELAUX
#undef MOE_SELAUX_K
  return cudaGetLastError();
}

cudaError_t launch_aux_finalize(const moe_config &cfg, const float *partials, int n_blocks,
                                float *out3, float *importance, float *load, float2 *aux_vec,
                                DeviceStatus *st, cudaStream_t s, float *raw_totals) {
  // E <= 256: a block per expert; beyond: the column form.
  if (cfg.E <= 256)
    launch_pdl_c(kPdlFinalize, k_aux_finalize, cfg.E, kFinThreads, 0, s, cfg.T, cfg.E, n_blocks,
        partials, aux_vec, importance, load, out3, st, raw_totals);
  else
    launch_pdl_c(kPdlFinalize, k_aux_finalize_cols, dim3((cfg.E + 31) / 32, 4), kFinColThreads, 0,
        s, cfg.T, cfg.E, n_blocks, partials, aux_vec, importance, load, out3, st, raw_totals);
  return cudaGetLastError();
}

cudaError_t launch_hier_select(int T, int a, int b, int kp, int ks, bool noisy,
                               const int32_t *idx_p, const float *g_p, const float *cs,
                               const float *ss, const float *Hs, const int32_t *poff,
                               const int32_t *pos_p, int32_t *idx, float *gate,
                               float *partials, DeviceStatus *st, cudaStream_t s) {
  if (kp > kHierMaxKp || ks > 8 || kp * b > 1024) return cudaErrorInvalidValue;
  const int TB = hier_tokens(kp, b);
  const dim3 grid((T + TB - 1) / TB);
  const size_t dsm = partials ? (size_t)TB * kp * b * 4 : 0;
  const int vpl = (b + 31) / 32;
#define MOE_HIER_K(V, KM)                                                                     \
  do {                                                                                         \
    cudaError_t e_ = cudaFuncSetAttribute(k_hier_select<V, KM>,                               \
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                                          (int)dsm);                                           \
    if (e_ != cudaSuccess) return e_;                                                          \
    launch_pdl(k_hier_select<V, KM>, grid, kHierWarps * 32, dsm, s, T, a, b, kp, ks,          \
               noisy ? 1 : 0, idx_p, g_p, cs, ss, Hs, poff, pos_p, idx, gate, partials, st);  \
  } while (0)
#define MOE_HIER(V)               \
  do {                            \
    if (ks <= 2)                  \
      MOE_HIER_K(V, 2);           \
    else if (ks <= 4)             \
      MOE_HIER_K(V, 4);           \
    else                          \
      MOE_HIER_K(V, 8);           \
  } while (0)
  if (vpl <= 1) MOE_HIER(1);
  else if (vpl <= 2) MOE_HIER(2);
  else if (vpl <= 4) MOE_HIER(4);
  else if (vpl <= 8) MOE_HIER(8);
  else if (vpl <= 16) MOE_HIER(16);
  else MOE_HIER(32);
#undef MOE_HIER
#undef MOE_HIER_K
  return cudaGetLastError();
}

int hier_rows(int T, int kp, int b) {
  const int TB = hier_tokens(kp, b);
  return (T + TB - 1) / TB;
}

cudaError_t launch_hier_tail(int T, int a, int b, const float2 *aux_s, const float2 *aux_p,
                             float *out2, DeviceStatus *st, const DeviceStatus *st_p,
                             cudaStream_t s) {
  if (a * b > kHierTailThreads) return cudaErrorInvalidValue;
  launch_pdl(k_hier_tail, 1, kHierTailThreads, 0, s, T, a, b, aux_s, aux_p, out2, st, st_p);
  return cudaGetLastError();
}

}  // namespace moe

// ----------------------------------------------------------------------------- diagnostic: Phi
// The load estimator's normal CDF, evaluated elementwise, so that its accuracy
// can be checked against a reference CDF on any grid.
namespace moe {
namespace {

__global__ void __launch_bounds__(256)
k_normal_cdf(long long n, const float *__restrict__ u, float *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = normal_cdf(u[i]);
}

}  // namespace
}  // namespace moe

extern "C" int moe_eval_normal_cdf(const float *u, float *out, int64_t n, moe_stream_t stream) {
  using namespace moe;
  if (n < 0 || (n > 0 && (!u || !out))) return MOE_ERR_ARG;
  if (n == 0) return MOE_OK;
  const long long blocks = (n + 255) / 256;
  const int grid = (int)(blocks < 4 * 152 ? blocks : 4 * 152);
  if (launch_pdl(k_normal_cdf, grid, 256, 0, (cudaStream_t)stream, (long long)n, u, out) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
