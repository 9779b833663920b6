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

// ----------------------------------------------------------------------------- selection
// One warp per token; expert e lives in lane e % 32, slot e / 32.
template <int VPL>
__global__ void __launch_bounds__(256)
k_select(int T, int E, int k, int mode, const float *__restrict__ H, int32_t *__restrict__ idx,
         float *__restrict__ gate, float *__restrict__ thr, float *__restrict__ rowstat) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float *h = H + (size_t)t * E;
  float v[VPL];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int e = lane + 32 * i;
    v[i] = e < E ? h[e] : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float se = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) se += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);

  // Rounds of warp-wide argmax in (value desc, index asc) order. A NaN never
  // wins; if only NaNs remain the round yields E (out of range), which the
  // consumers reject. The router has already flagged the NaN.
  uint32_t taken = 0;
  const int rounds = k < E ? k + 1 : k;
  float topv[kMaxK + 1];
  int topi[kMaxK + 1];
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int bi = E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      int e = lane + 32 * i;
      bool ok = e < E && !((taken >> i) & 1u);
      if (ok && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    topv[r] = bv;
    topi[r] = bi;
  }
  if (lane == 0) {
    if (mode == MOE_GATE_SWITCH) {
      idx[t] = topi[0];
      gate[t] = expf(topv[0] - mx) / se;
    } else {
      float z = 0.f;
      for (int j = 0; j < k; ++j) z += expf(topv[j] - topv[0]);
      for (int j = 0; j < k; ++j) {
        idx[(size_t)t * k + j] = topi[j];
        gate[(size_t)t * k + j] = expf(topv[j] - topv[0]) / z;
      }
    }
    thr[2 * (size_t)t] = topv[k - 1];
    thr[2 * (size_t)t + 1] = k < E ? topv[k] : -INFINITY;
    rowstat[2 * (size_t)t] = mx;
    rowstat[2 * (size_t)t + 1] = se;
  }
}

// ----------------------------------------------------------------------------- balancing partials
// Thread per expert; tokens of one block walked in order. partials layout:
// [block][4][E]: importance, load, first-choice count, sum of Softmax(H).
constexpr int kAuxThreads = 128;

__global__ void __launch_bounds__(kAuxThreads)
k_aux_partials(int T, int E, int k, int noisy, const float *__restrict__ c,
               const float *__restrict__ sg, const float *__restrict__ H,
               const float *__restrict__ rowstat, const int32_t *__restrict__ idx,
               const float *__restrict__ gate, const float *__restrict__ thr,
               float *__restrict__ partials) {
  const int e = blockIdx.x * kAuxThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (e >= E) return;
  const int tb = b * kAuxTokBlock, te = min(T, tb + kAuxTokBlock);
  float imp = 0.f, ld = 0.f, first = 0.f, pb = 0.f;
  for (int t = tb; t < te; ++t) {
    int chosen = -1;
    for (int j = 0; j < k; ++j)
      if (idx[(size_t)t * k + j] == e) chosen = j;
    if (chosen >= 0) imp += gate[(size_t)t * k + chosen];
    if (idx[(size_t)t * k] == e) first += 1.f;
    size_t o = (size_t)t * E + e;
    float p;
    if (k == E) {
      p = 1.f;
    } else {
      float s = noisy ? sg[o] : 0.f;
      if (s == 0.f) {
        p = chosen >= 0 ? 1.f : 0.f;
      } else {
        float th = chosen >= 0 ? thr[2 * (size_t)t + 1] : thr[2 * (size_t)t];
        float u = (c[o] - th) / s;
        p = 0.5f * erfcf(-u * 0.70710678118654752f);
      }
    }
    ld += p;
    pb += expf(H[o] - rowstat[2 * (size_t)t]) / rowstat[2 * (size_t)t + 1];
  }
  float *out = partials + (size_t)b * 4 * E;
  out[e] = imp;
  out[E + e] = ld;
  out[2 * E + e] = first;
  out[3 * E + e] = pb;
}

constexpr int kFinThreads = 256;

__device__ double block_sum_fixed(double v, double *sh) {
  // Fixed-shape tree: identical order on every run.
  sh[threadIdx.x] = v;
  __syncthreads();
  for (int s = kFinThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
    __syncthreads();
  }
  double r = sh[0];
  __syncthreads();
  return r;
}

// One block: sums the partials over token blocks in order (fp64), then CV^2 and
// the Switch loss. aux_vec: [4][E] fp32 copies (importance, load, f, Pbar).
__global__ void __launch_bounds__(kFinThreads)
k_aux_finalize(int T, int E, int nb, const float *__restrict__ partials, float *__restrict__ out3,
               float *__restrict__ importance, float *__restrict__ load,
               float *__restrict__ aux_vec) {
  __shared__ double sh[kFinThreads];
  double s_imp = 0, s_ld = 0, s_fp = 0;
  for (int e = threadIdx.x; e < E; e += kFinThreads) {
    double a = 0, l = 0, f = 0, p = 0;
    for (int b = 0; b < nb; ++b) {
      const float *q = partials + (size_t)b * 4 * E;
      a += q[e];
      l += q[E + e];
      f += q[2 * E + e];
      p += q[3 * E + e];
    }
    f /= T;
    p /= T;
    aux_vec[e] = (float)a;
    aux_vec[E + e] = (float)l;
    aux_vec[2 * E + e] = (float)f;
    aux_vec[3 * E + e] = (float)p;
    if (importance) importance[e] = (float)a;
    if (load) load[e] = (float)l;
    s_imp += a;
    s_ld += l;
    s_fp += f * p;
  }
  double m_imp = block_sum_fixed(s_imp, sh) / E;
  double m_ld = block_sum_fixed(s_ld, sh) / E;
  double fp = block_sum_fixed(s_fp, sh);
  // Second pass for the variances, re-summing the same partials in the same order.
  double v_imp = 0, v_ld = 0;
  for (int e = threadIdx.x; e < E; e += kFinThreads) {
    double a = 0, l = 0;
    for (int b = 0; b < nb; ++b) {
      const float *q = partials + (size_t)b * 4 * E;
      a += q[e];
      l += q[E + e];
    }
    v_imp += (a - m_imp) * (a - m_imp);
    v_ld += (l - m_ld) * (l - m_ld);
  }
  v_imp = block_sum_fixed(v_imp, sh) / E;
  v_ld = block_sum_fixed(v_ld, sh) / E;
  if (threadIdx.x == 0) {
    out3[0] = (float)(v_imp / (m_imp * m_imp));
    out3[1] = (float)(v_ld / (m_ld * m_ld));
    out3[2] = (float)(0.01 * E * fp);
  }
}

}  // namespace

cudaError_t launch_router(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                          const float *noise, const float *bias, float *c, float *sigma, float *H,
                          DeviceStatus *st, cudaStream_t s) {
  const bool noisy = Wn != nullptr;
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

cudaError_t launch_aux_partials(const moe_config &cfg, bool noisy, const float *c,
                                const float *sigma, const float *H, const float *rowstat,
                                const int32_t *idx, const float *gate, const float *thr,
                                float *partials, int n_blocks, cudaStream_t s) {
  dim3 grid((cfg.E + kAuxThreads - 1) / kAuxThreads, n_blocks);
  k_aux_partials<<<grid, kAuxThreads, 0, s>>>(cfg.T, cfg.E, cfg.k, noisy ? 1 : 0, c, sigma, H,
                                              rowstat, idx, gate, thr, partials);
  return cudaGetLastError();
}

cudaError_t launch_aux_finalize(const moe_config &cfg, const float *partials, int n_blocks,
                                float *out3, float *importance, float *load, float *aux_vec,
                                cudaStream_t s) {
  k_aux_finalize<<<1, kFinThreads, 0, s>>>(cfg.T, cfg.E, n_blocks, partials, out3, importance,
                                           load, aux_vec);
  return cudaGetLastError();
}

}  // namespace moe
