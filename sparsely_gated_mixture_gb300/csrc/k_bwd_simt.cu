// Backward of the expert networks on the CUDA cores: fp32 layers (the tensor
// cores have no fp32 input kind) and bf16 shapes the tensor-core kernels do
// not take (d or d_ff not a multiple of 64). Same quantities as the
// tensor-core path ("Outrageously Large Neural Networks", section 3.4:
// back-propagation through the experts; "Switch Transformer", step 6), in
// fp32 throughout:
//   gather:  dY[pr] = dy[t], dU[pr] = g * dy[t]            (padded rows, pad rows 0)
//   dgrad 0: D = dY W2[e]^T; <D, h> per 64-column block; dpre = g D [h > 0]
//   dgrad 1: dX = dpre W1[e]^T
//   wgrad:   dW2[e] = h^T dU, dW1[e] = x^T dpre, over the expert's real rows
//   dg:      <dy, U> of each kept choice from the partials plus <dy, b2>
//   dx:      dx = dy + the router's share + the kept choices' dX rows
// 64 x 64 output tiles, K in chunks of 16, 4 x 4 outputs per thread, fixed
// summation order (identical results from run to run).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int TM = 64, TN = 64, TK = 16, kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ T st_val(float v);
template <>
__device__ __forceinline__ float st_val<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 st_val<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ int find_blk(const int32_t *__restrict__ a, int n, int v) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid;
    else hi = mid;
  }
  return lo;
}

// One warp per padded row.
template <typename T>
__global__ void __launch_bounds__(256)
k_bs_gather(long long P_max, int E, int k, int d, const int32_t *__restrict__ offset,
            const int32_t *__restrict__ poff, const int32_t *__restrict__ row_token,
            const float *__restrict__ row_gate, const T *__restrict__ dy, float *__restrict__ dY,
            float *__restrict__ dU) {
  pdl_wait();
  const long long pr = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (pr < P_max && pr < poff[E]) {
    const int e = find_blk(poff, E, (int)pr);
    const int m = (int)(pr - poff[e]);
    const int rows = offset[e + 1] - offset[e];
    if (m < rows) {
      const int q = offset[e] + m;
      const size_t t = (size_t)(row_token[q] / k);
      const float g = row_gate[q];
      for (int c = lane; c < d; c += 32) {
        const float v = ld(dy, t * d + c);
        dY[pr * d + c] = v;
        dU[pr * d + c] = g * v;
      }
    } else {
      for (int c = lane; c < d; c += 32) {
        dY[pr * d + c] = 0.f;
        dU[pr * d + c] = 0.f;
      }
    }
  }
  pdl_trigger();
}

// out[pr, n] = sum_k A[pr, k] W[e*N + n, k] over one 64-row block of padded
// rows (all of one expert: the blocks are multiples of 64). MODE 0: A = dY,
// W = W2 (N = d_ff), epilogue: dgate partials and dpre; MODE 1: A = dpre,
// W = W1 (N = d), epilogue: dX on the real rows.
template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads)
k_bs_dgrad(int K, int N, int E, const int32_t *__restrict__ offset,
           const int32_t *__restrict__ poff, const float *__restrict__ row_gate,
           const float *__restrict__ A, const T *__restrict__ W, const T *__restrict__ hbuf,
           float *__restrict__ out, float *__restrict__ dgpart, DeviceStatus *st) {
  pdl_wait();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int pr0 = blockIdx.y * TM;
  if (pr0 >= poff[E]) {
    pdl_trigger();
    return;
  }
  const int e = find_blk(poff, E, pr0);
  const int rows = offset[e + 1] - offset[e];
  const int n0 = blockIdx.x * TN;
  const int tid = threadIdx.x;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = tid; i < TM * TK; i += kThreads) {
      const int m = i / TK, kk = i % TK, kx = k0 + kk;
      As[kk][m] = kx < K ? A[(size_t)(pr0 + m) * K + kx] : 0.f;
    }
    for (int i = tid; i < TN * TK; i += kThreads) {
      const int n = i / TK, kk = i % TK, kx = k0 + kk;
      Bs[kk][n] = (kx < K && n0 + n < N) ? ld(W, ((size_t)e * N + n0 + n) * K + kx) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][tm + i];
        b[i] = Bs[kk][tn + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = pr0 - poff[e] + tm + i;  // row within the expert's padded block
    const size_t pr = (size_t)pr0 + tm + i;
    const bool real = m < rows;
    const size_t q = (size_t)offset[e] + m;
    float part = 0.f;
    if (MODE == 0) {
      const float g = real ? row_gate[q] : 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tn + j;
        if (n >= N) continue;
        const float h = real ? ld(hbuf, q * N + n) : 0.f;
        part = fmaf(acc[i][j], h, part);
        const float p = h > 0.f ? g * acc[i][j] : 0.f;
        bad |= !isfinite(p);
        out[pr * N + n] = p;
      }
      // the 16 threads holding this row's 64 columns are 16 consecutive lanes
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if ((tid & 15) == 0) dgpart[pr * gridDim.x + blockIdx.x] = part;
    } else if (real) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tn + j;
        if (n >= N) continue;
        bad |= !isfinite(acc[i][j]);
        out[pr * N + n] = acc[i][j];
      }
    }
  }
  if (bad) record_error(st, MOE_ERR_NONFINITE, (long long)pr0);
  pdl_trigger();
}

// out[e][m][n] = sum over the expert's real rows r of A[offset[e] + r][m] *
// B[poff[e] + r][n]; A: the forward's packed rows (T), B: padded rows (fp32).
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_bs_wgrad(int M, int N, const int32_t *__restrict__ offset, const int32_t *__restrict__ poff,
           const T *__restrict__ A, const float *__restrict__ B, float *__restrict__ out,
           DeviceStatus *st) {
  pdl_wait();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int e = blockIdx.z;
  const int a0 = offset[e], rows = offset[e + 1] - a0, b0 = poff[e];
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tid = threadIdx.x;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int r0 = 0; r0 < rows; r0 += TK) {
    for (int i = tid; i < TK * TM; i += kThreads) {
      const int kk = i / TM, m = i % TM, r = r0 + kk;
      As[kk][m] = (r < rows && m0 + m < M) ? ld(A, (size_t)(a0 + r) * M + m0 + m) : 0.f;
    }
    for (int i = tid; i < TK * TN; i += kThreads) {
      const int kk = i / TN, n = i % TN, r = r0 + kk;
      Bs[kk][n] = (r < rows && n0 + n < N) ? B[(size_t)(b0 + r) * N + n0 + n] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][tm + i];
        b[i] = Bs[kk][tn + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn + j;
      if (n >= N) continue;
      bad |= !isfinite(acc[i][j]);
      out[((size_t)e * M + m) * N + n] = acc[i][j];
    }
  }
  if (bad) record_error(st, MOE_ERR_NONFINITE, (long long)e);
  pdl_trigger();
}

// dg[a] for the kept assignment a of packed row q (one warp per row).
template <typename T>
__global__ void __launch_bounds__(256)
k_bs_dg(int E, int k, int d, int n_blocks, const int32_t *__restrict__ offset,
        const int32_t *__restrict__ poff, const int32_t *__restrict__ row_token,
        const float *__restrict__ dgpart, const T *__restrict__ dy, const T *__restrict__ b2,
        float *__restrict__ dg) {
  pdl_wait();
  const long long q = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (q < offset[E]) {
    const int e = find_blk(offset, E, (int)q);
    const long long pr = poff[e] + (q - offset[e]);
    const int a = row_token[q];
    float s = 0.f;
    for (int nb = lane; nb < n_blocks; nb += 32) s += dgpart[pr * n_blocks + nb];
    if (b2) {
      const size_t t = (size_t)(a / k);
      for (int c = lane; c < d; c += 32) s = fmaf(ld(dy, t * d + c), ld(b2, (size_t)e * d + c), s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) dg[a] = s;
  }
  pdl_trigger();
}

// dx_t = dy_t + dxr_t + sum over kept choices (in order) of dX rows; one warp
// per token. Launched in plain stream order (after the side-stream join).
template <typename T>
__global__ void __launch_bounds__(256)
k_bs_dx(int T_, int d, int k, const int32_t *__restrict__ idx, const int32_t *__restrict__ pos,
        const uint8_t *__restrict__ keep, const int32_t *__restrict__ poff,
        const float *__restrict__ dX, const float *__restrict__ dxr, const T *__restrict__ dy,
        T *__restrict__ dx) {
  const long long t = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T_) return;
  long long rows[16];
  int nk = 0;
  for (int j = 0; j < k; ++j)
    if (keep[t * k + j]) rows[nk++] = (long long)poff[idx[t * k + j]] + pos[t * k + j];
  for (int c = lane; c < d; c += 32) {
    float v = ld(dy, (size_t)t * d + c);
    if (dxr) v += dxr[t * d + c];
    for (int j = 0; j < nk; ++j) v += dX[rows[j] * d + c];
    dx[t * d + c] = st_val<T>(v);
  }
}

int blocks_for(long long work, int per_block) {
  long long b = (work + per_block - 1) / per_block;
  return (int)(b < 1 ? 1 : (b > 0x7fffffffLL ? 0x7fffffffLL : b));
}

template <typename T>
cudaError_t run_simt_bwd(const moe_config &c, const BwdSimt &p, cudaStream_t s) {
  const T *dy = static_cast<const T *>(p.dy);
  cudaError_t err = launch_pdl(k_bs_gather<T>, blocks_for(p.P_max, 8), 256, 0, s, p.P_max, c.E,
                               c.k, c.d, p.offset, p.poff, p.row_token, p.row_gate, dy, p.dY,
                               p.dU);
  if (err != cudaSuccess) return err;
  const int rblk = (int)((p.P_max + TM - 1) / TM);
  const dim3 g0((c.d_ff + TN - 1) / TN, rblk);
  err = launch_pdl_c(kPdlGemm, k_bs_dgrad<T, 0>, g0, kThreads, 0, s, c.d, c.d_ff, c.E, p.offset,
                     p.poff, p.row_gate, (const float *)p.dY, static_cast<const T *>(p.W2),
                     static_cast<const T *>(p.hbuf), p.dP, p.dgpart, p.st);
  if (err != cudaSuccess) return err;
  return cudaSuccess;
}

}  // namespace

int simt_dgate_blocks(const moe_config &c) { return (c.d_ff + TN - 1) / TN; }

cudaError_t launch_bwd_simt_front(const moe_config &c, const BwdSimt &p, cudaStream_t s) {
  return c.act_dtype == MOE_BF16 ? run_simt_bwd<__nv_bfloat16>(c, p, s)
                                 : run_simt_bwd<float>(c, p, s);
}

template <typename T>
static cudaError_t simt_back(const moe_config &c, const BwdSimt &p, cudaStream_t s) {
  const int rblk = (int)((p.P_max + TM - 1) / TM);
  const dim3 g1((c.d + TN - 1) / TN, rblk);
  cudaError_t err = launch_pdl_c(kPdlGemm, k_bs_dgrad<T, 1>, g1, kThreads, 0, s, c.d_ff, c.d, c.E,
                                 p.offset, p.poff, (const float *)nullptr, (const float *)p.dP,
                                 static_cast<const T *>(p.W1), (const T *)nullptr, p.dX,
                                 (float *)nullptr, p.st);
  if (err != cudaSuccess) return err;
  const dim3 g2((c.d + TN - 1) / TN, (c.d_ff + TM - 1) / TM, c.E);
  err = launch_pdl_c(kPdlGemm, k_bs_wgrad<T>, g2, kThreads, 0, s, c.d_ff, c.d, p.offset, p.poff,
                     static_cast<const T *>(p.hbuf), (const float *)p.dU, p.dW2, p.st);
  if (err != cudaSuccess) return err;
  const dim3 g3((c.d_ff + TN - 1) / TN, (c.d + TM - 1) / TM, c.E);
  return launch_pdl_c(kPdlGemm, k_bs_wgrad<T>, g3, kThreads, 0, s, c.d, c.d_ff, p.offset,
                      p.poff, static_cast<const T *>(p.xbuf), (const float *)p.dP, p.dW1, p.st);
}

cudaError_t launch_bwd_simt_back(const moe_config &c, const BwdSimt &p, cudaStream_t s) {
  return c.act_dtype == MOE_BF16 ? simt_back<__nv_bfloat16>(c, p, s) : simt_back<float>(c, p, s);
}

cudaError_t launch_bwd_simt_dg(const moe_config &c, const BwdSimt &p, float *dg, cudaStream_t s) {
  const int nb = simt_dgate_blocks(c);
  if (c.act_dtype == MOE_BF16)
    return launch_pdl(k_bs_dg<__nv_bfloat16>, blocks_for((long long)c.T * c.k, 8), 256, 0, s, c.E,
                      c.k, c.d, nb, p.offset, p.poff, p.row_token, (const float *)p.dgpart,
                      static_cast<const __nv_bfloat16 *>(p.dy),
                      static_cast<const __nv_bfloat16 *>(p.b2), dg);
  return launch_pdl(k_bs_dg<float>, blocks_for((long long)c.T * c.k, 8), 256, 0, s, c.E, c.k, c.d,
                    nb, p.offset, p.poff, p.row_token, (const float *)p.dgpart,
                    static_cast<const float *>(p.dy), static_cast<const float *>(p.b2), dg);
}

cudaError_t launch_bwd_simt_dx(const moe_config &c, const BwdSimt &p, const int32_t *idx,
                               const int32_t *pos, const uint8_t *keep, const float *dxr,
                               void *dx, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks_for(c.T, 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  if (c.act_dtype == MOE_BF16)
    return cudaLaunchKernelEx(&cfg, k_bs_dx<__nv_bfloat16>, (int)c.T, (int)c.d, (int)c.k, idx, pos,
                              keep, (const int32_t *)p.poff, (const float *)p.dX, dxr,
                              static_cast<const __nv_bfloat16 *>(p.dy),
                              static_cast<__nv_bfloat16 *>(dx));
  return cudaLaunchKernelEx(&cfg, k_bs_dx<float>, (int)c.T, (int)c.d, (int)c.k, idx, pos, keep,
                            (const int32_t *)p.poff, (const float *)p.dX, dxr,
                            static_cast<const float *>(p.dy), static_cast<float *>(dx));
}

}  // namespace moe
