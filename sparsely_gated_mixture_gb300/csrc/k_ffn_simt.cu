// Stage 4 experts on the CUDA cores ("Switch Transformer", step 6: separate
// ReLU feed-forward networks per expert). Used for fp32 layers, where the
// tensor cores have no fp32 input kind, and for bf16 shapes the tensor-core
// kernel does not take. Grouped GEMM over the packed rows of each expert:
//   layer 1: hbuf[r] = ReLU(xbuf[r] W1[e] + b1[e])
//   layer 2: zbuf[r] = row_gate[r] * (hbuf[r] W2[e] + b2[e])
// 64 x 64 output tiles, K in chunks of 16, 4 x 4 outputs per thread, fp32
// accumulation in a fixed K order.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = kSimtBM, BN = 64, BK = 16, kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}

// LAYER 1: A = xbuf [rows, K=d], B = W1[e] [d, N=d_ff], out hbuf (T).
// LAYER 2: A = hbuf [rows, K=d_ff], B = W2[e] [d_ff, N=d], out zbuf (fp32).
template <typename T, int LAYER>
__global__ void __launch_bounds__(kThreads)
k_ffn_simt(int K, int N, const T *__restrict__ Ain, const int32_t *__restrict__ offset,
           const float *__restrict__ row_gate, const T *__restrict__ W, const T *__restrict__ bias,
           void *__restrict__ out, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN];
  const int e = blockIdx.z;
  const int r0 = offset[e], rows = offset[e + 1] - r0;
  const int m0 = blockIdx.y * BM;
  if (m0 >= rows) return;
  const int n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  const T *Wexp = W + (size_t)e * K * N;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += kThreads) {
      int m = i / BK, kk = i % BK;
      int k = k0 + kk;
      As[kk][m] = (m0 + m < rows && k < K) ? ld(Ain, (size_t)(r0 + m0 + m) * K + k) : 0.f;
    }
    for (int i = tid; i < BK * BN; i += kThreads) {
      int kk = i / BN, n = i % BN;
      int k = k0 + kk;
      Bs[kk][n] = (k < K && n0 + n < N) ? ld(Wexp, (size_t)k * N + n0 + n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tm + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tn + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + tm + i;
    if (m >= rows) continue;
    size_t r = (size_t)r0 + m;
    float g = LAYER == 2 ? row_gate[r] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tn + j;
      if (n >= N) continue;
      float v = acc[i][j] + (bias ? ld(bias, (size_t)e * N + n) : 0.f);
      if (LAYER == 1) {
        v = fmaxf(v, 0.f);
        T *o = static_cast<T *>(out);
        if constexpr (sizeof(T) == 2) o[r * N + n] = __float2bfloat16_rn(v);
        else o[r * N + n] = v;
      } else {
        v *= g;
        if (!isfinite(v)) record_error(st, MOE_ERR_NONFINITE, (long long)(r * N + n));
        static_cast<float *>(out)[r * N + n] = v;
      }
    }
  }
}

template <typename T>
cudaError_t run(const moe_config &cfg, int C, const void *xbuf, const int32_t *offset,
                const float *row_gate, const void *W1, const void *b1, const void *W2,
                const void *b2, void *hbuf, float *zbuf, DeviceStatus *st, cudaStream_t s) {
  const int mt = (C + BM - 1) / BM;
  dim3 g1((cfg.d_ff + BN - 1) / BN, mt, cfg.E);
  launch_pdl_c(kPdlGemm, k_ffn_simt<T, 1>, g1, kThreads, 0, s, cfg.d, cfg.d_ff, (const T *)xbuf,
      offset, row_gate, (const T *)W1, (const T *)b1, hbuf, st);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  dim3 g2((cfg.d + BN - 1) / BN, mt, cfg.E);
  launch_pdl_c(kPdlGemm, k_ffn_simt<T, 2>, g2, kThreads, 0, s, cfg.d_ff, cfg.d, (const T *)hbuf,
      offset, row_gate, (const T *)W2, (const T *)b2, zbuf, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_simt(const moe_config &cfg, int C, const void *xbuf, const int32_t *offset,
                            const float *row_gate, const void *W1, const void *b1, const void *W2,
                            const void *b2, void *hbuf, float *zbuf, DeviceStatus *st,
                            cudaStream_t s) {
  if (cfg.act_dtype == MOE_BF16)
    return run<__nv_bfloat16>(cfg, C, xbuf, offset, row_gate, W1, b1, W2, b2, hbuf, zbuf, st, s);
  return run<float>(cfg, C, xbuf, offset, row_gate, W1, b1, W2, b2, hbuf, zbuf, st, s);
}

}  // namespace moe
