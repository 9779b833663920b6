// Strictly balanced gating ("Outrageously Large", Strictly Balanced Gating
// (Batchwise Mask); the lesson's mask form of the gate, Ch. 2 and Ch. 4).
// P = G_sigma(x) = Softmax(H) over all E experts (H the clean router logits);
// for each expert the m tokens with the largest P (lower token first on ties)
// are its rows, m = max(1, min(T, floor(k T / E))); a token's gate on a picked
// expert is P renormalised over the token's own picks. Kernels, in order:
//   k_bal_softmax  P for every (token, expert), written expert-major
//                  (PT [E][T]) so that each expert's column is contiguous;
//   k_bal_select   a block per expert: radix select of the m-th largest P
//                  (three digit passes over the fp32 bit patterns, which
//                  order like the values for P >= 0), then one pass in token
//                  order that takes every larger value and the first ties,
//                  writes the expert's rows (their tokens) in token order, sets
//                  the token's bit in the mask, adds the expert's
//                  L_batchwise terms, and writes the row offsets e*m;
//   k_bal_tokens   a warp per token: the sum of P over its picks (expert
//                  order) and each pick's renormalised gate into the row's
//                  row_gate (the row found by binary search in the expert's
//                  token-ordered list), keeping the rows of its first picks;
//   k_bal_combine  a warp per token: y = x + the sum over its picks, in
//                  expert order, of the expert rows' outputs (fp32, rounded
//                  once);
//   k_bal_loss     the experts' L_batchwise terms summed in expert order.
// The rows then go through the flat gather and expert GEMMs.
#include "moe_internal.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kBalTok = 32;       // tokens per softmax block
constexpr int kBalChunk = 256;    // experts per shared-memory tile in the softmax
constexpr int kSelThreads = 1024;
constexpr int kRowWarps = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256)
k_bal_softmax(int T, int E, const float *__restrict__ H, float *__restrict__ PT) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[kBalTok][kBalChunk + 1];
  __shared__ float s_mx[kBalTok], s_inv[kBalTok];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kBalTok, nt = min(kBalTok, T - t0);
  for (int tt = warp; tt < nt; tt += 8) {
    const float *h = H + (size_t)(t0 + tt) * E;
    float mx = -INFINITY;
    for (int e = lane; e < E; e += 32) mx = fmaxf(mx, h[e]);
    mx = warp_max(mx);
    float se = 0.f;
    for (int e = lane; e < E; e += 32) se += expf(h[e] - mx);
    se = warp_sum(se);
    if (lane == 0) {
      s_mx[tt] = mx;
      s_inv[tt] = 1.f / se;
    }
  }
  __syncthreads();
  for (int c0 = 0; c0 < E; c0 += kBalChunk) {
    const int nc = min(kBalChunk, E - c0);
    for (int tt = warp; tt < nt; tt += 8) {
      const float *h = H + (size_t)(t0 + tt) * E + c0;
      const float mx = s_mx[tt], inv = s_inv[tt];
      for (int j = lane; j < nc; j += 32) tile[tt][j] = expf(h[j] - mx) * inv;
    }
    __syncthreads();
    for (int j = warp; j < nc; j += 8)  // expert c0 + j: its 32 tokens, one store
      if (lane < nt) PT[(size_t)(c0 + j) * T + t0 + lane] = tile[lane][j];
    __syncthreads();
  }
}

// Exclusive scan of one int per thread over a 1024-thread block; *total gets
// the block's sum. sh holds 33 ints.
__device__ int block_scan_excl(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = sh[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    sh[lane] = wi - w;
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const int r = sh[warp] + incl - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

// One block per expert e. Keys are the fp32 bit patterns of P (P >= 0, so
// key order is value order). The m-th largest key is found digit by digit
// (bits 31..21, 20..10, 9..0): each pass histograms the keys that match the
// digits found so far and picks the bin holding the remaining rank, counting
// from the top bin down.
__global__ void __launch_bounds__(kSelThreads)
k_bal_select(int T, int E, int k, int m, const float *__restrict__ PT,
             const float *__restrict__ thr, int32_t *__restrict__ row_token,
             int32_t *__restrict__ offset, uint32_t *__restrict__ mask,
             double *__restrict__ loss_part, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  __shared__ int hist[2048];
  __shared__ int sh[33];
  __shared__ int s_bin, s_above;
  __shared__ double s_loss[kSelThreads / 32];
  const int e = blockIdx.x, tid = threadIdx.x;
  const uint32_t *col = reinterpret_cast<const uint32_t *>(PT + (size_t)e * T);
  const int W = (E + 31) / 32;
  uint32_t prefix = 0, known = 0;
  int remaining = m;  // rank still to find among the keys matching prefix
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int p = 0; p < 3; ++p) {
    const int shift = shifts[p], nb = 1 << widths[p];
    for (int b = tid; b < 2048; b += kSelThreads) hist[b] = 0;
    __syncthreads();
    for (int t = tid; t < T; t += kSelThreads) {
      const uint32_t u = col[t];
      if ((u & known) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // Thread i holds bins 2r+1, 2r with r = nb/2 - 1 - i (top bins first).
    const int r = nb / 2 - 1 - tid;
    const int hi = r >= 0 ? hist[2 * r + 1] : 0, lo = r >= 0 ? hist[2 * r] : 0;
    int total;
    const int above = block_scan_excl(hi + lo, sh, &total);
    if (r >= 0 && above < remaining && remaining <= above + hi + lo) {
      if (remaining <= above + hi) {
        s_bin = 2 * r + 1;
        s_above = above;
      } else {
        s_bin = 2 * r;
        s_above = above + hi;
      }
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= (uint32_t)s_bin << shift;
    known |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  const uint32_t tau = prefix;  // the m-th largest key; take `remaining` of its ties
  int carry_eq = 0, carry_take = 0;
  double lsum = 0.0;
  const float th = thr ? thr[e] : 0.f;
  for (int base = 0; base < T; base += kSelThreads) {
    const int t = base + tid;
    const uint32_t u = t < T ? col[t] : 0u;
    const bool eq = t < T && u == tau;
    int tot_eq;
    const int eq_before = carry_eq + block_scan_excl(eq ? 1 : 0, sh, &tot_eq);
    const bool take = t < T && (u > tau || (eq && eq_before < remaining));
    int tot_take;
    const int pos = carry_take + block_scan_excl(take ? 1 : 0, sh, &tot_take);
    if (take) {
      if (pos < m) {
        const size_t row = (size_t)e * m + pos;
        row_token[row] = t * k;
        atomicOr(&mask[(size_t)t * W + (e >> 5)], 1u << (e & 31));
      } else {
        record_error(st, MOE_ERR_BOUNDS, (long long)e);
      }
    }
    if (thr && t < T) {
      const float pv = __uint_as_float(u);
      lsum += (double)(((pv > th) ? 1.f : 0.f) - (take ? 1.f : 0.f)) * ((double)pv - (double)th);
    }
    carry_eq += tot_eq;
    carry_take += tot_take;
  }
  if (tid == 0) {
    offset[e] = e * m;
    if (e == E - 1) offset[E] = E * m;
    if (carry_take != m) record_error(st, MOE_ERR_BOUNDS, (long long)e);
  }
  if (thr) {
#pragma unroll
    for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if ((tid & 31) == 0) s_loss[tid >> 5] = lsum;
    __syncthreads();
    if (tid == 0) {
      double s = 0.0;
      for (int w = 0; w < kSelThreads / 32; ++w) s += s_loss[w];
      loss_part[e] = s;
    }
  }
}

// The row of token t in expert e's token-ordered list (rows e*m .. e*m+m-1
// hold t*k for their tokens): binary search; -1 if absent.
__device__ __forceinline__ int find_row(const int32_t *__restrict__ row_token, int e, int m,
                                        int key) {
  int lo = 0, hi = m;
  const int32_t *l = row_token + (size_t)e * m;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(l + mid) < key) lo = mid + 1;
    else hi = mid;
  }
  return (lo < m && __ldg(l + lo) == key) ? e * m + lo : -1;
}

// Rows of a token's first kBalKeep picks, kept for the combine (later picks,
// rare, are looked up again there).
constexpr int kBalKeep = kBalKeepRows;

__global__ void __launch_bounds__(kRowWarps * 32)
k_bal_tokens(int T, int E, int k, int m, const float *__restrict__ PT,
             const uint32_t *__restrict__ mask, const int32_t *__restrict__ row_token,
             float *__restrict__ row_gate, int32_t *__restrict__ trows,
             int32_t *__restrict__ npick, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int W = (E + 31) / 32;
  float part = 0.f;  // this lane's experts, in expert order
  for (int w = lane; w < W; w += 32) {
    uint32_t bits = mask[(size_t)t * W + w];
    while (bits) {
      const int e = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      part += PT[(size_t)e * T + t];
    }
  }
  // The lanes' sums in a fixed order (lane order).
  float z = 0.f;
  for (int l = 0; l < 32; ++l) z += __shfl_sync(0xffffffffu, part, l);
  // Picks before this lane's words (for the pick number j of each pick).
  int cnt = 0;
  for (int w = lane; w < W; w += 32) cnt += __popc(mask[(size_t)t * W + w]);
  int before = 0, total = 0;
  for (int l = 0; l < 32; ++l) {
    const int c = __shfl_sync(0xffffffffu, cnt, l);
    if (l < lane) before += c;
    total += c;
  }
  if (lane == 0) npick[t] = total;
  if (z == 0.f) return;  // no expert took this token
  const float inv = 1.f / z;
  int j = before;
  for (int w = lane; w < W; w += 32) {
    uint32_t bits = mask[(size_t)t * W + w];
    while (bits) {
      const int e = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      const int row = find_row(row_token, e, m, t * k);
      if (row < 0) {
        record_error(st, MOE_ERR_BOUNDS, (long long)t);
        ++j;
        continue;
      }
      row_gate[row] = PT[(size_t)e * T + t] * inv;
      if (j < kBalKeep) trows[(size_t)t * kBalKeep + j] = row;
      ++j;
    }
  }
}

// y = x + the sum over the token's picks (expert order) of the rows' Z, fp32,
// rounded once. ACT: __nv_bfloat16 or float; the lanes take d in order.
template <typename ACT>
__global__ void __launch_bounds__(kRowWarps * 32)
k_bal_combine(int T, int d, int E, int k, int m, const ACT *__restrict__ x,
              const float *__restrict__ zbuf, const uint32_t *__restrict__ mask,
              const int32_t *__restrict__ row_token, const int32_t *__restrict__ trows,
              const int32_t *__restrict__ npick, ACT *__restrict__ y, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int W = (E + 31) / 32;
  const ACT *xr = x + (size_t)t * d;
  ACT *yr = y + (size_t)t * d;
  for (int c0 = 0; c0 < d; c0 += 32 * 8) {  // eight columns per lane at a time
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int c = c0 + lane + 32 * q;
      acc[q] = c < d ? (float)xr[c] : 0.f;
    }
    const int n = npick[t];
    int j = 0;
    for (int w = 0; w < W && j < n; ++w) {
      uint32_t bits = mask[(size_t)t * W + w];
      while (bits) {
        const int e = w * 32 + __ffs(bits) - 1;
        bits &= bits - 1;
        const int row = j < kBalKeep ? trows[(size_t)t * kBalKeep + j] : find_row(row_token, e, m,
                                                                                   t * k);
        ++j;
        if (row < 0) continue;  // reported by k_bal_tokens
        const float *zr = zbuf + (size_t)row * d;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = c0 + lane + 32 * q;
          if (c < d) acc[q] += zr[c];
        }
      }
    }
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int c = c0 + lane + 32 * q;
      if (c < d) {
        yr[c] = (ACT)acc[q];
        bad |= !isfinite(acc[q]);
      }
    }
    if (bad) record_error(st, MOE_ERR_NONFINITE, (long long)t);
  }
}

__global__ void k_bal_loss(int E, const double *__restrict__ part, float *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += part[e];
    out[0] = (float)s;
  }
}

// Threshold mask, the inference-time form of strictly balanced gating
// ("Outrageously Large", Strictly Balanced Gating: M_threshold(x, T)_i = 1
// iff x_i > T_i, applied to G_sigma(x) = Softmax(H), because at inference
// examples arrive one at a time and no batch can be ranked). A warp per token:
// P_i = exp(H_i - max) / sum_j exp(H_j - max) (the evaluation of
// k_bal_softmax), the picks are the experts with P_i > T_i (strict), listed
// in expert order, S = their sum of P and each pick's gate P_i / S. Choice j
// of token t: idx[t*kmax + j] = its j-th pick, or E (no choice) past the
// last; gate = P / S, or 0. The mask row holds bit i % 32 of word i / 32 for
// every pick. A token with more than kmax picks records MOE_ERR_BOUNDS
// (detail = t) and keeps its first kmax.
__global__ void __launch_bounds__(kRowWarps * 32)
k_thr_gate(int T, int E, int kmax, const float *__restrict__ H, const float *__restrict__ thr,
           int32_t *__restrict__ idx, float *__restrict__ gate, uint32_t *__restrict__ mask,
           DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float *h = H + (size_t)t * E;
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, h[e]);
  mx = warp_max(mx);
  float se = 0.f;
  for (int e = lane; e < E; e += 32) se += expf(h[e] - mx);
  se = warp_sum(se);
  const float inv = 1.f / se;
  const unsigned below = (1u << lane) - 1u;
  const int W = (E + 31) / 32;
  // Pass 1: the picks' count and S, 32 experts at a time in expert order.
  int cnt = 0;
  float S = 0.f;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    float pv = 0.f;
    bool take = false;
    if (e < E) {
      pv = expf(h[e] - mx) * inv;
      take = pv > thr[e];
    }
    const unsigned b = __ballot_sync(0xffffffffu, take);
    if (mask && lane == 0) mask[(size_t)t * W + (e0 >> 5)] = b;
    S += warp_sum(take ? pv : 0.f);
    cnt += __popc(b);
  }
  // Pass 2: each pick's choice slot and gate.
  int base = 0;
  for (int e0 = 0; e0 < E && base < kmax; e0 += 32) {
    const int e = e0 + lane;
    float pv = 0.f;
    bool take = false;
    if (e < E) {
      pv = expf(h[e] - mx) * inv;
      take = pv > thr[e];
    }
    const unsigned b = __ballot_sync(0xffffffffu, take);
    const int j = base + __popc(b & below);
    if (take && j < kmax) {
      idx[(size_t)t * kmax + j] = e;
      gate[(size_t)t * kmax + j] = pv / S;
    }
    base += __popc(b);
  }
  for (int j = cnt + lane; j < kmax; j += 32) {
    idx[(size_t)t * kmax + j] = E;
    gate[(size_t)t * kmax + j] = 0.f;
  }
  if (cnt > kmax && lane == 0) record_error(st, MOE_ERR_BOUNDS, (long long)t);
}

}  // namespace

int balanced_m(const moe_config &c) {
  const long long m = (long long)c.k * c.T / c.E;
  return (int)(m < 1 ? 1 : (m > c.T ? c.T : m));
}

cudaError_t launch_bal_gate(const moe_config &c, int m, const float *H, const float *thr,
                            float *PT, int32_t *row_token, float *row_gate, int32_t *offset,
                            uint32_t *mask, int32_t *trows, int32_t *npick, double *loss_part,
                            DeviceStatus *st, cudaStream_t s) {
  const int W = (c.E + 31) / 32;
  cudaError_t err = cudaMemsetAsync(mask, 0, (size_t)c.T * W * 4, s);
  if (err != cudaSuccess) return err;
  launch_pdl(k_bal_softmax, (c.T + kBalTok - 1) / kBalTok, 256, 0, s, c.T, c.E, H, PT);
  launch_pdl(k_bal_select, c.E, kSelThreads, 0, s, c.T, c.E, c.k, m, (const float *)PT, thr,
      row_token, offset, mask, loss_part, st);
  launch_pdl(k_bal_tokens, (c.T + kRowWarps - 1) / kRowWarps, kRowWarps * 32, 0, s, c.T, c.E,
      c.k, m, (const float *)PT, (const uint32_t *)mask, (const int32_t *)row_token, row_gate,
      trows, npick, st);
  return cudaGetLastError();
}

cudaError_t launch_bal_combine(const moe_config &c, int m, const void *x, const float *zbuf,
                               const uint32_t *mask, const int32_t *row_token,
                               const int32_t *trows, const int32_t *npick, void *y,
                               DeviceStatus *st, cudaStream_t s) {
  const dim3 grid((c.T + kRowWarps - 1) / kRowWarps);
  if (c.act_dtype == MOE_BF16)
    launch_pdl(k_bal_combine<__nv_bfloat16>, grid, kRowWarps * 32, 0, s, c.T, c.d, c.E, c.k, m,
        (const __nv_bfloat16 *)x, zbuf, mask, row_token, trows, npick, (__nv_bfloat16 *)y, st);
  else
    launch_pdl(k_bal_combine<float>, grid, kRowWarps * 32, 0, s, c.T, c.d, c.E, c.k, m,
        (const float *)x, zbuf, mask, row_token, trows, npick, (float *)y, st);
  return cudaGetLastError();
}

cudaError_t launch_thr_gate(const moe_config &c, const float *H, const float *thr, int32_t *idx,
                            float *gate, uint32_t *mask, DeviceStatus *st, cudaStream_t s) {
  launch_pdl(k_thr_gate, (c.T + kRowWarps - 1) / kRowWarps, kRowWarps * 32, 0, s, c.T, c.E, c.k,
      H, thr, idx, gate, mask, st);
  return cudaGetLastError();
}

cudaError_t launch_bal_loss(int E, const double *loss_part, float *out, cudaStream_t s) {
  launch_pdl(k_bal_loss, 1, 32, 0, s, E, loss_part, out);
  return cudaGetLastError();
}

}  // namespace moe
