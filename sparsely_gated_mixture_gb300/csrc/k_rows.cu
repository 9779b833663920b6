// Row movement around the experts.
//   gather  ("Switch Transformer", step 5: dispatch): row r of the packed
//           buffer receives token row_token[r] / k, so expert e's accepted
//           tokens sit contiguously, in token order, from offset[e].
//   combine ("Switch Transformer", step 7; "Outrageously Large", the output
//           y = sum_i G_i E_i(x), plus the residual): y[t] = x[t] + the kept
//           gate-weighted expert rows of t, added in choice order in fp32.
// Both are pure HBM streams: 16-byte vector loads and stores, one warp per row.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRowWarps = 8;

// Gather: copies d elements of `elem` bytes per row, in 16-byte vectors when
// the row length allows (the library requires 16-byte aligned base pointers).
template <typename V>
__global__ void __launch_bounds__(kRowWarps * 32)
k_gather(int A, int k, int nvec, const V *__restrict__ x, const int32_t *__restrict__ offset_end,
         const int32_t *__restrict__ row_token, V *__restrict__ xbuf, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (r >= A || r >= *offset_end) return;
  const int a = row_token[r];
  if (a < 0 || a >= A) {
    if (lane == 0) record_error(st, MOE_ERR_BOUNDS, (long long)r);
    return;
  }
  const int t = a / k;
  const V *src = x + (size_t)t * nvec;
  V *dst = xbuf + (size_t)r * nvec;
  int v = lane;
  for (; v + 96 < nvec; v += 128) {
    V a0 = src[v], a1 = src[v + 32], a2 = src[v + 64], a3 = src[v + 96];
    dst[v] = a0;
    dst[v + 32] = a1;
    dst[v + 64] = a2;
    dst[v + 96] = a3;
  }
  for (; v < nvec; v += 32) dst[v] = src[v];
}

// Gather for short rows (at most 32 * VPL 16-byte vectors): each warp moves
// RPW consecutive packed rows, their tokens and the row count read side by
// side, then every row's vectors loaded before any is stored, so a warp has
// RPW * VPL loads in flight instead of one row's worth.
template <int RPW, int VPL>
__global__ void __launch_bounds__(kRowWarps * 32)
k_gather_short(int A, int k, int nvec, const uint4 *__restrict__ x,
               const int32_t *__restrict__ offset_end, const int32_t *__restrict__ row_token,
               uint4 *__restrict__ xbuf, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * kRowWarps + (threadIdx.x >> 5)) * RPW;
  if (r0 >= A) return;
  const int end = min(*offset_end, A);
  int a_l = -1;
  if (lane < RPW && r0 + lane < A) a_l = row_token[r0 + lane];
  uint4 v[RPW][VPL];
  int tok[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int a = __shfl_sync(0xffffffffu, a_l, i);
    const bool live = r0 + i < end;
    const bool ok = live && a >= 0 && a < A;
    if (live && !ok && lane == 0) record_error(st, MOE_ERR_BOUNDS, (long long)(r0 + i));
    tok[i] = ok ? a / k : -1;
    if (tok[i] >= 0) {
      const uint4 *src = x + (size_t)tok[i] * nvec;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int c = lane + 32 * j;
        if (c < nvec) v[i][j] = src[c];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    if (tok[i] < 0) continue;
    uint4 *dst = xbuf + (size_t)(r0 + i) * nvec;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int c = lane + 32 * j;
      if (c < nvec) dst[c] = v[i][j];
    }
  }
}

template <typename T>
struct Act;
template <>
struct Act<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <>
struct Act<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Combine: one warp per token; each lane handles groups of 4 consecutive
// elements (VEC4) or single elements.
// The packed rows of token t's kept choices, in choice order, on every lane:
// lane j < k resolves choice j (keep, expert, slot -> row offset[e] + pos) so
// the k lookups run side by side, then the rows are read from the lanes in
// order. Returns their number; a bad index is recorded (MOE_ERR_BOUNDS) and
// skipped.
template <int KM>
__device__ __forceinline__ int token_rows(int t, int k, int E, const uint8_t *__restrict__ keep,
                                          const int32_t *__restrict__ idx,
                                          const int32_t *__restrict__ pos,
                                          const int32_t *__restrict__ offset, DeviceStatus *st,
                                          int lane, int (&rows)[KM]) {
  int r = -1;
  if (lane < k) {
    const size_t a = (size_t)t * k + lane;
    if (keep[a]) {
      const int e = idx[a];
      const int rr = (e >= 0 && e < E) ? offset[e] + pos[a] : -1;
      if (rr < 0 || rr >= offset[e + 1])
        record_error(st, MOE_ERR_BOUNDS, (long long)a);
      else
        r = rr;
    }
  }
  int nr = 0;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    if (j >= k) break;
    const int rj = __shfl_sync(0xffffffffu, r, j);
    if (rj >= 0) rows[nr++] = rj;
  }
  return nr;
}

template <typename T, bool VEC4>
__global__ void __launch_bounds__(kRowWarps * 32)
k_combine(int Tn, int d, int E, int k, const T *__restrict__ x, const float *__restrict__ zbuf,
          const int32_t *__restrict__ pos, const uint8_t *__restrict__ keep,
          const int32_t *__restrict__ idx, const int32_t *__restrict__ offset, T *__restrict__ y,
          DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  constexpr int kMaxK = 16;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  int rows[kMaxK];
  const int nr = token_rows<kMaxK>(t, k, E, keep, idx, pos, offset, st, lane, rows);
  const T *xr = x + (size_t)t * d;
  T *yr = y + (size_t)t * d;
  bool bad = false;
  if (VEC4) {
    for (int c = lane * 4; c < d; c += 128) {
      float acc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = Act<T>::to_f(xr[c + q]);
      for (int i = 0; i < nr; ++i) {
        float4 z = *reinterpret_cast<const float4 *>(zbuf + (size_t)rows[i] * d + c);
        acc[0] += z.x;
        acc[1] += z.y;
        acc[2] += z.z;
        acc[3] += z.w;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        bad |= !isfinite(acc[q]);
        yr[c + q] = Act<T>::from_f(acc[q]);
      }
    }
  } else {
    for (int c = lane; c < d; c += 32) {
      float acc = Act<T>::to_f(xr[c]);
      for (int i = 0; i < nr; ++i) acc += zbuf[(size_t)rows[i] * d + c];
      bad |= !isfinite(acc);
      yr[c] = Act<T>::from_f(acc);
    }
  }
  if (bad) record_error(st, MOE_ERR_NONFINITE, (long long)t);
}

// Combine for bf16 rows with d % 8 == 0: each lane handles NG groups of 8
// consecutive elements per step (16-byte loads of x and y; 32 bytes of each
// kept Z row per group, or 16 when Z is bf16 (ZB)), with every load of the
// step issued first; two groups when k <= 2 or Z is bf16, one for fp32 Z with
// k <= 4 (register budget). The sum runs in fp32 in choice order either way.
template <int KM, int NG, bool ZB>  // at most KM choices per token; NG groups per lane-step
__global__ void __launch_bounds__(kRowWarps * 32)
k_combine_bf16x8(int Tn, int d, int E, int k, const __nv_bfloat16 *__restrict__ x,
                 const void *__restrict__ zbuf, const int32_t *__restrict__ pos,
                 const uint8_t *__restrict__ keep, const int32_t *__restrict__ idx,
                 const int32_t *__restrict__ offset, __nv_bfloat16 *__restrict__ y,
                 DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  int rows[KM];
  const int nr = token_rows<KM>(t, k, E, keep, idx, pos, offset, st, lane, rows);
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * d);
  uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)t * d);
  const int nv = d / 8;
  bool bad = false;
  // NG 8-element groups per lane per step, all loads issued before the sums.
  for (int v0 = lane; v0 < nv; v0 += 32 * NG) {
    const int v1 = v0 + 32;
    const bool has1 = NG > 1 && v1 < nv;
    const uint4 xv0 = xr[v0];
    const uint4 xv1 = has1 ? xr[v1] : make_uint4(0, 0, 0, 0);
    // Z of each kept row: raw bf16 (16 bytes per group) or fp32 (32 bytes).
    uint4 zb[ZB ? KM : 1][NG];
    float4 zf[ZB ? 1 : KM][2 * NG];
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      if (i >= nr) break;
      if constexpr (ZB) {
        const uint4 *zr =
            reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(zbuf) +
                                            (size_t)rows[i] * d);
        zb[i][0] = zr[v0];
        if constexpr (NG > 1)
          if (has1) zb[i][1] = zr[v1];
      } else {
        const float4 *zr = reinterpret_cast<const float4 *>(static_cast<const float *>(zbuf) +
                                                            (size_t)rows[i] * d);
        zf[i][0] = zr[2 * v0];
        zf[i][1] = zr[2 * v0 + 1];
        if constexpr (NG > 1) {
          if (has1) {
            zf[i][2] = zr[2 * v1];
            zf[i][3] = zr[2 * v1 + 1];
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < NG; ++h) {
      if (h == 1 && !has1) break;
      const uint4 xv = h ? xv1 : xv0;
      const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&xv);
      float acc[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(xb[q]);
        acc[2 * q] = f.x;
        acc[2 * q + 1] = f.y;
      }
#pragma unroll
      for (int i = 0; i < KM; ++i) {
        if (i >= nr) break;
        if constexpr (ZB) {
          const __nv_bfloat162 *z2 = reinterpret_cast<const __nv_bfloat162 *>(&zb[i][h]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(z2[q]);
            acc[2 * q] += f.x;
            acc[2 * q + 1] += f.y;
          }
        } else {
          const float4 a0 = zf[i][2 * h], a1 = zf[i][2 * h + 1];
          acc[0] += a0.x; acc[1] += a0.y; acc[2] += a0.z; acc[3] += a0.w;
          acc[4] += a1.x; acc[5] += a1.y; acc[6] += a1.z; acc[7] += a1.w;
        }
      }
      uint4 out;
      __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        bad |= !isfinite(acc[2 * q]) || !isfinite(acc[2 * q + 1]);
        ob[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      }
      yr[h ? v1 : v0] = out;
    }
  }
  if (bad) record_error(st, MOE_ERR_NONFINITE, (long long)t);
}

}  // namespace

cudaError_t launch_gather(const moe_config &cfg, const void *x, const int32_t *offset,
                          const int32_t *row_token, void *xbuf, DeviceStatus *st, cudaStream_t s) {
  const int A = cfg.T * cfg.k;
  const size_t row_bytes = (size_t)cfg.d * elem_bytes(cfg.act_dtype);
  dim3 grid((A + kRowWarps - 1) / kRowWarps);
  const int32_t *end = offset + cfg.E;
  const int nv16 = (int)(row_bytes / 16);
  constexpr int kRpw = 4;
  const dim3 grid_s((A + kRowWarps * kRpw - 1) / (kRowWarps * kRpw));
  if (row_bytes % 16 == 0 && nv16 <= 64) {
    if (nv16 <= 32)
      launch_pdl(k_gather_short<kRpw, 1>, grid_s, kRowWarps * 32, 0, s, A, cfg.k, nv16,
          (const uint4 *)x, end, row_token, (uint4 *)xbuf, st);
    else
      launch_pdl(k_gather_short<kRpw, 2>, grid_s, kRowWarps * 32, 0, s, A, cfg.k, nv16,
          (const uint4 *)x, end, row_token, (uint4 *)xbuf, st);
  } else if (row_bytes % 16 == 0 && nv16 <= 128) {
    launch_pdl(k_gather_short<2, 4>, dim3((A + kRowWarps * 2 - 1) / (kRowWarps * 2)),
        kRowWarps * 32, 0, s, A, cfg.k, nv16, (const uint4 *)x, end, row_token, (uint4 *)xbuf,
        st);
  } else if (row_bytes % 16 == 0) {
    launch_pdl(k_gather<uint4>, grid, kRowWarps * 32, 0, s, A, cfg.k, (int)(row_bytes / 16),
        (const uint4 *)x, end, row_token, (uint4 *)xbuf, st);
  } else if (row_bytes % 4 == 0) {
    launch_pdl(k_gather<uint32_t>, grid, kRowWarps * 32, 0, s, A, cfg.k, (int)(row_bytes / 4),
        (const uint32_t *)x, end, row_token, (uint32_t *)xbuf, st);
  } else {
    launch_pdl(k_gather<uint16_t>, grid, kRowWarps * 32, 0, s, A, cfg.k, (int)(row_bytes / 2),
        (const uint16_t *)x, end, row_token, (uint16_t *)xbuf, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_config &cfg, const void *x, const void *zbuf, bool z_bf16,
                           const int32_t *pos, const uint8_t *keep, const int32_t *idx,
                           const int32_t *offset, void *y, DeviceStatus *st, cudaStream_t s) {
  dim3 grid((cfg.T + kRowWarps - 1) / kRowWarps);
  const bool v4 = cfg.d % 4 == 0;
  if (cfg.act_dtype == MOE_BF16) {
    auto xp = (const __nv_bfloat16 *)x;
    auto yp = (__nv_bfloat16 *)y;
    if (cfg.d % 8 == 0 && cfg.k <= 4) {
#define MOE_COMB(KM, NG, ZB)                                                                       \
  launch_pdl_c(kPdlCombine, k_combine_bf16x8<KM, NG, ZB>, grid, kRowWarps * 32, 0, s, cfg.T,       \
      cfg.d, cfg.E, cfg.k, xp, zbuf, pos, keep, idx, offset, yp, st)
      if (cfg.k <= 2) {
        if (z_bf16) MOE_COMB(2, 2, true);
        else MOE_COMB(2, 2, false);
      } else {
        if (z_bf16) MOE_COMB(4, 2, true);  // raw bf16 Z leaves room for two groups
        else MOE_COMB(4, 1, false);
      }
#undef MOE_COMB
    } else if (z_bf16) {
      return cudaErrorInvalidValue;  // bf16 Z is only produced for this form
    } else if (v4)
      launch_pdl_c(kPdlCombine, k_combine<__nv_bfloat16, true>, grid, kRowWarps * 32, 0, s, cfg.T,
          cfg.d, cfg.E, cfg.k, xp, (const float *)zbuf, pos, keep, idx, offset, yp, st);
    else
      launch_pdl_c(kPdlCombine, k_combine<__nv_bfloat16, false>, grid, kRowWarps * 32, 0, s, cfg.T,
          cfg.d, cfg.E, cfg.k, xp, (const float *)zbuf, pos, keep, idx, offset, yp, st);
  } else {
    if (z_bf16) return cudaErrorInvalidValue;
    auto xp = (const float *)x;
    auto yp = (float *)y;
    auto zf = (const float *)zbuf;
    if (v4)
      launch_pdl_c(kPdlCombine, k_combine<float, true>, grid, kRowWarps * 32, 0, s, cfg.T, cfg.d,
          cfg.E, cfg.k, xp, zf, pos, keep, idx, offset, yp, st);
    else
      launch_pdl_c(kPdlCombine, k_combine<float, false>, grid, kRowWarps * 32, 0, s, cfg.T, cfg.d,
          cfg.E, cfg.k, xp, zf, pos, keep, idx, offset, yp, st);
  }
  return cudaGetLastError();
}

}  // namespace moe
