// Stage 3: capacity and token-order slot assignment ("Switch Transformer",
// steps 3-4). The position of assignment a = t*k + j is the number of earlier
// assignments (in that flat, token-major order) to the same expert: an
// exclusive cumulative count. It is computed without atomics on the order:
//   k_slot_hist  -- per chunk of kSlotChunk assignments, count per expert;
//   k_slot_scan  -- per expert, exclusive sum over chunks (chunk bases) and
//                   the total n_e; the last block to finish then scans
//                   min(n_e, C) into row offsets and GEMM tile offsets;
//   k_slot_rank  -- one warp walks each chunk in order, 32 assignments at a
//                   time: __match_any_sync finds same-expert lanes, the rank
//                   among them is a popcount, a per-warp counter carries it.
// Kept assignments (pos < C) get row offset[e] + pos of the packed buffer.
#include "moe_internal.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr int kHistThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kScanBatch = 16;
constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(kHistThreads)
k_slot_hist(int A, int E, int allow_none, const int32_t *__restrict__ idx,
            int32_t *__restrict__ hist, DeviceStatus *st) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sh_hist[];
  if (blockIdx.x == 0 && threadIdx.x == 0) st->slot_ticket = 0;  // for k_slot_scan, next in order
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kSlotChunk;
  for (int i = threadIdx.x; i < kSlotChunk; i += blockDim.x) {
    int a = a0 + i;
    if (a >= A) break;
    int e = idx[a];
    if (e == E && allow_none) continue;  // an empty choice
    if (e < 0 || e >= E) {
      record_error(st, MOE_ERR_BOUNDS, (long long)a);
      continue;
    }
    atomicAdd(&sh_hist[e], 1);  // integer counts: order does not matter
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh_hist[e];
}

// Exclusive block scan of one int per thread (blockDim.x == kScanThreads).
__device__ int block_exclusive_scan(int v, int *sh_warp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = sh_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    sh_warp[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) sh_warp[32] = wi;
  }
  __syncthreads();
  int r = sh_warp[warp] + incl - v;
  *total = sh_warp[32];
  __syncthreads();
  return r;
}

// Block per 32 experts: lane l takes expert 32 blockIdx.x + l, warp w the
// chunk segment [w S, (w+1) S), S = ceil(n_chunks / 32), so hist rows are read
// coalesced. Segment totals are added across warps in shared memory, giving
// each warp its base; the warp then writes its chunks' bases. The block that
// finishes last (a ticket in the status word) scans min(n_e, C) and the tile
// counts over all experts, kScanThreads at a time, into offset and mtiles.
//
// Ranked form (counts_all given: the per-expert choice counts [W, E] of the W
// ranks whose batches, in rank order, make up the layer's batch): this rank's
// assignments to expert e come after base_e = sum over earlier ranks of their
// counts, so the capacity left to this rank is cap_e = max(0, C - base_e);
// the last block writes it to ecap, and the kept rows per expert are
// min(n_e, cap_e).
__global__ void __launch_bounds__(kScanThreads)
k_slot_scan(int E, int C, int n_chunks, int bm, int32_t *__restrict__ hist_base,
            int32_t *__restrict__ count, int32_t *__restrict__ offset,
            int32_t *__restrict__ mtiles, const int32_t *__restrict__ hist, DeviceStatus *st,
            const int32_t *__restrict__ counts_all, int rank, int32_t *__restrict__ ecap) {
  pdl_wait();
  pdl_trigger();
  constexpr int NW = kScanThreads / 32;
  __shared__ int seg[NW][33];
  __shared__ int sh_warp[33];
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int S = (n_chunks + NW - 1) / NW;
  const int c0 = min(n_chunks, warp * S), c1 = min(n_chunks, c0 + S);
  int tot = 0;
  if (e < E) {
    for (int cb = c0; cb < c1; cb += kScanBatch) {
      int h[kScanBatch];
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u)
        h[u] = cb + u < c1 ? hist[(size_t)(cb + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) tot += h[u];
    }
  }
  seg[warp][lane] = tot;
  __syncthreads();
  int n = 0;
  for (int w = 0; w < warp; ++w) n += seg[w][lane];
  if (e < E) {
    for (int c = c0; c < c1; ++c) {  // hist rows are L2-resident by now
      const int h = hist[(size_t)c * E + e];
      hist_base[(size_t)c * E + e] = n;
      n += h;
    }
    if (warp == NW - 1) count[e] = n;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&st->slot_ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const volatile int32_t *cnt = count;
  int carry_rows = 0, carry_tiles = 0;
  for (int e0 = 0; e0 < E; e0 += kScanThreads) {
    const int ee = e0 + threadIdx.x;
    int capv = C;
    if (counts_all && ee < E) {
      long long base = 0;
      for (int r = 0; r < rank; ++r) base += counts_all[(size_t)r * E + ee];
      capv = base >= C ? 0 : (int)(C - base);
      ecap[ee] = capv;
    }
    const int kept = ee < E ? min(cnt[ee], capv) : 0;
    const int tiles = (kept + bm - 1) / bm;
    int tot_rows, tot_tiles;
    const int off = block_exclusive_scan(kept, sh_warp, &tot_rows);
    const int toff = block_exclusive_scan(tiles, sh_warp, &tot_tiles);
    if (ee < E) {
      offset[ee] = carry_rows + off;
      mtiles[ee] = carry_tiles + toff;
    }
    carry_rows += tot_rows;
    carry_tiles += tot_tiles;
  }
  if (threadIdx.x == 0) {
    offset[E] = carry_rows;
    mtiles[E] = carry_tiles;
    st->slot_ticket = 0;
  }
}

// One block per chunk. Warp w ranks its 64 assignments in order (two rounds
// of 32: __match_any_sync groups equal experts, a popcount gives the rank,
// a per-warp counter carries it); an exclusive scan over the warps' counts
// then gives each warp its base, in warp order.
constexpr int kRankPerWarp = kSlotChunk / kRankWarps;

__global__ void __launch_bounds__(kRankWarps * 32)
k_slot_rank(int A, int E, int C, const int32_t *__restrict__ idx, const float *__restrict__ gate,
            const int32_t *__restrict__ hist_base, const int32_t *__restrict__ offset,
            int32_t *__restrict__ pos, uint8_t *__restrict__ keep, int32_t *__restrict__ row_token,
            float *__restrict__ row_gate, const int32_t *__restrict__ ecap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sh_cnt[];  // [kRankWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunk = blockIdx.x;
  for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) sh_cnt[i] = 0;
  __syncthreads();
  int32_t *cnt = sh_cnt + (size_t)warp * E;
  const unsigned lt = (1u << lane) - 1u;
  const int a0 = chunk * kSlotChunk + warp * kRankPerWarp;
  constexpr int R = kRankPerWarp / 32;
  int ee[R], rk[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int a = a0 + 32 * r + lane;
    int e = -1;
    if (a < A) {
      e = idx[a];
      if (e < 0 || e >= E) e = -1;  // an empty choice, or a bounds error k_slot_hist counts
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int before = e >= 0 ? cnt[e] : 0;
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) cnt[e] = before + __popc(peers);  // lowest peer updates
    __syncwarp();
    ee[r] = e;
    rk[r] = before + __popc(peers & lt);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
      const int v = sh_cnt[w * E + e];
      sh_cnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int a = a0 + 32 * r + lane;
    if (a >= A) continue;
    const int e = ee[r];
    if (e < 0) {
      pos[a] = -1;
      keep[a] = 0;
      continue;
    }
    const int p = hist_base[(size_t)chunk * E + e] + cnt[e] + rk[r];
    pos[a] = p;
    const bool kp = p < (ecap ? ecap[e] : C);
    keep[a] = kp ? 1 : 0;
    if (kp) {
      const int row = offset[e] + p;
      row_token[row] = a;
      row_gate[row] = gate[a];
    }
  }
}

}  // namespace

cudaError_t launch_slots(const moe_config &cfg, int C, const int32_t *idx, const float *gate,
                         int32_t *hist, int32_t *chunk_base, int32_t *count, int32_t *offset,
                         int32_t *mtiles, int32_t *pos, uint8_t *keep, int32_t *row_token,
                         float *row_gate, int n_chunks, DeviceStatus *st, cudaStream_t s,
                         bool allow_none, const SlotRanks *ranks) {
  const int A = cfg.T * cfg.k;
  launch_pdl(k_slot_hist, n_chunks, kHistThreads, cfg.E * sizeof(int32_t), s, A, cfg.E,
      allow_none ? 1 : 0, idx, hist, st);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int32_t *counts_all = ranks ? ranks->counts_all : nullptr;
  int32_t *ecap = ranks ? ranks->ecap : nullptr;
  launch_pdl(k_slot_scan, (cfg.E + 31) / 32, kScanThreads, 0, s, cfg.E, C, n_chunks, kTcBM,
      chunk_base, count, offset, mtiles, hist, st, counts_all, ranks ? ranks->rank : 0, ecap);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (!pos) return cudaSuccess;  // counts only
  size_t smem = (size_t)kRankWarps * cfg.E * sizeof(int32_t);
  if (smem > 48 * 1024) {
    err = cudaFuncSetAttribute(k_slot_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
  }
  launch_pdl(k_slot_rank, n_chunks, kRankWarps * 32, smem, s, A, cfg.E, C, idx, gate, chunk_base,
      offset, pos, keep, row_token, row_gate, (const int32_t *)ecap);
  return cudaGetLastError();
}

}  // namespace moe

// ----------------------------------------------------------------------------- allocation-free dispatch
// moe_dispatch_noalloc: the same slot assignment and gather as moe_dispatch,
// for callers that cannot give the library a workspace because they may not
// allocate device memory where they route tokens. Its scratch (the slot pass's
// histograms and chunk bases, tile offsets and a status word) is this file's
// own device array, which every GPU that loads the library keeps until exit.

namespace moe {
namespace {

constexpr size_t kNoAllocBytes = MOE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Device address of the scratch array on the current device. In host code the
// array's name is only a stand-in, so the address is looked up with the
// device current (cudaGetSymbolAddress), once per device and context: the
// cache entry remembers the context it was taken in, and a call made in
// another context -- after cudaDeviceReset, or under a context the caller
// made current -- looks the address up again. The first lookup in a context
// loads the library's module there.
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoAllocEntry {
  void *ctx = nullptr, *ptr = nullptr;
};
NoAllocEntry g_noalloc[kNoAllocMaxDevices];

int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
  void *ctx = current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocEntry &e = g_noalloc[dev];
  if (!e.ptr || !ctx || e.ctx != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      e = NoAllocEntry{};
      return MOE_ERR_CUDA;
    }
    // Re-read the context: the lookup itself may have created the primary one.
    e.ctx = current_context();
    e.ptr = p;
  }
  *out = e.ptr;
  return MOE_OK;
}

bool aligned16(const void *p) { return p && ((uintptr_t)p % 16) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch_noalloc(const moe_config *cfg, const int32_t *expert_idx,
                                    const float *gate, const void *x, int32_t *pos,
                                    uint8_t *keep, int32_t *expert_count, int32_t *expert_offset,
                                    void *xbuf, int32_t *row_token, float *row_gate,
                                    moe_stream_t stream) {
  using namespace moe;
  int32_t C = 0;
  int r = moe_capacity(cfg, &C);  // also validates cfg
  if (r != MOE_OK) return r;
  const void *ptrs[] = {expert_idx, gate, x, pos, keep, expert_count, expert_offset,
                        xbuf, row_token, row_gate};
  for (const void *p : ptrs)
    if (!aligned16(p)) return MOE_ERR_ARG;
  const size_t A = (size_t)cfg->T * cfg->k;
  const size_t n_chunks = (A + kSlotChunk - 1) / kSlotChunk;
  const size_t E = (size_t)cfg->E;
  // Scratch layout: status | hist [n_chunks, E] | chunk bases [n_chunks, E] | tile offsets [E+1]
  const size_t off_hist = 256;
  const size_t off_base = off_hist + round256(n_chunks * E * 4);
  const size_t off_tiles = off_base + round256(n_chunks * E * 4);
  const size_t need = off_tiles + round256((E + 1) * 4);
  if (need > kNoAllocBytes) return MOE_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  r = noalloc_scratch(&scratch);
  if (r != MOE_OK) return r;
  char *base = static_cast<char *>(scratch);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = reinterpret_cast<DeviceStatus *>(base);
  // Only the status word must start at zero; every other scratch word is
  // written before it is read within one call.
  if (cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_slots(*cfg, C, expert_idx, gate, reinterpret_cast<int32_t *>(base + off_hist),
                   reinterpret_cast<int32_t *>(base + off_base), expert_count, expert_offset,
                   reinterpret_cast<int32_t *>(base + off_tiles), pos, keep, row_token, row_gate,
                   (int)n_chunks, st, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gather(*cfg, x, expert_offset, row_token, xbuf, st, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" int moe_noalloc_last_status(moe_stream_t stream, int64_t *detail) {
  using namespace moe;
  void *scratch = nullptr;
  const int r = noalloc_scratch(&scratch);
  if (r != MOE_OK) return r;
  DeviceStatus h{};
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&h, scratch, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(scratch, 0, sizeof h) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = h.detail;
  return h.code;
}
