// Internal declarations shared by the translation units of libmoe.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ----------------------------------------------------------------------------- dependent launch
// Every kernel of the library is launched with programmatic dependent launch:
// it may become resident while the previous kernel on the stream drains, and
// it calls pdl_wait() before touching global memory that earlier work writes
// or reads (the wait returns once the previous grid has completed and its
// writes are visible), then pdl_trigger() so the next kernel can be scheduled
// early. A kernel whose predecessor is not a kernel (a memset, an event wait)
// starts in stream order and its wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch classes for the PDL switch: the environment variable MOE_PDL_MASK
// (read once; default all) keeps the attribute for the classes whose bit is
// set, so each kind of edge can be compared with plain stream order.
enum PdlClass { kPdlOther = 0, kPdlGemm = 1, kPdlCombine = 2, kPdlFinalize = 3 };
bool pdl_enabled(int cls = kPdlOther);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_c(int cls, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                size_t smem, cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled(cls) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  return launch_pdl_c(kPdlOther, kernel, grid, block, smem, s, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------- tiling constants
constexpr int kSlotChunk = 512;     // assignments ranked per warp in the slot pass
constexpr int kTcBM = 128;          // rows per tile of the tensor-core expert GEMM
constexpr int kSimtBM = 64;         // rows per tile of the CUDA-core expert GEMM

// ----------------------------------------------------------------------------- device status word
// Lives at offset 0 of the workspace. The first error wins; later ones are dropped.
struct DeviceStatus {
  int32_t code;
  uint32_t aux_ticket;  // blocks of the balancing finalize that are done (reset by the last)
  long long detail;
  uint32_t slot_ticket;  // blocks of the slot scan that are done (zeroed by the histogram pass)
  uint32_t reserved;
  // The CTA-pair expert GEMM's tile scheduler: tiles handed out past each
  // pair's first, and pairs done (the last pair resets both to zero).
  uint32_t gemm_next, gemm_done;
};

__device__ __forceinline__ void record_error(DeviceStatus *st, int code, long long detail) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    *reinterpret_cast<volatile long long *>(&st->detail) = detail;
  }
}

// ----------------------------------------------------------------------------- workspace layout
struct WsLayout {
  size_t status;
  size_t c, sigma, H, rowstat;            // router results kept for the balancing sums
  size_t bsplit;                          // router weights as three bf16 pieces (tensor-core router)
  size_t hist, chunk_base;                // slot pass: per-chunk per-expert counts and bases
  size_t count, offset, mtiles;           // per-expert totals, row offsets, GEMM tile prefix
  size_t ecap;                            // ranked dispatch: capacity left to this rank per expert
  size_t out3s;                           // scratch losses of moe_aux_totals
  size_t partials, aux_vec;               // balancing partial sums and final vectors
  size_t idx, gate, thr, pos, keep;       // moe_forward's own copies of the gate / slot outputs
  size_t row_token, row_gate;             // moe_forward's dispatch maps
  size_t xbuf, hbuf, zbuf;                // moe_forward's expert buffers
  size_t total;
  int n_chunks, n_aux_blocks;
};

WsLayout ws_layout(const moe_config &cfg);

// The calling thread's current CUDA context (a CUcontext, fetched through the
// runtime's driver entry point; the library does not link libcuda), or null if
// none is current. Host caches of per-context objects compare it to notice a
// context that was reset or replaced.
void *current_context();

template <typename T>
inline T *ws_at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

inline int elem_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

// ----------------------------------------------------------------------------- launchers
// Each returns a cudaError_t from the launch (cudaSuccess if nothing failed).

// Selection outputs the tensor-core router can produce in its own epilogue
// when one tile holds every expert of a row: expert_idx [T,k], gate [T,k],
// thr [T,2], rowstat [T,2] (row max, sum of exp(H - max)) and, when partials
// is not null, the balancing partial rows (one per 16 tokens, aux_rows).
struct RouterSelect {
  int32_t *idx;
  float *gate, *thr, *rowstat, *partials;
};

// k_gate.cu: router GEMM + noise + softplus, selection + softmax, balancing partials.
// With `sel` given, *selected tells whether the router also wrote the
// selection outputs (and the partials, if asked for); otherwise the caller
// launches the selection kernels.
cudaError_t launch_router(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                          const float *noise, const float *bias, float *c, float *sigma, float *H,
                          void *bsplit, DeviceStatus *st, cudaStream_t s,
                          const RouterSelect *sel = nullptr, bool *selected = nullptr);
cudaError_t launch_select(const moe_config &cfg, const float *H, int32_t *idx, float *gate,
                          float *thr, float *rowstat, DeviceStatus *st, cudaStream_t s);
cudaError_t launch_aux_partials(const moe_config &cfg, bool noisy, const float *c,
                                const float *sigma, const float *H, const float *rowstat,
                                const int32_t *idx, const float *gate, const float *thr,
                                float *partials, int n_blocks, cudaStream_t s);
// raw_totals [4][E] or null: the summed partial rows (importance, load, first
// choices, sum of Softmax(H)) in fp32 before any division by T.
cudaError_t launch_aux_finalize(const moe_config &cfg, const float *partials, int n_blocks,
                                float *out3, float *importance, float *load, float2 *aux_vec,
                                DeviceStatus *st, cudaStream_t s, float *raw_totals = nullptr);
int aux_rows(int T, int E);  // partial rows of the balancing sums
// Selection and balancing partials in one kernel (E <= 256).
cudaError_t launch_select_aux(const moe_config &cfg, bool noisy, const float *c, const float *sigma,
                              const float *H, int32_t *idx, float *gate, float *thr,
                              float *rowstat, float *partials, int n_blocks, cudaStream_t s);

// Hierarchical gate (k_gate.cu): two-level selection with the balancing
// partial rows (hier_rows(T, kp, b) rows of [4][a*b]), and the losses from the
// finalizes' sums.
// With poff and pos_p given, the secondary logits are the grouped router's
// compact rows: (t, q) at row poff[group] + pos_p[t*kp + q], stride b.
cudaError_t launch_hier_select(int T, int a, int b, int kp, int ks, bool noisy,
                               const int32_t *idx_p, const float *g_p, const float *cs,
                               const float *ss, const float *Hs, const int32_t *poff,
                               const int32_t *pos_p, int32_t *idx, float *gate,
                               float *partials, DeviceStatus *st, cudaStream_t s);
int hier_rows(int T, int kp, int b);
cudaError_t launch_hier_tail(int T, int a, int b, const float2 *aux_s, const float2 *aux_p,
                             float *out2, DeviceStatus *st, const DeviceStatus *st_p,
                             cudaStream_t s);

// k_balanced.cu: strictly balanced gating (batchwise mask). m rows per expert.
int balanced_m(const moe_config &c);
constexpr int kBalKeepRows = 8;  // rows kept per token for the combine
cudaError_t launch_bal_gate(const moe_config &c, int m, const float *H, const float *thr,
                            float *PT, int32_t *row_token, float *row_gate, int32_t *offset,
                            uint32_t *mask, int32_t *trows, int32_t *npick, double *loss_part,
                            DeviceStatus *st, cudaStream_t s);
cudaError_t launch_bal_combine(const moe_config &c, int m, const void *x, const float *zbuf,
                               const uint32_t *mask, const int32_t *row_token,
                               const int32_t *trows, const int32_t *npick, void *y,
                               DeviceStatus *st, cudaStream_t s);
cudaError_t launch_bal_loss(int E, const double *loss_part, float *out, cudaStream_t s);
// The threshold mask (k_balanced.cu): per token the experts whose softmax gate
// exceeds their threshold, in expert order, with gates renormalised over
// them; idx / gate [T, c.k] with E / 0 past a token's last pick; mask
// [T][ceil(E/32)] or null. More than c.k picks: MOE_ERR_BOUNDS.
cudaError_t launch_thr_gate(const moe_config &c, const float *H, const float *thr, int32_t *idx,
                            float *gate, uint32_t *mask, DeviceStatus *st, cudaStream_t s);

// k_router_tc.cu, grouped form: the hierarchical layer's secondary logits for
// the (token, primary pick) pairs only. xg holds group i's tokens in rows
// goff[i] .. goff[i+1]-1 (grow: packed row -> t*kp + q); Wg, Wn [d, a*b];
// noise [T, a*b]; outputs c, sigma, H [T*kp + a*128][b] at the padded row
// offsets written to poff [a+1]. Supported when a group's columns fill whole
// blocks (2b or b in {16, 32} or a multiple of 64), b % 4 == 0, bf16 x.
struct GroupedRouter {
  int T, d, a, b, kp;
  const void *xg;
  const int32_t *goff, *grow;
  const float *Wg, *Wn, *noise;
  float *c, *sigma, *H;
  int32_t *poff;
  void *bsplit;
};
bool router_grouped_supported(int d, int b, bool noisy, bool bf16);
cudaError_t launch_router_grouped(const GroupedRouter &r, DeviceStatus *st, cudaStream_t s);

// k_router_tc.cu: the router as three bf16 tensor-core GEMMs (exact split of W).
bool router_tc_supported(const moe_config &cfg);
size_t router_tc_split_bytes(const moe_config &cfg);
cudaError_t launch_router_tc(const moe_config &cfg, const void *x, const float *Wg, const float *Wn,
                             const float *noise, const float *bias, float *c, float *sigma,
                             float *H, void *bsplit, DeviceStatus *st, cudaStream_t s,
                             const RouterSelect *sel, bool *selected);

// k_slots.cu: capacity, token-order slots, dispatch maps.
// With allow_none, an expert index equal to E marks an empty choice (pos -1,
// keep 0, no row) instead of an index error. With ranks, this rank's
// assignments follow those of the earlier ranks (counts_all [W, E] device,
// rank in 0..W-1): the capacity left to it per expert, max(0, C - the earlier
// ranks' count), is written to ecap [E] and decides keep. With pos null only
// the counts (and offsets) are computed.
struct SlotRanks {
  const int32_t *counts_all;
  int rank;
  int32_t *ecap;
};
cudaError_t launch_slots(const moe_config &cfg, int C, const int32_t *idx, const float *gate,
                         int32_t *hist, int32_t *chunk_base, int32_t *count, int32_t *offset,
                         int32_t *mtiles, int32_t *pos, uint8_t *keep, int32_t *row_token,
                         float *row_gate, int n_chunks, DeviceStatus *st, cudaStream_t s,
                         bool allow_none = false, const SlotRanks *ranks = nullptr);

// k_rows.cu: gather of accepted token rows and the combine with the residual.
cudaError_t launch_gather(const moe_config &cfg, const void *x, const int32_t *offset,
                          const int32_t *row_token, void *xbuf, DeviceStatus *st,
                          cudaStream_t s);
cudaError_t launch_combine(const moe_config &cfg, const void *x, const void *zbuf, bool z_bf16,
                           const int32_t *pos, const uint8_t *keep, const int32_t *idx,
                           const int32_t *offset, void *y, DeviceStatus *st, cudaStream_t s);

// k_ffn_simt.cu: CUDA-core grouped expert GEMMs (fp32, and shapes the tensor-core path rejects).
cudaError_t launch_ffn_simt(const moe_config &cfg, int C, const void *xbuf, const int32_t *offset,
                            const float *row_gate, const void *W1, const void *b1, const void *W2,
                            const void *b2, void *hbuf, float *zbuf, DeviceStatus *st,
                            cudaStream_t s);

// k_ffn_tc.cu: tcgen05 / TMEM / TMA grouped expert GEMMs for bf16.
bool ffn_tc_supported(const moe_config &cfg);
cudaError_t launch_ffn_tc(const moe_config &cfg, int C, const void *xbuf, const int32_t *offset,
                          const int32_t *mtiles, const float *row_gate, const void *W1,
                          const void *b1, const void *W2, const void *b2, void *hbuf, void *zbuf,
                          bool z_bf16, DeviceStatus *st,
                          cudaStream_t s);  // z_bf16: Z in bf16 (else fp32)

// ----------------------------------------------------------------------------- backward
// Padded row blocks of the backward's row buffers: each expert's rows start at
// poff[e] and take max(64, roundup(rows, 64)) rows, pad rows zero.
constexpr int kBwdRowPad = 64;

// k_bwd_tc.cu: the expert backward GEMMs on tcgen05. mode 0: D = dY W2^T with
// the dgate partials and dpre (A = dY rows [a_rows, K = d], B = W2 as
// [E*N, K], N = d_ff); mode 1: dX = dpre W1^T (A = dpre rows [a_rows, K =
// d_ff], B = W1 as [E*N, K], N = d); mode 2: out[e] = A^T B over the padded
// rows (A: the forward's packed rows [a_rows, M], B: padded rows [b_rows, N]).
struct BwdGemm {
  int mode, K, N, M, E;
  long long a_rows, b_rows;
  long long k_len;  // mode 2: rows per expert to expect (for the kernel choice)
  const void *A, *B;
  const int32_t *offset, *poff;
  const float *row_gate;
  const void *hbuf;
  void *out;
  float *dgpart;
};
bool bwd_tc_supported(const moe_config &cfg);
cudaError_t launch_bwd_gemm(const BwdGemm &g, DeviceStatus *st, cudaStream_t s);

// k_bwd_simt.cu: the expert backward on the CUDA cores (fp32 layers, and bf16
// shapes the tensor-core kernels do not take); its row buffers are fp32.
struct BwdSimt {
  long long P_max;
  const int32_t *offset, *poff, *row_token;
  const float *row_gate;
  const void *dy, *W1, *W2, *b2, *xbuf, *hbuf;
  float *dY, *dU, *dP, *dX, *dgpart, *dW1, *dW2;
  DeviceStatus *st;
};
int simt_dgate_blocks(const moe_config &c);  // column blocks of the dgate partials
// gather and the dgrad through W2 (dpre, dgate partials)
cudaError_t launch_bwd_simt_front(const moe_config &c, const BwdSimt &p, cudaStream_t s);
// the dgrad through W1 and both weight gradients
cudaError_t launch_bwd_simt_back(const moe_config &c, const BwdSimt &p, cudaStream_t s);
cudaError_t launch_bwd_simt_dg(const moe_config &c, const BwdSimt &p, float *dg, cudaStream_t s);
cudaError_t launch_bwd_simt_dx(const moe_config &c, const BwdSimt &p, const int32_t *idx,
                               const int32_t *pos, const uint8_t *keep, const float *dxr,
                               void *dx, cudaStream_t s);

// k_bwd.cu: the CUDA-core kernels of the backward.
int sm_count();  // multiprocessors of the current device (k_ffn_tc.cu)
int xtd_splits(int T, int d, int NC);
int colsum_chunks(int C);
cudaError_t launch_bwd_offsets(int E, const int32_t *offset, int32_t *poff, cudaStream_t s);
cudaError_t launch_bwd_tail_zero(const moe_config &c, const int32_t *offset, void *xbuf,
                                 void *hbuf, cudaStream_t s);
cudaError_t launch_bwd_gather(const moe_config &c, long long P_max, const int32_t *offset,
                              const int32_t *poff, const int32_t *row_token,
                              const float *row_gate, const void *dy, void *dY, void *dU,
                              cudaStream_t s);
cudaError_t launch_bwd_dg(const moe_config &c, int n_blocks, const int32_t *offset,
                          const int32_t *poff, const int32_t *row_token, const float *dgpart,
                          const void *dy, const void *b2, float *dg, cudaStream_t s);
cudaError_t launch_bwd_coef(const moe_config &c, const float2 *aux_vec, float w_imp,
                            float w_load, float w_aux, float *coef, cudaStream_t s);
cudaError_t launch_bwd_gate(const moe_config &c, bool noisy, bool load_on, bool aux_on,
                            bool dg_total, const float *H, const float *cc, const float *sigma,
                            const float *noise, const float *rowstat, const float *thr,
                            const int32_t *idx, const float *gate, const uint8_t *keep,
                            const float *dg, const float *coef, float *dgate_out, float *dc,
                            float *dz, cudaStream_t s);
// x is act_dtype (bf16 or fp32).
cudaError_t launch_bwd_router(const moe_config &c, bool noisy, const void *x, const float *Wg,
                              const float *Wn, const float *dc, const float *dz, float *part,
                              float *bpart, float *dWg, float *dWn, float *dbias, float *dxr,
                              cudaStream_t s);
// src rows are bf16, or fp32 when src_f32.
cudaError_t launch_bwd_colsum(const moe_config &c, int cols, int chunks, const int32_t *offset,
                              const int32_t *poff, const float *row_gate, const void *src,
                              bool src_f32, float *part, float *out, cudaStream_t s);
cudaError_t launch_bwd_dx(const moe_config &c, const int32_t *idx, const int32_t *pos,
                          const uint8_t *keep, const int32_t *poff, const float *dX,
                          const float *dxr, const void *dy, void *dx, cudaStream_t s);

}  // namespace moe
