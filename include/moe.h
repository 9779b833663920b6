/*
 * moe.h -- C ABI of libmoe.so: the forward path of the sparsely-gated
 * Mixture-of-Experts layer on one NVIDIA GB300 (sm_103a), its hierarchical
 * and strictly balanced variants, and the flat layer's backward.
 *
 * The layer, as the pages state it ("Outrageously Large Neural Networks: The
 * Sparsely-Gated Mixture-of-Experts Layer", section 3.4; "Switch Transformer",
 * Implementation steps 1-8): T tokens of width d are routed to k of E experts,
 * each a ReLU feed-forward network of hidden width d_ff; each expert accepts at
 * most C = max(min_capacity, min(T, floor(k*T*capacity_factor/E))) of them,
 * in token order; the output is the input plus the gate-weighted sum of the
 * accepted experts' outputs; two balancing losses (importance and load) and
 * the Switch auxiliary loss are reported on the side.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every array argument is a DEVICE pointer owned by the caller, on the
 *   current CUDA device, row-major and contiguous, 16-byte aligned. The library
 *   never allocates, frees or copies host<->device (except moe_last_device_status,
 *   which reads the 32-byte status word back). Scratch space is the caller's
 *   workspace `ws` of moe_workspace_size() bytes (256-byte aligned).
 * Streams.  Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream) and returns without synchronising. moe_forward() runs the
 *   balancing-loss finalize on a side stream, forked from `stream` after the
 *   gate and joined back before it returns (so later work on `stream`, and
 *   stream capture, see one ordered forward); moe_backward forks its gate
 *   branch onto the side stream and joins it back before its last kernel.
 *   Each device has a pool of 8 side streams, made on the first such call
 *   that is not under stream capture (make one call before capturing if the
 *   captured graph should keep the overlap) and kept; each serves one caller
 *   stream, so calls on different streams -- from different host threads,
 *   one of them capturing a graph while another runs eagerly -- never share
 *   a side stream. When none fits (the pool is not made yet and `stream` is
 *   capturing; 8 other caller streams hold them; a side stream in another
 *   capture) the call runs everything on `stream`, with the same results.
 *   After cudaDeviceReset the next call makes a new pool.
 * Element types.  cfg->act_dtype (MOE_F32 or MOE_BF16) is the type of x, W1,
 *   b1, W2, b2, y, xbuf and hbuf. The router weights, router bias, noise,
 *   gates and zbuf are always fp32.
 * Errors.  A bad argument returns MOE_ERR_ARG (or MOE_ERR_UNSUPPORTED) before
 *   anything is enqueued. A failed launch returns MOE_ERR_CUDA; work enqueued
 *   before the failure (on `stream` and, in moe_forward and moe_backward, on
 *   the library's side stream) may still run, so synchronise the device before
 *   reusing the call's buffers. Conditions found
 *   on the device -- a non-finite router logit, expert output or layer output
 *   (the Switch page raises on each), an index out of range, or a bounded wait
 *   that ran out -- are recorded in a status word inside `ws`;
 *   moe_last_device_status() reads it. moe_gate() and moe_forward() clear it
 *   when they start, moe_last_device_status() after reading it; a caller whose
 *   first call on a fresh workspace is another stage zero-fills the workspace
 *   (or calls moe_last_device_status) first. Each bounded wait inside the
 *   tensor-core kernels gives up after 2 s, or after MOE_WAIT_LIMIT_NS
 *   nanoseconds if that environment variable is set when the call is made
 *   (a diagnostic: 0 makes the first wait that is not already satisfied run
 *   out); the kernel then records MOE_ERR_TIMEOUT, finishes its copies and
 *   MMAs in flight and returns, leaving the CUDA context usable.
 * Determinism.  Indices, slots and drop masks are exact; no floating-point
 *   atomics are used, so two calls on the same inputs give identical bits.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,         /* invalid argument (sizes, null or misaligned pointer) */
  MOE_ERR_UNSUPPORTED = 2, /* valid but not handled by the library */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  MOE_ERR_NONFINITE = 4,   /* device: a logit or an output was Inf/NaN */
  MOE_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_BOUNDS = 6       /* device: an index fell outside its array */
} moe_status;

typedef enum {
  MOE_GATE_TOPK_SOFTMAX = 0, /* G = Softmax(KeepTopK(H, k)) ("Outrageously Large", Eq. 5) */
  MOE_GATE_SWITCH = 1        /* k = 1; p = Softmax(H); gate = p[argmax] ("Switch", step 2) */
} moe_gate_mode;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef struct {
  int32_t T;               /* tokens, >= 1 */
  int32_t d;               /* token width, >= 1 */
  int32_t E;               /* experts, >= 1 */
  int32_t d_ff;            /* expert hidden width, >= 1 */
  int32_t k;               /* experts per token, 1 <= k <= E (1 for MOE_GATE_SWITCH) */
  float capacity_factor;   /* > 0 */
  int32_t min_capacity;    /* >= 1; the Switch page's reduced minimum is 1 */
  int32_t gate_mode;       /* moe_gate_mode */
  int32_t act_dtype;       /* moe_dtype */
} moe_config;

/* Human-readable name of a moe_status value (static string). */
const char *moe_status_string(int status);

/* Expert capacity C = max(min_capacity, min(T, floor(k*T*capacity_factor/E)))
 * ("Switch Transformer", step 3, with the top-k factor k). Host only. */
int moe_capacity(const moe_config *cfg, int32_t *C);

/* Bytes of workspace every entry point below needs for `cfg`. Host only. */
int moe_workspace_size(const moe_config *cfg, size_t *bytes);

/*
 * Stages 1-2: router and gate ("Outrageously Large", section 3.4, Eqs. 4-5;
 * "Switch Transformer", steps 1-2).
 *   c = x Wg + logit_bias; sigma = Softplus(x Wnoise); H = c + noise * sigma
 *   TOPK:   expert_idx[t,:] = the k largest H (descending; lower index on
 *           ties), gate[t,:] = softmax of those k values.
 *   SWITCH: expert_idx[t,0] = argmax H (first on ties), gate[t,0] = Softmax(H)
 *           at that expert (not renormalised).
 * x [T,d] (act_dtype); Wg, Wnoise [d,E] fp32; noise [T,E] fp32 (the
 * StandardNormal() draws, supplied so runs are deterministic); logit_bias [E]
 * fp32. Wnoise and noise are both NULL (no noise: sigma = 0, H = c) or both
 * given; logit_bias may be NULL. Outputs: expert_idx [T,k] int32, gate [T,k]
 * fp32, thr [T,2] fp32 = (k-th largest H, (k+1)-th largest H or -inf when
 * k == E). Also leaves in `ws` what moe_aux_loss() reads.
 */
int moe_gate(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
             const float *noise, const float *logit_bias, int32_t *expert_idx, float *gate,
             float *thr, void *ws, moe_stream_t stream);

/*
 * Stage 3 and dispatch ("Switch Transformer", steps 3-5): positions are
 * exclusive counts in token order, pos[t,j] = number of assignments (t',j')
 * before (t,j) in token-major order with the same expert; keep = pos < C.
 * Inputs: expert_idx [T,k], gate [T,k] from moe_gate, x [T,d].
 * Outputs: pos [T,k] int32; keep [T,k] uint8; expert_count [E] int32 = choices
 * per expert before capacity; expert_offset [E+1] int32 = exclusive sum of
 * min(expert_count, C); rows expert_offset[e] .. expert_offset[e+1]-1 of
 * xbuf [T*k, d] hold expert e's accepted tokens in token order;
 * row_token [T*k] int32 = t*k + j of each row; row_gate [T*k] fp32 = its gate.
 * Rows past expert_offset[E] are not written.
 */
int moe_dispatch(const moe_config *cfg, const int32_t *expert_idx, const float *gate,
                 const void *x, int32_t *pos, uint8_t *keep, int32_t *expert_count,
                 int32_t *expert_offset, void *xbuf, int32_t *row_token, float *row_gate,
                 void *ws, moe_stream_t stream);

/*
 * Stage 4, experts ("Switch Transformer", step 6; "Outrageously Large", the
 * expert networks E_i): for each expert e and each of its rows r,
 *   hbuf[r] = ReLU(xbuf[r] W1[e] + b1[e])             (act_dtype)
 *   zbuf[r] = row_gate[r] * (hbuf[r] W2[e] + b2[e])   (fp32)
 * W1 [E,d,d_ff], b1 [E,d_ff] (NULL = 0), W2 [E,d_ff,d], b2 [E,d] (NULL = 0);
 * expert_offset and row_gate as written by moe_dispatch; hbuf [T*k,d_ff],
 * zbuf [T*k,d]. bf16 runs on the tensor cores with fp32 accumulation.
 */
int moe_expert_ffn(const moe_config *cfg, const void *xbuf, const int32_t *expert_offset,
                   const float *row_gate, const void *W1, const void *b1, const void *W2,
                   const void *b2, void *hbuf, float *zbuf, void *ws, moe_stream_t stream);

/*
 * Stage 4, combine ("Switch Transformer", step 7; "Outrageously Large", the
 * output y = sum_i G(x)_i E_i(x)): y[t] = x[t] + sum over j with keep[t,j] of
 * zbuf[expert_offset[expert_idx[t,j]] + pos[t,j]], summed in j order in fp32
 * and rounded once to act_dtype. A token with no accepted choice gets y = x.
 */
int moe_combine(const moe_config *cfg, const void *x, const float *zbuf, const int32_t *pos,
                const uint8_t *keep, const int32_t *expert_idx, const int32_t *expert_offset,
                void *y, void *ws, moe_stream_t stream);

/*
 * Stage 5, balancing losses, from what moe_gate() left in `ws` (all before
 * capacity): importance[e] = sum_t G(x_t)_e ("Outrageously Large", Eq. 6);
 * load[e] = sum_t P(x_t,e) with P(x,e) = Phi((c_e - kth_excluding(H,k,e)) /
 * sigma_e) (Eqs. 8-10; the 0/1 indicator of selection when there is no noise);
 * out3[0] = CV(importance)^2, out3[1] = CV(load)^2 (population std, Eq. 7;
 * the caller applies its own weights w_importance, w_load); out3[2] =
 * 0.01 * E * sum_e f_e * Pbar_e with f_e the fraction of tokens whose first
 * choice is e and Pbar_e the mean of Softmax(H)_e ("Switch Transformer",
 * step 8). out3 [3] fp32; importance, load [E] fp32, each may be NULL.
 */
int moe_aux_loss(const moe_config *cfg, const void *ws, float *out3, float *importance,
                 float *load, moe_stream_t stream);

/*
 * Stages 1-5 in one call: moe_gate, moe_dispatch, moe_expert_ffn, moe_combine
 * and moe_aux_loss, with the intermediate buffers inside `ws`. y [T,d]
 * (act_dtype), aux_out3 [3] fp32 (may be NULL to skip stage 5), and optionally
 * (each may be NULL) expert_idx [T,k], gate [T,k], pos [T,k], keep [T,k].
 */
int moe_forward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                const float *noise, const float *logit_bias, const void *W1, const void *b1,
                const void *W2, const void *b2, void *y, float *aux_out3, int32_t *expert_idx,
                float *gate, int32_t *pos, uint8_t *keep, void *ws, moe_stream_t stream);

/*
 * Allocation-free variant of moe_dispatch. The pages have no counterpart: it
 * exists for callers that cannot call cudaMalloc where they route tokens --
 * for example an inference engine's plugin whose enqueue callback must not
 * allocate, or a runtime that fixes its device memory at start-up -- and so
 * cannot provide the workspace moe_dispatch needs.
 *
 * Same arguments, computation and outputs as moe_dispatch, minus `ws`. Its
 * scratch is a static device array of MOE_NOALLOC_SCRATCH_BYTES inside
 * libmoe.so (every GPU that loads the library holds it until the process
 * exits). The call needs 256 + 2 * ceil(T*k/512) * E * 4 + (E+1) * 4 bytes of
 * it (each term rounded up to 256) and returns MOE_ERR_UNSUPPORTED, enqueuing
 * nothing, if that is more. It allocates nothing and frees nothing.
 *
 * The first call on each device (and again after cudaDeviceReset, or in
 * another context) looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. All calls share the one array: calls whose work
 * overlaps on the GPU (other streams, other host threads) race and must be
 * serialised by the caller. An expert index outside [0, E) yields pos = -1
 * and keep = 0 for that assignment and is recorded (MOE_ERR_BOUNDS, detail =
 * the flat index t*k + j) in a status word inside the same array, which
 * moe_noalloc_last_status() reads; each call clears it when it starts.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
int moe_dispatch_noalloc(const moe_config *cfg, const int32_t *expert_idx, const float *gate,
                         const void *x, int32_t *pos, uint8_t *keep, int32_t *expert_count,
                         int32_t *expert_offset, void *xbuf, int32_t *row_token,
                         float *row_gate, moe_stream_t stream);

/*
 * The device-side status of the last moe_dispatch_noalloc on the current
 * device, its counterpart of moe_last_device_status (the pages have none
 * either): synchronises `stream` (the stream that call used), returns
 * MOE_OK or the first error recorded since the call started (MOE_ERR_BOUNDS
 * for an expert index outside [0, E)), writes its detail word to *detail if
 * non-NULL, and clears it. It copies 32 bytes device-to-host into a local
 * variable and allocates nothing.
 */
int moe_noalloc_last_status(moe_stream_t stream, int64_t *detail);

/*
 * Expert parallelism ("Outrageously Large Neural Networks", Distributed
 * Training: Solving the Shrinking Batch Problem: the experts are spread over
 * the devices, each device gates its own share of the batch, and every token
 * is sent to the device holding its expert and its output sent back, so each
 * expert sees the tokens of all devices). The layer's batch is the
 * concatenation, in rank order, of the W ranks' batches; capacity and the
 * token-order slots are those of moe_forward over that whole batch. A rank
 * calls, on its own T tokens (cfg->T), with E the number of all experts:
 *   1. moe_gate (or the gate of moe_forward's stages) on its tokens;
 *   2. moe_expert_counts: its choices per expert before capacity, and
 *      gathers the ranks' counts into counts_all [W, E] (a collective);
 *   3. moe_dispatch_ranked with the whole batch's capacity C: its assignment
 *      to expert e gets the slot after every earlier rank's, so it is kept
 *      iff base_e + pos < C with base_e the earlier ranks' count; the kept
 *      rows are packed per expert as moe_dispatch packs them, so the rows of
 *      the experts one rank holds are one contiguous range (an all-to-all
 *      sends them there and the outputs back);
 *   4. moe_expert_ffn on the rows it received, moe_combine on its own tokens
 *      with the outputs it got back;
 *   5. moe_aux_totals, a sum over the ranks (a collective) and
 *      moe_aux_from_totals for the balancing losses of the whole batch.
 * The module sparsely_gated_mixture_gb300.expert_parallel drives these.
 */

/*
 * Choices per expert before capacity (counts [E] int32) of this rank's
 * selection expert_idx [T,k] (an index outside [0, E) is a device-side
 * MOE_ERR_BOUNDS and not counted).
 */
int moe_expert_counts(const moe_config *cfg, const int32_t *expert_idx, int32_t *expert_count,
                      void *ws, moe_stream_t stream);

/*
 * moe_dispatch for rank `rank` of n_ranks: counts_all [n_ranks, E] int32
 * (device) holds every rank's moe_expert_counts, capacity the whole batch's
 * C (>= 1). pos[t,j] = this rank's exclusive count of earlier assignments to
 * the same expert (its local position; the slot in the whole batch adds
 * base_e); keep = pos < max(0, capacity - base_e). expert_count, expert_offset,
 * xbuf, row_token and row_gate as in moe_dispatch (kept rows only).
 */
int moe_dispatch_ranked(const moe_config *cfg, int32_t capacity, const int32_t *counts_all,
                        int32_t n_ranks, int32_t rank, const int32_t *expert_idx,
                        const float *gate, const void *x, int32_t *pos, uint8_t *keep,
                        int32_t *expert_count, int32_t *expert_offset, void *xbuf,
                        int32_t *row_token, float *row_gate, void *ws, moe_stream_t stream);

/*
 * The balancing sums of the last moe_gate (or moe_forward with aux_out3) on
 * `ws` over this rank's tokens: totals [4, E] fp32 = importance (sum of gates,
 * Eq. 6), load (sum of P(x, e), Eq. 10), the number of tokens whose first
 * choice is e, and the sum of Softmax(H)_e. Sums, not averages, so that
 * ranks' totals add up to the whole batch's.
 */
int moe_aux_totals(const moe_config *cfg, void *ws, float *totals, moe_stream_t stream);

/*
 * The losses of moe_aux_loss (out3 [3] fp32: CV(importance)^2, CV(load)^2,
 * the Switch loss) from totals [4, E] fp32 summed over all ranks, for a batch
 * of T_total tokens (f and Pbar are averaged over it). ws: this rank's
 * workspace (its status word and scratch).
 */
int moe_aux_from_totals(const moe_config *cfg, int64_t T_total, const float *totals,
                        float *out3, void *ws, moe_stream_t stream);

/*
 * Hierarchical layer ("Outrageously Large Neural Networks", Hierarchical
 * Mixture-of-Experts): a groups of b experts, flat expert i*b + j. A primary
 * noisy top-k gate over the a groups picks k_primary groups; in each picked
 * group i a secondary noisy top-k gate over its b experts picks
 * k_secondary; the output is y_H = x + sum_i sum_j G_primary(x)_i G_i(x)_j
 * E_ij(x), with capacity and token-order slots over the a*b experts exactly as
 * in moe_forward (k = k_primary * k_secondary choices per token, in primary
 * pick order, then secondary pick order).
 */
typedef struct {
  int32_t T;               /* tokens, >= 1 */
  int32_t d;               /* token width, >= 1 */
  int32_t a;               /* groups, >= 1 */
  int32_t b;               /* experts per group, >= 1; a * b <= 1024 */
  int32_t k_primary;       /* groups per token, 1 <= k_primary <= min(a, 8) */
  int32_t k_secondary;     /* experts per picked group, 1 <= k_secondary <= min(b, 8) */
  int32_t d_ff;            /* expert hidden width, >= 1 */
  float capacity_factor;   /* > 0; C = max(min_capacity, min(T, floor(k*T*cf/(a*b)))) */
  int32_t min_capacity;    /* >= 1 */
  int32_t act_dtype;       /* moe_dtype */
} moe_hier_config;

/* Bytes of workspace moe_forward_hier needs for `cfg`. Host only. */
int moe_hier_workspace_size(const moe_hier_config *cfg, size_t *bytes);

/*
 * The hierarchical layer in one call. Primary gate: Wp, Wp_noise [d,a] fp32,
 * noise_p [T,a] fp32; secondary gates: Ws, Ws_noise [d,a*b] fp32 (group i owns
 * columns i*b .. i*b+b-1), noise_s [T,a*b] fp32; each noise pair is both given
 * or both NULL (that gate without noise). Experts: W1 [a*b,d,d_ff], b1
 * [a*b,d_ff], W2 [a*b,d_ff,d], b2 [a*b,d] as in moe_forward (biases may be
 * NULL). Outputs: y [T,d] (act_dtype); aux_out2 [2] fp32 or NULL =
 * [CV(Importance_H)^2, CV(Load_H)^2] with Importance_H[i*b+j] = sum_x
 * G_primary(x)_i G_i(x)_j and Load_H[i*b+j] = Load_primary(X)_i *
 * Load_i(X^(i))_j / |X^(i)| (X^(i): the tokens whose primary gate picked
 * group i; Load_H is 0 for a group no token picked); optionally (each may be
 * NULL) expert_idx [T,k] (flat i*b + j), gate [T,k] (the products), pos and
 * keep [T,k]. Device-side errors go to the status word at the start of `ws`
 * (moe_last_device_status reads it); the call clears it first.
 */
int moe_forward_hier(const moe_hier_config *cfg, const void *x, const float *Wp,
                     const float *Wp_noise, const float *noise_p, const float *Ws,
                     const float *Ws_noise, const float *noise_s, const void *W1, const void *b1,
                     const void *W2, const void *b2, void *y, float *aux_out2,
                     int32_t *expert_idx, float *gate, int32_t *pos, uint8_t *keep, void *ws,
                     moe_stream_t stream);

/*
 * Strictly balanced gating ("Outrageously Large Neural Networks", Strictly
 * Balanced Gating (Batchwise Mask); the mask form of the gate). P =
 * Softmax(x Wg + logit_bias) over all E experts (dense, fp32, no noise); each
 * expert takes the m = max(1, min(T, floor(k*T/E))) tokens with the largest P
 * for it (lower token index first on ties), so every expert processes exactly
 * m rows and there is no capacity; a token's gate on a picked expert is P
 * renormalised over its own picks; y = x + sum over the picks of gate *
 * E_i(x) (a token no expert took keeps only the residual). Uses T, d, E, d_ff,
 * k and act_dtype of cfg (capacity_factor, min_capacity and gate_mode are not
 * used). thresholds [E] fp32 or NULL: the per-expert T_i of the threshold mask
 * P > T_i; loss_out [1] fp32 or NULL (needs thresholds) = L_batchwise = sum_t
 * sum_i (1[P > T_i] - M_batchwise[t,i]) * (P[t,i] - T_i). mask_out [T][ceil(E/32)]
 * uint32 or NULL: bit (i % 32) of word i / 32 of token t's row is
 * M_batchwise[t,i]. The status word at the start of `ws` is cleared first.
 */
int moe_balanced_workspace_size(const moe_config *cfg, size_t *bytes);
int moe_forward_balanced(const moe_config *cfg, const void *x, const float *Wg,
                         const float *logit_bias, const float *thresholds, const void *W1,
                         const void *b1, const void *W2, const void *b2, void *y,
                         float *loss_out, uint32_t *mask_out, void *ws, moe_stream_t stream);

/*
 * Threshold mask, the inference-time gate of strictly balanced gating
 * ("Outrageously Large Neural Networks", Strictly Balanced Gating: at
 * inference examples arrive one at a time, so the batchwise mask is replaced
 * by per-expert thresholds, M_threshold(x, T)_i = 1 iff x_i > T_i). With P =
 * Softmax(x Wg + logit_bias) over all E experts (dense, fp32, no noise), token
 * t picks every expert i with P[t,i] > thresholds[i] (strictly greater: P
 * equal to T_i is not taken); a pick's gate is P renormalised over the
 * token's own picks; y = x + sum over the picks, in expert order, of gate *
 * E_i(x) (fp32 sum, rounded once). A token that passes no threshold keeps
 * only the residual. No capacity: every pick is computed. Uses T, d, E, d_ff,
 * act_dtype and k of cfg, where k (1..min(E, 16)) is the caller's bound on
 * any token's picks, which sizes the workspace (a token's picks are fewer
 * than 1 / min_i T_i, so k >= that bound always holds); a token with more
 * than k picks records MOE_ERR_BOUNDS (detail = the token) and only its
 * first k picks (in expert order) reach y. capacity_factor, min_capacity and
 * gate_mode are not used. thresholds [E] fp32. Optional outputs (NULL to
 * skip): expert_idx [T,k] int32, a token's picks in expert order then E;
 * gate [T,k] fp32, their gates then 0; mask_out [T][ceil(E/32)] uint32, bit
 * (i % 32) of word i / 32 set for every pick. The status word at the start
 * of `ws` (moe_threshold_workspace_size bytes) is cleared first.
 */
int moe_threshold_workspace_size(const moe_config *cfg, size_t *bytes);
int moe_forward_threshold(const moe_config *cfg, const void *x, const float *Wg,
                          const float *logit_bias, const float *thresholds, const void *W1,
                          const void *b1, const void *W2, const void *b2, void *y,
                          int32_t *expert_idx, float *gate, uint32_t *mask_out, void *ws,
                          moe_stream_t stream);

/*
 * Backward of the flat layer ("Outrageously Large Neural Networks", section
 * 3.4, "Training the gating network": plain back-propagation, gradients reach
 * W_g through the selected softmax gates and W_noise through the smooth load
 * estimator; "Switch Transformer", step 8: f carries no gradient, P and the
 * selected gate do). The gradients of
 *   L = sum_t <dy_t, y_t> + w_importance * CV(Importance)^2
 *       + w_load * CV(Load)^2 + w_aux * 0.01 * E * sum_e f_e Pbar_e
 * with the forward's discrete choices held fixed (the top-k set, capacity
 * drops, the ReLU pattern): through the residual, the kept experts (dgrad and
 * wgrad of both layers), the kept top-k softmax (or the full softmax at the
 * Switch argmax), Importance (every selected choice, before capacity), the
 * load estimator P = Phi((c - thr) / sigma) (into c, sigma and the expert
 * whose noisy logit is thr; none without noise or when k = E), the Switch
 * loss's Pbar, sigma = Softplus(x W_noise) and c = x W_g + b.
 *
 * Precondition: `ws` holds the state the last moe_forward left in it for the
 * same cfg and inputs (x, Wg, Wnoise, noise, logit_bias, W1, b1, W2, b2), and
 * expert_idx, gate, pos, keep are the pointers given to that call (NULL where
 * it got NULL); that call had aux_out3 non-NULL if any loss weight here is
 * nonzero (the backward reads its balancing totals). The call may overwrite
 * `ws` rows past the forward's last expert row; it leaves the forward's other
 * results unchanged, so it may be repeated with another dy.
 * Every configuration moe_forward takes: bf16 layers with d and d_ff
 * multiples of 64 run the expert GEMMs on the tensor cores, the others
 * (fp32 layers, other widths) on the CUDA cores with fp32 row buffers.
 * Inputs: dy [T,d] act_dtype. Outputs (fp32 unless stated): dx [T,d]
 * act_dtype; dWg
 * [d,E]; dWnoise [d,E] (required iff Wnoise is given); dlogit_bias [E] (may
 * be NULL); dW1 [E,d,d_ff]; db1 [E,d_ff] (may be NULL); dW2 [E,d_ff,d]; db2
 * [E,d] (may be NULL); dgate [T,k] (may be NULL) = dL/dgate of each selected
 * gate value (<dy_t, U_e(x_t)> for a kept choice plus the Importance term).
 * bws is the backward's own workspace, moe_backward_workspace_size bytes,
 * 256-byte aligned. Device-side errors (a non-finite gradient, a bounded wait
 * that ran out) go to the status word of `ws`.
 */
int moe_backward_workspace_size(const moe_config *cfg, size_t *bytes);
int moe_backward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                 const float *noise, const void *W1, const void *W2, const void *b2,
                 const int32_t *expert_idx, const float *gate, const int32_t *pos,
                 const uint8_t *keep, const void *dy, float w_importance, float w_load,
                 float w_aux, void *dx, float *dWg, float *dWnoise, float *dlogit_bias,
                 float *dW1, float *db1, float *dW2, float *db2, float *dgate, void *ws,
                 void *bws, moe_stream_t stream);

/*
 * The gate's share of the backward, from given gate gradients: dgate [T,k]
 * fp32 = dL/dgate of each selected gate value (Importance term included) for
 * the selection expert_idx / gate (NULL: the copies in `ws`) of the last
 * moe_gate or moe_forward on `ws`; the load and Switch terms are added with
 * weights w_load, w_aux (these need the balancing totals of moe_aux_loss or
 * of moe_forward with aux_out3). Outputs: dWg [d,E], dWnoise [d,E] (iff
 * Wnoise), dlogit_bias [E] (may be NULL), dx_gate [T,d] (may be NULL): the
 * router's share of dx, all fp32. x [T,d] act_dtype; bws as for moe_backward.
 */
int moe_gate_backward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                      const float *noise, const int32_t *expert_idx, const float *gate,
                      const float *dgate, float w_load, float w_aux, float *dWg, float *dWnoise,
                      float *dlogit_bias, float *dx_gate, void *ws, void *bws,
                      moe_stream_t stream);

/*
 * Diagnostic: out[i] = Phi(u[i]) for i < n, the standard normal CDF exactly as
 * the balancing kernels evaluate it inside the load estimator P(x, i) =
 * Phi((c_i - kth_excluding(H, k, i)) / sigma_i) ("Outrageously Large", Eq. 9),
 * so its accuracy can be checked on any grid. u, out [n] fp32 device arrays
 * (n = 0: nothing is enqueued). The library's Phi is erfc(-u / sqrt 2) / 2
 * with erfc from the Chebyshev fit of Numerical Recipes (Press et al., 2nd
 * ed., section 6.2, "erfcc"), evaluated in fp32.
 */
int moe_eval_normal_cdf(const float *u, float *out, int64_t n, moe_stream_t stream);

/*
 * Synchronises `stream`, returns the first device-side error recorded in `ws`
 * since it was last cleared (MOE_OK if none), writes its detail word (e.g. the
 * offending flat index) to *detail if non-NULL, and clears it.
 */
int moe_last_device_status(void *ws, moe_stream_t stream, int64_t *detail);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
