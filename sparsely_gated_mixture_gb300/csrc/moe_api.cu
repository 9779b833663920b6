// C ABI of libmoe.so (declared in include/moe.h): argument checks, the
// workspace layout and the order of launches. No computation happens here;
// every stage runs in the kernels of the other translation units.
#include "moe_internal.cuh"

#include <mutex>

#include <math.h>
#include <stdlib.h>
#include <string.h>

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void *current_context() {
  using GetCurrent = int (*)(void **);  // CUresult cuCtxGetCurrent(CUcontext *)
  static const GetCurrent fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<GetCurrent>(ptr);
    cudaGetLastError();
    return static_cast<GetCurrent>(nullptr);
  }();
  void *ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

bool pdl_enabled(int cls) {
  static const unsigned mask = [] {
    const char *v = getenv("MOE_PDL_MASK");
    return v && *v ? (unsigned)strtoul(v, nullptr, 0) : ~0u;
  }();
  return (mask >> cls) & 1u;
}

WsLayout ws_layout(const moe_config &cfg) {
  WsLayout L{};
  const size_t T = cfg.T, E = cfg.E, k = cfg.k, d = cfg.d, dff = cfg.d_ff;
  const size_t A = T * k;
  const size_t eb = elem_bytes(cfg.act_dtype);
  L.n_chunks = (int)((A + kSlotChunk - 1) / kSlotChunk);
  L.n_aux_blocks = aux_rows((int)T, (int)cfg.E);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(sizeof(DeviceStatus));
  L.c = take(T * E * 4);
  L.sigma = take(T * E * 4);
  L.H = take(T * E * 4);
  L.rowstat = take(T * 2 * 4);
  L.bsplit = take(router_tc_split_bytes(cfg));
  L.hist = take((size_t)L.n_chunks * E * 4);
  L.chunk_base = take((size_t)L.n_chunks * E * 4);
  L.count = take(E * 4);
  L.offset = take((E + 1) * 4);
  L.mtiles = take((E + 1) * 4);
  L.ecap = take(E * 4);
  L.out3s = take(16);
  L.partials = take((size_t)L.n_aux_blocks * 4 * E * 4);
  L.aux_vec = take(4 * E * 8);
  L.idx = take(A * 4);
  L.gate = take(A * 4);
  L.thr = take(T * 2 * 4);
  L.pos = take(A * 4);
  L.keep = take(A);
  L.row_token = take(A * 4);
  L.row_gate = take(A * 4);
  L.xbuf = take(A * d * eb);
  L.hbuf = take(A * dff * eb);
  L.zbuf = take(A * d * 4);
  L.total = off;
  return L;
}

static int host_capacity(const moe_config &c) {
  double raw = floor((double)c.k * (double)c.T * (double)c.capacity_factor / (double)c.E);
  long v = (long)raw;
  if (v > c.T) v = c.T;
  if (v < c.min_capacity) v = c.min_capacity;
  return (int)v;
}

static int check_cfg(const moe_config *c) {
  if (!c) return MOE_ERR_ARG;
  if (c->T < 1 || c->d < 1 || c->E < 1 || c->d_ff < 1 || c->k < 1 || c->k > c->E) return MOE_ERR_ARG;
  if (!(c->capacity_factor > 0.f) || !isfinite(c->capacity_factor)) return MOE_ERR_ARG;
  if (c->min_capacity < 1) return MOE_ERR_ARG;
  if (c->gate_mode != MOE_GATE_TOPK_SOFTMAX && c->gate_mode != MOE_GATE_SWITCH) return MOE_ERR_ARG;
  if (c->gate_mode == MOE_GATE_SWITCH && c->k != 1) return MOE_ERR_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_ARG;
  if ((long long)c->T * c->k > 0x7fffffffLL || (long long)c->T * c->E > 0x7fffffffLL)
    return MOE_ERR_UNSUPPORTED;
  if (c->E > 1024 || c->k > 16) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Required pointers must be non-null; every given pointer 16-byte aligned.
#define MOE_REQ(p)                                      \
  do {                                                  \
    if (!(p) || !aligned((p), 16)) return MOE_ERR_ARG;  \
  } while (0)
#define MOE_OPT(p)                                      \
  do {                                                  \
    if ((p) && !aligned((p), 16)) return MOE_ERR_ARG;   \
  } while (0)
#define MOE_CUDA(call)                                  \
  do {                                                  \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA;     \
  } while (0)

static int gate_impl(const moe_config &c, const void *x, const float *Wg, const float *Wn,
                     const float *noise, const float *bias, int32_t *idx, float *gate, float *thr,
                     void *ws, bool partials, cudaStream_t s) {
  const WsLayout L = ws_layout(c);
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  float *cc = ws_at<float>(ws, L.c), *sg = ws_at<float>(ws, L.sigma), *H = ws_at<float>(ws, L.H);
  float *rs = ws_at<float>(ws, L.rowstat);
  float *part = ws_at<float>(ws, L.partials);  // launch_router clears the status word first
  const RouterSelect sel{idx, gate, thr, rs, partials ? part : nullptr};
  bool selected = false;
  MOE_CUDA(launch_router(c, x, Wg, Wn, noise, bias, cc, sg, H, ws_at<char>(ws, L.bsplit), st, s,
                         &sel, &selected));
  if (selected) return MOE_OK;  // the router's epilogue selected (and summed) itself
  if (partials && c.E <= 256) {
    MOE_CUDA(launch_select_aux(c, Wn != nullptr, cc, sg, H, idx, gate, thr, rs,
                               ws_at<float>(ws, L.partials), L.n_aux_blocks, s));
  } else {
    MOE_CUDA(launch_select(c, H, idx, gate, thr, rs, st, s));
    if (partials)
      MOE_CUDA(launch_aux_partials(c, Wn != nullptr, cc, sg, H, rs, idx, gate, thr,
                                   ws_at<float>(ws, L.partials), L.n_aux_blocks, s));
  }
  return MOE_OK;
}

// Inside moe_forward the expert outputs Z stay in bf16 when the layer runs on
// the tensor cores and combines 16 bytes at a time (the stage calls keep the
// fp32 zbuf of their contract): half the Z traffic, one more bf16 rounding per
// expert term before the fp32 combine.
static bool forward_z_bf16(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && ffn_tc_supported(c) && c.d % 8 == 0 && c.k <= 4;
}

static int ffn_impl(const moe_config &c, const void *xbuf, const int32_t *offset,
                    const int32_t *mtiles, const float *row_gate, const void *W1, const void *b1,
                    const void *W2, const void *b2, void *hbuf, void *zbuf, bool z_bf16,
                    DeviceStatus *st, cudaStream_t s) {
  const int C = host_capacity(c);
  if (c.act_dtype == MOE_BF16 && ffn_tc_supported(c)) {
    MOE_CUDA(launch_ffn_tc(c, C, xbuf, offset, mtiles, row_gate, W1, b1, W2, b2, hbuf, zbuf,
                           z_bf16, st, s));
  } else {
    if (z_bf16) return MOE_ERR_UNSUPPORTED;
    MOE_CUDA(launch_ffn_simt(c, C, xbuf, offset, row_gate, W1, b1, W2, b2, hbuf,
                             static_cast<float *>(zbuf), st, s));
  }
  return MOE_OK;
}

// Stages 3-4 of the forward from a selection: slots and dispatch, the expert
// GEMMs, combine (the intermediate buffers in `ws` laid out by L).
static int expert_path(const moe_config &c, const WsLayout &L, void *ws, const void *x,
                       const int32_t *idx, const float *g, int32_t *ps, uint8_t *kp,
                       const void *W1, const void *b1, const void *W2, const void *b2, void *y,
                       DeviceStatus *st, cudaStream_t s, bool allow_none = false) {
  int32_t *offset = ws_at<int32_t>(ws, L.offset);
  int32_t *row_token = ws_at<int32_t>(ws, L.row_token);
  float *row_gate = ws_at<float>(ws, L.row_gate);
  void *xbuf = ws_at<char>(ws, L.xbuf), *hbuf = ws_at<char>(ws, L.hbuf);
  float *zbuf = ws_at<float>(ws, L.zbuf);
  MOE_CUDA(launch_slots(c, host_capacity(c), idx, g, ws_at<int32_t>(ws, L.hist),
                        ws_at<int32_t>(ws, L.chunk_base), ws_at<int32_t>(ws, L.count), offset,
                        ws_at<int32_t>(ws, L.mtiles), ps, kp, row_token, row_gate, L.n_chunks, st,
                        s, allow_none));
  MOE_CUDA(launch_gather(c, x, offset, row_token, xbuf, st, s));
  const bool z_bf16 = forward_z_bf16(c);
  const int r = ffn_impl(c, xbuf, offset, ws_at<int32_t>(ws, L.mtiles), row_gate, W1, b1, W2,
                         b2, hbuf, zbuf, z_bf16, st, s);
  if (r != MOE_OK) return r;
  MOE_CUDA(launch_combine(c, x, zbuf, z_bf16, ps, kp, idx, offset, y, st, s));
  return MOE_OK;
}

// ----------------------------------------------------------------------------- hierarchical layer
// The secondary side is a flat layer over the a*b experts with k = kp*ks; the
// primary gate is a flat gate over the a groups. The workspace holds the
// flat layout of the former (status word first), then the latter's, then the
// hierarchical partial rows and the finalizes' scratch outputs.
static moe_config hier_secondary(const moe_hier_config &h) {
  moe_config c{};
  c.T = h.T;
  c.d = h.d;
  c.E = h.a * h.b;
  c.d_ff = h.d_ff;
  c.k = h.k_primary * h.k_secondary;
  c.capacity_factor = h.capacity_factor;
  c.min_capacity = h.min_capacity;
  c.gate_mode = MOE_GATE_TOPK_SOFTMAX;
  c.act_dtype = h.act_dtype;
  return c;
}

static moe_config hier_primary(const moe_hier_config &h) {
  moe_config c = hier_secondary(h);
  c.E = h.a;
  c.k = h.k_primary;
  return c;
}

struct HierLayout {
  WsLayout Ls, Lp;
  size_t off_p, parts, scratch, gc, gs, gH, gpoff, total;
  int rows;
};

static HierLayout hier_layout(const moe_hier_config &h) {
  HierLayout H;
  H.Ls = ws_layout(hier_secondary(h));
  H.Lp = ws_layout(hier_primary(h));
  H.rows = hier_rows(h.T, h.k_primary, h.b);
  size_t off = align_up(H.Ls.total, 256);
  H.off_p = off;
  off = align_up(off + H.Lp.total, 256);
  H.parts = off;
  off = align_up(off + (size_t)H.rows * 4 * (size_t)h.a * h.b * 4, 256);
  H.scratch = off;  // two finalize outputs of 3 floats
  off = align_up(off + 64, 256);
  // The grouped router's compact outputs: [T*kp + a*128 padded rows][b].
  const size_t grows = (size_t)h.T * h.k_primary + (size_t)h.a * 128;
  H.gc = off;
  off = align_up(off + grows * h.b * 4, 256);
  H.gs = off;
  off = align_up(off + grows * h.b * 4, 256);
  H.gH = off;
  off = align_up(off + grows * h.b * 4, 256);
  H.gpoff = off;
  H.total = align_up(off + (size_t)(h.a + 1) * 4, 256);
  return H;
}

static int check_hier(const moe_hier_config *h) {
  if (!h) return MOE_ERR_ARG;
  if (h->a < 1 || h->b < 1 || h->k_primary < 1 || h->k_secondary < 1 ||
      h->k_primary > h->a || h->k_secondary > h->b)
    return MOE_ERR_ARG;
  if (h->k_primary > 8 || h->k_secondary > 8 || (long long)h->a * h->b > 1024)
    return MOE_ERR_UNSUPPORTED;
  const moe_config cs = hier_secondary(*h), cp = hier_primary(*h);
  const int r = check_cfg(&cs);
  return r != MOE_OK ? r : check_cfg(&cp);
}

// ----------------------------------------------------------------------------- balanced gating
struct BalLayout {
  size_t status, c, sigma, H, bsplit, PT, mask, row_token, row_gate, offset, trows, npick, xbuf,
      hbuf, zbuf, loss, total;
  int m;
};

static BalLayout bal_layout(const moe_config &cfg) {
  BalLayout L{};
  const size_t T = cfg.T, E = cfg.E, d = cfg.d, dff = cfg.d_ff;
  const size_t eb = elem_bytes(cfg.act_dtype);
  L.m = balanced_m(cfg);
  const size_t R = E * (size_t)L.m, W = (E + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(sizeof(DeviceStatus));
  L.c = take(T * E * 4);
  L.sigma = take(T * E * 4);
  L.H = take(T * E * 4);
  L.bsplit = take(router_tc_split_bytes(cfg));
  L.PT = take(E * T * 4);
  L.mask = take(T * W * 4);
  L.row_token = take(R * 4);
  L.row_gate = take(R * 4);
  L.offset = take((E + 1) * 4);
  L.trows = take(T * kBalKeepRows * 4);
  L.npick = take(T * 4);
  L.xbuf = take(R * d * eb);
  L.hbuf = take(R * dff * eb);
  L.zbuf = take(R * d * 4);
  L.loss = take(E * 8);
  L.total = off;
  return L;
}

// ----------------------------------------------------------------------------- threshold mask
// The inference-time gate of strictly balanced gating runs the flat expert
// path with cfg.k choice slots per token (the caller's bound on a token's
// picks) and no capacity: C = T, so every pick keeps its row.
static moe_config thr_layer(const moe_config &c) {
  moe_config r = c;
  r.capacity_factor = (float)c.E;  // floor(k T E / E) >= T: the capacity is T
  r.min_capacity = 1;
  r.gate_mode = MOE_GATE_TOPK_SOFTMAX;
  return r;
}

// ----------------------------------------------------------------------------- backward
struct BwdLayout {
  size_t poff, dY, dU, dP, dX, dgpart, dg, coef, dc, dz, dxr, rpart, bpart, cpart, total;
  long long P_max;  // padded rows: T*k + 64*E bounds sum_e max(64, roundup(rows_e, 64))
  int n_blocks2, chunks;
};

// The expert backward runs on the tensor cores for bf16 layers whose widths
// are multiples of 64, else on the CUDA cores (fp32 row buffers).
static bool bwd_tc_shape(const moe_config &c) {
  return c.act_dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0;
}

static BwdLayout bwd_layout(const moe_config &cfg) {
  BwdLayout L{};
  const size_t T = cfg.T, E = cfg.E, k = cfg.k, d = cfg.d, dff = cfg.d_ff;
  const bool tc = bwd_tc_shape(cfg);
  const size_t rb = tc ? 2 : 4;  // bytes per element of the dY, g*dY and dpre rows
  L.P_max = (long long)T * k + (long long)kBwdRowPad * E;
  const size_t P = (size_t)L.P_max;
  L.n_blocks2 = tc ? (int)((dff + 255) / 256) : simt_dgate_blocks(cfg);
  // Router-gradient partials: sized for the larger of the clean (E columns)
  // and noisy (2E) cases, so the size does not depend on the noise arguments.
  const size_t rp_c = (size_t)xtd_splits(cfg.T, cfg.d, cfg.E) * E;
  const size_t rp_n = (size_t)xtd_splits(cfg.T, cfg.d, 2 * cfg.E) * 2 * E;
  const size_t rp = rp_c > rp_n ? rp_c : rp_n;
  L.chunks = colsum_chunks(host_capacity(cfg));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.poff = take((E + 1) * 4);
  L.dY = take(P * d * rb);
  L.dU = take(P * d * rb);
  L.dP = take(P * dff * rb);
  L.dX = take(P * d * 4);
  L.dgpart = take(P * L.n_blocks2 * 4);
  L.dg = take(T * k * 4);
  L.coef = take(3 * E * 4);
  L.dc = take(T * E * 4);
  L.dz = take(T * E * 4);
  L.dxr = take(T * d * 4);
  L.rpart = take(rp * d * 4);
  L.bpart = take(rp * 4);
  L.cpart = take((size_t)L.chunks * E * (d > dff ? d : dff) * 4);
  L.total = off;
  return L;
}

// Side streams. moe_forward and moe_backward fork part of their work onto a
// side stream and join it back before they return. Each device has a pool of
// kSidePool non-blocking side streams (with a fork / join event pair each),
// made together on the first call that is not under stream capture, and each
// side stream serves ONE caller stream (the legacy and per-thread default
// streams keyed by thread as well): calls on independent caller streams never
// share a side stream, so neither serialise on it nor drag one another's work
// into a graph being captured. A call runs everything on its own stream
// instead (same kernels, same results) when no side stream fits: the pool is
// not made yet and the caller is capturing, all kSidePool are taken by other
// caller streams, or the side stream's capture state does not match the
// caller's (idle when the caller is not capturing; idle or in the caller's
// own capture when it is). The pool belongs to the context it was made in; a
// call from another context (after cudaDeviceReset) makes a new one. The lock
// is held while a call enqueues on its side stream, so calls from several
// host threads do not interleave their records.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kSideMaxDevices = 64;
constexpr int kSidePool = 8;
struct DeviceSides {
  void *ctx = nullptr;
  bool made = false, failed = false;
  int used = 0;
  SideStream pool[kSidePool];
  cudaStream_t owner[kSidePool] = {};
  size_t owner_thread[kSidePool] = {};
};
static std::mutex g_side_mu;
static DeviceSides g_side[kSideMaxDevices];

// Identifies the calling thread for the default streams, which differ (per
// thread) or are shared (legacy) without a distinct handle.
static size_t side_thread_key(cudaStream_t caller) {
  if (caller != cudaStreamPerThread && caller != nullptr) return 0;
  static thread_local char tag;
  return caller == cudaStreamPerThread ? reinterpret_cast<size_t>(&tag) : 0;
}

static SideStream *side_stream(std::unique_lock<std::mutex> &lock, cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSideMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
  unsigned long long cid = 0;
  if (cudaStreamGetCaptureInfo(caller, &cst, &cid) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cst == cudaStreamCaptureStatusInvalidated) return nullptr;
  void *ctx = current_context();
  lock = std::unique_lock<std::mutex>(g_side_mu);
  DeviceSides &D = g_side[dev];
  if ((D.made || D.failed) && D.ctx != ctx) D = DeviceSides{};  // the old context's are gone
  if (!D.made) {
    if (D.failed || cst != cudaStreamCaptureStatusNone) {
      lock.unlock();
      return nullptr;
    }
    bool ok = true;
    for (int i = 0; i < kSidePool && ok; ++i) {
      SideStream &ss = D.pool[i];
      ok = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) == cudaSuccess;
    }
    D.ctx = ctx;
    if (!ok) {
      cudaGetLastError();
      for (SideStream &ss : D.pool) {
        if (ss.join) cudaEventDestroy(ss.join);
        if (ss.fork) cudaEventDestroy(ss.fork);
        if (ss.s) cudaStreamDestroy(ss.s);
        ss = SideStream{};
      }
      D.failed = true;
      lock.unlock();
      return nullptr;
    }
    D.made = true;
  }
  const size_t tkey = side_thread_key(caller);
  int slot = -1;
  for (int i = 0; i < D.used; ++i)
    if (D.owner[i] == caller && D.owner_thread[i] == tkey) slot = i;
  if (slot < 0 && D.used < kSidePool) {
    slot = D.used++;
    D.owner[slot] = caller;
    D.owner_thread[slot] = tkey;
  }
  if (slot < 0) {
    lock.unlock();
    return nullptr;
  }
  cudaStreamCaptureStatus sst = cudaStreamCaptureStatusNone;
  unsigned long long sid = 0;
  const bool side_ok =
      cudaStreamGetCaptureInfo(D.pool[slot].s, &sst, &sid) == cudaSuccess &&
      (sst == cudaStreamCaptureStatusNone ||
       (sst == cudaStreamCaptureStatusActive && cst == cudaStreamCaptureStatusActive &&
        sid == cid));
  if (!side_ok) {
    cudaGetLastError();
    lock.unlock();
    return nullptr;
  }
  return &D.pool[slot];
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_NONFINITE: return "non-finite router logit or output";
    case MOE_ERR_TIMEOUT: return "bounded device wait ran out";
    case MOE_ERR_BOUNDS: return "index out of range";
    default: return "unknown status";
  }
}

int moe_capacity(const moe_config *cfg, int32_t *C) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (!C) return MOE_ERR_ARG;
  *C = host_capacity(*cfg);
  return MOE_OK;
}

int moe_workspace_size(const moe_config *cfg, size_t *bytes) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = ws_layout(*cfg).total;
  return MOE_OK;
}

int moe_gate(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
             const float *noise, const float *logit_bias, int32_t *expert_idx, float *gate,
             float *thr, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(Wnoise); MOE_OPT(noise); MOE_OPT(logit_bias);
  MOE_REQ(expert_idx); MOE_REQ(gate); MOE_REQ(thr);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  if ((Wnoise == nullptr) != (noise == nullptr)) return MOE_ERR_ARG;
  return gate_impl(*cfg, x, Wg, Wnoise, noise, logit_bias, expert_idx, gate, thr, ws, true,
                   (cudaStream_t)stream);
}

int moe_dispatch(const moe_config *cfg, const int32_t *expert_idx, const float *gate,
                 const void *x, int32_t *pos, uint8_t *keep, int32_t *expert_count,
                 int32_t *expert_offset, void *xbuf, int32_t *row_token, float *row_gate,
                 void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(expert_idx); MOE_REQ(gate); MOE_REQ(x); MOE_REQ(pos); MOE_REQ(keep);
  MOE_REQ(expert_count); MOE_REQ(expert_offset); MOE_REQ(xbuf); MOE_REQ(row_token);
  MOE_REQ(row_gate);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  MOE_CUDA(launch_slots(c, host_capacity(c), expert_idx, gate, ws_at<int32_t>(ws, L.hist),
                        ws_at<int32_t>(ws, L.chunk_base), expert_count, expert_offset,
                        ws_at<int32_t>(ws, L.mtiles), pos, keep, row_token, row_gate, L.n_chunks,
                        st, s));
  MOE_CUDA(launch_gather(c, x, expert_offset, row_token, xbuf, st, s));
  return MOE_OK;
}

int moe_expert_ffn(const moe_config *cfg, const void *xbuf, const int32_t *expert_offset,
                   const float *row_gate, const void *W1, const void *b1, const void *W2,
                   const void *b2, void *hbuf, float *zbuf, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(xbuf); MOE_REQ(expert_offset); MOE_REQ(row_gate); MOE_REQ(W1); MOE_OPT(b1);
  MOE_REQ(W2); MOE_OPT(b2); MOE_REQ(hbuf); MOE_REQ(zbuf);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  return ffn_impl(*cfg, xbuf, expert_offset, nullptr, row_gate, W1, b1, W2, b2, hbuf, zbuf, false,
                  ws_at<DeviceStatus>(ws, L.status), (cudaStream_t)stream);
}

int moe_combine(const moe_config *cfg, const void *x, const float *zbuf, const int32_t *pos,
                const uint8_t *keep, const int32_t *expert_idx, const int32_t *expert_offset,
                void *y, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(zbuf); MOE_REQ(pos); MOE_REQ(keep); MOE_REQ(expert_idx);
  MOE_REQ(expert_offset); MOE_REQ(y);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  MOE_CUDA(launch_combine(*cfg, x, zbuf, false, pos, keep, expert_idx, expert_offset, y,
                          ws_at<DeviceStatus>(ws, L.status), (cudaStream_t)stream));
  return MOE_OK;
}

int moe_aux_loss(const moe_config *cfg, const void *ws, float *out3, float *importance,
                 float *load, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(out3); MOE_OPT(importance); MOE_OPT(load);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  void *w = const_cast<void *>(ws);
  MOE_CUDA(launch_aux_finalize(*cfg, ws_at<float>(w, L.partials), L.n_aux_blocks, out3,
                               importance, load, ws_at<float2>(w, L.aux_vec),
                               ws_at<DeviceStatus>(w, L.status), (cudaStream_t)stream));
  return MOE_OK;
}

int moe_forward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                const float *noise, const float *logit_bias, const void *W1, const void *b1,
                const void *W2, const void *b2, void *y, float *aux_out3, int32_t *expert_idx,
                float *gate, int32_t *pos, uint8_t *keep, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(Wnoise); MOE_OPT(noise); MOE_OPT(logit_bias);
  MOE_REQ(W1); MOE_OPT(b1); MOE_REQ(W2); MOE_OPT(b2); MOE_REQ(y); MOE_OPT(aux_out3);
  MOE_OPT(expert_idx); MOE_OPT(gate); MOE_OPT(pos); MOE_OPT(keep);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  if ((Wnoise == nullptr) != (noise == nullptr)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  int32_t *idx = expert_idx ? expert_idx : ws_at<int32_t>(ws, L.idx);
  float *g = gate ? gate : ws_at<float>(ws, L.gate);
  int32_t *ps = pos ? pos : ws_at<int32_t>(ws, L.pos);
  uint8_t *kp = keep ? keep : ws_at<uint8_t>(ws, L.keep);
  float *thr = ws_at<float>(ws, L.thr);
  r = gate_impl(c, x, Wg, Wnoise, noise, logit_bias, idx, g, thr, ws, aux_out3 != nullptr, s);
  if (r != MOE_OK) return r;
  // The balancing finalize needs only the gate's partial sums: it runs on the
  // side stream beside dispatch, the expert GEMMs and combine (on `stream`
  // itself if no side stream could be made).
  SideStream *side = nullptr;
  std::unique_lock<std::mutex> side_lock;
  if (aux_out3) {
    side = side_stream(side_lock, s);
    cudaStream_t fs = s;
    if (side) {
      MOE_CUDA(cudaEventRecord(side->fork, s));
      MOE_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
      fs = side->s;
    }
    MOE_CUDA(launch_aux_finalize(c, ws_at<float>(ws, L.partials), L.n_aux_blocks, aux_out3,
                                 nullptr, nullptr, ws_at<float2>(ws, L.aux_vec), st, fs));
  }
  r = expert_path(c, L, ws, x, idx, g, ps, kp, W1, b1, W2, b2, y, st, s);
  if (r != MOE_OK) return r;
  if (side) {
    // Join: work enqueued on `stream` after this call also waits for the losses.
    MOE_CUDA(cudaEventRecord(side->join, side->s));
    MOE_CUDA(cudaStreamWaitEvent(s, side->join, 0));
  }
  return MOE_OK;
}

int moe_expert_counts(const moe_config *cfg, const int32_t *expert_idx, int32_t *expert_count,
                      void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(expert_idx); MOE_REQ(expert_count);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const WsLayout L = ws_layout(c);
  MOE_CUDA(launch_slots(c, host_capacity(c), expert_idx, nullptr, ws_at<int32_t>(ws, L.hist),
                        ws_at<int32_t>(ws, L.chunk_base), expert_count,
                        ws_at<int32_t>(ws, L.offset), ws_at<int32_t>(ws, L.mtiles), nullptr,
                        nullptr, nullptr, nullptr, L.n_chunks, ws_at<DeviceStatus>(ws, L.status),
                        (cudaStream_t)stream));
  return MOE_OK;
}

int moe_dispatch_ranked(const moe_config *cfg, int32_t capacity, const int32_t *counts_all,
                        int32_t n_ranks, int32_t rank, const int32_t *expert_idx,
                        const float *gate, const void *x, int32_t *pos, uint8_t *keep,
                        int32_t *expert_count, int32_t *expert_offset, void *xbuf,
                        int32_t *row_token, float *row_gate, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (capacity < 1 || n_ranks < 1 || rank < 0 || rank >= n_ranks) return MOE_ERR_ARG;
  MOE_REQ(counts_all); MOE_REQ(expert_idx); MOE_REQ(gate); MOE_REQ(x); MOE_REQ(pos);
  MOE_REQ(keep); MOE_REQ(expert_count); MOE_REQ(expert_offset); MOE_REQ(xbuf);
  MOE_REQ(row_token); MOE_REQ(row_gate);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const WsLayout L = ws_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  const SlotRanks ranks{counts_all, rank, ws_at<int32_t>(ws, L.ecap)};
  MOE_CUDA(launch_slots(c, capacity, expert_idx, gate, ws_at<int32_t>(ws, L.hist),
                        ws_at<int32_t>(ws, L.chunk_base), expert_count, expert_offset,
                        ws_at<int32_t>(ws, L.mtiles), pos, keep, row_token, row_gate, L.n_chunks,
                        st, s, false, &ranks));
  MOE_CUDA(launch_gather(c, x, expert_offset, row_token, xbuf, st, s));
  return MOE_OK;
}

int moe_aux_totals(const moe_config *cfg, void *ws, float *totals, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(totals);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  MOE_CUDA(launch_aux_finalize(*cfg, ws_at<float>(ws, L.partials), L.n_aux_blocks,
                               ws_at<float>(ws, L.out3s), nullptr, nullptr,
                               ws_at<float2>(ws, L.aux_vec), ws_at<DeviceStatus>(ws, L.status),
                               (cudaStream_t)stream, totals));
  return MOE_OK;
}

int moe_aux_from_totals(const moe_config *cfg, int64_t T_total, const float *totals,
                        float *out3, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (T_total < 1 || T_total > 0x7fffffffLL) return MOE_ERR_ARG;
  MOE_REQ(totals); MOE_REQ(out3);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const WsLayout L = ws_layout(*cfg);
  moe_config whole = *cfg;
  whole.T = (int32_t)T_total;  // f and Pbar are averages over the whole batch
  MOE_CUDA(launch_aux_finalize(whole, totals, 1, out3, nullptr, nullptr,
                               ws_at<float2>(ws, L.aux_vec), ws_at<DeviceStatus>(ws, L.status),
                               (cudaStream_t)stream));
  return MOE_OK;
}

int moe_hier_workspace_size(const moe_hier_config *cfg, size_t *bytes) {
  const int r = check_hier(cfg);
  if (r != MOE_OK) return r;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = hier_layout(*cfg).total;
  return MOE_OK;
}

int moe_forward_hier(const moe_hier_config *cfg, const void *x, const float *Wp,
                     const float *Wp_noise, const float *noise_p, const float *Ws,
                     const float *Ws_noise, const float *noise_s, const void *W1, const void *b1,
                     const void *W2, const void *b2, void *y, float *aux_out2,
                     int32_t *expert_idx, float *gate, int32_t *pos, uint8_t *keep, void *ws,
                     moe_stream_t stream) {
  int r = check_hier(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wp); MOE_OPT(Wp_noise); MOE_OPT(noise_p); MOE_REQ(Ws);
  MOE_OPT(Ws_noise); MOE_OPT(noise_s); MOE_REQ(W1); MOE_OPT(b1); MOE_REQ(W2); MOE_OPT(b2);
  MOE_REQ(y); MOE_OPT(aux_out2); MOE_OPT(expert_idx); MOE_OPT(gate); MOE_OPT(pos); MOE_OPT(keep);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  if ((Wp_noise == nullptr) != (noise_p == nullptr) ||
      (Ws_noise == nullptr) != (noise_s == nullptr))
    return MOE_ERR_ARG;
  const moe_hier_config &h = *cfg;
  const moe_config cs = hier_secondary(h), cp = hier_primary(h);
  const HierLayout HL = hier_layout(h);
  const WsLayout &L = HL.Ls, &Lp = HL.Lp;
  cudaStream_t s = (cudaStream_t)stream;
  void *wsp = ws_at<char>(ws, HL.off_p);
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  DeviceStatus *st_p = ws_at<DeviceStatus>(wsp, Lp.status);
  float *scratch = ws_at<float>(ws, HL.scratch);
  // 1. The primary gate: the flat gate over the a groups (picks, gates and,
  //    for the losses, its balancing sums: Load_primary).
  int32_t *idx_p = ws_at<int32_t>(wsp, Lp.idx);
  float *g_p = ws_at<float>(wsp, Lp.gate);
  r = gate_impl(cp, x, Wp, Wp_noise, noise_p, nullptr, idx_p, g_p, ws_at<float>(wsp, Lp.thr), wsp,
                aux_out2 != nullptr, s);
  if (r != MOE_OK) return r;
  if (aux_out2)
    MOE_CUDA(launch_aux_finalize(cp, ws_at<float>(wsp, Lp.partials), Lp.n_aux_blocks, scratch,
                                 nullptr, nullptr, ws_at<float2>(wsp, Lp.aux_vec), st_p, s));
  // 2. The secondary logits (the router's first kernel clears the layer's
  //    status word). Grouped: only for the (token, primary pick) pairs -- the
  //    pairs packed by group with the flat slot pass (capacity T, so nothing
  //    drops; its status goes to the primary word) and gather, then the
  //    grouped router on each group's rows and weight columns. Otherwise the
  //    dense router over all a*b experts of every token.
  const bool bf16 = h.act_dtype == MOE_BF16;
  const bool grouped = router_grouped_supported(h.d, h.b, Ws_noise != nullptr, bf16);
  float *cc, *sg, *H;
  const int32_t *gpoff = nullptr, *pos_p = nullptr;
  if (grouped) {
    moe_config cpc = cp;
    cpc.capacity_factor = (float)h.a;  // C = T: every (token, pick) pair is kept
    const int32_t *goff = ws_at<int32_t>(wsp, Lp.offset);
    MOE_CUDA(launch_slots(cpc, h.T, idx_p, g_p, ws_at<int32_t>(wsp, Lp.hist),
                          ws_at<int32_t>(wsp, Lp.chunk_base), ws_at<int32_t>(wsp, Lp.count),
                          ws_at<int32_t>(wsp, Lp.offset), ws_at<int32_t>(wsp, Lp.mtiles),
                          ws_at<int32_t>(wsp, Lp.pos), ws_at<uint8_t>(wsp, Lp.keep),
                          ws_at<int32_t>(wsp, Lp.row_token), ws_at<float>(wsp, Lp.row_gate),
                          Lp.n_chunks, st_p, s));
    MOE_CUDA(launch_gather(cpc, x, goff, ws_at<int32_t>(wsp, Lp.row_token),
                           ws_at<char>(wsp, Lp.xbuf), st_p, s));
    cc = ws_at<float>(ws, HL.gc);
    sg = ws_at<float>(ws, HL.gs);
    H = ws_at<float>(ws, HL.gH);
    gpoff = ws_at<int32_t>(ws, HL.gpoff);
    pos_p = ws_at<int32_t>(wsp, Lp.pos);
    const GroupedRouter gr{h.T, h.d, h.a, h.b, h.k_primary, ws_at<char>(wsp, Lp.xbuf), goff,
                           ws_at<int32_t>(wsp, Lp.row_token), Ws, Ws_noise, noise_s, cc, sg, H,
                           ws_at<int32_t>(ws, HL.gpoff), ws_at<char>(ws, L.bsplit)};
    MOE_CUDA(launch_router_grouped(gr, st, s));
  } else {
    cc = ws_at<float>(ws, L.c);
    sg = ws_at<float>(ws, L.sigma);
    H = ws_at<float>(ws, L.H);
    MOE_CUDA(launch_router(cs, x, Ws, Ws_noise, noise_s, nullptr, cc, sg, H,
                           ws_at<char>(ws, L.bsplit), st, s));
  }
  // 3. The two-level selection and the hierarchical partial rows.
  int32_t *idx = expert_idx ? expert_idx : ws_at<int32_t>(ws, L.idx);
  float *g = gate ? gate : ws_at<float>(ws, L.gate);
  int32_t *ps = pos ? pos : ws_at<int32_t>(ws, L.pos);
  uint8_t *kp = keep ? keep : ws_at<uint8_t>(ws, L.keep);
  float *parts = aux_out2 ? ws_at<float>(ws, HL.parts) : nullptr;
  MOE_CUDA(launch_hier_select(h.T, h.a, h.b, h.k_primary, h.k_secondary, Ws_noise != nullptr,
                              idx_p, g_p, cc, sg, H, gpoff, pos_p, idx, g, parts, st, s));
  // 4. Importance_H and the in-group loads summed over the rows, then Load_H
  //    and the two CV^2 (the tail also carries a primary-gate error over).
  if (aux_out2)
    MOE_CUDA(launch_aux_finalize(cs, parts, HL.rows, scratch + 4, nullptr, nullptr,
                                 ws_at<float2>(ws, L.aux_vec), st, s));
  MOE_CUDA(launch_hier_tail(h.T, h.a, h.b, ws_at<float2>(ws, L.aux_vec),
                            ws_at<float2>(wsp, Lp.aux_vec), aux_out2, st, st_p, s));
  // 5. Capacity, dispatch, the experts and the combine over the a*b experts.
  return expert_path(cs, L, ws, x, idx, g, ps, kp, W1, b1, W2, b2, y, st, s);
}

int moe_balanced_workspace_size(const moe_config *cfg, size_t *bytes) {
  const int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = bal_layout(*cfg).total;
  return MOE_OK;
}

int moe_forward_balanced(const moe_config *cfg, const void *x, const float *Wg,
                         const float *logit_bias, const float *thresholds, const void *W1,
                         const void *b1, const void *W2, const void *b2, void *y,
                         float *loss_out, uint32_t *mask_out, void *ws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(logit_bias); MOE_OPT(thresholds); MOE_REQ(W1); MOE_OPT(b1);
  MOE_REQ(W2); MOE_OPT(b2); MOE_REQ(y); MOE_OPT(loss_out); MOE_OPT(mask_out);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  if (loss_out && !thresholds) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const BalLayout L = bal_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  float *H = ws_at<float>(ws, L.H);
  // The E*m expert rows exceed T*k when k*T < E (m is at least 1): the row
  // kernels and GEMMs bound their packed buffers by T*k rows and find a row's
  // token as (its key) / k, so they get a k that covers every row; rows key
  // their token t as t*kr.
  moe_config cr = c;
  {
    const long long need = ((long long)c.E * L.m + c.T - 1) / c.T;
    if (need > cr.k) cr.k = (int)need;
  }
  // 1. Clean router logits (this clears the status word first).
  MOE_CUDA(launch_router(c, x, Wg, nullptr, nullptr, logit_bias, ws_at<float>(ws, L.c),
                         ws_at<float>(ws, L.sigma), H, ws_at<char>(ws, L.bsplit), st, s));
  // 2. Dense softmax, the batchwise mask (m rows per expert, token order),
  //    the renormalised gates and the L_batchwise terms.
  uint32_t *mask = mask_out ? mask_out : ws_at<uint32_t>(ws, L.mask);
  int32_t *row_token = ws_at<int32_t>(ws, L.row_token);
  float *row_gate = ws_at<float>(ws, L.row_gate);
  int32_t *offset = ws_at<int32_t>(ws, L.offset);
  double *loss = ws_at<double>(ws, L.loss);
  int32_t *trows = ws_at<int32_t>(ws, L.trows), *npick = ws_at<int32_t>(ws, L.npick);
  MOE_CUDA(launch_bal_gate(cr, L.m, H, loss_out ? thresholds : nullptr, ws_at<float>(ws, L.PT),
                           row_token, row_gate, offset, mask, trows, npick, loss, st, s));
  // 3. The expert rows through the flat gather and expert GEMMs (fp32 Z).
  void *xbuf = ws_at<char>(ws, L.xbuf), *hbuf = ws_at<char>(ws, L.hbuf);
  float *zbuf = ws_at<float>(ws, L.zbuf);
  MOE_CUDA(launch_gather(cr, x, offset, row_token, xbuf, st, s));
  if (c.act_dtype == MOE_BF16 && ffn_tc_supported(c)) {
    MOE_CUDA(launch_ffn_tc(cr, L.m, xbuf, offset, nullptr, row_gate, W1, b1, W2, b2, hbuf, zbuf,
                           false, st, s));
  } else {
    MOE_CUDA(launch_ffn_simt(cr, L.m, xbuf, offset, row_gate, W1, b1, W2, b2, hbuf, zbuf, st, s));
  }
  // 4. y = x + the picks' outputs, and the loss.
  MOE_CUDA(launch_bal_combine(cr, L.m, x, zbuf, mask, row_token, trows, npick, y, st, s));
  if (loss_out) MOE_CUDA(launch_bal_loss(c.E, loss, loss_out, s));
  return MOE_OK;
}

int moe_threshold_workspace_size(const moe_config *cfg, size_t *bytes) {
  const int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = ws_layout(thr_layer(*cfg)).total;
  return MOE_OK;
}

int moe_forward_threshold(const moe_config *cfg, const void *x, const float *Wg,
                          const float *logit_bias, const float *thresholds, const void *W1,
                          const void *b1, const void *W2, const void *b2, void *y,
                          int32_t *expert_idx, float *gate, uint32_t *mask_out, void *ws,
                          moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(logit_bias); MOE_REQ(thresholds); MOE_REQ(W1); MOE_OPT(b1);
  MOE_REQ(W2); MOE_OPT(b2); MOE_REQ(y); MOE_OPT(expert_idx); MOE_OPT(gate); MOE_OPT(mask_out);
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  const moe_config c = thr_layer(*cfg);
  const WsLayout L = ws_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  float *H = ws_at<float>(ws, L.H);
  // 1. Clean router logits (this clears the status word first).
  MOE_CUDA(launch_router(c, x, Wg, nullptr, nullptr, logit_bias, ws_at<float>(ws, L.c),
                         ws_at<float>(ws, L.sigma), H, ws_at<char>(ws, L.bsplit), st, s));
  // 2. P = Softmax(H), the picks P_i > T_i and their renormalised gates.
  int32_t *idx = expert_idx ? expert_idx : ws_at<int32_t>(ws, L.idx);
  float *g = gate ? gate : ws_at<float>(ws, L.gate);
  MOE_CUDA(launch_thr_gate(c, H, thresholds, idx, g, mask_out, st, s));
  // 3. Slots (token order, no capacity), gather, expert GEMMs, combine.
  return expert_path(c, L, ws, x, idx, g, ws_at<int32_t>(ws, L.pos), ws_at<uint8_t>(ws, L.keep),
                     W1, b1, W2, b2, y, st, s, true);
}

int moe_backward_workspace_size(const moe_config *cfg, size_t *bytes) {
  const int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = bwd_layout(*cfg).total;
  return MOE_OK;
}

// The gate's backward from the total gate gradients (dg_total) or from the
// kept choices' <dy, U> plus the Importance term (coef), then the router's
// weight gradients and its share of dx.
static int gate_bwd_impl(const moe_config &c, const WsLayout &L, const BwdLayout &B, void *ws,
                         void *bws, const void *x, const float *Wg, const float *Wn,
                         const float *noise, const int32_t *idx, const float *g,
                         const uint8_t *kp, const float *dg, bool dg_total, float w_imp,
                         float w_load, float w_aux, float *dgate_out, float *dWg, float *dWn,
                         float *dbias, float *dxr, cudaStream_t s) {
  const bool noisy = Wn != nullptr;
  const bool load_on = noisy && c.k < c.E && w_load != 0.f;
  const bool aux_on = w_aux != 0.f;
  float *coef = ws_at<float>(bws, B.coef);
  MOE_CUDA(launch_bwd_coef(c, ws_at<float2>(ws, L.aux_vec), w_imp, w_load, w_aux, coef, s));
  float *dc = ws_at<float>(bws, B.dc), *dz = ws_at<float>(bws, B.dz);
  MOE_CUDA(launch_bwd_gate(c, noisy, load_on, aux_on, dg_total, ws_at<float>(ws, L.H),
                           ws_at<float>(ws, L.c), ws_at<float>(ws, L.sigma), noise,
                           ws_at<float>(ws, L.rowstat), ws_at<float>(ws, L.thr), idx, g, kp, dg,
                           coef, dgate_out, dc, noisy ? dz : nullptr, s));
  MOE_CUDA(launch_bwd_router(c, noisy, x, Wg, Wn, dc, noisy ? dz : nullptr,
                             ws_at<float>(bws, B.rpart), ws_at<float>(bws, B.bpart), dWg, dWn,
                             dbias, dxr, s));
  return MOE_OK;
}

int moe_gate_backward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                      const float *noise, const int32_t *expert_idx, const float *gate,
                      const float *dgate, float w_load, float w_aux, float *dWg, float *dWnoise,
                      float *dlogit_bias, float *dx_gate, void *ws, void *bws,
                      moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(Wnoise); MOE_OPT(noise); MOE_OPT(expert_idx); MOE_OPT(gate);
  MOE_REQ(dgate); MOE_REQ(dWg); MOE_OPT(dWnoise); MOE_OPT(dlogit_bias); MOE_OPT(dx_gate);
  if (!ws || !aligned(ws, 256) || !bws || !aligned(bws, 256)) return MOE_ERR_ARG;
  if ((Wnoise == nullptr) != (noise == nullptr) || (Wnoise == nullptr) != (dWnoise == nullptr))
    return MOE_ERR_ARG;
  if (!isfinite(w_load) || !isfinite(w_aux)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const WsLayout L = ws_layout(c);
  const BwdLayout B = bwd_layout(c);
  const int32_t *idx = expert_idx ? expert_idx : ws_at<int32_t>(ws, L.idx);
  const float *g = gate ? gate : ws_at<float>(ws, L.gate);
  return gate_bwd_impl(c, L, B, ws, bws, x, Wg, Wnoise, noise, idx, g, nullptr, dgate, true, 0.f,
                       w_load, w_aux, nullptr, dWg, dWnoise, dlogit_bias, dx_gate,
                       (cudaStream_t)stream);
}

int moe_backward(const moe_config *cfg, const void *x, const float *Wg, const float *Wnoise,
                 const float *noise, const void *W1, const void *W2, const void *b2,
                 const int32_t *expert_idx, const float *gate, const int32_t *pos,
                 const uint8_t *keep, const void *dy, float w_importance, float w_load,
                 float w_aux, void *dx, float *dWg, float *dWnoise, float *dlogit_bias,
                 float *dW1, float *db1, float *dW2, float *db2, float *dgate, void *ws,
                 void *bws, moe_stream_t stream) {
  int r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  MOE_REQ(x); MOE_REQ(Wg); MOE_OPT(Wnoise); MOE_OPT(noise); MOE_REQ(W1); MOE_REQ(W2);
  MOE_OPT(b2); MOE_OPT(expert_idx); MOE_OPT(gate); MOE_OPT(pos); MOE_OPT(keep); MOE_REQ(dy);
  MOE_REQ(dx); MOE_REQ(dWg); MOE_OPT(dWnoise); MOE_OPT(dlogit_bias); MOE_REQ(dW1); MOE_OPT(db1);
  MOE_REQ(dW2); MOE_OPT(db2); MOE_OPT(dgate);
  if (!ws || !aligned(ws, 256) || !bws || !aligned(bws, 256)) return MOE_ERR_ARG;
  if ((Wnoise == nullptr) != (noise == nullptr) || (Wnoise == nullptr) != (dWnoise == nullptr))
    return MOE_ERR_ARG;
  if (!isfinite(w_importance) || !isfinite(w_load) || !isfinite(w_aux)) return MOE_ERR_ARG;
  const moe_config &c = *cfg;
  const bool tc = bwd_tc_shape(c);
  if (tc && !bwd_tc_supported(c)) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(c);
  const BwdLayout B = bwd_layout(c);
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus *st = ws_at<DeviceStatus>(ws, L.status);
  const int32_t *idx = expert_idx ? expert_idx : ws_at<int32_t>(ws, L.idx);
  const float *g = gate ? gate : ws_at<float>(ws, L.gate);
  const int32_t *ps = pos ? pos : ws_at<int32_t>(ws, L.pos);
  const uint8_t *kp = keep ? keep : ws_at<uint8_t>(ws, L.keep);
  const int32_t *offset = ws_at<int32_t>(ws, L.offset);
  const int32_t *row_token = ws_at<int32_t>(ws, L.row_token);
  const float *row_gate = ws_at<float>(ws, L.row_gate);
  void *xbuf = ws_at<char>(ws, L.xbuf), *hbuf = ws_at<char>(ws, L.hbuf);
  int32_t *poff = ws_at<int32_t>(bws, B.poff);
  void *dY = ws_at<char>(bws, B.dY), *dU = ws_at<char>(bws, B.dU), *dP = ws_at<char>(bws, B.dP);
  float *dX = ws_at<float>(bws, B.dX), *dgpart = ws_at<float>(bws, B.dgpart);
  float *dg = ws_at<float>(bws, B.dg), *dxr = ws_at<float>(bws, B.dxr);
  const long long A_rows = (long long)c.T * c.k;
  const long long cap = host_capacity(c);  // rows per expert at most
  // CUDA-core form (fp32 rows): the same steps, in k_bwd_simt.cu.
  const BwdSimt sp{B.P_max, offset, poff, row_token, row_gate, dy, W1, W2, b2, xbuf, hbuf,
                   static_cast<float *>(dY), static_cast<float *>(dU), static_cast<float *>(dP),
                   dX, dgpart, dW1, dW2, st};
  // 1. Padded row blocks, finite K tails, the dy rows (plain and gate-scaled);
  // 2. through W2: D = dY W2^T, the gate partials <D, h> and dpre = g D [h > 0].
  MOE_CUDA(launch_bwd_offsets(c.E, offset, poff, s));
  if (tc) {
    MOE_CUDA(launch_bwd_tail_zero(c, offset, xbuf, hbuf, s));
    MOE_CUDA(launch_bwd_gather(c, B.P_max, offset, poff, row_token, row_gate, dy, dY, dU, s));
    BwdGemm g0{0, c.d, c.d_ff, 0, c.E, B.P_max, 0, 0, dY, W2, offset, poff, row_gate, hbuf, dP,
               dgpart};
    MOE_CUDA(launch_bwd_gemm(g0, st, s));
  } else {
    MOE_CUDA(launch_bwd_simt_front(c, sp, s));
  }
  // From here two independent branches. On the side stream (the library's,
  // as in moe_forward; `stream` itself if none could be made): the gate's
  // backward from the dgate partials -- <dy, U> per kept choice, the gate,
  // load and Switch terms, the router's weight gradients and its share of dx
  // -- and the bias column sums. Their small kernels fit beside the
  // persistent GEMM CTAs of the other branch, which stays on `stream`.
  SideStream *side = nullptr;
  std::unique_lock<std::mutex> side_lock;
  side = side_stream(side_lock, s);
  cudaStream_t fs = s;
  if (side) {
    MOE_CUDA(cudaEventRecord(side->fork, s));
    MOE_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    fs = side->s;
  }
  if (tc)
    MOE_CUDA(launch_bwd_dg(c, B.n_blocks2, offset, poff, row_token, dgpart, dy, b2, dg, fs));
  else
    MOE_CUDA(launch_bwd_simt_dg(c, sp, dg, fs));
  r = gate_bwd_impl(c, L, B, ws, bws, x, Wg, Wnoise, noise, idx, g, kp, dg, false, w_importance,
                    w_load, w_aux, dgate, dWg, dWnoise, dlogit_bias, dxr, fs);
  if (r != MOE_OK) return r;
  float *cpart = ws_at<float>(bws, B.cpart);
  if (db2)
    MOE_CUDA(launch_bwd_colsum(c, c.d, B.chunks, offset, poff, row_gate, dY, !tc, cpart, db2,
                               fs));
  if (db1)
    MOE_CUDA(launch_bwd_colsum(c, c.d_ff, B.chunks, offset, poff, nullptr, dP, !tc, cpart, db1,
                               fs));
  // 3. Through W1: dX = dpre W1^T; weight gradients dW2[e] = h^T (g dY),
  //    dW1[e] = x^T dpre.
  if (tc) {
    BwdGemm g1{1, c.d_ff, c.d, 0, c.E, B.P_max, 0, 0, dP, W1, offset, poff, nullptr, nullptr, dX,
               nullptr};
    MOE_CUDA(launch_bwd_gemm(g1, st, s));
    BwdGemm g2{2, 0, c.d, c.d_ff, c.E, A_rows, B.P_max, cap, hbuf, dU, offset, poff, nullptr,
               nullptr, dW2, nullptr};
    MOE_CUDA(launch_bwd_gemm(g2, st, s));
    BwdGemm g3{2, 0, c.d_ff, c.d, c.E, A_rows, B.P_max, cap, xbuf, dP, offset, poff, nullptr,
               nullptr, dW1, nullptr};
    MOE_CUDA(launch_bwd_gemm(g3, st, s));
  } else {
    MOE_CUDA(launch_bwd_simt_back(c, sp, s));
  }
  if (side) {
    MOE_CUDA(cudaEventRecord(side->join, side->s));
    MOE_CUDA(cudaStreamWaitEvent(s, side->join, 0));
  }
  // 4. dx = dy + the router's share + the kept experts' rows.
  if (tc)
    MOE_CUDA(launch_bwd_dx(c, idx, ps, kp, poff, dX, dxr, dy, dx, s));
  else
    MOE_CUDA(launch_bwd_simt_dx(c, sp, idx, ps, kp, dxr, dx, s));
  return MOE_OK;
}

int moe_last_device_status(void *ws, moe_stream_t stream, int64_t *detail) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  DeviceStatus h{};
  MOE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  MOE_CUDA(cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(ws, 0, sizeof h));
  if (detail) *detail = h.detail;
  return h.code;
}

}  // extern "C"
