// api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence of the
// fused MoE forward on the caller's stream.  No host synchronisation and no
// allocation happen here (except moe_get_device_status, which syncs).
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {
cudaError_t grouped_gemm_set_attributes();
cudaError_t small_gemm_set_attributes();
cudaError_t router_set_attributes();
cudaError_t route_fused_set_attributes();
cudaError_t dispatch_combine_set_attributes();
}  // namespace moe

using namespace moe;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

// ---------------------------------------------------------------- device --

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready;
  int sms;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].ready) {
    int major = 0, minor = 0, n = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(MOE_ERR_UNSUPPORTED, "built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    if ((e = router_set_attributes()) != cudaSuccess) return cuda_fail(e, "router attributes");
    if ((e = route_fused_set_attributes()) != cudaSuccess) return cuda_fail(e, "route attributes");
    if ((e = grouped_gemm_set_attributes()) != cudaSuccess) return cuda_fail(e, "gemm attributes");
    if ((e = small_gemm_set_attributes()) != cudaSuccess) return cuda_fail(e, "gemm attributes");
    if ((e = dispatch_combine_set_attributes()) != cudaSuccess)
      return cuda_fail(e, "dispatch/combine attributes");
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    g_dev[dev].sms = n;
    g_dev[dev].ready = true;
  }
  *sms = g_dev[dev].sms;
  return MOE_OK;
}

// bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
int encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides_bytes, const uint32_t* box, const char* what) {
  uint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                        dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return MOE_OK;
}

int map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
           uint32_t box_outer, const char* what) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_map(m, base, 2, dims, strides, box, what);
}

int map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
           uint32_t box0, uint32_t box1, const char* what) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {box0, box1, 1};
  return encode_map(m, base, 3, dims, strides, box, what);
}

// ------------------------------------------------------------ validation --

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const moe_shape* s, bool need_ffn) {
  if (!s) return fail(MOE_ERR_INVALID_ARG, "shape is null");
  if (s->T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", s->T);
  if (s->E < 1 || s->E > kMaxExperts)
    return fail(MOE_ERR_UNSUPPORTED, "E = %d: need 1 <= E <= %d", s->E, kMaxExperts);
  if (s->k < 1 || s->k > kMaxTopK || s->k > s->E)
    return fail(MOE_ERR_UNSUPPORTED, "k = %d: need 1 <= k <= min(8, E)", s->k);
  if (s->H < 8 || s->H % 8 != 0) return fail(MOE_ERR_UNSUPPORTED, "H = %d: need H >= 8, H %% 8 == 0", s->H);
  if (need_ffn && (s->F < 8 || s->F % 8 != 0))
    return fail(MOE_ERR_UNSUPPORTED, "F = %d: need F >= 8, F %% 8 == 0", s->F);
  if (s->expert_act != MOE_EXPERT_GELU && s->expert_act != MOE_EXPERT_SWIGLU)
    return fail(MOE_ERR_INVALID_ARG, "expert_act = %d: not a MOE_EXPERT_* value", s->expert_act);
  if (s->gating < MOE_GATE_TOPK_SOFTMAX || s->gating > MOE_GATE_SOFTMAX_TOPK_RENORM)
    return fail(MOE_ERR_INVALID_ARG, "gating = %d: not a MOE_GATE_* value", s->gating);
  if ((int64_t)s->T * s->k > (int64_t)1 << 24)
    return fail(MOE_ERR_UNSUPPORTED, "T * k = %lld exceeds 2^24", (long long)s->T * s->k);
  return MOE_OK;
}

#define REQUIRE_PTR(p)                                                               \
  do {                                                                               \
    if (!(p)) return fail(MOE_ERR_INVALID_ARG, "%s is null", #p);                    \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

int64_t capacity_of(const moe_shape* s) {
  const double cf = s->capacity_factor;
  if (!(cf > 0.0)) return -1;
  const double tk = (double)s->T * (double)s->k;
  double c = ceil(cf * tk / (double)s->E - 1e-9);
  if (c < 0.0) c = 0.0;
  if (c > tk) c = tk;
  return (int64_t)c;
}

// --------------------------------------------------------------- workspace --

// Workspace: [status block | per-tile expert counts | padded W_router |
// fused-route counts | h | Y | fp32 partials].  The status block holds the
// device status word (byte 0), the router's completion ticket (byte 64) and
// the fused route's grid counter (byte 128); all are cleared at the start of
// every call.  The padded W_router copy exists only when E % 8 != 0, the
// fused route's counts only for shapes it serves.
constexpr size_t kStatusBytes = 1024;
constexpr size_t kTicketOffset = 64;
constexpr size_t kGridCntOffset = 128;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
size_t hist_bytes(const moe_shape* s) {
  return align_up((size_t)((s->T + kSegTokens - 1) / kSegTokens) * s->E * 4, 1024);
}
// W_router's row pitch as the route reads it: E rounded up to 8 (16 bytes)
int router_ldw(const moe_shape* s) { return (s->E + 7) / 8 * 8; }
size_t wpad_bytes(const moe_shape* s) {
  return s->E % 8 ? align_up((size_t)s->H * router_ldw(s) * 2, 1024) : 0;
}
size_t h_bytes(const moe_shape* s) { return align_up((size_t)s->T * s->k * s->F * 2, 1024); }
size_t y_bytes(const moe_shape* s) { return align_up((size_t)s->T * s->k * s->H * 2, 1024); }

// The route runs on the CUDA cores in one launch for small batches, as one
// fused tensor-core launch for up to kFusedMaxTiles x 128 tokens (when its
// clusters all fit on the device at once; every sm_103 part holds 128 of its
// CTAs), else as router + dispatch kernels.
bool route_small(const moe_shape* s) { return s->T <= kSmallRouteTokens && s->E <= kSmallRouteExperts; }
int route_tiles(const moe_shape* s) { return (s->T + 127) / 128; }
bool route_fused_shape(const moe_shape* s) {
  return !route_small(s) && s->T > 0 && route_tiles(s) <= kFusedMaxTiles;
}
int route_npad(const moe_shape* s) { return (s->E + 15) / 16 * 16; }
// upper bound of the fused route's CTAs (64-token tiles x K splits), from
// the shape alone
int fused_ctas_bound(const moe_shape* s) {
  const int kb = (s->H + 63) / 64;
  const long long n = (long long)((s->T + 63) / 64) * (kb < kFusedMaxSplits ? kb : kFusedMaxSplits);
  return (int)(n < kFusedMaxCtas ? n : kFusedMaxCtas);
}
size_t fused_hist_bytes(const moe_shape* s) {
  return route_fused_shape(s) ? align_up((size_t)fused_ctas_bound(s) * route_npad(s), 1024) : 0;
}
size_t route_ws_bytes(const moe_shape* s) {
  return kStatusBytes + hist_bytes(s) + wpad_bytes(s) + fused_hist_bytes(s);
}
// small batches: fp32 partial expert outputs of a K-split second GEMM
size_t part_bytes(const moe_shape* s) {
  const size_t rows = (size_t)s->T * s->k;
  return rows <= (size_t)kSmallGemmRows ? align_up((size_t)kMaxKSplits * rows * s->H * 4, 1024) : 0;
}
size_t ws_bytes_for(const moe_shape* s) {
  return route_ws_bytes(s) + h_bytes(s) + y_bytes(s) + part_bytes(s);
}

int* status_ptr(void* ws) { return reinterpret_cast<int*>(ws); }
unsigned int* ticket_ptr(void* ws) {
  return reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + kTicketOffset);
}
int32_t* hist_ptr(void* ws) {
  return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kStatusBytes);
}
uint16_t* wpad_ptr(void* ws, const moe_shape* s) {
  return reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + kStatusBytes + hist_bytes(s));
}
uint8_t* fused_hist_ptr(void* ws, const moe_shape* s) {
  return reinterpret_cast<uint8_t*>(static_cast<char*>(ws) + kStatusBytes + hist_bytes(s) +
                                    wpad_bytes(s));
}
uint16_t* h_ptr(void* ws, const moe_shape* s) {
  return reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + route_ws_bytes(s));
}
float* part_ptr(void* ws, const moe_shape* s) {
  if (part_bytes(s) == 0) return nullptr;
  return reinterpret_cast<float*>(static_cast<char*>(ws) + route_ws_bytes(s) + h_bytes(s) +
                                  y_bytes(s));
}
uint16_t* y_ptr(void* ws, const moe_shape* s) {
  return reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + route_ws_bytes(s) + h_bytes(s));
}

// ------------------------------------------------------------------ steps --

// Optional timing hooks: ev[i] (a cudaEvent_t, may be null) is recorded on
// the stream at kernel boundary i (0 = before the router, 1..6 = after the
// router, dispatch, permute, GEMM1, GEMM2 and combine).  Recorded as external events
// so that, inside a stream capture, they become timed event-record nodes.
int mark(void* const* ev, int i, cudaStream_t st) {
  if (!ev || !ev[i]) return MOE_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  e = cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[i]), st,
                               cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                   : cudaEventRecordDefault);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaEventRecord");
}

int enqueue_route(const moe_shape* s, int sms, const uint16_t* x, const uint16_t* w_router,
                  const float* b_router, int32_t* ids, float* weights, int32_t* counts,
                  int32_t* offsets, int32_t* perm, int32_t* slot, void* ws, cudaStream_t st,
                  void* const* ev = nullptr) {
  int rc;
  // W_router rows that are not 16-byte aligned (E % 8 != 0) are read from a
  // zero-padded copy in the workspace (the padded experts are never chosen)
  const int ldw = router_ldw(s);
  if (s->E % 8) {
    uint16_t* wp = wpad_ptr(ws, s);
    cudaError_t e = launch_pad_router_weights(w_router, s->H, s->E, ldw, wp, sms, st, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "router weight padding launch");
    w_router = wp;
  }
  if (route_small(s)) {
    // small batch: logits on the CUDA cores and the dispatch by the last
    // CTA, one launch (a 32-token decode step routes in well under half the
    // time of the tensor-core router followed by the dispatch kernel)
    SmallRouteArgs sa;
    sa.x = x;
    sa.w = w_router;
    sa.ldw = ldw;
    sa.bias = b_router;
    sa.T = s->T;
    sa.H = s->H;
    sa.E = s->E;
    sa.k = s->k;
    sa.capacity = (int)capacity_of(s);
    sa.gating = s->gating;
    sa.ids = ids;
    sa.weights = weights;
    sa.counts = counts;
    sa.offsets = offsets;
    sa.perm = perm;
    sa.slot = slot;
    sa.ticket = ticket_ptr(ws);
    if ((rc = mark(ev, 0, st)) != MOE_OK) return rc;
    cudaError_t e = launch_router_small(sa, st, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");
    if ((rc = mark(ev, 1, st)) != MOE_OK) return rc;
    return mark(ev, 2, st);  // no separate dispatch kernel
  }
  CUtensorMap tm_x, tm_w;
  if ((rc = map_2d(&tm_w, w_router, (uint64_t)ldw, (uint64_t)s->H, 64, 64, "w_router")) != MOE_OK) return rc;
  const int mtiles = route_tiles(s);
  const int kblocks = (s->H + 63) / 64;
  FusedRoutePlan plan;
  if (route_fused_shape(s) && route_fused_pick(s->T, s->H, s->E, &plan)) {
    if ((rc = map_2d(&tm_x, x, (uint64_t)s->H, (uint64_t)s->T, 64, (uint32_t)plan.tm, "x (route)")) != MOE_OK)
      return rc;
    FusedRouteArgs fa;
    fa.T = s->T;
    fa.H = s->H;
    fa.E = s->E;
    fa.k = s->k;
    fa.npad = route_npad(s);
    fa.ep = route_npad(s);
    fa.tmem_cols = 32;
    while (fa.tmem_cols < fa.npad) fa.tmem_cols *= 2;
    fa.capacity = (int)capacity_of(s);
    fa.gating = s->gating;
    fa.bias = b_router;
    fa.ids = ids;
    fa.weights = weights;
    fa.counts = counts;
    fa.offsets = offsets;
    fa.perm = perm;
    fa.slot = slot;
    fa.grp_hist = fused_hist_ptr(ws, s);
    fa.grid_cnt = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kGridCntOffset);
    fa.status = status_ptr(ws);
    fa.wait_limit_ns = kWaitLimitNs;
    if ((rc = mark(ev, 0, st)) != MOE_OK) return rc;
    cudaError_t e = launch_route_fused(tm_x, tm_w, fa, plan, st, ev == nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    if ((rc = mark(ev, 1, st)) != MOE_OK) return rc;
    return mark(ev, 2, st);  // the dispatch ran in the same launch
  }
  if ((rc = map_2d(&tm_x, x, (uint64_t)s->H, (uint64_t)s->T, 64, 128, "x (router)")) != MOE_OK) return rc;
  RouterArgs ra;
  ra.T = s->T;
  ra.H = s->H;
  ra.E = s->E;
  ra.k = s->k;
  ra.npad = (s->E + 15) / 16 * 16;
  ra.tmem_cols = 32;
  while (ra.tmem_cols < ra.npad) ra.tmem_cols *= 2;
  // K splits per 128-token tile: as many as keep every cluster resident in a
  // single wave (a second wave would double the router's time)
  ra.splits = 1;
  while (ra.splits < 8 && mtiles * ra.splits * 2 <= sms && ra.splits * 2 <= kblocks) {
    int fit = 0;
    cudaError_t ce = router_max_clusters(s->E, ra.splits * 2, &fit);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaOccupancyMaxActiveClusters(router)");
    if (fit < mtiles) break;
    ra.splits *= 2;
  }
  ra.capacity = (int)capacity_of(s);
  ra.gating = s->gating;
  ra.bias = b_router;
  ra.ids = ids;
  ra.weights = weights;
  ra.hist = hist_ptr(ws);
  ra.counts = counts;
  ra.offsets = offsets;
  ra.ticket = ticket_ptr(ws);
  ra.scan_in_dispatch = dispatch_scans(mtiles, s->E) ? 1 : 0;
  ra.status = status_ptr(ws);
  ra.wait_limit_ns = kWaitLimitNs;
  if ((rc = mark(ev, 0, st)) != MOE_OK) return rc;
  cudaError_t e = launch_router(tm_x, tm_w, ra, st, ev == nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  if ((rc = mark(ev, 1, st)) != MOE_OK) return rc;

  DispatchArgs da;
  da.ids = ids;
  da.T = s->T;
  da.k = s->k;
  da.E = s->E;
  da.capacity = ra.capacity;
  da.seg_tokens = kSegTokens;
  da.scan = ra.scan_in_dispatch;
  da.base = hist_ptr(ws);
  da.counts = counts;
  da.offsets = offsets;
  da.perm = perm;
  da.slot = slot;
  da.status = status_ptr(ws);
  // the router precedes it on the stream: start early unless timing hooks
  // sit between the two kernels
  e = launch_dispatch(da, st, ev == nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  return mark(ev, 2, st);
}

// GEMM1 (+ activation) into h, then GEMM2 into `out`, over T*k rows grouped
// in n_seg segments: segment i (rows [seg_offsets[i], seg_offsets[i+1]))
// uses expert i % s->E.  combine_k1: GEMM2 writes y[perm[r]] = w * acc.
// pdl_first: GEMM1 starts early (programmatic dependent launch); false only
// when a timing event sits before it.
int enqueue_expert_gemms(const moe_shape* s, int n_seg, const uint16_t* xp, const uint16_t* w1,
                         const uint16_t* w2, const int32_t* seg_offsets, uint16_t* h,
                         uint16_t* out, bool combine_k1, const int32_t* perm,
                         const float* weights, int* status, cudaStream_t st, bool pdl_first,
                         bool pdl, void* const* ev, int ev_gemm1, int ev_gemm2,
                         float* part = nullptr, int* splits_used = nullptr) {
  int rc;
  const uint64_t rows = (uint64_t)s->T * s->k;
  const bool swiglu = s->expert_act == MOE_EXPERT_SWIGLU;
  if (splits_used) *splits_used = 1;

  // Small batch (every segment fits one 64-token tile): a GEMM may run on
  // the kernel that streams the weights as the MMA's M operand
  // (ffn_gemm_small.cu), which keeps more weight bytes in flight.  Measured
  // on a decode step it wins with at least two waves of column tiles
  // (GEMM1: 448 tiles, 0.155 -> 0.142 ms) and loses slightly below (GEMM2:
  // 128 tiles, 0.154 -> 0.156 ms), so a GEMM takes it only with at least
  // 2 * co-resident-pairs tiles.  When its fp32 partials can go to `part`
  // (the combine sums them), GEMM2 may split K in S <= kMaxKSplits parts to
  // reach that and fill its last wave best: decode GEMM2's 128 column tiles
  // are 1.7 waves on 76 pairs, with S = 4 its 512 tiles are 6.7.  Gated
  // experts keep GEMM1 on the main kernel.
  int small_pairs = 0;
  if (rows <= (uint64_t)kSmallGemmRows) {
    cudaError_t ce = small_gemm_max_pairs(&small_pairs);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaOccupancyMaxActiveClusters(small gemm)");
  }
  const int64_t small_tiles1 = (int64_t)n_seg * ((s->F + 255) / 256);
  const int64_t small_tiles2 = (int64_t)n_seg * ((s->H + 255) / 256);
  const bool small1 = small_pairs > 0 && !swiglu && small_tiles1 >= 2 * (int64_t)small_pairs;
  int S2 = 0;  // 0: GEMM2 on the main kernel
  if (small_pairs > 0 && part && !combine_k1) {
    const int kb2 = (s->F + 63) / 64;
    double best = 0.0;
    for (int S = 1; S <= kMaxKSplits && S <= kb2; ++S) {
      const int64_t n = small_tiles2 * S;
      if (n < 2 * (int64_t)small_pairs) continue;
      const double waves = (double)n / small_pairs;
      const double eff = waves / ceil(waves);
      if (eff > best + 1e-9) {
        best = eff;
        S2 = S;
      }
    }
  } else if (small_pairs > 0 && small_tiles2 >= 2 * (int64_t)small_pairs) {
    S2 = 1;
  }
  const bool small2 = S2 > 0;

  // token-row boxes: 32 rows for the small kernel, 128 (a CTA's half of a
  // 256-row pair tile) for the main one
  CUtensorMap tm_xp, tm_w1, tm_h, tm_w2;
  const uint64_t w1_cols = (uint64_t)s->F * (swiglu ? 2 : 1);  // SwiGLU: [W_gate | W_up]
  if ((rc = map_2d(&tm_xp, xp, (uint64_t)s->H, rows, 64, small1 ? 32 : 128, "xp")) != MOE_OK) return rc;
  if ((rc = map_3d(&tm_w1, w1, w1_cols, (uint64_t)s->H, (uint64_t)s->E, 64, 64, "W1")) != MOE_OK) return rc;
  if ((rc = map_2d(&tm_h, h, (uint64_t)s->F, rows, 64, small2 ? 32 : 128, "h")) != MOE_OK) return rc;
  // 64-row boxes for the main kernel's M = 128 tiles
  CUtensorMap tm_xp64, tm_h64;
  if ((rc = map_2d(&tm_xp64, xp, (uint64_t)s->H, rows, 64, 64, "xp")) != MOE_OK) return rc;
  if ((rc = map_2d(&tm_h64, h, (uint64_t)s->F, rows, 64, 64, "h")) != MOE_OK) return rc;
  if ((rc = map_3d(&tm_w2, w2, (uint64_t)s->H, (uint64_t)s->F, (uint64_t)s->E, 64, 64, "W2")) != MOE_OK) return rc;

  // pair tiles of the main kernel are 2*kGemmBM rows: a segment with n rows
  // owns ceil(n / 256)
  const int64_t row_blocks_ub = ((int64_t)rows + 2 * kGemmBM - 1) / (2 * kGemmBM) + n_seg;
  GemmArgs g;
  g.offsets = seg_offsets;
  g.E = n_seg;
  g.E_w = s->E;
  g.perm = perm;
  g.gate_w = weights;
  g.T = s->T;
  g.splits = 1;
  g.part = nullptr;
  g.part_stride = 0;
  g.status = status;
  g.wait_limit_ns = kWaitLimitNs;

  g.N = s->F;
  g.K = s->H;
  g.out = h;
  cudaError_t e;
  if (small1) {
    e = launch_small_gemm(kGemmGelu, tm_w1, tm_xp, g, (int)small_tiles1, st, pdl_first);
  } else {
    const int out_cols = swiglu ? kGemmBN / 2 : kGemmBN;  // h columns per pair tile
    const int64_t ub = row_blocks_ub * ((s->F + out_cols - 1) / out_cols);
    e = launch_grouped_gemm(swiglu ? kGemmSwiGLU : kGemmGelu, tm_xp, tm_w1, tm_xp64, g,
                            (int)(ub < (1 << 30) ? ub : (1 << 30)), st, pdl_first);
  }
  if (e != cudaSuccess) return cuda_fail(e, "expert GEMM1 launch");
  if ((rc = mark(ev, ev_gemm1, st)) != MOE_OK) return rc;

  g.N = s->H;
  g.K = s->F;
  g.out = out;
  if (small2) {
    const int mode2 = combine_k1 ? kGemmCombineK1 : S2 > 1 ? kGemmPartial : kGemmPlain;
    g.splits = S2;
    g.part = part;
    g.part_stride = (size_t)rows * s->H;
    e = launch_small_gemm(mode2, tm_w2, tm_h, g, (int)(small_tiles2 * S2), st, pdl);
    if (e == cudaSuccess && splits_used) *splits_used = S2;
  } else {
    const int64_t ub = row_blocks_ub * ((s->H + kGemmBN - 1) / kGemmBN);
    e = launch_grouped_gemm(combine_k1 ? kGemmCombineK1 : kGemmPlain, tm_h, tm_w2, tm_h64, g,
                            (int)(ub < (1 << 30) ? ub : (1 << 30)), st, pdl);
  }
  if (e != cudaSuccess) return cuda_fail(e, "expert GEMM2 launch");
  return mark(ev, ev_gemm2, st);
}

int enqueue_ffn_combine(const moe_shape* s, int sms, const uint16_t* x, const uint16_t* w1,
                        const uint16_t* w2, const float* weights, const int32_t* offsets,
                        const int32_t* perm, const int32_t* slot, uint16_t* y, void* ws,
                        cudaStream_t st, void* const* ev = nullptr) {
  int rc;
  // Every kernel starts early (programmatic dependent launch) unless timing
  // hooks sit between the kernels.
  const bool pdl = ev == nullptr;
  uint16_t* h = h_ptr(ws, s);
  uint16_t* Y = y_ptr(ws, s);
  uint16_t* xp = Y;  // the permuted tokens live where GEMM2 later writes Y

  PermuteArgs pa;
  pa.x = x;
  pa.perm = perm;
  pa.offsets = offsets;
  pa.T = s->T;
  pa.H = s->H;
  pa.k = s->k;
  pa.E = s->E;
  pa.xp = xp;
  // k = 1: GEMM2 writes y itself (fused combine); dropped tokens are zeroed here
  const bool fuse_combine = s->k == 1;
  pa.slot = slot;
  pa.y_zero = fuse_combine ? y : nullptr;
  cudaError_t e = launch_permute(pa, sms, st, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "permute launch");
  if ((rc = mark(ev, 3, st)) != MOE_OK) return rc;

  float* part = part_ptr(ws, s);
  int splits = 1;
  if ((rc = enqueue_expert_gemms(s, s->E, xp, w1, w2, offsets, h, fuse_combine ? y : Y,
                                 fuse_combine, perm, weights, status_ptr(ws), st, pdl, pdl, ev, 4,
                                 5, part, &splits)) != MOE_OK)
    return rc;
  if (fuse_combine) return mark(ev, 6, st);  // no combine kernel: the combine window is empty

  CombineArgs ca;
  ca.Y = Y;
  ca.w = weights;
  ca.slot = slot;
  ca.T = s->T;
  ca.H = s->H;
  ca.k = s->k;
  ca.y = y;
  ca.part = splits > 1 ? part : nullptr;  // GEMM2 left fp32 partials per K split
  ca.splits = splits;
  ca.part_stride = (size_t)s->T * s->k * s->H;
  e = launch_combine(ca, st, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return mark(ev, 6, st);
}

// Status word and ticket to zero (a one-warp kernel; with pdl it starts
// early, like the kernels after it).
int clear_status(void* ws, cudaStream_t st, bool pdl = true) {
  cudaError_t e = launch_clear_status(static_cast<int*>(ws), st, pdl);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "status clear launch");
}

int empty_routing(const moe_shape* s, int32_t* counts, int32_t* offsets, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)s->E, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(s->E + 1), st);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaMemsetAsync(counts/offsets)");
}

// ------------------------------------------------- allocation-free scratch --
// Scratch of moe_expert_ffn_combine_noalloc: the status block, h and the
// expert outputs, laid out as in a caller workspace.  In host code this name
// is only a handle: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

void* g_noalloc_ptr[kMaxDevices];  // device address per device, set once (g_mu)

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace

// =================================================================== C ABI

extern "C" {

int moe_version(void) { return (1 << 16) | 0; }

const char* moe_last_error_string(void) { return g_err; }

int64_t moe_expert_capacity(const moe_shape* s) {
  if (check_shape(s, false) != MOE_OK) return -1;
  return capacity_of(s);
}

size_t moe_workspace_size(const moe_shape* s) {
  if (check_shape(s, true) != MOE_OK) return 0;
  return ws_bytes_for(s);
}

size_t moe_route_workspace_size(const moe_shape* s) {
  if (check_shape(s, false) != MOE_OK) return 0;
  return route_ws_bytes(s);
}

int moe_forward_plan(const moe_shape* s, int32_t* dispatch_in_router, int32_t* combine_in_gemm) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  if (!dispatch_in_router || !combine_in_gemm)
    return fail(MOE_ERR_INVALID_ARG, "dispatch_in_router / combine_in_gemm is null");
  *dispatch_in_router = route_small(s) || route_fused_shape(s) ? 1 : 0;
  *combine_in_gemm = s->k == 1 ? 1 : 0;
  return MOE_OK;
}

int moe_route_plan(const moe_shape* s, int32_t* tile_tokens, int32_t* splits) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  if (!tile_tokens || !splits) return fail(MOE_ERR_INVALID_ARG, "tile_tokens / splits is null");
  *tile_tokens = 0;
  *splits = 0;
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  FusedRoutePlan plan;
  if (route_fused_shape(s) && route_fused_pick(s->T, s->H, s->E, &plan)) {
    *tile_tokens = plan.tm;
    *splits = plan.splits;
  }
  return MOE_OK;
}

int moe_route(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* b_router,
              int32_t* ids, float* weights, int32_t* counts, int32_t* offsets, int32_t* perm,
              int32_t* slot, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  REQUIRE_PTR(ws);
  if (ws_bytes < route_ws_bytes(s))
    return fail(MOE_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed (moe_route_workspace_size)",
                ws_bytes, route_ws_bytes(s));
  REQUIRE_PTR(counts);
  REQUIRE_PTR(offsets);
  if (b_router && !aligned16(b_router)) return fail(MOE_ERR_INVALID_ARG, "b_router is not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if ((rc = clear_status(ws, st)) != MOE_OK) return rc;
  if (s->T == 0) return empty_routing(s, counts, offsets, st);
  REQUIRE_PTR(x);
  REQUIRE_PTR(w_router);
  REQUIRE_PTR(ids);
  REQUIRE_PTR(weights);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(slot);
  return enqueue_route(s, sms, x, w_router, b_router, ids, weights, counts, offsets, perm, slot, ws, st);
}

int moe_dispatch(const moe_shape* s, const int32_t* ids, int32_t* counts, int32_t* offsets,
                 int32_t* perm, int32_t* slot, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  REQUIRE_PTR(ws);
  if (ws_bytes < route_ws_bytes(s))
    return fail(MOE_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed (moe_route_workspace_size)",
                ws_bytes, route_ws_bytes(s));
  REQUIRE_PTR(counts);
  REQUIRE_PTR(offsets);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if ((rc = clear_status(ws, st)) != MOE_OK) return rc;
  if (s->T == 0) return empty_routing(s, counts, offsets, st);
  REQUIRE_PTR(ids);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(slot);
  const int cap = (int)capacity_of(s);
  HistArgs ha;
  ha.ids = ids;
  ha.T = s->T;
  ha.k = s->k;
  ha.E = s->E;
  ha.seg_tokens = kSegTokens;
  ha.capacity = cap;
  ha.hist = hist_ptr(ws);
  ha.counts = counts;
  ha.offsets = offsets;
  ha.ticket = ticket_ptr(ws);
  ha.scan_in_dispatch = dispatch_scans((s->T + kSegTokens - 1) / kSegTokens, s->E) ? 1 : 0;
  ha.status = status_ptr(ws);
  cudaError_t e = launch_histogram(ha, st, /*pdl=*/true);
  if (e != cudaSuccess) return cuda_fail(e, "histogram launch");
  DispatchArgs da;
  da.ids = ids;
  da.T = s->T;
  da.k = s->k;
  da.E = s->E;
  da.capacity = cap;
  da.seg_tokens = kSegTokens;
  da.scan = ha.scan_in_dispatch;
  da.base = hist_ptr(ws);
  da.counts = counts;
  da.offsets = offsets;
  da.perm = perm;
  da.slot = slot;
  da.status = status_ptr(ws);
  e = launch_dispatch(da, st, /*pdl=*/true);  // follows the histogram kernel
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "dispatch launch");
}

int moe_expert_ffn_combine(const moe_shape* s, const uint16_t* x, const uint16_t* w1,
                           const uint16_t* w2, const float* weights, const int32_t* offsets,
                           const int32_t* perm, const int32_t* slot, uint16_t* y, void* ws,
                           size_t ws_bytes, void* stream) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  REQUIRE_PTR(ws);
  if (ws_bytes < ws_bytes_for(s))
    return fail(MOE_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, ws_bytes_for(s));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if ((rc = clear_status(ws, st)) != MOE_OK) return rc;
  if (s->T == 0) return MOE_OK;
  REQUIRE_PTR(x);
  REQUIRE_PTR(w1);
  REQUIRE_PTR(w2);
  REQUIRE_PTR(weights);
  REQUIRE_PTR(offsets);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(slot);
  REQUIRE_PTR(y);
  return enqueue_ffn_combine(s, sms, x, w1, w2, weights, offsets, perm, slot, y, ws, st);
}

int moe_dispatch_rows(const moe_shape* s, const uint16_t* x, const int32_t* perm,
                      const int32_t* offsets, uint16_t* xp, void* stream) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if (s->T == 0) return MOE_OK;
  REQUIRE_PTR(x);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(offsets);
  REQUIRE_PTR(xp);
  PermuteArgs pa;
  pa.x = x;
  pa.perm = perm;
  pa.offsets = offsets;
  pa.T = s->T;
  pa.H = s->H;
  pa.k = s->k;
  pa.E = s->E;
  pa.xp = xp;
  pa.slot = nullptr;
  pa.y_zero = nullptr;
  cudaError_t e = launch_permute(pa, sms, st, /*pdl=*/false);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute launch");
}

int moe_expert_ffn(const moe_shape* s, int32_t n_segments, const uint16_t* xp, const uint16_t* w1,
                   const uint16_t* w2, const int32_t* seg_offsets, uint16_t* Y, void* ws,
                   size_t ws_bytes, void* stream) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  if (n_segments < 1 || n_segments > kMaxExperts)
    return fail(MOE_ERR_INVALID_ARG, "n_segments = %d, must be 1..%d", n_segments, kMaxExperts);
  REQUIRE_PTR(ws);
  if (ws_bytes < ws_bytes_for(s))
    return fail(MOE_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, ws_bytes_for(s));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if ((rc = clear_status(ws, st)) != MOE_OK) return rc;
  if (s->T == 0) return MOE_OK;
  REQUIRE_PTR(xp);
  REQUIRE_PTR(w1);
  REQUIRE_PTR(w2);
  REQUIRE_PTR(seg_offsets);
  REQUIRE_PTR(Y);
  return enqueue_expert_gemms(s, n_segments, xp, w1, w2, seg_offsets, h_ptr(ws, s), Y, false,
                              nullptr, nullptr, status_ptr(ws), st, true, true, nullptr, 0, 0);
}

int moe_combine(const moe_shape* s, const uint16_t* Y, const float* weights, const int32_t* slot,
                uint16_t* y, void* stream) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if (s->T == 0) return MOE_OK;
  REQUIRE_PTR(Y);
  REQUIRE_PTR(weights);
  REQUIRE_PTR(slot);
  REQUIRE_PTR(y);
  CombineArgs ca;
  ca.Y = Y;
  ca.w = weights;
  ca.slot = slot;
  ca.T = s->T;
  ca.H = s->H;
  ca.k = s->k;
  ca.y = y;
  ca.part = nullptr;
  ca.splits = 1;
  ca.part_stride = 0;
  cudaError_t e = launch_combine(ca, st, /*pdl=*/false);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

int moe_expert_ffn_combine_noalloc(const moe_shape* s, const uint16_t* x, const uint16_t* w1,
                                   const uint16_t* w2, const float* weights,
                                   const int32_t* offsets, const int32_t* perm,
                                   const int32_t* slot, uint16_t* y, void* stream) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  const size_t need = ws_bytes_for(s);
  if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES)
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_expert_ffn_combine_noalloc: T*k = %lld rows at H = %d, F = %d need %zu "
                "bytes of scratch; the built-in scratch holds %u (use moe_expert_ffn_combine "
                "with a workspace)",
                (long long)s->T * s->k, s->H, s->F, need, (unsigned)MOE_NOALLOC_SCRATCH_BYTES);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch)) != MOE_OK) return rc;
  if ((rc = clear_status(scratch, st)) != MOE_OK) return rc;  // starts at zero every call
  if (s->T == 0) return MOE_OK;
  REQUIRE_PTR(x);
  REQUIRE_PTR(w1);
  REQUIRE_PTR(w2);
  REQUIRE_PTR(weights);
  REQUIRE_PTR(offsets);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(slot);
  REQUIRE_PTR(y);
  return enqueue_ffn_combine(s, sms, x, w1, w2, weights, offsets, perm, slot, y, scratch, st);
}

int moe_forward(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                const float* b_router, const uint16_t* w1, const uint16_t* w2, uint16_t* y,
                int32_t* ids, float* weights, int32_t* counts, int32_t* offsets, int32_t* perm,
                int32_t* slot, void* ws, size_t ws_bytes, void* stream) {
  return moe_forward_profiled(s, x, w_router, b_router, w1, w2, y, ids, weights, counts, offsets,
                              perm, slot, ws, ws_bytes, stream, nullptr);
}

int moe_forward_profiled(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                         const float* b_router, const uint16_t* w1, const uint16_t* w2,
                         uint16_t* y, int32_t* ids, float* weights, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* slot, void* ws,
                         size_t ws_bytes, void* stream, void* const* events) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  REQUIRE_PTR(ws);
  if (ws_bytes < ws_bytes_for(s))
    return fail(MOE_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, ws_bytes_for(s));
  REQUIRE_PTR(counts);
  REQUIRE_PTR(offsets);
  if (b_router && !aligned16(b_router)) return fail(MOE_ERR_INVALID_ARG, "b_router is not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = device_setup(&sms)) != MOE_OK) return rc;
  if ((rc = clear_status(ws, st, events == nullptr)) != MOE_OK) return rc;
  if (s->T == 0) return empty_routing(s, counts, offsets, st);
  REQUIRE_PTR(x);
  REQUIRE_PTR(w_router);
  REQUIRE_PTR(w1);
  REQUIRE_PTR(w2);
  REQUIRE_PTR(y);
  REQUIRE_PTR(ids);
  REQUIRE_PTR(weights);
  REQUIRE_PTR(perm);
  REQUIRE_PTR(slot);
  rc = enqueue_route(s, sms, x, w_router, b_router, ids, weights, counts, offsets, perm, slot, ws, st,
                     events);
  if (rc != MOE_OK) return rc;
  return enqueue_ffn_combine(s, sms, x, w1, w2, weights, offsets, perm, slot, y, ws, st, events);
}

int moe_get_device_status(void* ws, void* stream, int32_t* status) {
  if (!ws || !status) return fail(MOE_ERR_INVALID_ARG, "ws/status is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  *status = v;
  if (v == 0) return MOE_OK;
  if (v & MOE_DEV_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a device wait timed out (status 0x%x)", v);
  return fail(MOE_ERR_DEVICE, "device status 0x%x", v);
}

int moe_noalloc_device_status(void* stream, int32_t* status) {
  if (!status) return fail(MOE_ERR_INVALID_ARG, "status is null");
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_get_device_status(scratch, stream, status);
}

int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, void* stream) {
  if (!ws || !aligned16(ws) || ws_bytes < MOE_WS_MIN_BYTES)
    return fail(MOE_ERR_INVALID_ARG, "workspace null, misaligned or too small");
  if (limit_ns < 1000ull || limit_ns > 10000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns %llu outside [1e3, 1e10]", (unsigned long long)limit_ns);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  int rc = device_setup(&sms);
  if (rc != MOE_OK) return rc;
  if ((rc = clear_status(ws, st)) != MOE_OK) return rc;
  cudaError_t e = launch_wait_selftest(status_ptr(ws), limit_ns, st);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"
