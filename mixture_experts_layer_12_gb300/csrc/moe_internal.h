// moe_internal.h -- launch interfaces between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// Default limit of every bounded device wait (one second).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Token segments of the routing path: 128 tokens (one router tile).
constexpr int kSegTokens = 128;

// ---- router: logits (tcgen05, split-K over a thread-block cluster),
//      TopK and the top-k softmax, fused; logits stay on chip.  Also writes
//      each tile's per-expert counts to `hist`; the last tile to finish
//      scans them into counts / offsets and per-tile exclusive bases.
struct RouterArgs {
  int T, H, E, k;
  int npad;        // E rounded up to 16 (the MMA N)
  int tmem_cols;   // power of two >= max(32, npad)
  int splits;      // cluster size along K (1, 2, 4 or 8)
  int capacity;    // -1: unlimited
  int gating;      // MOE_GATE_*
  const float* bias;  // [E] or null
  int32_t* ids;       // [T, k]
  float* weights;     // [T, k]
  int32_t* hist;      // [ceil(T/128)][E] workspace
  int32_t* counts;    // [E]
  int32_t* offsets;   // [E+1]
  unsigned int* ticket;  // zero before the launch
  int scan_in_dispatch;  // 1: publish raw per-tile counts only (see dispatch_scans)
  int* status;
  uint64_t wait_limit_ns;
};
// Launches ceil(T/128) x splits CTAs in clusters of `splits`.
// tm_x: x [T, H] bf16, box {64, 128}, 128B swizzle.
// tm_w: w_router [H, ldw] bf16 (ldw = E rounded up to 8, zero past E),
// box {64, 64}, 128B swizzle.
cudaError_t launch_router(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a,
                          cudaStream_t st, bool pdl);
size_t router_smem_bytes(int E);

// ---- the whole route (router + dispatch) in one launch for batches of up
// to kFusedMaxTiles x 128 tokens (route_fused.cu): tiles of 64 or 128 tokens
// x S K splits, all resident at once; the S CTAs of a tile are one cluster
// and exchange their fp32 partial logits through distributed shared memory.
constexpr int kFusedMaxTiles = 128;   // T <= 16384 tokens
constexpr int kFusedMaxSplits = 8;    // K splits per tile (the cluster size)
constexpr int kFusedMaxCtas = 256;    // tiles x splits
struct FusedRouteArgs {
  int T, H, E, k;
  int npad;        // E rounded up to 16: MMA N and the partial's row pitch (floats)
  int ep;          // E rounded up to 16: row pitch of the per-CTA counts (bytes)
  int tmem_cols;   // power of two >= max(32, npad)
  int capacity;    // -1: unlimited
  int gating;      // MOE_GATE_*
  const float* bias;  // [E] or null
  int32_t* ids;       // [T, k]
  float* weights;     // [T, k]
  int32_t* counts;    // [E]
  int32_t* offsets;   // [E+1]
  int32_t* perm;      // [T*k]
  int32_t* slot;      // [T, k]
  uint8_t* grp_hist;  // workspace: [tiles * splits][ep] assignments per expert
  unsigned* grid_cnt; // zero before the launch
  int* status;
  uint64_t wait_limit_ns;
};
struct FusedRoutePlan {
  int tm;      // tokens per tile: 64 or 128
  int splits;  // K splits per tile = cluster size: 1, 2, 4 or 8
  int tiles;   // ceil(T / tm)
};
// The tile height and split that minimise the bytes each CTA streams, among
// those whose clusters all fit on the current device at once and with at
// most kFusedMaxCtas CTAs; false if none does (or before
// route_fused_set_attributes ran on the device).
bool route_fused_pick(int T, int H, int E, FusedRoutePlan* plan);
// tm_x: x [T, H] bf16, box {64, plan.tm}, 128B swizzle; tm_w as for
// launch_router.  Grid (splits, tiles), clusters of `splits`.
cudaError_t launch_route_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                               const FusedRouteArgs& a, const FusedRoutePlan& plan,
                               cudaStream_t st, bool pdl);

// ---- small-batch route (router + dispatch in one launch, CUDA cores):
// for T <= kSmallRouteTokens and E <= kSmallRouteExperts.
constexpr int kSmallRouteTokens = 128;
constexpr int kSmallRouteExperts = 64;
struct SmallRouteArgs {
  const uint16_t* x;  // [T, H] bf16
  const uint16_t* w;  // [H, ldw] bf16, columns past E zero
  int ldw;            // W_router row pitch in elements: E rounded up to 8
  const float* bias;  // [E] or null
  int T, H, E, k;
  int capacity;       // -1: unlimited
  int gating;         // MOE_GATE_*
  int32_t* ids;
  float* weights;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* slot;
  unsigned int* ticket;  // zero before the launch
};
cudaError_t launch_router_small(const SmallRouteArgs& a, cudaStream_t st, bool pdl);
// W_router [H, E] (E % 8 != 0) -> wp [H, ldw], ldw = E rounded up to 8,
// zero past E: the copy the route reads when the rows are not 16-byte
// aligned.
cudaError_t launch_pad_router_weights(const uint16_t* w, int H, int E, int ldw, uint16_t* wp,
                                      int sms, cudaStream_t st, bool pdl);
// Clusters of `splits` router CTAs that can be resident at once.
cudaError_t router_max_clusters(int E, int splits, int* out);

// ---- per-segment expert counts of caller-provided ids + the same scan.
struct HistArgs {
  const int32_t* ids;
  int T, k, E;
  int seg_tokens;
  int capacity;  // -1: unlimited
  int32_t* hist;
  int32_t* counts;
  int32_t* offsets;
  unsigned int* ticket;  // zero before the launch
  int scan_in_dispatch;  // 1: publish raw per-segment counts only (see dispatch_scans)
  int* status;
};
cudaError_t launch_histogram(const HistArgs& a, cudaStream_t st, bool pdl);

// ---- dispatch: one CTA per segment ranks its assignments within each
//      expert and scatters perm / slot (capacity clip applied).
// With scan = 1 (dispatch_scans: few segments) `base` holds the raw
// per-segment counts and every CTA derives its own bases and the expert
// offsets from them (CTA 0 also writes counts / offsets): the producer's
// last-CTA scan, a serial step between the two kernels, disappears.  With
// scan = 0 the producer's last CTA has already turned `base` into exclusive
// bases and written counts / offsets.
constexpr int kDispatchScanMaxCounts = 16384;  // nseg * E ints held in shared memory
inline bool dispatch_scans(int nseg, int E) {
  // every CTA reads all counts: nseg^2 * E reads in all, kept to 16 MB
  return (long long)nseg * E <= kDispatchScanMaxCounts &&
         (long long)nseg * nseg * E <= (1LL << 22);
}
struct DispatchArgs {
  const int32_t* ids;
  int T, k, E;
  int capacity;  // -1: unlimited
  int seg_tokens;
  int scan;
  const int32_t* base;  // [nseg][E]: raw counts (scan) or exclusive bases
  int32_t* counts;      // [E] (written when scan)
  int32_t* offsets;     // [E+1] (read, or written when scan)
  int32_t *perm, *slot;
  int* status;
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t st, bool pdl);
// The status block (256 ints at p) set to zero by a one-CTA kernel.
cudaError_t launch_clear_status(int* p, cudaStream_t st, bool pdl);

// ---- grouped expert GEMM (tcgen05 + TMA, persistent ragged scheduler).
struct GemmArgs {
  const int32_t* offsets;  // [E+1] row offsets of the E segments (device)
  int E;                   // row segments
  int E_w;                 // weight matrices: segment e uses W[e % E_w]
  int N;                   // output columns (SwiGLU: F; W1 then holds 2F columns)
  int K;                   // reduction length
  uint16_t* out;           // [rows, N] bf16, row r = dispatch row (kGemmCombineK1: y [T, N])
  const int32_t* perm;     // kGemmCombineK1: token of dispatch row r (k = 1: perm[r] = t)
  const float* gate_w;     // kGemmCombineK1: gate weight of token t
  int T;                   // kGemmCombineK1: tokens (rows of y)
  int splits;              // kGemmPartial: K splits (small kernel); 1 otherwise
  float* part;             // kGemmPartial: fp32 partial outputs, split-major
  size_t part_stride;      // kGemmPartial: elements between splits
  int* status;
  uint64_t wait_limit_ns;
};
// Both GEMMs read A rows in dispatch order through tm_a, box {64, 128}:
// GEMM1: tm_a = xp [T*k, H] (permuted tokens), tm_b = W1 [E, H, F] (or
//   [E, H, 2F] for SwiGLU), box {64, 64, 1}; GELU or SiLU(gate) * up.
// GEMM2: tm_a = h [T*k, F], tm_b = W2 [E, F, H] box {64, 64, 1}; no activation.
// Launches min(max_tiles, co-resident CTA pairs) persistent pairs
// (clusters of 2 CTAs); max_tiles bounds the number of 256x256 pair tiles.
constexpr int kGemmPlain = 0;   // GEMM2: no activation
constexpr int kGemmGelu = 1;    // GEMM1: GELU epilogue
constexpr int kGemmSwiGLU = 2;  // GEMM1: SiLU(gate) * up epilogue
constexpr int kGemmCombineK1 = 3;  // GEMM2 + combine for k = 1: y[perm[r]] = w * acc
constexpr int kGemmPartial = 4;    // small kernel only: split-K, fp32 part[split][r][:]
constexpr int kMaxKSplits = 4;
// pdl: launched with programmatic stream serialization.  Every kernel of
// this library executes griddepcontrol.wait before its first global-memory
// access, which waits for the whole predecessor grid (this library's or the
// caller's) to complete and its writes to become visible; the early launch
// overlaps only launch latency and shared-memory setup.
// tm_a: A [rows, K] bf16, box {64, 128}; tm_a64: the same tensor, box {64, 64}
// (the M = 128 tiles of short last row blocks).
cudaError_t launch_grouped_gemm(int mode, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const CUtensorMap& tm_a64, const GemmArgs& a, int max_tiles,
                                cudaStream_t st, bool pdl);
size_t grouped_gemm_smem_bytes();
constexpr int kGemmBM = 128;  // rows per CTA; a CTA pair covers 256
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;

// Small batches (at most kSmallGemmRows dispatch rows in all): the same
// GEMMs with the weights as the MMA's M operand and the tokens as its N
// (ffn_gemm_small.cu), modes kGemmGelu, kGemmPlain and kGemmCombineK1.
// tm_w: W [E, K, N] box {64, 64, 1}; tm_x: rows [T*k, K] box {64, 32}.
constexpr int kSmallGemmRows = 64;
cudaError_t launch_small_gemm(int mode, const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                              const GemmArgs& a, int max_tiles, cudaStream_t st, bool pdl);
// CTA pairs of the small kernel that are resident at once.
cudaError_t small_gemm_max_pairs(int* out);

// ---- row permutation (the expanded-x output of the dispatch step):
// xp[r] = x[perm[r] / k] for r < offsets[E]; rows past offsets[E] untouched.
struct PermuteArgs {
  const uint16_t* x;  // [T, H]
  const int32_t* perm;
  const int32_t* offsets;  // offsets[E] = number of kept rows (device)
  int T, H, k, E;
  uint16_t* xp;  // [T*k, H]
  // k = 1 with the combine fused into GEMM2: y rows of tokens whose only
  // slot was dropped (slot[t] < 0) are zeroed here; null otherwise
  const int32_t* slot;
  uint16_t* y_zero;
};
cudaError_t launch_permute(const PermuteArgs& a, int sms, cudaStream_t st, bool pdl);

// ---- combine: y[t] = sum_j w[t,j] * Y[slot[t,j]] (fp32), bf16 out.
struct CombineArgs {
  const uint16_t* Y;  // [rows, H]
  const float* w;     // [T, k]
  const int32_t* slot;
  int T, H, k;
  uint16_t* y;
  // when set: the expert outputs are the sum of `splits` fp32 partials
  // (part[s * part_stride + r * H + c]), rounded to bf16 before weighting
  const float* part;
  int splits;
  size_t part_stride;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl);

// ---- bounded-wait self test.
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st);

}  // namespace moe
