// dispatch_combine.cu -- token dispatch (stable counting sort by expert with
// a capacity clip) and the gate-weighted combine.
//
// Dispatch restates GatherTokensByExpert of "用Ascend C写一个MoE融合算子"
// (section "2. Dispatch + Expert + Combine 流水线", listing "Gather操作"):
// expert e's rows are its assignments in ascending (token, slot) order, each
// recorded with its original position (token_indices) and its top-k slot
// (token_weight_indices) -- here packed as perm[r] = t*k + j, with the
// inverse map slot[t][j].  Instead of one O(T*k) scan per expert, every
// assignment is ranked among the earlier assignments of its expert: per
// 128-token segment counts (from the router, or the histogram kernel) are
// scanned across segments, then one CTA per segment adds the in-segment
// rank -- the same order.  Assignments ranked at or beyond the capacity are
// dropped (token dropping, "CANN ops-transformer：MoE 路由算子的负载均衡策略",
// section "负载不均衡的根源"; capacity_factor of the article's section 4.3).
//
// Combine restates ScatterWithWeights (listing "Scatter + 加权":
// output(orig_pos, d) += weight * expert_out(i, d), accumulated over the
// token's k experts) as a gather: each token reads its kept rows, so no two
// threads write the same output and no atomics are needed; the sum is fp32
// in slot order j = 0..k-1.
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int DTHREADS = 1024;
constexpr int DWARPS = DTHREADS / 32;

// One CTA per segment of seg_tokens tokens (seg_tokens * k <= 1024
// assignments, one per thread).  An assignment's rank within its expert is
// the segment's exclusive base (all earlier segments' assignments to that
// expert, from the scan) + the assignments to the same expert earlier in
// this segment (warp match + per-warp counts scanned across warps).
__global__ void __launch_bounds__(DTHREADS, 1) dispatch_kernel(const DispatchArgs a) {
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_tot[kMaxExperts];
  __shared__ int s_wc[DWARPS * kMaxExperts];  // [warp][expert]
  extern __shared__ int s_cnt[];              // scan: [nseg][E] raw counts

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = a.E;
  const int seg = blockIdx.x;
  const int Tk = a.T * a.k;
  const int i0 = seg * a.seg_tokens * a.k;
  const int n = min(a.seg_tokens * a.k, Tk - i0);
  pdl_launch_dependents();
  pdl_wait();
  // this thread's assignment, loaded first so that its latency overlaps the
  // counts' below
  int e = tid < n ? __ldg(a.ids + i0 + tid) : -1;

  if (a.scan) {
    // this segment's bases (earlier segments' counts per expert) and the
    // totals, from all nseg x E counts: G lanes per expert (G | 32) split
    // the segments, then a butterfly sums them (integers: order-free)
    const int nseg = (int)gridDim.x;
    for (int i = tid; i < nseg * E; i += DTHREADS) s_cnt[i] = __ldcg(a.base + i);
    for (int idx = tid; idx < DWARPS * E; idx += DTHREADS) s_wc[idx] = 0;
    __syncthreads();
    int G = 32;
    while (G > 1 && G * E > DTHREADS) G >>= 1;
    const int ee = tid / G;
    const int part = tid % G;
    int pre = 0, tot = 0;
    if (ee < E)
      for (int sg = part; sg < nseg; sg += G) {
        const int v = s_cnt[sg * E + ee];
        tot += v;
        if (sg < seg) pre += v;
      }
    for (int off = G / 2; off > 0; off >>= 1) {
      pre += __shfl_xor_sync(0xffffffffu, pre, off);
      tot += __shfl_xor_sync(0xffffffffu, tot, off);
    }
    if (ee < E && part == 0) {
      s_base[ee] = pre;
      s_tot[ee] = tot;
    }
    __syncthreads();
    if (warp == 0) {
      // kept counts (capacity clip) and their exclusive scan: lane l holds
      // experts 8l .. 8l+7 (E <= 256)
      int loc[8];
      int sum = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e2 = lane * 8 + u;
        int n2 = 0;
        if (e2 < E) {
          n2 = s_tot[e2];
          if (a.capacity >= 0) n2 = min(n2, a.capacity);
        }
        loc[u] = n2;
        sum += n2;
      }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int run = incl - sum;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e2 = lane * 8 + u;
        if (e2 < E) {
          s_off[e2] = run;
          if (seg == 0) {
            a.offsets[e2] = run;
            a.counts[e2] = loc[u];
          }
        }
        run += loc[u];
      }
      if (lane == 31) {
        s_off[E] = incl;
        if (seg == 0) a.offsets[E] = incl;
      }
    }
  } else {
    for (int x = tid; x < E; x += DTHREADS) {
      s_base[x] = a.base[(size_t)seg * E + x];
      s_off[x] = a.offsets[x];
    }
    if (tid == 0) s_off[E] = a.offsets[E];
    for (int idx = tid; idx < DWARPS * E; idx += DTHREADS) s_wc[idx] = 0;
  }
  __syncthreads();

  if (e < 0 || e >= E) e = -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) s_wc[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int ee = tid; ee < E; ee += DTHREADS) {  // exclusive scan across warps
    int run = 0;
    for (int w = 0; w < DWARPS; ++w) {
      const int c = s_wc[w * E + ee];
      s_wc[w * E + ee] = run;
      run += c;
    }
  }
  __syncthreads();
  if (tid < n) {
    int sl = -1;
    if (e >= 0) {
      const int r = s_base[e] + s_wc[warp * E + e] + rank_w;
      if (a.capacity < 0 || r < a.capacity) {
        sl = s_off[e] + r;
        a.perm[sl] = i0 + tid;
      }
    }
    a.slot[i0 + tid] = sl;
  }
  // unused tail of perm, split across the segments
  const int N = s_off[E];
  const int per = (Tk - N + (int)gridDim.x - 1) / (int)gridDim.x;
  const int lo = N + seg * per;
  const int hi = min(Tk, lo + per);
  for (int i = lo + tid; i < hi; i += DTHREADS) a.perm[i] = -1;
}

constexpr int CTHREADS = 128;
constexpr int CCPT = 2;  // 16-byte column chunks per thread

// y[t, c..c+7] = sum_j w[t,j] * Y[slot[t,j], c..c+7] (fp32, j ascending).
// Grid (T, H / (CTHREADS * 8 * CCPT)): each thread takes CCPT 16-byte column
// chunks of one token (chunks CTHREADS * 8 columns apart, so every warp
// access is coalesced) and issues all k * CCPT loads before the sums: the
// kernel is latency-bound, so loads in flight per thread set its speed.
// KMAX >= k (1, 2, 4 or 8) sizes the per-thread arrays.
template <int KMAX>
__global__ void __launch_bounds__(CTHREADS) combine_kernel(const CombineArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int col0 = (blockIdx.y * CTHREADS * CCPT + threadIdx.x) * 8;
  if (col0 >= a.H) return;
  int r[KMAX];
  float w[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    r[j] = j < a.k ? __ldg(a.slot + (size_t)t * a.k + j) : -1;
    w[j] = r[j] >= 0 ? __ldg(a.w + (size_t)t * a.k + j) : 0.f;
  }
  uint4 v[KMAX][CCPT];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
#pragma unroll
    for (int c = 0; c < CCPT; ++c) {
      const int col = col0 + c * CTHREADS * 8;
      if (r[j] >= 0 && col < a.H)
        v[j][c] = __ldg(reinterpret_cast<const uint4*>(a.Y + (size_t)r[j] * a.H + col));
    }
#pragma unroll
  for (int c = 0; c < CCPT; ++c) {
    const int col = col0 + c * CTHREADS * 8;
    if (col >= a.H) break;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (r[j] < 0) continue;
      const float wt = w[j];
      acc[0] = fmaf(wt, bf16_lo(v[j][c].x), acc[0]);
      acc[1] = fmaf(wt, bf16_hi(v[j][c].x), acc[1]);
      acc[2] = fmaf(wt, bf16_lo(v[j][c].y), acc[2]);
      acc[3] = fmaf(wt, bf16_hi(v[j][c].y), acc[3]);
      acc[4] = fmaf(wt, bf16_lo(v[j][c].z), acc[4]);
      acc[5] = fmaf(wt, bf16_hi(v[j][c].z), acc[5]);
      acc[6] = fmaf(wt, bf16_lo(v[j][c].w), acc[6]);
      acc[7] = fmaf(wt, bf16_hi(v[j][c].w), acc[7]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(a.y + (size_t)t * a.H + col) = o;
  }
}

// The combine when the second expert GEMM ran split along K (small batches):
// a kept row's expert output is the sum of the splits' fp32 partials in
// split order, rounded to bf16 (as the unsplit GEMM rounds it), then
// weighted and summed over the token's slots in fp32 exactly as above.
__global__ void __launch_bounds__(CTHREADS) combine_partial_kernel(const CombineArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int col = (blockIdx.y * CTHREADS + threadIdx.x) * 8;
  if (col >= a.H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j = 0; j < a.k; ++j) {
    const int r = __ldg(a.slot + (size_t)t * a.k + j);
    if (r < 0) continue;
    const float wt = __ldg(a.w + (size_t)t * a.k + j);
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) {
      const float4* src =
          reinterpret_cast<const float4*>(a.part + sp * a.part_stride + (size_t)r * a.H + col);
      const float4 p0 = __ldg(src);
      const float4 p1 = __ldg(src + 1);
      v[0] += p0.x;
      v[1] += p0.y;
      v[2] += p0.z;
      v[3] += p0.w;
      v[4] += p1.x;
      v[5] += p1.y;
      v[6] += p1.z;
      v[7] += p1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t b = pack_bf16x2(v[i], v[i + 1]);  // the expert output in bf16
      acc[i] = fmaf(wt, bf16_lo(b), acc[i]);
      acc[i + 1] = fmaf(wt, bf16_hi(b), acc[i + 1]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(a.y + (size_t)t * a.H + col) = o;
}

// xp[r] = x[perm[r] / k] for the kept rows r < offsets[E]: the dispatch-
// ordered ("expanded") copy of the tokens that the expert GEMM reads with
// TMA.  One warp per row, 16-byte loads, eight in flight per lane; the copy
// is HBM/L2-bandwidth bound (2 H bytes read + 2 H bytes written per row).
constexpr int PTHREADS = 256;
__global__ void __launch_bounds__(PTHREADS) permute_kernel(const PermuteArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int rows = a.T * a.k;
  const int kept = min(max(__ldg(a.offsets + a.E), 0), rows);
  const int vec = a.H / 8;  // 16-byte chunks per row (H % 8 == 0)
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (PTHREADS / 32);
  for (int r = blockIdx.x * (PTHREADS / 32) + (threadIdx.x >> 5); r < kept; r += nw) {
    // perm is not re-validated by the caller-facing entry point: clamp so a
    // bad entry cannot address outside x
    const int tok = min(max(__ldg(a.perm + r) / a.k, 0), a.T - 1);
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)tok * a.H);
    uint4* dst = reinterpret_cast<uint4*>(a.xp + (size_t)r * a.H);
    int c = lane;
    for (; c + 224 < vec; c += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(src + c + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[c + 32 * u] = v[u];
    }
    for (; c < vec; c += 32) dst[c] = __ldg(src + c);
  }
  if (a.y_zero) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int t = blockIdx.x * (PTHREADS / 32) + (threadIdx.x >> 5); t < a.T; t += nw) {
      if (__ldg(a.slot + t) >= 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(a.y_zero + (size_t)t * a.H);
      for (int c = lane; c < vec; c += 32) dst[c] = z;
    }
  }
}

// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after limit_ns, records MOE_DEV_TIMEOUT and the kernel returns.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, status, limit_ns};
    (void)mbar_wait(&bar, 0, wc);
  }
  __syncthreads();
}

}  // namespace

// The router and GEMM kernels need the maximum shared-memory carveout; the
// small kernels between them ask for the same so the SMs are not
// reconfigured at every kernel boundary.
cudaError_t dispatch_combine_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kDispatchScanMaxCounts * sizeof(int)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  const void* combines[] = {(const void*)combine_kernel<1>, (const void*)combine_kernel<2>,
                           (const void*)combine_kernel<4>, (const void*)combine_kernel<8>,
                           (const void*)combine_partial_kernel};
  for (const void* f : combines)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

// Plain 1-D launch, optionally with programmatic serialization (pdl).
template <typename Kernel, typename Args>
cudaError_t launch_1d(Kernel k, dim3 grid, int threads, cudaStream_t st, bool pdl, const Args& a,
                      size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    set_pdl_attr(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, k, a);
}

// Zeroes a call's status block (status word, ticket and the fused route's
// counters: 256 ints) as a kernel: a memset node between two kernels costs
// several microseconds of serialisation, and a kernel can start early under
// programmatic dependent launch like every other kernel of the call.
__global__ void clear_status_kernel(int* p) {
  pdl_launch_dependents();
  pdl_wait();
  p[threadIdx.x] = 0;
}

cudaError_t launch_clear_status(int* p, cudaStream_t st, bool pdl) {
  return launch_1d(clear_status_kernel, dim3(1), 256, st, pdl, p);
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t st, bool pdl) {
  const int nseg = (a.T + a.seg_tokens - 1) / a.seg_tokens;
  const size_t smem = a.scan ? (size_t)nseg * a.E * sizeof(int) : 0;
  return launch_1d(dispatch_kernel, dim3((unsigned)nseg), DTHREADS, st, pdl, a, smem);
}

cudaError_t launch_permute(const PermuteArgs& a, int sms, cudaStream_t st, bool pdl) {
  const int64_t rows = (int64_t)a.T * a.k;
  const int64_t want = (rows + PTHREADS / 32 - 1) / (PTHREADS / 32);  // one row per warp
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * (2048 / PTHREADS);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  if (grid == 0) return cudaSuccess;
  return launch_1d(permute_kernel, dim3(grid), PTHREADS, st, pdl, a);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl) {
  if (a.part) {
    dim3 grid((unsigned)a.T, (unsigned)((a.H + CTHREADS * 8 - 1) / (CTHREADS * 8)), 1);
    return launch_1d(combine_partial_kernel, grid, CTHREADS, st, pdl, a);
  }
  const int cols_per_block = CTHREADS * 8 * CCPT;
  dim3 grid((unsigned)a.T, (unsigned)((a.H + cols_per_block - 1) / cols_per_block), 1);
  if (a.k <= 1) return launch_1d(combine_kernel<1>, grid, CTHREADS, st, pdl, a);
  if (a.k <= 2) return launch_1d(combine_kernel<2>, grid, CTHREADS, st, pdl, a);
  if (a.k <= 4) return launch_1d(combine_kernel<4>, grid, CTHREADS, st, pdl, a);
  return launch_1d(combine_kernel<8>, grid, CTHREADS, st, pdl, a);
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
