// router.cu -- fused router: logits = x · W_router (+ bias) on the tensor
// cores, per-token TopK (ties to the lower expert index) and the softmax
// over the k selected logits, in one kernel; the logits never reach HBM.
// The kernel also counts each 128-token tile's assignments per expert and
// the last tile to finish turns those counts into the dispatch offsets.
//
// Follows the router kernel of "用Ascend C写一个MoE融合算子", section
// "1. Routing + Gating 合并" (Mmad for x × W_router, TopK per sample, then
// Softmax over the top-k scores only), and the logit GEMM of
// "CANN ops-transformer：MoE 路由算子的负载均衡策略", section
// "Top-K 路由的并行化" (whose first-maximum '>' scan agrees with the
// lower-index tie rule).
//
// Design (sm_103a):
//   * a tile of 128 tokens x E experts (E <= 256) is one tcgen05.mma
//     accumulator (M = 128, N = E rounded up to 16) in TMEM, fed by a TMA
//     ring of up to 8 stages;
//   * the K = H reduction is split across a cluster of S CTAs (S = 1, 2, 4
//     or 8: the most whose clusters all fit in one wave) so
//     that ceil(T/128) x S CTAs stream x from HBM in parallel.  Each CTA
//     pushes the fp32 partial rows owned by rank r (rows [r*128/S, ...))
//     into rank r's shared memory with DSMEM stores; after one cluster
//     barrier every rank sums its rows' S partials locally in rank order
//     (deterministic);
//   * TopK: 8 lanes per token, each holding its share of the E logits
//     (4-expert chunks) in registers; k rounds of a local scan plus a
//     shuffle argmax over the 8 lanes.  Larger value first, equal values ->
//     lower index.  Gate
//     weights (fp32 expf): softmax over the k logits, or (the Softmax ->
//     Top-k order of section 2.1 of the article on CANN ops-transformer MoE
//     operators) softmax over all E then the k probabilities, with or
//     without renormalisation;
//   * per-tile expert counts go to the workspace (summed through DSMEM
//     atomics into rank 0).  For few tiles the dispatch kernel scans them;
//     otherwise the last tile to finish (an atomic ticket, no waiting) scans
//     them into counts / offsets (with the capacity clip) and per-tile
//     exclusive bases for the dispatch kernel.
#include <math.h>

#include "tc_common.cuh"

namespace moe {

// hist[seg][e] (assignment counts per 128-token segment) -> exclusive bases
// across segments, in place; counts[e] = min(total_e, cap); offsets =
// exclusive scan of counts.  Run by one whole CTA (blockDim.x threads) after
// every segment's counts are visible; `part` holds blockDim.x ints, `tot` E.
__device__ void scan_segment_counts(int32_t* hist, int nseg, int E, int cap, int32_t* counts,
                                    int32_t* offsets, int* part, int* tot) {
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int G = max(1, nt / E);       // threads per expert column
  const int cols = nt / G;            // columns per pass
  for (int e0 = 0; e0 < E; e0 += cols) {
    const int c = tid / G;
    const int g = tid % G;
    const int e = e0 + c;
    const bool act = c < cols && e < E;
    const int L = (nseg + G - 1) / G;
    const int s0 = min(nseg, g * L);
    const int s1 = min(nseg, s0 + L);
    int sum = 0;
    if (act)
      for (int sg = s0; sg < s1; ++sg) sum += __ldcg(hist + (size_t)sg * E + e);
    part[tid] = sum;
    __syncthreads();
    if (act) {
      int run = 0;
      for (int gg = 0; gg < g; ++gg) run += part[c * G + gg];
      for (int sg = s0; sg < s1; ++sg) {
        const int v = __ldcg(hist + (size_t)sg * E + e);
        hist[(size_t)sg * E + e] = run;
        run += v;
      }
      if (g == G - 1) tot[e] = run;
    }
    __syncthreads();
  }
  if (tid < 32) {
    const int lane = tid;
    int loc[8];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane * 8 + u;
      int n = 0;
      if (e < E) {
        n = tot[e];
        if (cap >= 0) n = min(n, cap);
      }
      loc[u] = n;
      sum += n;
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
      const int e = lane * 8 + u;
      if (e < E) {
        offsets[e] = run;
        counts[e] = loc[u];
      }
      run += loc[u];
    }
    if (lane == 31) offsets[E] = incl;
  }
}

namespace {

constexpr int RBM = 128;
constexpr int RBK = 64;
constexpr int RTHREADS = 256;  // warps 0-3: pipeline and TMEM; all 8: epilogue
constexpr int RMAX_STAGES = 8;

struct RCtrl {
  uint64_t full[RMAX_STAGES];
  uint64_t empty[RMAX_STAGES];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int hist[kMaxExperts];
  int part[RTHREADS];
  int tot[kMaxExperts];
};

template <int NB64>
struct RCfg {
  static constexpr int A_BYTES = RBM * RBK * 2;         // 16 KB
  static constexpr int B_CHUNK = RBK * 64 * 2;          // 8 KB
  static constexpr int B_BYTES = NB64 * B_CHUNK;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE) < RMAX_STAGES ? (196608 / STAGE) : RMAX_STAGES;
  static constexpr int PIPE = STAGES * STAGE;
  static constexpr int PITCH = NB64 * 64 + 4;           // floats per partial row
  static constexpr int RECV = RBM * PITCH * 4;          // S slots x 128/S rows = 128 rows
  static constexpr int DATA = PIPE > RECV ? PIPE : RECV;
  static constexpr size_t SMEM = 1024 + (size_t)DATA + sizeof(RCtrl);
};

__device__ bool rwait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      record_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// k-entry insertion list: larger value first, equal values keep the
// earlier (lower) expert; fully unrolled so it stays in registers.
struct TopK8 {
  float v[kMaxTopK];
  int id[kMaxTopK];
  int n;
  __device__ __forceinline__ void init() {
    n = 0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      v[j] = -INFINITY;
      id[j] = 0;
    }
  }
  // Inserts (val, e) before the first entry it beats strictly (or at the
  // end); from there every entry shifts down one slot unconditionally, so
  // displaced entries keep their order relative to equal values.
  __device__ __forceinline__ void push(float val, int e, int k) {
    float cv = val;
    int ci = e;
    bool shifting = false;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k && (shifting || j >= n || cv > v[j])) {
        shifting = true;
        const float tv = v[j];
        const int ti = id[j];
        v[j] = cv;
        id[j] = ci;
        cv = tv;
        ci = ti;
      }
    }
    n = min(n + 1, k);
  }
};

template <int NB64>
__global__ void __launch_bounds__(RTHREADS)
    router_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const RouterArgs a) {
  using C = RCfg<NB64>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  float* recv = reinterpret_cast<float*>(smem);  // reuses the pipeline buffers afterwards
  RCtrl& c = *reinterpret_cast<RCtrl*>(smem + C::DATA);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.splits;
  const int s = (int)cluster_ctarank();
  const int rpc = RBM / S;  // token rows owned by each rank
  const int m0 = blockIdx.y * RBM;
  const int KB = (a.H + RBK - 1) / RBK;
  const int kb0 = (int)(((long long)KB * s) / S);
  const int kb1 = (int)(((long long)KB * (s + 1)) / S);
  pdl_launch_dependents();  // the dispatch kernel may be scheduled now; it waits for us
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&c.full[i], 1);
      mbar_init(&c.empty[i], 1);
    }
    mbar_init(&c.done, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  for (int e = threadIdx.x; e < a.E; e += RTHREADS) c.hist[e] = 0;
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The setup above touched only shared memory and TMEM; from here on
  // global memory (x, the outputs) may belong to the predecessor grid.
  pdl_wait();
  const uint32_t tmem = c.tmem_base;
  const WaitCtl wc{&c.abort_flag, a.status, a.wait_limit_ns};

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: x tile [128 tokens x 64] and W_router [64 x E]
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    int stage = 0;
    uint32_t phase = 0;
    int armed = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&c.empty[stage], phase ^ 1u, wc)) break;
      mbar_arrive_expect_tx(&c.full[stage], C::STAGE);
      tma_load_2d(sA + stage * C::A_BYTES, &tm_x, &c.full[stage], kb * RBK, m0);
#pragma unroll
      for (int cb = 0; cb < NB64; ++cb)
        tma_load_2d(sB + stage * C::B_BYTES + cb * C::B_CHUNK, &tm_w, &c.full[stage], cb * 64,
                    kb * RBK);
      ++armed;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    for (int m = max(0, armed - C::STAGES); m < armed; ++m)
      rwait_drain(&c.full[m % C::STAGES], (uint32_t)((m / C::STAGES) & 1), a.wait_limit_ns,
                  a.status);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: logits[128 x npad] += x_tile · W_tile
    const uint32_t idesc = idesc_bf16_f32(RBM, a.npad, false, true);
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < nkb; ++i) {
      if (!mbar_wait(&c.full[stage], phase, wc)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
      const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
      for (int j = 0; j < RBK / 16; ++j) {
        const uint64_t ad = sdesc_sw128(a0 + j * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(b0 + j * 2048, C::B_CHUNK, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i | j) != 0 ? 1u : 0u);
      }
      umma_commit(&c.empty[stage]);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    umma_commit(&c.done);  // fires once every MMA issued above has completed
  }
  __syncwarp();

  // ---- all warps: accumulator complete; every rank's pipeline is idle
  int ok = 1;
  if (lane == 0) ok = rwait_drain(&c.done, 0, a.wait_limit_ns, a.status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_after();
  const bool have = ok && nkb > 0 && c.abort_flag == 0;
  cluster_sync_all();  // no rank still reads its pipeline buffers (now receive buffers)

  // ---- push this rank's partial of row `row` to the rank that owns it.
  // Warps w and w+4 read TMEM lanes 32(w%4) .. +31 (a warp's own lane
  // quadrant) and take alternate 16-column chunks, up to four loads in
  // flight per wait.
  {
    const int q = warp & 3;
    const int h = warp >> 2;
    const int row = q * 32 + lane;
    const int owner = row / rpc;
    const uint32_t dst =
        dsmem_map(smem_u32(recv + (size_t)(s * rpc + row % rpc) * C::PITCH), (uint32_t)owner);
    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
    const int nch = a.npad / 16;
    for (int c0 = h; c0 < nch; c0 += 8) {  // chunks c0, c0+2, c0+4, c0+6
      uint32_t v[4][16];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + 2 * u < nch) tmem_ld_x16(tb + (uint32_t)((c0 + 2 * u) * 16), v[u]);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + 2 * u < nch) {
          const int col = (c0 + 2 * u) * 16;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float f0 = have ? __uint_as_float(v[u][4 * g + 0]) : 0.f;
            const float f1 = have ? __uint_as_float(v[u][4 * g + 1]) : 0.f;
            const float f2 = have ? __uint_as_float(v[u][4 * g + 2]) : 0.f;
            const float f3 = have ? __uint_as_float(v[u][4 * g + 3]) : 0.f;
            dsmem_st_v4(dst + (uint32_t)((col + 4 * g) * 4), f0, f1, f2, f3);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
  }
  cluster_sync_all();  // every partial of this rank's rows has arrived

  // ---- per owned token: sum its S partial rows (ranks ascending, then +
  // bias; NaN -> -inf), TopK and the gate weights.  A group of 8 lanes takes
  // one token: lane g holds the 4-expert chunks g, g+8, g+16, ... in
  // registers.  Each of the k rounds scans the lane's untaken logits in
  // ascending expert order (strict '>' keeps the lower index on ties), a
  // 3-step shuffle argmax over the 8 lanes picks the round's expert (larger
  // value, then lower index) and its owner marks it taken.  All tokens of
  // the CTA are in flight at once.
  {
    constexpr int GS = 8;
    constexpr int NCH = 2 * NB64;  // chunks per lane when E = 64 * NB64
    constexpr int NV = NCH * 4;    // logits per lane
    static_assert(kMaxTopK <= GS, "lane g writes choice g");
    static_assert(NV <= 32, "taken mask");
    const int g = lane & (GS - 1);
    const unsigned gmask = 0xffu << (lane & ~(GS - 1));
    for (int li0 = 0; li0 < rpc; li0 += RTHREADS / GS) {
      const int li = li0 + (int)threadIdx.x / GS;
      const int t = m0 + s * rpc + li;
      if (li >= rpc || t >= a.T) continue;  // uniform over the group
      float lv[NV];
      uint32_t taken = 0;  // bit q: logit q unavailable (taken, or past E)
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int e0 = (g + cc * GS) * 4;
        if (e0 < a.E) {
          float4 acc = *reinterpret_cast<const float4*>(recv + (size_t)li * C::PITCH + e0);
          for (int r = 1; r < S; ++r) {
            const float4 p =
                *reinterpret_cast<const float4*>(recv + (size_t)(r * rpc + li) * C::PITCH + e0);
            acc.x += p.x;
            acc.y += p.y;
            acc.z += p.z;
            acc.w += p.w;
          }
          float v4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (e0 + i < a.E) {
              float v = v4[i];
              if (a.bias) v += __ldg(a.bias + e0 + i);
              lv[cc * 4 + i] = isnan(v) ? -INFINITY : v;
            } else {  // a zero-padded column of W_router: never selected
              lv[cc * 4 + i] = -INFINITY;
              taken |= 1u << (cc * 4 + i);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) lv[cc * 4 + i] = -INFINITY;
          taken |= 0xfu << (cc * 4);
        }
      }
      // k rounds (not unrolled: this code runs once per launch, cold in the
      // instruction cache, so its size is its cost); lane g keeps choice g
      int my_id = 0;
      float my_v = -INFINITY;
      float mx = 0.f;
#pragma unroll 1
      for (int j = 0; j < a.k; ++j) {
        float bv = -INFINITY;
        int bq = -1;
#pragma unroll
        for (int q = 0; q < NV; ++q)
          if (!((taken >> q) & 1u) && (bq < 0 || lv[q] > bv)) {
            bv = lv[q];
            bq = q;
          }
        // local index q = 4*cc + i  <->  expert 4*(g + 8*cc) + i
        int be = bq < 0 ? 0x7fffffff : ((g + (bq >> 2) * GS) << 2) + (bq & 3);
#pragma unroll
        for (int off = GS / 2; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(gmask, bv, off);
          const int oe = __shfl_xor_sync(gmask, be, off);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if (be != 0x7fffffff && ((be >> 2) & (GS - 1)) == g)
          taken |= 1u << (((be >> 5) << 2) | (be & 3));
        if (j == 0) mx = bv;
        if (j == g) {
          my_id = be;
          my_v = bv;
        }
      }
      // softmax over the k choices: lane g < k holds exp(l_g - l_0), the
      // group sums by butterfly
      float ex = g < a.k ? expf(my_v - mx) : 0.f;
      float z = ex;
#pragma unroll
      for (int off = GS / 2; off > 0; off >>= 1) z += __shfl_xor_sync(gmask, z, off);
      if (a.gating != MOE_GATE_TOPK_SOFTMAX) {
        // softmax over all E logits first: p_j = exp(l_j - max) / sum_e exp(l_e - max)
        float zall = 0.f;
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc)
          if ((g + cc * GS) * 4 < a.E)
#pragma unroll
            for (int i = 0; i < 4; ++i) zall += expf(lv[cc * 4 + i] - mx);
#pragma unroll
        for (int off = GS / 2; off > 0; off >>= 1) zall += __shfl_xor_sync(gmask, zall, off);
        ex = ex / zall;
        float zsel = ex;
#pragma unroll
        for (int off = GS / 2; off > 0; off >>= 1) zsel += __shfl_xor_sync(gmask, zsel, off);
        z = a.gating == MOE_GATE_SOFTMAX_TOPK ? 1.f : zsel;
      }
      const float my_w = ex / z;
      if (g < a.k) {
        a.ids[(size_t)t * a.k + g] = my_id;
        a.weights[(size_t)t * a.k + g] = my_w;
        atomicAdd(&c.hist[my_id], 1);
      }
    }
  }
  __syncthreads();

  // ---- this tile's expert counts: sum into rank 0, which publishes them
  if (S > 1) {
    const uint32_t h0 = dsmem_map(smem_u32(&c.hist[0]), 0);
    if (s != 0)
      for (int e = threadIdx.x; e < a.E; e += RTHREADS)
        if (c.hist[e]) atomicAdd_cluster_u32(h0 + 4u * (uint32_t)e, (uint32_t)c.hist[e]);
    cluster_sync_all();
  }
  if (s == 0) {
    for (int e = threadIdx.x; e < a.E; e += RTHREADS)
      a.hist[(size_t)blockIdx.y * a.E + e] = c.hist[e];
    if (a.scan_in_dispatch) return;  // the dispatch kernel scans (uniform over the CTA)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned prev = atomicAdd(a.ticket, 1u);
      c.is_last = (prev == gridDim.y - 1) ? 1 : 0;
    }
    __syncthreads();
    if (c.is_last) {
      __threadfence();
      scan_segment_counts(a.hist, (int)gridDim.y, a.E, a.capacity, a.counts, a.offsets, c.part,
                          c.tot);
    }
  }
}

template <int NB64>
cudaError_t launch_nb(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a,
                      cudaStream_t st, bool pdl) {
  using C = RCfg<NB64>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.splits, (unsigned)((a.T + RBM - 1) / RBM), 1);
  cfg.blockDim = dim3(RTHREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (pdl) set_pdl_attr(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, router_kernel<NB64>, tm_x, tm_w, a);
}

template <int NB64>
cudaError_t max_clusters_nb(int splits, int* out) {
  using C = RCfg<NB64>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, 1, 1);
  cfg.blockDim = dim3(RTHREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, router_kernel<NB64>, &cfg);
}

template <int NB64>
cudaError_t set_attr_nb() {
  return cudaFuncSetAttribute(router_kernel<NB64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)RCfg<NB64>::SMEM);
}

// ---- histogram of caller-provided ids (moe_dispatch): one CTA per
// 128-token segment, then the last CTA scans as the router does.
constexpr int HTHREADS = 1024;

__global__ void __launch_bounds__(HTHREADS) histogram_kernel(const HistArgs a) {
  __shared__ int s_hist[kMaxExperts];
  __shared__ int s_part[HTHREADS];
  __shared__ int s_tot[kMaxExperts];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();  // the predecessor grid (any) has completed
  for (int e = threadIdx.x; e < a.E; e += HTHREADS) s_hist[e] = 0;
  __syncthreads();
  const int n = min(a.seg_tokens, a.T - (int)blockIdx.x * a.seg_tokens) * a.k;
  const int32_t* ids = a.ids + (size_t)blockIdx.x * a.seg_tokens * a.k;
  bool bad = false;
  for (int i = threadIdx.x; i < n; i += HTHREADS) {
    const int e = __ldg(ids + i);
    if (e >= 0 && e < a.E)
      atomicAdd(&s_hist[e], 1);
    else
      bad = true;
  }
  if (bad) record_status(a.status, MOE_DEV_BAD_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += HTHREADS) a.hist[(size_t)blockIdx.x * a.E + e] = s_hist[e];
  if (a.scan_in_dispatch) return;  // the dispatch kernel scans
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (s_last) {
    __threadfence();
    scan_segment_counts(a.hist, (int)gridDim.x, a.E, a.capacity, a.counts, a.offsets, s_part,
                        s_tot);
  }
}

// ---- W_router [H, E] with E % 8 != 0: its rows are not 16-byte aligned,
// which TMA (and the 16-byte loads of the small-batch router) need, so the
// route reads a copy with ldw = E rounded up to 8 columns, zero-filled
// past E.  One thread per 8 columns of a row.
__global__ void __launch_bounds__(256) pad_router_weights_kernel(const uint16_t* __restrict__ w,
                                                                 int H, int E, int ldw,
                                                                 uint16_t* __restrict__ wp) {
  pdl_launch_dependents();
  pdl_wait();
  const int groups = ldw / 8;
  const long long n = (long long)H * groups;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int h = (int)(i / groups);
    const int e0 = (int)(i % groups) * 8;
    uint16_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = e0 + u < E ? w[(size_t)h * E + e0 + u] : (uint16_t)0;
    uint4 o;
    o.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
    o.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
    o.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
    o.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
    *reinterpret_cast<uint4*>(wp + (size_t)h * ldw + e0) = o;
  }
}

// ---- small batches (T <= kSmallRouteTokens, E <= 64): the whole route in
// one launch on the CUDA cores.  One CTA per token: each thread keeps
// partial logits for every expert over a strided slice of H (16-byte loads
// of x and of W_router's E-contiguous rows), then warps reduce by shuffle
// and the CTA sums the warps in order (a fixed order: deterministic).  The
// token's TopK and gate weights follow the tensor-core router exactly (same
// insertion list, gating modes, bias, NaN -> -inf).  The last CTA to finish
// (atomic ticket, nobody waits) then dispatches all T*k assignments: rank
// within the expert in (token, slot) order -- the serial scan of
// "Gather操作" -- the capacity clip, counts, offsets, slot and perm.
constexpr int SR_THREADS = 256;
constexpr int SR_WARPS = SR_THREADS / 32;
constexpr int SR_MAX_ASSIGN = kSmallRouteTokens * kMaxTopK;

template <int NE>  // experts rounded up to 8, 16, 32 or 64
__global__ void __launch_bounds__(SR_THREADS) router_small_kernel(const SmallRouteArgs a) {
  __shared__ float s_part[SR_WARPS][NE];
  __shared__ float s_logit[NE];
  __shared__ int s_last;
  __shared__ int s_pos[SR_MAX_ASSIGN];
  __shared__ int s_wc[SR_WARPS][NE];
  __shared__ int s_run[NE];
  __shared__ int s_off[NE + 1];
  pdl_launch_dependents();
  pdl_wait();  // the predecessor grid (any) has completed
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int t = blockIdx.x;
  const int E = a.E;
  const int Q = a.ldw / 8;  // 16-byte groups of experts in a W_router row

  // ---- logits of token t
  float acc[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) acc[e] = 0.f;
  const uint16_t* xr = a.x + (size_t)t * a.H;
  for (int h0 = tid * 8; h0 < a.H; h0 += SR_THREADS * 8) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + h0));
    const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                         bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint4* wrow = reinterpret_cast<const uint4*>(a.w + (size_t)(h0 + r) * a.ldw);
#pragma unroll
      for (int q = 0; q < NE / 8; ++q) {
        if (q < Q) {
          const uint4 wv = __ldg(wrow + q);
          acc[q * 8 + 0] = fmaf(xf[r], bf16_lo(wv.x), acc[q * 8 + 0]);
          acc[q * 8 + 1] = fmaf(xf[r], bf16_hi(wv.x), acc[q * 8 + 1]);
          acc[q * 8 + 2] = fmaf(xf[r], bf16_lo(wv.y), acc[q * 8 + 2]);
          acc[q * 8 + 3] = fmaf(xf[r], bf16_hi(wv.y), acc[q * 8 + 3]);
          acc[q * 8 + 4] = fmaf(xf[r], bf16_lo(wv.z), acc[q * 8 + 4]);
          acc[q * 8 + 5] = fmaf(xf[r], bf16_hi(wv.z), acc[q * 8 + 5]);
          acc[q * 8 + 6] = fmaf(xf[r], bf16_lo(wv.w), acc[q * 8 + 6]);
          acc[q * 8 + 7] = fmaf(xf[r], bf16_hi(wv.w), acc[q * 8 + 7]);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    float v = acc[e];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) s_part[warp][e] = v;
  }
  __syncthreads();
  if (tid < E) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < SR_WARPS; ++w) v += s_part[w][tid];
    if (a.bias) v += __ldg(a.bias + tid);
    s_logit[tid] = isnan(v) ? -INFINITY : v;
  }
  __syncthreads();

  // ---- TopK and gate weights (thread 0)
  if (tid == 0) {
    TopK8 tk;
    tk.init();
    for (int e = 0; e < E; ++e) tk.push(s_logit[e], e, a.k);
    const float mx = tk.v[0];
    float ex[kMaxTopK];
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      ex[j] = j < a.k ? expf(tk.v[j] - mx) : 0.f;
      z += ex[j];
    }
    if (a.gating != MOE_GATE_TOPK_SOFTMAX) {
      float zall = 0.f;
      for (int e = 0; e < E; ++e) zall += expf(s_logit[e] - mx);
      float zsel = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        ex[j] = ex[j] / zall;
        zsel += ex[j];
      }
      z = a.gating == MOE_GATE_SOFTMAX_TOPK ? 1.f : zsel;
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < a.k) {
        a.ids[(size_t)t * a.k + j] = tk.id[j];
        a.weights[(size_t)t * a.k + j] = ex[j] / z;
      }
    }
    __threadfence();
    s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;

  // ---- the last CTA: dispatch of all T*k assignments
  __threadfence();
  const int n = a.T * a.k;
  const unsigned lt = (1u << lane) - 1u;
  for (int e = tid; e < E; e += SR_THREADS) s_run[e] = 0;
  for (int c0 = 0; c0 < n; c0 += SR_THREADS) {
    for (int idx = tid; idx < SR_WARPS * NE; idx += SR_THREADS) (&s_wc[0][0])[idx] = 0;
    __syncthreads();
    const int i = c0 + tid;
    int e = i < n ? __ldcg(a.ids + i) : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    const int below = __popc(m & lt);  // same expert, earlier lane
    if (e >= 0 && below == 0) s_wc[warp][e] = __popc(m);
    __syncthreads();
    for (int ee = tid; ee < E; ee += SR_THREADS) {  // exclusive scan over warps
      int run = s_run[ee];
      for (int w = 0; w < SR_WARPS; ++w) {
        const int v = s_wc[w][ee];
        s_wc[w][ee] = run;
        run += v;
      }
      s_run[ee] = run;
    }
    __syncthreads();
    if (i < n) s_pos[i] = e >= 0 ? s_wc[warp][e] + below : -1;
    __syncthreads();
  }
  if (tid == 0) {  // counts after the capacity clip and their exclusive scan
    int run = 0;
    for (int e = 0; e < E; ++e) {
      const int kept = a.capacity >= 0 ? min(s_run[e], a.capacity) : s_run[e];
      a.counts[e] = kept;
      a.offsets[e] = run;
      s_off[e] = run;
      run += kept;
    }
    a.offsets[E] = run;
    s_off[E] = run;
  }
  __syncthreads();
  for (int i = tid; i < n; i += SR_THREADS) {
    const int e = __ldcg(a.ids + i);
    const int pos = s_pos[i];
    if (pos >= 0 && (a.capacity < 0 || pos < a.capacity)) {
      a.slot[i] = s_off[e] + pos;
      a.perm[s_off[e] + pos] = i;
    } else {
      a.slot[i] = -1;
    }
  }
  for (int i = s_off[E] + tid; i < n; i += SR_THREADS) a.perm[i] = -1;
}

}  // namespace

size_t router_smem_bytes(int E) {
  const int nb = (E + 63) / 64;
  switch (nb) {
    case 1: return RCfg<1>::SMEM;
    case 2: return RCfg<2>::SMEM;
    case 3: return RCfg<3>::SMEM;
    default: return RCfg<4>::SMEM;
  }
}

cudaError_t router_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(histogram_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if ((e = set_attr_nb<1>()) != cudaSuccess) return e;
  if ((e = set_attr_nb<2>()) != cudaSuccess) return e;
  if ((e = set_attr_nb<3>()) != cudaSuccess) return e;
  return set_attr_nb<4>();
}

// One CTA per token; with pdl, programmatic stream serialization.
template <typename Args>
cudaError_t launch_plain(void (*k)(Args), unsigned grid, int threads, cudaStream_t st, bool pdl,
                         const Args& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    set_pdl_attr(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_router_small(const SmallRouteArgs& a, cudaStream_t st, bool pdl) {
  const unsigned grid = (unsigned)a.T;
  if (a.E <= 8) return launch_plain(router_small_kernel<8>, grid, SR_THREADS, st, pdl, a);
  if (a.E <= 16) return launch_plain(router_small_kernel<16>, grid, SR_THREADS, st, pdl, a);
  if (a.E <= 32) return launch_plain(router_small_kernel<32>, grid, SR_THREADS, st, pdl, a);
  return launch_plain(router_small_kernel<64>, grid, SR_THREADS, st, pdl, a);
}

cudaError_t launch_router(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a,
                          cudaStream_t st, bool pdl) {
  switch ((a.E + 63) / 64) {
    case 1: return launch_nb<1>(tm_x, tm_w, a, st, pdl);
    case 2: return launch_nb<2>(tm_x, tm_w, a, st, pdl);
    case 3: return launch_nb<3>(tm_x, tm_w, a, st, pdl);
    default: return launch_nb<4>(tm_x, tm_w, a, st, pdl);
  }
}

// Co-resident clusters of `splits` router CTAs for E experts (cached per
// device, E bucket and cluster size).
cudaError_t router_max_clusters(int E, int splits, int* out) {
  static int cache[64][4][4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int nb = (E + 63) / 64 - 1;
  const int si = splits == 1 ? 0 : splits == 2 ? 1 : splits == 4 ? 2 : 3;
  if (dev >= 0 && dev < 64 && cache[dev][nb][si] > 0) {
    *out = cache[dev][nb][si];
    return cudaSuccess;
  }
  int n = 0;
  switch (nb + 1) {
    case 1: e = max_clusters_nb<1>(splits, &n); break;
    case 2: e = max_clusters_nb<2>(splits, &n); break;
    case 3: e = max_clusters_nb<3>(splits, &n); break;
    default: e = max_clusters_nb<4>(splits, &n); break;
  }
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev][nb][si] = n;
  *out = n;
  return cudaSuccess;
}

cudaError_t launch_pad_router_weights(const uint16_t* w, int H, int E, int ldw, uint16_t* wp,
                                      int sms, cudaStream_t st, bool pdl) {
  const long long n = (long long)H * (ldw / 8);
  long long blocks = (n + 255) / 256;
  const long long cap = (long long)(sms > 0 ? sms : 1) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    set_pdl_attr(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, pad_router_weights_kernel, w, H, E, ldw, wp);
}

cudaError_t launch_histogram(const HistArgs& a, cudaStream_t st, bool pdl) {
  const int nseg = (a.T + a.seg_tokens - 1) / a.seg_tokens;
  return launch_plain(histogram_kernel, (unsigned)nseg, HTHREADS, st, pdl, a);
}

}  // namespace moe
