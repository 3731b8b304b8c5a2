// route_fused.cu -- the whole route in one launch that fills the GPU:
// router logits on the tensor cores, per-token TopK and gate weights, and
// the dispatch (histogram, scan, stable counting sort with the capacity
// clip), for batches of up to kFusedMaxTiles x 128 tokens.
//
// Follows "用Ascend C写一个MoE融合算子": section "1. Routing + Gating 合并"
// (x × W_router, TopK per sample, Softmax over the top-k scores only) and
// listing "Gather操作" of section "2. Dispatch + Expert + Combine 流水线"
// (each expert's rows are its assignments in ascending (token, slot) order);
// token dropping past the capacity from "CANN ops-transformer：MoE 路由算子的
// 负载均衡策略", section "负载不均衡的根源".
//
// Design (sm_103a).  A batch of `tiles` tiles of TM tokens (TM = 64 or 128)
// runs as tiles x S CTAs, one per SM, all resident at once; the S CTAs of a
// tile form one thread-block cluster (S = 1, 2, 4 or 8 K splits, chosen on
// the host so that every cluster fits in one wave):
//   1. each CTA streams its K slice of the tile's x rows and of W_router by
//      TMA (128-byte swizzle, a ring of up to 12 stages that fills shared
//      memory) into one tcgen05.mma accumulator of TM tokens x E experts in
//      TMEM (M = TM: a 64-token tile runs the M = 64 form);
//   2. it stages that fp32 partial in its own shared memory (the ring, idle
//      after the MMAs); after one cluster barrier, rank s -- the owner of
//      rows [TM s / S, TM (s+1) / S) of the tile -- reads those rows of the
//      other ranks' partials through distributed shared memory and sums
//      the S partials of each row in rank order (deterministic); the
//      partials never reach L2;
//   3. TopK and the gate weights of the owned tokens by groups of 8 lanes
//      (route_topk.cuh); the logits never reach HBM;
//   4. the dispatch: each CTA ranks its own assignments within each expert
//      (warp match, then a scan across warps), publishes its per-expert
//      counts as bytes, and arrives on the grid's counter; once every CTA
//      has arrived it reads all counts, takes the exclusive sum over the
//      CTAs before it (its base, in token order) and the totals (capacity
//      clip, exclusive scan = offsets), and writes slot / perm of its own
//      assignments -- the serial scan's order, with no second kernel.
// Every wait on the CTA's own pipeline (TMA ring, MMA completion) and on the
// grid counter is bounded; on expiry MOE_DEV_TIMEOUT is recorded.  A CTA
// whose pipeline wait expired still stages (zeros) and reaches the cluster
// barrier, which every CTA of the cluster therefore passes; no CTA exits
// before the other ranks of its tile are done reading its shared memory.
#include "route_topk.cuh"

namespace moe {
namespace {

constexpr int FBM = 128;  // the largest tile (tokens); the MMA's M is the tile height
constexpr int FBK = 64;
constexpr int FTHREADS = 256;
constexpr int FWARPS = FTHREADS / 32;
constexpr int FMAX_STAGES = 12;
constexpr int FSMEM_LIMIT = 232448;  // dynamic shared memory of one CTA (227 KB)

struct FCtrl {
  uint64_t full[FMAX_STAGES];
  uint64_t empty[FMAX_STAGES];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
  int go;
};

// Shared memory of the steps after the MMAs, behind the staged partial
// logits [TM][npad + 4] fp32 (both overlay the TMA ring).
struct FPost {
  int ids[FBM * kMaxTopK];          // the group's choices, token-major; -1 past T
  int lrank[FBM * kMaxTopK];        // rank within the expert inside this CTA
  int wc[FWARPS][kMaxExperts];      // per-warp counts, then their exclusive scan
  int run[kMaxExperts];             // this CTA's assignments per expert
  int pre[kMaxExperts];             // assignments of the CTAs before this one
  int tot[kMaxExperts];             // all assignments
  int off[kMaxExperts + 1];         // expert offsets (capacity-clipped scan)
  int red[2][FWARPS * 256];         // per-warp sums of the experts' counts
};

template <int NB64, int TM>
struct FCfg {
  static_assert(TM == 64 || TM == 128, "tile height");
  // A slot: the tile's TM rows of a 64-wide K block (the MMA's M = TM)
  static constexpr int A_BYTES = TM * FBK * 2;
  static constexpr int B_CHUNK = FBK * 64 * 2;  // 8 KB
  static constexpr int B_BYTES = NB64 * B_CHUNK;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int FIT = (int)((FSMEM_LIMIT - 1024 - sizeof(FCtrl)) / STAGE);
  static constexpr int STAGES = FIT < FMAX_STAGES ? FIT : FMAX_STAGES;
  static constexpr int PIPE = STAGES * STAGE;
  static constexpr size_t SMEM = 1024 + (size_t)PIPE + sizeof(FCtrl);
  static_assert(SMEM <= (size_t)FSMEM_LIMIT, "shared memory");
  // staged partial: TM rows of npad + 4 floats (16-byte rows, banks spread)
  static constexpr int STG_BYTES = TM * (NB64 * 64 + 4) * 4;
  static_assert(STG_BYTES % 16 == 0, "aligned post-MMA state");
  static_assert(STG_BYTES + sizeof(FPost) <= (size_t)PIPE, "post-MMA state fits in the ring");
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 only: arrive on `cnt` (after the CTA's global writes, ordered by
// the preceding __syncthreads and this fence) and wait until it reaches
// `target`, at most limit_ns.  Returns false (and records the timeout) if it
// did not.
__device__ bool arrive_and_wait(unsigned* cnt, unsigned target, uint64_t limit_ns, int* status) {
  __threadfence();
  atomicAdd(cnt, 1u);
  if (ld_acquire_gpu(cnt) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(cnt) >= target) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      record_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ bool fwait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status) {
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

template <int NB64, int TM>
__global__ void __launch_bounds__(FTHREADS, 1)
    route_fused_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_w, const FusedRouteArgs a) {
  using C = FCfg<NB64, TM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  float* stg = reinterpret_cast<float*>(smem);                // after the MMAs
  FPost& P = *reinterpret_cast<FPost*>(smem + C::STG_BYTES);  // after the MMAs
  FCtrl& c = *reinterpret_cast<FCtrl*>(smem + C::PIPE);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = (int)gridDim.x;  // = the cluster size
  const int s = (int)blockIdx.x;  // = the rank in the cluster
  const int tile = (int)blockIdx.y;
  const int G = S * (int)gridDim.y;
  const int grp = tile * S + s;  // this CTA's group of tokens, in token order
  const int m0 = tile * TM;
  const int KB = (a.H + FBK - 1) / FBK;
  const int kb0 = (int)(((long long)KB * s) / S);
  const int kb1 = (int)(((long long)KB * (s + 1)) / S);
  const int nkb = kb1 - kb0;
  const int R = TM / S;  // owned rows of the tile (S divides TM)
  const int r0 = R * s;
  pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&c.full[i], 1);
      mbar_init(&c.empty[i], 1);
    }
    mbar_init(&c.done, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // shared memory and TMEM only so far; global memory may still belong to
  // the predecessor grid
  pdl_wait();
  const uint32_t tmem = c.tmem_base;
  const WaitCtl wc{&c.abort_flag, a.status, a.wait_limit_ns};

  // ---- 1. partial logits [TM x npad] over this CTA's K slice
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    int stage = 0;
    uint32_t phase = 0;
    int armed = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&c.empty[stage], phase ^ 1u, wc)) break;
      mbar_arrive_expect_tx(&c.full[stage], C::STAGE);
      tma_load_2d(sA + stage * C::A_BYTES, &tm_x, &c.full[stage], kb * FBK, m0);
#pragma unroll
      for (int cb = 0; cb < NB64; ++cb)
        tma_load_2d(sB + stage * C::B_BYTES + cb * C::B_CHUNK, &tm_w, &c.full[stage], cb * 64,
                    kb * FBK);
      ++armed;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // the ring is reused below: every armed stage's bytes must have landed
    for (int m = max(0, armed - C::STAGES); m < armed; ++m)
      fwait_drain(&c.full[m % C::STAGES], (uint32_t)((m / C::STAGES) & 1), a.wait_limit_ns,
                  a.status);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(TM, a.npad, false, true);
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < nkb; ++i) {
      if (!mbar_wait(&c.full[stage], phase, wc)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
      const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
      for (int j = 0; j < FBK / 16; ++j) {
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
  int ok = 1;
  if (lane == 0) ok = fwait_drain(&c.done, 0, a.wait_limit_ns, a.status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  // the ring that TMA (async proxy) filled is reused by plain stores below
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_after();
  const bool have = ok && nkb > 0 && c.abort_flag == 0;

  // ---- 2. the partial of the tile's TM rows into this CTA's shared memory.
  // Warps w and w+4 read TMEM lanes 32 (w % 4) .. +31 (their lane quadrant)
  // and take alternate 16-column chunks, four loads in flight per wait.  The
  // accumulator of an M = 128 MMA holds row r in lane r; that of M = 64 holds
  // row r in lane 32 (r / 16) + r % 16 (lanes 16..31 of a quadrant unused).
  const int sp = a.npad + 4;  // staging row pitch (floats)
  const int v4 = a.npad / 4;  // float4 per row
  {
    const int q = warp & 3;
    const int h = warp >> 2;
    const int row = TM == 128 ? q * 32 + lane : q * 16 + lane;
    const bool holds = TM == 128 || lane < 16;
    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
    const int nch = a.npad / 16;
    for (int c0 = h; c0 < nch; c0 += 8) {
      uint32_t v[4][16];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + 2 * u < nch) tmem_ld_x16(tb + (uint32_t)((c0 + 2 * u) * 16), v[u]);
      tmem_ld_wait();
      if (holds) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (c0 + 2 * u < nch) {
            float4* d4 = reinterpret_cast<float4*>(stg + row * sp + (c0 + 2 * u) * 16);
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
              float4 f;
              f.x = have ? __uint_as_float(v[u][4 * g4 + 0]) : 0.f;
              f.y = have ? __uint_as_float(v[u][4 * g4 + 1]) : 0.f;
              f.z = have ? __uint_as_float(v[u][4 * g4 + 2]) : 0.f;
              f.w = have ? __uint_as_float(v[u][4 * g4 + 3]) : 0.f;
              d4[g4] = f;
            }
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
  cluster_sync_all();  // every rank of the tile has staged its partial

  // ---- 3a. owned rows: the S partials in rank order (the other ranks'
  // read from their shared memory through DSMEM, a warp reading whole rows;
  // all loads of an element issued before the sums), + bias, NaN -> -inf,
  // columns past E at -inf; written over the staged row (rows no other rank
  // reads)
  for (int idx = tid; idx < R * v4; idx += FTHREADS) {
    const int li = idx / v4;
    const int col = (idx - li * v4) * 4;
    const int row = r0 + li;
    float4* mine = reinterpret_cast<float4*>(stg + row * sp + col);
    const uint32_t la = smem_u32(mine);
    float4 p[kFusedMaxSplits];
#pragma unroll
    for (int r = 0; r < kFusedMaxSplits; ++r)
      if (r < S && r != s) p[r] = dsmem_ld_v4(dsmem_map(la, (uint32_t)r));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kFusedMaxSplits; ++r) {
      if (r < S) {
        const float4 v = r == s ? *mine : p[r];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
    float o[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (col + i < a.E) {
        float vv = o[i];
        if (a.bias) vv += __ldg(a.bias + col + i);
        o[i] = isnan(vv) ? -INFINITY : vv;
      } else {
        o[i] = -INFINITY;
      }
    }
    *mine = make_float4(o[0], o[1], o[2], o[3]);
  }
  // done reading the other ranks' shared memory; every exit below waits
  // until all ranks of the tile are done with this CTA's
  cluster_arrive();
  __syncthreads();

  // ---- 3b. TopK and the gate weights of the owned tokens, 8 lanes per token
  {
    constexpr int GS = kTopkGroup;
    constexpr int NCH = 2 * NB64;  // chunks per lane when E = 64 * NB64
    const int g = lane & (GS - 1);
    const unsigned gmask = 0xffu << (lane & ~(GS - 1));
    for (int li0 = 0; li0 < R; li0 += FTHREADS / GS) {
      const int li = li0 + tid / GS;
      if (li >= R) continue;  // uniform over the group
      const int t = m0 + r0 + li;
      if (t >= a.T) {
        if (g < a.k) P.ids[li * a.k + g] = -1;
        continue;
      }
      const float* lrow = stg + (r0 + li) * sp;
      float lv[NCH * 4];
      uint32_t taken = 0;
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int e0 = (g + cc * GS) * 4;
        if (e0 < a.npad) {
          const float4 v = *reinterpret_cast<const float4*>(lrow + e0);
          lv[cc * 4 + 0] = v.x;
          lv[cc * 4 + 1] = v.y;
          lv[cc * 4 + 2] = v.z;
          lv[cc * 4 + 3] = v.w;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (e0 + i >= a.E) taken |= 1u << (cc * 4 + i);  // past E: never selected
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) lv[cc * 4 + i] = -INFINITY;
          taken |= 0xfu << (cc * 4);
        }
      }
      int my_id;
      float my_w;
      topk_gate_group<NCH>(lv, taken, g, gmask, a.k, a.E, a.gating, my_id, my_w);
      if (g < a.k) {
        a.ids[(size_t)t * a.k + g] = my_id;
        a.weights[(size_t)t * a.k + g] = my_w;
        P.ids[li * a.k + g] = my_id;
      }
    }
  }
  __syncthreads();

  // ---- 4a. rank of each assignment within its expert inside this CTA, in
  // (token, slot) order: warp match, then an exclusive scan across warps
  const int E = a.E;
  const int n = R * a.k;
  for (int e = tid; e < E; e += FTHREADS) P.run[e] = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += FTHREADS) {
    for (int idx = tid; idx < FWARPS * E; idx += FTHREADS) P.wc[idx / E][idx % E] = 0;
    __syncthreads();
    const int i = c0 + tid;
    const int e = i < n ? P.ids[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int below = __popc(peers & lt);
    if (e >= 0 && below == 0) P.wc[warp][e] = __popc(peers);
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += FTHREADS) {
      int run = P.run[e2];
      for (int w = 0; w < FWARPS; ++w) {
        const int v = P.wc[w][e2];
        P.wc[w][e2] = run;
        run += v;
      }
      P.run[e2] = run;
    }
    __syncthreads();
    if (i < n) P.lrank[i] = e >= 0 ? P.wc[warp][e] + below : -1;
    __syncthreads();
  }

  // ---- 4b. publish this CTA's counts (bytes: at most 128 tokens each)
  const int EP = a.ep;  // E rounded up to 16
  const int NC = EP / 16;
  for (int cgi = tid; cgi < NC; cgi += FTHREADS) {
    uint32_t w4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int e = cgi * 16 + q * 4 + b;
        word |= (uint32_t)(e < E ? P.run[e] : 0) << (8 * b);
      }
      w4[q] = word;
    }
    *reinterpret_cast<uint4*>(a.grp_hist + (size_t)grp * EP + cgi * 16) =
        make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
  __syncthreads();
  if (tid == 0) c.go = arrive_and_wait(a.grid_cnt, (unsigned)G, a.wait_limit_ns, a.status) ? 1 : 0;
  __syncthreads();
  if (!c.go) {
    cluster_wait();
    return;
  }

  // ---- 4c. bases (CTAs before this one) and totals from every CTA's counts.
  // Chunks of 16 experts, NCP = NC rounded up to a power of two (<= 16):
  // thread t takes chunk t % NCP (idle past NC) of CTAs t / NCP + j (256 /
  // NCP) -- at most NCP <= 16 loads, all issued before the sums -- then a
  // butterfly over the lanes of its warp that hold the same chunk, and one
  // sum over the 8 warps.
  {
    constexpr int MAXL = 16;
    int NCP = 1;
    while (NCP < NC) NCP <<= 1;
    const int cgi = tid & (NCP - 1);
    const int gstep = FTHREADS / NCP;
    uint4 hv[MAXL];
#pragma unroll
    for (int j = 0; j < MAXL; ++j) {
      const int gg = tid / NCP + j * gstep;
      if (cgi < NC && gg < G)
        hv[j] = __ldcg(reinterpret_cast<const uint4*>(a.grp_hist + (size_t)gg * EP + cgi * 16));
    }
    // packed sums: word q of a chunk holds the counts of experts 4q..4q+3 as
    // bytes; its even bytes (experts 4q, 4q+2) and odd bytes (4q+1, 4q+3) go
    // to two words of 16-bit lanes, so one add sums two experts (a lane
    // reaches at most 256 CTAs x 128 = 32768)
    uint32_t pre[8], tot[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pre[i] = tot[i] = 0u;
#pragma unroll
    for (int j = 0; j < MAXL; ++j) {
      const int gg = tid / NCP + j * gstep;
      if (cgi < NC && gg < G) {
        const uint32_t w4[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
        const bool before = gg < grp;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t ev = w4[q] & 0x00ff00ffu;
          const uint32_t od = (w4[q] >> 8) & 0x00ff00ffu;
          tot[2 * q] += ev;
          tot[2 * q + 1] += od;
          if (before) {
            pre[2 * q] += ev;
            pre[2 * q + 1] += od;
          }
        }
      }
    }
    // lanes l and l ^ off hold the same chunk for off >= NCP (NCP | 32)
    for (int off = 16; off >= NCP; off >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pre[i] += __shfl_xor_sync(0xffffffffu, pre[i], off);
        tot[i] += __shfl_xor_sync(0xffffffffu, tot[i], off);
      }
    }
    if (lane < NCP && lane < NC) {
      // word 2q + h, 16-bit lane l: expert 4q + 2l + h of chunk `lane`
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int w = 2 * (i >> 2) + (i & 1);
        const int sh = 16 * ((i >> 1) & 1);
        P.red[0][warp * 256 + lane * 16 + i] = (int)((pre[w] >> sh) & 0xffffu);
        P.red[1][warp * 256 + lane * 16 + i] = (int)((tot[w] >> sh) & 0xffffu);
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += FTHREADS) {
    int p = 0, t2 = 0;
#pragma unroll
    for (int w = 0; w < FWARPS; ++w) {
      p += P.red[0][w * 256 + e];
      t2 += P.red[1][w * 256 + e];
    }
    P.pre[e] = p;
    P.tot[e] = t2;
  }
  __syncthreads();
  if (warp == 0) {
    // kept counts (capacity clip) and their exclusive scan: lane l holds
    // experts 8l .. 8l+7 (E <= 256)
    int loc[8];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane * 8 + u;
      int k2 = 0;
      if (e < E) {
        k2 = P.tot[e];
        if (a.capacity >= 0) k2 = min(k2, a.capacity);
      }
      loc[u] = k2;
      sum += k2;
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
        P.off[e] = run;
        if (grp == 0) {
          a.offsets[e] = run;
          a.counts[e] = loc[u];
        }
      }
      run += loc[u];
    }
    if (lane == 31) {
      P.off[E] = incl;
      if (grp == 0) a.offsets[E] = incl;
    }
  }
  __syncthreads();

  // ---- 4d. slot / perm of this CTA's assignments; the unused tail of perm
  // split across the CTAs
  for (int i = tid; i < n; i += FTHREADS) {
    const int t = m0 + r0 + i / a.k;
    if (t >= a.T) continue;
    const int e = P.ids[i];
    int sl = -1;
    if (e >= 0) {
      const int r = P.pre[e] + P.lrank[i];
      if (a.capacity < 0 || r < a.capacity) {
        sl = P.off[e] + r;
        a.perm[sl] = t * a.k + i % a.k;
      }
    }
    a.slot[(size_t)t * a.k + i % a.k] = sl;
  }
  const int Tk = a.T * a.k;
  const int Nk = P.off[E];
  const int per = (Tk - Nk + G - 1) / G;
  const int lo = Nk + grp * per;
  const int hi = min(Tk, lo + per);
  for (int i = lo + tid; i < hi; i += FTHREADS) a.perm[i] = -1;
  cluster_wait();
}

template <int NB64, int TM>
void fused_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int splits, int tiles,
                  cudaStream_t st, bool pdl) {
  cfg = {};
  cfg.gridDim = dim3((unsigned)splits, (unsigned)tiles, 1);
  cfg.blockDim = dim3(FTHREADS, 1, 1);
  cfg.dynamicSmemBytes = FCfg<NB64, TM>::SMEM;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (pdl) set_pdl_attr(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
}

template <int NB64, int TM>
cudaError_t launch_fused_nb(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            const FusedRouteArgs& a, int splits, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  fused_config<NB64, TM>(cfg, attr, splits, (a.T + TM - 1) / TM, st, pdl);
  return cudaLaunchKernelEx(&cfg, route_fused_kernel<NB64, TM>, tm_x, tm_w, a);
}

// cluster sizes 1, 2, 4, 8 (the portable limit)
constexpr int kSplitSizes[4] = {1, 2, 4, 8};

template <int NB64, int TM>
cudaError_t fused_setup_nb(int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(route_fused_kernel<NB64, TM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)FCfg<NB64, TM>::SMEM);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < 4; ++i) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fused_config<NB64, TM>(cfg, attr, kSplitSizes[i], 1, nullptr, false);
    clusters[i] = 0;
    // a size the device refuses is simply never planned
    if (cudaOccupancyMaxActiveClusters(&clusters[i], route_fused_kernel<NB64, TM>, &cfg) !=
        cudaSuccess) {
      clusters[i] = 0;
      (void)cudaGetLastError();
    }
  }
  return cudaSuccess;
}

// [device][E bucket][tile height 64, 128][cluster size 1, 2, 4, 8]
int g_fused_clusters[64][4][2][4];

}  // namespace

cudaError_t route_fused_set_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n[4][2][4] = {};
  if ((e = fused_setup_nb<1, 64>(n[0][0])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<1, 128>(n[0][1])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<2, 64>(n[1][0])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<2, 128>(n[1][1])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<3, 64>(n[2][0])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<3, 128>(n[2][1])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<4, 64>(n[3][0])) != cudaSuccess) return e;
  if ((e = fused_setup_nb<4, 128>(n[3][1])) != cudaSuccess) return e;
  if (dev >= 0 && dev < 64)
    for (int i = 0; i < 4; ++i)
      for (int j = 0; j < 2; ++j)
        for (int q = 0; q < 4; ++q) g_fused_clusters[dev][i][j][q] = n[i][j][q];
  return cudaSuccess;
}

bool route_fused_pick(int T, int H, int E, FusedRoutePlan* plan) {
  int dev = 0;
  if (T <= 0 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const int nb = (E + 63) / 64 - 1;
  const long long npad = (E + 15) / 16 * 16;
  const int KB = (H + FBK - 1) / FBK;
  long long best = -1;
  for (int j = 1; j >= 0; --j) {  // 128-token tiles first: ties keep them
    const int tm = j ? 128 : 64;
    const long long tiles = (T + tm - 1) / tm;
    for (int i = 0; i < 4; ++i) {
      const int S = kSplitSizes[i];
      if (S > KB || tiles * S > kFusedMaxCtas) continue;
      if (tiles > g_fused_clusters[dev][nb][j][i]) continue;  // not all in one wave
      // bytes each CTA takes in (its K blocks of x rows and of W_router)
      const long long cost = (long long)((KB + S - 1) / S) * (tm + npad);
      if (best < 0 || cost < best) {
        best = cost;
        plan->tm = tm;
        plan->splits = S;
        plan->tiles = (int)tiles;
      }
    }
  }
  return best >= 0;
}

cudaError_t launch_route_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                               const FusedRouteArgs& a, const FusedRoutePlan& plan,
                               cudaStream_t st, bool pdl) {
  const int nb = (a.E + 63) / 64;
  const int S = plan.splits;
  if (plan.tm == 64) {
    switch (nb) {
      case 1: return launch_fused_nb<1, 64>(tm_x, tm_w, a, S, st, pdl);
      case 2: return launch_fused_nb<2, 64>(tm_x, tm_w, a, S, st, pdl);
      case 3: return launch_fused_nb<3, 64>(tm_x, tm_w, a, S, st, pdl);
      default: return launch_fused_nb<4, 64>(tm_x, tm_w, a, S, st, pdl);
    }
  }
  switch (nb) {
    case 1: return launch_fused_nb<1, 128>(tm_x, tm_w, a, S, st, pdl);
    case 2: return launch_fused_nb<2, 128>(tm_x, tm_w, a, S, st, pdl);
    case 3: return launch_fused_nb<3, 128>(tm_x, tm_w, a, S, st, pdl);
    default: return launch_fused_nb<4, 128>(tm_x, tm_w, a, S, st, pdl);
  }
}

}  // namespace moe
