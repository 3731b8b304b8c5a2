// router.cu -- fused router: logits = x · W_router (+ bias) on the tensor
// cores, per-token TopK (ties to the lower expert index) and the softmax
// over the k selected logits, in one kernel; the logits never reach HBM.
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
//     accumulator (M = 128, N = E rounded up to 16) in TMEM;
//   * the K = H reduction is split across a cluster of S CTAs (S = 1..8) so
//     that ceil(T/128) x S CTAs stream x from HBM in parallel; each CTA
//     copies its fp32 partial from TMEM to shared memory and the cluster
//     reduces the partials through distributed shared memory in a fixed
//     rank order (deterministic);
//   * CTA rank s then owns 128/S token rows: one warp per token, lane l
//     holds experts l, l+32, ...; k rounds of a warp-shuffle argmax
//     ((value, index) pairs, larger value wins, equal values -> lower
//     index) give the ids in descending-logit order; the softmax over those
//     k logits uses fp32 expf.
#include <math.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int RBM = 128;
constexpr int RBK = 64;
constexpr int RSTAGES = 4;
constexpr int RTHREADS = 128;

struct RCtrl {
  uint64_t full[RSTAGES];
  uint64_t empty[RSTAGES];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int NB64>
struct RCfg {
  static constexpr int A_BYTES = RBM * RBK * 2;         // 16 KB
  static constexpr int B_CHUNK = RBK * 64 * 2;          // 8 KB
  static constexpr int B_BYTES = NB64 * B_CHUNK;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int PIPE = RSTAGES * STAGE;
  static constexpr int PITCH = NB64 * 64 + 4;           // floats per partial row
  static constexpr int PART = RBM * PITCH * 4;
  static constexpr int DATA = PIPE > PART ? PIPE : PART;
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

template <int NB64>
__global__ void __launch_bounds__(RTHREADS)
    router_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const RouterArgs a) {
  using C = RCfg<NB64>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + RSTAGES * C::A_BYTES;
  float* part = reinterpret_cast<float*>(smem);  // reuses the pipeline buffers afterwards
  RCtrl& c = *reinterpret_cast<RCtrl*>(smem + C::DATA);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.splits;
  const int s = (int)cluster_ctarank();
  const int m0 = blockIdx.y * RBM;
  const int KB = (a.H + RBK - 1) / RBK;
  const int kb0 = (int)(((long long)KB * s) / S);
  const int kb1 = (int)(((long long)KB * (s + 1)) / S);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RSTAGES; ++i) {
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
      if (++stage == RSTAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    for (int m = max(0, armed - RSTAGES); m < armed; ++m)
      rwait_drain(&c.full[m % RSTAGES], (uint32_t)((m / RSTAGES) & 1), a.wait_limit_ns, a.status);
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
      if (++stage == RSTAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    umma_commit(&c.done);  // fires once every MMA issued above has completed
  }
  __syncwarp();

  // ---- all warps: wait for the accumulator, dump it to shared memory
  int ok = 1;
  if (lane == 0) ok = rwait_drain(&c.done, 0, a.wait_limit_ns, a.status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncthreads();  // the producer's drain is complete too
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_after();
  const bool have = ok && nkb > 0 && c.abort_flag == 0;
  {
    const int row = warp * 32 + lane;
    float* dst = part + row * C::PITCH;
    const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16);
    for (int col = 0; col < a.npad; col += 16) {
      uint32_t v[16];
      tmem_ld_x16(tb + (uint32_t)col, v);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float4 f;
        f.x = have ? __uint_as_float(v[4 * g + 0]) : 0.f;
        f.y = have ? __uint_as_float(v[4 * g + 1]) : 0.f;
        f.z = have ? __uint_as_float(v[4 * g + 2]) : 0.f;
        f.w = have ? __uint_as_float(v[4 * g + 3]) : 0.f;
        *reinterpret_cast<float4*>(dst + col + 4 * g) = f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
  }

  // ---- cluster: partials of every rank are complete and visible
  cluster_sync_all();

  constexpr int NU = 2 * NB64;  // 32-expert groups per lane
  const int rows_per_cta = RBM / S;
  for (int ri = warp; ri < rows_per_cta; ri += RTHREADS / 32) {
    const int row = s * rows_per_cta + ri;
    const int t = m0 + row;
    if (t >= a.T) continue;  // warp-uniform
    const uint32_t lbase = smem_u32(part + row * C::PITCH);
    float v[NU];
    uint32_t taken = 0;  // bit u: expert lane + 32u unavailable
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int e = lane + 32 * u;
      v[u] = -INFINITY;
      if (e < a.E) {
        float sum = dsmem_ld_f32(dsmem_map(lbase + 4u * (uint32_t)e, 0));
        for (int r = 1; r < S; ++r) sum += dsmem_ld_f32(dsmem_map(lbase + 4u * (uint32_t)e, (uint32_t)r));
        if (a.bias) sum += __ldg(a.bias + e);
        v[u] = isnan(sum) ? -INFINITY : sum;
      } else {
        taken |= 1u << u;
      }
    }
    int my_id = 0;
    float my_val = 0.f;
    for (int j = 0; j < a.k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const int e = lane + 32 * u;
        if (!((taken >> u) & 1u) && (v[u] > bv || (v[u] == bv && e < be))) {
          bv = v[u];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_id = be;
        my_val = bv;
      }
    }
    // softmax over the k selected logits; column 0 holds the maximum
    const float mx = __shfl_sync(0xffffffffu, my_val, 0);
    float ex = lane < a.k ? expf(my_val - mx) : 0.f;
    float z = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane < a.k) {
      a.ids[(size_t)t * a.k + lane] = my_id;
      a.weights[(size_t)t * a.k + lane] = ex / z;
    }
  }

  // keep this CTA's partial alive until every rank has read it
  cluster_sync_all();
}

template <int NB64>
cudaError_t launch_nb(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a,
                      cudaStream_t st) {
  using C = RCfg<NB64>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.splits, (unsigned)((a.T + RBM - 1) / RBM), 1);
  cfg.blockDim = dim3(RTHREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_kernel<NB64>, tm_x, tm_w, a);
}

template <int NB64>
cudaError_t set_attr_nb() {
  return cudaFuncSetAttribute(router_kernel<NB64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)RCfg<NB64>::SMEM);
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
  cudaError_t e;
  if ((e = set_attr_nb<1>()) != cudaSuccess) return e;
  if ((e = set_attr_nb<2>()) != cudaSuccess) return e;
  if ((e = set_attr_nb<3>()) != cudaSuccess) return e;
  return set_attr_nb<4>();
}

cudaError_t launch_router(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a,
                          cudaStream_t st) {
  switch ((a.E + 63) / 64) {
    case 1: return launch_nb<1>(tm_x, tm_w, a, st);
    case 2: return launch_nb<2>(tm_x, tm_w, a, st);
    case 3: return launch_nb<3>(tm_x, tm_w, a, st);
    default: return launch_nb<4>(tm_x, tm_w, a, st);
  }
}

}  // namespace moe
