// ffn_gemm_small.cu -- the expert GEMMs for small batches (at most
// kSmallGemmRows dispatch rows in all, e.g. a decode step), where every
// expert has only a few rows and the work is the stream of its weights.
//
// Same computation as ffn_gemm.cu (the two Mmad calls of the expert kernel
// in "用Ascend C写一个MoE融合算子", section "2. Dispatch + Expert + Combine
// 流水线", listing "Expert计算"), with the operands' roles swapped: the
// weights are the MMA's M operand and the tokens its N operand,
//   D[c, n] = sum_k W[e][k, c] * A[row0 + n, k],
// so a CTA pair's 256 x 64 tile is 256 output columns x 64 tokens.  A stage
// then holds 16 KB of weights and only 4 KB of token rows per CTA (instead
// of a 128-row A tile with a handful of real rows), and 10 stages fit: 160 KB
// of weights in flight per SM.  With T*k <= 64 every expert's rows fit one
// token tile, so each weight column is read exactly once.
//   * the weight tile is an MN-major A operand (two 64-column boxes, 128-byte
//     swizzle), the token tile a K-major B operand (32 rows per CTA);
//   * the accumulator comes out transposed: TMEM lane = output column,
//     register = token; each epilogue warp writes 32 consecutive columns
//     (64 bytes) of one token row per store.
// Warp roles, barriers and bounded waits as in ffn_gemm.cu.
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int SP_M = 256;                 // output columns per pair tile (MMA M)
constexpr int SM_CTA = SP_M / 2;          // output columns per CTA
constexpr int SN = kSmallGemmRows;        // tokens per pair tile (MMA N)
constexpr int SN_CTA = SN / 2;            // token rows each CTA holds
constexpr int SBK = 64;
constexpr int SA_CHUNK = SBK * 64 * 2;    // 8 KB: one 64-column weight box, 64 K rows
constexpr int SA_BYTES = (SM_CTA / 64) * SA_CHUNK;  // 16 KB
constexpr int SB_BYTES = SN_CTA * SBK * 2;          // 4 KB
constexpr int S_STAGE = SA_BYTES + SB_BYTES;
constexpr int S_STAGES = 10;
constexpr int S_ACC = 2;
constexpr int S_TMEM_COLS = S_ACC * SN;   // 128
constexpr int S_PRODUCER_WARP = 0;
constexpr int S_MMA_WARP = 1;
constexpr int S_EPI_WARP0 = 2;
constexpr int S_EPI_WARPS = 4;            // one per TMEM lane quadrant
constexpr int S_THREADS = 32 * (S_EPI_WARP0 + S_EPI_WARPS);
constexpr uint16_t S_PAIR_MASK = 0x3;
constexpr uint32_t S_IDESC = idesc_bf16_f32(SP_M, SN, /*a_mn=*/true, /*b_mn=*/false);

static_assert(SN % 32 == 0 && SN >= 32 && SN <= 256, "MMA N and the epilogue's 32-column loads");
static_assert(S_TMEM_COLS >= 32 && (S_TMEM_COLS & (S_TMEM_COLS - 1)) == 0, "TMEM allocation");
static_assert(SB_BYTES % 1024 == 0, "swizzle atoms of the token tile");

struct SCtrl {
  uint64_t full[S_STAGES];
  uint64_t empty[S_STAGES];
  uint64_t tfull[S_ACC];
  uint64_t tempty[S_ACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int n_tiles;
  int tile_start[kMaxExperts + 1];
  int row_off[kMaxExperts];
  int rows[kMaxExperts];
};

constexpr size_t S_SMEM = 1024 + (size_t)S_STAGES * S_STAGE + sizeof(SCtrl);

__device__ bool s_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status) {
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

// GELU(z) = 0.5 z (1 + erf(z / sqrt 2)) with erfc by Abramowitz & Stegun,
// formula 7.1.26 (|error| <= 1.5e-7), arranged so 1 + erf is never formed
// by cancellation (as in ffn_gemm.cu).
__device__ __forceinline__ float s_gelu(float z) {
  const float ax = fabsf(z) * 0.70710678118654752440f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f),
                       -0.284496736f),
               0.254829592f);
  const float c = poly * __expf(-ax * ax);
  return 0.5f * z * (z >= 0.0f ? 2.0f - c : c);
}

// Tiles of one pair increase monotonically: the segment cursor only moves
// forward.  Each segment with rows owns ceil(N / 256) column tiles, each in
// S K-splits (split fastest; the host keeps S <= KB so no range is empty);
// returns the column block, sets the split and its K range.
__device__ __forceinline__ int s_decode(const SCtrl& c, int tile, int& e, int S, int KB, int& sp,
                                        int& kb0, int& kb1) {
  while (tile >= c.tile_start[e + 1]) ++e;
  const int local = tile - c.tile_start[e];
  sp = local % S;
  kb0 = (int)(((long long)KB * sp) / S);
  kb1 = (int)(((long long)KB * (sp + 1)) / S);
  return local / S;
}

template <int MODE>
__global__ void __launch_bounds__(S_THREADS, 1)
    small_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_x, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                        // weight tiles
  uint8_t* sB = smem + S_STAGES * SA_BYTES;  // token tiles
  SCtrl& c = *reinterpret_cast<SCtrl*>(smem + S_STAGES * S_STAGE);
  constexpr bool COMBINE = MODE == kGemmCombineK1;
  constexpr bool PARTIAL = MODE == kGemmPartial;  // split-K: fp32 partial per split
  const int S = PARTIAL ? p.splits : 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int NB = (p.N + SP_M - 1) / SP_M;
  const int KB = (p.K + SBK - 1) / SBK;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {  // tile list: one token tile per segment, NB column tiles
    int cnt[8];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane * 8 + u;
      cnt[u] = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e);
        const int n = max(__ldg(p.offsets + e + 1) - o0, 0);
        c.row_off[e] = o0;
        c.rows[e] = min(n, SN);  // the host keeps every segment within SN rows
        cnt[u] = n > 0 ? NB * S : 0;
      }
      sum += cnt[u];
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
      if (e < p.E) c.tile_start[e] = run;
      run += cnt[u];
    }
    if (lane == 31) {
      c.tile_start[p.E] = incl;
      c.n_tiles = incl;
    }
  } else if (threadIdx.x == 32) {
    for (int i = 0; i < S_STAGES; ++i) {
      mbar_init(&c.full[i], 2);
      mbar_init(&c.empty[i], 1);
    }
    for (int i = 0; i < S_ACC; ++i) {
      mbar_init(&c.tfull[i], 1);
      mbar_init(&c.tempty[i], 2 * S_EPI_WARPS);
    }
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();
  const int n_tiles = c.n_tiles;
  if (pair >= n_tiles) return;  // uniform across the pair: nothing allocated yet

  if (warp == S_MMA_WARP) {
    tmem_alloc_pair(&c.tmem_base, S_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const WaitCtl wc{&c.abort_flag, p.status, p.wait_limit_ns};

  if (warp == S_PRODUCER_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
      const uint32_t full0 = dsmem_map(smem_u32(&c.full[0]), 0);
      const uint64_t pol_w = l2_evict_first_policy();  // each weight tile is read once
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int e = 0;
      bool ok = true;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
        int sp, kb0, kb1;
        const int nb = s_decode(c, tile, e, S, KB, sp, kb0, kb1);
        const int we = e % p.E_w;
        const int wcol = nb * SP_M + rank * SM_CTA;      // this CTA's 128 output columns
        const int trow = c.row_off[e] + rank * SN_CTA;   // this CTA's 32 token rows
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t full_cl = full0 + (uint32_t)(stage * sizeof(uint64_t));
          mbar_arrive_expect_tx_cluster(full_cl, S_STAGE);
#pragma unroll
          for (int cb = 0; cb < SM_CTA / 64; ++cb)
            tma_load_3d_pair_hint(sA + stage * SA_BYTES + cb * SA_CHUNK, &tm_w, full_cl,
                                  wcol + cb * 64, kb * SBK, we, pol_w);
          // token rows past the segment belong to the next one (or lie past
          // the last row: zero-filled); their columns are never stored
          tma_load_2d_pair(sB + stage * SB_BYTES, &tm_x, full_cl, kb * SBK, trow);
          ++issued;
          if (++stage == S_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (rank == 0) {
        for (int m = max(0, issued - S_STAGES); m < issued; ++m)
          s_wait_drain(&c.full[m % S_STAGES], (uint32_t)((m / S_STAGES) & 1), p.wait_limit_ns,
                       p.status);
      }
    }
    __syncwarp();
  } else if (warp == S_MMA_WARP) {
    if (rank == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int e = 0;
      bool ok = true;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
        int sp, kb0, kb1;
        s_decode(c, tile, e, S, KB, sp, kb0, kb1);
        if (!mbar_wait(&c.tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * SN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * SA_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * SB_BYTES);
#pragma unroll
          for (int j = 0; j < SBK / 16; ++j) {
            // weights: MN-major, 16 K rows = two 1024-byte atoms further;
            // tokens: K-major, 16 elements = 32 bytes into the swizzle row
            const uint64_t ad = sdesc_sw128(a0 + j * 2048, SA_CHUNK, 1024);
            const uint64_t bd = sdesc_sw128(b0 + j * 32, 16, 1024);
            umma_bf16_pair(d, ad, bd, S_IDESC, (kb != kb0 || j != 0) ? 1u : 0u);
          }
          umma_commit_pair_mc(&c.empty[stage], S_PAIR_MASK);
          if (++stage == S_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&c.tfull[acc], S_PAIR_MASK);
        if (++acc == S_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit_pair_mc(&c.drain, 0x1);
      s_wait_drain(&c.drain, 0, p.wait_limit_ns, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quadrant: output columns 32q .. 32q+31 of the CTA
    const uint32_t tempty0 = dsmem_map(smem_u32(&c.tempty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int e = 0;
    for (int tile = pair; tile < n_tiles; tile += n_pairs) {
      int sp, kb0, kb1;
      const int nb = s_decode(c, tile, e, S, KB, sp, kb0, kb1);
      int got = 1;
      if (lane == 0) got = mbar_wait(&c.tfull[acc], acc_phase, wc);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      const int col = nb * SP_M + rank * SM_CTA + q * 32 + lane;
      const uint32_t tbase = tmem + (uint32_t)(acc * SN) + ((uint32_t)(q * 32) << 16);
      const int nrows = c.rows[e];
      const int row0 = c.row_off[e];
#pragma unroll 1
      for (int n0 = 0; n0 < SN; n0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tbase + (uint32_t)n0, v);
        tmem_ld_wait();
        if (col < p.N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int n = n0 + i;
            if (n < nrows) {
              float f = __uint_as_float(v[i]);
              if constexpr (MODE == kGemmGelu) f = s_gelu(f);
              size_t orow = (size_t)(row0 + n);
              if constexpr (PARTIAL) {
                p.part[(size_t)sp * p.part_stride + orow * (size_t)p.N + col] = f;
                continue;
              }
              if constexpr (COMBINE) {
                // k = 1: the token's only expert row, scaled by its gate
                const int tok = __ldg(p.perm + row0 + n);
                if (tok < 0 || tok >= p.T) continue;  // perm is not re-validated
                f *= __ldg(p.gate_w + tok);
                orow = (size_t)tok;
              }
              p.out[orow * (size_t)p.N + col] = (uint16_t)(pack_bf16x2(f, 0.f) & 0xFFFFu);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
      if (++acc == S_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == S_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, S_TMEM_COLS);
  }
  cluster_sync_all();
}

template <int MODE>
cudaError_t s_launch(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const GemmArgs& a, int pairs,
                     cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(S_THREADS, 1, 1);
  cfg.dynamicSmemBytes = S_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (pdl) set_pdl_attr(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, small_gemm_kernel<MODE>, tm_w, tm_x, a);
}

int s_max_pairs_cache[64];

cudaError_t s_max_pairs(int dev, int* out) {
  if (dev >= 0 && dev < 64 && s_max_pairs_cache[dev] > 0) {
    *out = s_max_pairs_cache[dev];
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(S_THREADS, 1, 1);
  cfg.dynamicSmemBytes = S_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, small_gemm_kernel<kGemmGelu>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (dev >= 0 && dev < 64) s_max_pairs_cache[dev] = n;
  *out = n;
  return cudaSuccess;
}

}  // namespace

cudaError_t small_gemm_max_pairs(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return s_max_pairs(dev, out);
}

cudaError_t launch_small_gemm(int mode, const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                              const GemmArgs& a, int max_tiles, cudaStream_t st, bool pdl) {
  if (max_tiles <= 0) return cudaSuccess;
  int dev = 0, pairs = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = s_max_pairs(dev, &pairs)) != cudaSuccess) return e;
  if (pairs > max_tiles) pairs = max_tiles;
  switch (mode) {
    case kGemmGelu: return s_launch<kGemmGelu>(tm_w, tm_x, a, pairs, st, pdl);
    case kGemmCombineK1: return s_launch<kGemmCombineK1>(tm_w, tm_x, a, pairs, st, pdl);
    case kGemmPartial: return s_launch<kGemmPartial>(tm_w, tm_x, a, pairs, st, pdl);
    default: return s_launch<kGemmPlain>(tm_w, tm_x, a, pairs, st, pdl);
  }
}

cudaError_t small_gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(small_gemm_kernel<kGemmGelu>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_gemm_kernel<kGemmCombineK1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_gemm_kernel<kGemmPartial>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_gemm_kernel<kGemmPlain>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  return e;
}

}  // namespace moe
