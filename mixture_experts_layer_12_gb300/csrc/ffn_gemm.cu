// ffn_gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores.
//
// Computes, for every expert e and every dispatch row r of e
// (offsets[e] <= r < offsets[e+1]), with xp[r] = x[perm[r] / k] the
// dispatch-ordered copy of the tokens:
//   GEMM1 (GELU):   h[r, :] = GELU(xp[r, :] · W1[e])
//   GEMM1 (SwiGLU): h[r, :] = SiLU(xp[r] · W_gate[e]) * (xp[r] · W_up[e]),
//                   W1[e] = [W_gate | W_up]  (gated experts)
//   GEMM2 (plain):  Y[r, :] = h[r, :] · W2[e]
// which are the two Mmad calls of the expert kernel in "用Ascend C写一个
// MoE融合算子", section "2. Dispatch + Expert + Combine 流水线" (listing
// "Expert计算": M = tokens of the expert, N = ffn_hidden_dim, K = hidden_dim,
// then N = hidden_dim, K = ffn_hidden_dim, with GELU in between).
//
// Design (sm_103a):
//   * CTA pairs (clusters of 2) run the 2-SM form of tcgen05.mma
//     (cta_group::2, M = 256, N = 256, K = 16): each CTA holds 128 rows of A
//     and 128 columns of B per stage, so a 256x256 tile costs each SM 32 KB
//     of operands per 64-wide K step instead of 48 KB for 128x256.
//   * persistent pairs, tiles ordered expert-major and row-block fastest,
//     so pairs working at the same time share the expert's weight columns
//     through L2 (the pages' expert-block / token-block tiling, made ragged:
//     an expert owns ceil(n_e / 256) row blocks); the tile list is built on
//     the device from `offsets`, with no host synchronisation.  An expert's
//     last row block with at most 128 rows runs as an M = 128 MMA (64 rows
//     per CTA), a column block with at most 128 valid columns as N = 128,
//     so short blocks do not pay for padding.
//   * warp 0: producer.  One thread per CTA issues the TMA loads of the
//     stage: the A tile (128 rows of xp or h, one box) and the weight tile
//     (two 64-column boxes of W[e], N contiguous = MN-major operand); both
//     CTAs' loads signal the leader CTA's stage barrier.  (Gathering A rows
//     from x inside the kernel with cp.async cost more tensor-pipe time than
//     the separate row copy that produces xp.)
//   * warp 1: TMEM (two 128x256 fp32 accumulators per CTA, 512 columns);
//     in the leader one thread issues the MMAs from a 6-stage ring (the
//     load / compute / store overlap of the article's section 2.2
//     pipeline) and its commits release the stage / publish the
//     accumulator in both CTAs.
//   * warps 2-5: epilogue, one per TMEM lane quadrant; tcgen05.ld of the
//     CTA's 128 accumulator rows, GELU(erf) for GEMM1 (erfc by Abramowitz &
//     Stegun 7.1.26), bf16 rounding and 16-byte stores; double-buffered
//     against the next tile's MMAs.
// Every mbarrier wait is bounded (MOE_DEV_TIMEOUT on expiry).
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = kGemmBM;         // rows per CTA
constexpr int PAIR_M = 2 * BM;      // rows per pair tile (UMMA M)
constexpr int BN = kGemmBN;         // columns per pair tile (UMMA N)
constexpr int BN_CTA = BN / 2;      // B columns each CTA holds
constexpr int BK = kGemmBK;
constexpr int STAGES = 6;
constexpr int ACC = 2;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB: 128 rows x 128 B
constexpr int B_CHUNK = BK * 64 * 2;   // 8 KB: one 64-column box, 64 K rows
constexpr int B_BYTES = (BN_CTA / 64) * B_CHUNK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int PRODUCER_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int EPI_WARP0 = MMA_WARP + 1;
constexpr int EPI_WARPS = 4;  // one per TMEM lane quadrant (warp % 4)
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int TMEM_COLS = ACC * BN;  // 512
constexpr uint16_t PAIR_MASK = 0x3;
constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, BN, /*a_mn=*/false, /*b_mn=*/true);
// An expert's last row block with at most 128 rows runs as an M = 128 pair
// MMA (64 rows per CTA): half the tensor work of a padded 256-row tile.  Its
// accumulator sits in TMEM columns 0..127 of the slot: lanes 0-63 hold the
// CTA's 64 rows for output columns 0..127, lanes 64-127 the same rows for
// columns 128..255 (read back per warp: rows 32 (q & 1) + lane, columns
// 128 (q >> 1) + c for lane quadrant q).
constexpr uint32_t IDESC_HALF = idesc_bf16_f32(PAIR_M / 2, BN, /*a_mn=*/false, /*b_mn=*/true);
// A 256-row tile whose column block holds at most 128 valid columns (the
// last one when N % 256 is 1..128) runs as an N = 128 MMA: each CTA loads
// one 64-column B box, and lanes = rows, TMEM columns 0..127 = the block's
// columns, as for N = 256.
constexpr uint32_t IDESC_NHALF = idesc_bf16_f32(PAIR_M, BN / 2, /*a_mn=*/false, /*b_mn=*/true);

static_assert(BK == 64, "one 128-byte swizzle atom of K per stage");
static_assert(BN_CTA % 64 == 0 && BN <= 256, "UMMA N");
static_assert(TMEM_COLS <= 512, "TMEM capacity");
static_assert(EPI_WARPS == 4, "one warp per TMEM lane quadrant (warp % 4), all 256 columns");

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[ACC];
  uint64_t tempty[ACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int n_tiles;
  int tile_start[kMaxExperts + 1];
  int mblocks[kMaxExperts];
  int row_off[kMaxExperts];
  int rows[kMaxExperts];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl);

struct Tile {
  int e, nb;
  int row0;        // this CTA's first dispatch row
  int rows_valid;  // rows of this CTA's part that belong to the expert (may be <= 0)
  bool half;       // M = 128 tile: 64 rows per CTA
  bool nhalf;      // N = 128 tile (256 rows): 64 B columns per CTA
};

// Tiles of one pair increase monotonically, so the expert cursor only moves
// forward; experts without rows own no tiles and are skipped.
// Tiles of one pair increase monotonically, so the expert cursor only moves
// forward; experts without rows own no tiles and are skipped.  Within an
// expert the row blocks run fastest, so a weight tile's readers follow one
// another while it is in L2.  allow_half: the expert's last row block runs
// as an M = 128 tile when it holds at most 128 rows (not for SwiGLU, whose
// gate and up columns of one output would land in different lane halves).
// (Moving those tiles to the end of the list, to fill the last wave, was
// slower: their weight tiles had left L2 by then.)
// n_cols: output columns (N); the last column block runs as an N = 128
// tile when it holds at most 128 of them (allow_half, 256-row tiles only).
__device__ __forceinline__ Tile decode_tile(const Ctrl& c, int tile, int& e, int rank,
                                            bool allow_half, int n_cols) {
  while (tile >= c.tile_start[e + 1]) ++e;
  const int local = tile - c.tile_start[e];
  const int mbs = c.mblocks[e];
  const int mb = local % mbs;
  const int base = mb * PAIR_M;  // the block's first row within the expert
  Tile t;
  t.e = e;
  t.nb = local / mbs;
  t.half = allow_half && mb == mbs - 1 && c.rows[e] - base <= PAIR_M / 2;
  t.nhalf = allow_half && !t.half && n_cols - t.nb * BN <= BN / 2;
  const int per = t.half ? BM / 2 : BM;  // rows per CTA
  t.row0 = c.row_off[e] + base + rank * per;
  t.rows_valid = min(per, c.rows[e] - base - rank * per);
  return t;
}

// Wait that ignores the abort flag (used to drain in-flight copies and
// MMAs before the CTA releases its shared memory and TMEM); still bounded.
__device__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status) {
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

// GELU(z) = 0.5 z (1 + erf(z / sqrt 2))  (the exact, erf form), with erfc
// by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: for x >= 0, erfc(x) = 1 - erf(x) = (a1 t + a2 t^2 + a3 t^3 +
// a4 t^4 + a5 t^5) exp(-x^2), t = 1 / (1 + p x), |error| <= 1.5e-7.
// Written as 0.5 z (2 - erfc(|x|)) for z >= 0 and 0.5 z erfc(|x|) for z < 0,
// so 1 + erf is never formed by cancellation: the relative error stays below
// 5e-5 for z >= -3 and below 0.2% (half a bf16 step) for z >= -5, where
// |GELU| > 1.4e-6.  It costs one fast division, one exponential and five
// FMAs; erff cost ~8% of GEMM1's time on the prefill workload.
__device__ __forceinline__ float gelu_erf(float z) {
  const float ax = fabsf(z) * 0.70710678118654752440f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f),
                       -0.284496736f),
               0.254829592f);
  const float c = poly * __expf(-ax * ax);  // erfc(|z| / sqrt 2)
  return 0.5f * z * (z >= 0.0f ? 2.0f - c : c);
}

// SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)); the fast exponential and
// division are far inside the bf16 rounding of h, and for z < -88 the
// denominator overflows to +inf and the quotient to 0 (the limit).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_a64, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + STAGES * STAGE_BYTES);
  constexpr bool SWIGLU = MODE == kGemmSwiGLU;
  constexpr bool COMBINE = MODE == kGemmCombineK1;  // k = 1: scale by the gate, write y[t]
  constexpr bool HALF = !SWIGLU;  // M = 128 tiles for short last row blocks
  // output columns per pair tile: SwiGLU pairs 128 gate with 128 up columns
  constexpr int BN_OUT = SWIGLU ? BN / 2 : BN;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();  // 0 = leader of the pair
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int NB = (p.N + BN_OUT - 1) / BN_OUT;
  const int KB = (p.K + BK - 1) / BK;
  pdl_launch_dependents();
  pdl_wait();  // offsets, A rows and the output buffers belong to earlier kernels

  // ---- tile schedule from the dispatch offsets (warp 0), barriers (warp 1)
  if (warp == 0) {
    int cnt[8];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane * 8 + u;
      cnt[u] = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e);
        const int n = max(__ldg(p.offsets + e + 1) - o0, 0);
        const int mbs = (n + PAIR_M - 1) / PAIR_M;
        c.row_off[e] = o0;
        c.rows[e] = n;
        c.mblocks[e] = mbs;
        cnt[u] = mbs * NB;
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
    // Only the leader's `full`, `tempty` and `drain` are used.  full: one
    // expect-tx arrival per CTA; tempty: every epilogue warp of both CTAs.
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&c.full[i], 2);
      mbar_init(&c.empty[i], 1);
    }
    for (int i = 0; i < ACC; ++i) {
      mbar_init(&c.tfull[i], 1);
      mbar_init(&c.tempty[i], 2 * EPI_WARPS);
    }
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // the leader's barriers exist before the peer signals them
  const int n_tiles = c.n_tiles;
  if (pair >= n_tiles) return;  // uniform across the pair: nothing allocated yet

  if (warp == MMA_WARP) {
    tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const WaitCtl wc{&c.abort_flag, p.status, p.wait_limit_ns};

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------ producer (one thread)
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      if (HALF) tma_prefetch_desc(&tm_a64);
      tma_prefetch_desc(&tm_b);
      const uint32_t full0 = dsmem_map(smem_u32(&c.full[0]), 0);  // leader's barriers
      // An expert with a single row block reads each weight tile once: those
      // tiles go to L2 as evict-first and its A rows as evict-last (the
      // weight stream of a decode step).  With several row blocks the pairs
      // on the other blocks read the same weight tile a little later, so
      // the loads keep the default policy.
      const uint64_t pol_first = l2_evict_first_policy();
      const uint64_t pol_last = l2_evict_last_policy();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // k-blocks issued (all tiles)
      int e = 0;
      bool ok = true;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
        const Tile t = decode_tile(c, tile, e, rank, HALF, p.N);
        // B columns of this CTA: its half of the 256-wide tile, or for
        // SwiGLU the gate (rank 0) / up (rank 1) columns of the same 128
        // outputs (W1 = [W_gate | W_up], so up starts at column N)
        const int bcol = SWIGLU  ? rank * p.N + t.nb * BN_OUT
                         : t.nhalf ? t.nb * BN + rank * (BN_CTA / 2)
                                   : t.nb * BN + rank * BN_CTA;
        const int n_boxes = t.nhalf ? 1 : BN_CTA / 64;  // 64-column B boxes per CTA
        const int we = t.e % p.E_w;  // the segment's expert weights
        const bool once = c.mblocks[t.e] == 1;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t full_cl = full0 + (uint32_t)(stage * sizeof(uint64_t));
          // an M = 128 tile reads 64 A rows per CTA (the first 8 KB of the
          // stage, laid out as the first 64 rows of a 128-row box)
          const CUtensorMap* ma = t.half ? &tm_a64 : &tm_a;
          mbar_arrive_expect_tx_cluster(full_cl, (t.half ? A_BYTES / 2 : A_BYTES) + n_boxes * B_CHUNK);
          // rows past the expert's end belong to the next expert (or lie past
          // the last row: zero-filled); they are computed but never stored
          if (once) {
            tma_load_2d_pair_hint(sA + stage * A_BYTES, ma, full_cl, kb * BK, t.row0, pol_last);
#pragma unroll
            for (int cb = 0; cb < n_boxes; ++cb)
              tma_load_3d_pair_hint(sB + stage * B_BYTES + cb * B_CHUNK, &tm_b, full_cl,
                                    bcol + cb * 64, kb * BK, we, pol_first);
          } else {
            tma_load_2d_pair(sA + stage * A_BYTES, ma, full_cl, kb * BK, t.row0);
#pragma unroll
            for (int cb = 0; cb < n_boxes; ++cb)
              tma_load_3d_pair(sB + stage * B_BYTES + cb * B_CHUNK, &tm_b, full_cl, bcol + cb * 64,
                               kb * BK, we);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain (leader): the TMA bytes of the last STAGES armed stages of both
      // CTAs must have landed before shared memory is released (returns at
      // once on the normal path, where the MMA consumed every stage).
      if (rank == 0) {
        for (int m = max(0, issued - STAGES); m < issued; ++m)
          mbar_wait_drain(&c.full[m % STAGES], (uint32_t)((m / STAGES) & 1), p.wait_limit_ns,
                          p.status);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int e = 0;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
        const Tile tt = decode_tile(c, tile, e, rank, HALF, p.N);
        const uint32_t idesc = tt.half ? IDESC_HALF : tt.nhalf ? IDESC_NHALF : IDESC;
        if (!mbar_wait(&c.tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            // A: K-major, advance 16 elements = 32 bytes inside the swizzle row.
            // B: MN-major, advance 16 K rows = two 1024-byte atoms.
            const uint64_t ad = sdesc_sw128(a0 + j * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + j * 2048, B_CHUNK, 1024);
            umma_bf16_pair(d, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
          }
          umma_commit_pair_mc(&c.empty[stage], PAIR_MASK);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&c.tfull[acc], PAIR_MASK);
        if (++acc == ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs issued by this thread have completed once `drain` fires
      umma_commit_pair_mc(&c.drain, 0x1);
      mbar_wait_drain(&c.drain, 0, p.wait_limit_ns, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;                    // TMEM lane quadrant this warp may read
    const uint32_t tempty0 = dsmem_map(smem_u32(&c.tempty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int e = 0;
    for (int tile = pair; tile < n_tiles; tile += n_pairs) {
      const Tile t = decode_tile(c, tile, e, rank, HALF, p.N);
      int got = 1;
      if (lane == 0) got = mbar_wait(&c.tfull[acc], acc_phase, wc);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      // M = 128 tile: this warp's lanes hold rows 32 (q & 1) + lane for the
      // output columns 128 (q >> 1) .. +127 (TMEM columns 0..127)
      const int row = t.half ? (q & 1) * 32 + lane : q * 32 + lane;
      const int col_base = t.half ? (q >> 1) * 128 : 0;
      const int n_chunks = t.half || t.nhalf ? 4 : 8;  // 32-column chunks
      bool row_ok = row < t.rows_valid;
      uint16_t* orow = p.out + (size_t)(row_ok ? t.row0 + row : 0) * (size_t)p.N;
      float gw = 1.0f;
      if constexpr (COMBINE) {
        // the token's only expert row: y[t] = w[t] * (h W2)[r], no Y round trip
        const int tok = row_ok ? __ldg(p.perm + t.row0 + row) : -1;
        row_ok = row_ok && tok >= 0 && tok < p.T;  // perm is not re-validated: never write outside y
        if (row_ok) {
          gw = __ldg(p.gate_w + tok);
          orow = p.out + (size_t)tok * (size_t)p.N;
        }
      }
      const uint32_t tbase = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if constexpr (SWIGLU) {
        // accumulator columns [0,128) = x W_gate, [128,256) = x W_up of the
        // same 128 outputs, 32 at a time
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          const int col = ch * 32;
          uint32_t gv[32], uv[32];
          tmem_ld_x32(tbase + (uint32_t)col, gv);
          tmem_ld_x32(tbase + (uint32_t)(BN_OUT + col), uv);
          tmem_ld_wait();
          const int gcol = t.nb * BN_OUT + col;
          if (row_ok) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              if (gcol + g * 8 + 8 <= p.N) {
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  f[i] = silu(__uint_as_float(gv[g * 8 + i])) * __uint_as_float(uv[g * 8 + i]);
                uint4 pk;
                pk.x = pack_bf16x2(f[0], f[1]);
                pk.y = pack_bf16x2(f[2], f[3]);
                pk.z = pack_bf16x2(f[4], f[5]);
                pk.w = pack_bf16x2(f[6], f[7]);
                *reinterpret_cast<uint4*>(orow + gcol + g * 8) = pk;
              }
            }
          }
        }
      } else {
#pragma unroll 1
      for (int ch = 0; ch < n_chunks; ++ch) {
        const int col = ch * 32;
        uint32_t v[32];
        tmem_ld_x32(tbase + (uint32_t)col, v);
        tmem_ld_wait();
        const int gcol = t.nb * BN + col_base + col;
        if (row_ok) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (gcol + g * 8 + 8 <= p.N) {
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                f[i] = __uint_as_float(v[g * 8 + i]);
                if constexpr (MODE == kGemmGelu) f[i] = gelu_erf(f[i]);
                if constexpr (COMBINE) f[i] *= gw;
              }
              uint4 pk;
              pk.x = pack_bf16x2(f[0], f[1]);
              pk.y = pack_bf16x2(f[2], f[3]);
              pk.z = pack_bf16x2(f[4], f[5]);
              pk.w = pack_bf16x2(f[6], f[7]);
              *reinterpret_cast<uint4*>(orow + gcol + g * 8) = pk;
            }
          }
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // Both CTAs finish all remote signalling and the leader's MMAs before TMEM
  // is released and before either CTA's shared memory goes away.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
  cluster_sync_all();
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_a64,
                        const GemmArgs& a,
                        int pairs, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (pdl) set_pdl_attr(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE>, tm_a, tm_b, tm_a64, a);
}

// Co-resident CTA pairs of the GEMM kernel on this device (one per TPC).
int max_pairs_cache[64];

cudaError_t query_max_pairs(int dev, int* out) {
  if (dev >= 0 && dev < 64 && max_pairs_cache[dev] > 0) {
    *out = max_pairs_cache[dev];
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<kGemmGelu>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (dev >= 0 && dev < 64) max_pairs_cache[dev] = n;
  *out = n;
  return cudaSuccess;
}

}  // namespace

size_t grouped_gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_grouped_gemm(int mode, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const CUtensorMap& tm_a64,
                                const GemmArgs& a, int max_tiles, cudaStream_t st, bool pdl) {
  if (max_tiles <= 0) return cudaSuccess;
  int dev = 0, pairs = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = query_max_pairs(dev, &pairs)) != cudaSuccess) return e;
  if (pairs > max_tiles) pairs = max_tiles;
  switch (mode) {
    case kGemmGelu: return launch_pair<kGemmGelu>(tm_a, tm_b, tm_a64, a, pairs, st, pdl);
    case kGemmSwiGLU: return launch_pair<kGemmSwiGLU>(tm_a, tm_b, tm_a64, a, pairs, st, pdl);
    case kGemmCombineK1: return launch_pair<kGemmCombineK1>(tm_a, tm_b, tm_a64, a, pairs, st, pdl);
    default: return launch_pair<kGemmPlain>(tm_a, tm_b, tm_a64, a, pairs, st, pdl);
  }
}

cudaError_t grouped_gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemmGelu>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemmSwiGLU>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemmCombineK1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemmPlain>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  return e;
}

}  // namespace moe
