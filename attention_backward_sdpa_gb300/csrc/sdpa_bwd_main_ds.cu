// sdpa_bwd_main_ds.cu -- SDPA backward main kernel for head dims whose dK
// accumulator leaves no tensor memory for dQ (MLA: D_qk = 192, D_v = 128; and
// D_qk = D_v = 256).
//
// Same computation as sdpa_bwd_main.cu (cuDNN frontend docs, "SDPA Backward
// (SM120)", "Main-kernel pipeline: KV-stationary, five chained GEMMs"; D_qk
// sizes Q/K/dQ/dK and D_v sizes V/O/dO/dV as in "Head-size support and tile
// configs"), with dQ always on the two-kernel route of the "Determinism"
// section: every bf16 dS^T tile is stored and sdpa_bwd_dq.cu forms
// dQ = scale * dS K. Per 64-row query tile t:
//   G1  S^T  = K Q^T       -> slot columns [0,64)
//       P^T  = exp2(...)    -> bf16 into slot columns [64,96)
//   G2  dP^T = V dO^T      -> slot columns [0,64), once S^T has been read
//       dS^T = P^T (dP^T - delta) -> shared memory -> workspace (bulk store)
//   G3  dV  += P^T dO       (A = P^T from tensor memory)
//   G4  dK  += dS^T Q
// Tensor memory (512 columns): two 96-column slots at 96s, dV at [192,192+D_v),
// dK at [192+D_v, 192+D_v+D_qk): 2*96 + 128 + 192 = 512 for MLA.
//
// D_qk = D_v = 256 (SPLIT = 2): dK and dV alone would need all 512 columns, so
// a work unit accumulates one half of their columns, [128h, 128h+128), and the
// two units of a key tile each compute S^T and dP^T over the full head dim
// (G1 and G2 are done twice: 7 GEMMs per pair instead of 5). G3 and G4 read
// the matching half of dO and Q. Unit h = 0 alone stores dS^T, writes dBias and
// zeroes the rows of empty key tiles. Its shared memory holds K and V (64 KiB
// each), the two dS^T buffers and one Q and one dO stage (32 KiB each).
//
// Warps: 0-3 even tiles (slot 0), 4-7 odd tiles (slot 1), 8 TMA producer,
// 9 G1 issuer and tensor-memory owner, 10 G3/G4 issuer, 11 G2 issuer, 12 dS^T store,
// 13-15 idle (they complete the fourth warpgroup for the register split).
// Shared memory: K [D_qk/64][128][128 B], V [D_v/64][128][128 B], Q and dO
// stage rings ([D/64][64][128 B]), dS^T x2 [128 keys][64 q], row statistics.
#include <cuda.h>
#include <cuda_bf16.h>

#include "bias.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

namespace ds_kernel {

constexpr int THREADS = 512;
// Register budgets move between warpgroups: launched with 128 registers per
// thread, the compute warpgroups grow to 160 while the other two shrink to 96;
// 128 threads x (160 + 160 + 96 + 96) = 65536 = 512 threads x 128.
constexpr uint32_t REGS_COMPUTE = 160, REGS_OTHER = 96;
static_assert(128 * (2 * REGS_COMPUTE + 2 * REGS_OTHER) <= THREADS * 128, "register split");
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;

enum : int {
  BAR_KV = 0,
  BAR_QFULL = 1,     // + Q stage (up to 3): Q tile and row statistics landed
  BAR_QEMPTY = 4,    // + Q stage: G4 done reading Q
  BAR_DOFULL = 7,    // + dO stage (2)
  BAR_DOEMPTY = 9,   // + dO stage, 2 arrivals: G2 and G3 done reading dO
  BAR_SFULL = 11,    // + slot: S^T in tensor memory
  BAR_PREADY = 13,   // + slot, 128 arrivals: P^T written
  BAR_DPFULL = 15,   // + slot: dP^T in tensor memory
  BAR_SFREE = 17,    // + slot: G3 done reading P^T
  BAR_DSREADY = 19,  // + slot, 128 arrivals: dS^T in shared memory
  BAR_DSFREE = 21,   // + slot: G4 done reading dS^T
  BAR_DSCOPIED = 23, // + slot: dS^T stored to the workspace
  BAR_MMADONE = 25,
  BAR_SREAD = 26,    // + slot, 128 arrivals: S^T in registers (G2 may overwrite it)
  BAR_DPREAD = 28,   // + slot, 128 arrivals: dP^T in registers (G1 may overwrite it)
  NUM_BARS = 30
};

template <int DQK, int DV, int SPLIT = 1>
struct Layout {
  static constexpr int BLK_KV = BN * 128;
  static constexpr int BLK_Q = BQ * 128;
  static constexpr int TILE_K = BN * DQK * 2;
  static constexpr int TILE_V = BN * DV * 2;
  static constexpr int TILE_Q = BQ * DQK * 2;
  static constexpr int TILE_DO = BQ * DV * 2;
  static constexpr int TILE_DS = BN * BQ * 2;
  static constexpr int ACC_K = DQK / SPLIT, ACC_V = DV / SPLIT;  // accumulated columns
  static constexpr int FIXED = TILE_K + TILE_V + 2 * TILE_DS;
  static constexpr bool fits(int nq, int ndo) {
    return FIXED + nq * (TILE_Q + QSTAT_FLOATS * 4) + ndo * TILE_DO + NUM_BARS * 8 + 64 <= 232448;
  }
  // Q (with the row statistics) is held from G1 to G4, the whole tile, while
  // dO is released by G3; so Q gets the deeper ring. Three Q stages cover the
  // ~2000-cycle load latency at the tensor pipe's tile rate, two would not.
  // At D = 256 one stage of each is all that fits.
  static constexpr int NDO = fits(1, 2) ? 2 : 1;
  static constexpr int NQ = fits(3, NDO) ? 3 : (fits(2, NDO) ? 2 : 1);
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_K;
  static constexpr int OFF_DS = OFF_V + TILE_V;
  static constexpr int OFF_Q = OFF_DS + 2 * TILE_DS;
  static constexpr int OFF_DO = OFF_Q + NQ * TILE_Q;
  static constexpr int OFF_QS = OFF_DO + NDO * TILE_DO;
  static constexpr int OFF_BAR = OFF_QS + NQ * QSTAT_FLOATS * 4;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr uint32_t COL_DV = 192, COL_DK = 192 + ACC_V;
  __host__ __device__ static constexpr uint32_t col_s(int slot) { return 96u * slot; }
  __host__ __device__ static constexpr uint32_t col_p(int slot) { return 96u * slot + 64u; }
  static_assert(COL_DK + ACC_K <= 512, "tensor memory budget");
  static_assert(ACC_K % 64 == 0 && ACC_V % 64 == 0, "whole 64-column blocks per unit");
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(BYTES > 116 * 1024, "one CTA per SM");
  static_assert(TILE_Q % 1024 == 0 && TILE_DO % 1024 == 0 && TILE_K % 1024 == 0, "alignment");
};

}  // namespace ds_kernel

// BIAS: the additive bias in the replay and the fp32 dBias output, as in the
// D_qk 64/128 kernel (bias.cuh): loads of the next tile's bias column issued
// right after dS, dS' stored as dBias, and the dBias blocks no CTA computes
// zeroed by an idle warp (or by an empty unit's whole CTA).
template <int DQK, int DV, bool BIAS, bool F16 = false, int SPLIT = 1>
__global__ void __launch_bounds__(ds_kernel::THREADS, 1)
    sdpa_bwd_main_ds(const __grid_constant__ MainMaps maps, const ChainParams p) {
  using namespace ds_kernel;
  using L = Layout<DQK, DV, SPLIT>;
  constexpr int NQ = L::NQ, NDO = L::NDO;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  uint8_t* sK = smem + L::OFF_K;
  uint8_t* sV = smem + L::OFF_V;
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sDO = smem + L::OFF_DO;
  uint8_t* sDS = smem + L::OFF_DS;
  float* sQS = reinterpret_cast<float*>(smem + L::OFF_QS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  {
    // A key tile that no query sees only has zero gradients. Its rows are
    // written by an idle warp of the head's other CTAs (or here, when the
    // batch row has no query or no key); leave before any setup.
    const int BH0 = p.B * p.Hq;
    const int u0 = (int)blockIdx.x / SPLIT;
    const int kt0 = u0 / BH0, bh0 = u0 % BH0, b0 = bh0 / p.Hq;
    int Lq0, Lk0, lo0, hi0;
    batch_lengths(p, b0, Lq0, Lk0);
    visited_query_tiles(kt0, Lq0, Lk0, p.causal, p.bottom_right, p.window_left, p.window_right, lo0,
                        hi0);
    if (hi0 < lo0) {
      if (blockIdx.x % SPLIT != 0) return;  // the first half-unit writes the zeros
      // gsz = 1: the partial set of a query head is its bh index.
      if (!row_has_visible_pair(Lq0, Lk0))
        zero_key_tile_rows(p, p.dk_ws ? (long long)bh0 : (long long)b0 * p.Hkv + (bh0 % p.Hq) / p.G,
                                    kt0 * BN);
      if (BIAS && p.dbias != nullptr && !p.dbias_red)
        zero_unvisited_dbias_blocks(p, b0, bh0, 1, kt0, lo0, hi0, threadIdx.x, blockDim.x);
      return;
    }
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NUM_BARS; ++i) {
      const bool threads128 = (i == BAR_PREADY || i == BAR_PREADY + 1 || i == BAR_DSREADY ||
                               i == BAR_DSREADY + 1 || i == BAR_SREAD || i == BAR_SREAD + 1 ||
                               i == BAR_DPREAD || i == BAR_DPREAD + 1);
      const bool two = (i == BAR_DOEMPTY || i == BAR_DOEMPTY + 1);
      mbar_init(&bars[i], threads128 ? 128 : (two ? 2 : 1));
    }
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.d_o);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The dQ kernel may become resident on the SMs this grid's finished units
  // leave (it waits for this grid before loading dS). Each thread releases it
  // only after the preprocess, which clears its ticket and zero tile, has
  // completed; the producer lane does so after issuing the K/V loads.
  if (!(warp == 8 && lane == 0)) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
  }

  const int BH = p.B * p.Hq;
  const int half = (int)blockIdx.x % SPLIT;  // accumulated column half (SPLIT = 2)
  const int unit = (int)blockIdx.x / SPLIT;
  const int kt = unit / BH;   // key tile major: the longest units first under causal masks
  const int bh = unit % BH;
  const int b = bh / p.Hq, h = bh % p.Hq, hk = h / p.G;
  const int k0 = kt * BN;
  int Lq, Lk;
  batch_lengths(p, b, Lq, Lk);
  const int diag = p.bottom_right ? Lk - Lq : 0;
  const int Rp = p.window_right > 0 ? p.window_right : 0;
  const bool has_window = p.window_left >= 0;
  int qt_lo, qt_hi;
  visited_query_tiles(kt, Lq, Lk, p.causal, p.bottom_right, p.window_left, p.window_right, qt_lo,
                      qt_hi);
  const int n = qt_hi - qt_lo + 1;

  constexpr uint32_t ID_G1 = idesc_io(128, BQ, false, false, F16);
  constexpr uint32_t ID_G2 = idesc_io(128, BQ, false, false, F16);
  constexpr uint32_t ID_G3 = idesc_io(128, L::ACC_V, false, true, F16);
  constexpr uint32_t ID_G4 = idesc_io(128, L::ACC_K, false, true, F16);
  // Byte offsets of this unit's column half in a dO and a Q stage.
  const uint32_t off_dov = (uint32_t)(half * (L::ACC_V / 64) * L::BLK_Q);
  const uint32_t off_qk = (uint32_t)(half * (L::ACC_K / 64) * L::BLK_Q);
  const bool lead = half == 0;  // stores dS^T, writes dBias and the zero rows
  constexpr uint64_t T_KMAJ = sdesc_sw128_template(16, 1024);
  constexpr uint64_t T_MN_Q = sdesc_sw128_template(L::BLK_Q, 1024);

  if (warp >= 8) {
  regs_decrease<ds_kernel::REGS_OTHER>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(&bars[BAR_KV], L::TILE_K + L::TILE_V);
      for (int blk = 0; blk < DQK / 64; ++blk)
        tma_load_3d(sK + blk * L::BLK_KV, &maps.k, &bars[BAR_KV], blk * 64, k0, b * p.Hkv + hk);
      for (int blk = 0; blk < DV / 64; ++blk)
        tma_load_3d(sV + blk * L::BLK_KV, &maps.v, &bars[BAR_KV], blk * 64, k0, b * p.Hkv + hk);
      pdl_wait_prior_grid();
      pdl_launch_dependents();
      // Q(t) waits for G4(t - NQ), dO(t) for G2 and G3 of tile t - NDO; G3(t - 2)
      // is issued after G4(t - 3), so issuing Q(t) first never delays dO(t).
      for (int t = 0; t < n; ++t) {
        const int sq = t % NQ, sd = t % NDO;
        const int qt = qt_hi - t;
        if (t >= NQ &&
            !mbar_wait(&bars[BAR_QEMPTY + sq], ((t / NQ) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
          break;
        uint64_t* qfull = &bars[BAR_QFULL + sq];
        mbar_arrive_expect_tx(qfull, L::TILE_Q + QSTAT_FLOATS * 4);
        for (int blk = 0; blk < DQK / 64; ++blk)
          tma_load_3d(sQ + sq * L::TILE_Q + blk * L::BLK_Q, &maps.q, qfull, blk * 64, qt * BQ, bh);
        const float* src = p.qstat + ((long long)bh * p.n_qt + qt) * QSTAT_FLOATS;
        if (in_bounds(p.status, src, QSTAT_FLOATS * 4, p.qstat, qstat_bytes(p)))
          bulk_load(sQS + sq * QSTAT_FLOATS, src, QSTAT_FLOATS * 4, qfull);
        else
          mbar_complete_tx(qfull, QSTAT_FLOATS * 4);
        if (t >= NDO &&
            !mbar_wait(&bars[BAR_DOEMPTY + sd], ((t / NDO) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
          break;
        uint64_t* dofull = &bars[BAR_DOFULL + sd];
        mbar_arrive_expect_tx(dofull, L::TILE_DO);
        for (int blk = 0; blk < DV / 64; ++blk)
          tma_load_3d(sDO + sd * L::TILE_DO + blk * L::BLK_Q, &maps.d_o, dofull, blk * 64, qt * BQ, bh);
      }
    }
  } else if (warp >= 9 && warp <= 11) {
    // ------------------------------------------------------------ MMA issuers
    // A tcgen05.mma costs its issuing thread about 120 cycles, more than these
    // MMAs take on the tensor core, so three warps issue: 9 G1, 11 G2, 10 G3/G4.
    pdl_wait_prior_grid();
    const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
    bool ok = n > 0 && mbar_wait(&bars[BAR_KV], 0, abort_flag, WAIT_LIMIT_NS);
    if (warp == 9) {
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1, st = t % NQ, j = t >> 1;
        if (!mbar_wait(&bars[BAR_QFULL + st], (t / NQ) & 1, abort_flag, WAIT_LIMIT_NS)) break;
        // Slot columns [0,64) hold dP^T of tile t-2 until the warpgroup has it
        // in registers.
        if (t >= 2 && !mbar_wait(&bars[BAR_DPREAD + s], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS))
          break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          const uint32_t aQ = smem_u32(sQ + st * L::TILE_Q);
#pragma unroll
          for (int k = 0; k < DQK / 16; ++k) {
            const uint32_t kk = (k >> 2) * L::BLK_KV + (k & 3) * 32;
            const uint32_t kq = (k >> 2) * L::BLK_Q + (k & 3) * 32;
            mma_ss(tmem + L::col_s(s), sdesc_at(T_KMAJ, aK + kk), sdesc_at(T_KMAJ, aQ + kq), ID_G1,
                   k > 0);
          }
          mma_commit(&bars[BAR_SFULL + s]);
        }
        __syncwarp();
      }
    } else if (warp == 11) {
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1, st = t % NDO, j = t >> 1;
        if (!mbar_wait(&bars[BAR_DOFULL + st], (t / NDO) & 1, abort_flag, WAIT_LIMIT_NS)) break;
        // dP^T overwrites S^T once the warpgroup has it in registers (S_READ),
        // so G2 runs while the softmax is computed.
        if (!mbar_wait(&bars[BAR_SREAD + s], j & 1, abort_flag, WAIT_LIMIT_NS)) break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          const uint32_t aDO = smem_u32(sDO + st * L::TILE_DO);
#pragma unroll
          for (int k = 0; k < DV / 16; ++k) {
            const uint32_t kk = (k >> 2) * L::BLK_KV + (k & 3) * 32;
            const uint32_t kq = (k >> 2) * L::BLK_Q + (k & 3) * 32;
            mma_ss(tmem + L::col_s(s), sdesc_at(T_KMAJ, aV + kk), sdesc_at(T_KMAJ, aDO + kq), ID_G2,
                   k > 0);
          }
          mma_commit(&bars[BAR_DPFULL + s]);
          if (t + NDO < n) mma_commit(&bars[BAR_DOEMPTY + st]);  // G2's share of the release
        }
        __syncwarp();
      }
    } else {
      for (int u = 0; u < n && ok; ++u) {
        const int su = u & 1, sdu = u % NDO, squ = u % NQ, ju = u >> 1;
        if (!mbar_wait(&bars[BAR_PREADY + su], ju & 1, abort_flag, WAIT_LIMIT_NS)) break;
        // G3 reads dO(u) too; only the G2 issuer has waited for it so far.
        if (!mbar_wait(&bars[BAR_DOFULL + sdu], (u / NDO) & 1, abort_flag, WAIT_LIMIT_NS)) break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          // G3: dV[key, d] += sum_q P^T[key, q] dO[q, d]
          const uint32_t aDO = smem_u32(sDO + sdu * L::TILE_DO) + off_dov;
#pragma unroll
          for (int k = 0; k < BQ / 16; ++k)
            mma_ts(tmem + L::COL_DV, tmem + L::col_p(su) + 8 * k, sdesc_at(T_MN_Q, aDO + k * 2048),
                   ID_G3, (u > 0 || k > 0));
          if (u + NDO < n) mma_commit(&bars[BAR_DOEMPTY + sdu]);  // G3's share
          mma_commit(&bars[BAR_SFREE + su]);
        }
        __syncwarp();
        if (!mbar_wait(&bars[BAR_DSREADY + su], ju & 1, abort_flag, WAIT_LIMIT_NS)) break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          // G4: dK[key, d] += sum_q dS^T[key, q] Q[q, d]
          const uint32_t aQ = smem_u32(sQ + squ * L::TILE_Q) + off_qk;
          const uint32_t aDS = smem_u32(sDS + su * L::TILE_DS);
#pragma unroll
          for (int k = 0; k < BQ / 16; ++k)
            mma_ss(tmem + L::COL_DK, sdesc_at(T_KMAJ, aDS + k * 32), sdesc_at(T_MN_Q, aQ + k * 2048),
                   ID_G4, (u > 0 || k > 0));
          if (u + NQ < n) mma_commit(&bars[BAR_QEMPTY + squ]);
          mma_commit(&bars[BAR_DSFREE + su]);
        }
        __syncwarp();
      }
      if (n > 0 && elect_one()) mma_commit(&bars[BAR_MMADONE]);
      __syncwarp();
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------ dS^T store
    // Once a tile's dS^T is in shared memory, one thread stores it to the
    // workspace and releases the buffer when the copy has read it, so no
    // compute warp waits on the copy.
    if (lane == 0) {
      int band_lo, band_hi;
      ds_band_range(p, kt, band_lo, band_hi);
      const long long band_prefix = ds_band_prefix(p, kt);
      for (int t = 0; t < n; ++t) {
        const int s = t & 1, j = t >> 1;
        if (!mbar_wait(&bars[BAR_DSREADY + s], j & 1, abort_flag, WAIT_LIMIT_NS)) break;
        const int qt = qt_hi - t;
        uint8_t* dst = ds_tile(p, bh, band_prefix, band_lo, qt);
        if (lead && in_bounds(p.status, dst, DS_TILE_BYTES, p.ds_ws, ds_ws_bytes(p)))
          bulk_store(dst, sDS + s * L::TILE_DS, DS_TILE_BYTES);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(&bars[BAR_DSCOPIED + s]);
      }
      bulk_wait_group_read0();
    }
  } else if (warp == 13 && lead) {
    // This CTA's share of the head's empty key tiles (gsz = 1: the partial
    // set of a query head is its bh index).
    zero_group_share_of_empty_key_tiles(p, p.dk_ws ? (long long)bh : (long long)b * p.Hkv + hk,
                                                 kt, Lq, Lk, lane);
  } else if (BIAS && warp == 14 && lead) {
    // The dBias blocks of this key tile that no CTA computes.
    if (p.dbias != nullptr && !p.dbias_red) zero_unvisited_dbias_blocks(p, b, bh, 1, kt, qt_lo, qt_hi, lane, 32);
  }  // warp 15 (and 14 without a bias): idle members of the fourth warpgroup
  } else {
    regs_increase<ds_kernel::REGS_COMPUTE>();
    // ------------------------------------------------------------ compute warpgroups
    pdl_wait_prior_grid();
    const int slot = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int k = k0 + row;
    const bool row_dead = k >= Lk;
    const long long q_lo_vis = p.causal ? (long long)k - diag - Rp : -(1ll << 40);
    const long long q_hi_vis = has_window ? (long long)k - diag + p.window_left : (1ll << 40);
    uint8_t* ds_row = sDS + slot * L::TILE_DS + row * 128;
    float P[BQ];
    bool ok = true;
    constexpr float LOG2E_F = 1.4426950408889634f;
    const bool key_in = k < p.Skv;
    // Bias (BIAS): element offset of (head, first query, this key) of tile t
    // inside one batch, and that tile's column of this thread's key.
    auto bias_tile_off = [&](int tt) -> long long {
      return ((long long)h * p.Sq + (qt_hi - tt) * BQ) * p.Skv + k;
    };
    float bz[BIAS ? BQ : 1];
    if constexpr (BIAS) {
      if (slot < n)
        load_bias_column(p, (long long)b * p.bias_bstride + bias_tile_off(slot), key_in, (qt_hi - slot) * BQ, bz);
      else
        for (int i = 0; i < BQ; ++i) bz[i] = 0.f;
    }
    for (int t = slot; t < n && ok; t += 2) {
      const int j = t >> 1, st = t % NQ;
      const int qt = qt_hi - t, q0 = qt * BQ;
      const float* qs = sQS + st * QSTAT_FLOATS;
      const long long bias_off = BIAS ? bias_tile_off(t) : 0;
      const bool need_mask = (k0 + BN > Lk) ||
                             (p.causal && (long long)q0 < (long long)(k0 + BN - 1) - diag - Rp) ||
                             (has_window && (long long)(q0 + BQ - 1) > (long long)k0 - diag + p.window_left);
      if (!mbar_wait(&bars[BAR_QFULL + st], (t / NQ) & 1, abort_flag, WAIT_LIMIT_NS) ||
          !mbar_wait(&bars[BAR_SFULL + slot], j & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(t_lane + L::col_s(slot), ra);
        tmem_ld32(t_lane + L::col_s(slot) + 32, rb);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        tc_fence_before();
        mbar_arrive(&bars[BAR_SREAD + slot]);  // the S^T columns may be overwritten
        const float4* lse4 = reinterpret_cast<const float4*>(qs);
#pragma unroll
        for (int i4 = 0; i4 < BQ / 4; ++i4) {
          const float4 l = lse4[i4];
          const uint32_t* r = i4 < 8 ? ra : rb;
          const int i = (i4 & 7) * 4;
          float x[4] = {fmaf(__uint_as_float(r[i + 0]), p.scale_log2, -l.x),
                        fmaf(__uint_as_float(r[i + 1]), p.scale_log2, -l.y),
                        fmaf(__uint_as_float(r[i + 2]), p.scale_log2, -l.z),
                        fmaf(__uint_as_float(r[i + 3]), p.scale_log2, -l.w)};
          if constexpr (BIAS) {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = fmaf(bz[i4 * 4 + e], LOG2E_F, x[e]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) P[i4 * 4 + e] = ex2_approx(x[e]);
        }
      }
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < BQ; ++i) {
          const long long q = q0 + i;
          if (row_dead || q < q_lo_vis || q > q_hi_vis) P[i] = 0.f;
        }
      }
      // P^T columns of this slot are read by G3 of tile t-2 until it completes.
      if (j >= 1 && !mbar_wait(&bars[BAR_SFREE + slot], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_io2<F16>(P[c16 * 32 + 2 * i], P[c16 * 32 + 2 * i + 1]);
        tmem_st16(t_lane + L::col_p(slot) + c16 * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[BAR_PREADY + slot]);  // S^T read and P^T written

      if (!mbar_wait(&bars[BAR_DPFULL + slot], j & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      // The dS^T buffer is read by G4 and by the bulk store of tile t-2.
      if (j >= 1 && (!mbar_wait(&bars[BAR_DSFREE + slot], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS) ||
                     !mbar_wait(&bars[BAR_DSCOPIED + slot], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS))) {
        ok = false;
        break;
      }
      __syncwarp();
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(t_lane + L::col_s(slot), ra);
        tmem_ld32(t_lane + L::col_s(slot) + 32, rb);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        tc_fence_before();
        mbar_arrive(&bars[BAR_DPREAD + slot]);  // the dP^T columns may be overwritten
        const float4* delta4 = reinterpret_cast<const float4*>(qs + BQ);
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk) {  // 8 queries = 16 bytes of dS^T per chunk
          const uint32_t* r = chunk < 4 ? ra : rb;
          const int i = (chunk & 3) * 8;
          const float4 d0 = delta4[chunk * 2], d1 = delta4[chunk * 2 + 1];
          const int c = chunk * 8;
          const float ds[8] = {P[c + 0] * (__uint_as_float(r[i + 0]) - d0.x),
                               P[c + 1] * (__uint_as_float(r[i + 1]) - d0.y),
                               P[c + 2] * (__uint_as_float(r[i + 2]) - d0.z),
                               P[c + 3] * (__uint_as_float(r[i + 3]) - d0.w),
                               P[c + 4] * (__uint_as_float(r[i + 4]) - d1.x),
                               P[c + 5] * (__uint_as_float(r[i + 5]) - d1.y),
                               P[c + 6] * (__uint_as_float(r[i + 6]) - d1.z),
                               P[c + 7] * (__uint_as_float(r[i + 7]) - d1.w)};
          const uint32_t w0 = pack_io2<F16>(ds[0], ds[1]);
          const uint32_t w1 = pack_io2<F16>(ds[2], ds[3]);
          const uint32_t w2 = pack_io2<F16>(ds[4], ds[5]);
          const uint32_t w3 = pack_io2<F16>(ds[6], ds[7]);
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (row & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
          if constexpr (BIAS) {
            if (p.dbias != nullptr && key_in && lead) {
              const long long off = (long long)b * p.dbias_bstride + bias_off + (long long)c * p.Skv;
              const int rows_in = min(8, p.Sq - q0 - c);
              if (p.dbias_red) {
                float* dst = p.dbias + off;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (e < rows_in) atomicAdd(dst + (long long)e * p.Skv, ds[e]);
              } else if (p.dbias_out == 0) {
                float* dst = p.dbias + off;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (e < rows_in) __stcs(dst + (long long)e * p.Skv, ds[e]);
              } else {  // a 16-bit dBias (the io type): half the store bytes
                unsigned short* dst = reinterpret_cast<unsigned short*>(p.dbias) + off;
                const bool f16 = p.dbias_out == 2;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (e < rows_in) __stcs(dst + (long long)e * p.Skv, f32_to_16(ds[e], f16));
              }
            }
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[BAR_DSREADY + slot]);  // dP^T read, dS^T in shared memory
      if constexpr (BIAS) {
        // The next tile's bias column (unconditional, zeros past the last
        // tile, so that the old values are dead here), the one after into L2.
        const int tn = t + 2 < n ? t + 2 : t;
        load_bias_column(p, (long long)b * p.bias_bstride + bias_tile_off(tn), key_in && t + 2 < n,
                         (qt_hi - tn) * BQ, bz);
        if (t + 4 < n)
          prefetch_bias_tile(p, (long long)b * p.bias_bstride + bias_tile_off(t + 4) - k + k0,
                             (qt_hi - t - 4) * BQ, k0, row);
      }
    }

    // ---- epilogue: warpgroup 0 writes dV (D_v columns), warpgroup 1 scale * dK
    // (D_qk). Each thread converts its key row into the (now idle) dO or Q stage
    // ring in the 128-byte-swizzled box layout, and one thread per warpgroup
    // writes the rows with TMA stores, which drop rows past S_kv.
    if (n > 0 && ok) {
      ok = mbar_wait(&bars[BAR_MMADONE], 0, abort_flag, WAIT_LIMIT_NS);
      __syncwarp();
      tc_fence_after();
    }
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    const int D = slot ? L::ACC_K : L::ACC_V;  // this unit's columns
    const uint32_t col0 = slot ? L::COL_DK : L::COL_DV;
    const float mult = slot ? p.scale : 1.f;
    uint8_t* stg = slot ? sQ : sDO;
    static_assert(L::NQ * L::TILE_Q >= L::ACC_K / 64 * L::BLK_KV &&
                      L::NDO * L::TILE_DO >= L::ACC_V / 64 * L::BLK_KV,
                  "staging fits in the stage rings");
    for (int c32 = 0; c32 < D / 32; ++c32) {
      uint32_t r[32];
      if (n > 0 && warp_ok) {
        tmem_ld32(t_lane + col0 + c32 * 32, r);
        tmem_ld_wait(r);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      uint8_t* dst_row = stg + (c32 >> 1) * L::BLK_KV + row * 128;
#pragma unroll
      for (int v8 = 0; v8 < 4; ++v8) {
        uint4 o;
        o.x = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 0]) * mult, __uint_as_float(r[v8 * 8 + 1]) * mult);
        o.y = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 2]) * mult, __uint_as_float(r[v8 * 8 + 3]) * mult);
        o.z = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 4]) * mult, __uint_as_float(r[v8 * 8 + 5]) * mult);
        o.w = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 6]) * mult, __uint_as_float(r[v8 * 8 + 7]) * mult);
        const int piece = (c32 & 1) * 4 + v8;
        *reinterpret_cast<uint4*>(dst_row + ((piece ^ (row & 7)) << 4)) = o;
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + slot, 128);
    if (row == 0) {
      const long long head = p.dk_ws ? (long long)bh : (long long)b * p.Hkv + hk;
      const CUtensorMap* map = slot ? &maps.dk_out : &maps.dv_out;
      for (int blk = 0; blk < D / 64; ++blk)
        tma_store_3d(map, stg + blk * L::BLK_KV, (half * (D / 64) + blk) * 64, k0, (int)head);
      bulk_commit_group();
      bulk_wait_group_read0();  // the CTA may exit once the copies have read shared memory
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, bool BIAS, bool F16, int SPLIT>
static cudaError_t set_ds_smem() {
  return cudaFuncSetAttribute(sdpa_bwd_main_ds<DQK, DV, BIAS, F16, SPLIT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              ds_kernel::Layout<DQK, DV, SPLIT>::BYTES);
}

template <int DQK, int DV, int SPLIT>
static cudaError_t set_ds_smem_all() {
  cudaError_t e = set_ds_smem<DQK, DV, false, false, SPLIT>();
  if (e == cudaSuccess) e = set_ds_smem<DQK, DV, true, false, SPLIT>();
  if (e == cudaSuccess) e = set_ds_smem<DQK, DV, false, true, SPLIT>();
  if (e == cudaSuccess) e = set_ds_smem<DQK, DV, true, true, SPLIT>();
  return e;
}

cudaError_t main_ds_kernel_setup() {
  cudaError_t e = set_ds_smem_all<192, 128, 1>();
  if (e == cudaSuccess) e = set_ds_smem_all<256, 256, 2>();
  return e;
}

template <int DQK, int DV, int SPLIT>
static cudaError_t launch_main_ds_dims(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  // SPLIT units per (key tile, query head), key tile major.
  const dim3 grid((unsigned)(p.n_kt * p.B * p.Hq * SPLIT));
  const dim3 block(ds_kernel::THREADS);
  constexpr int bytes = ds_kernel::Layout<DQK, DV, SPLIT>::BYTES;
  if (p.bias != nullptr && p.f16)
    return launch_kernel(sdpa_bwd_main_ds<DQK, DV, true, true, SPLIT>, grid, block, bytes, s, true, maps, p);
  if (p.bias != nullptr)
    return launch_kernel(sdpa_bwd_main_ds<DQK, DV, true, false, SPLIT>, grid, block, bytes, s, true, maps, p);
  if (p.f16)
    return launch_kernel(sdpa_bwd_main_ds<DQK, DV, false, true, SPLIT>, grid, block, bytes, s, true, maps, p);
  return launch_kernel(sdpa_bwd_main_ds<DQK, DV, false, false, SPLIT>, grid, block, bytes, s, true, maps, p);
}

cudaError_t launch_main_ds(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  if (p.Dqk == 192 && p.Dv == 128) return launch_main_ds_dims<192, 128, 1>(maps, p, s);
  if (p.Dqk == 256 && p.Dv == 256) return launch_main_ds_dims<256, 256, 2>(maps, p, s);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
