// sdpa_bwd_main.cuh -- fused five-GEMM SDPA backward main kernel for sm_103a
// (D_qk = D_v = 64 or 128). Instantiated without a bias in sdpa_bwd_main.cu, with
// one in sdpa_bwd_main_bias.cu, and for the NVFP4 QAT backward in
// sdpa_bwd_main_qat.cu.
//
// What it computes (cuDNN frontend docs, "SDPA Backward (SM120)", section
// "Main-kernel pipeline: KV-stationary, five chained GEMMs"): one CTA owns one
// tile of BN = 128 keys of one query head (its KV head is h / G), keeps K and V
// of that tile in shared memory, and walks the visible query tiles of BQ = 64
// rows in descending order. Per query tile t:
//   G1  S^T  = K Q^T                       (tensor memory, fp32)
//       P^T  = exp2(S^T * scale*log2e - LSE*log2e), masked -> 0
//   G2  dP^T = V dO^T                      (tensor memory, fp32)
//       dS^T = P^T * (dP^T - delta)        -> bf16 in shared memory
//   G3  dV  += P^T dO                      (A = P^T read from tensor memory)
//   G4  dK  += dS^T Q
//   G5  dQ^T = K^T dS^T  -> one TMA bulk reduce-add into the fp32 dQ accumulator
// Masks follow "Causal, sliding-window, and padding masks": loop bounds skip
// fully masked tiles and only edge tiles mask in registers.
//
// Additive bias (BIAS; the Capabilities list of the same page): the bias
// enters the replay exponent, P^T = exp2(S^T * scale*log2e + bias*log2e -
// LSE*log2e), and dS' = P^T * (dP^T - delta) is also written out in fp32 as
// dBias. A thread owns one key, so a warp's 32 keys of one query row are 32
// consecutive elements of a bias or dBias row: each load and store of a tile
// column is one coalesced 64- or 128-byte access. A warpgroup requests the
// bias of its next tile as soon as it has formed dS of the current one (the
// registers are free then), so the loads are in flight while it waits for the
// next S^T, and the tile after that is prefetched into L2. dBias tiles that no
// CTA visits get their zeros from an otherwise idle warp of the CTA that owns
// their key tile (per-batch dBias), or from the preprocess kernel (one shared
// dBias, which the batch rows add into atomically).
//
// NVFP4 QAT (QAT; page "NVFP4 Attention QAT Backward", Overview): Q, K and V
// arrive already fake-quantized, so the GEMMs are unchanged; dS (hence dQ and
// dK) uses P itself (straight-through), while G3 takes P fake-quantized to
// NVFP4 in blocks of 16 consecutive keys of each query: the 16 keys of a block
// are 16 lanes of one warp (block maxima by shuffles, p_block_scales). The E4M3
// and E2M1 roundings are the hardware conversions (round to nearest even,
// saturating).
//
// Schedule. Two query tiles are in flight: tensor memory holds two slots, each
// with S^T and dP^T (dQ^T reuses the dP^T columns once dS is formed). Compute
// warpgroup 0 owns the even tiles (slot 0), warpgroup 1 the odd ones (slot 1).
// One MMA warp issues G1/G2 of tile t while the other issues G3/G4/G5 of tile
// t-1, so the tensor core works on one tile while a warpgroup replays the
// softmax of the other. A third warpgroup moves each dQ^T tile from tensor
// memory to shared memory and hands it to the TMA engine as one bulk reduction
// (in deterministic mode after waiting its turn on the query tile's counter).
//
// Warps: 0-3 slot-0 compute, 4-7 slot-1 compute, 8-11 dQ, 12 TMA producer,
// 13 score-GEMM issuer and tensor-memory owner, 14 gradient-GEMM issuer, 15 the
// dS^T store on the two-kernel route, otherwise idle (it completes the fourth
// warpgroup so that register budgets can be moved
// between warpgroups: launched with 128 registers per thread, the compute
// warpgroups grow to 160 while the dQ and control warpgroups shrink to 96;
// 128 threads x (160 + 160 + 96 + 96) = 65536 = 512 threads x 128).
//
// Shared memory (128-byte swizzle, every tile 1024-byte aligned):
//   K, V        [D/64 blocks][128 key rows][128 B]
//   Q, dO x3/4  [D/64 blocks][64 query rows][128 B]   (stage ring: 4 stages on the
//                                                      two-kernel route, which
//                                                      needs no dQ staging)
//   dS^T x2     [128 key rows][64 queries x 2 B]      (one per slot)
//   dQ staging  [64 queries][D] fp32                  (bulk reduction source)
//   qstat x3/4  LSE*log2e[64], delta[64]
// Tensor memory (512 columns x 128 lanes, fp32):
//   slot s: S^T at 128s + [0,64) (P^T written back as bf16 into [0,32) by the
//           same threads that read S^T), dP^T then dQ^T at 128s + [64,128)
//   dV at [256, 256+D), dK at [256+D, 256+2D)
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "bias.cuh"
#include "common.cuh"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace sdpa {

constexpr int MAIN_THREADS = 512;
constexpr uint32_t REGS_COMPUTE = 160, REGS_DQ = 96, REGS_CTRL = 96;
static_assert(128 * (2 * REGS_COMPUTE + REGS_DQ + REGS_CTRL) <= MAIN_THREADS * 128,
              "register split exceeds the launch budget");
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;  // 4 s: far above any legal wait

enum : int {
  BAR_K = 0,            // the K tile has landed (G1, G5)
  BAR_QFULL = 1,        // + stage (up to 4)
  BAR_QEMPTY = 5,       // + stage (up to 4)
  BAR_SFULL = 9,        // + slot (2)
  BAR_DPFULL = 11,      // + slot
  BAR_PREADY = 13,      // + slot, 128 arrivals
  BAR_SFREE = 15,       // + slot
  BAR_DSREADY = 17,     // + slot, 128 arrivals
  BAR_DQFULL = 19,      // + slot
  BAR_DQEMPTY = 21,     // + slot, 128 arrivals
  BAR_MMADONE = 23,     // every MMA of the CTA has completed (epilogue may read dK/dV)
  BAR_DSCOPIED = 24,    // + slot: the slot's dS^T tile has been read out to global (dS route)
  BAR_DPREAD = 26,      // + slot, 128 arrivals: dP^T has been loaded into registers
  BAR_STAGEREADY = 28,  // + staging half (2), 128 arrivals: the half is written
  BAR_STAGEFREE = 30,   // + staging half (2): its bulk reduction has read it
  BAR_V = 32,           // the V tile has landed (G2)
  NUM_BARS = 33
};

// NST Q/dO stages; the dQ staging buffer exists only on the dQ-reduction route
// (on the two-kernel route its space holds a fourth stage).
template <int D, bool DS_OUT>
struct MainLayout {
  static constexpr int NST = DS_OUT ? 4 : 3;
  static constexpr int BLK_KV = BN * 128;          // one 64-column block of a 128-row tile
  static constexpr int BLK_Q = BQ * 128;           // one 64-column block of a 64-row tile
  static constexpr int TILE_KV = BN * D * 2;
  static constexpr int TILE_Q = BQ * D * 2;
  static constexpr int TILE_DS = BN * BQ * 2;
  static constexpr int TILE_DQ = DS_OUT ? 0 : BQ * D * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_KV;
  static constexpr int OFF_Q = OFF_V + TILE_KV;
  static constexpr int OFF_DO = OFF_Q + NST * TILE_Q;
  static constexpr int OFF_DS = OFF_DO + NST * TILE_Q;
  static constexpr int OFF_DQ = OFF_DS + 2 * TILE_DS;
  static constexpr int OFF_QS = OFF_DQ + TILE_DQ;
  static constexpr int OFF_BAR = OFF_QS + NST * QSTAT_FLOATS * 4;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + D;
  __host__ __device__ static constexpr uint32_t col_s(int slot) { return 128u * slot; }
  __host__ __device__ static constexpr uint32_t col_dp(int slot) { return 128u * slot + 64u; }
  static_assert(COL_DK + D <= 512, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
  // More than half an SM's shared memory: one CTA per SM, so a CTA never waits
  // for tensor memory held by a co-resident CTA that may be waiting on it.
  static_assert(BYTES > 116 * 1024, "one CTA per SM");
};

__device__ __forceinline__ void set_main_status(int* status, int bit) { atomicOr(status, bit); }

// NVFP4 local scales of P's 16-key blocks for all BQ (= 64) query columns of
// this lane's key: the 16 keys of a block are the 16 lanes of one half warp
// (l = lane & 15). Four rounds of recursive halving (exchange half of the
// columns with lane l ^ o, keep the maxima of the other half) leave lane l with
// the block maxima of columns 4l .. 4l+3; it turns them into scales,
// E4M3(amax / 6) with a correctly rounded division, and four rounds of
// recursive doubling hand every lane all 64 scales. (A half-warp reduction
// instruction per column measured four times slower.)
__device__ __forceinline__ void p_block_scales(const float (&P)[BQ], float (&sc)[BQ], int l) {
  static_assert(BQ == 64, "four halving rounds take 64 columns to 4");
#pragma unroll
  for (int i = 0; i < BQ; ++i) sc[i] = P[i];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int o = 8 >> r, n = BQ >> r;
    const bool up = (l & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? sc[i] : sc[i + n / 2];
      const float keep = up ? sc[i + n / 2] : sc[i];
      sc[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  const float2 s01 = nvfp4_scales(sc[0], sc[1]), s23 = nvfp4_scales(sc[2], sc[3]);
  sc[0] = s01.x;
  sc[1] = s01.y;
  sc[2] = s23.x;
  sc[3] = s23.y;
#pragma unroll
  for (int r = 3; r >= 0; --r) {
    const int o = 8 >> r, n = 4 << (3 - r);
    const bool up = (l & o) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float recv = __shfl_xor_sync(0xffffffffu, sc[i], o);
      const float own = sc[i];
      sc[i] = up ? recv : own;
      sc[i + n] = up ? own : recv;
    }
  }
}

// Fake NVFP4 of two P values with their blocks' scales. P is itself the
// ex2.approx replay of the softmax, so each value's division by its scale is a
// product with the reciprocal (within an ulp or two of the correctly rounded
// quotient; an E2M1 rounding can differ only for a value that close to a
// rounding boundary, well inside P's own error).
__device__ __forceinline__ uint32_t fake_nvfp4_p_pair(float p0, float p1, float s0, float s1) {
  float r0, r1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(s0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(s1));
  const float2 q = round_e2m1x2(s0 > 0.f ? p0 * r0 : 0.f, s1 > 0.f ? p1 * r1 : 0.f);
  return pack_bf16x2(q.x * s0, q.y * s1);
}

// DS_OUT selects the deterministic two-kernel route: instead of G5 and the dQ
// reduction, every dS^T tile is stored to the workspace for the dQ kernel.
// BIAS adds the additive bias to the replay and writes dBias (when p.dbias).
// QAT writes G3's P^T fake-quantized to NVFP4. F16: fp16 io tensors (and
// fp16 P^T / dS^T MMA operands) instead of bf16.
template <int D, bool DS_OUT, bool BIAS, bool QAT = false, bool F16 = false>
__global__ void __launch_bounds__(MAIN_THREADS, 1)
    sdpa_bwd_main(const __grid_constant__ MainMaps maps, const ChainParams p) {
  using L = MainLayout<D, DS_OUT>;
  constexpr int NSTAGE = L::NST;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (tid == 0) set_main_status(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  if (!p.deterministic) {
    // A key tile that no query sees only has zero gradients. Its rows are
    // written by an idle warp of the group's other CTAs (or here, when the
    // batch row has no query or no key); leave before any setup.
    const int NG0 = p.B * p.Hkv * p.n_part;
    const int kt0 = blockIdx.x / NG0, gi0 = blockIdx.x % NG0, b0 = gi0 / (p.Hkv * p.n_part);
    int Lq0, Lk0, lo0, hi0;
    batch_lengths(p, b0, Lq0, Lk0);
    visited_query_tiles(kt0, Lq0, Lk0, p.causal, p.bottom_right, p.window_left, p.window_right, lo0,
                        hi0);
    if (hi0 < lo0) {
      if (!row_has_visible_pair(Lq0, Lk0))
        zero_key_tile_rows(p, p.dk_ws ? (long long)gi0 : (long long)(gi0 / p.n_part), kt0 * BN);
      if (BIAS && p.dbias != nullptr && !p.dbias_red) {
        const int hk0 = (gi0 / p.n_part) % p.Hkv;
        zero_unvisited_dbias_blocks(p, b0, b0 * p.Hq + hk0 * p.G + (gi0 % p.n_part) * p.gsz, p.gsz, kt0,
                                    lo0, hi0, threadIdx.x, blockDim.x);
      }
      return;
    }
  }
  uint8_t* sK = smem + L::OFF_K;
  uint8_t* sV = smem + L::OFF_V;
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sDO = smem + L::OFF_DO;
  uint8_t* sDS = smem + L::OFF_DS;
  float* sDQ = reinterpret_cast<float*>(smem + L::OFF_DQ);
  float* sQS = reinterpret_cast<float*>(smem + L::OFF_QS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int* unit_slot = reinterpret_cast<int*>(smem + L::OFF_MISC + 8);

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NUM_BARS; ++i) {
      const bool threads128 = (i == BAR_PREADY || i == BAR_PREADY + 1 || i == BAR_DSREADY ||
                               i == BAR_DSREADY + 1 || i == BAR_DQEMPTY || i == BAR_DQEMPTY + 1 ||
                               i == BAR_STAGEREADY || i == BAR_STAGEREADY + 1 || i == BAR_DPREAD ||
                               i == BAR_DPREAD + 1);
      mbar_init(&bars[i], threads128 ? 128 : 1);
    }
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.d_o);
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }

  // Work unit. Deterministic mode claims units from a ticket so that a unit is
  // only ever claimed after every unit it waits on (the same query tile, a
  // lower key tile) has been claimed by a running CTA.
  if (p.deterministic) {
    pdl_wait_prior_grid();  // the ticket is cleared by the preprocess kernel
    if (tid == 0) *unit_slot = atomicAdd(p.ticket, 1);
  } else if (tid == 0) {
    *unit_slot = blockIdx.x;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int unit = *unit_slot;
  if constexpr (DS_OUT) {
    // The dQ kernel may become resident on the SMs this grid's finished units
    // leave (its setup and first K loads need nothing from here; it waits for
    // this grid before loading dS). Each thread releases it only after the
    // preprocess has completed, which clears the dQ kernel's ticket and zero
    // tile; the producer lane does so after issuing its first loads.
    if (!(warp == 12 && lane == 0)) {
      pdl_wait_prior_grid();
      pdl_launch_dependents();
    }
  }

  // A unit is one key tile of one head group: gsz query heads of one KV head
  // (group gi = (b * Hkv + hk) * n_part + g covers query heads
  // hk * G + g * gsz ...). Units are ordered key tile major: every group's key
  // tile 0 first. Under a causal mask low key tiles see the most query tiles,
  // so the longest units start first.
  const int NG = p.B * p.Hkv * p.n_part;
  const int kt = unit / NG;
  const int gi = unit % NG;
  const int kvh_g = gi / p.n_part;                 // b * Hkv + hk
  const int b = kvh_g / p.Hkv, hk = kvh_g % p.Hkv;
  const int bh0 = b * p.Hq + hk * p.G + (gi % p.n_part) * p.gsz;  // the group's first query head
  const int k0 = kt * BN;
  // dK/dV destination: the KV head, or the group's partial set.
  const long long out_head = p.dk_ws ? (long long)gi : (long long)kvh_g;

  int Lq, Lk;
  batch_lengths(p, b, Lq, Lk);
  const int diag = p.bottom_right ? Lk - Lq : 0;
  const int Rp = p.window_right > 0 ? p.window_right : 0;
  const bool has_window = p.window_left >= 0;
  int qt_lo, qt_hi;
  visited_query_tiles(kt, Lq, Lk, p.causal, p.bottom_right, p.window_left, p.window_right, qt_lo,
                      qt_hi);
  // Tiles t = 0 .. n-1 walk the visible query tiles (descending) of the group's
  // heads in turn: head bh0 + t / n1, query tile qt_hi - t % n1.
  const int n1 = qt_hi >= qt_lo ? qt_hi - qt_lo + 1 : 0;  // query tiles per head
  const int n = p.gsz * n1;

  if (warp >= 12) {
    regs_decrease<REGS_CTRL>();
    if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      // K first, then the first tile's Q and dO, then V: G1 of the first tile
      // needs only K and Q, so its score GEMM and softmax can run while V and
      // dO are still landing. Q, dO, K and V are inputs of the chain; only the
      // row statistics come from the preprocess kernel, so they alone wait for it.
      auto load_q_do = [&](int t) {
        const int st = t % NSTAGE, hj = t / n1;
        const int qt = qt_hi - (t - hj * n1), bh = bh0 + hj;
        uint64_t* full = &bars[BAR_QFULL + st];
        mbar_arrive_expect_tx(full, 2 * L::TILE_Q + QSTAT_FLOATS * 4);
        for (int blk = 0; blk < D / 64; ++blk) {
          tma_load_3d(sQ + st * L::TILE_Q + blk * L::BLK_Q, &maps.q, full, blk * 64, qt * BQ, bh);
          tma_load_3d(sDO + st * L::TILE_Q + blk * L::BLK_Q, &maps.d_o, full, blk * 64, qt * BQ, bh);
        }
      };
      auto load_qstat = [&](int t) {
        const int st = t % NSTAGE, hj = t / n1;
        const int qt = qt_hi - (t - hj * n1), bh = bh0 + hj;
        const float* src = p.qstat + ((long long)bh * p.n_qt + qt) * QSTAT_FLOATS;
        if (in_bounds(p.status, src, QSTAT_FLOATS * 4, p.qstat, qstat_bytes(p)))
          bulk_load(sQS + st * QSTAT_FLOATS, src, QSTAT_FLOATS * 4, &bars[BAR_QFULL + st]);
        else
          mbar_complete_tx(&bars[BAR_QFULL + st], QSTAT_FLOATS * 4);
      };
      // On the dQ-reduction route a K/V tile is read by this unit only, when
      // its KV group is one unit; marking it evict-first keeps the fp32 dQ
      // accumulator in L2 (the two-kernel route, whose dQ kernel reads K
      // again, measured slightly slower with the hints and keeps the default).
      const bool once = !DS_OUT && p.n_part == 1;
      const uint64_t pol_k = once ? l2_evict_first() : l2_evict_normal();
      const uint64_t pol_v = pol_k;
      mbar_arrive_expect_tx(&bars[BAR_K], L::TILE_KV);
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d_hint(sK + blk * L::BLK_KV, &maps.k, &bars[BAR_K], blk * 64, k0, b * p.Hkv + hk, pol_k);
      load_q_do(0);
      mbar_arrive_expect_tx(&bars[BAR_V], L::TILE_KV);
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d_hint(sV + blk * L::BLK_KV, &maps.v, &bars[BAR_V], blk * 64, k0, b * p.Hkv + hk, pol_v);
      pdl_wait_prior_grid();  // row statistics come from the preprocess kernel
      if constexpr (DS_OUT) pdl_launch_dependents();
      load_qstat(0);
      for (int t = 1; t < n; ++t) {
        const int st = t % NSTAGE;
        if (t >= NSTAGE && !mbar_wait(&bars[BAR_QEMPTY + st], ((t / NSTAGE) - 1) & 1, abort_flag,
                                      WAIT_LIMIT_NS))
          break;
        load_q_do(t);
        load_qstat(t);
      }
    }
    } else if (warp == 13 || warp == 14) {
      // ---------------------------------------------------------- MMA issuers
      // A tcgen05.mma costs its issuing thread on the order of 100 cycles, more
      // than a 64-column MMA takes on the tensor core, so two warps issue: warp
      // 13 the score GEMMs G1/G2 of every tile, warp 14 the gradient GEMMs
      // G3/G4/G5. Each warp stays converged and issues from one elected lane;
      // mbarriers carry every dependency between the two streams.
      pdl_wait_prior_grid();
      constexpr uint32_t ID_G12 = idesc_io(128, BQ, false, false, F16);  // S^T, dP^T
      constexpr uint32_t ID_G34 = idesc_io(128, D, false, true, F16);    // dV, dK
      constexpr uint32_t ID_G5 = idesc_io(128, BQ, true, true, F16);     // dQ^T (rows >= D unused)
      constexpr uint64_t T_KMAJ = sdesc_sw128_template(16, 1024);          // K-major operands
      constexpr uint64_t T_MN_Q = sdesc_sw128_template(L::BLK_Q, 1024);    // MN-major, 64-row tiles
      constexpr uint64_t T_MN_KV = sdesc_sw128_template(L::BLK_KV, 1024);  // MN-major, 128-row tiles
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      // Both issuers need K (G1, G5); G2 also needs V, waited for before its first use.
      bool ok = n > 0 && mbar_wait(&bars[BAR_K], 0, abort_flag, WAIT_LIMIT_NS);
      if (warp == 13) {
        for (int t = 0; t < n && ok; ++t) {
          const int s = t & 1, st = t % NSTAGE, j = t >> 1;
          const uint32_t aQ = smem_u32(sQ + st * L::TILE_Q);
          const uint32_t aDO = smem_u32(sDO + st * L::TILE_Q);
          ok = mbar_wait(&bars[BAR_QFULL + st], (t / NSTAGE) & 1, abort_flag, WAIT_LIMIT_NS);
          // The slot's S^T columns hold P^T of tile t-2 until its G3 completes.
          if (ok && t >= 2) ok = mbar_wait(&bars[BAR_SFREE + s], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS);
          if (!ok) break;
          __syncwarp();
          tc_fence_after();
          if (elect_one()) {
            // G1: S^T[key, q] = sum_d K[key, d] Q[q, d]   (both K-major)
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t kk = (k >> 2) * L::BLK_KV + (k & 3) * 32;
              const uint32_t kq = (k >> 2) * L::BLK_Q + (k & 3) * 32;
              mma_ss(tmem + L::col_s(s), sdesc_at(T_KMAJ, aK + kk), sdesc_at(T_KMAJ, aQ + kq), ID_G12,
                     k > 0);
            }
            mma_commit(&bars[BAR_SFULL + s]);
          }
          __syncwarp();
          // The slot's dP^T columns are read by the compute warpgroup of tile t-2
          // until it has them in registers (DP_READ), and on the dQ-reduction
          // route then hold dQ^T of tile t-2 until the dQ warpgroup has read it.
          if (t >= 2 && !mbar_wait(&bars[BAR_DPREAD + s], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS))
            break;
          if (!DS_OUT && t >= 2 &&
              !mbar_wait(&bars[BAR_DQEMPTY + s], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS))
            break;
          if (t == 0 && !mbar_wait(&bars[BAR_V], 0, abort_flag, WAIT_LIMIT_NS)) break;
          __syncwarp();
          tc_fence_after();
          if (elect_one()) {
            // G2: dP^T[key, q] = sum_d V[key, d] dO[q, d]
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t kk = (k >> 2) * L::BLK_KV + (k & 3) * 32;
              const uint32_t kq = (k >> 2) * L::BLK_Q + (k & 3) * 32;
              mma_ss(tmem + L::col_dp(s), sdesc_at(T_KMAJ, aV + kk), sdesc_at(T_KMAJ, aDO + kq), ID_G12,
                     k > 0);
            }
            mma_commit(&bars[BAR_DPFULL + s]);
          }
          __syncwarp();
        }
      } else {
        for (int u = 0; u < n && ok; ++u) {
          const int su = u & 1, stu = u % NSTAGE, ju = u >> 1;
          const uint32_t aQ = smem_u32(sQ + stu * L::TILE_Q);
          const uint32_t aDO = smem_u32(sDO + stu * L::TILE_Q);
          const uint32_t aDS = smem_u32(sDS + su * L::TILE_DS);
          if (!mbar_wait(&bars[BAR_PREADY + su], ju & 1, abort_flag, WAIT_LIMIT_NS)) break;
          __syncwarp();
          tc_fence_after();
          if (elect_one()) {
            // G3: dV[key, d] += sum_q P^T[key, q] dO[q, d]; P^T pairs in columns [0,32) of the slot.
#pragma unroll
            for (int k = 0; k < BQ / 16; ++k)
              mma_ts(tmem + L::COL_DV, tmem + L::col_s(su) + 8 * k, sdesc_at(T_MN_Q, aDO + k * 2048),
                     ID_G34, (u > 0 || k > 0));
            mma_commit(&bars[BAR_SFREE + su]);
          }
          __syncwarp();
          if (!mbar_wait(&bars[BAR_DSREADY + su], ju & 1, abort_flag, WAIT_LIMIT_NS)) break;
          __syncwarp();
          tc_fence_after();
          if (elect_one()) {
            // G4: dK[key, d] += sum_q dS^T[key, q] Q[q, d]   (dS^T K-major, Q MN-major)
#pragma unroll
            for (int k = 0; k < BQ / 16; ++k)
              mma_ss(tmem + L::COL_DK, sdesc_at(T_KMAJ, aDS + k * 32), sdesc_at(T_MN_Q, aQ + k * 2048),
                     ID_G34, (u > 0 || k > 0));
            // Stage u is refilled for tile u+3 once G4 is done (G1/G2 of tile u
            // completed before P_READY / DS_READY could arrive).
            if (u + NSTAGE < n) mma_commit(&bars[BAR_QEMPTY + stu]);
            if (!DS_OUT) {
              // G5: dQ^T[d, q] = sum_key K[key, d] dS^T[key, q]   (both MN-major)
#pragma unroll
              for (int k = 0; k < BN / 16; ++k)
                mma_ss(tmem + L::col_dp(su), sdesc_at(T_MN_KV, aK + k * 2048),
                       sdesc_at(T_MN_KV, aDS + k * 2048), ID_G5, k > 0);
            }
            // dQ^T ready (dQ route) / the slot's dS^T buffer no longer read by MMAs.
            mma_commit(&bars[BAR_DQFULL + su]);
          }
          __syncwarp();
        }
        // After the last tile (also releases the epilogue on abort).
        if (n > 0 && elect_one()) mma_commit(&bars[BAR_MMADONE]);
        __syncwarp();
      }
    } else if (!DS_OUT && warp == 15) {
      // Idle on this route: this CTA's share of the group's empty key tiles,
      // and the dBias blocks of its key tile that no CTA computes.
      if (!p.deterministic) zero_group_share_of_empty_key_tiles(p, out_head, kt, Lq, Lk, lane);
      if (BIAS && p.dbias != nullptr && !p.dbias_red)
        zero_unvisited_dbias_blocks(p, b, bh0, p.gsz, kt, qt_lo, qt_hi, lane, 32);
    } else if (DS_OUT && warp == 15) {
      // ------------------------------------------------------------ dS^T store
      // Two-kernel route: once a tile's dS^T is in shared memory, one thread
      // stores it to the workspace (the dQ kernel's input) and releases the
      // buffer when the copy has read it, so no compute warp waits on the copy.
      if (lane == 0) {
        int band_lo, band_hi;
        ds_band_range(p, kt, band_lo, band_hi);
        const long long band_prefix = ds_band_prefix(p, kt);
        for (int t = 0; t < n; ++t) {
          const int s = t & 1, j = t >> 1;
          if (!mbar_wait(&bars[BAR_DSREADY + s], j & 1, abort_flag, WAIT_LIMIT_NS)) break;
          const int hj = t / n1;
          const int qt = qt_hi - (t - hj * n1), bh = bh0 + hj;
          uint8_t* dst = ds_tile(p, bh, band_prefix, band_lo, qt);
          if (in_bounds(p.status, dst, DS_TILE_BYTES, p.ds_ws, ds_ws_bytes(p)))
            bulk_store(dst, sDS + s * L::TILE_DS, DS_TILE_BYTES);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&bars[BAR_DSCOPIED + s]);
        }
        bulk_wait_group_read0();
      }
    }  // otherwise warp 15: idle member of the control warpgroup
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ warpgroup
    regs_decrease<REGS_DQ>();
    // Idle on the two-kernel route: warp 9 writes this CTA's share of the
    // group's empty key tiles.
    if (DS_OUT && warp == 9 && !p.deterministic)
      zero_group_share_of_empty_key_tiles(p, out_head, kt, Lq, Lk, lane);
    // ... and the dBias blocks of this key tile that no CTA computes.
    if (BIAS && DS_OUT && p.dbias != nullptr && !p.dbias_red)
      zero_unvisited_dbias_blocks(p, b, bh0, p.gsz, kt, qt_lo, qt_hi, threadIdx.x - 256, 128);
    pdl_wait_prior_grid();
    const int quarter = warp & 3;
    const int d = quarter * 32 + lane;                 // dQ^T lane = head-dim column
    const bool has_rows = quarter * 32 < D;            // warp-uniform
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const bool leader = (warp == 8 && lane == 0);
    const uint64_t pol_acc = l2_evict_last();  // the convert reads the accumulator next
    int* pending_counter = nullptr;  // deterministic mode: turn not yet released
    int pending_turn = 0;
    int* pending_next = nullptr;     // ... and the current tile's, once the next is issued
    int pending_next_turn = 0;
    bool ok = true;
    for (int t = 0; t < (DS_OUT ? 0 : n) && ok; ++t) {
      const int s = t & 1, j = t >> 1;
      const int hj = t / n1;
      const int qt = qt_hi - (t - hj * n1), bh = bh0 + hj;
      if (!mbar_wait(&bars[BAR_DQFULL + s], j & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      uint32_t va[32], vb[32];
      if (has_rows) {
        tmem_ld32(t_lane + L::col_dp(s), va);
        tmem_ld32(t_lane + L::col_dp(s) + 32, vb);
        tmem_ld_wait(va);
        tmem_ld_wait(vb);
      }
      tc_fence_before();
      mbar_arrive(&bars[BAR_DQEMPTY + s]);
      // The staging buffer is used as two 16 KiB halves (query rows 0-31 and
      // 32-63, contiguous in the accumulator), each with its own bulk reduction:
      // the first half's copy runs while the second is written, and a half is
      // refilled as soon as its own copy has read it.
      float* dst = p.dq_accum + ((long long)bh * p.n_qt + qt) * (long long)BQ * D;
      if (leader && p.deterministic) {
        // Ordered relay: key tiles add into this query tile in ascending
        // order. This tile's turn is released once both of its reductions have
        // completed, which is checked after the next tile's reductions have
        // been issued, so the completion latency overlaps the next tile instead
        // of stalling this warpgroup. A key tile only ever waits on lower key
        // tiles, so the delayed release only skews the chain.
        const int kv_lo = has_window ? (int)max(0ll, floor_div((long long)qt * BQ + diag -
                                                                   p.window_left, BN))
                                     : 0;
        const int turn = kt - kv_lo + p.relay_turn_skew;
        int* counter = p.counters + (long long)bh * p.n_qt + qt;
        const uint64_t t0 = globaltimer_ns();
        const bool counter_ok = in_bounds(p.status, counter, sizeof(int), p.counters,
                                          (size_t)p.n_counters * sizeof(int));
        if (!counter_ok) counter = p.counters;  // stays in range; the status word reports it
        while (counter_ok && ld_acquire_gpu(counter) != turn) {
          __nanosleep(32);
          if (globaltimer_ns() - t0 > p.relay_wait_ns) {
            // Gives up on the turn (the adds may then come out of order) and
            // reports it; the kernel still completes.
            set_main_status(p.status, STATUS_TIMEOUT);
            break;
          }
        }
        fence_proxy_async_global();
        if (pending_counter != nullptr) pending_next = counter, pending_next_turn = turn;
        else pending_counter = counter, pending_turn = turn;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float* stg = sDQ + hf * (L::TILE_DQ / 8);
        if (t >= 1 &&
            !mbar_wait(&bars[BAR_STAGEFREE + hf], (t - 1) & 1, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        if (has_rows) {
          const uint32_t* v = hf ? vb : va;
#pragma unroll
          for (int q = 0; q < 32; ++q) stg[q * D + d] = __uint_as_float(v[q]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[BAR_STAGEREADY + hf]);
        if (leader) {
          mbar_wait(&bars[BAR_STAGEREADY + hf], t & 1, abort_flag, WAIT_LIMIT_NS);
          if (in_bounds(p.status, dst + hf * 32 * D, L::TILE_DQ / 2, p.dq_accum, dq_accum_bytes(p)))
            bulk_reduce_add_f32_hint(dst + hf * 32 * D, stg, L::TILE_DQ / 2, pol_acc);
          bulk_commit_group();
          // The previously issued half's reduction has read its buffer.
          if (t >= 1 || hf == 1) {
            bulk_wait_group_read1();
            mbar_arrive(&bars[BAR_STAGEFREE + (hf ^ 1)]);
          }
          if (p.deterministic && hf == 1 && pending_next != nullptr) {
            // Both halves of the previous tile complete -> release its turn.
            bulk_wait_group2();
            fence_proxy_async_global();
            st_release_gpu(pending_counter, pending_turn + 1);
            pending_counter = pending_next;
            pending_turn = pending_next_turn;
            pending_next = nullptr;
          }
        }
      }
      if (!ok) break;
    }
    if (leader) {
      // The relay releases the last turn only once the reductions have landed;
      // otherwise the CTA may leave as soon as they have read shared memory
      // (the writes complete before the grid does).
      if (p.deterministic) bulk_wait_group0();
      else bulk_wait_group_read0();
      if (pending_counter != nullptr) {
        fence_proxy_async_global();
        st_release_gpu(pending_counter, pending_turn + 1);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warpgroups
    regs_increase<REGS_COMPUTE>();
    pdl_wait_prior_grid();
    const int slot = warp >> 2;        // warpgroup: even (0) or odd (1) query tiles
    const int quarter = warp & 3;      // tensor-memory lane quarter
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int k = k0 + row;            // this thread's key (S^T / dP^T lane)
    const bool row_dead = k >= Lk;
    const long long q_lo_vis = p.causal ? (long long)k - diag - Rp : -(1ll << 40);
    const long long q_hi_vis = has_window ? (long long)k - diag + p.window_left : (1ll << 40);
    const float scale_log2 = p.scale_log2;
    uint8_t* ds_row = sDS + slot * L::TILE_DS + row * 128;
    float P[BQ];
    bool ok = true;
    constexpr float LOG2E_F = 1.4426950408889634f;
    const bool key_in = k < p.Skv;

    // Bias (BIAS): element offset of (head, first query, this key) of tile t
    // inside one batch, and that tile's column of this thread's key.
    auto bias_tile_off = [&](int tt) -> long long {
      const int hq = bh0 + tt / n1 - b * p.Hq;
      return ((long long)hq * p.Sq + (qt_hi - tt % n1) * BQ) * p.Skv + k;
    };
    float bz[BIAS ? BQ : 1];
    if constexpr (BIAS) {
      if (slot < n)
        load_bias_column(p, (long long)b * p.bias_bstride + bias_tile_off(slot), key_in,
                         (qt_hi - slot % n1) * BQ, bz);
      else
        for (int i = 0; i < BQ; ++i) bz[i] = 0.f;
    }

    for (int t = slot; t < n && ok; t += 2) {
      const int j = t >> 1, st = t % NSTAGE;
      const int qt = qt_hi - (t % n1), q0 = qt * BQ;
      const float* qs = sQS + st * QSTAT_FLOATS;
      const bool need_mask = (k0 + BN > Lk) ||
                             (p.causal && (long long)q0 < (long long)(k0 + BN - 1) - diag - Rp) ||
                             (has_window && (long long)(q0 + BQ - 1) > (long long)k0 - diag + p.window_left);
      const long long bias_off = BIAS ? bias_tile_off(t) : 0;

      // ---- softmax replay: P^T from S^T. The row statistics were written by
      // TMA, so this thread waits on the stage's transaction barrier itself.
      if (!mbar_wait(&bars[BAR_QFULL + st], (t / NSTAGE) & 1, abort_flag, WAIT_LIMIT_NS) ||
          !mbar_wait(&bars[BAR_SFULL + slot], j & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(t_lane + L::col_s(slot), ra);
        tmem_ld32(t_lane + L::col_s(slot) + 32, rb);
        const float4* lse4 = reinterpret_cast<const float4*>(qs);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
#pragma unroll
        for (int i4 = 0; i4 < BQ / 4; ++i4) {
          const float4 l = lse4[i4];
          const uint32_t* r = i4 < 8 ? ra : rb;
          const int i = (i4 & 7) * 4;
          if constexpr (BIAS) {
            P[i4 * 4 + 0] = ex2_approx(fmaf(bz[i4 * 4 + 0], LOG2E_F, fmaf(__uint_as_float(r[i + 0]), scale_log2, -l.x)));
            P[i4 * 4 + 1] = ex2_approx(fmaf(bz[i4 * 4 + 1], LOG2E_F, fmaf(__uint_as_float(r[i + 1]), scale_log2, -l.y)));
            P[i4 * 4 + 2] = ex2_approx(fmaf(bz[i4 * 4 + 2], LOG2E_F, fmaf(__uint_as_float(r[i + 2]), scale_log2, -l.z)));
            P[i4 * 4 + 3] = ex2_approx(fmaf(bz[i4 * 4 + 3], LOG2E_F, fmaf(__uint_as_float(r[i + 3]), scale_log2, -l.w)));
          } else {
            P[i4 * 4 + 0] = ex2_approx(fmaf(__uint_as_float(r[i + 0]), scale_log2, -l.x));
            P[i4 * 4 + 1] = ex2_approx(fmaf(__uint_as_float(r[i + 1]), scale_log2, -l.y));
            P[i4 * 4 + 2] = ex2_approx(fmaf(__uint_as_float(r[i + 2]), scale_log2, -l.z));
            P[i4 * 4 + 3] = ex2_approx(fmaf(__uint_as_float(r[i + 3]), scale_log2, -l.w));
          }
        }
      }
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < BQ; ++i) {
          const long long q = q0 + i;
          if (row_dead || q < q_lo_vis || q > q_hi_vis) P[i] = 0.f;
        }
      }
      // QAT: G3 reads P fake-quantized over blocks of 16 keys (16 lanes).
      float psc[QAT ? BQ : 1];
      if constexpr (QAT) p_block_scales(P, psc, lane & 15);
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        uint32_t w[16];
        if constexpr (QAT) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = fake_nvfp4_p_pair(P[c16 * 32 + 2 * i], P[c16 * 32 + 2 * i + 1], psc[c16 * 32 + 2 * i],
                                     psc[c16 * 32 + 2 * i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_io2<F16>(P[c16 * 32 + 2 * i], P[c16 * 32 + 2 * i + 1]);
        }
        tmem_st16(t_lane + L::col_s(slot) + c16 * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[BAR_PREADY + slot]);

      // ---- dS^T = P^T * (dP^T - delta) -> shared memory (K-major, swizzled)
      if (!mbar_wait(&bars[BAR_DPFULL + slot], j & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      // This slot's dS^T buffer is read by G4/G5 of tile t-2 until they complete
      // (and, on the dS route, by the bulk store of tile t-2).
      if (j >= 1 && !mbar_wait(&bars[BAR_DQFULL + slot], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      if (DS_OUT && j >= 1 &&
          !mbar_wait(&bars[BAR_DSCOPIED + slot], (j - 1) & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(t_lane + L::col_dp(slot), ra);
        tmem_ld32(t_lane + L::col_dp(slot) + 32, rb);
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
            // dBias = dS' in fp32: one column segment of this thread's key.
            if (p.dbias != nullptr && key_in) {
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
      mbar_arrive(&bars[BAR_DSREADY + slot]);
      if constexpr (BIAS) {
        // The next tile's bias column now (its loads overlap the wait for its
        // S^T), and the tile after it into L2.
        // (Unconditional, zeros past the last tile, so that the old values are
        // dead here rather than carried through this tile's dS step.)
        const int tn = t + 2 < n ? t + 2 : t;
        load_bias_column(p, (long long)b * p.bias_bstride + bias_tile_off(tn), key_in && t + 2 < n,
                         (qt_hi - tn % n1) * BQ, bz);
        if (t + 4 < n) {
          const int t4 = t + 4, q04 = (qt_hi - t4 % n1) * BQ;
          prefetch_bias_tile(p, (long long)b * p.bias_bstride + bias_tile_off(t4) - k + k0, q04, k0, row);
        }
      }
    }

    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK. Each
    // thread converts its key row into the warpgroup's half of the (now idle)
    // Q/dO stage ring, in the 128-byte-swizzled box layout, and one thread per
    // warpgroup writes the rows with TMA stores, which drop rows past S_kv.
    // Every lane runs the (warp-collective) tensor-memory loads.
    if (n > 0 && ok) {
      ok = mbar_wait(&bars[BAR_MMADONE], 0, abort_flag, WAIT_LIMIT_NS);
      __syncwarp();
      tc_fence_after();
    }
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    const uint32_t col0 = slot ? L::COL_DK : L::COL_DV;
    const float mult = slot ? p.scale : 1.f;
    uint8_t* stg = slot ? sDO : sQ;
    static_assert(L::NST * L::TILE_Q >= D / 64 * L::BLK_KV, "staging fits in a stage ring");
#pragma unroll
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
      const long long head = out_head;
      const CUtensorMap* map = slot ? &maps.dk_out : &maps.dv_out;
      // Final dK/dV rows are not read again (partial sets are, by the group
      // reduction); the reduction route keeps its accumulator in L2 instead.
      const uint64_t pol = (!DS_OUT && p.n_part == 1) ? l2_evict_first() : l2_evict_normal();
      for (int blk = 0; blk < D / 64; ++blk)
        tma_store_3d_hint(map, stg + blk * L::BLK_KV, blk * 64, k0, (int)head, pol);
      bulk_commit_group();
      bulk_wait_group_read0();  // the CTA may exit once the copies have read shared memory
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) set_main_status(p.status, STATUS_TIMEOUT);
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DS_OUT, bool BIAS, bool QAT = false, bool F16 = false>
static cudaError_t set_main_smem() {
  return cudaFuncSetAttribute(sdpa_bwd_main<D, DS_OUT, BIAS, QAT, F16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, MainLayout<D, DS_OUT>::BYTES);
}

// One CTA per (key tile, head group) work unit.
template <bool BIAS, bool F16 = false>
static cudaError_t launch_main_variant(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.n_kt * p.B * p.Hkv * p.n_part));
  const dim3 block(MAIN_THREADS);
  // D_qk = D_v up to 64 runs on the 64-column kernels, up to 128 on the 128-column
  // ones: TMA zero-fills the columns past D on loads and drops them on stores.
  if (p.Dqk <= 64)
    return launch_kernel(sdpa_bwd_main<64, false, BIAS, false, F16>, grid, block,
                         MainLayout<64, false>::BYTES, s, true, maps, p);
  if (p.ds_route)
    return launch_kernel(sdpa_bwd_main<128, true, BIAS, false, F16>, grid, block,
                         MainLayout<128, true>::BYTES, s, true, maps, p);
  return launch_kernel(sdpa_bwd_main<128, false, BIAS, false, F16>, grid, block,
                       MainLayout<128, false>::BYTES, s, true, maps, p);
}

template <bool BIAS, bool F16 = false>
static cudaError_t main_variant_setup() {
  cudaError_t e = set_main_smem<64, false, BIAS, false, F16>();
  if (e == cudaSuccess) e = set_main_smem<128, false, BIAS, false, F16>();
  if (e == cudaSuccess) e = set_main_smem<128, true, BIAS, false, F16>();
  return e;
}

}  // namespace sdpa
