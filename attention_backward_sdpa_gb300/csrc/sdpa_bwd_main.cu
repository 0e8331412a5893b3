// sdpa_bwd_main.cu -- fused five-GEMM SDPA backward main kernel for sm_103a.
//
// What it computes (cuDNN frontend docs, "SDPA Backward (SM120)", section
// "Main-kernel pipeline: KV-stationary, five chained GEMMs"): one CTA owns one
// tile of BN = 128 keys of one query head (its KV head is h / G), keeps K and V
// of that tile in shared memory, and walks the visible query tiles of BM = 128
// rows in descending order. Per query tile:
//   G1  S^T  = K Q^T                       (tensor memory, fp32)
//       P^T  = exp2(S^T * scale*log2e - LSE*log2e), masked -> 0
//   G2  dP^T = V dO^T                      (tensor memory, fp32)
//       dS^T = P^T * (dP^T - delta)        -> bf16 in shared memory
//   G3  dV  += P^T dO                      (A = P^T in tensor memory)
//   G4  dK  += dS^T Q
//   G5  dQ_t = dS K   -> fp32 reductions into the dQ accumulator
// The roles of the page's SM120 design (register-resident accumulators, 8 math
// warps with ldmatrix) are replaced by the Blackwell ones: tcgen05.mma issued
// by one thread with all accumulators in tensor memory, a TMA producer warp,
// and two 128-thread compute warpgroups that move S/dP/dQ between tensor memory
// and registers. Masks follow "Causal, sliding-window, and padding masks":
// loop bounds skip fully masked tiles, and only edge tiles mask in registers.
//
// Shared memory (bytes, every tile 1024-byte aligned, 128-byte swizzle):
//   K, V          [D/64 blocks][128 key rows][128 B]
//   Q, dO  x2     [D/64 blocks][128 query rows][128 B]   (double-buffered)
//   dS^T          [2 blocks of 64 queries][128 key rows][128 B]
//   qstat x2      LSE*log2e[128], delta[128]             (double-buffered)
// Tensor memory (512 fp32 columns x 128 lanes):
//   [0,128)    S^T (lanes = keys); P^T is written back as bf16 into the
//              columns each warpgroup has already read ([0,32) and [64,96))
//   [128,256)  dP^T, then dQ (lanes = queries) once dS has been formed
//   [256, 256+Dv)          dV accumulator
//   [256+Dv, 256+Dv+Dqk)   dK accumulator
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

constexpr int MAIN_THREADS = 320;  // warps 0-7 compute, 8 TMA producer, 9 MMA issuer
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;  // 4 s: far above any legal wait

enum : int {
  BAR_KV = 0,
  BAR_QFULL = 1,   // +stage
  BAR_QEMPTY = 3,  // +stage
  BAR_SFULL = 5,
  BAR_DPFULL = 6,
  BAR_PREADY = 7,
  BAR_G3DONE = 8,
  BAR_DSREADY = 9,
  BAR_DQFULL = 10,
  BAR_DQEMPTY = 11,
  BAR_RELAYGO = 12,
  BAR_RELAYDONE = 13,
  NUM_BARS = 14
};

template <int DQK, int DV>
struct MainLayout {
  static constexpr int TILE_K = BN * DQK * 2;
  static constexpr int TILE_V = BN * DV * 2;
  static constexpr int TILE_Q = BM * DQK * 2;
  static constexpr int TILE_DO = BM * DV * 2;
  static constexpr int TILE_DS = BN * BM * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_K;
  static constexpr int OFF_Q = OFF_V + TILE_V;
  static constexpr int OFF_DO = OFF_Q + 2 * TILE_Q;
  static constexpr int OFF_DS = OFF_DO + 2 * TILE_DO;
  static constexpr int OFF_QS = OFF_DS + TILE_DS;
  static constexpr int OFF_BAR = OFF_QS + 2 * QSTAT_FLOATS * 4;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + DV;
  static_assert(COL_DK + DQK <= 512, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
  // More than half an SM's shared memory: one CTA per SM, so a CTA never waits
  // for tensor memory held by a co-resident CTA that may be waiting on it.
  static_assert(BYTES > 116 * 1024, "one CTA per SM");
};

__device__ __forceinline__ void set_status(int* status, int bit) { atomicOr(status, bit); }

template <int DQK, int DV>
__global__ void __launch_bounds__(MAIN_THREADS, 1)
    sdpa_bwd_main(const __grid_constant__ MainMaps maps, const ChainParams p) {
  using L = MainLayout<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (tid == 0) set_status(p.status, STATUS_SMEM_ALIGN);
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
  int* unit_slot = reinterpret_cast<int*>(smem + L::OFF_MISC + 8);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bars[BAR_KV], 1);
    mbar_init(&bars[BAR_QFULL + 0], 1);
    mbar_init(&bars[BAR_QFULL + 1], 1);
    mbar_init(&bars[BAR_QEMPTY + 0], 1);
    mbar_init(&bars[BAR_QEMPTY + 1], 1);
    mbar_init(&bars[BAR_SFULL], 1);
    mbar_init(&bars[BAR_DPFULL], 1);
    mbar_init(&bars[BAR_PREADY], 256);
    mbar_init(&bars[BAR_G3DONE], 1);
    mbar_init(&bars[BAR_DSREADY], 256);
    mbar_init(&bars[BAR_DQFULL], 1);
    mbar_init(&bars[BAR_DQEMPTY], 256);
    mbar_init(&bars[BAR_RELAYGO], 1);
    mbar_init(&bars[BAR_RELAYDONE], 256);
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

  // Units are ordered key tile major: every head's key tile 0 first. Under a
  // causal mask low key tiles see the most query tiles, so the longest units
  // start first.
  const int BH = p.B * p.Hq;
  const int kt = unit / BH;
  const int bh = unit % BH;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hk = h / p.G;
  const int k0 = kt * BN;

  int Lq, Lk;
  batch_lengths(p, b, Lq, Lk);
  const int diag = p.bottom_right ? Lk - Lq : 0;
  const int Rp = p.window_right > 0 ? p.window_right : 0;
  const bool has_window = p.window_left >= 0;
  int qt_lo = 0, qt_hi = -1;
  if (k0 < Lk && Lq > 0) {
    const int k_last = min(k0 + BN - 1, Lk - 1);
    long long q_min = 0, q_max = Lq - 1;
    if (p.causal) q_min = max(0ll, (long long)k0 - diag - Rp);
    if (has_window) q_max = min(q_max, (long long)k_last - diag + p.window_left);
    if (q_min <= q_max) {
      qt_lo = (int)(q_min / BM);
      qt_hi = (int)(q_max / BM);
    }
  }
  const int n_iter = qt_hi - qt_lo + 1;  // may be 0

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_iter > 0) {
      mbar_arrive_expect_tx(&bars[BAR_KV], L::TILE_K + L::TILE_V);
      for (int blk = 0; blk < DQK / 64; ++blk)
        tma_load_3d(sK + blk * 16384, &maps.k, &bars[BAR_KV], blk * 64, k0, b * p.Hkv + hk);
      for (int blk = 0; blk < DV / 64; ++blk)
        tma_load_3d(sV + blk * 16384, &maps.v, &bars[BAR_KV], blk * 64, k0, b * p.Hkv + hk);
      pdl_wait_prior_grid();  // row statistics come from the preprocess kernel
      for (int it = 0; it < n_iter; ++it) {
        const int st = it & 1;
        if (it >= 2 && !mbar_wait(&bars[BAR_QEMPTY + st], ((it >> 1) - 1) & 1, abort_flag,
                                  WAIT_LIMIT_NS))
          break;
        const int qt = qt_hi - it;
        uint64_t* full = &bars[BAR_QFULL + st];
        mbar_arrive_expect_tx(full, L::TILE_Q + L::TILE_DO + QSTAT_FLOATS * 4);
        uint8_t* q_dst = sQ + st * L::TILE_Q;
        uint8_t* do_dst = sDO + st * L::TILE_DO;
        for (int blk = 0; blk < DQK / 64; ++blk)
          tma_load_3d(q_dst + blk * 16384, &maps.q, full, blk * 64, qt * BM, bh);
        for (int blk = 0; blk < DV / 64; ++blk)
          tma_load_3d(do_dst + blk * 16384, &maps.d_o, full, blk * 64, qt * BM, bh);
        bulk_load(sQS + st * QSTAT_FLOATS, p.qstat + ((long long)bh * p.n_qt + qt) * QSTAT_FLOATS,
                  QSTAT_FLOATS * 4, full);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    pdl_wait_prior_grid();
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t ID_SS_KK = idesc_bf16_f32(128, 128, false, false);  // G1, G2
      constexpr uint32_t ID_DV = idesc_bf16_f32(128, DV, false, true);       // G3
      constexpr uint32_t ID_DK = idesc_bf16_f32(128, DQK, false, true);      // G4
      constexpr uint32_t ID_DQ = idesc_bf16_f32(128, DQK, true, true);       // G5
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
      bool ok = mbar_wait(&bars[BAR_KV], 0, abort_flag, WAIT_LIMIT_NS);
      for (int it = 0; it < n_iter && ok; ++it) {
        const int st = it & 1, ph = it & 1;
        const uint32_t aQ = smem_u32(sQ + st * L::TILE_Q), aDO = smem_u32(sDO + st * L::TILE_DO);
        ok = mbar_wait(&bars[BAR_QFULL + st], (it >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
        // S region is rewritten by G1: the previous G3 (reads P^T there) must be done.
        if (ok && it > 0) ok = mbar_wait(&bars[BAR_G3DONE], ph ^ 1, abort_flag, WAIT_LIMIT_NS);
        if (!ok) break;
        tc_fence_after();
        // G1: S^T[key, query] = sum_d K[key, d] Q[query, d]  (both K-major)
#pragma unroll
        for (int s = 0; s < DQK / 16; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          mma_ss(tmem + L::COL_S, sdesc_sw128(aK + ko, 16, 1024), sdesc_sw128(aQ + ko, 16, 1024),
                 ID_SS_KK, s > 0);
        }
        mma_commit(&bars[BAR_SFULL]);
        // dP/dQ region: the previous dQ must have been read out.
        if (it > 0 && !mbar_wait(&bars[BAR_DQEMPTY], ph ^ 1, abort_flag, WAIT_LIMIT_NS)) break;
        tc_fence_after();
        // G2: dP^T[key, query] = sum_d V[key, d] dO[query, d]
#pragma unroll
        for (int s = 0; s < DV / 16; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          mma_ss(tmem + L::COL_DP, sdesc_sw128(aV + ko, 16, 1024),
                 sdesc_sw128(aDO + ko, 16, 1024), ID_SS_KK, s > 0);
        }
        mma_commit(&bars[BAR_DPFULL]);
        if (!mbar_wait(&bars[BAR_PREADY], ph, abort_flag, WAIT_LIMIT_NS)) break;
        tc_fence_after();
        // G3: dV[key, d] += sum_q P^T[key, q] dO[q, d]; P^T (bf16 pairs) sits in
        // columns [0,32) for queries 0..63 and [64,96) for queries 64..127.
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          const uint32_t a_col = L::COL_S + (s < 4 ? 8 * s : 64 + 8 * (s - 4));
          mma_ts(tmem + L::COL_DV, tmem + a_col, sdesc_sw128(aDO + s * 2048, 16384, 1024), ID_DV,
                 (it > 0 || s > 0));
        }
        mma_commit(&bars[BAR_G3DONE]);
        if (!mbar_wait(&bars[BAR_DSREADY], ph, abort_flag, WAIT_LIMIT_NS)) break;
        tc_fence_after();
        // G4: dK[key, d] += sum_q dS^T[key, q] Q[q, d]   (dS^T K-major, Q MN-major)
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          mma_ss(tmem + L::COL_DK, sdesc_sw128(aDS + ko, 16, 1024),
                 sdesc_sw128(aQ + s * 2048, 16384, 1024), ID_DK, (it > 0 || s > 0));
        }
        // G5: dQ[q, d] = sum_key dS[q, key] K[key, d]   (dS and K both MN-major)
#pragma unroll
        for (int s = 0; s < BN / 16; ++s) {
          mma_ss(tmem + L::COL_DP, sdesc_sw128(aDS + s * 2048, 16384, 1024),
                 sdesc_sw128(aK + s * 2048, 16384, 1024), ID_DQ, s > 0);
        }
        mma_commit(&bars[BAR_DQFULL]);
        if (it + 2 < n_iter) mma_commit(&bars[BAR_QEMPTY + st]);  // only if the stage is refilled
      }
    }
  } else {
    // ------------------------------------------------------------ compute warpgroups
    pdl_wait_prior_grid();
    const int wg = warp >> 2;          // 0: queries 0..63 of the tile, 1: 64..127
    const int quarter = warp & 3;      // tensor-memory lane quarter
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int k = k0 + row;            // this thread's key (S^T / dP^T lane)
    const bool row_dead = k >= Lk;
    const long long q_lo_vis = p.causal ? (long long)k - diag - Rp : -(1ll << 40);
    const long long q_hi_vis = has_window ? (long long)k - diag + p.window_left : (1ll << 40);
    const float scale_log2 = p.scale_log2;
    float P[64];
    bool ok = true;

    for (int it = 0; it < n_iter && ok; ++it) {
      const int st = it & 1, ph = it & 1;
      const int qt = qt_hi - it, q0 = qt * BM;
      const float* qs = sQS + st * QSTAT_FLOATS;
      const bool need_mask = (k0 + BN > Lk) ||
                             (p.causal && (long long)q0 < (long long)(k0 + BN - 1) - diag - Rp) ||
                             (has_window && (long long)(q0 + BM - 1) > (long long)k0 - diag + p.window_left);

      // ---- softmax replay: P^T from S^T. The row statistics were written by
      // TMA, so this thread waits on the stage's transaction barrier itself.
      if (!mbar_wait(&bars[BAR_QFULL + st], (it >> 1) & 1, abort_flag, WAIT_LIMIT_NS) ||
          !mbar_wait(&bars[BAR_SFULL], ph, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld32(t_lane + L::COL_S + wg * 64 + half * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = wg * 64 + half * 32 + j;
          P[half * 32 + j] = ex2_approx(fmaf(__uint_as_float(r[j]), scale_log2, -qs[c]));
        }
      }
      if (need_mask) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const long long q = q0 + wg * 64 + j;
          if (row_dead || q < q_lo_vis || q > q_hi_vis) P[j] = 0.f;
        }
      }
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = pack_bf16x2(P[c16 * 32 + 2 * i], P[c16 * 32 + 2 * i + 1]);
        tmem_st16(t_lane + L::COL_S + wg * 64 + c16 * 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[BAR_PREADY]);

      // ---- dS^T = P^T * (dP^T - delta) -> shared memory (K-major, swizzled)
      if (!mbar_wait(&bars[BAR_DPFULL], ph, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      uint8_t* ds_row = sDS + wg * 16384 + row * 128;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld32(t_lane + L::COL_DP + wg * 64 + half * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = half * 32 + ch * 8 + 2 * i;
            const int c = wg * 64 + j;
            const float d0 = P[j] * (__uint_as_float(r[ch * 8 + 2 * i]) - qs[BM + c]);
            const float d1 = P[j + 1] * (__uint_as_float(r[ch * 8 + 2 * i + 1]) - qs[BM + c + 1]);
            w[i] = pack_bf16x2(d0, d1);
          }
          const int chunk = half * 4 + ch;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[BAR_DSREADY]);

      // ---- dQ tile -> fp32 reductions (lanes are now queries)
      if (!mbar_wait(&bars[BAR_DQFULL], ph, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      constexpr int QC = DQK / 2;  // dQ columns per warpgroup
      uint32_t dq[QC];
#pragma unroll
      for (int c32 = 0; c32 < QC / 32; ++c32) {
        uint32_t r[32];
        tmem_ld32(t_lane + L::COL_DP + wg * QC + c32 * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) dq[c32 * 32 + j] = r[j];
      }
      tc_fence_before();
      mbar_arrive(&bars[BAR_DQEMPTY]);  // tensor memory may be reused; values are in registers

      int turn = 0;
      int* counter = nullptr;
      if (p.deterministic) {
        // Ordered relay: key tiles add into this query tile in ascending order.
        const int kv_lo = has_window
                              ? (int)max(0ll, floor_div((long long)q0 + diag - p.window_left, BN))
                              : 0;
        turn = kt - kv_lo;
        counter = p.counters + (long long)bh * p.n_qt + qt;
        if (tid == 0) {
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(counter) != turn) {
            __nanosleep(64);
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
              set_status(p.status, STATUS_TIMEOUT);
              break;
            }
          }
          mbar_arrive(&bars[BAR_RELAYGO]);
        }
        if (!mbar_wait(&bars[BAR_RELAYGO], ph, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      }
      float* dst = p.dq_accum + ((long long)bh * p.n_qt + qt) * (long long)BM * DQK;
#pragma unroll
      for (int i = 0; i < QC / 4; ++i) {
        const int cq = (wg * QC) / 4 + i;  // column quad
        red_add_v4(dst + ((long long)cq * BM + row) * 4, __uint_as_float(dq[4 * i]),
                   __uint_as_float(dq[4 * i + 1]), __uint_as_float(dq[4 * i + 2]),
                   __uint_as_float(dq[4 * i + 3]));
      }
      if (p.deterministic) {
        __threadfence();
        mbar_arrive(&bars[BAR_RELAYDONE]);
        if (tid == 0) {
          mbar_wait(&bars[BAR_RELAYDONE], ph, abort_flag, WAIT_LIMIT_NS);
          st_release_gpu(counter, turn + 1);
        }
      }
    }

    // ---- epilogue: dV and scale * dK from tensor memory, bf16, one key row per thread.
    // Every lane runs the (warp-collective) tensor-memory loads; only the stores
    // are predicated on the row being inside the tensor.
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    const bool store_row = k < p.Skv;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const int D = which ? DQK : DV;
      const uint32_t col0 = which ? L::COL_DK : L::COL_DV;
      const float mult = which ? p.scale : 1.f;
      __nv_bfloat16* base = which ? (p.dk_ws ? p.dk_ws : p.dk) : (p.dv_ws ? p.dv_ws : p.dv);
      const long long head = p.dk_ws ? (long long)bh : (long long)b * p.Hkv + hk;
      __nv_bfloat16* out = base + (head * p.Skv + k) * (long long)D + wg * (D / 2);
      for (int c32 = 0; c32 < D / 64; ++c32) {
        uint32_t r[32];
        if (n_iter > 0 && warp_ok) {
          tmem_ld32(t_lane + col0 + wg * (D / 2) + c32 * 32, r);
          tmem_ld_wait(r);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (store_row) {
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[v8 * 8 + 0]) * mult, __uint_as_float(r[v8 * 8 + 1]) * mult);
            o.y = pack_bf16x2(__uint_as_float(r[v8 * 8 + 2]) * mult, __uint_as_float(r[v8 * 8 + 3]) * mult);
            o.z = pack_bf16x2(__uint_as_float(r[v8 * 8 + 4]) * mult, __uint_as_float(r[v8 * 8 + 5]) * mult);
            o.w = pack_bf16x2(__uint_as_float(r[v8 * 8 + 6]) * mult, __uint_as_float(r[v8 * 8 + 7]) * mult);
            *reinterpret_cast<uint4*>(out + c32 * 32 + v8 * 8) = o;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, STATUS_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t main_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(sdpa_bwd_main<64, 64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       MainLayout<64, 64>::BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(sdpa_bwd_main<128, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MainLayout<128, 128>::BYTES);
}

// One CTA per (key tile, batch, query head) work unit.
cudaError_t launch_main(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.n_kt * p.B * p.Hq));
  if (p.Dqk == 64)
    return launch_kernel(sdpa_bwd_main<64, 64>, grid, dim3(MAIN_THREADS), MainLayout<64, 64>::BYTES,
                         s, true, maps, p);
  return launch_kernel(sdpa_bwd_main<128, 128>, grid, dim3(MAIN_THREADS),
                       MainLayout<128, 128>::BYTES, s, true, maps, p);
}

}  // namespace sdpa
