// sdpa_fwd.cu -- fused SDPA forward (O and the natural-log LSE) for sm_103a.
//
// What it computes: the forward whose outputs the backward consumes ("SDPA
// Backward (SM120)", API Usage: `o` and the natural-log `stats`; the masks of
// "Causal, sliding-window, and padding masks"; GQA/MQA head mapping; the sink
// token of the Capabilities list, which joins every row's softmax denominator
// without a value row):
//   S = scale Q K^T (masked entries removed), LSE = log(sum_k exp(S) [+ exp(sink)]),
//   O = sum_k exp(S - LSE) V.
// A row with no visible key and no sink gets LSE = -inf and O = 0; with a sink
// LSE = sink and O = 0.
//
// Schedule. One CTA owns 128 query rows of one (batch, query head) and walks the
// key tiles (128 keys) that any of its rows sees, in ascending order. Per key tile j:
//   G1  S   = Q K_j^T        -> tensor-memory slot j % 2 (128 fp32 columns)
//       P   = exp2(S * scale * log2e - m)   (the softmax warpgroup, one row per thread)
//           -> bf16 into the slot's first 64 columns
//   G2  O  += P V_j           (A = P from tensor memory, B = V_j MN-major)
// m is a per-row running reference that is raised only when the row's maximum
// exceeds it by more than 8 (in log2 units). Until then P stays below 2^8, which
// bf16 and fp32 hold exactly enough, so the O accumulator is rescaled only on
// those rare raises (after the previous G2 has completed). The row sum l is kept
// in fp32 alongside; at the end O / l and LSE = (m + log2 l) * ln 2.
//
// Warps: 0-3 the softmax warpgroup (thread = query row = tensor-memory lane), 4 the
// TMA producer (Q once, K/V stage ring), 5 the MMA issuer and tensor-memory owner,
// 6-7 idle. Tensor memory: slots at [0,128) and [128,256), O at [256, 256+D_v).
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

namespace fwd_kernel {

constexpr int THREADS = 256;
constexpr int BM = 128;  // query rows per CTA
constexpr int BK = 128;  // keys per tile
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;
constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units

enum : int {
  BAR_QFULL = 0,
  BAR_KVFULL = 1,   // + stage (up to 4)
  BAR_KVEMPTY = 5,  // + stage: G2 of the tile completed (K read by G1 before it)
  BAR_SFULL = 9,    // + slot: S in tensor memory
  BAR_PREADY = 11,  // + slot, 128 arrivals: P written
  BAR_PVDONE = 13,  // + slot: G2 of the slot's tile completed
  NUM_BARS = 15
};

template <int DQK, int DV>
struct Layout {
  static constexpr int BLK = 128 * 128;            // one 64-column block of a 128-row tile
  static constexpr int TILE_Q = BM * DQK * 2;
  static constexpr int TILE_K = BK * DQK * 2;
  static constexpr int TILE_V = BK * DV * 2;
  static constexpr int STAGE = TILE_K + TILE_V;
  static constexpr int NS_FIT = (232448 - TILE_Q - NUM_BARS * 8 - 64) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = TILE_Q;
  static constexpr int OFF_BAR = OFF_KV + NS * STAGE;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // More than half an SM's shared memory keeps one CTA per SM, so the 512
  // tensor-memory columns are never contended.
  static constexpr int BYTES_RAW = OFF_MISC + 64;
  static constexpr int BYTES = BYTES_RAW > 120 * 1024 ? BYTES_RAW : 120 * 1024;
  static constexpr uint32_t COL_O = 256;
  static_assert(NS >= 2, "stage ring");
  static_assert(COL_O + DV <= 512, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(TILE_Q % 1024 == 0 && TILE_K % 1024 == 0 && TILE_V % 1024 == 0, "alignment");
  static_assert(DV <= DQK, "O staging reuses the Q tile");
};

}  // namespace fwd_kernel

template <int DQK, int DV>
__global__ void __launch_bounds__(fwd_kernel::THREADS, 1)
    sdpa_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p) {
  using namespace fwd_kernel;
  using L = Layout<DQK, DV>;
  constexpr int NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sKV = smem + L::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  // Work item: query tile qt (descending, so that under a causal mask the
  // longest items start first) of head bh.
  const int BH = p.B * p.Hq;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, h = bh % p.Hq, kvh = b * p.Hkv + h / p.G;
  const int q0 = qt * BM;
  int Lq = p.Sq, Lk = p.Skv;
  if (p.seq_q_lens) Lq = min(max(p.seq_q_lens[b], 0), p.Sq);
  if (p.seq_kv_lens) Lk = min(max(p.seq_kv_lens[b], 0), p.Skv);
  const long long diag = p.bottom_right ? (long long)Lk - Lq : 0;
  const long long Rp = p.window_right > 0 ? p.window_right : 0;
  const bool has_window = p.window_left >= 0;
  // Key tiles any live row of this tile sees: [kt_lo, kt_hi].
  int kt_lo = 0, kt_hi = -1;
  {
    const long long q_last = min(q0 + BM, Lq) - 1;
    if (q0 < Lq && Lk > 0) {
      long long k_hi = Lk - 1, k_lo = 0;
      if (p.causal) k_hi = min(k_hi, q_last + diag + Rp);
      if (has_window) k_lo = max(0ll, (long long)q0 + diag - p.window_left);
      if (k_lo <= k_hi) {
        kt_lo = (int)(k_lo / BK);
        kt_hi = (int)(k_hi / BK);
      }
    }
  }
  const int n = kt_hi - kt_lo + 1;  // may be 0

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NUM_BARS; ++i)
      mbar_init(&bars[i], (i == BAR_PREADY || i == BAR_PREADY + 1) ? 128 : 1);
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    prefetch_tmap(&maps.o);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(&bars[BAR_QFULL], L::TILE_Q);
      for (int blk = 0; blk < DQK / 64; ++blk)
        tma_load_3d(sQ + blk * L::BLK, &maps.q, &bars[BAR_QFULL], blk * 64, q0, bh);
      for (int j = 0; j < n; ++j) {
        const int st = j % NS;
        if (j >= NS &&
            !mbar_wait(&bars[BAR_KVEMPTY + st], ((j / NS) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
          break;
        const int k0 = (kt_lo + j) * BK;
        uint8_t* sK = sKV + st * L::STAGE;
        uint8_t* sV = sK + L::TILE_K;
        uint64_t* full = &bars[BAR_KVFULL + st];
        mbar_arrive_expect_tx(full, L::STAGE);
        for (int blk = 0; blk < DQK / 64; ++blk)
          tma_load_3d(sK + blk * L::BLK, &maps.k, full, blk * 64, k0, kvh);
        for (int blk = 0; blk < DV / 64; ++blk)
          tma_load_3d(sV + blk * L::BLK, &maps.v, full, blk * 64, k0, kvh);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Order: G1(0), then for j >= 1: G1(j), G2(j-1); finally G2(n-1). G1(j)
    // reuses the slot of tile j-2, whose P G2(j-2) read; G2(j-1) needs P(j-1).
    constexpr uint32_t ID_S = idesc_bf16_f32(BM, BK, false, false);  // S = Q K^T
    constexpr uint32_t ID_O = idesc_bf16_f32(BM, DV, false, true);   // O += P V
    constexpr uint64_t T_KMAJ = sdesc_sw128_template(16, 1024);
    constexpr uint64_t T_MN_V = sdesc_sw128_template(L::BLK, 1024);
    bool ok = n > 0 && mbar_wait(&bars[BAR_QFULL], 0, abort_flag, WAIT_LIMIT_NS);
    const uint32_t aQ = smem_u32(sQ);
    for (int j = 0; j <= n && ok; ++j) {
      if (j < n) {
        const int st = j % NS, s = j & 1;
        ok = mbar_wait(&bars[BAR_KVFULL + st], (j / NS) & 1, abort_flag, WAIT_LIMIT_NS);
        if (ok && j >= 2) ok = mbar_wait(&bars[BAR_PVDONE + s], ((j - 2) >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
        if (!ok) break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          const uint32_t aK = smem_u32(sKV + st * L::STAGE);
#pragma unroll
          for (int k = 0; k < DQK / 16; ++k) {
            const uint32_t ko = (k >> 2) * L::BLK + (k & 3) * 32;
            mma_ss(tmem + 128u * s, sdesc_at(T_KMAJ, aQ + ko), sdesc_at(T_KMAJ, aK + ko), ID_S, k > 0);
          }
          mma_commit(&bars[BAR_SFULL + s]);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int u = j - 1, su = u & 1, stu = u % NS;
        if (!mbar_wait(&bars[BAR_PREADY + su], (u >> 1) & 1, abort_flag, WAIT_LIMIT_NS)) break;
        __syncwarp();
        tc_fence_after();
        if (elect_one()) {
          const uint32_t aV = smem_u32(sKV + stu * L::STAGE + L::TILE_K);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_ts(tmem + L::COL_O, tmem + 128u * su + 8 * k, sdesc_at(T_MN_V, aV + k * 2048), ID_O,
                   (u > 0 || k > 0));
          mma_commit(&bars[BAR_PVDONE + su]);
          if (u + NS < n) mma_commit(&bars[BAR_KVEMPTY + stu]);
        }
        __syncwarp();
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax warpgroup
    const int row = warp * 32 + lane;
    const int q = q0 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    const float c = p.scale_log2;
    const bool live = q < Lq;
    // Running reference m (log2 units) and row sum l; the sink starts them.
    float m = -INFINITY, l = 0.f;
    if (p.sink) {
      m = p.sink[h] * 1.4426950408889634f;
      l = 1.f;
    }
    bool ok = true;
    const long long k_vis_hi = p.causal ? (long long)q + diag + Rp : (1ll << 40);
    const long long k_vis_lo = has_window ? (long long)q + diag - p.window_left : -(1ll << 40);
    for (int j = 0; j < n && ok; ++j) {
      const int s = j & 1;
      const int k0 = (kt_lo + j) * BK;
      if (!mbar_wait(&bars[BAR_SFULL + s], (j >> 1) & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c32 = 0; c32 < 4; ++c32) tmem_ld32(t_lane + 128u * s + c32 * 32, sr[c32]);
#pragma unroll
      for (int c32 = 0; c32 < 4; ++c32) tmem_ld_wait(sr[c32]);
      // Visible keys of this row within the tile: [v_lo, v_hi] relative to k0.
      int v_lo = 0, v_hi = BK - 1;
      if (!live) {
        v_hi = -1;
      } else {
        v_hi = (int)min((long long)BK - 1, min((long long)Lk - 1, k_vis_hi) - k0);
        v_lo = (int)max(0ll, k_vis_lo - k0);
      }
      // A tile whose keys this row all sees (every tile but the edges) takes the
      // unmasked path: the maximum of the raw scores, then one FFMA + ex2 each.
      const bool full = v_lo == 0 && v_hi == BK - 1;
      float mt = -INFINITY;
      if (full) {
#pragma unroll
        for (int i = 0; i < BK; ++i) mt = fmaxf(mt, __uint_as_float(sr[i >> 5][i & 31]));
        mt *= c;  // c > 0
      } else {
#pragma unroll
        for (int i = 0; i < BK; ++i)
          if (i >= v_lo && i <= v_hi) mt = fmaxf(mt, __uint_as_float(sr[i >> 5][i & 31]) * c);
      }
      // Raise the reference when the tile's maximum exceeds it by more than the
      // threshold (or when it is the row's first visible key).
      const bool raise = mt > m + RESCALE_THRESHOLD || (m == -INFINITY && mt > -INFINITY);
      const float m_new = raise ? mt : m;
      const float alpha = raise ? ex2_approx(m - m_new) : 1.f;  // 0 when m was -inf
      // O holds this row's contributions of tiles < j when l > 0 and j > 0. Its
      // lane is rescaled once G2(j-1) has completed (no G2 reads or writes O
      // meanwhile: G2(j) waits for this warpgroup's P_READY(j)).
      const bool rescale_o = raise && j > 0 && l > 0.f;
      if (__any_sync(0xffffffffu, rescale_o)) {
        if (!mbar_wait(&bars[BAR_PVDONE + (s ^ 1)], ((j - 1) >> 1) & 1, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float f = rescale_o ? alpha : 1.f;
#pragma unroll 1
        for (int c32 = 0; c32 < DV / 32; ++c32) {
          uint32_t o[32];
          tmem_ld32(t_lane + L::COL_O + c32 * 32, o);
          tmem_ld_wait(o);
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w0[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            w1[i] = __float_as_uint(__uint_as_float(o[16 + i]) * f);
          }
          tmem_st16(t_lane + L::COL_O + c32 * 32, w0);
          tmem_st16(t_lane + L::COL_O + c32 * 32 + 16, w1);
        }
        tmem_st_wait();
      }
      l *= alpha;
      m = m_new;
      // P = exp2(x - m) on visible keys, written as bf16 pairs into the slot's
      // first 64 columns (this thread's own lane, already read above).
      float rs0 = 0.f, rs1 = 0.f;
      const float neg_m = -m;
#pragma unroll
      for (int c16 = 0; c16 < 4; ++c16) {
        uint32_t w[16];
        if (full) {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2]), c, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2 + 1]), c, neg_m));
            rs0 += p0;
            rs1 += p1;
            w[i2] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const int i = c16 * 32 + 2 * i2;
            const float p0 = (i >= v_lo && i <= v_hi)
                                 ? ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2]), c, neg_m)) : 0.f;
            const float p1 = (i + 1 >= v_lo && i + 1 <= v_hi)
                                 ? ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2 + 1]), c, neg_m)) : 0.f;
            rs0 += p0;
            rs1 += p1;
            w[i2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(t_lane + 128u * s + c16 * 16, w);
      }
      l += rs0 + rs1;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[BAR_PREADY + s]);
    }

    // ---- epilogue: O / l (bf16) staged row by row into the Q tile in the
    // 128-byte-swizzled box layout and written by TMA (rows past S_q dropped);
    // LSE in natural-log units.
    const bool have_o = n > 0 && ok;
    if (have_o) {
      ok = mbar_wait(&bars[BAR_PVDONE + ((n - 1) & 1)], ((n - 1) >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
    }
    const bool warp_ok = __all_sync(0xffffffffu, ok);
    if (have_o && warp_ok) tc_fence_after();
    const float inv_l = (l > 0.f && live) ? 1.f / l : 0.f;
    uint8_t* dst_row = sQ + row * 128;
#pragma unroll 1
    for (int c32 = 0; c32 < DV / 32; ++c32) {
      uint32_t o[32];
      if (have_o && warp_ok) {
        tmem_ld32(t_lane + L::COL_O + c32 * 32, o);
        tmem_ld_wait(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
#pragma unroll
      for (int v8 = 0; v8 < 4; ++v8) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[v8 * 8 + 0]) * inv_l, __uint_as_float(o[v8 * 8 + 1]) * inv_l);
        w.y = pack_bf16x2(__uint_as_float(o[v8 * 8 + 2]) * inv_l, __uint_as_float(o[v8 * 8 + 3]) * inv_l);
        w.z = pack_bf16x2(__uint_as_float(o[v8 * 8 + 4]) * inv_l, __uint_as_float(o[v8 * 8 + 5]) * inv_l);
        w.w = pack_bf16x2(__uint_as_float(o[v8 * 8 + 6]) * inv_l, __uint_as_float(o[v8 * 8 + 7]) * inv_l);
        const int piece = (c32 & 1) * 4 + v8;
        *reinterpret_cast<uint4*>(dst_row + (c32 >> 1) * L::BLK + ((piece ^ (row & 7)) << 4)) = w;
      }
    }
    if (q < p.Sq) {
      float lse = -INFINITY;
      if (l > 0.f) lse = (m + __log2f(l)) * 0.6931471805599453f;  // a padded row with a sink: the sink
      p.lse[(long long)bh * p.Sq + q] = lse;
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (row == 0) {
      for (int blk = 0; blk < DV / 64; ++blk) tma_store_3d(&maps.o, sQ + blk * L::BLK, blk * 64, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV>
static cudaError_t set_fwd_smem() {
  return cudaFuncSetAttribute(sdpa_fwd_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fwd_kernel::Layout<DQK, DV>::BYTES);
}

cudaError_t fwd_kernel_setup() {
  cudaError_t e = set_fwd_smem<64, 64>();
  if (e == cudaSuccess) e = set_fwd_smem<128, 128>();
  if (e == cudaSuccess) e = set_fwd_smem<192, 128>();
  return e;
}

cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.n_qt * p.B * p.Hq));
  const dim3 block(fwd_kernel::THREADS);
  if (p.Dqk == 64 && p.Dv == 64)
    return launch_kernel(sdpa_fwd_kernel<64, 64>, grid, block, fwd_kernel::Layout<64, 64>::BYTES, s,
                         false, maps, p);
  if (p.Dqk == 128 && p.Dv == 128)
    return launch_kernel(sdpa_fwd_kernel<128, 128>, grid, block, fwd_kernel::Layout<128, 128>::BYTES,
                         s, false, maps, p);
  if (p.Dqk == 192 && p.Dv == 128)
    return launch_kernel(sdpa_fwd_kernel<192, 128>, grid, block, fwd_kernel::Layout<192, 128>::BYTES,
                         s, false, maps, p);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
