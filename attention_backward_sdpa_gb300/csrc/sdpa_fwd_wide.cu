// sdpa_fwd_wide.cu -- the fused SDPA forward at head dim 256 (D_qk = D_v = 256).
//
// It computes what sdpa_fwd.cu computes -- O and the natural-log LSE of the
// masked softmax ("SDPA Backward (SM120)", API Usage: `o` and `stats`), with the
// masks of "Causal, sliding-window, and padding masks", the GQA/MQA head map,
// the sink logit and the additive bias of the Capabilities list -- for the head
// size that kernel's tensor-memory plan cannot hold. There each half of a row's
// keys keeps an O accumulator of its own (2 x D_v columns) beside two 128-column
// score slots; at D_v = 256 a single O already takes half of tensor memory.
// Here:
//   - tensor memory: the two S/P slots at [0, 256), one O at [256, 512);
//   - one softmax reference m per row, shared by the two softmax warpgroups
//     (warps w and w + 4 read the same lanes; warpgroup h takes keys
//     [64 h, 64 h + 64) of each tile). Each takes the maximum of its 64 scores,
//     the two exchange it in shared memory at a named barrier, and both apply
//     the same raise rule to the same m (raised only when the tile's maximum
//     exceeds it by more than 8 in log2 units), so the P of both halves lands in
//     O on one scale. On a raise each warpgroup rescales its 128 columns of O;
//     the row sums l_0, l_1 stay per warpgroup and add at the end;
//   - P packed into the slot's first 64 columns (warpgroup h at [32 h, 32 h + 32)),
//     written after the exchange, when both have read their scores;
//   - shared memory holds Q (64 KB), one K tile and one V tile (64 KB each), 192
//     KB in all, moved in 16 KB pieces with a barrier pair each: K by 64-column
//     block, V by 32-key row group. Two producers: warp 8 loads Q and each
//     piece of K(j + 1) as soon as G1(j)'s MMAs over that piece have completed;
//     warp 11 does the same for V(j + 1) after G2(j). Several pieces are then in
//     flight at once: with whole tiles (one load in flight per buffer) the
//     loads' latency paced the kernel at about 4,950 cycles a tile against
//     2,048 of tensor work.
//   Per key tile j (slot s = j % 2):
//     G1  S_s = Q K_j^T                        (16 MMAs 128x128x16, warp 9)
//         P = exp2(S scale log2e [+ bias log2e] - m) -> bf16 pairs in slot s
//     G2  O (+)= P V_j                         (8 MMAs 128x256x16, warp 10)
// The schedule is persistent, as in sdpa_fwd.cu: one CTA per SM takes items
// (128 query rows of one batch and query head, longest first) from a ticket and
// publishes each to the other roles through a ring of four entries.
#include <cuda.h>
#include <cuda_bf16.h>

#include "sdpa_fwd.cuh"

namespace sdpa {

namespace fwd_wide {

using fwd_shared::BK;
using fwd_shared::BM;
using fwd_shared::RESCALE_THRESHOLD;
using fwd_shared::WAIT_LIMIT_NS;
constexpr int D = 256;
constexpr int THREADS = 384;
constexpr int BLK = 128 * 128;         // one 64-column block of a 128-row tile (16 KB)
constexpr int TILE = 128 * D * 2;      // a Q, K or V tile (64 KB)
constexpr uint32_t COL_O = 256;        // O accumulator columns [256, 512)
constexpr int RING = 4;                // items published by the ticket taker
constexpr int RING_READERS = 4;        // warps 0 (for the softmax warpgroups), 9, 10 and 11
// Register split: launched at 168 per thread, the control warpgroup drops to 72
// (the per-piece issue loops spilled at 56) and the softmax warpgroups grow to
// 216: 128 x (72 + 216 + 216) = 64,512 = 384 x 168.
constexpr uint32_t REGS_CTRL = 72, REGS_SOFTMAX = 216;
static_assert(128 * (REGS_CTRL + 2 * REGS_SOFTMAX) <= THREADS * 168, "register split");

// K and V move in pieces of 16 KB, each with a barrier pair of its own: K(j)
// by 64-column block (G1's MMAs walk the head dim, four MMAs per block), V(j)
// by 32-key row group (G2's MMAs walk the keys, two MMAs per group). A piece is
// replaced as soon as the MMAs that read it have completed, so the next tile's
// first pieces load while the current GEMM still reads the last ones.
constexpr int NPIECE = 4;
constexpr int PIECE = TILE / NPIECE;
enum : int {
  BAR_QFULL = 0,   // the item's Q landed
  BAR_QEMPTY = 1,  // the item's last G1 completed: Q may be replaced
  BAR_KFULL = 2,   // + block: K(j)'s 64-column block landed
  BAR_KEMPTY = 6,  // + block: G1(j)'s MMAs over the block completed
  BAR_VFULL = 10,  // + row group: V(j)'s 32 keys landed
  BAR_VEMPTY = 14, // + row group: G2(j)'s MMAs over those keys completed
  BAR_SFULL = 18,  // + slot: S in tensor memory
  BAR_PREADY = 20, // + slot, 256 arrivals: P written (both warpgroups)
  BAR_PVDONE = 22, // + slot: G2 of the slot's tile completed
  BAR_RFULL = 24,  // + ring entry: an item published
  BAR_REMPTY = BAR_RFULL + RING,  // + ring entry, RING_READERS arrivals
  NUM_BARS = BAR_REMPTY + RING
};

constexpr int OFF_Q = 0;
constexpr int OFF_K = TILE;
constexpr int OFF_V = 2 * TILE;
constexpr int OFF_BAR = 3 * TILE;
constexpr int OFF_XT = OFF_BAR + NUM_BARS * 8;  // tile maxima: [2 parity][2 warpgroup][128 rows]
constexpr int OFF_XL = OFF_XT + 2 * 256 * 4;    // row sums at the end: [2 warpgroup][128 rows]
constexpr int OFF_MISC = OFF_XL + 256 * 4;      // tensor-memory base, abort flag, ring
constexpr int BYTES = OFF_MISC + 64;
static_assert(BYTES <= 232448, "shared memory budget");
static_assert(BYTES > 116 * 1024, "one CTA per SM: the 512 tensor-memory columns are never contended");

}  // namespace fwd_wide

// Tickets of this kernel's launches, one counter pair per launch slot, used as
// in sdpa_fwd.cu (the last CTA of a launch resets its slot).
__device__ int g_fwd_wide_ticket[fwd_shared::FWD_SLOTS];
__device__ int g_fwd_wide_done[fwd_shared::FWD_SLOTS];

// BIAS adds the additive bias (FwdParams::bias) to the scaled scores. F16: fp16
// io tensors (and fp16 P for the PV GEMM) instead of bf16.
template <bool BIAS, bool F16>
__global__ void __launch_bounds__(fwd_wide::THREADS, 1)
    sdpa_fwd_wide_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p, const int ticket_slot) {
  using namespace fwd_wide;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + OFF_MISC + 16);  // [RING] items
  volatile int* sitem = ring + RING;  // [2] the softmax warpgroups' current item, by parity
  const int n_items = p.n_qt * p.B * p.Hq;

  // Item e of this CTA, read from the ring by one thread (which releases the
  // entry): -1 at the end, or when a wait gave up.
  auto ring_take = [&](int e) -> int {
    const int r = e % RING;
    if (!mbar_wait(&bars[BAR_RFULL + r], (e / RING) & 1, abort_flag, WAIT_LIMIT_NS)) return -1;
    const int it = ring[r];
    mbar_arrive(&bars[BAR_REMPTY + r]);
    return it;
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NUM_BARS; ++i)
      mbar_init(&bars[i], (i == BAR_PREADY || i == BAR_PREADY + 1) ? 256
                          : (i >= BAR_REMPTY && i < BAR_REMPTY + RING) ? RING_READERS : 1);
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
  }
  if (warp == 11 && lane == 0) prefetch_tmap(&maps.v);
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Every role walks the same items, in the order the ticket taker drew them,
  // and counts the key tiles over all of them (g), so that the K and V buffers,
  // the two slots and their barrier phases run on across items; ni counts the
  // items with at least one key tile (the Q buffer's phases). Items whose rows
  // see no key are written by the softmax warps alone. The producers and the
  // MMA issuers run on lane 0 of their warps.
  if (warp >= 8) {
    regs_decrease<REGS_CTRL>();
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------- tickets, Q and K
      int g = 0, ni = 0;
      bool ok = true;
      for (int e = 0; ok; ++e) {
        const int r = e % RING;
        if (e >= RING && !mbar_wait(&bars[BAR_REMPTY + r], ((e / RING) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
          break;
        int it = atomicAdd(&g_fwd_wide_ticket[ticket_slot], 1);
        if (it >= n_items) it = -1;
        ring[r] = it;
        mbar_arrive(&bars[BAR_RFULL + r]);
        if (it < 0) break;
        const FwdItem w = fwd_item(p, it);
        if (w.n <= 0) continue;
        for (int j = 0; j < w.n && ok; ++j, ++g) {
          // Block b of K(g) replaces that of K(g - 1) once G1(g - 1)'s MMAs over
          // it have completed. On an item's first tile that G1 was the previous
          // item's last, whose completion also frees Q.
          const int k0 = (w.kt_lo + j) * BK;
          for (int b = 0; b < NPIECE && ok; ++b) {
            if (g >= 1) ok = mbar_wait(&bars[BAR_KEMPTY + b], (g - 1) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[BAR_KFULL + b], PIECE);
            tma_load_3d(sK + b * BLK, &maps.k, &bars[BAR_KFULL + b], b * 64, k0, w.kvh);
          }
          if (ok && j == 0) {
            if (ni >= 1) ok = mbar_wait(&bars[BAR_QEMPTY], (ni - 1) & 1, abort_flag, WAIT_LIMIT_NS);
            if (ok) {
              mbar_arrive_expect_tx(&bars[BAR_QFULL], TILE);
              for (int blk = 0; blk < D / 64; ++blk)
                tma_load_3d(sQ + blk * BLK, &maps.q, &bars[BAR_QFULL], blk * 64, w.q0, w.bh);
            }
          }
        }
        ++ni;
      }
    } else if (warp == 11 && lane == 0) {
      // ---------------------------------------------------- V
      int g = 0;
      bool ok = true;
      for (int e = 0; ok; ++e) {
        const int it = ring_take(e);
        if (it < 0) break;
        const FwdItem w = fwd_item(p, it);
        for (int j = 0; j < w.n && ok; ++j, ++g) {
          // Keys 32 r .. 32 r + 31 of V(g) replace those of V(g - 1) once G2(g - 1)'s
          // MMAs over them have completed: four 32-row boxes, one per 64-column
          // block (the V map's boxes are 32 rows high).
          const int k0 = (w.kt_lo + j) * BK;
          for (int r = 0; r < NPIECE && ok; ++r) {
            if (g >= 1) ok = mbar_wait(&bars[BAR_VEMPTY + r], (g - 1) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[BAR_VFULL + r], PIECE);
            for (int blk = 0; blk < D / 64; ++blk)
              tma_load_3d(sV + blk * BLK + r * 32 * 128, &maps.v, &bars[BAR_VFULL + r], blk * 64, k0 + 32 * r,
                          w.kvh);
          }
        }
      }
    } else if (warp == 9 && lane == 0) {
      // ---------------------------------------------------- G1: S = Q K^T
      constexpr uint32_t ID_S = idesc_io(BM, BK, false, false, F16);
      constexpr uint64_t T_KMAJ = sdesc_sw128_template(16, 1024);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK);
      int g = 0, ni = 0;
      bool ok = true;
      for (int e = 0; ok; ++e) {
        const int it = ring_take(e);
        if (it < 0) break;
        const FwdItem w = fwd_item(p, it);
        if (w.n <= 0) continue;
        ok = mbar_wait(&bars[BAR_QFULL], ni & 1, abort_flag, WAIT_LIMIT_NS);
        for (int j = 0; j < w.n && ok; ++j, ++g) {
          const int s = g & 1;
          // The slot held P(g - 2) until G2(g - 2) read it.
          if (g >= 2) ok = mbar_wait(&bars[BAR_PVDONE + s], ((g - 2) >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
          for (int b = 0; b < NPIECE && ok; ++b) {
            ok = mbar_wait(&bars[BAR_KFULL + b], g & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int k = 4 * b + kk;
              const uint32_t ko = b * BLK + kk * 32;
              mma_ss(tmem + 128u * s, sdesc_at(T_KMAJ, aQ + ko), sdesc_at(T_KMAJ, aK + ko), ID_S, k > 0);
            }
            mma_commit(&bars[BAR_KEMPTY + b]);
          }
          if (!ok) break;
          mma_commit(&bars[BAR_SFULL + s]);
          if (j == w.n - 1) mma_commit(&bars[BAR_QEMPTY]);
        }
        ++ni;
      }
    } else if (warp == 10 && lane == 0) {
      // ---------------------------------------------------- G2: O += P V
      constexpr uint32_t ID_O = idesc_io(BM, D, false, true, F16);
      constexpr uint64_t T_MN_V = sdesc_sw128_template(BLK, 1024);
      const uint32_t aV = smem_u32(sV);
      int g = 0;
      bool ok = true;
      for (int e = 0; ok; ++e) {
        const int it = ring_take(e);
        if (it < 0) break;
        const FwdItem w = fwd_item(p, it);
        for (int u = 0; u < w.n && ok; ++u, ++g) {
          const int s = g & 1;
          // (The previous item's epilogue has read O before any P of this item
          // is written: the same threads do both, in that order.)
          ok = mbar_wait(&bars[BAR_PREADY + s], (g >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
          // Keys 16 k .. 16 k + 15 of P sit in the slot's columns [8 k, 8 k + 8);
          // row group r of V holds keys 32 r .. 32 r + 31 (MMAs 2 r and 2 r + 1).
          for (int r = 0; r < NPIECE && ok; ++r) {
            ok = mbar_wait(&bars[BAR_VFULL + r], g & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const int k = 2 * r + kk;
              mma_ts(tmem + COL_O, tmem + 128u * s + 8u * k, sdesc_at(T_MN_V, aV + k * 2048), ID_O,
                     (u > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&bars[BAR_VEMPTY + r]);
          }
          if (!ok) break;
          mma_commit(&bars[BAR_PVDONE + s]);
        }
      }
    }
  } else {
    regs_increase<REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax warpgroups
    const int half = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    float* xt = reinterpret_cast<float*>(smem + OFF_XT);
    float* xl = reinterpret_cast<float*>(smem + OFF_XL);
    const float c = p.scale_log2;
    const long long Rp = p.window_right > 0 ? p.window_right : 0;
    const bool has_window = p.window_left >= 0;
    const int i0 = half * 64;  // this warpgroup's first key within a tile
    // With a bias the scores are rewritten in place as x = s * c + bias * log2e,
    // and everything below reads them with the factor cs = 1 instead of c.
    const float cs = BIAS ? 1.f : c;
    uint16_t* const o_base = static_cast<uint16_t*>(p.o);
    const size_t o_bytes = (size_t)p.B * p.Hq * p.Sq * D * 2;
    // O rows go out in 32-byte stores when every 16-column piece is 32-byte
    // aligned (the base 32-byte aligned, D_v a multiple of 16), else 16-byte ones.
    const bool o_sector = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0 && (p.Dv & 15) == 0;
    int g = 0;
    bool ok = true;
    bool have_next = false;  // the item for this e was taken during the previous epilogue
    for (int e = 0; ok; ++e) {
      // One thread takes the item for all eight warps, so that they never
      // disagree on it (a wait that gives up can do so in one reader and not
      // in another) and meet at the same named barriers: during the previous
      // item's epilogue, whose barrier hands it over, else here with a barrier
      // of its own. Double-buffered by parity: a slot is rewritten only after a
      // later barrier that every reader of it has passed.
      if (!have_next) {
        if (warp == 0 && lane == 0) sitem[e & 1] = ring_take(e);
        named_bar_sync(3, 256);
      }
      have_next = false;
      const int it = sitem[e & 1];
      if (it < 0) break;
      const FwdItem w = fwd_item(p, it);
      const int q = w.q0 + row;
      const long long orow = (long long)w.bh * p.Sq + q;  // O / LSE row
      if (w.n <= 0) {
        // No row of this item sees a key: O = 0 and LSE = -inf, or the sink logit.
        if (half == 0 && q < p.Sq) {
          uint4* o = reinterpret_cast<uint4*>(o_base + orow * D);
          if (in_bounds(p.status, o, (size_t)D * 2, p.o, o_bytes))
            for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[orow] = p.sink ? p.sink[w.h] : -INFINITY;
        }
        continue;
      }
      const bool live = q < w.Lq;
      // The row's reference (common to both warpgroups) and this warpgroup's sum;
      // the sink joins warpgroup 0's sum.
      float m = -INFINITY, l = 0.f;
      if (p.sink) {
        m = p.sink[w.h] * 1.4426950408889634f;
        l = half == 0 ? 1.f : 0.f;
      }
      const long long k_vis_hi = p.causal ? (long long)q + w.diag + Rp : (1ll << 40);
      const long long k_vis_lo = has_window ? (long long)q + w.diag - p.window_left : -(1ll << 40);
      const long long bias_row =
          BIAS ? (long long)(w.bh / p.Hq) * p.bias_bstride + ((long long)w.h * p.Sq + q) * p.Skv : 0;
      for (int j = 0; j < w.n; ++j, ++g) {
        const int s = g & 1;
        const int k0 = (w.kt_lo + j) * BK;
        uint32_t braw[BIAS ? 64 : 1];
        bool bpacked = false;
        if constexpr (BIAS) {
          load_fwd_bias_row(p, bias_row, k0 + i0, live, braw, bpacked);
          const int kp = k0 + 2 * BK + i0;  // the row's segment of the tile after next into L2
          if (live && j + 2 < w.n && kp < p.Skv) {
            const char* a = static_cast<const char*>(p.bias) + (bias_row + kp) * (p.bias_fp32 ? 4 : 2);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
            if (p.bias_fp32 && kp + 32 < p.Skv) asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 128));
          }
        }
        // A wait that gave up (here or at a rescale) reaches every softmax thread
        // through the OR of the exchange barrier, so that all 256 leave the tile
        // loop at the same tile and meet again at the epilogue's barriers.
        const bool wok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[BAR_SFULL + s], (g >> 1) & 1,
                                                                  abort_flag, WAIT_LIMIT_NS));
        uint32_t sr[2][32];
        float mt_h = -INFINITY;
        int v_lo = 0, v_hi = -1;
        bool full = false;
        if (wok) {
          tc_fence_after();
          tmem_ld32(t_lane + 128u * s + i0, sr[0]);
          tmem_ld32(t_lane + 128u * s + i0 + 32, sr[1]);
          tmem_ld_wait(sr[0]);
          tmem_ld_wait(sr[1]);
          if constexpr (BIAS) add_bias_row(p, c, braw, bpacked, sr);
          // Visible keys of this row within the tile: [v_lo, v_hi] relative to k0.
          if (live) {
            v_hi = (int)min((long long)BK - 1, min((long long)w.Lk - 1, k_vis_hi) - k0);
            v_lo = (int)max(0ll, k_vis_lo - k0);
          }
          // Unmasked path when this warpgroup's 64 keys are visible to the whole
          // warp (warp-uniform: the tensor-memory stores below are .sync.aligned).
          full = __all_sync(0xffffffffu, v_lo <= i0 && v_hi >= i0 + 63);
          float mp[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) mp[a] = -INFINITY;
          if (full) {
#pragma unroll
            for (int i = 0; i < 64; ++i) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(sr[i >> 5][i & 31]));
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i0 + i >= v_lo && i0 + i <= v_hi) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(sr[i >> 5][i & 31]));
          }
          mt_h = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                       fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * cs;  // cs > 0
        }
        // Exchange of the two warpgroups' maxima (double-buffered by tile parity:
        // a thread rewrites a parity only after the next tile's barrier, which
        // every reader of this one has passed).
        float* xg = xt + (g & 1) * 256;
        xg[half * 128 + row] = mt_h;
        if (named_bar_sync_or(2, 256, !wok)) {
          ok = false;
          break;
        }
        const float mt = fmaxf(xg[row], xg[128 + row]);
        // Raise the reference when the tile's maximum exceeds it by more than the
        // threshold (or when it is the row's first visible key): the same
        // decision in both warpgroups.
        const bool raise = mt > m + RESCALE_THRESHOLD || (m == -INFINITY && mt > -INFINITY);
        const float m_new = raise ? mt : m;
        const float alpha = raise ? ex2_approx(m - m_new) : 1.f;  // 0 when m was -inf
        // O holds this item's earlier tiles once m is finite and j > 0; each
        // warpgroup rescales its 128 columns once G2(g - 1) has completed.
        const bool rescale_o = raise && j > 0 && m > -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          const bool w2 = __all_sync(0xffffffffu, mbar_wait(&bars[BAR_PVDONE + ((g - 1) & 1)], ((g - 1) >> 1) & 1,
                                                            abort_flag, WAIT_LIMIT_NS));
          if (w2) {
            tc_fence_after();
            const float f = rescale_o ? alpha : 1.f;
#pragma unroll 1
            for (int c32 = 0; c32 < 4; ++c32) {
              const uint32_t col = COL_O + 128u * half + c32 * 32;
              uint32_t o[32];
              tmem_ld32(t_lane + col, o);
              tmem_ld_wait(o);
              uint32_t w0[16], w1[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                w0[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                w1[i] = __float_as_uint(__uint_as_float(o[16 + i]) * f);
              }
              tmem_st16(t_lane + col, w0);
              tmem_st16(t_lane + col + 16, w1);
            }
            tmem_st_wait();
          } else {
            ok = false;  // left at the next tile's exchange or the epilogue's barrier
          }
        }
        l *= alpha;
        m = m_new;
        if (!ok) continue;
        // P = exp2(x - m) on visible keys, as io-type pairs into the slot's
        // columns [32 half, 32 half + 32): warpgroup 1 writes over scores of
        // warpgroup 0, which the exchange barrier shows were read.
        float rs[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) rs[a] = 0.f;
        // (m stays -inf only if every visible score so far is -inf, which only a
        // bias can make; P is 0 then, and exp2(-inf + 0) gives it without a NaN.)
        const float neg_m = m == -INFINITY ? 0.f : -m;
#pragma unroll
        for (int c16 = 0; c16 < 2; ++c16) {
          uint32_t wv[16];
          if (full) {
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2]), cs, neg_m));
              const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2 + 1]), cs, neg_m));
              rs[(2 * i2) & 7] += p0;
              rs[(2 * i2 + 1) & 7] += p1;
              wv[i2] = pack_io2<F16>(p0, p1);
            }
          } else {
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const int i = i0 + c16 * 32 + 2 * i2;
              const float p0 = (i >= v_lo && i <= v_hi)
                                   ? ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2]), cs, neg_m)) : 0.f;
              const float p1 = (i + 1 >= v_lo && i + 1 <= v_hi)
                                   ? ex2_approx(fmaf(__uint_as_float(sr[c16][2 * i2 + 1]), cs, neg_m)) : 0.f;
              rs[(2 * i2) & 7] += p0;
              rs[(2 * i2 + 1) & 7] += p1;
              wv[i2] = pack_io2<F16>(p0, p1);
            }
          }
          __syncwarp();
          tmem_st16(t_lane + 128u * s + half * 32 + c16 * 16, wv);
        }
        l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[BAR_PREADY + s]);
      }

      // ---- epilogue: O = O / (l_0 + l_1), each warpgroup writing its 128
      // columns of the row straight from registers (16-byte stores; rows past
      // S_q are not written), and LSE = (m + log2 L) ln 2. Tensor memory is read
      // before this warpgroup's next P_READY, which the next item's first G2
      // waits for before it overwrites O.
      if (ok) ok = mbar_wait(&bars[BAR_PVDONE + ((g - 1) & 1)], ((g - 1) >> 1) & 1, abort_flag, WAIT_LIMIT_NS);
      const bool warp_ok = __all_sync(0xffffffffu, ok);
      if (warp_ok) tc_fence_after();
      xl[half * 128 + row] = l;
      // The next item, handed to every softmax warp by the barrier below.
      if (warp == 0 && lane == 0) sitem[(e + 1) & 1] = ring_take(e + 1);
      have_next = true;
      // Every softmax thread learns whether any of them gave up, so that all
      // leave the item loop together after this epilogue.
      const bool any_fail = named_bar_sync_or(1, 256, !warp_ok);
      const float lt = xl[row] + xl[128 + row];
      named_bar_sync(1, 256);  // the exchange area is free for the next item
      const float inv_l = (lt > 0.f && live) ? 1.f / lt : 0.f;
      uint16_t* const orow_ptr = o_base + orow * D;
      const bool row_ok = q < p.Sq && in_bounds(p.status, orow_ptr, (size_t)D * 2, p.o, o_bytes);
#pragma unroll 1
      for (int c32 = 0; c32 < 4; ++c32) {
        const int cbase = half * 128 + c32 * 32;  // first O column of this chunk
        uint32_t o[32];
        if (warp_ok) {
          tmem_ld32(t_lane + COL_O + cbase, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint4 wv[4];
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          wv[v8].x = pack_io2<F16>(__uint_as_float(o[v8 * 8 + 0]) * inv_l, __uint_as_float(o[v8 * 8 + 1]) * inv_l);
          wv[v8].y = pack_io2<F16>(__uint_as_float(o[v8 * 8 + 2]) * inv_l, __uint_as_float(o[v8 * 8 + 3]) * inv_l);
          wv[v8].z = pack_io2<F16>(__uint_as_float(o[v8 * 8 + 4]) * inv_l, __uint_as_float(o[v8 * 8 + 5]) * inv_l);
          wv[v8].w = pack_io2<F16>(__uint_as_float(o[v8 * 8 + 6]) * inv_l, __uint_as_float(o[v8 * 8 + 7]) * inv_l);
        }
        if (o_sector) {
          // Whole 32-byte sectors: 16-column pieces, each inside the row.
#pragma unroll
          for (int v16 = 0; v16 < 2; ++v16)
            if (row_ok && cbase + v16 * 16 < p.Dv) st_global_32b(orow_ptr + cbase + v16 * 16, wv[2 * v16], wv[2 * v16 + 1]);
        } else {
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            const int cc = cbase + v8 * 8;  // column of this 16-byte piece
            if (row_ok && cc < p.Dv) *reinterpret_cast<uint4*>(orow_ptr + cc) = wv[v8];
          }
        }
      }
      tc_fence_before();
      if (half == 0 && q < p.Sq) {
        float lse = -INFINITY;
        if (lt > 0.f) lse = (m + __log2f(lt)) * 0.6931471805599453f;  // a padded row with a sink: the sink
        p.lse[orow] = lse;
      }
      if (any_fail) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
  if (tid == 0) {
    // Every ticket taker of this launch has drawn its last ticket once all CTAs
    // have come here: the last one resets the slot.
    if (atomicAdd(&g_fwd_wide_done[ticket_slot], 1) == (int)gridDim.x - 1) {
      g_fwd_wide_ticket[ticket_slot] = 0;
      g_fwd_wide_done[ticket_slot] = 0;
    }
  }
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BIAS, bool F16>
static cudaError_t set_fwd_wide_smem() {
  return cudaFuncSetAttribute(sdpa_fwd_wide_kernel<BIAS, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fwd_wide::BYTES);
}

cudaError_t fwd_wide_setup() {
  cudaError_t e = set_fwd_wide_smem<false, false>();
  if (e == cudaSuccess) e = set_fwd_wide_smem<true, false>();
  if (e == cudaSuccess) e = set_fwd_wide_smem<false, true>();
  if (e == cudaSuccess) e = set_fwd_wide_smem<true, true>();
  return e;
}

template <bool BIAS, bool F16>
static cudaError_t launch_wide_variant(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms,
                                       int slot) {
  const long long items = (long long)p.n_qt * p.B * p.Hq;
  const dim3 grid((unsigned)(items < sms ? items : sms));
  return launch_kernel(sdpa_fwd_wide_kernel<BIAS, F16>, grid, dim3(fwd_wide::THREADS), fwd_wide::BYTES, s,
                       false, maps, p, slot);
}

cudaError_t launch_fwd_wide(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms, int slot) {
  if (p.Dqk != fwd_wide::D || p.Dv != fwd_wide::D || sms <= 0 || slot < 0 || slot >= fwd_shared::FWD_SLOTS)
    return cudaErrorInvalidValue;
  if (p.bias)
    return p.f16 ? launch_wide_variant<true, true>(maps, p, s, sms, slot)
                 : launch_wide_variant<true, false>(maps, p, s, sms, slot);
  return p.f16 ? launch_wide_variant<false, true>(maps, p, s, sms, slot)
               : launch_wide_variant<false, false>(maps, p, s, sms, slot);
}

}  // namespace sdpa
