// sdpa_fwd_shared.cu -- the fused SDPA forward with one O accumulator shared by
// both softmax warpgroups, served for the MLA head pair (D_qk = 192, D_v = 128).
//
// It computes what sdpa_fwd.cu computes (O and the natural-log LSE of the
// masked softmax: "SDPA Backward (SM120)", API Usage, `o` and `stats`; the masks
// of "Causal, sliding-window, and padding masks"; GQA/MQA; the sink logit and
// the additive bias of the Capabilities list):
//   S = scale Q K^T [+ bias] (masked entries removed),
//   LSE = log(sum_k exp(S) [+ exp(sink)]),   O = sum_k exp(S - LSE) V.
// sdpa_fwd.cu keeps an O per key half, which leaves tensor memory two S slots;
// this kernel trades that for a per-tile exchange of the row maximum and a third
// slot. At D_qk = 192 the score GEMM is half again as long, the two-slot loop
// (G1 of tile j + 2 waits for G2 of tile j) binds, and the third slot measured
// 1,086 against 876 TFLOP/s on the MLA workload; at D_qk = 128 the softmax binds
// instead, and the exchange cost 6 % there, so those head dims stay on
// sdpa_fwd.cu.
//
// Schedule. A work item is 128 query rows of one (batch, query head); the CTA
// walks the key tiles (128 keys) that any of its rows sees, in ascending order.
// Per key tile j:
//   G1  S = Q K_j^T          -> tensor-memory slot j % 3 (128 fp32 columns)
//       P = exp2(S * scale * log2e - m)   (two softmax warpgroups, 64 keys each)
//           -> io-type pairs, warpgroup h into the slot's columns [32 h, 32 h + 32)
//   G2  O += P V_j           (A = P from tensor memory, B = V_j MN-major)
// The two warpgroups share O and one reference m per row: each takes the
// maximum of its 64 scores, they exchange it at a named barrier, and both raise
// m only when the tile's maximum exceeds it by more than 8 (log2 units). Until
// a raise P stays below 2^8, which bf16 and fp32 hold exactly enough, so O is
// rescaled only on those rare raises (after the previous G2 has completed), each
// warpgroup its D_v / 2 columns. The row sums l_0, l_1 stay per warpgroup; at
// the end O = O / (l_0 + l_1) and LSE = (m + log2(l_0 + l_1)) * ln 2.
// One O leaves room for three S/P slots, so G1 of tile j + 3, not j + 2, is the
// one that waits for G2 of tile j: three tiles in flight between the score GEMM,
// the softmax and the PV GEMM.
//
// Warps: 0-7 two softmax warpgroups (a row's keys split between warps w and w+4,
// which read the same tensor-memory lanes; one warp per SMSP did not hide the
// instruction latencies), 8 the TMA producer of Q and the K ring (a K tile is
// replaced once its G1 has read it), 9 the G1 issuer and tensor-memory owner,
// 10 the G2 issuer, 11 the TMA producer of the V ring (a V tile is replaced once
// its G2 has read it). Tensor memory: S/P slots at [0,128), [128,256) and
// [256,384), O at [384, 384 + D_v).
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include "sdpa_fwd.cuh"

namespace sdpa {

namespace fwd_sh {

constexpr int THREADS = 384;
using fwd_shared::BM;
using fwd_shared::BK;
using fwd_shared::WAIT_LIMIT_NS;
using fwd_shared::RESCALE_THRESHOLD;
constexpr int NSLOT = 3;  // S/P slots in tensor memory

// Register split: launched with 168 per thread (384 threads), the control
// warpgroup (warps 8-11) drops to 56 and the two softmax warpgroups grow to 224:
// 128 x (56 + 224 + 224) = 64,512 = 384 x 168.
constexpr uint32_t REGS_CTRL = 56, REGS_SOFTMAX = 224;
static_assert(128 * (REGS_CTRL + 2 * REGS_SOFTMAX) <= THREADS * 168, "register split");
constexpr int RING = 4;           // items published by the producer (persistent form)
constexpr int RING_READERS = 4;   // warps that read them: 0 (for warps 0-7), 9, 10 and 11

enum : int {
  BAR_QFULL = 0,                 // the item's Q tile landed
  BAR_QEMPTY = 1,                // the item's last G1 completed: Q may be replaced
  BAR_KFULL = 2,                 // + stage (up to 4): the K tile landed
  BAR_KEMPTY = 6,                // + stage: G1 of the tile completed, K may be replaced
  BAR_VFULL = 10,                // + stage: the V tile landed
  BAR_VEMPTY = 14,               // + stage: G2 of the tile completed, V may be replaced
  BAR_SFULL = 18,                // + slot: S in tensor memory
  BAR_PREADY = BAR_SFULL + NSLOT,  // + slot, 256 arrivals: P written (both warpgroups)
  BAR_PVDONE = BAR_PREADY + NSLOT, // + slot: G2 of the slot's tile completed
  BAR_RFULL = BAR_PVDONE + NSLOT,  // + ring entry: an item published
  BAR_REMPTY = BAR_RFULL + RING,   // + ring entry, RING_READERS arrivals: read by every role
  NUM_BARS = BAR_REMPTY + RING
};

template <int DQK, int DV>
struct Layout {
  static constexpr int BLK = 128 * 128;            // one 64-column block of a 128-row tile
  static constexpr int TILE_Q = BM * DQK * 2;
  static constexpr int TILE_K = BK * DQK * 2;
  static constexpr int TILE_V = BK * DV * 2;
  static constexpr int STAGE = TILE_K + TILE_V;  // one stage of each ring
  static constexpr int NS_FIT = (232448 - TILE_Q - NUM_BARS * 8 - 2 * 256 * 4 - 64) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE_Q;               // K ring: NS tiles
  static constexpr int OFF_V = OFF_K + NS * TILE_K;  // V ring: NS tiles
  static constexpr int OFF_BAR = OFF_V + NS * TILE_V;
  // The warpgroups' exchange area: [2 tile parities][2 warpgroups][128 rows]
  // floats, the tile maxima every tile and the row sums at an item's end.
  static constexpr int OFF_XT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_MISC = OFF_XT + 2 * 256 * 4;
  // More than half an SM's shared memory keeps one CTA per SM, so the 512
  // tensor-memory columns are never contended.
  static constexpr int BYTES_RAW = OFF_MISC + 64;
  static constexpr int BYTES = BYTES_RAW > 120 * 1024 ? BYTES_RAW : 120 * 1024;
  // Three 128-column S/P slots, then the one O accumulator.
  static constexpr uint32_t COL_O = 128 * NSLOT;
  static_assert(NS >= 2, "stage ring");
  static_assert(COL_O + DV <= 512 && DV <= 128, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(TILE_Q % 1024 == 0 && TILE_K % 1024 == 0 && TILE_V % 1024 == 0, "alignment");
  static_assert(DV <= DQK, "O staging reuses the Q tile");
};

}  // namespace fwd_sh

// Work tickets of the persistent forward (PERSIST), one counter pair per launch
// slot: a CTA's producer takes items (longest first) from g_fwd_sh_ticket[slot], and
// the last CTA to finish puts both counters back to zero for the slot's next
// launch. The host hands out the 64 slots in turn, so launches share a counter
// only if 64 forward launches run on one device at once.
constexpr int FWD_SLOTS = fwd_shared::FWD_SLOTS;
__device__ int g_fwd_sh_ticket[FWD_SLOTS];
__device__ int g_fwd_sh_done[FWD_SLOTS];

// BIAS adds the additive bias (FwdParams::bias) to the scaled scores. F16:
// fp16 io tensors (and fp16 P for the PV GEMM) instead of bf16. PERSIST: one
// CTA per SM takes items from the launch's ticket, and the K/V ring, the S/P
// slots and their barrier phases run on from one item to the next; otherwise
// one item per CTA (blockIdx.x).
template <int DQK, int DV, bool BIAS, bool F16 = false, bool PERSIST = false>
__global__ void __launch_bounds__(fwd_sh::THREADS, 1)
    sdpa_fwd_shared_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p, const int ticket_slot) {
  using namespace fwd_sh;
  using L = Layout<DQK, DV>;
  constexpr int NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sKr = smem + L::OFF_K;  // K ring
  uint8_t* sVr = smem + L::OFF_V;  // V ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);  // [RING] items
  volatile int* sitem = ring + RING;  // [2] the softmax warpgroups' current item, by parity
  const int n_items = p.n_qt * p.B * p.Hq;
  // Items a CTA walks at most: one without PERSIST, so that the compiler sees
  // a single pass and keeps no state across items.
  constexpr int E_MAX = PERSIST ? 0x7fffffff : 1;
  // Item e of this CTA, for a whole warp: from the ring the producer fills
  // (PERSIST; lane 0 waits, reads and releases the entry, and hands the item to
  // the other lanes), else blockIdx.x then the end (-1).
  auto ring_take = [&](int e) -> int {  // one thread
    if constexpr (!PERSIST) return e == 0 ? (int)blockIdx.x : -1;
    const int r = e % RING;
    if (!mbar_wait(&bars[BAR_RFULL + r], (e / RING) & 1, abort_flag, WAIT_LIMIT_NS)) return -1;
    const int it = ring[r];
    mbar_arrive(&bars[BAR_REMPTY + r]);
    return it;
  };
  auto next_item = [&](int e) -> int {
    int it = -1;
    if ((threadIdx.x & 31) == 0) it = ring_take(e);
    return __shfl_sync(0xffffffffu, it, 0);
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NUM_BARS; ++i)
      mbar_init(&bars[i], (i >= BAR_PREADY && i < BAR_PREADY + NSLOT) ? 256
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

  // Every role walks the same items, in the order the producer took them, and
  // counts the key tiles it has passed over all of them (g), so that the K and
  // V rings, the three S/P slots and their barrier phases run on across items;
  // ni counts the items with at least one key tile (the Q buffer's phases).
  // Items whose rows see no key are written by the softmax warps alone.
  if (warp >= 8) {
    // Producer and MMA issuers need few registers; the softmax warpgroups get them.
    regs_decrease<REGS_CTRL>();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int g = 0, ni = 0;
        bool ok = true;
        // K(g) replaces the ring's K(g - NS) once G1(g - NS) has read it.
        auto load_k = [&](const FwdItem& w, int j) -> bool {
          const int st = g % NS;
          if (g >= NS && !mbar_wait(&bars[BAR_KEMPTY + st], ((g / NS) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
            return false;
          const int k0 = (w.kt_lo + j) * BK;
          uint8_t* sK = sKr + st * L::TILE_K;
          uint64_t* full = &bars[BAR_KFULL + st];
          mbar_arrive_expect_tx(full, L::TILE_K);
          for (int blk = 0; blk < DQK / 64; ++blk) tma_load_3d(sK + blk * L::BLK, &maps.k, full, blk * 64, k0, w.kvh);
          ++g;
          return true;
        };
        for (int e = 0; e < E_MAX && ok; ++e) {
          int it;
          if constexpr (PERSIST) {
            // Take the next item and publish it to the other roles.
            const int r = e % RING;
            if (e >= RING && !mbar_wait(&bars[BAR_REMPTY + r], ((e / RING) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
              break;
            it = atomicAdd(&g_fwd_sh_ticket[ticket_slot], 1);
            if (it >= n_items) it = -1;
            ring[r] = it;
            mbar_arrive(&bars[BAR_RFULL + r]);
          } else {
            it = e == 0 ? (int)blockIdx.x : -1;
          }
          if (it < 0) break;
          const FwdItem w = fwd_item(p, it);
          if (w.n <= 0) continue;
          // The item's first key tiles only wait for stages that earlier items
          // release, so they load before its Q, which waits for the previous
          // item's last G1; later tiles wait for stages this item releases,
          // which needs its Q first.
          const int pre = w.n < NS ? w.n : NS;
          for (int j = 0; j < pre && ok; ++j) ok = load_k(w, j);
          if (ok && ni >= 1) ok = mbar_wait(&bars[BAR_QEMPTY], (ni - 1) & 1, abort_flag, WAIT_LIMIT_NS);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[BAR_QFULL], L::TILE_Q);
          for (int blk = 0; blk < DQK / 64; ++blk)
            tma_load_3d(sQ + blk * L::BLK, &maps.q, &bars[BAR_QFULL], blk * 64, w.q0, w.bh);
          for (int j = pre; j < w.n && ok; ++j) ok = load_k(w, j);
          ++ni;
        }
      }
    } else if (warp == 11) {
      // ------------------------------------------------------------ V producer
      // V(g) replaces the ring's V(g - NS) once G2(g - NS) has read it: V is
      // needed a softmax later than K, so its ring runs behind K's.
      if (lane == 0) {
        int g = 0;
        bool ok = true;
        for (int e = 0; e < E_MAX && ok; ++e) {
          const int it = ring_take(e);
          if (it < 0) break;
          const FwdItem w = fwd_item(p, it);
          for (int j = 0; j < w.n && ok; ++j, ++g) {
            const int st = g % NS;
            if (g >= NS) ok = mbar_wait(&bars[BAR_VEMPTY + st], ((g / NS) - 1) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            const int k0 = (w.kt_lo + j) * BK;
            uint8_t* sV = sVr + st * L::TILE_V;
            uint64_t* full = &bars[BAR_VFULL + st];
            mbar_arrive_expect_tx(full, L::TILE_V);
            for (int blk = 0; blk < DV / 64; ++blk)
              tma_load_3d(sV + blk * L::BLK, &maps.v, full, blk * 64, k0, w.kvh);
          }
        }
      }
    } else if (warp == 9 || warp == 10) {
      // ------------------------------------------------------------ MMA issuers
      // A tcgen05.mma costs its issuing thread on the order of 100 cycles, about
      // what a 128-column MMA takes on the tensor core, so the 16 MMAs of a tile
      // are issued by two warps: 9 the score GEMM G1, 10 the PV GEMM G2. G1 of
      // tile g reuses the slot of tile g-3, whose P G2(g-3) read; G2(g) needs P(g).
      constexpr uint32_t ID_S = idesc_io(BM, BK, false, false, F16);  // S = Q K^T
      constexpr uint32_t ID_O = idesc_io(BM, DV, false, true, F16);   // O += P V
      constexpr uint64_t T_KMAJ = sdesc_sw128_template(16, 1024);
      constexpr uint64_t T_MN_V = sdesc_sw128_template(L::BLK, 1024);
      int g = 0, ni = 0;
      bool ok = true;
      const uint32_t aQ = smem_u32(sQ);
      for (int e = 0; e < E_MAX && ok; ++e) {
        const int it = next_item(e);
        if (it < 0) break;
        const FwdItem w = fwd_item(p, it);
        if (w.n <= 0) continue;
        if (warp == 9) {
          ok = mbar_wait(&bars[BAR_QFULL], ni & 1, abort_flag, WAIT_LIMIT_NS);
          for (int j = 0; j < w.n && ok; ++j, ++g) {
            const int st = g % NS, s = g % NSLOT;
            ok = mbar_wait(&bars[BAR_KFULL + st], (g / NS) & 1, abort_flag, WAIT_LIMIT_NS);
            if (ok && g >= NSLOT)
              ok = mbar_wait(&bars[BAR_PVDONE + s], ((g - NSLOT) / NSLOT) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            if (elect_one()) {
              const uint32_t aK = smem_u32(sKr + st * L::TILE_K);
  #pragma unroll
              for (int k = 0; k < DQK / 16; ++k) {
                const uint32_t ko = (k >> 2) * L::BLK + (k & 3) * 32;
                mma_ss(tmem + 128u * s, sdesc_at(T_KMAJ, aQ + ko), sdesc_at(T_KMAJ, aK + ko), ID_S, k > 0);
              }
              mma_commit(&bars[BAR_SFULL + s]);
              mma_commit(&bars[BAR_KEMPTY + st]);
              // After the item's last G1 the Q buffer takes the next item's Q.
              if (j == w.n - 1) mma_commit(&bars[BAR_QEMPTY]);
            }
            __syncwarp();
          }
        } else {
          for (int u = 0; u < w.n && ok; ++u, ++g) {
            const int su = g % NSLOT, stu = g % NS;
            // P(g) written implies S(g) computed, so V(g) has landed as well;
            // waiting on the stage barrier too makes that explicit for this warp.
            // (The previous item's epilogue has read O before any P of this item
            // is written: the same threads do both, in that order.)
            ok = mbar_wait(&bars[BAR_PREADY + su], (g / NSLOT) & 1, abort_flag, WAIT_LIMIT_NS) &&
                 mbar_wait(&bars[BAR_VFULL + stu], (g / NS) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            if (elect_one()) {
              const uint32_t aV = smem_u32(sVr + stu * L::TILE_V);
              // O += P V: keys 16 k .. 16 k + 15 of P sit in the slot's columns
              // [8 k, 8 k + 8) (warpgroup h's 64 keys at [32 h, 32 h + 32)).
  #pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                mma_ts(tmem + L::COL_O, tmem + 128u * su + 8u * k, sdesc_at(T_MN_V, aV + k * 2048), ID_O,
                       (u > 0 || k > 0) ? 1u : 0u);
              mma_commit(&bars[BAR_PVDONE + su]);
              mma_commit(&bars[BAR_VEMPTY + stu]);
            }
            __syncwarp();
          }
        }
        ++ni;
      }
    }
  } else {
    regs_increase<REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax warpgroups
    // Warps w and w + 4 read the same tensor-memory lanes (w % 4): warpgroup
    // `half` takes keys [64 half, 64 half + 64) of each tile. The two share the
    // one O accumulator and so one reference m per row: each takes the maximum
    // of its 64 scores, the two exchange it at a named barrier, and both apply
    // the same raise rule to the same m. The row sums stay per warpgroup.
    const int half = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    float* xt = reinterpret_cast<float*>(smem + L::OFF_XT);  // [2 parity][2 half][128]
    const float c = p.scale_log2;
    const uint32_t col_o = L::COL_O + half * (DV / 2);  // this warpgroup's columns of O
    const long long Rp = p.window_right > 0 ? p.window_right : 0;
    const bool has_window = p.window_left >= 0;
    const int i0 = half * 64;  // this warpgroup's first key within a tile
    // With a bias the scores are rewritten in place as x = s * c + bias * log2e,
    // and everything below reads them with the factor cs = 1 instead of c.
    const float cs = BIAS ? 1.f : c;
    uint16_t* const o_base = static_cast<uint16_t*>(p.o);
    const size_t o_bytes = (size_t)p.B * p.Hq * p.Sq * p.Dv * 2;
    // O rows go out in 32-byte stores when every 16-column piece is 32-byte
    // aligned (the base 32-byte aligned, D_v a multiple of 16), else 16-byte ones.
    const bool o_sector = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0 && (p.Dv & 15) == 0;
    int g = 0;
    bool ok = true;
    bool have_next = false;  // the item for this e was taken during the previous epilogue
    for (int e = 0; e < E_MAX && ok; ++e) {
      // Warp 0 takes the item for all eight warps, so that they never disagree
      // on it (a wait that gives up can do so in one reader and not in another)
      // and meet at the same named barriers: during the previous item's
      // epilogue, whose barrier hands it over, else here with a barrier of its
      // own. Double-buffered by parity: a slot is rewritten only after a later
      // barrier that every reader of it has passed.
      int it;
      if constexpr (PERSIST) {
        if (!have_next) {
          if (warp == 0) {
            const int t = next_item(e);
            if (lane == 0) sitem[e & 1] = t;
          }
          named_bar_sync(3, 256);
        }
        have_next = false;
        it = sitem[e & 1];
      } else {
        it = next_item(e);
      }
      if (it < 0) break;
      const FwdItem w = fwd_item(p, it);
      const int q = w.q0 + row;
      const long long orow = (long long)w.bh * p.Sq + q;  // O / LSE row
      if (w.n <= 0) {
        // No row of this item sees a key (every row past the query length, or
        // a mask that leaves none): O = 0 and LSE = -inf, or the sink logit.
        if (half == 0 && q < p.Sq) {
          uint4* o = reinterpret_cast<uint4*>(o_base + orow * p.Dv);
          if (in_bounds(p.status, o, (size_t)p.Dv * 2, p.o, o_bytes))
            for (int i = 0; i < p.Dv / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
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
        const int s = g % NSLOT;
        const int k0 = (w.kt_lo + j) * BK;
        uint32_t braw[BIAS ? 64 : 1];
        bool bpacked = false;
        if constexpr (BIAS) {
          load_fwd_bias_row(p, bias_row, k0 + i0, live, braw, bpacked);
          // The row's segment of the tile after next into L2 (one or two lines).
          const int kp = k0 + 2 * BK + i0;
          if (live && j + 2 < w.n && kp < p.Skv) {
            const char* a = static_cast<const char*>(p.bias) + (bias_row + kp) * (p.bias_fp32 ? 4 : 2);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
            if (p.bias_fp32 && kp + 32 < p.Skv) asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 128));
          }
        }
        // A wait that gave up (here or at a rescale) reaches every softmax thread
        // through the OR of the exchange barrier, so that all 256 leave the tile
        // loop at the same tile and meet again at the epilogue's barriers.
        const bool wok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[BAR_SFULL + s], (g / NSLOT) & 1,
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
          // warp (every tile but the mask edges). The choice is warp-uniform: the
          // tensor-memory stores below are .sync.aligned, and a warp split
          // between the two paths would reach them diverged.
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
        // decision in both warpgroups. Until a raise P stays below 2^8, which
        // bf16 and fp32 hold exactly enough, so O is rescaled only on a raise.
        const bool raise = mt > m + RESCALE_THRESHOLD || (m == -INFINITY && mt > -INFINITY);
        const float m_new = raise ? mt : m;
        const float alpha = raise ? ex2_approx(m - m_new) : 1.f;  // 0 when m was -inf
        // O holds this item's earlier tiles once m is finite and j > 0; each
        // warpgroup rescales its D_v / 2 columns once G2(g - 1) has completed
        // (G2(g) waits for this tile's P_READY).
        const bool rescale_o = raise && j > 0 && m > -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          const int gp = g - 1;
          const bool w2 = __all_sync(0xffffffffu, mbar_wait(&bars[BAR_PVDONE + gp % NSLOT], (gp / NSLOT) & 1,
                                                            abort_flag, WAIT_LIMIT_NS));
          if (w2) {
            tc_fence_after();
            const float f = rescale_o ? alpha : 1.f;
#pragma unroll 1
            for (int c32 = 0; c32 < DV / 64; ++c32) {
              const uint32_t col = col_o + c32 * 32;
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

      // ---- epilogue: O = O / (l_0 + l_1), each warpgroup writing its D_v / 2
      // columns of the row straight from registers (16-byte stores; columns past
      // D_v and rows past S_q are not written), and LSE = (m + log2 L) ln 2.
      // Tensor memory is read before this warpgroup's next P_READY, which G2 of
      // the next item's first tile waits for before it overwrites O.
      if (ok) {
        const int gp = g - 1;
        ok = mbar_wait(&bars[BAR_PVDONE + gp % NSLOT], (gp / NSLOT) & 1, abort_flag, WAIT_LIMIT_NS);
      }
      const bool warp_ok = __all_sync(0xffffffffu, ok);
      if (warp_ok) tc_fence_after();
      // The row sums go through the exchange area of the next tile's parity: its
      // last readers (the tile before last) have passed the last tile's barrier,
      // and the next tile writes it only after this epilogue's barriers.
      float* xl = xt + (g & 1) * 256;
      xl[half * 128 + row] = l;
      if constexpr (PERSIST) {
        // The next item, handed to every softmax warp by the barrier below.
        if (warp == 0) {
          const int t = next_item(e + 1);
          if (lane == 0) sitem[(e + 1) & 1] = t;
        }
        have_next = true;
      }
      // Every softmax thread learns whether any of them gave up, so that all
      // leave the item loop together after this epilogue.
      const bool any_fail = named_bar_sync_or(1, 256, !warp_ok);
      const float lt = xl[row] + xl[128 + row];
      named_bar_sync(1, 256);  // the exchange area is free for the next tile
      const float inv_l = (lt > 0.f && live) ? 1.f / lt : 0.f;
      uint16_t* const orow_ptr = o_base + orow * p.Dv;
      const bool row_ok = q < p.Sq && in_bounds(p.status, orow_ptr, (size_t)p.Dv * 2, p.o, o_bytes);
#pragma unroll 1
      for (int c32 = 0; c32 < DV / 64; ++c32) {
        const int cbase = half * (DV / 2) + c32 * 32;  // first O column of this chunk
        uint32_t o[32];
        if (warp_ok) {
          tmem_ld32(t_lane + L::COL_O + cbase, o);
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
  if (PERSIST && tid == 0) {
    // Every producer of this launch has taken its last ticket once all CTAs
    // have come here: the last one resets the slot.
    if (atomicAdd(&g_fwd_sh_done[ticket_slot], 1) == (int)gridDim.x - 1) {
      g_fwd_sh_ticket[ticket_slot] = 0;
      g_fwd_sh_done[ticket_slot] = 0;
    }
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BIAS, bool F16>
static cudaError_t set_fwd_shared_smem() {
  return cudaFuncSetAttribute(sdpa_fwd_shared_kernel<192, 128, BIAS, F16, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_sh::Layout<192, 128>::BYTES);
}

cudaError_t fwd_shared_setup() {
  cudaError_t e = set_fwd_shared_smem<false, false>();
  if (e == cudaSuccess) e = set_fwd_shared_smem<true, false>();
  if (e == cudaSuccess) e = set_fwd_shared_smem<false, true>();
  if (e == cudaSuccess) e = set_fwd_shared_smem<true, true>();
  return e;
}

template <bool BIAS, bool F16>
static cudaError_t launch_shared_variant(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms,
                                         int slot) {
  const long long items = (long long)p.n_qt * p.B * p.Hq;
  const dim3 grid((unsigned)(items < sms ? items : sms));
  return launch_kernel(sdpa_fwd_shared_kernel<192, 128, BIAS, F16, true>, grid, dim3(fwd_sh::THREADS),
                       fwd_sh::Layout<192, 128>::BYTES, s, false, maps, p, slot);
}

cudaError_t launch_fwd_shared(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms, int slot) {
  if (p.Dqk != 192 || p.Dv != 128 || sms <= 0 || slot < 0 || slot >= fwd_shared::FWD_SLOTS)
    return cudaErrorInvalidValue;
  if (p.bias)
    return p.f16 ? launch_shared_variant<true, true>(maps, p, s, sms, slot)
                 : launch_shared_variant<true, false>(maps, p, s, sms, slot);
  return p.f16 ? launch_shared_variant<false, true>(maps, p, s, sms, slot)
               : launch_shared_variant<false, false>(maps, p, s, sms, slot);
}

}  // namespace sdpa
