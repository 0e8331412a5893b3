// sdpa_fwd.cu -- fused SDPA forward (O and the natural-log LSE) for sm_103a.
//
// What it computes: the forward whose outputs the backward consumes ("SDPA
// Backward (SM120)", API Usage: `o` and the natural-log `stats`; the masks of
// "Causal, sliding-window, and padding masks"; GQA/MQA head mapping; the sink
// token of the Capabilities list, which joins every row's softmax denominator
// without a value row; and the additive bias of the same list, added to the
// scaled scores):
//   S = scale Q K^T [+ bias] (masked entries removed),
//   LSE = log(sum_k exp(S) [+ exp(sink)]),   O = sum_k exp(S - LSE) V.
// With a bias each softmax thread loads its row's 64 bias values of a tile
// (16-byte loads along the keys) before it waits for that tile's S.
// A row with no visible key and no sink gets LSE = -inf and O = 0; with a sink
// LSE = sink and O = 0.
//
// Schedule. One CTA owns 128 query rows of one (batch, query head) and walks the
// key tiles (128 keys) that any of its rows sees, in ascending order. Per key tile j:
//   G1  S   = Q K_j^T        -> tensor-memory slot j % 2 (128 fp32 columns)
//       P   = exp2(S * scale * log2e - m)   (two softmax warpgroups, half a row each)
//           -> bf16 pairs, half h into the slot's columns [64 h, 64 h + 32)
//   G2  O_h += P[:, half h] V_j[half h, :]   (A = P from tensor memory, B = V_j
//           MN-major; keys 0-63 into O_0, 64-127 into O_1)
// Each half h of a row keeps its own softmax state: a running reference m_h
// that is raised only when the half's maximum exceeds it by more than 8 (in
// log2 units), an fp32 sum l_h and the accumulator O_h. Until a raise P stays
// below 2^8, which bf16 and fp32 hold exactly enough, so O_h is rescaled only on
// those rare raises (after the previous G2 has completed). At the end, with
// M = max(m_0, m_1) and a_h = 2^(m_h - M): O = (O_0 a_0 + O_1 a_1) / L,
// L = l_0 a_0 + l_1 a_1, LSE = (M + log2 L) * ln 2.
//
// Warps: 0-7 two softmax warpgroups (a row's keys split between warps w and w+4,
// which read the same tensor-memory lanes; one warp per SMSP did not hide the
// instruction latencies), 8 the TMA producer (Q once, K/V stage ring), 9 the G1
// issuer and tensor-memory owner, 10 the G2 issuer, 11 idle. Tensor memory: S/P slots at
// [0,128) and [128,256), O_0 at [256, 256+D_v), O_1 at [384, 384+D_v).
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include "sdpa_fwd.cuh"

namespace sdpa {

namespace fwd_kernel {

constexpr int THREADS = 384;
using fwd_shared::BM;
using fwd_shared::BK;
using fwd_shared::WAIT_LIMIT_NS;
using fwd_shared::RESCALE_THRESHOLD;
constexpr int NSLOT = 2;  // S/P slots in tensor memory

// Register split: launched with 168 per thread (384 threads), the control
// warpgroup (warps 8-11) drops to 56 and the two softmax warpgroups grow to 224:
// 128 x (56 + 224 + 224) = 64,512 = 384 x 168.
constexpr uint32_t REGS_CTRL = 56, REGS_SOFTMAX = 224;
static_assert(128 * (REGS_CTRL + 2 * REGS_SOFTMAX) <= THREADS * 168, "register split");
constexpr int RING = 4;           // items published by the producer (persistent form)
constexpr int RING_READERS = 3;   // warps that read them: 0 (for warps 0-7), 9 and 10

enum : int {
  BAR_QFULL = 0,                 // the item's Q tile landed
  BAR_QEMPTY = 1,                // the item's last G1 completed: Q may be replaced
  BAR_KVFULL = 2,                // + stage (up to 4)
  BAR_KVEMPTY = 6,               // + stage: G2 of the tile completed (K read by G1 before it)
  BAR_SFULL = 10,                // + slot: S in tensor memory
  BAR_PREADY = BAR_SFULL + NSLOT,  // + slot, 256 arrivals: P written (both halves)
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
  static constexpr int STAGE = TILE_K + TILE_V;
  static constexpr int NS_FIT = (232448 - TILE_Q - NUM_BARS * 8 - 2 * 256 * 4 - 64) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = TILE_Q;
  static constexpr int OFF_BAR = OFF_KV + NS * STAGE;
  static constexpr int OFF_XCH = OFF_BAR + NUM_BARS * 8;   // the halves' (m, l) at the end
  static constexpr int OFF_MISC = OFF_XCH + 2 * 256 * 4;
  // More than half an SM's shared memory keeps one CTA per SM, so the 512
  // tensor-memory columns are never contended.
  static constexpr int BYTES_RAW = OFF_MISC + 64;
  static constexpr int BYTES = BYTES_RAW > 120 * 1024 ? BYTES_RAW : 120 * 1024;
  // Two O accumulators, one per half of the keys: O_h at COL_O + 128 h.
  static constexpr uint32_t COL_O = 128 * NSLOT;
  static_assert(NS >= 2, "stage ring");
  static_assert(COL_O + 128 + DV <= 512 && DV <= 128, "tensor memory budget");
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(TILE_Q % 1024 == 0 && TILE_K % 1024 == 0 && TILE_V % 1024 == 0, "alignment");
  static_assert(DV <= DQK, "O staging reuses the Q tile");
};

}  // namespace fwd_kernel

// Work tickets of the persistent forward (PERSIST), one counter pair per launch
// slot: a CTA's producer takes items (longest first) from g_fwd_ticket[slot], and
// the last CTA to finish puts both counters back to zero for the slot's next
// launch. The host hands out the 64 slots in turn, so launches share a counter
// only if 64 forward launches run on one device at once.
constexpr int FWD_SLOTS = fwd_shared::FWD_SLOTS;
__device__ int g_fwd_ticket[FWD_SLOTS];
__device__ int g_fwd_done[FWD_SLOTS];

// BIAS adds the additive bias (FwdParams::bias) to the scaled scores. F16:
// fp16 io tensors (and fp16 P for the PV GEMM) instead of bf16. PERSIST: one
// CTA per SM takes items from the launch's ticket, and the K/V ring, the S/P
// slots and their barrier phases run on from one item to the next; otherwise
// one item per CTA (blockIdx.x).
template <int DQK, int DV, bool BIAS, bool F16 = false, bool PERSIST = false>
__global__ void __launch_bounds__(fwd_kernel::THREADS, 1)
    sdpa_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p, const int ticket_slot) {
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
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);  // [RING] items
  volatile int* sitem = ring + RING;  // [2] the softmax warpgroups' current item, by parity
  const int n_items = p.n_qt * p.B * p.Hq;
  // Items a CTA walks at most: one without PERSIST, so that the compiler sees
  // a single pass and keeps no state across items.
  constexpr int E_MAX = PERSIST ? 0x7fffffff : 1;
  // Item e of this CTA, for a whole warp: from the ring the producer fills
  // (PERSIST; lane 0 waits, reads and releases the entry, and hands the item to
  // the other lanes), else blockIdx.x then the end (-1).
  auto next_item = [&](int e) -> int {
    if constexpr (!PERSIST) return e == 0 ? (int)blockIdx.x : -1;
    int it = -1;
    if ((threadIdx.x & 31) == 0) {
      const int r = e % RING;
      if (mbar_wait(&bars[BAR_RFULL + r], (e / RING) & 1, abort_flag, WAIT_LIMIT_NS)) {
        it = ring[r];
        mbar_arrive(&bars[BAR_REMPTY + r]);
      }
    }
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
    prefetch_tmap(&maps.v);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Every role walks the same items, in the order the producer took them, and
  // counts the key tiles it has passed over all of them (g), so that the K/V
  // stage ring, the two S/P slots and their barrier phases run on across items;
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
        auto load_kv = [&](const FwdItem& w, int j) -> bool {
          const int st = g % NS;
          if (g >= NS && !mbar_wait(&bars[BAR_KVEMPTY + st], ((g / NS) - 1) & 1, abort_flag, WAIT_LIMIT_NS))
            return false;
          const int k0 = (w.kt_lo + j) * BK;
          uint8_t* sK = sKV + st * L::STAGE;
          uint8_t* sV = sK + L::TILE_K;
          uint64_t* full = &bars[BAR_KVFULL + st];
          mbar_arrive_expect_tx(full, L::STAGE);
          for (int blk = 0; blk < DQK / 64; ++blk) tma_load_3d(sK + blk * L::BLK, &maps.k, full, blk * 64, k0, w.kvh);
          for (int blk = 0; blk < DV / 64; ++blk) tma_load_3d(sV + blk * L::BLK, &maps.v, full, blk * 64, k0, w.kvh);
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
            it = atomicAdd(&g_fwd_ticket[ticket_slot], 1);
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
          for (int j = 0; j < pre && ok; ++j) ok = load_kv(w, j);
          if (ok && ni >= 1) ok = mbar_wait(&bars[BAR_QEMPTY], (ni - 1) & 1, abort_flag, WAIT_LIMIT_NS);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[BAR_QFULL], L::TILE_Q);
          for (int blk = 0; blk < DQK / 64; ++blk)
            tma_load_3d(sQ + blk * L::BLK, &maps.q, &bars[BAR_QFULL], blk * 64, w.q0, w.bh);
          for (int j = pre; j < w.n && ok; ++j) ok = load_kv(w, j);
          ++ni;
        }
      }
    } else if (warp == 9 || warp == 10) {
      // ------------------------------------------------------------ MMA issuers
      // A tcgen05.mma costs its issuing thread on the order of 100 cycles, about
      // what a 128-column MMA takes on the tensor core, so the 16 MMAs of a tile
      // are issued by two warps: 9 the score GEMM G1, 10 the PV GEMM G2. G1 of
      // tile g reuses the slot of tile g-2, whose P G2(g-2) read; G2(g) needs P(g).
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
            ok = mbar_wait(&bars[BAR_KVFULL + st], (g / NS) & 1, abort_flag, WAIT_LIMIT_NS);
            if (ok && g >= NSLOT)
              ok = mbar_wait(&bars[BAR_PVDONE + s], ((g - NSLOT) / NSLOT) & 1, abort_flag, WAIT_LIMIT_NS);
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
                 mbar_wait(&bars[BAR_KVFULL + stu], (g / NS) & 1, abort_flag, WAIT_LIMIT_NS);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            if (elect_one()) {
              const uint32_t aV = smem_u32(sKV + stu * L::STAGE + L::TILE_K);
              // O_h += P[:, keys of half h] V[keys of half h, :]; P of half h sits in
              // the slot's columns [64 h, 64 h + 32).
  #pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                mma_ts(tmem + L::COL_O + 128u * (k >> 2), tmem + 128u * su + 64u * (k >> 2) + 8 * (k & 3),
                       sdesc_at(T_MN_V, aV + k * 2048), ID_O, (u > 0 || (k & 3) > 0));
              mma_commit(&bars[BAR_PVDONE + su]);
              mma_commit(&bars[BAR_KVEMPTY + stu]);
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
    // `half` takes keys [64 half, 64 half + 64) of each tile. Each half keeps a
    // softmax of its own (reference m, sum l, accumulator O_half): no exchange
    // per tile; the two are combined once per item at its end.
    const int half = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + L::OFF_XCH);  // epilogue: [m, l][2 half][128]
    const float c = p.scale_log2;
    const uint32_t col_o = L::COL_O + 128u * half;  // this half's O accumulator
    const long long Rp = p.window_right > 0 ? p.window_right : 0;
    const bool has_window = p.window_left >= 0;
    const int i0 = half * 64;  // this half's first key within a tile
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
      float m = -INFINITY, l = 0.f;  // this half's reference and sum (the sink goes to half 0)
      if (p.sink && half == 0) {
        m = p.sink[w.h] * 1.4426950408889634f;
        l = 1.f;
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
        if (!mbar_wait(&bars[BAR_SFULL + s], (g / NSLOT) & 1, abort_flag, WAIT_LIMIT_NS)) { ok = false; break; }
        __syncwarp();
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32(t_lane + 128u * s + i0, sr[0]);
        tmem_ld32(t_lane + 128u * s + i0 + 32, sr[1]);
        tmem_ld_wait(sr[0]);
        tmem_ld_wait(sr[1]);
        if constexpr (BIAS) add_bias_row(p, c, braw, bpacked, sr);
        // Visible keys of this row within the tile: [v_lo, v_hi] relative to k0.
        int v_lo = 0, v_hi = BK - 1;
        if (!live) {
          v_hi = -1;
        } else {
          v_hi = (int)min((long long)BK - 1, min((long long)w.Lk - 1, k_vis_hi) - k0);
          v_lo = (int)max(0ll, k_vis_lo - k0);
        }
        // Unmasked path when this half is fully visible for the whole warp (every
        // tile but the mask edges). The choice is warp-uniform: the tensor-memory
        // stores below are .sync.aligned, and a warp split between the two paths
        // would reach them diverged.
        const bool full = __all_sync(0xffffffffu, v_lo <= i0 && v_hi >= i0 + 63);
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
        const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * cs;  // cs > 0
        // Raise the reference when the tile's maximum exceeds it by more than the
        // threshold (or when it is the row's first visible key).
        const bool raise = mt > m + RESCALE_THRESHOLD || (m == -INFINITY && mt > -INFINITY);
        const float m_new = raise ? mt : m;
        const float alpha = raise ? ex2_approx(m - m_new) : 1.f;  // 0 when m was -inf
        // O_half holds contributions of this item's earlier tiles once m is
        // finite and j > 0. It is rescaled once G2(g-1) has completed (G2(g)
        // waits for this tile's P_READY).
        const bool rescale_o = raise && j > 0 && m > -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          if (!mbar_wait(&bars[BAR_PVDONE + (g - 1) % NSLOT], ((g - 1) / NSLOT) & 1, abort_flag,
                         WAIT_LIMIT_NS)) {
            ok = false;
          }
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          const float f = rescale_o ? alpha : 1.f;
#pragma unroll 1
          for (int c32 = 0; c32 < DV / 32; ++c32) {
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
        }
        l *= alpha;
        m = m_new;
        // P = exp2(x - m) on visible keys, as bf16 pairs into the slot's columns
        // [64 half, 64 half + 32): inside this half's own S columns, which this
        // warp has already read. (Writing into the other half's S columns raced
        // with that half's warp, which may still be a tile behind.)
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
          tmem_st16(t_lane + 128u * s + half * 64 + c16 * 16, wv);
        }
        l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[BAR_PREADY + s]);
      }
      // (A wait that ran out sets the abort flag, so every other wait returns at
      // once; all 256 threads still reach the epilogue's barriers below.)

      // ---- epilogue: the halves combine, O = (O_0 a_0 + O_1 a_1) / (l_0 a_0 + l_1 a_1)
      // with a_h = 2^(m_h - M), M = max(m_0, m_1), each half writing D_v / 2
      // columns of its row straight from registers (16-byte stores; columns
      // past D_v and rows past S_q are not written). LSE in natural-log units.
      // Tensor memory is read before this warpgroup's next P_READY, which G2
      // of the next item's first tile waits for before it overwrites O.
      if (ok) ok = mbar_wait(&bars[BAR_PVDONE + (g - 1) % NSLOT], ((g - 1) / NSLOT) & 1, abort_flag,
                             WAIT_LIMIT_NS);
      const bool warp_ok = __all_sync(0xffffffffu, ok);
      if (warp_ok) tc_fence_after();
      xch[half * 128 + row] = m;
      xch[256 + half * 128 + row] = l;
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
      const float m0 = xch[row], m1 = xch[128 + row];
      const float l0 = xch[256 + row], l1 = xch[384 + row];
      named_bar_sync(1, 256);  // the exchange area is free for the next item
      const float M = fmaxf(m0, m1);
      const float a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - M);
      const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
      const float lt = l0 * a0 + l1 * a1;
      const float inv_l = (lt > 0.f && live) ? 1.f / lt : 0.f;
      const float f0 = a0 * inv_l, f1 = a1 * inv_l;
      uint16_t* const orow_ptr = o_base + orow * p.Dv;
      const bool row_ok = q < p.Sq && in_bounds(p.status, orow_ptr, (size_t)p.Dv * 2, p.o, o_bytes);
#pragma unroll 1
      for (int c32 = 0; c32 < DV / 64; ++c32) {
        const int cbase = half * (DV / 2) + c32 * 32;  // first O column of this chunk
        uint32_t o0[32], o1[32];
        if (warp_ok) {
          tmem_ld32(t_lane + L::COL_O + cbase, o0);
          tmem_ld32(t_lane + L::COL_O + 128 + cbase, o1);
          tmem_ld_wait(o0);
          tmem_ld_wait(o1);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o0[i] = o1[i] = 0u;
        }
        uint4 wv[4];
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            y[e] = __uint_as_float(o0[v8 * 8 + e]) * f0 + __uint_as_float(o1[v8 * 8 + e]) * f1;
          wv[v8].x = pack_io2<F16>(y[0], y[1]);
          wv[v8].y = pack_io2<F16>(y[2], y[3]);
          wv[v8].z = pack_io2<F16>(y[4], y[5]);
          wv[v8].w = pack_io2<F16>(y[6], y[7]);
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
        if (lt > 0.f) lse = (M + __log2f(lt)) * 0.6931471805599453f;  // a padded row with a sink: the sink
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
    if (atomicAdd(&g_fwd_done[ticket_slot], 1) == (int)gridDim.x - 1) {
      g_fwd_ticket[ticket_slot] = 0;
      g_fwd_done[ticket_slot] = 0;
    }
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, bool BIAS, bool F16>
static cudaError_t set_fwd_smem() {
  return cudaFuncSetAttribute(sdpa_fwd_kernel<DQK, DV, BIAS, F16, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_kernel::Layout<DQK, DV>::BYTES);
}

template <bool BIAS, bool F16>
static cudaError_t fwd_setup_variant() {
  cudaError_t e = set_fwd_smem<64, 64, BIAS, F16>();
  if (e == cudaSuccess) e = set_fwd_smem<128, 128, BIAS, F16>();
  return e;
}

cudaError_t fwd_kernel_setup() {
  cudaError_t e = fwd_setup_variant<false, false>();
  if (e == cudaSuccess) e = fwd_setup_variant<true, false>();
  if (e == cudaSuccess) e = fwd_setup_variant<false, true>();
  if (e == cudaSuccess) e = fwd_setup_variant<true, true>();
  if (e == cudaSuccess) e = fwd_shared_setup();
  if (e == cudaSuccess) e = fwd_wide_setup();
  return e;
}

template <bool BIAS, bool F16>
static cudaError_t launch_fwd_variant(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms,
                                      int slot) {
  // Persistent: one CTA per SM (more than half its shared memory each) taking
  // items from the launch's ticket.
  constexpr bool PERSIST = true;
  const long long items = (long long)p.n_qt * p.B * p.Hq;
  const dim3 grid((unsigned)(PERSIST ? (items < sms ? items : sms) : items));
  const dim3 block(fwd_kernel::THREADS);
  // D_qk = D_v up to 64 runs on the 64-column kernel, up to 128 on the 128-column
  // one: TMA zero-fills the columns past D on loads and drops them on stores.
  if (p.Dqk <= 64 && p.Dv == p.Dqk)
    return launch_kernel(sdpa_fwd_kernel<64, 64, BIAS, F16, PERSIST>, grid, block,
                         fwd_kernel::Layout<64, 64>::BYTES, s, false, maps, p, slot);
  if (p.Dqk <= 128 && p.Dv == p.Dqk)
    return launch_kernel(sdpa_fwd_kernel<128, 128, BIAS, F16, PERSIST>, grid, block,
                         fwd_kernel::Layout<128, 128>::BYTES, s, false, maps, p, slot);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, cudaStream_t s) {
  static std::atomic<unsigned> next_slot{0};
  const int slot = (int)(next_slot.fetch_add(1, std::memory_order_relaxed) % fwd_shared::FWD_SLOTS);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return cudaErrorInvalidValue;
  // The MLA pair: one O shared by the softmax warpgroups and three score slots
  // (sdpa_fwd_shared.cu). Head dim 256: one shared O, single K and V buffers
  // (sdpa_fwd_wide.cu).
  if (p.Dqk == 192 && p.Dv == 128) return launch_fwd_shared(maps, p, s, sms, slot);
  if (p.Dqk == 256 && p.Dv == 256) return launch_fwd_wide(maps, p, s, sms, slot);
  if (p.bias)
    return p.f16 ? launch_fwd_variant<true, true>(maps, p, s, sms, slot)
                 : launch_fwd_variant<true, false>(maps, p, s, sms, slot);
  return p.f16 ? launch_fwd_variant<false, true>(maps, p, s, sms, slot)
               : launch_fwd_variant<false, false>(maps, p, s, sms, slot);
}

}  // namespace sdpa
