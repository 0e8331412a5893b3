// sdpa_bwd_dq.cu -- deterministic dQ from stored dS tiles (the "two-kernel
// split" of the cuDNN frontend page "SDPA Backward (SM120)", section
// "Determinism": the main kernel streams dS to a workspace and a Q-stationary
// kernel computes dQ = scale * dS K over an ascending key walk).
//
// A unit is 128 query rows (two 64-row query tiles) of one (batch, query
// head). For each unit a CTA walks, in ascending order, every 128-key tile that the main kernel
// visited for either of its query tiles (the same loop bounds), and for each
// loads the key tile K (TMA) and the two stored dS^T tiles (bulk copies of the
// main kernel's swizzled shared-memory images; a tile the main kernel did not
// visit is replaced by zeros). Per key tile it issues
//     dQ[q, d] += sum_key dS[q, key] K[key, d]
// as eight tcgen05.mma (M = 128 queries, N = D, K = 16 keys; both operands
// MN-major), accumulating in tensor memory. The fixed walk order makes dQ
// bitwise reproducible; there are no atomics and no fp32 accumulator in memory.
//
// Warps: 0-3 epilogue (tensor memory -> scale -> bf16 -> dQ; before that, the
// CTA's slice of the GQA dK/dV group reduction), 4 dS loads and unit claims,
// 5 MMA, 6 K loads.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "gqa.cuh"
#include "ptx.cuh"

namespace sdpa {

// One 32-byte store of two 16-byte halves (the address 32-byte aligned).
__device__ __forceinline__ void dq_store_32b(void* ptr, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a.x), "r"(a.y),
               "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

constexpr int DQ_THREADS = 224;
constexpr uint64_t DQ_WAIT_LIMIT_NS = 4000000000ull;

// K tiles (from L2: every query unit of a head reads them) and dS tiles (from
// HBM, read once) have rings of their own, so that the dS loads, whose latency
// paces the kernel, can run further ahead.
template <int D>
struct DqLayout {
  static constexpr int NK = (D <= 128) ? 3 : 2;         // K buffers (64 KiB each at D = 256)
  static constexpr int NDS = (D <= 128) ? 4 : 3;        // dS buffers
  static constexpr int TILE_K = BN * D * 2;             // [D/64 blocks][128 keys][128 B]
  static constexpr int TILE_DS = 2 * DS_TILE_BYTES;     // two dS^T tiles: [2][128 keys][64 q]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_DS = NK * TILE_K;
  static constexpr int OFF_BAR = OFF_DS + NDS * TILE_DS;
  // full/empty per K and dS buffer, acc full/empty x2, unit ring full/empty x URING
  static constexpr int URING = 4;
  static constexpr int NUM_BARS = 2 * NK + 2 * NDS + 4 + 2 * URING;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem base, abort flag, unit ring
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr uint32_t ACC_COLS = D <= 128 ? 128 : 256;   // one accumulator, padded
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;          // double-buffered
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "tensor memory budget");
};

// Work unit u (128 query rows of one (batch, query head)), in claiming order:
// query-tile pair descending, so that under a causal mask (where later query
// rows see more key tiles) the longest units are claimed first, and heads of
// the same pair next to each other.
struct DqUnit {
  int bh, qp, b, hk, qt0, qt1, Lq, Lk, kv_first, n;
};

__device__ __forceinline__ DqUnit dq_unit(const ChainParams& p, int u) {
  DqUnit w;
  const int n_qp = ceil_div(p.n_qt, 2);
  const int BH = p.B * p.Hq;
  w.qp = n_qp - 1 - u / BH;
  w.bh = u % BH;
  w.b = w.bh / p.Hq;
  w.hk = (w.bh % p.Hq) / p.G;
  w.qt0 = 2 * w.qp;
  w.qt1 = 2 * w.qp + 1;  // may be past the last tile
  batch_lengths(p, w.b, w.Lq, w.Lk);
  // Key tiles visited for either query tile, ascending: a contiguous range.
  // The walk starts at a lower bound (no key tile below it can see query row
  // 64*qt0 under a sliding window) and stops just past the range.
  int first = p.n_kt, last = -1;
  int kt_start = 0;
  if (p.window_left >= 0) {
    const int diag = p.bottom_right ? w.Lk - w.Lq : 0;
    kt_start = (int)max(0ll, floor_div((long long)w.qt0 * BQ + diag - p.window_left, BN) - 1);
  }
  for (int kt = kt_start; kt < p.n_kt; ++kt) {
    int lo, hi;
    visited_query_tiles(kt, w.Lq, w.Lk, p.causal, p.bottom_right, p.window_left, p.window_right, lo, hi);
    if ((lo <= w.qt0 && w.qt0 <= hi) || (w.qt1 < p.n_qt && lo <= w.qt1 && w.qt1 <= hi)) {
      first = min(first, kt);
      last = kt;
    } else if (last >= 0) {
      break;
    }
  }
  w.kv_first = first;
  w.n = last - first + 1;  // may be <= 0
  return w;
}

// Persistent: one CTA per SM. The load warp claims units from a global ticket
// (longest first, so the CTAs finish together) and publishes each to the MMA
// warp and the epilogue through a small ring in shared memory; it runs ahead
// across unit boundaries through one stage ring. The MMA warp alternates
// between two tensor-memory accumulators (counted over non-empty units only)
// so that the epilogue of one unit overlaps the next.
template <int D, bool F16 = false>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    sdpa_bwd_dq_from_ds(const __grid_constant__ CUtensorMap k_map, const ChainParams p) {
  using L = DqLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(p.status, STATUS_SMEM_ALIGN);
    return;
  }
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kempty = kfull + L::NK;
  uint64_t* dsfull = kempty + L::NK;
  uint64_t* dsempty = dsfull + L::NDS;
  uint64_t* acc_full = dsempty + L::NDS;    // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2], 128 arrivals
  uint64_t* ufull = acc_empty + 2;          // [URING]
  uint64_t* uempty = ufull + L::URING;      // [URING], 6 arrivals (K loads, MMA, 4 epilogue warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);
  const int n_units = ceil_div(p.n_qt, 2) * p.B * p.Hq;
  // Reads ring entry i (a unit, or -1 at the end) and releases it; all lanes of a warp.
  auto ring_get = [&](int i, int& unit) -> bool {
    const int r = i % L::URING;
    if (!mbar_wait(&ufull[r], (i / L::URING) & 1, abort_flag, DQ_WAIT_LIMIT_NS)) return false;
    unit = ring[r];
    __syncwarp();
    if (lane == 0) mbar_arrive(&uempty[r]);
    return true;
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < L::NK; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < L::NDS; ++i) {
      mbar_init(&dsfull[i], 1);
      mbar_init(&dsempty[i], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 128);
    mbar_init(&acc_empty[1], 128);
    for (int i = 0; i < L::URING; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], 6);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The main kernel lets this grid launch while its last units run (once each
  // of its CTAs has passed the wait for the preprocess, which clears the ticket
  // and the zero tile): setup, unit claims and K loads proceed, and the roles
  // that read the main kernel's output (dS tiles, GQA partial sets) wait for
  // its completion first.

  if (warp == 4) {
    // ------------------------------------------------------------ dS loads, unit claims
    if (lane == 0) {
      int step = 0;
      bool main_done = false;
      for (int e = 0;; ++e) {
        // The ticket was cleared by the preprocess kernel; on this route the
        // main kernel does not use it.
        const int u = atomicAdd(p.ticket, 1);
        const int r = e % L::URING;
        if (e >= L::URING &&
            !mbar_wait(&uempty[r], ((e / L::URING) - 1) & 1, abort_flag, DQ_WAIT_LIMIT_NS))
          goto loads_done;
        ring[r] = u < n_units ? u : -1;
        mbar_arrive(&ufull[r]);
        if (u >= n_units) break;
        const DqUnit w = dq_unit(p, u);
        long long band_prefix = w.n > 0 ? ds_band_prefix(p, w.kv_first) : 0;
        for (int i = 0; i < w.n; ++i, ++step) {
          const int st = step % L::NDS;
          const int kt = w.kv_first + i;
          if (step >= L::NDS &&
              !mbar_wait(&dsempty[st], ((step / L::NDS) - 1) & 1, abort_flag, DQ_WAIT_LIMIT_NS))
            goto loads_done;
          uint8_t* stage = smem + L::OFF_DS + st * L::TILE_DS;
          if (!main_done) {
            pdl_wait_prior_grid();  // the dS tiles come from the main kernel
            main_done = true;
          }
          mbar_arrive_expect_tx(&dsfull[st], L::TILE_DS);
          int lo, hi;
          visited_query_tiles(kt, w.Lq, w.Lk, p.causal, p.bottom_right, p.window_left, p.window_right, lo, hi);
          // Without length arrays the band is the visited range itself.
          int band_lo = lo, band_hi = hi;
          if (p.seq_q_lens != nullptr || p.seq_kv_lens != nullptr) ds_band_range(p, kt, band_lo, band_hi);
          for (int half = 0; half < 2; ++half) {
            const int qt = w.qt0 + half;
            const bool stored = qt < p.n_qt && lo <= qt && qt <= hi;
            const uint8_t* src = stored ? ds_tile(p, w.bh, band_prefix, band_lo, qt) : p.zero_tile;
            if (stored ? in_bounds(p.status, src, DS_TILE_BYTES, p.ds_ws, ds_ws_bytes(p))
                       : in_bounds(p.status, src, DS_TILE_BYTES, p.zero_tile, DS_TILE_BYTES))
              bulk_load(stage + half * DS_TILE_BYTES, src, DS_TILE_BYTES, &dsfull[st]);
            else
              mbar_complete_tx(&dsfull[st], DS_TILE_BYTES);
          }
          if (band_hi >= band_lo) band_prefix += band_hi - band_lo + 1;
        }
      }
    loads_done:;
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ K loads
    bool ok = true;
    int step = 0;
    if (lane == 0) prefetch_tmap(&k_map);
    for (int e = 0; ok; ++e) {
      int u;
      if (!ring_get(e, u) || u < 0) break;
      const DqUnit w = dq_unit(p, u);
      for (int i = 0; i < w.n; ++i, ++step) {
        const int st = step % L::NK;
        if (step >= L::NK &&
            !mbar_wait(&kempty[st], ((step / L::NK) - 1) & 1, abort_flag, DQ_WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* stage = smem + L::OFF_K + st * L::TILE_K;
          mbar_arrive_expect_tx(&kfull[st], L::TILE_K);
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_3d(stage + blk * (BN * 128), &k_map, &kfull[st], blk * 64,
                        (w.kv_first + i) * BN, w.b * p.Hkv + w.hk);
        }
        __syncwarp();
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA
    constexpr uint32_t ID = idesc_io(128, D, true, true, F16);
    constexpr uint64_t T_MN = sdesc_sw128_template(BN * 128, 1024);  // 16 KB block stride
    bool ok = true;
    int step = 0, done_units = 0;
    for (int e = 0; ok; ++e) {
      int u;
      if (!ring_get(e, u) || u < 0) break;
      const DqUnit w = dq_unit(p, u);
      if (w.n <= 0) continue;
      const int buf = done_units & 1;
      const uint32_t acc = tmem + buf * L::ACC_COLS;
      // The accumulator was read out by the epilogue two non-empty units ago.
      if (done_units >= 2 &&
          !mbar_wait(&acc_empty[buf], ((done_units >> 1) - 1) & 1, abort_flag, DQ_WAIT_LIMIT_NS)) {
        ok = false;
        break;
      }
      __syncwarp();
      tc_fence_after();
      for (int i = 0; i < w.n; ++i, ++step) {
        const int sk = step % L::NK, sd = step % L::NDS;
        ok = mbar_wait(&kfull[sk], (step / L::NK) & 1, abort_flag, DQ_WAIT_LIMIT_NS) &&
             mbar_wait(&dsfull[sd], (step / L::NDS) & 1, abort_flag, DQ_WAIT_LIMIT_NS);
        __syncwarp();
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t aK = smem_u32(smem + L::OFF_K + sk * L::TILE_K);
          const uint32_t aS = smem_u32(smem + L::OFF_DS + sd * L::TILE_DS);
          // A = dS as (M = 128 queries, K = keys): the stored dS^T tiles are
          // [key][query] with queries contiguous, i.e. MN-major, the two 64-query
          // tiles 16 KB apart. B = K as (N = d, K = keys): MN-major as well.
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_ss(acc, sdesc_at(T_MN, aS + k * 2048), sdesc_at(T_MN, aK + k * 2048), ID,
                   (i > 0 || k > 0));
          mma_commit(&kempty[sk]);
          mma_commit(&dsempty[sd]);
          if (i == w.n - 1) mma_commit(&acc_full[buf]);
        }
        __syncwarp();
      }
      ++done_units;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // dQ of each unit as its accumulator completes. This CTA's slice of the GQA
    // group sums (dK/dV, which depend only on the main kernel) is split into one
    // piece per unit, each reduced while that unit's MMAs run.
    // The GQA slice is cut into as many pieces as the CTA's fair share of units;
    // pieces left over when the CTA runs out of units are reduced at the end.
    const int n_pieces = (n_units + (int)gridDim.x - 1) / (int)gridDim.x;
    int unit_idx = 0;
    pdl_wait_prior_grid();  // the GQA partial sets come from the main kernel
    const int row = warp * 32 + lane;          // query within the 128-row unit
    // A thread writes its own dQ row: in 32-byte stores (whole sectors) when dQ's
    // base is 32-byte aligned (its rows, D x 2 bytes, then are too), else 16-byte.
    const bool dq_sector = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    int done_units = 0;
    bool ok = true;
    for (int e = 0;; ++e) {
      int u;
      if (!ring_get(e, u)) {
        ok = false;
        break;
      }
      if (u < 0) break;
      const DqUnit w = dq_unit(p, u);
      const int q = w.qt0 * BQ + row;
      __nv_bfloat16* out = p.dq + ((long long)w.bh * p.Sq + q) * D;
      const bool have = w.n > 0;
      const int buf = done_units & 1;
      gqa_reduce_slice<F16>(p, blockIdx.x, gridDim.x, tid, 128, unit_idx++, n_pieces);
      if (have && ok) {
        ok = mbar_wait(&acc_full[buf], (done_units >> 1) & 1, abort_flag, DQ_WAIT_LIMIT_NS);
        __syncwarp();
        tc_fence_after();
      }
      const bool warp_ok = __all_sync(0xffffffffu, ok);
#pragma unroll
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t r[32];
        if (have && warp_ok) {
          tmem_ld32(t_lane + buf * L::ACC_COLS + c32 * 32, r);
          tmem_ld_wait(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (q < p.Sq) {
          uint4 o[4];
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            o[v8].x = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 0]) * p.scale, __uint_as_float(r[v8 * 8 + 1]) * p.scale);
            o[v8].y = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 2]) * p.scale, __uint_as_float(r[v8 * 8 + 3]) * p.scale);
            o[v8].z = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 4]) * p.scale, __uint_as_float(r[v8 * 8 + 5]) * p.scale);
            o[v8].w = pack_io2<F16>(__uint_as_float(r[v8 * 8 + 6]) * p.scale, __uint_as_float(r[v8 * 8 + 7]) * p.scale);
          }
          if (dq_sector) {
            dq_store_32b(out + c32 * 32, o[0], o[1]);
            dq_store_32b(out + c32 * 32 + 16, o[2], o[3]);
          } else {
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8) *reinterpret_cast<uint4*>(out + c32 * 32 + v8 * 8) = o[v8];
          }
        }
      }
      if (have) {
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        ++done_units;
      }
    }
    for (; unit_idx < n_pieces; ++unit_idx)
      gqa_reduce_slice<F16>(p, blockIdx.x, gridDim.x, tid, 128, unit_idx, n_pieces);
  }

  pdl_wait_prior_grid();  // this grid ends after the main kernel's
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16>
static cudaError_t set_dq_smem() {
  return cudaFuncSetAttribute(sdpa_bwd_dq_from_ds<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DqLayout<D>::BYTES);
}

cudaError_t dq_kernel_setup() {
  cudaError_t e = set_dq_smem<128, false>();
  if (e == cudaSuccess) e = set_dq_smem<192, false>();
  if (e == cudaSuccess) e = set_dq_smem<256, false>();
  if (e == cudaSuccess) e = set_dq_smem<128, true>();
  if (e == cudaSuccess) e = set_dq_smem<192, true>();
  if (e == cudaSuccess) e = set_dq_smem<256, true>();
  return e;
}

template <bool F16>
static cudaError_t launch_dq_variant(const CUtensorMap& k_map, const ChainParams& p, cudaStream_t s,
                                     dim3 grid) {
  if (p.Dqk == 192)
    return launch_kernel(sdpa_bwd_dq_from_ds<192, F16>, grid, dim3(DQ_THREADS), DqLayout<192>::BYTES, s,
                         true, k_map, p);
  if (p.Dqk == 256)
    return launch_kernel(sdpa_bwd_dq_from_ds<256, F16>, grid, dim3(DQ_THREADS), DqLayout<256>::BYTES, s,
                         true, k_map, p);
  return launch_kernel(sdpa_bwd_dq_from_ds<128, F16>, grid, dim3(DQ_THREADS), DqLayout<128>::BYTES, s,
                       true, k_map, p);
}

// Persistent: one CTA per SM (at most one per unit).
cudaError_t launch_dq_from_ds(const CUtensorMap& k_map, const ChainParams& p, cudaStream_t s,
                              int num_sms) {
  const int units = ceil_div(p.n_qt, 2) * p.B * p.Hq;
  const dim3 grid((unsigned)(units < num_sms ? units : num_sms));
  return p.f16 ? launch_dq_variant<true>(k_map, p, s, grid) : launch_dq_variant<false>(k_map, p, s, grid);
}

}  // namespace sdpa
