// sdpa_bwd_aux.cu -- the bandwidth-bound kernels of the SDPA backward chain.
//
//   preprocess  delta = rowsum(dO * O) in fp32 and the replay statistic
//               LSE * log2(e) (+inf for masked rows and LSE = -inf), staged
//               per query tile; clears the fp32 dQ accumulator (rows below
//               the query length) and the deterministic-mode counters;
//               clears a dBias that B > 1 batch rows add into atomically.
//               ("The kernel chain": dot.)
//   dq_convert  dQ = bf16(scale * dq_accum), dropping the accumulator's
//               padding rows. ("The kernel chain": cvt.)
// The dQ convert also carries the GQA group reduction of dK/dV (gqa.cuh).
//
// Both move 16-byte vectors with consecutive threads on consecutive
// addresses; grids are sized to a few CTAs per SM and stride over the work.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "gqa.cuh"
#include "ptx.cuh"

namespace sdpa {

// ---------------------------------------------------------------- dBias zeros
// One dBias shared by B > 1 batch rows receives their terms by atomic adds, so
// it must be all zeros before the main kernel starts: the batch-row-0 tiles of
// this kernel clear it, query tile by query tile (16-byte stores where the
// rows allow). A per-batch dBias is not touched here: the main kernel writes
// every element of the blocks it computes and zeros the others.
__device__ void zero_shared_dbias_rows(const ChainParams& p, unsigned bh, int qt) {
  const int b = (int)(bh / (unsigned)p.Hq), h = (int)(bh % (unsigned)p.Hq);
  if (b != 0) return;
  const int q0 = qt * BQ, rows = min(BQ, p.Sq - q0);
  float* base = p.dbias + ((long long)h * p.Sq + q0) * p.Skv;
  const long long n = (long long)rows * p.Skv;  // contiguous rows
  long long i0 = 0;
  while (i0 < n && ((reinterpret_cast<uintptr_t>(base + i0) & 15u) != 0)) ++i0;  // scalar head
  if ((long long)threadIdx.x < i0) base[threadIdx.x] = 0.f;
  const long long n4 = (n - i0) / 4;
  float4* v = reinterpret_cast<float4*>(base + i0);
  for (long long i = threadIdx.x; i < n4; i += blockDim.x) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = i0 + 4 * n4 + threadIdx.x; i < n; i += blockDim.x) base[i] = 0.f;  // tail
}

// ---------------------------------------------------------------- preprocess
// Persistent and TMA-staged: a CTA walks the 64-row query tiles t = blockIdx.x,
// + gridDim.x, ... with PRE_STAGES tiles in flight. One thread issues each
// tile's O and dO rows (the rows below the query length: contiguous, 16-byte
// multiples) as two bulk copies into a shared-memory stage ring, and clears
// the tile's dQ accumulator rows with bulk stores from a zeroed buffer; all
// threads reduce the rows from shared memory. Two CTAs per SM keep about
// 192 KB of loads in flight per SM (one short CTA per tile, reading into
// registers, left half the HBM bandwidth idle).
// TPR = DV/8 lanes per row (8 io elements each), 256 / TPR rows per pass;
// lanes past D_v/8 (D_v not a power-of-two multiple of 8) read nothing.
constexpr int PRE_THREADS = 256;
constexpr int PRE_STAGES = 3;
constexpr int PRE_ZERO = 16384;                      // zero source of the accumulator clear
template <int TPR>
struct PreLayout {
  static constexpr int TILE = BQ * TPR * 8 * 2;      // one 64-row io tile at D_v <= 8 * TPR
  static constexpr int OFF_O = 0;
  static constexpr int OFF_DO = OFF_O + PRE_STAGES * TILE;
  static constexpr int OFF_ZERO = OFF_DO + PRE_STAGES * TILE;
  static constexpr int OFF_BAR = OFF_ZERO + PRE_ZERO;
  static constexpr int BYTES = OFF_BAR + PRE_STAGES * 8;
  // Up to D_v = 128 two CTAs share an SM; at 256 one CTA takes 208 KiB.
  static constexpr int CTAS_PER_SM = BYTES <= 113 * 1024 ? 2 : 1;
};

template <int TPR, bool F16>
__global__ void __launch_bounds__(PRE_THREADS, 2) sdpa_bwd_preprocess(const ChainParams p) {
  // The main kernel may start its prologue (barrier setup, TMEM allocation,
  // K/V loads) while this grid runs; it waits for completion before reading
  // anything written here.
  pdl_launch_dependents();

  using PL = PreLayout<TPR>;
  constexpr int PRE_TILE = PL::TILE;
  constexpr int PRE_OFF_O = PL::OFF_O, PRE_OFF_DO = PL::OFF_DO, PRE_OFF_ZERO = PL::OFF_ZERO;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PL::OFF_BAR);
  const uint8_t* zero = smem + PRE_OFF_ZERO;
  const int DV = p.Dv;
  constexpr int RPP = PRE_THREADS / TPR;   // rows per pass
  constexpr int PASSES = BQ / RPP;         // passes per 64-row tile
  constexpr float LOG2E = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const unsigned group_mask = (TPR == 32 ? 0xFFFFFFFFu : ((1u << TPR) - 1u) << (lane / TPR * TPR));
  const int sub = threadIdx.x % TPR;
  const int rsub = threadIdx.x / TPR;
  const unsigned n_tiles = (unsigned)p.B * p.Hq * p.n_qt;
  __shared__ float sink_terms[BQ];  // per-row sink terms of the current tile
  __shared__ int abort_flag;         // a stage wait that ran out (then results are invalid)

  for (int i = threadIdx.x; i < PRE_ZERO / 16; i += PRE_THREADS)
    reinterpret_cast<uint4*>(smem + PRE_OFF_ZERO)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int st = 0; st < PRE_STAGES; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zeros are read by bulk stores
  __syncthreads();

  // Query rows of tile t below the length, i.e. the rows the bulk copies fill.
  auto live_rows = [&](unsigned t, unsigned& bh, int& qt, int& Lq) {
    bh = t / (unsigned)p.n_qt;
    qt = (int)(t - bh * (unsigned)p.n_qt);
    int Lk;
    batch_lengths(p, (int)(bh / (unsigned)p.Hq), Lq, Lk);
    return max(0, min(BQ, Lq - qt * BQ));
  };
  // Thread 0: the loads of this CTA's k-th tile into stage k % PRE_STAGES.
  auto issue = [&](unsigned k) {
    const unsigned t = blockIdx.x + k * gridDim.x;
    if (t >= n_tiles) return;
    unsigned bh;
    int qt, Lq;
    const int rows = live_rows(t, bh, qt, Lq);
    uint64_t* bar = &full[k % PRE_STAGES];
    if (rows == 0) {
      mbar_arrive(bar);
      return;
    }
    const uint32_t bytes = (uint32_t)rows * DV * 2;
    const long long row0 = (long long)bh * p.Sq + (long long)qt * BQ;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    if (in_bounds(p.status, p.o + row0 * DV, bytes, p.o, io_q_bytes(p, DV)) &&
        in_bounds(p.status, p.d_o + row0 * DV, bytes, p.d_o, io_q_bytes(p, DV)) && bytes <= PRE_TILE) {
      // O is read only here (dO is read again by the main kernel): on the
      // reduction route it makes way for the dQ accumulator cleared below.
      bulk_load_hint(smem + PRE_OFF_O + (k % PRE_STAGES) * PRE_TILE, p.o + row0 * DV, bytes, bar,
                     p.dq_accum ? l2_evict_first() : l2_evict_normal());
      bulk_load(smem + PRE_OFF_DO + (k % PRE_STAGES) * PRE_TILE, p.d_o + row0 * DV, bytes, bar);
    } else {
      mbar_complete_tx(bar, 2 * bytes);
    }
  };
  if (threadIdx.x == 0)
    for (unsigned k = 0; k < PRE_STAGES; ++k) issue(k);

  unsigned k = 0;
  for (unsigned t = blockIdx.x; t < n_tiles; t += gridDim.x, ++k) {
    unsigned bh;
    int qt, Lq;
    const int rows = live_rows(t, bh, qt, Lq);
    // dQ-reduction route: clear this tile's accumulator rows below Lq (the
    // convert kernel writes zeros for rows at or past Lq without reading them).
    if (threadIdx.x == 0 && p.dq_accum && rows > 0) {
      uint8_t* acc = reinterpret_cast<uint8_t*>(p.dq_accum + ((long long)bh * p.n_qt + qt) * BQ * p.dq_acc_cols);
      const uint32_t total = (uint32_t)rows * p.dq_acc_cols * 4;
      if (in_bounds(p.status, acc, total, p.dq_accum, dq_accum_bytes(p)))
        for (uint32_t off = 0; off < total; off += PRE_ZERO)
          bulk_store_hint(acc + off, zero, total - off < (uint32_t)PRE_ZERO ? total - off : (uint32_t)PRE_ZERO,
                          l2_evict_last());  // the main kernel's reductions follow
      bulk_commit_group();
    }
    if (p.dbias_red) zero_shared_dbias_rows(p, bh, qt);
    float lv[PASSES];  // the rows' LSE, requested before the wait for the stage
#pragma unroll
    for (int u = 0; u < PASSES; ++u) {
      const int q = qt * BQ + u * RPP + rsub;
      lv[u] = (q < Lq && sub == 0) ? p.lse[(long long)bh * p.Sq + q] : 0.f;
    }
    const int st = (int)(k % PRE_STAGES);
    if (!mbar_wait(&full[st], (k / PRE_STAGES) & 1, &abort_flag, 4000000000ull)) {
      atomicOr(p.status, STATUS_TIMEOUT);
      break;  // every thread leaves (the flag is shared); nothing waits on this kernel's threads
    }
    const uint8_t* so = smem + PRE_OFF_O + st * PRE_TILE;
    const uint8_t* sd = smem + PRE_OFF_DO + st * PRE_TILE;
    float* qs = p.qstat + (long long)t * QSTAT_FLOATS;
    const bool qs_ok = in_bounds(p.status, qs, QSTAT_FLOATS * 4, p.qstat, qstat_bytes(p));
    const float sink2 = p.dsink_part ? p.sink[bh % (unsigned)p.Hq] * LOG2E : 0.f;
#pragma unroll
    for (int u = 0; u < PASSES; ++u) {
      const int qi = u * RPP + rsub;
      const int q = qt * BQ + qi;
      float dot = 0.f;
      if (qi < rows && sub * 8 < DV) {
        float fo[8], fd[8];
        unpack8<F16>(*reinterpret_cast<const uint4*>(so + (qi * DV + sub * 8) * 2), fo);
        unpack8<F16>(*reinterpret_cast<const uint4*>(sd + (qi * DV + sub * 8) * 2), fd);
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(fo[i], fd[i], dot);
      }
#pragma unroll
      for (int sft = TPR / 2; sft > 0; sft >>= 1) dot += __shfl_xor_sync(group_mask, dot, sft, TPR);
      if (sub == 0) {
        float lse2 = INFINITY, delta = 0.f;
        if (q < Lq) {
          const float l = lv[u];
          lse2 = (l == -INFINITY) ? INFINITY : l * LOG2E;
          delta = dot;
        }
        if (qs_ok) {
          qs[qi] = lse2;
          qs[BQ + qi] = delta;
        }
        // Sink term of this row: exp(sink - LSE) * delta (0 for a row past the
        // length, whose delta is 0, or with LSE = -inf, whose lse2 is +inf).
        if (p.dsink_part) sink_terms[qi] = exp2f(sink2 - lse2) * delta;
      }
    }
    // Every thread has read the stage (and the sink terms are written): the
    // stage takes the tile PRE_STAGES ahead.
    __syncthreads();
    if (threadIdx.x == 0) {
      if (p.dsink_part) {
        // The tile's 64 terms in ascending row order, by one thread: bitwise
        // reproducible, and so is the fixed-order sum of the tiles (dsink kernel).
        float acc = 0.f;
        for (int i = 0; i < BQ; ++i) acc += sink_terms[i];
        p.dsink_part[t] = acc;
      }
      issue(k + PRE_STAGES);
    }
    if (p.dsink_part) __syncthreads();  // sink_terms is rewritten by the next tile
  }
  if (threadIdx.x == 0) bulk_wait_group_read0();  // the zero buffer outlives its readers

  // Clear the stand-in zero dS tile (two-kernel route) and the counters (+ ticket).
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.zero_tile) {
    float4* zt = reinterpret_cast<float4*>(p.zero_tile);
    for (long long i = tid; i < DS_TILE_BYTES / 16; i += nthreads) zt[i] = z;
  }
  for (long long i = tid; i < p.n_counters; i += nthreads) p.counters[i] = 0;
}

// ---------------------------------------------------------------- dq convert
// dq_accum: [B*Hq][n_qt*BQ][Dqk] fp32, row-major; rows past S_q are padding.
// One 64-row query tile per CTA: 64 rows x DQK/8 chunks of 8 columns, every
// thread's loads issued before any store, index arithmetic once per tile. Rows
// at or past the batch row's query length are written as zeros without being
// read (the preprocess kernel did not clear them). The kernel also carries a
// slice of the GQA group reduction of dK/dV (gqa.cuh).
// ACC: the accumulator's row width (64 or 128, that of the main kernel that
// ran); D_qk (<= ACC, a multiple of 8) is the width of dQ.
template <int ACC, bool F16>
__global__ void __launch_bounds__(256) sdpa_bwd_dq_convert(const ChainParams p) {
  pdl_wait_prior_grid();
  gqa_reduce_slice<F16>(p, blockIdx.x, gridDim.x, threadIdx.x, blockDim.x);
  const int DQK = p.Dqk;
  const int CPR = DQK / 8;                      // 8-column chunks per row of dQ
  constexpr int MAX_ITEMS = BQ * (ACC / 8) / 256;
  const unsigned bh = blockIdx.x / (unsigned)p.n_qt;
  const int qt = (int)(blockIdx.x - bh * (unsigned)p.n_qt);
  int Lq, Lk;
  batch_lengths(p, (int)(bh / (unsigned)p.Hq), Lq, Lk);
  const int rows = min(BQ, p.Sq - qt * BQ);         // rows of dQ in this tile
  const int live = max(0, min(rows, Lq - qt * BQ)); // rows holding accumulated values
  const float* src = p.dq_accum + ((long long)bh * p.n_qt + qt) * BQ * ACC;
  __nv_bfloat16* dst = p.dq + ((long long)bh * p.Sq + (long long)qt * BQ) * DQK;
  if (!in_bounds(p.status, src, (size_t)BQ * ACC * 4, p.dq_accum, dq_accum_bytes(p)) ||
      !in_bounds(p.status, dst, (size_t)rows * DQK * 2, p.dq, io_q_bytes(p, DQK)))
    return;
  float4 a[MAX_ITEMS], c[MAX_ITEMS];
#pragma unroll
  for (int u = 0; u < MAX_ITEMS; ++u) {
    const int i = threadIdx.x + u * 256, r = i / CPR, c8 = i % CPR;
    if (r < live) {
      a[u] = *reinterpret_cast<const float4*>(src + r * ACC + c8 * 8);
      c[u] = *reinterpret_cast<const float4*>(src + r * ACC + c8 * 8 + 4);
    } else {
      a[u] = c[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int u = 0; u < MAX_ITEMS; ++u) {
    const int i = threadIdx.x + u * 256, r = i / CPR, c8 = i % CPR;
    if (r < rows) {
      uint4 out;
      out.x = pack_io2<F16>(a[u].x * p.scale, a[u].y * p.scale);
      out.y = pack_io2<F16>(a[u].z * p.scale, a[u].w * p.scale);
      out.z = pack_io2<F16>(c[u].x * p.scale, c[u].y * p.scale);
      out.w = pack_io2<F16>(c[u].z * p.scale, c[u].w * p.scale);
      *reinterpret_cast<uint4*>(dst + r * DQK + c8 * 8) = out;
    }
  }
}

// ---------------------------------------------------------------- dsink
// dsink[h] = -sum_{b,q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q] ("SDPA
// Backward (SM120)", the `dsink` step of the kernel chain and the sink-token
// capability). The preprocess kernel left one fixed-order partial per 64-row
// tile; one CTA per head sums the head's B * n_qt partials: each thread a fixed
// strided subset in ascending order, then a fixed-shape tree. Every run adds
// in the same order, so dsink is bitwise reproducible.
constexpr int DSINK_THREADS = 256;

__global__ void __launch_bounds__(DSINK_THREADS) sdpa_bwd_dsink(const ChainParams p) {
  __shared__ float part[DSINK_THREADS];
  const int h = blockIdx.x;
  const int n = p.B * p.n_qt;  // partials of head h: index b * n_qt + qt
  float acc = 0.f;
  for (int i = threadIdx.x; i < n; i += DSINK_THREADS) {
    const int b = i / p.n_qt, qt = i - b * p.n_qt;
    acc += p.dsink_part[((long long)b * p.Hq + h) * p.n_qt + qt];
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = DSINK_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.dsink[h] = -part[0];
}

__global__ void __launch_bounds__(256) sdpa_dbias_cast(const float* __restrict__ src,
                                                       unsigned short* __restrict__ dst, long long n,
                                                       int f16) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256)
    dst[i] = f32_to_16(src[i], f16 != 0);
}

cudaError_t launch_dbias_cast(const float* src, void* dst, long long n, bool f16, int num_sms,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long want = (n + 255) / 256, cap = (long long)num_sms * 8;
  return launch_kernel(sdpa_dbias_cast, dim3((unsigned)(want < cap ? want : cap)), dim3(256), 0, s, false,
                       src, static_cast<unsigned short*>(dst), n, f16 ? 1 : 0);
}

cudaError_t launch_dsink(const ChainParams& p, cudaStream_t s) {
  return launch_kernel(sdpa_bwd_dsink, dim3((unsigned)p.Hq), dim3(DSINK_THREADS), 0, s, false, p);
}

// The convert takes one 64-row query tile per CTA and leaves the balancing of
// the tiles to the hardware dispatcher.
// Persistent: two CTAs per SM (fewer when there are fewer tiles).
template <int TPR, bool F16>
static cudaError_t launch_preprocess_tpr(const ChainParams& p, cudaStream_t s, int num_sms) {
  const long long tiles = (long long)p.B * p.Hq * p.n_qt;
  const long long cap = (long long)PreLayout<TPR>::CTAS_PER_SM * num_sms;
  const dim3 grid((unsigned)(tiles < cap ? tiles : cap));
  return launch_kernel(sdpa_bwd_preprocess<TPR, F16>, grid, dim3(PRE_THREADS), PreLayout<TPR>::BYTES, s,
                       false, p);
}

template <bool F16>
static cudaError_t launch_preprocess_io(const ChainParams& p, cudaStream_t s, int num_sms) {
  if (p.Dv <= 32) return launch_preprocess_tpr<4, F16>(p, s, num_sms);
  if (p.Dv <= 64) return launch_preprocess_tpr<8, F16>(p, s, num_sms);
  if (p.Dv <= 128) return launch_preprocess_tpr<16, F16>(p, s, num_sms);
  return launch_preprocess_tpr<32, F16>(p, s, num_sms);
}

template <int TPR, bool F16>
static cudaError_t set_pre_smem() {
  return cudaFuncSetAttribute(sdpa_bwd_preprocess<TPR, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PreLayout<TPR>::BYTES);
}

cudaError_t preprocess_kernel_setup() {
  cudaError_t e = set_pre_smem<4, false>();
  if (e == cudaSuccess) e = set_pre_smem<8, false>();
  if (e == cudaSuccess) e = set_pre_smem<16, false>();
  if (e == cudaSuccess) e = set_pre_smem<32, false>();
  if (e == cudaSuccess) e = set_pre_smem<4, true>();
  if (e == cudaSuccess) e = set_pre_smem<8, true>();
  if (e == cudaSuccess) e = set_pre_smem<16, true>();
  if (e == cudaSuccess) e = set_pre_smem<32, true>();
  return e;
}

cudaError_t launch_preprocess(const ChainParams& p, cudaStream_t s, int num_sms) {
  return p.f16 ? launch_preprocess_io<true>(p, s, num_sms) : launch_preprocess_io<false>(p, s, num_sms);
}

template <bool F16>
static cudaError_t launch_dq_convert_io(const ChainParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.B * p.Hq * p.n_qt));
  if (p.dq_acc_cols == 64) return launch_kernel(sdpa_bwd_dq_convert<64, F16>, grid, dim3(256), 0, s, true, p);
  return launch_kernel(sdpa_bwd_dq_convert<128, F16>, grid, dim3(256), 0, s, true, p);
}

cudaError_t launch_dq_convert(const ChainParams& p, cudaStream_t s) {
  return p.f16 ? launch_dq_convert_io<true>(p, s) : launch_dq_convert_io<false>(p, s);
}

}  // namespace sdpa
