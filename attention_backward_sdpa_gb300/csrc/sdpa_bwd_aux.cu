// sdpa_bwd_aux.cu -- the bandwidth-bound kernels of the SDPA backward chain.
//
//   preprocess  delta = rowsum(dO * O) in fp32 and the replay statistic
//               LSE * log2(e) (+inf for masked rows and LSE = -inf), staged
//               per query tile; clears the fp32 dQ accumulator and the
//               deterministic-mode counters. ("The kernel chain": dot.)
//   dq_convert  dQ = bf16(scale * dq_accum), dropping the accumulator's
//               padding rows. ("The kernel chain": cvt.)
//   gqa_reduce  dK/dV of each KV head = fp32 sum of its group's per-query-head
//               partials in ascending head order, rounded to bf16.
//               ("GQA/MQA group reduction".)
//
// All three move 16-byte vectors with consecutive threads on consecutive
// addresses; grids are sized to a few CTAs per SM and stride over the work.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ---------------------------------------------------------------- preprocess
template <int DV>
__global__ void __launch_bounds__(256) sdpa_bwd_preprocess(const ChainParams p) {
  // The main kernel may start its prologue (barrier setup, TMEM allocation,
  // K/V loads) while this grid runs; it waits for completion before reading
  // anything written here.
  pdl_launch_dependents();

  constexpr int TPR = DV / 8;  // threads per query row, 8 bf16 each
  constexpr float LOG2E = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const unsigned group_mask = (TPR == 32 ? 0xFFFFFFFFu : ((1u << TPR) - 1u) << (lane / TPR * TPR));
  const int sub = threadIdx.x % TPR;
  const long long rows = (long long)p.B * p.Hq * p.n_qt * BQ;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;

  for (long long r = tid / TPR; r < rows; r += nthreads / TPR) {
    const int qi = (int)(r % BQ);
    const long long t = r / BQ;
    const int qt = (int)(t % p.n_qt);
    const long long bh = t / p.n_qt;
    const int b = (int)(bh / p.Hq);
    const int q = qt * BQ + qi;
    int Lq, Lk;
    batch_lengths(p, b, Lq, Lk);
    float dot = 0.f;
    if (q < Lq) {
      const long long off = (bh * p.Sq + q) * (long long)DV + sub * 8;
      float fo[8], fd[8];
      unpack8(*reinterpret_cast<const uint4*>(p.o + off), fo);
      unpack8(*reinterpret_cast<const uint4*>(p.d_o + off), fd);
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(fo[i], fd[i], dot);
    }
#pragma unroll
    for (int s = TPR / 2; s > 0; s >>= 1) dot += __shfl_xor_sync(group_mask, dot, s, TPR);
    if (sub == 0) {
      float lse2 = INFINITY, delta = 0.f;
      if (q < Lq) {
        const float l = p.lse[bh * p.Sq + q];
        lse2 = (l == -INFINITY) ? INFINITY : l * LOG2E;
        delta = dot;
      }
      float* qs = p.qstat + t * QSTAT_FLOATS;
      qs[qi] = lse2;
      qs[BQ + qi] = delta;
    }
  }

  // Clear the dQ accumulator (dQ-reduction route), the stand-in zero dS tile
  // (two-kernel route), and the counters (+ ticket).
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.dq_accum) {
    float4* acc = reinterpret_cast<float4*>(p.dq_accum);
    const long long n4 = (long long)p.B * p.Hq * p.n_qt * BQ * p.Dqk / 4;
    for (long long i = tid; i < n4; i += nthreads) acc[i] = z;
  }
  if (p.zero_tile) {
    float4* zt = reinterpret_cast<float4*>(p.zero_tile);
    for (long long i = tid; i < DS_TILE_BYTES / 16; i += nthreads) zt[i] = z;
  }
  for (long long i = tid; i < p.n_counters; i += nthreads) p.counters[i] = 0;
}

// ---------------------------------------------------------------- dq convert
// dq_accum: [B*Hq][n_qt*BQ][Dqk] fp32, row-major; rows past S_q are padding.
template <int DQK>
__global__ void __launch_bounds__(256) sdpa_bwd_dq_convert(const ChainParams p) {
  pdl_wait_prior_grid();
  constexpr int PER_ROW = DQK / 8;
  const long long total = (long long)p.B * p.Hq * p.Sq * PER_ROW;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long rows_pad = (long long)p.n_qt * BQ;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
    const int c8 = (int)(i % PER_ROW);
    const long long r = i / PER_ROW;  // (b*Hq + h)*Sq + q
    const long long bh = r / p.Sq;
    const int q = (int)(r % p.Sq);
    const float* src = p.dq_accum + (bh * rows_pad + q) * DQK + c8 * 8;
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 c = *reinterpret_cast<const float4*>(src + 4);
    uint4 out;
    out.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    out.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    out.z = pack_bf16x2(c.x * p.scale, c.y * p.scale);
    out.w = pack_bf16x2(c.z * p.scale, c.w * p.scale);
    *reinterpret_cast<uint4*>(p.dq + r * DQK + c8 * 8) = out;
  }
}

// ---------------------------------------------------------------- GQA reduce
__global__ void __launch_bounds__(256) sdpa_bwd_gqa_reduce(const ChainParams p) {
  pdl_wait_prior_grid();
  const long long rows = (long long)p.B * p.Hkv * p.Skv;
  const long long nk = rows * (p.Dqk / 8), nv = rows * (p.Dv / 8);
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nk + nv; i += nthreads) {
    const bool is_k = i < nk;
    const long long vec = is_k ? i : i - nk;
    const int D = is_k ? p.Dqk : p.Dv;
    const __nv_bfloat16* ws = is_k ? p.dk_ws : p.dv_ws;
    __nv_bfloat16* out = is_k ? p.dk : p.dv;
    const long long row = vec / (D / 8);
    const int c8 = (int)(vec % (D / 8));
    const int k = (int)(row % p.Skv);
    const long long bhk = row / p.Skv;
    const int hk = (int)(bhk % p.Hkv);
    const long long b = bhk / p.Hkv;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < p.G; ++j) {  // ascending query head: fixed order
      const long long h = (long long)hk * p.G + j;
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(ws + ((b * p.Hq + h) * p.Skv + k) * D + c8 * 8), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += f[e];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + row * D + c8 * 8) = o;
  }
}

cudaError_t launch_preprocess(const ChainParams& p, int grid, cudaStream_t s) {
  return p.Dv == 64 ? launch_kernel(sdpa_bwd_preprocess<64>, dim3(grid), dim3(256), 0, s, false, p)
                    : launch_kernel(sdpa_bwd_preprocess<128>, dim3(grid), dim3(256), 0, s, false, p);
}

cudaError_t launch_gqa_reduce(const ChainParams& p, int grid, cudaStream_t s) {
  return launch_kernel(sdpa_bwd_gqa_reduce, dim3(grid), dim3(256), 0, s, true, p);
}

cudaError_t launch_dq_convert(const ChainParams& p, int grid, cudaStream_t s) {
  return p.Dqk == 64 ? launch_kernel(sdpa_bwd_dq_convert<64>, dim3(grid), dim3(256), 0, s, true, p)
                     : launch_kernel(sdpa_bwd_dq_convert<128>, dim3(grid), dim3(256), 0, s, true, p);
}

}  // namespace sdpa
