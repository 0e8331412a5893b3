// bias.cuh -- additive-bias helpers of the backward main kernels (cuDNN
// frontend docs, "SDPA Backward (SM120)": the bias capability). In both main
// kernels a compute thread owns one key of a 128-key tile, so one query column
// of a tile's bias or dBias is 32 consecutive elements across a warp.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace sdpa {

// Bias column of one query tile for this thread's key: bz[i] = bias(q0 + i, k)
// (0 past S_q or S_kv); bf16, fp16 or fp32 elements. `off` is the element offset of (batch row, head, q0, k).
template <int N>
__device__ __forceinline__ void load_bias_column(const ChainParams& p, long long off, bool key_in,
                                                 int q0, float (&bz)[N]) {
  const long long ld = p.Skv;
  const int rows = key_in ? min(N, p.Sq - q0) : 0;
  if (p.bias_fp32) {
    const float* src = static_cast<const float*>(p.bias) + off;
    if (rows == N) {
#pragma unroll
      for (int i = 0; i < N; ++i) bz[i] = __ldcs(src + i * ld);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) bz[i] = i < rows ? __ldcs(src + i * ld) : 0.f;
    }
  } else {
    // (One loop per element type: a per-element choice cost the replay a
    // select on every value.)
    const unsigned short* src = static_cast<const unsigned short*>(p.bias) + off;
    if (p.bias_f16) {
#pragma unroll
      for (int i = 0; i < N; ++i) bz[i] = i < rows ? __half2float(__ushort_as_half(__ldcs(src + i * ld))) : 0.f;
    } else if (rows == N) {
#pragma unroll
      for (int i = 0; i < N; ++i) bz[i] = __uint_as_float((uint32_t)__ldcs(src + i * ld) << 16);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i)
        bz[i] = i < rows ? __uint_as_float((uint32_t)__ldcs(src + i * ld) << 16) : 0.f;
    }
  }
}

// Zeros `rows` rows of `cols` elements of ESZ bytes (4 or 2), `ld` elements
// apart, with threads thr = 0 .. nthr-1 (nthr a multiple of 32). A full
// 128-column block row is 32 (fp32) or 16 (16-bit) 16-byte stores, one per lane
// of a warp; other shapes take element stores. (The element size is a template
// argument: computed at run time it cost the biased kernel 10 % through this
// loop.)
template <int ESZ>
__device__ __forceinline__ void zero_elem_rows(char* base, int rows, int cols, long long ld, int thr,
                                               int nthr) {
  constexpr int VPR = BN * ESZ / 16;  // 16-byte vectors per full row
  if (cols == BN && (reinterpret_cast<uintptr_t>(base) & 15u) == 0 && ((ld * ESZ) & 15) == 0) {
    const int rstep = nthr / VPR, c = (thr % VPR) * 16;
    for (int r = thr / VPR; r < rows; r += rstep)
      *reinterpret_cast<uint4*>(base + (long long)r * ld * ESZ + c) = make_uint4(0u, 0u, 0u, 0u);
  } else {
    for (int r = 0; r < rows; ++r)
      for (int c = thr; c < cols; c += nthr) {
        if (ESZ == 4)
          reinterpret_cast<float*>(base)[(long long)r * ld + c] = 0.f;
        else
          reinterpret_cast<unsigned short*>(base)[(long long)r * ld + c] = 0;
      }
  }
}

// Per-batch dBias: zeros of the (query tile, key tile kt) blocks of query heads
// bh0 .. bh0 + gsz - 1 whose query tile lies outside [qt_lo, qt_hi], i.e. the
// blocks of this key tile that no CTA computes.
__device__ inline void zero_unvisited_dbias_blocks(const ChainParams& p, int b, int bh0, int gsz, int kt,
                                                   int qt_lo, int qt_hi, int thr, int nthr) {
  const int k0 = kt * BN, cols = min(BN, p.Skv - k0);
  for (int hj = 0; hj < gsz; ++hj) {
    const int hq = bh0 + hj - b * p.Hq;
    for (int qt = 0; qt < p.n_qt; ++qt) {
      if (qt >= qt_lo && qt <= qt_hi) continue;
      const int q0 = qt * BQ;
      const long long e0 = (long long)b * p.dbias_bstride + ((long long)hq * p.Sq + q0) * p.Skv + k0;
      if (p.dbias_out)
        zero_elem_rows<2>(reinterpret_cast<char*>(p.dbias) + e0 * 2, min(BQ, p.Sq - q0), cols, p.Skv, thr, nthr);
      else
        zero_elem_rows<4>(reinterpret_cast<char*>(p.dbias) + e0 * 4, min(BQ, p.Sq - q0), cols, p.Skv, thr, nthr);
    }
  }
}

// L2 prefetch of one BQ x BN bias tile (rows q0.., keys k0..) by 128 threads:
// each takes one (bf16) or two (fp32) of its 128-byte lines.
__device__ __forceinline__ void prefetch_bias_tile(const ChainParams& p, long long tile_off, int q0,
                                                   int k0, int thread) {
  const int esz = p.bias_fp32 ? 4 : 2;
  const int lines_per_row = BN * esz / 128;
  for (int line = thread; line < BQ * lines_per_row; line += 128) {
    const int r = line / lines_per_row, key = (line % lines_per_row) * (128 / esz);
    if (q0 + r < p.Sq && k0 + key < p.Skv) {
      const char* a = static_cast<const char*>(p.bias) +
                      (tile_off + (long long)r * p.Skv + key) * esz;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
}

}  // namespace sdpa
