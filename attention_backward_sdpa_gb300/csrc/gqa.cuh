// gqa.cuh -- the fixed-order GQA/MQA group reduction of dK/dV ("GQA/MQA group
// reduction" section of the cuDNN frontend page "SDPA Backward (SM120)"):
// dK[b, kv head, key] = sum over the group's n_part partial sets (each the sum
// of gsz query heads, in ascending head order), in ascending order,
// accumulated in fp32 and rounded once to bf16 (bitwise reproducible by
// construction). Run by the dQ kernels over slices of the output rows,
// overlapping their other work.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

// Eight io elements (bf16, or fp16 when F16) widened to fp32.
template <bool F16 = false>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = io_lo<F16>(w[i]);
    f[2 * i + 1] = io_hi<F16>(w[i]);
  }
}

// Rows [row_begin, row_end) of one output (dK with D = D_qk or dV with D = D_v,
// a multiple of 8), one 8-column chunk per item, items strided over `nthreads`
// threads.
template <bool F16>
__device__ __forceinline__ void gqa_reduce_rows(const ChainParams& p, const __nv_bfloat16* ws,
                                                __nv_bfloat16* out, int D, unsigned row_begin,
                                                unsigned row_end, unsigned thread,
                                                unsigned nthreads) {
  const unsigned CPR = (unsigned)D / 8;  // chunks per row
  const unsigned items = (row_end > row_begin ? row_end - row_begin : 0) * CPR;
  const long long head_stride = (long long)p.Skv * D;
  const int G = p.n_part;
  for (unsigned it = thread; it < items; it += nthreads) {
    const unsigned row = row_begin + it / CPR, c8 = it % CPR;
    const unsigned bhk = row / (unsigned)p.Skv, k = row - bhk * (unsigned)p.Skv;
    const unsigned b = bhk / (unsigned)p.Hkv, hk = bhk - b * (unsigned)p.Hkv;
    const __nv_bfloat16* src =
        ws + (long long)(b * p.Hkv + hk) * G * head_stride + (long long)k * D + c8 * 8;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)  // issue the group's loads together
      if (j < G) v[j] = *reinterpret_cast<const uint4*>(src + j * head_stride);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // ascending partial set: fixed order
      if (j < G) {
        float f[8];
        unpack8<F16>(v[j], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
    }
    for (int j = 8; j < G; ++j) {  // more partial sets: the rest, same order
      float f[8];
      unpack8<F16>(*reinterpret_cast<const uint4*>(src + j * head_stride), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += f[e];
    }
    uint4 o;
    o.x = pack_io2<F16>(acc[0], acc[1]);
    o.y = pack_io2<F16>(acc[2], acc[3]);
    o.z = pack_io2<F16>(acc[4], acc[5]);
    o.w = pack_io2<F16>(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + (long long)row * D + c8 * 8) = o;
  }
}

// Piece `piece` of `n_pieces` of the slice of output rows assigned to CTA
// `cta` of `n_ctas` (both outputs). Pieces let a kernel spread the work.
template <bool F16 = false>
__device__ __forceinline__ void gqa_reduce_slice(const ChainParams& p, unsigned cta, unsigned n_ctas,
                                                 unsigned thread, unsigned nthreads,
                                                 unsigned piece = 0, unsigned n_pieces = 1) {
  if (p.dk_ws == nullptr) return;  // MHA: the main kernel wrote dK/dV directly
  const unsigned rows = (unsigned)p.B * p.Hkv * p.Skv;
  const unsigned per = (rows + n_ctas - 1) / n_ctas;
  const unsigned lo = cta * per, hi = (lo + per < rows) ? lo + per : rows;
  if (lo >= hi || piece >= n_pieces) return;
  const unsigned pp = (hi - lo + n_pieces - 1) / n_pieces;
  const unsigned plo = lo + piece * pp, phi = (plo + pp < hi) ? plo + pp : hi;
  if (plo >= phi) return;
  gqa_reduce_rows<F16>(p, p.dk_ws, p.dk, p.Dqk, plo, phi, thread, nthreads);
  gqa_reduce_rows<F16>(p, p.dv_ws, p.dv, p.Dv, plo, phi, thread, nthreads);
}

}  // namespace sdpa
