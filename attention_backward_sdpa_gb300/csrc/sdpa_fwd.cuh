// sdpa_fwd.cuh -- what the three forward kernels share: the work-item decode of
// the persistent schedule, the bias row loader, a named barrier that also ORs a
// predicate, the constants of the schedule, and the launchers of the other two
// forward kernels, which launch_fwd (sdpa_fwd.cu) calls by head dims.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa {

namespace fwd_shared {
constexpr int BM = 128;  // query rows per item
constexpr int BK = 128;  // keys per tile
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;
constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units: P stays below 2^8 until a raise
constexpr int FWD_SLOTS = 64;             // launch slots of the persistent tickets
}  // namespace fwd_shared

// One 32-byte streaming load (the address 32-byte aligned) into r[at .. at + 7].
__device__ __forceinline__ void ld_global_cs_32b(const void* ptr, uint32_t (&r)[64], int at) {
  asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[at]), "=r"(r[at + 1]), "=r"(r[at + 2]), "=r"(r[at + 3]), "=r"(r[at + 4]),
                 "=r"(r[at + 5]), "=r"(r[at + 6]), "=r"(r[at + 7])
               : "l"(ptr));
}

// This row's bias for keys kb .. kb + 63 as 32-bit words: on the 16-byte path
// 16-bit pairs (`packed`, 32 words) or fp32 values (64 words); otherwise fp32
// values from scalar loads, 0 past S_kv.
__device__ __forceinline__ void load_fwd_bias_row(const FwdParams& p, long long row_off, int kb, bool live,
                                                  uint32_t (&raw)[64], bool& packed) {
  const bool vec = p.bias_vec && kb + 64 <= p.Skv;  // uniform across the warp
  packed = vec && !p.bias_fp32;
  if (!live) {
#pragma unroll
    for (int i = 0; i < 64; ++i) raw[i] = 0u;
    return;
  }
  const int esz = p.bias_fp32 ? 4 : 2;
  // 32-byte loads (a thread reads whole 32-byte sectors of its row) when every
  // row segment is 32-byte aligned: the base, and rows whose byte length is a
  // multiple of 32 (kb is a multiple of 64 keys). Uniform across the launch.
  const bool v32 = vec && (reinterpret_cast<uintptr_t>(p.bias) & 31u) == 0 && ((long long)p.Skv * esz) % 32 == 0;
  if (v32) {
    const char* src = static_cast<const char*>(p.bias) + (row_off + kb) * esz;
    if (p.bias_fp32) {
#pragma unroll
      for (int v = 0; v < 8; ++v) ld_global_cs_32b(src + 32 * v, raw, 8 * v);
    } else {
#pragma unroll
      for (int v = 0; v < 4; ++v) ld_global_cs_32b(src + 32 * v, raw, 8 * v);
#pragma unroll
      for (int i = 32; i < 64; ++i) raw[i] = 0u;
    }
  } else if (vec) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(p.bias) + (row_off + kb) * esz);
    if (p.bias_fp32) {
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        const uint4 x = __ldcs(src + v);
        raw[4 * v] = x.x; raw[4 * v + 1] = x.y; raw[4 * v + 2] = x.z; raw[4 * v + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint4 x = __ldcs(src + v);
        raw[4 * v] = x.x; raw[4 * v + 1] = x.y; raw[4 * v + 2] = x.z; raw[4 * v + 3] = x.w;
      }
#pragma unroll
      for (int i = 32; i < 64; ++i) raw[i] = 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      float x = 0.f;
      if (kb + i < p.Skv)
        x = p.bias_fp32 ? __ldcs(static_cast<const float*>(p.bias) + row_off + kb + i)
                        : bias16_to_f32(__ldcs(static_cast<const unsigned short*>(p.bias) + row_off + kb + i),
                                        p.bias_f16 != 0);
      raw[i] = __float_as_uint(x);
    }
  }
}

// A thread's 64 scores of a tile rewritten as x = s * c + bias * log2e, the bias
// widened from 16-bit pairs (`packed`; fp16 when p.bias_f16, else bf16) or taken
// as fp32 words. One loop per element form (the choice is uniform across the
// warp), so that widening an element is a fixed instruction or two: a
// per-element choice between the bf16 and the fp16 widening cost the biased
// forward about a third of its speed.
__device__ __forceinline__ void add_bias_row(const FwdParams& p, float c, const uint32_t (&braw)[64], bool packed,
                                             uint32_t (&sr)[2][32]) {
  constexpr float LOG2E_F = 1.4426950408889634f;
  if (packed && p.bias_f16) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const uint32_t wd = braw[i >> 1];
      const float bv = __half2float(__ushort_as_half((unsigned short)((i & 1) ? (wd >> 16) : (wd & 0xFFFFu))));
      sr[i >> 5][i & 31] = __float_as_uint(fmaf(__uint_as_float(sr[i >> 5][i & 31]), c, bv * LOG2E_F));
    }
  } else if (packed) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const uint32_t wd = braw[i >> 1];
      const float bv = __uint_as_float((i & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
      sr[i >> 5][i & 31] = __float_as_uint(fmaf(__uint_as_float(sr[i >> 5][i & 31]), c, bv * LOG2E_F));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      sr[i >> 5][i & 31] =
          __float_as_uint(fmaf(__uint_as_float(sr[i >> 5][i & 31]), c, __uint_as_float(braw[i]) * LOG2E_F));
  }
}

// One work item: 128 query rows (query tile qt, descending so that under a
// causal mask the longest items come first) of one (batch, query head), and the
// range [kt_lo, kt_lo + n) of 128-key tiles that any of its live rows sees.
struct FwdItem {
  int qt, bh, h, kvh, q0, Lq, Lk, kt_lo, n;
  long long diag;
};

__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int it) {
  FwdItem w;
  const int BH = p.B * p.Hq;
  w.qt = p.n_qt - 1 - it / BH;
  w.bh = it % BH;
  const int b = w.bh / p.Hq;
  w.h = w.bh % p.Hq;
  w.kvh = b * p.Hkv + w.h / p.G;
  w.q0 = w.qt * fwd_shared::BM;
  w.Lq = p.Sq;
  w.Lk = p.Skv;
  if (p.seq_q_lens) w.Lq = min(max(p.seq_q_lens[b], 0), p.Sq);
  if (p.seq_kv_lens) w.Lk = min(max(p.seq_kv_lens[b], 0), p.Skv);
  w.diag = p.bottom_right ? (long long)w.Lk - w.Lq : 0;
  const long long Rp = p.window_right > 0 ? p.window_right : 0;
  int kt_lo = 0, kt_hi = -1;
  const long long q_last = min(w.q0 + fwd_shared::BM, w.Lq) - 1;
  if (w.q0 < w.Lq && w.Lk > 0) {
    long long k_hi = w.Lk - 1, k_lo = 0;
    if (p.causal) k_hi = min(k_hi, q_last + w.diag + Rp);
    if (p.window_left >= 0) k_lo = max(0ll, (long long)w.q0 + w.diag - p.window_left);
    if (k_lo <= k_hi) {
      kt_lo = (int)(k_lo / fwd_shared::BK);
      kt_hi = (int)(k_hi / fwd_shared::BK);
    }
  }
  w.kt_lo = kt_lo;
  w.n = kt_hi - kt_lo + 1;  // may be 0
  return w;
}

// One 32-byte global store of two 16-byte halves (the address 32-byte aligned):
// a thread writes a whole 32-byte sector of its O row at once.
__device__ __forceinline__ void st_global_32b(void* ptr, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a.x), "r"(a.y),
               "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// Named barrier over nthreads threads that also ORs a predicate over them.
__device__ __forceinline__ bool named_bar_sync_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}


// The other forward kernels, each a persistent grid of `sms` CTAs taking items
// from ticket slot `slot`: the shared-O kernel for the MLA pair (D_qk = 192,
// D_v = 128; sdpa_fwd_shared.cu) and the head-dim-256 kernel (sdpa_fwd_wide.cu).
cudaError_t launch_fwd_shared(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms, int slot);
cudaError_t fwd_shared_setup();
cudaError_t launch_fwd_wide(const FwdMaps& maps, const FwdParams& p, cudaStream_t s, int sms, int slot);
cudaError_t fwd_wide_setup();

}  // namespace sdpa
