// common.cuh -- parameters and workspace geometry shared by the SDPA backward
// kernels and their host launcher.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <utility>

namespace sdpa {

// Tile sizes of the KV-stationary main kernel: one CTA owns BN keys of one
// query head and walks the query tiles of BQ rows.
constexpr int BN = 128;
constexpr int BQ = 64;

// Row statistics staged per query tile: BQ values of LSE * log2(e) (+inf for
// masked or empty rows) followed by BQ values of delta.
constexpr int QSTAT_FLOATS = 2 * BQ;

// Device status bits (OR-ed into the per-device status word).
constexpr int STATUS_TIMEOUT = 1;
constexpr int STATUS_SMEM_ALIGN = 2;
constexpr int STATUS_BOUNDS = 4;  // debug-bounds build: an access outside its region was skipped

struct ChainParams {
  int B, Hq, Hkv, Sq, Skv, Dqk, Dv;
  int G;            // Hq / Hkv
  // Main-kernel work units of the D_qk 64/128 kernels cover gsz query heads of
  // one KV group (their dK/dV summed in tensor memory); n_part = G / gsz
  // partial dK/dV sets per KV head then remain for the group reduction (none
  // when n_part == 1). The D_qk 192 kernel always has gsz = 1.
  int gsz, n_part;
  int n_qt, n_kt;   // ceil(Sq / BQ), ceil(Skv / BN)
  float scale;      // softmax scale
  float scale_log2; // scale * log2(e)
  int causal, bottom_right, window_left, window_right, deterministic;
  int f16;          // io tensors are fp16 (the __nv_bfloat16 pointers below then hold fp16)
  const int32_t* seq_q_lens;   // (B,) or null
  const int32_t* seq_kv_lens;  // (B,) or null

  // inputs
  const __nv_bfloat16* o;
  const __nv_bfloat16* d_o;
  const float* lse;
  // outputs
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;

  // workspace regions
  float* qstat;         // [B*Hq][n_qt][QSTAT_FLOATS]
  float* dq_accum;      // [B*Hq][n_qt*BQ][dq_acc_cols] row-major, rows padded to whole tiles
  int dq_acc_cols;      // 64 or 128: the column count of the main kernel that runs (D_qk <= it)
  int* counters;        // [B*Hq][n_qt] turn counters (deterministic mode)
  int* ticket;          // work-unit ticket
  __nv_bfloat16* dk_ws; // n_part > 1: [B][Hkv][n_part][Skv][Dqk] partials, else null
  __nv_bfloat16* dv_ws; // n_part > 1: [B][Hkv][n_part][Skv][Dv]
  int n_counters;       // B*Hq*n_qt + 1 (counters plus ticket)

  // Sink tokens (optional): the forward's LSE already folds the sink logits in,
  // so dQ/dK/dV need nothing; dsink[h] = -sum_{b,q} exp(sink[h] - LSE) * delta.
  const float* sink;    // (Hq,) sink logits, or null
  float* dsink;         // (Hq,) output, or null
  float* dsink_part;    // [B*Hq][n_qt] per-tile partial sums (fixed order within a tile)

  // Additive bias (optional), added to the scaled scores before the softmax:
  // element (b, h, q, k) at bias[b * bias_bstride + (h * Sq + q) * Skv + k],
  // bf16 or fp32; bias_bstride = 0 when one bias batch serves every batch row.
  // dbias (fp32, same indexing with dbias_bstride) receives dS = P * (dP - delta);
  // with dbias_red the batch rows' terms are added atomically into one batch.
  const void* bias;     // or null
  int bias_fp32;
  int bias_f16;         // 16-bit bias elements are fp16 (else bf16)
  long long bias_bstride;
  float* dbias;         // or null (holds bf16 / fp16 elements when dbias_out is 1 / 2)
  long long dbias_bstride;
  int dbias_red;
  int dbias_out;        // element type written: 0 fp32, 1 bf16, 2 fp16 (0 whenever dbias_red)

  // Two-kernel route: the main kernel stores each bf16 dS^T tile (its swizzled
  // shared-memory image, DS_TILE_BYTES) at ds_tile(p, bh, ...) below, and the
  // dQ kernel reads them back in ascending key-tile order. zero_tile is
  // DS_TILE_BYTES of zeros standing in for tiles the main kernel never visits.
  // The tiles of one (batch, query head) are stored key tile by key tile, each
  // key tile's band of query tiles contiguous (ds_tile below): with ds_band the
  // band is the query tiles the key tile visits at the full lengths, which
  // contains every range it visits under shorter lengths when the mask is
  // top-left aligned or no length array is given; otherwise (a bottom-right mask
  // with per-batch lengths moves the diagonal) the band is every query tile.
  // ds_band_tiles is the band size summed over the key tiles.
  int ds_route;
  int ds_band;
  long long ds_band_tiles;
  uint8_t* ds_ws;
  uint8_t* zero_tile;

  int* status;          // per-device status word
  // Ordered relay (deterministic mode, D_qk up to 128 but not 128): how long a
  // key tile waits for its turn before it gives up and reports a timeout, and a
  // skew added to every expected turn (0; a nonzero skew makes the first key
  // tile of each query tile wait for a turn that no tile releases, which is how
  // the bounded wait is tested).
  unsigned long long relay_wait_ns;
  int relay_turn_skew;
};

constexpr int DS_TILE_BYTES = BN * BQ * 2;  // one dS^T tile: 128 keys x 64 queries, bf16

// Query tiles [qt_lo, qt_hi] (of BQ rows) that key tile kt visits for batch row
// b: loop bounds of "Causal, sliding-window, and padding masks". Empty when
// qt_lo > qt_hi. Shared by the main kernel and the dQ kernel so that both walk
// exactly the same (key tile, query tile) pairs.
__host__ __device__ inline void visited_query_tiles(int kt, int Lq, int Lk, int causal,
                                                    int bottom_right, int window_left,
                                                    int window_right, int& qt_lo, int& qt_hi) {
  qt_lo = 0;
  qt_hi = -1;
  const int k0 = kt * BN;
  if (k0 >= Lk || Lq <= 0) return;
  const long long diag = bottom_right ? (long long)Lk - Lq : 0;
  const long long Rp = window_right > 0 ? window_right : 0;
  const long long k_last = (k0 + BN - 1 < Lk - 1) ? k0 + BN - 1 : Lk - 1;
  long long q_min = 0, q_max = Lq - 1;
  if (causal) q_min = (k0 - diag - Rp > 0) ? k0 - diag - Rp : 0;
  if (window_left >= 0 && k_last - diag + window_left < q_max) q_max = k_last - diag + window_left;
  if (q_min > q_max) return;
  qt_lo = (int)(q_min / BQ);
  qt_hi = (int)(q_max / BQ);
}

// Debug-bounds build (compiled with -DSDPA_DEBUG_BOUNDS): the kernels check
// every raw-pointer global access (bulk copies, reductions, counters, direct
// stores) against the region it belongs to; an access outside it sets
// STATUS_BOUNDS in the status word and is skipped, with no trap. In the normal
// build the check is the constant true and compiles away.
__device__ __forceinline__ bool in_bounds(int* status, const void* ptr, size_t bytes, const void* base,
                                          size_t extent) {
#ifdef SDPA_DEBUG_BOUNDS
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr), b0 = reinterpret_cast<uintptr_t>(base);
  if (base == nullptr || a < b0 || a + bytes > b0 + extent) {
    atomicOr(status, STATUS_BOUNDS);
    return false;
  }
#else
  (void)status; (void)ptr; (void)bytes; (void)base; (void)extent;
#endif
  return true;
}

// Region sizes in bytes, from the parameters (for the debug-bounds checks).
__host__ __device__ inline size_t qstat_bytes(const ChainParams& p) {
  return (size_t)p.B * p.Hq * p.n_qt * QSTAT_FLOATS * sizeof(float);
}
__host__ __device__ inline size_t dq_accum_bytes(const ChainParams& p) {
  return (size_t)p.B * p.Hq * p.n_qt * BQ * p.dq_acc_cols * sizeof(float);
}
__host__ __device__ inline size_t io_q_bytes(const ChainParams& p, int D) {  // (B, H_q, S_q, D) io tensor
  return (size_t)p.B * p.Hq * p.Sq * D * 2;
}
__host__ __device__ inline size_t kv_out_bytes(const ChainParams& p, int D, bool partials) {  // dK / dV (or partial sets)
  return (size_t)p.B * (partials ? p.Hq : p.Hkv) * p.Skv * D * 2;
}

// Band of query tiles [lo, hi] of key tile kt in the dS workspace (see ChainParams).
__host__ __device__ inline void ds_band_range(const ChainParams& p, int kt, int& lo, int& hi) {
  if (!p.ds_band) {
    lo = 0;
    hi = p.n_qt - 1;
    return;
  }
  visited_query_tiles(kt, p.Sq, p.Skv, p.causal, p.bottom_right, p.window_left, p.window_right, lo, hi);
}

// Index (in tiles, within one (batch, query head)) of the first tile of key
// tile kt's band: the band sizes of key tiles 0 .. kt-1 summed.
__host__ __device__ inline long long ds_band_prefix(const ChainParams& p, int kt) {
  long long s = 0;
  for (int k = 0; k < kt; ++k) {
    int lo, hi;
    ds_band_range(p, k, lo, hi);
    if (hi >= lo) s += hi - lo + 1;
  }
  return s;
}

__host__ __device__ inline size_t ds_ws_bytes(const ChainParams& p) {
  return (size_t)p.B * p.Hq * p.ds_band_tiles * DS_TILE_BYTES;
}

// Address of the stored dS^T tile (bh, kt, qt); `prefix` = ds_band_prefix(p, kt)
// and `band_lo` the first query tile of kt's band (callers compute both once per key
// tile). qt must lie in the band.
__host__ __device__ inline uint8_t* ds_tile(const ChainParams& p, int bh, long long prefix, int band_lo,
                                            int qt) {
  return p.ds_ws + ((long long)bh * p.ds_band_tiles + prefix + (qt - band_lo)) * (long long)DS_TILE_BYTES;
}

// Forward pass (sdpa_fwd.cu): O and the natural-log LSE of the masked softmax.
struct FwdParams {
  int B, Hq, Hkv, Sq, Skv, Dqk, Dv;
  int G;            // Hq / Hkv
  int n_qt;         // ceil(Sq / 128): 128-row query tiles
  float scale_log2; // scale * log2(e)
  int f16;          // io tensors are fp16
  int causal, bottom_right, window_left, window_right;
  const int32_t* seq_q_lens;  // (B,) or null
  const int32_t* seq_kv_lens; // (B,) or null
  const float* sink;          // (Hq,) sink logits, or null
  // Additive bias (optional), as in ChainParams: element (b, h, q, k) at
  // bias[b * bias_bstride + (h * Sq + q) * Skv + k], bf16 or fp32.
  const void* bias;
  int bias_fp32;
  int bias_f16;               // 16-bit bias elements are fp16 (else bf16)
  long long bias_bstride;
  int bias_vec;               // rows allow 16-byte loads (S_kv * size % 16 == 0, base aligned)
  float* lse;                 // (B, Hq, Sq) output
  void* o;                    // (B, Hq, Sq, Dv) output (io type), also behind FwdMaps::o
  int* status;                // device status word
};
struct FwdMaps {
  CUtensorMap q, k, v, o;  // 128-row boxes
};
cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, cudaStream_t s);
cudaError_t fwd_kernel_setup();

// TMA tensor maps of the main kernels: inputs K and V with H_kv heads, Q and dO
// with H_q; outputs dK and dV (H_kv heads, or the per-query-head partials of
// the GQA workspace), written in 128-row boxes.
struct MainMaps {
  CUtensorMap q, k, v, d_o, dk_out, dv_out;
};

// Host launchers, one per kernel, defined beside their kernels. `pdl` launches
// with programmatic stream serialization (the kernel waits on its predecessor
// with griddepcontrol.wait before touching dependent data).
cudaError_t launch_preprocess(const ChainParams& p, cudaStream_t s, int num_sms);
cudaError_t preprocess_kernel_setup();  // per device: opt in to the preprocess's shared memory
cudaError_t launch_main(const MainMaps& maps, const ChainParams& p, cudaStream_t s);
cudaError_t launch_dq_convert(const ChainParams& p, cudaStream_t s);
cudaError_t launch_dsink(const ChainParams& p, cudaStream_t s);
// fp32 -> 16-bit (bf16, or fp16 when f16) copy of n elements: the io-type dBias
// of a shared bias, whose batch rows add into an fp32 buffer first.
cudaError_t launch_dbias_cast(const float* src, void* dst, long long n, bool f16, int num_sms,
                              cudaStream_t s);
cudaError_t launch_dq_from_ds(const CUtensorMap& k_map, const ChainParams& p, cudaStream_t s,
                              int num_sms);
cudaError_t dq_kernel_setup();  // per device: opt in to the dQ kernel's shared memory
cudaError_t launch_main_ds(const MainMaps& maps, const ChainParams& p, cudaStream_t s);
cudaError_t main_ds_kernel_setup();
cudaError_t main_kernel_setup();  // per device: opt in to the main kernel's shared memory
cudaError_t launch_main_bias(const MainMaps& maps, const ChainParams& p, cudaStream_t s);
cudaError_t launch_main_f16(const MainMaps& maps, const ChainParams& p, cudaStream_t s);
cudaError_t main_f16_kernel_setup();
cudaError_t main_bias_kernel_setup();
cudaError_t launch_main_qat(const MainMaps& maps, const ChainParams& p, cudaStream_t s);
cudaError_t main_qat_kernel_setup();
// NVFP4 fake quantization of n_blocks blocks of 16 consecutive bf16 values.
cudaError_t launch_nvfp4_fake_quant(const void* x, void* y, long long n_blocks, int num_sms,
                                    cudaStream_t s);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// floor(a / b) for b > 0 and any sign of a.
__host__ __device__ inline long long floor_div(long long a, long long b) {
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// A 16-bit bias element (bf16, or fp16 when f16) widened to fp32.
__device__ __forceinline__ float bias16_to_f32(unsigned short v, bool f16) {
  return f16 ? __half2float(__ushort_as_half(v)) : __uint_as_float((uint32_t)v << 16);
}

// fp32 to a 16-bit dBias element (bf16, or fp16 when f16), round to nearest even.
__device__ __forceinline__ unsigned short f32_to_16(float x, bool f16) {
  return f16 ? __half_as_ushort(__float2half_rn(x)) : __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Valid lengths of batch row b (the full S when no length array is given).
__device__ inline void batch_lengths(const ChainParams& p, int b, int& Lq, int& Lk) {
  Lq = p.seq_q_lens ? min(max(p.seq_q_lens[b], 0), p.Sq) : p.Sq;
  Lk = p.seq_kv_lens ? min(max(p.seq_kv_lens[b], 0), p.Skv) : p.Skv;
}

// Zero rows [k0, min(k0 + BN, S_kv)) of dK and dV (`head` indexes the KV heads,
// or the partial sets of the group reduction when dk_ws is set) for a key tile
// that no query sees: such keys have exactly zero gradient, and the outputs are
// overwritten in full. Called by every thread of a CTA; 16-byte stores,
// consecutive threads on consecutive addresses.
// Key tiles that no query of their batch row sees (padding, windows) only have
// zero gradients. On the non-deterministic launch their CTAs leave at once and
// the head group's other CTAs write those rows with an otherwise idle warp:
// the r-th key tile with a visible query (ascending) takes the tiles with none
// whose index among them is r modulo the number of visible ones. Every batch
// row with at least one query and one key has a visible pair (the diagonal
// q + diag is inside the causal band and the window), so only a row with no
// query or no key leaves its CTAs to zero their own rows.
__device__ inline bool row_has_visible_pair(int Lq, int Lk) { return Lq > 0 && Lk > 0; }

// One warp: zeroes the dK/dV rows of this CTA's share of the empty key tiles of
// its head group (dK/dV destination `head`), classifying tiles with the same
// visited_query_tiles() that every kernel walks.
__device__ inline void zero_group_share_of_empty_key_tiles(const ChainParams& p, long long head, int kt_self,
                                                    int Lq, int Lk, int lane) {
  int rank = 0, n_vis = 0;
  for (int base = 0; base < p.n_kt; base += 32) {
    const int kt = base + lane;
    int lo = 0, hi = -1;
    if (kt < p.n_kt)
      visited_query_tiles(kt, Lq, Lk, p.causal, p.bottom_right, p.window_left, p.window_right, lo, hi);
    const unsigned vis = __ballot_sync(0xffffffffu, kt < p.n_kt && hi >= lo);
    if (kt_self >= base && kt_self < base + 32) rank = n_vis + __popc(vis & ((1u << (kt_self - base)) - 1u));
    n_vis += __popc(vis);
  }
  if (n_vis == 0) return;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  int j = 0;  // index among the empty tiles
  for (int base = 0; base < p.n_kt; base += 32) {
    const int kt = base + lane;
    int lo = 0, hi = -1;
    if (kt < p.n_kt)
      visited_query_tiles(kt, Lq, Lk, p.causal, p.bottom_right, p.window_left, p.window_right, lo, hi);
    unsigned empty = __ballot_sync(0xffffffffu, kt < p.n_kt && hi < lo);
    while (empty != 0u) {
      const int e = base + __ffs(empty) - 1;
      empty &= empty - 1u;
      if (j++ % n_vis != rank) continue;
      const int k0 = e * BN;
      const int rows = min(BN, p.Skv - k0);
      uint4* dk = reinterpret_cast<uint4*>((p.dk_ws ? p.dk_ws : p.dk) + (head * p.Skv + k0) * p.Dqk);
      uint4* dv = reinterpret_cast<uint4*>((p.dv_ws ? p.dv_ws : p.dv) + (head * p.Skv + k0) * p.Dv);
      if (!in_bounds(p.status, dk, (size_t)rows * p.Dqk * 2, p.dk_ws ? p.dk_ws : p.dk,
                     kv_out_bytes(p, p.Dqk, p.dk_ws != nullptr)) ||
          !in_bounds(p.status, dv, (size_t)rows * p.Dv * 2, p.dv_ws ? p.dv_ws : p.dv,
                     kv_out_bytes(p, p.Dv, p.dv_ws != nullptr)))
        continue;
      for (int i = lane; i < rows * (p.Dqk / 8); i += 32) dk[i] = z;
      for (int i = lane; i < rows * (p.Dv / 8); i += 32) dv[i] = z;
    }
  }
}

__device__ inline void zero_key_tile_rows(const ChainParams& p, long long head, int k0) {
  const int rows = min(BN, p.Skv - k0);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  uint4* dk = reinterpret_cast<uint4*>((p.dk_ws ? p.dk_ws : p.dk) + (head * p.Skv + k0) * p.Dqk);
  uint4* dv = reinterpret_cast<uint4*>((p.dv_ws ? p.dv_ws : p.dv) + (head * p.Skv + k0) * p.Dv);
  if (!in_bounds(p.status, dk, (size_t)rows * p.Dqk * 2, p.dk_ws ? p.dk_ws : p.dk,
                 kv_out_bytes(p, p.Dqk, p.dk_ws != nullptr)) ||
      !in_bounds(p.status, dv, (size_t)rows * p.Dv * 2, p.dv_ws ? p.dv_ws : p.dv,
                 kv_out_bytes(p, p.Dv, p.dv_ws != nullptr)))
    return;
  for (int i = threadIdx.x; i < rows * (p.Dqk / 8); i += blockDim.x) dk[i] = z;
  for (int i = threadIdx.x; i < rows * (p.Dv / 8); i += blockDim.x) dv[i] = z;
}

}  // namespace sdpa
