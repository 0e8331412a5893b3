// sdpa_bwd_api.cu -- host side of libsdpa_bwd.so: the C ABI declared in
// include/sdpa_bwd.h.
//
// One call validates its arguments, carves the workspace, encodes the six TMA
// tensor maps and enqueues the kernel chain on the caller's stream
// (cuDNN frontend docs, "SDPA Backward (SM120)", section "The kernel chain"):
//   preprocess -> main -> dq (convert, or dS x K on the two-kernel route)
// with the GQA group reduction of dK/dV folded into the dq kernel.
// Every launch after the first uses programmatic dependent launch, so each
// kernel's prologue overlaps its predecessor's tail; each kernel waits for its
// predecessor's completion (griddepcontrol.wait) before touching its outputs.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sdpa_bwd.h"
#include "common.cuh"
#include "tmap.h"

namespace sdpa {

// Per-device status word written by kernels that give up on a bounded wait.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
bool g_device_checked[kMaxDevices] = {};
bool g_device_ok[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Profiling state.
bool g_profile = false;

// Ordered-relay wait limit and turn skew (sdpa_bwd_debug_relay).
constexpr unsigned long long kRelayWaitDefaultNs = 4000000000ull;
unsigned long long g_relay_wait_ns = kRelayWaitDefaultNs;
int g_relay_turn_skew = 0;
float g_prof_ms[3] = {};
int g_prof_n[3] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Routes of the chain:
//   kTwoKernel main kernel with dS stored, then the Q-stationary dQ kernel:
//              the deterministic route for D_qk = 128 as on the pages (the
//              relay serves every other D_qk up to 128), and the only route
//              for D_qk = 192 and 256, whose dK accumulators leave no tensor
//              memory for dQ in the main kernel.
//   kReduce    main kernel with the fp32 dQ accumulator (the ordered relay
//              when deterministic), then the convert.
enum class Route { kReduce, kTwoKernel };

Route choose_route(int deterministic, int Dqk) {
  return (Dqk > 128 || (deterministic && Dqk == 128)) ? Route::kTwoKernel : Route::kReduce;
}

// The problem shape and mask as far as they size the workspace.
struct Shape {
  int B, Hq, Hkv, Sq, Skv, Dqk, Dv;
  int causal, bottom_right, window_left, window_right;
  int padded;  // per-batch length arrays are given
};

// Band mode of the dS workspace (ChainParams::ds_band) and the band size per
// (batch, query head) in tiles.
void ds_band_geometry(const Shape& sh, int& band, long long& tiles) {
  ChainParams p{};
  p.Sq = sh.Sq;
  p.Skv = sh.Skv;
  p.n_qt = ceil_div(sh.Sq, BQ);
  p.n_kt = ceil_div(sh.Skv, BN);
  p.causal = sh.causal ? 1 : 0;
  p.bottom_right = sh.bottom_right ? 1 : 0;
  p.window_left = sh.window_left < 0 ? -1 : sh.window_left;
  p.window_right = (sh.causal && sh.window_right > 0) ? sh.window_right : -1;
  p.ds_band = (sh.bottom_right && sh.padded) ? 0 : 1;
  band = p.ds_band;
  tiles = ds_band_prefix(p, p.n_kt);
}

struct Carve {
  size_t qstat, dq_accum, ds_ws, zero_tile, counters, dk_ws, dv_ws, dsink_part;
  size_t q_hat, k_hat, v_hat;  // NVFP4 QAT: the fake-quantized Q, K, V
  int ds_band;
  long long ds_band_tiles;
  size_t total;
};

Carve carve(const Shape& sh, Route route, bool qat = false) {
  const int B = sh.B, Hq = sh.Hq, Hkv = sh.Hkv, Sq = sh.Sq, Skv = sh.Skv, Dqk = sh.Dqk, Dv = sh.Dv;
  const size_t n_qt = (size_t)ceil_div(Sq, BQ);
  const size_t bh = (size_t)B * Hq;
  Carve c{};
  size_t off = 0;
  c.qstat = off;
  off = align256(off + bh * n_qt * QSTAT_FLOATS * sizeof(float));
  if (route != Route::kReduce) {
    ds_band_geometry(sh, c.ds_band, c.ds_band_tiles);
    c.dq_accum = SIZE_MAX;
    c.ds_ws = off;
    off = align256(off + bh * (size_t)c.ds_band_tiles * (size_t)DS_TILE_BYTES);
    c.zero_tile = off;
    off = align256(off + DS_TILE_BYTES);
  } else {
    c.ds_ws = c.zero_tile = SIZE_MAX;
    c.dq_accum = off;  // rows of 64 or 128 columns: the width of the main kernel that runs
    off = align256(off + bh * n_qt * BQ * (size_t)(Dqk <= 64 ? 64 : 128) * sizeof(float));
  }
  c.counters = off;  // turn counters, then the work ticket
  off = align256(off + (bh * n_qt + 1) * sizeof(int));
  c.dsink_part = off;  // sink-token partials (one float per 64-row tile); used only by sdpa_bwd_sink
  off = align256(off + bh * n_qt * sizeof(float));
  if (Hkv < Hq) {
    c.dk_ws = off;
    off = align256(off + bh * (size_t)Skv * Dqk * 2);
    c.dv_ws = off;
    off = align256(off + bh * (size_t)Skv * Dv * 2);
  } else {
    c.dk_ws = c.dv_ws = SIZE_MAX;
  }
  c.q_hat = c.k_hat = c.v_hat = SIZE_MAX;
  if (qat) {
    c.q_hat = off;
    off = align256(off + bh * (size_t)Sq * Dqk * 2);
    c.k_hat = off;
    off = align256(off + (size_t)B * Hkv * Skv * Dqk * 2);
    c.v_hat = off;
    off = align256(off + (size_t)B * Hkv * Skv * Dv * 2);
  }
  c.total = off;
  return c;
}

bool dims_supported(int Dqk, int Dv) {
  // D_qk = D_v, a multiple of 8 up to 128: the 64- or 128-column kernels, the
  // columns past D zero-filled by TMA; the MLA pair 192/128; and 256/256 (the
  // backward only: units that accumulate half of the dK/dV columns each).
  return (Dqk == Dv && Dqk % 8 == 0 && Dqk >= 8 && Dqk <= 128) || (Dqk == 192 && Dv == 128) ||
         (Dqk == 256 && Dv == 256);
}

int basic_checks(int B, int Hq, int Hkv, int Sq, int Skv, int Dqk, int Dv) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || Dqk <= 0 || Dv <= 0)
    return SDPA_ERR_INVALID;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID;
  if (!dims_supported(Dqk, Dv)) return SDPA_ERR_UNSUPPORTED;
  // TMA coordinates, the flattened (batch, head) axis and the element index of
  // every tensor are 32-bit.
  const long long limit = 1ll << 31;
  if ((long long)B * Hq * Sq * (Dqk > Dv ? Dqk : Dv) >= limit ||
      (long long)B * Hkv * Skv * (Dqk > Dv ? Dqk : Dv) >= limit ||
      (long long)B * Hq * ceil_div(Skv, BN) >= limit)
    return SDPA_ERR_INVALID;
  return SDPA_OK;
}

// Sets up per-device state once: device capability check and the status word.
int device_state(int dev, int** status_out, int* sms_out) {
  if (dev < 0 || dev >= kMaxDevices) return SDPA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_device_checked[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SDPA_ERR_CUDA;
    g_device_ok[dev] = (prop.major == 10 && prop.minor == 3);
    g_num_sms[dev] = prop.multiProcessorCount;
    if (g_device_ok[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return SDPA_ERR_CUDA;
      g_status_ptr[dev] = static_cast<int*>(p);
      if (main_kernel_setup() != cudaSuccess || main_ds_kernel_setup() != cudaSuccess ||
          preprocess_kernel_setup() != cudaSuccess ||
          dq_kernel_setup() != cudaSuccess || fwd_kernel_setup() != cudaSuccess)
        return SDPA_ERR_CUDA;
    }
    g_device_checked[dev] = true;
  }
  if (!g_device_ok[dev]) return SDPA_ERR_UNSUPPORTED;
  *status_out = g_status_ptr[dev];
  *sms_out = g_num_sms[dev];
  return SDPA_OK;
}

// 3-D map {D, S, B*H} of a contiguous (B, H, S, D) bf16 tensor; boxes of 64
// columns (128 bytes, the swizzle span) by `rows` sequence positions.
bool make_bhsd_map(CUtensorMap* m, const void* base, int D, int S, long long BH, int rows,
                   bool f16 = false) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)S, (uint64_t)BH};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)S * D * 2};
  const uint32_t box[3] = {64, (uint32_t)rows, 1};
  return make_tmap(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                   dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// NVTX range names of the chain's launches (seen by profilers and tracers;
// a no-op without one attached).
const char* const kRangeNames[3] = {"sdpa_bwd.preprocess", "sdpa_bwd.main", "sdpa_bwd.dq"};

// Opens an NVTX range around each launch and, while profiling is on, records
// one event pair per launch; the pairs are resolved once at the end of the
// call, so no synchronization sits between launches (a busy stream keeps host
// launch latency out of the intervals).
struct ProfEvents {
  cudaEvent_t ev[3][2] = {};
  bool used[3] = {};
  cudaStream_t s;
  explicit ProfEvents(cudaStream_t s_) : s(s_) {}
  void begin(int slot) {
    nvtxRangePushA(kRangeNames[slot]);
    if (!g_profile) return;
    cudaEventCreate(&ev[slot][0]);
    cudaEventCreate(&ev[slot][1]);
    cudaEventRecord(ev[slot][0], s);
    used[slot] = true;
  }
  void end(int slot) {
    if (g_profile && used[slot]) cudaEventRecord(ev[slot][1], s);
    nvtxRangePop();
  }
  ~ProfEvents() {
    for (int i = 0; i < 3; ++i) {
      if (!used[i]) continue;
      cudaEventSynchronize(ev[i][1]);
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ev[i][0], ev[i][1]) == cudaSuccess) {
        std::lock_guard<std::mutex> lock(g_mu);
        g_prof_ms[i] += ms;
        g_prof_n[i] += 1;
      }
      cudaEventDestroy(ev[i][0]);
      cudaEventDestroy(ev[i][1]);
    }
  }
};

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" {

int sdpa_bwd_version(void) { return 200; }

const char* sdpa_status_string(int status) {
  switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case SDPA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case SDPA_ERR_WORKSPACE: return "workspace too small";
    case SDPA_ERR_CUDA: return "CUDA runtime error";
    case SDPA_ERR_TIMEOUT: return "device-side wait timed out";
    case SDPA_ERR_BOUNDS: return "debug-bounds build: an out-of-range access was skipped";
    default: return "unknown status";
  }
}

size_t sdpa_bwd_workspace_size(int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v,
                               int causal, int bottom_right, int window_left, int window_right,
                               int deterministic, int padded) {
  if (basic_checks(B, H_q, H_kv, S_q, S_kv, D_qk, D_v) != SDPA_OK) return 0;
  if (S_q == 0 || S_kv == 0) return 0;
  const Shape sh{B, H_q, H_kv, S_q, S_kv, D_qk, D_v, causal, bottom_right, window_left, window_right,
                 padded};
  return carve(sh, choose_route(deterministic, D_qk)).total;
}

size_t sdpa_bwd_nvfp4_qat_workspace_size(int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk,
                                         int D_v) {
  if (basic_checks(B, H_q, H_kv, S_q, S_kv, D_qk, D_v) != SDPA_OK) return 0;
  if (D_qk != 128 || D_v != 128 || S_q == 0 || S_kv == 0) return 0;
  const Shape sh{B, H_q, H_kv, S_q, S_kv, D_qk, D_v, 0, 0, -1, -1, 0};
  return carve(sh, Route::kReduce, true).total;
}

int sdpa_bwd_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = on != 0;
  for (int i = 0; i < 3; ++i) {
    g_prof_ms[i] = 0.f;
    g_prof_n[i] = 0;
  }
  return SDPA_OK;
}

int sdpa_bwd_profile_read(float* ms, int* launches, int n) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < n && i < 3; ++i) {
    if (ms) ms[i] = g_prof_ms[i];
    if (launches) launches[i] = g_prof_n[i];
  }
  return 3;
}

int sdpa_bwd_debug_relay(unsigned long long wait_limit_ns, int turn_skew) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_relay_wait_ns = wait_limit_ns == 0 ? kRelayWaitDefaultNs : wait_limit_ns;
  g_relay_turn_skew = turn_skew;
  return SDPA_OK;
}

int sdpa_bwd_check_device_status(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  int* status = nullptr;
  int sms = 0;
  int rc = device_state(dev, &status, &sms);
  if (rc != SDPA_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SDPA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDPA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return (v & STATUS_BOUNDS) ? SDPA_ERR_BOUNDS : SDPA_ERR_TIMEOUT;
  }
  return SDPA_OK;
}

}  // extern "C"

namespace {

// Optional additive bias of sdpa_bwd_bias(); all null/zero for the other calls.
struct BiasArgs {
  const void* bias = nullptr;
  int dtype = SDPA_DTYPE_BF16;
  int batch = 0;  // 1 or B
  void* dbias = nullptr;
  int dbias_dtype = SDPA_DTYPE_F32;
};

// The whole chain; sink/dsink are null for sdpa_bwd().
int run_chain(const void* q, const void* k, const void* v, const void* o, const void* d_o,
              const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int S_q,
              int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
              int window_left, int window_right, int deterministic, const int32_t* seq_q_lens,
              const int32_t* seq_kv_lens, void* workspace, size_t workspace_bytes,
              const float* sink, float* dsink, const BiasArgs& ba, void* stream_,
              bool qat = false, bool f16 = false) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int rc = basic_checks(B, H_q, H_kv, S_q, S_kv, D_qk, D_v);
  if (rc != SDPA_OK) return rc;
  // The QAT path is bf16 (the page's QAT kernels take BF16 activations only).
  if (f16 && qat) return SDPA_ERR_UNSUPPORTED;
  // NVFP4 QAT: D 128, the dQ-reduction route, no bias or sink.
  if (qat && (D_qk != 128 || D_v != 128)) return SDPA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !d_o || !lse || !dq || !dk || !dv) return SDPA_ERR_INVALID;
  if (dsink && !sink) return SDPA_ERR_INVALID;
  if (ba.bias) {
    if (ba.dtype != SDPA_DTYPE_BF16 && ba.dtype != SDPA_DTYPE_F32 && ba.dtype != SDPA_DTYPE_F16)
      return SDPA_ERR_INVALID;
    if (ba.batch != 1 && ba.batch != B) return SDPA_ERR_INVALID;
    // A one-batch dBias summed over B > 1 batch rows is added atomically: not
    // reproducible, so deterministic mode rejects it.
    if (deterministic && ba.dbias && ba.batch == 1 && B > 1) return SDPA_ERR_INVALID;
    if (ba.dbias_dtype != SDPA_DTYPE_F32 && ba.dbias_dtype != SDPA_DTYPE_BF16 &&
        ba.dbias_dtype != SDPA_DTYPE_F16)
      return SDPA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(ba.bias) % (ba.dtype == SDPA_DTYPE_F32 ? 4 : 2) != 0 ||
        reinterpret_cast<uintptr_t>(ba.dbias) % (ba.dbias_dtype == SDPA_DTYPE_F32 ? 4 : 2) != 0)
      return SDPA_ERR_ALIGN;
  }
  for (const void* ptr : {q, k, v, o, d_o, (const void*)dq, (const void*)dk, (const void*)dv})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return SDPA_ERR_ALIGN;
  for (const void* ptr : {(const void*)lse, (const void*)sink, (const void*)dsink})
    if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) return SDPA_ERR_ALIGN;
  if (window_right >= 0 && !causal) return SDPA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt((float)D_qk);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  int* status = nullptr;
  int sms = 0;
  rc = device_state(dev, &status, &sms);
  if (rc != SDPA_OK) return rc;

  const size_t dq_bytes = (size_t)B * H_q * S_q * D_qk * 2;
  const size_t dk_bytes = (size_t)B * H_kv * S_kv * D_qk * 2;
  const size_t dv_bytes = (size_t)B * H_kv * S_kv * D_v * 2;
  if (S_q == 0 || S_kv == 0) {  // no (query, key) pair: every gradient is zero
    // (and O = 0, so delta = 0 and dsink = 0)
    if (cudaMemsetAsync(dq, 0, dq_bytes, stream) != cudaSuccess ||
        cudaMemsetAsync(dk, 0, dk_bytes, stream) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, dv_bytes, stream) != cudaSuccess ||
        (dsink && cudaMemsetAsync(dsink, 0, (size_t)H_q * sizeof(float), stream) != cudaSuccess) ||
        (ba.dbias && cudaMemsetAsync(ba.dbias, 0, (size_t)ba.batch * H_q * S_q * S_kv *
                                                      (ba.dbias_dtype == SDPA_DTYPE_F32 ? 4 : 2),
                                     stream) != cudaSuccess))
      return SDPA_ERR_CUDA;
    return SDPA_OK;
  }

  const Route route = choose_route(deterministic, D_qk);
  const bool ds_route = route != Route::kReduce;
  const Shape sh{B, H_q, H_kv, S_q, S_kv, D_qk, D_v, causal, bottom_right, window_left, window_right,
                 (seq_q_lens || seq_kv_lens) ? 1 : 0};
  const Carve cv = carve(sh, route, qat);
  bool own_ws = false;
  if (workspace == nullptr) {
    if (cudaMallocAsync(&workspace, cv.total, stream) != cudaSuccess) return SDPA_ERR_CUDA;
    own_ws = true;
  } else {
    if (workspace_bytes < cv.total) return SDPA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SDPA_ERR_ALIGN;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  ChainParams p{};
  float* dbias_tmp = nullptr;  // fp32 sum of a shared bias's dBias before its io-type cast
  p.B = B; p.Hq = H_q; p.Hkv = H_kv; p.Sq = S_q; p.Skv = S_kv; p.Dqk = D_qk; p.Dv = D_v;
  p.G = H_q / H_kv;
  // Head-group size of the D_qk 64/128 main kernel: the largest divisor of G
  // that still leaves at least 1.5 work units per SM. Fewer, longer units pay
  // the per-unit start and drain less often and leave fewer partial dK/dV sets
  // to reduce; below 1.5 units per SM the greedy dispatch of uneven (causal)
  // units loses more to imbalance than that saves.
  p.gsz = 1;
  if (D_qk <= 128) {
    for (int c = p.G; c > 1; --c) {
      if (p.G % c == 0 && (long long)ceil_div(S_kv, BN) * B * H_kv * (p.G / c) * 2 >= 3ll * sms) {
        p.gsz = c;
        break;
      }
    }
  }
  p.n_part = p.G / p.gsz;
  p.n_qt = ceil_div(S_q, BQ);
  p.n_kt = ceil_div(S_kv, BN);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.bottom_right = bottom_right ? 1 : 0;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.window_right = (causal && window_right > 0) ? window_right : -1;
  // The two-kernel route is deterministic by construction (no cross-CTA
  // reduction); `deterministic` inside the kernels selects the ordered relay.
  p.deterministic = (deterministic && !ds_route) ? 1 : 0;
  p.f16 = f16 ? 1 : 0;
  p.ds_route = ds_route ? 1 : 0;
  p.ds_band = cv.ds_band;
  p.ds_band_tiles = cv.ds_band_tiles;
  p.seq_q_lens = seq_q_lens;
  p.seq_kv_lens = seq_kv_lens;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.d_o = static_cast<const __nv_bfloat16*>(d_o);
  p.lse = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.qstat = reinterpret_cast<float*>(ws + cv.qstat);
  p.dq_accum = ds_route ? nullptr : reinterpret_cast<float*>(ws + cv.dq_accum);
  p.dq_acc_cols = D_qk <= 64 ? 64 : 128;
  p.ds_ws = ds_route ? ws + cv.ds_ws : nullptr;
  p.zero_tile = ds_route ? ws + cv.zero_tile : nullptr;
  p.counters = reinterpret_cast<int*>(ws + cv.counters);
  p.n_counters = B * H_q * p.n_qt + 1;
  p.ticket = p.counters + (p.n_counters - 1);
  // Partial dK/dV sets ([B][H_kv][n_part][S_kv][D], within the region sized for
  // one set per query head) when a KV group spans several work units.
  p.dk_ws = p.n_part > 1 ? reinterpret_cast<__nv_bfloat16*>(ws + cv.dk_ws) : nullptr;
  p.dv_ws = p.n_part > 1 ? reinterpret_cast<__nv_bfloat16*>(ws + cv.dv_ws) : nullptr;
  p.status = status;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    p.relay_wait_ns = g_relay_wait_ns;
    p.relay_turn_skew = g_relay_turn_skew;
  }
  p.sink = dsink ? sink : nullptr;
  p.dsink = dsink;
  p.dsink_part = dsink ? reinterpret_cast<float*>(ws + cv.dsink_part) : nullptr;
  if (ba.bias) {
    const long long per_batch = (long long)H_q * S_q * S_kv;
    const bool shared = ba.batch == 1 && B > 1;
    p.bias = ba.bias;
    p.bias_fp32 = ba.dtype == SDPA_DTYPE_F32 ? 1 : 0;
    p.bias_f16 = ba.dtype == SDPA_DTYPE_F16 ? 1 : 0;
    p.bias_bstride = shared ? 0 : per_batch;
    p.dbias = static_cast<float*>(ba.dbias);
    p.dbias_bstride = shared ? 0 : per_batch;
    p.dbias_red = (ba.dbias && shared) ? 1 : 0;
    // A 16-bit dBias is written directly (each element once), except for a
    // shared bias: its batch rows add into an fp32 buffer, cast at the end.
    if (ba.dbias && ba.dbias_dtype != SDPA_DTYPE_F32) {
      if (shared) {
        if (cudaMallocAsync(reinterpret_cast<void**>(&p.dbias), (size_t)per_batch * sizeof(float), stream) !=
            cudaSuccess) {
          if (own_ws) cudaFreeAsync(workspace, stream);
          return SDPA_ERR_CUDA;
        }
        dbias_tmp = p.dbias;
      } else {
        p.dbias_out = ba.dbias_dtype == SDPA_DTYPE_F16 ? 2 : 1;
      }
    }
  }

  MainMaps maps;
  const long long BHq = (long long)B * H_q, BHkv = (long long)B * H_kv;
  // QAT: the GEMMs read the fake-quantized copies, written first.
  const void* qg = qat ? static_cast<const void*>(ws + cv.q_hat) : q;
  const void* kg = qat ? static_cast<const void*>(ws + cv.k_hat) : k;
  const void* vg = qat ? static_cast<const void*>(ws + cv.v_hat) : v;
  if (!make_bhsd_map(&maps.q, qg, D_qk, S_q, BHq, BQ, f16) ||
      !make_bhsd_map(&maps.k, kg, D_qk, S_kv, BHkv, BN, f16) ||
      !make_bhsd_map(&maps.v, vg, D_v, S_kv, BHkv, BN, f16) ||
      !make_bhsd_map(&maps.d_o, d_o, D_v, S_q, BHq, BQ, f16) ||
      !make_bhsd_map(&maps.dk_out, p.dk_ws ? static_cast<void*>(p.dk_ws) : dk, D_qk, S_kv,
                     p.dk_ws ? BHq : BHkv, BN, f16) ||
      !make_bhsd_map(&maps.dv_out, p.dv_ws ? static_cast<void*>(p.dv_ws) : dv, D_v, S_kv,
                     p.dv_ws ? BHq : BHkv, BN, f16)) {
    if (dbias_tmp) cudaFreeAsync(dbias_tmp, stream);
    if (own_ws) cudaFreeAsync(workspace, stream);
    return SDPA_ERR_CUDA;
  }

  cudaError_t e = cudaSuccess;
  ProfEvents prof(stream);
  prof.begin(0);
  if (qat) {
    e = launch_nvfp4_fake_quant(q, ws + cv.q_hat, BHq * S_q * D_qk / 16, sms, stream);
    if (e == cudaSuccess) e = launch_nvfp4_fake_quant(k, ws + cv.k_hat, BHkv * S_kv * D_qk / 16, sms, stream);
    if (e == cudaSuccess) e = launch_nvfp4_fake_quant(v, ws + cv.v_hat, BHkv * S_kv * D_v / 16, sms, stream);
  }
  if (e == cudaSuccess) e = launch_preprocess(p, stream, sms);
  prof.end(0);
  if (e == cudaSuccess) {
    prof.begin(1);
    e = D_qk > 128 ? launch_main_ds(maps, p, stream)
                    : (qat ? launch_main_qat(maps, p, stream) : launch_main(maps, p, stream));
    prof.end(1);
  }
  if (e == cudaSuccess) {  // dQ (and, under GQA, the dK/dV group reduction)
    prof.begin(2);
    e = ds_route ? launch_dq_from_ds(maps.k, p, stream, sms) : launch_dq_convert(p, stream);
    prof.end(2);
  }
  if (e == cudaSuccess && dsink) {
    nvtxRangePushA("sdpa_bwd.dsink");
    e = launch_dsink(p, stream);
    nvtxRangePop();
  }
  if (dbias_tmp) {
    if (e == cudaSuccess)
      e = launch_dbias_cast(dbias_tmp, ba.dbias, (long long)H_q * S_q * S_kv,
                            ba.dbias_dtype == SDPA_DTYPE_F16, sms, stream);
    cudaFreeAsync(dbias_tmp, stream);
  }
  if (own_ws) cudaFreeAsync(workspace, stream);
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

extern "C" {

int sdpa_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o,
             const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int S_q,
             int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
             int window_left, int window_right, int deterministic, const int32_t* seq_q_lens,
             const int32_t* seq_kv_lens, void* workspace, size_t workspace_bytes, void* stream) {
  return run_chain(q, k, v, o, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                   causal, bottom_right, window_left, window_right, deterministic, seq_q_lens,
                   seq_kv_lens, workspace, workspace_bytes, nullptr, nullptr, BiasArgs{}, stream);
}

}  // extern "C"

namespace {

int run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
            int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
            int bottom_right, int window_left, int window_right, const int32_t* seq_q_lens,
            const int32_t* seq_kv_lens, const float* sink, const BiasArgs& ba, void* stream_,
            bool f16 = false) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int rc = basic_checks(B, H_q, H_kv, S_q, S_kv, D_qk, D_v);
  if (rc != SDPA_OK) return rc;
  // Every pair the backward serves: D_v up to 128 (and the MLA pair) on the
  // kernel with two O halves in tensor memory, 256/256 on the one with a single O.
  if (!q || !k || !v || !o || !lse) return SDPA_ERR_INVALID;
  for (const void* ptr : {q, k, v, (const void*)o})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return SDPA_ERR_ALIGN;
  for (const void* ptr : {(const void*)lse, (const void*)sink})
    if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) return SDPA_ERR_ALIGN;
  if (ba.bias) {
    if (ba.dtype != SDPA_DTYPE_BF16 && ba.dtype != SDPA_DTYPE_F32 && ba.dtype != SDPA_DTYPE_F16)
      return SDPA_ERR_INVALID;
    if (ba.batch != 1 && ba.batch != B) return SDPA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(ba.bias) % (ba.dtype == SDPA_DTYPE_F32 ? 4 : 2) != 0)
      return SDPA_ERR_ALIGN;
  }
  if (window_right >= 0 && !causal) return SDPA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt((float)D_qk);
  if (S_q == 0) return SDPA_OK;  // no rows

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  int* status = nullptr;
  int sms = 0;
  rc = device_state(dev, &status, &sms);
  if (rc != SDPA_OK) return rc;

  FwdParams p{};
  p.B = B; p.Hq = H_q; p.Hkv = H_kv; p.Sq = S_q; p.Skv = S_kv; p.Dqk = D_qk; p.Dv = D_v;
  p.G = H_q / H_kv;
  p.n_qt = ceil_div(S_q, 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.f16 = f16 ? 1 : 0;
  p.causal = causal ? 1 : 0;
  p.bottom_right = bottom_right ? 1 : 0;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.window_right = (causal && window_right > 0) ? window_right : -1;
  p.seq_q_lens = seq_q_lens;
  p.seq_kv_lens = seq_kv_lens;
  p.sink = sink;
  if (ba.bias) {
    const int esz = ba.dtype == SDPA_DTYPE_F32 ? 4 : 2;
    p.bias = ba.bias;
    p.bias_fp32 = esz == 4;
    p.bias_f16 = ba.dtype == SDPA_DTYPE_F16 ? 1 : 0;
    p.bias_bstride = (ba.batch == 1) ? 0 : (long long)H_q * S_q * S_kv;
    p.bias_vec = ((long long)S_kv * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(ba.bias) % 16 == 0;
  }
  p.lse = lse;
  p.o = o;
  p.status = status;
  FwdMaps maps;
  const long long BHq = (long long)B * H_q, BHkv = (long long)B * H_kv;
  // An empty key axis still needs valid K/V maps: point them at Q (never read).
  const int Skv_map = S_kv > 0 ? S_kv : 1;
  const void* kb = S_kv > 0 ? k : q;
  const void* vb = S_kv > 0 ? v : q;
  if (!make_bhsd_map(&maps.q, q, D_qk, S_q, BHq, 128, f16) ||
      !make_bhsd_map(&maps.k, kb, D_qk, Skv_map, S_kv > 0 ? BHkv : BHq, 128, f16) ||
      // (the head-dim-256 kernel loads V in 32-key row groups)
      !make_bhsd_map(&maps.v, vb, D_v, Skv_map, S_kv > 0 ? BHkv : BHq, D_v == 256 ? 32 : 128, f16) ||
      !make_bhsd_map(&maps.o, o, D_v, S_q, BHq, 128, f16))
    return SDPA_ERR_CUDA;
  nvtxRangePushA("sdpa_fwd");
  const cudaError_t e = launch_fwd(maps, p, stream);
  nvtxRangePop();
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

extern "C" {

int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
             int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
             int bottom_right, int window_left, int window_right, const int32_t* seq_q_lens,
             const int32_t* seq_kv_lens, const float* sink, void* stream) {
  return run_fwd(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale, causal, bottom_right,
                 window_left, window_right, seq_q_lens, seq_kv_lens, sink, BiasArgs{}, stream);
}

int sdpa_fwd_typed(int io_dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale,
                   int causal, int bottom_right, int window_left, int window_right,
                   const int32_t* seq_q_lens, const int32_t* seq_kv_lens, const float* sink,
                   const void* bias, int bias_dtype, int bias_batch, void* stream) {
  if (io_dtype != SDPA_DTYPE_BF16 && io_dtype != SDPA_DTYPE_F16) return SDPA_ERR_INVALID;
  BiasArgs ba;
  ba.bias = bias;
  ba.dtype = bias_dtype;
  ba.batch = bias_batch;
  return run_fwd(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale, causal, bottom_right,
                 window_left, window_right, seq_q_lens, seq_kv_lens, sink, ba, stream,
                 io_dtype == SDPA_DTYPE_F16);
}

int sdpa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                  int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
                  int bottom_right, int window_left, int window_right, const int32_t* seq_q_lens,
                  const int32_t* seq_kv_lens, const float* sink, const void* bias, int bias_dtype,
                  int bias_batch, void* stream) {
  if (!bias) return SDPA_ERR_INVALID;
  BiasArgs ba;
  ba.bias = bias;
  ba.dtype = bias_dtype;
  ba.batch = bias_batch;
  return run_fwd(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale, causal, bottom_right,
                 window_left, window_right, seq_q_lens, seq_kv_lens, sink, ba, stream);
}

int sdpa_bwd_sink(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                  int S_q, int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
                  int window_left, int window_right, int deterministic,
                  const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                  size_t workspace_bytes, const float* sink, float* dsink, void* stream) {
  if (!sink || !dsink) return SDPA_ERR_INVALID;
  return run_chain(q, k, v, o, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                   causal, bottom_right, window_left, window_right, deterministic, seq_q_lens,
                   seq_kv_lens, workspace, workspace_bytes, sink, dsink, BiasArgs{}, stream);
}

int sdpa_bwd_typed(int io_dtype, const void* q, const void* k, const void* v, const void* o,
                   const void* d_o, const float* lse, void* dq, void* dk, void* dv, int B, int H_q,
                   int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
                   int bottom_right, int window_left, int window_right, int deterministic,
                   const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                   size_t workspace_bytes, const float* sink, float* dsink, const void* bias,
                   int bias_dtype, int bias_batch, void* dbias, int dbias_dtype, void* stream) {
  if (io_dtype != SDPA_DTYPE_BF16 && io_dtype != SDPA_DTYPE_F16) return SDPA_ERR_INVALID;
  if (dsink && !sink) return SDPA_ERR_INVALID;
  if (!bias && dbias) return SDPA_ERR_INVALID;
  BiasArgs ba;
  ba.bias = bias;
  ba.dtype = bias_dtype;
  ba.batch = bias_batch;
  ba.dbias = dbias;
  ba.dbias_dtype = dbias_dtype;
  return run_chain(q, k, v, o, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                   causal, bottom_right, window_left, window_right, deterministic, seq_q_lens,
                   seq_kv_lens, workspace, workspace_bytes, dsink ? sink : nullptr, dsink, ba,
                   stream, false, io_dtype == SDPA_DTYPE_F16);
}

int sdpa_bwd_nvfp4_qat(const void* q, const void* k, const void* v, const void* o_hp,
                       const void* d_o, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale,
                       int causal, int bottom_right, int window_left, int window_right,
                       const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return run_chain(q, k, v, o_hp, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                   causal, bottom_right, window_left, window_right, 0, seq_q_lens, seq_kv_lens,
                   workspace, workspace_bytes, nullptr, nullptr, BiasArgs{}, stream, true);
}

int sdpa_nvfp4_fake_quant(const void* x, void* y, long long n, void* stream) {
  if (!x || !y || n < 0 || n % 16 != 0) return SDPA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(y) % 16 != 0)
    return SDPA_ERR_ALIGN;
  if (n == 0) return SDPA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  int* status = nullptr;
  int sms = 0;
  const int rc = device_state(dev, &status, &sms);
  if (rc != SDPA_OK) return rc;
  return launch_nvfp4_fake_quant(x, y, n / 16, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SDPA_OK : SDPA_ERR_CUDA;
}

int sdpa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                  int S_q, int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
                  int window_left, int window_right, int deterministic,
                  const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                  size_t workspace_bytes, const float* sink, float* dsink, const void* bias,
                  int bias_dtype, int bias_batch, float* dbias, void* stream) {
  if (!bias || (dsink && !sink)) return SDPA_ERR_INVALID;
  BiasArgs ba;
  ba.bias = bias;
  ba.dtype = bias_dtype;
  ba.batch = bias_batch;
  ba.dbias = dbias;
  return run_chain(q, k, v, o, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                   causal, bottom_right, window_left, window_right, deterministic, seq_q_lens,
                   seq_kv_lens, workspace, workspace_bytes, dsink ? sink : nullptr, dsink, ba,
                   stream);
}

}  // extern "C"
