// sdpa_bwd_noalloc.cu -- an SDPA backward entry point that allocates no device
// memory: its workspace is a fixed array compiled into the library.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the
// point where they run the backward. Examples are plugins and foreign-function
// hooks called by a framework that has already reserved the whole device memory
// pool for its own allocator (a cudaMalloc there fails or fragments the pool),
// and latency-critical code that cannot accept cudaMalloc's implicit device
// synchronization. They still pass their own inputs and outputs; only the
// scratch memory of the chain (row statistics, the fp32 dQ accumulator, the
// turn counters and the GQA partials) comes from the static array below.
//
// Costs and limits:
//   - The array takes NOALLOC_SCRATCH_BYTES of device memory on each GPU where
//     the code module holding it is loaded, until the process exits. Under
//     CUDA's default lazy module loading that happens at the first call on
//     that GPU (the address lookup below), and the chain's kernel modules load
//     at their first launch; both need device memory. A caller whose framework
//     later reserves the whole device pool should therefore make one small
//     call on each GPU before the pool is reserved (or run with
//     CUDA_MODULE_LOADING=EAGER, which loads every module, the array included,
//     when the CUDA context is created).
//   - A problem whose workspace (sdpa_bwd_workspace_size) exceeds the array is
//     rejected with SDPA_ERR_WORKSPACE before anything is launched.
//   - All calls on a device share the one array, which keeps the contents the
//     last call left. The kernels clear what must start at zero (accumulator,
//     counters) and overwrite everything else on every call, but two calls whose
//     work overlaps on the device (different streams, no ordering between them)
//     race on the array and corrupt each other's results.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current). Make that first call
//     before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sdpa_bwd.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device; the host-side symbol itself is not a device address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDPA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SDPA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return SDPA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return SDPA_OK;
}

}  // namespace

extern "C" {

int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                     int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
                     int bottom_right, int window_left, int window_right, int deterministic,
                     const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* stream) {
  const size_t need = sdpa_bwd_workspace_size(B, H_q, H_kv, S_q, S_kv, D_qk, D_v, causal, bottom_right,
                                              window_left, window_right, deterministic,
                                              (seq_q_lens || seq_kv_lens) ? 1 : 0);
  if (need > NOALLOC_SCRATCH_BYTES) return SDPA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SDPA_OK) return rc;
  // Same chain as sdpa_bwd with the static array as the caller-provided
  // workspace: sdpa_bwd allocates only when it is given no workspace.
  return sdpa_bwd(q, k, v, o, d_o, lse, dq, dk, dv, B, H_q, H_kv, S_q, S_kv, D_qk, D_v, scale,
                  causal, bottom_right, window_left, window_right, deterministic, seq_q_lens,
                  seq_kv_lens, scratch, NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
