// sdpa_bwd_main_f16.cu -- the main kernels (sdpa_bwd_main.cuh) with fp16 io
// tensors ("SDPA Backward (SM120)", support surface: FP16 / BF16), in their own
// translation unit so that they compile in parallel with the others.
#include "sdpa_bwd_main.cuh"

namespace sdpa {

cudaError_t main_f16_kernel_setup() { return main_variant_setup<false, true>(); }

cudaError_t launch_main_f16(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  return launch_main_variant<false, true>(maps, p, s);
}

}  // namespace sdpa
