// sdpa_bwd_main_bias.cu -- the main kernels with an additive bias and the
// dBias output (sdpa_bwd_main.cuh, BIAS = true), in their own translation
// unit so that they compile in parallel with the others.
#include "sdpa_bwd_main.cuh"

namespace sdpa {

cudaError_t main_bias_kernel_setup() { return main_variant_setup<true>(); }

cudaError_t launch_main_bias(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  return launch_main_variant<true>(maps, p, s);
}

}  // namespace sdpa
