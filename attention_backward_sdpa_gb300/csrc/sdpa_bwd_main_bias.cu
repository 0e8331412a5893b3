// sdpa_bwd_main_bias.cu -- the main kernels with an additive bias and the
// dBias output (sdpa_bwd_main.cuh, BIAS = true), in their own translation
// unit so that they compile in parallel with the others.
#include "sdpa_bwd_main.cuh"

namespace sdpa {

cudaError_t main_bias_kernel_setup() {
  cudaError_t e = main_variant_setup<true, false>();
  if (e == cudaSuccess) e = main_variant_setup<true, true>();
  return e;
}

cudaError_t launch_main_bias(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  return p.f16 ? launch_main_variant<true, true>(maps, p, s) : launch_main_variant<true, false>(maps, p, s);
}

}  // namespace sdpa
