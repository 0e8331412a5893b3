// sdpa_bwd_main.cu -- the main kernels without a bias (sdpa_bwd_main.cuh) and
// the launcher that picks between them and the biased ones.
#include "sdpa_bwd_main.cuh"

namespace sdpa {

cudaError_t main_kernel_setup() {
  cudaError_t e = main_variant_setup<false>();
  if (e == cudaSuccess) e = main_bias_kernel_setup();
  if (e == cudaSuccess) e = main_qat_kernel_setup();
  if (e == cudaSuccess) e = main_f16_kernel_setup();
  return e;
}

cudaError_t launch_main(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  if (p.bias != nullptr) return launch_main_bias(maps, p, s);
  if (p.f16) return launch_main_f16(maps, p, s);
  return launch_main_variant<false>(maps, p, s);
}

}  // namespace sdpa
