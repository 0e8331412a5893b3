// sdpa_bwd_main_qat.cu -- the NVFP4 QAT backward's kernels ("NVFP4 Attention
// QAT Backward" page, Overview): the main kernel with G3 reading P
// fake-quantized to NVFP4 (sdpa_bwd_main.cuh, QAT = true; D = 128, dQ-reduction
// route), and the fake quantization of Q, K and V that runs before it.
#include "gqa.cuh"
#include "nvfp4.cuh"
#include "sdpa_bwd_main.cuh"

namespace sdpa {

cudaError_t main_qat_kernel_setup() { return set_main_smem<128, false, false, true>(); }

cudaError_t launch_main_qat(const MainMaps& maps, const ChainParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.n_kt * p.B * p.Hkv * p.n_part));
  return launch_kernel(sdpa_bwd_main<128, false, false, true>, grid, dim3(MAIN_THREADS),
                       MainLayout<128, false>::BYTES, s, true, maps, p);
}

// One thread per block of 16 consecutive bf16 values (two 16-byte vectors;
// consecutive threads on consecutive blocks). The block's local scale is
// E4M3(amax / 6); each value becomes E2M1(x / scale) * scale, exact in bf16.
__global__ void __launch_bounds__(256) sdpa_nvfp4_fake_quant(const uint4* __restrict__ x,
                                                             uint4* __restrict__ y,
                                                             long long n_blocks) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n_blocks;
       i += (long long)gridDim.x * 256) {
    const uint4 a = x[2 * i], b = x[2 * i + 1];
    float v[16];
    float (&v0)[8] = *reinterpret_cast<float(*)[8]>(v);
    float (&v1)[8] = *reinterpret_cast<float(*)[8]>(v + 8);
    unpack8(a, v0);
    unpack8(b, v1);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const float sc = nvfp4_scales(amax, amax).x;
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = fake_nvfp4_pair_bf16(v[2 * j], v[2 * j + 1], sc, sc);
    y[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
    y[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

cudaError_t launch_nvfp4_fake_quant(const void* x, void* y, long long n_blocks, int num_sms,
                                    cudaStream_t s) {
  if (n_blocks <= 0) return cudaSuccess;
  const long long want = (n_blocks + 255) / 256, cap = (long long)num_sms * 8;
  const dim3 grid((unsigned)(want < cap ? want : cap));
  return launch_kernel(sdpa_nvfp4_fake_quant, grid, dim3(256), 0, s, false,
                       static_cast<const uint4*>(x), static_cast<uint4*>(y), n_blocks);
}

}  // namespace sdpa
