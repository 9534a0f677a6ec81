// Test-only probe: evaluates the library's exp2_poly and CUDA's exp2f on the same inputs.
#include "../../attention_flashattention_sdpa_gb300/csrc/ptx.cuh"

__global__ void exp2_probe_kernel(const float* x, float* poly, float* ref, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    poly[i] = sdpa::ptx::exp2_poly(x[i]);
    ref[i] = exp2f(x[i]);
  }
}

extern "C" int exp2_probe(const float* x, float* poly, float* ref, int n) {
  exp2_probe_kernel<<<(n + 255) / 256, 256>>>(x, poly, ref, n);
  return (int)cudaDeviceSynchronize();
}
