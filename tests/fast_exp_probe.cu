// Test probe (built by tests/test_fast_exp.py, not part of libgdr): evaluates the
// tensor-core kernels' fast_exp (tc_common.cuh) and CUDA's expf on the same inputs.
#include <cuda_runtime.h>

#include "../gated_delta_rule_03_gb300/csrc/tc_common.cuh"

__global__ void probe_kernel(const float *x, float *fast, float *ref, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        fast[i] = gdr::tc::fast_exp(x[i]);
        ref[i] = expf(x[i]);
    }
}

extern "C" int fast_exp_probe(const float *x, float *fast, float *ref, int n) {
    if (n <= 0) return 0;
    probe_kernel<<<(n + 255) / 256, 256>>>(x, fast, ref, n);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}
