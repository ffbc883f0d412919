// test_hooks.cu -- ssm_test_math: evaluates one of the device math helpers of
// common.cuh elementwise, so tests can hold each to its stated error bound over a
// dense grid of its domain (the scan's parity runs only check them indirectly).
#include "common.cuh"
#include "ssm_scan.h"

namespace {

__global__ void math_kernel(int fn, const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = x[i];
    float r;
    switch (fn) {
        case SSM_MATH_EXP: r = ssm::exp_acc(v); break;
        case SSM_MATH_LOG1P01: r = ssm::log1p01(v); break;
        case SSM_MATH_EXPM1: r = ssm::expm1_acc(v); break;
        case SSM_MATH_SOFTPLUS: r = ssm::softplus_acc<true>(v); break;
        case SSM_MATH_SILU: r = ssm::silu_acc<true>(v); break;
        case SSM_MATH_SOFTPLUS_SFU: r = ssm::softplus_acc<false>(v); break;
        default: r = ssm::silu_acc<false>(v); break;
    }
    y[i] = r;
}

}  // namespace

extern "C" int ssm_test_math(int fn, const float* x, float* y, int64_t n, void* stream) {
    if (fn < SSM_MATH_EXP || fn > SSM_MATH_SILU_SFU) return SSM_ERR_ALGO;
    if (n < 0) return SSM_ERR_DIM;
    if (n == 0) return SSM_OK;
    if (!x || !y) return SSM_ERR_NULL;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > ((int64_t)1 << 31) - 1) return SSM_ERR_DIM;
    math_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(fn, x, y, n);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}
