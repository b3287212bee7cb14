// Test probe: the largest relative error of ex2.approx.f32 against fp64 exp2
// over arguments in [-100, 0] (the range in which the logits kernels decide an
// accept test in fp32; their error bound assumes at most 2^-20).  Built and
// run by the GPU tests only.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void ex2_error_kernel(unsigned long long *worst, uint32_t n_grid, uint32_t n_bits) {
    double local = 0.0;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_grid + n_bits; i += stride) {
        float a;
        if (i < n_grid) {
            a = -100.0f * (float)((double)i / (double)n_grid);  // an even grid over the range
        } else {
            // evenly spaced float bit patterns between -0 and -100 (dense near 0)
            const uint32_t lo = 0x80000000u, hi = 0xC2C80000u;  // -0.0f and -100.0f
            a = __uint_as_float(lo + (uint32_t)(((uint64_t)(i - n_grid) * (hi - lo)) / n_bits));
        }
        float y;
        asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(a));
        const double ref = exp2((double)a);
        const double rel = fabs((double)y - ref) / ref;
        local = rel > local ? rel : local;
    }
    atomicMax(worst, (unsigned long long)__double_as_longlong(local));  // non-negative: bit order is value order
}

extern "C" int ex2_worst_relative_error(double *out) {
    unsigned long long *d = nullptr, h = 0;
    if (cudaMalloc(&d, sizeof(h)) != cudaSuccess) return -1;
    cudaMemset(d, 0, sizeof(h));
    ex2_error_kernel<<<1024, 256>>>(d, 1u << 26, 1u << 26);
    const bool ok = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(d);
    if (!ok) return -1;
    union { unsigned long long u; double f; } v;
    v.u = h;
    *out = v.f;
    return 0;
}
