// sv_debug.cuh -- input checks of a debug build of the library (compiled only
// with -DSV_DEBUG=1; the default build neither contains nor runs them).
//
// The "spec-verify" page takes probabilities as given: they need not be
// normalised, but the rules assume finite, non-negative masses (section
// "Correctness"; section "Requirements and limits" asks for draft and target
// probabilities warped identically).  NaN, negative or infinite entries give
// unspecified results in the regular build.  A debug build scans every input
// row once before the verification kernels run and raises
// SV_STATUS_BAD_VALUE when one holds such an entry (for logits: a NaN or an
// infinity).  The verification itself is unchanged.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr uint32_t kStatusBadValue = 32u;
constexpr int kCheckThreads = 256;
constexpr int64_t kCheckMaxGrid = 1 << 20;

// CTAs take rows r = blockIdx.x, blockIdx.x + gridDim.x, ... of `rows` rows
// of V floats starting `stride` floats apart; plain scalar loads, so any
// alignment and page-locked host rows are fine.  finite_only: reject only NaN
// and infinities (logits may be negative).
__global__ void __launch_bounds__(kCheckThreads)
    check_values_kernel(const float *base, int64_t stride, int64_t rows, int64_t V,
                        int finite_only, uint32_t *status) {
    int bad = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *row = base + r * stride;
        for (int64_t v = threadIdx.x; v < V; v += kCheckThreads) {
            const float x = row[v];
            // a NaN fails every comparison, so it is rejected by both tests
            bad |= finite_only ? !(fabsf(x) < __int_as_float(0x7f800000))
                               : !(x >= 0.f && x < __int_as_float(0x7f800000));
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kStatusBadValue);
}

// Enqueues the check of `rows` rows on stream st (nothing for an empty set).
inline int check_values(const float *base, int64_t stride, int64_t rows, int64_t V,
                        bool finite_only, uint32_t *status, cudaStream_t st) {
    if (!base || rows <= 0 || V <= 0) return 0;
    const int64_t grid = rows < kCheckMaxGrid ? rows : kCheckMaxGrid;
    check_values_kernel<<<(unsigned)grid, kCheckThreads, 0, st>>>(base, stride, rows, V,
                                                                   finite_only ? 1 : 0, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sv
