// sv_alpha.cuh -- per-position acceptance-rate diagnostic (sm_103a).
//
// For each sequence b and draft position i < K: alpha[b][i] =
// sum_v min(p_i(v) / P_i, q_i(v) / Q_i), P_i and Q_i the row totals, and the
// expected accepted length E[b] = sum_{m=1..K} prod_{j<m} alpha[b][j] -- the
// quantities of the rejection-sampling theorem behind the "spec-verify"
// page's analytic accepted-length law (section "Measured").  Diagnostic only:
// it reads every p_i and q_i row in full, twice.
//
// Three launches on one stream, the later two programmatic dependents:
//  1. one CTA per (b, i) row pair sums P_i and Q_i in double-fp32 (the exact
//     four-element sums of quad_mass, combined with Dekker additions);
//  2. one CTA per row pair sums min(p * (1/P), q * (1/Q)) the same way, with
//     the reciprocals rounded once to fp32 -- each term carries at most two
//     fp32 roundings, so |alpha - exact| <= 2 * 2^-24 * alpha ~ 1.2e-7;
//  3. one thread per sequence forms E[b] in fp64.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kAlphaWarps = 8;
constexpr int kAlphaThreads = kAlphaWarps * 32;

struct AlphaParams {
    const float *p;
    int64_t ps;
    const float *q;
    int64_t qs;
    int32_t B, K;
    int64_t V;
    int32_t nseg;
    float2 *norm;       // workspace [B][K][2]: P_i, Q_i as double-fp32
    double *alpha;      // [B][K]
    double *expected;   // [B] or null
};

__device__ __forceinline__ dd warp_sum_dd(dd v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = dd_add(v, shfl_xor_dd(v, m));
    return v;
}

// Sum over the CTA of one dd per warp (lane 0's); the result is valid in warp 0.
__device__ __forceinline__ dd cta_sum_dd(dd v, dd *sh, int warp, int lane) {
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    dd t = lane < kAlphaWarps ? sh[lane] : dd{0.f, 0.f};
    if (warp == 0) t = warp_sum_dd(t);
    return t;
}

// Per-lane sums over one row pair: f(pv, qv) gives the four terms of a float4
// pair; aligned full segments take 16-byte loads, the rest scalar loads.
template <class F>
__device__ __forceinline__ void row_pair_sums(const float *pr, const float *qr, int64_t V, int nseg,
                                              bool vec, int warp, int lane, F f, dd &s0, dd &s1) {
    for (int s = warp; s < nseg; s += kAlphaWarps) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t n = V - base < kSeg ? V - base : kSeg;
        if (vec && n == kSeg) {
#pragma unroll 4
            for (int k = 0; k < kVecPerLane; ++k) {
                const int64_t e = base + 4 * (lane + 32 * k);
                f(ld_stream4(pr + e), ld_stream4(qr + e), s0, s1);
            }
        } else {
            for (int64_t e = base + 4 * lane; e < base + n; e += 128) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
                a.x = ld_stream1(pr + e);
                c.x = ld_stream1(qr + e);
                if (e + 1 < base + n) { a.y = ld_stream1(pr + e + 1); c.y = ld_stream1(qr + e + 1); }
                if (e + 2 < base + n) { a.z = ld_stream1(pr + e + 2); c.z = ld_stream1(qr + e + 2); }
                if (e + 3 < base + n) { a.w = ld_stream1(pr + e + 3); c.w = ld_stream1(qr + e + 3); }
                f(a, c, s0, s1);
            }
        }
    }
}

__device__ __forceinline__ bool alpha_vec(const AlphaParams &A) {
    return aligned16(A.p) && aligned16(A.q) && (A.ps & 3) == 0 && (A.qs & 3) == 0;
}

__global__ void __launch_bounds__(kAlphaThreads) alpha_norm_kernel(const AlphaParams A) {
    __shared__ dd sh[2][kAlphaWarps];
    grid_dependents_may_launch();
    const int b = blockIdx.x / A.K, i = blockIdx.x - b * A.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *pr = A.p + ((int64_t)b * (A.K + 1) + i) * A.ps;
    const float *qr = A.q + ((int64_t)b * A.K + i) * A.qs;
    dd sp = {0.f, 0.f}, sq = {0.f, 0.f};
    row_pair_sums(pr, qr, A.V, A.nseg, alpha_vec(A), warp, lane,
                  [](float4 a, float4 c, dd &s0, dd &s1) {
                      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                      s0 = dd_add(s0, quad_mass<false>(a, z));
                      s1 = dd_add(s1, quad_mass<false>(c, z));
                  },
                  sp, sq);
    sp = warp_sum_dd(sp);
    sq = warp_sum_dd(sq);
    const dd P = cta_sum_dd(sp, sh[0], warp, lane);
    const dd Q = cta_sum_dd(sq, sh[1], warp, lane);
    if (threadIdx.x == 0) {
        float2 *o = A.norm + ((int64_t)b * A.K + i) * 2;
        o[0] = make_float2(P.hi, P.lo);
        o[1] = make_float2(Q.hi, Q.lo);
    }
}

__global__ void __launch_bounds__(kAlphaThreads) alpha_min_kernel(const AlphaParams A) {
    __shared__ dd sh[kAlphaWarps];
    grid_dependents_may_launch();
    wait_for_primary_grid();  // the totals
    const int b = blockIdx.x / A.K, i = blockIdx.x - b * A.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float2 *o = A.norm + ((int64_t)b * A.K + i) * 2;
    const float2 P2 = ld_l2(o), Q2 = ld_l2(o + 1);
    const double P = (double)P2.x + (double)P2.y, Q = (double)Q2.x + (double)Q2.y;
    if (!(P > 0.0) || !(Q > 0.0)) {  // a row with no mass: no acceptance
        if (threadIdx.x == 0) A.alpha[(int64_t)b * A.K + i] = 0.0;
        return;
    }
    const float ip = (float)(1.0 / P), iq = (float)(1.0 / Q);
    const float *pr = A.p + ((int64_t)b * (A.K + 1) + i) * A.ps;
    const float *qr = A.q + ((int64_t)b * A.K + i) * A.qs;
    dd s = {0.f, 0.f}, unused = {0.f, 0.f};
    row_pair_sums(pr, qr, A.V, A.nseg, alpha_vec(A), warp, lane,
                  [ip, iq](float4 a, float4 c, dd &s0, dd &) {
                      const float4 m = make_float4(fminf(a.x * ip, c.x * iq), fminf(a.y * ip, c.y * iq),
                                                   fminf(a.z * ip, c.z * iq), fminf(a.w * ip, c.w * iq));
                      s0 = dd_add(s0, quad_mass<false>(m, make_float4(0.f, 0.f, 0.f, 0.f)));
                  },
                  s, unused);
    s = warp_sum_dd(s);
    const dd t = cta_sum_dd(s, sh, warp, lane);
    if (threadIdx.x == 0) A.alpha[(int64_t)b * A.K + i] = (double)t.hi + (double)t.lo;
}

__global__ void alpha_length_kernel(const AlphaParams A) {
    wait_for_primary_grid();  // every alpha
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= A.B) return;
    double mean = 0.0, reach = 1.0;
    for (int i = 0; i < A.K; ++i) {
        reach *= A.alpha[(int64_t)b * A.K + i];  // P(n > i)
        mean += reach;
    }
    A.expected[b] = mean;
}

}  // namespace sv
