// sv_alpha.cuh -- per-position acceptance-rate diagnostic (sm_103a).
//
// For each sequence b and draft position i < K: alpha[b][i] =
// sum_v min(p_i(v) / P_i, q_i(v) / Q_i), P_i and Q_i the row totals, and the
// expected accepted length E[b] = sum_{m=1..K} prod_{j<m} alpha[b][j] -- the
// quantities of the rejection-sampling theorem behind the "spec-verify"
// page's analytic accepted-length law (section "Measured").  Diagnostic only:
// it reads every p_i and q_i row in full.
//
// alpha needs the totals before the minima, so each row pair is read twice;
// only the first read comes from DRAM.  One thread-block cluster of
// kAlphaCluster CTAs takes a (b, i) row pair, CTA r an r-th of its segments:
//  1. each CTA sums its slice of P_i and Q_i in double-fp32 (the exact
//     four-element sums of quad_mass, combined with Dekker additions) and
//     writes the pair of partials into every CTA of the cluster (distributed
//     shared memory); after a cluster barrier every CTA adds the partials in
//     rank order, so all hold the same P_i, Q_i;
//  2. each CTA sums min(p * (1/P), q * (1/Q)) over its slice again -- the
//     slice it read moments before, now an L2 hit -- with the reciprocals
//     rounded once to fp32: each term carries at most two fp32 roundings, so
//     |alpha - exact| <= 2 * 2^-24 * alpha ~ 1.2e-7; the partials go to the
//     cluster's first CTA, which adds them in rank order;
//  3. a dependent launch, one thread per sequence, forms E[b] in fp64.
// The launch's shared memory (which also keeps the first segments of each
// CTA's slice for the second sweep) and registers bound the CTAs resident
// per SM, so that the row pairs being read at once stay mostly inside L2
// until their second read.
#pragma once

#include <cooperative_groups.h>

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

// Per-lane sums over segments [s0, s1) of a row pair: f(pv, qv) takes the
// four terms of a float4 pair; aligned full segments take 16-byte loads, the
// rest scalar loads.  kKeep: the first kAlphaKeepSegs full segments of the
// slice are also stored in (1) or read from (2) the shared-memory copy, so the
// second sweep reads them from shared memory instead of L2.
constexpr int kAlphaKeepSegs = 4;  // 2 rows x 4 x 4 KB = 32 KB of the shared memory reserved
template <int kKeep, class F>
__device__ __forceinline__ void slice_pair_sums(const float *pr, const float *qr, int64_t V, int s0,
                                                int s1, bool vec, int warp, int lane, F f, dd &x0,
                                                dd &x1, float4 *keep) {
    for (int s = s0 + warp; s < s1; s += kAlphaWarps) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t n = V - base < kSeg ? V - base : kSeg;
        const int j = s - s0;  // the segment's place in the slice
        if (vec && n == kSeg && kKeep == 2 && j < kAlphaKeepSegs) {
            const float4 *kp = keep + (size_t)j * 2 * (kSeg / 4);
#pragma unroll 4
            for (int k = 0; k < kVecPerLane; ++k)
                f(kp[lane + 32 * k], kp[kSeg / 4 + lane + 32 * k], x0, x1);
        } else if (vec && n == kSeg) {
            float4 *kp = keep + (size_t)j * 2 * (kSeg / 4);
#pragma unroll 4
            for (int k = 0; k < kVecPerLane; ++k) {
                const int64_t e = base + 4 * (lane + 32 * k);
                const float4 a = ld_stream4(pr + e), c = ld_stream4(qr + e);
                if (kKeep == 1 && j < kAlphaKeepSegs) {
                    kp[lane + 32 * k] = a;
                    kp[kSeg / 4 + lane + 32 * k] = c;
                }
                f(a, c, x0, x1);
            }
        } else {
            for (int64_t e = base + 4 * lane; e < base + n; e += 128) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
                a.x = ld_stream1(pr + e);
                c.x = ld_stream1(qr + e);
                if (e + 1 < base + n) { a.y = ld_stream1(pr + e + 1); c.y = ld_stream1(qr + e + 1); }
                if (e + 2 < base + n) { a.z = ld_stream1(pr + e + 2); c.z = ld_stream1(qr + e + 2); }
                if (e + 3 < base + n) { a.w = ld_stream1(pr + e + 3); c.w = ld_stream1(qr + e + 3); }
                f(a, c, x0, x1);
            }
        }
    }
}

__device__ __forceinline__ bool alpha_vec(const AlphaParams &A) {
    return aligned16(A.p) && aligned16(A.q) && (A.ps & 3) == 0 && (A.qs & 3) == 0;
}

constexpr int kAlphaCluster = 8;
// The launch's dynamic shared memory, sized for kAlphaCtasPerSm CTAs per SM,
// holds each CTA's first kAlphaKeepSegs segments for the second sweep, which
// spares that sweep a quarter of its L2 re-reads.  Registers (42 a thread)
// and the shared-memory carveout hold the residency to 5 CTAs per SM (ncu's
// occupancy limits), 95 row pairs read at once.  Measured per call at B=256
// V=128256 K=5: sized for 4 per SM without kept segments 441.5 us, for 4
// keeping 6 segments 373.0, for 6 keeping 4 343.3; 7 or 8 per SM need at most
// 32 registers and spill (446.4, 440.8).
constexpr int kAlphaCtasPerSm = 6;
constexpr int kAlphaSmemBytes = 200 * 1024 / kAlphaCtasPerSm;
static_assert(kAlphaKeepSegs * 2 * kSeg * 4 <= kAlphaSmemBytes, "the kept segments fit the reserved memory");

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// One cluster per (b, i) row pair (blockIdx.x / kAlphaCluster); see the top
// of this file.
__global__ void __cluster_dims__(kAlphaCluster, 1, 1) __launch_bounds__(kAlphaThreads)
    alpha_pair_kernel(const AlphaParams A) {
    namespace cg = cooperative_groups;
    __shared__ dd sh[2][kAlphaWarps];
    __shared__ dd pq[kAlphaCluster][2];   // every CTA's (P, Q) partials, written by their CTAs
    __shared__ dd am[kAlphaCluster];      // the alpha partials (first CTA only)
    __shared__ float recip[2];
    // the cluster's CTAs have all started before any writes into another's
    // shared memory (the wait is below, after this CTA's own first pass)
    cluster_arrive_relaxed();
    grid_dependents_may_launch();
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int64_t pair = (int64_t)(blockIdx.x / kAlphaCluster);
    const int b = (int)(pair / A.K), i = (int)(pair - (int64_t)b * A.K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = (A.nseg + kAlphaCluster - 1) / kAlphaCluster;
    const int s0 = min(A.nseg, rank * per), s1 = min(A.nseg, s0 + per);
    const float *pr = A.p + ((int64_t)b * (A.K + 1) + i) * A.ps;
    const float *qr = A.q + ((int64_t)b * A.K + i) * A.qs;
    const bool vec = alpha_vec(A);
    extern __shared__ __align__(16) float4 keep[];
    dd sp = {0.f, 0.f}, sq = {0.f, 0.f};
    slice_pair_sums<1>(pr, qr, A.V, s0, s1, vec, warp, lane,
                    [](float4 a, float4 c, dd &x0, dd &x1) {
                        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                        x0 = dd_add(x0, quad_mass<false>(a, z));
                        x1 = dd_add(x1, quad_mass<false>(c, z));
                    },
                    sp, sq, keep);
    sp = warp_sum_dd(sp);
    sq = warp_sum_dd(sq);
    const dd P_part = cta_sum_dd(sp, sh[0], warp, lane);
    const dd Q_part = cta_sum_dd(sq, sh[1], warp, lane);
    cluster_wait();
    if (threadIdx.x < kAlphaCluster) {  // warp 0's lanes hold the totals: into CTA threadIdx.x
        dd *dst = cluster.map_shared_rank(&pq[0][0], (int)threadIdx.x);
        dst[2 * rank] = P_part;
        dst[2 * rank + 1] = Q_part;
    }
    cluster.sync();
    if (threadIdx.x == 0) {
        dd P = pq[0][0], Q = pq[0][1];
        for (int r = 1; r < kAlphaCluster; ++r) {
            P = dd_add(P, pq[r][0]);
            Q = dd_add(Q, pq[r][1]);
        }
        const double Pd = (double)P.hi + (double)P.lo, Qd = (double)Q.hi + (double)Q.lo;
        // a row with no mass: no acceptance (0 marks it)
        recip[0] = Pd > 0.0 && Qd > 0.0 ? (float)(1.0 / Pd) : 0.f;
        recip[1] = Pd > 0.0 && Qd > 0.0 ? (float)(1.0 / Qd) : 0.f;
    }
    __syncthreads();
    const float ip = recip[0], iq = recip[1];
    dd m = {0.f, 0.f}, unused = {0.f, 0.f};
    if (ip != 0.f)
        slice_pair_sums<2>(pr, qr, A.V, s0, s1, vec, warp, lane,
                        [ip, iq](float4 a, float4 c, dd &x0, dd &) {
                            const float4 v = make_float4(fminf(a.x * ip, c.x * iq), fminf(a.y * ip, c.y * iq),
                                                         fminf(a.z * ip, c.z * iq), fminf(a.w * ip, c.w * iq));
                            x0 = dd_add(x0, quad_mass<false>(v, make_float4(0.f, 0.f, 0.f, 0.f)));
                        },
                        m, unused, keep);
    m = warp_sum_dd(m);
    const dd M_part = cta_sum_dd(m, sh[0], warp, lane);
    if (threadIdx.x == 0) cluster.map_shared_rank(&am[0], 0)[rank] = M_part;
    cluster.sync();  // after this no CTA touches another's shared memory
    if (rank == 0 && threadIdx.x == 0) {
        dd t = am[0];
        for (int r = 1; r < kAlphaCluster; ++r) t = dd_add(t, am[r]);
        A.alpha[pair] = ip != 0.f ? (double)t.hi + (double)t.lo : 0.0;
    }
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
