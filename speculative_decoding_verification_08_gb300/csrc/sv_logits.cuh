// sv_logits.cuh -- sampling verification straight from logits (sm_103a).
//
// The "spec-verify" page requires the target and draft distributions to be
// warped identically (section "Requirements and limits"); here the warp is
// part of the op: p_i = softmax(zp_i / tau), q_i = softmax(zq_i / tau), and the
// sampling rule of section "Method" runs on those rows without ever writing
// them to memory.  (Greedy needs no warp: softmax is strictly increasing, so
// argmax p_i = argmax zp_i, and the greedy entry point takes logits as they
// are.)
//
// One thread-block cluster of up to 8 CTAs per sequence walks its rows in
// order; CTA r of the cluster streams segments r*8 + w, r*8 + w + 8*C, ... (w
// its warp, C the cluster size).  For position i each CTA streams its share of
// the row pair (zp_i, zq_i) once, keeping per lane an online maximum and a
// compensated (Kahan) fp32 sum of exp2((z - max) * c), c = log2(e) / tau.  The CTA writes
// its (max, sum) pair into a shared slot (two slots, alternating by row), one
// cluster barrier follows, and every CTA combines all C slots in rank order
// through distributed shared memory -- so every CTA holds bit-identical
// normalisers and reaches the same accept decision u * q_i(t_i) < p_i(t_i)
// (made on the recomputed gathers).  After the first rejection the cluster
// streams that row pair a second time, forming r = max(0, p - q) per element
// in fp32 and, from fp32 sums of four, the double-fp32 block and segment sums
// of r in the workspace;
// when all K are accepted it streams zp_K twice (normaliser, then the masses
// of p_K).  After a last cluster barrier CTA 0 draws: the same segment ->
// block -> element search as the probability path, its element step
// recomputing the masses with the same instructions.
//
// Every CTA of a cluster makes the same sequence of barrier calls: the
// decisions between them depend only on values every CTA computes identically,
// and no CTA leaves while another may still read its shared memory (the last
// reads of it precede the last barrier).
//
// Accuracy: each mass carries the error of exp2.approx (~2^-22), of the fp32
// subtraction and scaling of its argument (about |z - max| * c * 2^-24 in the
// exponent) and of the fp32 normalisation -- around 1e-6 relative at most for
// the elements that carry mass; sums of four add at most 3 * 2^-24 relative,
// and the row totals are compensated.  Accept decisions can therefore differ from an
// fp64 softmax only when |u*q - p| is within ~1e-5 of p, and drawn tokens only
// when u*R lies within ~2e-6 (in units of normalised mass) of a boundary.
#pragma once

#include <cooperative_groups.h>

#include "sv_device.cuh"

namespace sv {

constexpr int kLgWarps = 8;
constexpr int kLgMaxCluster = 8;  // portable cluster size
constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kLgThreads = kLgWarps * 32;

struct LogitsParams {
    const float *zp;
    int64_t ps;
    const float *zq;
    int64_t qs;
    const int32_t *t;
    const float *u_acc;
    const double *u_res;
    int32_t B, K;
    int64_t V;
    int32_t nseg;
    float c;            // log2(e) / tau
    int32_t *n_out;
    int32_t *next_out;
    uint32_t *status;
    float2 *seg;        // workspace [B][nseg]
    float2 *blk;        // workspace [B][nseg][8]
    int32_t csize;      // CTAs per sequence (the cluster size)
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// exp((z - m) / tau) as used everywhere in this file (no contraction, so every
// recomputation gives the same bits).
__device__ __forceinline__ float warp_e(float z, float m, float c) {
    return ex2(__fmul_rn(__fsub_rn(z, m), c));
}

// Sum of four fp32 masses in one fixed order (the same everywhere in this
// file, so the element step of the draw reproduces the block sums).
__device__ __forceinline__ float sum4(float4 m) {
    return __fadd_rn(__fadd_rn(m.x, m.y), __fadd_rn(m.z, m.w));
}

// Running (max, sum of exp) of one row, per lane: the sum is compensated
// (Kahan), s.hi the running sum and s.lo the compensation.
struct Online {
    float m = kNegInf;
    dd s = {0.f, 0.f};
    __device__ void add4(float4 x, float c) {
        const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
        if (mx == kNegInf) return;  // padding only
        if (mx > m) {
            if (s.hi != 0.f) {
                const float f = warp_e(m, mx, c);
                s = dd{__fmul_rn(s.hi, f), __fmul_rn(s.lo, f)};
            }
            m = mx;
        }
        const float q = sum4(make_float4(warp_e(x.x, m, c), warp_e(x.y, m, c), warp_e(x.z, m, c),
                                         warp_e(x.w, m, c)));
        const float y = __fsub_rn(q, s.lo);
        const float t = __fadd_rn(s.hi, y);
        s.lo = __fsub_rn(__fsub_rn(t, s.hi), y);
        s.hi = t;
    }
    // the lane's sum as a double-fp32 value (s.hi - s.lo, exactly split)
    __device__ dd total() const { return two_sum(s.hi, -s.lo); }
    // merges another (max, sum) into this one
    __device__ void merge(float m2, dd s2, float c) {
        if (m2 == kNegInf) return;
        if (m == kNegInf) {
            m = m2;
            s = s2;
            return;
        }
        const float M = fmaxf(m, m2);
        const float f1 = warp_e(m, M, c), f2 = warp_e(m2, M, c);
        const dd a = fast_two_sum(__fmul_rn(s.hi, f1), __fmul_rn(s.lo, f1));
        const dd b = fast_two_sum(__fmul_rn(s2.hi, f2), __fmul_rn(s2.lo, f2));
        m = M;
        s = dd_add(a, b);
    }
};

// Loads element e of a row (or 0-padding past n), vectorised when possible.
__device__ __forceinline__ float4 load4(const float *row, int64_t e, int64_t end, bool vec) {
    if (vec && e + 3 < end) return ld_stream4(row + e);
    float4 x;
    const float ninf = kNegInf;
    x.x = e < end ? ld_stream1(row + e) : ninf;
    x.y = e + 1 < end ? ld_stream1(row + e + 1) : ninf;
    x.z = e + 2 < end ? ld_stream1(row + e + 2) : ninf;
    x.w = e + 3 < end ? ld_stream1(row + e + 3) : ninf;
    return x;
}

// CTA-wide (max, sum) of one or two rows' lane states.
struct RowNorm {
    float m;
    dd s;
};

// CTA-wide (max, sum) of two rows' lane states, combined in warp order.
__device__ void cta_norms(Online a, Online b, RowNorm &na, RowNorm &nb, float c, int warp,
                          int lane, RowNorm (*sh)[kLgWarps]) {
    a.s = a.total();
    b.s = b.total();
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float ma = __shfl_xor_sync(0xffffffffu, a.m, d);
        const dd sa = shfl_xor_dd(a.s, d);
        a.merge(ma, sa, c);
        const float mb = __shfl_xor_sync(0xffffffffu, b.m, d);
        const dd sb = shfl_xor_dd(b.s, d);
        b.merge(mb, sb, c);
    }
    if (lane == 0) {
        sh[0][warp] = RowNorm{a.m, a.s};
        sh[1][warp] = RowNorm{b.m, b.s};
    }
    __syncthreads();
    Online x, y;
    for (int w = 0; w < kLgWarps; ++w) {
        x.merge(sh[0][w].m, sh[0][w].s, c);
        y.merge(sh[1][w].m, sh[1][w].s, c);
    }
    na = RowNorm{x.m, x.s};
    nb = RowNorm{y.m, y.s};
    __syncthreads();  // sh is reused by the next row
}

__device__ __forceinline__ bool lg_vec(const LogitsParams &L) {
    return aligned16(L.zp) && aligned16(L.zq) && (L.ps & 3) == 0 && (L.qs & 3) == 0;
}

// This CTA's (max, sum) of its segments of row pair (a, b) (b may be null).
__device__ void row_norms(const float *a, const float *b, const LogitsParams &L, bool vec, int rank,
                          int warp, int lane, RowNorm &na, RowNorm &nb, RowNorm (*sh)[kLgWarps]) {
    Online oa, ob;
    const float4 none = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
    for (int s = rank * kLgWarps + warp; s < L.nseg; s += L.csize * kLgWarps) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t end = min(L.V, base + kSeg);
        float4 xa[kVecPerLane], xb[kVecPerLane];  // every load of the segment first
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const int64_t e = base + 4 * (lane + 32 * k);
            xa[k] = e < end ? load4(a, e, end, vec) : none;
            xb[k] = (b && e < end) ? load4(b, e, end, vec) : none;
        }
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            oa.add4(xa[k], L.c);
            if (b) ob.add4(xb[k], L.c);
        }
    }
    cta_norms(oa, ob, na, nb, L.c, warp, lane, sh);
}

// The cluster's normalisers: each CTA publishes its pair in slot[parity],
// one cluster barrier, then every CTA combines all of them in rank order.
__device__ void cluster_norms(RowNorm &na, RowNorm &nb, RowNorm (*slot)[2], int parity,
                              float c) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    if (threadIdx.x == 0) {
        slot[parity][0] = na;
        slot[parity][1] = nb;
    }
    cl.sync();
    Online x, y;
    const int C = (int)cl.num_blocks();
    for (int r = 0; r < C; ++r) {
        const RowNorm *o = cl.map_shared_rank(&slot[parity][0], r);
        const RowNorm pa = o[0], pb = o[1];
        x.merge(pa.m, pa.s, c);
        y.merge(pb.m, pb.s, c);
    }
    na = RowNorm{x.m, x.s};
    nb = RowNorm{y.m, y.s};
}

// Mass of one element: the residual max(0, p - q) of the warped rows, or p
// alone (b == null), with 1/S rounded once to fp32.
__device__ __forceinline__ float lg_mass(float za, float zb, bool pair, const RowNorm &na,
                                         const RowNorm &nb, float ia, float ib, float c) {
    const float pa = __fmul_rn(warp_e(za, na.m, c), ia);
    if (!pair) return pa;
    const float qb = __fmul_rn(warp_e(zb, nb.m, c), ib);
    return fmaxf(__fsub_rn(pa, qb), 0.f);
}

// Streams the masses of a row (pair) into segment and block sums of sequence
// bseq; warp w of `warps` takes segments w, w + warps, ...
__device__ void mass_sums(const float *a, const float *b, const LogitsParams &L, int bseq, bool vec,
                          const RowNorm &na, const RowNorm &nb, float ia, float ib, int warp,
                          int warps, int lane) {
    float2 *seg = L.seg + (int64_t)bseq * L.nseg;
    float2 *blk = L.blk + (int64_t)bseq * L.nseg * kBlocks;
    for (int s = warp; s < L.nseg; s += warps) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t end = min(L.V, base + kSeg);
        dd v[kBlocks];
        float4 xa[kBlocks], xb[kBlocks];  // every load of the segment first
#pragma unroll
        for (int k = 0; k < kBlocks; ++k) {
            const int64_t e = base + 4 * (lane + 32 * k);
            xa[k] = e < end ? load4(a, e, end, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
            xb[k] = (b && e < end) ? load4(b, e, end, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kBlocks; ++k) {
            const int64_t e = base + 4 * (lane + 32 * k);
            float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < end) {
                const float4 x = xa[k], y = xb[k];
                m.x = lg_mass(x.x, y.x, b, na, nb, ia, ib, L.c);
                m.y = e + 1 < end ? lg_mass(x.y, y.y, b, na, nb, ia, ib, L.c) : 0.f;
                m.z = e + 2 < end ? lg_mass(x.z, y.z, b, na, nb, ia, ib, L.c) : 0.f;
                m.w = e + 3 < end ? lg_mass(x.w, y.w, b, na, nb, ia, ib, L.c) : 0.f;
            }
            v[k] = dd{sum4(m), 0.f};
        }
        store_sums(seg, blk, s, v, lane);
    }
}

// Element step of the draw on a logit row (pair): the same masses, recomputed.
__device__ int lg_search_block(const float *a, const float *b, int64_t base, int64_t V,
                               const RowNorm &na, const RowNorm &nb, float ia, float ib, float c,
                               dd prefix, dd T, int lane) {
    const int64_t e0 = base + 4 * lane;
    const int64_t end = min(V, base + 128);
    float mh[4];
    int last_nz = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        mh[j] = 0.f;
        if (e0 + j < end) {
            mh[j] = lg_mass(__ldcg(a + e0 + j), b ? __ldcg(b + e0 + j) : 0.f, b, na, nb, ia, ib, c);
            if (mh[j] != 0.f) last_nz = (int)(e0 - base) + j;
        }
    }
    const dd mine = {sum4(make_float4(mh[0], mh[1], mh[2], mh[3])), 0.f};
    const dd inc = warp_incl_scan(mine, lane);
    const unsigned msk = __ballot_sync(0xffffffffu, mine.hi != 0.f && dd_gt(dd_add(prefix, inc), T));
    if (msk) {
        const int Ln = __ffs(msk) - 1;
        dd excl = shfl_up_dd(inc, 1);
        if (lane == 0) excl = {0.f, 0.f};
        int found = -1;
        if (lane == Ln) {
            dd run = dd_add(prefix, excl);
            int lastj = -1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (found < 0 && mh[j] != 0.f) {
                    lastj = j;
                    run = dd_add(run, dd{mh[j], 0.f});
                    if (dd_gt(run, T)) found = 4 * lane + j;
                }
            }
            if (found < 0) found = 4 * lane + lastj;
        }
        found = __shfl_sync(0xffffffffu, found, Ln);
        return (int)(base + found);
    }
#pragma unroll
    for (int mm = 16; mm > 0; mm >>= 1) last_nz = max(last_nz, __shfl_xor_sync(0xffffffffu, last_nz, mm));
    return last_nz < 0 ? -1 : (int)(base + last_nz);
}

__global__ void __launch_bounds__(kLgThreads, 2) logits_sample_kernel(const LogitsParams L) {
    namespace cg = cooperative_groups;
    __shared__ RowNorm sh[2][kLgWarps];
    __shared__ RowNorm slot[2][2];  // this CTA's (p, q) normaliser pair, by row parity
    __shared__ int sh_tok[kMaxK];
    __shared__ float sh_u[kMaxK];
    __shared__ int sh_bad;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / L.csize;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec = lg_vec(L);
    if (threadIdx.x == 0) sh_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < L.K; i += kLgThreads) {
        const int32_t x = L.t[(int64_t)b * L.K + i];
        sh_tok[i] = x;
        sh_u[i] = L.u_acc[(int64_t)b * L.K + i];
        if (x < 0 || (int64_t)x >= L.V) atomicOr(&sh_bad, 1);
    }
    __syncthreads();
    if (sh_bad) {  // the same verdict in every CTA of the cluster: nobody waits
        if (rank == 0 && threadIdx.x == 0) {
            atomicOr(L.status, kStatusBadToken);
            L.n_out[b] = 0;
            L.next_out[b] = -1;
        }
        return;
    }
    int n = L.K, parity = 0;
    RowNorm np, nq;
    for (int i = 0; i < L.K; ++i) {
        const float *a = L.zp + ((int64_t)b * (L.K + 1) + i) * L.ps;
        const float *c = L.zq + ((int64_t)b * L.K + i) * L.qs;
        row_norms(a, c, L, vec, rank, warp, lane, np, nq, sh);
        cluster_norms(np, nq, slot, parity, L.c);
        parity ^= 1;
        const int x = sh_tok[i];
        const float pt = __fmul_rn(warp_e(__ldg(a + x), np.m, L.c), __frcp_rn(np.s.hi));
        const float qt = __fmul_rn(warp_e(__ldg(c + x), nq.m, L.c), __frcp_rn(nq.s.hi));
        if (!accepts(sh_u[i], qt, pt)) {
            n = i;
            break;
        }
    }
    const float *a = L.zp + ((int64_t)b * (L.K + 1) + n) * L.ps;
    const float *c = n < L.K ? L.zq + ((int64_t)b * L.K + n) * L.qs : nullptr;
    if (n == L.K) {
        row_norms(a, nullptr, L, vec, rank, warp, lane, np, nq, sh);
        cluster_norms(np, nq, slot, parity, L.c);
    }
    const float ia = __frcp_rn(np.s.hi), ib = c ? __frcp_rn(nq.s.hi) : 0.f;
    mass_sums(a, c, L, b, vec, np, nq, ia, ib, rank * kLgWarps + warp, L.csize * kLgWarps, lane);
    cl.sync();  // every segment's sums are in the workspace (release / acquire)
    if (rank != 0 || warp != 0) return;
    // the draw, by warp 0 of CTA 0
    DrawInputs in = {};
    in.u = split_uniform(L.u_res[b]);
    const float2 *seg = L.seg + (int64_t)b * L.nseg;
    const float2 *blk = L.blk + (int64_t)b * L.nseg * kBlocks;
    int next = draw_core(L.nseg, L.V, seg, blk, nullptr, nullptr, in, lane,
                         [&](int64_t base, dd prefix, dd T) {
                             return lg_search_block(a, c, base, L.V, np, nq, ia, ib, L.c, prefix,
                                                    T, lane);
                         });
    if (next < 0 && c) {
        // p_n == q_n: the residual has no mass; draw from p_n (the probability
        // path's fallback)
        mass_sums(a, nullptr, L, b, vec, np, nq, ia, ib, 0, 1, lane);  // this warp alone
        __threadfence_block();
        __syncwarp();
        next = draw_core(L.nseg, L.V, seg, blk, nullptr, nullptr, in, lane,
                         [&](int64_t base, dd prefix, dd T) {
                             return lg_search_block(a, nullptr, base, L.V, np, nq, ia, ib, L.c,
                                                    prefix, T, lane);
                         });
    }
    if (lane == 0) {
        if (next < 0) atomicOr(L.status, kStatusZeroMass);
        L.n_out[b] = n;
        L.next_out[b] = next;
    }
}

}  // namespace sv
