// sv_device.cuh -- device code of the batched speculative-decoding
// verification kernels (sm_103a).
//
// One launch verifies B sequences.  The grid is B x C CTAs: CTA (b, c) owns
// chunk c of every row of sequence b, where a row of V probabilities is cut
// into 1024-element segments and a chunk is a run of consecutive segments.
// Each warp streams whole segments with 16-byte loads; no CTA ever waits on
// another.  The last CTA of a sequence to finish (atomic ticket) reads the
// per-row or per-segment partials the others left in the workspace and writes
// that sequence's (n_accepted, next_token).
//
//  * Greedy rule ("spec-verify" page, section "Method", greedy bullet): CTA
//    (b, c) walks rows 0, 1, ... of sequence b, keeping for its chunk the
//    largest value and its lowest index.  As soon as any lane has seen an
//    element that beats the draft token t_i (larger, or equal at a lower
//    index) it records "row i missed" in a per-sequence flag (atomicMax of an
//    encoding that favours smaller rows); every warp re-reads the flag before
//    each segment and every CTA before each row, so rows after the first miss
//    are not streamed.  Only comparisons are involved, so the result is exact
//    in any order.
//  * Sampling rule (same section, sampling bullet): warp 0 of every CTA
//    gathers p_i(t_i), q_i(t_i) for the K positions and finds the first
//    rejection n with the exact fp64 test u*q < p.  The CTA then streams its
//    chunk of the residual max(0, p_n - q_n) (or of p_K when all K were
//    accepted) and stores one double-fp32 sum per segment.  The last CTA scans
//    the segment sums, finds the segment where the running mass first exceeds
//    T = u_resample * total, and re-reads only that segment to locate the token.
//
// Mass sums use error-free transformations in fp32 instead of fp64 (fp64
// throughput on this part is a small fraction of fp32): each element
// p - q with p > q >= 0 is split exactly into hi + lo (Dekker's FastTwoSum on
// p and -q), each lane accumulates its 32 elements per segment with the
// Ogita-Rump-Oishi "Sum2" cascade (Knuth's TwoSum), and partials are combined
// with double-fp32 addition (Dekker).  The relative error of every prefix is
// below about 1e-11 for these non-negative terms.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSeg = 1024;                  // elements per segment (one warp task)
constexpr int kVecPerLane = kSeg / 4 / 32;  // float4 loads per lane per segment
constexpr int kMaxK = 64;
constexpr int kFlagBase = kMaxK + 1;        // miss flag stores kFlagBase - row; 0 = none

constexpr uint32_t kStatusBadToken = 1u;
constexpr uint32_t kStatusZeroMass = 2u;
constexpr uint32_t kStatusOverflow = 4u;
constexpr uint32_t kStatusBadMode = 8u;

enum Rule : int { kGreedy = 0, kSample = 1, kPerSequence = 2 };

struct Params {
    const float *p;
    int64_t ps;                 // target row stride (elements)
    const float *q;
    int64_t qs;                 // draft row stride (elements)
    const int32_t *t;           // [B][K]
    const float *u_acc;         // [B][K]
    const double *u_res;        // [B]
    const uint8_t *mode;        // [B], per-sequence rule (kPerSequence only)
    int32_t B, K;
    int64_t V;
    int32_t nseg;               // segments per row
    int32_t chunks;             // CTAs per sequence
    int32_t spc;                // segments per chunk
    int32_t *n_out;
    int32_t *next_out;
    int32_t *tokens;            // optional commit target [B][max_len]
    int32_t *lengths;
    int32_t max_len;
    // workspace
    uint32_t *status;
    uint32_t *ticket;           // [B]
    int32_t *miss;              // [B]
    unsigned long long *best;   // [B][K+1] packed (value, index) keys
    float2 *seg;                // [B][nseg] double-fp32 segment sums
};

// ---------------------------------------------------------------------------
// double-fp32 arithmetic (every operation explicitly rounded, never fused)

struct dd {
    float hi, lo;
};

__device__ __forceinline__ dd two_sum(float a, float b) {  // Knuth
    float s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ dd fast_two_sum(float a, float b) {  // Dekker, |a| >= |b|
    float s = __fadd_rn(a, b);
    float e = __fsub_rn(b, __fsub_rn(s, a));
    return {s, e};
}

__device__ __forceinline__ dd dd_add(dd x, dd y) {
    dd s = two_sum(x.hi, y.hi);
    float e = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
    return fast_two_sum(s.hi, e);
}

__device__ __forceinline__ double dd_to_double(dd x) {
    return __dadd_rn((double)x.hi, (double)x.lo);
}

__device__ __forceinline__ dd shfl_xor_dd(dd x, int m) {
    return {__shfl_xor_sync(0xffffffffu, x.hi, m), __shfl_xor_sync(0xffffffffu, x.lo, m)};
}

__device__ __forceinline__ dd shfl_up_dd(dd x, int d) {
    return {__shfl_up_sync(0xffffffffu, x.hi, d), __shfl_up_sync(0xffffffffu, x.lo, d)};
}

// Running per-lane sum of exact element masses (Sum2 cascade): s is the fp32
// running sum, c collects every rounding error and the low parts.
struct Acc {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float hi, float lo) {
        dd t = two_sum(s, hi);
        s = t.hi;
        c = __fadd_rn(c, __fadd_rn(t.lo, lo));
    }
    __device__ __forceinline__ dd value() const { return fast_two_sum(s, c); }
};

// Exact residual mass of one element: max(0, p - q) as hi + lo.  For
// p > q >= 0, |p| >= |q|, so FastTwoSum(p, -q) is exact.  With kResidual
// false the mass is p itself (bonus draw and the zero-residual fallback).
template <bool kResidual>
__device__ __forceinline__ void elem_mass(float p, float q, float &hi, float &lo) {
    if (kResidual) {
        float d = __fsub_rn(p, q);
        float e = __fsub_rn(__fsub_rn(p, d), q);
        bool pos = p > q;
        hi = pos ? d : 0.f;
        lo = pos ? e : 0.f;
    } else {
        hi = p;
        lo = 0.f;
    }
}

// ---------------------------------------------------------------------------
// memory helpers

__device__ __forceinline__ float4 ld_stream4(const float *ptr) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(ptr));
    return v;
}

__device__ __forceinline__ float ld_stream1(const float *ptr) {
    float v;
    asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

// Loads that must see other CTAs' writes of this launch (L2, never L1).
template <class T>
__device__ __forceinline__ T ld_l2(const T *ptr) {
    return __ldcg(ptr);
}

__device__ __forceinline__ bool aligned16(const float *ptr) {
    return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

// Order-preserving 32-bit code of a float (-0 folded onto +0), so that
// unsigned comparison matches float comparison for non-NaN values.
__device__ __forceinline__ uint32_t ordered_bits(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value, index) packed so that a larger key is a larger value, or an equal
// value at a lower index; 0 means "no element".
__device__ __forceinline__ unsigned long long pack_key(float v, int32_t idx) {
    if (idx < 0) return 0ull;
    return ((unsigned long long)ordered_bits(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ int32_t key_index(unsigned long long key) {
    return (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        unsigned long long o = __shfl_xor_sync(0xffffffffu, k, m);
        k = o > k ? o : k;
    }
    return k;
}

// ---------------------------------------------------------------------------
// shared state of one CTA

struct Shared {
    int32_t tok[kMaxK];
    int32_t n;
    int32_t bad;
    int32_t flag;
    int32_t is_last;
    int32_t cand;
    int32_t pick;
    int32_t zero;
    unsigned long long wkey[kWarps];
    dd wsum[kWarps];
    dd base;
};

__device__ __forceinline__ const float *prow(const Params &P, int b, int i) {
    return P.p + ((int64_t)b * (P.K + 1) + i) * P.ps;
}

__device__ __forceinline__ const float *qrow(const Params &P, int b, int i) {
    return P.q + ((int64_t)b * P.K + i) * P.qs;
}

// Loads t[b][0..K) into shared memory and flags out-of-range ids.
__device__ __forceinline__ void load_tokens(const Params &P, int b, Shared &sh) {
    if (threadIdx.x == 0) sh.bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < P.K; i += kThreads) {
        int32_t x = P.t[(int64_t)b * P.K + i];
        sh.tok[i] = x;
        if (x < 0 || (int64_t)x >= P.V) sh.bad = 1;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// greedy: argmax of one segment, lane view

__device__ __forceinline__ void take(float x, int32_t e, float &bv, int32_t &bi) {
    if (x > bv) {  // strict: within a lane indices only increase
        bv = x;
        bi = e;
    }
}

__device__ __forceinline__ void argmax_segment(const float *row, int64_t base, int64_t V,
                                               bool vec, int lane, float &bv, int32_t &bi) {
    if (vec && base + kSeg <= V) {
        float4 x[kVecPerLane];
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) x[k] = ld_stream4(row + base + 4 * (lane + 32 * k));
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            int32_t e = (int32_t)(base + 4 * (lane + 32 * k));
            take(x[k].x, e, bv, bi);
            take(x[k].y, e + 1, bv, bi);
            take(x[k].z, e + 2, bv, bi);
            take(x[k].w, e + 3, bv, bi);
        }
    } else {
        int64_t end = base + kSeg < V ? base + kSeg : V;
        for (int64_t e0 = base; e0 < end; e0 += 32 * 8) {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int64_t e = e0 + lane + 32 * j;
                x[j] = e < end ? ld_stream1(row + e) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int64_t e = e0 + lane + 32 * j;
                if (e < end) take(x[j], (int32_t)e, bv, bi);
            }
        }
    }
}

__device__ void greedy_body(const Params &P, int b, int c, Shared &sh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    load_tokens(P, b, sh);
    if (sh.bad) return;
    const int s_lo = c * P.spc;
    const int s_hi = min(P.nseg, s_lo + P.spc);
    for (int i = 0; i <= P.K; ++i) {
        if (threadIdx.x == 0) sh.flag = ld_l2(P.miss + b);
        __syncthreads();
        const int flag = sh.flag;
        __syncthreads();
        if (flag > kFlagBase - i) break;  // an earlier row already missed
        const float *row = prow(P, b, i);
        const bool vec = aligned16(row);
        const bool has_t = i < P.K;
        const int32_t ti = has_t ? sh.tok[i] : -1;
        const float pt = has_t ? __ldg(row + ti) : 0.f;
        bool signalled = !has_t;
        float bv = -__int_as_float(0x7f800000);  // -inf
        int32_t bi = -1;
        for (int s = s_lo + warp; s < s_hi; s += kWarps) {
            if (s != s_lo + warp) {
                int f = 0;
                if (lane == 0) f = ld_l2(P.miss + b);
                f = __shfl_sync(0xffffffffu, f, 0);
                if (f > kFlagBase - i) break;
            }
            argmax_segment(row, (int64_t)s * kSeg, P.V, vec, lane, bv, bi);
            if (!signalled) {
                bool beats = bi >= 0 && (bv > pt || (bv == pt && bi < ti));
                if (__any_sync(0xffffffffu, beats)) {
                    if (lane == 0) atomicMax(P.miss + b, kFlagBase - i);
                    signalled = true;
                }
            }
        }
        unsigned long long key = warp_max_u64(pack_key(bv, bi));
        if (lane == 0) sh.wkey[warp] = key;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long k = sh.wkey[0];
            for (int w = 1; w < kWarps; ++w) k = sh.wkey[w] > k ? sh.wkey[w] : k;
            if (k) atomicMax(P.best + (int64_t)b * (P.K + 1) + i, k);
        }
        // the next iteration's leading barrier orders sh.wkey reuse
    }
}

// ---------------------------------------------------------------------------
// sampling: accept scan (warp 0) and residual segment sums

__device__ void accept_scan(const Params &P, int b, Shared &sh) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int n = P.K;
        bool bad = false;
        for (int i0 = 0; i0 < P.K; i0 += 32) {
            const int i = i0 + lane;
            bool rej = false;
            if (i < P.K) {
                const int32_t x = P.t[(int64_t)b * P.K + i];
                if (x < 0 || (int64_t)x >= P.V) {
                    bad = true;
                } else {
                    const float pt = __ldg(prow(P, b, i) + x);
                    const float qt = __ldg(qrow(P, b, i) + x);
                    const float u = __ldg(P.u_acc + (int64_t)b * P.K + i);
                    // exact: the fp64 product of two fp32 values is exact
                    rej = !(__dmul_rn((double)u, (double)qt) < (double)pt);
                }
            }
            unsigned m = __ballot_sync(0xffffffffu, rej);
            if (m && n == P.K) n = i0 + __ffs(m) - 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            sh.n = n;
            sh.bad = bad ? 1 : 0;
        }
    }
    __syncthreads();
}

// Sum of one segment's masses (lane-strided 16-byte loads); every lane gets
// the warp total.
template <bool kResidual>
__device__ __forceinline__ dd segment_sum(const float *pr, const float *qr, int64_t base,
                                          int64_t V, bool vec, int lane) {
    Acc acc;
    if (vec && base + kSeg <= V) {
        float4 a[kVecPerLane], d[kVecPerLane];
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            a[k] = ld_stream4(pr + base + 4 * (lane + 32 * k));
            if (kResidual) d[k] = ld_stream4(qr + base + 4 * (lane + 32 * k));
        }
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            float hi, lo;
            float4 qq = kResidual ? d[k] : make_float4(0.f, 0.f, 0.f, 0.f);
            elem_mass<kResidual>(a[k].x, qq.x, hi, lo); acc.add(hi, lo);
            elem_mass<kResidual>(a[k].y, qq.y, hi, lo); acc.add(hi, lo);
            elem_mass<kResidual>(a[k].z, qq.z, hi, lo); acc.add(hi, lo);
            elem_mass<kResidual>(a[k].w, qq.w, hi, lo); acc.add(hi, lo);
        }
    } else {
        int64_t end = base + kSeg < V ? base + kSeg : V;
        for (int64_t e = base + lane; e < end; e += 32) {
            float hi, lo;
            elem_mass<kResidual>(ld_stream1(pr + e), kResidual ? ld_stream1(qr + e) : 0.f, hi, lo);
            acc.add(hi, lo);
        }
    }
    dd v = acc.value();
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = dd_add(v, shfl_xor_dd(v, m));
    return v;
}

// Segment sums of segments [s_lo, s_hi) of one row, warp-strided, stored to
// seg[] by lane 0 of the warp that computed them.
template <bool kResidual>
__device__ void stream_segments(const Params &P, const float *pr, const float *qr, float2 *seg,
                                int s_lo, int s_hi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec = aligned16(pr) && (!kResidual || aligned16(qr));
    for (int s = s_lo + warp; s < s_hi; s += kWarps) {
        dd v = segment_sum<kResidual>(pr, qr, (int64_t)s * kSeg, P.V, vec, lane);
        if (lane == 0) seg[s] = make_float2(v.hi, v.lo);
    }
}

__device__ void sample_body(const Params &P, int b, int c, Shared &sh) {
    accept_scan(P, b, sh);
    if (sh.bad) return;
    const int n = sh.n;
    const int s_lo = c * P.spc;
    const int s_hi = min(P.nseg, s_lo + P.spc);
    float2 *seg = P.seg + (int64_t)b * P.nseg;
    if (n < P.K)
        stream_segments<true>(P, prow(P, b, n), qrow(P, b, n), seg, s_lo, s_hi);
    else
        stream_segments<false>(P, prow(P, b, P.K), nullptr, seg, s_lo, s_hi);
    __threadfence();  // segment sums visible before this CTA's ticket
}

// ---------------------------------------------------------------------------
// block-wide helpers for the deciding CTA

// Exclusive scan of one dd per thread (thread order); total to *total.
__device__ dd block_excl_scan(dd v, dd *total, Shared &sh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    dd inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        dd o = shfl_up_dd(inc, d);
        if (lane >= d) inc = dd_add(o, inc);
    }
    if (lane == 31) sh.wsum[warp] = inc;
    __syncthreads();
    dd wbase = {0.f, 0.f}, all = {0.f, 0.f};
    for (int w = 0; w < kWarps; ++w) {
        if (w == warp) wbase = all;
        all = dd_add(all, sh.wsum[w]);
    }
    __syncthreads();
    *total = all;
    dd lane_excl = shfl_up_dd(inc, 1);
    if (lane == 0) lane_excl = {0.f, 0.f};
    return dd_add(wbase, lane_excl);
}

__device__ int block_min_int(int v, Shared &sh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, m));
    if (lane == 0) sh.wkey[warp] = (unsigned long long)(uint32_t)v;
    __syncthreads();
    int r = (int)(uint32_t)sh.wkey[0];
    for (int w = 1; w < kWarps; ++w) r = min(r, (int)(uint32_t)sh.wkey[w]);
    __syncthreads();
    return r;
}

__device__ int block_max_int(int v, Shared &sh) {
    return -block_min_int(-v, sh);
}

// Rescans one segment with lane-contiguous 32-element blocks (warp 0 only):
// returns the smallest index v in it whose running mass base + C_v exceeds T,
// or the last index with non-zero mass if none does (a rounding boundary), or
// -1 if the segment has no mass.
template <bool kResidual>
__device__ int rescan_segment(const float *pr, const float *qr, int64_t base, int64_t V,
                              dd prefix, double T) {
    const int lane = threadIdx.x & 31;
    const int64_t lo = base + 32 * lane;
    const int64_t hi = lo + 32 < V ? lo + 32 : V;
    const int64_t seg_end = base + kSeg < V ? base + kSeg : V;
    float mh[32], ml[32];
    Acc acc;
    int last_nz = -1;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int64_t e = lo + j;
        float pv = 0.f, qv = 0.f;
        if (e < hi) {
            pv = __ldcg(pr + e);
            if (kResidual) qv = __ldcg(qr + e);
        }
        elem_mass<kResidual>(pv, qv, mh[j], ml[j]);
        if (e >= hi) mh[j] = ml[j] = 0.f;
        if (mh[j] != 0.f) last_nz = (int)(e - base);
        acc.add(mh[j], ml[j]);
    }
    (void)seg_end;
    dd mine = acc.value();
    // lane-exclusive prefix within the segment
    dd inc = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        dd o = shfl_up_dd(inc, d);
        if (lane >= d) inc = dd_add(o, inc);
    }
    dd excl = shfl_up_dd(inc, 1);
    if (lane == 0) excl = {0.f, 0.f};
    dd start = dd_add(prefix, excl);
    dd end = dd_add(prefix, inc);
    const bool crosses = mine.hi != 0.f && dd_to_double(end) > T;
    const unsigned m = __ballot_sync(0xffffffffu, crosses);
    int pick = -1;
    if (m) {
        const int L = __ffs(m) - 1;
        int found = -1;
        if (lane == L) {
            dd run = start;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (found < 0 && mh[j] != 0.f) {
                    run = dd_add(run, fast_two_sum(mh[j], ml[j]));
                    if (dd_to_double(run) > T) found = (int)(lo + j - base);
                }
            }
            if (found < 0) found = last_nz;  // lane total crossed but steps did not
        }
        pick = __shfl_sync(0xffffffffu, found, L);
    } else {
        int l = last_nz;
#pragma unroll
        for (int mm = 16; mm > 0; mm >>= 1) l = max(l, __shfl_xor_sync(0xffffffffu, l, mm));
        pick = l;
    }
    return pick < 0 ? -1 : (int)(base + pick);
}

// Inverse-CDF draw over the segment sums seg[0..nseg) of the row pair
// (pr, qr): returns the token, or -1 if the total mass is zero.
template <bool kResidual>
__device__ int draw_from_segments(const Params &P, const float2 *seg, const float *pr,
                                  const float *qr, double u, Shared &sh) {
    const int per = (P.nseg + kThreads - 1) / kThreads;
    const int r0 = min(P.nseg, (int)threadIdx.x * per);
    const int r1 = min(P.nseg, r0 + per);
    dd run = {0.f, 0.f};
    for (int s = r0; s < r1; ++s) {
        float2 v = ld_l2(seg + s);
        run = dd_add(run, dd{v.x, v.y});
    }
    dd total;
    dd excl = block_excl_scan(run, &total, sh);
    if (total.hi == 0.f) return -1;
    const double T = __dmul_rn(u, dd_to_double(total));
    int cand = 0x7fffffff;
    dd acc = excl;
    for (int s = r0; s < r1; ++s) {
        float2 v = ld_l2(seg + s);
        dd nxt = dd_add(acc, dd{v.x, v.y});
        if (v.x != 0.f && dd_to_double(nxt) > T) {
            cand = s;
            break;
        }
        acc = nxt;
    }
    const int first = block_min_int(cand, sh);
    if (first == cand && cand != 0x7fffffff) sh.base = acc;  // prefix before segment `first`
    int target = first;
    if (first == 0x7fffffff) {
        // T reached the total through rounding: the last segment with mass
        int lastnz = -1;
        for (int s = r0; s < r1; ++s)
            if (ld_l2(seg + s).x != 0.f) lastnz = s;
        target = block_max_int(lastnz, sh);
        if (threadIdx.x == 0) sh.base = dd{0.f, 0.f};
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // for the rounding fallback, T' = +inf forces "last non-zero element"
        const double Tt = first == 0x7fffffff ? __longlong_as_double(0x7ff0000000000000ll) : T;
        int j = rescan_segment<kResidual>(pr, qr, (int64_t)target * kSeg, P.V, sh.base, Tt);
        if (threadIdx.x == 0) sh.pick = j;
    }
    __syncthreads();
    return sh.pick;
}

// ---------------------------------------------------------------------------
// decisions of the last CTA of a sequence

__device__ void commit_round(const Params &P, int b, int n, int next, Shared &sh) {
    if (!P.tokens || next < 0) return;
    if (threadIdx.x == 0) {
        const int len = P.lengths[b];
        const bool ok = len >= 0 && (int64_t)len + n + 1 <= P.max_len;
        sh.flag = ok ? len : -1;
        if (!ok) atomicOr(P.status, kStatusOverflow);
    }
    __syncthreads();
    const int len = sh.flag;
    if (len >= 0) {
        int32_t *row = P.tokens + (int64_t)b * P.max_len;
        for (int i = threadIdx.x; i < n; i += kThreads) row[len + i] = P.t[(int64_t)b * P.K + i];
        if (threadIdx.x == 0) {
            row[len + n] = next;
            P.lengths[b] = len + n + 1;
        }
    }
}

__device__ void greedy_decide(const Params &P, int b, Shared &sh) {
    int n = 0, next = -1;
    if (!sh.bad) {
        const int f = ld_l2(P.miss + b);
        n = f ? kFlagBase - f : P.K;
        const unsigned long long key = ld_l2(P.best + (int64_t)b * (P.K + 1) + n);
        next = key ? key_index(key) : 0;
    }
    if (threadIdx.x == 0) {
        if (sh.bad) atomicOr(P.status, kStatusBadToken);
        P.n_out[b] = n;
        P.next_out[b] = next;
        P.miss[b] = 0;
    }
    for (int i = threadIdx.x; i <= P.K; i += kThreads) P.best[(int64_t)b * (P.K + 1) + i] = 0ull;
    commit_round(P, b, n, next, sh);
}

__device__ void sample_decide(const Params &P, int b, Shared &sh) {
    int n = 0, next = -1;
    if (!sh.bad) {
        n = sh.n;
        const double u = P.u_res[b];
        float2 *seg = P.seg + (int64_t)b * P.nseg;
        if (n < P.K) {
            next = draw_from_segments<true>(P, seg, prow(P, b, n), qrow(P, b, n), u, sh);
            if (next < 0) {
                // zero residual mass (unnormalised rows): draw from p_n itself
                __syncthreads();
                stream_segments<false>(P, prow(P, b, n), nullptr, seg, 0, P.nseg);
                __threadfence_block();
                __syncthreads();
                next = draw_from_segments<false>(P, seg, prow(P, b, n), nullptr, u, sh);
            }
        } else {
            next = draw_from_segments<false>(P, seg, prow(P, b, P.K), nullptr, u, sh);
        }
    }
    if (threadIdx.x == 0) {
        if (sh.bad) atomicOr(P.status, kStatusBadToken);
        else if (next < 0) atomicOr(P.status, kStatusZeroMass);
        P.n_out[b] = sh.bad ? 0 : n;
        P.next_out[b] = next;
    }
    commit_round(P, b, sh.bad ? 0 : n, next, sh);
}

// Returns true in every thread of the CTA that arrives last for sequence b.
__device__ __forceinline__ bool arrive_last(const Params &P, int b, Shared &sh) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(P.ticket + b, 1u);
        sh.is_last = prev == (uint32_t)(P.chunks - 1);
        if (sh.is_last) __threadfence();
    }
    __syncthreads();
    return sh.is_last != 0;
}

template <int kRule>
__global__ void __launch_bounds__(kThreads) verify_kernel(const Params P) {
    __shared__ Shared sh;
    const int b = blockIdx.x / P.chunks;
    const int c = blockIdx.x - b * P.chunks;
    const int rule = kRule == kPerSequence ? (int)P.mode[b] : kRule;
    if (rule == kGreedy) greedy_body(P, b, c, sh);
    else if (rule == kSample) sample_body(P, b, c, sh);
    if (!arrive_last(P, b, sh)) return;
    if (rule == kGreedy) {
        greedy_decide(P, b, sh);
    } else if (rule == kSample) {
        sample_decide(P, b, sh);
    } else if (threadIdx.x == 0) {
        atomicOr(P.status, kStatusBadMode);
        P.n_out[b] = 0;
        P.next_out[b] = -1;
    }
    if (threadIdx.x == 0) P.ticket[b] = 0u;
}

}  // namespace sv
