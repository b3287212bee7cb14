// sv_device.cuh -- device code of the batched speculative-decoding
// verification kernels (sm_103a): the arithmetic and helpers every path
// shares, and the plain-load path.
//
// A row of V probabilities is cut into 1024-element segments, each made of
// eight 128-element blocks.  Two launch paths give identical outputs:
//  * sv_item.cuh: one persistent launch over (sequence, chunk) items, rows
//    moved into shared memory by bulk copies (16-byte aligned device rows);
//  * this file: scan -> plain-load stream -> decide (any alignment, and rows
//    in page-locked host memory).
// In the three-launch chain the scan kernel caches per-sequence data (the
// first rejection n of a sampling sequence; the draft tokens and p_i(t_i) of
// a greedy one), the stream kernel's warps take the batch's segments in turn
// and leave partials in the workspace, and the decide kernel, a programmatic
// dependent, turns them into (n_accepted, next_token).
//
//  * Greedy rule ("spec-verify" page, section "Method", greedy bullet): a
//    segment of row i is reduced to its largest value and lowest index.  An
//    element that beats the draft token t_i (larger, or equal at a lower
//    index) records "row i missed" in a per-sequence flag (atomicMax of an
//    encoding that favours smaller rows); streaming stops after the first row
//    known to have missed.  Row maxima go into per-row 64-bit keys with
//    atomicMax.  Only comparisons are involved, so the result is exact in any
//    order.
//  * Sampling rule (same section, sampling bullet): the first rejection n
//    comes from a lane-parallel gather of p_i(t_i), q_i(t_i) and the exact
//    test u*q < p (`accepts`).  The residual max(0, p_n - q_n), or p_K when all K
//    were accepted, is streamed once and leaves a double-fp32 sum per segment
//    and per block.  The draw finds the segment where the running mass first
//    exceeds T = u_resample * total, then the block within it, then re-reads
//    that one block to locate the token.
//
// Mass sums use error-free transformations in fp32 instead of fp64 (fp64
// throughput on this part is a small fraction of fp32).  Each residual
// max(0, p - q) is exact as hi + lo: FastTwoSum(max(p, q), -q) (Dekker), with
// max(p, q) >= q >= 0.  Four consecutive masses are added with a packed
// fp32x2 TwoSum tree that keeps every rounding error; lanes' block partials
// are combined with double-fp32 addition.  The relative error of any prefix
// is below about 1e-11 for these non-negative terms.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSeg = 1024;                  // elements per segment (one item)
constexpr int kVecPerLane = kSeg / 4 / 32;  // float4 loads per lane per segment row
constexpr int kBlocks = kSeg / 128;         // 128-element blocks per segment
constexpr int kMaxK = 64;
constexpr int kFlagBase = kMaxK + 1;        // miss flag stores kFlagBase - row; 0 = none
constexpr int32_t kNBad = 0x7fffffff;       // cached n: 0 unknown, n + 1, or kNBad

// Occupancy targets (CTAs per SM the register budget must allow) and how many
// 16-byte loads per row a lane keeps in flight in the sampling stream.
#ifndef SV_MIN_CTAS_PER_SM
#define SV_MIN_CTAS_PER_SM 4
#endif
#ifndef SV_GREEDY_MIN_CTAS_PER_SM
#define SV_GREEDY_MIN_CTAS_PER_SM 5
#endif
#ifndef SV_SAMPLE_BATCH
#define SV_SAMPLE_BATCH 4
#endif
constexpr int kSampleBatch = SV_SAMPLE_BATCH;
static_assert(kVecPerLane % kSampleBatch == 0, "batch must divide the per-lane loads");

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
    int32_t nseg;               // segments per row = items per sequence
    int32_t items;              // B * nseg
    int32_t warps;              // warps in the stream kernel's grid
    int32_t *n_out;
    int32_t *next_out;
    int32_t *tokens;            // optional commit target [B][max_len]
    int32_t *lengths;
    int32_t max_len;
    int32_t rows_on_host;       // host side: p or q is page-locked host memory
    int32_t ichunks;            // item kernel: items (chunks) per sequence
    int32_t isegs;              // item kernel: segments per big item
    int32_t ibig;               // item kernel: big items per sequence (the first ones of its row)
    int32_t itail;              // item kernel: segments per small item (the rest of the row), 0: none
    // workspace
    uint32_t *status;
    uint32_t *queue;            // item kernel: next item to hand out, and exited CTAs
    int32_t *miss;              // [B] greedy: kFlagBase - first missed row
    int32_t *nstate;            // [B] first rejection + 1 (sampling), 1 (greedy), kNBad
    int32_t *done;              // [B] item kernel: items of the sequence retired this round
    float *ptok;                // [B][K] greedy: p_i(t_i)
    unsigned long long *best;   // [B][K+1] packed (value, index) keys
    float2 *seg;                // [B][nseg] double-fp32 segment sums
    float2 *blk;                // [B][nseg][kBlocks] double-fp32 128-element block sums
    float2 *udd;                // [B] u_resample split into two fp32 parts
    int2 *order;                // [B] item kernel, mixed rounds: {sequence, mode} in the
                                // order sequences are taken (greedy ones first)
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

__device__ __forceinline__ dd shfl_dd(dd x, int src) {
    return {__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}

__device__ __forceinline__ dd shfl_xor_dd(dd x, int m) {
    return {__shfl_xor_sync(0xffffffffu, x.hi, m), __shfl_xor_sync(0xffffffffu, x.lo, m)};
}

__device__ __forceinline__ dd shfl_up_dd(dd x, int d) {
    return {__shfl_up_sync(0xffffffffu, x.hi, d), __shfl_up_sync(0xffffffffu, x.lo, d)};
}

// Inclusive warp scan in lane order.
template <int kWidth = 32>  // scans lanes [0, kWidth) (lanes past it get partial sums)
__device__ __forceinline__ dd warp_incl_scan(dd v, int lane) {
#pragma unroll
    for (int d = 1; d < kWidth; d <<= 1) {
        dd o = shfl_up_dd(v, d);
        if (lane >= d) v = dd_add(o, v);
    }
    return v;
}

// Packed pairs of fp32 values in one 64-bit register, and Blackwell's packed
// fp32x2 add/subtract (two results per instruction, each correctly rounded).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float a, float b) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ void unpack2(f32x2 x, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Exact sum of the masses of four consecutive elements as a double-fp32
// pair.  Residual masses max(0, p - q) come out exactly as hi + lo from
// FastTwoSum(max(p, q), -q) -- exact because max(p, q) >= q >= 0, and exactly
// zero when p <= q, so no compare or select is needed.  The four (hi, lo)
// values are then added with a packed TwoSum tree ((x + y), (z + w)) and one
// scalar TwoSum, every rounding error kept.
template <bool kResidual>
__device__ __forceinline__ dd quad_mass(float4 p, float4 q) {
    f32x2 ha, hb, la, lb;
    if (kResidual) {
        const f32x2 ma = pack2(fmaxf(p.x, q.x), fmaxf(p.z, q.z));
        const f32x2 mb = pack2(fmaxf(p.y, q.y), fmaxf(p.w, q.w));
        const f32x2 qa = pack2(q.x, q.z), qb = pack2(q.y, q.w);
        ha = sub2(ma, qa);
        la = sub2(sub2(ma, ha), qa);
        hb = sub2(mb, qb);
        lb = sub2(sub2(mb, hb), qb);
    } else {
        ha = pack2(p.x, p.z);
        hb = pack2(p.y, p.w);
        la = lb = 0ull;
    }
    // packed TwoSum: (x + y, z + w) and its rounding errors
    const f32x2 sum = add2(ha, hb);
    const f32x2 bb = sub2(sum, ha);
    const f32x2 err = add2(sub2(ha, sub2(sum, bb)), sub2(hb, bb));
    const f32x2 low = kResidual ? add2(add2(la, lb), err) : err;
    float s1, s2, c1, c2;
    unpack2(sum, s1, s2);
    unpack2(low, c1, c2);
    const dd t = two_sum(s1, s2);
    return fast_two_sum(t.hi, __fadd_rn(t.lo, __fadd_rn(c1, c2)));
}

// Reduce-scatter of eight per-lane block partials v[k] (k = 128-element
// block of the segment): afterwards lane l holds the warp total of block
// bk(l) = 4 * bit4(l) + 2 * bit3(l) + bit2(l) (lanes with l % 4 == 0 hold the
// eight blocks), and every lane holds the segment total.  12 double-fp32
// additions instead of 40 for eight separate warp reductions.
__device__ __forceinline__ void reduce_blocks(const dd v[kBlocks], int lane, dd &blk, int &bk,
                                              dd &total) {
    const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
    dd a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const dd send = h4 ? v[j] : v[j + 4];
        const dd keep = h4 ? v[j + 4] : v[j];
        a[j] = dd_add(keep, shfl_xor_dd(send, 16));
    }
    dd c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const dd send = h3 ? a[j] : a[j + 2];
        const dd keep = h3 ? a[j + 2] : a[j];
        c[j] = dd_add(keep, shfl_xor_dd(send, 8));
    }
    dd x = dd_add(h2 ? c[1] : c[0], shfl_xor_dd(h2 ? c[0] : c[1], 4));
    x = dd_add(x, shfl_xor_dd(x, 2));
    x = dd_add(x, shfl_xor_dd(x, 1));
    blk = x;
    bk = (h4 ? 4 : 0) + (h3 ? 2 : 0) + (h2 ? 1 : 0);
    dd t = dd_add(x, shfl_xor_dd(x, 4));
    t = dd_add(t, shfl_xor_dd(t, 8));
    total = dd_add(t, shfl_xor_dd(t, 16));
}

// Stores segment s's total and its eight block totals.
__device__ __forceinline__ void store_sums(float2 *seg, float2 *blk, int64_t s, const dd v[kBlocks],
                                           int lane) {
    dd b, total;
    int bk;
    reduce_blocks(v, lane, b, bk, total);
    if ((lane & 3) == 0) blk[s * kBlocks + bk] = make_float2(b.hi, b.lo);
    if (lane == 0) seg[s] = make_float2(total.hi, total.lo);
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

// Exact residual mass of one element: max(0, p - q) as hi + lo, computed as
// FastTwoSum(max(p, q), -q) -- exact since max(p, q) >= q >= 0, and exactly
// zero when p <= q.  With kResidual false the mass is p itself (bonus draw and
// the zero-residual fallback).
template <bool kResidual>
__device__ __forceinline__ void elem_mass(float p, float q, float &hi, float &lo) {
    if (kResidual) {
        const float m = fmaxf(p, q);
        hi = __fsub_rn(m, q);
        lo = __fsub_rn(__fsub_rn(m, hi), q);
    } else {
        hi = p;
        lo = 0.f;
    }
}

// ---------------------------------------------------------------------------
// mbarrier, bulk-copy and timing primitives (inline PTX)

constexpr uint32_t kStatusTimeout = 16u;
constexpr uint64_t kWaitLimitNs = 250000000ull;  // any single wait gives up after 250 ms

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One try: the thread may sleep in it for up to kTrySuspendNs and is woken
// as soon as the phase completes, so a waiting warp issues a few instructions
// per wait instead of spinning.
constexpr uint32_t kTrySuspendNs = 1000000u;

__device__ __forceinline__ bool mbar_try(unsigned long long *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kTrySuspendNs)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete, for at most
// kWaitLimitNs of wall-clock time.  The clock is read only once a first try
// has failed: a phase that is already complete costs one try_wait.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Idle-wait bookkeeping for polls of shared state: idle(ns) sleeps about ns
// and returns false once no progress has been made for kWaitLimitNs.
struct IdleClock {
    uint64_t since = 0;
    __device__ void progress() { since = 0; }
    __device__ bool idle(uint32_t ns = 128) {
        const uint64_t now = global_ns();
        if (since == 0) since = now;
        if (now - since > kWaitLimitNs) return false;
        __nanosleep(ns);
        return true;
    }
};

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

// Loads that must see other warps' writes of this launch (L2, never L1).
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
    return ((unsigned long long)ordered_bits(v) << 32) |
           (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
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

__device__ __forceinline__ const float *prow(const Params &P, int b, int i) {
    return P.p + ((int64_t)b * (P.K + 1) + i) * P.ps;
}

__device__ __forceinline__ const float *qrow(const Params &P, int b, int i) {
    return P.q + ((int64_t)b * P.K + i) * P.qs;
}

// Draft tokens of sequence b in two per-lane registers (positions lane and
// lane + 32); returns true in every lane if one of them is outside [0, V).
__device__ __forceinline__ bool load_tokens(const Params &P, int b, int lane, int32_t &t0,
                                            int32_t &t1) {
    const int32_t *tb = P.t + (int64_t)b * P.K;
    t0 = lane < P.K ? tb[lane] : 0;
    t1 = lane + 32 < P.K ? tb[lane + 32] : 0;
    bool bad = (lane < P.K && (t0 < 0 || (int64_t)t0 >= P.V)) ||
               (lane + 32 < P.K && (t1 < 0 || (int64_t)t1 >= P.V));
    return __any_sync(0xffffffffu, bad);
}

// ---------------------------------------------------------------------------
// greedy item: argmax of segment s over rows 0, 1, ... of sequence b

__device__ __forceinline__ void take(float x, int32_t e, float &bv, int32_t &bi) {
    if (x > bv) {  // strict: within a lane indices only increase
        bv = x;
        bi = e;
    }
}

__device__ __forceinline__ void argmax_segment(const float *row, int64_t base, int64_t V,
                                               int lane, float &bv, int32_t &bi) {
    if (aligned16(row) && base + kSeg <= V) {
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

__device__ void greedy_item(const Params &P, int b, int s, int lane) {
    int32_t t0, t1;
    if (load_tokens(P, b, lane, t0, t1)) return;  // the decide kernel reports it
    const float pt0 = lane < P.K ? __ldg(prow(P, b, lane) + t0) : 0.f;
    const float pt1 = lane + 32 < P.K ? __ldg(prow(P, b, lane + 32) + t1) : 0.f;
    const int64_t base = (int64_t)s * kSeg;
    for (int i = 0; i <= P.K; ++i) {
        int f = 0;
        if (lane == 0) f = ld_l2(P.miss + b);  // waited for only after the row's loads
        float bv = -__int_as_float(0x7f800000);  // -inf
        int32_t bi = -1;
        argmax_segment(prow(P, b, i), base, P.V, lane, bv, bi);
        bool missed = false;
        if (i < P.K) {
            const float pti = __shfl_sync(0xffffffffu, i < 32 ? pt0 : pt1, i & 31);
            const int32_t ti = __shfl_sync(0xffffffffu, i < 32 ? t0 : t1, i & 31);
            const bool beats = bi >= 0 && (bv > pti || (bv == pti && bi < ti));
            missed = __any_sync(0xffffffffu, beats);
            if (missed && lane == 0) atomicMax(P.miss + b, kFlagBase - i);
        }
        const unsigned long long key = warp_max_u64(pack_key(bv, bi));
        if (lane == 0 && key) atomicMax(P.best + (int64_t)b * (P.K + 1) + i, key);
        f = __shfl_sync(0xffffffffu, f, 0);
        if (missed || f >= kFlagBase - i) break;  // a row <= i missed: no later row is needed
    }
}

// ---------------------------------------------------------------------------
// sampling item: first rejection n, then one segment of the draw distribution

// First rejection of sequence b as n + 1 (n = K when all K are accepted), or
// kNBad when a draft id is outside [0, V): a lane-parallel gather of
// p_i(t_i), q_i(t_i) and the exact accept test for every position.
// The accept test u * q < p, decided exactly (the product of two fp32 values
// is exact in fp64, which is how the test is defined).  fmaf(-u, q, p) rounds
// p - u*q once, and a rounding never changes the sign of a nonzero value, so
// a nonzero result decides alone; only a zero result -- p equal to the exact
// product, or a difference below half the smallest subnormal -- needs the
// fp64 comparison, whose pipe is slow on this part.
__device__ __forceinline__ bool accepts(float u, float q, float p) {
    const float r = __fmaf_rn(-u, q, p);
    if (r != 0.f) return r > 0.f;
    return __dmul_rn((double)u, (double)q) < (double)p;
}

__device__ int32_t first_rejection(const Params &P, int b, int lane) {
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
                rej = !accepts(u, qt, pt);
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (m && n == P.K) n = i0 + __ffs(m) - 1;
    }
    return __any_sync(0xffffffffu, bad) ? kNBad : n + 1;
}

// Masses of one segment (lane-strided 16-byte loads), summed per lane and per
// 128-element block: lane l's k-th float4 holds elements 128k + 4l .. +3, and
// on the scalar path its j-th element is 32j + l, in block j / 4.
template <bool kResidual>
__device__ __forceinline__ void segment_partials(const float *pr, const float *qr, int64_t base,
                                                 int64_t V, int lane, dd v[kBlocks]) {
    if (aligned16(pr) && (!kResidual || aligned16(qr)) && base + kSeg <= V) {
#pragma unroll
        for (int h = 0; h < kVecPerLane; h += kSampleBatch) {
            float4 a[kSampleBatch], d[kSampleBatch];
#pragma unroll
            for (int k = 0; k < kSampleBatch; ++k) {
                a[k] = ld_stream4(pr + base + 4 * (lane + 32 * (h + k)));
                if (kResidual) d[k] = ld_stream4(qr + base + 4 * (lane + 32 * (h + k)));
            }
#pragma unroll
            for (int k = 0; k < kSampleBatch; ++k)
                v[h + k] = quad_mass<kResidual>(a[k], kResidual ? d[k] : make_float4(0.f, 0.f, 0.f, 0.f));
        }
    } else {
        Acc acc[kBlocks];
        const int64_t end = base + kSeg < V ? base + kSeg : V;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const int64_t e = base + lane + 32 * j;
            if (e < end) {
                float hi, lo;
                elem_mass<kResidual>(ld_stream1(pr + e), kResidual ? ld_stream1(qr + e) : 0.f, hi, lo);
                acc[j / 4].add(hi, lo);
            }
        }
#pragma unroll
        for (int k = 0; k < kBlocks; ++k) v[k] = acc[k].value();
    }
}

template <bool kResidual>
__device__ __forceinline__ void segment_sum_store(const Params &P, int b, const float *pr,
                                                  const float *qr, int s, int lane) {
    dd v[kBlocks];
    segment_partials<kResidual>(pr, qr, (int64_t)s * kSeg, P.V, lane, v);
    store_sums(P.seg + (int64_t)b * P.nseg, P.blk + (int64_t)b * P.nseg * kBlocks, s, v, lane);
}

__device__ void sample_item(const Params &P, int b, int s, int32_t ns, int lane) {
    if (ns == kNBad) return;  // the decide kernel reports it
    const int n = ns - 1;
    if (n < P.K) segment_sum_store<true>(P, b, prow(P, b, n), qrow(P, b, n), s, lane);
    else segment_sum_store<false>(P, b, prow(P, b, P.K), nullptr, s, lane);
}

// ---------------------------------------------------------------------------
// decisions (one warp, once per sequence)

constexpr int kSegRegs = 8;  // segment sums a lane keeps in registers (V <= 262144)

// Comparisons with the draw threshold are made in double-fp32: a > b for
// normalised pairs (|lo| <= ulp(hi) / 2).
__device__ __forceinline__ bool dd_gt(dd a, dd b) {
    return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

// u * R as a double-fp32 pair (u given as two fp32 parts; fmaf keeps the
// products' rounding errors).
__device__ __forceinline__ dd threshold(dd u, dd R) {
    const float p = __fmul_rn(u.hi, R.hi);
    float e = __fmaf_rn(u.hi, R.hi, -p);
    e = __fmaf_rn(u.hi, R.lo, e);
    e = __fmaf_rn(u.lo, R.hi, e);
    return fast_two_sum(p, e);
}

// Within one 128-element block starting at element `base` of the row pair:
// the smallest index whose running mass prefix + C_v exceeds T, or the last
// index with mass if none does (a rounding boundary), or -1.  Lane l holds
// elements 4l .. 4l + 3; one warp scan finds the lane, which walks its four.
template <bool kResidual>
__device__ int search_block(const float *pr, const float *qr, int64_t base, int64_t V, dd prefix,
                            dd T, int lane) {
    const int64_t n = V - base < 128 ? V - base : 128;
    const int64_t e0 = 4 * lane;
    float pv[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (n == 128 && aligned16(pr + base) && (!kResidual || aligned16(qr + base))) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(pr + base + e0));
        pv[0] = a.x; pv[1] = a.y; pv[2] = a.z; pv[3] = a.w;
        if (kResidual) {
            const float4 d = __ldcg(reinterpret_cast<const float4 *>(qr + base + e0));
            qv[0] = d.x; qv[1] = d.y; qv[2] = d.z; qv[3] = d.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            pv[j] = e0 + j < n ? __ldcg(pr + base + e0 + j) : 0.f;
            if (kResidual) qv[j] = e0 + j < n ? __ldcg(qr + base + e0 + j) : 0.f;
        }
    }
    float mh[4], ml[4];
    int last_nz = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        elem_mass<kResidual>(pv[j], qv[j], mh[j], ml[j]);
        if (mh[j] != 0.f) last_nz = (int)e0 + j;
    }
    // the same four-element sum the stream kernels formed for the block sums
    const dd mine = quad_mass<kResidual>(make_float4(pv[0], pv[1], pv[2], pv[3]),
                                         make_float4(qv[0], qv[1], qv[2], qv[3]));
    const dd inc = warp_incl_scan(mine, lane);
    const unsigned m = __ballot_sync(0xffffffffu, mine.hi != 0.f && dd_gt(dd_add(prefix, inc), T));
    if (m) {
        const int L = __ffs(m) - 1;
        dd excl = shfl_up_dd(inc, 1);
        if (lane == 0) excl = {0.f, 0.f};
        int found = -1;
        if (lane == L) {
            dd run = dd_add(prefix, excl);
            int lastj = -1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (found < 0 && mh[j] != 0.f) {
                    lastj = j;
                    run = dd_add(run, fast_two_sum(mh[j], ml[j]));
                    if (dd_gt(run, T)) found = (int)e0 + j;
                }
            }
            if (found < 0) found = (int)e0 + lastj;  // the lane crossed, its steps did not
        }
        found = __shfl_sync(0xffffffffu, found, L);
        return (int)(base + found);
    }
#pragma unroll
    for (int mm = 16; mm > 0; mm >>= 1) last_nz = max(last_nz, __shfl_xor_sync(0xffffffffu, last_nz, mm));
    return last_nz < 0 ? -1 : (int)(base + last_nz);
}

// Given lanes holding consecutive sums v (lane order = index order) and their
// inclusive warp scan inc, starting at running mass `prefix`: the first lane
// whose inclusive sum exceeds T (-1 if none) and the running mass before it.
__device__ __forceinline__ int crossing_of_scan(dd v, dd inc, dd prefix, dd T, int lane, dd &before) {
    const unsigned m = __ballot_sync(0xffffffffu, v.hi != 0.f && dd_gt(dd_add(prefix, inc), T));
    if (!m) return -1;
    const int L = __ffs(m) - 1;
    dd excl = shfl_up_dd(inc, 1);
    if (lane == 0) excl = {0.f, 0.f};
    before = shfl_dd(dd_add(prefix, excl), L);
    return L;
}

__device__ __forceinline__ int first_crossing(dd v, dd prefix, dd T, int lane, dd &before) {
    return crossing_of_scan(v, warp_incl_scan(v, lane), prefix, T, lane, before);
}

// The same over the eight block sums of a segment, held by lanes 0..7.
__device__ __forceinline__ int first_crossing8(dd v, dd prefix, dd T, int lane, dd &before) {
    return crossing_of_scan(v, warp_incl_scan<kBlocks>(v, lane), prefix, T, lane, before);
}

// Asks the memory system to bring [p, p + bytes) into L2 (no destination, no
// completion): a later load of it then waits on L2, not on DRAM.  p and bytes
// are multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ dd split_uniform(double ur) {
    const float uh = __double2float_rn(ur);
    return {uh, __double2float_rn(__dsub_rn(ur, (double)uh))};
}

// Where a draw finds the sequence's uniform and its block sums.
struct DrawInputs {
    dd u;                     // the uniform split into two fp32 parts, unless u_res is set
    const double *u_res;      // else: loaded here once the segment loads are out
    bool seg_local;           // seg points to shared memory written by this CTA
    const float2 *blk_sh;     // block sums in shared memory (else read from blk) ...
    unsigned long long *bar;  // ... staged by a bulk copy completing on this mbarrier phase
    uint32_t parity;          //     (no wait when bar is null)
    bool prefetch;            // rows are 16-byte-aligned device memory: once the segment
                              // is known, ask L2 for it while the block is searched
};

__device__ __forceinline__ float2 load_sum(const float2 *p, bool local) {
    return local ? *p : ld_l2(p);
}

// Inverse-CDF draw over the segment sums seg[0..nseg) and block sums blk of a
// row of V masses (one warp): the token, -1 if the total mass is zero, -2 if
// the staged block sums never arrived.  The segment (lane l owns segments
// [l * per, (l + 1) * per)), the block within it (lanes 0..7), then
// in_block(base, prefix, T), which finds the element within the 128-element
// block at `base`: one load round trip each, or two in all when the block
// sums were staged while the segment sums loaded.  With in.prefetch, rows
// pf0 and pf1 (either may be null) are asked into L2 at the chosen segment.
template <class InBlock>
__device__ int draw_core(int nseg, int64_t V, const float2 *seg, const float2 *blk,
                         const float *pf0, const float *pf1, const DrawInputs &in, int lane,
                         InBlock in_block) {
    const int per = (nseg + 31) / 32;
    const int r0 = min(nseg, lane * per), r1 = min(nseg, r0 + per);
    dd v[kSegRegs];
#pragma unroll
    for (int r = 0; r < kSegRegs; ++r) {
        v[r] = dd{0.f, 0.f};
        if (r0 + r < r1) {
            const float2 x = load_sum(seg + r0 + r, in.seg_local);
            v[r] = dd{x.x, x.y};
        }
    }
    const dd u = in.u_res ? split_uniform(__ldg(in.u_res)) : in.u;
    static_assert(kSegRegs == 8, "the lane total below is a tree over eight sums");
    dd own = dd_add(dd_add(dd_add(v[0], v[1]), dd_add(v[2], v[3])),
                    dd_add(dd_add(v[4], v[5]), dd_add(v[6], v[7])));
    for (int s = r0 + kSegRegs; s < r1; ++s) {  // rows longer than 32 * kSegRegs segments
        const float2 x = load_sum(seg + s, in.seg_local);
        own = dd_add(own, dd{x.x, x.y});
    }
    const dd inc = warp_incl_scan(own, lane);
    const dd total = shfl_dd(inc, 31);
    // the staged copy has to land before this warp returns, whatever the outcome
    if (in.bar && !__all_sync(0xffffffffu, mbar_wait(in.bar, in.parity))) return -2;
    if (total.hi == 0.f) return -1;
    const dd T = threshold(u, total);
    const dd zero = {0.f, 0.f};
    dd before;
    const int L = crossing_of_scan(own, inc, zero, T, lane, before);
    // the segment, the running mass before it, and the time T is past every segment
    int sg = -1;
    dd sbefore = zero;
    if (L >= 0 && per <= kSegRegs) {
        // every lane walks its own segments from its exclusive prefix (the
        // same additions lane L alone would make); lane L's result is used
        dd excl = shfl_up_dd(inc, 1);
        if (lane == 0) excl = zero;
        dd acc = dd_add(zero, excl), last_before = acc, fbefore = zero;
        int last = -1, found = -1;
#pragma unroll
        for (int r = 0; r < kSegRegs; ++r) {
            if (r0 + r < r1 && found < 0) {
                const dd x = v[r];
                const dd nx = dd_add(acc, x);
                if (x.hi != 0.f) {
                    last = r0 + r;
                    last_before = acc;
                    if (dd_gt(nx, T)) {
                        found = r0 + r;
                        fbefore = acc;
                    }
                }
                acc = nx;
            }
        }
        if (found < 0) {
            found = last;
            fbefore = last_before;
        }
        sg = __shfl_sync(0xffffffffu, found, L);
        sbefore = shfl_dd(fbefore, L);
    } else if (L >= 0) {
        // rows longer than 32 * kSegRegs segments: lane L walks, loading the rest
        if (lane == L) {
            dd acc = before, last_before = before;
            int last = -1;
            for (int s = r0; s < r1; ++s) {
                const int r = s - r0;
                dd x = zero;
                if (r < kSegRegs) {
#pragma unroll
                    for (int i = 0; i < kSegRegs; ++i)
                        if (i == r) x = v[i];
                } else {
                    const float2 y = load_sum(seg + s, in.seg_local);
                    x = dd{y.x, y.y};
                }
                const dd nx = dd_add(acc, x);
                if (x.hi != 0.f) {
                    last = s;
                    last_before = acc;
                    if (dd_gt(nx, T)) {
                        sg = s;
                        sbefore = acc;
                        break;
                    }
                }
                acc = nx;
            }
            if (sg < 0) {
                sg = last;
                sbefore = last_before;
            }
        }
        sg = __shfl_sync(0xffffffffu, sg, L);
        sbefore = shfl_dd(sbefore, L);
    }
    dd Tt = T;
    if (sg < 0) {
        // T reached the total through rounding: the last segment with mass,
        // searched with an infinite threshold (its last element with mass)
        int lastnz = -1;
        for (int s = r0; s < r1; ++s)
            if (load_sum(seg + s, in.seg_local).x != 0.f) lastnz = s;
#pragma unroll
        for (int mm = 16; mm > 0; mm >>= 1) lastnz = max(lastnz, __shfl_xor_sync(0xffffffffu, lastnz, mm));
        sg = lastnz;
        Tt = dd{__int_as_float(0x7f800000), 0.f};
    }
    if (in.prefetch && lane < 2) {
        const int c = min(kSeg, (int)(V - (int64_t)sg * kSeg)) & ~3;
        const float *row = lane == 0 ? pf0 : pf1;
        if (c && row) prefetch_l2(row + (int64_t)sg * kSeg, 4u * (uint32_t)c);
    }
    // block within the segment
    dd bv = zero;
    if (lane < kBlocks) {
        const float2 x = in.blk_sh ? in.blk_sh[sg * kBlocks + lane]
                                   : ld_l2(blk + (int64_t)sg * kBlocks + lane);
        bv = dd{x.x, x.y};
    }
    dd bbefore;
    int bk = first_crossing8(bv, sbefore, Tt, lane, bbefore);
    if (bk < 0) {
        // block sums and the segment sum disagree in the last bits: the last
        // block with mass, with an infinite threshold
        const unsigned nz = __ballot_sync(0xffffffffu, lane < kBlocks && bv.hi != 0.f);
        bk = nz ? 31 - __clz(nz) : kBlocks - 1;
        bbefore = zero;
        Tt = dd{__int_as_float(0x7f800000), 0.f};
    }
    return in_block((int64_t)sg * kSeg + 128 * bk, bbefore, Tt);
}

// The draw over a probability row pair (pr, qr), or over pr alone.
template <bool kResidual>
__device__ int draw_from_sums(const Params &P, const float2 *seg, const float2 *blk,
                              const float *pr, const float *qr, const DrawInputs &in, int lane) {
    return draw_core(P.nseg, P.V, seg, blk, pr, qr, in, lane, [&](int64_t base, dd prefix, dd T) {
        return search_block<kResidual>(pr, qr, base, P.V, prefix, T, lane);
    });
}

// Commit step of a round ("spec-verify", section "Usage": keep
// draft_tokens[:n_accepted], append next_token).
__device__ void commit_round(const Params &P, int b, int n, int next, int lane) {
    if (!P.tokens || next < 0) return;
    int len = 0;
    if (lane == 0) {
        len = P.lengths[b];
        const bool ok = len >= 0 && (int64_t)len + n + 1 <= P.max_len;
        if (!ok) {
            atomicOr(P.status, kStatusOverflow);
            len = -1;
        }
    }
    len = __shfl_sync(0xffffffffu, len, 0);
    if (len < 0) return;
    int32_t *row = P.tokens + (int64_t)b * P.max_len;
    for (int i = lane; i < n; i += 32) row[len + i] = P.t[(int64_t)b * P.K + i];
    if (lane == 0) {
        row[len + n] = next;
        P.lengths[b] = len + n + 1;
    }
}

__device__ void greedy_decide(const Params &P, int b, int lane) {
    int32_t t0, t1;
    const bool bad = load_tokens(P, b, lane, t0, t1);
    int n = 0, next = -1;
    if (!bad) {
        const int f = ld_l2(P.miss + b);
        n = f ? kFlagBase - f : P.K;
        const unsigned long long key = ld_l2(P.best + (int64_t)b * (P.K + 1) + n);
        next = key ? key_index(key) : 0;
    }
    if (lane == 0) {
        if (bad) atomicOr(P.status, kStatusBadToken);
        P.n_out[b] = n;
        P.next_out[b] = next;
        P.miss[b] = 0;
        P.nstate[b] = 0;
    }
    for (int i = lane; i <= P.K; i += 32) P.best[(int64_t)b * (P.K + 1) + i] = 0ull;
    commit_round(P, b, n, next, lane);
}

__device__ void sample_decide(const Params &P, int b, int lane) {
    const int ns = ld_l2(P.nstate + b);
    const float2 uf = ld_l2(P.udd + b);  // loaded alongside, used only if the sequence is valid
    DrawInputs in = {};
    in.u = dd{uf.x, uf.y};
    const bool bad = ns == kNBad;
    int n = 0, next = -1;
    if (!bad) {
        n = ns - 1;
        const float2 *seg = P.seg + (int64_t)b * P.nseg;
        const float2 *blk = P.blk + (int64_t)b * P.nseg * kBlocks;
        if (n < P.K) {
            next = draw_from_sums<true>(P, seg, blk, prow(P, b, n), qrow(P, b, n), in, lane);
            if (next < 0) {
                // zero residual mass (unnormalised rows): draw from p_n itself
                const float *pr = prow(P, b, n);
                for (int s = 0; s < P.nseg; ++s) segment_sum_store<false>(P, b, pr, nullptr, s, lane);
                __threadfence_block();
                __syncwarp();
                next = draw_from_sums<false>(P, seg, blk, pr, nullptr, in, lane);
            }
        } else {
            next = draw_from_sums<false>(P, seg, blk, prow(P, b, P.K), nullptr, in, lane);
        }
    }
    if (lane == 0) {
        if (bad) atomicOr(P.status, kStatusBadToken);
        else if (next < 0) atomicOr(P.status, kStatusZeroMass);
        P.n_out[b] = n;
        P.next_out[b] = next;
        P.nstate[b] = 0;
    }
    commit_round(P, b, n, next, lane);
}

// ---------------------------------------------------------------------------
// kernels

__device__ __forceinline__ void grid_dependents_may_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void wait_for_primary_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One warp per sequence, cached in the workspace for the later kernels: the
// first rejection of a sampling sequence; for a greedy sequence, whether its
// draft ids are valid and the target probability of each draft token.
template <int kRule>
__global__ void __launch_bounds__(kThreads) scan_kernel(const Params P) {
    grid_dependents_may_launch();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b >= P.B) return;
    const int rule = kRule == kPerSequence ? (int)P.mode[b] : kRule;
    int32_t ns = 0;
    if (rule == kSample) {
        ns = first_rejection(P, b, lane);
        if (lane == 0) {
            const double u = P.u_res[b];
            const float uh = __double2float_rn(u);
            P.udd[b] = make_float2(uh, __double2float_rn(__dsub_rn(u, (double)uh)));
        }
    } else if (rule == kGreedy) {
        int32_t t0, t1;
        const bool bad = load_tokens(P, b, lane, t0, t1);
        if (!bad) {
            float *pt = P.ptok + (int64_t)b * P.K;
            if (lane < P.K) pt[lane] = __ldg(prow(P, b, lane) + t0);
            if (lane + 32 < P.K) pt[lane + 32] = __ldg(prow(P, b, lane + 32) + t1);
        }
        ns = bad ? kNBad : 1;
    } else {
        return;
    }
    if (lane == 0) P.nstate[b] = ns;
}

template <int kRule>
__device__ __forceinline__ void stream_body(const Params &P) {
    // the decide kernel may be scheduled as soon as this grid's CTAs retire
    grid_dependents_may_launch();
    // the scan kernel's cached per-sequence data
    wait_for_primary_grid();
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
    // per-item sequence data is fetched one item ahead
    int item = w;
    int32_t ns_next = 0, rule_next = kRule;
    if (item < P.items && lane == 0) {
        const int b = item / P.nseg;
        if (kRule == kPerSequence) rule_next = P.mode[b];
        if (kRule != kGreedy) ns_next = ld_l2(P.nstate + b);
    }
    for (; item < P.items; item += P.warps) {
        const int b = item / P.nseg;
        const int s = item - b * P.nseg;
        const int rule = __shfl_sync(0xffffffffu, rule_next, 0);
        const int32_t ns = __shfl_sync(0xffffffffu, ns_next, 0);
        const int nxt = item + P.warps;
        if (nxt < P.items && lane == 0) {
            const int bn = nxt / P.nseg;
            if (kRule == kPerSequence) rule_next = P.mode[bn];
            if (kRule != kGreedy) ns_next = ld_l2(P.nstate + bn);
        }
        if (rule == kGreedy) greedy_item(P, b, s, lane);
        else if (rule == kSample) sample_item(P, b, s, ns, lane);
    }
}

template <int kRule>
__global__ void __launch_bounds__(kThreads, SV_MIN_CTAS_PER_SM) stream_kernel(const Params P) {
    stream_body<kRule>(P);
}

// The greedy stream needs fewer registers, so more warps fit per SM.
template <>
__global__ void __launch_bounds__(kThreads, SV_GREEDY_MIN_CTAS_PER_SM)
stream_kernel<kGreedy>(const Params P) {
    stream_body<kGreedy>(P);
}

// One warp per sequence: turns the partials into (n_accepted, next_token),
// commits a round if asked, and leaves the workspace zeroed for the next call.
constexpr int kDecideWarps = 2;  // small CTAs spread the per-sequence work over the SMs

template <int kRule>
__global__ void __launch_bounds__(kDecideWarps * 32) decide_kernel(const Params P) {
    wait_for_primary_grid();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kDecideWarps + (threadIdx.x >> 5);
    if (b >= P.B) return;
    const int rule = kRule == kPerSequence ? (int)P.mode[b] : kRule;
    if (rule == kGreedy) {
        greedy_decide(P, b, lane);
    } else if (rule == kSample) {
        sample_decide(P, b, lane);
    } else if (lane == 0) {
        atomicOr(P.status, kStatusBadMode);
        P.n_out[b] = 0;
        P.next_out[b] = -1;
    }
}

}  // namespace sv
