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
// One persistent launch in which every warp is a worker.  Work comes in
// groups, one per (sequence b, position i, kind), each group one task per
// 1024-element segment of the row:
//   norm(b, i), i < K  the normalisers of the row pair (zp_i, zq_i): the task
//                      streams its segment of both rows once and stores, per
//                      row, the segment's maximum M and the double-fp32 sum of
//                      exp2((z - M) * c), c = log2(e) / tau (fp32 sums of four,
//                      then a fixed tree and a butterfly over the lanes);
//   norm(b, K)         the same on the bonus row zp_K alone;
//   mass(b, n)         the masses r = max(0, p_n - q_n) (or p_K) of the chosen
//                      row (pair), formed in fp32 from the normalisers, summed
//                      in fours and stored as double-fp32 block and segment
//                      sums.
// One queue counter hands tasks (bulk-copy workers: chunks of 4, 8 or 32
// segments, chosen per call) out in order.  The first B groups are
// norm(b, 0); every later group is appended by the worker that finishes the
// last task of the sequence's previous group (an arrival counter per
// sequence).  That worker merges the segment pairs in segment order -- so the
// normalisers do not depend on which worker ran which task -- and decides:
// after norm(b, i) it makes the accept test u * q_i(t_i) < p_i(t_i) on the
// gathered logits and appends norm(b, i + 1) on acceptance, else mass(b, i)
// (a precise group first when the fp32 test is too close to call); after
// norm(b, K) it appends mass(b, K); after mass(b, n) it draws with the same
// segment -> block -> element search as the probability path, its element
// step recomputing the masses with the same instructions.  A sequence's
// groups form a chain that runs while other sequences' groups fill the
// machine.  To shorten the chains: mass groups, which end a chain, wait in a
// pending list while the first groups alone occupy every worker; producers
// claim their next chunk only once the current one is issued; and where the
// chains are long against the batch, a norm group appended while workers run
// short of work covers two positions.  The only wait is that of a worker whose
// next task belongs to a group not yet appended; it is bounded
// (kStatusTimeout), moves pending mass groups into the queue, and ends once
// every sequence has its token.
//
// Accuracy: each mass carries the error of exp2.approx (~2^-22), of the fp32
// subtraction and scaling of its argument (about |z - max| * c * 2^-24 in the
// exponent) and of the fp32 normalisation -- around 1e-6 relative at most for
// the elements that carry mass; the fp32 sums within a lane (four masses, or a
// lane's 32 normaliser terms) add at most 3 * 2^-24 and 5 * 2^-24 relative,
// and everything above them is summed in double-fp32.  An accept test whose
// margin is inside the fast probabilities' error bound is made again in fp64
// (lg_fast_decides), so accept decisions equal an fp64 softmax's; drawn
// tokens may differ only when u*R lies within ~2e-6 (in units of normalised
// mass) of a boundary.
#pragma once

#include "sv_device.cuh"
#include "sv_tma.cuh"
#include "sv_trace.cuh"

namespace sv {

constexpr int kLgWarps = 8;
constexpr int kLgThreads = kLgWarps * 32;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr uint32_t kLgNorm = 1u, kLgMass = 2u, kLgPrecise = 3u;  // group kinds

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
    double tau;         // the temperature (the precise recomputation's exp((z - M) / tau))
    int32_t *n_out;
    int32_t *next_out;
    uint32_t *status;
    float2 *seg;        // workspace [B][nseg] segment sums of the mass pass
    float2 *blk;        // workspace [B][nseg][8] block sums of the mass pass; before a
                        // sequence's mass pass the first half of its rows holds the
                        // norm tasks' (max, sum) pairs, two float4 per segment
    float4 *fnorm;      // workspace [B][2] normalisers of the chosen row (pair)
    unsigned long long *grp;    // workspace [B * (3K + 2)] group slots (0 = not appended)
    int32_t *arrive;    // workspace [B] the sequence's arrivals so far, weighted so that every
                        // group adds 2 nseg (a group is complete at a multiple of 2 nseg)
    unsigned long long *head;   // next task (plain-load workers) or chunk (bulk-copy workers)
    unsigned long long *tail;   // groups appended after the first B
    uint32_t *ndone;    // sequences finished
    uint32_t *nexit;    // workers that left
    int64_t ngroups;    // B * (3K + 2): a sequence appends at most 3K + 1 slots (a norm group
                        // of at most two slots per position after the first, a precise group
                        // per near-threshold test, a mass one)
    unsigned long long *pend;       // workspace [B] deferred mass groups (0 = not yet written)
    unsigned long long *pend_head;  // deferred mass groups moved into the queue so far
    unsigned long long *pend_tail;  // mass groups deferred so far
    int32_t defer;      // nonzero: mass groups are deferred (see lg_append_mass)
    int32_t chunk;      // bulk-copy workers: segments per chunk (a multiple of kLgStageSegs)
    int64_t claims;     // queue claims per group slot (chunks, or tasks for the plain-load workers)
    int64_t spec_claims;  // a norm group spans two positions while fewer claims than this are
                          // appended and not yet taken (0: never)
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

// A running (max, sum of exp2((z - max) * c)) pair of a row, merged from
// per-segment pairs.
struct Online {
    float m = kNegInf;
    dd s = {0.f, 0.f};
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
    // merges the lanes' states in a fixed butterfly and gives every lane the
    // result lane 0 holds
    __device__ void warp_merge(float c) {
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
            const dd s2 = shfl_xor_dd(s, d);
            merge(m2, s2, c);
        }
        m = __shfl_sync(0xffffffffu, m, 0);
        s = shfl_dd(s, 0);
    }
};

// Loads element e of a row (or -inf padding past end), vectorised when possible.
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

// A row's normalisers: the maximum logit and the sum of exp2((z - m) * c).
struct RowNorm {
    float m;
    dd s;
};

// Normalisers of one 1024-element segment of a row held as eight float4 per
// lane (lane l: elements 4 * (l + 32k) .. + 3, -inf past the row's end): the
// segment's maximum M (warp-wide first, so every term below is independent)
// and S = sum exp2((z - M) * c) -- a fixed fp32 tree over the lane's 32 terms
// (at most 5 * 2^-24 relative error), then a double-fp32 butterfly over the
// lanes (dd_add is commutative, so every lane ends with the same bits).
__device__ __forceinline__ RowNorm seg_norm(const float4 (&x)[kVecPerLane], float c) {
    float mx = kNegInf;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k)
        mx = fmaxf(mx, fmaxf(fmaxf(x[k].x, x[k].y), fmaxf(x[k].z, x[k].w)));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    if (mx == kNegInf) return RowNorm{kNegInf, {0.f, 0.f}};  // padding only (warp-uniform)
    float g[kVecPerLane];
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k)
        g[k] = sum4(make_float4(warp_e(x[k].x, mx, c), warp_e(x[k].y, mx, c),
                                warp_e(x[k].z, mx, c), warp_e(x[k].w, mx, c)));
    static_assert(kVecPerLane == 8, "the lane sum below is a tree over eight");
    dd t = {__fadd_rn(__fadd_rn(__fadd_rn(g[0], g[1]), __fadd_rn(g[2], g[3])),
                      __fadd_rn(__fadd_rn(g[4], g[5]), __fadd_rn(g[6], g[7]))),
            0.f};
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) t = dd_add(t, shfl_xor_dd(t, d));
    return RowNorm{mx, t};
}

__device__ __forceinline__ bool lg_vec(const LogitsParams &L) {
    return aligned16(L.zp) && aligned16(L.zq) && (L.ps & 3) == 0 && (L.qs & 3) == 0;
}

// Mass of one element: the residual max(0, p - q) of the warped rows, or p
// alone (pair false), with 1/S rounded once to fp32.
__device__ __forceinline__ float lg_mass(float za, float zb, bool pair, const RowNorm &na,
                                         const RowNorm &nb, float ia, float ib, float c) {
    const float pa = __fmul_rn(warp_e(za, na.m, c), ia);
    if (!pair) return pa;
    const float qb = __fmul_rn(warp_e(zb, nb.m, c), ib);
    return fmaxf(__fsub_rn(pa, qb), 0.f);
}

// The fp32 accept test u * qt < pt decides only when its margin is larger
// than the error of the fast probabilities can be; every other test is made
// again in fp64 (a precise group).  Relative error of a fast probability
// exp2(a) / S_hi, first order, with slack:
//   the argument a: three fp32 roundings (z - M, c = log2(e) / tau, the
//     product), |da| <= 3 * 2^-24 * |a|, so ln 2 * 3 * 2^-24 * |a| (kLn2ArgRel);
//   ex2.approx.f32: at most kEx2Rel (2^-20; the GPU tests measure its error
//     over a dense sweep of arguments against fp64 and require half of it);
//   the normaliser S: every term carries its own argument error -- at most
//     ln 2 * 3 * 2^-24 * 64 relative for the terms with |a| <= 64; the others
//     are below 2^-64 each and cannot matter at 2^-31 terms -- and ex2
//     error, plus up to nine rescalings by exp2 factors and fp32 sums of four
//     and of eight (kRowRel);
//   the reciprocal, S_lo and the product: 3 * 2^-24.
// Results below 2^-100 (where subnormal outputs lose relative accuracy) are
// never decided in fp32.
constexpr float kU24 = 5.9604645e-08f;          // 2^-24
constexpr float kLn2ArgRel = 1.2395e-07f;       // ln 2 * 3 * 2^-24, rounded up
constexpr float kEx2Rel = 9.5367432e-07f;       // 2^-20
constexpr float kRowRel = 64.f * kLn2ArgRel + 10.f * kEx2Rel + 48.f * kU24 + 1e-12f;
constexpr float kTiny = 7.8886091e-31f;         // 2^-100

// True when u * qt < pt (fp32, as accepts() decides it) is certain to agree
// with the exact test on the exact softmax; ap, aq are the tokens' fp32
// arguments.
__device__ __forceinline__ bool lg_fast_decides(float u, float pt, float qt, float ap, float aq) {
    const float rp = kLn2ArgRel * fabsf(ap) + kEx2Rel + kRowRel + 3.f * kU24;
    const float rq = kLn2ArgRel * fabsf(aq) + kEx2Rel + kRowRel + 3.f * kU24;
    const float uq = u * qt;
    const float margin = fabsf(fmaf(-u, qt, pt));
    const float bound = 1.01f * (pt * rp + uq * rq) + 2.f * kU24 * fmaxf(pt, uq) + kTiny;
    return margin > bound;  // false for NaN too
}

// fp64 sum of exp((x - M) / tau) over a lane's elements of one segment
// (-inf marks padding): the precise recomputation's terms, the oracle's
// formula.
__device__ __forceinline__ double precise_terms(const float4 (&x)[kVecPerLane], float M, double tau) {
    double s = 0.0;
    const double m = (double)M;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
        if (x[k].x != kNegInf) s += exp(((double)x[k].x - m) / tau);
        if (x[k].y != kNegInf) s += exp(((double)x[k].y - m) / tau);
        if (x[k].z != kNegInf) s += exp(((double)x[k].z - m) / tau);
        if (x[k].w != kNegInf) s += exp(((double)x[k].w - m) / tau);
    }
    return s;
}

// Sum over the warp in a fixed butterfly (every lane ends with the same bits).
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// Masses of segment s of a row (pair) into its segment and block sums (one warp).
__device__ void lg_mass_segment(const float *a, const float *b, const LogitsParams &L, float2 *seg,
                                float2 *blk, int64_t s, bool vec, const RowNorm &na,
                                const RowNorm &nb, float ia, float ib, int lane) {
    const int64_t base = s * kSeg;
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

// ---------------------------------------------------------------------------
// the task queue

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Arrival of n tasks on a sequence's counter: release (the stores this thread
// made or observed before it) and acquire (the earlier arrivals' stores) in
// one atomic; returns the count before it.
__device__ __forceinline__ int arrive_acq_rel(int32_t *p, int n) {
    int v;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(v) : "l"(p), "r"(n) : "memory");
    return v;
}

// A group slot: bit 63 marks it present, then the slot's place in its span
// (bit 44), the span less one (bits 42-43), kind (bits 40-41), the slot's
// position (32-39) and sequence (0-31).  A norm group of span 2 is two
// consecutive slots, positions i and i + 1, whose tasks count as one group.
__device__ __forceinline__ unsigned long long lg_group(int b, int i, uint32_t kind, int span = 1,
                                                       int r = 0) {
    return (1ull << 63) | ((unsigned long long)r << 44) | ((unsigned long long)(span - 1) << 42) |
           ((unsigned long long)kind << 40) | ((unsigned long long)(uint32_t)i << 32) |
           (unsigned long long)(uint32_t)b;
}

// The span bits of a slot: span - 1, and the slot's place r in bit 2.
__device__ __forceinline__ int lg_span_bits(unsigned long long d) { return (int)((d >> 42) & 7u); }

// One arrival of `tasks` tasks on sequence b's count (lane 0; acquire and
// release): every group adds 2 nseg in all (a task of a span-2 group counts
// 1, any other 2), so a group is complete when the count reaches a multiple
// of 2 nseg.
__device__ __forceinline__ bool lg_arrive(const LogitsParams &L, int b, int tasks, int span) {
    const int w = span == 2 ? tasks : 2 * tasks;
    return (arrive_acq_rel(L.arrive + b, w) + w) % (2 * L.nseg) == 0;
}

// The queue's claim counter and appended slots as one snapshot (relaxed;
// only a hint).
__device__ __forceinline__ ulonglong2 lg_queue_snapshot(const LogitsParams &L) {
    return __ldcg(reinterpret_cast<const ulonglong2 *>(L.head));  // head, then tail
}

// Appends a group (one lane; its earlier stores are visible to every reader
// of the group).
__device__ __forceinline__ void lg_append(const LogitsParams &L, unsigned long long gdesc) {
    const unsigned long long slot = (unsigned long long)L.B + atomicAdd(L.tail, 1ull);
    if (slot >= (unsigned long long)L.ngroups) {  // cannot happen: at most K + 1 per sequence
        atomicOr(L.status, kStatusOverflow);
        return;
    }
    st_release(L.grp + slot, gdesc);
}

// Appends sequence b's norm group at position i (one lane).  While the queue,
// as seen in the snapshot ht, holds fewer than spec_claims claims that no
// worker has taken, workers are about to wait for work: the group then also
// covers position i + 1 (when there is one), whose normalisers are ready if
// position i is accepted and are not used otherwise.
__device__ __forceinline__ void lg_append_norm(const LogitsParams &L, int b, int i, ulonglong2 ht) {
    const long long appended =
        (long long)(((unsigned long long)L.B + ht.y) * (unsigned long long)L.claims);
    if (i < L.K && appended - (long long)ht.x < L.spec_claims) {
        const unsigned long long slot = (unsigned long long)L.B + atomicAdd(L.tail, 2ull);
        if (slot + 1 >= (unsigned long long)L.ngroups) {  // cannot happen (see ngroups)
            atomicOr(L.status, kStatusOverflow);
            return;
        }
        st_release(L.grp + slot, lg_group(b, i, kLgNorm, 2, 0));
        st_release(L.grp + slot + 1, lg_group(b, i + 1, kLgNorm, 2, 1));
    } else {
        lg_append(L, lg_group(b, i, kLgNorm));
    }
}

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The mass group that ends sequence b's chain (one lane; the normalisers it
// needs are in fnorm).  A sequence's normaliser groups form its chain of
// dependent steps, and a mass group has no successor: when the call defers,
// the mass group waits in the pending list, so that the chains' next groups
// are not queued behind it, until a worker that finds no work moves it in
// (lg_release_mass).
__device__ void lg_append_mass(const LogitsParams &L, unsigned long long gdesc) {
    if (!L.defer) {
        lg_append(L, gdesc);
        return;
    }
    const unsigned long long slot = atomicAdd(L.pend_tail, 1ull);
    if (slot >= (unsigned long long)L.B) {  // cannot happen: one mass group per sequence
        atomicOr(L.status, kStatusOverflow);
        return;
    }
    st_release(L.pend + slot, gdesc);
}

// Deferred mass groups moved into the queue at once (one claim of the
// pending list and one of the queue for all of them).
constexpr int kLgReleaseBatch = 4;

// Moves the oldest deferred mass groups, up to kLgReleaseBatch of them, into
// the queue (one lane), unless there are none or another worker takes them
// first.
__device__ void lg_release_mass(const LogitsParams &L) {
    const unsigned long long h = ld_relaxed64(L.pend_head);
    const unsigned long long t = ld_relaxed64(L.pend_tail);
    if (h >= t) return;
    const unsigned long long n = t - h < (unsigned long long)kLgReleaseBatch ? t - h : kLgReleaseBatch;
    if (atomicCAS(L.pend_head, h, h + n) != h) return;
    const unsigned long long slot = (unsigned long long)L.B + atomicAdd(L.tail, n);
    for (unsigned long long k = 0; k < n; ++k) {
        // a pending slot is taken just before it is written: wait for it (bounded)
        IdleClock clk;
        unsigned long long d;
        while (!(d = ld_acquire(L.pend + h + k))) {
            if (!clk.idle(64)) {
                atomicOr(L.status, kStatusTimeout);
                return;
            }
        }
        L.pend[h + k] = 0ull;  // zero again for the next call
        if (slot + k >= (unsigned long long)L.ngroups) {  // cannot happen (see ngroups)
            atomicOr(L.status, kStatusOverflow);
            return;
        }
        st_release(L.grp + slot + k, d);
    }
}

// A worker that has waited this long for its claimed group moves deferred
// mass groups into the queue (a shorter wait would let them in while the
// chains' groups are still on their way; a longer one idles the worker).
constexpr uint64_t kLgReleaseNs = 3000;

// Group g (one lane): the first B are implicit; a later one is waited for
// until appended, or until every sequence is finished (0).  Once the wait
// has lasted kLgReleaseNs, the worker moves deferred mass groups into the
// queue, so a wait always ends: every unfinished sequence either has a group
// in the queue or a deferred mass group that a waiting worker appends.
__device__ unsigned long long lg_wait_group(const LogitsParams &L, uint64_t g) {
    if (g < (uint64_t)L.B) return lg_group((int)g, 0, kLgNorm);
    IdleClock clk;
    const uint64_t t0 = global_ns();
    while (true) {
        const unsigned long long d = ld_acquire(L.grp + g);
        if (d) return d;
        if (ld_relaxed(L.ndone) >= (uint32_t)L.B) return 0ull;
        if (L.defer && global_ns() - t0 >= kLgReleaseNs) lg_release_mass(L);
        if (!clk.idle(256)) {
            atomicOr(L.status, kStatusTimeout);
            return 0ull;
        }
    }
}

// A sequence's result (one lane).
__device__ __forceinline__ void lg_finish(const LogitsParams &L, int b, int n, int next,
                                          uint32_t flags) {
    if (flags) atomicOr(L.status, flags);
    L.n_out[b] = n;
    L.next_out[b] = next;
    __threadfence();
    atomicAdd(L.ndone, 1u);
}

__device__ __forceinline__ const float *lg_row_p(const LogitsParams &L, int b, int i) {
    return L.zp + ((int64_t)b * (L.K + 1) + i) * L.ps;
}

__device__ __forceinline__ const float *lg_row_q(const LogitsParams &L, int b, int i) {
    return i < L.K ? L.zq + ((int64_t)b * L.K + i) * L.qs : nullptr;
}

// The (max, sum) slot of segment s of sequence b for the r-th position of a
// span: two float4, p then q (the two places fill the sequence's block sums).
__device__ __forceinline__ float4 *lg_pair(const LogitsParams &L, int b, int64_t s, int r = 0) {
    return reinterpret_cast<float4 *>(L.blk + (int64_t)b * L.nseg * kBlocks) + 2 * (s + r * (int64_t)L.nseg);
}

// Stores a norm task's segment pairs (oa, ob), the same in every lane (lane 0).
__device__ __forceinline__ void lg_store_pair(const LogitsParams &L, int b, int64_t s, int r,
                                              const RowNorm &oa, const RowNorm &ob) {
    float4 *pr = lg_pair(L, b, s, r);
    pr[0] = make_float4(oa.m, oa.s.hi, oa.s.lo, 0.f);
    pr[1] = make_float4(ob.m, ob.s.hi, ob.s.lo, 0.f);
}

// Decides position i of sequence b from its row (pair)'s normalisers na, nb
// and the draft token's logits gp, gq (lane 0): true if the fast test accepts
// the draft token; otherwise the sequence's next group is appended (a precise
// one for a test too close to call in fp32, a mass one after a rejection or
// at the bonus position K) with the normalisers it needs in fnorm.
__device__ __forceinline__ bool lg_decide_fast(const LogitsParams &L, int b, int i, const Online &na,
                                               const Online &nb, float gp, float gq, float u) {
    SV_TRACE_EVENT(kTrLgDecide, (uint32_t)b | ((uint32_t)i << 16) | (kLgNorm << 24));
    if (i == L.K) {
        L.fnorm[2 * b] = make_float4(na.m, na.s.hi, na.s.lo, 0.f);
        lg_append_mass(L, lg_group(b, i, kLgMass));
        return false;
    }
    const float ap = __fmul_rn(__fsub_rn(gp, na.m), L.c), aq = __fmul_rn(__fsub_rn(gq, nb.m), L.c);
    const float pt = __fmul_rn(ex2(ap), __frcp_rn(na.s.hi));  // warp_e(gp, na.m, L.c) / S
    const float qt = __fmul_rn(ex2(aq), __frcp_rn(nb.s.hi));
    const bool sure = lg_fast_decides(u, pt, qt, ap, aq);
    if (sure && accepts(u, qt, pt)) return true;
    // too close to call in fp32 (the position is decided again in fp64; the
    // fast normalisers are kept for a later mass group), or rejected
    L.fnorm[2 * b] = make_float4(na.m, na.s.hi, na.s.lo, 0.f);
    L.fnorm[2 * b + 1] = make_float4(nb.m, nb.s.hi, nb.s.lo, 0.f);
    if (sure)
        lg_append_mass(L, lg_group(b, i, kLgMass));
    else
        lg_append(L, lg_group(b, i, kLgPrecise));
    return false;
}

// The last arrival of sequence b's norm group of kSpan positions from i0
// (slots g0, ...): merges the segment pairs of each position in segment order
// (lane l takes segments l, l + 32, ..., then a fixed butterfly), makes the
// accept tests in position order and appends the sequence's next group (or
// finishes it on an invalid draft id).  Lane 1 + k holds position i0 + k's
// draft token x and uniform u; y0, y1 the draft ids (position 0).
template <int kSpan>
__device__ __forceinline__ void lg_norm_decide(const LogitsParams &L, int b, int i0, uint64_t g0,
                                               int32_t x, float u, int32_t y0, int32_t y1, int lane) {
    const int p = i0 + lane - 1;
    float gp = 0.f, gq = 0.f;
    if (lane >= 1 && lane <= kSpan && p < L.K && x >= 0 && (int64_t)x < L.V) {
        gp = __ldcg(lg_row_p(L, b, p) + x);
        gq = __ldcg(lg_row_q(L, b, p) + x);
    }
    // the queue's state, for the next group's span (with the pairs' round trip)
    ulonglong2 ht = make_ulonglong2(0ull, 0ull);
    if (lane == 3 && L.spec_claims > 0) ht = lg_queue_snapshot(L);
    const bool c0 = i0 < L.K, c1 = kSpan == 2 && i0 + 1 < L.K;
    Online na, nb, ma, mb;
#pragma unroll 4
    for (int64_t k = lane; k < L.nseg; k += 32) {
        const float4 *pr = lg_pair(L, b, k, 0);
        const float4 pa = __ldcg(pr);
        const float4 pb = c0 ? __ldcg(pr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (kSpan == 2) {
            const float4 *qr = lg_pair(L, b, k, 1);
            const float4 qa = __ldcg(qr);
            const float4 qb = c1 ? __ldcg(qr + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            ma.merge(qa.x, dd{qa.y, qa.z}, L.c);
            if (c1) mb.merge(qb.x, dd{qb.y, qb.z}, L.c);
        }
        na.merge(pa.x, dd{pa.y, pa.z}, L.c);
        if (c0) nb.merge(pb.x, dd{pb.y, pb.z}, L.c);
    }
    if (lane == 0) SV_TRACE_EVENT(kTrLgMerged, (uint32_t)b | ((uint32_t)i0 << 16));
    na.warp_merge(L.c);
    if (c0) nb.warp_merge(L.c);
    if constexpr (kSpan == 2) {
        ma.warp_merge(L.c);
        if (c1) mb.warp_merge(L.c);
    }
    bool bad = false;
    if (i0 == 0 && L.K > 0) {  // every draft id is checked once, before the first decision
        static_assert(kMaxK <= 64, "two draft ids per lane");
        bad = (lane < L.K && (y0 < 0 || (int64_t)y0 >= L.V)) ||
              (lane + 32 < L.K && (y1 < 0 || (int64_t)y1 >= L.V));
        bad = __any_sync(0xffffffffu, bad);
    }
    const float u0 = __shfl_sync(0xffffffffu, u, 1), gp0 = __shfl_sync(0xffffffffu, gp, 1),
                gq0 = __shfl_sync(0xffffffffu, gq, 1);
    float u1 = 0.f, gp1 = 0.f, gq1 = 0.f;
    if constexpr (kSpan == 2) {
        u1 = __shfl_sync(0xffffffffu, u, 2);
        gp1 = __shfl_sync(0xffffffffu, gp, 2);
        gq1 = __shfl_sync(0xffffffffu, gq, 2);
    }
    ht.x = __shfl_sync(0xffffffffu, ht.x, 3);
    ht.y = __shfl_sync(0xffffffffu, ht.y, 3);
    if (lane != 0) return;
    if (bad) {
        atomicExch(L.arrive + b, 0);  // no later group: the count is back at zero
        lg_finish(L, b, 0, -1, kStatusBadToken);
    } else if (lg_decide_fast(L, b, i0, na, nb, gp0, gq0, u0) &&
               (kSpan == 1 || lg_decide_fast(L, b, i0 + 1, ma, mb, gp1, gq1, u1))) {
        lg_append_norm(L, b, i0 + kSpan, ht);
    }
    if (g0 >= (uint64_t)L.B) {  // every task of the group has read its slots
        L.grp[g0] = 0ull;
        if (kSpan == 2) L.grp[g0 + 1] = 0ull;
    }
}

// `tasks` norm tasks of slot g (sequence b, position i; span bits sj) have
// stored their pairs: arrives for them, and the group's last arrival decides
// (lg_norm_decide).  The decision's inputs that no task writes -- the span's
// draft tokens, their uniforms and, at position 0, every draft id -- are
// loaded while lane 0's arrival is in flight, so the last arrival waits for
// one round trip (the tokens' logits, the segment pairs and the queue's state
// together), not two.
__device__ __noinline__ void lg_norm_arrive(const LogitsParams &L, int b, int i, uint64_t g, int sj,
                                            int tasks, int lane) {
    const int span = (sj & 3) + 1, r = sj >> 2;
    const int i0 = i - r;  // the span's first position; its slots are g - r, ...
    // lane 1 + k loads position i0 + k's draft token and uniform
    int32_t x = -1, y0 = 0, y1 = 0;
    float u = 0.f;
    const int p = i0 + lane - 1;
    if (lane >= 1 && lane <= span && p < L.K) {
        x = __ldg(L.t + (int64_t)b * L.K + p);
        u = __ldg(L.u_acc + (int64_t)b * L.K + p);
    }
    if (i0 == 0 && L.K > 0) {
        if (lane < L.K) y0 = __ldg(L.t + (int64_t)b * L.K + lane);
        if (lane + 32 < L.K) y1 = __ldg(L.t + (int64_t)b * L.K + lane + 32);
    }
    int last = 0;
    if (lane == 0) last = lg_arrive(L, b, tasks, span);
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();  // lane 0's acquire, before every lane's reads below
    if (lane == 0) SV_TRACE_EVENT(kTrLgLast, (uint32_t)b | ((uint32_t)i0 << 16));
    if (span == 1)
        lg_norm_decide<1>(L, b, i0, g, x, u, y0, y1, lane);
    else
        lg_norm_decide<2>(L, b, i0, g - r, x, u, y0, y1, lane);
}

// The chosen row (pair)'s normalisers, read by lane 0 (after the group's
// publication) and given to every lane.
__device__ __forceinline__ void lg_load_norms(const LogitsParams &L, int b, bool pair, int lane,
                                              RowNorm &np, RowNorm &nq) {
    float4 f0 = make_float4(0.f, 0.f, 0.f, 0.f), f1 = f0;
    if (lane == 0) {
        f0 = __ldcg(L.fnorm + 2 * b);
        if (pair) f1 = __ldcg(L.fnorm + 2 * b + 1);
    }
    np = {__shfl_sync(0xffffffffu, f0.x, 0),
          {__shfl_sync(0xffffffffu, f0.y, 0), __shfl_sync(0xffffffffu, f0.z, 0)}};
    nq = {__shfl_sync(0xffffffffu, f1.x, 0),
          {__shfl_sync(0xffffffffu, f1.y, 0), __shfl_sync(0xffffffffu, f1.z, 0)}};
}

// The precise group's per-segment fp64 sums (p, q), in a segment's pair slot.
__device__ __forceinline__ double2 *lg_precise_slot(const LogitsParams &L, int b, int64_t s) {
    return reinterpret_cast<double2 *>(lg_pair(L, b, s));
}

// `tasks` precise tasks of group g (sequence b, position i) have stored their
// sums: arrives for them; the group's last arrival adds the segments' sums in
// segment order (lane l takes segments l, l + 32, ..., then a fixed
// butterfly), forms p_i(t_i) and q_i(t_i) in fp64 as the oracle does --
// exp((z - M) / tau) / S with M the row's maximum -- and makes the accept
// test (double)u * q < p; then the sequence goes on as after a fast test.
__device__ __noinline__ void lg_precise_arrive(const LogitsParams &L, int b, int i, uint64_t g,
                                               int tasks, int lane) {
    int last = 0;
    if (lane == 0) last = lg_arrive(L, b, tasks, 1);
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();  // lane 0's acquire, before every lane's reads below
    ulonglong2 ht = make_ulonglong2(0ull, 0ull);
    if (L.spec_claims > 0) ht = lg_queue_snapshot(L);  // (only lane 0 uses it)
    double sp = 0.0, sq = 0.0;
    for (int64_t k = lane; k < L.nseg; k += 32) {
        const double2 v = __ldcg(lg_precise_slot(L, b, k));
        sp += v.x;
        sq += v.y;
    }
    sp = warp_sum_f64(sp);
    sq = warp_sum_f64(sq);
    if (lane != 0) return;
    SV_TRACE_EVENT(kTrLgDecide, (uint32_t)b | ((uint32_t)i << 16) | (kLgPrecise << 24));
    const int32_t x = L.t[(int64_t)b * L.K + i];  // checked at position 0
    const float u = L.u_acc[(int64_t)b * L.K + i];
    const float Mp = __ldcg(L.fnorm + 2 * b).x, Mq = __ldcg(L.fnorm + 2 * b + 1).x;
    const double zp = (double)__ldcg(lg_row_p(L, b, i) + x), zq = (double)__ldcg(lg_row_q(L, b, i) + x);
    const double p = exp((zp - (double)Mp) / L.tau) / sp;
    const double q = exp((zq - (double)Mq) / L.tau) / sq;
    if ((double)u * q < p)
        lg_append_norm(L, b, i + 1, ht);
    else
        lg_append_mass(L, lg_group(b, i, kLgMass));  // the fast normalisers are in fnorm
    L.grp[g] = 0ull;  // every task of the group has read it (a precise group is never one of the first B)
}

// `tasks` mass tasks of group g have stored their sums (and every lane's
// stores are ordered before this call): arrives for them; the group's last
// arrival draws and finishes the sequence.
__device__ __noinline__ void lg_mass_arrive(const LogitsParams &L, int b, int n, uint64_t g, int tasks, bool vec,
                               const RowNorm &np, const RowNorm &nq, float ia, float ib, int lane,
                               int kind = (int)kLgMass) {
    if (kind == (int)kLgPrecise) {  // (the bulk-copy workers' precise chunks arrive here)
        lg_precise_arrive(L, b, n, g, tasks, lane);
        return;
    }
    const float *a = lg_row_p(L, b, n);
    const float *c = lg_row_q(L, b, n);
    float2 *seg = L.seg + (int64_t)b * L.nseg;
    float2 *blk = L.blk + (int64_t)b * L.nseg * kBlocks;
    int last = 0;
    if (lane == 0) last = lg_arrive(L, b, tasks, 1);
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();  // lane 0's acquire, before every lane's reads below
    if (lane == 0) {
        atomicExch(L.arrive + b, 0);  // the sequence's last group: back to zero
        SV_TRACE_EVENT(kTrLgDecide, (uint32_t)b | ((uint32_t)n << 16) | (kLgMass << 24));
    }
    DrawInputs in = {};
    in.u = split_uniform(L.u_res[b]);
    int next = draw_core(L.nseg, L.V, seg, blk, nullptr, nullptr, in, lane,
                         [&](int64_t base, dd prefix, dd T) {
                             return lg_search_block(a, c, base, L.V, np, nq, ia, ib, L.c, prefix,
                                                    T, lane);
                         });
    if (next < 0 && c) {
        // p_n == q_n: the residual has no mass; draw from p_n (the probability
        // path's fallback), its sums formed by this warp alone
        for (int64_t k = 0; k < L.nseg; ++k)
            lg_mass_segment(a, nullptr, L, seg, blk, k, vec, np, nq, ia, ib, lane);
        __threadfence_block();
        __syncwarp();
        next = draw_core(L.nseg, L.V, seg, blk, nullptr, nullptr, in, lane,
                         [&](int64_t base, dd prefix, dd T) {
                             return lg_search_block(a, nullptr, base, L.V, np, nq, ia, ib, L.c,
                                                    prefix, T, lane);
                         });
    }
    if (lane == 0) {
        if (g >= (uint64_t)L.B) L.grp[g] = 0ull;
        lg_finish(L, b, n, next, next < 0 ? kStatusZeroMass : 0u);
    }
}

// ---------------------------------------------------------------------------
// plain-load workers (rows that are not 16-byte aligned, or in host memory):
// every warp takes one segment task at a time and loads it itself

__device__ void lg_norm_task(const LogitsParams &L, int b, int i, int64_t s, uint64_t g, int sj,
                             bool vec, int lane) {
    const float *a = lg_row_p(L, b, i);
    const float *c = lg_row_q(L, b, i);
    const int64_t base = s * kSeg;
    const int64_t end = min(L.V, base + kSeg);
    const float4 none = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
    float4 xa[kVecPerLane], xb[kVecPerLane];
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
        const int64_t e = base + 4 * (lane + 32 * k);
        xa[k] = e < end ? load4(a, e, end, vec) : none;
        xb[k] = (c && e < end) ? load4(c, e, end, vec) : none;
    }
    const RowNorm oa = seg_norm(xa, L.c);
    const RowNorm ob = c ? seg_norm(xb, L.c) : RowNorm{kNegInf, {0.f, 0.f}};
    if (lane == 0) lg_store_pair(L, b, s, sj >> 2, oa, ob);
    lg_norm_arrive(L, b, i, g, sj, 1, lane);
}

__device__ void lg_mass_task(const LogitsParams &L, int b, int n, int64_t s, uint64_t g, bool vec,
                             int lane) {
    const float *a = lg_row_p(L, b, n);
    const float *c = lg_row_q(L, b, n);
    RowNorm np, nq;
    lg_load_norms(L, b, c != nullptr, lane, np, nq);  // after lane 0's acquire of the group
    const float ia = __frcp_rn(np.s.hi), ib = c ? __frcp_rn(nq.s.hi) : 0.f;
    lg_mass_segment(a, c, L, L.seg + (int64_t)b * L.nseg, L.blk + (int64_t)b * L.nseg * kBlocks,
                    s, vec, np, nq, ia, ib, lane);
    __threadfence();  // this lane's sums, before the arrival
    __syncwarp();
    lg_mass_arrive(L, b, n, g, 1, vec, np, nq, ia, ib, lane);
}

__device__ __noinline__ void lg_precise_task(const LogitsParams &L, int b, int i, int64_t s, uint64_t g,
                                             bool vec, int lane) {
    const float *a = lg_row_p(L, b, i);
    const float *c = lg_row_q(L, b, i);
    const int64_t base = s * kSeg;
    const int64_t end = min(L.V, base + kSeg);
    const float4 none = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
    float4 xa[kVecPerLane], xb[kVecPerLane];
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
        const int64_t e = base + 4 * (lane + 32 * k);
        xa[k] = e < end ? load4(a, e, end, vec) : none;
        xb[k] = e < end ? load4(c, e, end, vec) : none;
    }
    float Mp = 0.f, Mq = 0.f;
    if (lane == 0) {  // after lane 0's acquire of the group
        Mp = __ldcg(L.fnorm + 2 * b).x;
        Mq = __ldcg(L.fnorm + 2 * b + 1).x;
    }
    Mp = __shfl_sync(0xffffffffu, Mp, 0);
    Mq = __shfl_sync(0xffffffffu, Mq, 0);
    const double sp = warp_sum_f64(precise_terms(xa, Mp, L.tau));
    const double sq = warp_sum_f64(precise_terms(xb, Mq, L.tau));
    if (lane == 0) *lg_precise_slot(L, b, s) = make_double2(sp, sq);
    __threadfence();
    __syncwarp();
    lg_precise_arrive(L, b, i, g, 1, lane);
}

__global__ void __launch_bounds__(kLgThreads, 2) logits_task_kernel(const LogitsParams L) {
    const int lane = threadIdx.x & 31;
    const bool vec = lg_vec(L);
    const uint64_t nseg = (uint64_t)L.nseg;
    wait_for_primary_grid();
    unsigned long long h = 0;
    if (lane == 0) h = atomicAdd(L.head, 1ull);
    h = __shfl_sync(0xffffffffu, h, 0);
    while (true) {
        const uint64_t g = h / nseg;
        if (g >= (uint64_t)L.ngroups) break;
        unsigned long long d = 0;
        if (lane == 0) d = lg_wait_group(L, g);
        d = __shfl_sync(0xffffffffu, d, 0);
        if (!d) break;
        // the next task is claimed now: its number is needed only after this one
        unsigned long long hn = 0;
        if (lane == 0) hn = atomicAdd(L.head, 1ull);
        const int b = (int)(uint32_t)d;
        const int i = (int)((d >> 32) & 0xffu);
        const int64_t s = (int64_t)(h % nseg);
        const uint32_t kind = (uint32_t)((d >> 40) & 3u);
        if (kind == kLgNorm)
            lg_norm_task(L, b, i, s, g, lg_span_bits(d), vec, lane);
        else if (kind == kLgPrecise)
            lg_precise_task(L, b, i, s, g, vec, lane);
        else
            lg_mass_task(L, b, i, s, g, vec, lane);
        h = __shfl_sync(0xffffffffu, hn, 0);
    }
    // the last worker out returns the queue counters to zero for the next call
    if (lane == 0) {
        __threadfence();
        if (atomicAdd(L.nexit, 1u) == gridDim.x * kLgWarps - 1) {
            atomicExch(L.head, 0ull);
            atomicExch(L.tail, 0ull);
            atomicExch(L.pend_head, 0ull);
            atomicExch(L.pend_tail, 0ull);
            atomicExch(L.ndone, 0u);
            atomicExch(L.nexit, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// bulk-copy workers (16-byte-aligned device rows): per CTA one producer warp
// takes chunks of L.chunk segment tasks of one group from the queue and
// moves their row segments into a ring of shared-memory stages (kLgStageSegs
// segments of each row per stage) with cp.async.bulk; kLgConsumers consumer
// warps take the stages' segments in order, one segment per ticket, and run
// the tasks on them.  The producer waits for the group of its next chunk
// (bounded, as above); the copies already issued keep the consumers busy
// meanwhile.

struct LgStage {
    const float *g0;  // global start of the stage's p part and of its q part (null: one row)
    const float *g1;
    unsigned long long g;  // group
    int64_t s;        // first segment
    int kind;         // kLgNorm, kLgMass, 0 = stop
    int b, i;
    int ns;           // segments in the stage (1 .. kLgStageSegs)
    int n;            // elements of the stage's part of a row
    int c;            // elements delivered by the copies (a multiple of 4)
    int slot;         // the chunk's counter in LgShared::left
    int tasks;        // stages of the chunk
    int sj;           // the slot's span bits (norm stages)
    float4 np, nq;    // mass stages: the row (pair)'s normalisers (m, s.hi, s.lo)
};

// Chunks whose stages are counted in shared memory at once: a chunk's counter
// is reused kLgSlots chunks later, and only once it is back at zero.
constexpr int kLgSlots = 32;

// The ring: kLgStages stages, each kLgStageSegs consecutive segments of the
// row pair (or of one row), p's part first.
#ifndef SV_LG_STAGE_SEGS
#define SV_LG_STAGE_SEGS 4
#endif
#ifndef SV_LG_STAGES
#define SV_LG_STAGES 3
#endif
constexpr int kLgStageSegs = SV_LG_STAGE_SEGS;
constexpr int kLgStages = SV_LG_STAGES;
constexpr int kLgPartBytes = kLgStageSegs * kSeg * 4;
constexpr int kLgStageBytes = 2 * kLgPartBytes;
static_assert(kLgStages <= 32, "stage bookkeeping is a 32-bit mask");
// A stage is taken by kLgStageSegs consumers, one segment each (a ticket is a
// share of a stage), so no warp holds a stage for more than one segment's
// work.  A share's parity wait is unambiguous while no consumer can take a
// share of the same position two fills ahead: the other consumers can hold
// at most (stages - 1) * shares + shares - 1 filled shares beyond it, so
// consumers <= stages * shares + 1.  Seven consumers (registers allow no
// more at two CTAs per SM).
constexpr int kLgShares = kLgStageSegs;
constexpr int kLgConsumers = 7;
static_assert(kLgConsumers <= kLgStages * kLgShares + 1, "too few ring stages for the consumers");
constexpr int kLgProducerWarp = kLgConsumers;

// A chunk the producer has taken.
struct LgChunk {
    unsigned long long g, d;  // group and its record
    uint64_t ci;              // chunk index within the group
    float4 np, nq;            // mass chunks: the normalisers
};

struct LgShared {
    int ticket;  // next stage a consumer takes (ring position = ticket % kLgStages)
    unsigned long long full[kLgStages];
    unsigned long long empty[kLgStages];
    LgStage meta[kLgStages];
    int left[kLgSlots];  // stage shares of the chunk not yet done (0: free)
};
static_assert(sizeof(LgShared) <= kTmaBufOffset, "shared header too large");
constexpr int kLgRingThreads = (kLgConsumers + 1) * 32;
constexpr int kLgRingSmemBytes = kTmaBufOffset + kLgStages * kLgStageBytes;

struct LgProducer {
    LgShared &sh;
    unsigned char *buf;
    uint32_t *status;
    int lane;
    int k = 0;           // next stage
    uint32_t phase = 0;  // flips each time k wraps
    uint32_t used = 0;   // bit i: stage i has been filled at least once
    uint32_t parity = 0; // bit i: phase of the last fill of stage i
    bool ok = true;

    __device__ LgProducer(LgShared &sh_, unsigned char *buf_, uint32_t *status_, int lane_)
        : sh(sh_), buf(buf_), status(status_), lane(lane_) {}

    // Fills the next stage once its consumer released it (warp-uniform; lane 0 acts).
    __device__ void issue(const LgStage &m) {
        if (!ok) return;
        bool good = true;
        if (lane == 0) {
            good = mbar_wait(&sh.empty[k], phase ^ 1u);
            if (good) {
                sh.meta[k] = m;
                const uint32_t part = 4u * (uint32_t)m.c;
                mbar_arrive_expect_tx(&sh.full[k], m.g1 ? 2u * part : part);
                unsigned char *dst = buf + (size_t)k * kLgStageBytes;
                if (part) {
                    bulk_copy_g2s(dst, m.g0, part, &sh.full[k]);
                    if (m.g1) bulk_copy_g2s(dst + kLgPartBytes, m.g1, part, &sh.full[k]);
                }
            } else {
                atomicOr(status, kStatusTimeout);
            }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
            ok = false;
            return;
        }
        used |= 1u << k;
        parity = (parity & ~(1u << k)) | (phase << k);
        if (++k == kLgStages) {
            k = 0;
            phase ^= 1u;
        }
    }
};

// Issues the stages of chunk ci (segments [ci * L.chunk, ...)) of group g.
__device__ void lg_issue_chunk(const LogitsParams &L, LgShared &sh, LgProducer &pr,
                               const LgChunk &ch, uint32_t &nchunks_here, int lane) {
    const uint64_t g = ch.g, ci = ch.ci;
    const unsigned long long d = ch.d;
    const int64_t s0 = (int64_t)ci * L.chunk;
    const int64_t s1 = min((int64_t)L.nseg, s0 + L.chunk);
    // the chunk's stage counter: free once the chunk kLgSlots before it is done
    const int slot = (int)(nchunks_here++ % kLgSlots);
    bool free = true;
    if (lane == 0) {
        IdleClock clk;
        while (*(volatile int *)&sh.left[slot] != 0) {
            if (!clk.idle(64)) {
                atomicOr(L.status, kStatusTimeout);
                free = false;
                break;
            }
        }
        if (free)
            *(volatile int *)&sh.left[slot] =
                (int)((s1 - s0 + kLgStageSegs - 1) / kLgStageSegs) * kLgShares;
    }
    if (!__shfl_sync(0xffffffffu, free, 0)) {
        pr.ok = false;
        return;
    }
    LgStage m = {};
    m.g = g;
    m.b = (int)(uint32_t)d;
    m.i = (int)((d >> 32) & 0xffu);
    m.kind = (int)((d >> 40) & 3u);
    m.sj = lg_span_bits(d);
    m.slot = slot;
    m.tasks = (int)(s1 - s0);
    m.np = ch.np;
    m.nq = ch.nq;
    const float *a = lg_row_p(L, m.b, m.i);
    const float *c = lg_row_q(L, m.b, m.i);
    // a precise stage (rare) is read by its consumer from global memory and
    // takes the consumers' out-of-line path: no copy, and the temperature in
    // np.w (an fp32 value, so exact)
    const bool precise = m.kind == (int)kLgPrecise;
    if (precise) m.np.w = (float)L.tau;
    for (int64_t s = s0; s < s1; s += kLgStageSegs) {
        const int64_t base = s * kSeg;
        m.s = s;
        m.ns = (int)min((int64_t)kLgStageSegs, s1 - s);
        m.n = (int)min((int64_t)m.ns * kSeg, L.V - base);
        m.c = precise ? 0 : m.n & ~3;
        m.g0 = a + base;
        m.g1 = c ? c + base : nullptr;
        pr.issue(m);
    }
}

// Chunks are taken in queue order (the first B groups, then the appended
// ones as they come).  The next chunk is claimed only once the current one's
// stages are issued: a claim taken earlier would tie an appended group's
// chunk to a worker that is still busy while others wait for work, and that
// worker's delay would be the group's (the ring's stages in flight cover the
// claim's round trip).
__device__ void lg_produce(const LogitsParams &L, LgShared &sh, unsigned char *buf, int lane) {
    LgProducer pr(sh, buf, L.status, lane);
    const uint64_t nchunk = (uint64_t)((L.nseg + L.chunk - 1) / L.chunk);
    uint32_t nchunks_here = 0;
    unsigned long long h = 0;
    if (lane == 0) h = atomicAdd(L.head, 1ull);
    h = __shfl_sync(0xffffffffu, h, 0);
    while (pr.ok) {
        LgChunk ch = {};
        ch.g = h / nchunk;
        if (ch.g >= (uint64_t)L.ngroups) break;
        unsigned long long d = 0;
        if (lane == 0) {
            SV_TRACE_EVENT(kTrLgClaim, (uint32_t)ch.g | ((uint32_t)(h % nchunk) << 24));
            d = lg_wait_group(L, ch.g);
            SV_TRACE_EVENT(kTrLgReady, (uint32_t)ch.g);
            if (d && ((d >> 40) & 3u) >= kLgMass) {  // mass and precise; after the group's acquire
                const int b = (int)(uint32_t)d;
                ch.np = __ldcg(L.fnorm + 2 * b);
                if ((int)((d >> 32) & 0xffu) < L.K) ch.nq = __ldcg(L.fnorm + 2 * b + 1);
            }
        }
        ch.d = __shfl_sync(0xffffffffu, d, 0);
        if (!ch.d) break;
        ch.np = make_float4(__shfl_sync(0xffffffffu, ch.np.x, 0), __shfl_sync(0xffffffffu, ch.np.y, 0),
                            __shfl_sync(0xffffffffu, ch.np.z, 0), 0.f);
        ch.nq = make_float4(__shfl_sync(0xffffffffu, ch.nq.x, 0), __shfl_sync(0xffffffffu, ch.nq.y, 0),
                            __shfl_sync(0xffffffffu, ch.nq.z, 0), 0.f);
        ch.ci = h % nchunk;
        lg_issue_chunk(L, sh, pr, ch, nchunks_here, lane);
        if (lane == 0) {
            SV_TRACE_EVENT(kTrLgIssued, (uint32_t)ch.g);
            h = atomicAdd(L.head, 1ull);
        }
        h = __shfl_sync(0xffffffffu, h, 0);
    }
    // tell every consumer to stop (each stop stage serves kLgShares of them)
    for (int w = 0; w < (kLgConsumers + kLgShares - 1) / kLgShares; ++w) {
        LgStage m = {};
        pr.issue(m);
    }
    if (!pr.ok && lane == 0) {
        // a wait gave up: let the copies still in flight land before returning
        for (int i = 0; i < kLgStages; ++i)
            if (pr.used & (1u << i)) mbar_wait(&sh.full[i], (pr.parity >> i) & 1u);
    }
}

// Element e of a staged segment (the copy delivered the first c elements;
// the last 1-3 of a ragged row come from global memory), pad past n.
__device__ __forceinline__ float4 lg_stage4(const float *sm, const float *g, int n, int c, int e,
                                            float pad) {
    if (e + 3 < c) return *reinterpret_cast<const float4 *>(sm + e);
    float4 x;
    x.x = e < n ? part_elem(sm, g, c, e) : pad;
    x.y = e + 1 < n ? part_elem(sm, g, c, e + 1) : pad;
    x.z = e + 2 < n ? part_elem(sm, g, c, e + 2) : pad;
    x.w = e + 3 < n ? part_elem(sm, g, c, e + 3) : pad;
    return x;
}

// Normalisers of a staged segment that is not a full 1024 elements (the last
// of a row; out of line, so the full-segment loop stays small).
__device__ __noinline__ RowNorm lg_ragged_norm(const float *sm, const float *g, int n, int c,
                                               float cc, int lane) {
    float4 x[kVecPerLane];
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) x[j] = lg_stage4(sm, g, n, c, 4 * (lane + 32 * j), kNegInf);
    return seg_norm(x, cc);
}

// Masses of a staged segment that is not a full 1024 elements, into the
// segment's sums (out of line, as above).
__device__ __noinline__ void lg_ragged_mass(const float *sp, const float *sq, const LgStage &m,
                                            const RowNorm &np, const RowNorm &nq, float ia,
                                            float ib, float2 *seg, float2 *blk, float cc,
                                            int lane) {
    if (m.kind == (int)kLgPrecise) {
        // a precise stage (no copy, so it always comes here): the segment's
        // fp64 sums from global memory into its slot; m.np.x and m.nq.x are
        // the rows' maxima, m.np.w the temperature (a float, exactly)
        float4 xa[kVecPerLane], xb[kVecPerLane];
#pragma unroll
        for (int v = 0; v < kVecPerLane; ++v) {
            xa[v] = lg_stage4(sp, m.g0, m.n, 0, 4 * (lane + 32 * v), kNegInf);
            xb[v] = lg_stage4(sq, m.g1, m.n, 0, 4 * (lane + 32 * v), kNegInf);
        }
        const double tau = (double)m.np.w;
        const double s0 = warp_sum_f64(precise_terms(xa, m.np.x, tau));
        const double s1 = warp_sum_f64(precise_terms(xb, m.nq.x, tau));
        if (lane == 0)
            *reinterpret_cast<double2 *>(reinterpret_cast<float4 *>(blk) + 2 * m.s) = make_double2(s0, s1);
        return;
    }
    const bool pair = m.g1 != nullptr;
    dd v[kBlocks];
#pragma unroll
    for (int j = 0; j < kBlocks; ++j) {
        const int e = 4 * (lane + 32 * j);
        float4 ms = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < m.n) {
            const float4 x = lg_stage4(sp, m.g0, m.n, m.c, e, 0.f);
            const float4 y = pair ? lg_stage4(sq, m.g1, m.n, m.c, e, 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
            ms.x = lg_mass(x.x, y.x, pair, np, nq, ia, ib, cc);
            ms.y = e + 1 < m.n ? lg_mass(x.y, y.y, pair, np, nq, ia, ib, cc) : 0.f;
            ms.z = e + 2 < m.n ? lg_mass(x.z, y.z, pair, np, nq, ia, ib, cc) : 0.f;
            ms.w = e + 3 < m.n ? lg_mass(x.w, y.w, pair, np, nq, ia, ib, cc) : 0.f;
        }
        v[j] = dd{sum4(ms), 0.f};
    }
    store_sums(seg, blk, m.s, v, lane);
}

// Waits (bounded) until the stage of share ticket t holds its fill (the same
// two-step wait as wait_ticket, per stage ticket t / kLgShares, on this ring's
// size; kLgConsumers keeps it unambiguous).
__device__ __forceinline__ bool lg_wait_ticket(unsigned long long *full, unsigned long long *empty,
                                               int t) {
    const int ts = t / kLgShares;
    const int k = ts % kLgStages;
    const uint32_t phase = (uint32_t)(ts / kLgStages) & 1u;
    return mbar_wait(&empty[k], phase ^ 1u) && mbar_wait(&full[k], phase);
}

// Counts this warp's stage (its global stores made before the call) in its
// chunk; true for the warp that completes the chunk, which then arrives for
// all of the chunk's stages.  The CTA-scope fences make every counted stage's
// stores part of what the completing warp's release at GPU scope publishes.
__device__ __forceinline__ bool lg_chunk_done(LgShared &sh, int slot, int lane) {
    __threadfence_block();
    __syncwarp();
    int done = 0;
    if (lane == 0) done = atomicSub(&sh.left[slot], 1) == 1;
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done) __threadfence_block();
    return done;
}

__device__ void lg_consume(const LogitsParams &L, LgShared &sh, unsigned char *buf, int lane) {
    const RowNorm none = {kNegInf, {0.f, 0.f}};
    while (true) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&sh.ticket, 1);
        t = __shfl_sync(0xffffffffu, t, 0);
        const int k = (t / kLgShares) % kLgStages;
        const int j = t % kLgShares;  // this share's segment of the stage
        const float *sp = reinterpret_cast<const float *>(buf + (size_t)k * kLgStageBytes);
        const float *sq = reinterpret_cast<const float *>(buf + (size_t)k * kLgStageBytes + kLgPartBytes);
        if (!__all_sync(0xffffffffu, lg_wait_ticket(sh.full, sh.empty, t))) {
            if (lane == 0) atomicOr(L.status, kStatusTimeout);
            return;
        }
        const LgStage m = sh.meta[k];
        if (m.kind == 0) {  // released, so a stop may follow it round the ring
            release_stage(sh.empty, k, lane);
            return;
        }
        const bool pair = m.g1 != nullptr;
        const int o = j * kSeg;  // the segment's offset in the stage
        if (m.kind == (int)kLgNorm) {
            if (j < m.ns) {
                RowNorm oa, ob = none;
                if (o + kSeg <= m.c) {  // a full segment, straight from shared memory
                    const float4 *p4 = reinterpret_cast<const float4 *>(sp + o);
                    const float4 *q4 = reinterpret_cast<const float4 *>(sq + o);
                    float4 xa[kVecPerLane], xb[kVecPerLane];
#pragma unroll
                    for (int v = 0; v < kVecPerLane; ++v) {
                        xa[v] = p4[lane + 32 * v];
                        if (pair) xb[v] = q4[lane + 32 * v];
                    }
                    release_stage(sh.empty, k, lane);
                    oa = seg_norm(xa, L.c);
                    if (pair) ob = seg_norm(xb, L.c);
                } else {
                    const int n = min(kSeg, m.n - o), c = max(0, min(kSeg, m.c - o));
                    oa = lg_ragged_norm(sp + o, m.g0 + o, n, c, L.c, lane);
                    if (pair) ob = lg_ragged_norm(sq + o, m.g1 + o, n, c, L.c, lane);
                    release_stage(sh.empty, k, lane);
                }
                if (lane == 0) lg_store_pair(L, m.b, m.s + j, m.sj >> 2, oa, ob);
            } else {
                release_stage(sh.empty, k, lane);
            }
            if (lg_chunk_done(sh, m.slot, lane)) {
                if (lane == 0) SV_TRACE_EVENT(kTrLgChunkDone, (uint32_t)m.g);
                lg_norm_arrive(L, m.b, m.i, m.g, m.sj, m.tasks, lane);
            }
        } else {  // mass and precise stages (a precise one has no copy: see lg_issue_chunk)
            const RowNorm np = {m.np.x, {m.np.y, m.np.z}}, nq = {m.nq.x, {m.nq.y, m.nq.z}};
            const float ia = __frcp_rn(np.s.hi), ib = pair ? __frcp_rn(nq.s.hi) : 0.f;
            float2 *seg = L.seg + (int64_t)m.b * L.nseg;
            float2 *blk = L.blk + (int64_t)m.b * L.nseg * kBlocks;
            if (j < m.ns && o + kSeg <= m.c) {
                const float4 *p4 = reinterpret_cast<const float4 *>(sp + o);
                const float4 *q4 = reinterpret_cast<const float4 *>(sq + o);
                dd v[kBlocks];
#pragma unroll
                for (int w = 0; w < kBlocks; ++w) {
                    const float4 x = p4[lane + 32 * w];
                    const float4 y = pair ? q4[lane + 32 * w] : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[w] = dd{sum4(make_float4(lg_mass(x.x, y.x, pair, np, nq, ia, ib, L.c),
                                               lg_mass(x.y, y.y, pair, np, nq, ia, ib, L.c),
                                               lg_mass(x.z, y.z, pair, np, nq, ia, ib, L.c),
                                               lg_mass(x.w, y.w, pair, np, nq, ia, ib, L.c))),
                              0.f};
                }
                release_stage(sh.empty, k, lane);
                store_sums(seg, blk, m.s + j, v, lane);
            } else if (j < m.ns) {
                LgStage mj = m;
                mj.s = m.s + j;
                mj.n = min(kSeg, m.n - o);
                mj.c = max(0, min(kSeg, m.c - o));
                mj.g0 = m.g0 + o;
                mj.g1 = pair ? m.g1 + o : nullptr;
                lg_ragged_mass(sp + o, sq + o, mj, np, nq, ia, ib, seg, blk, L.c, lane);
                release_stage(sh.empty, k, lane);
            } else {
                release_stage(sh.empty, k, lane);
            }
            if (lg_chunk_done(sh, m.slot, lane)) {
                if (lane == 0) SV_TRACE_EVENT(kTrLgChunkDone, (uint32_t)m.g);
                lg_mass_arrive(L, m.b, m.i, m.g, m.tasks, true, np, nq, ia, ib, lane, m.kind);
            }
        }
    }
}

__global__ void __launch_bounds__(kLgRingThreads, 2) logits_ring_kernel(const LogitsParams L) {
    extern __shared__ __align__(1024) unsigned char smem[];
    LgShared &sh = *reinterpret_cast<LgShared *>(smem);
    unsigned char *buf = smem + kTmaBufOffset;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kLgStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], kLgShares);  // released by every share
        }
        sh.ticket = 0;
        SV_TRACE_INIT();
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x < kLgSlots) sh.left[threadIdx.x] = 0;
    __syncthreads();
    wait_for_primary_grid();
    SV_TRACE_START(false);
    if (warp == kLgProducerWarp)
        lg_produce(L, sh, buf, lane);
    else
        lg_consume(L, sh, buf, lane);
    // the last CTA out returns the queue counters to zero for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(L.nexit, 1u) == gridDim.x - 1) {
            atomicExch(L.head, 0ull);
            atomicExch(L.tail, 0ull);
            atomicExch(L.pend_head, 0ull);
            atomicExch(L.pend_tail, 0ull);
            atomicExch(L.ndone, 0u);
            atomicExch(L.nexit, 0u);
        }
    }
    SV_TRACE_FINISH();
}

}  // namespace sv
