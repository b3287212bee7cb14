// sv_tma.cuh -- the streaming stage of a verification round as a bulk-copy
// pipeline (sm_103a), used for 16-byte-aligned device rows when the batch has
// fewer sequences than SMs (larger batches run sv_item.cuh's single launch);
// the ring primitives here serve both.
//
// A persistent CTA has one producer warp and eight consumer warps.  The
// producer takes chunks (kChunkSegs consecutive 1024-element segments of one
// sequence) from a device-wide counter, reads what the scan kernel cached for
// the sequence (the first rejection n of a sampling sequence, or the draft
// tokens and p_i(t_i) of a greedy one) one chunk ahead of use, and moves the
// chunk's row segments from HBM into a ring of shared-memory stages with
// cp.async.bulk.  Consumers reduce the stages: the double-fp32 mass sum of a
// residual (or bonus-row) segment, or a greedy segment's maximum folded into
// the row's 64-bit key while a draft-token miss raises the sequence's flag.
// Loads stay in flight while consumers compute, so the bytes in flight are
// set by the ring, not by any warp's registers.  Nothing here fences or waits
// for another CTA: the decide kernel that follows turns the partials into
// outputs.
//
// Greedy sequences are streamed one row at a time: the producer keeps up to
// kSlots greedy chunks open and moves one to its next row only after every
// stage of the current row was consumed and neither this CTA nor the
// per-sequence flag has seen a miss at or before that row, so rows past the
// first miss are not read.
//
// Every wait (on an mbarrier or on the consumers) is bounded by kWaitLimitNs
// of wall-clock time: on timeout the warp sets SV_STATUS_TIMEOUT (the round's
// outputs are then not meaningful) and leaves its loop; the producer then
// waits, again bounded, for its copies still in flight.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kTmaConsumers = 8;
constexpr int kProducerWarp = kTmaConsumers;
constexpr int kTmaThreads = (kTmaConsumers + 1) * 32;
// Shared-memory ring stages; consumers take full stages in order through a
// shared ticket, so a stage's turn-around is copy latency plus the processing
// time of whichever consumer is free, not of one fixed warp.
#ifndef SV_STAGES
#define SV_STAGES 11
#endif
constexpr int kStages = SV_STAGES;
// wait_ticket tells a stage's fills apart by barrier parity, which is only
// unambiguous while no consumer can take ticket t + 2 * kStages before ticket
// t's stage is released.  The other consumers can hold at most kStages - 1
// filled tickets beyond t, so that holds while consumers <= kStages + 1.
static_assert(kTmaConsumers <= kStages + 1, "too few ring stages for the consumers");
constexpr int kPartBytes = kSeg * 4;        // one segment of one row
constexpr int kStageBytes = 2 * kPartBytes;
constexpr int kChunkSegs = 8;               // segments per chunk
constexpr int kChunkSlots = 32;             // greedy chunks a CTA tracks until they are consumed
constexpr int kSlots = 4;                   // greedy chunks a producer keeps open

enum StageKind : int { kStop = 0, kPair = 1, kMass = 2, kArgmax = 3 };

struct StageMeta {
    const float *g0;  // global start of part 0 / part 1 (elements past c0/c1 are read from here)
    const float *g1;
    int kind;
    int b;
    int s;            // first segment (kMass / kArgmax: parts are segments s and s + 1)
    int nparts;
    int n0, n1;       // elements in part 0 / 1
    int c0, c1;       // elements of part 0 / 1 delivered by the bulk copy (multiple of 4)
    int row;          // greedy: row index
    int cslot;        // chunk slot the stage belongs to
    int tok;          // greedy: draft token of the row, -1 for the bonus row
    float pt;         // greedy: p_row(tok)
};

struct TmaShared {
    int ticket;  // next stage a consumer takes (ring position = ticket % kStages)
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    StageMeta meta[kStages];
    int cs_state[kChunkSlots];     // greedy chunk slots: 0 free, 1 open
    int cs_consumed[kChunkSlots];  // stages of the chunk processed so far
    int cs_missed[kChunkSlots];    // kFlagBase - row of a miss seen in the chunk
    int g_tok[kSlots][kMaxK];      // greedy: draft tokens and p_i(t_i) of open chunks
    float g_pt[kSlots][kMaxK];
};

constexpr int kTmaBufOffset = 4096;  // stage buffers start here in dynamic shared memory
static_assert(sizeof(TmaShared) <= kTmaBufOffset, "shared header too large");
constexpr int kTmaSmemBytes = kTmaBufOffset + kStages * kStageBytes;

// ---------------------------------------------------------------------------
// producer

// What the producer knows about a chunk, per lane: positions lane and
// lane + 32 of a greedy sequence's draft tokens and their target probability.
struct ChunkPre {
    int c;          // chunk index (>= P.nchunks: none)
    int b, s0, s1;
    int rule;
    int32_t ns;     // from the scan kernel: n + 1 (sampling), 1 (greedy), kNBad
    int32_t t0, t1;
    float pt0, pt1;
};

struct Producer {
    const Params &P;
    TmaShared &sh;
    unsigned char *buf;
    int lane;
    int cps;             // chunks per sequence
    int k = 0;           // next stage
    uint32_t phase = 0;  // flips each time k wraps
    uint32_t used = 0;   // bit i: stage i has been filled at least once
    uint32_t parity = 0; // bit i: phase of the last fill of stage i
    bool ok = true;

    __device__ Producer(const Params &P_, TmaShared &sh_, unsigned char *buf_, int lane_)
        : P(P_), sh(sh_), buf(buf_), lane(lane_) {
        cps = (P.nseg + kChunkSegs - 1) / kChunkSegs;
    }

    __device__ void fail() {
        if (ok && lane == 0) atomicOr(P.status, kStatusTimeout);
        ok = false;
    }

    // Fills the next stage: waits until its consumer released it, publishes
    // the metadata and starts the copies.  Warp-uniform; lane 0 acts.
    __device__ void issue(const StageMeta &m) {
        if (!ok) return;
        bool good = true;
        if (lane == 0) {
            good = mbar_wait(&sh.empty[k], phase ^ 1u);
            if (good) {
                sh.meta[k] = m;
                const uint32_t bytes = 4u * (uint32_t)(m.c0 + m.c1);
                mbar_arrive_expect_tx(&sh.full[k], bytes);
                unsigned char *dst = buf + (size_t)k * kStageBytes;
                if (m.c0) bulk_copy_g2s(dst, m.g0, 4u * m.c0, &sh.full[k]);
                if (m.c1) bulk_copy_g2s(dst + kPartBytes, m.g1, 4u * m.c1, &sh.full[k]);
            }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
            fail();
            return;
        }
        used |= 1u << k;
        parity = (parity & ~(1u << k)) | (phase << k);
        if (++k == kStages) {
            k = 0;
            phase ^= 1u;
        }
    }

    __device__ static void part(const float *row, int s, int64_t V, const float *&g, int &n, int &c) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t rem = V - base;
        n = (int)(rem < kSeg ? rem : kSeg);
        c = n & ~3;
        g = row + base;
    }

    __device__ int grab() {
        int c = 0;
        if (lane == 0) c = (int)atomicAdd(P.queue, 1u);
        return __shfl_sync(0xffffffffu, c, 0);
    }

    // The scan kernel's cached data for a chunk's sequence, loaded one chunk
    // before it is needed.
    template <int kRule>
    __device__ ChunkPre load(int c) {
        ChunkPre x = {};
        x.c = c;
        if (c >= P.nchunks) return x;
        x.b = c / cps;
        const int g = c - x.b * cps;
        x.s0 = g * kChunkSegs;
        x.s1 = min(P.nseg, x.s0 + kChunkSegs);
        x.rule = kRule == kPerSequence ? (int)P.mode[x.b] : kRule;
        x.ns = ld_l2(P.nstate + x.b);
        if (x.rule == kGreedy) {
            const int64_t tb = (int64_t)x.b * P.K;
            if (lane < P.K) {
                x.t0 = P.t[tb + lane];
                x.pt0 = ld_l2(P.ptok + tb + lane);
            }
            if (lane + 32 < P.K) {
                x.t1 = P.t[tb + lane + 32];
                x.pt1 = ld_l2(P.ptok + tb + lane + 32);
            }
        }
        return x;
    }

    // A free chunk slot for a greedy chunk (one of them is always free while
    // fewer than kSlots greedy chunks are open).
    __device__ int take_chunk_slot() {
        const bool free = *(volatile int *)&sh.cs_state[lane] == 0;
        const unsigned m = __ballot_sync(0xffffffffu, free);
        return m ? __ffs(m) - 1 : -1;
    }

    __device__ void open_chunk(int x) {
        if (lane == 0) {
            sh.cs_consumed[x] = 0;
            sh.cs_missed[x] = 0;
            *(volatile int *)&sh.cs_state[x] = 1;
        }
        __syncwarp();
    }

    __device__ void free_chunk(int x) {
        if (lane == 0) *(volatile int *)&sh.cs_state[x] = 0;
        __syncwarp();
    }

    // Sampling chunk: residual pairs of row n, or pairs of p_K segments.
    __device__ int sample_chunk(const ChunkPre &ci) {
        const int x = -1;  // sampling stages are not tracked per chunk
        const int n = ci.ns - 1;
        int stages = 0;
        if (n < P.K) {
            const float *pr = prow(P, ci.b, n), *qr = qrow(P, ci.b, n);
            for (int s = ci.s0; s < ci.s1; ++s) {
                StageMeta m = {};
                m.kind = kPair;
                m.b = ci.b;
                m.s = s;
                m.nparts = 2;
                m.cslot = x;
                part(pr, s, P.V, m.g0, m.n0, m.c0);
                part(qr, s, P.V, m.g1, m.n1, m.c1);
                issue(m);
                ++stages;
            }
        } else {
            const float *pr = prow(P, ci.b, P.K);
            for (int s = ci.s0; s < ci.s1; s += 2) {
                StageMeta m = {};
                m.kind = kMass;
                m.b = ci.b;
                m.s = s;
                m.nparts = s + 1 < ci.s1 ? 2 : 1;
                m.cslot = x;
                part(pr, s, P.V, m.g0, m.n0, m.c0);
                if (m.nparts == 2) part(pr, s + 1, P.V, m.g1, m.n1, m.c1);
                issue(m);
                ++stages;
            }
        }
        return stages;
    }

    // Greedy chunk row: pairs of segments of row `row`.
    __device__ int greedy_row(int b, int s0, int s1, int x, int gs, int row) {
        const float *pr = prow(P, b, row);
        int stages = 0;
        for (int s = s0; s < s1; s += 2) {
            StageMeta m = {};
            m.kind = kArgmax;
            m.b = b;
            m.s = s;
            m.nparts = s + 1 < s1 ? 2 : 1;
            m.row = row;
            m.cslot = x;
            m.tok = row < P.K ? sh.g_tok[gs][row] : -1;
            m.pt = row < P.K ? sh.g_pt[gs][row] : 0.f;
            part(pr, s, P.V, m.g0, m.n0, m.c0);
            if (m.nparts == 2) part(pr, s + 1, P.V, m.g1, m.n1, m.c1);
            issue(m);
            ++stages;
        }
        return stages;
    }
};

template <int kRule>
__device__ void tma_produce(const Params &P, TmaShared &sh, unsigned char *buf, int lane) {
    Producer pr(P, sh, buf, lane);
    IdleClock clk;
    // open greedy chunks (warp-uniform copies in every lane)
    bool gactive[kSlots];
    int gx[kSlots], gb[kSlots], gs0[kSlots], gs1[kSlots], grow[kSlots], gissued[kSlots];
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
        gactive[i] = false;
        gx[i] = gb[i] = gs0[i] = gs1[i] = grow[i] = gissued[i] = 0;
    }
    // chunk pipeline: `cur` is loaded, `nxt` has its loads in flight
    ChunkPre cur = pr.load<kRule>(pr.grab());
    ChunkPre nxt = pr.load<kRule>(pr.grab());
    while (pr.ok) {
        bool did = false;
        // (a) open greedy chunks whose current row is fully consumed
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
            if (!gactive[i]) continue;
            const int x = gx[i];
            if (*(volatile int *)&sh.cs_consumed[x] < gissued[i]) continue;
            __threadfence_block();
            int f = *(volatile int *)&sh.cs_missed[x];
            if (f < kFlagBase - grow[i] && grow[i] < P.K) {
                int g = 0;
                if (lane == 0) g = ld_l2(P.miss + gb[i]);
                f = max(f, __shfl_sync(0xffffffffu, g, 0));
            }
            if (f >= kFlagBase - grow[i] || grow[i] == P.K) {
                gactive[i] = false;
                pr.free_chunk(x);
                did = true;
                continue;
            }
            grow[i] += 1;
            gissued[i] += pr.greedy_row(gb[i], gs0[i], gs1[i], x, i, grow[i]);
            did = true;
        }
        // (b) start the next chunk
        int gfree = -1;
#pragma unroll
        for (int i = kSlots - 1; i >= 0; --i)
            if (!gactive[i]) gfree = i;
        const bool have = cur.c < P.nchunks;
        if (have && (cur.rule != kGreedy || gfree >= 0)) {
            const ChunkPre ci = cur;
            cur = nxt;
            nxt = pr.load<kRule>(pr.grab());
            if (ci.ns == kNBad || ci.ns == 0) {
                // invalid draft ids or mode: nothing to stream, the decide kernel reports it
            } else if (ci.rule == kSample) {
                pr.sample_chunk(ci);
            } else if (ci.rule == kGreedy) {
                const int x = pr.take_chunk_slot();
                const int i = gfree;
                if (lane < P.K) {
                    sh.g_tok[i][lane] = ci.t0;
                    sh.g_pt[i][lane] = ci.pt0;
                }
                if (lane + 32 < P.K) {
                    sh.g_tok[i][lane + 32] = ci.t1;
                    sh.g_pt[i][lane + 32] = ci.pt1;
                }
                pr.open_chunk(x);
                gactive[i] = true;
                gx[i] = x;
                gb[i] = ci.b;
                gs0[i] = ci.s0;
                gs1[i] = ci.s1;
                grow[i] = 0;
                gissued[i] = pr.greedy_row(ci.b, ci.s0, ci.s1, x, i, 0);
            }
            did = true;
        } else if (!have) {
            bool any = false;
#pragma unroll
            for (int i = 0; i < kSlots; ++i) any |= gactive[i];
            if (!any) break;
        }
        if (did) {
            clk.progress();
        } else if (!clk.idle()) {
            pr.fail();
        }
    }
    // tell every consumer to stop
    for (int i = 0; i < kTmaConsumers; ++i) {  // one stop per consumer
        StageMeta m = {};
        m.kind = kStop;
        pr.issue(m);
    }
    if (!pr.ok && lane == 0) {
        // a wait gave up: let the copies still in flight land before returning
        // (the last fill of each stage completes once its bytes have arrived)
        for (int i = 0; i < kStages; ++i)
            if (pr.used & (1u << i)) mbar_wait(&sh.full[i], (pr.parity >> i) & 1u);
    }
}

// ---------------------------------------------------------------------------
// consumers

// Element e of a stage part: from shared memory if the copy delivered it,
// else straight from global memory (the last 1-3 elements of a ragged row).
__device__ __forceinline__ float part_elem(const float *sm, const float *g, int c, int e) {
    return e < c ? sm[e] : __ldg(g + e);
}

// Per-lane, per-block partial sums of one stage part (see segment_partials).
template <bool kResidual>
__device__ __forceinline__ void stage_partials(const float *sp, const float *sq, int n, int c0,
                                               int c1, const float *g0, const float *g1, int lane,
                                               dd v[kBlocks]) {
    if (n == kSeg && c0 == kSeg && (!kResidual || c1 == kSeg)) {
        const float4 *p4 = reinterpret_cast<const float4 *>(sp);
        const float4 *q4 = reinterpret_cast<const float4 *>(sq);
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const float4 a = p4[lane + 32 * k];
            const float4 d = kResidual ? q4[lane + 32 * k] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[k] = quad_mass<kResidual>(a, d);
        }
    } else {
        Acc acc[kBlocks];
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const int e = lane + 32 * j;
            if (e < n) {
                float hi, lo;
                elem_mass<kResidual>(part_elem(sp, g0, c0, e), kResidual ? part_elem(sq, g1, c1, e) : 0.f,
                                     hi, lo);
                acc[j / 4].add(hi, lo);
            }
        }
#pragma unroll
        for (int k = 0; k < kBlocks; ++k) v[k] = acc[k].value();
    }
}

__device__ __forceinline__ void stage_argmax(const float *sp, int n, int c, const float *g,
                                             int64_t base, int lane, float &bv, int32_t &bi) {
    if (n == kSeg && c == kSeg) {
        const float4 *p4 = reinterpret_cast<const float4 *>(sp);
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const float4 x = p4[lane + 32 * k];
            const int32_t e = (int32_t)(base + 4 * (lane + 32 * k));
            take(x.x, e, bv, bi);
            take(x.y, e + 1, bv, bi);
            take(x.z, e + 2, bv, bi);
            take(x.w, e + 3, bv, bi);
        }
    } else {
        for (int e = lane; e < n; e += 32) take(part_elem(sp, g, c, e), (int32_t)(base + e), bv, bi);
    }
}

// Waits (bounded) until ring position t % kStages holds the fill of ticket t.
// Consumers take tickets as they free up, so one may hold ticket t while the
// fill of ticket t - kStages is still in flight; a parity wait on the full
// barrier cannot tell that fill's phase from the one before it and would pass
// at once.  Waiting first for the release of the stage's previous fill (the
// empty barrier's phase t / kStages - 1; the next phase needs this consumer's
// own arrival) leaves the full barrier at most one phase ahead of the wanted
// one, where its parity is unambiguous.
__device__ __forceinline__ bool wait_ticket(unsigned long long *full, unsigned long long *empty,
                                            int t) {
    const int k = t % kStages;
    const uint32_t phase = (uint32_t)(t / kStages) & 1u;
    return mbar_wait(&empty[k], phase ^ 1u) && mbar_wait(&full[k], phase);
}

// Hands ring position k back to the producer once every lane of the warp has
// read what it needs from it (the values are in registers by then), so the
// next copy into it overlaps this warp's reduction and stores.
__device__ __forceinline__ void release_stage(unsigned long long *empty, int k, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[k]);
}

__device__ void tma_consume(const Params &P, TmaShared &sh, unsigned char *buf, int w, int lane) {
    (void)w;
    while (true) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&sh.ticket, 1);
        t = __shfl_sync(0xffffffffu, t, 0);
        const int k = t % kStages;
        const float *sp = reinterpret_cast<const float *>(buf + (size_t)k * kStageBytes);
        const float *sq = reinterpret_cast<const float *>(buf + (size_t)k * kStageBytes + kPartBytes);
        // every lane observes the phase, so every lane's reads of the stage
        // are ordered after the copy that filled it
        if (!__all_sync(0xffffffffu, wait_ticket(sh.full, sh.empty, t))) {
            if (lane == 0) atomicOr(P.status, kStatusTimeout);
            return;
        }
        const StageMeta m = sh.meta[k];
        if (m.kind == kStop) {  // released, so a stop may follow it round the ring
            release_stage(sh.empty, k, lane);
            return;
        }
        float2 *seg = P.seg + (int64_t)m.b * P.nseg;
        float2 *blk = P.blk + (int64_t)m.b * P.nseg * kBlocks;
        if (m.kind == kPair) {
            dd v[kBlocks];
            stage_partials<true>(sp, sq, m.n0, m.c0, m.c1, m.g0, m.g1, lane, v);
            release_stage(sh.empty, k, lane);
            store_sums(seg, blk, m.s, v, lane);
        } else if (m.kind == kMass) {
            dd v[kBlocks], v1[kBlocks];
            stage_partials<false>(sp, nullptr, m.n0, m.c0, 0, m.g0, nullptr, lane, v);
            if (m.nparts == 2) stage_partials<false>(sq, nullptr, m.n1, m.c1, 0, m.g1, nullptr, lane, v1);
            release_stage(sh.empty, k, lane);
            store_sums(seg, blk, m.s, v, lane);
            if (m.nparts == 2) store_sums(seg, blk, m.s + 1, v1, lane);
        } else {  // kArgmax
            float bv = -__int_as_float(0x7f800000);
            int32_t bi = -1;
            stage_argmax(sp, m.n0, m.c0, m.g0, (int64_t)m.s * kSeg, lane, bv, bi);
            if (m.nparts == 2)
                stage_argmax(sq, m.n1, m.c1, m.g1, (int64_t)(m.s + 1) * kSeg, lane, bv, bi);
            release_stage(sh.empty, k, lane);
            if (m.tok >= 0) {
                const bool beats = bi >= 0 && (bv > m.pt || (bv == m.pt && bi < m.tok));
                if (__any_sync(0xffffffffu, beats) && lane == 0) {
                    atomicMax(P.miss + m.b, kFlagBase - m.row);
                    atomicMax(&sh.cs_missed[m.cslot], kFlagBase - m.row);
                }
            }
            const unsigned long long key = warp_max_u64(pack_key(bv, bi));
            if (lane == 0 && key) atomicMax(P.best + (int64_t)m.b * (P.K + 1) + m.row, key);
        }
        __syncwarp();
        if (lane == 0 && m.cslot >= 0) {
            __threadfence_block();  // this stage's results before its count
            atomicAdd(&sh.cs_consumed[m.cslot], 1);
        }
    }
}

template <int kRule>
__global__ void __launch_bounds__(kTmaThreads, 2) tma_stream_kernel(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    TmaShared &sh = *reinterpret_cast<TmaShared *>(smem);
    unsigned char *buf = smem + kTmaBufOffset;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        sh.ticket = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x < kChunkSlots) {
        sh.cs_state[threadIdx.x] = 0;
        sh.cs_consumed[threadIdx.x] = 0;
        sh.cs_missed[threadIdx.x] = 0;
    }
    __syncthreads();
    grid_dependents_may_launch();
    wait_for_primary_grid();  // the scan kernel's cached per-sequence data
    if (warp == kProducerWarp) tma_produce<kRule>(P, sh, buf, lane);
    else tma_consume(P, sh, buf, warp, lane);
}

}  // namespace sv
