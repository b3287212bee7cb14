// sv_seq.cuh -- a whole verification round as one persistent kernel in which
// each CTA owns whole sequences (sm_103a); used when the batch has at least
// one sequence per SM and every row starts on a 16-byte boundary.
//
// Because all of a sequence's work stays in one CTA, its completion is a
// shared-memory count, its greedy row maxima and miss flag are shared-memory
// atomics, and no device-scope fence or cross-CTA wait is needed.  Each CTA
// runs three roles:
//  * a producer warp takes the next sequence from a device-wide counter, finds
//    what it needs (sampling: the first rejection n from gathered p_i(t_i),
//    q_i(t_i) and the exact fp64 accept test; greedy: the draft tokens and
//    p_i(t_i)) one sequence ahead of use, and streams its rows' 4 KB segments
//    into a ring of shared-memory stages with cp.async.bulk;
//  * eight consumer warps reduce the stages -- the double-fp32 segment and
//    block sums of a residual (or bonus) row, or a greedy segment's maximum
//    folded into the row's key in shared memory;
//  * a decider warp turns a sequence whose stages are all consumed into
//    (n_accepted, next_token) while the producer already streams the next one.
//
// Greedy rows are streamed in order; the producer stops before a row once this
// CTA has seen a miss in an earlier row, and after a row once it has seen a
// miss in that row, so at most the ring's depth of a row past the first miss
// is read.  Every wait is bounded by kWaitLimitNs of wall-clock time (then
// SV_STATUS_TIMEOUT is set and the warp leaves its loop).
#pragma once

#include "sv_tma.cuh"

namespace sv {

constexpr int kSeqSlots = 2;                      // sequences a CTA holds at once
constexpr int kSeqProducerWarp = kTmaConsumers;
constexpr int kSeqDeciderWarp = kTmaConsumers + 1;
constexpr int kSeqThreads = (kTmaConsumers + 2) * 32;

struct SeqSlot {
    int state;     // 0 free, 1 streaming, 2 every stage issued (`issued` final)
    int b;
    int rule;
    int ns;        // sampling: n + 1; greedy: 1; kNBad: invalid draft ids; 0: bad mode
    int issued;
    int consumed;
    int miss;      // greedy: kFlagBase - first missed row seen
    int pad;
    unsigned long long keys[kMaxK + 1];  // greedy: packed (value, index) maximum per row
};

struct SeqShared {
    int ticket;  // next stage a consumer takes (ring position = ticket % kStages)
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    StageMeta meta[kStages];
    SeqSlot slot[kSeqSlots];
    int producer_done;
};

constexpr int kSeqBufOffset = 4096;
static_assert(sizeof(SeqShared) <= kSeqBufOffset, "shared header too large");
constexpr int kSeqSmemBytes = kSeqBufOffset + kStages * kStageBytes;

// ---------------------------------------------------------------------------
// producer

// Per-lane view of a sequence's draft positions lane and lane + 32.
struct SeqPre {
    int b;  // >= P.B: none
    int rule;
    int32_t t0, t1;
    float u0, u1, pt0, pt1, qt0, qt1;
    bool bad;
};

struct SeqProducer {
    const Params &P;
    SeqShared &sh;
    unsigned char *buf;
    int lane;
    int k = 0;
    uint32_t phase = 0;
    uint32_t used = 0, parity = 0;
    bool ok = true;

    __device__ SeqProducer(const Params &P_, SeqShared &sh_, unsigned char *buf_, int lane_)
        : P(P_), sh(sh_), buf(buf_), lane(lane_) {}

    __device__ void fail() {
        if (ok && lane == 0) atomicOr(P.status, kStatusTimeout);
        ok = false;
    }

    __device__ void issue(const StageMeta &m) {
        if (!ok) return;
        bool good = true;
        if (lane == 0) {
            good = mbar_wait(&sh.empty[k], phase ^ 1u);
            if (good) {
                sh.meta[k] = m;
                mbar_arrive_expect_tx(&sh.full[k], 4u * (uint32_t)(m.c0 + m.c1));
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

    __device__ int grab() {
        int b = 0;
        if (lane == 0) b = (int)atomicAdd(P.queue, 1u);
        return __shfl_sync(0xffffffffu, b, 0);
    }

    template <int kRule>
    __device__ SeqPre begin(int b) {
        SeqPre x = {};
        x.b = b;
        if (b >= P.B) return x;
        x.rule = kRule == kPerSequence ? (int)P.mode[b] : kRule;
        const int64_t tb = (int64_t)b * P.K;
        if (lane < P.K) x.t0 = P.t[tb + lane];
        if (lane + 32 < P.K) x.t1 = P.t[tb + lane + 32];
        if (x.rule == kSample) {
            if (lane < P.K) x.u0 = __ldg(P.u_acc + tb + lane);
            if (lane + 32 < P.K) x.u1 = __ldg(P.u_acc + tb + lane + 32);
        }
        return x;
    }

    __device__ void gather(SeqPre &x) {
        if (x.b >= P.B || (x.rule != kSample && x.rule != kGreedy)) return;
        const bool b0 = lane < P.K && (x.t0 < 0 || (int64_t)x.t0 >= P.V);
        const bool b1 = lane + 32 < P.K && (x.t1 < 0 || (int64_t)x.t1 >= P.V);
        x.bad = __any_sync(0xffffffffu, b0 || b1);
        if (x.bad) return;
        if (lane < P.K) x.pt0 = __ldg(prow(P, x.b, lane) + x.t0);
        if (lane + 32 < P.K) x.pt1 = __ldg(prow(P, x.b, lane + 32) + x.t1);
        if (x.rule == kSample) {
            if (lane < P.K) x.qt0 = __ldg(qrow(P, x.b, lane) + x.t0);
            if (lane + 32 < P.K) x.qt1 = __ldg(qrow(P, x.b, lane + 32) + x.t1);
        }
    }

    // n + 1 for sampling (exact fp64 accept test), 1 for greedy, kNBad for
    // invalid draft ids, 0 for an invalid mode.
    __device__ int finish(const SeqPre &x) {
        if (x.rule != kSample && x.rule != kGreedy) return 0;
        if (x.bad) return kNBad;
        if (x.rule == kGreedy) return 1;
        const bool r0 = lane < P.K && !(__dmul_rn((double)x.u0, (double)x.qt0) < (double)x.pt0);
        const bool r1 = lane + 32 < P.K && !(__dmul_rn((double)x.u1, (double)x.qt1) < (double)x.pt1);
        const unsigned m0 = __ballot_sync(0xffffffffu, r0);
        const unsigned m1 = __ballot_sync(0xffffffffu, r1);
        const int n = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : P.K);
        return n + 1;
    }

    __device__ static void part(const float *row, int s, int64_t V, const float *&g, int &n, int &c) {
        const int64_t base = (int64_t)s * kSeg;
        const int64_t rem = V - base;
        n = (int)(rem < kSeg ? rem : kSeg);
        c = n & ~3;
        g = row + base;
    }

    __device__ int stream_sample(int b, int n, int x) {
        int stages = 0;
        if (n < P.K) {
            const float *pr = prow(P, b, n), *qr = qrow(P, b, n);
            for (int s = 0; s < P.nseg && ok; ++s) {
                StageMeta m = {};
                m.kind = kPair;
                m.b = b;
                m.s = s;
                m.nparts = 2;
                m.cslot = x;
                part(pr, s, P.V, m.g0, m.n0, m.c0);
                part(qr, s, P.V, m.g1, m.n1, m.c1);
                issue(m);
                ++stages;
            }
        } else {
            const float *pr = prow(P, b, P.K);
            for (int s = 0; s < P.nseg && ok; s += 2) {
                StageMeta m = {};
                m.kind = kMass;
                m.b = b;
                m.s = s;
                m.nparts = s + 1 < P.nseg ? 2 : 1;
                m.cslot = x;
                part(pr, s, P.V, m.g0, m.n0, m.c0);
                if (m.nparts == 2) part(pr, s + 1, P.V, m.g1, m.n1, m.c1);
                issue(m);
                ++stages;
            }
        }
        return stages;
    }

    __device__ int stream_greedy(int b, const SeqPre &c, int x) {
        int stages = 0;
        for (int i = 0; i <= P.K && ok; ++i) {
            int tok = -1;
            float pt = 0.f;
            if (i < P.K) {
                tok = __shfl_sync(0xffffffffu, i < 32 ? c.t0 : c.t1, i & 31);
                pt = __shfl_sync(0xffffffffu, i < 32 ? c.pt0 : c.pt1, i & 31);
            }
            const float *pr = prow(P, b, i);
            bool stop = false;
            for (int s = 0; s < P.nseg && ok; s += 2) {
                if (*(volatile int *)&sh.slot[x].miss > kFlagBase - i) {  // an earlier row missed
                    stop = true;
                    break;
                }
                StageMeta m = {};
                m.kind = kArgmax;
                m.b = b;
                m.s = s;
                m.nparts = s + 1 < P.nseg ? 2 : 1;
                m.row = i;
                m.cslot = x;
                m.tok = tok;
                m.pt = pt;
                part(pr, s, P.V, m.g0, m.n0, m.c0);
                if (m.nparts == 2) part(pr, s + 1, P.V, m.g1, m.n1, m.c1);
                issue(m);
                ++stages;
            }
            if (stop || *(volatile int *)&sh.slot[x].miss >= kFlagBase - i) break;
        }
        return stages;
    }
};

template <int kRule>
__device__ void seq_produce(const Params &P, SeqShared &sh, unsigned char *buf, int lane) {
    SeqProducer pr(P, sh, buf, lane);
    IdleClock clk;
    SeqPre cur = pr.begin<kRule>(pr.grab());
    pr.gather(cur);
    SeqPre nxt = pr.begin<kRule>(pr.grab());
    while (pr.ok && cur.b < P.B) {
        // a free sequence slot (the decider frees them)
        int x = -1;
        while (pr.ok) {
            unsigned m = 0;
#pragma unroll
            for (int i = 0; i < kSeqSlots; ++i)
                if (*(volatile int *)&sh.slot[i].state == 0) m |= 1u << i;
            if (m) {
                x = __ffs(m) - 1;
                clk.progress();
                break;
            }
            if (!clk.idle()) pr.fail();
        }
        if (x < 0) break;
        const SeqPre c = cur;
        const int ns = pr.finish(c);
        SeqSlot &sl = sh.slot[x];
        for (int i = lane; i <= P.K; i += 32) sl.keys[i] = 0ull;
        if (lane == 0) {
            sl.b = c.b;
            sl.rule = c.rule;
            sl.ns = ns;
            sl.issued = 0;
            sl.consumed = 0;
            sl.miss = 0;
            __threadfence_block();
            *(volatile int *)&sl.state = 1;
        }
        __syncwarp();
        // the next sequence's loads go out while this one streams
        cur = nxt;
        pr.gather(cur);
        nxt = pr.begin<kRule>(pr.grab());
        int stages = 0;
        if (ns != 0 && ns != kNBad) {
            if (c.rule == kSample) stages = pr.stream_sample(c.b, ns - 1, x);
            else stages = pr.stream_greedy(c.b, c, x);
        }
        if (lane == 0) {
            sl.issued = stages;
            __threadfence_block();
            *(volatile int *)&sl.state = 2;
        }
        __syncwarp();
    }
    // stop the consumers, then the decider
    for (int i = 0; i < kTmaConsumers; ++i) {  // one stop per consumer
        StageMeta m = {};
        m.kind = kStop;
        pr.issue(m);
    }
    if (lane == 0) {
        __threadfence_block();
        *(volatile int *)&sh.producer_done = pr.ok ? 1 : 2;
        // the last CTA to stop taking sequences resets the counter for the next round
        __threadfence();
        if (atomicAdd(P.queue + 1, 1u) == gridDim.x - 1) {
            atomicExch(P.queue, 0u);
            atomicExch(P.queue + 1, 0u);
        }
    }
    if (!pr.ok && lane == 0) {
        for (int i = 0; i < kStages; ++i)
            if (pr.used & (1u << i)) mbar_wait(&sh.full[i], (pr.parity >> i) & 1u);
    }
}

// ---------------------------------------------------------------------------
// consumers

__device__ void seq_consume(const Params &P, SeqShared &sh, unsigned char *buf, int w, int lane) {
    (void)w;
    while (true) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&sh.ticket, 1);
        t = __shfl_sync(0xffffffffu, t, 0);
        const int k = t % kStages;
        const float *sp = reinterpret_cast<const float *>(buf + (size_t)k * kStageBytes);
        const float *sq = reinterpret_cast<const float *>(buf + (size_t)k * kStageBytes + kPartBytes);
        if (!__all_sync(0xffffffffu, wait_ticket(sh.full, sh.empty, t))) {
            if (lane == 0) atomicOr(P.status, kStatusTimeout);
            return;
        }
        const StageMeta m = sh.meta[k];
        if (m.kind == kStop) return;
        SeqSlot &sl = sh.slot[m.cslot];
        if (m.kind == kPair || m.kind == kMass) {
            float2 *seg = P.seg + (int64_t)m.b * P.nseg;
            float2 *blk = P.blk + (int64_t)m.b * P.nseg * kBlocks;
            dd v[kBlocks];
            if (m.kind == kPair) {
                stage_partials<true>(sp, sq, m.n0, m.c0, m.c1, m.g0, m.g1, lane, v);
                store_sums(seg, blk, m.s, v, lane);
            } else {
                stage_partials<false>(sp, nullptr, m.n0, m.c0, 0, m.g0, nullptr, lane, v);
                store_sums(seg, blk, m.s, v, lane);
                if (m.nparts == 2) {
                    stage_partials<false>(sq, nullptr, m.n1, m.c1, 0, m.g1, nullptr, lane, v);
                    store_sums(seg, blk, m.s + 1, v, lane);
                }
            }
        } else {  // kArgmax
            float bv = -__int_as_float(0x7f800000);
            int32_t bi = -1;
            stage_argmax(sp, m.n0, m.c0, m.g0, (int64_t)m.s * kSeg, lane, bv, bi);
            if (m.nparts == 2)
                stage_argmax(sq, m.n1, m.c1, m.g1, (int64_t)(m.s + 1) * kSeg, lane, bv, bi);
            if (m.tok >= 0) {
                const bool beats = bi >= 0 && (bv > m.pt || (bv == m.pt && bi < m.tok));
                if (__any_sync(0xffffffffu, beats) && lane == 0) atomicMax(&sl.miss, kFlagBase - m.row);
            }
            const unsigned long long key = warp_max_u64(pack_key(bv, bi));
            if (lane == 0 && key) atomicMax(&sl.keys[m.row], key);
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();  // this stage's results before its count
            atomicAdd(&sl.consumed, 1);
            mbar_arrive(&sh.empty[k]);
        }
    }
}

// ---------------------------------------------------------------------------
// decider

__device__ void seq_decide_one(const Params &P, SeqSlot &sl, int lane) {
    const int b = sl.b, rule = sl.rule, ns = sl.ns;
    int n = 0, next = -1;
    uint32_t st = 0;
    if (rule == kGreedy) {
        if (ns == kNBad) {
            st = kStatusBadToken;
        } else {
            n = sl.miss ? kFlagBase - sl.miss : P.K;
            const unsigned long long key = sl.keys[n];
            next = key ? key_index(key) : 0;
        }
    } else if (rule == kSample) {
        if (ns == kNBad) {
            st = kStatusBadToken;
        } else {
            n = ns - 1;
            const double ur = P.u_res[b];
            const float uh = __double2float_rn(ur);
            const dd u = {uh, __double2float_rn(__dsub_rn(ur, (double)uh))};
            const float2 *seg = P.seg + (int64_t)b * P.nseg;
            const float2 *blk = P.blk + (int64_t)b * P.nseg * kBlocks;
            if (n < P.K) {
                next = draw_from_sums<true>(P, seg, blk, prow(P, b, n), qrow(P, b, n), u, lane);
                if (next < 0) {
                    // zero residual mass (unnormalised rows): draw from p_n itself
                    const float *pr = prow(P, b, n);
                    for (int s = 0; s < P.nseg; ++s) segment_sum_store<false>(P, b, pr, nullptr, s, lane);
                    __threadfence_block();
                    __syncwarp();
                    next = draw_from_sums<false>(P, seg, blk, pr, nullptr, u, lane);
                }
            } else {
                next = draw_from_sums<false>(P, seg, blk, prow(P, b, P.K), nullptr, u, lane);
            }
            if (next < 0) st = kStatusZeroMass;
        }
    } else {
        st = kStatusBadMode;
    }
    if (lane == 0) {
        if (st) atomicOr(P.status, st);
        P.n_out[b] = n;
        P.next_out[b] = next;
    }
    commit_round(P, b, n, next, lane);
}

__device__ void seq_decide(const Params &P, SeqShared &sh, int lane) {
    IdleClock clk;
    while (true) {
        bool did = false;
#pragma unroll
        for (int i = 0; i < kSeqSlots; ++i) {
            SeqSlot &sl = sh.slot[i];
            if (*(volatile int *)&sl.state != 2) continue;
            __threadfence_block();
            if (*(volatile int *)&sl.consumed < *(volatile int *)&sl.issued) continue;
            __threadfence_block();
            seq_decide_one(P, sl, lane);
            __syncwarp();
            if (lane == 0) *(volatile int *)&sl.state = 0;
            __syncwarp();
            did = true;
        }
        if (did) {
            clk.progress();
            continue;
        }
        const int pd = *(volatile int *)&sh.producer_done;
        bool busy = false;
#pragma unroll
        for (int i = 0; i < kSeqSlots; ++i) busy |= *(volatile int *)&sh.slot[i].state != 0;
        if (pd == 2 || (pd && !busy)) return;
        if (!clk.idle()) {
            if (lane == 0) atomicOr(P.status, kStatusTimeout);
            return;
        }
    }
}

template <int kRule>
__global__ void __launch_bounds__(kSeqThreads, 2) seq_round_kernel(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    SeqShared &sh = *reinterpret_cast<SeqShared *>(smem);
    unsigned char *buf = smem + kSeqBufOffset;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        for (int i = 0; i < kSeqSlots; ++i) sh.slot[i].state = 0;
        sh.producer_done = 0;
        sh.ticket = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == kSeqProducerWarp) seq_produce<kRule>(P, sh, buf, lane);
    else if (warp == kSeqDeciderWarp) seq_decide(P, sh, lane);
    else seq_consume(P, sh, buf, warp, lane);
}

}  // namespace sv
