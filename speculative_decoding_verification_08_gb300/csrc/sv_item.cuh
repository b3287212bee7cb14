// sv_item.cuh -- a whole verification round as one persistent kernel over
// (sequence, chunk) work items (sm_103a); used when every row starts on a
// 16-byte boundary and lies in device memory.
//
// A work item is one of a sequence's `ichunks` parts: a run of consecutive
// 1024-element segments of the rows that sequence needs.  When a row takes
// several items, its first ~three quarters come in big items of `isegs`
// segments and the rest in small ones of `itail`; every sequence's big items
// are numbered before any small one.  Items are handed out in order from a
// device-wide counter, so every CTA streams until the batch is done, and the
// last items handed out -- the ones that set when the round ends -- are short.
// Each CTA runs three roles:
//  * a producer warp takes the next item, finds what the item needs one item
//    ahead of use (sampling: the first rejection n from gathered p_i(t_i),
//    q_i(t_i) and the exact accept test; greedy: the draft tokens and
//    p_i(t_i)), and streams the item's row segments into a ring of
//    shared-memory stages with cp.async.bulk;
//  * eight consumer warps reduce the stages -- the double-fp32 segment and
//    block sums of a residual (or bonus) row, stored to the workspace, or a
//    greedy segment's maximum folded into the item's per-row key in shared
//    memory, a draft-token miss raising the sequence's flag;
//  * a retire warp frees an item whose stages are all consumed: it merges the
//    item's greedy keys into the sequence's keys and counts the item as done
//    (after a device-scope fence that also publishes the consumers' sums);
//    the CTA whose item completes a sequence queues the sequence for
//  * a decide warp, which turns it into (n_accepted, next_token) and clears the
//    sequence's state for the next round.  Nothing waits for another CTA: the
//    last item to finish decides, and retiring never waits for a decision.
//
// Greedy items stream their rows in order and stop before a row once a miss in
// an earlier row is known (seen by this CTA, or recorded for the sequence by
// any CTA), and after a row once this CTA has seen a miss in it.  Every wait is
// bounded by kWaitLimitNs of wall-clock time (then SV_STATUS_TIMEOUT is set,
// the warp leaves its loop, and the workspace has to be initialised again
// before its next use).
#pragma once

#include "sv_tma.cuh"
#include "sv_trace.cuh"

namespace sv {

// Items a CTA holds at once: the one streaming, ones whose stages are still in
// the ring, and ones waiting for the retire warp.
#ifndef SV_ITEM_SLOTS
#define SV_ITEM_SLOTS 4
#endif
constexpr int kItemSlots = SV_ITEM_SLOTS;
constexpr int kItemDecideWarps = 2;
constexpr int kItemThreads = (kTmaConsumers + 2 + kItemDecideWarps) * 32;
// Warp w issues on scheduler w % 4.  The producer's issue rate bounds the
// stream, so it shares its scheduler only with the two decide warps (mostly
// idle); the eight consumers and the retire warp fill the other three.
constexpr int kItemProducerWarp = 0;
constexpr int kItemDecideWarpA = 4;
constexpr int kItemDecideWarpB = 8;
constexpr int kItemRetireWarp = 11;
static_assert(kItemThreads == 12 * 32, "role map assumes twelve warps");
constexpr int kDecideQueue = 16;  // sequences a CTA has completed but not yet decided
// Poll intervals of the retire and decide warps: they wait on shared state,
// not on a barrier, and a few hundred ns of delay costs them nothing, while
// every poll takes issue slots from the producer.
constexpr uint32_t kRetirePollNs = 256;
constexpr uint32_t kDecidePollNs = 256;

struct ItemSlot {
    int state;     // 0 free, 1 streaming, 2 every stage issued (`issued` final)
    int b;
    int rule;
    int ns;        // sampling: n + 1; greedy: 1; kNBad: invalid draft ids; 0: bad mode
    int issued;
    int consumed;
    int miss;      // greedy: kFlagBase - first missed row seen in this item
    int sbuf;      // shared-memory sum buffer holding this item's sums, or -1
    unsigned long long keys[kMaxK + 1];  // greedy: packed (value, index) maximum per row
    unsigned long long tkey0;  // greedy: pack_key(p_0(t_0), t_0) once known, else 0
};

// ItemMeta::tok of a greedy row-0 stage issued before the draft data arrived:
// the token's key is read from the item slot (ItemSlot::tkey0) instead.
constexpr int kTokInSlot = -2;

// What a consumer needs to know about a stage beyond its item slot (the
// sequence, n and hence the row pointers live there): 32 bytes, written with
// two 16-byte stores.
struct __align__(16) ItemMeta {
    int s;       // first segment of the stage
    int slot;    // item slot the stage belongs to
    int kind;    // StageKind
    int nparts;  // segments in the stage (kMass, kArgmax: 1 or 2)
    int row;     // greedy: row index
    int tok;     // greedy: the row's draft token, -1 for the bonus row, kTokInSlot
    float pt;    // greedy: p_row(tok)
    int pad;
};

struct ItemShared {
    int ticket;  // next stage a consumer takes (ring position = ticket % kStages)
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    ItemMeta meta[kStages];
    ItemSlot slot[kItemSlots];
    int producer_done;
    int retire_done;          // 1 once the retire warp has left (2: after a timeout)
    int dq_head;              // decide queue: entries pushed so far (retire warp only)
    int dq_claim;             // entries claimed by the decide warps
    int4 dq[kDecideQueue];    // (b, rule, ns, h + 1 while entry h waits; 0 once read)
    unsigned long long dbar[kItemDecideWarps];  // each decide warp's staging copy
    int sbuf_busy[kItemDecideWarps];            // sum buffers taken by whole-row items
};

// Dynamic shared memory: the header, two sum buffers (segment sums, then block
// sums, of rows of up to kDecideSegs segments), the stage ring.  When an item
// is a whole row (one item per sequence) its consumers write its sums into a
// buffer the producer took for it, and the decide reads them there; otherwise
// buffer d is decide warp d's landing area for the block sums it stages.
constexpr int kItemHeaderBytes = 4096;
constexpr int kDecideSegs = 128;
constexpr int kSumSegOffset = 0;
constexpr int kSumBlkOffset = kDecideSegs * 8;
constexpr int kSumUOffset = kSumBlkOffset + kDecideSegs * kBlocks * 8;  // the item's u_resample
constexpr int kSumBufBytes = kSumUOffset + 16;

constexpr int kItemBufOffset = kItemHeaderBytes + kItemDecideWarps * kSumBufBytes;
static_assert(sizeof(ItemShared) <= kItemHeaderBytes, "shared header too large");
constexpr int kItemSmemBytes = kItemBufOffset + kStages * kStageBytes;

__device__ __forceinline__ int ld_volatile(const int32_t *p) {
    return *reinterpret_cast<const volatile int32_t *>(p);
}

// Loads of read-only inputs issued where they stand: a volatile asm statement
// keeps its place among the producer's other asm (barrier waits, copies), so
// the compiler cannot sink it to the value's first use an item later, and the
// warp waits only if the value is still missing when it is used.
__device__ __forceinline__ int32_t ld_early(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_early(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ double ld_early(const double *p) {
    double v;
    asm volatile("ld.global.nc.f64 %0, [%1];" : "=d"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint8_t ld_early(const uint8_t *p) {
    uint16_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return (uint8_t)v;
}

// A load from L2 (not L1) of data a primary grid wrote before this grid's wait.
__device__ __forceinline__ int2 ld_l2(const int2 *p) {
    int2 v;
    asm volatile("ld.global.cg.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// producer

// Per-lane view of an item's sequence: draft positions lane and lane + 32.
struct ItemPre {
    int b;  // >= P.B: no item
    int s0, s1;  // the item's segments [s0, s1)
    int rule;
    int32_t t0, t1;
    float u0, u1, pt0, pt1, qt0, qt1;
    double ur;  // sampling: u_resample (lane 0)
    bool bad;
};

__device__ __forceinline__ int seg_len(int64_t V, int s) {
    const int64_t rem = V - (int64_t)s * kSeg;
    return (int)(rem < kSeg ? rem : kSeg);
}

struct ItemProducer {
    const Params &P;
    ItemShared &sh;
    unsigned char *buf;
    int lane;
    // ring position, its phase and the stages filled so far (lane 0's copies)
    int k = 0;
    uint32_t phase = 0;
    int fills = 0;
    bool ok = true;

    __device__ ItemProducer(const Params &P_, ItemShared &sh_, unsigned char *buf_, int lane_)
        : P(P_), sh(sh_), buf(buf_), lane(lane_) {}

    // Lane 0 only: waits (bounded) for the next ring position, writes its
    // record and copies c0 elements from g0 and c1 from g1 into it.
    __device__ bool put(const ItemMeta &m, const float *g0, int c0, const float *g1, int c1) {
        if (!mbar_wait(&sh.empty[k], phase ^ 1u)) return false;
        uint4 *dst = reinterpret_cast<uint4 *>(&sh.meta[k]);
        dst[0] = make_uint4((uint32_t)m.s, (uint32_t)m.slot, (uint32_t)m.kind, (uint32_t)m.nparts);
        dst[1] = make_uint4((uint32_t)m.row, (uint32_t)m.tok, __float_as_uint(m.pt), 0u);
        mbar_arrive_expect_tx(&sh.full[k], 4u * (uint32_t)(c0 + c1));
        unsigned char *d = buf + (size_t)k * kStageBytes;
        if (c0) bulk_copy_g2s(d, g0, 4u * c0, &sh.full[k]);
        if (c1) bulk_copy_g2s(d + kPartBytes, g1, 4u * c1, &sh.full[k]);
        ++fills;
        SV_TRACE_EVENT(kTrStage, fills);
        if (++k == kStages) {
            k = 0;
            phase ^= 1u;
        }
        return true;
    }

    // Lane 0's verdict to the warp; the status bit is raised once.
    __device__ void sync_ok() {
        const bool was = ok;
        ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
        (void)was;
    }

    // CTA c starts with items c, c + G and c + 2G (G = gridDim.x); later ones
    // come from the counter.  take() returns the oldest of two items fetched
    // ahead and issues the next atomic, whose value is read two items later:
    // under a saturated memory system a round trip can outlast one item.
    // Among the last kLateClaimG * G items no claim is taken ahead: one is
    // taken when it is needed, so that no CTA is left holding several of the
    // round's last items while others have none (per round: mixed B=1024
    // V=128256 K=8 206.7 -> 204.1 us, sampling B=128 V=262144 K=16
    // 58.2 -> 56.3 us).
    static constexpr int kLateClaimG = 4;
    int pending = 0, pending2 = 0;
    static constexpr int kClaimLater = -1;
    __device__ int take() {
        int got = __shfl_sync(0xffffffffu, pending, 0);
        if (got == kClaimLater) {  // not claimed ahead (the end of the queue): claim it now
            if (lane == 0) got = 3 * (int)gridDim.x + (int)atomicAdd(P.queue, 1u);
            got = __shfl_sync(0xffffffffu, got, 0);
        }
        pending = pending2;
        const int64_t total = (int64_t)P.B * P.ichunks;
        if ((int64_t)got >= total - (int64_t)kLateClaimG * gridDim.x)
            pending2 = kClaimLater;
        else if (lane == 0)
            pending2 = 3 * (int)gridDim.x + (int)atomicAdd(P.queue, 1u);
        return got;
    }

    // The item's sequence and segment range (no load but a mixed round's
    // order entry).
    template <int kRule>
    __device__ ItemPre locate(int item) {
        ItemPre x = {};
        x.b = P.B;
        if (item >= P.B * P.ichunks) return x;
        // every sequence's big items first (sequence-major), then the small ones
        int b;
        const int nbig = P.B * P.ibig;
        if (item < nbig) {
            b = item / P.ibig;
            const int c = item - b * P.ibig;
            x.s0 = c * P.isegs;
            x.s1 = min(P.nseg, x.s0 + P.isegs);
        } else {
            const int nsmall = P.ichunks - P.ibig;
            const int j = item - nbig;
            b = j / nsmall;
            const int c = j - b * nsmall;
            x.s0 = P.ibig * P.isegs + c * P.itail;
            x.s1 = min(P.nseg, x.s0 + P.itail);
        }
        if constexpr (kRule == kPerSequence) {
            // mixed rounds take the sequences in the order mode_order_kernel
            // wrote: every greedy one first
            const int2 e = ld_l2(P.order + b);
            b = e.x;
            x.rule = e.y;
        } else {
            x.rule = kRule;
        }
        x.b = b;
        return x;
    }

    // Loads of the item's per-position data (issued, not waited for).
    template <int kRule>
    __device__ void load_draft(ItemPre &x) {
        if (x.b >= P.B) return;
        const int64_t tb = (int64_t)x.b * P.K;
        if (lane < P.K) x.t0 = ld_early(P.t + tb + lane);
        if (lane + 32 < P.K) x.t1 = ld_early(P.t + tb + lane + 32);
        if (kRule != kGreedy && P.u_acc) {  // (loaded for every rule in a mixed round)
            if (lane < P.K) x.u0 = ld_early(P.u_acc + tb + lane);
            if (lane + 32 < P.K) x.u1 = ld_early(P.u_acc + tb + lane + 32);
        }
        if (kRule != kGreedy && lane == 0) x.ur = ld_early(P.u_res + x.b);
    }

    // locate() and load_draft().
    template <int kRule>
    __device__ ItemPre begin(int item) {
        ItemPre x = locate<kRule>(item);
        load_draft<kRule>(x);
        return x;
    }

    __device__ void gather(ItemPre &x) {
        if (x.b >= P.B || (x.rule != kSample && x.rule != kGreedy)) return;
        const bool b0 = lane < P.K && (x.t0 < 0 || (int64_t)x.t0 >= P.V);
        const bool b1 = lane + 32 < P.K && (x.t1 < 0 || (int64_t)x.t1 >= P.V);
        x.bad = __any_sync(0xffffffffu, b0 || b1);
        if (x.bad) return;
        if (lane < P.K) x.pt0 = ld_early(prow(P, x.b, lane) + x.t0);
        if (lane + 32 < P.K) x.pt1 = ld_early(prow(P, x.b, lane + 32) + x.t1);
        if (x.rule == kSample) {
            if (lane < P.K) x.qt0 = ld_early(qrow(P, x.b, lane) + x.t0);
            if (lane + 32 < P.K) x.qt1 = ld_early(qrow(P, x.b, lane + 32) + x.t1);
        }
    }

    // n + 1 for sampling (exact accept test), 1 for greedy, kNBad for
    // invalid draft ids, 0 for an invalid mode.
    __device__ int finish(const ItemPre &x) {
        if (x.rule != kSample && x.rule != kGreedy) return 0;
        if (x.bad) return kNBad;
        if (x.rule == kGreedy) return 1;
        const bool r0 = lane < P.K && !accepts(x.u0, x.qt0, x.pt0);
        const bool r1 = lane + 32 < P.K && !accepts(x.u1, x.qt1, x.pt1);
        const unsigned m0 = __ballot_sync(0xffffffffu, r0);
        const unsigned m1 = __ballot_sync(0xffffffffu, r1);
        const int n = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : P.K);
        return n + 1;
    }

    __device__ int copy_len(int s) const { return seg_len(P.V, s) & ~3; }

    // Stages of a sampling item: its residual row pair (p_n, q_n), one
    // segment of each row per stage, or the bonus row p_K, two segments per
    // stage.
    __device__ int sample_stages(const ItemPre &c, int n) const {
        const int len = c.s1 - c.s0;
        return n < P.K ? len : (len + 1) / 2;
    }

    // Stages [j0, j1) of a sampling item; the stage loop runs on lane 0 alone.
    __device__ int stream_sample(const ItemPre &c, int n, int x, int j0, int j1) {
        int stages = 0;
        if (lane == 0 && ok) {
            ItemMeta m = {};
            m.slot = x;
            m.tok = -1;
            if (n < P.K) {
                const float *pr = prow(P, c.b, n), *qr = qrow(P, c.b, n);
                m.kind = kPair;
                m.nparts = 2;
                for (int s = c.s0 + j0; s < c.s0 + j1; ++s) {
                    m.s = s;
                    const int cc = copy_len(s);
                    if (!put(m, pr + (int64_t)s * kSeg, cc, qr + (int64_t)s * kSeg, cc)) {
                        ok = false;
                        break;
                    }
                    ++stages;
                }
            } else {
                const float *pr = prow(P, c.b, P.K);
                m.kind = kMass;
                for (int s = c.s0 + 2 * j0; s < min(c.s1, c.s0 + 2 * j1); s += 2) {
                    m.s = s;
                    m.nparts = s + 1 < c.s1 ? 2 : 1;
                    const int c1 = m.nparts == 2 ? copy_len(s + 1) : 0;
                    if (!put(m, pr + (int64_t)s * kSeg, copy_len(s), pr + (int64_t)(s + 1) * kSeg, c1)) {
                        ok = false;
                        break;
                    }
                    ++stages;
                }
            }
        }
        sync_ok();
        return __shfl_sync(0xffffffffu, stages, 0);
    }

    // Lane 0 only: greedy row i's stages for segments [from, to) of item
    // slot x, two segments per stage, until a miss in an earlier row shows up
    // in the slot or in `flag` (the sequence's flag as last read).
    __device__ int put_greedy_row(int b, int x, int i, int tok, float pt, int from, int to, int flag,
                                  bool &stop) {
        const float *pr = prow(P, b, i);
        ItemMeta m = {};
        m.kind = kArgmax;
        m.slot = x;
        m.row = i;
        m.tok = tok;
        m.pt = pt;
        int stages = 0;
        for (int s = from; s < to; s += 2) {
            if (max(*(volatile int *)&sh.slot[x].miss, flag) > kFlagBase - i) {
                stop = true;  // an earlier row missed
                break;
            }
            m.s = s;
            m.nparts = s + 1 < to ? 2 : 1;
            const int c1 = m.nparts == 2 ? copy_len(s + 1) : 0;
            if (!put(m, pr + (int64_t)s * kSeg, copy_len(s), pr + (int64_t)(s + 1) * kSeg, c1)) {
                ok = false;
                stop = true;
                break;
            }
            ++stages;
        }
        return stages;
    }

    // Greedy rows first..K of the item's segments, in order.  The sequence's
    // flag is read one row ahead of its use, so the check costs no wait.
    __device__ int stream_greedy(const ItemPre &c, int x, int first = 0, int seen = 0) {
        int stages = 0;
        bool stop = !ok;
        for (int i = first; i <= P.K && !stop; ++i) {
            int tok = -1;
            float pt = 0.f;
            if (i < P.K) {
                tok = __shfl_sync(0xffffffffu, i < 32 ? c.t0 : c.t1, i & 31);
                pt = __shfl_sync(0xffffffffu, i < 32 ? c.pt0 : c.pt1, i & 31);
            }
            if (lane == 0) {
                const int flag_now = seen;
                seen = ld_volatile(P.miss + c.b);  // used at the next row
                stages += put_greedy_row(c.b, x, i, tok, pt, c.s0, c.s1, flag_now, stop);
                if (*(volatile int *)&sh.slot[x].miss >= kFlagBase - i) stop = true;
            }
            stop = __shfl_sync(0xffffffffu, stop, 0) != 0;
        }
        sync_ok();
        return __shfl_sync(0xffffffffu, stages, 0);
    }

    // A greedy item whose draft ids are on their way.  Row 0 is read whatever
    // the draft, so its first `early` stages go out before the gather waits
    // for the ids, and `late` more while p_0(t_0) is on its way; the row's
    // token key then goes into the slot, before the rest of the row (which
    // is tested as it arrives, so a miss shows up before row 1 and no row-1
    // stage is issued for nothing); rows 1..K as above.  ns becomes kNBad
    // when a draft id is invalid (nothing past the early stages is read).
    __device__ int stream_greedy_lazy(ItemPre &c, int x, int early, int late, int &ns) {
        const int split = min(c.s1, c.s0 + 2 * early);
        const int split2 = min(c.s1, split + 2 * late);
        const int tok0 = P.K > 0 ? kTokInSlot : -1;
        int stages = 0, seen = 0;
        bool stop = !ok;
        if (lane == 0 && !stop) {
            seen = ld_volatile(P.miss + c.b);
            stages = put_greedy_row(c.b, x, 0, tok0, 0.f, c.s0, split, 0, stop);
        }
        sync_ok();
        gather(c);
        if (c.bad) {
            ns = kNBad;
            return __shfl_sync(0xffffffffu, stages, 0);
        }
        if (lane == 0 && ok) {
            stages += put_greedy_row(c.b, x, 0, tok0, 0.f, split, split2, 0, stop);
            if (P.K > 0) *(volatile unsigned long long *)&sh.slot[x].tkey0 = pack_key(c.pt0, c.t0);
            if (!stop) stages += put_greedy_row(c.b, x, 0, tok0, 0.f, split2, c.s1, 0, stop);
            if (*(volatile int *)&sh.slot[x].miss >= kFlagBase) stop = true;
        }
        sync_ok();
        stages = __shfl_sync(0xffffffffu, stages, 0);
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if (__shfl_sync(0xffffffffu, stop, 0) || !ok) return stages;
        return stages + stream_greedy(c, x, 1, seen);
    }

    // Lane 0 of the warp waits (bounded) for a free item slot: its index, or
    // -1 once a wait gave up.
    __device__ int free_slot(IdleClock &clk) {
        while (ok) {
            unsigned m = 0;
#pragma unroll
            for (int i = 0; i < kItemSlots; ++i)
                if (*(volatile int *)&sh.slot[i].state == 0) m |= 1u << i;
            if (m) {
                clk.progress();
                return __ffs(m) - 1;
            }
            if (!clk.idle()) ok = false;
        }
        return -1;
    }
};

// After the last item: stop the consumers, then the retire warp; the last CTA
// to stop taking items resets the counter for the next round.
__device__ void item_produce_end(const Params &P, ItemShared &sh, ItemProducer &pr, int lane) {
    // this CTA reads no more rows into its ring: the next grid may start taking
    // SM slots as they free up (it waits for this grid to end before it reads)
    grid_dependents_may_launch();
    if (lane == 0 && pr.ok) {
        ItemMeta m = {};
        m.kind = kStop;
        for (int i = 0; i < kTmaConsumers && pr.ok; ++i)  // one stop per consumer
            pr.ok = pr.put(m, nullptr, 0, nullptr, 0);
        SV_TRACE_EVENT(kTrProducerEnd, 0);
    }
    pr.sync_ok();
    if (!pr.ok && lane == 0) atomicOr(P.status, kStatusTimeout);
    if (lane == 0) {
        __threadfence_block();
        *(volatile int *)&sh.producer_done = pr.ok ? 1 : 2;
        __threadfence();
        if (atomicAdd(P.queue + 1, 1u) == gridDim.x - 1) {
            atomicExch(P.queue, 0u);
            atomicExch(P.queue + 1, 0u);
        }
    }
    if (!pr.ok && lane == 0) {
        // a wait gave up: let the copies still in flight land before leaving
        // (ring position i last held fill i + kStages * r, r = its round)
        for (int i = 0; i < kStages && i < pr.fills; ++i) {
            const int r = (pr.fills - 1 - i) / kStages;
            mbar_wait(&sh.full[i], (uint32_t)r & 1u);
        }
    }
}

// The greedy producer.  A CTA holds one item at a time and claims the next
// once the current one's copies are out (CTA c starts with item c; claimed
// earlier, the items measured slower, and later claims near the end of the
// queue gained nothing).  A greedy item needs no draft data before its first
// copies, so there is nothing to fetch ahead, and the last items go to the
// CTAs that finish first.  Per item: the slot is published first, then the
// draft ids are loaded while kGreedyEarly row-0 stages go out, then
// kGreedyLate more while p_0(t_0) is loaded (so the producer does not wait
// for either load), then the token's key and the rest.  The first item's slot
// is set up before the wait for the previous grid (`prewait`): nothing in
// global memory is touched until that wait.
constexpr int kGreedyEarly = 2;
constexpr int kGreedyLate = 2;

__device__ void item_produce_greedy(const Params &P, ItemShared &sh, unsigned char *buf, int lane,
                                    bool prewait) {
    ItemProducer pr(P, sh, buf, lane);
    IdleClock clk;
    int item = (int)blockIdx.x;
    while (pr.ok) {
        ItemPre c = pr.locate<kGreedy>(item);
        if (c.b >= P.B) break;
        const int x = __shfl_sync(0xffffffffu, pr.free_slot(clk), 0);
        pr.sync_ok();
        if (x < 0) break;
        ItemSlot &sl = sh.slot[x];
        for (int i = lane; i <= P.K; i += 32) sl.keys[i] = 0ull;
        unsigned claim = 0;
        if (lane == 0) {
            SV_TRACE_EVENT(kTrItemBegin, c.b);
            sl.b = c.b;
            sl.rule = kGreedy;
            sl.ns = 1;
            sl.issued = 0;
            sl.consumed = 0;
            sl.miss = 0;
            sl.sbuf = -1;
            sl.tkey0 = 0ull;
            __threadfence_block();
            *(volatile int *)&sl.state = 1;
        }
        __syncwarp();
        if (prewait) {
            wait_for_primary_grid();
            SV_TRACE_START_WARP();
            prewait = false;
        }
        pr.load_draft<kGreedy>(c);
        int ns = 1;
        const int stages = pr.stream_greedy_lazy(c, x, kGreedyEarly, kGreedyLate, ns);
        if (lane == 0) {
            SV_TRACE_EVENT(kTrItemIssued, stages);
            sl.ns = ns;
            sl.issued = stages;
            __threadfence_block();
            *(volatile int *)&sl.state = 2;
            claim = atomicAdd(P.queue, 1u);
        }
        __syncwarp();
        item = (int)gridDim.x + (int)__shfl_sync(0xffffffffu, claim, 0);
    }
    if (prewait) {  // no item at all (or a wait gave up before the first)
        wait_for_primary_grid();
        SV_TRACE_START_WARP();
    }
    item_produce_end(P, sh, pr, lane);
}

template <int kRule>
__device__ void item_produce(const Params &P, ItemShared &sh, unsigned char *buf,
                             unsigned char *sumbufs, int lane) {
    ItemProducer pr(P, sh, buf, lane);
    IdleClock clk;
    // Items in flight: cur (gathered, streams now), nxt (gathered), nxt2
    // (begun).  Each step's loads get at least one item's streaming time.
    pr.pending = (int)(blockIdx.x + gridDim.x);
    pr.pending2 = (int)(blockIdx.x + 2 * gridDim.x);
    ItemPre cur = pr.begin<kRule>((int)blockIdx.x);
    ItemPre nxt = pr.begin<kRule>(pr.take());
    pr.gather(cur);
    pr.gather(nxt);
    ItemPre nxt2 = pr.begin<kRule>(pr.take());
    while (pr.ok && cur.b < P.B) {
        // a free item slot (the retire warp frees them)
        const int x = pr.free_slot(clk);
        if (x < 0) break;
        const ItemPre c = cur;
        const int ns = pr.finish(c);
        // a whole-row sampling item keeps its sums in a shared-memory buffer
        int sb = -1;
        if (c.rule == kSample && ns != kNBad && ns != 0 && P.ichunks == 1 && P.nseg <= kDecideSegs) {
            while (pr.ok) {
#pragma unroll
                for (int i = 0; i < kItemDecideWarps && sb < 0; ++i)
                    if (*(volatile int *)&sh.sbuf_busy[i] == 0) sb = i;
                if (sb >= 0) {
                    clk.progress();
                    break;
                }
                if (!clk.idle()) pr.ok = false;
            }
            if (sb < 0) break;
        }
        ItemSlot &sl = sh.slot[x];
        for (int i = lane; i <= P.K; i += 32) sl.keys[i] = 0ull;
        if (lane == 0) {
            SV_TRACE_EVENT(kTrItemBegin, c.b);
            sl.b = c.b;
            sl.rule = c.rule;
            sl.ns = ns;
            sl.issued = 0;
            sl.consumed = 0;
            sl.miss = 0;
            sl.sbuf = sb;
            if (sb >= 0) {
                sh.sbuf_busy[sb] = 1;
                *reinterpret_cast<double *>(sumbufs + sb * kSumBufBytes + kSumUOffset) = c.ur;
            }
            __threadfence_block();
            *(volatile int *)&sl.state = 1;
        }
        __syncwarp();
        // later items' loads go out while this one streams
        cur = nxt;
        nxt = nxt2;
        pr.gather(nxt);
        nxt2 = pr.begin<kRule>(pr.take());
        int stages = 0;
        if (ns != 0 && ns != kNBad) {
            if (c.rule == kSample) stages = pr.stream_sample(c, ns - 1, x, 0, pr.sample_stages(c, ns - 1));
            else stages = pr.stream_greedy(c, x);
        }
        if (lane == 0) {
            SV_TRACE_EVENT(kTrItemIssued, stages);
            sl.issued = stages;
            __threadfence_block();
            *(volatile int *)&sl.state = 2;
        }
        __syncwarp();
    }
    item_produce_end(P, sh, pr, lane);
}

// ---------------------------------------------------------------------------
// consumers

__device__ void item_consume(const Params &P, ItemShared &sh, unsigned char *buf,
                             unsigned char *sumbufs, int lane) {
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
        const ItemMeta m = sh.meta[k];
        if (m.kind == kStop) {  // released, so a stop may follow it round the ring
            release_stage(sh.empty, k, lane);
            return;
        }
        ItemSlot &sl = sh.slot[m.slot];
        const int b = sl.b;
        const int n0 = seg_len(P.V, m.s), c0 = n0 & ~3;
        const int n1 = m.nparts == 2 ? seg_len(P.V, m.s + 1) : 0, c1 = n1 & ~3;
        if (m.kind == kPair || m.kind == kMass) {
            const int sb = sl.sbuf;
            float2 *seg = sb >= 0 ? reinterpret_cast<float2 *>(sumbufs + sb * kSumBufBytes + kSumSegOffset)
                                  : P.seg + (int64_t)b * P.nseg;
            float2 *blk = sb >= 0 ? reinterpret_cast<float2 *>(sumbufs + sb * kSumBufBytes + kSumBlkOffset)
                                  : P.blk + (int64_t)b * P.nseg * kBlocks;
            dd v[kBlocks];
            if (m.kind == kPair) {
                const int n = sl.ns - 1;
                const int64_t off = (int64_t)m.s * kSeg;
                stage_partials<true>(sp, sq, n0, c0, c0, prow(P, b, n) + off, qrow(P, b, n) + off, lane, v);
                release_stage(sh.empty, k, lane);
                store_sums(seg, blk, m.s, v, lane);
            } else {
                const float *g = prow(P, b, P.K) + (int64_t)m.s * kSeg;
                dd v1[kBlocks];
                stage_partials<false>(sp, nullptr, n0, c0, 0, g, nullptr, lane, v);
                if (m.nparts == 2)
                    stage_partials<false>(sq, nullptr, n1, c1, 0, g + kSeg, nullptr, lane, v1);
                release_stage(sh.empty, k, lane);
                store_sums(seg, blk, m.s, v, lane);
                if (m.nparts == 2) store_sums(seg, blk, m.s + 1, v1, lane);
            }
        } else {  // kArgmax
            const float *g = prow(P, b, m.row) + (int64_t)m.s * kSeg;
            float bv = -__int_as_float(0x7f800000);
            int32_t bi = -1;
            stage_argmax(sp, n0, c0, g, (int64_t)m.s * kSeg, lane, bv, bi);
            if (m.nparts == 2)
                stage_argmax(sq, n1, c1, g + kSeg, (int64_t)(m.s + 1) * kSeg, lane, bv, bi);
            release_stage(sh.empty, k, lane);
            const unsigned long long key = warp_max_u64(pack_key(bv, bi));
            // the draft token loses the row when a larger key (a larger value,
            // or an equal one at a lower index) is in it; a row-0 stage taken
            // before the token's key is known goes untested, which only costs
            // the early stop (the decide reads the row maxima)
            const unsigned long long tk =
                m.tok >= 0 ? pack_key(m.pt, m.tok)
                           : (m.tok == kTokInSlot ? *(volatile unsigned long long *)&sl.tkey0 : 0ull);
            // (once per row: a later stage that misses too changes nothing)
            if (lane == 0 && tk && key > tk && *(volatile int *)&sl.miss < kFlagBase - m.row) {
                atomicMax(&sl.miss, kFlagBase - m.row);
                atomicMax(P.miss + b, kFlagBase - m.row);  // other CTAs stop sooner
            }
            if (lane == 0 && key) atomicMax(&sl.keys[m.row], key);
        }
        __syncwarp();
        if (lane == 0) {
            // this stage's results before its count; the retire warp's
            // device-scope fence then publishes them to the deciding CTA
            __threadfence_block();
            atomicAdd(&sl.consumed, 1);
        }
    }
}

// ---------------------------------------------------------------------------
// decider

// (n_accepted, next_token) of sequence b, all of whose items are done, then
// its state cleared for the next round.  A sampling draw stages the row's
// block sums into `blk_sh` (when they fit) while it loads the segment sums;
// `dphase` is the parity of the decide warp's staging barrier.
__device__ void item_decide_sequence(const Params &P, unsigned long long *dbar, float2 *stage_sh,
                                     const unsigned char *sums, uint32_t &dphase, int b, int rule,
                                     int ns, int lane) {
    int n = 0, next = -1;
    uint32_t st = 0;
    unsigned long long *best = P.best + (int64_t)b * (P.K + 1);
    if (rule == kGreedy) {
        if (ns == kNBad) {
            st = kStatusBadToken;
        } else {
            // every row's key and draft token in one round trip.  An item stops
            // streaming a row only after a miss in an earlier row, so every row
            // up to the first miss is whole, and the first row whose maximum is
            // not its draft token is that miss.
            const int64_t tb = (int64_t)b * P.K;
            const unsigned long long k0 = lane <= P.K ? ld_l2(best + lane) : 0ull;
            const unsigned long long k1 = lane + 32 <= P.K ? ld_l2(best + lane + 32) : 0ull;
            const unsigned long long k2 = lane + 64 <= P.K ? ld_l2(best + lane + 64) : 0ull;
            const int32_t t0 = lane < P.K ? ld_early(P.t + tb + lane) : -1;
            const int32_t t1 = lane + 32 < P.K ? ld_early(P.t + tb + lane + 32) : -1;
            const unsigned m0 = __ballot_sync(0xffffffffu, lane < P.K && key_index(k0) != t0);
            const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 < P.K && key_index(k1) != t1);
            n = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : P.K);
            const unsigned long long mine = n < 32 ? k0 : (n < 64 ? k1 : k2);
            const unsigned long long key = __shfl_sync(0xffffffffu, mine, n & 31);
            next = key ? key_index(key) : 0;
        }
    } else if (rule == kSample) {
        if (ns == kNBad) {
            st = kStatusBadToken;
        } else {
            n = ns - 1;
            const float2 *seg = P.seg + (int64_t)b * P.nseg;
            const float2 *blk = P.blk + (int64_t)b * P.nseg * kBlocks;
            DrawInputs in = {};
            in.u_res = P.u_res + b;
            in.prefetch = true;  // this kernel runs on aligned device rows only
            if (sums) {
                // this CTA streamed the whole row: its sums (and u) are in shared memory
                seg = reinterpret_cast<const float2 *>(sums + kSumSegOffset);
                in.seg_local = true;
                in.blk_sh = reinterpret_cast<const float2 *>(sums + kSumBlkOffset);
                in.u_res = nullptr;
                in.u = split_uniform(*reinterpret_cast<const double *>(sums + kSumUOffset));
            } else if (P.nseg <= kDecideSegs) {
                const uint32_t bytes = (uint32_t)P.nseg * kBlocks * 8u;
                if (lane == 0) {
                    // other CTAs wrote these sums through the generic proxy
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    mbar_arrive_expect_tx(dbar, bytes);
                    bulk_copy_g2s(stage_sh, blk, bytes, dbar);
                }
                in.blk_sh = stage_sh;
                in.bar = dbar;
                in.parity = dphase;
                dphase ^= 1u;
            }
            const float *pr = prow(P, b, n < P.K ? n : P.K);
            if (n < P.K) {
                next = draw_from_sums<true>(P, seg, blk, pr, qrow(P, b, n), in, lane);
                if (next == -1) {
                    // zero residual mass (unnormalised rows): draw from p_n itself
                    for (int s = 0; s < P.nseg; ++s) segment_sum_store<false>(P, b, pr, nullptr, s, lane);
                    __threadfence_block();
                    __syncwarp();
                    in.seg_local = false;
                    in.blk_sh = nullptr;
                    in.bar = nullptr;
                    next = draw_from_sums<false>(P, P.seg + (int64_t)b * P.nseg, blk, pr, nullptr, in,
                                                 lane);
                }
            } else {
                next = draw_from_sums<false>(P, seg, blk, pr, nullptr, in, lane);
            }
            if (next == -2) st = kStatusTimeout;
            else if (next < 0) st = kStatusZeroMass;
            if (next < 0) next = -1;
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
    // every item of b has retired, so nothing else touches its state now
    if (rule == kGreedy)
        for (int r = lane; r <= P.K; r += 32) best[r] = 0ull;
    if (lane == 0) {
        P.miss[b] = 0;
        P.done[b] = 0;
    }
}

// Lane l holds the item's keys of rows l, l + 32 and l + 64 (0 past row K).
__device__ bool item_retire(const Params &P, int b, int rule, int ns, int miss,
                            unsigned long long k0, unsigned long long k1, unsigned long long k2,
                            int lane) {
    if (rule == kGreedy && ns == 1) {
        unsigned long long *best = P.best + (int64_t)b * (P.K + 1);
        if (k0) atomicMax(best + lane, k0);
        if (k1) atomicMax(best + lane + 32, k1);
        if (k2) atomicMax(best + lane + 64, k2);
        if (lane == 0 && miss) atomicMax(P.miss + b, miss);
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        // one acquire-release count: this item's results (the warp's, after
        // __syncwarp) before it, and for the last item every other item's
        // results after it
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(P.done + b) : "memory");
        last = old == P.ichunks - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();  // lane 0's acquire, before every lane's reads of the other items' results
    return last != 0;
}

template <int kRule>
__device__ void item_retire_loop(const Params &P, ItemShared &sh, int lane) {
    IdleClock clk;
    bool ok = true;
    while (ok) {
        bool did = false;
#pragma unroll
        for (int i = 0; i < kItemSlots; ++i) {
            ItemSlot &sl = sh.slot[i];
            if (*(volatile int *)&sl.state != 2) continue;
            __threadfence_block();
            if (*(volatile int *)&sl.consumed < *(volatile int *)&sl.issued) continue;
            __threadfence_block();
            const int b = sl.b, rule = sl.rule, ns = sl.ns, miss = sl.miss, sb = sl.sbuf;
            const unsigned long long k0 = lane <= P.K ? sl.keys[lane] : 0ull;
            const unsigned long long k1 = lane + 32 <= P.K ? sl.keys[lane + 32] : 0ull;
            const unsigned long long k2 = lane + 64 <= P.K ? sl.keys[lane + 64] : 0ull;
            __syncwarp();
            if (lane == 0) *(volatile int *)&sl.state = 0;  // the producer may refill it now
            __syncwarp();
            did = true;
            if (lane == 0) SV_TRACE_EVENT(kTrItemRetired, b);
            // a whole-row item with its sums in shared memory is its sequence
            if (sb < 0 && !item_retire(P, b, rule, ns, miss, k0, k1, k2, lane)) continue;
            if (kRule != kSample && rule == kGreedy) {
                // a greedy decision is one round trip: made here, not queued
                // (the decide warps' poll would cost more than it saves)
                uint32_t unused = 0;
                if (lane == 0) SV_TRACE_EVENT(kTrDecideBegin, b);
                item_decide_sequence(P, nullptr, nullptr, nullptr, unused, b, rule, ns, lane);
                if (lane == 0) SV_TRACE_EVENT(kTrDecideEnd, b);
                continue;
            }
            // queue the sequence for the decide warps (once its entry's previous
            // occupant has been read)
            const int h = sh.dq_head;
            int4 *e = &sh.dq[h % kDecideQueue];
            IdleClock room;
            while (*(volatile int *)&e->w != 0) {
                if (!room.idle()) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) {
                e->x = b;
                e->y = rule | ((sb + 1) << 8);
                e->z = ns;
                __threadfence_block();
                *(volatile int *)&e->w = h + 1;
                *(volatile int *)&sh.dq_head = h + 1;
            }
            __syncwarp();
        }
        if (!ok) break;
        if (did) {
            clk.progress();
            continue;
        }
        const int pd = *(volatile int *)&sh.producer_done;
        bool busy = false;
#pragma unroll
        for (int i = 0; i < kItemSlots; ++i) busy |= *(volatile int *)&sh.slot[i].state != 0;
        if (pd == 2) break;
        if (pd && !busy) {
            if (lane == 0) {
                __threadfence_block();
                *(volatile int *)&sh.retire_done = 1;
            }
            return;
        }
        if (!clk.idle(kRetirePollNs)) ok = false;
    }
    if (lane == 0) {
        atomicOr(P.status, kStatusTimeout);
        *(volatile int *)&sh.retire_done = 2;
    }
}

// A decide warp claims queue entries in turn and decides their sequences; it
// leaves once the retire warp has left and its claim is past the last entry.
__device__ void item_decide_loop(const Params &P, ItemShared &sh, unsigned long long *dbar,
                                 unsigned char *sumbufs, int d, int lane) {
    uint32_t dphase = 0;
    while (true) {
        int c = 0;
        if (lane == 0) c = atomicAdd(&sh.dq_claim, 1);
        c = __shfl_sync(0xffffffffu, c, 0);
        int4 *e = &sh.dq[c % kDecideQueue];
        IdleClock clk;
        bool have = false;
        while (true) {
            if (*(volatile int *)&e->w == c + 1) {
                have = true;
                break;
            }
            const int rd = *(volatile int *)&sh.retire_done;
            if (rd == 2) return;
            if (rd == 1) {
                __threadfence_block();
                if (c >= *(volatile int *)&sh.dq_head) return;
                continue;
            }
            if (!clk.idle(kDecidePollNs)) {
                if (lane == 0) atomicOr(P.status, kStatusTimeout);
                return;
            }
        }
        if (!have) return;
        __threadfence_block();
        const int b = e->x, rule = e->y & 0xff, sb = (e->y >> 8) - 1, ns = e->z;
        __syncwarp();
        if (lane == 0) *(volatile int *)&e->w = 0;  // the entry may be reused
        if (sb < 0) __threadfence();  // the other items' results after their counts
        if (lane == 0) SV_TRACE_EVENT(kTrDecideBegin, b);
        item_decide_sequence(P, dbar,
                             reinterpret_cast<float2 *>(sumbufs + d * kSumBufBytes + kSumBlkOffset),
                             sb >= 0 ? sumbufs + sb * kSumBufBytes : nullptr, dphase, b, rule, ns,
                             lane);
        if (lane == 0) SV_TRACE_EVENT(kTrDecideEnd, b);
        if (sb >= 0) {
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                *(volatile int *)&sh.sbuf_busy[sb] = 0;  // the producer may reuse the buffer
            }
        }
    }
}

// Mixed rounds: the order in which item_round_kernel<kPerSequence> takes the
// sequences -- every greedy one first, then the rest, each group in batch
// order -- written as {sequence, mode} to P.order.  Taking all the greedy
// rows first measured faster than batch order on half-greedy batches (likely
// because the round then ends on sampling items, whose sizes are known when
// they are taken, rather than on greedy ones that may stop early).  One CTA; it lets the
// item kernel be placed at once (that kernel reads P.order after its wait).
constexpr int kOrderThreads = 256;

__global__ void __launch_bounds__(kOrderThreads) mode_order_kernel(const Params P) {
    grid_dependents_may_launch();
    wait_for_primary_grid();
    __shared__ int wsum[kOrderThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (P.B + kOrderThreads - 1) / kOrderThreads;
    const int lo = min(P.B, tid * per), hi = min(P.B, lo + per);
    int g = 0;
    for (int b = lo; b < hi; ++b) g += P.mode[b] == 0;
    int incl = g;  // inclusive scan of the greedy counts over the block
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kOrderThreads / 32; ++w) {
        const int c = wsum[w];
        if (w < warp) before += c;
        total += c;
    }
    int gpos = before + incl - g;     // greedy sequences before lo
    int rpos = total + (lo - gpos);   // the others: after every greedy one
    for (int b = lo; b < hi; ++b) {
        const int m = P.mode[b];
        P.order[m == 0 ? gpos++ : rpos++] = make_int2(b, m);
    }
}

template <int kRule>
__global__ void __launch_bounds__(kItemThreads, 2) item_round_kernel(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    ItemShared &sh = *reinterpret_cast<ItemShared *>(smem);
    unsigned char *buf = smem + kItemBufOffset;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        for (int i = 0; i < kItemDecideWarps; ++i) {
            mbar_init(&sh.dbar[i], 1);
            sh.sbuf_busy[i] = 0;
        }
        for (int i = 0; i < kDecideQueue; ++i) sh.dq[i] = make_int4(0, 0, 0, 0);
        for (int i = 0; i < kItemSlots; ++i) sh.slot[i].state = 0;
        sh.producer_done = 0;
        sh.retire_done = 0;
        sh.dq_head = 0;
        sh.dq_claim = 0;
        sh.ticket = 0;
        SV_TRACE_INIT();
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // launched as a programmatic dependent: the set-up above may overlap the
    // previous grid; nothing in global memory is touched before it is done
    // (the greedy producer waits on its own, after setting up its first slot)
    constexpr bool kPrewait = kRule == kGreedy;
    if (!(kPrewait && warp == kItemProducerWarp)) {
        wait_for_primary_grid();
        SV_TRACE_START(kPrewait);
    }
    if (warp == kItemProducerWarp) {
        if constexpr (kRule == kGreedy) item_produce_greedy(P, sh, buf, lane, kPrewait);
        else item_produce<kRule>(P, sh, buf, smem + kItemHeaderBytes, lane);
    }
    else if (warp == kItemRetireWarp) item_retire_loop<kRule>(P, sh, lane);
    else if (warp == kItemDecideWarpA || warp == kItemDecideWarpB) {
        const int d = warp == kItemDecideWarpA ? 0 : 1;
        // (a greedy round's decisions are all made by the retire warp; idle
        // decide warps would only hold the CTA's exit back)
        if constexpr (kRule != kGreedy)
            item_decide_loop(P, sh, &sh.dbar[d], smem + kItemHeaderBytes, d, lane);
    }
    else item_consume(P, sh, buf, smem + kItemHeaderBytes, lane);
    SV_TRACE_FINISH();
}

}  // namespace sv
