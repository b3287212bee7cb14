// sv_tma.cuh -- the shared-memory stage ring that the single-launch item
// kernel (sv_item.cuh) and the logits kernels (sv_logits.cuh) stream rows
// through (sm_103a): stage sizes, the stage kinds, and the per-stage
// reductions and ring waits the consumer warps use.
//
// A producer warp moves row segments from HBM into the ring's shared-memory
// stages with cp.async.bulk; consumer warps take full stages in order through
// a shared ticket and reduce them: the double-fp32 mass sum of a residual (or
// bonus-row) segment, or a greedy segment's maximum as a packed (value, index)
// key.  Loads stay in flight while consumers compute, so the bytes in flight
// are set by the ring, not by any warp's registers.
//
// Every wait on a ring barrier is bounded by kWaitLimitNs of wall-clock time:
// on timeout the caller sets SV_STATUS_TIMEOUT (the round's outputs are then
// not meaningful) and leaves its loop.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kTmaConsumers = 8;
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

enum StageKind : int { kStop = 0, kPair = 1, kMass = 2, kArgmax = 3 };

constexpr int kTmaBufOffset = 4096;  // stage buffers start here in dynamic shared memory

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

}  // namespace sv
