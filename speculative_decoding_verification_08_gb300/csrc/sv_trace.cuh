// sv_trace.cuh -- a timeline of the single-launch item kernel, compiled only
// with -DSV_TRACE=1 (the default build neither contains nor runs it).
//
// Each CTA appends (time, event) records to its own region of a static
// device buffer: a slot comes from a shared-memory counter, the time from
// %globaltimer (ns, one clock for the whole GPU), and the record is a plain
// 16-byte store, so recording costs no global round trip.  Consecutive
// launches keep appending: a CTA starts at the slot where the CTA with its
// index in the previous launch stopped (read after the wait for that grid,
// written back when the CTA ends), so one read covers several rounds and the
// time between them.  The host clears the buffer and the slot counts before
// the traced calls (sv_trace_reset) and copies the records back after
// (sv_trace_read); empty slots have time 0.  What the records are for: where
// a round's time goes between a CTA's placement behind the previous grid,
// its start, its first and last copy, the last item's retirement, the last
// decision and the CTA's exit.
#pragma once

#include <stdint.h>

#ifndef SV_TRACE
#define SV_TRACE 0
#endif

namespace sv {

// Event ids (bits 56..63 of a record's second word; bits 32..55 hold the CTA,
// bits 0..31 the event's argument).
enum TraceEvent : uint32_t {
    kTrCtaBegin = 0,     // set-up done and the previous grid waited for (argument 0)
    kTrItemBegin = 1,    // the producer starts streaming an item (argument: its sequence)
    kTrStage = 2,        // one stage's copies issued (argument: the CTA's fills so far)
    kTrItemIssued = 3,   // every stage of the item issued (argument: its stage count)
    kTrItemRetired = 4,  // the retire warp freed an item (argument: its sequence)
    kTrDecideBegin = 5,  // a decide warp took a sequence (argument: the sequence)
    kTrDecideEnd = 6,    // ... and wrote its outputs (argument: the sequence)
    kTrProducerEnd = 7,  // the producer issued its stop stages (argument 0)
    kTrCtaPlaced = 8,    // the CTA began its set-up, before the wait (argument 0)
    kTrCtaEnd = 9,       // every warp of the CTA is done (argument 0)
    // sampling from logits (the bulk-copy workers)
    kTrLgClaim = 10,     // a producer claimed a chunk (argument: group | chunk << 24)
    kTrLgReady = 11,     // ... and its group is appended (argument: group)
    kTrLgIssued = 12,    // ... and every stage of it is issued (argument: group)
    kTrLgChunkDone = 13, // a consumer completed a chunk (argument: group)
    kTrLgDecide = 14,    // a group's last arrival decided (argument: sequence | position << 16 | kind << 24)
    kTrLgLast = 15,      // an arrival found it is its group's last (argument: sequence | position << 16)
    kTrLgMerged = 16,    // ... and has merged its lane's segment pairs (argument: sequence | position << 16)
};

constexpr int kTraceCtaCap = 2048;  // records per CTA over all traced launches
constexpr int kTraceMaxCtas = 1024;
constexpr size_t kTraceRecords = (size_t)kTraceCtaCap * kTraceMaxCtas;

#if SV_TRACE
static __device__ ulonglong2 sv_trace_buf[kTraceRecords];
static __device__ unsigned int sv_trace_next[kTraceMaxCtas];  // each CTA's next slot
static __shared__ unsigned int sv_trace_slot;                 // this CTA's next slot
static __shared__ unsigned long long sv_trace_placed;         // time of the CTA's placement

__device__ __forceinline__ unsigned long long trace_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void trace_at(unsigned long long t, uint32_t ev, uint32_t arg) {
    const uint32_t c = blockIdx.x;
    if (c >= (uint32_t)kTraceMaxCtas) return;
    const uint32_t i = atomicAdd(&sv_trace_slot, 1u);
    if (i >= (uint32_t)kTraceCtaCap) return;
    sv_trace_buf[(size_t)c * kTraceCtaCap + i] =
        make_ulonglong2(t, ((uint64_t)ev << 56) | ((uint64_t)c << 32) | arg);
}

__device__ __forceinline__ void trace(uint32_t ev, uint32_t arg) { trace_at(trace_now(), ev, arg); }

// Thread 0, before the wait for the previous grid: the placement time.
__device__ __forceinline__ void trace_init() {
    sv_trace_slot = 0u;
    sv_trace_placed = trace_now();
}

// Every thread, after the wait: the CTA's slot continues from the previous
// launch's, then the placement and start records.  A warp that waits on its
// own (the greedy producer, after its first slot is set up) takes the
// records instead, and the other warps wait at the named barrier for it.
__device__ __forceinline__ void trace_start_records() {
    if (blockIdx.x < (unsigned)kTraceMaxCtas) {
        sv_trace_slot = *(volatile unsigned int *)&sv_trace_next[blockIdx.x];
        trace_at(sv_trace_placed, kTrCtaPlaced, 0u);
        trace(kTrCtaBegin, 0u);
    }
}
__device__ __forceinline__ void trace_start(bool warp_of_thread0_waits_alone) {
    if (threadIdx.x == 0 && !warp_of_thread0_waits_alone) trace_start_records();
    asm volatile("bar.sync 1;" ::: "memory");
}
__device__ __forceinline__ void trace_start_warp() {
    if ((threadIdx.x & 31) == 0) trace_start_records();
    __syncwarp();
    asm volatile("bar.sync 1;" ::: "memory");
}

// Every thread, as the kernel's last statement: the exit record and the slot
// count the next launch continues from.
__device__ __forceinline__ void trace_finish() {
    __syncthreads();
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceMaxCtas) {
        trace(kTrCtaEnd, 0u);
        const unsigned int s = sv_trace_slot;
        sv_trace_next[blockIdx.x] = s < (unsigned)kTraceCtaCap ? s : (unsigned)kTraceCtaCap;
    }
}
#define SV_TRACE_INIT() ::sv::trace_init()
#define SV_TRACE_START(alone) ::sv::trace_start(alone)
#define SV_TRACE_START_WARP() ::sv::trace_start_warp()
#define SV_TRACE_FINISH() ::sv::trace_finish()
#define SV_TRACE_EVENT(ev, arg) ::sv::trace((ev), (uint32_t)(arg))
#else
#define SV_TRACE_INIT() ((void)0)
#define SV_TRACE_START(alone) ((void)0)
#define SV_TRACE_START_WARP() ((void)0)
#define SV_TRACE_FINISH() ((void)0)
#define SV_TRACE_EVENT(ev, arg) ((void)0)
#endif

}  // namespace sv
