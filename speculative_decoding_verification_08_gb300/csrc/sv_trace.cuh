// sv_trace.cuh -- a timeline of the single-launch item kernel, compiled only
// with -DSV_TRACE=1 (the default build neither contains nor runs it).
//
// Each CTA appends (time, event) records to its own region of a static
// device buffer: a slot comes from a shared-memory counter, the time from
// %globaltimer (ns, one clock for the whole GPU), and the record is a plain
// 16-byte store, so recording costs no global round trip.  The host clears
// the buffer before a traced call (sv_trace_reset) and copies it back after
// (sv_trace_read); empty slots have time 0.  What the records are for: where
// a round's time goes between the first CTA's start, each CTA's first and
// last copy, the last item's retirement and the last decision.
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
};

constexpr int kTraceCtaCap = 512;   // records per CTA (later ones are dropped)
constexpr int kTraceMaxCtas = 1024;
constexpr size_t kTraceRecords = (size_t)kTraceCtaCap * kTraceMaxCtas;

#if SV_TRACE
static __device__ ulonglong2 sv_trace_buf[kTraceRecords];
static __shared__ unsigned int sv_trace_slot;  // this CTA's next record

__device__ __forceinline__ void trace(uint32_t ev, uint32_t arg) {
    const uint32_t c = blockIdx.x;
    if (c >= (uint32_t)kTraceMaxCtas) return;
    const uint32_t i = atomicAdd(&sv_trace_slot, 1u);
    if (i >= (uint32_t)kTraceCtaCap) return;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    sv_trace_buf[(size_t)c * kTraceCtaCap + i] =
        make_ulonglong2(t, ((uint64_t)ev << 56) | ((uint64_t)c << 32) | arg);
}
#define SV_TRACE_INIT() (::sv::sv_trace_slot = 0u)
#define SV_TRACE_EVENT(ev, arg) ::sv::trace((ev), (uint32_t)(arg))
#else
#define SV_TRACE_INIT() ((void)0)
#define SV_TRACE_EVENT(ev, arg) ((void)0)
#endif

}  // namespace sv
