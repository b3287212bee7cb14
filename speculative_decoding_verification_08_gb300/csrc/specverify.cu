// specverify.cu -- host side of libspecverify.so: argument checks, workspace
// layout and kernel launches behind the C ABI declared in specverify.h.
//
// The operation ("spec-verify" page, section "Method") is verification of K
// draft tokens against target probabilities for B sequences at once; the
// kernels and their design live in sv_device.cuh.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "sv_alpha.cuh"
#include "sv_device.cuh"
#include "sv_item.cuh"
#include "sv_logits.cuh"
#include "specverify.h"

// A debug build (-DSV_DEBUG=1) checks the inputs' values before each call's
// kernels and reports NaN, negative or infinite probabilities as
// SV_STATUS_BAD_VALUE; the default build contains no such check.
#ifndef SV_DEBUG
#define SV_DEBUG 0
#endif
#if SV_DEBUG
#include "sv_debug.cuh"
#endif
// A trace build (-DSV_TRACE=1) records a timeline of the item kernel
// (sv_trace.cuh); sv_trace_reset and sv_trace_read return SV_EINVAL otherwise.
static_assert(SV_TRACE_CTA_RECORDS == sv::kTraceCtaCap && SV_TRACE_RECORDS == sv::kTraceRecords,
              "trace buffer sizes in specverify.h and sv_trace.cuh differ");

// Segments (1024 elements) per item of the single-launch kernel: sampling
// rows are streamed whole by one CTA (a draw then needs no other CTA's sums
// early, and an item switch costs the producer more than the finer balance
// gains); greedy rows in chunks, so that a miss found in one chunk stops the
// others and the batch's bytes spread over every SM.  Greedy and mixed rounds
// take separate sizes: at V = 128256 (126 segments) greedy rows measured
// fastest as two 48-segment items and two small ones, mixed rows with
// 32-segment items.
#ifndef SV_ITEM_SEGS_SAMPLE
#define SV_ITEM_SEGS_SAMPLE 128
#endif
#ifndef SV_ITEM_TAIL_PCT
#define SV_ITEM_TAIL_PCT 25
#endif
#ifndef SV_ITEM_TAIL_SEGS
#define SV_ITEM_TAIL_SEGS 16
#endif
#ifndef SV_ITEM_SEGS
#define SV_ITEM_SEGS 32
#endif
#ifndef SV_ITEM_SEGS_GREEDY
#define SV_ITEM_SEGS_GREEDY 48
#endif
// Batches with fewer sequences than SMs: items sized so that the grid gets
// about SV_ITEM_SMALL_B_PER_CTA items per CTA, a multiple of 8 segments from
// SV_ITEM_SMALL_B_MIN_SEGS to 64 (SV_ITEM_SMALL_B_SEGS > 0 fixes the size
// instead).  At B = 128, V = 262144 and B = 64, V = 32000 two items per CTA
// measured fastest, and faster than a three-launch pipeline over fixed
// 8-segment chunks (scan, bulk-copy stream, decide).
#ifndef SV_ITEM_SMALL_B_SEGS
#define SV_ITEM_SMALL_B_SEGS 0
#endif
#ifndef SV_ITEM_SMALL_B_PER_CTA
#define SV_ITEM_SMALL_B_PER_CTA 2
#endif
#ifndef SV_ITEM_SMALL_B_MIN_SEGS
#define SV_ITEM_SMALL_B_MIN_SEGS 8
#endif

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t num_segments(int64_t V) { return (V + sv::kSeg - 1) / sv::kSeg; }

bool sizes_ok(int32_t B, int32_t K, int64_t V) {
    return B >= 0 && K >= 0 && K <= SV_MAX_K && V >= 1 && V <= INT32_MAX;
}

// Workspace layout:
// [header | miss[B] | nstate[B] | done[B] | ptok[B][K] | best[B][K+1] | arrive[B] |
//  groups[B][3K+2] | pend[B] | seg[B][nseg] | blk[B][nseg][8] | udd[B] | norm[B][K][2] |
//  fnorm[B][2] | order[B]], every region 256-byte aligned; everything before seg
// must start at zero (and every call leaves it so).  Header: status (u32 at 0), the
// chunk queue and its exit count (u32 at 4 and 8), the logits path's task
// counter and appended groups (u64 at 16 and 24), finished sequences and
// exited workers (u32 at 32 and 36), deferred mass groups moved into the queue
// and deferred (u64 at 40 and 48).
struct Layout {
    size_t status, queue, miss, nstate, done, ptok, best, arrive, groups, pend, seg, blk, udd,
        norm, fnorm, order, total;
};
constexpr size_t kLgHead = 16, kLgTail = 24, kLgDone = 32, kLgExit = 36, kLgPendHead = 40,
                 kLgPendTail = 48;
// sv_verify_sample_logits' chunk size: 32 segments when the first groups give
// every worker at least kLgChunkBig claims of 32, else 8 when they give every
// worker at least kLgChunkSmall claims of 8, else 4 (a measured rule at
// V=128256: 32 is best at B=512, 768 and 1024, where the first groups give
// each worker 6.7 to 13.5 claims of 32; 8 at B=256, 3.4 claims, where 16
// measured slower than 8; 4 at B <= 64 with V=32000)
constexpr int64_t kLgChunkBig = 4, kLgChunkSmall = 1;



Layout layout(int32_t B, int32_t K, int64_t V) {
    Layout L;
    size_t off = 0;
    L.status = off;
    L.queue = off + sizeof(uint32_t);
    off += kAlign;
    L.miss = off;
    off += round_up((size_t)B * sizeof(int32_t));
    L.nstate = off;
    off += round_up((size_t)B * sizeof(int32_t));
    L.done = off;
    off += round_up((size_t)B * sizeof(int32_t));
    L.ptok = off;
    off += round_up((size_t)B * (size_t)K * sizeof(float));
    L.best = off;
    off += round_up((size_t)B * (size_t)(K + 1) * sizeof(unsigned long long));
    L.arrive = off;
    off += round_up((size_t)B * sizeof(int32_t));
    L.groups = off;
    off += round_up((size_t)B * (size_t)(3 * K + 2) * sizeof(unsigned long long));
    L.pend = off;
    off += round_up((size_t)B * sizeof(unsigned long long));
    L.seg = off;
    off += round_up((size_t)B * (size_t)num_segments(V) * sizeof(float2));
    L.blk = off;
    off += round_up((size_t)B * (size_t)num_segments(V) * sv::kBlocks * sizeof(float2));
    L.udd = off;
    off += round_up((size_t)B * sizeof(float2));
    L.norm = off;
    off += round_up((size_t)B * (size_t)K * 2 * sizeof(float2));
    L.fnorm = off;
    off += round_up((size_t)B * 2 * sizeof(float4));
    L.order = off;
    off += round_up((size_t)B * sizeof(int2));
    L.total = off;
    return L;
}

std::atomic<int32_t> g_ctas_per_sm{0};
thread_local int64_t g_last_grid = 0;
thread_local int32_t g_last_kernels = 0;

struct DeviceInfo {
    int sms = 0;
    int occupancy[3] = {0, 0, 0};      // resident CTAs per SM, register stream kernels
    int item_occupancy[3] = {0, 0, 0};  // resident CTAs per SM, single-launch item kernels
};

template <int kRule>
int item_occupancy_of() {
    if (cudaFuncSetAttribute(sv::item_round_kernel<kRule>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sv::kItemSmemBytes) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sv::item_round_kernel<kRule>,
                                                      sv::kItemThreads,
                                                      sv::kItemSmemBytes) != cudaSuccess)
        return 0;
    return n;
}

std::mutex g_info_mu;
DeviceInfo g_info[64];

template <int kRule>
int occupancy_of() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sv::stream_kernel<kRule>, sv::kThreads,
                                                      0) != cudaSuccess)
        return 0;
    return n;
}

// SM count and per-kernel residency of the current device, queried once.
bool device_info(int rule, int *sms, int *occ, int *item_occ) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_info_mu);
    DeviceInfo &d = g_info[dev];
    if (d.sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return false;
        d.occupancy[sv::kGreedy] = occupancy_of<sv::kGreedy>();
        d.occupancy[sv::kSample] = occupancy_of<sv::kSample>();
        d.occupancy[sv::kPerSequence] = occupancy_of<sv::kPerSequence>();
        d.item_occupancy[sv::kGreedy] = item_occupancy_of<sv::kGreedy>();
        d.item_occupancy[sv::kSample] = item_occupancy_of<sv::kSample>();
        d.item_occupancy[sv::kPerSequence] = item_occupancy_of<sv::kPerSequence>();
        d.sms = n;
    }
    *sms = d.sms;
    *occ = d.occupancy[rule] > 0 ? d.occupancy[rule] : 1;
    *item_occ = d.item_occupancy[rule];
    return true;
}

// The alpha kernel's dynamic shared memory limit, raised once per device.
bool alpha_attr_set() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    static std::atomic<int> done[64];
    if (done[dev].load()) return true;
    if (cudaFuncSetAttribute(sv::alpha_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sv::kAlphaSmemBytes) != cudaSuccess)
        return false;
    done[dev].store(1);
    return true;
}

// SM count and the residency of the two logits kernels on the current device.
bool logits_info(int *sms, int *task_occ, int *ring_occ) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_info_mu);
    static int cached_sms[64], cached_task[64], cached_ring[64];
    if (cached_sms[dev] == 0) {
        int n = 0, o = 0, r = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return false;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv::logits_task_kernel,
                                                          sv::kLgThreads, 0) != cudaSuccess ||
            o <= 0)
            return false;
        if (cudaFuncSetAttribute(sv::logits_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 sv::kLgRingSmemBytes) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, sv::logits_ring_kernel,
                                                          sv::kLgRingThreads,
                                                          sv::kLgRingSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            r = 0;
        }
        cached_task[dev] = o;
        cached_ring[dev] = r;
        cached_sms[dev] = n;
    }
    *sms = cached_sms[dev];
    *task_occ = cached_task[dev];
    *ring_occ = cached_ring[dev];
    return true;
}

// Launches kernel on stream st as a programmatic dependent of the previous
// launch: it may be scheduled while that grid's CTAs retire and waits on the
// device (griddepcontrol.wait) before it reads their results.
template <class Kernel, class Args>
int launch_dependent(Kernel kernel, unsigned grid, unsigned threads, size_t smem,
                     const Args &P, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, P) == cudaSuccess ? SV_OK : SV_ECUDA;
}

bool aligned_rows(const float *base, int64_t stride) {
    return base && (reinterpret_cast<uintptr_t>(base) & 15u) == 0 && (stride & 3) == 0;
}

// One round on rows the bulk copies cannot take (not 16-byte aligned, or in
// host memory): three kernels chained on the stream -- scan (per-sequence
// data), the register stream over segments, decide.  The later two are
// programmatic dependents.
template <int kRule>
int launch_round(const sv::Params &P, unsigned grid, cudaStream_t st) {
    const unsigned per_seq = (unsigned)((P.B + sv::kWarps - 1) / sv::kWarps);
    sv::scan_kernel<kRule><<<per_seq, sv::kThreads, 0, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;
    const int rc = launch_dependent(sv::stream_kernel<kRule>, grid, sv::kThreads, 0, P, st);
    if (rc != SV_OK) return rc;
    const unsigned decide_grid = (unsigned)((P.B + sv::kDecideWarps - 1) / sv::kDecideWarps);
    return launch_dependent(sv::decide_kernel<kRule>, decide_grid, sv::kDecideWarps * 32, 0, P, st);
}

// Picks the round's kernels.  With every row 16-byte aligned and in device
// memory: one persistent launch over (sequence, chunk) items (a mixed round
// adds the one-CTA ordering kernel before it).  Otherwise: scan -> register
// stream -> decide.  Persistent grids hold as many CTAs as the SMs fit at once
// (or the tuning override), never more than there is work for.
int launch(int rule, sv::Params P, sv_stream_t stream) {
    const int64_t nseg = num_segments(P.V);
    const int64_t items = (int64_t)P.B * nseg;
    if (items > INT32_MAX / 2) return SV_EINVAL;
    P.nseg = (int32_t)nseg;
    P.items = (int32_t)items;
    int sms = 0, occ = 0, item_occ = 0;
    if (!device_info(rule, &sms, &occ, &item_occ)) return SV_ECUDA;
    const bool small_b = P.B < sms;
    int64_t isegs = rule == sv::kSample   ? SV_ITEM_SEGS_SAMPLE
                    : rule == sv::kGreedy ? SV_ITEM_SEGS_GREEDY
                                          : SV_ITEM_SEGS;
    if (small_b) {
        const int64_t ctas = std::max<int64_t>(1, (int64_t)sms * item_occ);
        isegs = SV_ITEM_SMALL_B_SEGS > 0
                    ? SV_ITEM_SMALL_B_SEGS
                    : std::min<int64_t>(64, std::max<int64_t>(
                                                SV_ITEM_SMALL_B_MIN_SEGS,
                                                nseg * P.B / (SV_ITEM_SMALL_B_PER_CTA * ctas) / 8 * 8));
    }
    P.isegs = (int32_t)std::min<int64_t>(nseg, isegs);
    P.ichunks = (int32_t)((nseg + P.isegs - 1) / P.isegs);
    P.ibig = P.ichunks;
    P.itail = 0;
    if (P.ichunks > 1 && SV_ITEM_TAIL_PCT > 0) {
        // guided sizes: big chunks cover about the first (100 - SV_ITEM_TAIL_PCT) %
        // of a row, small ones the rest; the small ones are queued after every
        // big one, so the last items handed out are short
        const int64_t big = std::max<int64_t>(
            1, (nseg * (100 - SV_ITEM_TAIL_PCT) + 50 * (int64_t)P.isegs) / (100 * (int64_t)P.isegs));
        const int64_t rest = nseg - big * P.isegs;
        if (rest > 0) {
            P.ibig = (int32_t)big;
            P.itail = (int32_t)std::min<int64_t>(
                std::min<int64_t>(SV_ITEM_TAIL_SEGS, std::max<int32_t>(1, P.isegs / 2)), rest);
            P.ichunks = (int32_t)(big + (rest + P.itail - 1) / P.itail);
        }
    }
    // bulk copies read device memory only: rows on the host take the plain loads
    const bool aligned = !P.rows_on_host && aligned_rows(P.p, P.ps) &&
                         (rule == sv::kGreedy || P.K == 0 || aligned_rows(P.q, P.qs));
    const int32_t forced = g_ctas_per_sm.load();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (aligned && item_occ > 0) {
        int64_t grid = (int64_t)sms * (forced > 0 ? std::min<int64_t>(forced, item_occ) : item_occ);
        grid = std::min<int64_t>(grid, (int64_t)P.B * P.ichunks);
        P.warps = (int32_t)(grid * sv::kWarps);
        g_last_grid = grid;
        g_last_kernels = 1;
        // a programmatic dependent of whatever precedes it on the stream: its
        // CTAs may be placed while that grid drains, and wait for it to end
        // before they touch global memory
        switch (rule) {
            case sv::kGreedy:
                return launch_dependent(sv::item_round_kernel<sv::kGreedy>, (unsigned)grid,
                                        sv::kItemThreads, sv::kItemSmemBytes, P, st);
            case sv::kSample:
                return launch_dependent(sv::item_round_kernel<sv::kSample>, (unsigned)grid,
                                        sv::kItemThreads, sv::kItemSmemBytes, P, st);
            default: {
                // the order the items take the sequences in (greedy ones first)
                int rc = launch_dependent(sv::mode_order_kernel, 1u, sv::kOrderThreads, 0, P, st);
                if (rc != SV_OK) return rc;
                g_last_kernels = 2;
                return launch_dependent(sv::item_round_kernel<sv::kPerSequence>, (unsigned)grid,
                                        sv::kItemThreads, sv::kItemSmemBytes, P, st);
            }
        }
    }
    int64_t grid = (int64_t)sms * (forced > 0 ? forced : occ);
    const int64_t needed = (items + sv::kWarps - 1) / sv::kWarps;
    if (grid > needed) grid = needed;
    P.warps = (int32_t)(grid * sv::kWarps);
    g_last_grid = grid;
    g_last_kernels = 3;
    switch (rule) {
        case sv::kGreedy: return launch_round<sv::kGreedy>(P, (unsigned)grid, st);
        case sv::kSample: return launch_round<sv::kSample>(P, (unsigned)grid, st);
        default: return launch_round<sv::kPerSequence>(P, (unsigned)grid, st);
    }
}

// The sizes each workspace's per-sequence state was last laid out for.  A
// call leaves that state zeroed, but for its own sizes: the regions move with
// B, K and V, so a call with other sizes first clears everything between the
// status word and the sums.  A workspace seen by sv_workspace_init is known to
// be all zero.
struct StateKey {
    int32_t B = -1, K = -1;
    int64_t V = -1;
    bool zeroed = false;
};
std::mutex g_ws_mu;
std::unordered_map<uintptr_t, StateKey> g_ws_state;

void note_zeroed(const void *ws) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    StateKey k;
    k.zeroed = true;
    g_ws_state[reinterpret_cast<uintptr_t>(ws)] = k;
}

int prepare_state(const sv::Params &P, void *ws, cudaStream_t st) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    StateKey &k = g_ws_state[reinterpret_cast<uintptr_t>(ws)];
    if (!k.zeroed && (k.B != P.B || k.K != P.K || k.V != P.V)) {
        const Layout L = layout(P.B, P.K, P.V);
        if (cudaMemsetAsync(static_cast<char *>(ws) + L.queue, 0, L.seg - L.queue, st) != cudaSuccess)
            return SV_ECUDA;
    }
    k.zeroed = false;
    k.B = P.B;
    k.K = P.K;
    k.V = P.V;
    return SV_OK;
}

// Where a pointer lives, as the runtime knows it: device (or managed) memory,
// page-locked host memory the GPU reads over the host link, or neither
// (pageable host memory, which the kernels must not be given).
enum Residence { kOnDevice = 0, kOnHost = 1, kUnusable = 2 };

template <class T>
Residence place(T *&ptr) {
    if (!ptr) return kOnDevice;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return kUnusable;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return kOnDevice;
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return kUnusable;
    // the address the device uses for this page-locked block
    const char *base = static_cast<const char *>(a.hostPointer);
    const ptrdiff_t off = reinterpret_cast<const char *>(ptr) - base;
    ptr = reinterpret_cast<T *>(static_cast<char *>(a.devicePointer) + off);
    return kOnHost;
}

// Checks where every caller array lives and rewrites host addresses to their
// device-side aliases.  Rows in page-locked host memory select the plain-load
// path (the kernels then read only the rows the rule needs over the link).
int place_arrays(sv::Params &P) {
    Residence r[10] = {place(P.p),       place(P.q),        place(P.t),      place(P.u_acc),
                       place(P.u_res),   place(P.mode),     place(P.n_out),  place(P.next_out),
                       place(P.tokens),  place(P.lengths)};
    for (Residence x : r)
        if (x == kUnusable) return SV_EINVAL;
    P.rows_on_host = (r[0] == kOnHost || r[1] == kOnHost) ? 1 : 0;
    return SV_OK;
}

int bind_workspace(sv::Params &P, void *ws, size_t bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return SV_EWORKSPACE;
    void *w = ws;
    if (place(w) != kOnDevice) return SV_EWORKSPACE;  // atomics and counters live here
    const Layout L = layout(P.B, P.K, P.V);
    if (bytes < L.total) return SV_EWORKSPACE;
    char *base = static_cast<char *>(ws);
    P.status = reinterpret_cast<uint32_t *>(base + L.status);
    P.miss = reinterpret_cast<int32_t *>(base + L.miss);
    P.nstate = reinterpret_cast<int32_t *>(base + L.nstate);
    P.done = reinterpret_cast<int32_t *>(base + L.done);
    P.queue = reinterpret_cast<uint32_t *>(base + L.queue);
    P.ptok = reinterpret_cast<float *>(base + L.ptok);
    P.best = reinterpret_cast<unsigned long long *>(base + L.best);
    P.seg = reinterpret_cast<float2 *>(base + L.seg);
    P.blk = reinterpret_cast<float2 *>(base + L.blk);
    P.udd = reinterpret_cast<float2 *>(base + L.udd);
    P.order = reinterpret_cast<int2 *>(base + L.order);
    return SV_OK;
}

// Debug builds: the value check of p (and of q when with_q) on the stream,
// ahead of the verification kernels; a no-op otherwise.
int debug_check(const sv::Params &P, bool with_q, bool finite_only, cudaStream_t st) {
#if SV_DEBUG
    if (sv::check_values(P.p, P.ps, (int64_t)P.B * (P.K + 1), P.V, finite_only, P.status, st))
        return SV_ECUDA;
    if (with_q && P.K > 0 &&
        sv::check_values(P.q, P.qs, (int64_t)P.B * P.K, P.V, finite_only, P.status, st))
        return SV_ECUDA;
#else
    (void)P, (void)with_q, (void)finite_only, (void)st;
#endif
    return SV_OK;
}

int common_checks(const float *p, int64_t ps, const int32_t *t, int32_t B, int32_t K, int64_t V,
                  const int32_t *n_out, const int32_t *next_out) {
    if (!sizes_ok(B, K, V)) return SV_EINVAL;
    if (B == 0) return SV_OK;
    if (!p || !n_out || !next_out || ps < V) return SV_EINVAL;
    if (K > 0 && !t) return SV_EINVAL;
    return SV_OK;
}

sv::Params make_params(const float *p, int64_t ps, const float *q, int64_t qs, const int32_t *t,
                       const float *u_acc, const double *u_res, const uint8_t *mode, int32_t B,
                       int32_t K, int64_t V, int32_t *n_out, int32_t *next_out) {
    sv::Params P{};
    P.p = p;
    P.ps = ps;
    P.q = q;
    P.qs = qs;
    P.t = t;
    P.u_acc = u_acc;
    P.u_res = u_res;
    P.mode = mode;
    P.B = B;
    P.K = K;
    P.V = V;
    P.n_out = n_out;
    P.next_out = next_out;
    return P;
}

}  // namespace

extern "C" {

size_t sv_workspace_size(int32_t B, int32_t K, int64_t V) {
    if (!sizes_ok(B, K, V)) return 0;
    return layout(B, K, V).total;
}

int sv_workspace_init(void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return SV_EWORKSPACE;
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return SV_ECUDA;
    note_zeroed(workspace);
    return SV_OK;
}

int sv_verify_greedy(const float *p, int64_t p_row_stride, const int32_t *t, int32_t B, int32_t K,
                     int64_t V, int32_t *n_accepted, int32_t *next_token, void *workspace,
                     size_t workspace_bytes, sv_stream_t stream) {
    int rc = common_checks(p, p_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    sv::Params P = make_params(p, p_row_stride, nullptr, 0, t, nullptr, nullptr, nullptr, B, K, V,
                               n_accepted, next_token);
    if ((rc = bind_workspace(P, workspace, workspace_bytes)) != SV_OK) return rc;
    if ((rc = place_arrays(P)) != SV_OK) return rc;
    if ((rc = prepare_state(P, workspace, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    if ((rc = debug_check(P, false, false, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    return launch(sv::kGreedy, P, stream);
}

int sv_verify_sample(const float *p, int64_t p_row_stride, const float *q, int64_t q_row_stride,
                     const int32_t *t, const float *u_accept, const double *u_resample, int32_t B,
                     int32_t K, int64_t V, int32_t *n_accepted, int32_t *next_token,
                     void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    int rc = common_checks(p, p_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    if (!u_resample) return SV_EINVAL;
    if (K > 0 && (!q || !u_accept || q_row_stride < V)) return SV_EINVAL;
    sv::Params P = make_params(p, p_row_stride, q, q_row_stride, t, u_accept, u_resample, nullptr,
                               B, K, V, n_accepted, next_token);
    if ((rc = bind_workspace(P, workspace, workspace_bytes)) != SV_OK) return rc;
    if ((rc = place_arrays(P)) != SV_OK) return rc;
    if ((rc = prepare_state(P, workspace, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    if ((rc = debug_check(P, true, false, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    return launch(sv::kSample, P, stream);
}

int sv_verify_round(const uint8_t *mode, const float *p, int64_t p_row_stride, const float *q,
                    int64_t q_row_stride, const int32_t *t, const float *u_accept,
                    const double *u_resample, int32_t B, int32_t K, int64_t V,
                    int32_t *n_accepted, int32_t *next_token, int32_t *tokens, int32_t *lengths,
                    int32_t max_len, void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    int rc = common_checks(p, p_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    if (!mode || !u_resample) return SV_EINVAL;
    if (K > 0 && (!q || !u_accept || q_row_stride < V)) return SV_EINVAL;
    if (tokens && (!lengths || max_len < 1)) return SV_EINVAL;
    sv::Params P = make_params(p, p_row_stride, q, q_row_stride, t, u_accept, u_resample, mode, B,
                               K, V, n_accepted, next_token);
    P.tokens = tokens;
    P.lengths = lengths;
    P.max_len = max_len;
    if ((rc = bind_workspace(P, workspace, workspace_bytes)) != SV_OK) return rc;
    if ((rc = place_arrays(P)) != SV_OK) return rc;
    if ((rc = prepare_state(P, workspace, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    if ((rc = debug_check(P, true, false, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    return launch(sv::kPerSequence, P, stream);
}

int sv_alpha(const float *p, int64_t p_row_stride, const float *q, int64_t q_row_stride,
             int32_t B, int32_t K, int64_t V, double *alpha, double *expected_length,
             void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    if (!sizes_ok(B, K, V)) return SV_EINVAL;
    if (B == 0) return SV_OK;
    if (!p || p_row_stride < V) return SV_EINVAL;
    if (K > 0 && (!q || q_row_stride < V || !alpha)) return SV_EINVAL;
    if ((int64_t)B * K > INT32_MAX) return SV_EINVAL;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return SV_EWORKSPACE;
    const Layout L = layout(B, K, V);
    if (workspace_bytes < L.total) return SV_EWORKSPACE;
    void *w = workspace;
    if (place(w) != kOnDevice) return SV_EWORKSPACE;
    sv::AlphaParams A{};
    A.p = p;
    A.ps = p_row_stride;
    A.q = q;
    A.qs = q_row_stride;
    A.B = B;
    A.K = K;
    A.V = V;
    A.nseg = (int32_t)num_segments(V);
    A.alpha = alpha;
    A.expected = expected_length;
    if (place(A.p) == kUnusable || place(A.q) == kUnusable || place(A.alpha) == kUnusable ||
        place(A.expected) == kUnusable)
        return SV_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
#if SV_DEBUG
    uint32_t *status = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + L.status);
    if (sv::check_values(A.p, A.ps, (int64_t)B * (K + 1), V, false, status, st) ||
        (K > 0 && sv::check_values(A.q, A.qs, (int64_t)B * K, V, false, status, st)))
        return SV_ECUDA;
#endif
    const int64_t ctas = (int64_t)B * K * sv::kAlphaCluster;
    if (ctas > INT32_MAX) return SV_EINVAL;
    g_last_grid = ctas;
    g_last_kernels = 0;
    if (K > 0) {
        // one cluster of kAlphaCluster CTAs per row pair (its dimensions are
        // compiled into the kernel); the dynamic shared memory caps the CTAs
        // resident per SM
        if (!alpha_attr_set() ) return SV_ECUDA;
        sv::alpha_pair_kernel<<<(unsigned)ctas, sv::kAlphaThreads, sv::kAlphaSmemBytes, st>>>(A);
        if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;
        g_last_kernels = 1;
    }
    if (A.expected) {
        if (K == 0) {
            if (cudaMemsetAsync(A.expected, 0, (size_t)B * sizeof(double), st) != cudaSuccess)
                return SV_ECUDA;
        } else {
            int rc = launch_dependent(sv::alpha_length_kernel, (unsigned)((B + 255) / 256), 256u, 0,
                                      A, st);
            if (rc != SV_OK) return rc;
            g_last_kernels = 2;
        }
    }
    return SV_OK;
}

int sv_verify_sample_logits(const float *zp, int64_t zp_row_stride, const float *zq,
                            int64_t zq_row_stride, const int32_t *t, const float *u_accept,
                            const double *u_resample, int32_t B, int32_t K, int64_t V,
                            float temperature, int32_t *n_accepted, int32_t *next_token,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    int rc = common_checks(zp, zp_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    if (!u_resample || !(temperature > 0.f) || !std::isfinite(temperature)) return SV_EINVAL;
    if (K > 0 && (!zq || !u_accept || zq_row_stride < V)) return SV_EINVAL;
    sv::Params P = make_params(zp, zp_row_stride, zq, zq_row_stride, t, u_accept, u_resample,
                               nullptr, B, K, V, n_accepted, next_token);
    if ((rc = bind_workspace(P, workspace, workspace_bytes)) != SV_OK) return rc;
    if ((rc = place_arrays(P)) != SV_OK) return rc;
    if ((rc = prepare_state(P, workspace, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    if ((rc = debug_check(P, true, true, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    const Layout W = layout(B, K, V);
    char *ws = static_cast<char *>(workspace);
    sv::LogitsParams L{};
    L.zp = P.p;
    L.ps = P.ps;
    L.zq = P.q;
    L.qs = P.qs;
    L.t = P.t;
    L.u_acc = P.u_acc;
    L.u_res = P.u_res;
    L.B = B;
    L.K = K;
    L.V = V;
    L.nseg = (int32_t)num_segments(V);
    L.c = (float)(1.4426950408889634 / (double)temperature);
    L.tau = (double)temperature;
    L.n_out = P.n_out;
    L.next_out = P.next_out;
    L.status = P.status;
    L.seg = P.seg;
    L.blk = P.blk;
    L.fnorm = reinterpret_cast<float4 *>(ws + W.fnorm);
    L.grp = reinterpret_cast<unsigned long long *>(ws + W.groups);
    L.arrive = reinterpret_cast<int32_t *>(ws + W.arrive);
    L.head = reinterpret_cast<unsigned long long *>(ws + kLgHead);
    L.tail = reinterpret_cast<unsigned long long *>(ws + kLgTail);
    L.ndone = reinterpret_cast<uint32_t *>(ws + kLgDone);
    L.nexit = reinterpret_cast<uint32_t *>(ws + kLgExit);
    L.pend = reinterpret_cast<unsigned long long *>(ws + W.pend);
    L.pend_head = reinterpret_cast<unsigned long long *>(ws + kLgPendHead);
    L.pend_tail = reinterpret_cast<unsigned long long *>(ws + kLgPendTail);
    L.ngroups = (int64_t)B * (3 * K + 2);
    // one persistent grid of as many CTAs as the SMs hold: bulk-copy workers
    // for 16-byte-aligned device rows, plain-load workers otherwise
    int sms = 0, task_occ = 0, ring_occ = 0;
    if (!logits_info(&sms, &task_occ, &ring_occ)) return SV_ECUDA;
    const bool ring = ring_occ > 0 && !P.rows_on_host && aligned_rows(P.p, P.ps) &&
                      (K == 0 || aligned_rows(P.q, P.qs));
    const int occ = ring ? ring_occ : task_occ;
    const int32_t forced = g_ctas_per_sm.load();
    const unsigned grid = (unsigned)sms * (unsigned)(forced > 0 ? std::min(forced, occ) : occ);
    g_last_grid = grid;
    g_last_kernels = 1;
    // mass groups are deferred when the first B groups alone give every
    // worker a claim (otherwise no chain waits behind another's mass group)
    const int64_t workers = (int64_t)grid * (ring ? 1 : sv::kLgWarps);
    // segments per chunk (one claim, one group read and one arrival each):
    // 32 while the first groups give every worker several claims, fewer when
    // they do not, so that a group spreads over more workers and its
    // sequence's steps are shorter
    auto chunks = [&](int64_t c) { return (int64_t)B * ((L.nseg + c - 1) / c); };
    L.chunk = chunks(32) >= kLgChunkBig * workers ? 32 : chunks(8) >= kLgChunkSmall * workers ? 8 : 4;
    const int64_t claims = ring ? (L.nseg + L.chunk - 1) / L.chunk : L.nseg;
    L.claims = claims;
    // a norm group spans two positions while fewer claims than workers wait
    // in the queue, in calls whose chains (K decisions) are long against each
    // worker's share of the first groups (B x claims / workers): there the
    // workers run short of work for much of the call, and a second
    // position's reads are cheap next to a step of the chain
    const bool spans = (int64_t)K * workers >= (int64_t)B * claims;
    L.spec_claims = spans ? workers : 0;
    L.defer = (int64_t)B * claims >= workers;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (ring)
        return launch_dependent(sv::logits_ring_kernel, grid, sv::kLgRingThreads,
                                sv::kLgRingSmemBytes, L, st);
    return launch_dependent(sv::logits_task_kernel, grid, sv::kLgThreads, 0, L, st);
}

int sv_get_status(void *workspace, sv_stream_t stream, uint32_t *flags) {
    if (!workspace || !flags) return SV_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SV_ECUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(v), st) != cudaSuccess) return SV_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ECUDA;
    *flags = v;
    return SV_OK;
}

int sv_set_ctas_per_sm(int32_t ctas_per_sm) {
    if (ctas_per_sm < 0) return SV_EINVAL;
    g_ctas_per_sm.store(ctas_per_sm);
    return SV_OK;
}

int64_t sv_last_grid_size(void) { return g_last_grid; }

int32_t sv_last_kernel_count(void) { return g_last_kernels; }

const char *sv_status_string(int code) {
    switch (code) {
        case SV_ETOOLARGE: return "sizes exceed the 4 MiB static scratch of sv_verify_sample_noalloc";
        case SV_OK: return "ok";
        case SV_EINVAL: return "invalid argument";
        case SV_EWORKSPACE: return "workspace missing, misaligned or too small";
        case SV_ECUDA: return "CUDA launch or stream error";
        case (int)SV_STATUS_BAD_TOKEN: return "draft token id outside [0, V)";
        case (int)SV_STATUS_ZERO_MASS: return "distribution to draw from has zero mass";
        case (int)SV_STATUS_OVERFLOW: return "commit would pass max_len";
        case (int)SV_STATUS_BAD_MODE: return "round mode other than 0 (greedy) or 1 (sampling)";
        case (int)SV_STATUS_TIMEOUT: return "a bounded wait inside a kernel gave up";
        case (int)SV_STATUS_BAD_VALUE:
            return "an input probability is negative, NaN or infinite (debug builds)";
        default: return "unknown code";
    }
}

int sv_version(void) { return 1; }

int sv_trace_reset(sv_stream_t stream) {
#if SV_TRACE
    void *buf = nullptr, *next = nullptr;
    if (cudaGetSymbolAddress(&buf, sv::sv_trace_buf) != cudaSuccess ||
        cudaGetSymbolAddress(&next, sv::sv_trace_next) != cudaSuccess)
        return SV_ECUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(buf, 0, sizeof(ulonglong2) * sv::kTraceRecords, st) != cudaSuccess ||
        cudaMemsetAsync(next, 0, sizeof(unsigned int) * sv::kTraceMaxCtas, st) != cudaSuccess)
        return SV_ECUDA;
    return SV_OK;
#else
    (void)stream;
    return SV_EINVAL;
#endif
}

int sv_trace_read(void *records, size_t max_records, size_t *count, sv_stream_t stream) {
    if (count) *count = 0;
    if (!records || !count) return SV_EINVAL;
#if SV_TRACE
    const size_t n = std::min(max_records, sv::kTraceRecords);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyFromSymbolAsync(records, sv::sv_trace_buf, n * sizeof(ulonglong2), 0,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return SV_ECUDA;
    *count = n;
    return SV_OK;
#else
    (void)max_records, (void)stream;
    return SV_EINVAL;
#endif
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point: the sampling kernel with its scratch in a fixed
// device array instead of a caller-provided workspace, for callers that cannot
// allocate device memory while they enqueue work.

static __device__ __align__(256) unsigned char sv_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of sv_noalloc_scratch in the current device's context.  In
// host code the array's name is only a host-side stand-in, so the kernel must
// be given this address, never the name.  It is looked up on every call: a
// cached address would outlive a device reset (the array is then placed
// again, possibly elsewhere) and would be wrong in another context on the same
// device.  Once the library's device code is loaded in the context, the lookup
// allocates nothing.
int noalloc_scratch_address(void **out) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, sv_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return SV_ECUDA;
    }
    *out = ptr;
    return SV_OK;
}

}  // namespace

extern "C" int sv_verify_sample_noalloc(const float *p, int64_t p_row_stride, const float *q,
                                        int64_t q_row_stride, const int32_t *t,
                                        const float *u_accept, const double *u_resample,
                                        int32_t B, int32_t K, int64_t V, int32_t *n_accepted,
                                        int32_t *next_token, sv_stream_t stream) {
    int rc = common_checks(p, p_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    if (!u_resample) return SV_EINVAL;
    if (K > 0 && (!q || !u_accept || q_row_stride < V)) return SV_EINVAL;
    const Layout L = layout(B, K, V);
    if (L.total > (size_t)SV_NOALLOC_SCRATCH_BYTES) return SV_ETOOLARGE;
    void *scratch = nullptr;
    if ((rc = noalloc_scratch_address(&scratch)) != SV_OK) return rc;
    // status, miss flags, cached n and keys must start at zero; the array keeps
    // whatever the previous call (possibly with other sizes) left there
    if (cudaMemsetAsync(scratch, 0, L.seg, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SV_ECUDA;
    sv::Params P = make_params(p, p_row_stride, q, q_row_stride, t, u_accept, u_resample,
                               nullptr, B, K, V, n_accepted, next_token);
    if ((rc = bind_workspace(P, scratch, SV_NOALLOC_SCRATCH_BYTES)) != SV_OK) return rc;
    if ((rc = place_arrays(P)) != SV_OK) return rc;
    if ((rc = debug_check(P, true, false, reinterpret_cast<cudaStream_t>(stream))) != SV_OK) return rc;
    return launch(sv::kSample, P, stream);
}
