// specverify.cu -- host side of libspecverify.so: argument checks, workspace
// layout and kernel launches behind the C ABI declared in specverify.h.
//
// The operation ("spec-verify" page, section "Method") is verification of K
// draft tokens against target probabilities for B sequences at once; the
// kernels and their design live in sv_device.cuh.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "sv_device.cuh"
#include "specverify.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t num_segments(int64_t V) { return (V + sv::kSeg - 1) / sv::kSeg; }

bool sizes_ok(int32_t B, int32_t K, int64_t V) {
    return B >= 0 && K >= 0 && K <= SV_MAX_K && V >= 1 && V <= INT32_MAX;
}

// Workspace layout: [status | ticket[B] | miss[B] | best[B][K+1] | seg[B][nseg]],
// every region 256-byte aligned.
struct Layout {
    size_t status, ticket, miss, best, seg, total;
};

Layout layout(int32_t B, int32_t K, int64_t V) {
    Layout L;
    size_t off = 0;
    L.status = off;
    off += kAlign;
    L.ticket = off;
    off += round_up((size_t)B * sizeof(uint32_t));
    L.miss = off;
    off += round_up((size_t)B * sizeof(int32_t));
    L.best = off;
    off += round_up((size_t)B * (size_t)(K + 1) * sizeof(unsigned long long));
    L.seg = off;
    off += round_up((size_t)B * (size_t)num_segments(V) * sizeof(float2));
    L.total = off;
    return L;
}

std::atomic<int32_t> g_segs_per_cta{0};
thread_local int64_t g_last_grid = 0;

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

// Segments per CTA: 16 (two per warp) when the batch alone fills the GPU a few
// times over, fewer when B is small so that every SM still gets work.
int32_t choose_spc(int32_t B, int64_t nseg) {
    int32_t forced = g_segs_per_cta.load();
    if (forced > 0) return forced;
    const int64_t want_ctas = (int64_t)sm_count() * 8;
    int64_t spc = 16;
    while (spc > 1 && (int64_t)B * ((nseg + spc - 1) / spc) < want_ctas) spc >>= 1;
    return (int32_t)spc;
}

int launch(int rule, sv::Params P, sv_stream_t stream) {
    const int64_t nseg = num_segments(P.V);
    P.nseg = (int32_t)nseg;
    P.spc = choose_spc(P.B, nseg);
    P.chunks = (int32_t)((nseg + P.spc - 1) / P.spc);
    const int64_t grid = (int64_t)P.B * P.chunks;
    if (grid > INT32_MAX) return SV_EINVAL;
    g_last_grid = grid;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (rule) {
        case sv::kGreedy:
            sv::verify_kernel<sv::kGreedy><<<(unsigned)grid, sv::kThreads, 0, st>>>(P);
            break;
        case sv::kSample:
            sv::verify_kernel<sv::kSample><<<(unsigned)grid, sv::kThreads, 0, st>>>(P);
            break;
        default:
            sv::verify_kernel<sv::kPerSequence><<<(unsigned)grid, sv::kThreads, 0, st>>>(P);
            break;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

int bind_workspace(sv::Params &P, void *ws, size_t bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return SV_EWORKSPACE;
    const Layout L = layout(P.B, P.K, P.V);
    if (bytes < L.total) return SV_EWORKSPACE;
    char *base = static_cast<char *>(ws);
    P.status = reinterpret_cast<uint32_t *>(base + L.status);
    P.ticket = reinterpret_cast<uint32_t *>(base + L.ticket);
    P.miss = reinterpret_cast<int32_t *>(base + L.miss);
    P.best = reinterpret_cast<unsigned long long *>(base + L.best);
    P.seg = reinterpret_cast<float2 *>(base + L.seg);
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
    return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

int sv_verify_greedy(const float *p, int64_t p_row_stride, const int32_t *t, int32_t B, int32_t K,
                     int64_t V, int32_t *n_accepted, int32_t *next_token, void *workspace,
                     size_t workspace_bytes, sv_stream_t stream) {
    int rc = common_checks(p, p_row_stride, t, B, K, V, n_accepted, next_token);
    if (rc != SV_OK || B == 0) return rc;
    sv::Params P = make_params(p, p_row_stride, nullptr, 0, t, nullptr, nullptr, nullptr, B, K, V,
                               n_accepted, next_token);
    if ((rc = bind_workspace(P, workspace, workspace_bytes)) != SV_OK) return rc;
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
    return launch(sv::kPerSequence, P, stream);
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

int sv_set_segments_per_cta(int32_t segs_per_cta) {
    if (segs_per_cta < 0) return SV_EINVAL;
    g_segs_per_cta.store(segs_per_cta);
    return SV_OK;
}

int64_t sv_last_grid_size(void) { return g_last_grid; }

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
        default: return "unknown code";
    }
}

int sv_version(void) { return 1; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point: the sampling kernel with its scratch in a fixed
// device array instead of a caller-provided workspace, for callers that cannot
// allocate device memory while they enqueue work.

static __device__ __align__(256) unsigned char sv_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of sv_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in, so
// the kernel must be given this address, never the name.
int noalloc_scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return SV_ECUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, sv_noalloc_scratch) != cudaSuccess || !ptr)
            return SV_ECUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
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
    // status, tickets, miss flags and keys must start at zero; the array keeps
    // whatever the previous call (possibly with other sizes) left there
    if (cudaMemsetAsync(scratch, 0, L.seg, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SV_ECUDA;
    sv::Params P = make_params(p, p_row_stride, q, q_row_stride, t, u_accept, u_resample,
                               nullptr, B, K, V, n_accepted, next_token);
    if ((rc = bind_workspace(P, scratch, SV_NOALLOC_SCRATCH_BYTES)) != SV_OK) return rc;
    return launch(sv::kSample, P, stream);
}
