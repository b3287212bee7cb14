/*
 * specverify.h -- C ABI of the batched speculative-decoding verification
 * library (libspecverify.so, CUDA, sm_103a).
 *
 * What the calls compute is defined on the "spec-verify" page (Hugging Face
 * kernels page phanerozoic/spec-verify):
 *   - section "Usage": n_accepted, next_token = verify_greedy(target_probs
 *     [K+1, V], draft_tokens [K]); the caller keeps draft_tokens[:n_accepted]
 *     and appends next_token;
 *   - section "Method": the greedy rule and the speculative-sampling rule of
 *     Leviathan et al. / Chen et al., with randomness entering only through
 *     explicit uniforms;
 *   - section "Correctness": probabilities need not be normalised and masses
 *     are summed exactly;
 *   - section "Requirements and limits": target_probs [K+1, V] f32 and, for
 *     sampling, draft_probs [K, V] warped identically to the target.
 * These entry points batch that operation over B independent sequences.
 *
 * Common conventions
 *   Memory.  Every array argument is device memory of the current device or
 *     page-locked host memory (cudaHostAlloc / cudaHostRegister), owned by
 *     the caller, and must stay valid until the stream reaches the end of the
 *     call; pageable host memory is rejected with SV_EINVAL.  When p or q is
 *     in host memory the kernels read it where it is, over the host link, and
 *     only the rows the rule needs cross it (the plain-load path is used).
 *     The workspace must be device memory (else SV_EWORKSPACE).  Inputs are
 *     read-only; outputs must not alias inputs.  The library allocates no
 *     memory.
 *   Layout.  p holds B*(K+1) rows of V f32 target probabilities; row (b, i),
 *     i in [0, K], starts at p + (b*(K+1) + i) * p_row_stride.  q holds B*K
 *     rows of draft probabilities; row (b, i), i in [0, K), starts at
 *     q + (b*K + i) * q_row_stride.  Strides are in elements and >= V.  t,
 *     u_accept are [B][K] row-major; u_resample, mode, n_accepted, next_token,
 *     lengths are [B]; tokens is [B][max_len].  Rows whose start is 16-byte
 *     aligned are read with 16-byte vector loads; others are still correct.
 *   Values.  Probabilities are finite and >= 0 and need not sum to 1 (NaN or
 *     negative entries give unspecified results).  u_accept in [0, 1) (f32),
 *     u_resample in [0, 1) (f64).
 *   Asynchrony.  Every call only enqueues work on `stream` (NULL = the legacy
 *     default stream) and returns; nothing is synchronised and nothing is
 *     copied to the host except by sv_get_status.
 *   Workspace.  Scratch of sv_workspace_size(B, K, V) bytes, 256-byte
 *     aligned, zeroed once with sv_workspace_init before its first use.  Each
 *     call leaves it ready for the next one.  One workspace serves one call at
 *     a time: calls that share a workspace must be ordered on one stream.
 *   Return codes.  SV_OK, or a negative SV_E* code for errors detected on the
 *     host before anything is enqueued (SV_EINVAL: a null pointer or an array
 *     in pageable host memory, B < 0,
 *     K < 0 or K > SV_MAX_K, V < 1 or V > 2^31-1, a stride < V, max_len < 1;
 *     SV_EWORKSPACE: workspace null, misaligned or too small; SV_ECUDA: the
 *     launch failed).  B = 0 is a no-op.
 *   Device-detected errors never trap.  The affected sequence gets
 *     next_token = -1 and a status bit is OR-ed into the workspace's status
 *     word, read (and cleared) by sv_get_status:
 *       SV_STATUS_BAD_TOKEN  a draft id outside [0, V): n_accepted = 0,
 *                            next_token = -1 for that sequence;
 *       SV_STATUS_ZERO_MASS  the distribution to draw from has zero mass;
 *       SV_STATUS_OVERFLOW   a commit would pass max_len (nothing written);
 *                            from sv_verify_sample_logits: its workspace
 *                            held a count it cannot have left there (a
 *                            workspace reused without re-initialising it
 *                            after SV_STATUS_TIMEOUT, or overwritten);
 *       SV_STATUS_BAD_MODE   a round mode other than 0 or 1 (n = 0, next = -1);
 *       SV_STATUS_TIMEOUT    a bounded wait inside a kernel gave up (the
 *                            round's outputs are not meaningful);
 *       SV_STATUS_BAD_VALUE  only from a library built with -DSV_DEBUG=1,
 *                            which checks every input row before a call's
 *                            kernels: a probability that is negative, NaN
 *                            or infinite (for sv_verify_sample_logits: a
 *                            logit that is NaN or infinite).  The regular
 *                            build does not look, and such inputs give
 *                            unspecified results.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *sv_stream_t;

#define SV_OK 0
#define SV_EINVAL (-1)
#define SV_EWORKSPACE (-2)
#define SV_ECUDA (-3)

#define SV_STATUS_BAD_TOKEN 1u
#define SV_STATUS_ZERO_MASS 2u
#define SV_STATUS_OVERFLOW 4u
#define SV_STATUS_BAD_MODE 8u
#define SV_STATUS_TIMEOUT 16u
#define SV_STATUS_BAD_VALUE 32u

#define SV_MAX_K 64

/* Bytes of workspace the calls need for B sequences, K drafts, vocabulary V
 * (0 for invalid sizes).  Covers greedy, sampling and mixed rounds alike. */
size_t sv_workspace_size(int32_t B, int32_t K, int64_t V);

/* Zeroes a workspace on `stream` (once, before its first use).  Returns
 * SV_EWORKSPACE for a null or misaligned pointer, SV_ECUDA on failure.
 * Afterwards the workspace serves any calls it is large enough for, one at a
 * time in stream order: every call leaves its per-sequence state zeroed, and a
 * call whose sizes differ from the previous call's on the same workspace first
 * clears that state (one memset on its stream).  After a call reported
 * SV_STATUS_TIMEOUT the state is undefined: initialise the workspace again. */
int sv_workspace_init(void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* Greedy verification ("spec-verify", section "Method", greedy bullet):
 * for each sequence b, accepts t[b][i] while it equals argmax(p row (b, i))
 * (ties go to the lowest index); at the first miss i writes n_accepted[b] = i
 * and next_token[b] = argmax(p row (b, i)); when all K match writes
 * n_accepted[b] = K and next_token[b] = argmax(p row (b, K)).  Only the rows
 * up to the first miss need to be read, and the kernel stops reading the
 * others once a miss is known.  t may be NULL when K = 0. */
int sv_verify_greedy(const float *p, int64_t p_row_stride, const int32_t *t,
                     int32_t B, int32_t K, int64_t V,
                     int32_t *n_accepted, int32_t *next_token,
                     void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* Speculative-sampling verification ("spec-verify", section "Method",
 * sampling bullet; Leviathan et al. / Chen et al.): for i = 0, 1, ... accepts
 * t[b][i] iff u_accept[b][i] * q_i(t_i) < p_i(t_i), evaluated exactly (raw,
 * unnormalised values).  At the first rejection i it draws next_token from
 * max(0, p_i - q_i) by inverse CDF with u_resample[b]: the smallest v whose
 * running mass exceeds u_resample[b] times the total; if that total is zero it
 * draws from p_i instead.  When all K are accepted it draws the bonus from p_K
 * with the same uniform.  Masses are summed with fp64-level accuracy (double
 * fp32 arithmetic, relative error below 1e-10); the drawn token can differ
 * from an exact fp64 sum only when u_resample * total lies within that error
 * of a boundary between two tokens.  q, t, u_accept may be NULL when K = 0. */
int sv_verify_sample(const float *p, int64_t p_row_stride,
                     const float *q, int64_t q_row_stride,
                     const int32_t *t, const float *u_accept, const double *u_resample,
                     int32_t B, int32_t K, int64_t V,
                     int32_t *n_accepted, int32_t *next_token,
                     void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* One verification round over a mixed batch: mode[b] = 0 applies the greedy
 * rule and mode[b] = 1 the sampling rule to sequence b (other values set
 * SV_STATUS_BAD_MODE).  If tokens is not NULL the round is also committed
 * ("spec-verify", section "Usage": keep draft_tokens[:n_accepted], append
 * next_token): t[b][0..n) and next_token[b] are written to
 * tokens[b][lengths[b] ..] and lengths[b] grows by n + 1.  A sequence whose
 * next_token is -1 is not committed; one that would pass max_len is left
 * unchanged and sets SV_STATUS_OVERFLOW.  q and u_accept are read only for
 * sampling sequences but must be valid [B][K][..] arrays when K > 0. */
int sv_verify_round(const uint8_t *mode, const float *p, int64_t p_row_stride,
                    const float *q, int64_t q_row_stride,
                    const int32_t *t, const float *u_accept, const double *u_resample,
                    int32_t B, int32_t K, int64_t V,
                    int32_t *n_accepted, int32_t *next_token,
                    int32_t *tokens, int32_t *lengths, int32_t max_len,
                    void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* Allocation-free sampling verification.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory
 * at call time: code that enqueues work from inside a framework hook or
 * plugin interface that forbids allocation while enqueuing, and serving loops
 * that must not call cudaMalloc because it can synchronise the device or fail
 * under memory pressure at the worst moment.
 *
 * It computes exactly what sv_verify_sample computes (same kernel, same
 * arguments minus the workspace) but takes its scratch from a fixed array of
 * SV_NOALLOC_SCRATCH_BYTES (4 MiB) compiled into the library: every GPU that
 * loads the library holds that array until the process exits.  Sizes whose
 * sv_workspace_size(B, K, V) exceeds it are rejected with SV_ETOOLARGE before
 * anything is enqueued (at V = 128256, K = 5 that is more than 444 sequences).
 * The call allocates nothing: it issues one cudaMemsetAsync that clears the
 * part of the array that must start at zero, then the kernel launch.
 * Every call looks up the array's device address in the current device's
 * context (a host-side lookup), so a device reset, or a different context on
 * the same device, never leaves the call with a stale address.  The first
 * call on a device (or in a new context) also loads the library's device
 * code there, which the CUDA runtime does with an allocation of its own:
 * make that first call before any stream capture, and before the point after
 * which nothing may allocate.  All calls share the one array, which keeps the previous call's
 * contents: two calls whose work overlaps on the GPU (different streams, or
 * different host threads without ordering) race on it and give wrong results.
 * Device-detected errors show up as next_token = -1; their status bits are not
 * reported by this entry point. */
#define SV_ETOOLARGE (-4)
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)
int sv_verify_sample_noalloc(const float *p, int64_t p_row_stride,
                             const float *q, int64_t q_row_stride,
                             const int32_t *t, const float *u_accept,
                             const double *u_resample, int32_t B, int32_t K, int64_t V,
                             int32_t *n_accepted, int32_t *next_token, sv_stream_t stream);

/* Waits for `stream`, copies the workspace's status bits to *flags (host
 * memory) and clears them.  Returns SV_ECUDA if the stream reported an error. */
int sv_get_status(void *workspace, sv_stream_t stream, uint32_t *flags);

/* Launch shape used by the calls above.  The kernels are persistent: their
 * grid holds ctas_per_sm CTAs per SM (0, the default, uses the largest count
 * the SMs can hold at once).  The setting is process-wide and meant
 * for tuning sweeps. */
int sv_set_ctas_per_sm(int32_t ctas_per_sm);

/* Sampling verification straight from logits: p_i = softmax(zp_i / T),
 * q_i = softmax(zq_i / T) with T = temperature (the identical warp the
 * "spec-verify" page requires of both distributions, section "Requirements and
 * limits"), then the sampling rule of sv_verify_sample on those rows; the
 * warped rows are never written to memory.  zp holds B*(K+1) rows and zq B*K
 * rows of V f32 logits, laid out like p and q above.  Rows are read in order:
 * the pair (zp_i, zq_i) once for its normalisers and the accept test of
 * position i, the rejected pair (or zp_K) a second time for the draw.  In
 * calls whose chains of positions are long against the batch (K x resident
 * workers >= B x claims per row pair), the next position's pair may be read
 * together with position i's while the GPU would otherwise wait, and is then
 * not used if position i is rejected.
 * Arithmetic is fp32 with exp2.approx and double-fp32 sums.  An accept test
 * is decided in fp32 only when its margin |u*q - p| exceeds a bound on the
 * fast probabilities' error (derived from the fp32 exponent arguments, an
 * ex2.approx error of at most 2^-20 and the normalisers' sums); otherwise the
 * position's normalisers are recomputed in fp64 across the grid and the test
 * is made in fp64, as in an exact softmax.  Accept decisions therefore equal
 * those of an fp64 softmax except where two fp64 summation orders may round
 * differently (|u*q - p| within ~1e-13 * p); a drawn token may differ only
 * when u*R lies within ~2e-6 of normalised mass of a boundary.  temperature
 * must be positive and finite (else SV_EINVAL); logits must be finite.
 * Greedy needs no warp: argmax softmax(z/T) = argmax z, so sv_verify_greedy
 * takes logits directly.  Workspace and status as above. */
int sv_verify_sample_logits(const float *zp, int64_t zp_row_stride,
                            const float *zq, int64_t zq_row_stride,
                            const int32_t *t, const float *u_accept, const double *u_resample,
                            int32_t B, int32_t K, int64_t V, float temperature,
                            int32_t *n_accepted, int32_t *next_token,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* Acceptance-rate diagnostic: for each sequence b and draft position i < K,
 *   alpha[b][i] = sum_v min(p_i(v) / P_i, q_i(v) / Q_i),
 * P_i, Q_i the totals of rows p (b, i) and q (b, i) (a row with zero total
 * gives alpha = 0), and, when expected_length is not NULL,
 *   expected_length[b] = sum_{m=1..K} prod_{j<m} alpha[b][j],
 * the mean number of accepted draft tokens of a sampling round: the
 * rejection-sampling theorem behind the "spec-verify" page's analytic
 * accepted-length law (section "Measured").  Not part of a verification
 * round: it reads every row p_0..p_{K-1} and q_0..q_{K-1} in full (once from
 * memory; the second sweep over a row pair, after its totals, hits L2).
 * Layout and memory rules as above; alpha is [B][K] f64, expected_length [B]
 * f64.  |alpha - exact| <= 2 * 2^-24 * alpha (fp32 scaling of each term,
 * double-fp32 sums).  Uses the workspace of sv_workspace_size(B, K, V); any
 * call may use a workspace between verification calls. */
int sv_alpha(const float *p, int64_t p_row_stride, const float *q, int64_t q_row_stride,
             int32_t B, int32_t K, int64_t V, double *alpha, double *expected_length,
             void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* Number of CTAs the last call on this thread launched (its grid size). */
int64_t sv_last_grid_size(void);

/* Number of kernels the last call on this thread enqueued: 1 for the
 * single-launch verification path, 3 for the scan / stream / decide chain,
 * 2 for the mixed round (ordering kernel and item kernel), up to 2 for
 * sv_alpha. */
int32_t sv_last_kernel_count(void);

/* Text for an SV_* return code or SV_STATUS_* bit. */
const char *sv_status_string(int code);

/* Library ABI version (this header: 1). */
int sv_version(void);

/* Timeline of the single-launch item kernel, for performance work; the pages
 * have no counterpart.  Only a library built with -DSV_TRACE=1 records it;
 * in any other build both calls return SV_EINVAL.  Each CTA appends records
 * of two uint64 words to its own region of a static device buffer
 * (SV_TRACE_RECORDS records, SV_TRACE_CTA_RECORDS per CTA index over all
 * launches since the last reset; later ones are dropped): word 0 is
 * %globaltimer in ns, word 1 holds the event id in bits 56..63, the CTA in
 * bits 32..55 and the event's argument in bits 0..31.  Consecutive launches
 * append after one another, each CTA's records starting with event 8.
 * Events: 0 CTA start (after the wait for the previous grid), 1 item start
 * (sequence), 2 stage issued (count), 3 item fully issued (stages), 4 item
 * retired (sequence), 5 decision start (sequence), 6 decision end
 * (sequence), 7 producer done, 8 CTA placed (before that wait), 9 CTA exit;
 * and for the bulk-copy workers of sv_verify_sample_logits: 10 chunk claimed
 * (group | chunk << 24), 11 its group appended (group), 12 its stages issued
 * (group), 13 chunk completed by a consumer (group), 14 a group's last
 * arrival decided (sequence | position << 16 | kind << 24; kinds 1 normalisers,
 * 2 masses and draw, 3 fp64 recheck), 15 an arrival found it is its group's
 * last (sequence | position << 16; normaliser groups), 16 that arrival has
 * merged its lane's segment normalisers (the same argument).
 *   sv_trace_reset: enqueues the clearing of the buffer and of the per-CTA
 *     slot counts on `stream` (empty records have time 0).  Calls that
 *     record while another is traced mix their records.
 *   sv_trace_read: copies the first min(max_records, SV_TRACE_RECORDS)
 *     records into `records` (host memory of 16 * max_records bytes), waits
 *     for `stream`, and sets *count to the number copied. */
#define SV_TRACE_CTA_RECORDS 2048
#define SV_TRACE_RECORDS (2048u * 1024u)
int sv_trace_reset(sv_stream_t stream);
int sv_trace_read(void *records, size_t max_records, size_t *count, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
