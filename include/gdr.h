/* gdr.h -- C ABI of the GB300 gated delta-rule training library (libgdr.so).
 *
 * Chunked training (forward and backward) of gated delta-rule linear
 * attention over packed variable-length documents, head dimension 128, on one
 * GPU (sm_103a), in two variants:
 *
 *   KDA  (Kimi Delta Attention): a per-channel log-decay gate g[t][h][0..127].
 *        flashinfer PR #8218 "feat(cake_kda): with grad, add non-deterministic
 *        Cake KDA context-parallel (KCP) autograd backend", opening description
 *        and "Workload" paragraph: packed documents, q/k/v BF16 [T,H,128] with q
 *        and k L2-normalized, g FP32 [T,H,128] pre-activated (no sigmoid, no
 *        softplus, no in-kernel L2 norm), beta BF16 [T,H].
 *   GDN  (Gated DeltaNet): a scalar log-decay per (token, value head) and
 *        grouped Q/K heads.  flashinfer PR #7723 "perf(cake_gdn): prefetch
 *        offset adjoint walk, default LPT segment plan", opening description:
 *        BF16 q/k/v/out/dout, FP32 g and beta, (H_qk, HV) runtime parameters,
 *        dq/dk reduced in FP32 over the value heads of each Q/K head and
 *        converted to the output type once.
 *
 * The recurrence, per (document, value head), state S (K x V = 128 x 128,
 * stored S[k][v]) reset to h0[doc] (or zero) at every document start:
 *     S_t = (I - beta_t k_t k_t^T) diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *     ht[doc] = S after the document's last token.
 * exp(g_t) scales the K index (rows) of S.  For GDN, value head j uses Q/K
 * head j / (HV / Hqk) (contiguous groups).
 *
 * Conventions (all entry points):
 *   - Pointers without a _host suffix are DEVICE pointers; buffers are dense,
 *     row-major, and owned by the caller.  The library never allocates device
 *     memory and never synchronizes the host with the device: every call only
 *     enqueues work on `stream` and returns.
 *   - Layouts.  q, k, dq, dk: [T][Hqk][128] BF16 (KDA: Hqk = HV = H).
 *     v, out, dout, dv: [T][HV][128] BF16.  KDA g, dg: [T][H][128] FP32;
 *     GDN g, dg: [T][HV] FP32.  KDA beta, dbeta: [T][H] BF16; GDN beta, dbeta:
 *     [T][HV] FP32.  States h0, ht, dht, dh0: [N][HV][128][128] FP32, S[k][v].
 *   - cu_seqlens: int32 [N+1] with cu[0] = 0, non-decreasing, cu[N] = T.
 *     Empty documents are allowed (their state passes h0 -> ht).  The device
 *     copy and the host copy (cu_seqlens_host) must hold the same values; the
 *     host copy sizes the launches, the device copy drives the kernels.
 *   - Gate precondition: g finite and >= -10 (the per-block gate
 *     factorization keeps every exponent below FP32 overflow for 8 tokens x
 *     10 = 80 < 88.7).  Outside that range results are unspecified.
 *   - Range precondition of the forward's FP16 operands.  The intermediates
 *     w, Q Gamma, Kd^T and Aqk (functions of q, k, g, beta: of order |q| |k|)
 *     are stored, and the forward walk's copies of the state and of Delta
 *     (of the order of the values v) are multiplied, in FP16, which has the
 *     11-bit significand of the TF32 products but a largest finite value of
 *     65504: q, k rows of norm up to about 100 and state entries below that
 *     bound are required (unit-norm q, k and values v of moderate size, as in
 *     training, satisfy it by orders of magnitude).  The backward's adjoints
 *     are gradients and stay in FP32 / TF32.
 *   - Workspaces.  `saved` carries the forward's intermediates to the
 *     backward; `scratch` holds temporaries.  Sizes come from
 *     *_workspace_bytes.  Both must be 256-byte aligned.
 *   - Alignment of the tensors: q, k, v, g and dout start on a 16-byte
 *     boundary (the kernels copy their rows in 16-byte pieces), out, dq, dk
 *     and dv on a 4-byte boundary; otherwise GDR_INVALID_ARG.  `saved` belongs to
 *     the caller between a forward with save_for_bwd = 1 and the backward.
 *   - Errors are returned as gdr_status, never thrown; a call that returns an
 *     error has enqueued nothing (except GDR_CUDA_ERROR from a launch).
 *   - Calls on one stream are ordered; calls that share a workspace must not
 *     overlap on the GPU.  Inside a call, packs whose longest documents have
 *     at least 64 chunks run their document groups (see gdr_doc_groups) on
 *     internal streams of the current device: two per group (its walks; its
 *     prep or gradient slices), at most eight, created on first use and
 *     shared by all callers, the walks at the highest priorities.  They are
 *     forked from and joined back to the caller's stream with events; the
 *     call's work is still ordered after the stream's earlier work and before
 *     its later work, also under stream capture.
 *   - Results are deterministic (no floating-point atomics).
 *   - Per-device state.  The library keeps, per device, its internal streams
 *     and events, an error word and (for kda_fwd_noalloc) the address of its
 *     device array, all created on first use.  cudaDeviceReset destroys them
 *     behind the library's back: do not call into the library on a device
 *     after a cudaDeviceReset of that device in the same process.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gdr_bf16; /* raw bfloat16 bits */
typedef int gdr_status;

#define GDR_OK 0
#define GDR_INVALID_ARG 1          /* null pointer, bad size, bad head counts, misaligned workspace */
#define GDR_BAD_CU_SEQLENS 2       /* cu[0] != 0, decreasing, or cu[N] != T */
#define GDR_WORKSPACE_TOO_SMALL 3  /* saved_bytes / scratch_bytes below *_workspace_bytes */
#define GDR_UNSUPPORTED 4          /* device is not sm_103 (GB300 / B300) */
#define GDR_STALE_WORKSPACE 5      /* `saved` not filled by a matching forward with save_for_bwd = 1
                                    * (returned by the backward, or by gdr_check_device for the
                                    * device-side header check) */
#define GDR_CUDA_ERROR 6           /* a CUDA launch or runtime call failed */
#define GDR_DEVICE_TIMEOUT 7       /* a kernel's bounded wait ran out (reported by gdr_check_device) */

/* Human-readable name of a status code (static string). */
const char* gdr_status_string(gdr_status status);

/* In-kernel q/k L2 normalization (argument qk_l2norm of the calls below; the
 * pages' "use_qk_l2norm_in_kernel", flashinfer PR #8638 "perf(cake_gdn_kcp):
 * ... graph-replay checkpoint recompute hands its tapes to the backward",
 * workload description).  When non-zero, every (token, Q/K head) vector x of
 * q and of k enters the recurrence as n = x * (sum_c x_c^2 + 1e-6)^(-1/2)
 * (FP32, rounded to BF16 once), and dq, dk are the gradients with respect to
 * the raw q, k (dx = r (dn - n (n . dn)), applied in FP32 before the single
 * rounding).  The forward keeps the normalized q, k and their scales in
 * `saved`; the flag must be the same for the workspace query, the forward and
 * the backward (a mismatch with the forward returns GDR_STALE_WORKSPACE). */

/* Workspace sizes for a KDA problem (host-only; no CUDA calls).
 * saved_bytes: the forward's intermediates kept for the backward (chunk and
 * segment tables, w, u, Q*Gamma, Kd, Delta, Aqk, At, T, gamma, the per-chunk
 * state tape, per-segment state maps of split documents, and with qk_l2norm
 * the normalized q, k).
 * scratch_bytes: temporaries of the backward.  A forward called without a
 * `saved` buffer keeps its intermediates in `scratch`, which must then hold
 * saved_bytes.  Returns GDR_BAD_CU_SEQLENS or GDR_INVALID_ARG on bad input. */
gdr_status kda_workspace_bytes(int64_t T, int32_t H, int32_t N, const int32_t* cu_seqlens_host, int qk_l2norm,
                               size_t* saved_bytes, size_t* scratch_bytes);

/* KDA forward.  Writes out [T][H][128] and, when non-null, ht [N][H][128][128].
 * h0 may be null (zero initial state).  When save_for_bwd is non-zero, the
 * intermediates go to `saved` (saved_bytes >= the queried size) and the
 * buffer is stamped for kda_bwd; otherwise `saved` may be null and the
 * intermediates go to `scratch`. */
gdr_status kda_fwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const gdr_bf16* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t H,
                   float scale, int qk_l2norm, const float* h0, gdr_bf16* out, float* ht, void* saved,
                   size_t saved_bytes, int save_for_bwd, void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* KDA backward from a forward with save_for_bwd = 1 on the same inputs.
 * dout [T][H][128]; dht may be null (zero).  Writes dq, dk, dv [T][H][128]
 * BF16, dg [T][H][128] FP32, dbeta [T][H] BF16 and, when non-null, dh0.
 *
 * Saved-buffer stamp.  A saving forward writes a header at the start of
 * `saved`: a magic word, T, N, the head counts, the variant, the segment
 * length, the qk_l2norm flag, a hash of cu_seqlens_host and the number of
 * the saving forward in this process (1, 2, ...); it also records the header
 * in a host registry keyed by the buffer's address.  The backward checks it
 * twice.  On the host, before enqueueing anything: a buffer this process last
 * filled with other arguments returns GDR_STALE_WORKSPACE.  On the device
 * (asynchronously, no host synchronization): the header must match the
 * backward's arguments, and for a registered address also the forward's
 * number, so that a buffer overwritten in place by another saved buffer is
 * caught; a mismatch makes the next gdr_check_device return
 * GDR_STALE_WORKSPACE, and the backward's outputs are then unspecified (its
 * kernels follow only tables it plans itself, so a bad buffer yields wrong
 * numbers, never an out-of-bounds access).  The contents are
 * position-independent: a saved buffer copied to another address (not
 * registered) is accepted by its header alone. */
gdr_status kda_bwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const gdr_bf16* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t H,
                   float scale, int qk_l2norm, const float* h0, const gdr_bf16* dout, const float* dht,
                   const void* saved, size_t saved_bytes, gdr_bf16* dq, gdr_bf16* dk, gdr_bf16* dv, float* dg,
                   gdr_bf16* dbeta, float* dh0, void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* No-allocation KDA forward.  The paper has no counterpart; this entry point
 * exists for callers that cannot allocate device memory at call time: code
 * running under CUDA stream capture in global mode (where cudaMalloc is not
 * permitted), engines and plugins whose host framework owns every device byte
 * and forbids side allocations, and real-time paths that must not take the
 * allocator's locks or risk an out-of-memory failure mid-step.
 *
 * Same arguments and results as kda_fwd with save_for_bwd = 0 and
 * qk_l2norm = 0, but the
 * forward's intermediates live in one fixed 64 MiB device array inside the
 * library (held by every GPU that loads the library until the process exits)
 * instead of caller-provided workspaces, and nothing is saved for a backward.
 * Limit: the problem's intermediates (the saved_bytes that kda_workspace_bytes
 * reports for the same T, H, cu_seqlens) must fit in 64 MiB -- about 270
 * (chunk, head) pairs, e.g. 4096 tokens at H = 4; larger problems are rejected
 * with GDR_WORKSPACE_TOO_SMALL before anything is enqueued.  The call itself
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array, which keeps
 * the previous call's contents; no byte of it needs to start at zero (each
 * call writes everything it reads).  Calls that overlap on the GPU (for
 * example on two streams) race on the array and must be serialized. */
gdr_status kda_fwd_noalloc(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g,
                           const gdr_bf16* beta, const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                           int32_t N, int64_t T, int32_t H, float scale, const float* h0, gdr_bf16* out, float* ht,
                           cudaStream_t stream);

/* GDN counterparts: Hqk Q/K heads, HV value heads (HV % Hqk == 0), scalar
 * FP32 gate g [T][HV] and FP32 beta [T][HV]; dq/dk are [T][Hqk][128], summed
 * in FP32 over the value heads of each Q/K head. */
gdr_status gdn_workspace_bytes(int64_t T, int32_t Hqk, int32_t HV, int32_t N, const int32_t* cu_seqlens_host,
                               int qk_l2norm, size_t* saved_bytes, size_t* scratch_bytes);

gdr_status gdn_fwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t Hqk,
                   int32_t HV, float scale, int qk_l2norm, const float* h0, gdr_bf16* out, float* ht, void* saved,
                   size_t saved_bytes, int save_for_bwd, void* scratch, size_t scratch_bytes, cudaStream_t stream);

gdr_status gdn_bwd(const gdr_bf16* q, const gdr_bf16* k, const gdr_bf16* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N, int64_t T, int32_t Hqk,
                   int32_t HV, float scale, int qk_l2norm, const float* h0, const gdr_bf16* dout, const float* dht,
                   const void* saved, size_t saved_bytes, gdr_bf16* dq, gdr_bf16* dk, gdr_bf16* dv, float* dg,
                   float* dbeta, float* dh0, void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* Diagnostic (no counterpart on the pages): synchronizes the current device
 * and reports whether any kernel of this library gave up a bounded wait on
 * its own asynchronous copies or tensor-core operations since the last check
 * (GDR_DEVICE_TIMEOUT; the word is then cleared), whether a backward found a
 * saved-buffer header that does not match it (GDR_STALE_WORKSPACE, also
 * cleared), or a CUDA error occurred (GDR_CUDA_ERROR).  Kernels never spin
 * without a time limit; a kernel that times out skips the dependent work, so
 * its outputs are then incomplete. */
gdr_status gdr_check_device(void);

/* Failure-detection diagnostics (no counterpart on the pages; they exist so
 * that callers and tests can exercise the timeout path without faulting or
 * hanging a GPU).
 * gdr_inject_device_error(code): writes a non-zero `code` into the current
 * device's error word, as a kernel whose bounded wait ran out would; the next
 * gdr_check_device returns GDR_DEVICE_TIMEOUT.  code <= 0: GDR_INVALID_ARG.
 * gdr_selftest_wait(limit_ns, stream): enqueues one kernel that waits, with
 * the same bounded mbarrier wait as the walks, on a barrier that nothing
 * completes; after limit_ns nanoseconds (1 <= limit_ns <= 1e8, else
 * GDR_INVALID_ARG) it records the timeout in the error word and exits.
 * Device error codes: 3 forward walk, 4 backward walk, 5 this self-test,
 * 6 state-side gradient products, 7 chunk-local gradients, 9 the grouped-GDN
 * prep (all reported as GDR_DEVICE_TIMEOUT); 8 a saved-buffer header that
 * does not match the backward (reported as GDR_STALE_WORKSPACE). */
gdr_status gdr_inject_device_error(int code);

/* Host-side plan of the backward's document groups (no device work).  The
 * backward ranks the documents longest first (ties: lower index first; above
 * 4096 documents the given order), numbers chunks in that order, and runs
 * each group's walk and gradient kernels on a stream of its own: each of the
 * first 3 documents with at least 64 chunks is a group, the remaining
 * documents form one more (a single group when that leaves one).  Writes
 * *n_groups (at most 4) and the group bounds: group i holds ranks
 * [rank_bounds[i], rank_bounds[i+1]) and chunks [chunk_bounds[i],
 * chunk_bounds[i+1]); both arrays need room for 5 entries.  Errors:
 * GDR_INVALID_ARG for null pointers or N < 0, GDR_BAD_CU_SEQLENS for a
 * cu_seqlens that does not start at 0 or decreases. */
gdr_status gdr_doc_groups(int32_t N, const int32_t* cu_seqlens_host, int32_t* rank_bounds, int64_t* chunk_bounds,
                          int32_t* n_groups);
gdr_status gdr_selftest_wait(uint64_t limit_ns, cudaStream_t stream);

/* Benchmark support (no counterpart on the pages): opt-in per-kernel timing.
 * gdr_profile_enable(1) clears previous records and makes every subsequent
 * kernel launch of this library record a pair of CUDA events on its stream;
 * gdr_profile_enable(0) stops recording and keeps the records for the report.  gdr_profile_report synchronizes the
 * recorded events and writes one line per kernel, "<name> <launches>
 * <total_ms> <token_heads>\n" (the sum over its launches of their durations
 * and of the (token, value head) pairs each worked on; launches of different
 * document groups may overlap in time), in first-launch order, NUL-terminated,
 * into buf; it returns GDR_INVALID_ARG if buf_bytes is too small.  Kernel
 * names: plan, check, l2norm, prep, walk_fwd_sum, merge_fwd, walk_fwd, walk_bwd_sum,
 * merge_bwd, walk_bwd, grad_state, grad, group_reduce (the _sum and merge
 * launches run only for split packs, l2norm only with qk_l2norm). */
int gdr_profile_enable(int on);
gdr_status gdr_profile_report(char* buf, size_t buf_bytes);

/* gdr_launch_count(): the number of kernel launches the compute calls of this
 * library have enqueued since it was loaded (all devices, all threads); a
 * benchmark reads it before and after a timed region.
 * gdr_set_serial(on): while on != 0, every compute call enqueues all its
 * launches on the caller's stream, its document groups one after another
 * (same kernels, same results, no overlap between groups), so that
 * per-kernel event timing measures each launch alone.  Process-wide; returns
 * the previous setting.  Default off. */
uint64_t gdr_launch_count(void);
int gdr_set_serial(int on);

/* gdr_set_segment_chunks(chunks): the state walks split a long document into
 * segments walked in parallel (summary walks give each segment's affine map
 * of its start state, a merge chains the segments' start states, then every
 * segment's walk runs from its own start state; flashinfer PR #7723,
 * "perf(cake_gdn): prefetch offset adjoint walk, default LPT segment plan",
 * segment plan).  By default (chunks = 0) a pack is split only when the
 * longest document's walk chain (about 8.3 us per chunk, forward and backward
 * together) outlasts the rest of the pack's work spread over the SMs (about
 * 50 us of SM time per chunk and head); its segments then have about
 * max(64, total chunks x heads / SM count) chunks, and documents no longer
 * than one segment stay whole.  chunks > 0 forces segments
 * of about that many chunks (tests and tuning).  Process-wide, read by every
 * *_workspace_bytes, forward and backward call; the saved-buffer stamp
 * records it, so a backward planned with another setting than its forward
 * returns GDR_STALE_WORKSPACE.  Returns the previous setting. */
int gdr_set_segment_chunks(int chunks);

/* Host-side segment plan of the state walks (no device work): writes the
 * segment length in chunks that the compute calls would use for this pack
 * and value-head count (*seg_chunks = 0 when no document is split) and the
 * number of walk segments (*n_segments: one per document no longer than a
 * segment, ceil(chunks / segment length) for a longer one).  Reads the
 * gdr_set_segment_chunks setting and the device's SM count (152 when no
 * device answers).  Errors: GDR_INVALID_ARG for null pointers, N < 0 or
 * HV <= 0; GDR_BAD_CU_SEQLENS for a cu_seqlens that does not start at 0 or
 * decreases. */
gdr_status gdr_segment_plan(int32_t N, const int32_t* cu_seqlens_host, int32_t HV, int32_t* seg_chunks,
                            int64_t* n_segments);

/* gdr_set_slice_chunks(chunks): a document group that holds one unsplit
 * document longer than a slice walks it slice by slice (the state, or the
 * adjoint, passed on exactly in FP32 between the slices' launches), so that
 * the forward walk starts once the first slice is prepared and the
 * backward's gradient kernels of a slice run while the walk goes on with the
 * next; the results are bit for bit those of the whole walk.  The first and
 * the last slice are shorter (half a slice in the forward walk, a quarter in
 * the backward walk, at least 2 chunks; the last one may take one chunk
 * more), the chunks between them go in equal slices of about the slice
 * length, and every slice starts at an even chunk; a document shorter than
 * two end slices and two chunks is cut into whole slices.  chunks > 0 sets
 * the slice length (rounded down to an even number, at least 2); 0 restores
 * the default of 128 chunks.  Process-wide; returns the previous setting. */
int gdr_set_slice_chunks(int chunks);

/* Host-side slice plan of a pipelined walk (no device work), as the forward
 * (direction 0) or the backward (direction 1) walk cuts a document of
 * nchunks chunks at the current slice length: writes *n_slices and the slice
 * bounds 0 = bounds[0] < bounds[1] < ... < bounds[*n_slices] = nchunks
 * (slice i holds chunks [bounds[i], bounds[i+1]); the backward walks them
 * last slice first).  nchunks = 0 gives no slice (bounds[0] = 0).  bounds
 * needs room for *n_slices + 1 entries; cap is its length.  Errors:
 * GDR_INVALID_ARG for null pointers, nchunks < 0, a direction other than 0
 * or 1, or a cap too small for the plan. */
gdr_status gdr_walk_slices(int32_t nchunks, int32_t direction, int32_t* bounds, int32_t cap, int32_t* n_slices);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
