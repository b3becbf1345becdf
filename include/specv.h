/*
 * specv.h -- C ABI of the GB300 speculative-decoding verification library
 * (libspecv.so).
 *
 * Two operations, both defined on the pages this library restates:
 *
 *   spec_verify    batched lossless draft verification.  For each request b
 *                  and draft position j < ell_b it forms the temperature
 *                  softmax p of target row j and q of draft row j over the full
 *                  vocabulary, accepts draft token x_j when u_j * q(x_j) <
 *                  p(x_j) (i.e. with probability min(1, p/q)), stops at the
 *                  first rejection n, and emits one more token: a draw from the
 *                  normalised residual max(p_n - q_n, 0) after a rejection, or a
 *                  bonus draw from p of target row ell_b when every tested
 *                  draft was accepted.
 *                  Sources: "UraionSpec: A Faithful Implementation of
 *                  Confidence-Scheduled Speculative Decoding" §2.1, eq.
 *                  (acceptance); "breaking down dspark and its lineage", section
 *                  "Preserving the target distribution during verification";
 *                  "AngelSpec" §1 and §4.1 (verified prefix plus one
 *                  target-generated bonus token).
 *
 *   spec_schedule  confidence-scheduled verify lengths.  Prefix survival
 *                  s_{b,k} = prod_{t<=k} c_{b,t} (s_{b,0} = 1), estimated progress
 *                  A_b(n) = sum_{k<=n} s_{b,k}, candidates taken in order of
 *                  survival (ties: shallower position, then lower request), and
 *                  the budget N = sum_b (ell_b + 1) chosen to maximise
 *                  tau(N) / C(N) against a piecewise-linear round-cost table.
 *                  Sources: "AngelSpec" §4.2, eqs. (19)-(24); "UraionSpec" §3.5,
 *                  Algorithm 1 (hardware-aware prefix scheduler).
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless marked host.  The caller
 *     owns every buffer; the library never allocates or frees device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  No call synchronises the stream except
 *     spec_read_status.
 *   - A negative return value is an error detected on the host: nothing was
 *     launched and no output was written.  Errors found in device data (a bad
 *     token id, a NaN row, ...) mark the affected request (out_accept_len = -1,
 *     its tokens -1) and set a status word in the workspace, read with
 *     spec_read_status.  For spec_verify the word holds the status of the most
 *     recent call on that workspace (each call resets it); for the schedulers
 *     it is sticky until read.
 *   - Every device wait in the kernels is bounded; on expiry the call reports
 *     SPEC_ERR_TIMEOUT in the status word and the kernel returns.
 */
#ifndef SPECV_H
#define SPECV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* spec_stream_t; /* a cudaStream_t */

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

enum {
    SPEC_OK = 0,
    SPEC_ERR_NULL = -1,        /* a required pointer is NULL */
    SPEC_ERR_SHAPE = -2,       /* B, gamma, V or min_len out of range */
    SPEC_ERR_ALIGN = -3,       /* a pointer is not aligned to its element size / 16 B */
    SPEC_ERR_TEMPERATURE = -4, /* temperature not 0 and not in [1e-4, 1e4], or NaN */
    SPEC_ERR_VERIFY_LEN = -5,  /* device: verify_len[b] outside [0, gamma] */
    SPEC_ERR_TOKEN = -6,       /* device: draft token outside [0, V) at a tested position */
    SPEC_ERR_WORKSPACE = -7,   /* workspace smaller than the *_workspace_bytes value */
    SPEC_ERR_COST_TABLE = -8,  /* cost table: n outside [1, 32], knots not increasing, cost <= 0 */
    SPEC_ERR_NONFINITE = -9,   /* device: a needed logit row has a NaN, +inf, no finite value, or (T > 0)
                                  a largest |z| * log2(e) / T beyond the fp32 range */
    SPEC_ERR_TIMEOUT = -10,    /* device: a bounded wait expired (results of the call invalid) */
    SPEC_ERR_CUDA = -11,       /* a CUDA runtime call failed (launch, attribute query) */
    SPEC_ERR_UNIFORM = -12,    /* device: a used uniform outside [0, 1) */
    SPEC_ERR_CONFIDENCE = -13, /* device: a confidence outside [0, 1] or NaN */
    SPEC_ERR_ROW_INDEX = -14   /* device: packed rows of a request outside the packed arrays */
};

/* Limits of this build. */
#define SPEC_MAX_BATCH 4096
#define SPEC_MAX_GAMMA 32
#define SPEC_MAX_SCHED_CANDIDATES 16384 /* B * (gamma - min_len) for spec_schedule */

/* ------------------------------------------------------------- verification */

/* Bytes of device workspace spec_verify needs for these sizes (0 if the sizes
 * are out of range).  Depends only on (B, gamma, V, dt). */
size_t spec_verify_workspace_bytes(int B, int gamma, int V, spec_dtype dt);

/*
 * Batched verification of B requests with up to gamma draft tokens each.
 *
 *   target_logits  [B, gamma+1, V] row-major, dt; row j of request b holds the
 *                  target logits for draft position j (row gamma: the position
 *                  after the last draft).  Aligned to the element size.
 *   draft_logits   [B, gamma, V] row-major, dt; may be NULL when temperature == 0
 *                  or gamma == 0 (never read then).
 *   draft_tokens   [B, gamma] int32; only positions j < ell_b are read.
 *   verify_len     [B] int32, ell_b in [0, gamma]; NULL means gamma for all.
 *                  Rows j > ell_b (target) and j >= ell_b (draft) are not read.
 *   temperature    0 = greedy (accept while x_j == argmax of target row j,
 *                  lowest index on ties; emit the argmax of row n); otherwise
 *                  p = softmax(z / T) with T in [1e-4, 1e4].
 *   uniforms       [B, gamma+2] fp32 in [0,1): slot j < gamma is the accept test
 *                  of position j, slot gamma the residual draw, slot gamma+1 the
 *                  bonus draw.  Not read (may be NULL) when temperature == 0.
 *   out_tokens     [B, gamma+1] int32: x_0..x_{n-1}, then the drawn token at
 *                  position n, then -1.
 *   out_accept_len [B] int32: n, the number of accepted drafts (-1 if the
 *                  request's inputs were invalid).
 *   workspace      device scratch of at least spec_verify_workspace_bytes(),
 *                  16-byte aligned; holds the status word of the most recent
 *                  call (reset by each call, read and cleared by
 *                  spec_read_status).  Its contents need no initialisation.
 *                  Two calls sharing one workspace must be ordered on the same
 *                  stream.
 * Draws use the inverse CDF: the token is the smallest v whose running sum of
 * weights exceeds u * (sum of weights).  Returns SPEC_OK or a host-detected
 * error (nothing launched).  B == 0 returns SPEC_OK without launching.
 * Stream order: the call's kernels are programmatic dependent launches, each
 * waiting (griddepcontrol.wait) for the work before it on `stream` before
 * touching global memory, and each letting the next kernel be scheduled early.
 * A caller's own kernel launched right after with programmatic stream
 * serialization must likewise wait before reading the outputs; ordinary
 * launches, copies and events see them complete.
 */
int spec_verify(const void* target_logits, const void* draft_logits, spec_dtype dt, int B,
                int gamma, int V, const int32_t* draft_tokens, const int32_t* verify_len,
                float temperature, const float* uniforms, int32_t* out_tokens,
                int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                spec_stream_t stream);

/*
 * Verification on packed logits ("AngelSpec" §4.2, "Packing and correctness":
 * after the budget is chosen, the unequal request prefixes are packed into one
 * dense verification batch and only those positions reach the target model).
 * Same method, outputs, workspace and errors as spec_verify; only where the
 * logit rows live differs:
 *   target_logits  [K_target, V], dt: request b's target rows 0..ell_b are rows
 *                  target_row[b] .. target_row[b] + ell_b.
 *   draft_logits   [K_draft, V], dt: request b's draft rows 0..ell_b-1 are rows
 *                  draft_row[b] .. draft_row[b] + ell_b - 1 (not read when
 *                  temperature == 0; may then be NULL, as may draft_row).
 *   target_row, draft_row  [B] int32 device arrays (the row index).  Any
 *                  placement is allowed (dense request-major packing is what
 *                  spec_pack_rows writes); a request whose rows fall outside
 *                  [0, K) is marked invalid with SPEC_ERR_ROW_INDEX and none of
 *                  its rows are read.
 *   verify_len     [B] int32 as for spec_verify (NULL: gamma for all).
 * Fixed launch shapes for given (B, gamma, V, dt, temperature), no host
 * synchronisation: capturable in a CUDA graph, one per batch shape.
 */
int spec_verify_packed(const void* target_logits, int K_target, const void* draft_logits, int K_draft,
                       const int32_t* target_row, const int32_t* draft_row, spec_dtype dt, int B,
                       int gamma, int V, const int32_t* draft_tokens, const int32_t* verify_len,
                       float temperature, const float* uniforms, int32_t* out_tokens,
                       int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                       spec_stream_t stream);

/*
 * Dense request-major packing of ragged prefixes (the layout of the packed
 * batch in "AngelSpec" §4.2): from verify_len [B] (device), writes
 *   target_row[b] = sum_{b' < b} (ell_b' + 1),   draft_row[b] = sum_{b' < b} ell_b',
 *   totals[0] = K_target = sum_b (ell_b + 1),    totals[1] = K_draft = sum_b ell_b
 * (all device int32; a verify length outside [0, gamma] counts as no rows).
 * One launch, no host synchronisation.  Requires B <= 4096.
 */
int spec_pack_rows(const int32_t* verify_len, int B, int gamma, int32_t* target_row, int32_t* draft_row,
                   int32_t* totals, spec_stream_t stream);

/*
 * Diagnostics of the last spec_verify that used `workspace` (same B, gamma, V,
 * dt; stream-ordered after it).  Each output is a device pointer or NULL:
 *   px, qx      [B, gamma] fp64: p(x_j), q(x_j) for j < ell_b, NaN elsewhere
 *               (and at temperature 0).
 *   resid_mass  [B] fp64: the total weight of the final draw, sum_v max(p - q, 0)
 *               after a rejection, sum_v p_v (= 1 up to rounding) for a bonus
 *               draw; NaN at temperature 0 or for an invalid request.
 *   status      [B] int32: per-request status (SPEC_OK or a device error code).
 */
int spec_verify_stats(const void* workspace, size_t workspace_bytes, int B, int gamma, int V,
                      spec_dtype dt, double* px, double* qx, double* resid_mass, int32_t* status,
                      spec_stream_t stream);

/* --------------------------------------------------------------- scheduling */

/* Piecewise-linear round cost C(N): knots (tokens[i], cost_ms[i]), i < n, with
 * strictly increasing tokens and positive costs; linear between knots, flat
 * beyond both ends.  Evaluated in fp64 as
 *   cost_ms[i] + ((N - tokens[i]) * (cost_ms[i+1] - cost_ms[i])) / (tokens[i+1] - tokens[i])
 * for tokens[i] <= N < tokens[i+1]. */
typedef struct {
    int n;
    double tokens[32];
    double cost_ms[32];
} spec_cost_table;

typedef enum {
    SPEC_SCHED_EXACT = 0,      /* first budget N that maximises tau(N)/C(N) over every N */
    SPEC_SCHED_ALGORITHM1 = 1, /* Algorithm 1: add candidates while tau/C strictly improves */
    SPEC_SCHED_DCUT = 2        /* D-cut: the table's "tokens" are budget ratios rho_i in (0, 1]
                                  (strictly increasing) and its costs C(B, rho_i); the budget is
                                  K_i = max(B(min_len+1), ceil(rho_i * B(gamma+1))) and the first
                                  maximum of tau(K_i) / C_i is taken ("AngelSpec" §4.2,
                                  eqs. (22)-(24)) */
} spec_sched_mode;

/* Bytes of device workspace spec_schedule needs (its status word). */
size_t spec_schedule_workspace_bytes(int B, int gamma);

/*
 * Per-request verify lengths for B requests with gamma draft positions.
 *   confidence      [B, gamma] fp32 in [0, 1]; confidence[b][k-1] is c_{b,k}.
 *   cost            HOST pointer, copied by value into the launch.
 *   min_len         every request keeps at least min_len drafts (0 <= min_len <= gamma).
 *   sts_temperature HOST [gamma] fp32 > 0 or NULL: Sequential Temperature
 *                   Scaling ("UraionSpec" §2.4): the scheduler uses the calibrated
 *                   confidence c_{b,k}^(1/T_k) (fp64 pow) in place of c_{b,k}.
 *   out_verify_len  [B] int32 in [min_len, gamma] (all -1 if a confidence is invalid).
 * Numbers: survival products are fp64, left to right; each survival is then
 * rounded to a multiple of 2^-46 (nearest, ties to even).  Candidates are
 * ordered by that value (ties: shallower position, then lower request) and
 * progress values are exact integer sums of it, so tau(N) does not depend on
 * the order of summation; objectives tau / C are fp64 with explicit rounding.
 * Results are reproducible bit for bit.  The status word in `workspace` is
 * sticky: set on an error, cleared by spec_read_status (zero the workspace
 * once before first use).  Requires B <= 4096, gamma <= 32,
 * B * (gamma - min_len) <= 16384.  One thread-block cluster per call.
 */
int spec_schedule(const float* confidence, int B, int gamma, const spec_cost_table* cost,
                  int min_len, spec_sched_mode mode, const float* sts_temperature,
                  int32_t* out_verify_len, void* workspace, size_t workspace_bytes,
                  spec_stream_t stream);

/*
 * Static verify lengths ("breaking down dspark and its lineage", section
 * "Verify smarter, not longer": a static confidence threshold, zero recovering
 * fixed-length verification; "UraionSpec" §3.5, the fixed-length and
 * static-threshold StaticScheduler).  Request b keeps its leading positions k
 * whose (optionally STS-calibrated) confidence is at least `threshold`, at most
 * max_len and at least min_len of them: threshold <= 0 gives fixed length
 * max_len, and then confidence may be NULL.  0 <= min_len <= max_len <= gamma.
 * Requests are independent: one with a confidence outside [0, 1] (or NaN) gets
 * verify length -1 and the status word SPEC_ERR_CONFIDENCE; the others are
 * scheduled as usual.  Other arguments as for spec_schedule; any B <= 4096.
 */
int spec_schedule_static(const float* confidence, int B, int gamma, float threshold, int max_len,
                         int min_len, const float* sts_temperature, int32_t* out_verify_len,
                         void* workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * Host-side STS fit ("UraionSpec" §2.4 and §3.6): for positions k = 1..gamma
 * in order, the temperature T_k on the grid (i+1)/10, i = 0..99 (the 100
 * points of 0.1..10) minimising the 15-bin expected calibration error of the
 * cumulative survival prod_{j<k} c_j^(1/T_j) * c_k^(1/T) against the labels
 * [accept_len >= k]; earlier positions keep their chosen T; ties go to the
 * smaller T.  All HOST pointers: confidence [n, gamma] fp32, accept_len [n]
 * int32 (observed with verify_len = gamma), out_temperature [gamma] fp32,
 * out_ece [gamma] fp64 or NULL.  Runs on the CPU, fp64.
 */
int spec_sts_fit(const float* confidence, const int32_t* accept_len, int n, int gamma,
                 float* out_temperature, double* out_ece);

/* ------------------------------------------------- verification, no workspace */

/* Size of the device scratch array that spec_verify_static uses (8 MiB on each
 * device that loads the library, held until the process exits). */
#define SPEC_STATIC_WORKSPACE_BYTES (8u << 20)

/*
 * spec_verify without a workspace argument, for callers that cannot allocate
 * device memory where they verify (an allocator that must not grow inside a
 * capture or a latency-critical loop, a plugin handed only input and output
 * buffers, a runtime with a memory budget fixed at start-up).  It has no
 * counterpart on the pages: it is the same verification as spec_verify, with
 * the scratch taken from a statically sized array in device memory instead
 * of from the caller.
 *
 * Arguments, outputs and results are those of spec_verify.  It allocates
 * nothing (no cudaMalloc, no cudaFree).
 *   - Returns SPEC_ERR_WORKSPACE, launching nothing, when
 *     spec_verify_workspace_bytes(B, gamma, V, dt) exceeds
 *     SPEC_STATIC_WORKSPACE_BYTES (e.g. B=64, gamma=16, V=131072 bf16 needs
 *     about 1.1 MiB; B=256, gamma=16, V=131072 about 4.3 MiB).
 *   - Every call looks up the array's device address on the current device
 *     (so an address never outlives a cudaDeviceReset).  The first lookup on a
 *     device may load the library's device code; make that first call before
 *     any stream capture.
 *   - Every call on a device uses the same array and leaves its contents
 *     behind.  Nothing in it needs to start at zero.  Calls that can overlap
 *     on the GPU (different streams without ordering, or several host threads)
 *     race on it: order them on one stream.
 *   - The device status word lives in that array and cannot be read through
 *     this call; invalid requests are still reported per request
 *     (out_accept_len = -1).
 */
int spec_verify_static(const void* target_logits, const void* draft_logits, spec_dtype dt, int B, int gamma,
                       int V, const int32_t* draft_tokens, const int32_t* verify_len, float temperature,
                       const float* uniforms, int32_t* out_tokens, int32_t* out_accept_len,
                       spec_stream_t stream);

/*
 * Self-test of the bounded waits.  The streaming kernel waits on mbarriers for
 * its own bulk copies; every such wait gives up after 2 s of the GPU's global
 * timer and the call then reports SPEC_ERR_TIMEOUT instead of hanging.  This
 * call runs the same wait routine with a limit of limit_ns (1e3 .. 2e9):
 *   status[0], elapsed_ns[0]: a wait on a barrier nothing completes; expect
 *                             SPEC_ERR_TIMEOUT after about limit_ns;
 *   status[1], elapsed_ns[1]: a wait on a completed phase; expect SPEC_OK at once.
 * status [2] int32 and elapsed_ns [2] uint64 are device pointers.  One launch
 * of one warp.
 */
int spec_selftest_wait(long long limit_ns, int32_t* status, unsigned long long* elapsed_ns,
                       spec_stream_t stream);

/*
 * Test hook of the streaming kernel's timeout path (off by default).  While
 * `on` is nonzero, later spec_verify calls (made from any thread) treat the
 * first copy wait of every warp of the streaming kernel as expired, without
 * waiting for it.  The warps then let their copies in flight land (each wait
 * bounded as usual) and stop; the call marks every request invalid
 * (out_accept_len = -1) and its status word reads SPEC_ERR_TIMEOUT.  No copy
 * is lost and nothing hangs; it exercises the path that a bulk copy which
 * never completes would take.  Returns SPEC_OK.
 */
int spec_selftest_expire_first_wait(int on);

/* ------------------------------------------------------------------ status */

/* Synchronises `stream`, reads the device status word of `workspace` into
 * *status and clears it: for a verification workspace the status of the most
 * recent call on it, for a scheduler workspace the first error since the last
 * read.  Returns SPEC_OK or SPEC_ERR_CUDA. */
int spec_read_status(void* workspace, spec_stream_t stream, int* status);

/* A static English description of a status code. */
const char* spec_status_string(int status);

/* ---------------------------------------------------------------- profiling */

/* Registers two cudaEvent_t handles (as void*) that later spec_verify calls
 * record on their stream immediately before and after the row-statistics
 * kernel (the HBM-streaming pass), so a caller can time that kernel alone.
 * Pass NULL, NULL to stop.  Process-wide setting: calls racing with it on
 * other threads may record the old or the new pair. */
int spec_profile_events(void* before_row_stats, void* after_row_stats);

/* Number of kernels one spec_verify call launches for these arguments
 * (depends on temperature == 0 and B == 0 only). */
int spec_verify_kernel_count(int B, float temperature);

#ifdef __cplusplus
}
#endif

#endif /* SPECV_H */
