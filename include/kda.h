/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) mixer core.
 *
 * What the library computes, per sequence n, head h and token t (channel
 * c = h*128 + i, i < 128):
 *
 *   1. short causal conv + SiLU on each of the planes q, k, v
 *        x~[c] = sum_{j<4} conv_w[p][c][j] * x_p[t-3+j][c],  a = x~ * sigmoid(x~)
 *      inputs before the sequence start come from the conv ring (slot 0
 *      oldest); "Kimi Delta Attention (KDA) -- analysis & C kernel plan",
 *      section "The KDA layer, precisely" (q = SiLU(ShortConv_4(W_q x)) ...);
 *      "ferrox-models 0.8.0, module kda" (depthwise causal Conv1d, padding
 *      kernel_size-1, no bias; KdaState keeps the raw projected inputs).
 *   2. q^ = a_q / sqrt(sum a_q^2 + l2_eps) * q_scale,  k^ = a_k / sqrt(sum a_k^2 + l2_eps),
 *      v^ = a_v  ("ferrox-models 0.8.0, module kda": L2-normalise q and k with
 *      eps 1e-6, then scale q by head_dim^-0.5).
 *   3. g[c] = gate_lower_bound * sigmoid(exp(A_log[h]) * (z[t][c] + dt_bias[c]))
 *      ("Kimi K3 - Retention gate - OpenModelAtlas", gate formula and the
 *      gate.py excerpt naive_kda_lowerbound_gate);  beta = sigmoid(b[t][h]).
 *   4. S' = Diag(exp(g)) S;  S = S' + beta k^ (v^ - S'^T k^)^T;  o_core = S^T q^
 *      ("Kimi Delta Attention (KDA) -- analysis & C kernel plan", section
 *      "Recurrence"); S is 128 x 128 fp32 per (sequence, head), rows = key.
 *   5. o = o_core / sqrt(mean_i o_core^2 + norm_eps) * norm_w[i] * sigmoid(gout[t][c])
 *      (same page, section "The KDA layer, precisely": RMSNormGated with a
 *      sigmoid gate; "ferrox-models 0.8.0, module kda", fact 2).
 *
 * Conventions shared by every entry point
 *   - The caller owns every buffer.  The library allocates no device memory
 *     (kda_prefill_noalloc's fixed scratch array aside) and the prefill and
 *     decode calls never synchronise: all work is ordered on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream), and the small tables
 *     a call needs (cu_seqlens, the chunk table) are built on the device from
 *     kernel arguments, never copied from host memory.  A call may fan work
 *     out to streams it is given or creates, and joins them back into
 *     `stream` before it returns (kda_prefill's overlapped windows,
 *     kda_prefill_host's copy streams).  kda_workspace_status and
 *     kda_noalloc_status synchronise `stream` by design.
 *   - The library keeps a few caches, and no other state:
 *       per device: the SM count and kernel attributes it has set;
 *       per host thread and device: the overlapped windows' high-priority
 *       stream and seven events, created on the thread's first windowed call
 *       and released when the thread exits;
 *       per CUDA context: the address of kda_prefill_noalloc's scratch array.
 *   - Every pointer marked "device" must be a device (or managed) address
 *     aligned to 16 bytes, except b which needs only element alignment.
 *   - Token tensors are token-major: element (t, c) at t*(H*128) + c.
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned as a status; nothing is written in that case.  Launch
 *     errors are reported as KDA_ERR_CUDA; asynchronous faults surface at the
 *     caller's next synchronisation.  No kernel traps or asserts.
 *   - Results are deterministic: repeated calls on the same inputs give the
 *     same bytes (no atomics in any reduction).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2, /* head_dim != 128, conv_kernel != 4, algo/bound mismatch */
    KDA_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_TIMEOUT = 5      /* a bounded in-kernel wait gave up (read via kda_workspace_status) */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/* Prefill algorithm.  AUTO picks CHUNKED for bf16 I/O with the softplus gate
 * or with the bounded gate and a bound >= -5.5 (the bounded gate's
 * tensor-core diagonal blocks need every 16-token rescaling factor below
 * e^88), and SCAN otherwise.  SCAN is the fp32 sequential recurrence.
 * Segments: the recurrence of a single sequence whose heads leave SMs idle
 * can run as P segments in parallel: each segment's map S -> M S + B (the
 * state exchange a context-parallel split of one sequence needs), composed by
 * a scan, then every segment again from its true starting state.  This
 * computes the same function up to rounding and takes the single-pass
 * workspace plus 3P - 5 states of H x 128 x 128 fp32 (included in
 * kda_prefill_workspace_bytes).  AUTO segments when P >= 5 segments of at
 * least 8 chunks fit (2P - 3 CTAs per head on the device's SMs), or P >= 3
 * for a sequence of 64 to 128 chunks (measured on GB300: below and above that
 * range the overlapped windows are as fast or faster with 3 or 4 segments);
 * otherwise a single sequence runs as the overlapped windows of
 * kda_prefill_windows.
 * CHUNKED_SEGMENTS segments from P = 3; CHUNKED never segments.
 * kda_prefill_algo reports CHUNKED for all three. */
typedef enum { KDA_ALGO_AUTO = 0, KDA_ALGO_SCAN = 1, KDA_ALGO_CHUNKED = 2, KDA_ALGO_CHUNKED_SEGMENTS = 3 } kda_algo;

/* Decay gate.
 *   BOUNDED: g = gate_lower_bound * sigmoid(exp(A_log) (z + dt_bias)), in
 *     (lb, 0). This is the Kimi K3 gate ("Kimi K3 - Retention gate -
 *     OpenModelAtlas", gate formula).
 *   SOFTPLUS: g = -exp(A_log) softplus(z + dt_bias), unbounded below. This is
 *     the earlier Kimi-Linear gate ("Kimi Delta Attention (KDA) -- analysis &
 *     C kernel plan", status note; fused_kda_gate with bias = dt_bias). With it
 *     gate_lower_bound is ignored.  The chunked form (bf16 I/O) then sums the
 *     diagonal 16 x 16 blocks of each chunk position pair by position pair on
 *     the CUDA cores, as the retention-gate page says the old gate needed
 *     ("Kimi K3 - Retention gate", section "Why"), so that no rescaling factor
 *     leaves fp32 range; its chunk preparation is about 1.5x slower than with
 *     the bounded gate. */
typedef enum { KDA_GATE_BOUNDED = 0, KDA_GATE_SOFTPLUS = 1 } kda_gate;

typedef struct {
    int32_t num_heads;      /* H >= 1 */
    int32_t head_dim;       /* must be 128 */
    int32_t conv_kernel;    /* must be 4 */
    int32_t io_dtype;       /* kda_dtype of q,k,v,z,b,gout,o and the ring */
    int32_t algo;           /* kda_algo, prefill only */
    float gate_lower_bound; /* lb < 0, -5 for Kimi K3 */
    float l2_eps;           /* 1e-6 */
    float norm_eps;         /* RMSNorm eps, 1e-5 */
    float q_scale;          /* 0 selects head_dim^-0.5 */
    const float* conv_w;    /* device [3][H*128][4] fp32, planes q,k,v; tap 3 = current token */
    const float* A_log;     /* device [H] fp32 */
    const float* dt_bias;   /* device [H*128] fp32 */
    const float* norm_w;    /* device [128] fp32, shared by all heads */
    int32_t gate_kind;      /* kda_gate */
    /* Test hook, 0 in normal use.  Every in-kernel wait gives up after 2 s
     * (the call then reports KDA_ERR_TIMEOUT through kda_workspace_status).
     * A nonzero value shortens the waits between the chunk preparation's two
     * warp groups to that many microseconds, so that a test can make a
     * bounded wait run out on demand; the waits that let the kernel's own
     * copies and tensor-core work finish before it frees its resources keep
     * the 2 s limit. */
    uint32_t wait_limit_us;
} kda_params;

/* The prefill algorithm (KDA_ALGO_SCAN or KDA_ALGO_CHUNKED) that kda_prefill
 * runs for these parameters, or -1 when it would reject them. */
int32_t kda_prefill_algo(const kda_params* p);

/* Bytes of device workspace kda_prefill needs for this problem (0 when
 * total_tokens == 0 and n_seqs == 0).  Returns 0 as well for arguments
 * kda_prefill would reject. */
size_t kda_prefill_workspace_bytes(const kda_params* p, int32_t n_seqs, int64_t total_tokens);

/*
 * Stateful varlen prefill: steps 1-5 over n_seqs packed sequences.
 *   q,k,v,z,gout : device [total_tokens][H*128] io_dtype, raw projections
 *                  (z = decay-gate logits, gout = output-gate logits)
 *   b            : device [total_tokens][H] io_dtype, beta logits
 *   cu_seqlens_host : HOST [n_seqs+1] int64, cu[0] = 0, non-decreasing,
 *                  cu[n_seqs] = total_tokens; sequence n is tokens [cu[n], cu[n+1])
 *   S_in         : device [n_seqs][H][128][128] fp32 initial state or NULL (zero)
 *   S_out        : device, same shape, final state; may equal S_in
 *   ring_in      : device [n_seqs][3 planes q,k,v][3 slots][H*128] io_dtype or
 *                  NULL (zero); slot 0 is the oldest raw input
 *   ring_out     : device, same shape, the last three raw inputs of each
 *                  sequence (older slots carried from ring_in when the
 *                  sequence is shorter than three); may equal ring_in; may be
 *                  NULL to skip
 *   o            : device [total_tokens][H*128] io_dtype
 *   workspace    : device, >= kda_prefill_workspace_bytes(), 256-byte aligned;
 *                  owned by the caller, reused freely between calls that do
 *                  not overlap on the GPU
 * Zero-length sequences copy their state (and ring) through unchanged.
 */
kda_status kda_prefill(const kda_params* p,
                       const void* q, const void* k, const void* v, const void* z,
                       const void* b, const void* gout,
                       const int64_t* cu_seqlens_host, int32_t n_seqs, int64_t total_tokens,
                       const float* S_in, float* S_out,
                       const void* ring_in, void* ring_out,
                       void* o, void* workspace, size_t workspace_bytes, void* stream);

/* Number of windows kda_prefill runs these arguments as: 1 for the single
 * pass, S >= 2 when one long sequence's recurrence would leave SMs idle
 * (chunked path, one sequence, fewer heads than SMs, at least 2048 tokens
 * with up to 64 heads or 16384 with more, and a workspace that holds two
 * windows' records).  Then the sequence runs as S <= 4 windows (S <= 3
 * above 48 heads) of whole chunks, of at least 1024 tokens (up to 64 heads) or
 * 8192 tokens each except the last, which is 1/d as long as the others (d = 6
 * above 64 heads, 4 above 32, 2 up to 32): its recurrence runs alone.
 * Window w's chunk preparation overlaps the recurrence of window w - 1 on a
 * second, high-priority stream, and the result is bit-identical to the single
 * pass.  That stream and seven
 * events are created on a host thread's first windowed call on a device and
 * kept for the thread's lifetime (one set per thread and device, never
 * shared between threads).  A call that runs as segments (see kda_algo)
 * reports 1.  The query needs a current CUDA device (it reads the SM count);
 * -1 for arguments kda_prefill would reject. */
int32_t kda_prefill_windows(const kda_params* p, int32_t n_seqs, int64_t total_tokens, size_t workspace_bytes);

/* The number of segments P >= 3 kda_prefill runs the recurrence of one
 * sequence as (see kda_algo), or 0 when it does not segment; -1 for arguments
 * kda_prefill would reject.  Like kda_prefill_windows it reads the current
 * device's SM count and takes the caller's workspace size.  A segmented call
 * launches the chunk preparation, two recurrence passes and the scan of the
 * segment maps (besides the metadata and ring kernels every call runs). */
int32_t kda_prefill_segments(const kda_params* p, int32_t n_seqs, int64_t total_tokens, size_t workspace_bytes);

/* Same as kda_prefill, and records caller-created CUDA events on `stream` at
 * the stage boundaries, for profiling: stage_events[0] before the pre-stage,
 * [1] after the pre-stage (conv, norms, gate, beta), [2] after the chunk
 * preparation (chunked path; right after [1] on the scan path), [3] after
 * the recurrence (on the chunked path it includes the RMSNormGated output),
 * [4] after the separate RMSNormGated epilogue (scan path; right after [3]
 * on the chunked path), [5] after the conv-ring update.  stage_events holds
 * KDA_PREFILL_EVENTS cudaEvent_t handles (any may be NULL to skip it) or is
 * NULL.  With events the call always runs the single pass (one window), so
 * that every stage boundary is a point on `stream`. */
#define KDA_PREFILL_EVENTS 6
kda_status kda_prefill_with_events(const kda_params* p,
                                   const void* q, const void* k, const void* v, const void* z,
                                   const void* b, const void* gout,
                                   const int64_t* cu_seqlens_host, int32_t n_seqs,
                                   int64_t total_tokens, const float* S_in, float* S_out,
                                   const void* ring_in, void* ring_out, void* o, void* workspace,
                                   size_t workspace_bytes, void* stream, void* const* stage_events);

/*
 * Batched one-token decode for n_sessions independent sessions (one token
 * each): steps 1-5 with the state and ring updated in place.
 *   q,k,v,z,gout : device [n_sessions][H*128] io_dtype
 *   b            : device [n_sessions][H] io_dtype
 *   S            : device [n_sessions][H][128][128] fp32, read and overwritten
 *   ring         : device [n_sessions][3][3][H*128] io_dtype, rolled in place
 *   o            : device [n_sessions][H*128] io_dtype
 * Equal, up to rounding, to kda_prefill with one token per sequence.
 */
kda_status kda_decode(const kda_params* p, int32_t n_sessions,
                      const void* q, const void* k, const void* v, const void* z,
                      const void* b, const void* gout,
                      float* S, void* ring, void* o, void* stream);

/*
 * Multi-token decode (speculative verify) over a state pool.
 *
 * Each of the n_sessions sessions advances by n_tokens consecutive tokens,
 * 1 <= n_tokens <= KDA_DECODE_MAX_TOKENS, and produces one output row per
 * token. The recurrence stays sequential over the register-resident state
 * inside one launch. This follows the batched verify-rows call and its
 * rollback on "memra-engine 0.124.0, module kda" (kda_verify_rows_cached,
 * kda_verify_rollback_rows, KdaRowsStash). The step per token is the decode
 * step above.
 *
 *   q,k,v,z,gout : device [n_sessions][n_tokens][H*128] io_dtype
 *   b            : device [n_sessions][n_tokens][H] io_dtype
 *   slots        : device int32 [n_sessions], the pool slot of each session,
 *                  or NULL (session i uses slot i).
 *                  - Slots must be distinct.
 *                  - A slot outside [0, n_slots) skips its session: its
 *                    state, ring and output rows are left untouched.
 *   S_in, S_out  : device state pools [n_slots][H][128][128] fp32. S_in is
 *                  read and S_out written; they may alias (in-place update).
 *   ring_in, ring_out : device ring pools [n_slots][3][3][H*128] io_dtype,
 *                  slot 0 oldest. They may alias.
 *   o            : device [n_sessions][n_tokens][H*128] io_dtype
 *
 * Rollback (snapshot and replay). Keep S_in and ring_in, i.e. write to
 * separate S_out and ring_out. If only the first j tokens of a round are
 * accepted, call again with those j tokens from S_in and ring_in. This gives
 * the state after token j-1, equal to kda_prefill over the same tokens up to
 * rounding.
 *
 * Errors:
 *   - KDA_ERR_INVALID_ARG: n_tokens out of range, null or misaligned pointers,
 *     or n_slots < n_sessions without slots.
 *   - KDA_ERR_UNSUPPORTED: head_dim or conv_kernel not supported.
 */
#define KDA_DECODE_MAX_TOKENS 64
kda_status kda_decode_multi(const kda_params* p, int32_t n_sessions, int32_t n_tokens,
                            const void* q, const void* k, const void* v, const void* z,
                            const void* b, const void* gout, const int32_t* slots, int32_t n_slots,
                            const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                            void* o, void* stream);

/*
 * kda_prefill without a workspace, for callers that cannot allocate device
 * memory when they run: a plugin inside an engine that owns every byte of
 * device memory, or a serving loop that must not call cudaMalloc/cudaFree
 * because they can synchronise the whole device.  The sources describe no
 * counterpart; this is an interface addition of this library.
 * Same arguments, checks and results as kda_prefill, minus the workspace.  The
 * scratch is a fixed device array of KDA_NOALLOC_SCRATCH_BYTES, held by every
 * GPU that loads the library until the process exits.  The first call in a
 * CUDA context (one per device for runtime-API callers) looks up that
 * array's address (cudaGetSymbolAddress) and caches it with the context:
 * make that first call before any stream capture.  Every call shares the
 * array and leaves its contents behind (each call clears the error word and
 * writes every other byte it reads), so calls that can overlap on the GPU
 * race: issue them in order on one stream.
 * Returns KDA_ERR_WORKSPACE when the problem needs more scratch than the
 * array holds (kda_prefill_workspace_bytes reports the need), and
 * KDA_ERR_UNSUPPORTED for more than 512 sequences in one call (their order is
 * sorted on the host stack).  Calls no memory-allocating routine.  A
 * bounded-wait timeout inside a call is read with kda_noalloc_status.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
kda_status kda_prefill_noalloc(const kda_params* p,
                               const void* q, const void* k, const void* v, const void* z,
                               const void* b, const void* gout,
                               const int64_t* cu_seqlens_host, int32_t n_seqs, int64_t total_tokens,
                               const float* S_in, float* S_out,
                               const void* ring_in, void* ring_out, void* o, void* stream);

/* Synchronises `stream` and reads the error word in kda_prefill_noalloc's
 * scratch array on the current device: KDA_OK, or KDA_ERR_TIMEOUT when a
 * bounded in-kernel wait gave up in an earlier call (the word is then
 * cleared).  Like kda_prefill_noalloc, allocates nothing.  No counterpart in
 * the sources. */
kda_status kda_noalloc_status(void* stream);

/*
 * Prefill of a packed batch held in HOST memory, with the host<->device
 * copies overlapped with the kernels.  An interface addition of this library:
 * the sources time the mixer with its inputs already on the device.
 *
 * The batch is cut into segments of segment_tokens consecutive tokens.  Each
 * segment runs as kda_prefill over the pieces of the sequences inside it,
 * continuing every sequence from the state and ring its previous piece left
 * in S_out / ring_out.  The result equals kda_prefill of the whole batch up
 * to rounding (the chunk boundaries move with the segment boundaries).  Three
 * staging sets in `scratch` rotate: while `stream` runs segment s,
 * `h2d_stream` copies segment s+1 in and `d2h_stream` copies the output of
 * segment s-1 out.
 *
 *   q,k,v,z,gout : HOST [total_tokens][H*128] io_dtype
 *   b            : HOST [total_tokens][H] io_dtype
 *   o            : HOST [total_tokens][H*128] io_dtype, written
 *                  The host arrays should be page-locked (cudaHostAlloc or
 *                  cudaHostRegister); pageable memory gives correct results
 *                  but the copies then do not overlap.
 *   cu_seqlens_host, n_seqs, total_tokens : as for kda_prefill
 *   S_in, ring_in : device, as for kda_prefill (NULL = zero); may alias the outputs
 *   S_out, ring_out : device, as for kda_prefill; both required (they carry
 *                  each sequence across segments)
 *   segment_tokens : tokens per segment, >= 1
 *   scratch      : device, >= kda_prefill_host_scratch_bytes(), 256-byte
 *                  aligned.  Its first 256 bytes are the error word that
 *                  kda_workspace_status(scratch, stream) reads; it covers
 *                  every segment of the call.
 *   stream       : the work starts after what is already queued on it, and it
 *                  is ordered after every copy when the call returns:
 *                  synchronise it before reading o.
 *   h2d_stream, d2h_stream : caller-created streams for the copies, or NULL
 *                  (then the copies run on `stream` and nothing overlaps).
 *
 * Errors: the checks of kda_prefill plus KDA_ERR_INVALID_ARG for a NULL
 * S_out or ring_out or segment_tokens < 1, and KDA_ERR_WORKSPACE for missing,
 * short or misaligned scratch.  Every check runs before anything is queued.
 */
size_t kda_prefill_host_scratch_bytes(const kda_params* p, const int64_t* cu_seqlens_host, int32_t n_seqs,
                                      int64_t total_tokens, int64_t segment_tokens);
kda_status kda_prefill_host(const kda_params* p,
                            const void* q, const void* k, const void* v, const void* z,
                            const void* b, const void* gout,
                            const int64_t* cu_seqlens_host, int32_t n_seqs, int64_t total_tokens,
                            const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                            void* o, int64_t segment_tokens, void* scratch, size_t scratch_bytes,
                            void* stream, void* h2d_stream, void* d2h_stream);

/* Synchronises `stream` and reads the error word the prefill kernels keep in
 * `workspace`: KDA_OK, or KDA_ERR_TIMEOUT when a bounded in-kernel wait gave
 * up during an earlier call on that workspace (the word is then cleared). */
kda_status kda_workspace_status(void* workspace, void* stream);

/* Static string naming a status. */
const char* kda_status_str(kda_status s);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
