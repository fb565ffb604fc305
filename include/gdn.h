/*
 * gdn.h - C ABI of the GB300 (sm_103a) chunked Gated-DeltaNet prefill library.
 *
 * One hybrid Qwen3.5-style Gated-DeltaNet (GDN) layer. Per v-head h, reading
 * q/k head h / (Hv/Hk), the layer
 *   1. applies a causal short convolution (kernel 4) to each q, k and v
 *      channel, with the last three raw inputs carried as the conv state;
 *   2. L2-normalises q and k per head;
 *   3. runs the gated delta rule
 *        S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *        o_t = S_t q_t,
 *      in chunked (WY / UT) form on 64-token blocks.
 * Sources: the layer's state is the per-session "Gated-DeltaNet state"
 * ("The shadow reader", section "One session's state"); a captured state holds
 * the fp32 recurrent state and the last three conv inputs ("qwen3_5: run
 * prompts that share prefixes once per prefix", section "Purpose"); the state
 * advances only in whole grid chunks at absolute positions c * C, with the
 * sub-grid tail pending and forks that restore the state ("The shadow reader",
 * section "Exact on a grid").
 *
 * Conventions for every call:
 *  - All pointers to tensors are DEVICE pointers (cudaMalloc / PyTorch CUDA
 *    memory) unless stated otherwise, 16-byte aligned, C-contiguous. The
 *    caller owns every buffer; the library allocates no device memory.
 *  - Every call validates all arguments on the host before any device work. On
 *    an error status nothing (device memory or host structs) has been changed.
 *  - Device work is enqueued on `stream` and is asynchronous: a call returning
 *    GDN_OK means the work was launched. GDN_ERR_CUDA reports a failed launch;
 *    in that case state buffers may be partially written.
 *  - Results are deterministic. A session's state after a sequence of on-grid
 *    calls depends only on the token values and the grid, not on how the
 *    tokens were split into calls, nor on which other sessions share a call.
 *  - gdn_last_error() returns a message for the last failing call on the
 *    calling host thread.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t). NULL means the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad flag, negative size */
    GDN_ERR_SHAPE = 2,          /* unsupported head count, head dim, grid, dtype */
    GDN_ERR_OFF_GRID = 3,       /* on-grid call on a session whose committed length is off grid */
    GDN_ERR_STATE_MISMATCH = 4, /* session / slot belongs to another layer description, or slot is missing */
    GDN_ERR_WORKSPACE = 5,      /* workspace too small */
    GDN_ERR_CUDA = 6,           /* a CUDA call or launch failed */
    GDN_ERR_TIMEOUT = 7,        /* a bounded device wait ran out (see gdn_device_status) */
    GDN_ERR_NOT_FOUND = 8,      /* no saved state at the given path */
    GDN_ERR_IO = 9              /* a file could not be written or read */
} gdn_status;

enum { GDN_FP32 = 0, GDN_BF16 = 1 };
enum { GDN_CONV_NONE = 0, GDN_CONV_SILU = 1 };

/* Flag of the prefill calls: also process the final partial grid chunk. */
#define GDN_ALLOW_PARTIAL 1u

/* Maximum sessions in one varlen / decode call. */
#define GDN_MAX_SESSIONS 4096

/* The layer. ch = 2 * n_qk_heads * d_k + n_v_heads * d_v conv channels, in the
 * order q | k | v. */
typedef struct gdn_layer_desc {
    int32_t n_qk_heads; /* Hk >= 1 */
    int32_t n_v_heads;  /* Hv, a multiple of Hk (GQA: v-head h reads q/k head h / (Hv/Hk)) */
    int32_t d_k;        /* 64 or 128 */
    int32_t d_v;        /* equal to d_k */
    int32_t grid_c;     /* commit grid C: a multiple of 64 in [64, 4096] (the pages use 64 and 512) */
    int32_t in_dtype;   /* GDN_BF16 or GDN_FP32: x_q, x_k, x_v, conv weights and conv state */
    int32_t out_dtype;  /* GDN_FP32 or GDN_BF16 */
    int32_t conv_act;   /* GDN_CONV_NONE (default) or GDN_CONV_SILU after the conv */
    float q_scale;      /* multiplies the normalised q (1.0) */
    float l2_eps;       /* added to |y|^2 inside the square root of the L2 norm (1e-6), > 0 */
} gdn_layer_desc;

/* A session's recurrent state, or a checkpoint slot (same layout).
 * Host struct; S and conv point to caller-owned device memory. */
typedef struct gdn_session {
    float *S;          /* fp32 [Hv][d_k][d_v]: the state S transposed (row = key dim) */
    void *conv;        /* in_dtype [3][ch]: raw inputs of the last three positions, oldest first */
    int64_t committed; /* tokens consumed so far = absolute position of the next token; -1 = missing slot */
    uint64_t tag;      /* gdn_desc_tag() of the layer this state belongs to */
} gdn_session;

/* Hash of every field of the description; sessions and slots carry it and
 * calls refuse a state whose tag differs (another layer, grid or format). */
uint64_t gdn_desc_tag(const gdn_layer_desc *desc);

/* GDN_OK if the description is supported. */
gdn_status gdn_desc_check(const gdn_layer_desc *desc);

/* Bytes of S and of the conv state for one session of this layer (0 if invalid). */
size_t gdn_state_bytes(const gdn_layer_desc *desc);
size_t gdn_conv_state_bytes(const gdn_layer_desc *desc);

/* Binds S and conv (device buffers of gdn_state_bytes / gdn_conv_state_bytes)
 * to *session, zeroes them on `stream`, sets committed = 0 and the tag. */
gdn_status gdn_session_init(const gdn_layer_desc *desc, gdn_session *session, float *S,
                            void *conv, gdn_stream_t stream);

/* Workspace bytes a prefill call needs for up to `max_tokens` tokens in total
 * over up to `max_sessions` sessions, for any 16-byte-aligned workspace pointer
 * (the size includes room for the library to align it further): the per-block
 * records the prologue hands to the state pass and, for d = 128, the flags by
 * which the one-launch prefill publishes them. Scratch of one call: its
 * contents are not needed afterwards and need no clearing before, and calls
 * that overlap on the GPU must not share it. */
size_t gdn_workspace_size(const gdn_layer_desc *desc, int64_t max_tokens, int32_t max_sessions);

/* Prefill of one session.
 *   xq, xk: in_dtype [n_tokens][Hk * d_k]; xv: in_dtype [n_tokens][Hv * d_v];
 *   g: fp32 [n_tokens][Hv] log-decay (g <= 0); beta: fp32 [n_tokens][Hv];
 *   conv_w: in_dtype [ch][4], tap 3 multiplies the current token;
 *   out: out_dtype [n_tokens][Hv][d_v].
 * Without GDN_ALLOW_PARTIAL the session must be on grid (committed % C == 0)
 * and the call consumes the largest multiple of C of the given tokens; the
 * rest (< C) is the pending tail, which the caller keeps and sends again with
 * the next call. With GDN_ALLOW_PARTIAL every token is consumed, the last grid
 * chunk may be partial and the session may be left off grid: the next call on
 * it must be another partial call, a decode step or a restore.
 * Rows of `out` for consumed tokens are written; the others are untouched.
 * *n_consumed (host) receives the consumed count; session->committed grows by it.
 * Arithmetic: fp32 conv, norm, gates, triangular solve, accumulation and state;
 * with bf16 inputs the block and state products take 16-bit operands (bf16
 * hi/lo pairs for Q K^T, fp16 elsewhere, 11 significant bits), so conv outputs,
 * U and state entries must stay within about 1e4 in magnitude (the fp16 range).
 * fp32 inputs run fp32 throughout. */
gdn_status gdn_prefill_chunks(const gdn_layer_desc *desc, gdn_session *session, const void *xq,
                              const void *xk, const void *xv, const float *g, const float *beta,
                              const void *conv_w, int64_t n_tokens, uint32_t flags, void *out,
                              int64_t *n_consumed, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream);

/* Prefill of n_sessions sessions in one pass (packed / varlen batch).
 * Session i's tokens are rows [cu_seqlens[i], cu_seqlens[i+1]) of the packed
 * xq, xk, xv, g, beta and out (same per-row layouts as gdn_prefill_chunks).
 * cu_seqlens is a HOST array of n_sessions + 1 non-decreasing offsets starting
 * at 0. The sessions must be distinct. Each session follows the rules of
 * gdn_prefill_chunks; n_consumed (host) has n_sessions entries. Every session's
 * result is bit-identical to a gdn_prefill_chunks call on it alone. */
gdn_status gdn_prefill_varlen(const gdn_layer_desc *desc, gdn_session *sessions, int32_t n_sessions,
                              const int64_t *cu_seqlens, const void *xq, const void *xk,
                              const void *xv, const float *g, const float *beta,
                              const void *conv_w, uint32_t flags, void *out, int64_t *n_consumed,
                              void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* gdn_prefill_chunks (gdn_prefill_varlen) that also writes each session's
 * result into a checkpoint slot, as gdn_state_capture(session -> slot) after
 * the call would, but in the same pass: the state kernel stores the final
 * state and conv state twice, and no copy launch follows. A turn of a
 * conversation that keeps a checkpoint at every turn end is one call ("The
 * shadow reader": a checkpoint of the recurrent state at each turn's prompt
 * end). Slots need buffers of this layer, distinct from every session and
 * from each other; their committed and tag are set as a capture sets them.
 * A refused call changes no slot. */
gdn_status gdn_prefill_chunks_checkpoint(const gdn_layer_desc *desc, gdn_session *session, gdn_session *slot,
                                         const void *xq, const void *xk, const void *xv, const float *g,
                                         const float *beta, const void *conv_w, int64_t n_tokens, uint32_t flags,
                                         void *out, int64_t *n_consumed, void *workspace, size_t workspace_bytes,
                                         gdn_stream_t stream);
gdn_status gdn_prefill_varlen_checkpoint(const gdn_layer_desc *desc, gdn_session *sessions, gdn_session *slots,
                                         int32_t n_sessions, const int64_t *cu_seqlens, const void *xq,
                                         const void *xk, const void *xv, const float *g, const float *beta,
                                         const void *conv_w, uint32_t flags, void *out, int64_t *n_consumed,
                                         void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Prefill of n_branches branches that all continue one prefix: branch i's
 * tokens are rows [cu_seqlens[i], cu_seqlens[i+1]) of the packed inputs (as in
 * gdn_prefill_varlen). Every branch starts from the prefix session's state,
 * which the kernels read in place (no copy per branch) and never change; the
 * branch's own buffers receive its result, and its committed becomes the
 * prefix's plus what it consumed. Branch i's result is bit-identical to
 * gdn_state_restore(branch i, prefix) followed by gdn_prefill_chunks on its
 * tokens (the shared-prefix continuation of "The shadow reader" and of
 * "Long context and sessions", section "Checkpoints"). A branch with nothing
 * to process becomes a copy of the prefix. The grid rule applies to the
 * prefix's committed length. Branches and the prefix must be distinct
 * sessions; a branch may be a missing slot (committed < 0) of this layer. */
gdn_status gdn_prefill_branches(const gdn_layer_desc *desc, const gdn_session *prefix, gdn_session *branches,
                                int32_t n_branches, const int64_t *cu_seqlens, const void *xq, const void *xk,
                                const void *xv, const float *g, const float *beta, const void *conv_w,
                                uint32_t flags, void *out, int64_t *n_consumed, void *workspace,
                                size_t workspace_bytes, gdn_stream_t stream);

/* Bytes of the library's built-in scratch used by gdn_prefill_chunks_noalloc
 * (held on every GPU that loads the library, until the process exits). */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)

/* gdn_prefill_chunks for callers that cannot allocate device memory. The
 * pages have no counterpart of this call; it exists for code whose device
 * memory is planned up front by a host framework that owns the allocator, and
 * for latency-critical callers that must not call cudaMalloc / cudaFree (those
 * calls can synchronise the device). Arguments and results are those of
 * gdn_prefill_chunks without the workspace: the scratch is a fixed
 * GDN_NOALLOC_SCRATCH_BYTES array inside the library, and the call allocates
 * nothing. A call whose processed tokens need more than that
 * (gdn_workspace_size(desc, tokens processed, 1) > GDN_NOALLOC_SCRATCH_BYTES;
 * 1,536 tokens for 16 heads of d = 128) is refused with GDN_ERR_WORKSPACE
 * before any device work. The first call on a device looks up the scratch's
 * device address (cudaGetSymbolAddress) with that device current: make that
 * first call before any stream capture. All calls in the process share the
 * one scratch per device, so calls that overlap on the GPU (different streams
 * without ordering between them) race and give wrong results; serialise them.
 * No scratch content needs clearing between calls. */
gdn_status gdn_prefill_chunks_noalloc(const gdn_layer_desc *desc, gdn_session *session, const void *xq,
                                      const void *xk, const void *xv, const float *g, const float *beta,
                                      const void *conv_w, int64_t n_tokens, uint32_t flags, void *out,
                                      int64_t *n_consumed, gdn_stream_t stream);

/* Checkpoint: bitwise copy of src's S and conv state into slot (device to
 * device), and of its committed length and tag. The slot is marked missing
 * (committed = -1) first and only filled in when the copy was launched, so a
 * failed capture leaves a missing slot, never a stale one ("Long context and
 * sessions", section "Checkpoints"; saveSlot in "Sessions on one engine"). */
gdn_status gdn_state_capture(const gdn_layer_desc *desc, const gdn_session *src, gdn_session *slot,
                             gdn_stream_t stream);

/* Puts a captured state back: bitwise copy of slot into dst (S, conv,
 * committed). Refuses a missing slot or one of another layer description. */
gdn_status gdn_state_restore(const gdn_layer_desc *desc, gdn_session *dst, const gdn_session *slot,
                             gdn_stream_t stream);

/* Copies the session's conv state (in_dtype [3][ch], oldest row first) to
 * `out`, which may be device memory or pinned host memory. */
gdn_status gdn_conv_state(const gdn_layer_desc *desc, const gdn_session *session, void *out,
                          gdn_stream_t stream);

/* ---- Serialised states (host memory and files) ----
 *
 * A blob is a 128-byte header followed by S (fp32 [Hv][d_k][d_v]) and the
 * conv state (in_dtype [3][ch]), gdn_state_blob_bytes(desc) bytes in all.
 * Header, little-endian: "GDNSTATE" (8 bytes), version 1 (u32), header bytes
 * 128 (u32), layer tag (u64), n_qk_heads, n_v_heads, d_k, d_v, grid_c,
 * in_dtype (6 x i32), committed (i64), S bytes (u64), conv bytes (u64),
 * payload checksum (u64; 0 = not computed), completion marker (u64), zero
 * padding. The completion marker is written last, after the payload is in
 * place; a blob without it reads as missing, never as an older state.
 * Restoring refuses a blob of another layer description (tag, shapes, grid),
 * of another format version, a blob without its completion marker and one
 * whose checksum does not match, with GDN_ERR_STATE_MISMATCH, and changes
 * nothing then. */
size_t gdn_state_blob_bytes(const gdn_layer_desc *desc);

/* Serialises a session (or slot) into `blob` (host memory, pinned for an
 * asynchronous copy, of blob_bytes >= gdn_state_blob_bytes). The header is
 * written at once with the marker cleared; the payload copies and then the
 * marker follow in `stream` order. The blob must stay allocated, and must not
 * be read as complete, until the stream has passed the call. */
gdn_status gdn_state_serialize(const gdn_layer_desc *desc, const gdn_session *session, void *blob,
                               size_t blob_bytes, gdn_stream_t stream);

/* Restores a blob into `dst` (its own device buffers): validates the header
 * on the host, then enqueues the copies on `stream` and sets dst->committed
 * and dst->tag. The blob must stay allocated until the stream has passed the
 * copies. */
gdn_status gdn_state_deserialize(const gdn_layer_desc *desc, const void *blob, size_t blob_bytes,
                                 gdn_session *dst, gdn_stream_t stream);

/* Saves a session to the file `path` with a payload checksum. Write
 * protocol: the old file is removed first, the blob goes to "<path>.tmp",
 * is flushed to disk and renamed over `path`, then the directory is flushed:
 * after a failure at any point the path holds either the new state or
 * nothing. Synchronises `stream`. GDN_ERR_IO on a file error. */
gdn_status gdn_state_save(const gdn_layer_desc *desc, const gdn_session *session, const char *path,
                          gdn_stream_t stream);

/* Loads the file `path` into `dst` (validation as gdn_state_deserialize, and
 * the checksum); synchronises `stream`. GDN_ERR_NOT_FOUND if there is no file,
 * GDN_ERR_IO if it cannot be read. */
gdn_status gdn_state_load(const gdn_layer_desc *desc, const char *path, gdn_session *dst, gdn_stream_t stream);

/* One token for each of n_sessions sessions (a decode step; leaves sessions
 * off grid). Row i of xq, xk ([n][Hk*d_k]), xv ([n][Hv*d_v]), g, beta ([n][Hv])
 * and out ([n][Hv][d_v]) belongs to sessions[i]; committed grows by one.
 * Defined by the gated delta rule for one token (the recurrence of "Gated
 * Delta Networks", section 3, with the layer's conv and L2 norm). The call
 * allocates nothing and never waits on the host, and its kernels reach the
 * states only through the sessions' device addresses: it can be captured in
 * a CUDA graph on `stream` and replayed with new inputs copied into the same
 * buffers. A replay advances the device states only; `committed` counts the
 * host calls. Errors as for the prefill calls; nothing is launched on error. */
gdn_status gdn_decode_step(const gdn_layer_desc *desc, gdn_session *sessions, int32_t n_sessions,
                           const void *xq, const void *xk, const void *xv, const float *g,
                           const float *beta, const void *conv_w, void *out, gdn_stream_t stream);

/* Raw-gate inputs: g and beta of every token from its raw projections, on the
 * GPU, for the prefill and decode calls above (which take g and beta as given,
 * the form the pages use). The parametrisation is the usual one of
 * Gated-DeltaNet layers, a reading outside the pages: per token t and v-head h,
 *   g[t][h]    = -exp(A_log[h]) * softplus(a[t][h] + dt_bias[h]),
 *   beta[t][h] = 1 / (1 + exp(-b[t][h])),   softplus(x) = log(1 + exp(x)).
 * a, b, g, beta: fp32 device [n_tokens][Hv]; A_log, dt_bias: fp32 device [Hv]
 * (4-byte aligned). g and beta may be the same buffers as a and b. Stream-
 * ordered; errors as for the prefill calls. */
gdn_status gdn_gates(const gdn_layer_desc *desc, const float *a, const float *b, const float *A_log,
                     const float *dt_bias, int64_t n_tokens, float *g, float *beta, gdn_stream_t stream);

/* Per-kernel timing with CUDA events, for benchmarks (off by default).
 * gdn_timing_begin(max_launches) creates 2 * max_launches events and starts
 * recording: every kernel the library launches afterwards, on whatever stream
 * the call names, is bracketed by an event pair on that stream (launches past
 * max_launches are counted but not timed). gdn_timing_end waits for the
 * recorded events, stops recording, and writes per kernel kind its launch
 * count, timed launches and summed device milliseconds into out[0..max_kinds),
 * with *n_kinds the number of kinds that launched. Process-global and not
 * thread-safe: one benchmark thread at a time. */
typedef struct gdn_kernel_time {
    char name[32];        /* kernel kind: prep_wy, prep_wy_tail (the prologue of a call's last blocks, run
                             beside the state pass of its first ones), conv_commit, state_output, state_copy,
                             decode, gates */
    int64_t launches;     /* launches while recording */
    int64_t timed;        /* launches with an event pair */
    double total_ms;      /* summed device time of the timed launches */
} gdn_kernel_time;

gdn_status gdn_timing_begin(int32_t max_launches);
gdn_status gdn_timing_end(gdn_kernel_time *out, int32_t max_kinds, int32_t *n_kinds);

/* Outcome of the device-side bounded waits. Kernels that wait on their own
 * asynchronous operand copies give up after a bounded number of polls instead
 * of hanging; they then record the fact in a device error word, leave their
 * results incomplete and exit. This call synchronises `stream`, reads and
 * clears that word, and returns GDN_ERR_TIMEOUT if it was set, else GDN_OK.
 * (A timeout does not happen in normal operation.) */
gdn_status gdn_device_status(gdn_stream_t stream);

/* Test hook for the timeout path above: while enabled, prefill launches of the
 * bf16 path give up after `wait_limit` polls, and one kernel never issues its
 * first operand copy, so its wait runs out without any fault: enable = 1, the
 * state kernel; enable = 2, the tcgen05 prologue (d_k = d_v = 128). enable = 0
 * restores normal operation; other values are refused with
 * GDN_ERR_INVALID_ARG. Process-global; for tests only. */
gdn_status gdn_debug_inject_wait_timeout(int32_t enable, int64_t wait_limit);

/* Message of the last failing call on this host thread ("" if none). */
const char *gdn_last_error(void);

/* Name of a status code. */
const char *gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
