/*
 * gdr.h -- C ABI of libgdr, the GB300 (sm_103a) gated delta rule library.
 *
 * The gated delta rule (Gated DeltaNet recurrence) keeps, per sequence and
 * head, a d_k x d_v state S and for every token t computes
 *     S'_t = alpha_t S_{t-1},  vhat_t = S'_t^T k_t,
 *     S_t  = S'_t + beta_t k_t (v_t - vhat_t)^T,  o_t = S_t^T q_t
 * ("Linear attention" (arsalanzafar.ai), section "How it works", Eqs. (1)-(4),
 * keys x values layout; the state is updated before it is read, "How linear
 * attention works: a small memory matrix and the gated delta rule", section
 * "Writing a key-value association"). alpha_t = exp(log_alpha_t).
 * No score scale and no normalisation of q or k are applied: the caller
 * passes the vectors to use.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise, to
 *     memory owned by the caller. The library never allocates device memory
 *     at run time and never frees caller memory. What it does keep between
 *     calls, for the life of the process: per device, the SM count and
 *     whether the cooperative launch of the fused schedule fits (cached on
 *     first use, thread-safe); per host thread and device, one side stream
 *     and 8 events for the phased schedule (created by the first phased call
 *     on that thread and device, never destroyed); and the static scratch
 *     array of gdr_chunk_fwd_noalloc, which the module reserves on every
 *     device it is loaded on. No result depends on any of them.
 *   - Tensors are dense and row-major. q, k, v, o, S0, S, S_final and the
 *     workspace start on a 16-byte boundary; log_alpha, beta and cu_seqlens
 *     on a 4-byte boundary (so per-token slices of the gates are accepted).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and is asynchronous: outputs are valid once the stream has
 *     reached the call. Only the status readers (gdr_read_device_status,
 *     gdr_noalloc_read_device_status) synchronise.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     returned as a negative status; nothing is written in that case.
 *   - gdr_dtype selects the storage type of q, k, v and o. Gates and states
 *     are always fp32.
 *   - Gate preconditions (not checked on the device): log_alpha finite and
 *     <= 0 (alpha = 0 is expressed as a large negative value, never -inf),
 *     beta finite. Accuracy is specified for beta in [0, 1].
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *gdr_stream_t; /* the same handle as cudaStream_t */

typedef enum {
    GDR_F32 = 0,  /* q, k, v, o in fp32 (exact fp32 arithmetic path) */
    GDR_BF16 = 1  /* q, k, v, o in bf16 (tensor-core path, fp32 accumulation) */
} gdr_dtype;

enum {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = -1,    /* null pointer, negative or inconsistent size */
    GDR_ERR_UNSUPPORTED = -2,    /* dtype, d_k, d_v or chunk outside the supported set */
    GDR_ERR_ALIGNMENT = -3,      /* a pointer is not aligned as required */
    GDR_ERR_WORKSPACE = -4,      /* workspace missing or smaller than required */
    GDR_ERR_CUDA = -5,           /* a CUDA runtime call or kernel launch failed */
    GDR_ERR_DEVICE_TIMEOUT = -6, /* a device-side wait gave up (read via gdr_read_device_status) */
    GDR_ERR_BAD_SEQLENS = -7     /* cu_seqlens not 0 ... total_tokens non-decreasing (device-checked) */
};

/*
 * Human-readable name of a status code. The returned string is static.
 */
const char *gdr_status_string(int status);

/*
 * Bytes of device workspace gdr_chunk_fwd needs for these sizes (a host-only
 * computation; no CUDA call). Returns 0 when the sizes are unsupported or
 * invalid, in which case gdr_chunk_fwd rejects them too.
 */
size_t gdr_chunk_fwd_workspace_size(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                    int d_v, int chunk, int dtype);

/*
 * Chunked prefill over packed sequences.
 *
 * What it computes: for every sequence n and head h, the recurrence above run
 * over the sequence's tokens from the initial state S0[n, h] (zero if S0 is
 * NULL); o receives every o_t and S_final[n, h] the state after the last
 * token. The result is the token recurrence's, computed chunk by chunk
 * ("Attention as Matrix Algebra: From Softmax to the Delta Rule", section 8
 * "Training the delta rule in chunks": a unit lower-triangular solve turns
 * values into pseudo-values, then chunked linear attention carries the state
 * across chunks), extended with the decay gate: inside a chunk
 * g_t = sum of log_alpha up to t, (I + L) with L_ti = beta_t exp(g_t - g_i)
 * k_t.k_i (i < t), and the state between chunks decays by exp(g_last).
 * Chunks never straddle sequences; a sequence's last chunk may be partial.
 *
 * Arguments
 *   q, k          [total_tokens, H, d_k]  dtype
 *   v             [total_tokens, H, d_v]  dtype
 *   log_alpha     [total_tokens, H]       fp32, log of the decay gate (<= 0)
 *   beta          [total_tokens, H]       fp32, write strength
 *   S0            [num_seqs, H, d_k, d_v] fp32 (d_v contiguous), or NULL for zero
 *   cu_seqlens    [num_seqs + 1] int32 token offsets, cu_seqlens[0] = 0,
 *                 non-decreasing, cu_seqlens[num_seqs] = total_tokens; or NULL for
 *                 num_seqs sequences of total_tokens / num_seqs tokens each
 *                 (then num_seqs must divide total_tokens). A sequence of zero
 *                 tokens is allowed: its S_final equals its S0. cu_seqlens lives in
 *                 device memory, so it is validated on the device: a violation sets
 *                 GDR_ERR_BAD_SEQLENS in the workspace status word (see
 *                 gdr_read_device_status) and the contents of o and S_final are then
 *                 unspecified; no access leaves the buffers described here.
 *   num_seqs, total_tokens, H   sizes (num_seqs >= 1, total_tokens >= 0, H >= 1)
 *   d_k           64 or 128
 *   d_v           a multiple of 32 in [32, 256] (bf16 tensor-core path: 128 or 256
 *                 with d_k = 128; other shapes use the exact fp32-arithmetic path)
 *   chunk         64
 *   dtype         gdr_dtype of q, k, v and o
 *   o             [total_tokens, H, d_v]  dtype (written)
 *   S_final       [num_seqs, H, d_k, d_v] fp32 (written). It may be the same buffer
 *                 as S0 (in-place update); any other overlap is not allowed.
 *   workspace     device scratch of at least gdr_chunk_fwd_workspace_size() bytes,
 *                 16-byte aligned; its first bytes hold the device status word.
 *                 Calls that share a workspace must be ordered on one stream.
 *   stream        stream to enqueue on
 * Returns GDR_OK or a negative status from the list above.
 *
 * Schedules. On the bf16 tensor-core path the per-chunk solve and the
 * sequential chain over the chunks run in one of three ways, chosen from the
 * sizes and the device's SM count:
 *   - fused (sequences of equal length, cu_seqlens NULL, when the chains leave
 *     enough SMs free): one cooperative kernel launch on `stream` whose CTAs
 *     share the work; it needs the whole GPU at one CTA per SM.
 *   - phased: the chunks are split into phases and the solve of the next phase
 *     runs on a second stream of the library's own (one per host thread and
 *     device, created on first use) while the chain of the current phase runs
 *     on `stream`. That stream forks from `stream` and joins back into it inside
 *     the call, so the call behaves as one operation on `stream`, including
 *     under stream capture. A call made while `stream` is being captured, before
 *     the calling thread has made an uncaptured call on that device, runs as a
 *     single phase on `stream` alone.
 *   - segmented (few long chains: at most 38 sequence-head-128-column chains
 *     over sequences of 64 chunks or more on average, when the estimated time
 *     beats the others): every sequence is cut into n segments; a first chain
 *     launch summarises every segment but the last as an affine map of its
 *     entering state, a scan chains the segments' start states in fp32, and a
 *     second chain launch runs every segment from its start state. All on
 *     `stream`, no side stream.
 * The environment variable GDR_PREFILL_PHASES (1 to 8), read at each call,
 * forces the phased schedule with that many phases, and GDR_PREFILL_SEGMENTS
 * (2 to 8) the segmented schedule with that many segments where the workspace
 * holds it. The fused and phased schedules give the same bits: the state passes
 * between phases in fp32, exactly as between chunks, and they perform the same
 * arithmetic. The segmented schedule rounds differently (the summaries and the
 * scan), within the same tolerance.
 */
int gdr_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *S0, const int32_t *cu_seqlens,
                  int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v, int chunk,
                  int dtype, void *o, float *S_final, void *workspace, size_t workspace_bytes,
                  gdr_stream_t stream);

/*
 * One decode step: one new token for each of N sequences, the state updated in
 * place. Per (n, h) it reads S once and writes it once, fusing the decay, the
 * read vhat = alpha S^T k, the delta write S <- alpha S + k u^T with
 * u = beta (v - vhat), and the output o = S_new^T q
 * ("Attention as Matrix Algebra", section 9: a generation step reads about
 * d_k d_v numbers; "Linear attention" (arsalanzafar.ai), Eqs. (1)-(4)).
 *
 * Arguments
 *   q, k        [N, H, d_k]  dtype
 *   v           [N, H, d_v]  dtype
 *   log_alpha   [N, H] fp32;  beta [N, H] fp32
 *   S           [N, H, d_k, d_v] fp32, read and overwritten with the new state
 *   o           [N, H, d_v]  dtype (written); must not overlap S
 *   N >= 0, H >= 1, d_k in {64, 128}, d_v in {64, 128, 256}
 * Returns GDR_OK or a negative status. N = 0 enqueues nothing.
 */
int gdr_decode_step(const void *q, const void *k, const void *v, const float *log_alpha,
                    const float *beta, float *S, void *o, int64_t N, int H, int d_k, int d_v,
                    int dtype, gdr_stream_t stream);

/*
 * Variants of the recurrence, chosen through gdr_options by the _ex entry
 * points below.
 *
 *   GDR_RULE_DELTA      the gated delta rule above (the default):
 *                         S_t = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T.
 *                       With log_alpha = 0 it is the ungated delta rule.
 *   GDR_RULE_ADDITIVE   the decayed additive write (gated linear attention with a write
 *                       strength):  S_t = alpha_t S_{t-1} + beta_t k_t v_t^T.
 *                       This is the decay-gate form of "From KV Cache to a State
 *                       Matrix" (section "Why DeltaNet may forget too slowly") together
 *                       with the gradient step of size beta on the dot-product loss
 *                       ("From attention weights to a state matrix", "Associating keys
 *                       and values"). The chunk form then needs no triangular solve:
 *                       the transform T is diag(beta) and the state does not enter the
 *                       pseudo-values. With log_alpha = 0 and beta = 1 it is plain
 *                       linear attention, S_t = S_{t-1} + k_t v_t^T.
 * In both, o_t = S_t^T q_t, read after the update.
 */
enum { GDR_RULE_DELTA = 0, GDR_RULE_ADDITIVE = 1 };

/*
 * Options of the _ex entry points. A null pointer means all defaults.
 *   rule             GDR_RULE_DELTA or GDR_RULE_ADDITIVE (else GDR_ERR_UNSUPPORTED)
 *   out_gate         the layer's output step, applied to o before it is stored
 *                    ("Linear attention" (arsalanzafar.ai), "A naive PyTorch
 *                    implementation": the output normalised over the head
 *                    dimension, times SiLU of the input-dependent output gate):
 *                      o_tj <- o_tj / sqrt(mean_j' o_tj'^2 + eps) * w_j * z_tj * sigmoid(z_tj)
 *                    per token t and head, j over the head's d_v entries. out_gate
 *                    holds z, laid out like o ([tokens, H, d_v] for gdr_chunk_fwd_ex,
 *                    [N, H, d_v] for gdr_decode_step_ex), in o's dtype, 16-byte
 *                    aligned. Null: no output step (then the two fields below must
 *                    be null and zero). The state is not affected.
 *   out_norm_weight  w: [d_v] fp32, 16-byte aligned; null means all ones.
 *   out_norm_eps     eps >= 0 (finite); 0 means 1e-6.
 *   prologue         GDR_PROLOGUE_NONE (q, k, log_alpha and beta are used as given)
 *                    or GDR_PROLOGUE_LAYER: the layer's steps before the recurrence
 *                    ("Linear attention", "A naive PyTorch implementation") run
 *                    inside the kernels. q and k are then the raw projections and
 *                    each token's head vector is scaled to unit length,
 *                    x / max(|x|, 1e-12); the log_alpha argument holds the forget
 *                    gate's pre-activation a and beta holds the write gate's b, and
 *                      log alpha = -A_h softplus(a),   beta = sigmoid(b).
 *   gate_A           A: [H] fp32 per-head rate (A_h > 0; the layer keeps log A and
 *                    exponentiates it), 4-byte aligned; null means all ones. Only
 *                    with GDR_PROLOGUE_LAYER.
 *   decay            GDR_DECAY_HEAD (default): one forget rate per token and head,
 *                    log_alpha [tokens, H] ([N, H] for decode). GDR_DECAY_CHANNEL: one
 *                    rate per token, head and key channel, log_alpha [tokens, H, d_k]
 *                    ([N, H, d_k] for decode), fp32, 4-byte aligned: row c of the
 *                    state decays by its own alpha_t[c], S'_t = diag(alpha_t) S_{t-1},
 *                    the other steps unchanged ("Attention as Matrix Algebra: From
 *                    Softmax to the Delta Rule", section 10 "Where this goes next":
 *                    Kimi Delta Attention gives each feature channel its own rate).
 *                    With GDR_PROLOGUE_LAYER the pre-activation a has that shape too.
 *                    Prefill with per-channel rates takes the per-channel tensor-core
 *                    path (GDR_PATH_CHANNEL_TENSOR) for bf16 with d_k = d_v = 128,
 *                    else the exact fp32 path (GDR_PATH_EXACT);
 *                    gdr_chunk_fwd_workspace_size_ex sizes the workspace of either,
 *                    and gdr_chunk_fwd_path_ex says which one a call takes. Other
 *                    values: GDR_ERR_INVALID_ARG.
 */
enum { GDR_PROLOGUE_NONE = 0, GDR_PROLOGUE_LAYER = 1 };
enum { GDR_DECAY_HEAD = 0, GDR_DECAY_CHANNEL = 1 };
typedef struct gdr_options {
    int rule;
    float out_norm_eps;
    const void *out_gate;
    const float *out_norm_weight;
    int prologue;
    int decay;
    const float *gate_A;
} gdr_options;

/*
 * Workspace bytes of a gdr_chunk_fwd_ex call with these sizes and options
 * (the options decide the kernel path: per-channel rates take the exact one);
 * 0 for unsupported sizes or options. With a null options pointer it equals
 * gdr_chunk_fwd_workspace_size.
 */
size_t gdr_chunk_fwd_workspace_size_ex(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                       int d_v, int chunk, int dtype, const gdr_options *options);

/*
 * gdr_chunk_fwd with options: the same arguments, layouts, ownership and
 * errors, for the rule and output step in *options. gdr_chunk_fwd is this call
 * with a null options pointer. out_gate must not overlap o (it may not be o).
 */
int gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     const float *beta, const float *S0, const int32_t *cu_seqlens,
                     int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v, int chunk,
                     int dtype, void *o, float *S_final, void *workspace, size_t workspace_bytes,
                     const gdr_options *options, gdr_stream_t stream);

/*
 * gdr_decode_step with options, as gdr_chunk_fwd_ex. For GDR_RULE_ADDITIVE
 * the step is S <- alpha S + beta k v^T, o = S_new^T q (one read and one
 * write of S, as for the delta rule). The output step, if any, is fused into
 * the same kernel.
 */
int gdr_decode_step_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, float *S, void *o, int64_t N, int H, int d_k, int d_v,
                       int dtype, const gdr_options *options, gdr_stream_t stream);

/*
 * gdr_chunk_fwd for callers that cannot allocate device memory.
 *
 * (The pages have no counterpart: this is a deployment convenience, not part
 * of the method.) Some callers cannot hand gdr_chunk_fwd a workspace: a
 * plugin loaded into a runtime that owns the device allocator and offers its
 * plugins no way to allocate, or a serving loop whose memory policy forbids
 * device allocations after start-up. This entry point takes the same
 * arguments as gdr_chunk_fwd minus the workspace and computes the same
 * result, using as scratch a static array inside the library of
 * GDR_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library
 * holds until the process exits. It allocates nothing.
 *
 *   - Sizes whose workspace (gdr_chunk_fwd_workspace_size) exceeds
 *     GDR_NOALLOC_SCRATCH_BYTES are rejected with GDR_ERR_WORKSPACE before
 *     anything is enqueued; other argument errors are those of gdr_chunk_fwd.
 *   - The device current on the calling thread must be the one the pointers
 *     and the stream belong to. Every call looks up the array's device
 *     address there (cudaGetSymbolAddress, which allocates nothing); the
 *     first call on a device also loads the library's module on it, so make
 *     that first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing needs clearing: each call writes all the scratch it reads).
 *     Calls that overlap on the GPU race on it: order them on one stream.
 *   - The device-side checks (a rejected cu_seqlens: GDR_ERR_BAD_SEQLENS; a
 *     bounded wait that gave up: GDR_ERR_DEVICE_TIMEOUT) leave their status
 *     in the first word of the array, and then o and S_final are not
 *     written. gdr_noalloc_read_device_status reads it.
 */
#define GDR_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
int gdr_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *S0, const int32_t *cu_seqlens,
                          int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v,
                          int chunk, int dtype, void *o, float *S_final, gdr_stream_t stream);

/*
 * The device status word that the last gdr_chunk_fwd_noalloc call on the
 * current device left in the library's scratch array (GDR_OK,
 * GDR_ERR_BAD_SEQLENS or GDR_ERR_DEVICE_TIMEOUT), written to *status (a HOST
 * pointer). Like gdr_read_device_status it synchronises `stream` first, so it
 * must not be called inside stream capture; it allocates nothing. Returns
 * GDR_OK if the status was read, GDR_ERR_INVALID_ARG for a null status
 * pointer, GDR_ERR_CUDA if the device cannot be read.
 */
int gdr_noalloc_read_device_status(int *status, gdr_stream_t stream);

/*
 * Which kernel path gdr_chunk_fwd takes for these sizes, for diagnostics and
 * benchmarks (host-only, no CUDA call): GDR_PATH_EXACT (plain fp32 arithmetic:
 * a planning kernel, a per-chunk kernel and a per-sequence chain kernel) or
 * GDR_PATH_TENSOR (bf16 tensor cores: a chunk-parallel solve and per-sequence
 * chains, as one cooperative kernel or as separate kernels after a planning
 * kernel; see gdr_chunk_fwd_schedule).
 * Returns a negative status for unsupported sizes.
 */
enum { GDR_PATH_EXACT = 0, GDR_PATH_TENSOR = 1, GDR_PATH_CHANNEL_TENSOR = 2 };
int gdr_chunk_fwd_path(int d_k, int d_v, int dtype);

/*
 * The kernel path of a gdr_chunk_fwd_ex call with these sizes and options (null:
 * the defaults, the same answer as gdr_chunk_fwd_path). With per-channel rates
 * (decay = GDR_DECAY_CHANNEL) it is GDR_PATH_CHANNEL_TENSOR (bf16 tensor cores:
 * a planning kernel, a chunk-parallel kernel that builds every chunk's operands
 * with per-channel decay folded in, and a per-sequence chain kernel) for bf16
 * with d_k = d_v = 128, else GDR_PATH_EXACT. Host-only, no
 * CUDA call. Returns a negative status for unsupported sizes or options, as
 * gdr_chunk_fwd_ex would.
 */
int gdr_chunk_fwd_path_ex(int d_k, int d_v, int dtype, const gdr_options *options);

/*
 * Number of kernels one uncaptured gdr_chunk_fwd call with these sizes
 * launches on the current device (the schedule depends on the device's SM
 * count), for diagnostics and benchmarks. varlen: nonzero when the call passes
 * cu_seqlens. Returns a negative status for unsupported or invalid sizes, or
 * GDR_ERR_CUDA if the device cannot be read.
 */
int gdr_chunk_fwd_kernel_launches(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                  int d_v, int chunk, int dtype, int varlen);

/*
 * Schedule of an uncaptured gdr_chunk_fwd call with these sizes on the current
 * device, for diagnostics and benchmarks: 0 for the fused schedule of the
 * tensor-core path (one cooperative kernel that runs the chains beside the solve;
 * over equal lengths it is the call's only kernel, its plan being closed form;
 * with varlen a planning kernel runs first, the solve kernel and the chain kernel
 * of one phase follow, and the planning kernel, which sees the lengths, hands the
 * call to either the cooperative kernel or that pair, the other returning at
 * once); 1 .. 8, the number of phases of the phased
 * schedule (the exact path is one phase); or GDR_SCHEDULE_SEGMENTED + n for
 * the segmented schedule of few long chains, each sequence cut into n (2 .. 8)
 * segments whose state transitions are summarised and chained by a scan
 * (planning kernel, solve, summary chain, scan, chain). varlen as above.
 * Returns a negative status for unsupported or invalid sizes, or GDR_ERR_CUDA
 * if the device cannot be read.
 */
enum { GDR_SCHEDULE_SEGMENTED = 16 };

/*
 * The schedule gdr_chunk_fwd_schedule would report on a device with `sms` SMs
 * (cooperative: nonzero if that device can run the fused schedule's cooperative
 * launch), for tests and capacity planning. It makes no CUDA call. The
 * environment variables that force a schedule apply here too. Returns a
 * negative status for unsupported or invalid sizes, or GDR_ERR_INVALID_ARG if
 * sms < 1. (The phased schedule also needs a side stream, which a real call may
 * not get under stream capture; see gdr_chunk_fwd.)
 */
int gdr_chunk_fwd_schedule_model(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                 int d_v, int chunk, int dtype, int varlen, int sms,
                                 int cooperative);
int gdr_chunk_fwd_schedule(int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v,
                           int chunk, int dtype, int varlen);

/*
 * Reads the device status word that the last gdr_chunk_fwd call on this
 * workspace left (GDR_OK, GDR_ERR_BAD_SEQLENS or GDR_ERR_DEVICE_TIMEOUT) into
 * *status (a HOST pointer). It synchronises `stream` first, so it must not be
 * called inside stream capture. Returns GDR_OK if the status was read.
 */
int gdr_read_device_status(const void *workspace, int *status, gdr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
