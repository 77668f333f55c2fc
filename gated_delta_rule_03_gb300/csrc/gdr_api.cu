// gdr_api.cu -- the C ABI of libgdr: argument validation, workspace layout, dispatch.
//
// Every check that can be made without touching the device is made here, before
// anything is enqueued; a rejected call writes nothing. Checks that need device
// memory (cu_seqlens) are made by the kernels, which report through the status
// word at the start of the workspace.
#include <string.h>

#include "internal.h"

namespace gdr {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool use_tensor_path(int dk, int dv, int dtype) {
    return dtype == GDR_BF16 && dk == 128 && (dv == 128 || dv == 256);
}

bool use_channel_tc(int dk, int dv, int dtype, int prologue) {
    (void)prologue;  // the operands kernel folds the prologue in
    return dtype == GDR_BF16 && dk == 128 && dv == 128;
}

WsLayout ws_layout(int64_t num_seqs, int64_t total_tokens, int H, int dk, int dv, int dtype,
                   int decay, int prologue) {
    WsLayout L;
    memset(&L, 0, sizeof(L));
    L.tensor_path = decay == GDR_DECAY_HEAD && use_tensor_path(dk, dv, dtype);
    L.channel_tc = decay == GDR_DECAY_CHANNEL && use_channel_tc(dk, dv, dtype, prologue);
    L.max_chunks = total_tokens / kChunk + num_seqs;
    size_t off = 0;
    L.ctl = off;
    off += 256;
    L.plan = off;
    off = align_up(off + sizeof(int4) * (size_t)L.max_chunks, 256);
    L.seq_chunk = off;
    off = align_up(off + sizeof(int32_t) * (size_t)kMaxPhases * (size_t)(num_seqs + 1), 256);
    if (L.channel_tc) {
        const size_t units = (size_t)L.max_chunks * (size_t)H;
        L.T = off;  // A^T in the second of two 64x64 bf16 matrices per unit
        off = align_up(off + units * 2 * kChunk * kChunk * 2, 256);
        L.G = off;  // 384 floats per unit: exp(g_C) per channel first
        off = align_up(off + units * 384 * sizeof(float), 256);
        L.QW = off;
        off = align_up(off + units * kChunk * 256 * 2, 256);
        L.KT = off;
        off = align_up(off + units * kChunk * 128 * 2, 256);
        L.UT = off;
        off = align_up(off + units * 128 * kChunk * 2, 256);
    } else if (!L.tensor_path) {
        const size_t per = (size_t)L.max_chunks * (size_t)H * kChunk;
        L.W = off;
        off = align_up(off + sizeof(float) * per * dk, 256);
        L.U = off;
        off = align_up(off + sizeof(float) * per * dv, 256);
        L.A = off;
        off = align_up(off + sizeof(float) * per * kChunk, 256);
        L.g = off;  // gamma, kdec, and the prologue's 1/|q|, 1/|k| per chunk token
        off = align_up(off + sizeof(float) * per * 4, 256);
        L.gc = off;  // per-channel rates: the cumulative log decay per chunk token and channel
        if (decay == GDR_DECAY_CHANNEL) off = align_up(off + sizeof(float) * per * dk, 256);
    } else {
        L.T = off;  // two 64x64 bf16 matrices per (chunk, head)
        off = align_up(off + (size_t)L.max_chunks * (size_t)H * 2 * kChunk * kChunk * 2, 256);
        L.G = off;  // 384 floats per (chunk, head): decay factors, the prologue's norms
        off = align_up(off + (size_t)L.max_chunks * (size_t)H * 384 * sizeof(float), 256);
        L.S = off;  // the state handed from one phase to the next
        off = align_up(off + (size_t)num_seqs * (size_t)H * dk * dv * sizeof(float), 256);
        L.F = off;  // one flag per (chunk, head) unit (fused schedule)
        off = align_up(off + (size_t)L.max_chunks * (size_t)H * sizeof(int32_t), 256);
        L.order = off;  // the claim order of the fused schedule over packed sequences
        off = align_up(off + (size_t)L.max_chunks * sizeof(int4), 256);
        L.trig = off;
        off = align_up(off + (size_t)num_seqs * sizeof(int32_t), 256);
        L.segmentable = tc_segmentable(num_seqs, total_tokens, H, dv);
        L.seg = off;  // the segmented schedule's state sets
        if (L.segmentable)
            off = align_up(off + (size_t)(4 * kMaxPhases - 3) * (size_t)num_seqs * H * dk * dv *
                                     sizeof(float), 256);
    }
    L.total = off;
    return L;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

static int check_prefill_sizes(int64_t num_seqs, int64_t total_tokens, int H, int dk, int dv,
                               int chunk, int dtype) {
    if (num_seqs < 1 || total_tokens < 0 || H < 1) return GDR_ERR_INVALID_ARG;
    if (total_tokens > INT32_MAX || num_seqs > INT32_MAX / 2) return GDR_ERR_INVALID_ARG;
    if (dtype != GDR_F32 && dtype != GDR_BF16) return GDR_ERR_UNSUPPORTED;
    if (dk != 64 && dk != 128) return GDR_ERR_UNSUPPORTED;
    if (dv < 32 || dv > 256 || dv % 32 != 0) return GDR_ERR_UNSUPPORTED;
    if (chunk != kChunk) return GDR_ERR_UNSUPPORTED;
    // grid limits: (num_seqs * H) blocks in x
    if ((int64_t)H * num_seqs > INT32_MAX / 4) return GDR_ERR_INVALID_ARG;
    if ((int64_t)H * (total_tokens / kChunk + num_seqs) > INT32_MAX / 4) return GDR_ERR_INVALID_ARG;
    return GDR_OK;
}

// The checked contents of an options block (defaults for a null pointer).
struct Opts {
    int rule = GDR_RULE_DELTA;
    const void *out_gate = nullptr;
    const float *out_norm_weight = nullptr;
    float out_norm_eps = 0.f;
    int prologue = GDR_PROLOGUE_NONE;
    const float *gate_A = nullptr;
    int decay = GDR_DECAY_HEAD;
};

// Known rule, prologue and decay; the output-step fields need a gate; pointers aligned.
static int check_options(const gdr_options *opt, Opts *o) {
    *o = Opts();
    if (!opt) return GDR_OK;
    if (opt->decay != GDR_DECAY_HEAD && opt->decay != GDR_DECAY_CHANNEL) return GDR_ERR_INVALID_ARG;
    o->decay = opt->decay;
    if (opt->rule != GDR_RULE_DELTA && opt->rule != GDR_RULE_ADDITIVE) return GDR_ERR_UNSUPPORTED;
    o->rule = opt->rule;
    if (opt->prologue != GDR_PROLOGUE_NONE && opt->prologue != GDR_PROLOGUE_LAYER)
        return GDR_ERR_UNSUPPORTED;
    if (opt->gate_A && opt->prologue != GDR_PROLOGUE_LAYER) return GDR_ERR_INVALID_ARG;
    if ((uintptr_t)opt->gate_A & 3u) return GDR_ERR_ALIGNMENT;
    o->prologue = opt->prologue;
    o->gate_A = opt->gate_A;
    if (!opt->out_gate) {
        if (opt->out_norm_weight || opt->out_norm_eps != 0.f) return GDR_ERR_INVALID_ARG;
        return GDR_OK;
    }
    const float eps = opt->out_norm_eps;
    if (!(eps >= 0.f && eps < 3.0e38f)) return GDR_ERR_INVALID_ARG;  // also rejects NaN
    if (((uintptr_t)opt->out_gate & 15u) || ((uintptr_t)opt->out_norm_weight & 15u))
        return GDR_ERR_ALIGNMENT;
    o->out_gate = opt->out_gate;
    o->out_norm_weight = opt->out_norm_weight;
    o->out_norm_eps = eps == 0.f ? 1e-6f : eps;
    return GDR_OK;
}

static bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + bn && pb < pa + an;
}

}  // namespace gdr

using namespace gdr;

extern "C" {

const char *gdr_status_string(int status) {
    switch (status) {
        case GDR_OK: return "GDR_OK";
        case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: null pointer or invalid size";
        case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: dtype, d_k, d_v or chunk not supported";
        case GDR_ERR_ALIGNMENT: return "GDR_ERR_ALIGNMENT: pointer not aligned as required";
        case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace missing or too small";
        case GDR_ERR_CUDA: return "GDR_ERR_CUDA: CUDA call or kernel launch failed";
        case GDR_ERR_DEVICE_TIMEOUT: return "GDR_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
        case GDR_ERR_BAD_SEQLENS: return "GDR_ERR_BAD_SEQLENS: cu_seqlens not 0..total_tokens non-decreasing";
        default: return "GDR_ERR_UNKNOWN";
    }
}

size_t gdr_chunk_fwd_workspace_size(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                    int d_v, int chunk, int dtype) {
    if (check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype) != GDR_OK) return 0;
    return ws_layout(num_seqs, total_tokens, H, d_k, d_v, dtype).total;
}

size_t gdr_chunk_fwd_workspace_size_ex(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                       int d_v, int chunk, int dtype, const gdr_options *options) {
    Opts op;
    if (check_options(options, &op) != GDR_OK) return 0;
    if (check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype) != GDR_OK) return 0;
    return ws_layout(num_seqs, total_tokens, H, d_k, d_v, dtype, op.decay, op.prologue).total;
}

int gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     const float *beta, const float *S0, const int32_t *cu_seqlens,
                     int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v, int chunk,
                     int dtype, void *o, float *S_final, void *workspace, size_t workspace_bytes,
                     const gdr_options *options, gdr_stream_t stream) {
    Opts op;
    int st = check_options(options, &op);
    if (st != GDR_OK) return st;
    st = check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype);
    if (st != GDR_OK) return st;
    if (!cu_seqlens && total_tokens % num_seqs != 0) return GDR_ERR_INVALID_ARG;
    if (!S_final || !workspace) return workspace ? GDR_ERR_INVALID_ARG : GDR_ERR_WORKSPACE;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !o))
        return GDR_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, S0, o, S_final, workspace};
    for (const void *p : ptrs16)
        if (p && !aligned16(p)) return GDR_ERR_ALIGNMENT;
    const void *ptrs4[] = {log_alpha, beta, cu_seqlens};
    for (const void *p : ptrs4)
        if (p && !aligned4(p)) return GDR_ERR_ALIGNMENT;
    const WsLayout L = ws_layout(num_seqs, total_tokens, H, d_k, d_v, dtype, op.decay, op.prologue);
    if (workspace_bytes < L.total) return GDR_ERR_WORKSPACE;
    const size_t esz = dtype == GDR_F32 ? 4 : 2;
    const size_t o_bytes = (size_t)total_tokens * H * d_v * esz;
    const size_t s_bytes = (size_t)num_seqs * H * d_k * d_v * sizeof(float);
    if (S0 && S0 != S_final && overlaps(S0, s_bytes, S_final, s_bytes)) return GDR_ERR_INVALID_ARG;
    if (o && overlaps(o, o_bytes, S_final, s_bytes)) return GDR_ERR_INVALID_ARG;
    if (overlaps(workspace, L.total, S_final, s_bytes)) return GDR_ERR_INVALID_ARG;
    if (o && overlaps(workspace, L.total, o, o_bytes)) return GDR_ERR_INVALID_ARG;
    if (op.out_gate && o && overlaps(op.out_gate, o_bytes, o, o_bytes)) return GDR_ERR_INVALID_ARG;

    PrefillArgs a;
    a.q = q; a.k = k; a.v = v;
    a.log_alpha = log_alpha; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = cu_seqlens;
    a.num_seqs = num_seqs; a.total_tokens = total_tokens;
    a.H = H; a.dk = d_k; a.dv = d_v; a.chunk = chunk; a.dtype = dtype;
    a.rule = op.rule;
    a.out_gate = op.out_gate;
    a.out_norm_weight = op.out_norm_weight;
    a.out_norm_eps = op.out_norm_eps;
    a.prologue = op.prologue;
    a.gate_A = op.gate_A;
    a.decay = op.decay;
    a.o = o; a.S_final = S_final;
    a.ws = (char *)workspace;
    a.stream = (cudaStream_t)stream;
    const int phases = L.tensor_path ? tc_schedule(a) : 1;
    // (the fused schedule over equal lengths plans itself: its plan is closed form)
    if (!(L.tensor_path && phases == 0 && !cu_seqlens)) {
        st = launch_plan(a, L, phases);
        if (st != GDR_OK) return st;
    }
    st = L.channel_tc ? launch_prefill_channel_tc(a, L)
                      : (L.tensor_path ? launch_prefill_tc(a, L, phases) : launch_prefill_exact(a, L));
    // the output step, where the chain did not fuse it (it does on the tensor-core paths
    // when one chain CTA holds all d_v = 128 entries of a token)
    if (st == GDR_OK && a.out_gate && !((L.tensor_path || L.channel_tc) && d_v == 128))
        st = launch_out_norm_gate(o, a.out_gate, a.out_norm_weight, a.out_norm_eps,
                                  total_tokens * H, d_v, dtype, a.stream);
    return st;
}

int gdr_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *S0, const int32_t *cu_seqlens,
                  int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v, int chunk,
                  int dtype, void *o, float *S_final, void *workspace, size_t workspace_bytes,
                  gdr_stream_t stream) {
    return gdr_chunk_fwd_ex(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H,
                            d_k, d_v, chunk, dtype, o, S_final, workspace, workspace_bytes,
                            nullptr, stream);
}

int gdr_decode_step_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, float *S, void *o, int64_t N, int H, int d_k, int d_v,
                       int dtype, const gdr_options *options, gdr_stream_t stream) {
    Opts op;
    const int st = check_options(options, &op);
    if (st != GDR_OK) return st;
    if (N < 0 || H < 1 || N > INT32_MAX || (int64_t)N * H > INT32_MAX) return GDR_ERR_INVALID_ARG;
    if (dtype != GDR_F32 && dtype != GDR_BF16) return GDR_ERR_UNSUPPORTED;
    if ((d_k != 64 && d_k != 128) || (d_v != 64 && d_v != 128 && d_v != 256))
        return GDR_ERR_UNSUPPORTED;
    if (N == 0) return GDR_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return GDR_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, S, o};
    for (const void *p : ptrs16)
        if (!aligned16(p)) return GDR_ERR_ALIGNMENT;
    if (!aligned4(log_alpha) || !aligned4(beta)) return GDR_ERR_ALIGNMENT;
    const size_t esz = dtype == GDR_F32 ? 4 : 2;
    if (overlaps(o, (size_t)N * H * d_v * esz, S, (size_t)N * H * d_k * d_v * sizeof(float)))
        return GDR_ERR_INVALID_ARG;
    if (op.out_gate && overlaps(op.out_gate, (size_t)N * H * d_v * esz, o, (size_t)N * H * d_v * esz))
        return GDR_ERR_INVALID_ARG;
    return launch_decode(q, k, v, log_alpha, beta, S, o, N, H, d_k, d_v, dtype, op.rule, op.out_gate,
                         op.out_norm_weight, op.out_norm_eps, op.prologue, op.gate_A, op.decay,
                         (cudaStream_t)stream);
}

int gdr_decode_step(const void *q, const void *k, const void *v, const float *log_alpha,
                    const float *beta, float *S, void *o, int64_t N, int H, int d_k, int d_v,
                    int dtype, gdr_stream_t stream) {
    return gdr_decode_step_ex(q, k, v, log_alpha, beta, S, o, N, H, d_k, d_v, dtype, nullptr, stream);
}

int gdr_chunk_fwd_path(int d_k, int d_v, int dtype) {
    const int st = check_prefill_sizes(1, 0, 1, d_k, d_v, kChunk, dtype);
    if (st != GDR_OK) return st;
    return use_tensor_path(d_k, d_v, dtype) ? GDR_PATH_TENSOR : GDR_PATH_EXACT;
}

int gdr_chunk_fwd_path_ex(int d_k, int d_v, int dtype, const gdr_options *options) {
    Opts op;
    int st = check_options(options, &op);
    if (st != GDR_OK) return st;
    st = check_prefill_sizes(1, 0, 1, d_k, d_v, kChunk, dtype);
    if (st != GDR_OK) return st;
    if (op.decay == GDR_DECAY_CHANNEL)
        return use_channel_tc(d_k, d_v, dtype, op.prologue) ? GDR_PATH_CHANNEL_TENSOR : GDR_PATH_EXACT;
    return use_tensor_path(d_k, d_v, dtype) ? GDR_PATH_TENSOR : GDR_PATH_EXACT;
}

int gdr_chunk_fwd_kernel_launches(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                  int d_v, int chunk, int dtype, int varlen) {
    const int st = check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype);
    if (st != GDR_OK) return st;
    if (!use_tensor_path(d_k, d_v, dtype)) return 3;  // plan, per-chunk prep, chain
    if (total_tokens == 0) return 1;  // the plan; the state copy is not a kernel of ours
    const int P = tc_schedule_query(num_seqs, total_tokens, H, d_v, varlen != 0);
    if (P < 0) return GDR_ERR_CUDA;
    // fused: the cooperative kernel alone (equal lengths: it plans itself), or for packed
    // sequences the plan, the cooperative kernel, then the solve and chain of one phase,
    // which the plan may hand the call to; P phases: plan, P solves, P chains;
    // segmented: plan, solve, summary chain, scan, chain
    return P == 0 ? (varlen ? 4 : 1) : (P > kSegmentedBase ? 5 : 1 + 2 * P);
}

int gdr_chunk_fwd_schedule(int64_t num_seqs, int64_t total_tokens, int H, int d_k, int d_v,
                           int chunk, int dtype, int varlen) {
    const int st = check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype);
    if (st != GDR_OK) return st;
    if (!use_tensor_path(d_k, d_v, dtype) || total_tokens == 0) return 1;
    const int P = tc_schedule_query(num_seqs, total_tokens, H, d_v, varlen != 0);
    return P < 0 ? GDR_ERR_CUDA : P;
}

int gdr_chunk_fwd_schedule_model(int64_t num_seqs, int64_t total_tokens, int H, int d_k,
                                 int d_v, int chunk, int dtype, int varlen, int sms,
                                 int cooperative) {
    const int st = check_prefill_sizes(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype);
    if (st != GDR_OK) return st;
    if (sms < 1) return GDR_ERR_INVALID_ARG;
    if (!use_tensor_path(d_k, d_v, dtype) || total_tokens == 0) return 1;
    return tc_schedule_for(num_seqs, total_tokens, H, d_v, sms, varlen != 0, cooperative != 0);
}

int gdr_read_device_status(const void *workspace, int *status, gdr_stream_t stream) {
    if (!workspace || !status) return GDR_ERR_INVALID_ARG;
    int32_t word = 0;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    *status = word;
    return GDR_OK;
}

}  // extern "C"
