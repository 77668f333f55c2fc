// internal.h -- declarations shared by the translation units of libgdr (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdr.h"

namespace gdr {

constexpr int kChunk = 64;  // tokens per chunk (the only chunk size the kernels support)
constexpr int kMaxPhases = 8;  // most phases a tensor-core prefill is split into
// Schedules of the tensor-core path: 0 fused, 1 .. kMaxPhases phased, kSegmentedBase + n
// segmented into n segments per sequence.
constexpr int kSegmentedBase = GDR_SCHEDULE_SEGMENTED;
// The fused schedule over packed sequences: at most this many sequences (the planning
// kernel keeps their chunk counts in shared memory), and the control word that counts
// the solve's claims.
constexpr int kMaxClaimSeqs = 128;
constexpr int kClaimWord = 32;
// For packed sequences the host launches the fused kernel and, after it, the phased
// schedule's two kernels (one phase); the planning kernel sets ctl[kPairWord] to 1 when
// the pair is to do the work (the fused kernel then returns at once), else to 0 (the
// pair then returns at once).
constexpr int kPairWord = 33;
// phases of the chunk plan a schedule needs (a segment is a phase)
inline int plan_phases(int schedule) {
    return schedule == 0 ? 1 : (schedule > kSegmentedBase ? schedule - kSegmentedBase : schedule);
}
// Few chains (sequences x heads x 128-column value slices) over long sequences: the
// workspace then holds the segmented schedule's state sets.
inline bool tc_segmentable(int64_t num_seqs, int64_t total_tokens, int H, int dv) {
    return num_seqs > 0 && num_seqs * H * (dv / 128) <= 38 && total_tokens >= num_seqs * 64 * kChunk;
}

// Everything gdr_chunk_fwd receives, after host validation.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;
    int64_t num_seqs, total_tokens;
    int H, dk, dv, chunk, dtype;
    int rule;  // GDR_RULE_DELTA or GDR_RULE_ADDITIVE
    // the output step (null out_gate: none): o <- rmsnorm(o) * w * silu(z)
    const void *out_gate;
    const float *out_norm_weight;
    float out_norm_eps;
    // the layer's prologue (unit-length q and k, gates from pre-activations)
    int prologue;
    const float *gate_A;
    int decay;  // GDR_DECAY_HEAD, or GDR_DECAY_CHANNEL: log_alpha [tokens, H, d_k]
    void *o;
    float *S_final;
    char *ws;
    cudaStream_t stream;
};

// Byte offsets of the workspace regions. The control words come first:
//   int32 ctl[0] = device status (GDR_OK / GDR_ERR_*), ctl[1] = number of chunks,
//   ctl[2 + f] = first chunk of phase f (f = 0 .. phases).
// Chunks are numbered phase-major (see plan_kernel); a single phase is the plain
// sequence-by-sequence order.
struct WsLayout {
    int64_t max_chunks;   // upper bound on sum over sequences of ceil(len / chunk)
    size_t ctl;           // int32[64]
    size_t plan;          // int4[max_chunks]: (sequence, first token, tokens, chunk index)
    size_t seq_chunk;     // int32[kMaxPhases][num_seqs + 1]: first chunk of each sequence per phase
    size_t W, U, A, g;    // fp32 per-chunk intermediates of the exact path (g: gamma, kdec)
    size_t gc;            // exact path, per-channel rates: fp32 [chunk * H][C][d_k] cumulative
                          // log decay per key channel
    size_t T;             // tensor-core path: bf16 [max_chunks * H][2][64][64] T' and A^T per unit
    size_t G;             // tensor-core path: fp32 [max_chunks * H][256] decay factors per unit
    size_t S;             // tensor-core path: fp32 [num_seqs][H][dk][dv] state between phases
    size_t F;             // tensor-core path: int32 [max_chunks * H] unit-solved flags
                          // (fused schedule)
    size_t order;         // tensor-core path: int4 [max_chunks] the claim order of the fused
                          // schedule over packed sequences: (chunk, first token, tokens,
                          // sequence) per claim row
    size_t trig;          // tensor-core path: int32 [num_seqs] the claim count at which the
                          // chain CTAs of each sequence stop solving and start their chains
    size_t seg;           // tensor-core path, few long chains: the segmented schedule's
                          // fp32 state sets, [NH][d_k][d_v] each: (kMaxPhases - 1) each
                          // of P, R and discard, kMaxPhases of start; 0 bytes otherwise
    bool segmentable;
    size_t QW, KT, UT;    // tensor-core path with per-channel rates: per unit, bf16
                          // [64][256] e^g . Q | -W, [64][128] e^{g_C - g} . K, [128][64] Utilde^T
                          // (T holds A^T, G exp(g_C) per channel)
    size_t total;
    bool tensor_path;     // bf16 tensor-core kernels with one rate per head
    bool channel_tc;      // bf16 tensor-core kernels with one rate per key channel
};

bool use_tensor_path(int dk, int dv, int dtype);
// Per-channel rates on the tensor cores: bf16, d_k = d_v = 128, no layer prologue (the other
// cases take the exact path).
bool use_channel_tc(int dk, int dv, int dtype, int prologue);
WsLayout ws_layout(int64_t num_seqs, int64_t total_tokens, int H, int dk, int dv, int dtype,
                   int decay = GDR_DECAY_HEAD, int prologue = GDR_PROLOGUE_NONE);

// Launchers (return GDR_OK or GDR_ERR_CUDA).
// The planning kernel for a schedule (the fused schedule, 0, plans one phase and clears
// the unit flags; the segmented one plans a phase per segment).
int launch_plan(const PrefillArgs &a, const WsLayout &L, int phases);
// The SM count of the current device (0 if it cannot be read), cached.
int current_device_sms();
int launch_prefill_exact(const PrefillArgs &a, const WsLayout &L);
int launch_prefill_tc(const PrefillArgs &a, const WsLayout &L, int phases);
// The tensor-core path with one forget rate per key channel: the per-channel chunk kernel
// over every unit, then the chains (one phase).
int launch_prefill_channel_tc(const PrefillArgs &a, const WsLayout &L);

// The schedule of a tensor-core prefill: 0 for the fused cooperative launch,
// 1 .. kMaxPhases phases of the two-kernel schedule, or kSegmentedBase + n for n
// segments per sequence.
int tc_schedule_for(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms, bool varlen,
                    bool cooperative);
// The schedule a call with these arguments runs on the current device (falls back to
// one phase when the second stream of the phased schedule cannot be had).
int tc_schedule(const PrefillArgs &a);
// The schedule an uncaptured call with these sizes runs on the current device (or -1).
int tc_schedule_query(int64_t num_seqs, int64_t total_tokens, int H, int dv, bool varlen);
int launch_decode(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, float *S, void *o, int64_t N, int H, int dk, int dv,
                  int dtype, int rule, const void *out_gate, const float *out_norm_weight,
                  float out_norm_eps, int prologue, const float *gate_A, int decay,
                  cudaStream_t stream);
// The output step over `rows` rows of d_v entries of o, in place (prefill paths that do
// not fuse it).
int launch_out_norm_gate(void *o, const void *z, const float *w, float eps, int64_t rows, int dv,
                         int dtype, cudaStream_t stream);

// The layer's gate activations (the prologue): log alpha = -A softplus(a), beta = sigmoid(b).
__device__ __forceinline__ float prologue_log_alpha(float a, float A) {
    const float sp = a > 20.f ? a : log1pf(expf(a));  // softplus, exact to fp32 beyond 20
    return -A * sp;
}
__device__ __forceinline__ float prologue_beta(float b) { return 1.f / (1.f + expf(-b)); }
// 1 / max(|x|, 1e-12) from the sum of squares
__device__ __forceinline__ float prologue_inv_norm(float ss) { return 1.f / fmaxf(sqrtf(ss), 1e-12f); }

// Type helpers for kernels.
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA; }

}  // namespace gdr
