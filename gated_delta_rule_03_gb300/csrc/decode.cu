// decode.cu -- one decode step of the gated delta rule, streaming the fp32 state once.
//
// Per (sequence, head) the state S (d_k x d_v, d_v contiguous) is read once and
// written once. With alpha = exp(log_alpha):
//   a   = S^T k,  b = S^T q                 (reads of the old state)
//   u   = beta (v - alpha a)                (the correction; vhat = alpha S^T k)
//   S'  = alpha S + k u^T                   (decay and delta write)
//   o   = S'^T q = alpha b + (k.q) u        (read-out after the update)
// which is Eqs. (1)-(4) of "Linear attention" (arsalanzafar.ai), "How it works",
// for a single token. The additive rule (S' = alpha S + beta k v^T) is the same step
// with u = beta v. With the layer's prologue, k and q are scaled to unit length in
// shared memory and the gates come from their pre-activations. With one rate per key
// channel (PC; log_alpha [N, H, d_k]) alpha becomes diag(alpha): a = S^T (alpha . k),
// b = S^T (alpha . q), o = b + (k.q) u and row r of S decays by alpha_r; each thread
// loads the rates of its own rows beside its part of the state. The layer's output step (o / rms(o) * w * silu(z), over the head's
// value entries) is applied before o is stored when a gate z is given. The kernel is
// HBM-bound: a generation step reads about
// d_k d_v numbers ("Attention as Matrix Algebra", section 9).
//
// Layout: one CTA per (n, h); d_k*d_v/64 threads, each holding 16 rows x 4
// consecutive columns (16 float4) of S in registers. A warp reads whole
// 512-byte row segments, so every load and store is a coalesced 16-byte
// access. All 16 loads of a thread are issued before any arithmetic, so a CTA
// keeps its whole 64 KB tile in flight. Loads and stores use the streaming
// cache hint: the state is far larger than L2 and is not reused in the step.
#include "internal.h"

namespace gdr {

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    static __device__ __forceinline__ void store(float *p, float4 x) {
        *reinterpret_cast<float4 *>(p) = x;
    }
    static __device__ __forceinline__ float4 load(const float *p) {
        return *reinterpret_cast<const float4 *>(p);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float4 x) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p) = packed;
    }
    static __device__ __forceinline__ float4 load(const __nv_bfloat16 *p) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// z sigmoid(z)
__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

template <typename Tin, int DK, int DV, bool PC>
__global__ void __launch_bounds__(DK * DV / 64)
decode_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const float *__restrict__ log_alpha,
                   const float *__restrict__ beta, float *__restrict__ S, Tin *__restrict__ o,
                   float read, const Tin *__restrict__ z, const float *__restrict__ w, float eps,
                   int prologue, const float *__restrict__ gate_A, int H) {
    // read = 1: the delta rule's correction u = beta (v - alpha S^T k); read = 0: the
    // additive write u = beta v
    constexpr int NT = DK * DV / 64;  // threads
    constexpr int TPR = DV / 4;       // threads per state row (one float4 each)
    constexpr int RG = NT / TPR;      // row groups (= DK / 16)
    constexpr int RPT = DK / RG;      // rows per thread (= 16)
    static_assert(RPT == 16, "each thread holds 16 rows");

    __shared__ float ks[DK], qs[DK], vs[DV], os[DV];
    __shared__ float4 red_k[RG][TPR], red_q[RG][TPR];
    __shared__ float s_kq, s_rstd, s_nk, s_nq;

    const int64_t nh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % TPR;  // column group: columns 4cg .. 4cg+3
    const int rg = tid / TPR;  // rows rg, rg + RG, ...

    float4 *Sp = reinterpret_cast<float4 *>(S + nh * (DK * DV));
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) s[m] = __ldcs(Sp + (rg + m * RG) * TPR + cg);
    // per-channel rates of this thread's rows, loaded beside the state (activated below)
    float rate[PC ? RPT : 1];
    if (PC) {
#pragma unroll
        for (int m = 0; m < RPT; ++m) rate[m] = log_alpha[nh * DK + rg + m * RG];
    }

    for (int i = tid; i < DK; i += NT) {
        ks[i] = to_f32(k[nh * DK + i]);
        qs[i] = to_f32(q[nh * DK + i]);
    }
    for (int j = tid; j < DV; j += NT) vs[j] = to_f32(v[nh * DV + j]);
    float alpha = 1.f, b;
    if (prologue) {  // the layer's gate activations from the pre-activations a, b
        if (!PC) alpha = expf(prologue_log_alpha(log_alpha[nh], gate_A ? gate_A[nh % H] : 1.f));
        b = prologue_beta(beta[nh]);
    } else {
        if (!PC) alpha = expf(log_alpha[nh]);
        b = beta[nh];
    }
    if (PC) {  // alpha stays 1; the rates go with the rows
        const float A = prologue && gate_A ? gate_A[nh % H] : 1.f;
#pragma unroll
        for (int m = 0; m < RPT; ++m) rate[m] = expf(prologue ? prologue_log_alpha(rate[m], A) : rate[m]);
    }
    const float ra = read * alpha;
    __syncthreads();
    if (prologue) {  // unit-length k and q: warp 0 sums k's squares, warp 1 q's
        if (tid < 64) {
            const float *x = tid < 32 ? ks : qs;
            float ss = 0.f;
            for (int i = tid & 31; i < DK; i += 32) ss = fmaf(x[i], x[i], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if ((tid & 31) == 0) (tid < 32 ? s_nk : s_nq) = prologue_inv_norm(ss);
        }
        __syncthreads();
        for (int i = tid; i < DK; i += NT) {
            ks[i] *= s_nk;
            qs[i] *= s_nq;
        }
        __syncthreads();
    }

    if (tid < 32) {
        float p = 0.f;
        for (int i = tid; i < DK; i += 32) p = fmaf(ks[i], qs[i], p);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (tid == 0) s_kq = p;
    }

    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const float kr = ks[rg + m * RG] * (PC ? rate[m] : 1.f), qr = qs[rg + m * RG] * (PC ? rate[m] : 1.f);
        pk.x = fmaf(s[m].x, kr, pk.x); pk.y = fmaf(s[m].y, kr, pk.y);
        pk.z = fmaf(s[m].z, kr, pk.z); pk.w = fmaf(s[m].w, kr, pk.w);
        pq.x = fmaf(s[m].x, qr, pq.x); pq.y = fmaf(s[m].y, qr, pq.y);
        pq.z = fmaf(s[m].z, qr, pq.z); pq.w = fmaf(s[m].w, qr, pq.w);
    }
    red_k[rg][cg] = pk;
    red_q[rg][cg] = pq;
    __syncthreads();

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), bq = a;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        const float4 x = red_k[r][cg], y = red_q[r][cg];
        a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        bq.x += y.x; bq.y += y.y; bq.z += y.z; bq.w += y.w;
    }
    const float kq = s_kq;
    const float4 vv = *reinterpret_cast<const float4 *>(&vs[4 * cg]);
    float4 u;
    u.x = b * (vv.x - ra * a.x);
    u.y = b * (vv.y - ra * a.y);
    u.z = b * (vv.z - ra * a.z);
    u.w = b * (vv.w - ra * a.w);
    float4 out;
    out.x = fmaf(alpha, bq.x, kq * u.x);
    out.y = fmaf(alpha, bq.y, kq * u.y);
    out.z = fmaf(alpha, bq.z, kq * u.z);
    out.w = fmaf(alpha, bq.w, kq * u.w);
    if (z) {  // the output step: o / rms(o) * w * silu(z) over the head's DV entries
        if (rg == 0) *reinterpret_cast<float4 *>(&os[4 * cg]) = out;
        __syncthreads();
        if (tid < 32) {
            float ss = 0.f;
            for (int j = tid; j < DV; j += 32) ss = fmaf(os[j], os[j], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (tid == 0) s_rstd = rsqrtf(ss * (1.f / DV) + eps);
        }
        __syncthreads();
        if (rg == 0) {
            const float r = s_rstd;
            const float4 zz = Vec4<Tin>::load(z + nh * DV + 4 * cg);
            const float4 ww = w ? *reinterpret_cast<const float4 *>(w + 4 * cg) : make_float4(1.f, 1.f, 1.f, 1.f);
            out.x *= r * ww.x * silu(zz.x);
            out.y *= r * ww.y * silu(zz.y);
            out.z *= r * ww.z * silu(zz.z);
            out.w *= r * ww.w * silu(zz.w);
        }
    }
    if (rg == 0) Vec4<Tin>::store(o + nh * DV + 4 * cg, out);
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const float kr = ks[rg + m * RG];
        const float rm = PC ? rate[m] : alpha;
        float4 x;
        x.x = fmaf(rm, s[m].x, kr * u.x);
        x.y = fmaf(rm, s[m].y, kr * u.y);
        x.z = fmaf(rm, s[m].z, kr * u.z);
        x.w = fmaf(rm, s[m].w, kr * u.w);
        __stcs(Sp + (rg + m * RG) * TPR + cg, x);
    }
}

template <typename Tin, int DK, int DV>
static int launch_decode_t(const void *q, const void *k, const void *v, const float *la,
                           const float *beta, float *S, void *o, int64_t NH, float read,
                           const void *z, const float *w, float eps, int prologue,
                           const float *gate_A, int H, bool per_channel, cudaStream_t stream) {
    if (per_channel)
        decode_step_kernel<Tin, DK, DV, true><<<(unsigned)NH, DK * DV / 64, 0, stream>>>(
            (const Tin *)q, (const Tin *)k, (const Tin *)v, la, beta, S, (Tin *)o, read,
            (const Tin *)z, w, eps, prologue, gate_A, H);
    else
        decode_step_kernel<Tin, DK, DV, false><<<(unsigned)NH, DK * DV / 64, 0, stream>>>(
            (const Tin *)q, (const Tin *)k, (const Tin *)v, la, beta, S, (Tin *)o, read,
            (const Tin *)z, w, eps, prologue, gate_A, H);
    return cuda_status(cudaGetLastError());
}

template <typename Tin>
static int launch_decode_dtype(const void *q, const void *k, const void *v, const float *la,
                               const float *beta, float *S, void *o, int64_t NH, int dk, int dv,
                               float read, const void *z, const float *w, float eps, int prologue,
                               const float *gate_A, int H, bool pc, cudaStream_t stream) {
#define GDR_DECODE_CASE(DK_, DV_)                                                         \
    if (dk == DK_ && dv == DV_)                                                           \
        return launch_decode_t<Tin, DK_, DV_>(q, k, v, la, beta, S, o, NH, read, z, w, eps, \
                                              prologue, gate_A, H, pc, stream);
    GDR_DECODE_CASE(64, 64)
    GDR_DECODE_CASE(64, 128)
    GDR_DECODE_CASE(64, 256)
    GDR_DECODE_CASE(128, 64)
    GDR_DECODE_CASE(128, 128)
    GDR_DECODE_CASE(128, 256)
#undef GDR_DECODE_CASE
    return GDR_ERR_UNSUPPORTED;
}

int launch_decode(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, float *S, void *o, int64_t N, int H, int dk, int dv,
                  int dtype, int rule, const void *out_gate, const float *out_norm_weight,
                  float out_norm_eps, int prologue, const float *gate_A, int decay,
                  cudaStream_t stream) {
    const int64_t NH = N * H;
    const float read = rule == GDR_RULE_ADDITIVE ? 0.f : 1.f;
    const bool pc = decay == GDR_DECAY_CHANNEL;
    if (dtype == GDR_BF16)
        return launch_decode_dtype<__nv_bfloat16>(q, k, v, log_alpha, beta, S, o, NH, dk, dv,
                                                  read, out_gate, out_norm_weight, out_norm_eps,
                                                  prologue, gate_A, H, pc, stream);
    return launch_decode_dtype<float>(q, k, v, log_alpha, beta, S, o, NH, dk, dv, read, out_gate,
                                      out_norm_weight, out_norm_eps, prologue, gate_A, H, pc, stream);
}

}  // namespace gdr
