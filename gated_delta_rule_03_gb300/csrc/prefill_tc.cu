// prefill_tc.cu -- chunked prefill of the gated delta rule on the 5th-generation tensor
// cores (tcgen05), for bf16 q/k/v with d_k = 128 and d_v a multiple of 128.
//
// What it computes is the chunk form of the recurrence: the chunk algorithm of
// "Attention as Matrix Algebra: From Softmax to the Delta Rule", section 8
// ("Training the delta rule in chunks"), with the decay gate carried through the
// same substitution. Per chunk of C = 64 tokens entering with state S (d_k x d_v):
//   g_t = sum_{i<=t} log alpha_i,  gamma_t = exp(g_t),  Gamma_ti = exp(g_t - g_i)
//   L_ti = beta_t Gamma_ti k_t.k_i (i < t),  T = (I + L)^{-1} diag(beta)
//   Utilde = T V,  W = T diag(gamma) K,  U = Utilde - W S
//   O = diag(gamma) Q S + (Q K^T . Gamma . [i <= t]) U
//   S <- gamma_C S + Ktilde^T U,  Ktilde_i = exp(g_C - g_i) k_i
//
// Work mapping. One CTA per (sequence, head, 128-column slice of d_v); the value
// columns of S evolve independently. Every dense product is a tcgen05.mma chain with
// bf16 operands in 128-byte-swizzled shared memory and fp32 accumulators in TMEM,
// in the transposed orientation so that M is always 128:
//   G      = [K; Q] K^T                       (M=128: 64 keys then 64 queries; N=64)
//   U~^T   = V^T T^T,  W^T = K^T (T diag gamma)^T                       (N=64, K=64)
//   (WS)^T = S^T W^T,  O^T = S^T (diag(gamma) Q)^T                      (N=64, K=128)
//   S_upd^T = U^T Ktilde,  O^T += U^T A^T                         (N=128|64, K=64)
// q, k and v arrive by TMA as 64x64 bf16 boxes; the same tiles serve as K-major
// operands (Gram) and as MN-major operands (products over tokens).
//
// Warp roles (16 warps; an SM sub-partition holds one warp of each warpgroup), one
// pipeline:
//   warp 0      producer: TMA loads of q, k, v and the gates of chunk c into one of
//               two stages; cumulative log-decay by a warp scan. (Warps 1-3 idle.)
//   warps 4-7   "prep" (everything that does not depend on S): G, the masked L and A,
//               the unit lower-triangular solve (fp32, CUDA cores), T and
//               T diag(gamma), U~ and W, W^T to shared memory, and the in-place
//               scaling of the stage's Q rows by gamma and K rows by exp(g_C - g).
//               Its own elected thread issues G and U~/W.
//   warps 8-15  "state" (the sequential chain): WS, U = U~ - WS, S_upd, the bf16 copy
//               of S^T that feeds the next chunk, and the outputs. The fp32 master S^T
//               lives in TMEM: while WS runs it is scaled by gamma_C in place, and
//               S_upd accumulates U^T Ktilde onto it. Its own elected thread issues
//               WS, QS, S_upd and AU.
// Prep runs up to one chunk ahead of state, so the state chain -- WS, U, S_upd, the
// state update -- is the critical path per chunk.
//
// Two equivalent forms of the decay factors, chosen per chunk:
//  * ratio form, when the chunk's cumulative log-decay g_C (its minimum) stays above
//    -80 so that gamma and 1/gamma are finite normal floats: Gamma_ti = gamma_t / gamma_i
//    needs no per-entry exponential, and the decay moves off Q and K entirely --
//      A U = (1/gamma_C) (Q K^T . [i <= t]) (diag(kdec) U),  S_upd = K^T (diag(kdec) U),
//      O_t = gamma_t ((S^T q_t) + ((A U)_t)/gamma_t) computed as gamma_t times the
//      accumulator of Q S + (1/gamma_C)(masked Q K^T)(diag(kdec) U),
//    with kdec_t = exp(g_C - g_t); q, k stay as loaded.
//  * exponential form otherwise: Gamma_ti = exp(g_t - g_i) per entry (exponents <= 0),
//    and the stage's Q rows are scaled by gamma and K rows by kdec in place.
// Both compute the same products; only the placement of the decay factors differs.
// Padding rows of a partial last chunk get beta = 0 and log alpha = 0: their rows of
// T, W, U~ and U are zero, they change nothing and they are not stored.
// Every wait is bounded; a role that gives up marks the call GDR_ERR_DEVICE_TIMEOUT in
// the status word, and the others give up in turn, drain and free TMEM.
#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int C = kChunk;   // 64 tokens per chunk
constexpr int DK = 128;     // key dimension
constexpr int NV = 128;     // value columns per CTA
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPrepWarp0 = 4, kPrepThreads = 128;
constexpr int kStateWarp0 = 8, kStateThreads = 256;
constexpr int kBarPrep = 1, kBarState = 2;  // named barrier ids
constexpr int LP = C + 1;                   // fp32 pitch of the solve matrices

// Shared memory map (bytes from a 1024-aligned base). A stage holds one chunk's inputs.
constexpr uint32_t STAGE_BYTES = 51200;
constexpr uint32_t ST_KQ = 0;        // K_b0 | Q_b0 | K_b1 | Q_b1, 8 KB each (b = d_k half)
constexpr uint32_t ST_V = 32768;     // V_b0 | V_b1 (b = half of this CTA's d_v slice)
constexpr uint32_t ST_GATE = 49152;  // fp32 g, gamma, beta, kdec = exp(g_C - g), 1/gamma [64 each]
constexpr int G_G = 0, G_GAM = 64, G_BETA = 128, G_KDEC = 192, G_GINV = 256;  // float offsets
// Gamma_ti = gamma_t / gamma_i exactly when no gamma underflows: the chunk's cumulative
// decay g_C (its minimum, since log alpha <= 0) stays above this bound. Otherwise each
// Gamma_ti is its own exponential of g_t - g_i <= 0.
constexpr float kRatioSafeLogDecay = -80.f;
constexpr uint32_t OFF_ST = 2 * STAGE_BYTES;     // S^T bf16 [d_v 128][d_k 128], two K-blocks
constexpr uint32_t OFF_WT = OFF_ST + 32768;      // W^T bf16 [d_k 128][t 64]
constexpr uint32_t OFF_UT = OFF_WT + 16384;      // U^T bf16 [d_v 128][t 64]; output staging
constexpr uint32_t OFF_AM = OFF_UT + 16384;      // A bf16 [t][i], two 8 KB buffers
constexpr uint32_t OFF_LF = OFF_AM + 16384;      // L fp32 [64][LP]; then T | T diag(gamma)
constexpr uint32_t OFF_NF = OFF_LF + C * LP * 4; // (I + L)^{-1} fp32 [64][LP]
constexpr uint32_t OFF_SG = OFF_NF + C * LP * 4;  // state's copy of gamma[64], kdec[64]
constexpr uint32_t OFF_BAR = OFF_SG + 2 * C * 4;
constexpr uint32_t SMEM_USED = OFF_BAR + 128;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for the 1024-byte alignment
static_assert(OFF_LF % 1024 == 0 && OFF_ST % 1024 == 0 && STAGE_BYTES % 1024 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory");

// mbarrier slots at OFF_BAR (8 bytes each), then the TMEM slot and role flags.
enum {
    B_FULL0 = 0, B_FULL1,    // producer -> prep/state: stage loaded (tx bytes + gates)
    B_EMPTY0, B_EMPTY1,      // state -> producer: stage free again
    B_G,                     // G done                        (prep issuer commit)
    B_UW0, B_UW1,            // U~ (buffer c%2) and W done     (prep issuer commit)
    B_WQ,                    // W^T stored, Q/K scaled         (128 prep arrivals)
    B_WS,                    // WS done                        (state issuer commit)
    B_S,                     // S_upd done                     (state issuer commit)
    B_O,                     // QS + AU done                   (state issuer commit)
    B_DRAIN0, B_DRAIN1,      // drain after an abort
    B_COUNT
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t OFF_FLAGS = OFF_TMEM_SLOT + 4;  // int: prep_fail, state_fail, any_fail

// TMEM columns (fp32 over 128 lanes; TM_S holds the master state S^T).
constexpr uint32_t TM_G = 0, TM_U = 64 /* two buffers */, TM_W = 192, TM_WS = 256, TM_O = 320,
                   TM_S = 384, TM_COLS = 512;

constexpr uint32_t TMA_BYTES = 6 * 64 * 64 * 2;  // K, Q, V: two 64x64 bf16 boxes each

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// exp(x) through the hardware base-2 exponential (flushes subnormal results to zero).
__device__ __forceinline__ float fast_exp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// ---------------------------------------------------------------- warp-level 16x16 products
// The unit lower-triangular solve combines 16x16 blocks. These products are far below
// the tensor-core MMA's minimum tile (M = 64) and sit on a short dependency chain, so
// they use the warp-synchronous m16n8k8 TF32 MMA with fp32 accumulation (operands
// rounded to TF32, 2^-11 relative; the solve's result is rounded to bf16 afterwards).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d (+)= A * B for 16x16 row-major blocks A (pitch pa) and B (pitch pb); d holds the
// result's two 16x8 halves in the m16n8 accumulator layout.
__device__ __forceinline__ void warp_gemm16(const float *__restrict__ A, int pa,
                                            const float *__restrict__ B, int pb, float (&d)[2][4],
                                            int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a[4] = {to_tf32(A[g * pa + 8 * ks + q]), to_tf32(A[(g + 8) * pa + 8 * ks + q]),
                               to_tf32(A[g * pa + 8 * ks + q + 4]),
                               to_tf32(A[(g + 8) * pa + 8 * ks + q + 4])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {to_tf32(B[(8 * ks + q) * pb + 8 * nt + g]),
                                   to_tf32(B[(8 * ks + q + 4) * pb + 8 * nt + g])};
            mma_tf32_16x8x8(d[nt], a, b);
        }
    }
}

// M = scale * d for a 16x16 row-major block M (pitch pm).
__device__ __forceinline__ void warp_store16(float *__restrict__ M, int pm, const float (&d)[2][4],
                                             int lane, float scale) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        M[g * pm + 8 * nt + 2 * q] = scale * d[nt][0];
        M[g * pm + 8 * nt + 2 * q + 1] = scale * d[nt][1];
        M[(g + 8) * pm + 8 * nt + 2 * q] = scale * d[nt][2];
        M[(g + 8) * pm + 8 * nt + 2 * q + 1] = scale * d[nt][3];
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Writes 32 fp32 values as bf16 into columns [32*half, 32*half + 32) of row `row` of a
// 128-byte-swizzled block of 64-wide rows.
__device__ __forceinline__ void store_row32_sw128(unsigned char *block, int row, int half,
                                                  const float (&v)[32]) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const int chunk = 4 * half + jj;
        uint4 w;
        w.x = pack_bf16x2(v[8 * jj + 0], v[8 * jj + 1]);
        w.y = pack_bf16x2(v[8 * jj + 2], v[8 * jj + 3]);
        w.z = pack_bf16x2(v[8 * jj + 4], v[8 * jj + 5]);
        w.w = pack_bf16x2(v[8 * jj + 6], v[8 * jj + 7]);
        *reinterpret_cast<uint4 *>(block + row * 128 + (((chunk ^ row) & 7) << 4)) = w;
    }
}

// Nf = (I + L)^{-1} for the strictly lower-triangular 64x64 L in Lf (fp32, pitch LP),
// by the 128 prep threads. 16x16 diagonal blocks by forward substitution in fp32 (one
// column per thread), then the off-diagonal blocks with warp-level TF32 products. Only
// the lower triangle (with its unit diagonal) of Nf is written; Lf's strictly lower
// off-diagonal blocks are overwritten on the way.
__device__ __forceinline__ void unit_lower_inverse(float *__restrict__ Lf,
                                                   float *__restrict__ Nf, int ptid) {
    if (ptid < C) {
        const int base = 16 * (ptid >> 4), c = ptid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < r; ++k) s = fmaf(-Lf[(base + r) * LP + base + k], x[k], s);
            x[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Nf[(base + r) * LP + base + c] = x[r];
    }
    named_sync(kBarPrep, kPrepThreads);
    // Off-diagonal blocks. With M_ik = N_ii L_ik (i > k), N_ij = -sum_{k=j}^{i-1} M_ik N_kj:
    // first all six M blocks in one round (written over the L blocks, which are not read
    // again), then the blocks by distance from the diagonal, each by one warp as a
    // single chain of accumulated products.
    const int w = ptid >> 5, lane = ptid & 31;
    float *__restrict__ Mf = Lf;
    {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int b = w + 4 * r;  // blocks (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
            if (b < 6) {
                const int i = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
                const int k = b < 3 ? b : (b < 5 ? b - 3 : 0);
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                warp_gemm16(Nf + 16 * i * LP + 16 * i, LP, Lf + 16 * i * LP + 16 * k, LP, acc, lane);
                __syncwarp();
                warp_store16(Mf + 16 * i * LP + 16 * k, LP, acc, lane, 1.f);
            }
        }
    }
    named_sync(kBarPrep, kPrepThreads);
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        if (w < 4 - d) {
            const int i = d + w, j = w;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int k = j; k < i; ++k)
                warp_gemm16(Mf + 16 * i * LP + 16 * k, LP, Nf + 16 * k * LP + 16 * j, LP, acc, lane);
            warp_store16(Nf + 16 * i * LP + 16 * j, LP, acc, lane, -1.f);
        }
        named_sync(kBarPrep, kPrepThreads);
    }
}

struct TcParams {
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;
    int64_t num_seqs, total_tokens;
    int H, dv, n_slices;
    __nv_bfloat16 *o;
    float *S_final;
    int32_t *ctl;
};

// MMA issue helpers (one thread). Descriptors per the layouts described above.
__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t kq) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = kq + (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tmem + TM_G, sw128_desc(off, 16, 1024), sw128_desc(off, 16, 1024),
                 idesc_bf16(128, 64, 0, 0), kk > 0);
    }
}

__device__ __forceinline__ void issue_uw(uint32_t tmem, uint32_t kq, uint32_t v, uint32_t tm,
                                         uint32_t tg, uint32_t ubuf) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem + TM_U + 64 * ubuf, sw128_desc(v + kk * 2048, 8192, 1024),
                 sw128_desc(tm + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem + TM_W, sw128_desc(kq + kk * 2048, 16384, 1024),
                 sw128_desc(tg + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
}

__device__ __forceinline__ void issue_ws(uint32_t tmem, uint32_t st, uint32_t wt) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + TM_WS, sw128_desc(st + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                 sw128_desc(wt + kk * 2048, 8192, 1024), idesc_bf16(128, 64, 0, 1), kk > 0);
}

__device__ __forceinline__ void issue_qs(uint32_t tmem, uint32_t st, uint32_t kq) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + TM_O, sw128_desc(st + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                 sw128_desc(kq + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32, 16, 1024),
                 idesc_bf16(128, 64, 0, 0), kk > 0);
}

__device__ __forceinline__ void issue_supd_au(uint32_t tmem, uint32_t ut, uint32_t kq,
                                              uint32_t am, uint32_t bar_s, uint32_t bar_empty,
                                              uint32_t bar_o) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem + TM_S, sw128_desc(ut + kk * 32, 16, 1024),
                 sw128_desc(kq + kk * 2048, 16384, 1024), idesc_bf16(128, 128, 0, 1), 1);
    mma_commit(bar_s);
    mma_commit(bar_empty);  // S_upd and the earlier QS were the stage's last readers
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem + TM_O, sw128_desc(ut + kk * 32, 16, 1024), sw128_desc(am + kk * 32, 16, 1024),
                 idesc_bf16(128, 64, 0, 0), 1);
    mma_commit(bar_o);
}

__global__ void __launch_bounds__(kThreads, 1)
tc_prefill_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const TcParams p) {
    if (p.ctl[0] != GDR_OK) return;  // cu_seqlens rejected by the planning kernel
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that every access
    // through it stays a shared-memory access the compiler can schedule freely
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM_SLOT);
    volatile int *flags = reinterpret_cast<volatile int *>(sm + OFF_FLAGS);  // prep, state, any

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int slice = blockIdx.x % p.n_slices;
    const int nh = blockIdx.x / p.n_slices;
    const int n = nh / p.H, h = nh % p.H;
    int64_t seq_begin, seq_end;
    if (p.cu_seqlens) {
        seq_begin = p.cu_seqlens[n];
        seq_end = p.cu_seqlens[n + 1];
    } else {
        const int64_t len = p.total_tokens / p.num_seqs;
        seq_begin = (int64_t)n * len;
        seq_end = seq_begin + len;
    }
    const int n_chunks = (int)((seq_end - seq_begin + C - 1) / C);
    const int col0 = slice * NV;  // first value column of this CTA

    if (tid == 0) {
        mbar_init(bar(B_FULL0), 2);
        mbar_init(bar(B_FULL1), 2);
        mbar_init(bar(B_EMPTY0), 2);
        mbar_init(bar(B_EMPTY1), 2);
        mbar_init(bar(B_G), 1);
        mbar_init(bar(B_UW0), 1);
        mbar_init(bar(B_UW1), 1);
        mbar_init(bar(B_WQ), kPrepThreads);
        mbar_init(bar(B_WS), 1);
        mbar_init(bar(B_S), 1);
        mbar_init(bar(B_O), 1);
        mbar_init(bar(B_DRAIN0), 1);
        mbar_init(bar(B_DRAIN1), 1);
        fence_mbar_init();
        flags[0] = flags[1] = flags[2] = 0;
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ============================================================ producer
        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t stage = sbase + s * STAGE_BYTES;
            bool ok = true;
            if (c >= 2 && lane == 0) ok = mbar_wait(bar(B_EMPTY0 + s), (u - 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                flags[2] = 1;
                break;
            }
            const int64_t t0 = seq_begin + (int64_t)c * C;
            const int len = (int)((seq_end - t0) < C ? (seq_end - t0) : C);
            if (lane == 0) {
                const uint32_t fb = bar(B_FULL0 + s);
                mbar_arrive_expect_tx(fb, TMA_BYTES);
                const int tt = (int)t0;
                tma_load_3d(stage + ST_KQ + 0, &map_k, fb, 0, h, tt);
                tma_load_3d(stage + ST_KQ + 16384, &map_k, fb, 64, h, tt);
                tma_load_3d(stage + ST_KQ + 8192, &map_q, fb, 0, h, tt);
                tma_load_3d(stage + ST_KQ + 24576, &map_q, fb, 64, h, tt);
                tma_load_3d(stage + ST_V + 0, &map_v, fb, col0, h, tt);
                tma_load_3d(stage + ST_V + 8192, &map_v, fb, col0 + 64, h, tt);
            }
            // gates of tokens 2*lane and 2*lane + 1, cumulative log-decay by a warp scan
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
            if (2 * lane < len) {
                const size_t off = (size_t)(t0 + 2 * lane) * p.H + h;
                a0 = p.log_alpha[off];
                b0 = p.beta[off];
            }
            if (2 * lane + 1 < len) {
                const size_t off = (size_t)(t0 + 2 * lane + 1) * p.H + h;
                a1 = p.log_alpha[off];
                b1 = p.beta[off];
            }
            float sum = a0 + a1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float up = __shfl_up_sync(0xffffffffu, sum, off);
                if (lane >= off) sum += up;
            }
            const float g0 = sum - a1, g1 = sum;
            const float g_last = __shfl_sync(0xffffffffu, sum, 31);
            float *gate = reinterpret_cast<float *>(sm + s * STAGE_BYTES + ST_GATE);
            gate[G_G + 2 * lane] = g0;
            gate[G_G + 2 * lane + 1] = g1;
            gate[G_GAM + 2 * lane] = fast_exp(g0);
            gate[G_GAM + 2 * lane + 1] = fast_exp(g1);
            gate[G_BETA + 2 * lane] = b0;
            gate[G_BETA + 2 * lane + 1] = b1;
            gate[G_KDEC + 2 * lane] = fast_exp(g_last - g0);
            gate[G_KDEC + 2 * lane + 1] = fast_exp(g_last - g1);
            gate[G_GINV + 2 * lane] = fast_exp(-g0);
            gate[G_GINV + 2 * lane + 1] = fast_exp(-g1);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_FULL0 + s));
        }
    } else if (warp >= kPrepWarp0 && warp < kStateWarp0) {
        // ============================================================ prep
        const int ptid = tid - 32 * kPrepWarp0;
        const int row = 32 * (warp & 3) + lane;  // this thread's TMEM lane
        const bool issuer = ptid == 0;
        volatile int *fail = &flags[0];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        float *__restrict__ Lf = reinterpret_cast<float *>(sm + OFF_LF);
        float *__restrict__ Nf = reinterpret_cast<float *>(sm + OFF_NF);
        auto check = [&](bool ok) -> bool {  // role-wide agreement after a wait
            if (!ok) { *fail = 1; flags[2] = 1; }
            named_sync(kBarPrep, kPrepThreads);
            return *fail == 0;
        };
        if (issuer && n_chunks > 0) {
            if (mbar_wait(bar(B_FULL0), 0)) {
                tc_fence_after();
                issue_gram(tmem, sbase + ST_KQ);
                mma_commit(bar(B_G));
            } else {
                *fail = 1;
                flags[2] = 1;
            }
        }
        __syncwarp();
        bool next_g_issued = true;  // (issuer) G of chunk c already issued
        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t stage = sbase + s * STAGE_BYTES;
            const float *gate = reinterpret_cast<const float *>(sm + s * STAGE_BYTES + ST_GATE);
            if (issuer && !next_g_issued) {
                if (mbar_wait(bar(B_FULL0 + s), u & 1)) {
                    tc_fence_after();
                    issue_gram(tmem, stage + ST_KQ);
                    mma_commit(bar(B_G));
                } else {
                    *fail = 1;
                    flags[2] = 1;
                }
            }
            __syncwarp();
            bool ok = mbar_wait(bar(B_G), c & 1) && mbar_wait(bar(B_FULL0 + s), u & 1);
            if (!check(ok)) break;
            tc_fence_after();

            // ---- L (fp32, strictly lower) from K K^T, masked A (bf16) from Q K^T
            {
                const int t = row < C ? row : row - C;
                // Gamma_ti as gamma_t / gamma_i when that is exact, else exp(g_t - g_i)
                const bool ratio = gate[G_G + C - 1] > kRatioSafeLogDecay;
                const float gt = ratio ? gate[G_GAM + t] : gate[G_G + t];
                const float bt = gate[G_BETA + t];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float v[32], gi[32];
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) gi[ii] = gate[(ratio ? G_GINV : G_G) + 32 * hh + ii];
                    tmem_load32(lane_base + TM_G + 32 * hh, v);
                    if (ratio && row >= C) {  // A in ratio form: (1/gamma_C) q_t.k_i
                        const float ginv_c = gate[G_GINV + C - 1];
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) v[ii] *= ginv_c;
                    } else {
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) {
                            const float dec = ratio ? gt * gi[ii] : fast_exp(gt - gi[ii]);
                            v[ii] *= dec;
                        }
                    }
                    if (row < C) {  // L: strictly lower entries only (the solve reads no others)
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii)
                            if (32 * hh + ii < t) Lf[t * LP + 32 * hh + ii] = bt * v[ii];
                    } else {        // A: causal mask i <= t, zeros above
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii)
                            if (32 * hh + ii > t) v[ii] = 0.f;
                        store_row32_sw128(sm + OFF_AM + (c & 1) * 8192, t, hh, v);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);

            // ---- T = (I + L)^{-1} diag(beta) and T diag(gamma), bf16, over L's space
            unit_lower_inverse(Lf, Nf, ptid);
            {
                const int t = ptid >> 1, hh = ptid & 1;
                float tv[32], tg[32];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    tv[ii] = Nf[t * LP + 32 * hh + ii];
                    tg[ii] = gate[G_GAM + 32 * hh + ii];
                }
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * hh + ii;
                    const float x = (i <= t) ? tv[ii] * gate[G_BETA + i] : 0.f;
                    tv[ii] = x;
                    tg[ii] *= x;
                }
                store_row32_sw128(sm + OFF_LF, t, hh, tv);
                store_row32_sw128(sm + OFF_LF + 8192, t, hh, tg);
            }
            fence_async_smem();
            named_sync(kBarPrep, kPrepThreads);

            // ---- U~ and W; then, if its stage has landed, G of the next chunk
            if (issuer) {
                tc_fence_after();
                issue_uw(tmem, stage + ST_KQ, stage + ST_V, sbase + OFF_LF, sbase + OFF_LF + 8192,
                         c & 1);
                mma_commit(bar(B_UW0 + (c & 1)));
                next_g_issued = false;
                if (c + 1 < n_chunks) {
                    const int s1 = (c + 1) & 1;
                    if (mbar_try_wait(bar(B_FULL0 + s1), ((c + 1) >> 1) & 1)) {
                        tc_fence_after();
                        issue_gram(tmem, sbase + s1 * STAGE_BYTES + ST_KQ);
                        mma_commit(bar(B_G));
                        next_g_issued = true;
                    }
                }
            }
            __syncwarp();
            ok = mbar_wait(bar(B_UW0 + (c & 1)), u & 1);
            if (c > 0) ok = ok && mbar_wait(bar(B_WS), (c - 1) & 1);  // W^T buffer free
            if (!check(ok)) break;
            tc_fence_after();

            // ---- W^T to shared memory; scale the stage's Q rows by gamma, K rows by kdec
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[32];
                tmem_load32(lane_base + TM_W + 32 * hh, v);
                store_row32_sw128(sm + OFF_WT, row, hh, v);
            }
            if (!(gate[G_G + C - 1] > kRatioSafeLogDecay))  // exponential form only
#pragma unroll 2
            for (int base = 0; base < 2048; base += 8 * kPrepThreads) {
                uint4 w[8];
                float f[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t o = (base + k * kPrepThreads + ptid) * 16;
                    const int r = (o % 16384) / 128;  // rows 0..63 keys, 64..127 queries
                    f[k] = r < C ? gate[G_KDEC + r] : gate[G_GAM + r - C];
                    w[k] = *reinterpret_cast<const uint4 *>(sm + s * STAGE_BYTES + ST_KQ + o);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t *uw = &w[k].x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 fl = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&uw[e]));
                        uw[e] = pack_bf16x2(fl.x * f[k], fl.y * f[k]);
                    }
                    const uint32_t o = (base + k * kPrepThreads + ptid) * 16;
                    *reinterpret_cast<uint4 *>(sm + s * STAGE_BYTES + ST_KQ + o) = w[k];
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_WQ));
        }
        if (*fail && issuer) {  // let issued MMAs land before TMEM and shared memory go away
            mma_commit(bar(B_DRAIN0));
            mbar_wait(bar(B_DRAIN0), 0);
        }
    } else if (warp >= kStateWarp0) {
        // ============================================================ state
        const int stid = tid - 32 * kStateWarp0;
        const int half = (warp - kStateWarp0) >> 2;  // which 64 of the d_k entries / 32 of the tokens
        const int row = 32 * (warp & 3) + lane;      // TMEM lane = value column col0 + row
        const bool issuer = stid == 0;
        volatile int *fail = &flags[1];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        float *__restrict__ sgate = reinterpret_cast<float *>(sm + OFF_SG);  // gamma | kdec
        auto check = [&](bool ok) -> bool {
            if (!ok) { *fail = 1; flags[2] = 1; }
            named_sync(kBarState, kStateThreads);
            return *fail == 0;
        };
        // master state S^T: lane col0 + row, columns TM_S + d for d in [64*half, 64*half + 64)
        const size_t s_off = ((size_t)n * p.H + h) * DK * p.dv + col0 + row;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[i] = p.S0 ? p.S0[s_off + (size_t)(64 * half + 32 * hh + i) * p.dv] : 0.f;
            tmem_store32(lane_base + TM_S + 64 * half + 32 * hh, v);
            store_row32_sw128(sm + OFF_ST + half * 16384, row, hh, v);
        }
        tc_fence_before();
        fence_async_smem();
        named_sync(kBarState, kStateThreads);
        if (issuer && n_chunks > 0) {
            if (mbar_wait(bar(B_WQ), 0)) {
                tc_fence_after();
                issue_ws(tmem, sbase + OFF_ST, sbase + OFF_WT);
                mma_commit(bar(B_WS));
                issue_qs(tmem, sbase + OFF_ST, sbase + ST_KQ);
            } else {
                *fail = 1;
                flags[2] = 1;
            }
        }
        __syncwarp();
        for (int c = 0; c < n_chunks; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t stage = sbase + s * STAGE_BYTES;
            const float *gate = reinterpret_cast<const float *>(sm + s * STAGE_BYTES + ST_GATE);
            const int64_t t0 = seq_begin + (int64_t)c * C;
            const int len = (int)((seq_end - t0) < C ? (seq_end - t0) : C);

            // ---- while WS runs: copy this chunk's gates, decay the master state in place
            bool ok = mbar_wait(bar(B_FULL0 + s), u & 1);  // this stage's gates are visible
            if (!check(ok)) break;
            tc_fence_after();
            const bool ratio = gate[G_G + C - 1] > kRatioSafeLogDecay;
            if (stid < C) {
                sgate[stid] = gate[G_GAM + stid];
                sgate[C + stid] = gate[G_KDEC + stid];
            }
            {
                const float gC = gate[G_GAM + C - 1];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float v[32];
                    tmem_load32(lane_base + TM_S + 64 * half + 32 * hh, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= gC;
                    tmem_store32(lane_base + TM_S + 64 * half + 32 * hh, v);
                }
            }

            // ---- U^T = U~^T - (WS)^T
            ok = mbar_wait(bar(B_WS), c & 1) && mbar_wait(bar(B_UW0 + (c & 1)), u & 1);
            if (!check(ok)) break;
            tc_fence_after();
            if (issuer) mbar_arrive(bar(B_EMPTY0 + s));  // the stage's gates are no longer read
            {
                float a[32], b[32];
                tmem_load32(lane_base + TM_U + 64 * (c & 1) + 32 * half, a);
                tmem_load32(lane_base + TM_WS + 32 * half, b);
                if (ratio) {  // U' = diag(kdec) U
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = (a[i] - b[i]) * sgate[C + 32 * half + i];
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] -= b[i];
                }
                store_row32_sw128(sm + OFF_UT, row, half, a);
            }
            fence_async_smem();
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            if (issuer) {
                tc_fence_after();
                issue_supd_au(tmem, sbase + OFF_UT, stage + ST_KQ, sbase + OFF_AM + (c & 1) * 8192,
                              bar(B_S), bar(B_EMPTY0 + s), bar(B_O));
            }
            __syncwarp();

            // ---- the new state (gamma_C S + U^T Ktilde, accumulated in TMEM): its bf16 copy
            ok = mbar_wait(bar(B_S), c & 1);
            if (!check(ok)) break;
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[32];
                tmem_load32(lane_base + TM_S + 64 * half + 32 * hh, v);
                store_row32_sw128(sm + OFF_ST + half * 16384, row, hh, v);
            }
            fence_async_smem();
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            if (issuer) {
                if (c + 1 < n_chunks) {
                    if (mbar_wait(bar(B_WQ), (c + 1) & 1)) {
                        tc_fence_after();
                        issue_ws(tmem, sbase + OFF_ST, sbase + OFF_WT);
                        mma_commit(bar(B_WS));
                    } else {
                        *fail = 1;
                        flags[2] = 1;
                    }
                }
            }
            __syncwarp();

            // ---- outputs: O^T from TMEM -> staging tile [t][128] -> coalesced stores
            ok = mbar_wait(bar(B_O), c & 1);
            if (!check(ok)) break;
            tc_fence_after();
            {
                __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_UT);
                float v[32];
                tmem_load32(lane_base + TM_O + 32 * half, v);
                if (ratio) {  // O_t = gamma_t x accumulator
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) v[ii] *= sgate[32 * half + ii];
                }
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) stg[(32 * half + ii) * NV + row] = __float2bfloat16_rn(v[ii]);
            }
            tc_fence_before();
            named_sync(kBarState, kStateThreads);
            if (issuer && c + 1 < n_chunks) {  // O accumulator free again
                tc_fence_after();
                issue_qs(tmem, sbase + OFF_ST, sbase + ((c + 1) & 1) * STAGE_BYTES + ST_KQ);
            }
            {
                const uint4 *stg = reinterpret_cast<const uint4 *>(sm + OFF_UT);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int idx = stid + k * kStateThreads;  // 64 rows x 16 chunks of 16 bytes
                    const int t = idx >> 4, ch = idx & 15;
                    if (t < len)
                        *reinterpret_cast<uint4 *>(p.o + ((size_t)(t0 + t) * p.H + h) * p.dv + col0 +
                                                   ch * 8) = stg[idx];
                }
            }
            named_sync(kBarState, kStateThreads);  // staging consumed before U^T reuses it
        }
        if (*fail == 0) {
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[32];
                tmem_load32(lane_base + TM_S + 64 * half + 32 * hh, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) p.S_final[s_off + (size_t)(64 * half + 32 * hh + i) * p.dv] = v[i];
            }
        } else if (issuer) {
            mma_commit(bar(B_DRAIN1));
            mbar_wait(bar(B_DRAIN1), 0);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (flags[2] != 0 && tid == 0) {
        atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
        // loads still in flight land before the shared memory is released
        for (int s = 0; s < 2 && s < n_chunks; ++s) {
            const int last_c = ((n_chunks - 1 - s) / 2) * 2 + s;  // last chunk that used stage s
            mbar_wait(bar(B_FULL0 + s), (last_c >> 1) & 1);
        }
    }
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ----------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Tensor map over a packed [T, H, d] bf16 tensor, 64 (features) x 1 (head) x 64 (tokens) boxes.
bool make_map(CUtensorMap *map, const void *base, int d, int H, int64_t T) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * H * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill_tc(const PrefillArgs &a, const WsLayout &L) {
    const size_t s_bytes = (size_t)a.num_seqs * a.H * a.dk * a.dv * sizeof(float);
    if (a.total_tokens == 0) {  // nothing to compute: S_final = S0 (or zero)
        cudaError_t e = cudaSuccess;
        if (!a.S0) e = cudaMemsetAsync(a.S_final, 0, s_bytes, a.stream);
        else if (a.S0 != a.S_final)
            e = cudaMemcpyAsync(a.S_final, a.S0, s_bytes, cudaMemcpyDeviceToDevice, a.stream);
        return cuda_status(e);
    }
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.dk, a.H, a.total_tokens) || !make_map(&mk, a.k, a.dk, a.H, a.total_tokens) ||
        !make_map(&mv, a.v, a.dv, a.H, a.total_tokens))
        return GDR_ERR_CUDA;
    TcParams p;
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.H = a.H;
    p.dv = a.dv;
    p.n_slices = a.dv / NV;
    p.o = (__nv_bfloat16 *)a.o;
    p.S_final = a.S_final;
    p.ctl = (int32_t *)(a.ws + L.ctl);
    if (cudaFuncSetAttribute(tc_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    const unsigned grid = (unsigned)(a.num_seqs * a.H * p.n_slices);
    tc_prefill_kernel<<<grid, kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mv, p);
    return cuda_status(cudaGetLastError());
}

}  // namespace gdr
