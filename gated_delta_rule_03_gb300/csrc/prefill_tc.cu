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
// Mapping. One CTA per (sequence, head, 128-column slice of d_v); the value columns of
// S evolve independently, so slices never talk to each other. The CTA walks the
// chunks of its sequence in order. Every dense product is one tcgen05.mma chain
// (bf16 operands from shared memory, fp32 accumulators in TMEM), computed in the
// transposed orientation so that M is always 128 (d_k or the d_v slice):
//   G   = [K; Q] K^T          (M=128 rows: 64 keys then 64 queries, N=64, K=d_k)
//   U~^T = V^T T^T,  W^T = K^T (T diag gamma)^T                  (M=128, N=64, K=64)
//   (WS)^T = S^T W^T,  O^T = S^T (diag(gamma) Q)^T               (M=128, N=64, K=128)
//   S_upd^T = U^T Ktilde,  O^T += U^T A^T                        (M=128, N=128|64, K=64)
// q, k and v arrive by TMA as 64x64 bf16 boxes in the 128-byte-swizzled layout; the
// same tiles serve as K-major operands (Gram) and MN-major operands (products over
// tokens). The fp32 master copy of S^T lives in registers (thread = one d_v lane,
// 64 of the d_k entries); a bf16 copy in shared memory feeds the next chunk's
// products. Exponents g_t - g_i are formed only for i <= t, so they are <= 0.
// The unit lower-triangular solve runs in fp32 on the CUDA cores: 16x16 diagonal
// blocks by forward substitution, then the off-diagonal blocks by block products.
//
// Padding rows of a partial last chunk get beta = 0 and log alpha = 0, which makes
// their rows of T, W, U~ and U zero: they change nothing and are not stored.
// Every mbarrier wait is bounded; on a timeout the CTA records
// GDR_ERR_DEVICE_TIMEOUT in the status word, drains, frees its TMEM and returns.
#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace gdr {
namespace {

using namespace sm100;

constexpr int C = kChunk;      // 64 tokens per chunk
constexpr int DK = 128;        // key dimension
constexpr int NV = 128;        // value columns per CTA
constexpr int kThreads = 256;  // 8 warps: 2 warpgroups x 4 TMEM lane quarters
constexpr int LP = C + 1;      // fp32 pitch of the solve matrices
constexpr int PP = 17;         // fp32 pitch of the solve scratch

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_KQ = 0;          // K_b0 | Q_b0 | K_b1 | Q_b1, 8 KB each (b = d_k half)
constexpr uint32_t OFF_V = 32768;       // V_b0 | V_b1 (b = d_v half of the slice)
constexpr uint32_t OFF_ST = 49152;      // S^T bf16, [d_v 128][d_k 128]: two 16 KB K-blocks
constexpr uint32_t OFF_WT = 81920;      // W^T bf16, [d_k 128][t 64]
constexpr uint32_t OFF_UT = 98304;      // U^T bf16, [d_v 128][t 64]
constexpr uint32_t OFF_AM = 114688;     // A = masked QK^T . Gamma, bf16 [t 64][i 64]
constexpr uint32_t OFF_TM = 122880;     // T bf16 [t][i]
constexpr uint32_t OFF_TG = 131072;     // T diag(gamma) bf16 [t][i]
constexpr uint32_t OFF_LF = 139264;     // L fp32 [64][LP]
constexpr uint32_t OFF_NF = OFF_LF + C * LP * 4;        // (I+L)^{-1} fp32 [64][LP]
constexpr uint32_t OFF_PF = OFF_NF + C * LP * 4;        // solve scratch fp32 [48][PP]
constexpr uint32_t OFF_GATE = OFF_PF + 48 * PP * 4;     // g, gamma, beta, kdec: 4 x 64 fp32
constexpr uint32_t OFF_BAR = OFF_GATE + 4 * C * 4;      // 2 mbarriers + TMEM slot + flags
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;       // slack for the 1024-byte alignment

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t TM_G = 0, TM_U = 64, TM_W = 128, TM_WS = 192, TM_O = 256, TM_S = 384;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t TMA_BYTES = 6 * 64 * 64 * 2;  // K, Q, V: two 64x64 bf16 boxes each

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

// Nf = (I + L)^{-1} for the strictly lower-triangular 64x64 L in Lf (fp32, pitch LP).
// Only the lower triangle (with its unit diagonal) of Nf is written.
__device__ void unit_lower_inverse(const float *Lf, float *Nf, float *Pf, int tid) {
    if (tid < C) {  // 16x16 diagonal blocks: forward substitution, one column per thread
        const int base = 16 * (tid >> 4), c = tid & 15;
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
    __syncthreads();
    // Off-diagonal blocks, by distance d from the diagonal:
    // N_ij = -N_ii * sum_{k=j}^{i-1} L_ik N_kj   (block indices, j = i - d)
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        for (int idx = tid; idx < nb * 256; idx += kThreads) {
            const int blk = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
            const int i = d + blk, j = i - d;
            float s = 0.f;
            for (int k = 16 * j; k < 16 * i; ++k)
                s = fmaf(Lf[(16 * i + r) * LP + k], Nf[k * LP + 16 * j + c], s);
            Pf[(blk * 16 + r) * PP + c] = s;
        }
        __syncthreads();
        for (int idx = tid; idx < nb * 256; idx += kThreads) {
            const int blk = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
            const int i = d + blk, j = i - d;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                s = fmaf(Nf[(16 * i + r) * LP + 16 * i + m], Pf[(blk * 16 + m) * PP + c], s);
            Nf[(16 * i + r) * LP + 16 * j + c] = -s;
        }
        __syncthreads();
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

__global__ void __launch_bounds__(kThreads, 1)
tc_prefill_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const TcParams p) {
    if (p.ctl[0] != GDR_OK) return;  // cu_seqlens rejected by the planning kernel
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    float *Lf = reinterpret_cast<float *>(sm + OFF_LF);
    float *Nf = reinterpret_cast<float *>(sm + OFF_NF);
    float *Pf = reinterpret_cast<float *>(sm + OFF_PF);
    float *g_s = reinterpret_cast<float *>(sm + OFF_GATE);
    float *gam_s = g_s + C;
    float *beta_s = gam_s + C;
    float *kdec_s = beta_s + C;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 16);
    int *abort_flag = reinterpret_cast<int *>(sm + OFF_BAR + 20);
    const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;  // this thread's TMEM lane (d_v or d_k index)

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
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *abort_flag = 0;
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    // Master state: S[d][col0 + row] for d in [64*half, 64*half + 64).
    float S[64];
    const size_t s_off = ((size_t)n * p.H + h) * DK * p.dv + col0 + row;
#pragma unroll
    for (int i = 0; i < 64; ++i)
        S[i] = p.S0 ? p.S0[s_off + (size_t)(64 * half + i) * p.dv] : 0.f;
    {
        float v[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = S[32 * hh + i];
            store_row32_sw128(sm + OFF_ST + half * 16384, row, hh, v);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);

    uint32_t ph_tma = 0, ph_mma = 0;
    bool tma_pending = false, mma_pending = false;

    // All threads wait for a barrier phase; false (for every thread) if any gave up.
    auto wait_all = [&](uint32_t bar, uint32_t &phase, bool &pending) -> bool {
        const bool ok = mbar_wait(bar, phase);
        if (!ok) *abort_flag = 1;
        phase ^= 1;
        __syncthreads();
        if (*abort_flag) return false;
        pending = false;
        tc_fence_after();
        return true;
    };

    for (int c = 0; c < n_chunks; ++c) {
        const int64_t t0 = seq_begin + (int64_t)c * C;
        const int len = (int)((seq_end - t0) < C ? (seq_end - t0) : C);

        // ---- loads: q, k, v tiles by TMA; gates by plain loads
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_tma, TMA_BYTES);
            const int tt = (int)t0;
            tma_load_3d(sbase + OFF_KQ + 0, &map_k, bar_tma, 0, h, tt);
            tma_load_3d(sbase + OFF_KQ + 16384, &map_k, bar_tma, 64, h, tt);
            tma_load_3d(sbase + OFF_KQ + 8192, &map_q, bar_tma, 0, h, tt);
            tma_load_3d(sbase + OFF_KQ + 24576, &map_q, bar_tma, 64, h, tt);
            tma_load_3d(sbase + OFF_V + 0, &map_v, bar_tma, col0, h, tt);
            tma_load_3d(sbase + OFF_V + 8192, &map_v, bar_tma, col0 + 64, h, tt);
        }
        tma_pending = true;
        if (tid < C) {
            float la = 0.f, b = 0.f;
            if (tid < len) {
                const size_t off = (size_t)(t0 + tid) * p.H + h;
                la = p.log_alpha[off];
                b = p.beta[off];
            }
            g_s[tid] = la;
            beta_s[tid] = b;
        }
        __syncthreads();
        if (warp == 0) {  // inclusive prefix sum of log alpha, two tokens per lane
            const float a0 = g_s[2 * lane], a1 = g_s[2 * lane + 1];
            float s = a0 + a1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float up = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += up;
            }
            const float g0 = s - a1, g1 = s;
            const float g_last = __shfl_sync(0xffffffffu, s, 31);
            g_s[2 * lane] = g0;
            g_s[2 * lane + 1] = g1;
            gam_s[2 * lane] = __expf(g0);
            gam_s[2 * lane + 1] = __expf(g1);
            kdec_s[2 * lane] = __expf(g_last - g0);
            kdec_s[2 * lane + 1] = __expf(g_last - g1);
        }
        if (!wait_all(bar_tma, ph_tma, tma_pending)) break;

        // ---- G = [K; Q] K^T
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = sbase + OFF_KQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + TM_G, sw128_desc(off, 16, 1024), sw128_desc(off, 16, 1024),
                         idesc_bf16(128, 64, 0, 0), kk > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma, mma_pending)) break;

        // ---- L (fp32, for the solve) from K K^T; masked A from Q K^T
        {
            float v[32];
            tmem_load32(lane_base + TM_G + 32 * half, v);
            if (row < C) {
                const int t = row;
                const float gt = g_s[t], bt = beta_s[t];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * half + ii;
                    Lf[t * LP + i] = (i < t) ? bt * __expf(gt - g_s[i]) * v[ii] : 0.f;
                }
            } else {
                const int t = row - C;
                const float gt = g_s[t];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * half + ii;
                    v[ii] = (i <= t) ? __expf(gt - g_s[i]) * v[ii] : 0.f;
                }
                store_row32_sw128(sm + OFF_AM, t, half, v);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + L)^{-1} diag(beta), and T diag(gamma), as bf16 MMA operands
        unit_lower_inverse(Lf, Nf, Pf, tid);
        {
            const int t = tid >> 2, cq = tid & 3;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int chunk = 2 * cq + jj;
                float tv[8], tg[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * chunk + e;
                    const float x = (i <= t) ? Nf[t * LP + i] * beta_s[i] : 0.f;
                    tv[e] = x;
                    tg[e] = x * gam_s[i];
                }
                const uint32_t o = t * 128 + (((chunk ^ t) & 7) << 4);
                uint4 w;
                w.x = pack_bf16x2(tv[0], tv[1]); w.y = pack_bf16x2(tv[2], tv[3]);
                w.z = pack_bf16x2(tv[4], tv[5]); w.w = pack_bf16x2(tv[6], tv[7]);
                *reinterpret_cast<uint4 *>(sm + OFF_TM + o) = w;
                w.x = pack_bf16x2(tg[0], tg[1]); w.y = pack_bf16x2(tg[2], tg[3]);
                w.z = pack_bf16x2(tg[4], tg[5]); w.w = pack_bf16x2(tg[6], tg[7]);
                *reinterpret_cast<uint4 *>(sm + OFF_TG + o) = w;
            }
        }
        fence_async_smem();
        __syncthreads();

        // ---- U~^T = V^T T^T and W^T = K^T (T diag gamma)^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + TM_U, sw128_desc(sbase + OFF_V + kk * 2048, 8192, 1024),
                         sw128_desc(sbase + OFF_TM + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0),
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + TM_W, sw128_desc(sbase + OFF_KQ + kk * 2048, 16384, 1024),
                         sw128_desc(sbase + OFF_TG + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0),
                         kk > 0);
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma, mma_pending)) break;

        // ---- W^T to shared memory; scale Q rows by gamma and K rows by exp(g_C - g)
        {
            float v[32];
            tmem_load32(lane_base + TM_W + 32 * half, v);
            store_row32_sw128(sm + OFF_WT, row, half, v);
        }
        for (int ci = tid; ci < 2048; ci += kThreads) {
            const uint32_t o = ci * 16;
            const int r = (o % 16384) / 128;  // rows 0..63 keys, 64..127 queries
            const float f = r < C ? kdec_s[r] : gam_s[r - C];
            uint4 w = *reinterpret_cast<uint4 *>(sm + OFF_KQ + o);
            uint32_t *u = &w.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&u[e]);
                const float2 fl = __bfloat1622float2(b2);
                u[e] = pack_bf16x2(fl.x * f, fl.y * f);
            }
            *reinterpret_cast<uint4 *>(sm + OFF_KQ + o) = w;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- (WS)^T = S^T W^T and O^T = S^T (diag(gamma) Q)^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t a = sw128_desc(sbase + OFF_ST + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_bf16(tmem + TM_WS, a, sw128_desc(sbase + OFF_WT + kk * 2048, 8192, 1024),
                         idesc_bf16(128, 64, 0, 1), kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t a = sw128_desc(sbase + OFF_ST + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_bf16(tmem + TM_O, a,
                         sw128_desc(sbase + OFF_KQ + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32, 16, 1024),
                         idesc_bf16(128, 64, 0, 0), kk > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma, mma_pending)) break;

        // ---- U^T = U~^T - (WS)^T
        {
            float a[32], b[32];
            tmem_load32(lane_base + TM_U + 32 * half, a);
            tmem_load32(lane_base + TM_WS + 32 * half, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] -= b[i];
            store_row32_sw128(sm + OFF_UT, row, half, a);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- S_upd^T = U^T Ktilde and O^T += U^T A^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = sw128_desc(sbase + OFF_UT + kk * 32, 16, 1024);
                mma_bf16(tmem + TM_S, a, sw128_desc(sbase + OFF_KQ + kk * 2048, 16384, 1024),
                         idesc_bf16(128, 128, 0, 1), kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = sw128_desc(sbase + OFF_UT + kk * 32, 16, 1024);
                mma_bf16(tmem + TM_O, a, sw128_desc(sbase + OFF_AM + kk * 32, 16, 1024),
                         idesc_bf16(128, 64, 0, 0), 1);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma, mma_pending)) break;

        // ---- S <- gamma_C S + S_upd (fp32 master), its bf16 copy, and the outputs
        {
            const float gC = gam_s[C - 1];
            float v[32];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                tmem_load32(lane_base + TM_S + 64 * half + 32 * hh, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    S[32 * hh + i] = fmaf(gC, S[32 * hh + i], v[i]);
                    v[i] = S[32 * hh + i];
                }
                store_row32_sw128(sm + OFF_ST + half * 16384, row, hh, v);
            }
            tmem_load32(lane_base + TM_O + 32 * half, v);
            __nv_bfloat16 *op = p.o + ((size_t)t0 * p.H + h) * p.dv + col0 + row;
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int t = 32 * half + ii;
                if (t < len) op[(size_t)t * p.H * p.dv] = __float2bfloat16_rn(v[ii]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    if (*abort_flag) {
        // A wait gave up: record it, then give outstanding copies and MMAs a bounded
        // chance to land before the shared memory and TMEM are released.
        if (tid == 0) {
            atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
            if (tma_pending) mbar_wait(bar_tma, ph_tma ^ 1);
            if (mma_pending) mbar_wait(bar_mma, ph_mma ^ 1);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) p.S_final[s_off + (size_t)(64 * half + i) * p.dv] = S[i];
    }
    tc_fence_before();
    __syncthreads();
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
