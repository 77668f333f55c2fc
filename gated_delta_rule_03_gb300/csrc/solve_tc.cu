// solve_tc.cu -- the chunk-parallel half of the tensor-core prefill: for every
// (chunk, head) the decayed key Gram matrix, its unit lower-triangular inverse, the
// pseudo-value transform that the sequential chain kernel applies to the values, and
// the masked intra-chunk query-key products.
//
// This is the UT/WY step of "Attention as Matrix Algebra: From Softmax to the Delta
// Rule", section 8 ("Training the delta rule in chunks": one triangular solve per
// chunk turns values into pseudo-values), with the decay gate carried through. Per
// chunk of C = 64 tokens, g_t the cumulative log-decay within the chunk:
//   L_ti = beta_t exp(g_t - g_i) k_t.k_i   (i < t),     T = (I + L)^{-1} diag(beta)
//   T'   = diag(kdec) T  with kdec_t = exp(g_C - g_t)   in the ratio form,
//   T'   = T                                            in the exponential form,
// and the transposed causal query-key products (i <= t, else 0)
//   A^T_it = (1/gamma_C) k_i.q_t                    in the ratio form,
//   A^T_it = exp(g_t - g_i) k_i.q_t                 in the exponential form,
// both stored as bf16 [64][64] row-major: matrix 2u is T' and 2u + 1 is A^T of unit u,
// units ordered chunk-major, head-minor. Each unit's decay factors go out with them
// (fp32 [256]: g[64], gamma[64], kdec[64], then 1 for the ratio form and 0 otherwise),
// so that the chain kernel uses the same values and the same form. (The two forms are described in prefill_tc.cu;
// they differ only in where the decay factors are applied, and both kernels choose
// the same form for a chunk.)
//
// Mapping. A CTA of 4 warps takes units two at a time. One tcgen05.mma chain forms
// [K_a; K_b] [K_a; K_b; Q_a; Q_b]^T (M = 128, N = 256, K = d_k = 128) in TMEM from
// TMA-loaded bf16 tiles: its diagonal 64x64 blocks are the units' Gram matrices K K^T
// and K Q^T. Warps 0-1 read unit a's rows (TMEM lanes 0-63), warps 2-3 unit b's (lanes
// 64-127). The solve is fp32 on the CUDA cores: 16x16 diagonal blocks by forward
// substitution, the off-diagonal blocks with warp-level TF32 products. While a pair is
// solved, the next pair's keys and queries are already loading. Two CTAs share an SM.
#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace sm100;
using namespace tc;

constexpr int C = kChunk;
constexpr int kThreads = 128;
constexpr int kBarSolve = 1;  // named barrier of the whole CTA
constexpr int LP = C + 1;     // fp32 pitch of the solve matrices

// per d_k half b (32 KB): K_a | K_b | Q_a | Q_b, 8 KB each; rows 0-127 are the MMA's A
// operand, rows 0-255 its B operand
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_LF = 65536;                // L fp32 [64][LP] (then the M blocks)
constexpr uint32_t OFF_NF = OFF_LF + C * LP * 4;  // (I + L)^{-1} fp32 [64][LP]
constexpr uint32_t OFF_GATE = OFF_NF + C * LP * 4;
constexpr int G_G = 0, G_GAM = 64, G_GINV = 128, G_BETA = 192, G_KDEC = 256, G_UNIT = 320;
constexpr uint32_t OFF_BAR = OFF_GATE + 2 * G_UNIT * 4;  // per unit: g, gamma, 1/gamma, beta, kdec
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES * 2 <= 227 * 1024, "two CTAs per SM");
enum { B_FULL = 0, B_MMA, B_DRAIN, B_COUNT };
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t OFF_FAIL = OFF_TMEM_SLOT + 4;
constexpr uint32_t TM_COLS = 256;

// ---------------------------------------------------------------- warp-level 16x16 products
// The unit lower-triangular solve combines 16x16 blocks. These products are far below
// the tensor-core MMA's minimum tile and sit on a short dependency chain, so they use
// the warp-synchronous m16n8k8 TF32 MMA with fp32 accumulation (operands rounded to
// TF32, 2^-11 relative; the solve's result is rounded to bf16 afterwards).
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

// Nf = (I + L)^{-1} for the strictly lower-triangular 64x64 L in Lf (fp32, pitch LP),
// by the CTA's 128 threads. 16x16 diagonal blocks by forward substitution (one column
// per thread), then the off-diagonal blocks: with M_ik = N_ii L_ik (i > k),
// N_ij = -sum_{k=j}^{i-1} M_ik N_kj. All six M blocks are formed in one round (written
// over the L blocks, which are not read again), then the N blocks by distance from the
// diagonal, each by one warp as a single chain of accumulated products. Only the lower
// triangle (with its unit diagonal) of Nf is written.
__device__ __forceinline__ void unit_lower_inverse(float *__restrict__ Lf, float *__restrict__ Nf,
                                                   int tid) {
    if (tid < C) {
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
    named_sync(kBarSolve, kThreads);
    const int w = tid >> 5, lane = tid & 31;
    float *__restrict__ Mf = Lf;
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
    named_sync(kBarSolve, kThreads);
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        if (w < 4 - d) {
            const int i = d + w, j = w;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int k = j; k < i; ++k)
                warp_gemm16(Mf + 16 * i * LP + 16 * k, LP, Nf + 16 * k * LP + 16 * j, LP, acc, lane);
            warp_store16(Nf + 16 * i * LP + 16 * j, LP, acc, lane, -1.f);
        }
        named_sync(kBarSolve, kThreads);
    }
}

struct SolveParams {
    const float *log_alpha, *beta;
    const int4 *plan;  // per chunk: sequence, first token, tokens, index within the sequence
    int32_t *ctl;      // [0] status, [1] number of chunks
    int H;
    __nv_bfloat16 *Tout;  // [chunks * H][2][64][64]: T' then A^T per unit
    float *Gout;          // [chunks * H][256]: g, gamma, kdec, form flag per unit
};

__global__ void __launch_bounds__(kThreads, 2)
tc_solve_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const SolveParams p) {
    if (p.ctl[0] != GDR_OK) return;
    const int n_units = p.ctl[1] * p.H;
    const int n_pairs = (n_units + 1) / 2;
    if ((int)blockIdx.x >= n_pairs) return;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM_SLOT);
    volatile int *fail = reinterpret_cast<volatile int *>(sm + OFF_FAIL);
    float *__restrict__ Lf = reinterpret_cast<float *>(sm + OFF_LF);
    float *__restrict__ Nf = reinterpret_cast<float *>(sm + OFF_NF);
    float *__restrict__ gates = reinterpret_cast<float *>(sm + OFF_GATE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // unit u -> (chunk, head); the second unit of an odd last pair repeats the first
    auto unit_of = [&](int pair, int which) {
        const int u = 2 * pair + which;
        return u < n_units ? u : 2 * pair;
    };
    auto load_pair = [&](int pair) {  // one thread
        mbar_arrive_expect_tx(bar(B_FULL), 8 * 8192);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const int u = unit_of(pair, which);
            const int4 pl = p.plan[u / p.H];
            const int h = u % p.H;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t blk = sbase + OFF_K + b * 32768 + which * 8192;
                tma_load_3d(blk, &map_k, bar(B_FULL), 64 * b, h, pl.y);
                tma_load_3d(blk + 16384, &map_q, bar(B_FULL), 64 * b, h, pl.y);
            }
        }
    };

    if (tid == 0) {
        mbar_init(bar(B_FULL), 1);
        mbar_init(bar(B_MMA), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
        *fail = 0;
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);

    if (tid == 0) load_pair(blockIdx.x);
    int it = 0;
    for (int pair = blockIdx.x; pair < n_pairs; pair += gridDim.x, ++it) {
        // ---- gates of both units (warp 0: unit a, warp 1: unit b), by the shared scan
        if (warp < 2) {
            const int u = 2 * pair + warp;
            float *g = gates + warp * G_UNIT;
            if (u < n_units) {
                const int4 pl = p.plan[u / p.H];
                const int h = u % p.H, len = pl.z;
                float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
                if (2 * lane < len) {
                    const size_t off = (size_t)(pl.y + 2 * lane) * p.H + h;
                    a0 = p.log_alpha[off];
                    b0 = p.beta[off];
                }
                if (2 * lane + 1 < len) {
                    const size_t off = (size_t)(pl.y + 2 * lane + 1) * p.H + h;
                    a1 = p.log_alpha[off];
                    b1 = p.beta[off];
                }
                const ChunkScan sc = chunk_scan(a0, a1, lane);
                g[G_G + 2 * lane] = sc.g0;
                g[G_G + 2 * lane + 1] = sc.g1;
                g[G_GAM + 2 * lane] = fast_exp(sc.g0);
                g[G_GAM + 2 * lane + 1] = fast_exp(sc.g1);
                g[G_GINV + 2 * lane] = fast_exp(-sc.g0);
                g[G_GINV + 2 * lane + 1] = fast_exp(-sc.g1);
                g[G_BETA + 2 * lane] = b0;
                g[G_BETA + 2 * lane + 1] = b1;
                g[G_KDEC + 2 * lane] = fast_exp(sc.g_last - sc.g0);
                g[G_KDEC + 2 * lane + 1] = fast_exp(sc.g_last - sc.g1);
            }
        }
        // ---- the pair's keys and queries have landed: one MMA chain for both units
        if (tid == 0) {
            bool ok = mbar_wait(bar(B_FULL), it & 1);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = sbase + OFF_K + (kk >> 2) * 32768 + (kk & 3) * 32;
                    mma_bf16(tmem, sw128_desc(off, 16, 1024), sw128_desc(off, 16, 1024),
                             idesc_bf16(128, 256, 0, 0), kk > 0);
                }
                mma_commit(bar(B_MMA));
                ok = mbar_wait(bar(B_MMA), it & 1);
            }
            if (ok && pair + (int)gridDim.x < n_pairs) load_pair(pair + gridDim.x);  // stage free
            if (!ok) *fail = 1;
        }
        __syncthreads();
        if (*fail) break;
        tc_fence_after();

#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            const int u = 2 * pair + which;
            if (u >= n_units) break;  // uniform over the CTA
            const float *g = gates + which * G_UNIT;
            const bool ratio = g[G_G + C - 1] > kRatioSafeLogDecay;
            {
                float *go = p.Gout + (size_t)u * 256;
                if (tid < C) {
                    go[tid] = g[G_G + tid];
                    go[64 + tid] = g[G_GAM + tid];
                    go[128 + tid] = g[G_KDEC + tid];
                } else {
                    go[192 + tid - C] = (tid == C) ? (ratio ? 1.f : 0.f) : 0.f;
                }
            }
            // ---- L (fp32, strictly lower) from this unit's K K^T block, and its A^T
            if ((warp >> 1) == which) {
                const int t = 32 * (warp & 1) + lane;
                const float gt = ratio ? g[G_GAM + t] : g[G_G + t];
                const float bt = g[G_BETA + t];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (hh > (warp & 1)) break;  // columns >= 32 are above the diagonal of rows < 32
                    float v[32];
                    tmem_load32(lane_base + 64 * which + 32 * hh, v);
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) {
                        const int i = 32 * hh + ii;
                        const float dec = ratio ? gt * g[G_GINV + i] : fast_exp(gt - g[G_G + i]);
                        if (i < t) Lf[t * LP + i] = bt * dec * v[ii];
                    }
                }
                // row i = t of A^T: key i against queries tq >= i
                const float gi = g[G_G + t];
                const float ginv_c = g[G_GINV + C - 1];
                uint4 *dst = reinterpret_cast<uint4 *>(p.Tout + ((size_t)(2 * u + 1) * C + t) * C);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float v[32];
                    if (hh < (warp & 1)) {  // rows i >= 32: queries tq < 32 are all masked
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) v[ii] = 0.f;
                    } else {
                        tmem_load32(lane_base + 128 + 64 * which + 32 * hh, v);
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) {
                            const int tq = 32 * hh + ii;
                            const float dec = ratio ? ginv_c : fast_exp(g[G_G + tq] - gi);
                            v[ii] = (tq >= t) ? v[ii] * dec : 0.f;
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        dst[4 * hh + jj] = make_uint4(pack_bf16x2(v[8 * jj], v[8 * jj + 1]),
                                                      pack_bf16x2(v[8 * jj + 2], v[8 * jj + 3]),
                                                      pack_bf16x2(v[8 * jj + 4], v[8 * jj + 5]),
                                                      pack_bf16x2(v[8 * jj + 6], v[8 * jj + 7]));
                }
            }
            tc_fence_before();  // the TMEM reads are done before the next pair's MMA is issued
            named_sync(kBarSolve, kThreads);
            unit_lower_inverse(Lf, Nf, tid);
            // ---- T' = diag(kdec) (I + L)^{-1} diag(beta) (ratio form; no kdec otherwise), bf16
            {
                const int t = tid >> 1, hh = tid & 1;
                const float kd = ratio ? g[G_KDEC + t] : 1.f;
                float x[32];
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * hh + ii;
                    x[ii] = (i <= t) ? Nf[t * LP + i] * g[G_BETA + i] * kd : 0.f;
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.Tout + ((size_t)(2 * u) * C + t) * C + 32 * hh);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    dst[jj] = make_uint4(pack_bf16x2(x[8 * jj], x[8 * jj + 1]),
                                         pack_bf16x2(x[8 * jj + 2], x[8 * jj + 3]),
                                         pack_bf16x2(x[8 * jj + 4], x[8 * jj + 5]),
                                         pack_bf16x2(x[8 * jj + 6], x[8 * jj + 7]));
            }
            named_sync(kBarSolve, kThreads);  // Nf and Lf free for the next unit
        }
    }

    __syncthreads();
    if (*fail && tid == 0) {
        atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
        mma_commit(bar(B_DRAIN));  // issued MMAs and loads land before TMEM and smem go away
        mbar_wait(bar(B_DRAIN), 0);
        mbar_wait(bar(B_FULL), it & 1);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

namespace tc {

int launch_solve_tc(const PrefillArgs &a, const WsLayout &L, const CUtensorMap &map_q,
                    const CUtensorMap &map_k) {
    SolveParams p;
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.plan = reinterpret_cast<const int4 *>(a.ws + L.plan);
    p.ctl = reinterpret_cast<int32_t *>(a.ws + L.ctl);
    p.H = a.H;
    p.Tout = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.T);
    p.Gout = reinterpret_cast<float *>(a.ws + L.G);
    if (cudaFuncSetAttribute(tc_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int64_t pairs = (L.max_chunks * a.H + 1) / 2;  // upper bound; the kernel reads the count
    const int64_t grid = pairs < 2 * (int64_t)sms ? pairs : 2 * (int64_t)sms;
    tc_solve_kernel<<<(unsigned)grid, kThreads, SMEM_BYTES, a.stream>>>(map_q, map_k, p);
    return cuda_status(cudaGetLastError());
}

}  // namespace tc
}  // namespace gdr
