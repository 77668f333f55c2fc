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
// so that the chain kernel uses the same values and the same form. (The two forms are
// described in prefill_tc.cu; they differ only in where the decay factors are applied.)
//
// Mapping. A CTA of 8 warps takes units two at a time; two CTAs share an SM. One
// tcgen05.mma chain forms [K_a; K_b] [K_a; K_b; Q_a; Q_b]^T (M = 128, N = 256, K = d_k =
// 128) in TMEM from TMA-loaded bf16 tiles: its diagonal 64x64 blocks are the units' K K^T
// and K Q^T. All 8 warps read them out at once (warps 0-1: L of unit a from TMEM lanes
// 0-63; 2-3: L of unit b, lanes 64-127; 4-5 and 6-7: A^T of a and b), then warp 0
// inverts unit a while warp 4 inverts unit b, and all 8 warps write T'. The inverse is
// fp32 on the CUDA cores in 16x16 blocks, by one warp and without barriers: the diagonal
// blocks by forward substitution, the others with warp-level TF32 products. While a
// pair is solved, the next pair's keys and queries are loading and its decay gates are
// in flight to registers.
#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace sm100;
using namespace tc;

constexpr int C = kChunk;
constexpr int kThreads = 256;
// A 16x16 fp32 block is stored row-major with its columns permuted per row: element
// (r, c) at r*16 + (c ^ sw(r)), sw(r) = 8*bit1(r) + 4*bit2(r). The permutation moves
// groups of four columns, so row segments of 2 and 4 stay contiguous, and it makes both
// fragment reads of the m16n8k8 TF32 MMA -- rows g, columns q (A) and rows q, columns g
// (B), g < 8, q < 4 -- fall on 32 different banks.
__host__ __device__ constexpr int sw(int r) { return (((r >> 1) & 1) << 3) | (((r >> 2) & 1) << 2); }
__host__ __device__ constexpr int el(int r, int c) { return r * 16 + (c ^ sw(r)); }
constexpr int BF = 256;             // floats per block
// Lower-triangular 4x4 arrangement of 16x16 blocks: block (i, k), k <= i, at index
// i(i+1)/2 + k. A unit has sixteen block slots: the ten of L, where M_ik = N_ii L_ik
// replaces L_ik (i > k) and N_ii replaces L_ii, then six for N_ik (i > k). Slots are
// BF + 4 floats apart (16-byte aligned) so that the four diagonal blocks, read at the
// same element by the forward substitution, start on different banks.
constexpr int BS = BF + 4;
__host__ __device__ constexpr int blk(int i, int k) { return (i * (i + 1) / 2 + k) * BS; }
__host__ __device__ constexpr int nblk(int i, int k) {  // N_ik, i > k
    return (10 + (i - k == 1 ? k : (i - k == 2 ? 3 + k : 5))) * BS;
}
constexpr int UNIT_FLOATS = 16 * BS;

// per d_k half b (32 KB): K_a | K_b | Q_a | Q_b, 8 KB each; rows 0-127 are the MMA's A
// operand, rows 0-255 its B operand
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_LN = 65536;                             // two units' L, N blocks
constexpr uint32_t OFF_GATE = OFF_LN + 2 * UNIT_FLOATS * 4;
constexpr int G_G = 0, G_GAM = 64, G_GINV = 128, G_BETA = 192, G_KDEC = 256, G_UNIT = 320;
constexpr uint32_t OFF_BAR = OFF_GATE + 2 * G_UNIT * 4;  // per unit: g, gamma, 1/gamma, beta, kdec
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert((SMEM_BYTES + 1024) * 2 <= 228 * 1024, "two CTAs per SM");
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
    // not volatile: independent products may interleave (the outputs keep it alive)
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d (+)= A * B for 16x16 blocks A and B (layout el); d holds the result's two 16x8
// halves in the m16n8 accumulator layout.
__device__ __forceinline__ void warp_gemm16(const float *__restrict__ A, const float *__restrict__ B,
                                            float (&d)[2][4], int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a[4] = {to_tf32(A[el(g, 8 * ks + q)]), to_tf32(A[el(g + 8, 8 * ks + q)]),
                               to_tf32(A[el(g, 8 * ks + q + 4)]), to_tf32(A[el(g + 8, 8 * ks + q + 4)])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {to_tf32(B[el(8 * ks + q, 8 * nt + g)]),
                                   to_tf32(B[el(8 * ks + q + 4, 8 * nt + g)])};
            mma_tf32_16x8x8(d[nt], a, b);
        }
    }
}

// M = scale * d for a 16x16 block M, d in the accumulator layout.
__device__ __forceinline__ void warp_store16(float *__restrict__ M, const float (&d)[2][4], int lane,
                                             float scale) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2 *>(M + el(g, 8 * nt + 2 * q)) = make_float2(scale * d[nt][0], scale * d[nt][1]);
        *reinterpret_cast<float2 *>(M + el(g + 8, 8 * nt + 2 * q)) =
            make_float2(scale * d[nt][2], scale * d[nt][3]);
    }
}

// N = (I + L)^{-1} for the strictly lower-triangular 64x64 L held as blocks in U (see
// blk, nblk), by one warp:
//   1. N_ii by forward substitution: lane l takes columns 2(l%8), 2(l%8)+1 of block l/8.
//   2. M_ik = N_ii L_ik for the six blocks below the diagonal (over L_ik).
//   3. N_ij = -sum_{k=j}^{i-1} M_ik N_kj by distance from the diagonal, with the partial
//      sums that do not need the previous level formed one level early, so that the
//      dependent chain is four block products long.
__device__ __forceinline__ void warp_lower_inverse(float *__restrict__ U, int lane) {
    {
        const int b = lane >> 3, c0 = 2 * (lane & 7);
        float *D = U + blk(b, b);
        float x0[16], x1[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            x0[r] = (r == c0) ? 1.f : 0.f;
            x1[r] = (r == c0 + 1) ? 1.f : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 15; ++k) {
            const float a0 = x0[k], a1 = x1[k];
#pragma unroll
            for (int r = k + 1; r < 16; ++r) {
                const float l = D[el(r, k)];
                x0[r] = fmaf(-l, a0, x0[r]);
                x1[r] = fmaf(-l, a1, x1[r]);
            }
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r) *reinterpret_cast<float2 *>(D + el(r, c0)) = make_float2(x0[r], x1[r]);
        __syncwarp();
    }
    typedef float Acc[2][4];
    auto zero = [](Acc &a) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) a[nt][e] = 0.f;
    };
    Acc a0, a1, a2, a3, a4, a5;
    // M_10, M_21, M_32, M_20, M_31, M_30
    zero(a0); zero(a1); zero(a2); zero(a3); zero(a4); zero(a5);
    warp_gemm16(U + blk(1, 1), U + blk(1, 0), a0, lane);
    warp_gemm16(U + blk(2, 2), U + blk(2, 1), a1, lane);
    warp_gemm16(U + blk(3, 3), U + blk(3, 2), a2, lane);
    warp_gemm16(U + blk(2, 2), U + blk(2, 0), a3, lane);
    warp_gemm16(U + blk(3, 3), U + blk(3, 1), a4, lane);
    warp_gemm16(U + blk(3, 3), U + blk(3, 0), a5, lane);
    __syncwarp();
    warp_store16(U + blk(1, 0), a0, lane, 1.f);
    warp_store16(U + blk(2, 1), a1, lane, 1.f);
    warp_store16(U + blk(3, 2), a2, lane, 1.f);
    warp_store16(U + blk(2, 0), a3, lane, 1.f);
    warp_store16(U + blk(3, 1), a4, lane, 1.f);
    warp_store16(U + blk(3, 0), a5, lane, 1.f);
    __syncwarp();
    // level 1: N_10, N_21, N_32; partial sums P20 = M_20 N_00, P31 = M_31 N_11, P30 = M_30 N_00
    zero(a0); zero(a1); zero(a2); zero(a3); zero(a4); zero(a5);
    warp_gemm16(U + blk(1, 0), U + blk(0, 0), a0, lane);
    warp_gemm16(U + blk(2, 1), U + blk(1, 1), a1, lane);
    warp_gemm16(U + blk(3, 2), U + blk(2, 2), a2, lane);
    warp_gemm16(U + blk(2, 0), U + blk(0, 0), a3, lane);
    warp_gemm16(U + blk(3, 1), U + blk(1, 1), a4, lane);
    warp_gemm16(U + blk(3, 0), U + blk(0, 0), a5, lane);
    warp_store16(U + nblk(1, 0), a0, lane, -1.f);
    warp_store16(U + nblk(2, 1), a1, lane, -1.f);
    warp_store16(U + nblk(3, 2), a2, lane, -1.f);
    __syncwarp();
    // level 2: N_20 = -(P20 + M_21 N_10), N_31 = -(P31 + M_32 N_21); P30 += M_31 N_10
    warp_gemm16(U + blk(2, 1), U + nblk(1, 0), a3, lane);
    warp_gemm16(U + blk(3, 2), U + nblk(2, 1), a4, lane);
    warp_gemm16(U + blk(3, 1), U + nblk(1, 0), a5, lane);
    warp_store16(U + nblk(2, 0), a3, lane, -1.f);
    warp_store16(U + nblk(3, 1), a4, lane, -1.f);
    __syncwarp();
    // level 3: N_30 = -(P30 + M_32 N_20)
    warp_gemm16(U + blk(3, 2), U + nblk(2, 0), a5, lane);
    warp_store16(U + nblk(3, 0), a5, lane, -1.f);
    __syncwarp();
}

// Element (t, i), i <= t, of N = (I + L)^{-1} in the unit's block slots.
__device__ __forceinline__ float n_entry(const float *__restrict__ U, int t, int i) {
    const int bt = t >> 4, bi = i >> 4;
    const int base = bt == bi ? blk(bt, bt) : nblk(bt, bi);
    return U[base + el(t & 15, i & 15)];
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
    float *__restrict__ gates = reinterpret_cast<float *>(sm + OFF_GATE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // unit u -> (chunk, head); the second unit of an odd last pair repeats the first
    auto unit_of = [&](int pair, int which) {
        const int u = 2 * pair + which;
        return u < n_units ? u : 2 * pair;
    };
    int loads_issued = 0, loads_landed = 0;  // (thread 0) for the drain after an abort
    auto load_pair = [&](int pair) {  // one thread
        ++loads_issued;
        mbar_arrive_expect_tx(bar(B_FULL), 8 * 8192);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const int u = unit_of(pair, which);
            const int4 pl = p.plan[u / p.H];
            const int h = u % p.H;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t blkaddr = sbase + OFF_K + b * 32768 + which * 8192;
                tma_load_3d(blkaddr, &map_k, bar(B_FULL), 64 * b, h, pl.y);
                tma_load_3d(blkaddr + 16384, &map_q, bar(B_FULL), 64 * b, h, pl.y);
            }
        }
    };
    // decay gates of one unit of `pair` (warp 0: unit a, warp 1: unit b), into registers
    float ga0 = 0.f, ga1 = 0.f, gb0 = 0.f, gb1 = 0.f;
    auto fetch_gates = [&](int pair) {
        ga0 = ga1 = gb0 = gb1 = 0.f;
        const int u = 2 * pair + warp;
        if (u < n_units) {
            const int4 pl = p.plan[u / p.H];
            const int h = u % p.H, len = pl.z;
            if (2 * lane < len) {
                const size_t off = (size_t)(pl.y + 2 * lane) * p.H + h;
                ga0 = p.log_alpha[off];
                gb0 = p.beta[off];
            }
            if (2 * lane + 1 < len) {
                const size_t off = (size_t)(pl.y + 2 * lane + 1) * p.H + h;
                ga1 = p.log_alpha[off];
                gb1 = p.beta[off];
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
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

    // the Gram chain of `pair` (thread 0), once its keys and queries have landed
    auto issue_gram = [&](int it_) -> bool {
        if (!mbar_wait(bar(B_FULL), it_ & 1)) return false;
        ++loads_landed;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = sbase + OFF_K + (kk >> 2) * 32768 + (kk & 3) * 32;
            mma_bf16(tmem, sw128_desc(off, 16, 1024), sw128_desc(off, 16, 1024), idesc_bf16(128, 256, 0, 0),
                     kk > 0);
        }
        mma_commit(bar(B_MMA));
        return true;
    };
    if (tid == 0) {
        load_pair(blockIdx.x);
        if (!issue_gram(0)) *fail = 1;
    }
    if (warp < 2) fetch_gates(blockIdx.x);
    int it = 0;
    for (int pair = blockIdx.x; pair < n_pairs; pair += gridDim.x, ++it) {
        const int next = pair + (int)gridDim.x;
        // ---- gates of both units (warp 0: unit a, warp 1: unit b) by the shared scan;
        // then the next pair's gates are fetched
        if (warp < 2) {
            float *g = gates + warp * G_UNIT;
            const ChunkScan sc = chunk_scan(ga0, ga1, lane);
            g[G_G + 2 * lane] = sc.g0;
            g[G_G + 2 * lane + 1] = sc.g1;
            g[G_GAM + 2 * lane] = fast_exp(sc.g0);
            g[G_GAM + 2 * lane + 1] = fast_exp(sc.g1);
            g[G_GINV + 2 * lane] = fast_exp(-sc.g0);
            g[G_GINV + 2 * lane + 1] = fast_exp(-sc.g1);
            g[G_BETA + 2 * lane] = gb0;
            g[G_BETA + 2 * lane + 1] = gb1;
            g[G_KDEC + 2 * lane] = fast_exp(sc.g_last - sc.g0);
            g[G_KDEC + 2 * lane + 1] = fast_exp(sc.g_last - sc.g1);
            if (next < n_pairs) fetch_gates(next);
        }
        // ---- the pair's Gram chain (issued before) has completed: its stage takes the next pair
        if (tid == 0) {
            if (*fail == 0 && mbar_wait(bar(B_MMA), it & 1)) {
                if (next < n_pairs) load_pair(next);
            } else {
                *fail = 1;
            }
        }
        __syncthreads();
        if (*fail) break;
        tc_fence_after();

        // ---- read-out: L blocks of both units (warps 0-3), A^T and the factors (warps 4-7)
        {
            const int which = (warp >> 1) & 1;  // unit of this warp's TMEM lanes
            const int u = 2 * pair + which;
            const float *g = gates + which * G_UNIT;
            const bool ratio = g[G_G + C - 1] > kRatioSafeLogDecay;
            const int t = 32 * (warp & 1) + lane;  // token row (TMEM lane 64 which + t)
            if (u < n_units) {
                if (warp < 4) {
                    // L_ti = beta_t Gamma_ti k_t.k_i (i < t) into the unit's blocks
                    float *Lb = reinterpret_cast<float *>(sm + OFF_LN) + which * UNIT_FLOATS;
                    const float gt = ratio ? g[G_GAM + t] : g[G_G + t];
                    const float bt = g[G_BETA + t];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh > (warp & 1)) break;  // columns >= 32 lie above rows < 32
                        float v[32], f[32];
                        tmem_load32(lane_base + 64 * which + 32 * hh, v);
                        const float4 *gv = reinterpret_cast<const float4 *>(g + (ratio ? G_GINV : G_G) + 32 * hh);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 x = gv[j];
                            f[4 * j] = x.x; f[4 * j + 1] = x.y; f[4 * j + 2] = x.z; f[4 * j + 3] = x.w;
                        }
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) {
                            const int i = 32 * hh + ii;
                            const float dec = ratio ? gt * f[ii] : fast_exp(gt - f[ii]);
                            v[ii] = (i < t) ? bt * dec * v[ii] : 0.f;
                        }
                        // whole 16-wide rows of the blocks left of and on the diagonal (the
                        // zeros on and above the diagonal are never read)
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const int ib = 2 * hh + m;
                            if (ib <= (t >> 4)) {
                                float *blockp = Lb + blk(t >> 4, ib);
#pragma unroll
                                for (int e4 = 0; e4 < 4; ++e4)
                                    *reinterpret_cast<float4 *>(blockp + el(t & 15, 4 * e4)) =
                                        make_float4(v[16 * m + 4 * e4], v[16 * m + 4 * e4 + 1],
                                                    v[16 * m + 4 * e4 + 2], v[16 * m + 4 * e4 + 3]);
                            }
                        }
                    }
                } else {
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
                    // the unit's decay factors for the chain kernel: g and gamma (threads
                    // t < 32), kdec and the form flag (t >= 32), two tokens each
                    float *go = p.Gout + (size_t)u * 256;
                    if (t < 32) {
                        go[2 * t] = g[G_G + 2 * t];
                        go[2 * t + 1] = g[G_G + 2 * t + 1];
                        go[64 + 2 * t] = g[G_GAM + 2 * t];
                        go[64 + 2 * t + 1] = g[G_GAM + 2 * t + 1];
                    } else {
                        const int t2 = t - 32;
                        go[128 + 2 * t2] = g[G_KDEC + 2 * t2];
                        go[128 + 2 * t2 + 1] = g[G_KDEC + 2 * t2 + 1];
                        go[192 + 2 * t2] = (t2 == 0) ? (ratio ? 1.f : 0.f) : 0.f;
                        go[192 + 2 * t2 + 1] = 0.f;
                    }
                }
            }
        }
        tc_fence_before();  // the TMEM reads are done before the next pair's MMA is issued
        __syncthreads();
        if (tid == 0 && next < n_pairs && !issue_gram(it + 1)) *fail = 1;

        // ---- warp 0 inverts unit a, warp 4 unit b
        if ((warp & 3) == 0 && 2 * pair + (warp >> 2) < n_units)
            warp_lower_inverse(reinterpret_cast<float *>(sm + OFF_LN) + (warp >> 2) * UNIT_FLOATS, lane);
        __syncthreads();
        // ---- T' = diag(kdec) (I + L)^{-1} diag(beta) (ratio form; no kdec otherwise), bf16:
        // warps 0-3 unit a, warps 4-7 unit b, one half row per thread
        {
            const int which = warp >> 2, u = 2 * pair + which;
            if (u < n_units) {
                const float *U = reinterpret_cast<const float *>(sm + OFF_LN) + which * UNIT_FLOATS;
                const float *g = gates + which * G_UNIT;
                const bool ratio = g[G_G + C - 1] > kRatioSafeLogDecay;
                const int gtid = tid & 127, t = gtid >> 1, hh = gtid & 1;
                const float kd = ratio ? g[G_KDEC + t] : 1.f;
                float x[32], bv[32];
                const float4 *bp = reinterpret_cast<const float4 *>(g + G_BETA + 32 * hh);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 b4 = bp[j];
                    bv[4 * j] = b4.x; bv[4 * j + 1] = b4.y; bv[4 * j + 2] = b4.z; bv[4 * j + 3] = b4.w;
                }
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = 32 * hh + ii;
                    x[ii] = (i <= t) ? n_entry(U, t, i) * bv[ii] * kd : 0.f;
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.Tout + ((size_t)(2 * u) * C + t) * C + 32 * hh);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    dst[jj] = make_uint4(pack_bf16x2(x[8 * jj], x[8 * jj + 1]),
                                         pack_bf16x2(x[8 * jj + 2], x[8 * jj + 3]),
                                         pack_bf16x2(x[8 * jj + 4], x[8 * jj + 5]),
                                         pack_bf16x2(x[8 * jj + 6], x[8 * jj + 7]));
            }
        }
        __syncthreads();  // blocks and gates free for the next pair
    }

    __syncthreads();
    if (*fail && tid == 0) {
        atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
        mma_commit(bar(B_DRAIN));  // issued MMAs and loads land before TMEM and smem go away
        mbar_wait(bar(B_DRAIN), 0);
        if (loads_issued > loads_landed) mbar_wait(bar(B_FULL), loads_landed & 1);
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
    const int64_t grid = pairs < 2 * (int64_t)sms ? pairs : 2 * (int64_t)sms;  // two CTAs per SM
    tc_solve_kernel<<<(unsigned)grid, kThreads, SMEM_BYTES, a.stream>>>(map_q, map_k, p);
    return cuda_status(cudaGetLastError());
}

}  // namespace tc
}  // namespace gdr
