// solve_tc.cuh -- the chunk-parallel half of the tensor-core prefill: for every
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
// Mapping. One CTA per SM walks unit pairs as a pipeline of warp roles joined by
// mbarriers:
//   warp 4      loads a pair's keys and queries by TMA into one of two stage slots and
//               issues its Gram chain [K_a; K_b] [K_a; K_b; Q_a; Q_b]^T (tcgen05, M = 128,
//               N = 256, K = d_k = 128) into one of two TMEM slots; the diagonal 64x64
//               blocks are each unit's K K^T and K Q^T;
//   warps 0-3   read a TMEM slot out (warps 0-1: unit a, TMEM lanes 0-63; 2-3: unit b,
//               lanes 64-127): the unit's decay factors, its decayed L into fp32 16x16
//               blocks of one of four solver slots, and its masked, decayed A^T straight
//               to the workspace;
//   warps 5-8   one solver warp per slot: the inverse of I + L, then T' in bf16.
// The inverse is fp32 on the CUDA cores in 16x16 blocks, by one warp and without
// barriers: the diagonal blocks by forward substitution, the others with warp-level TF32
// products.
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace solve {

using namespace sm100;
using namespace tc;

constexpr int C = kChunk;
constexpr int kThreads = 288;  // 9 warps
constexpr int kProducerWarp = 4, kSolverWarp0 = 5, kSolvers = 4;
// fused launch only: one publisher warp per solver slot releases the slot's units
constexpr int kPublisherWarp0 = kSolverWarp0 + kSolvers;
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

// Stage slot (64 KB), per d_k half b (32 KB): K_a | K_b | Q_a | Q_b, 8 KB each; rows
// 0-127 are the Gram chain's A operand, rows 0-255 its B operand.
constexpr uint32_t STAGE = 65536;
constexpr uint32_t OFF_LS = 2 * STAGE;  // solver slots: blocks, then the unit's gates
constexpr int G_G = 0, G_GAM = 64, G_GINV = 128, G_BETA = 192, G_KDEC = 256, G_UNIT = 320;
constexpr uint32_t LSLOT = 18432;  // blocks, gates; 1024-aligned (its first 8 KB stage T')
static_assert(UNIT_FLOATS * 4 + G_UNIT * 4 <= LSLOT && UNIT_FLOATS * 4 >= 8192, "solver slot");
constexpr uint32_t OFF_BAR = OFF_LS + kSolvers * LSLOT;
enum {
    B_STF0 = 0, B_STF1,  // stage slot loaded                  (tx bytes)
    B_STE0, B_STE1,      // stage slot read by the Gram chain   (commit)
    B_TMF0, B_TMF1,      // TMEM slot holds a pair's Gram       (commit)
    B_TME0, B_TME1,      // TMEM slot read out                  (128 read-out arrivals)
    B_LF0, B_LF1, B_LF2, B_LF3,  // solver slot filled          (64 read-out arrivals)
    B_LE0, B_LE1, B_LE2, B_LE3,  // solver slot free again      (solver lane 0)
    B_PUB0, B_PUB1, B_PUB2, B_PUB3,      // fused: slot's unit stored        (32 solver lanes)
    B_PUBE0, B_PUBE1, B_PUBE2, B_PUBE3,  // fused: slot's unit published     (publisher)
    B_PID0, B_PID1, B_PID2, B_PID3, B_PID4, B_PID5, B_PID6, B_PID7,  // pair id k in ring[k % 8]
    B_DRAIN,
    B_COUNT
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t OFF_FAIL = OFF_TMEM_SLOT + 4;
constexpr uint32_t OFF_RING = OFF_FAIL + 16;  // int[8]: the pairs this CTA claimed
constexpr uint32_t SMEM_USED = OFF_RING + 32;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 232448 && LSLOT % 1024 == 0 && OFF_LS % 1024 == 0, "shared memory");
constexpr uint32_t TM_COLS = 512;  // two 256-column slots

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

// T' = diag(kd) N diag(beta) in bf16 (kd = kdec in the ratio form, else 1), by one warp,
// into a 128-byte-swizzled [64][64] tile at `tile` (the layout a TMA store reads) that
// overlays the first 8 KB of U: N's ten blocks are read into registers in the m16n8
// accumulator layout first, the blocks above the diagonal are zero.
__device__ __forceinline__ void warp_stage_tprime(float *__restrict__ U, const float *__restrict__ g,
                                                  bool ratio, unsigned char *tile, int lane) {
    const int gq = lane >> 2, q = lane & 3;
    float n[10][2][4];
#pragma unroll
    for (int bt = 0; bt < 4; ++bt)
#pragma unroll
        for (int bi = 0; bi <= bt; ++bi) {
            const float *B = U + (bt == bi ? blk(bt, bt) : nblk(bt, bi));
            const int idx = bt * (bt + 1) / 2 + bi;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 lo = *reinterpret_cast<const float2 *>(B + el(gq, 8 * nt + 2 * q));
                const float2 hi = *reinterpret_cast<const float2 *>(B + el(gq + 8, 8 * nt + 2 * q));
                n[idx][nt][0] = lo.x; n[idx][nt][1] = lo.y; n[idx][nt][2] = hi.x; n[idx][nt][3] = hi.y;
            }
        }
    __syncwarp();
#pragma unroll
    for (int bt = 0; bt < 4; ++bt) {
        float kd[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) kd[h] = ratio ? g[G_KDEC + 16 * bt + gq + 8 * h] : 1.f;
#pragma unroll
        for (int bi = 0; bi < 4; ++bi)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int i0 = 16 * bi + 8 * nt + 2 * q;  // columns i0, i0 + 1
                const float b0 = g[G_BETA + i0], b1 = g[G_BETA + i0 + 1];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = 16 * bt + gq + 8 * h;
                    float x0 = 0.f, x1 = 0.f;
                    if (bi <= bt) {
                        const int idx = bt * (bt + 1) / 2 + bi;
                        // within a diagonal block the entries above the diagonal are zero
                        x0 = (i0 <= t) ? n[idx][nt][2 * h] * b0 * kd[h] : 0.f;
                        x1 = (i0 + 1 <= t) ? n[idx][nt][2 * h + 1] * b1 * kd[h] : 0.f;
                    }
                    *reinterpret_cast<uint32_t *>(tile + t * 128 + ((((i0 >> 3) ^ t) & 7) << 4) + (i0 & 7) * 2) =
                        pack_bf16x2(x0, x1);
                }
            }
    }
}

struct SolveParams {
    const float *log_alpha, *beta;
    const int4 *plan;  // per chunk: sequence, first token, tokens, index within the sequence
    int32_t *ctl;      // [0] status, [1] number of chunks, [2 + f] first chunk of phase f
    int H;
    int phase;            // the units of this phase's chunks are solved
    // fused launch (beside the chain): units in chunk-major order over `seqs` sequences of
    // `seq_chunks` chunks each, and a ready flag per unit, set once its results are stored
    int seqs, seq_chunks;
    int32_t *flags;
    int32_t *pair_counter;  // pairs are claimed from it at run time (zeroed by the plan)
    __nv_bfloat16 *Tout;  // [chunks * H][2][64][64]: T' then A^T per unit
    float *Gout;          // [chunks * H][256]: g, gamma, kdec, form flag per unit
};

// The solve on CTA `cta` of `ncta`. kFused: the CTA shares a cooperative launch with the
// chain (which may have more warps: warps past the ninth only pass the block barriers),
// takes the units in chunk-major order so that the chains find their chunks solved in
// the order they need them, and publishes each unit with a release of its flag.
template <bool kFused>
__device__ __forceinline__ void solve_body(const CUtensorMap &map_q, const CUtensorMap &map_k,
                                           const CUtensorMap &map_t, const SolveParams &p, int cta,
                                           int ncta) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM_SLOT);
    volatile int *fail = reinterpret_cast<volatile int *>(sm + OFF_FAIL);
    auto lslot = [&](int s) { return reinterpret_cast<float *>(sm + OFF_LS + s * LSLOT); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_STF0 + i), 1);
            mbar_init(bar(B_STE0 + i), 1);
            mbar_init(bar(B_TMF0 + i), 1);
            mbar_init(bar(B_TME0 + i), 128);
        }
        for (int i = 0; i < kSolvers; ++i) {
            mbar_init(bar(B_LF0 + i), 64);
            mbar_init(bar(B_LE0 + i), 1);
        }
        for (int i = 0; i < kSolvers; ++i) {
            mbar_init(bar(B_PUB0 + i), 32);
            mbar_init(bar(B_PUBE0 + i), 1);
        }
        for (int i = 0; i < 8; ++i) mbar_init(bar(B_PID0 + i), 1);
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
        *fail = 0;
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_t);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Everything above overlaps the tail of the planning kernel (programmatic launch);
    // the plan and the status word are read only after it has completed.
    griddep_wait();
    griddep_launch_dependents();
    // this phase's units are u0 + [0, n_units); local indices below, u0 added for addressing
    const int u0 = kFused ? 0 : p.ctl[2 + p.phase] * p.H;
    const int n_units =
        p.ctl[0] == GDR_OK ? (kFused ? p.ctl[1] * p.H : p.ctl[3 + p.phase] * p.H - u0) : 0;
    const int n_pairs = (n_units + 1) / 2;
    // The CTA's k-th pair, or -1 after its last. The producer claims pairs one at a time
    // from the call's counter, as its stage slots free up, so that faster CTAs take more
    // of them, and hands each on through ring[k % 8] and its barrier; -1 marks the end.
    // (The producer can be at most six pairs ahead of the slowest role, seven with the
    // second end mark, so a ring slot and its barrier phase are never reused while a
    // role still needs them.)
    volatile int *ring = reinterpret_cast<volatile int *>(sm + OFF_RING);
    auto pair_id = [&](int k) -> int {
        if (!mbar_wait(bar(B_PID0 + (k & 7)), (k >> 3) & 1)) {
            *fail = 1;
            return -1;
        }
        return ring[k & 7];
    };
    // the unit at local index x: the phase's units in order, or (fused) chunk j of
    // sequence n for head h at x = (j * seqs + n) * H + h
    auto unit_at = [&](int x) {
        if (!kFused) return u0 + x;
        const int h = x % p.H, r = x / p.H;
        return ((r % p.seqs) * p.seq_chunks + r / p.seqs) * p.H + h;
    };

    if (warp == kProducerWarp) {
        // ============================================================ loads and Gram chains
        if (lane == 0) {
            int loads = 0, landed = 0;
            for (int k = 0; !*fail; ++k) {
                // claim pair k once stage slot k % 2 is free (Gram k - 2 has read it), hand
                // it on, and load it
                const int sl = k & 1;
                if (k >= 2 && !mbar_wait(bar(B_STE0 + sl), ((k >> 1) - 1) & 1)) { *fail = 1; break; }
                int pr = n_pairs > 0 ? atomicAdd(p.pair_counter, 1) : n_pairs;
                if (pr >= n_pairs) pr = -1;
                ring[k & 7] = pr;
                mbar_arrive(bar(B_PID0 + (k & 7)));
                if (pr < 0) {
                    // the end, for pair k + 1 too: each solver and publisher walks every
                    // other pair, so half of them next ask for pair k + 1
                    ring[(k + 1) & 7] = -1;
                    mbar_arrive(bar(B_PID0 + ((k + 1) & 7)));
                }
                if (pr >= 0) {
                    mbar_arrive_expect_tx(bar(B_STF0 + sl), 8 * 8192);
                    ++loads;
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        int u = 2 * pr + which;
                        if (u >= n_units) u = 2 * pr;  // a missing unit b repeats a
                        u = unit_at(u);
                        const int4 pl = p.plan[u / p.H];
                        const int h = u % p.H;
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const uint32_t dst = sbase + sl * STAGE + b * 32768 + which * 8192;
                            tma_load_3d(dst, &map_k, bar(B_STF0 + sl), 64 * b, h, pl.y);
                            tma_load_3d(dst + 16384, &map_q, bar(B_STF0 + sl), 64 * b, h, pl.y);
                        }
                    }
                }
                if (k >= 1) {  // Gram of pair j = k - 1 into TMEM slot j % 2 (free once read out)
                    const int j = k - 1, sl = j & 1;
                    if (!mbar_wait(bar(B_STF0 + sl), (j >> 1) & 1)) { *fail = 1; break; }
                    ++landed;
                    if (j >= 2 && !mbar_wait(bar(B_TME0 + sl), ((j >> 1) - 1) & 1)) { *fail = 1; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = sbase + sl * STAGE + (kk >> 2) * 32768 + (kk & 3) * 32;
                        mma_bf16(tmem + 256 * sl, sw128_desc(off, 16, 1024), sw128_desc(off, 16, 1024),
                                 idesc_bf16(128, 256, 0, 0), kk > 0);
                    }
                    mma_commit(bar(B_STE0 + sl));
                    mma_commit(bar(B_TMF0 + sl));
                }
                if (pr < 0) break;
            }
            if (*fail) {  // issued MMAs and loads land before TMEM and shared memory go away
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0);
                for (int j = landed; j < loads; ++j) mbar_wait(bar(B_STF0 + (j & 1)), (j >> 1) & 1);
            }
        }
    } else if (warp < 4) {
        // ============================================================ read-out
        const int which = warp >> 1;          // unit a (0) or b (1) of each pair
        const int t = 32 * (warp & 1) + lane; // token row = TMEM lane 64 which + t
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        // decay gates of this warp pair's unit of pair k, into registers (warp 2 which)
        float ga0 = 0.f, ga1 = 0.f, gb0 = 0.f, gb1 = 0.f;
        auto fetch_gates = [&](int pr) {
            ga0 = ga1 = gb0 = gb1 = 0.f;
            const int u = 2 * pr + which;
            if (pr >= 0 && u < n_units) {
                const int ug = unit_at(u);
                const int4 pl = p.plan[ug / p.H];
                const int h = ug % p.H, len = pl.z;
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
        int pr = pair_id(0);
        if ((warp & 1) == 0) fetch_gates(pr);
        for (int k = 0; pr >= 0; ++k) {
            const int sl = k & 1;
            const int lu = 2 * k + which, ls = lu % kSolvers;  // local unit and its solver slot
            const bool exists = 2 * pr + which < n_units;
            const int u = unit_at(2 * pr + which);
            const int pr_next = pair_id(k + 1);  // handed on before the Gram of pair k
            float *U = lslot(ls);
            float *g = U + UNIT_FLOATS;
            bool ok = true;
            if (exists && lu >= kSolvers) ok = mbar_wait(bar(B_LE0 + ls), ((lu / kSolvers) - 1) & 1);
            if (!ok) *fail = 1;
            if ((warp & 1) == 0) {  // the unit's gates, by the shared scan; then the next pair's
                const ChunkScan sc = chunk_scan(ga0, ga1, lane);
                if (exists && ok) {
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
                }
                fetch_gates(pr_next);
            }
            named_sync(1 + which, 64);  // the gates are visible to both warps of the unit
            ok = mbar_wait(bar(B_TMF0 + sl), (k >> 1) & 1);
            if (!ok) *fail = 1;
            tc_fence_after();
            if (exists && ok && !*fail) {
                const bool ratio = g[G_G + C - 1] > kRatioSafeLogDecay;
                const uint32_t col = 256 * sl + 64 * which;
                // L_ti = beta_t Gamma_ti k_t.k_i (i < t), whole 16-wide block rows
                {
                    const float gt = ratio ? g[G_GAM + t] : g[G_G + t];
                    const float bt = g[G_BETA + t];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh > (warp & 1)) break;  // columns >= 32 lie above rows < 32
                        float v[32], f[32];
                        tmem_load32(lane_base + col + 32 * hh, v);
                        const float4 *gv = reinterpret_cast<const float4 *>(g + (ratio ? G_GINV : G_G) + 32 * hh);
#pragma unroll
                        for (int jv = 0; jv < 8; ++jv) {
                            const float4 x = gv[jv];
                            f[4 * jv] = x.x; f[4 * jv + 1] = x.y; f[4 * jv + 2] = x.z; f[4 * jv + 3] = x.w;
                        }
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) {
                            const int i = 32 * hh + ii;
                            const float dec = ratio ? gt * f[ii] : fast_exp(gt - f[ii]);
                            v[ii] = (i < t) ? bt * dec * v[ii] : 0.f;
                        }
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const int ib = 2 * hh + m;
                            if (ib <= (t >> 4)) {
                                float *blockp = U + blk(t >> 4, ib);
#pragma unroll
                                for (int e4 = 0; e4 < 4; ++e4)
                                    *reinterpret_cast<float4 *>(blockp + el(t & 15, 4 * e4)) =
                                        make_float4(v[16 * m + 4 * e4], v[16 * m + 4 * e4 + 1],
                                                    v[16 * m + 4 * e4 + 2], v[16 * m + 4 * e4 + 3]);
                            }
                        }
                    }
                }
                // row i = t of A^T: key i against queries tq >= i, straight to the workspace
                {
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
                            tmem_load32(lane_base + col + 128 + 32 * hh, v);
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
                // the unit's decay factors for the chain kernel: g and gamma (warp 2 which),
                // kdec and the form flag (warp 2 which + 1), two tokens per lane
                float *go = p.Gout + (size_t)u * 256;
                if ((warp & 1) == 0) {
                    *reinterpret_cast<float2 *>(go + 2 * lane) = make_float2(g[G_G + 2 * lane], g[G_G + 2 * lane + 1]);
                    *reinterpret_cast<float2 *>(go + 64 + 2 * lane) =
                        make_float2(g[G_GAM + 2 * lane], g[G_GAM + 2 * lane + 1]);
                } else {
                    *reinterpret_cast<float2 *>(go + 128 + 2 * lane) =
                        make_float2(g[G_KDEC + 2 * lane], g[G_KDEC + 2 * lane + 1]);
                    *reinterpret_cast<float2 *>(go + 192 + 2 * lane) =
                        make_float2(lane == 0 ? (ratio ? 1.f : 0.f) : 0.f, 0.f);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_TME0 + sl));              // the TMEM slot is read
            if (exists) mbar_arrive(bar(B_LF0 + ls));   // the solver slot is filled
            pr = pr_next;
        }
    } else if (warp >= kSolverWarp0 && warp < kSolverWarp0 + kSolvers) {
        // ============================================================ solvers
        const int sv = warp - kSolverWarp0;
        for (int lu = sv;; lu += kSolvers) {
            const int which = lu & 1, pr = pair_id(lu >> 1);
            if (pr < 0) break;
            if (2 * pr + which >= n_units) continue;  // the missing half of an odd last pair
            const int u = unit_at(2 * pr + which);
            if (!mbar_wait(bar(B_LF0 + sv), (lu / kSolvers) & 1)) { *fail = 1; break; }
            float *U = lslot(sv);
            const float *g = U + UNIT_FLOATS;
            warp_lower_inverse(U, lane);
            // T' = diag(kdec) (I + L)^{-1} diag(beta) (ratio form; no kdec otherwise), bf16,
            // staged over the slot and stored by TMA
            const bool ratio = g[G_G + C - 1] > kRatioSafeLogDecay;
            unsigned char *tile = reinterpret_cast<unsigned char *>(U);
            warp_stage_tprime(U, g, ratio, tile, lane);
            if (kFused) {
                // T' to the workspace by plain stores (16-byte segments, row-major), then to
                // the slot's publisher, whose gpu-scope release of the unit's flag covers
                // these stores and the read-out's A^T and factors (stored before B_LF)
                __syncwarp();
                uint4 *dst = reinterpret_cast<uint4 *>(p.Tout + (size_t)2 * u * C * C);
#pragma unroll 4
                for (int sg = lane; sg < C * 8; sg += 32) {
                    const int r = sg >> 3, c8 = sg & 7;
                    dst[sg] = *reinterpret_cast<const uint4 *>(tile + r * 128 + (((c8 ^ r) & 7) << 4));
                }
                // the publisher has released this slot's previous unit
                const bool ok = lu < kSolvers || mbar_wait(bar(B_PUBE0 + sv), ((lu / kSolvers) - 1) & 1);
                if (!ok) *fail = 1;
                mbar_arrive(bar(B_PUB0 + sv));
                __syncwarp();
                if (!ok) break;
            } else {
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&map_t, smem_u32(tile), 0, 0, 2 * u);
                    bulk_commit_group();
                    bulk_wait_group_read<0>();  // the slot may be refilled once the store has read it
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(bar(B_LE0 + sv));
        }
        if (lane == 0) bulk_wait_group_all();  // the T' stores have completed
    } else if (kFused && warp >= kPublisherWarp0 && warp < kPublisherWarp0 + kSolvers) {
        // ============================================================ publishers (fused)
        const int sv = warp - kPublisherWarp0;
        if (lane == 0) {
            for (int lu = sv;; lu += kSolvers) {
                const int which = lu & 1, pr = pair_id(lu >> 1);
                if (pr < 0) break;
                if (2 * pr + which >= n_units) continue;
                if (!mbar_wait(bar(B_PUB0 + sv), (lu / kSolvers) & 1)) { *fail = 1; break; }
                release_flag_gpu(p.flags + unit_at(2 * pr + which));
                mbar_arrive(bar(B_PUBE0 + sv));
            }
        }
    }

    __syncthreads();
    if (*fail && tid == 0) atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace solve
}  // namespace gdr
