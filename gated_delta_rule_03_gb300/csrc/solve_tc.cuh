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
// (fp32 [384]: g[64], gamma[64], kdec[64], then 1 for the ratio form and 0 otherwise,
// then the layer prologue's 1/|k_t| and 1/|q_t|, ones without it), so that the chain
// kernel uses the same values and the same form. With the prologue, L is formed from
// unit-length keys (k_t.k_i / (|k_t| |k_i|)); A^T stays the raw products, the chain
// applying 1/|k_i| through the pseudo-values and 1/|q_t| on the output rows. (The two forms are
// described in chain_tc.cuh; they differ only in where the decay factors are applied.)
//
// Mapping. Each warpgroup of a CTA solves one (chunk, head) unit at a time, on its own:
// group g of the launch's G groups takes units g, g + G, g + 2G, ..., and warp w of the
// group owns the unit's token rows 16w .. 16w + 15 throughout.
//   * load: the unit's keys and queries by TMA (128-byte-swizzled 64 x 64 bf16 tiles),
//     issued for the next unit as soon as this one's have been read;
//   * gates: warp 0 scans the log-decays of the unit (loaded while the previous unit
//     was worked on) into the decay factors;
//   * products: warp w forms its 16 rows of K K^T (keys up to its own block, for L) and
//     of K Q^T (queries from its own block on, for A^T) with warp-level bf16 MMAs,
//     ten 8-column tiles each, so that the four warps share the work evenly; L goes to
//     shared memory as fp32 16 x 16 blocks, A^T and the factors to the workspace;
//   * inverse: the unit lower-triangular (I + L)^{-1} on the CUDA cores in 16 x 16
//     blocks: warp w inverts diagonal block w by forward substitution, then the blocks
//     below the diagonal follow level by level (warp w computes block row w, with
//     warp-level TF32 products), the group meeting at a named barrier between levels;
//   * T': warp w writes block row w of diag(kdec) (I + L)^{-1} diag(beta) in bf16.
// Four groups per SM keep four units in flight, so that one unit's latencies (the load,
// the level barriers) are covered by the others'.
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace solve {

using namespace sm100;
using namespace tc;

constexpr int C = kChunk;
constexpr int kGroups = 4;                 // warpgroups per CTA, one unit each at a time
constexpr int kThreads = kGroups * 128;    // the standalone kernel's block
constexpr int kSolveWarps = kGroups * 4;   // warps of a fused launch's block that solve

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
// BF + 4 floats apart (16-byte aligned) so that blocks read at the same element by
// different warps start on different banks.
constexpr int BS = BF + 4;
__host__ __device__ constexpr int blk(int i, int k) { return (i * (i + 1) / 2 + k) * BS; }
__host__ __device__ constexpr int nblk(int i, int k) {  // N_ik, i > k
    return (10 + (i - k == 1 ? k : (i - k == 2 ? 3 + k : 5))) * BS;
}
constexpr int UNIT_FLOATS = 16 * BS;

// Shared memory of one group (the CTA holds kGroups of them, 1024-aligned):
//   keys then queries, each two 64-feature halves of 64 token rows (8 KB, 128-byte
//   swizzled as TMA writes them); the blocks; the unit's gates; the load barrier and the
//   group's failure flag.
constexpr uint32_t G_K = 0, G_Q = 16384;
constexpr uint32_t G_BLK = 32768;
constexpr uint32_t G_GATES = G_BLK + UNIT_FLOATS * 4;
constexpr int GG_G = 0, GG_GAM = 64, GG_GINV = 128, GG_BETA = 192, GG_KDEC = 256,
              GG_NK = 320, GG_NQ = 384;  // floats
constexpr uint32_t G_BAR = G_GATES + 7 * 64 * 4;
constexpr int kFactorFloats = 384;  // per unit in the workspace
constexpr uint32_t G_FAIL = G_BAR + 8;
constexpr uint32_t GROUP_BYTES = (G_FAIL + 8 + 1023) / 1024 * 1024;
constexpr uint32_t SMEM_BYTES = kGroups * GROUP_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448 && G_GATES % 16 == 0 && G_BAR % 8 == 0, "shared memory");

// ---------------------------------------------------------------- warp-level products
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

typedef float Acc16[2][4];
__device__ __forceinline__ void zero16(Acc16 &a) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) a[nt][e] = 0.f;
}

// ---------------------------------------------------------------- bf16 products of the Gram
// ldmatrix of four 8x8 bf16 matrices: lane l supplies a row address of matrix l / 8.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += A B for a 16x16 bf16 A (row-major) and a 16x8 B (held by column), fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared address of the 16-byte segment (row r, features 8c .. 8c + 7) of a 64-feature
// half tile as TMA writes it with the 128-byte swizzle (segment c of row r at c ^ r % 8).
__device__ __forceinline__ uint32_t sw128_at(uint32_t half, int r, int c) {
    return half + (uint32_t)(r * 128 + (((c ^ r) & 7) << 4));
}

struct SolveParams {
    const float *log_alpha, *beta;
    const int4 *plan;  // per chunk: sequence, first token, tokens, index within the sequence
    int32_t *ctl;      // [0] status, [1] number of chunks, [2 + f] first chunk of phase f
    int H;
    int phase;            // the units of this phase's chunks are solved (-1: every unit)
    // fused launch (beside the chain): units in chunk-major order over `seqs` sequences of
    // `seq_chunks` chunks each, and a ready flag per unit, set once its results are stored
    int seqs, seq_chunks;
    int32_t *flags;
    int additive;           // the additive rule: L = 0, so T = diag(beta)
    int prologue;           // the layer prologue: unit-length q, k; gates from a, b
    const float *gate_A;    // its per-head rate (null: 1)
    __nv_bfloat16 *Tout;  // [chunks * H][2][64][64]: T' then A^T per unit
    float *Gout;          // [chunks * H][kFactorFloats]: g, gamma, kdec, form, 1/|k|, 1/|q|
};

// One warp's part of the solve: warp W of a group (block row W of every unit), its loop
// over the group's units. The block row is a template parameter so that every
// loop bound and mask below is a constant and the loads can be issued early.
template <bool kFused>
struct GroupSolver {
    const SolveParams &p;
    const CUtensorMap *map_q, *map_k;
    uint32_t gbase;            // the group's shared memory
    float *U, *gt;             // its blocks and gates
    volatile int *gfail;
    int grp, lane, u0, n_units;
    int gid, gstride;          // units gid, gid + gstride, ... are this group's

    // the unit at local index x: the phase's units in order, or (fused) chunk j of
    // sequence n for head h at x = (j * seqs + n) * H + h
    __device__ __forceinline__ int unit_at(int x) const {
        if (!kFused) return u0 + x;
        const int h = x % p.H, r = x / p.H;
        return ((r % p.seqs) * p.seq_chunks + r / p.seqs) * p.H + h;
    }
    __device__ __forceinline__ void gsync() const { named_sync(1 + grp, 128); }
    __device__ __forceinline__ uint32_t bar_ld() const { return gbase + G_BAR; }
    // the plan entry of unit x (any x >= n_units: none); every lane of the caller loads it
    __device__ __forceinline__ int4 plan_of(int x) const {
        return x < n_units ? p.plan[unit_at(x) / p.H] : make_int4(0, 0, 0, 0);
    }
    __device__ __forceinline__ void issue_load(int x, const int4 &pl) const {  // leader
        const int h = unit_at(x) % p.H;
        mbar_arrive_expect_tx(bar_ld(), 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(gbase + G_K + b * 8192, map_k, bar_ld(), 64 * b, h, pl.y);
            tma_load_3d(gbase + G_Q + b * 8192, map_q, bar_ld(), 64 * b, h, pl.y);
        }
    }
    // the stored gates of unit x, two tokens per lane of warp 0 (padding past the end of
    // the sequence: log alpha = 0, beta = 0). The loads are only issued here; the values
    // are first used a whole unit later (gates_of), so their latency is hidden.
    __device__ __forceinline__ void fetch_gates(int x, const int4 &pl, float (&raw)[4]) const {
        raw[0] = raw[1] = raw[2] = raw[3] = 0.f;
        if (x >= n_units) return;
        const int h = unit_at(x) % p.H;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (2 * lane + e < pl.z) {
                const size_t off = (size_t)(pl.y + 2 * lane + e) * p.H + h;
                raw[e] = p.log_alpha[off];
                raw[2 + e] = p.beta[off];
            }
        }
    }
    // log alpha and beta from the stored values (the prologue's activations, if any)
    template <bool kPro>
    __device__ __forceinline__ void gates_of(int x, const int4 &pl, const float (&raw)[4],
                                             float (&gv)[4]) const {
        const float A = kPro && p.gate_A ? p.gate_A[unit_at(x) % p.H] : 1.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool in = 2 * lane + e < pl.z;
            gv[e] = kPro && in ? prologue_log_alpha(raw[e], A) : raw[e];
            gv[2 + e] = kPro && in ? prologue_beta(raw[2 + e]) : raw[2 + e];
        }
    }

    // kPro: the layer prologue (a template parameter, so that the plain path carries none
    // of its work)
    template <int W, bool kPro>
    __device__ __forceinline__ void run() const {
        const int gq = lane >> 2, q = lane & 3;  // m16n8 fragment coordinates
        const bool leader = W == 0 && lane == 0;
        int loads = 0, landed = 0;
        // This group's units are gid, gid + gstride, ...: fixed in advance, so that warp 0
        // can fetch a unit's plan entry and gates a whole unit before it needs them (a
        // claim from a shared counter would put two dependent global round trips on the
        // group's critical path). The units are equal in work.
        int x = gid;
        int4 pl_cur = make_int4(0, 0, 0, 0), pl_next = make_int4(0, 0, 0, 0);
        float raw[4] = {0.f, 0.f, 0.f, 0.f};  // warp 0: stored gates of unit x
        if (W == 0) {
            pl_cur = plan_of(x);
            if (leader && x < n_units) {
                issue_load(x, pl_cur);
                ++loads;
            }
            fetch_gates(x, pl_cur, raw);
            pl_next = plan_of(x + gstride);
        }
        uint32_t ld_phase = 0;
        while (x < n_units) {
            const int u = unit_at(x);
            // ---- gates of unit x: the shared scan of warp 0
            if (W == 0) {
                float gv[4];
                gates_of<kPro>(x, pl_cur, raw, gv);
                const ChunkScan sc = chunk_scan(gv[0], gv[1], lane);
                *reinterpret_cast<float2 *>(gt + GG_G + 2 * lane) = make_float2(sc.g0, sc.g1);
                *reinterpret_cast<float2 *>(gt + GG_GAM + 2 * lane) = make_float2(fast_exp(sc.g0), fast_exp(sc.g1));
                *reinterpret_cast<float2 *>(gt + GG_GINV + 2 * lane) = make_float2(fast_exp(-sc.g0), fast_exp(-sc.g1));
                *reinterpret_cast<float2 *>(gt + GG_BETA + 2 * lane) = make_float2(gv[2], gv[3]);
                *reinterpret_cast<float2 *>(gt + GG_KDEC + 2 * lane) =
                    make_float2(fast_exp(sc.g_last - sc.g0), fast_exp(sc.g_last - sc.g1));
            }
            if (!mbar_wait(bar_ld(), ld_phase)) *gfail = 1;
            ld_phase ^= 1;
            gsync();  // the gates are visible; every thread saw the load land (or gave up)
            if (*gfail) break;
            if (leader) ++landed;
            const bool ratio = gt[GG_G + C - 1] > kRatioSafeLogDecay;
            // 1/|k_r| (threads 0-63 of the group) and 1/|q_r| (64-127): the prologue's unit
            // lengths, from the staged rows; ones without it
            if (kPro) {
                const int i = 32 * W + lane, r = i & 63;
                float inv = 1.f;
                {
                    const uint32_t tile = gbase + (i < 64 ? G_K : G_Q);
                    float ss = 0.f;
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            uint4 u;
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                                         : "r"(sw128_at(tile + b * 8192, r, s)));
                            const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uw[e]));
                                ss = fmaf(x.x, x.x, fmaf(x.y, x.y, ss));
                            }
                        }
                    inv = prologue_inv_norm(ss);
                }
                gt[(i < 64 ? GG_NK : GG_NQ) + r] = inv;
            }

            // ---- rows 16W .. 16W + 15 of K K^T (keys i < 16W + 16) and of K Q^T (queries
            // t >= 16W): ten 8-column tiles; tile pair j2 <= W holds keys 16 j2 .. 16 j2 + 15,
            // the others queries 16 (j2 - 1) .. 16 (j2 - 1) + 15
            float acc[10][4];
#pragma unroll
            for (int j = 0; j < 10; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int b = ks >> 2, c = 2 * (ks & 3);  // d_k half, 8-feature segment
                uint32_t a[4];
                ldsm_x4(sw128_at(gbase + G_K + b * 8192, 16 * W + (lane & 15), c + (lane >> 4)), a);
#pragma unroll
                for (int j2 = 0; j2 < 5; ++j2) {
                    const bool keys = j2 <= W;
                    const int r0 = keys ? 16 * j2 : 16 * (j2 - 1);
                    const uint32_t half = gbase + (keys ? G_K : G_Q) + b * 8192;
                    uint32_t bf[4];
                    ldsm_x4(sw128_at(half, r0 + (lane & 7) + 8 * (lane >> 4), c + ((lane >> 3) & 1)), bf);
                    mma_bf16_16x8x16(acc[2 * j2], a, bf[0], bf[1]);
                    mma_bf16_16x8x16(acc[2 * j2 + 1], a, bf[2], bf[3]);
                }
            }
            if (kPro) gsync();  // every row's 1/|k| is in place
            // the gates this warp needs: its rows' (t = 16W + gq + 8hh) and the columns' of
            // its tiles (i0 = 8j + 2q, two each)
            float rg[2], rb[2], rgi[2], rkd[2], cg[8][2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = 16 * W + gq + 8 * hh;
                rg[hh] = ratio ? gt[GG_GAM + t] : gt[GG_G + t];
                rgi[hh] = gt[GG_G + t];
                // L = 0 for the additive rule; 1/|k_t| of the prologue folded into beta_t
                rb[hh] = p.additive ? 0.f : (kPro ? gt[GG_BETA + t] * gt[GG_NK + t] : gt[GG_BETA + t]);
                rkd[hh] = ratio ? gt[GG_KDEC + t] : 1.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = *reinterpret_cast<const float2 *>(gt + (ratio && j < 2 * (W + 1) ? GG_GINV : GG_G) + 8 * j + 2 * q);
                cg[j][0] = f.x;
                cg[j][1] = f.y;
            }
            const float ginv_c = gt[GG_GINV + C - 1];
            // L_ti = beta_t Gamma_ti k_t.k_i (i < t) into block row W
#pragma unroll
            for (int j = 0; j < 2 * (W + 1); ++j) {
                const int i0 = 8 * j + 2 * q;
                float *B = U + blk(W, j >> 1);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int t = 16 * W + gq + 8 * hh;
                    const float d0 = ratio ? rg[hh] * cg[j][0] : fast_exp(rg[hh] - cg[j][0]);
                    const float d1 = ratio ? rg[hh] * cg[j][1] : fast_exp(rg[hh] - cg[j][1]);
                    const float nk0 = kPro ? gt[GG_NK + i0] : 1.f, nk1 = kPro ? gt[GG_NK + i0 + 1] : 1.f;
                    const float v0 = i0 < t ? rb[hh] * d0 * nk0 * acc[j][2 * hh] : 0.f;
                    const float v1 = i0 + 1 < t ? rb[hh] * d1 * nk1 * acc[j][2 * hh + 1] : 0.f;
                    *reinterpret_cast<float2 *>(B + el(gq + 8 * hh, 8 * (j & 1) + 2 * q)) = make_float2(v0, v1);
                }
            }
            // A^T_it (t >= i) for keys i = 16W + gq + 8hh and queries t from 16W on, bf16 to
            // the workspace; the queries before 16W are zero
            __nv_bfloat16 *arow = p.Tout + (size_t)(2 * u + 1) * C * C;
#pragma unroll
            for (int j = 2 * (W + 1); j < 10; ++j) {
                const int t0 = 8 * (j - 2) + 2 * q;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = 16 * W + gq + 8 * hh;
                    const float d0 = ratio ? ginv_c : fast_exp(cg[j - 2][0] - rgi[hh]);
                    const float d1 = ratio ? ginv_c : fast_exp(cg[j - 2][1] - rgi[hh]);
                    const float v0 = t0 >= i ? acc[j][2 * hh] * d0 : 0.f;
                    const float v1 = t0 + 1 >= i ? acc[j][2 * hh + 1] * d1 : 0.f;
                    *reinterpret_cast<uint32_t *>(arow + i * C + t0) = pack_bf16x2(v0, v1);
                }
            }
#pragma unroll
            for (int s = 0; s < W; ++s) {  // rows 16W .. 16W + 15, columns 0 .. 16W - 1
                const int idx = lane + 32 * s, r = 16 * W + (idx & 15), seg = idx >> 4;
                *reinterpret_cast<uint4 *>(arow + r * C + 8 * seg) = make_uint4(0, 0, 0, 0);
            }
            // the unit's decay factors for the chain: g (warp 0), gamma (1), kdec (2), form (3);
            // 1/|k| (warp 0) and 1/|q| (warp 1)
            {
                float *go = p.Gout + (size_t)u * kFactorFloats;
                float2 v;
                if (W == 0) v = *reinterpret_cast<const float2 *>(gt + GG_G + 2 * lane);
                else if (W == 1) v = *reinterpret_cast<const float2 *>(gt + GG_GAM + 2 * lane);
                else if (W == 2) v = *reinterpret_cast<const float2 *>(gt + GG_KDEC + 2 * lane);
                else v = make_float2(lane == 0 ? (ratio ? 1.f : 0.f) : 0.f, 0.f);
                *reinterpret_cast<float2 *>(go + 64 * W + 2 * lane) = v;
                if (kPro && W < 2)  // (the chain reads them only with the prologue)
                    *reinterpret_cast<float2 *>(go + 256 + 64 * W + 2 * lane) =
                        *reinterpret_cast<const float2 *>(gt + (W == 0 ? GG_NK : GG_NQ) + 2 * lane);
            }
            gsync();  // keys and queries are read; L is complete
            // the next unit: its keys and queries land while the inverse runs; its gates
            // and the plan entry of the one after are fetched for later
            if (W == 0) {
                const int xn = x + gstride;
                if (leader && xn < n_units) {
                    fence_async_smem();  // the reads above come before the TMA overwrites the tiles
                    issue_load(xn, pl_next);
                    ++loads;
                }
                fetch_gates(xn, pl_next, raw);
                pl_cur = pl_next;
                pl_next = plan_of(xn + gstride);
            }

            // ---- (I + L)^{-1}: diagonal block W by forward substitution, lane l on column
            // l % 16 (the upper half of the warp repeats the lower and stores nothing)
            {
                float *D = U + blk(W, W);
                const int c0 = lane & 15;
                float xv[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) xv[r] = (r == c0) ? 1.f : 0.f;
#pragma unroll
                for (int k = 0; k < 15; ++k) {
                    const float ak = xv[k];
#pragma unroll
                    for (int r = k + 1; r < 16; ++r) xv[r] = fmaf(-D[el(r, k)], ak, xv[r]);
                }
                __syncwarp();
                if (lane < 16) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) D[el(r, c0)] = xv[r];
                }
                __syncwarp();
            }
            // M_Wk = N_WW L_Wk over L_Wk (k < W): the warp's own blocks
            if (W >= 1) {
                Acc16 m[W > 0 ? W : 1];
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    zero16(m[k]);
                    warp_gemm16(U + blk(W, W), U + blk(W, k), m[k], lane);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < W; ++k) warp_store16(U + blk(W, k), m[k], lane, 1.f);
            }
            gsync();  // every N_kk is in place
            // level 1: N_{W,W-1} = -M_{W,W-1} N_{W-1,W-1}, and the partial sums that need
            // only the diagonal: P20 = M_20 N_00 (warp 2), P31 = M_31 N_11, P30 = M_30 N_00 (3)
            Acc16 pa, pb;
            zero16(pa);
            zero16(pb);
            if (W >= 1) {
                constexpr int Wm = W > 0 ? W - 1 : 0;
                Acc16 n1;
                zero16(n1);
                warp_gemm16(U + blk(W, Wm), U + blk(Wm, Wm), n1, lane);
                if (W == 2) warp_gemm16(U + blk(2, 0), U + blk(0, 0), pa, lane);
                if (W == 3) {
                    warp_gemm16(U + blk(3, 1), U + blk(1, 1), pa, lane);
                    warp_gemm16(U + blk(3, 0), U + blk(0, 0), pb, lane);
                }
                warp_store16(U + nblk(W > 0 ? W : 1, Wm), n1, lane, -1.f);
            }
            gsync();  // N_10, N_21, N_32 are in place
            // level 2: N_20 = -(P20 + M_21 N_10) (warp 2); N_31 = -(P31 + M_32 N_21) and
            // P30 += M_31 N_10 (warp 3)
            if (W == 2) {
                warp_gemm16(U + blk(2, 1), U + nblk(1, 0), pa, lane);
                warp_store16(U + nblk(2, 0), pa, lane, -1.f);
            } else if (W == 3) {
                warp_gemm16(U + blk(3, 2), U + nblk(2, 1), pa, lane);
                warp_gemm16(U + blk(3, 1), U + nblk(1, 0), pb, lane);
                warp_store16(U + nblk(3, 1), pa, lane, -1.f);
            }
            gsync();  // N_20 is in place
            // level 3: N_30 = -(P30 + M_32 N_20) (warp 3)
            if (W == 3) {
                warp_gemm16(U + blk(3, 2), U + nblk(2, 0), pb, lane);
                warp_store16(U + nblk(3, 0), pb, lane, -1.f);
            }
            __syncwarp();

            // ---- T' block row W: diag(kd) N diag(beta), bf16 pairs to the workspace (the
            // blocks right of the diagonal, and the diagonal block's upper part, are zero)
            {
                __nv_bfloat16 *trow = p.Tout + (size_t)2 * u * C * C;
                float cb[4][2][2];  // beta of columns 16 bi + 8 nt + 2q (+1)
#pragma unroll
                for (int bi = 0; bi < 4; ++bi)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float2 bb = *reinterpret_cast<const float2 *>(gt + GG_BETA + 16 * bi + 8 * nt + 2 * q);
                        cb[bi][nt][0] = bb.x;
                        cb[bi][nt][1] = bb.y;
                    }
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int i0 = 16 * bi + 8 * nt + 2 * q;
                        float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
                        if (bi <= W) {
                            const float *B = U + (bi == W ? blk(W, W) : nblk(W > bi ? W : 1, W > bi ? bi : 0));
                            lo = *reinterpret_cast<const float2 *>(B + el(gq, 8 * nt + 2 * q));
                            hi = *reinterpret_cast<const float2 *>(B + el(gq + 8, 8 * nt + 2 * q));
                        }
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int t = 16 * W + gq + 8 * hh;
                            const float2 v = hh ? hi : lo;
                            const float x0 = i0 <= t ? v.x * cb[bi][nt][0] * rkd[hh] : 0.f;
                            const float x1 = i0 + 1 <= t ? v.y * cb[bi][nt][1] * rkd[hh] : 0.f;
                            *reinterpret_cast<uint32_t *>(trow + t * C + i0) = pack_bf16x2(x0, x1);
                        }
                    }
                }
            }
            gsync();  // unit u is stored; the blocks and gates may be reused
            if (kFused && leader) release_flag_gpu(p.flags + u);
            x += gstride;
        }
        if (leader) {
            if (*gfail) atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
            // a load still in flight lands before the shared memory goes away
            for (int j = landed; j < loads; ++j) mbar_wait(bar_ld(), j & 1);
        }
    }
};

// The solve on one CTA, rank `rank` of the launch's `ranks` solve CTAs. kFused: the
// CTA shares a cooperative launch with the chain (whose block has more warps: those past
// the solve's return at once; no block-wide barrier follows), takes the units in
// chunk-major order so that the chains find their chunks solved in the order they need
// them (every group runs at the same pace), and publishes each unit with a release of
// its flag.
template <bool kFused>
__device__ __forceinline__ void solve_body(const CUtensorMap &map_q, const CUtensorMap &map_k,
                                           const SolveParams &p, int rank, int ranks) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp >= kSolveWarps) return;
    const int grp = warp >> 2, w = warp & 3;  // group, and the warp's block row in it
    unsigned char *gs = sm + grp * GROUP_BYTES;
    const uint32_t gbase = smem_u32(gs);
    volatile int *fail = reinterpret_cast<volatile int *>(gs + G_FAIL);
    if (w == 0 && lane == 0) {
        mbar_init(gbase + G_BAR, 1);
        fence_mbar_init();
        *fail = 0;
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
    }
    named_sync(1 + grp, 128);

    // Everything above overlaps the tail of the planning kernel (programmatic launch);
    // the plan and the status word are read only after it has completed.
    griddep_wait();
    griddep_launch_dependents();
    // this phase's units are u0 + [0, n_units); local indices, u0 added for addressing
    // (phase -1: every unit of the call)
    const bool all = kFused || p.phase < 0;
    const int u0 = all ? 0 : p.ctl[2 + p.phase] * p.H;
    const int n_units =
        p.ctl[0] == GDR_OK ? (all ? p.ctl[1] * p.H : p.ctl[3 + p.phase] * p.H - u0) : 0;
    const GroupSolver<kFused> gsv{p, &map_q, &map_k, gbase,
                                  reinterpret_cast<float *>(gs + G_BLK), reinterpret_cast<float *>(gs + G_GATES),
                                  fail, grp, lane, u0, n_units, rank * kGroups + grp, ranks * kGroups};
    switch (w) {
        case 0: p.prologue ? gsv.template run<0, true>() : gsv.template run<0, false>(); break;
        case 1: p.prologue ? gsv.template run<1, true>() : gsv.template run<1, false>(); break;
        case 2: p.prologue ? gsv.template run<2, true>() : gsv.template run<2, false>(); break;
        default: p.prologue ? gsv.template run<3, true>() : gsv.template run<3, false>(); break;
    }
}

}  // namespace solve
}  // namespace gdr
