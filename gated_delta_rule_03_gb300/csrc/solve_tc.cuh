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
//   * products: one tcgen05 MMA chain per unit, [K; Q] K^T (M = 128: the 64 keys, then
//     the 64 queries; N = 64 keys; K = d_k) into the group's 64 TMEM columns, issued
//     by the group's leader as soon as the unit's tiles have landed -- for the next
//     unit, during this unit's inverse. TMEM lane quarter w belongs to warp w: warps
//     0 and 1 read the key rows t of K K^T and write L to shared memory as fp32
//     16 x 16 blocks; warps 2 and 3 read the query rows t of Q K^T and write A^T to the
//     workspace (neighbouring queries swap one value each so that every store is a
//     bf16 pair along t); the factors go to the workspace too;
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
//   the unit's keys and queries: for each 64-feature half b of d_k, the 64 key rows then
//   the 64 query rows (8 KB each, 128-byte swizzled as TMA writes them), so that half b
//   is the 128-row A operand [K; Q] of the Gram and its first 64 rows the B operand K;
//   the blocks; the unit's gates; the load and Gram barriers and the group's failure
//   flag (group 0 also keeps the CTA's TMEM address after them).
constexpr uint32_t G_KQ = 0;
constexpr uint32_t G_BLK = 32768;
constexpr uint32_t G_GATES = G_BLK + UNIT_FLOATS * 4;
constexpr int GG_G = 0, GG_GAM = 64, GG_GINV = 128, GG_BETA = 192, GG_KDEC = 256,
              GG_NK = 320, GG_NQ = 384;  // floats
constexpr uint32_t G_BAR = G_GATES + 7 * 64 * 4;
constexpr uint32_t G_BAR_MMA = G_BAR + 8;
constexpr int kFactorFloats = 384;  // per unit in the workspace
constexpr uint32_t G_FAIL = G_BAR_MMA + 8;
constexpr uint32_t G_TMEM_SLOT = G_FAIL + 8;
constexpr uint32_t G_XSLOT = G_TMEM_SLOT + 8;  // claimed units: the group's next unit
constexpr uint32_t GROUP_BYTES = (G_XSLOT + 8 + 1023) / 1024 * 1024;
constexpr uint32_t SMEM_BYTES = kGroups * GROUP_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448 && G_GATES % 16 == 0 && G_BAR % 8 == 0, "shared memory");
// TMEM: 64 fp32 columns per group for its Gram (rows = the 128 lanes)
constexpr uint32_t kGramCols = 64, kTmemCols = kGroups * kGramCols;
static_assert(kTmemCols == 256, "TMEM allocation is a power of two");
constexpr int kBarSolve = 5;  // named barrier of all the solve warps of a CTA

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

// Shared address of the 16-byte segment (row r, features 8c .. 8c + 7) of a 64-feature
// half tile as TMA writes it with the 128-byte swizzle (segment c of row r at c ^ r % 8).
__device__ __forceinline__ uint32_t sw128_at(uint32_t half, int r, int c) {
    return half + (uint32_t)(r * 128 + (((c ^ r) & 7) << 4));
}

// (I + L)^{-1} of one unit, in place in its 16 x 16 blocks (the layout above). On entry
// the ten lower blocks hold L: strictly lower triangular, the diagonal blocks zero on and
// above their diagonal. On return blk(i, i) holds N_ii and nblk(i, k) holds N_ik (i > k)
// of N = (I + L)^{-1} (blk(i, k), i > k, then holds M_ik = N_ii L_ik). Warp W of four
// computes block row W: the diagonal block by forward substitution (lane l on column
// l % 16; the upper half of the warp repeats the lower and stores nothing), then the
// blocks below the diagonal level by level with warp-level TF32 products. sync() is a
// barrier of the four warps; after_diag() runs on every thread once the diagonal blocks'
// inverses are in place (before the levels).
template <int W, typename Sync, typename Hook>
__device__ __forceinline__ void invert_unit(float *__restrict__ U, int lane, Sync sync, Hook after_diag) {
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
    sync();  // every N_kk is in place
    after_diag();
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
    sync();  // N_10, N_21, N_32 are in place
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
    sync();  // N_20 is in place
    // level 3: N_30 = -(P30 + M_32 N_20) (warp 3)
    if (W == 3) {
        warp_gemm16(U + blk(3, 2), U + nblk(2, 0), pb, lane);
        warp_store16(U + nblk(3, 0), pb, lane, -1.f);
    }
    __syncwarp();
}

struct SolveParams {
    const float *log_alpha, *beta;
    const int4 *plan;  // per chunk: sequence, first token, tokens, index within the sequence
    int32_t *ctl;      // [0] status, [1] number of chunks, [2 + f] first chunk of phase f
    int H;
    int phase;            // the units of this phase's chunks are solved (-1: every unit)
    // fused launch (beside the chain): units in chunk-major order over `seqs` sequences of
    // `seq_chunks` chunks (seq_len tokens) each, and a ready flag per unit, set once its
    // results are stored; the plan of such a call is closed-form and not read
    int seqs, seq_chunks, seq_len;
    int32_t *flags;
    // fused launch over packed sequences: the units are claimed one at a time from a
    // counter shared by the grid, in the order of the plan's claim rows (row r: chunk
    // order[r].x, first token .y, tokens .z; its H units are heads 0 .. H - 1)
    const int4 *order;
    int32_t *claim;
    int only_pair;  // solve nothing unless ctl[kPairWord] hands the call to this launch
    int additive;           // the additive rule: L = 0, so T = diag(beta)
    int prologue;           // the layer prologue: unit-length q, k; gates from a, b
    const float *gate_A;    // its per-head rate (null: 1)
    __nv_bfloat16 *Tout;  // [chunks * H][2][64][64]: T' then A^T per unit
    float *Gout;          // [chunks * H][kFactorFloats]: g, gamma, kdec, form, 1/|k|, 1/|q|
};

// One warp's part of the solve: warp W of a group (block row W of every unit), its loop
// over the group's units. The block row is a template parameter so that every
// loop bound and mask below is a constant and the loads can be issued early.
template <bool kFused, bool kClaim = false>
struct GroupSolver {
    const SolveParams &p;
    const CUtensorMap *map_q, *map_k;
    uint32_t gbase;            // the group's shared memory
    float *U, *gt;             // its blocks and gates
    volatile int *gfail;
    int grp, lane, u0, n_units;
    int gid, gstride;          // units gid, gid + gstride, ... are this group's
    uint32_t tmem_d;           // the group's TMEM columns (lane field 0)
    int stop;                  // kClaim: no claim once the group holds a unit >= stop

    // the unit at local index x: the phase's units in order, or (fused) chunk j of
    // sequence n for head h at x = (j * seqs + n) * H + h
    __device__ __forceinline__ int unit_at(int x) const {
        if (kClaim) return p.order[x / p.H].x * p.H + x % p.H;
        if (!kFused) return u0 + x;
        const int h = x % p.H, r = x / p.H;
        return ((r % p.seqs) * p.seq_chunks + r / p.seqs) * p.H + h;
    }
    __device__ __forceinline__ void gsync() const { named_sync(1 + grp, 128); }
    __device__ __forceinline__ uint32_t bar_ld() const { return gbase + G_BAR; }
    __device__ __forceinline__ uint32_t bar_mma() const { return gbase + G_BAR_MMA; }
    // the plan entry of unit x (any x >= n_units: none); every lane of the caller loads it
    __device__ __forceinline__ int4 plan_of(int x) const {
        if (kClaim) return x < n_units ? p.order[x / p.H] : make_int4(0, 0, 0, 0);
        if (kFused) {  // chunk c of the call is chunk c % seq_chunks of sequence c / seq_chunks
            if (x >= n_units) return make_int4(0, 0, 0, 0);
            const int c = unit_at(x) / p.H, n = c / p.seq_chunks, j = c % p.seq_chunks;
            const int rem = p.seq_len - j * C;
            return make_int4(n, n * p.seq_len + j * C, rem < C ? rem : C, j);
        }
        return x < n_units ? p.plan[unit_at(x) / p.H] : make_int4(0, 0, 0, 0);
    }
    // kClaim: warp 0 claims the next unit (lane 0's atomic; the index is read later, so
    // that its latency is not waited for); n_units when the group claims no more
    __device__ __forceinline__ int claim_issue(int held) const {
        return lane == 0 && held < n_units && held < stop ? claim_next(p.claim) : n_units;
    }
    __device__ __forceinline__ int claim_read(int c) const {
        const int x = __shfl_sync(0xffffffffu, c, 0);
        return x < n_units ? x : n_units;
    }
    __device__ __forceinline__ volatile int *xslot() const {
        return reinterpret_cast<volatile int *>(reinterpret_cast<volatile unsigned char *>(gfail) - G_FAIL +
                                                G_XSLOT);
    }
    __device__ __forceinline__ void issue_load(int x, const int4 &pl) const {  // leader
        const int h = unit_at(x) % p.H;
        mbar_arrive_expect_tx(bar_ld(), 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(gbase + G_KQ + b * 16384, map_k, bar_ld(), 64 * b, h, pl.y);
            tma_load_3d(gbase + G_KQ + b * 16384 + 8192, map_q, bar_ld(), 64 * b, h, pl.y);
        }
    }
    // [K; Q] K^T of the unit whose keys and queries are in the tiles, into the group's
    // TMEM columns: D row t < 64 holds k_t . k_i, row 64 + t holds q_t . k_i (i < 64).
    // Issued by the leader once the tiles have landed; completes on bar_mma.
    __device__ __forceinline__ void issue_gram() const {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t at = gbase + G_KQ + (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem_d, sw128_desc(at, 16, 1024), sw128_desc(at, 16, 1024),
                     idesc_bf16(128, 64, 0, 0), kk > 0);
        }
        mma_commit(bar_mma());
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
        // (leader) loads issued and seen landed, Grams issued and consumed
        int loads = 0, landed = 0, grams = 0, consumed = 0;
        // This group's units are gid, gid + gstride, ...: fixed in advance, so that warp 0
        // can fetch a unit's plan entry and gates a whole unit before it needs them (a
        // claim from a shared counter would put two dependent global round trips on the
        // group's critical path). The units are equal in work.
        // (kClaim: the group's units come from the grid's claim counter instead; warp 0
        // claims them a unit ahead and passes each to the group through shared memory.)
        int x = gid;
        int x_next = 0, claimed = 0;  // kClaim, warp 0: the next unit; the pending claim
        int4 pl_cur = make_int4(0, 0, 0, 0), pl_next = make_int4(0, 0, 0, 0);
        float raw[4] = {0.f, 0.f, 0.f, 0.f};  // warp 0: stored gates of unit x
        if (kClaim) {
            if (W == 0) {
                x = claim_read(claim_issue(-1));
                if (lane == 0) *xslot() = x;
                claimed = claim_issue(x);
            }
            gsync();
            x = *xslot();
        }
        if (W == 0) {
            pl_cur = plan_of(x);
            if (leader && x < n_units) {
                issue_load(x, pl_cur);
                ++loads;
            }
            fetch_gates(x, pl_cur, raw);
            if (!kClaim) pl_next = plan_of(x + gstride);
        }
        // the first unit's Gram, once its keys and queries have landed
        if (leader && x < n_units) {
            if (mbar_wait(bar_ld(), 0)) {
                ++landed;
                issue_gram();
                ++grams;
            } else {
                *gfail = 1;
            }
        }
        uint32_t ld_phase = 0, mma_phase = 0;
        while (x < n_units) {
            const int u = unit_at(x);
            // (kClaim: known to warp 0 only, after the first barrier below)
            bool has_next = x + gstride < n_units;
            bool gram_next = false;  // (leader) the next unit's Gram is issued
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
            // the unit's tiles have landed (their bytes visible to this thread) and its
            // Gram is done
            if (!(mbar_wait(bar_ld(), ld_phase) && mbar_wait(bar_mma(), mma_phase))) *gfail = 1;
            ld_phase ^= 1;
            mma_phase ^= 1;
            if (leader) ++consumed;
            gsync();  // the gates are visible; every thread saw the Gram done (or gave up)
            if (*gfail) break;
            tc_fence_after();
            if (kClaim && W == 0) {  // the unit after this one, claimed during the last
                x_next = claim_read(claimed);
                has_next = x_next < n_units;
                pl_next = plan_of(x_next);
            }
            const bool ratio = gt[GG_G + C - 1] > kRatioSafeLogDecay;
            // 1/|k_r| (threads 0-63 of the group) and 1/|q_r| (64-127): the prologue's unit
            // lengths, from the staged rows; ones without it
            if (kPro) {
                const int i = 32 * W + lane, r = i & 63;
                float inv = 1.f;
                {
                    const uint32_t tile = gbase + G_KQ + (i < 64 ? 0u : 8192u);
                    float ss = 0.f;
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            uint4 u;
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                                         : "r"(sw128_at(tile + b * 16384, r, s)));
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
                gsync();  // every row's 1/|k| is in place
            }

            // ---- read out the Gram: warp W holds TMEM lanes 32W .. 32W + 31, read 16
            // columns (keys) at a time
            const uint32_t lanes = tmem_d + ((uint32_t)(32 * W) << 16);
            if (W < 2) {
                // key row t of K K^T: L_ti = beta_t Gamma_ti k_t.k_i (i < t) into the blocks
                // of block row t / 16
                const int t = 32 * W + lane, br = t >> 4, r = t & 15;
                const float rg = ratio ? gt[GG_GAM + t] : gt[GG_G + t];
                // L = 0 for the additive rule; 1/|k_t| of the prologue folded into beta_t
                const float rb = p.additive ? 0.f : (kPro ? gt[GG_BETA + t] * gt[GG_NK + t] : gt[GG_BETA + t]);
                // the warp-wide TMEM loads run for every block column of the warp's two block
                // rows (2W and 2W + 1); a row's lanes store only its own blocks
#pragma unroll 1
                for (int jb = 0; jb <= 2 * W + 1; ++jb) {  // block column jb: keys 16 jb .. +15
                    float d[16];
                    tmem_load16(lanes + 16 * jb, d);
                    if (jb > br) continue;
                    float *B = U + blk(br, jb);
#pragma unroll
                    for (int cg = 0; cg < 4; ++cg) {
                        const int i0 = 16 * jb + 4 * cg;
                        const float4 cf = *reinterpret_cast<const float4 *>(gt + (ratio ? GG_GINV : GG_G) + i0);
                        const float4 nk4 = kPro ? *reinterpret_cast<const float4 *>(gt + GG_NK + i0)
                                                : make_float4(1.f, 1.f, 1.f, 1.f);
                        const float c[4] = {cf.x, cf.y, cf.z, cf.w}, nk[4] = {nk4.x, nk4.y, nk4.z, nk4.w};
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float dec = ratio ? rg * c[e] : fast_exp(rg - c[e]);
                            v[e] = i0 + e < t ? rb * dec * nk[e] * d[4 * cg + e] : 0.f;
                        }
                        *reinterpret_cast<float4 *>(B + el(r, 4 * cg)) = make_float4(v[0], v[1], v[2], v[3]);
                    }
                }
            } else {
                // query row t of Q K^T: A^T_it for keys i <= t, else 0, bf16 to the workspace.
                // Lanes t and t ^ 1 swap one value per key pair, so that the even lane stores
                // (A^T_{2p, t}, A^T_{2p, t+1}) and the odd lane (A^T_{2p+1, t-1}, A^T_{2p+1, t}).
                const int t = 32 * (W - 2) + lane;
                const bool odd = lane & 1;
                const float g_t = gt[GG_G + t], ginv_c = gt[GG_GINV + C - 1];
                __nv_bfloat16 *arow = p.Tout + (size_t)(2 * u + 1) * C * C + (t & ~1);
#pragma unroll 1
                for (int kb = 0; kb < 4; ++kb) {  // keys 16 kb .. 16 kb + 15
                    float d[16];
                    tmem_load16(lanes + 16 * kb, d);
#pragma unroll
                    for (int pp = 0; pp < 8; ++pp) {
                        const int i0 = 16 * kb + 2 * pp;
                        float dec0 = ginv_c, dec1 = ginv_c;
                        if (!ratio) {
                            const float2 gi = *reinterpret_cast<const float2 *>(gt + GG_G + i0);
                            dec0 = fast_exp(g_t - gi.x);
                            dec1 = fast_exp(g_t - gi.y);
                        }
                        const float v0 = i0 <= t ? dec0 * d[2 * pp] : 0.f;
                        const float v1 = i0 + 1 <= t ? dec1 * d[2 * pp + 1] : 0.f;
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                        const uint32_t w = odd ? pack_bf16x2(recv, v1) : pack_bf16x2(v0, recv);
                        *reinterpret_cast<uint32_t *>(arow + (i0 + (odd ? 1 : 0)) * C) = w;
                    }
                }
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
            tc_fence_before();
            gsync();  // L is complete; the tiles and the Gram's TMEM columns are read
            // the next unit: its keys and queries land while the inverse runs (its Gram is
            // issued once they have); its gates and the plan entry of the one after are
            // fetched for later
            if (W == 0) {
                const int xn = kClaim ? x_next : x + gstride;
                if (leader && xn < n_units) {
                    if (kPro) fence_async_smem();  // the norms' reads come before the TMA writes
                    issue_load(xn, pl_next);
                    ++loads;
                }
                fetch_gates(xn, pl_next, raw);
            }

            // ---- (I + L)^{-1} in the blocks
            invert_unit<W>(U, lane, [&] { gsync(); }, [&] {
                // the next unit's Gram, if its tiles have landed (else at the end of this
                // unit); the Gram's TMEM columns were read before the load was issued
                if (leader && has_next && mbar_test_wait(bar_ld(), ld_phase)) {
                    ++landed;
                    issue_gram();
                    ++grams;
                    gram_next = true;
                }
            });

            // ---- T' block row W: diag(kd) N diag(beta), bf16 pairs to the workspace (the
            // blocks right of the diagonal, and the diagonal block's upper part, are zero)
            {
                __nv_bfloat16 *trow = p.Tout + (size_t)2 * u * C * C;
                float rkd[2];  // kdec of this thread's rows t = 16W + gq + 8hh (ratio form)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) rkd[hh] = ratio ? gt[GG_KDEC + 16 * W + gq + 8 * hh] : 1.f;
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
            if (kClaim && W == 0 && lane == 0) *xslot() = x_next;
            gsync();  // unit u is stored; the blocks and gates may be reused
            if (kFused && leader) release_flag_gpu(p.flags + u);
            if (leader && has_next && !gram_next) {
                if (mbar_wait(bar_ld(), ld_phase)) {
                    ++landed;
                    issue_gram();
                    ++grams;
                } else {
                    *gfail = 1;
                }
            }
            if (kClaim) {
                x = *xslot();
                if (W == 0) {
                    pl_cur = pl_next;
                    claimed = claim_issue(x);
                }
            } else {
                if (W == 0) {
                    pl_cur = pl_next;
                    pl_next = plan_of(x + 2 * gstride);
                }
                x += gstride;
            }
        }
        if (leader) {
            if (*gfail) atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
            // a load still in flight lands, and a Gram still in flight completes, before the
            // shared memory and TMEM go away
            for (int j = landed; j < loads; ++j) mbar_wait(bar_ld(), j & 1);
            if (grams > consumed) mbar_wait(bar_mma(), (grams - 1) & 1);
        }
    }
};

// The solve on one CTA, rank `rank` of the launch's `ranks` solve CTAs. kFused: the
// CTA shares a cooperative launch with the chain (whose block has more warps: those past
// the solve's return at once; no block-wide barrier follows), takes the units in
// chunk-major order so that the chains find their chunks solved in the order they need
// them (every group runs at the same pace), and publishes each unit with a release of
// its flag. kClaim (with kFused): the units are claimed from the grid's counter in the
// plan's claim order instead, each group stopping after the first unit it holds at or
// past `stop`; with then_chain the CTA goes on to run a chain, so its TMEM allocation
// right is kept and its barriers are ended for the chain to reuse the shared memory.
template <bool kFused, bool kClaim = false>
__device__ __forceinline__ void solve_body(const CUtensorMap &map_q, const CUtensorMap &map_k,
                                           const SolveParams &p, int rank, int ranks,
                                           int stop = 0x7fffffff, bool then_chain = false) {
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
        mbar_init(gbase + G_BAR_MMA, 1);
        fence_mbar_init();
        *fail = 0;
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_q);
    }
    // the CTA's TMEM: 64 columns per group (its address kept in group 0's area)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G_TMEM_SLOT);
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        if (!then_chain) tmem_relinquish();
    }
    tc_fence_before();
    named_sync(kBarSolve, kSolveWarps * 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Everything above overlaps the tail of the planning kernel (programmatic launch);
    // the plan and the status word are read only after it has completed.
    griddep_wait();
    griddep_launch_dependents();
    // this phase's units are u0 + [0, n_units); local indices, u0 added for addressing
    // (phase -1: every unit of the call)
    const bool all = kFused || p.phase < 0;
    const int u0 = all ? 0 : p.ctl[2 + p.phase] * p.H;
    const bool runs = p.ctl[0] == GDR_OK && (!p.only_pair || p.ctl[kPairWord] == 1);
    const int n_units = runs ? (all ? p.ctl[1] * p.H : p.ctl[3 + p.phase] * p.H - u0) : 0;
    const GroupSolver<kFused, kClaim> gsv{p, &map_q, &map_k, gbase,
                                          reinterpret_cast<float *>(gs + G_BLK), reinterpret_cast<float *>(gs + G_GATES),
                                          fail, grp, lane, u0, n_units, rank * kGroups + grp, ranks * kGroups,
                                          tmem + (uint32_t)grp * kGramCols, stop};
    switch (w) {
        case 0: p.prologue ? gsv.template run<0, true>() : gsv.template run<0, false>(); break;
        case 1: p.prologue ? gsv.template run<1, true>() : gsv.template run<1, false>(); break;
        case 2: p.prologue ? gsv.template run<2, true>() : gsv.template run<2, false>(); break;
        default: p.prologue ? gsv.template run<3, true>() : gsv.template run<3, false>(); break;
    }
    // every group is done with its TMEM columns (their Grams completed or drained)
    __syncwarp();
    tc_fence_before();
    named_sync(kBarSolve, kSolveWarps * 32);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (then_chain) {  // nothing waits on the group's barriers any more
        if (w == 0 && lane == 0) {
            mbar_inval(gbase + G_BAR);
            mbar_inval(gbase + G_BAR_MMA);
        }
        named_sync(kBarSolve, kSolveWarps * 32);
    }
}

}  // namespace solve
}  // namespace gdr
