// channel_tc.cuh -- the chunk-parallel half of the tensor-core prefill with one forget
// rate per key channel (bf16, d_k = d_v = 128): every operand of the chain, per
// (chunk, head) unit.
//
// With one rate per token, head and key channel (Kimi Delta Attention, "Attention as
// Matrix Algebra: From Softmax to the Delta Rule", section 10) row c of the state decays
// by alpha_t[c], and the chunk form of section 8 keeps its shape with the decay moved
// into the key channels. Per chunk of C = 64 tokens, g_t[c] = sum_{i <= t} log alpha_i[c]:
//   L_ti = beta_t sum_c k_t[c] k_i[c] exp(g_t[c] - g_i[c])   (i < t)
//   A_ti =        sum_c q_t[c] k_i[c] exp(g_t[c] - g_i[c])   (i <= t)
//   T = (I + L)^{-1} diag(beta),  W = T (e^g . K),  Utilde = T V
//   U = Utilde - W S,  O = (e^g . Q) S + A U,  S <- diag(e^{g_C}) S + (e^{g_C - g} . K)^T U
// (e^g . K: row t scaled by exp(g_t[c]) in channel c). Every factor in the last three
// lines is at most 1.
//
// The Gram entries factor around a reference token r of the chunk (token 31):
// exp(g_t[c] - g_i[c]) = exp(g_t[c] - g_r[c]) exp(g_r[c] - g_i[c]), so that
//   [L/beta; A] = [K'; Q'] K''^T,  K' = e^{g - g_r} . K,  Q' = e^{g - g_r} . Q,
//   K'' = e^{g_r - g} . K,
// one tcgen05 MMA chain (M = 128, N = 64, K = d_k). The factors can exceed 1 but stay
// finite while -g_r[c] < 80 and g_r[c] - g_C[c] < 80 in every channel; a chunk that
// decays further (over about e^-160 in some channel) takes every entry as its own sum
// with exp(g_t[c] - g_i[c]) <= 1 on the CUDA cores instead. W is formed from K' too,
// W = T K' with column c scaled by exp(g_r[c]) on the way out (exp(0) without the
// factored Gram).
//
// With the layer prologue ("Linear attention", "A naive PyTorch implementation") the rates
// and beta arrive as pre-activations, log alpha = -A_h softplus(a) per channel and
// beta = sigmoid(b), and q, k are scaled to unit length per token: the kernel takes the
// norms from the staged bf16 rows and scales every row it writes, so that the chain
// needs no change.
//
// Four warps per CTA, four CTAs per SM (52 KB of shared memory and 128 TMEM columns each),
// each CTA taking units blockIdx.x, blockIdx.x + gridDim.x, ... in turn; TMEM lane quarter
// w belongs to warp w. Outputs (the chain kernel loads them by TMA, 128-byte swizzled
// 64 x 64 boxes):
//   QW [units * 64][256] bf16: e^g . Q in columns 0..127, -W in columns 128..255;
//   KT [units * 64][128] bf16: e^{g_C - g} . K;
//   UT [units * 128][64] bf16: Utilde^T (row j: value column j over the chunk's tokens);
//   AT [units][2][64][64] bf16: A^T in matrix 2u + 1 (row i, column t);
//   G  [units][384] fp32: exp(g_C[c]) in floats 0..127.
// Padding rows of a partial last chunk get log alpha = 0 and beta = 0: their rows of T,
// W, Utilde are zero and they change nothing.
#pragma once

#include "solve_tc.cuh"

namespace gdr {
namespace channel {

using namespace sm100;
using namespace tc;
using solve::Acc16;
using solve::blk;
using solve::el;
using solve::invert_unit;
using solve::nblk;

constexpr int C = kChunk;
constexpr int DK = 128, DV = 128;
constexpr int kThreads = 128;
constexpr int kCtasPerSm = 4;  // resident CTAs per SM (shared memory and TMEM are sized for it)
// The reference token of the factored Gram, and the bound that keeps its factors finite.
constexpr int kRefToken = 31;
constexpr float kFactorLogBound = 80.f;

// Shared memory map (bytes from a 1024-aligned base). Regions are reused as the unit
// moves on: V is loaded over the query rows once Q is spent (after the Gram MMA, or after
// the element-wise pass without the factored Gram); the blocks of the inverse go over
// K'' once the Gram has completed, and T' over the blocks once every warp holds its
// block row in registers.
constexpr uint32_t P_KQ = 0;       // per d_k half b at 16384 b: 64 key rows, then 64 query rows
constexpr uint32_t P_V = 8192;     // V's 64-column halves at P_V and P_V + 16384
constexpr uint32_t P_KC = 32768;   // the Gram's B operand K'': two 64-column halves of 8 KB
constexpr uint32_t P_BLK = P_KC;   // the unit's 16 x 16 blocks (the solve's layout)
constexpr uint32_t P_TP = P_KC;    // T' bf16 [t][i], 128-byte swizzled
constexpr uint32_t P_MISC = P_KC + (solve::UNIT_FLOATS * 4 + 1023) / 1024 * 1024;
                                   // floats: beta[64], g_C[128], g_r[128], the prologue's
                                   // 1/|k_t|[64] and 1/|q_t|[64],
                                   // the "V load gave up" flag
constexpr int M_BETA = 0, M_GC = 64, M_GREF = 192, M_RK = 320, M_RQ = 384, M_FLAG = 448;
constexpr uint32_t P_BARS = P_MISC + 456 * 4;  // load, Gram, products, V reload, drain
constexpr uint32_t P_TMEM = P_BARS + 40;
constexpr uint32_t P_USED = P_TMEM + 16;
constexpr uint32_t SMEM_BYTES = P_USED + 1024;
static_assert(P_TP % 1024 == 0 && P_BARS % 8 == 0 && SMEM_BYTES + 1024 <= 233472 / kCtasPerSm,
              "shared memory: four CTAs per SM");
// TMEM columns: the Gram, then W^T in the same columns once the Gram is read; Utilde^T
constexpr uint32_t TM_GRAM = 0, TM_W = 0, TM_UT = 64, TM_COLS = 128;

struct ChannelParams {
    const float *log_alpha;  // [tokens, H, DK]
    const float *beta;       // [tokens, H]
    const int4 *plan;        // per chunk: sequence, first token, tokens, index
    int32_t *ctl;
    int H;
    int additive;            // the additive rule: L = 0, W = 0
    const float *gate_A;     // the layer prologue's per-head rate A_h (null: 1)
    __nv_bfloat16 *QW, *KT, *UT, *AT;
    float *G;
    long long wait_cycles;   // bound of every wait (SM cycles)
    int rates_vec;           // log_alpha starts on a 16-byte boundary (every row then does):
                             // its rows are read 16 bytes at a time, else 4
    int prefetch_rates;      // map_la is a tensor map of log_alpha (needs a 16-byte base)
    int fault_chunk;         // test knob: head 0's CTA of this chunk skips its key and query
                             // loads, so that its wait gives up (-1: never)
};

// Element (row, col) of a 128-byte-swizzled block of 64-wide bf16 rows at `block`.
__device__ __forceinline__ float sw_elem(const unsigned char *block, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(block + sw128_offset(row, col)));
}

// Brings the box of `map` at (c0, c1, c2) into L2: a hint with no completion to wait for.
__device__ __forceinline__ void prefetch_box_l2(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// The two bf16 halves of a packed pair, as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x and 1/x from the hardware approximations (about 2 ulp; subnormal results flush to
// zero). Every value they see here is within e^{+-80}.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// T' = (I + L)^{-1} diag(beta), block row W of warp W, as bf16 into the swizzled [t][i]
// tile `tp` (the B operand of the products; zeros right of the diagonal). The tile lies
// over the blocks: every warp reads its row into registers, then `sync` (the whole CTA),
// then the stores.
template <int W, typename Sync>
__device__ __forceinline__ void store_t_prime(const float *__restrict__ U, const float *__restrict__ beta,
                                              unsigned char *tp, int lane, Sync sync) {
    const int gq = lane >> 2, q = lane & 3;
    float2 lo[4][2], hi[4][2];
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            lo[bi][nt] = hi[bi][nt] = make_float2(0.f, 0.f);
            if (bi <= W) {
                const float *B = U + (bi == W ? blk(W, W) : nblk(W > bi ? W : 1, W > bi ? bi : 0));
                lo[bi][nt] = *reinterpret_cast<const float2 *>(B + el(gq, 8 * nt + 2 * q));
                hi[bi][nt] = *reinterpret_cast<const float2 *>(B + el(gq + 8, 8 * nt + 2 * q));
            }
        }
    }
    sync();
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int i0 = 16 * bi + 8 * nt + 2 * q;
            const float b0 = beta[i0], b1 = beta[i0 + 1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = 16 * W + gq + 8 * hh;
                const float2 v = hh ? hi[bi][nt] : lo[bi][nt];
                const float x0 = i0 <= t ? v.x * b0 : 0.f;
                const float x1 = i0 + 1 <= t ? v.y * b1 : 0.f;
                *reinterpret_cast<uint32_t *>(tp + sw128_offset(t, i0)) = pack_bf16x2(x0, x1);
            }
        }
    }
}

// A persistent CTA over units (chunk-major, head-minor). map_q, map_k, map_v: the inputs;
// map_la: the rates, when p.prefetch_rates (used only to bring the next unit's into L2).
// kPro: the layer prologue (a compile-time variant, so that the plain path carries none
// of its work).
template <bool kPro>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
channel_prep_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_la,
                    const ChannelParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *misc = reinterpret_cast<float *>(sm + P_MISC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P_TMEM);
    auto bar = [&](int i) { return sb + P_BARS + 8u * (uint32_t)i; };
    auto wait = [&](int i, uint32_t parity) { return mbar_wait_for(bar(i), parity, p.wait_cycles); };
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bar(i), 1);
        misc[M_FLAG] = 0.f;
        fence_mbar_init();
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        if (p.prefetch_rates) prefetch_tensormap(&map_la);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // Everything above overlaps the tail of the planning kernel (programmatic launch).
    griddep_wait();
    griddep_launch_dependents();
    const int n_chunks = p.ctl[0] == GDR_OK ? p.ctl[1] : 0;
    const int64_t n_units = (int64_t)n_chunks * p.H;
    bool fail = false;
    // Barrier phases (a barrier completes once for each unit that uses it), and (thread 0,
    // which issues every copy) the copies issued and not yet seen landed: a failure drains
    // those before the shared memory goes.
    uint32_t ph_kq = 0, ph_gram = 0, ph_mma = 0, ph_v = 0;
    bool kq_pending = false, v_pending = false;
    // the keys and queries of unit x (chunk-major, head-minor), whose first token is t0x,
    // unless the test knob drops them; thread 0
    auto issue_kq = [&](int64_t x, int t0x) {
        const int cx = (int)(x / p.H), hx = (int)(x % p.H);
        if (cx == p.fault_chunk && hx == 0) return;
        mbar_arrive_expect_tx(bar(0), 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sb + P_KQ + 16384 * b, &map_k, bar(0), 64 * b, hx, t0x);
            tma_load_3d(sb + P_KQ + 16384 * b + 8192, &map_q, bar(0), 64 * b, hx, t0x);
        }
        kq_pending = true;
    };
    if (tid == 0 && (int64_t)blockIdx.x < n_units) issue_kq(blockIdx.x, p.plan[blockIdx.x / p.H].y);
    // Units blockIdx.x, blockIdx.x + gridDim.x, ...: the next unit's keys and queries are
    // copied in while this one's outputs are stored.
    for (int64_t x = blockIdx.x; x < n_units; x += gridDim.x) {
        const int c = (int)(x / p.H), h = (int)(x % p.H);
        const int4 pl = p.plan[c];
        const int t0 = pl.y, len = pl.z;
        const size_t u = (size_t)x;
        const int64_t x_next = x + gridDim.x;
        // the next unit's first token: thread 0 copies its keys and queries in and brings
        // its rates into L2 while this unit's outputs are stored
        const int t0_next = (tid == 0 && x_next < n_units) ? p.plan[x_next / p.H].y : 0;
        if (tid == 0) misc[M_FLAG] = 0.f;
        // V over the query rows, once they are spent
        auto load_v = [&] {
            mbar_arrive_expect_tx(bar(3), 2 * 8192);
            tma_load_3d(sb + P_V, &map_v, bar(3), 0, h, t0);
            tma_load_3d(sb + P_V + 16384, &map_v, bar(3), 64, h, t0);
            v_pending = true;
        };
        if (tid < C) {
            float bt = 0.f;
            if (tid < len) {
                bt = p.beta[(size_t)(t0 + tid) * p.H + h];
                if (kPro) bt = prologue_beta(bt);
            }
            misc[M_BETA + tid] = bt;
        }
        const float gate_a = kPro && p.gate_A ? p.gate_A[h] : 1.f;
        // g by tiles: thread (o, grp) owns channels 8o .. 8o + 7 over tokens 8grp .. 8grp + 7
        const int o = tid & 15, grp = tid >> 4;
        float g[8][8];
        {
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = 8 * grp + j;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                if (t < len) {
                    const float *src = p.log_alpha + ((size_t)(t0 + t) * p.H + h) * DK + 8 * o;
                    if (p.rates_vec) {
                        a = reinterpret_cast<const float4 *>(src)[0];
                        b = reinterpret_cast<const float4 *>(src)[1];
                    } else {
                        a = make_float4(src[0], src[1], src[2], src[3]);
                        b = make_float4(src[4], src[5], src[6], src[7]);
                    }
                    if (kPro) {  // log alpha = -A_h softplus(a), per channel
                        a = make_float4(prologue_log_alpha(a.x, gate_a), prologue_log_alpha(a.y, gate_a),
                                        prologue_log_alpha(a.z, gate_a), prologue_log_alpha(a.w, gate_a));
                        b = make_float4(prologue_log_alpha(b.x, gate_a), prologue_log_alpha(b.y, gate_a),
                                        prologue_log_alpha(b.z, gate_a), prologue_log_alpha(b.w, gate_a));
                    }
                }
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
#pragma unroll
                for (int e = 0; e < 8; ++e) g[j][e] = acc[e];
            }
            // each group's sums, over K'' (written only after the scan)
            float4 *sums = reinterpret_cast<float4 *>(sm + P_KC) + (grp * DK + 8 * o) / 4;
            sums[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            sums[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        __syncthreads();
        {
            float base[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) base[e] = 0.f;
            const float4 *sums = reinterpret_cast<const float4 *>(sm + P_KC) + 2 * o;
            for (int gg = 0; gg < grp; ++gg) {
                const float4 a = sums[gg * (DK / 4)], b = sums[gg * (DK / 4) + 1];
                base[0] += a.x; base[1] += a.y; base[2] += a.z; base[3] += a.w;
                base[4] += b.x; base[5] += b.y; base[6] += b.z; base[7] += b.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) g[j][e] += base[e];
            float4 *gref = reinterpret_cast<float4 *>(misc + M_GREF + 8 * o);
            float4 *gcs = reinterpret_cast<float4 *>(misc + M_GC + 8 * o);
            constexpr int jr = kRefToken % 8;
            if (grp == kRefToken / 8) {
                gref[0] = make_float4(g[jr][0], g[jr][1], g[jr][2], g[jr][3]);
                gref[1] = make_float4(g[jr][4], g[jr][5], g[jr][6], g[jr][7]);
            }
            if (grp == 7) {
                gcs[0] = make_float4(g[7][0], g[7][1], g[7][2], g[7][3]);
                gcs[1] = make_float4(g[7][4], g[7][5], g[7][6], g[7][7]);
            }
        }
        __syncthreads();
        float gc[8], gr[8];
        bool col_ok = true;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            gc[e] = misc[M_GC + 8 * o + e];
            gr[e] = misc[M_GREF + 8 * o + e];
            col_ok = col_ok && -gr[e] < kFactorLogBound && gr[e] - gc[e] < kFactorLogBound;
        }
        const bool factored = __syncthreads_and(col_ok) != 0;
        if (!wait(0, ph_kq)) {
            fail = true;
        } else {
            ph_kq ^= 1;
            kq_pending = false;
        }
        fail = __syncthreads_or(fail) != 0;
        if (!fail && kPro) {
            // 1/|k_t| and 1/|q_t| from the staged bf16 rows: the 16 threads of a token group
            // (one half-warp) each sum 8 channels, then combine
            const int b = o >> 3, cc = o & 7;
            const unsigned char *kh = sm + P_KQ + 16384 * b, *qh = kh + 8192;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = 8 * grp + j;
                const uint32_t off = (uint32_t)(t * 128 + ((cc ^ (t & 7)) << 4));
                const uint4 kr = *reinterpret_cast<const uint4 *>(kh + off);
                const uint4 qr = *reinterpret_cast<const uint4 *>(qh + off);
                const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qv[4] = {qr.x, qr.y, qr.z, qr.w};
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float k0 = bf16_lo(kw[w]), k1 = bf16_hi(kw[w]);
                    const float q0 = bf16_lo(qv[w]), q1 = bf16_hi(qv[w]);
                    sk = fmaf(k0, k0, fmaf(k1, k1, sk));
                    sq = fmaf(q0, q0, fmaf(q1, q1, sq));
                }
#pragma unroll
                for (int off2 = 1; off2 < 16; off2 <<= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, off2);
                    sq += __shfl_xor_sync(0xffffffffu, sq, off2);
                }
                if (o == 0) {
                    misc[M_RK + t] = prologue_inv_norm(sk);
                    misc[M_RQ + t] = prologue_inv_norm(sq);
                }
            }
            __syncthreads();
        }
        float *U = reinterpret_cast<float *>(sm + P_BLK);
        __nv_bfloat16 *arow = p.AT + (u * 2 + 1) * C * C;
        if (!fail && !factored) {
            // ---- the unfactored Gram on the CUDA cores, every entry as its own sum. g goes
            // to the unit's slot of QW in the workspace (fp32 [C][DK], 32 KB), which the
            // element-wise pass below fills only after this loop has read it.
            float *gs = reinterpret_cast<float *>(p.QW + (u * C) * 256);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 *row = reinterpret_cast<float4 *>(gs + (8 * grp + j) * DK + 8 * o);
                row[0] = make_float4(g[j][0], g[j][1], g[j][2], g[j][3]);
                row[1] = make_float4(g[j][4], g[j][5], g[j][6], g[j][7]);
            }
            for (int e = tid; e < 10 * solve::BS; e += kThreads) U[e] = 0.f;  // the ten L blocks
            __syncthreads();
            for (int e = tid; e < C * C; e += kThreads) {
                const int t = e >> 6, i = e & 63;  // A^T row i, column t: this thread's entry
                float kk = 0.f, qk = 0.f;
                if (i <= t) {
                    for (int d = 0; d < DK; ++d) {
                        const unsigned char *half = sm + P_KQ + 16384 * (d >> 6);
                        const float f = fast_exp(gs[t * DK + d] - gs[i * DK + d]);
                        const float ki = sw_elem(half, i, d & 63) * f;
                        kk = fmaf(sw_elem(half, t, d & 63), ki, kk);
                        qk = fmaf(sw_elem(half + 8192, t, d & 63), ki, qk);
                    }
                    if (kPro) {
                        const float rki = misc[M_RK + i];
                        kk *= misc[M_RK + t] * rki;
                        qk *= misc[M_RQ + t] * rki;
                    }
                    if (i < t && !p.additive) U[blk(t >> 4, i >> 4) + el(t & 15, i & 15)] = misc[M_BETA + t] * kk;
                }
                arow[i * C + t] = __float2bfloat16_rn(qk);
            }
            __syncthreads();  // every read of the g table before the QW stores below
        }
        if (!fail) {
            // ---- element-wise: the chain's e^g . Q and e^{g_C - g} . K to the workspace,
            // the products' tiles in place: K' = e^{g - sh} . K (and with the factored Gram
            // Q' = e^{g - sh} . Q, K'' = e^{sh - g} . K), sh = g_r with the factored Gram,
            // else 0. Thread (o, grp): one 16-byte row segment of 8 channels per token.
            // With the factored Gram every factor comes from s = e^{g - g_r} (within e^{+-80}):
            // e^{g - g_r} = s, e^{g_r - g} = 1 / s, e^g = e^{g_r} s, e^{g_C - g} = e^{g_C - g_r} / s.
            const int b = o >> 3, cc = o & 7;
            unsigned char *kh = sm + P_KQ + 16384 * b, *qh = kh + 8192, *kc = sm + P_KC + 8192 * b;
            __nv_bfloat16 *qw = p.QW + (u * C) * 256 + 8 * o;
            __nv_bfloat16 *kt = p.KT + (u * C) * DK + 8 * o;
            constexpr float kLog2e = 1.4426950408889634f;
            if (factored) {
                float shl[8], eq[8], ek[8];  // -g_r log2(e), e^{g_r}, e^{g_C - g_r}
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    shl[e] = -gr[e] * kLog2e;
                    eq[e] = fast_exp(gr[e]);
                    ek[e] = fast_exp(gc[e] - gr[e]);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = 8 * grp + j;
                    const uint32_t off = (uint32_t)(t * 128 + ((cc ^ (t & 7)) << 4));
                    const uint4 kr = *reinterpret_cast<const uint4 *>(kh + off);
                    const uint4 qr = *reinterpret_cast<const uint4 *>(qh + off);
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qv[4] = {qr.x, qr.y, qr.z, qr.w};
                    const float rk = kPro ? misc[M_RK + t] : 1.f, rq = kPro ? misc[M_RQ + t] : 1.f;
                    uint32_t o_qw[4], o_kt[4], o_k1[4], o_q1[4], o_k2[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float k0 = bf16_lo(kw[w]) * rk, k1 = bf16_hi(kw[w]) * rk;
                        const float q0 = bf16_lo(qv[w]) * rq, q1 = bf16_hi(qv[w]) * rq;
                        const int e0 = 2 * w, e1 = 2 * w + 1;
                        const float s0 = fast_exp2(fmaf(g[j][e0], kLog2e, shl[e0]));
                        const float s1 = fast_exp2(fmaf(g[j][e1], kLog2e, shl[e1]));
                        const float r0 = fast_rcp(s0), r1 = fast_rcp(s1);
                        o_qw[w] = pack_bf16x2(q0 * s0 * eq[e0], q1 * s1 * eq[e1]);
                        o_kt[w] = pack_bf16x2(k0 * r0 * ek[e0], k1 * r1 * ek[e1]);
                        o_k1[w] = pack_bf16x2(k0 * s0, k1 * s1);
                        o_q1[w] = pack_bf16x2(q0 * s0, q1 * s1);
                        o_k2[w] = pack_bf16x2(k0 * r0, k1 * r1);
                    }
                    *reinterpret_cast<uint4 *>(qw + (size_t)t * 256) = make_uint4(o_qw[0], o_qw[1], o_qw[2], o_qw[3]);
                    *reinterpret_cast<uint4 *>(kt + (size_t)t * DK) = make_uint4(o_kt[0], o_kt[1], o_kt[2], o_kt[3]);
                    *reinterpret_cast<uint4 *>(kh + off) = make_uint4(o_k1[0], o_k1[1], o_k1[2], o_k1[3]);
                    *reinterpret_cast<uint4 *>(qh + off) = make_uint4(o_q1[0], o_q1[1], o_q1[2], o_q1[3]);
                    *reinterpret_cast<uint4 *>(kc + off) = make_uint4(o_k2[0], o_k2[1], o_k2[2], o_k2[3]);
                }
            } else {
                // each factor as its own exponential (no factor above 1 to divide by)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = 8 * grp + j;
                    const uint32_t off = (uint32_t)(t * 128 + ((cc ^ (t & 7)) << 4));
                    const uint4 kr = *reinterpret_cast<const uint4 *>(kh + off);
                    const uint4 qr = *reinterpret_cast<const uint4 *>(qh + off);
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qv[4] = {qr.x, qr.y, qr.z, qr.w};
                    const float rk = kPro ? misc[M_RK + t] : 1.f, rq = kPro ? misc[M_RQ + t] : 1.f;
                    uint32_t o_qw[4], o_kt[4], o_k1[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float k0 = bf16_lo(kw[w]) * rk, k1 = bf16_hi(kw[w]) * rk;
                        const float q0 = bf16_lo(qv[w]) * rq, q1 = bf16_hi(qv[w]) * rq;
                        const int e0 = 2 * w, e1 = 2 * w + 1;
                        const float x0 = fast_exp(g[j][e0]), x1 = fast_exp(g[j][e1]);
                        o_qw[w] = pack_bf16x2(q0 * x0, q1 * x1);
                        o_kt[w] = pack_bf16x2(k0 * fast_exp(gc[e0] - g[j][e0]), k1 * fast_exp(gc[e1] - g[j][e1]));
                        o_k1[w] = pack_bf16x2(k0 * x0, k1 * x1);
                    }
                    *reinterpret_cast<uint4 *>(qw + (size_t)t * 256) = make_uint4(o_qw[0], o_qw[1], o_qw[2], o_qw[3]);
                    *reinterpret_cast<uint4 *>(kt + (size_t)t * DK) = make_uint4(o_kt[0], o_kt[1], o_kt[2], o_kt[3]);
                    *reinterpret_cast<uint4 *>(kh + off) = make_uint4(o_k1[0], o_k1[1], o_k1[2], o_k1[3]);
                }
            }
            fence_async_smem();
            __syncthreads();
            if (!factored && tid == 0) load_v();  // the query rows are spent
            if (factored) {
                if (tid == 0) {  // [K'; Q'] K''^T: row t < 64 of D is L_t. / beta_t, row 64 + t is A_t.
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t at = sb + P_KQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t bt = sb + P_KC + (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_bf16(tmem + TM_GRAM, sw128_desc(at, 16, 1024), sw128_desc(bt, 16, 1024),
                                 idesc_bf16(128, 64, 0, 0), kk > 0);
                    }
                    mma_commit(bar(1));
                }
                if (!wait(1, ph_gram)) fail = true;
                ph_gram ^= 1;
                // a Gram that did not complete is neither read nor written over
                fail = __syncthreads_or(fail) != 0;
            }
            if (factored && !fail) {
                if (tid == 0) load_v();  // the query rows are spent
                tc_fence_after();
                // the Gram's rows, warp w on TMEM lanes 32w .. 32w + 31, 16 columns at a time
                const uint32_t lanes = tmem + TM_GRAM + ((uint32_t)(32 * warp) << 16);
                if (warp < 2) {
                    const int t = 32 * warp + lane, br = t >> 4, r = t & 15;
                    const float rb = p.additive ? 0.f : misc[M_BETA + t];
#pragma unroll 1
                    for (int jb = 0; jb <= 2 * warp + 1; ++jb) {  // warp-uniform trip count
                        float d[16];
                        tmem_load16(lanes + 16 * jb, d);
                        if (jb > br) continue;
                        float *B = U + blk(br, jb);
#pragma unroll
                        for (int cg = 0; cg < 4; ++cg) {
                            float v[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) v[e] = 16 * jb + 4 * cg + e < t ? rb * d[4 * cg + e] : 0.f;
                            *reinterpret_cast<float4 *>(B + el(r, 4 * cg)) = make_float4(v[0], v[1], v[2], v[3]);
                        }
                    }
                } else {
                    // A^T_it for keys i <= t: neighbouring lanes swap one value per key pair
                    // so that each store is a bf16 pair along the queries t
                    const int t = 32 * (warp - 2) + lane;
                    const bool odd = lane & 1;
                    __nv_bfloat16 *ar = arow + (t & ~1);
#pragma unroll 1
                    for (int kb = 0; kb < 4; ++kb) {
                        float d[16];
                        tmem_load16(lanes + 16 * kb, d);
#pragma unroll
                        for (int pp = 0; pp < 8; ++pp) {
                            const int i0 = 16 * kb + 2 * pp;
                            const float v0 = i0 <= t ? d[2 * pp] : 0.f;
                            const float v1 = i0 + 1 <= t ? d[2 * pp + 1] : 0.f;
                            const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                            *reinterpret_cast<uint32_t *>(ar + (i0 + (odd ? 1 : 0)) * C) =
                                odd ? pack_bf16x2(recv, v1) : pack_bf16x2(v0, recv);
                        }
                    }
                }
                tc_fence_before();  // the reads come before W^T's MMA into the same columns
            }
            fail = __syncthreads_or(fail) != 0;  // (also: the L blocks are complete)
        }
        if (!fail) {
            // ---- (I + L)^{-1}, then T' = (I + L)^{-1} diag(beta) into the swizzled tile
            auto sync4 = [] { __syncthreads(); };
            auto none = [] {};
            const float *beta_s = misc + M_BETA;
            unsigned char *tp = sm + P_TP;
            switch (warp) {
                case 0: invert_unit<0>(U, lane, sync4, none); store_t_prime<0>(U, beta_s, tp, lane, sync4); break;
                case 1: invert_unit<1>(U, lane, sync4, none); store_t_prime<1>(U, beta_s, tp, lane, sync4); break;
                case 2: invert_unit<2>(U, lane, sync4, none); store_t_prime<2>(U, beta_s, tp, lane, sync4); break;
                default: invert_unit<3>(U, lane, sync4, none); store_t_prime<3>(U, beta_s, tp, lane, sync4); break;
            }
            fence_async_smem();
            __syncthreads();
            // ---- W^T = K'^T T'^T (M = d_k) and Utilde^T = V^T T'^T (M = d_v)
            if (tid == 0) {
                const bool v_ok = wait(3, ph_v);
                if (v_ok) {
                    ph_v ^= 1;
                    v_pending = false;
                }
                if (v_ok) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + TM_W, sw128_desc(sb + P_KQ + kk * 2048, 16384, 1024),
                                 sw128_desc(sb + P_TP + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + TM_UT, sw128_desc(sb + P_V + kk * 2048, 16384, 1024),
                                 sw128_desc(sb + P_TP + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
                    mma_commit(bar(2));
                } else {
                    misc[M_FLAG] = 1.f;  // (the V load gave up: nothing was issued)
                }
            }
            __syncthreads();
            const bool issued = misc[M_FLAG] == 0.f;
            if (!issued) fail = true;
            if (issued) {
                if (!wait(2, ph_mma)) fail = true;
                ph_mma ^= 1;
            }
            tc_fence_after();
            fail = __syncthreads_or(fail) != 0;
            if (!fail) {
                // the products have read K' and V: the next unit's keys and queries may land
                if (tid == 0 && x_next < n_units) {
                    issue_kq(x_next, t0_next);
                    if (p.prefetch_rates) prefetch_box_l2(&map_la, 0, (int)(x_next % p.H), t0_next);
                }
                // -W rows: lane j = d_k index of warp w's quarter; column t of W^T scaled by
                // exp(sh_j); lanes j, j ^ 1 swap one value per token pair so that each store
                // is a bf16 pair along d_k
                const int j = 32 * warp + lane;
                const bool odd = lane & 1;
                const float sc = p.additive ? 0.f : -fast_exp(factored ? misc[M_GREF + j] : 0.f);
                __nv_bfloat16 *wq = p.QW + (u * C) * 256 + 128 + (j & ~1);
                const uint32_t lw = tmem + TM_W + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
                for (int tb = 0; tb < 4; ++tb) {
                    float d[16];
                    tmem_load16(lw + 16 * tb, d);
#pragma unroll
                    for (int pp = 0; pp < 8; ++pp) {
                        const int tt = 16 * tb + 2 * pp;
                        const float v0 = sc * d[2 * pp], v1 = sc * d[2 * pp + 1];
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                        *reinterpret_cast<uint32_t *>(wq + (size_t)(tt + (odd ? 1 : 0)) * 256) =
                            odd ? pack_bf16x2(recv, v1) : pack_bf16x2(v0, recv);
                    }
                }
                // Utilde^T rows: lane j = value column, its 64 tokens as one 128-byte row
                const uint32_t lu = tmem + TM_UT + ((uint32_t)(32 * warp) << 16);
                uint4 *ur = reinterpret_cast<uint4 *>(p.UT + (u * DV + j) * C);
#pragma unroll 1
                for (int tb = 0; tb < 4; ++tb) {
                    float d[16];
                    tmem_load16(lu + 16 * tb, d);
                    ur[2 * tb] = make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                            pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7]));
                    ur[2 * tb + 1] = make_uint4(pack_bf16x2(d[8], d[9]), pack_bf16x2(d[10], d[11]),
                                                pack_bf16x2(d[12], d[13]), pack_bf16x2(d[14], d[15]));
                }
                // the state's decay over the chunk, per channel
                p.G[u * 384 + j] = fast_exp(misc[M_GC + j]);
            }
        }
        if (fail) {
            if (tid == 0) {
                atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
                // loads and MMAs still in flight land before the shared memory and TMEM go
                if (kq_pending) wait(0, ph_kq);
                if (v_pending) wait(3, ph_v);
                mma_commit(bar(4));
                wait(4, 0);
            }
            break;
        }
        // the unit's TMEM columns, blocks and gates are free for the next one
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace channel
}  // namespace gdr
