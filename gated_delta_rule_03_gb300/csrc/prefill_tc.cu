// prefill_tc.cu -- chunked prefill of the gated delta rule on the 5th-generation tensor
// cores (tcgen05), for bf16 q/k/v with d_k = 128 and d_v a multiple of 128: the
// sequential chain over the chunks of each (sequence, head), and the host launcher of
// the whole tensor-core path.
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
// The chunk-parallel part -- L and the triangular solve, giving T -- runs first, for all
// chunks at once (solve_tc.cu). This file holds everything that follows it.
//
// Two equivalent forms of the decay factors, chosen per chunk:
//  * ratio form, when the chunk's cumulative log-decay g_C (its minimum) stays above
//    -80 so that gamma and 1/gamma are finite normal floats. With kdec_t = exp(g_C - g_t)
//    and U' = diag(kdec) U the decay moves off Q and K:
//      T' = diag(kdec) T,  U' = T' V - T' diag(gamma) K S,  S_upd = K^T U',
//      O_t = gamma_t [ (S^T q_t) + (1/gamma_C) ((Q K^T . [i <= t]) U')_t ].
//  * exponential form otherwise: T' = T, U' = U, Gamma_ti = exp(g_t - g_i) per entry,
//    and the stage's Q rows are scaled by gamma and K rows by kdec in place.
// Both compute the same products; only the placement of the decay factors differs.
//
// Work mapping. One CTA per (sequence, head, 128-column slice of d_v); the value columns
// of S evolve independently. Every dense product is a tcgen05.mma chain with fp32
// accumulators in TMEM and bf16 operands either in 128-byte-swizzled shared memory or,
// for the two operands the chain itself produces (S^T and U'^T), in TMEM. A tcgen05.mma
// instruction costs about as much to issue whatever its N, so products that share an
// operand are issued as one wide chain:
//   U'~^T       = V^T T'^T,  W'^T = K^T (T' diag gamma)^T           (N = 64, K = 64)
//   [O^T | X^T] = S^T [Q; -W']^T               (A = S^T from TMEM;  N = 128, K = d_k)
//   [S^T | O^T] += U'^T [K | A^T]              (A = U'^T from TMEM; N = 192, K = 64)
// with U' = U'~ + X, all with M = d_v = 128. A^T (the causal, decay-weighted key-query
// products), T' and the chunk's decay factors (g, gamma, kdec and the form) come from
// the solve. Two tiles change orientation on the way (-W'^T into -W' rows next to Q,
// and O^T into o rows): both are read from TMEM in the m16n8 fragment layout and
// written transposed with stmatrix; o leaves by TMA store.
//
// Loads. Each input goes into a ring of its own, freed as soon as its last reader is
// done, so that the next chunks load while this one is worked on:
//   V, T'            2 slots, freed when U'~ and W' are done;
//   K, A^T, factors  3 slots, freed when the chunk is done;
//   Q (and -W')      2 slots, freed when [QS | WS] is done.
//
// Warp roles (18 warps; TMEM lane quarter = warp % 4):
//   warps 0-3   epilogue: O^T of chunk c from TMEM (times gamma_t in the ratio form),
//               transposed into a staging tile, stored by TMA.
//   warps 4-7   prep: T' diag(gamma), -W' into the Q slot, the in-place scaling of Q
//               and K (exponential form).
//   warps 8-15  state, the sequential chain: the bf16 S^T and U'^T operands in TMEM,
//               and the decay of the fp32 master S^T (in TMEM);
//   warp 17     the MMA issuer: [QS | WS] once S^T is in place, [S_upd | AU] once U'^T
//               is, and U'~, W' of the next chunk in between, where the tensor pipe would
//               otherwise wait for the state's conversion.
//   warp 16     producer: the TMA and bulk loads of the three rings, in chunk order, each
//               as soon as its slot is free.
// The critical path per chunk is: S^T copy -> [QS | WS] -> U'^T copy -> [S_upd | AU].
// The decay of the master by the next chunk's gamma_C runs while [QS | WS] does.
// Padding rows of a partial last chunk get log alpha = 0 and beta = 0: their rows of
// T', W', U' are zero, they change nothing and they are not stored.
// Every wait is bounded; a role that gives up marks the call GDR_ERR_DEVICE_TIMEOUT in
// the status word, and the others give up in turn, drain and free TMEM.
#include <stdlib.h>

#include <mutex>

#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace sm100;
using namespace tc;

constexpr int C = kChunk;   // 64 tokens per chunk
constexpr int DK = 128;     // key dimension
constexpr int NV = 128;     // value columns per CTA
constexpr int kWarps = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiThreads = 128;                      // warps 0-3
constexpr int kPrepWarp0 = 4, kPrepThreads = 128;     // warps 4-7
constexpr int kStateWarp0 = 8;   // warps 8-15
constexpr int kProducerWarp = 16, kMmaWarp = 17;
constexpr int kStateWarps = 8;
constexpr int kBarPrep = 1, kBarEpi = 3;  // named barrier ids

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t RQ = 0, RQ_SLOT = 32768;        // per d_k half b (16 KB): Q_b then -W'_b
constexpr uint32_t RK = 65536, RK_SLOT = 25600;    // K_b0 | K_b1 | A^T (8 KB each) | factors
constexpr uint32_t RK_A = 16384, RK_G = 24576;     // offsets of A^T and the factors in a K slot
constexpr uint32_t RV = RK + 3 * RK_SLOT, RV_SLOT = 24576;  // V_b0 | V_b1 | T'
constexpr uint32_t RV_T = 16384;
constexpr int G_GAM = 64, G_KDEC = 128, G_FORM = 192;  // float offsets in the factors (g at 0)
constexpr uint32_t OFF_TG = RV + 2 * RV_SLOT;   // T' diag(gamma) bf16 [t][i]
constexpr uint32_t OFF_OST = OFF_TG + 8192;     // output staging [t][128]: two 8 KB tiles
constexpr uint32_t OFF_EG = OFF_OST + 16384;    // epilogue gates: gamma[4][64], form flag[4]
constexpr uint32_t OFF_BAR = OFF_EG + 2048;
static_assert(RK % 1024 == 0 && RK_SLOT % 1024 == 0 && RV % 1024 == 0 && OFF_TG % 1024 == 0 &&
                  OFF_OST % 1024 == 0,
              "alignment");

// mbarrier slots at OFF_BAR (8 bytes each), then the TMEM slot and role flags.
enum {
    B_QF0 = 0, B_QF1,        // Q slot loaded                              (tx bytes)
    B_QE0, B_QE1,            // Q slot free: [QS | WS] done                (MMA warp commit)   
    B_KF0, B_KF1, B_KF2,     // K slot loaded                              (tx bytes)
    B_KE0, B_KE1, B_KE2,     // K slot free: chunk done (prep 128 arrivals + state commit)
    B_VF0, B_VF1,            // V slot loaded                              (tx bytes)
    B_VE0, B_VE1,            // V slot free: U'~ and W' done               (MMA warp commit)
    B_WD0, B_WD1,            // W' of chunk c done                         (MMA warp commit)
    B_WQ0, B_WQ1,            // -W' of chunk c stored, Q/K scaled          (128 prep arrivals)
    B_WS,                    // [QS | WS] done                             (MMA warp commit)   
    B_SO,                    // [S_upd | AU] done                          (MMA warp commit)   
    B_OFREE,                 // O read by the epilogue                     (128 arrivals)
    B_TGR0, B_TGR1,          // T' diag(gamma) of chunk c staged           (128 prep arrivals)
    B_SREADY, B_UREADY,      // S^T / U'^T operands written to TMEM        (8 state warps)
    B_EG0, B_EG1, B_EG2, B_EG3,  // epilogue gates of chunk c in slot c%4  (128 prep arrivals)
    B_DRAIN,                 // drain after an abort
    B_COUNT
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t OFF_FLAGS = OFF_TMEM_SLOT + 4;  // int: prep, state, epilogue, any failure
constexpr uint32_t SMEM_USED = OFF_FLAGS + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for the 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory");

// TMEM columns (fp32 over 128 lanes unless noted). [S | O] and [O | X] are each one
// MMA's D; U'^T (bf16 pairs) is written over X once X has been read.
constexpr uint32_t TM_S = 0, TM_O = 128, TM_X = 192, TM_U = 256 /* two buffers */, TM_W = 384,
                   TM_SA = 448 /* S^T as bf16 pairs */, TM_COLS = 512;


struct TcParams {
    const float *S_in;         // state before this phase's chunks (null: zero)
    const float *factors;      // per solve unit: g, gamma, kdec, form (256 floats)
    const int32_t *cu_seqlens;
    const int32_t *seq_chunk;  // first chunk of each sequence in this phase (planning kernel)
    int64_t num_seqs, total_tokens;
    int H, dv, n_slices;
    int phase, phases;         // this launch runs chunks [floor(f m / P), floor((f+1) m / P))
    __nv_bfloat16 *o;
    float *S_out;              // state after this phase's chunks (may alias S_in)
    int32_t *ctl;
};

// Shared address of the 16-byte row segment (row r, 8 columns from c8*8) of a
// 128-byte-swizzled block of 64-wide bf16 rows.
__device__ __forceinline__ uint32_t sw128_seg(uint32_t block, int r, int c8) {
    return block + (uint32_t)(r * 128 + (((c8 ^ r) & 7) << 4));
}

// Writes a 16-lane x 64-column fp32 TMEM tile (fragment registers of
// tmem_load_16x256b_x8, times `scale`) transposed: the element at (lane l, column t) goes
// to row t, column l of 128-byte-swizzled bf16 rows. row_block(l8) gives the block that
// holds the 8-column segment starting at lane l8 and its segment index within the row.
template <typename RowBlock>
__device__ __forceinline__ void transpose_store16(const uint32_t (&r)[32], float scale_sign,
                                                  const float *col_scale, int lane, int l0,
                                                  RowBlock row_block) {
    const int i = lane >> 3, rr = lane & 7;  // this thread addresses row rr of matrix i
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        uint32_t p[4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int j = 2 * jj + m;  // column block
            const int t0 = 8 * j + 2 * (lane & 3);
            const float s0 = col_scale ? col_scale[t0] * scale_sign : scale_sign;
            const float s1 = col_scale ? col_scale[t0 + 1] * scale_sign : scale_sign;
            p[2 * m] = pack_bf16x2(__uint_as_float(r[4 * j]) * s0, __uint_as_float(r[4 * j + 1]) * s1);
            p[2 * m + 1] = pack_bf16x2(__uint_as_float(r[4 * j + 2]) * s0, __uint_as_float(r[4 * j + 3]) * s1);
        }
        // matrix i: lanes l0 + 8(i & 1) .. +7, columns 8(2jj + (i >> 1)) .. +7
        const int row = 8 * (2 * jj + (i >> 1)) + rr;
        uint32_t block;
        int c8;
        row_block(l0 + 8 * (i & 1), block, c8);
        stmatrix_x4_trans(sw128_seg(block, row, c8), p[0], p[1], p[2], p[3]);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_t,
                const __grid_constant__ CUtensorMap map_o, const TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that every access
    // through it stays a shared-memory access the compiler can schedule freely
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM_SLOT);
    volatile int *flags = reinterpret_cast<volatile int *>(sm + OFF_FLAGS);
    auto note_fail = [&](int role) { flags[role] = 1; flags[3] = 1; };

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
    // this phase's chunks of the sequence: local chunk c is the sequence's chunk cb + c
    const int64_t m = (seq_end - seq_begin + C - 1) / C;
    const int64_t cb = (int64_t)p.phase * m / p.phases;
    const int n_chunks = (int)((int64_t)(p.phase + 1) * m / p.phases - cb);
    seq_begin += cb * C;
    const int col0 = slice * NV;  // first value column of this CTA
    auto chunk_len = [&](int c) {
        const int64_t rem = seq_end - (seq_begin + (int64_t)c * C);
        return (int)(rem < C ? rem : C);
    };
    // ring slots of chunk c
    auto qslot = [&](int c) { return (uint32_t)(RQ + (c & 1) * RQ_SLOT); };
    auto kslot = [&](int c) { return (uint32_t)(RK + (c % 3) * RK_SLOT); };
    auto vslot = [&](int c) { return (uint32_t)(RV + (c & 1) * RV_SLOT); };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_QF0 + i), 1);
            mbar_init(bar(B_QE0 + i), 1);
            mbar_init(bar(B_VF0 + i), 1);
            mbar_init(bar(B_VE0 + i), 1);
            mbar_init(bar(B_WD0 + i), 1);
            mbar_init(bar(B_WQ0 + i), kPrepThreads);
            mbar_init(bar(B_TGR0 + i), kPrepThreads);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(bar(B_KF0 + i), 1);
            mbar_init(bar(B_KE0 + i), kPrepThreads + 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(B_EG0 + i), kPrepThreads);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_WS), 1);
        mbar_init(bar(B_SO), 1);
        mbar_init(bar(B_OFREE), kEpiThreads);
        mbar_init(bar(B_SREADY), kStateWarps);
        mbar_init(bar(B_UREADY), kStateWarps);
        fence_mbar_init();
        flags[0] = flags[1] = flags[2] = flags[3] = 0;
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        prefetch_tensormap(&map_t);
        prefetch_tensormap(&map_o);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    float *__restrict__ eg = reinterpret_cast<float *>(sm + OFF_EG);  // gamma[4][64], flag[4]

    // Everything above overlaps the tail of the kernel ahead in the stream (programmatic
    // launch); what that kernel writes (status, plan, solve results, the state of the
    // previous phase) is read only after it has completed.
    griddep_wait();
    griddep_launch_dependents();
    const bool live = p.ctl[0] == GDR_OK;  // cu_seqlens rejected, or a solve gave up

    if (!live) {
        // nothing is read or written
    } else if (warp == kProducerWarp) {
        // ============================================================ producer
        if (lane == 0) {
            const int unit0 = p.seq_chunk[n] * p.H + h;  // chunk c is solve unit unit0 + c * H
            for (int c = 0; c < n_chunks; ++c) {
                const int tt = (int)(seq_begin + (int64_t)c * C), unit = unit0 + c * p.H;
                // V, T' (slot free once U'~ and W' of chunk c - 2 are done)
                if (c >= 2 && !mbar_wait(bar(B_VE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t vs = sbase + vslot(c), vf = bar(B_VF0 + (c & 1));
                mbar_arrive_expect_tx(vf, 3 * 8192);
                tma_load_3d(vs, &map_v, vf, col0, h, tt);
                tma_load_3d(vs + 8192, &map_v, vf, col0 + 64, h, tt);
                tma_load_3d(vs + RV_T, &map_t, vf, 0, 0, 2 * unit);
                // K, A^T, factors (slot free once chunk c - 3 is done)
                if (c >= 3 && !mbar_wait(bar(B_KE0 + c % 3), (c / 3 - 1) & 1)) { note_fail(3); break; }
                const uint32_t ks = sbase + kslot(c), kf = bar(B_KF0 + c % 3);
                mbar_arrive_expect_tx(kf, 3 * 8192 + 1024);
                tma_load_3d(ks, &map_k, kf, 0, h, tt);
                tma_load_3d(ks + 8192, &map_k, kf, 64, h, tt);
                tma_load_3d(ks + RK_A, &map_t, kf, 0, 0, 2 * unit + 1);
                bulk_load(ks + RK_G, p.factors + (size_t)unit * 256, 1024, kf);
                // Q (slot free once [QS | WS] of chunk c - 2 is done)
                if (c >= 2 && !mbar_wait(bar(B_QE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t qs = sbase + qslot(c), qf = bar(B_QF0 + (c & 1));
                mbar_arrive_expect_tx(qf, 2 * 8192);
                tma_load_3d(qs, &map_q, qf, 0, h, tt);
                tma_load_3d(qs + 16384, &map_q, qf, 64, h, tt);
            }
        }
    } else if (warp < kPrepWarp0) {
        // ============================================================ epilogue
        const int etid = tid;
        volatile int *fail = &flags[2];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        for (int c = 0; c < n_chunks; ++c) {
            // Slot c%4 moves on to chunk c + 4 only after this role has read O of chunk
            // c + 1, so the parity below is unambiguous.
            const bool ok = mbar_wait(bar(B_EG0 + (c & 3)), (c >> 2) & 1) && mbar_wait(bar(B_SO), c & 1);
            if (!ok) note_fail(2);
            named_sync(kBarEpi, kEpiThreads);
            if (*fail) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_load_16x256b_x8(lane_base + TM_O, r0);
            tmem_load_16x256b_x8(lane_base + (16u << 16) + TM_O, r1);
            tc_fence_before();
            mbar_arrive(bar(B_OFREE));
            // the staging tile: the TMA store of chunk c - 1 must have read it
            if (etid == 0) bulk_wait_group_read<0>();
            named_sync(kBarEpi, kEpiThreads);
            const uint32_t stg = sbase + OFF_OST;
            const bool ratio = eg[256 + (c & 3)] != 0.f;
            const float *gam = ratio ? eg + 64 * (c & 3) : nullptr;
            auto row_block = [&](int l8, uint32_t &block, int &c8) {
                const int dv = 32 * warp + l8;  // value column within the slice
                block = stg + (dv >> 6) * 8192;
                c8 = (dv & 63) >> 3;
            };
            transpose_store16(r0, 1.f, gam, lane, 0, row_block);
            transpose_store16(r1, 1.f, gam, lane, 16, row_block);
            fence_async_smem();
            named_sync(kBarEpi, kEpiThreads);
            const int64_t t0 = seq_begin + (int64_t)c * C;
            const int len = chunk_len(c);
            if (len == C) {
                if (etid == 0) {
                    tma_store_3d(&map_o, stg, col0, h, (int)t0);
                    tma_store_3d(&map_o, stg + 8192, col0 + 64, h, (int)t0);
                    bulk_commit_group();
                }
            } else {  // a partial last chunk: only its own rows, by plain stores
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int idx = etid + k * kEpiThreads;  // 64 rows x 16 segments of 16 bytes
                    const int row = idx >> 4, seg = idx & 15;
                    if (row < len) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            sm + OFF_OST + (seg >> 3) * 8192 + row * 128 + ((((seg & 7) ^ row) & 7) << 4));
                        *reinterpret_cast<uint4 *>(p.o + ((size_t)(t0 + row) * p.H + h) * p.dv + col0 +
                                                   seg * 8) = v;
                    }
                }
            }
        }
        if (etid == 0) bulk_wait_group_all();  // the stores have completed before exit
    } else if (warp < kStateWarp0) {
        // ============================================================ prep
        const int ptid = tid - 32 * kPrepWarp0;
        const int q = warp & 3;  // TMEM lane quarter
        volatile int *fail = &flags[0];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        auto check = [&](bool ok) -> bool {  // role-wide agreement after a wait
            if (!ok) note_fail(0);
            named_sync(kBarPrep, kPrepThreads);
            return *fail == 0;
        };
        for (int c = 0; c < n_chunks; ++c) {
            const int u = c >> 1;
            const uint32_t vs = sbase + vslot(c), ks = sbase + kslot(c), qs = sbase + qslot(c);
            unsigned char *vs_p = sm + vslot(c), *ks_p = sm + kslot(c), *qs_p = sm + qslot(c);
            const float *gate = reinterpret_cast<const float *>(ks_p + RK_G);
            if (!check(mbar_wait(bar(B_VF0 + (c & 1)), u & 1) && mbar_wait(bar(B_KF0 + c % 3), (c / 3) & 1)))
                break;
            const bool ratio = gate[G_FORM] != 0.f;
            {
                // ---- T' diag(gamma) (bf16), same swizzled layout as T'; epilogue gates
                const int t = ptid >> 1;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * (ptid & 1) + jj;  // 16-byte segment: columns 8j..8j+7
                    const uint32_t off = (uint32_t)(t * 128 + (((j ^ t) & 7) << 4));
                    uint4 w = *reinterpret_cast<const uint4 *>(vs_p + RV_T + off);
                    uint32_t *uw = &w.x;
                    const float4 ga = *reinterpret_cast<const float4 *>(gate + G_GAM + 8 * j);
                    const float4 gb = *reinterpret_cast<const float4 *>(gate + G_GAM + 8 * j + 4);
                    const float gj[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&uw[e]));
                        uw[e] = pack_bf16x2(f.x * gj[2 * e], f.y * gj[2 * e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_TG + off) = w;
                }
                if (ptid < C) eg[64 * (c & 3) + ptid] = gate[G_GAM + ptid];
                if (ptid == 0) eg[256 + (c & 3)] = ratio ? 1.f : 0.f;
                mbar_arrive(bar(B_EG0 + (c & 3)));
            }
            // T' diag(gamma) is staged: the MMA warp issues U'~ and W' when the chain
            // reaches them (the single TG buffer is reused only after U'~, W' are done)
            fence_async_smem();
            mbar_arrive(bar(B_TGR0 + (c & 1)));
            // W' done; the Q slot's -W' half free once [QS | WS] of chunk c - 2 is done
            bool ok = mbar_wait(bar(B_WD0 + (c & 1)), u & 1);
            if (ok && c >= 2) ok = mbar_wait(bar(B_QE0 + (c & 1)), (u - 1) & 1);
            if (!check(ok)) break;
            tc_fence_after();

            // ---- -W' (rows t) into the Q slot
            {
                uint32_t r[32];
                auto row_block = [&](int l8, uint32_t &block, int &c8) {
                    const int dk = 32 * q + l8;
                    block = qs + (dk >> 6) * 16384 + 8192;
                    c8 = (dk & 63) >> 3;
                };
                tmem_load_16x256b_x8(lane_base + TM_W, r);
                transpose_store16(r, -1.f, nullptr, lane, 0, row_block);
                tmem_load_16x256b_x8(lane_base + (16u << 16) + TM_W, r);
                transpose_store16(r, -1.f, nullptr, lane, 16, row_block);
            }
            // Q has landed ([QS | WS] follows B_WQ, and the exponential form scales it here)
            if (!check(mbar_wait(bar(B_QF0 + (c & 1)), u & 1))) break;
            if (!ratio) {
                // exponential form: 16-byte segments of Q (gamma) and K (kdec), in place
#pragma unroll 4
                for (int k = 0; k < 16; ++k) {
                    const int idx = ptid + k * kPrepThreads;  // 0..2047
                    const bool isq = idx < 1024;
                    unsigned char *ptr = isq ? qs_p + (idx >> 9) * 16384 + (idx & 511) * 16
                                             : ks_p + (idx - 1024) * 16;
                    const int r = ((isq ? (idx & 511) : (idx - 1024)) * 16 % 8192) / 128;  // token row
                    const float f = isq ? gate[G_GAM + r] : gate[G_KDEC + r];
                    uint4 w = *reinterpret_cast<const uint4 *>(ptr);
                    uint32_t *uw = &w.x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 fl = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&uw[e]));
                        uw[e] = pack_bf16x2(fl.x * f, fl.y * f);
                    }
                    *reinterpret_cast<uint4 *>(ptr) = w;
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_WQ0 + (c & 1)));
            mbar_arrive(bar(B_KE0 + c % 3));  // this thread reads the K slot no more
        }
    } else if (warp == kMmaWarp) {
        // ============================================================ state MMA issuer
        if (lane == 0) {
            // U'~^T = V^T T'^T into buffer j % 2 and W'^T = K^T (T' diag gamma)^T of chunk j,
            // once prep has staged T' diag(gamma) (it saw V, T' and K land). They are issued
            // where the tensor pipe would otherwise idle: after [QS | WS] of chunk j - 1,
            // while the state converts U'^T, or else after [S_upd | AU] of chunk j - 1.
            // W' first: prep transposes it while U'~ is computed.
            auto issue_uw = [&](int j) {
                const uint32_t vs = sbase + vslot(j), ks = sbase + kslot(j);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_W, sw128_desc(ks + kk * 2048, 8192, 1024),
                             sw128_desc(sbase + OFF_TG + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0),
                             kk > 0);
                mma_commit(bar(B_WD0 + (j & 1)));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_U + 64 * (j & 1), sw128_desc(vs + kk * 2048, 8192, 1024),
                             sw128_desc(vs + RV_T + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
                // U'~ needs no barrier of its own: the state reads it after B_WS, which
                // this thread commits after these MMAs
                mma_commit(bar(B_VE0 + (j & 1)));  // V and T' are read
            };
            auto tg_ready = [&](int j) { return bar(B_TGR0 + (j & 1)); };
            if (n_chunks > 0) {
                if (mbar_wait(tg_ready(0), 0)) issue_uw(0);
                else note_fail(1);
            }
            for (int c = 0; c < n_chunks && !flags[3]; ++c) {
                // [O^T | X^T] = S^T [Q; -W']^T once S^T, -W' and (for the O buffer) the
                // epilogue of chunk c - 1 are ready
                bool ok = mbar_wait(bar(B_SREADY), c & 1) && mbar_wait(bar(B_WQ0 + (c & 1)), (c >> 1) & 1);
                if (ok && c > 0) ok = mbar_wait(bar(B_OFREE), (c - 1) & 1);
                if (!ok) { note_fail(1); break; }
                tc_fence_after();
                const uint32_t qw = sbase + qslot(c);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ta(tmem + TM_O, tmem + TM_SA + 8 * kk,
                                sw128_desc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                                idesc_bf16(128, 128, 0, 0), kk > 0);
                mma_commit(bar(B_WS));
                mma_commit(bar(B_QE0 + (c & 1)));  // Q and -W' are read
                // W', U'~ of the next chunk now, while the state converts U'^T, if prep
                // stages T' diag(gamma) within a few hundred cycles (TM_U buffer (c+1)%2 was
                // converted before [S_upd | AU] of chunk c - 1; W' of chunk c was read before
                // B_WQ); else after [S_upd | AU]
                bool uw_next = c + 1 >= n_chunks;
                if (!uw_next) {
                    const uint32_t tb = tg_ready(c + 1), par = ((c + 1) >> 1) & 1;
                    const long long t0 = clock64();
                    bool ready = mbar_test_wait(tb, par);
                    while (!ready && clock64() - t0 < 400) ready = mbar_test_wait(tb, par);
                    if (ready) {
                        issue_uw(c + 1);
                        uw_next = true;
                    }
                }
                // [S^T | O^T] += U'^T [K | A^T] once U'^T (and the decayed master) is in place
                if (!mbar_wait(bar(B_UREADY), c & 1)) { note_fail(1); break; }
                tc_fence_after();
                const uint32_t ks = sbase + kslot(c);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // tokens 16kk..16kk+15: columns X + 32(kk/2) + 8(kk%2)
                    mma_bf16_ta(tmem + TM_S, tmem + TM_X + 32 * (kk >> 1) + 8 * (kk & 1),
                                sw128_desc(ks + kk * 2048, 8192, 1024), idesc_bf16(128, 192, 0, 1), 1);
                mma_commit(bar(B_SO));
                mma_commit(bar(B_KE0 + c % 3));  // the state's last reads of the K slot
                if (!uw_next) {
                    if (!mbar_wait(tg_ready(c + 1), ((c + 1) >> 1) & 1)) { note_fail(1); break; }
                    issue_uw(c + 1);
                }
            }
            if (flags[3]) {  // let issued MMAs land before TMEM and shared memory go away
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0);
            }
        }
    } else if (warp >= kStateWarp0 && warp < kStateWarp0 + kStateWarps) {
        // ============================================================ state
        const int half = (warp - kStateWarp0) >> 2;  // which 64 of the d_k entries / 32 of the tokens
        const int row = 32 * (warp & 3) + lane;      // TMEM lane = value column col0 + row
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        // each state warp's arrival on B_SREADY / B_UREADY after its TMEM stores
        auto warp_arrive = [&](int b) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(b));
        };
        // this thread's 64 entries of S^T: lane col0 + row, d_k columns [64*half, 64*half + 64);
        // they live in the fp32 master in TMEM
        const size_t s_off = ((size_t)n * p.H + h) * DK * p.dv + col0 + row;
        const uint32_t s_tm = lane_base + TM_S + 64 * half;
        {  // the incoming state (or zero) into the master; the same thread later writes
           // the same entries of S_out, so S_out may be S_in
            const float *src = p.S_in ? p.S_in + s_off + (size_t)(64 * half) * p.dv : nullptr;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = src ? src[(size_t)(32 * hh + i) * p.dv] : 0.f;
                tmem_store32(s_tm + 32 * hh, x);
            }
        }
        // Step c finishes chunk c - 1 (when c > 0), then starts chunk c (when c < n_chunks).
        for (int c = 0; c <= n_chunks; ++c) {
            if (c > 0) {
                const int cp = c - 1;
                // ---- U'^T = U'~^T + X^T, as bf16 pairs over this thread's read part of X
                if (!mbar_wait(bar(B_WS), cp & 1)) { note_fail(1); break; }
                tc_fence_after();
                {
                    float a[32], b[32];
                    tmem_load32(lane_base + TM_U + 64 * (cp & 1) + 32 * half, a);
                    tmem_load32(lane_base + TM_X + 32 * half, b);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(a[2 * i] + b[2 * i], a[2 * i + 1] + b[2 * i + 1]);
                    tmem_store16(lane_base + TM_X + 32 * half, w);
                }
                warp_arrive(B_UREADY);
                // ---- the new state (gamma_C S + U'^T K, accumulated in TMEM)
                if (!mbar_wait(bar(B_SO), cp & 1)) { note_fail(1); break; }
                tc_fence_after();
            }
            if (c == n_chunks) {  // the outgoing state (no chunks: the incoming one)
                float *dst = p.S_out + s_off + (size_t)(64 * half) * p.dv;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[32];
                    tmem_load32(s_tm + 32 * hh, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(size_t)(32 * hh + i) * p.dv] = x[i];
                }
                break;
            }
            // ---- bf16 S^T into TMEM for [QS | WS] of chunk c; then the master decayed by
            // gamma_C of chunk c while [QS | WS] runs
            float x[2][32];
            tmem_load64(s_tm, x);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(x[hh][2 * i], x[hh][2 * i + 1]);
                tmem_store16(lane_base + TM_SA + 32 * half + 16 * hh, w);
            }
            warp_arrive(B_SREADY);
            if (!mbar_wait(bar(B_KF0 + c % 3), (c / 3) & 1)) { note_fail(1); break; }
            const float gC = reinterpret_cast<const float *>(sm + kslot(c) + RK_G)[G_GAM + C - 1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[hh][i] *= gC;
                tmem_store32(s_tm + 32 * hh, x[hh]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (flags[3] != 0 && tid == 0) {
        atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
        // loads still in flight land before the shared memory is released: the last
        // chunk loaded into each slot (a wait on a phase that never completes gives up)
        for (int c = n_chunks - 1; c >= 0 && c >= n_chunks - 3; --c) {
            if (c >= n_chunks - 2) {
                mbar_wait(bar(B_QF0 + (c & 1)), (c >> 1) & 1);
                mbar_wait(bar(B_VF0 + (c & 1)), (c >> 1) & 1);
            }
            mbar_wait(bar(B_KF0 + c % 3), (c / 3) & 1);
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

bool encode_3d(CUtensorMap *map, const void *base, const cuuint64_t (&dims)[3],
               const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace tc {

bool make_map_thd(CUtensorMap *map, const void *base, int d, int H, int64_t T) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * H * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    return encode_3d(map, base, dims, strides, box);
}

bool make_map_units(CUtensorMap *map, const void *base, int64_t units) {
    const cuuint64_t dims[3] = {64, 64, (cuuint64_t)units};
    const cuuint64_t strides[2] = {64 * 2, 64 * 64 * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    return encode_3d(map, base, dims, strides, box);
}

}  // namespace tc

// ---------------------------------------------------------------- phases

// The solve of every chunk must finish before the chain reaches it, but nothing else
// orders the two kernels. A call is therefore split into phases, each taking a fixed
// share of every sequence's chunks: the chain of phase f runs on the caller's stream
// while the solve of phase f + 1 runs on a second stream, on the SMs the chain leaves
// free (one chain CTA per SM). Events order solve f before chain f; the second stream
// forks from and joins back into the caller's stream, so the call stays one
// stream-ordered operation and can be captured into a CUDA graph. No kernel waits on
// another kernel.

namespace {

constexpr int kMaxDevices = 256;

// The second stream and the events of the current host thread on one device. Kept per
// thread so that calls from several threads never share a stream that one of them may
// be capturing. Created on first use; never destroyed (they go with the context).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[kMaxPhases] = {};
    bool ready = false, failed = false;
};
thread_local SideStream t_side[kMaxDevices];

int device_sms(int dev) {
    static int sms[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        sms[dev] = v;
    }
    return sms[dev];
}

// The current thread's side stream on the current device, or null. Resources are not
// created while `caller` is being captured; such a call runs as one phase.
SideStream *side_stream(cudaStream_t caller) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream &sd = t_side[dev];
    if (sd.ready) return &sd;
    if (sd.failed) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
        return nullptr;
    bool ok = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < kMaxPhases; ++i)
        ok = cudaEventCreateWithFlags(&sd.ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        sd.failed = true;  // run single-phase from now on; nothing half-made is used
        return nullptr;
    }
    sd.ready = true;
    return &sd;
}

}  // namespace

// The solve keeps pace with the chain when the free SMs solve one chunk of every
// (sequence, head) no slower than a chain CTA takes one step: about 2.2 us of one SM per
// solve unit against about 1.8 us per chain step, so 1.25 units per chunk step per free
// SM. Every phase restarts the chain's pipeline (pipeline fill and drain, about 7 us,
// and a launch behind an event, about 5 us), so a phase keeps at least 32 chunks of the
// average sequence. GDR_PREFILL_PHASES=1..8 in the
// environment overrides the choice (a tuning and testing knob; the result does not
// depend on the phase count).
int tc_phases_for(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms) {
    if (const char *env = getenv("GDR_PREFILL_PHASES")) {
        const int v = atoi(env);
        if (v >= 1 && v <= kMaxPhases) return v;
    }
    const int64_t units_per_step = num_seqs * H;
    const int64_t chain_ctas = units_per_step * (dv / NV);
    const int64_t free_sms = sms - chain_ctas;
    if (free_sms < 8 || 5 * units_per_step > 4 * free_sms) return 1;
    const int64_t avg_chunks = total_tokens / num_seqs / kChunk;
    const int64_t P = avg_chunks / 32;
    return P < 1 ? 1 : (P > kMaxPhases ? kMaxPhases : (int)P);
}

int tc_phases(const PrefillArgs &a) {
    int dev = -1;
    if (a.total_tokens == 0 || cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int P = tc_phases_for(a.num_seqs, a.total_tokens, a.H, a.dv, device_sms(dev));
    return P > 1 && side_stream(a.stream) ? P : 1;
}

int launch_prefill_tc(const PrefillArgs &a, const WsLayout &L, int phases) {
    const size_t s_bytes = (size_t)a.num_seqs * a.H * a.dk * a.dv * sizeof(float);
    if (a.total_tokens == 0) {  // nothing to compute: S_final = S0 (or zero)
        cudaError_t e = cudaSuccess;
        if (!a.S0) e = cudaMemsetAsync(a.S_final, 0, s_bytes, a.stream);
        else if (a.S0 != a.S_final)
            e = cudaMemcpyAsync(a.S_final, a.S0, s_bytes, cudaMemcpyDeviceToDevice, a.stream);
        return cuda_status(e);
    }
    CUtensorMap mq, mk, mv, mt, mo;
    if (!tc::make_map_thd(&mq, a.q, a.dk, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mk, a.k, a.dk, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mv, a.v, a.dv, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mo, a.o, a.dv, a.H, a.total_tokens) ||
        !tc::make_map_units(&mt, a.ws + L.T, 2 * L.max_chunks * a.H))
        return GDR_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int n_slices = a.dv / NV;
    const int64_t chain_ctas = a.num_seqs * a.H * n_slices;
    SideStream *sd = nullptr;
    if (phases > 1) {
        sd = side_stream(a.stream);
        if (!sd) return GDR_ERR_CUDA;  // tc_phases made it; it cannot have gone
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDR_ERR_CUDA;
    const int free_sms = (int)(device_sms(dev) - chain_ctas);

    // solve of phase 0 on the caller's stream, with the whole GPU
    int st = tc::launch_solve_tc(a, L, mq, mk, mt, 0, 0, a.stream, true);
    if (st != GDR_OK) return st;
    if (phases > 1) {  // solves of phases 1 .. P-1 on the side stream, after the solve of
                       // phase 0 (which has had every SM) and beside the chains
        cudaError_t e = cudaEventRecord(sd->ev[0], a.stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sd->stream, sd->ev[0], 0);
        if (e != cudaSuccess) return GDR_ERR_CUDA;
        for (int f = 1; f < phases; ++f) {
            st = tc::launch_solve_tc(a, L, mq, mk, mt, f, free_sms, sd->stream, false);
            if (st != GDR_OK) return st;
            if (cudaEventRecord(sd->ev[f], sd->stream) != cudaSuccess) return GDR_ERR_CUDA;
        }
    }
    TcParams p;
    p.factors = reinterpret_cast<const float *>(a.ws + L.G);
    p.cu_seqlens = a.cu_seqlens;
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.H = a.H;
    p.dv = a.dv;
    p.n_slices = n_slices;
    p.phases = phases;
    p.o = (__nv_bfloat16 *)a.o;
    p.ctl = (int32_t *)(a.ws + L.ctl);
    float *S_mid = reinterpret_cast<float *>(a.ws + L.S);
    for (int f = 0; f < phases; ++f) {
        if (f > 0 && cudaStreamWaitEvent(a.stream, sd->ev[f], 0) != cudaSuccess) return GDR_ERR_CUDA;
        p.phase = f;
        p.seq_chunk = reinterpret_cast<const int32_t *>(a.ws + L.seq_chunk) + (size_t)f * (a.num_seqs + 1);
        p.S_in = f == 0 ? a.S0 : S_mid;
        p.S_out = f == phases - 1 ? a.S_final : S_mid;
        // a programmatic dependent of the kernel ahead of it (the solve of phase 0, or the
        // chain of the previous phase); it waits for that kernel before reading its results
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)chain_ctas);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, tc_chain_kernel, mq, mk, mv, mt, mo, p) != cudaSuccess)
            return GDR_ERR_CUDA;
    }
    return GDR_OK;
}

}  // namespace gdr
