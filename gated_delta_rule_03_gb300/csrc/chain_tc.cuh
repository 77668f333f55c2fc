// chain_tc.cuh -- chunked prefill of the gated delta rule on the 5th-generation tensor
// cores (tcgen05), for bf16 q/k/v with d_k = 128 and d_v a multiple of 128: the
// sequential chain over the chunks of each (sequence, head). Its kernels and the host
// launcher of the whole tensor-core path are in prefill_tc.cu.
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
#pragma once

#include "tc_common.cuh"

namespace gdr {
namespace chain {

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
constexpr uint32_t RK = 65536, RK_SLOT = 26624;    // K_b0 | K_b1 | A^T (8 KB each) | factors
constexpr uint32_t RK_A = 16384, RK_G = 24576;     // offsets of A^T and the factors in a K slot
constexpr uint32_t RV = RK + 3 * RK_SLOT, RV_SLOT = 24576;  // V_b0 | V_b1 | T'
constexpr uint32_t RV_T = 16384;
// float offsets in a unit's factors (g at 0); 1/|k|, 1/|q| of the layer prologue (else 1)
constexpr int G_GAM = 64, G_KDEC = 128, G_FORM = 192, G_NK = 256, G_NQ = 320;
constexpr uint32_t kFactorBytes = 384 * 4;
static_assert(RK_G + kFactorBytes <= RK_SLOT, "K slot");
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
// int[7]: the last chunk whose loads the producer issued into each slot (V/T' 0-1,
// K/A^T/factors 2-4, Q 5-6), -1 for none; the drain after a failure waits for them
constexpr uint32_t OFF_ISSUED = OFF_FLAGS + 16;
constexpr uint32_t SMEM_USED = OFF_ISSUED + 32;
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
    const int32_t *flags;      // fused launch: per solve unit, set once the unit is solved
    int additive;              // the additive rule: W' = 0 (the state does not enter U')
    int prologue;              // the layer prologue: 1/|k|, 1/|q| from the factors apply
    // Segments of the sequences (the segmented schedule): mode 0 is the plain chain of a
    // (sequence, head, slice) over this launch's phase. Mode 1 runs, for every segment f
    // but the last (the phase f of `phases`), the segment's transition P_f (one more
    // slice: zero values from the identity; d_k = NV) and its local state R_f (the value
    // slices from zero), without output. Mode 2 runs every segment f from its start
    // state S_start[f] (a copy of S_in for the first, so that S_out may be S_in), with
    // output; the last segment's state goes to S_out, the others' to S_discard. Every
    // per-segment buffer holds [segment][sequence * H + head][d_k][d_v] (P_f transposed,
    // in columns [0, d_k)).
    int mode;
    float *S_P, *S_R;
    const float *S_start;
    float *S_discard;
    // the layer's output step on o (null out_gate: none; only when d_v = NV, one slice)
    const __nv_bfloat16 *out_gate;
    const float *out_norm_weight;
    float out_norm_eps;
    // Bound of every wait in SM cycles (kWaitCycles; twice that for a solved unit), and a
    // test of the give-up path: the producer of the launch's CTA 0 skips the K-slot load of
    // chunk fault_chunk (-1: never), so that the roles waiting on it give up, mark the
    // call GDR_ERR_DEVICE_TIMEOUT and drain.
    long long wait_cycles;
    int fault_chunk;
    int only_pair;  // run nothing unless ctl[kPairWord] hands the call to this launch
};

// Every wait's bound, and the give-up test knob (host side, prefill_tc.cu).
void chain_wait_policy(TcParams &p);

// A chain CTA of a fused launch waits here until the solve has published unit u (its
// T', A^T and factors stored); false if the call failed meanwhile or the wait ran out.
__device__ __forceinline__ bool wait_unit_solved(const int32_t *flag, const int32_t *ctl,
                                                 long long limit) {
    const long long t0 = clock64();
    while (acquire_load_gpu(flag) == 0) {
        if (*reinterpret_cast<const volatile int32_t *>(ctl) != GDR_OK || clock64() - t0 > limit)
            return false;
        __nanosleep(64);
    }
    fence_proxy_async_global();  // the TMA loads that follow see what the flag published
    return true;
}

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

// The chain of CTA `cta`: (sequence, head, d_v slice) = (cta / n_slices / H, ...).
// kFused: the CTA shares a cooperative launch with the solve and waits for each chunk's
// unit to be published before loading its results.
// kSeg: a launch of the segmented schedule (p.mode 1 or 2); without it p.mode is 0 and
// the segment branches compile away.
// kPC: one forget rate per key channel (d_k = d_v = 128, one slice): every operand comes
// precomputed from the per-channel chunk kernel (channel_tc.cuh), in the same slots --
// e^g . Q and -W in the Q slot, e^{g_C - g} . K, A^T and exp(g_C) per channel in the K
// slot, Utilde^T in the V slot -- so the chain issues only [QS | WS] and [S_upd | AU],
// prep has nothing to stage, U' = Utilde + X reads Utilde from shared memory, and the
// master decays column by column.
template <bool kFused, bool kSeg = false, bool kPC = false>
__device__ __forceinline__ void chain_body(const CUtensorMap &map_q, const CUtensorMap &map_k,
                                           const CUtensorMap &map_v, const CUtensorMap &map_t,
                                           const CUtensorMap &map_o, const TcParams &p, int cta) {
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
    volatile int *issued = reinterpret_cast<volatile int *>(sm + OFF_ISSUED);
    const long long wait_limit = p.wait_cycles;
    auto wait = [&](uint32_t b, uint32_t parity) { return mbar_wait_for(b, parity, wait_limit); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // this CTA's chain: segment (phase), sequence-head, value slice; state in and out
    const int NH = (int)p.num_seqs * p.H;
    const size_t mat_floats = (size_t)DK * p.dv;
    int phase = p.phase, slice, nh;
    bool zero_v = false, no_out = false;  // mode 1: the transition slice / no output
    const int32_t *seq_chunk = p.seq_chunk;
    const float *S_in_m;  // this chain's [d_k][d_v] start state, or null (zero)
    float *S_out_m;       // where its end state goes
    if (!kSeg || p.mode == 0) {
        slice = cta % p.n_slices;
        nh = cta / p.n_slices;
        S_in_m = p.S_in ? p.S_in + nh * mat_floats : nullptr;
        S_out_m = p.S_out + nh * mat_floats;
    } else {
        const int per = p.n_slices + (p.mode == 1 ? 1 : 0);
        phase = cta / (NH * per);
        nh = (cta % (NH * per)) / per;
        const int s1 = cta % per;
        seq_chunk = p.seq_chunk + (size_t)phase * (p.num_seqs + 1);
        const size_t mat = ((size_t)phase * NH + nh) * mat_floats;
        if (p.mode == 1) {
            zero_v = s1 == 0;
            no_out = true;
            slice = zero_v ? 0 : s1 - 1;
            S_in_m = nullptr;  // (the transition starts from the identity)
            S_out_m = (zero_v ? p.S_P : p.S_R) + mat;
        } else {
            slice = s1;
            S_in_m = p.S_start + mat;
            S_out_m = phase == p.phases - 1 ? p.S_out + nh * mat_floats : p.S_discard + mat;
        }
    }
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
    const int64_t cb = (int64_t)phase * m / p.phases;
    const int n_chunks = (int)((int64_t)(phase + 1) * m / p.phases - cb);
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
        for (int i = 0; i < 7; ++i) issued[i] = -1;
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
    // (not live: cu_seqlens rejected, a solve gave up, or the call is another launch's)
    const bool live = p.ctl[0] == GDR_OK && (!p.only_pair || p.ctl[kPairWord] == 1);

    if (!live) {
        // nothing is read or written
    } else if (warp == kProducerWarp) {
        // ============================================================ producer
        if (lane == 0) {
            // chunk c is solve unit unit0 + c * H (equal lengths in a fused launch: closed form)
            const int first = kFused && !p.cu_seqlens ? n * (int)m : seq_chunk[n];
            const int unit0 = first * p.H + h;
            for (int c = 0; kPC && c < n_chunks; ++c) {
                // per-channel operands: Utilde^T (V slot), e^{g_C - g} . K, A^T and exp(g_C)
                // (K slot), e^g . Q and -W (Q slot); units of 64 (or 128) rows
                const int unit = unit0 + c * p.H;
                if (c >= 2 && !wait(bar(B_VE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t vs = sbase + vslot(c), vf = bar(B_VF0 + (c & 1));
                mbar_arrive_expect_tx(vf, 2 * 8192);
                tma_load_3d(vs, &map_v, vf, 0, 0, 128 * unit);
                tma_load_3d(vs + 8192, &map_v, vf, 0, 0, 128 * unit + 64);
                issued[c & 1] = c;
                if (c >= 3 && !wait(bar(B_KE0 + c % 3), (c / 3 - 1) & 1)) { note_fail(3); break; }
                const uint32_t ks = sbase + kslot(c), kf = bar(B_KF0 + c % 3);
                if (!(c == p.fault_chunk && cta == 0)) {
                    mbar_arrive_expect_tx(kf, 3 * 8192 + 512);
                    tma_load_3d(ks, &map_k, kf, 0, 0, 64 * unit);
                    tma_load_3d(ks + 8192, &map_k, kf, 64, 0, 64 * unit);
                    tma_load_3d(ks + RK_A, &map_t, kf, 0, 0, 2 * unit + 1);
                    bulk_load(ks + RK_G, p.factors + (size_t)unit * 384, 512, kf);
                    issued[2 + c % 3] = c;
                }
                if (c >= 2 && !wait(bar(B_QE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t qs = sbase + qslot(c), qf = bar(B_QF0 + (c & 1));
                mbar_arrive_expect_tx(qf, 4 * 8192);
                tma_load_3d(qs, &map_q, qf, 0, 0, 64 * unit);
                tma_load_3d(qs + 8192, &map_q, qf, 128, 0, 64 * unit);
                tma_load_3d(qs + 16384, &map_q, qf, 64, 0, 64 * unit);
                tma_load_3d(qs + 24576, &map_q, qf, 192, 0, 64 * unit);
                issued[5 + (c & 1)] = c;
            }
            for (int c = 0; !kPC && c < n_chunks; ++c) {
                const int tt = (int)(seq_begin + (int64_t)c * C), unit = unit0 + c * p.H;
                if (kFused && !wait_unit_solved(p.flags + unit, p.ctl, 2 * wait_limit)) { note_fail(3); break; }
                // V, T' (slot free once U'~ and W' of chunk c - 2 are done)
                if (c >= 2 && !wait(bar(B_VE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t vs = sbase + vslot(c), vf = bar(B_VF0 + (c & 1));
                mbar_arrive_expect_tx(vf, zero_v ? 8192 : 3 * 8192);
                if (!zero_v) {  // (the transition slice has zero values)
                    tma_load_3d(vs, &map_v, vf, col0, h, tt);
                    tma_load_3d(vs + 8192, &map_v, vf, col0 + 64, h, tt);
                }
                tma_load_3d(vs + RV_T, &map_t, vf, 0, 0, 2 * unit);
                issued[c & 1] = c;
                // K, A^T, factors (slot free once chunk c - 3 is done)
                if (c >= 3 && !wait(bar(B_KE0 + c % 3), (c / 3 - 1) & 1)) { note_fail(3); break; }
                const uint32_t ks = sbase + kslot(c), kf = bar(B_KF0 + c % 3);
                // the factors: the decay's 1 KB, plus 1/|k|, 1/|q| with the prologue
                const uint32_t fbytes = p.prologue ? kFactorBytes : 1024u;
                if (!(c == p.fault_chunk && cta == 0)) {
                    mbar_arrive_expect_tx(kf, 3 * 8192 + fbytes);
                    tma_load_3d(ks, &map_k, kf, 0, h, tt);
                    tma_load_3d(ks + 8192, &map_k, kf, 64, h, tt);
                    tma_load_3d(ks + RK_A, &map_t, kf, 0, 0, 2 * unit + 1);
                    bulk_load(ks + RK_G, p.factors + (size_t)unit * 384, fbytes, kf);
                    issued[2 + c % 3] = c;
                }
                // Q (slot free once [QS | WS] of chunk c - 2 is done)
                if (c >= 2 && !wait(bar(B_QE0 + (c & 1)), ((c >> 1) - 1) & 1)) { note_fail(3); break; }
                const uint32_t qs = sbase + qslot(c), qf = bar(B_QF0 + (c & 1));
                mbar_arrive_expect_tx(qf, no_out ? 0 : 2 * 8192);
                if (!no_out) {  // (a segment summary reads no Q)
                    tma_load_3d(qs, &map_q, qf, 0, h, tt);
                    tma_load_3d(qs + 16384, &map_q, qf, 64, h, tt);
                }
                issued[5 + (c & 1)] = c;
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
            const bool ok = wait(bar(B_EG0 + (c & 3)), (c >> 2) & 1) && wait(bar(B_SO), c & 1);
            if (!ok) note_fail(2);
            named_sync(kBarEpi, kEpiThreads);
            if (*fail) break;
            tc_fence_after();
            if (no_out) {  // a segment summary: no O was computed
                tc_fence_before();
                mbar_arrive(bar(B_OFREE));
                continue;
            }
            uint32_t r0[32], r1[32];
            tmem_load_16x256b_x8(lane_base + TM_O, r0);
            tmem_load_16x256b_x8(lane_base + (16u << 16) + TM_O, r1);
            tc_fence_before();
            mbar_arrive(bar(B_OFREE));
            // the staging tile: the TMA store of chunk c - 1 must have read it
            if (etid == 0) bulk_wait_group_read<0>();
            named_sync(kBarEpi, kEpiThreads);
            const uint32_t stg = sbase + OFF_OST;
            // the output rows' scales (prep), when there are any
            const float *gam = eg[256 + (c & 3)] != 0.f ? eg + 64 * (c & 3) : nullptr;
            auto row_block = [&](int l8, uint32_t &block, int &c8) {
                const int dv = 32 * warp + l8;  // value column within the slice
                block = stg + (dv >> 6) * 8192;
                c8 = (dv & 63) >> 3;
            };
            transpose_store16(r0, 1.f, gam, lane, 0, row_block);
            transpose_store16(r1, 1.f, gam, lane, 16, row_block);
            const int64_t t0 = seq_begin + (int64_t)c * C;
            const int len = chunk_len(c);
            if (p.out_gate) {
                // the layer's output step on the staged rows (the CTA holds all d_v = 128
                // entries of its tokens): thread 2r + f takes the 64 entries of row r in
                // staging tile f, the pair sums the row's squares
                named_sync(kBarEpi, kEpiThreads);
                const int r = etid >> 1, f = etid & 1;
                unsigned char *tile = sm + OFF_OST + f * 8192;
                auto seg_at = [&](int s) {
                    return reinterpret_cast<uint4 *>(tile + r * 128 + (((s ^ r) & 7) << 4));
                };
                float ss = 0.f;
                if (r < len) {
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint4 u = *seg_at(s);
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uw[e]));
                            ss = fmaf(x.x, x.x, fmaf(x.y, x.y, ss));
                        }
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (r < len) {
                    const float rs = rsqrtf(ss * (1.f / NV) + p.out_norm_eps);
                    const __nv_bfloat16 *zr = p.out_gate + ((size_t)(t0 + r) * p.H + h) * p.dv + col0 + 64 * f;
                    const float *wr = p.out_norm_weight ? p.out_norm_weight + col0 + 64 * f : nullptr;
#pragma unroll 2
                    for (int s = 0; s < 8; ++s) {
                        const uint4 u = *seg_at(s);
                        const uint4 zu = *reinterpret_cast<const uint4 *>(zr + 8 * s);
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w}, zw[4] = {zu.x, zu.y, zu.z, zu.w};
                        uint32_t ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&uw[e]));
                            const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&zw[e]));
                            const float w0 = wr ? wr[8 * s + 2 * e] : 1.f, w1 = wr ? wr[8 * s + 2 * e + 1] : 1.f;
                            ow[e] = pack_bf16x2(x.x * rs * w0 * (g.x / (1.f + __expf(-g.x))),
                                                x.y * rs * w1 * (g.y / (1.f + __expf(-g.y))));
                        }
                        *seg_at(s) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
            }
            fence_async_smem();
            named_sync(kBarEpi, kEpiThreads);
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
        for (int c = 0; kPC && c < n_chunks; ++c) {
            // nothing to stage: the epilogue's rows need no scale (e^g is in the queries),
            // and this role's reads of the K slot are done once it has landed
            if (!check(wait(bar(B_KF0 + c % 3), (c / 3) & 1))) break;
            if (ptid == 0) eg[256 + (c & 3)] = 0.f;
            mbar_arrive(bar(B_EG0 + (c & 3)));
            mbar_arrive(bar(B_KE0 + c % 3));
        }
        for (int c = 0; !kPC && c < n_chunks; ++c) {
            const int u = c >> 1;
            const uint32_t vs = sbase + vslot(c), ks = sbase + kslot(c), qs = sbase + qslot(c);
            unsigned char *vs_p = sm + vslot(c), *ks_p = sm + kslot(c), *qs_p = sm + qslot(c);
            const float *gate = reinterpret_cast<const float *>(ks_p + RK_G);
            if (!check(wait(bar(B_VF0 + (c & 1)), u & 1) && wait(bar(B_KF0 + c % 3), (c / 3) & 1)))
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
                    // gamma_i (times the prologue's 1/|k_i|: the unit-length keys enter W' here)
                    const float4 ga = *reinterpret_cast<const float4 *>(gate + G_GAM + 8 * j);
                    const float4 gb = *reinterpret_cast<const float4 *>(gate + G_GAM + 8 * j + 4);
                    float gj[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    if (p.prologue) {
                        const float4 na = *reinterpret_cast<const float4 *>(gate + G_NK + 8 * j);
                        const float4 nb = *reinterpret_cast<const float4 *>(gate + G_NK + 8 * j + 4);
                        const float nj[8] = {na.x, na.y, na.z, na.w, nb.x, nb.y, nb.z, nb.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) gj[e] *= nj[e];
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&uw[e]));
                        uw[e] = pack_bf16x2(f.x * gj[2 * e], f.y * gj[2 * e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_TG + off) = w;
                }
                // the scale of output row t: gamma_t (ratio form) times the prologue's 1/|q_t|
                if (ptid < C)
                    eg[64 * (c & 3) + ptid] = p.prologue ? (ratio ? gate[G_GAM + ptid] : 1.f) * gate[G_NQ + ptid]
                                                         : gate[G_GAM + ptid];
                if (ptid == 0) eg[256 + (c & 3)] = (ratio || p.prologue) ? 1.f : 0.f;
                mbar_arrive(bar(B_EG0 + (c & 3)));
            }
            // T' diag(gamma) is staged: the MMA warp issues U'~ and W' when the chain
            // reaches them (the single TG buffer is reused only after U'~, W' are done)
            fence_async_smem();
            mbar_arrive(bar(B_TGR0 + (c & 1)));
            // W' done; the Q slot's -W' half free once [QS | WS] of chunk c - 2 is done
            bool ok = wait(bar(B_WD0 + (c & 1)), u & 1);
            if (ok && c >= 2) ok = wait(bar(B_QE0 + (c & 1)), (u - 1) & 1);
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
                const float wsign = p.additive ? 0.f : -1.f;  // W' (finite) times 0 for the additive rule
                tmem_load_16x256b_x8(lane_base + TM_W, r);
                transpose_store16(r, wsign, nullptr, lane, 0, row_block);
                tmem_load_16x256b_x8(lane_base + (16u << 16) + TM_W, r);
                transpose_store16(r, wsign, nullptr, lane, 16, row_block);
            }
            // Q has landed ([QS | WS] follows B_WQ, and the exponential form scales it here)
            if (!check(wait(bar(B_QF0 + (c & 1)), u & 1))) break;
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
                if (!zero_v) {  // U'~ = T'V (zero for the transition slice, never read)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + TM_U + 64 * (j & 1), sw128_desc(vs + kk * 2048, 8192, 1024),
                                 sw128_desc(vs + RV_T + kk * 32, 16, 1024), idesc_bf16(128, 64, 1, 0), kk > 0);
                }
                // U'~ needs no barrier of its own: the state reads it after B_WS, which
                // this thread commits after these MMAs
                mma_commit(bar(B_VE0 + (j & 1)));  // V and T' are read
            };
            auto tg_ready = [&](int j) { return bar(B_TGR0 + (j & 1)); };
            if (!kPC && n_chunks > 0) {
                if (wait(tg_ready(0), 0)) issue_uw(0);
                else note_fail(1);
            }
            for (int c = 0; c < n_chunks && !flags[3]; ++c) {
                // [O^T | X^T] = S^T [Q; -W']^T once the epilogue has read O of chunk c - 1,
                // -W' is in place and S^T is written: checked in the order they usually
                // complete, so that only the last wait is on the chain's critical path
                bool ok = c == 0 || wait(bar(B_OFREE), (c - 1) & 1);
                // -W: staged by prep, or (per-channel) loaded with the queries
                ok = ok && wait(bar((kPC ? B_QF0 : B_WQ0) + (c & 1)), (c >> 1) & 1) && wait(bar(B_SREADY), c & 1);
                if (!ok) { note_fail(1); break; }
                tc_fence_after();
                const uint32_t qw = sbase + qslot(c);
                if (no_out) {  // a segment summary: X^T = -S^T W'^T alone (rows -W' of the slot)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tmem + TM_X, tmem + TM_SA + 8 * kk,
                                    sw128_desc(qw + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32, 16, 1024),
                                    idesc_bf16(128, 64, 0, 0), kk > 0);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tmem + TM_O, tmem + TM_SA + 8 * kk,
                                    sw128_desc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                                    idesc_bf16(128, 128, 0, 0), kk > 0);
                }
                mma_commit(bar(B_WS));
                mma_commit(bar(B_QE0 + (c & 1)));  // Q and -W' are read
                // W', U'~ of the next chunk now, while the state converts U'^T, if prep
                // stages T' diag(gamma) within a few hundred cycles (TM_U buffer (c+1)%2 was
                // converted before [S_upd | AU] of chunk c - 1; W' of chunk c was read before
                // B_WQ); else after [S_upd | AU]
                bool uw_next = kPC || c + 1 >= n_chunks;
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
                if (!wait(bar(B_UREADY), c & 1)) { note_fail(1); break; }
                tc_fence_after();
                if (kPC) mbar_arrive(bar(B_VE0 + (c & 1)));  // the state has read Utilde^T
                const uint32_t ks = sbase + kslot(c);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // tokens 16kk..16kk+15: columns X + 32(kk/2) + 8(kk%2)
                    mma_bf16_ta(tmem + TM_S, tmem + TM_X + 32 * (kk >> 1) + 8 * (kk & 1),
                                sw128_desc(ks + kk * 2048, 8192, 1024),
                                idesc_bf16(128, no_out ? 128 : 192, 0, 1), 1);  // (summary: S only)
                mma_commit(bar(B_SO));
                mma_commit(bar(B_KE0 + c % 3));  // the state's last reads of the K slot
                if (!uw_next) {
                    if (!wait(tg_ready(c + 1), ((c + 1) >> 1) & 1)) { note_fail(1); break; }
                    issue_uw(c + 1);
                }
            }
            if (flags[3]) {  // let issued MMAs land before TMEM and shared memory go away
                mma_commit(bar(B_DRAIN));
                wait(bar(B_DRAIN), 0);
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
        const size_t s_off = col0 + row;  // within this chain's [d_k][d_v] matrix
        const uint32_t s_tm = lane_base + TM_S + 64 * half;
        {  // the incoming state (zero, or the identity for a transition) into the master;
           // the same thread later writes the same entries of S_out, so S_out may be S_in
            const float *src = S_in_m ? S_in_m + s_off + (size_t)(64 * half) * p.dv : nullptr;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = src ? src[(size_t)(32 * hh + i) * p.dv]
                               : (zero_v && 64 * half + 32 * hh + i == row ? 1.f : 0.f);
                tmem_store32(s_tm + 32 * hh, x);
            }
        }
        // Step c finishes chunk c - 1 (when c > 0), then starts chunk c (when c < n_chunks).
        for (int c = 0; c <= n_chunks; ++c) {
            if (c > 0) {
                const int cp = c - 1;
                // ---- U'^T = U'~^T + X^T, as bf16 pairs over this thread's read part of X
                if (!wait(bar(B_WS), cp & 1)) { note_fail(1); break; }
                // (per-channel: Utilde^T is read from the V slot, which nobody else waits for)
                if (kPC && !wait(bar(B_VF0 + (cp & 1)), (cp >> 1) & 1)) { note_fail(1); break; }
                tc_fence_after();
                {
                    float a[32], b[32];
                    if (zero_v) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a[i] = 0.f;
                    } else if (kPC) {
                        // row `row` of Utilde^T (a 128-byte-swizzled box of 64 rows per half of
                        // d_v), tokens 32 half .. 32 half + 31: four 16-byte segments
                        const uint32_t box = sbase + vslot(cp) + (row >> 6) * 8192;
                        const int rr = row & 63;
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4) {
                            uint4 w4;
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(w4.x), "=r"(w4.y), "=r"(w4.z), "=r"(w4.w)
                                         : "r"(sw128_seg(box, rr, 4 * half + s4)));
                            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ww[e]));
                                a[8 * s4 + 2 * e] = f.x;
                                a[8 * s4 + 2 * e + 1] = f.y;
                            }
                        }
                    } else {
                        tmem_load32(lane_base + TM_U + 64 * (cp & 1) + 32 * half, a);
                    }
                    tmem_load32(lane_base + TM_X + 32 * half, b);
                    uint32_t w[16];
                    if (p.prologue) {  // U'_i 1/|k_i|: the unit-length keys of the state update
                        const float *nk = reinterpret_cast<const float *>(sm + kslot(cp) + RK_G) + G_NK + 32 * half;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = pack_bf16x2((a[2 * i] + b[2 * i]) * nk[2 * i], (a[2 * i + 1] + b[2 * i + 1]) * nk[2 * i + 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(a[2 * i] + b[2 * i], a[2 * i + 1] + b[2 * i + 1]);
                    }
                    tmem_store16(lane_base + TM_X + 32 * half, w);
                }
                warp_arrive(B_UREADY);
                // ---- the new state (gamma_C S + U'^T K, accumulated in TMEM)
                if (!wait(bar(B_SO), cp & 1)) { note_fail(1); break; }
                tc_fence_after();
            }
            if (c == n_chunks) {  // the outgoing state (no chunks: the incoming one)
                float *dst = S_out_m + s_off + (size_t)(64 * half) * p.dv;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[32];
                    tmem_load32(s_tm + 32 * hh, x);
                    if (zero_v) {  // a transition is stored transposed: P^T[row][k]
                        float4 *t = reinterpret_cast<float4 *>(S_out_m + (size_t)row * p.dv + 64 * half + 32 * hh);
#pragma unroll
                        for (int i = 0; i < 8; ++i) t[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) dst[(size_t)(32 * hh + i) * p.dv] = x[i];
                    }
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
            if (!wait(bar(B_KF0 + c % 3), (c / 3) & 1)) { note_fail(1); break; }
            const float *fac = reinterpret_cast<const float *>(sm + kslot(c) + RK_G);
            if (kPC) {  // exp(g_C) per key channel: column 64 half + 32 hh + i of S^T
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 f = *reinterpret_cast<const float4 *>(fac + 64 * half + 32 * hh + 4 * i4);
                        x[hh][4 * i4] *= f.x;
                        x[hh][4 * i4 + 1] *= f.y;
                        x[hh][4 * i4 + 2] *= f.z;
                        x[hh][4 * i4 + 3] *= f.w;
                    }
                    tmem_store32(s_tm + 32 * hh, x[hh]);
                }
            } else {
                const float gC = fac[G_GAM + C - 1];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[hh][i] *= gC;
                    tmem_store32(s_tm + 32 * hh, x[hh]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (flags[3] != 0 && tid == 0) {
        atomicExch(p.ctl, GDR_ERR_DEVICE_TIMEOUT);
        // loads still in flight land before the shared memory is released: for each slot,
        // the last chunk the producer issued into it (earlier ones in the slot completed
        // before that one was issued)
        for (int i = 0; i < 7; ++i) {
            const int c = issued[i];
            if (c < 0) continue;
            if (i < 2) wait(bar(B_VF0 + i), (c >> 1) & 1);
            else if (i < 5) wait(bar(B_KF0 + (i - 2)), (c / 3) & 1);
            else wait(bar(B_QF0 + (i - 5)), (c >> 1) & 1);
        }
    }
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace chain
}  // namespace gdr
