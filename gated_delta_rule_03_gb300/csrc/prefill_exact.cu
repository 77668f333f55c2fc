// prefill_exact.cu -- chunked prefill in plain fp32 arithmetic (no tensor cores).
//
// This is the path for fp32 inputs, whose accuracy target (1e-4 relative) bf16
// or tf32 tensor-core products cannot meet, and for shapes the tensor-core
// kernel does not cover. It computes the chunk form of the gated delta rule:
// the ungated chunk algorithm of "Attention as Matrix Algebra: From Softmax to
// the Delta Rule", section 8 ("Training the delta rule in chunks"), with the
// decay gate carried through the same substitution. Per chunk of C tokens,
// entering with state S:
//   gamma_t = prod_{j<=t} alpha_j,  Gamma_ti = prod_{i<j<=t} alpha_j  (= exp(g_t - g_i))
//   L_ti = beta_t Gamma_ti k_t.k_i (i < t),  T = (I + L)^{-1} diag(beta)
//   W = T diag(gamma) K,  Utilde = T V                  (prep kernel, all chunks at once)
//   U = Utilde - W S
//   O = diag(gamma) Q S + (Q K^T . Gamma . [i <= t]) U
//   S <- gamma_C S + Ktilde^T U,  Ktilde_i = exp(g_C - g_i) k_i   (chain kernel, in order)
// The decay factors are products of the per-token alpha_j = exp(log alpha_j), never
// differences of cumulative log-decays: a cumulative sum that has passed a huge
// negative log alpha (alpha = 0 written as -1e4) keeps no digits for the small
// differences after it, whereas the products stay exact to a few ulp (and exactly 0
// across such a token). Padding rows of a partial chunk get beta = 0 and alpha = 1:
// they change nothing and their outputs are not stored.
//
// Kernels, in stream order:
//   plan   -- validates cu_seqlens, lists the chunks (sequence, first token,
//             length) and each sequence's first chunk; writes the status word.
//   prep   -- one CTA per (chunk, head): W, Utilde, the masked A = QK^T . Gamma,
//             gamma and kdec_i = Gamma_{C-1,i}.
//   chain  -- one CTA per (sequence, head, 32 value columns): walks the chunks
//             of its sequence in order, carrying its 32 columns of S (the
//             columns of S evolve independently) in shared memory.
#include "internal.h"

namespace gdr {

// ----------------------------------------------------------------------------- plan

// Exclusive prefix sum of one int per thread over a block of 1024 threads; *total gets
// the block's sum. Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += up;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int up = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += up;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int ex = inc - x + (warp ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();  // warp_sums may be reused
    return ex;
}

// The chunk plan, phase-major. Sequence n, of m_n chunks, gives its chunks
// [floor(f m_n / P), floor((f + 1) m_n / P)) to phase f. Chunks are numbered phase by
// phase and, within a phase, sequence by sequence, so that the chunks of one phase are
// contiguous and so are the chunks of one sequence within a phase. Outputs:
//   plan[chunk]                       (sequence, first token, tokens, index in the sequence)
//   seq_chunk[f * (num_seqs + 1) + n] first chunk of sequence n in phase f; the entry at
//                                     n = num_seqs is the end of phase f
//   ctl[0] status, ctl[1] number of chunks, ctl[2 + f] first chunk of phase f (f <= P)
//   zero[0 .. n_zero)                 cleared (the fused schedule's unit-solved flags)
// A single block of 1024 threads: sequences in blocks of 1024 for the prefix sums, then a
// group of threads per sequence writes its plan entries.
//
// With `order` (the fused schedule over packed sequences, one phase, at most
// kMaxClaimSeqs sequences) it also lists the claim order of the solve and the chains'
// triggers. Sequence n of m_n chunks starts its chains s_n = m_max - m_n chain steps
// after the longest, so that all end together; its chunk j is due at step s_n + j, and
// the rows (n, j) are claimed in order of that step (ties by sequence). A sequence's
// chain CTAs solve until the claims reach trig[n], then run their chains. The trigger
// is no earlier than the sequence's first row (H x that row's place in the order), and
// late enough that the units still unclaimed can be solved in the m_n steps left: in
// those steps every chain k runs min(m_k, m_n) of its steps, and each SM that runs no
// chain solves about one unit per chain step (a unit takes about 2 us of an SM when
// four are in flight on it, a chain step beside the solve about 1.8 us), so
// trig[n] >= U - (sms m_n - chains_per_seq sum_k min(m_k, m_n)) for U units in all.
// The claim counter ctl[kClaimWord] starts at zero. When the SMs the chains leave free
// over the longest chain's steps could solve less than half of the units (equal or
// nearly equal lengths over many chains), little of the solve would overlap the chains
// and the two-kernel pair that follows the fused launch is faster: ctl[kPairWord] = 1
// hands the call to it (else 0).
__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t *__restrict__ cu, int64_t num_seqs, int64_t total_tokens,
            int64_t max_chunks, int phases, int4 *__restrict__ plan,
            int32_t *__restrict__ seq_chunk, int32_t *__restrict__ ctl,
            int32_t *__restrict__ zero, int64_t n_zero, int4 *__restrict__ order,
            int32_t *__restrict__ trig, int H, int chains_per_seq, int sms) {
    __shared__ int s_warp[32];
    __shared__ int s_off[kMaxPhases + 1];
    __shared__ int s_bad;
    __shared__ int s_m[kMaxClaimSeqs], s_mmax;  // (claim order) chunks per sequence, and most
    const int tid = threadIdx.x;
    const int64_t row = num_seqs + 1;  // seq_chunk entries per phase
    // the solve kernel after this one may be launched now (programmatic launch): it sets
    // itself up and waits for this grid to complete before reading the plan
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) s_bad = 0;
    for (int64_t i = tid; i < n_zero; i += blockDim.x) zero[i] = 0;
    __syncthreads();
    const int64_t seq_len = cu ? 0 : total_tokens / num_seqs;
    // first token and length of sequence n; false if cu_seqlens is out of range there
    auto seq_range = [&](int64_t n, int64_t &t0, int64_t &len) {
        if (!cu) {
            t0 = n * seq_len;
            len = seq_len;
            return true;
        }
        t0 = cu[n];
        const int64_t t1 = cu[n + 1];
        len = t1 - t0;
        if (len < 0 || t0 < 0 || t1 > total_tokens) {
            len = 0;
            return false;
        }
        return true;
    };
    // pass 1: each sequence's first chunk in each phase, relative to the phase's start
    int carry[kMaxPhases];
#pragma unroll
    for (int f = 0; f < kMaxPhases; ++f) carry[f] = 0;
    for (int64_t base = 0; base < num_seqs; base += blockDim.x) {
        const int64_t n = base + tid;
        int64_t m = 0;
        if (n < num_seqs) {
            int64_t t0, len;
            if (!seq_range(n, t0, len)) s_bad = 1;
            m = (len + kChunk - 1) / kChunk;
        }
#pragma unroll
        for (int f = 0; f < kMaxPhases; ++f) {
            if (f >= phases) break;
            const int cnt = (int)((f + 1) * m / phases - f * m / phases);
            int tot;
            const int ex = block_exclusive_scan(cnt, s_warp, &tot);
            if (n < num_seqs) seq_chunk[f * row + n] = carry[f] + ex;
            carry[f] += tot;
        }
    }
    if (tid == 0) {
        int acc = 0;
#pragma unroll
        for (int f = 0; f < kMaxPhases; ++f) {
            if (f >= phases) break;
            s_off[f] = acc;
            acc += carry[f];
        }
        s_off[phases] = acc;
        if (cu && (cu[0] != 0 || cu[num_seqs] != total_tokens)) s_bad = 1;
        if (acc > max_chunks) s_bad = 1;
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    if (!bad) {
        // pass 2: absolute chunk numbers (each thread revisits its own entries)
        for (int64_t base = 0; base < num_seqs; base += blockDim.x) {
            const int64_t n = base + tid;
            if (n < num_seqs)
                for (int f = 0; f < phases; ++f) seq_chunk[f * row + n] += s_off[f];
        }
        if (tid < phases) seq_chunk[tid * row + num_seqs] = s_off[tid + 1];
        __syncthreads();
        // pass 3: the plan entries; G groups of 1024 / G threads, a group per sequence
        int G = 1;
        while (G < 32 && 2 * G <= num_seqs) G *= 2;
        const int gsize = (int)blockDim.x / G, g = tid / gsize, gt = tid % gsize;
        for (int64_t n = g; n < num_seqs; n += G) {
            int64_t t0, len;
            seq_range(n, t0, len);
            const int64_t m = (len + kChunk - 1) / kChunk;
            for (int f = 0; f < phases; ++f) {
                const int64_t cb = f * m / phases, ce = (f + 1) * m / phases;
                const int64_t first = seq_chunk[f * row + n];
                for (int64_t j = cb + gt; j < ce; j += gsize) {
                    const int64_t rem = len - j * kChunk;
                    plan[first + (j - cb)] = make_int4((int)n, (int)(t0 + j * kChunk),
                                                       (int)(rem < kChunk ? rem : kChunk), (int)j);
                }
            }
        }
        // pass 4: the claim order and the triggers
        if (order && num_seqs <= kMaxClaimSeqs) {
            if (tid == 0) s_mmax = 0;
            __syncthreads();
            for (int n = tid; n < num_seqs; n += blockDim.x) {
                s_m[n] = seq_chunk[n + 1] - seq_chunk[n];
                atomicMax(&s_mmax, s_m[n]);
            }
            __syncthreads();
            const int mmax = s_mmax, rows = s_off[1];
            const int64_t units = (int64_t)rows * H;
            if (tid == 0) {
                const int64_t free_all = (int64_t)sms * mmax - (int64_t)chains_per_seq * rows;
                ctl[kPairWord] = 2 * free_all < units ? 1 : 0;
            }
            for (int n = g; n < num_seqs; n += G) {
                const int m = s_m[n], sn = mmax - m;
                int64_t t0, len;
                seq_range(n, t0, len);
                for (int j = gt; j < m; j += gsize) {
                    // rows of sequence k due before row (n, j), or at the same step if k < n
                    const int due = sn + j;
                    int pos = 0;
                    for (int k = 0; k < num_seqs; ++k) {
                        int c = due - (mmax - s_m[k]) + (k < n ? 1 : 0);
                        pos += c < 0 ? 0 : (c > s_m[k] ? s_m[k] : c);
                    }
                    const int64_t rem = len - (int64_t)j * kChunk;
                    order[pos] = make_int4(seq_chunk[n] + j, (int)(t0 + (int64_t)j * kChunk),
                                           (int)(rem < kChunk ? rem : kChunk), n);
                    if (j == 0) {
                        int64_t steps = 0;  // chain steps of all sequences in the last m steps
                        for (int k = 0; k < num_seqs; ++k) steps += s_m[k] < m ? s_m[k] : m;
                        const int64_t free_steps = (int64_t)sms * m - (int64_t)chains_per_seq * steps;
                        const int64_t late = units - (free_steps > 0 ? free_steps : 0);
                        const int64_t first = (int64_t)pos * H;
                        trig[n] = (int)(late > first ? late : first);
                    }
                }
                // a sequence without chunks solves to the end; its chain only copies S0
                if (m == 0 && gt == 0) trig[n] = (int)units;
            }
        }
    }
    if (order && bad)  // no chain runs; no CTA solves first
        for (int64_t n = tid; n < num_seqs && n < kMaxClaimSeqs; n += blockDim.x) trig[n] = 0;
    if (tid == 0) {
        ctl[0] = bad ? GDR_ERR_BAD_SEQLENS : GDR_OK;
        ctl[1] = bad ? 0 : s_off[phases];
        for (int f = 0; f <= phases; ++f) ctl[2 + f] = bad ? 0 : s_off[f];
        ctl[kClaimWord] = 0;
    }
}

int launch_plan(const PrefillArgs &a, const WsLayout &L, int phases) {
    const bool fused = phases == 0;
    // the fused schedule over packed sequences claims its units in a planned order
    const bool claim = fused && L.tensor_path && a.cu_seqlens;
    plan_kernel<<<1, 1024, 0, a.stream>>>(a.cu_seqlens, a.num_seqs, a.total_tokens, L.max_chunks,
                                          plan_phases(phases), (int4 *)(a.ws + L.plan),
                                          (int32_t *)(a.ws + L.seq_chunk),
                                          (int32_t *)(a.ws + L.ctl),
                                          L.tensor_path ? (int32_t *)(a.ws + L.F) : nullptr,
                                          !L.tensor_path ? 0
                                          : (fused ? L.max_chunks * a.H : 0),
                                          claim ? (int4 *)(a.ws + L.order) : nullptr,
                                          claim ? (int32_t *)(a.ws + L.trig) : nullptr, a.H,
                                          a.H * (a.dv / 128), current_device_sms());
    return cuda_status(cudaGetLastError());
}

// ----------------------------------------------------------------------------- prep

// Four consecutive elements at p (16-byte aligned for fp32, 8-byte for bf16) as fp32.
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

constexpr int kPrepThreads = 256;

template <int DK> struct PrepSmem {
    static constexpr int KP = DK + 1;  // padded row pitch (floats)
    static constexpr int CP = kChunk + 1;
    static constexpr size_t floats = 2 * kChunk * KP + 4 * kChunk * CP + 5 * kChunk;
    static constexpr size_t bytes = floats * sizeof(float);
    // per-channel rates: the cumulative log decay [C][KP] after the rest
    static constexpr size_t bytes_per_channel = bytes + kChunk * KP * sizeof(float);
};

template <typename Tin, int DK>
__global__ void __launch_bounds__(kPrepThreads)
exact_prep_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                  const float *__restrict__ log_alpha, const float *__restrict__ beta, int H,
                  int dv, const int4 *__restrict__ plan, const int32_t *__restrict__ ctl,
                  float *__restrict__ Wws, float *__restrict__ Uws, float *__restrict__ Aws,
                  float *__restrict__ gws, int additive, int prologue,
                  const float *__restrict__ gate_A, float *__restrict__ gcws) {
    // gws receives, per chunk, gamma[C], kdec[C], then 1/|q_t| and 1/|k_t| (ones without
    // the prologue). With the additive rule the write does not read the state: L = 0 (so
    // T = diag(beta)) and W = 0. With the layer's prologue the rows of q and k are scaled
    // to unit length here and the gates come from their pre-activations.
    // With one rate per key channel (gcws non-null; log_alpha [tokens, H, DK]) the decay
    // moves inside the key products: g_t is a vector, the Gram entries are
    // sum_d k_t[d] k_i[d] exp(g_t[d] - g_i[d]) (likewise q_t.k_i), W = T (gamma . K) by
    // rows, and gcws receives g per chunk token and channel for the chain; gamma and kdec
    // are then ones. Every exponent is g_t - g_i with i <= t, or g_t: all factors <= 1.
    using SM = PrepSmem<DK>;
    constexpr int KP = SM::KP, CP = SM::CP, C = kChunk;
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (ctl[0] != GDR_OK || c >= ctl[1]) return;
    const int4 p = plan[c];
    const int64_t t0 = p.y;
    const int len = p.z;

    extern __shared__ float smem[];
    float *ks = smem;                 // [C][KP]
    float *qs = ks + C * KP;          // [C][KP]
    float *Lm = qs + C * KP;          // [C][CP] strictly lower: beta_t Gamma_ti k_t.k_i
    float *Am = Lm + C * CP;          // [C][CP] lower incl. diagonal: Gamma_ti q_t.k_i
    float *Tm = Am + C * CP;          // [C][CP] T = (I + L)^{-1} diag(beta)
    float *Gm = Tm + C * CP;          // [C][CP] Gamma_ti (i <= t)
    float *al = Gm + C * CP;          // [C] alpha (1 on padding rows)
    float *bs = al + C;               // [C] beta (0 on padding rows)
    float *gam = bs + C;              // [C] gamma
    float *nq = gam + C;              // [C] 1/|q_t| (prologue), else 1
    float *nk = nq + C;               // [C] 1/|k_t|
    float *Gs = nk + C;               // [C][KP] per-channel rates: g_t[d] (after the rest)
    const bool per_channel = gcws != nullptr;

    {  // keys and queries, four elements a load, every load issued before any is used
        constexpr int NK = C * DK / 4 / kPrepThreads;
        float4 kv4[NK], qv4[NK];
#pragma unroll
        for (int r = 0; r < NK; ++r) {
            const int e = 4 * (tid + r * kPrepThreads), t = e / DK, d = e % DK;
            kv4[r] = qv4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < len) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DK + d;
                kv4[r] = load4(k + off);
                qv4[r] = load4(q + off);
            }
        }
#pragma unroll
        for (int r = 0; r < NK; ++r) {
            const int e = 4 * (tid + r * kPrepThreads), t = e / DK, d = e % DK;
            float *kr = ks + t * KP + d, *qr = qs + t * KP + d;
            kr[0] = kv4[r].x; kr[1] = kv4[r].y; kr[2] = kv4[r].z; kr[3] = kv4[r].w;
            qr[0] = qv4[r].x; qr[1] = qv4[r].y; qr[2] = qv4[r].z; qr[3] = qv4[r].w;
        }
    }
    if (tid < C) {
        float b = 0.f, a = 1.f;
        if (tid < len) {
            const size_t off = (size_t)(t0 + tid) * H + h;
            if (prologue) {
                b = prologue_beta(beta[off]);
                if (!per_channel) a = expf(prologue_log_alpha(log_alpha[off], gate_A ? gate_A[h] : 1.f));
            } else {
                b = beta[off];
                if (!per_channel) a = expf(log_alpha[off]);
            }
        }
        bs[tid] = b;
        al[tid] = a;  // (per-channel rates: 1, so the per-head factors below are ones)
    }
    if (per_channel) {  // log alpha per token and channel (0 on padding rows)
        const float A = prologue && gate_A ? gate_A[h] : 1.f;
        for (int idx = tid; idx < C * DK; idx += blockDim.x) {
            const int t = idx / DK, d = idx % DK;
            float la = 0.f;
            if (t < len) {
                const float x = log_alpha[((size_t)(t0 + t) * H + h) * DK + d];
                la = prologue ? prologue_log_alpha(x, A) : x;
            }
            Gs[t * KP + d] = la;
        }
        __syncthreads();
        if (tid < DK) {  // inclusive prefix sum over the chunk's tokens, one channel a thread
            float acc = 0.f;
            for (int t = 0; t < C; ++t) {
                acc += Gs[t * KP + tid];
                Gs[t * KP + tid] = acc;
            }
        }
    }
    __syncthreads();
    if (prologue) {  // unit-length rows: four threads per row of k and of q
        const int t = tid >> 2, part = tid & 3;
        float sk = 0.f, sq = 0.f;
        for (int d = part; d < DK; d += 4) {
            sk = fmaf(ks[t * KP + d], ks[t * KP + d], sk);
            sq = fmaf(qs[t * KP + d], qs[t * KP + d], sq);
        }
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        const float ik = prologue_inv_norm(sk), iq = prologue_inv_norm(sq);
        for (int d = part; d < DK; d += 4) {
            ks[t * KP + d] *= ik;
            qs[t * KP + d] *= iq;
        }
        if (part == 0) {
            nk[t] = ik;
            nq[t] = iq;
        }
    } else if (tid < C) {
        nk[tid] = 1.f;
        nq[tid] = 1.f;
    }
    __syncthreads();
    if (tid < C) {  // row t of Gamma by a running product from the diagonal down; then gamma_t
        const int t = tid;
        float prod = 1.f;
        for (int i = t; i >= 0; --i) {
            Gm[t * CP + i] = prod;      // prod_{i<j<=t} alpha_j
            prod *= al[i];
        }
        gam[t] = prod;                  // prod_{j<=t} alpha_j
    }
    __syncthreads();

    if (per_channel) {
        for (int idx = tid; idx < C * C; idx += blockDim.x) {
            const int t = idx / C, i = idx % C;
            float kk = 0.f, qk = 0.f;
            if (i <= t) {
                for (int d = 0; d < DK; ++d) {
                    const float ki = ks[i * KP + d] * expf(Gs[t * KP + d] - Gs[i * KP + d]);
                    kk = fmaf(ks[t * KP + d], ki, kk);
                    qk = fmaf(qs[t * KP + d], ki, qk);
                }
            }
            Lm[t * CP + i] = (i < t && !additive) ? bs[t] * kk : 0.f;
            Am[t * CP + i] = qk;
        }
    } else {
        // 4 x 4 blocks of (t, i) per thread: per feature, 4 keys and 4 queries of rows t and 4
        // keys of rows i serve 32 products; blocks right of the diagonal are zero
        static_assert(C * C / 16 == kPrepThreads, "one 4 x 4 block per thread");
        const int t0 = 4 * (tid / (C / 4)), i0 = 4 * (tid % (C / 4));
        float kk[4][4], qk[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) kk[a][b] = qk[a][b] = 0.f;
        if (i0 <= t0 + 3) {
#pragma unroll 4
            for (int d = 0; d < DK; ++d) {
                float kt[4], qt[4], ki[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    kt[a] = ks[(t0 + a) * KP + d];
                    qt[a] = qs[(t0 + a) * KP + d];
                    ki[a] = ks[(i0 + a) * KP + d];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        kk[a][b] = fmaf(kt[a], ki[b], kk[a][b]);
                        qk[a][b] = fmaf(qt[a], ki[b], qk[a][b]);
                    }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int t = t0 + a, i = i0 + b;
                const float dec = i <= t ? Gm[t * CP + i] : 0.f;
                Lm[t * CP + i] = (i < t && !additive) ? bs[t] * dec * kk[a][b] : 0.f;
                Am[t * CP + i] = dec * qk[a][b];
            }
    }
    __syncthreads();

    // Forward substitution, one column of T per thread: (I + L) x = beta_j e_j. The column
    // stays in registers (both loops unrolled, so every index is a constant; x_i = 0 for
    // i < j), each row's sum in four partial sums.
    if (tid < C) {
        const int j = tid;
        float x[C];
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int i = 0; i + 3 < t; i += 4) {
                s0 = fmaf(Lm[t * CP + i], x[i], s0);
                s1 = fmaf(Lm[t * CP + i + 1], x[i + 1], s1);
                s2 = fmaf(Lm[t * CP + i + 2], x[i + 2], s2);
                s3 = fmaf(Lm[t * CP + i + 3], x[i + 3], s3);
            }
#pragma unroll
            for (int i = t & ~3; i < t; ++i) s0 = fmaf(Lm[t * CP + i], x[i], s0);
            x[t] = t == j ? bs[j] : (t > j ? -((s0 + s1) + (s2 + s3)) : 0.f);
        }
#pragma unroll
        for (int t = 0; t < C; ++t) Tm[t * CP + j] = x[t];
    }
    __syncthreads();

    const size_t cb = (size_t)c * H + h;
    float *Wout = Wws + cb * C * DK;
    if (per_channel) {
        for (int idx = tid; idx < C * DK; idx += blockDim.x) {
            const int t = idx / DK, d = idx % DK;
            float s = 0.f;
            for (int i = 0; i <= t; ++i)  // rows gamma_i[d] k_i[d]
                s = fmaf(Tm[t * CP + i] * expf(Gs[i * KP + d]), ks[i * KP + d], s);
            Wout[idx] = additive ? 0.f : s;
        }
    } else {
        // 4 x 4 blocks of (t, d) per thread; T is zero right of its diagonal, so a block's
        // sums run to its last row, each in the order of the unblocked loop
        constexpr int NBD = DK / 4;
        for (int blk = tid; blk < (C / 4) * NBD; blk += kPrepThreads) {
            const int tb = 4 * (blk / NBD), d0 = 4 * (blk % NBD);
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
            for (int i = 0; i <= tb + 3; ++i) {
                const float gi = gam[i];
                float tv[4], kv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    tv[a] = Tm[(tb + a) * CP + i] * gi;
                    kv[a] = ks[i * KP + d0 + a];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(tv[a], kv[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
                *reinterpret_cast<float4 *>(Wout + (tb + a) * DK + d0) =
                    additive ? make_float4(0.f, 0.f, 0.f, 0.f)
                             : make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
    }
    if (per_channel)
        for (int idx = tid; idx < C * DK; idx += blockDim.x)
            gcws[cb * C * DK + idx] = Gs[(idx / DK) * KP + idx % DK];
    // Utilde = T V, 64 value columns at a time staged in shared memory over the queries
    // (spent once the Gram is formed); padding rows of V are zero
    float *Uout = Uws + cb * C * dv;
    float *Vs = qs;  // [C][64 + 1]
    constexpr int VB = 64, VP = VB + 1;
    static_assert(VP <= KP, "a value block fits in the query tile");
    for (int jb = 0; jb < dv; jb += VB) {
        const int nb = dv - jb < VB ? dv - jb : VB;
        __syncthreads();  // (the queries, or the previous block, are read)
#pragma unroll
        for (int r = 0; r < C * VB / 4 / kPrepThreads; ++r) {  // four elements a load
            const int e = 4 * (tid + r * kPrepThreads), i = e / VB, j = e % VB;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < len && j < nb) x = load4(v + ((size_t)(t0 + i) * H + h) * dv + jb + j);
            float *vr = Vs + i * VP + j;
            vr[0] = x.x; vr[1] = x.y; vr[2] = x.z; vr[3] = x.w;
        }
        __syncthreads();
        // 4 x 4 blocks of (t, j) per thread, as for W
        const int nbj = nb / 4;
        for (int blk = tid; blk < (C / 4) * nbj; blk += kPrepThreads) {
            const int tb = 4 * (blk / nbj), j4 = 4 * (blk % nbj);
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
            for (int i = 0; i <= tb + 3; ++i) {
                float tv[4], vv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    tv[a] = Tm[(tb + a) * CP + i];
                    vv[a] = Vs[i * VP + j4 + a];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(tv[a], vv[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
                *reinterpret_cast<float4 *>(Uout + (size_t)(tb + a) * dv + jb + j4) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
    }
    float *Aout = Aws + cb * C * C;
    for (int idx = tid; idx < C * C; idx += blockDim.x) Aout[idx] = Am[(idx / C) * CP + idx % C];
    if (tid < C) {
        gws[cb * 4 * C + tid] = gam[tid];
        gws[cb * 4 * C + C + tid] = Gm[(C - 1) * CP + tid];  // kdec_i = Gamma_{C-1,i}
        gws[cb * 4 * C + 2 * C + tid] = nq[tid];
        gws[cb * 4 * C + 3 * C + tid] = nk[tid];
    }
}

// ----------------------------------------------------------------------------- chain

constexpr int kChainCols = 32;  // value columns per chain CTA
constexpr int kChainThreads = 256;


template <int DK> struct ChainSmem {
    static constexpr int KP = DK + 1;
    static constexpr int SP = kChainCols + 4;  // (rows of S and U on 16-byte boundaries)
    static constexpr size_t floats = DK * SP + 3 * kChunk * KP + kChunk * (kChunk + 1) +
                                     kChunk * SP + 5 * kChunk;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <typename Tin, int DK>
__global__ void __launch_bounds__(kChainThreads)
exact_chain_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const float *__restrict__ S0, const int32_t *__restrict__ cu,
                   int64_t num_seqs, int64_t total_tokens, int H, int dv,
                   const int32_t *__restrict__ seq_chunk, const int32_t *__restrict__ ctl,
                   const float *__restrict__ Wws, const float *__restrict__ Uws,
                   const float *__restrict__ Aws, const float *__restrict__ gws,
                   const float *__restrict__ gcws, Tin *__restrict__ o, float *__restrict__ S_final) {
    // gcws (per-channel rates, else null): g_t[d] per chunk token and channel. Then
    // q_t is scaled by gamma_t[d] = exp(g_t[d]), k_i by exp(g_C[d] - g_i[d]) for the
    // state update, and row d of S decays by exp(g_C[d]); gamma and kdec are ones.
    using SM = ChainSmem<DK>;
    constexpr int KP = SM::KP, SP = SM::SP, C = kChunk, NC = kChainCols, CP = C + 1;
    if (ctl[0] != GDR_OK) return;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int j0 = blockIdx.y * NC;
    const int tid = threadIdx.x;
    int64_t t_begin, t_end;
    if (cu) {
        t_begin = cu[n];
        t_end = cu[n + 1];
    } else {
        const int64_t sl = total_tokens / num_seqs;
        t_begin = (int64_t)n * sl;
        t_end = t_begin + sl;
    }
    const int c_first = seq_chunk[n];
    const int n_chunks = seq_chunk[n + 1] - c_first;

    extern __shared__ float smem[];
    float *Ss = smem;            // [DK][SP]  the state's columns j0 .. j0+31
    float *Wc = Ss + DK * SP;    // [C][KP]
    float *qs = Wc + C * KP;     // [C][KP]
    float *ks = qs + C * KP;     // [C][KP]
    float *Ac = ks + C * KP;     // [C][CP]
    float *Uc = Ac + C * CP;     // [C][SP]  Utilde, then U
    static_assert((DK * SP + 3 * C * KP + C * CP) % 4 == 0, "U rows on 16-byte boundaries");
    float *gam = Uc + C * SP;    // [C] gamma_t
    float *kdec = gam + C;       // [C] Gamma_{C-1,i}
    float *nqk = kdec + C;       // [2][C] 1/|q_t|, 1/|k_t| (the prologue; else 1)

    const size_t s_base = ((size_t)n * H + h) * DK * dv;
    for (int idx = tid; idx < DK * NC; idx += blockDim.x) {
        const int d = idx / NC, j = idx % NC;
        Ss[d * SP + j] = S0 ? S0[s_base + (size_t)d * dv + j0 + j] : 0.f;
    }
    __syncthreads();

    for (int cc = 0; cc < n_chunks; ++cc) {
        const size_t cb = (size_t)(c_first + cc) * H + h;
        const int64_t tc0 = t_begin + (int64_t)cc * C;
        const int len = (int)((t_end - tc0) < C ? (t_end - tc0) : C);
        if (tid < 2 * C) nqk[tid] = gws[cb * 4 * C + 2 * C + tid];
        // W, q and k, A and Utilde of the chunk: every load of a thread is issued before
        // any is used, four elements at a time
        constexpr int NK = C * DK / 4 / kChainThreads, NA = C * C / 4 / kChainThreads,
                      NU = C * NC / 4 / kChainThreads;
        float4 wv[NK], kv4[NK], qv4[NK], gv4[NK], gl4[NK], av[NA], uv[NU];
#pragma unroll
        for (int r = 0; r < NK; ++r) {
            const int e = 4 * (tid + r * kChainThreads), t = e / DK, d = e % DK;
            wv[r] = load4(Wws + cb * C * DK + e);
            kv4[r] = qv4[r] = gv4[r] = gl4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < len) {
                const size_t off = ((size_t)(tc0 + t) * H + h) * DK + d;
                kv4[r] = load4(k + off);
                qv4[r] = load4(q + off);
                if (gcws) {
                    gv4[r] = load4(gcws + cb * C * DK + t * DK + d);
                    gl4[r] = load4(gcws + cb * C * DK + (C - 1) * DK + d);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < NA; ++r) av[r] = load4(Aws + cb * C * C + 4 * (tid + r * kChainThreads));
#pragma unroll
        for (int r = 0; r < NU; ++r) {
            const int e = 4 * (tid + r * kChainThreads), t = e / NC, j = e % NC;
            uv[r] = load4(Uws + cb * C * dv + (size_t)t * dv + j0 + j);
        }
        __syncthreads();  // (nqk)
#pragma unroll
        for (int r = 0; r < NK; ++r) {
            const int e = 4 * (tid + r * kChainThreads), t = e / DK, d = e % DK;
            const float w4[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
            const float k4[4] = {kv4[r].x, kv4[r].y, kv4[r].z, kv4[r].w};
            const float q4[4] = {qv4[r].x, qv4[r].y, qv4[r].z, qv4[r].w};
            const float g4[4] = {gv4[r].x, gv4[r].y, gv4[r].z, gv4[r].w};
            const float c4[4] = {gl4[r].x, gl4[r].y, gl4[r].z, gl4[r].w};
            const float nk = t < len ? nqk[C + t] : 0.f, nq = t < len ? nqk[t] : 0.f;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                float kv = k4[x] * nk, qv = q4[x] * nq;
                if (gcws) {
                    qv *= expf(g4[x]);
                    kv *= expf(c4[x] - g4[x]);
                }
                Wc[t * KP + d + x] = w4[x];
                ks[t * KP + d + x] = kv;
                qs[t * KP + d + x] = qv;
            }
        }
#pragma unroll
        for (int r = 0; r < NA; ++r) {
            const int e = 4 * (tid + r * kChainThreads), t = e / C, i = e % C;
            Ac[t * CP + i] = av[r].x;
            Ac[t * CP + i + 1] = av[r].y;
            Ac[t * CP + i + 2] = av[r].z;
            Ac[t * CP + i + 3] = av[r].w;
        }
#pragma unroll
        for (int r = 0; r < NU; ++r) {
            const int e = 4 * (tid + r * kChainThreads), t = e / NC, j = e % NC;
            Uc[t * SP + j] = uv[r].x;
            Uc[t * SP + j + 1] = uv[r].y;
            Uc[t * SP + j + 2] = uv[r].z;
            Uc[t * SP + j + 3] = uv[r].w;
        }
        if (tid < C) {
            gam[tid] = gws[cb * 4 * C + tid];
            kdec[tid] = gws[cb * 4 * C + C + tid];
        }
        __syncthreads();

        // U = Utilde - W S  and  QS, one token row and 8 columns per thread.
        const int t = tid >> 2, jg = (tid & 3) * 8;
        float u[8], qsv[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            u[x] = 0.f;
            qsv[x] = 0.f;
        }
#pragma unroll 4
        for (int d = 0; d < DK; ++d) {
            const float w = Wc[t * KP + d], qq = qs[t * KP + d];
            const float4 sa = *reinterpret_cast<const float4 *>(Ss + d * SP + jg);
            const float4 sb = *reinterpret_cast<const float4 *>(Ss + d * SP + jg + 4);
            const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                u[x] = fmaf(w, sv[x], u[x]);
                qsv[x] = fmaf(qq, sv[x], qsv[x]);
            }
        }
        __syncthreads();  // every thread has read S and Utilde is still intact
#pragma unroll
        for (int x = 0; x < 8; ++x) Uc[t * SP + jg + x] -= u[x];
        __syncthreads();
        // O = gamma_t QS + A U
        if (t < len) {
            float outv[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) outv[x] = gam[t] * qsv[x];
            for (int i = 0; i <= t; ++i) {
                const float aw = Ac[t * CP + i];
                const float4 ua = *reinterpret_cast<const float4 *>(Uc + i * SP + jg);
                const float4 ub = *reinterpret_cast<const float4 *>(Uc + i * SP + jg + 4);
                const float uv8[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                for (int x = 0; x < 8; ++x) outv[x] = fmaf(aw, uv8[x], outv[x]);
            }
            Tin *op = o + ((size_t)(tc0 + t) * H + h) * dv + j0 + jg;
#pragma unroll
            for (int x = 0; x < 8; ++x) op[x] = from_f32<Tin>(outv[x]);
        }
        // S <- gamma_C S + Ktilde^T U
        {
            constexpr int TPR = 256 / DK;          // threads per state row
            constexpr int CPT = NC / TPR;          // columns per thread
            const int d = tid / TPR, jb = (tid % TPR) * CPT;
            const float gC = gcws ? expf(gcws[cb * C * DK + (C - 1) * DK + d]) : gam[C - 1];
            static_assert(CPT % 4 == 0, "state columns in 16-byte groups");
            float acc[CPT];
#pragma unroll
            for (int x4 = 0; x4 < CPT / 4; ++x4) {
                const float4 s4 = *reinterpret_cast<const float4 *>(Ss + d * SP + jb + 4 * x4);
                acc[4 * x4] = gC * s4.x;
                acc[4 * x4 + 1] = gC * s4.y;
                acc[4 * x4 + 2] = gC * s4.z;
                acc[4 * x4 + 3] = gC * s4.w;
            }
#pragma unroll 4
            for (int i = 0; i < C; ++i) {
                const float kt = kdec[i] * ks[i * KP + d];
#pragma unroll
                for (int x4 = 0; x4 < CPT / 4; ++x4) {
                    const float4 u4 = *reinterpret_cast<const float4 *>(Uc + i * SP + jb + 4 * x4);
                    acc[4 * x4] = fmaf(kt, u4.x, acc[4 * x4]);
                    acc[4 * x4 + 1] = fmaf(kt, u4.y, acc[4 * x4 + 1]);
                    acc[4 * x4 + 2] = fmaf(kt, u4.z, acc[4 * x4 + 2]);
                    acc[4 * x4 + 3] = fmaf(kt, u4.w, acc[4 * x4 + 3]);
                }
            }
            __syncthreads();  // all reads of the old S (QS above) are done
#pragma unroll
            for (int x4 = 0; x4 < CPT / 4; ++x4)
                *reinterpret_cast<float4 *>(Ss + d * SP + jb + 4 * x4) =
                    make_float4(acc[4 * x4], acc[4 * x4 + 1], acc[4 * x4 + 2], acc[4 * x4 + 3]);
        }
        __syncthreads();
    }

    for (int idx = tid; idx < DK * NC; idx += blockDim.x) {
        const int d = idx / NC, j = idx % NC;
        S_final[s_base + (size_t)d * dv + j0 + j] = Ss[d * SP + j];
    }
}

// ----------------------------------------------------------------------------- launch

template <typename Tin, int DK>
static int launch_exact_t(const PrefillArgs &a, const WsLayout &L) {
    const int32_t *ctl = (const int32_t *)(a.ws + L.ctl);
    float *W = (float *)(a.ws + L.W), *U = (float *)(a.ws + L.U);
    float *A = (float *)(a.ws + L.A), *g = (float *)(a.ws + L.g);
    cudaError_t e;
    const bool per_channel = a.decay == GDR_DECAY_CHANNEL;
    const size_t prep_smem = per_channel ? PrepSmem<DK>::bytes_per_channel : PrepSmem<DK>::bytes;
    float *gc = per_channel ? (float *)(a.ws + L.gc) : nullptr;
    e = cudaFuncSetAttribute(exact_prep_kernel<Tin, DK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    e = cudaFuncSetAttribute(exact_chain_kernel<Tin, DK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ChainSmem<DK>::bytes);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    if (L.max_chunks > 0) {
        dim3 grid((unsigned)L.max_chunks, (unsigned)a.H);
        exact_prep_kernel<Tin, DK><<<grid, kPrepThreads, prep_smem, a.stream>>>(
            (const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, a.log_alpha, a.beta, a.H, a.dv,
            (const int4 *)(a.ws + L.plan), ctl, W, U, A, g, a.rule == GDR_RULE_ADDITIVE ? 1 : 0,
            a.prologue, a.gate_A, gc);
        e = cudaGetLastError();
        if (e != cudaSuccess) return GDR_ERR_CUDA;
    }
    dim3 grid2((unsigned)(a.num_seqs * a.H), (unsigned)(a.dv / kChainCols));
    exact_chain_kernel<Tin, DK><<<grid2, kChainThreads, ChainSmem<DK>::bytes, a.stream>>>(
        (const Tin *)a.q, (const Tin *)a.k, a.S0, a.cu_seqlens, a.num_seqs, a.total_tokens, a.H,
        a.dv, (const int32_t *)(a.ws + L.seq_chunk), ctl, W, U, A, g, gc, (Tin *)a.o, a.S_final);
    return cuda_status(cudaGetLastError());
}

int launch_prefill_exact(const PrefillArgs &a, const WsLayout &L) {
    if (a.dtype == GDR_BF16) {
        if (a.dk == 64) return launch_exact_t<__nv_bfloat16, 64>(a, L);
        return launch_exact_t<__nv_bfloat16, 128>(a, L);
    }
    if (a.dk == 64) return launch_exact_t<float, 64>(a, L);
    return launch_exact_t<float, 128>(a, L);
}

}  // namespace gdr
