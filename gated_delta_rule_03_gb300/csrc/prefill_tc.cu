// prefill_tc.cu -- the kernels of the tensor-core prefill and its host launcher.
//
// The work is split in two (see solve_tc.cuh and chain_tc.cuh): a chunk-parallel solve
// of every (chunk, head) unit, and the sequential chain of each (sequence, head, d_v
// slice). They run in one of two ways:
//  * fused: one cooperative launch holds every chain CTA and, on the remaining SMs, solve
//    CTAs that take the units in chunk-major order; a chain CTA waits (bounded) on each
//    unit's flag before loading its results. Cooperative launch guarantees that all the
//    CTAs are resident together, so the waits always end. Used for batches of equal
//    lengths whose chains leave enough SMs free. For packed sequences of different
//    lengths the solve CTAs claim units from a counter in the order the planning kernel
//    lists (each chain's chunks by the step at which it needs them, when all chains end
//    together), and a chain CTA solves too until the claims reach its sequence's
//    trigger; only then does it start its chain. No solving CTA waits on a chain, so
//    every claimed unit is published. The phased pair follows that launch, and the plan
//    hands the call to one of the two.
//  * phased: separate solve and chain kernels over phases of the chunks (below).
//  * segmented: for a few long chains, which leave most SMs idle under the other two.
//    The state after a run of chunks is affine in the state before it, S_end = P S + R,
//    with P (d_k x d_k) the product of the chunks' transitions gamma_C I - Ktilde^T W
//    and R the end state from zero. Each sequence is cut into n segments; one kernel
//    runs every segment but the last from the identity with zero values (giving P) and
//    from zero (giving R), all segments at once; a scan chains the segments' start
//    states, S_{f+1} = P_f S_f + R_f, in fp32; a second kernel runs every segment from
//    its start state, with output. Chain steps per call fall from m to about 2 m / n.
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include <cooperative_groups.h>

#include "chain_tc.cuh"
#include "solve_tc.cuh"

namespace gdr {
namespace chain {
namespace {

// kSeg: the segmented schedule's launches (summary and chain modes)
template <bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_t,
                const __grid_constant__ CUtensorMap map_o, const TcParams p) {
    // The plan's choice between the fused kernel and this pair: the plan completed before
    // the fused kernel ahead of this launch began, so the word is read at once. A launch
    // left out lets the next one start, and ends only after the kernel ahead of it.
    if (p.only_pair && p.ctl[kPairWord] != 1) {
        griddep_launch_dependents();
        griddep_wait();
        return;
    }
    chain_body<false, kSeg>(map_q, map_k, map_v, map_t, map_o, p, (int)blockIdx.x);
}

static_assert(solve::kSolveWarps * 32 <= kThreads, "the fused launch runs the solve on the chain's block");
constexpr uint32_t FUSED_SMEM_BYTES = SMEM_BYTES > solve::SMEM_BYTES ? SMEM_BYTES : solve::SMEM_BYTES;

// CTAs [0, chain_ctas) run chains, the others the solve. kClaim (packed sequences): the
// solve CTAs claim units from the grid's counter in the plan's claim order, and a chain
// CTA first solves too, until the claims reach the trigger trig[n] of its sequence n
// (the plan puts it where the chain is due to start), then runs its chain.
template <bool kClaim>
__global__ void __launch_bounds__(kThreads, 1)
tc_fused_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_t,
                const __grid_constant__ CUtensorMap map_o, const TcParams p,
                const solve::SolveParams sp, int chain_ctas, const int32_t *trig) {
    if (!kClaim) {
        // Equal lengths: no planning kernel runs ahead of this launch (its plan is closed
        // form). Every CTA clears its share of the unit flags and CTA 0 resets the control
        // words; the grid barrier of the cooperative launch then makes them visible to all
        // before any unit is published or waited on.
        const int n_flags = sp.seqs * sp.seq_chunks * p.H;
        for (int i = (int)(blockIdx.x * blockDim.x + threadIdx.x); i < n_flags; i += (int)(gridDim.x * blockDim.x))
            sp.flags[i] = 0;
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            const int chunks = sp.seqs * sp.seq_chunks;
            p.ctl[0] = GDR_OK;
            p.ctl[1] = chunks;
            p.ctl[2] = 0;
            p.ctl[3] = chunks;
        }
        cooperative_groups::this_grid().sync();
    }
    if (kClaim && p.ctl[kPairWord] == 1) return;  // the two-kernel pair after it runs the call
    if ((int)blockIdx.x < chain_ctas) {
        if (kClaim) {
            const int stop = trig[(int)blockIdx.x / p.n_slices / p.H];
            if (stop > 0) solve::solve_body<true, true>(map_q, map_k, sp, 0, 1, stop, true);
        }
        chain_body<true>(map_q, map_k, map_v, map_t, map_o, p, (int)blockIdx.x);
    } else {
        solve::solve_body<true, kClaim>(map_q, map_k, sp, (int)blockIdx.x - chain_ctas,
                                        (int)gridDim.x - chain_ctas);
    }
}

// The segmented schedule's scan over the segment summaries of one (sequence, head) and
// 16 value columns: X_0 = S_in (or zero), X_{f+1} = P_f X_f + R_f for f < segs, each X_f
// stored as start[f]. P_f is stored transposed in the first d_k columns of its
// [d_k][d_v] matrix. Thread (rb, cb) owns rows 4rb..4rb+3 and columns 2cb, 2cb+1 of X;
// P_f^T is staged in shared memory, the next one loading (cp.async) while this one is
// used.
constexpr int kScanCols = 16, kScanThreads = 256;
constexpr uint32_t SCAN_SMEM_BYTES = (2 * DK * DK + DK * kScanCols) * sizeof(float);

__device__ __forceinline__ void scan_stage_p(float *dst, const float *src, int dv, int tid) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
#pragma unroll 4
    for (int e = tid; e < DK * DK / 4; e += kScanThreads) {
        const int r = e / (DK / 4), c4 = e % (DK / 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s + 16u * e),
                     "l"(src + (size_t)r * dv + 4 * c4)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(kScanThreads)
seg_scan_kernel(const float *__restrict__ S_in, const float *__restrict__ P,
                const float *__restrict__ R, float *__restrict__ start, int NH, int dv, int segs) {
    extern __shared__ float4 scan_smem[];
    float *sPT = reinterpret_cast<float *>(scan_smem);  // 2 x [DK][DK]: P_f^T[k][i]
    float *sX = sPT + 2 * DK * DK;                       // [DK][kScanCols]
    griddep_wait();  // the summaries are complete
    griddep_launch_dependents();
    const int nh = blockIdx.x, c0 = blockIdx.y * kScanCols, tid = threadIdx.x;
    const int cb = tid & 7, rb = tid >> 3;
    const size_t mat = (size_t)DK * dv, set = (size_t)NH * mat;
    if (segs > 0) scan_stage_p(sPT, P + nh * mat, dv, tid);
    for (int e = tid; e < DK * kScanCols; e += kScanThreads) {
        const int r = e / kScanCols, c = e % kScanCols;
        const size_t at = nh * mat + (size_t)r * dv + c0 + c;
        sX[e] = S_in ? S_in[at] : 0.f;
        start[at] = sX[e];
    }
    for (int f = 0; f < segs; ++f) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();  // P_f^T and X_f are in place; P_{f-1}^T is read no more
        if (f + 1 < segs) scan_stage_p(sPT + ((f + 1) & 1) * DK * DK, P + (f + 1) * set + nh * mat, dv, tid);
        const float *pt = sPT + (f & 1) * DK * DK + 4 * rb;
        const float *Rf = R + f * set + nh * mat + (size_t)(4 * rb) * dv + c0 + 2 * cb;
        float2 r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = *reinterpret_cast<const float2 *>(Rf + (size_t)i * dv);
        float y[4][2] = {};
#pragma unroll 8
        for (int k = 0; k < DK; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(pt + k * DK);
            const float2 x = *reinterpret_cast<const float2 *>(sX + k * kScanCols + 2 * cb);
            y[0][0] = fmaf(a.x, x.x, y[0][0]); y[0][1] = fmaf(a.x, x.y, y[0][1]);
            y[1][0] = fmaf(a.y, x.x, y[1][0]); y[1][1] = fmaf(a.y, x.y, y[1][1]);
            y[2][0] = fmaf(a.z, x.x, y[2][0]); y[2][1] = fmaf(a.z, x.y, y[2][1]);
            y[3][0] = fmaf(a.w, x.x, y[3][0]); y[3][1] = fmaf(a.w, x.y, y[3][1]);
        }
        __syncthreads();  // every thread has read X_f
        float *dst = start + (f + 1) * set + nh * mat + (size_t)(4 * rb) * dv + c0 + 2 * cb;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = make_float2(y[i][0] + r[i].x, y[i][1] + r[i].y);
            *reinterpret_cast<float2 *>(sX + (4 * rb + i) * kScanCols + 2 * cb) = v;
            *reinterpret_cast<float2 *>(dst + (size_t)i * dv) = v;
        }
    }
}

}  // namespace
}  // namespace chain

namespace {

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
               const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3],
               CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, type, 3, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace tc {

bool make_map_thd(CUtensorMap *map, const void *base, int d, int H, int64_t T) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * H * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    return encode_3d(map, base, dims, strides, box);
}

bool make_map_rows_f32(CUtensorMap *map, const float *base, int d, int H, int64_t T) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)d * H * 4};
    const cuuint32_t box[3] = {(cuuint32_t)d, 1, 64};
    return encode_3d(map, base, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
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

// The SM count of a device, cached on first use. Threads that race on the first use
// both query and store the same value; the atomics make that race well defined.
std::atomic<int> g_sms[kMaxDevices];

int device_sms(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
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

int current_device_sms() {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess ? device_sms(dev) : 0;
}

// Fused over packed sequences (solve units claimed in the plan's order, chain CTAs
// solving until their chains are due): every chain CTA and at least 16 solve-only CTAs
// fit on the GPU at once, over at most kMaxClaimSeqs sequences (the plan's limit), of
// 32 chunks or more on average (shorter work does not pay for the cooperative launch and
// the ramp of the solve ahead of the chains).
static bool claim_fits(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms) {
    return num_seqs <= kMaxClaimSeqs && num_seqs * H * (dv / chain::NV) + 16 <= sms &&
           total_tokens >= num_seqs * 32 * kChunk;
}

// Fused: the chain CTAs plus at least 1.2 solve CTAs per (sequence, head) must fit on
// the GPU at one CTA per SM. A solve CTA finishes a unit about every 2 us and a chain
// step takes about 1.5 us, so with that many solve CTAs the solve about keeps pace with
// the chains. Only for equal-length sequences (the chunk-major unit order is then
// closed-form).
static bool fused_fits(int64_t num_seqs, int H, int dv, int sms) {
    const int64_t units_per_step = num_seqs * H;
    const int64_t free_sms = sms - units_per_step * (dv / chain::NV);
    return 5 * free_sms >= 6 * units_per_step && free_sms >= 8;
}

// Phased: the solve keeps pace with the chain when the free SMs solve one chunk of every
// (sequence, head) no slower than a chain CTA takes one step (1.25 units per chunk step
// per free SM at the rates above). Every phase restarts the chain's pipeline (fill and
// drain, about 7 us, and a launch behind an event, about 5 us), so a phase keeps at least
// 32 chunks of the average sequence.
static int phased_count(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms) {
    const int64_t units_per_step = num_seqs * H;
    const int64_t free_sms = sms - units_per_step * (dv / chain::NV);
    if (free_sms < 8 || 5 * units_per_step > 4 * free_sms) return 1;
    const int64_t P = total_tokens / num_seqs / kChunk / 32;
    return P < 1 ? 1 : (P > kMaxPhases ? kMaxPhases : (int)P);
}

// GDR_PREFILL_PHASES=1..8 in the environment forces the phased schedule with that many
// phases (a tuning and testing knob: the result does not depend on the schedule).
static int forced_phases() {
    if (const char *env = getenv("GDR_PREFILL_PHASES")) {
        const int v = atoi(env);
        if (v >= 1 && v <= kMaxPhases) return v;
    }
    return 0;
}

// Segmented: worth it when the chains leave most SMs idle. Segment count: the summary
// launch's (sequence, head, slice + 1) CTAs of n - 1 segments, and the second launch's
// (sequence, head, slice) CTAs of n segments, each fit on the GPU at once. It runs the
// solve of every unit first (about 2.3 SM-us per unit) and 2 m / n chain steps, against
// m chain steps of the other schedules (about 1.5 us per chunk step).
static int segment_count(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms) {
    if (!tc_segmentable(num_seqs, total_tokens, H, dv)) return 0;
    const int64_t nh = num_seqs * H, slices = dv / chain::NV;
    int64_t n = 1 + sms / (nh * (slices + 1));
    if (n > kMaxPhases) n = kMaxPhases;
    while (n > 1 && n * nh * slices > sms) --n;
    if (n < 3) return 0;
    const double m = (double)total_tokens / (double)num_seqs / kChunk;
    const double units = m * (double)nh;
    const double chained = 1.5 * m;
    const double segmented = 2.3 * units / sms + 3.0 * m / (double)n + 15.0;
    return segmented < 0.8 * chained ? (int)n : 0;
}

// GDR_PREFILL_SEGMENTS=2..8 forces the segmented schedule with that many segments where
// the workspace holds it (a tuning and testing knob, like GDR_PREFILL_PHASES).
static int forced_segments() {
    if (const char *env = getenv("GDR_PREFILL_SEGMENTS")) {
        const int v = atoi(env);
        if (v >= 2 && v <= kMaxPhases) return v;
    }
    return 0;
}

// Whether the fused schedule's cooperative launch fits on a device, cached on first use
// (0 unknown, 1 yes, 2 no; racing first uses compute and store the same answer).
static std::atomic<int> g_cooperative_ok[kMaxDevices];

// The chain kernels' wait bound, and a test of their give-up path: with
// GDR_DEBUG_CHAIN_FAULT=<chunk> in the environment, the producer of each chain launch's
// CTA 0 skips the K-slot load of that chunk, and every wait gives up after 2e7 SM cycles
// (about 10 ms) instead of 2e9. The roles waiting on the missing load then give up, mark
// the call GDR_ERR_DEVICE_TIMEOUT in the status word and drain; nothing faults or hangs.
namespace chain {
void chain_wait_policy(TcParams &p) {
    p.wait_cycles = sm100::kWaitCycles;
    p.fault_chunk = -1;
    if (const char *env = getenv("GDR_DEBUG_CHAIN_FAULT")) {
        char *end = nullptr;
        const long c = strtol(env, &end, 10);
        if (end != env && *end == '\0' && c >= 0 && c < (1l << 30)) {
            p.fault_chunk = (int)c;
            p.wait_cycles = 20000000;
        }
    }
}
}  // namespace chain

template <typename K>
static bool one_block_fits(K kernel) {
    int blocks = 0;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)chain::FUSED_SMEM_BYTES) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, chain::kThreads,
                                                         chain::FUSED_SMEM_BYTES) == cudaSuccess &&
           blocks >= 1;
}

// (both forms of the fused kernel)
static bool cooperative_ok(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    int known = g_cooperative_ok[dev].load(std::memory_order_relaxed);
    if (!known) {
        int coop = 0;
        const bool yes =
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            one_block_fits(chain::tc_fused_kernel<false>) && one_block_fits(chain::tc_fused_kernel<true>);
        known = yes ? 1 : 2;
        g_cooperative_ok[dev].store(known, std::memory_order_relaxed);
    }
    return known == 1;
}

int tc_schedule_for(int64_t num_seqs, int64_t total_tokens, int H, int dv, int sms, bool varlen,
                    bool cooperative) {
    if (total_tokens == 0) return 1;
    if (const int n = forced_segments())
        if (tc_segmentable(num_seqs, total_tokens, H, dv)) return kSegmentedBase + n;
    if (const int P = forced_phases()) return P;
    if (const int n = segment_count(num_seqs, total_tokens, H, dv, sms)) return kSegmentedBase + n;
    if (varlen && cooperative && claim_fits(num_seqs, total_tokens, H, dv, sms)) return 0;
    if (!varlen && cooperative && fused_fits(num_seqs, H, dv, sms)) return 0;
    return phased_count(num_seqs, total_tokens, H, dv, sms);
}

int tc_schedule(const PrefillArgs &a) {
    int dev = -1;
    if (a.total_tokens == 0 || cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int P = tc_schedule_for(a.num_seqs, a.total_tokens, a.H, a.dv, device_sms(dev),
                                  a.cu_seqlens != nullptr, cooperative_ok(dev));
    if (P == 0 || P > kSegmentedBase) return P;
    return P > 1 && side_stream(a.stream) ? P : 1;
}

int tc_schedule_query(int64_t num_seqs, int64_t total_tokens, int H, int dv, bool varlen) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return tc_schedule_for(num_seqs, total_tokens, H, dv, device_sms(dev), varlen, cooperative_ok(dev));
}

// The fused launch: every chain CTA and, on the remaining SMs, solve CTAs (claiming
// their units, and with chain CTAs solving first, for packed sequences).
static int launch_fused(const PrefillArgs &a, const WsLayout &L, const CUtensorMap &mq,
                        const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mt,
                        const CUtensorMap &mo) {
    using namespace chain;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDR_ERR_CUDA;
    const int n_slices = a.dv / NV;
    const int chain_ctas = (int)(a.num_seqs * a.H * n_slices);
    const int grid = device_sms(dev);
    int32_t *flags = reinterpret_cast<int32_t *>(a.ws + L.F);
    TcParams p = {};
    chain_wait_policy(p);
    const bool claim = a.cu_seqlens != nullptr;
    p.S_in = a.S0;
    p.factors = reinterpret_cast<const float *>(a.ws + L.G);
    p.cu_seqlens = a.cu_seqlens;
    p.seq_chunk = reinterpret_cast<const int32_t *>(a.ws + L.seq_chunk);
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.H = a.H;
    p.dv = a.dv;
    p.n_slices = n_slices;
    p.phase = 0;
    p.phases = 1;
    p.o = (__nv_bfloat16 *)a.o;
    p.S_out = a.S_final;
    p.ctl = (int32_t *)(a.ws + L.ctl);
    p.flags = flags;
    p.additive = a.rule == GDR_RULE_ADDITIVE;
    p.prologue = a.prologue;
    if (a.dv == NV) {  // the output step fused into the chain's epilogue
        p.out_gate = (const __nv_bfloat16 *)a.out_gate;
        p.out_norm_weight = a.out_norm_weight;
        p.out_norm_eps = a.out_norm_eps;
    }
    solve::SolveParams sp = {};
    sp.log_alpha = a.log_alpha;
    sp.beta = a.beta;
    sp.plan = reinterpret_cast<const int4 *>(a.ws + L.plan);
    sp.ctl = p.ctl;
    sp.H = a.H;
    sp.Tout = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.T);
    sp.Gout = reinterpret_cast<float *>(a.ws + L.G);
    sp.phase = 0;
    sp.seqs = (int)a.num_seqs;
    sp.seq_chunks = (int)((a.total_tokens / a.num_seqs + kChunk - 1) / kChunk);
    sp.seq_len = (int)(a.total_tokens / a.num_seqs);
    sp.flags = flags;
    sp.order = reinterpret_cast<const int4 *>(a.ws + L.order);
    sp.claim = p.ctl + kClaimWord;
    sp.additive = a.rule == GDR_RULE_ADDITIVE;
    sp.prologue = a.prologue;
    sp.gate_A = a.gate_A;
    const int32_t *trig = reinterpret_cast<const int32_t *>(a.ws + L.trig);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = FUSED_SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cuda_status(claim ? cudaLaunchKernelEx(&cfg, tc_fused_kernel<true>, mq, mk, mv, mt, mo, p,
                                                  sp, chain_ctas, trig)
                             : cudaLaunchKernelEx(&cfg, tc_fused_kernel<false>, mq, mk, mv, mt, mo, p,
                                                  sp, chain_ctas, trig));
}

// The segmented schedule over `segs` segments per sequence.
static int launch_segmented(const PrefillArgs &a, const WsLayout &L, int segs, const CUtensorMap &mq,
                            const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mt,
                            const CUtensorMap &mo) {
    using namespace chain;
    if (!L.segmentable || a.dk != DK) return GDR_ERR_CUDA;  // the schedule asks for neither
    // the solve of every unit, with the whole GPU
    int st = tc::launch_solve_tc(a, L, mq, mk, -1, 0, a.stream, true);
    if (st != GDR_OK) return st;
    if (cudaFuncSetAttribute(tc_chain_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SCAN_SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int n_slices = a.dv / NV;
    const int64_t NH = a.num_seqs * a.H;
    const size_t set = (size_t)NH * a.dk * a.dv;  // floats of one state set
    float *sets = reinterpret_cast<float *>(a.ws + L.seg);
    float *S_P = sets, *S_R = sets + (kMaxPhases - 1) * set;
    float *S_discard = sets + 2 * (kMaxPhases - 1) * set, *S_start = sets + 3 * (kMaxPhases - 1) * set;
    TcParams p = {};
    chain_wait_policy(p);
    p.factors = reinterpret_cast<const float *>(a.ws + L.G);
    p.cu_seqlens = a.cu_seqlens;
    p.seq_chunk = reinterpret_cast<const int32_t *>(a.ws + L.seq_chunk);
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.H = a.H;
    p.dv = a.dv;
    p.n_slices = n_slices;
    p.phases = segs;
    p.o = (__nv_bfloat16 *)a.o;
    p.ctl = (int32_t *)(a.ws + L.ctl);
    p.additive = a.rule == GDR_RULE_ADDITIVE;
    p.prologue = a.prologue;
    p.S_P = S_P;
    p.S_R = S_R;
    p.S_start = S_start;
    p.S_discard = S_discard;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    // the summaries (P_f, R_f) of every segment but the last, without output
    p.mode = 1;
    cfg.gridDim = dim3((unsigned)((segs - 1) * NH * (n_slices + 1)));
    if (cudaLaunchKernelEx(&cfg, tc_chain_kernel<true>, mq, mk, mv, mt, mo, p) != cudaSuccess)
        return GDR_ERR_CUDA;
    // the segments' start states
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = dim3((unsigned)NH, (unsigned)(a.dv / kScanCols));
    scfg.blockDim = dim3(kScanThreads);
    scfg.dynamicSmemBytes = SCAN_SMEM_BYTES;
    scfg.stream = a.stream;
    scfg.attrs = &attr;
    scfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&scfg, seg_scan_kernel, (const float *)a.S0, (const float *)S_P,
                           (const float *)S_R, S_start, (int)NH, a.dv, segs - 1) != cudaSuccess)
        return GDR_ERR_CUDA;
    // every segment from its start state, with output
    p.mode = 2;
    p.S_out = a.S_final;
    if (a.dv == NV) {  // the output step fused into the chain's epilogue
        p.out_gate = (const __nv_bfloat16 *)a.out_gate;
        p.out_norm_weight = a.out_norm_weight;
        p.out_norm_eps = a.out_norm_eps;
    }
    cfg.gridDim = dim3((unsigned)(segs * NH * n_slices));
    if (cudaLaunchKernelEx(&cfg, tc_chain_kernel<true>, mq, mk, mv, mt, mo, p) != cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}

int launch_prefill_tc(const PrefillArgs &a, const WsLayout &L, int phases) {
    using namespace chain;
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
    // Packed sequences on the fused schedule: the fused launch, then the two-kernel pair
    // of one phase; the plan has chosen on the device which of the two does the work.
    const bool only_pair = phases == 0 && a.cu_seqlens;
    if (phases == 0) {
        const int st = launch_fused(a, L, mq, mk, mv, mt, mo);
        if (st != GDR_OK || !only_pair) return st;
        phases = 1;
    }
    if (phases > kSegmentedBase)
        return launch_segmented(a, L, phases - kSegmentedBase, mq, mk, mv, mt, mo);
    if (cudaFuncSetAttribute(tc_chain_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    int st = tc::launch_solve_tc(a, L, mq, mk, 0, 0, a.stream, true, only_pair);
    if (st != GDR_OK) return st;
    if (phases > 1) {  // solves of phases 1 .. P-1 on the side stream, after the solve of
                       // phase 0 (which has had every SM) and beside the chains
        cudaError_t e = cudaEventRecord(sd->ev[0], a.stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sd->stream, sd->ev[0], 0);
        if (e != cudaSuccess) return GDR_ERR_CUDA;
        for (int f = 1; f < phases; ++f) {
            st = tc::launch_solve_tc(a, L, mq, mk, f, free_sms, sd->stream, false);
            if (st != GDR_OK) return st;
            if (cudaEventRecord(sd->ev[f], sd->stream) != cudaSuccess) return GDR_ERR_CUDA;
        }
    }
    TcParams p = {};
    chain_wait_policy(p);
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
    p.additive = a.rule == GDR_RULE_ADDITIVE;
    p.prologue = a.prologue;
    p.only_pair = only_pair;
    if (a.dv == NV) {  // the output step fused into the chain's epilogue
        p.out_gate = (const __nv_bfloat16 *)a.out_gate;
        p.out_norm_weight = a.out_norm_weight;
        p.out_norm_eps = a.out_norm_eps;
    }
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
        if (cudaLaunchKernelEx(&cfg, tc_chain_kernel<false>, mq, mk, mv, mt, mo, p) != cudaSuccess)
            return GDR_ERR_CUDA;
    }
    return GDR_OK;
}

}  // namespace gdr
