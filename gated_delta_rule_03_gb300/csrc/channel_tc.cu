// channel_tc.cu -- the tensor-core prefill with one forget rate per key channel: the
// per-channel chunk kernel (channel_tc.cuh), the chain in its per-channel mode
// (chain_tc.cuh), and their host launcher.
#include <cstdlib>

#include "chain_tc.cuh"
#include "channel_tc.cuh"

namespace gdr {
namespace chain {
namespace {

__global__ void __launch_bounds__(kThreads, 1)
tc_chain_channel_kernel(const __grid_constant__ CUtensorMap map_qw, const __grid_constant__ CUtensorMap map_kt,
                        const __grid_constant__ CUtensorMap map_ut, const __grid_constant__ CUtensorMap map_t,
                        const __grid_constant__ CUtensorMap map_o, const TcParams p) {
    chain_body<false, false, true>(map_qw, map_kt, map_ut, map_t, map_o, p, (int)blockIdx.x);
}

}  // namespace
}  // namespace chain

// The operands kernel's wait bound, and a test of its give-up path: with
// GDR_DEBUG_PREP_FAULT=<chunk> in the environment, head 0's CTA of that chunk skips its key
// and query loads and every wait gives up after 2e7 SM cycles (about 10 ms) instead of
// 2e9. That CTA then marks the call GDR_ERR_DEVICE_TIMEOUT in the status word and drains;
// the chain kernel, seeing the status, writes nothing. Nothing faults or hangs.
static void channel_wait_policy(channel::ChannelParams &p) {
    p.wait_cycles = sm100::kWaitCycles;
    p.fault_chunk = -1;
    if (const char *env = getenv("GDR_DEBUG_PREP_FAULT")) {
        char *end = nullptr;
        const long c = strtol(env, &end, 10);
        if (end != env && *end == '\0' && c >= 0 && c < (1l << 30)) {
            p.fault_chunk = (int)c;
            p.wait_cycles = 20000000;
        }
    }
}

int launch_prefill_channel_tc(const PrefillArgs &a, const WsLayout &L) {
    using namespace chain;
    const size_t s_bytes = (size_t)a.num_seqs * a.H * a.dk * a.dv * sizeof(float);
    if (a.total_tokens == 0) {  // nothing to compute: S_final = S0 (or zero)
        cudaError_t e = cudaSuccess;
        if (!a.S0) e = cudaMemsetAsync(a.S_final, 0, s_bytes, a.stream);
        else if (a.S0 != a.S_final)
            e = cudaMemcpyAsync(a.S_final, a.S0, s_bytes, cudaMemcpyDeviceToDevice, a.stream);
        return cuda_status(e);
    }
    if (a.dk != channel::DK || a.dv != channel::DV) return GDR_ERR_UNSUPPORTED;
    const int64_t units = L.max_chunks * a.H;
    CUtensorMap mq, mk, mv, mla, mo, mqw, mkt, mut, mt;
    if (!tc::make_map_thd(&mq, a.q, a.dk, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mk, a.k, a.dk, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mv, a.v, a.dv, a.H, a.total_tokens) ||

        !tc::make_map_thd(&mo, a.o, a.dv, a.H, a.total_tokens) ||
        !tc::make_map_thd(&mqw, a.ws + L.QW, 256, 1, units * kChunk) ||
        !tc::make_map_thd(&mkt, a.ws + L.KT, 128, 1, units * kChunk) ||
        !tc::make_map_thd(&mut, a.ws + L.UT, kChunk, 1, units * 128) ||
        !tc::make_map_units(&mt, a.ws + L.T, 2 * units))
        return GDR_ERR_CUDA;
    // log_alpha need only be 4-byte aligned: 16-byte loads of it, and its tensor map for
    // the L2 prefetch, where its base is 16-byte aligned
    const bool rates_vec = ((uintptr_t)a.log_alpha & 15u) == 0;
    const bool rates_map = rates_vec &&
                           tc::make_map_rows_f32(&mla, a.log_alpha, a.dk, a.H, a.total_tokens);
    if (!rates_map) mla = mq;  // (not read)
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;

    // every unit's operands, a programmatic dependent of the planning kernel
    // the plain kernel or the one with the layer prologue folded in
    auto prep = a.prologue ? channel::channel_prep_kernel<true> : channel::channel_prep_kernel<false>;
    if (cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)channel::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return GDR_ERR_CUDA;
    channel::ChannelParams cp = {};
    cp.log_alpha = a.log_alpha;
    cp.beta = a.beta;
    cp.plan = reinterpret_cast<const int4 *>(a.ws + L.plan);
    cp.ctl = reinterpret_cast<int32_t *>(a.ws + L.ctl);
    cp.H = a.H;
    cp.additive = a.rule == GDR_RULE_ADDITIVE;
    cp.gate_A = a.gate_A;
    cp.QW = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.QW);
    cp.KT = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.KT);
    cp.UT = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.UT);
    cp.AT = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.T);
    cp.G = reinterpret_cast<float *>(a.ws + L.G);
    cp.rates_vec = rates_vec;
    cp.prefetch_rates = rates_map;
    channel_wait_policy(cp);
    // persistent CTAs, as many as are resident at once
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GDR_ERR_CUDA;
    const int64_t resident = (int64_t)channel::kCtasPerSm * sms;
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3((unsigned)(units < resident ? units : resident));
    pcfg.blockDim = dim3(channel::kThreads);
    pcfg.dynamicSmemBytes = channel::SMEM_BYTES;
    pcfg.stream = a.stream;
    pcfg.attrs = &attr;
    pcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&pcfg, prep, mq, mk, mv, mla, cp) != cudaSuccess)
        return GDR_ERR_CUDA;

    // the chains, one CTA per (sequence, head), a programmatic dependent of the above
    if (cudaFuncSetAttribute(tc_chain_channel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    TcParams p = {};
    chain_wait_policy(p);
    p.S_in = a.S0;
    p.factors = reinterpret_cast<const float *>(a.ws + L.G);
    p.cu_seqlens = a.cu_seqlens;
    p.seq_chunk = reinterpret_cast<const int32_t *>(a.ws + L.seq_chunk);
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.H = a.H;
    p.dv = a.dv;
    p.n_slices = 1;
    p.phase = 0;
    p.phases = 1;
    p.o = (__nv_bfloat16 *)a.o;
    p.S_out = a.S_final;
    p.ctl = reinterpret_cast<int32_t *>(a.ws + L.ctl);
    p.additive = a.rule == GDR_RULE_ADDITIVE;
    p.prologue = 0;
    p.out_gate = (const __nv_bfloat16 *)a.out_gate;
    p.out_norm_weight = a.out_norm_weight;
    p.out_norm_eps = a.out_norm_eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.num_seqs * a.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, tc_chain_channel_kernel, mqw, mkt, mut, mt, mo, p));
}

}  // namespace gdr
