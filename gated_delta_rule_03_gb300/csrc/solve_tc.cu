// solve_tc.cu -- the standalone chunk-parallel solve kernel and its launcher (the
// solve itself is in solve_tc.cuh, shared with the fused launch in prefill_tc.cu).
#include "solve_tc.cuh"

namespace gdr {
namespace solve {
namespace {

__global__ void __launch_bounds__(kThreads, 1)
tc_solve_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const SolveParams p) {
    // The plan's choice between the fused kernel and this pair: the plan completed before
    // the fused kernel ahead of this launch began, so the word is read at once. A launch
    // left out lets the next one start, and ends only after the kernel ahead of it.
    if (p.only_pair && p.ctl[kPairWord] != 1) {
        griddep_launch_dependents();
        griddep_wait();
        return;
    }
    solve_body<false>(map_q, map_k, p, (int)blockIdx.x, (int)gridDim.x);
}

}  // namespace
}  // namespace solve

namespace tc {

int launch_solve_tc(const PrefillArgs &a, const WsLayout &L, const CUtensorMap &map_q,
                    const CUtensorMap &map_k, int phase, int max_ctas,
                    cudaStream_t stream, bool programmatic, bool only_pair) {
    using namespace solve;
    SolveParams p = {};
    p.log_alpha = a.log_alpha;
    p.beta = a.beta;
    p.plan = reinterpret_cast<const int4 *>(a.ws + L.plan);
    p.ctl = reinterpret_cast<int32_t *>(a.ws + L.ctl);
    p.H = a.H;
    p.Tout = reinterpret_cast<__nv_bfloat16 *>(a.ws + L.T);
    p.Gout = reinterpret_cast<float *>(a.ws + L.G);
    p.phase = phase;
    p.additive = a.rule == GDR_RULE_ADDITIVE;
    p.prologue = a.prologue;
    p.gate_A = a.gate_A;
    p.only_pair = only_pair;
    if (cudaFuncSetAttribute(tc_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
        return GDR_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GDR_ERR_CUDA;
    // upper bound on the CTAs that find work (the kernel reads the unit count)
    const int64_t busy = (L.max_chunks * a.H + kGroups - 1) / kGroups;
    int64_t grid = busy < (int64_t)sms ? busy : (int64_t)sms;  // at most one CTA per SM
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cuda_status(cudaLaunchKernelEx(&cfg, tc_solve_kernel, map_q, map_k, p));
}

}  // namespace tc
}  // namespace gdr
