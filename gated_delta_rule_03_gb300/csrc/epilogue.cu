// epilogue.cu -- the layer's output step on o, for the prefill paths that do not fuse it
// into their own epilogue (the exact path, and the tensor-core path when d_v spans two
// chain CTAs).
//
// Per token and head, over the head's d_v value entries ("Linear attention"
// (arsalanzafar.ai), "A naive PyTorch implementation": the output normalised over the
// head dimension, times SiLU of the input-dependent output gate):
//   o_j <- o_j / sqrt(mean_j' o_j'^2 + eps) * w_j * z_j * sigmoid(z_j)
// One warp per (token, head) row, in place, fp32 arithmetic.
#include "internal.h"

namespace gdr {
namespace {

template <typename T, int PER>  // PER = d_v / 32 entries per lane
__global__ void __launch_bounds__(256)
out_norm_gate_kernel(T *__restrict__ o, const T *__restrict__ z, const float *__restrict__ w,
                     float eps, int64_t rows) {
    constexpr int DV = 32 * PER;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;  // whole warps leave together
    T *orow = o + row * DV;
    const T *zrow = z + row * DV;
    float x[PER];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        x[e] = to_f32(orow[lane + 32 * e]);
        ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = rsqrtf(ss * (1.f / DV) + eps);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int j = lane + 32 * e;
        const float g = to_f32(zrow[j]);
        const float wj = w ? w[j] : 1.f;
        orow[j] = from_f32<T>(x[e] * r * wj * (g / (1.f + __expf(-g))));
    }
}

template <typename T>
int launch_t(void *o, const void *z, const float *w, float eps, int64_t rows, int dv,
             cudaStream_t stream) {
    const unsigned grid = (unsigned)((rows + 7) / 8);
#define GDR_OUT_CASE(P)                                                                    \
    if (dv == 32 * P) {                                                                    \
        out_norm_gate_kernel<T, P><<<grid, 256, 0, stream>>>((T *)o, (const T *)z, w, eps, rows); \
        return cuda_status(cudaGetLastError());                                            \
    }
    GDR_OUT_CASE(1) GDR_OUT_CASE(2) GDR_OUT_CASE(3) GDR_OUT_CASE(4)
    GDR_OUT_CASE(5) GDR_OUT_CASE(6) GDR_OUT_CASE(7) GDR_OUT_CASE(8)
#undef GDR_OUT_CASE
    return GDR_ERR_UNSUPPORTED;
}

}  // namespace

int launch_out_norm_gate(void *o, const void *z, const float *w, float eps, int64_t rows, int dv,
                         int dtype, cudaStream_t stream) {
    if (rows == 0) return GDR_OK;
    if (dtype == GDR_BF16) return launch_t<__nv_bfloat16>(o, z, w, eps, rows, dv, stream);
    return launch_t<float>(o, z, w, eps, rows, dv, stream);
}

}  // namespace gdr
