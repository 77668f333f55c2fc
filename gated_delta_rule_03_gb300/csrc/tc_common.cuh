// tc_common.cuh -- pieces shared by the two tensor-core prefill kernels (the
// chunk-parallel solve in solve_tc.cu and the sequential chain in prefill_tc.cu).
//
// Both kernels derive the per-chunk decay factors from the same warp scan of the
// same log-decay values, so every decision taken on them (the ratio or the
// exponential form, below) comes out identical in the two kernels.
#pragma once

#include <cuda.h>

#include "internal.h"
#include "sm100.cuh"

namespace gdr {
namespace tc {

// Gamma_ti = gamma_t / gamma_i is exact only while no gamma underflows: the chunk's
// cumulative log-decay g_C (its minimum, since log alpha <= 0) stays above this bound.
// Such chunks use the ratio form; the others take each Gamma_ti as exp(g_t - g_i).
constexpr float kRatioSafeLogDecay = -80.f;

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// exp(x) through the hardware base-2 exponential (flushes subnormal results to zero).
__device__ __forceinline__ float fast_exp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Writes 32 fp32 values as bf16 into columns [32*half, 32*half + 32) of row `row` of a
// 128-byte-swizzled block of 64-wide bf16 rows (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B: the 16-byte chunk j of row r sits at chunk j ^ (r % 8)).
__device__ __forceinline__ void store_row32_sw128(unsigned char *block, int row, int half,
                                                  const float (&v)[32]) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const int chunk = 4 * half + jj;
        uint4 w;
        w.x = pack_bf16x2(v[8 * jj + 0], v[8 * jj + 1]);
        w.y = pack_bf16x2(v[8 * jj + 2], v[8 * jj + 3]);
        w.z = pack_bf16x2(v[8 * jj + 4], v[8 * jj + 5]);
        w.w = pack_bf16x2(v[8 * jj + 6], v[8 * jj + 7]);
        *reinterpret_cast<uint4 *>(block + row * 128 + (((chunk ^ row) & 7) << 4)) = w;
    }
}

// Cumulative log-decay of one chunk by one warp: lane l holds the log-decays a0, a1 of
// tokens 2l and 2l + 1 (zero past the end of the sequence) and gets back g_{2l},
// g_{2l+1} and the chunk's total g_C.
struct ChunkScan {
    float g0, g1, g_last;
};

__device__ __forceinline__ ChunkScan chunk_scan(float a0, float a1, int lane) {
    float sum = a0 + a1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, sum, off);
        if (lane >= off) sum += up;
    }
    ChunkScan r;
    r.g0 = sum - a1;
    r.g1 = sum;
    r.g_last = __shfl_sync(0xffffffffu, sum, 31);
    return r;
}

// ---------------------------------------------------------------- host side

// Tensor map over a packed [T, H, d] bf16 tensor with 64 (features) x 1 (head) x 64
// (tokens) boxes, 128-byte swizzle.
bool make_map_thd(CUtensorMap *map, const void *base, int d, int H, int64_t T);
// Tensor map over [units][64][64] bf16 matrices, one whole matrix per box, 128-byte swizzle.
bool make_map_units(CUtensorMap *map, const void *base, int64_t units);
// Tensor map over a packed [T, H, d] fp32 tensor with d (features) x 1 (head) x 64 (tokens)
// boxes, no swizzle (d * 4 a multiple of 16, d at most 256).
bool make_map_rows_f32(CUtensorMap *map, const float *base, int d, int H, int64_t T);

// The chunk-parallel solve: T' and A^T for every (chunk, head) of one phase into the
// workspace, on `stream`, with at most max_ctas CTAs (all SMs when max_ctas <= 0);
// `programmatic` launches it as a programmatic dependent of the kernel ahead of it;
// `only_pair`: it solves nothing unless the plan handed the call to the two-kernel pair.
int launch_solve_tc(const PrefillArgs &a, const WsLayout &L, const CUtensorMap &map_q,
                    const CUtensorMap &map_k, int phase, int max_ctas,
                    cudaStream_t stream, bool programmatic, bool only_pair = false);

}  // namespace tc
}  // namespace gdr
