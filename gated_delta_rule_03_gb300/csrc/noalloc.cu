// noalloc.cu -- gdr_chunk_fwd_noalloc: chunked prefill for callers that cannot allocate.
//
// gdr_chunk_fwd needs a caller-provided device workspace. Some callers have no
// way to provide one: a plugin loaded into a host runtime that owns the device
// allocator and gives its plugins no allocation hook, or a serving loop whose
// memory policy forbids any device allocation once it has started. This entry
// point serves them with a scratch area that is part of the library itself: a
// file-scope __device__ array of GDR_NOALLOC_SCRATCH_BYTES, reserved on every
// GPU that loads the library and held until the process exits.
//
// The array's name is only a host-side stand-in in host code; the device
// address of the current device's copy is fetched once per device with
// cudaGetSymbolAddress (the first call on a device does this set-up, which is
// why that first call should come before any stream capture) and is then
// passed to the kernels as their workspace. Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
//
// Every call shares the one array and it keeps the previous call's contents.
// The kernels write every word of scratch they later read during the same
// call (the status word, the chunk plan and the per-chunk intermediates), so
// nothing has to be cleared between calls. Calls that overlap on the GPU (on
// different streams without ordering, or from several threads) race on the
// array and give wrong results; order them on one stream.
#include <mutex>

#include "internal.h"

static __device__ __align__(256) unsigned char g_gdr_noalloc_scratch[GDR_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];  // device address of the array, per device ordinal
}  // namespace

// Device address of the scratch array on the current device (set-up on first use).
static int noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gdr_noalloc_scratch) != cudaSuccess || !p)
            return GDR_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDR_OK;
}

extern "C" int gdr_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                     const float *log_alpha, const float *beta, const float *S0,
                                     const int32_t *cu_seqlens, int64_t num_seqs,
                                     int64_t total_tokens, int H, int d_k, int d_v, int chunk,
                                     int dtype, void *o, float *S_final, gdr_stream_t stream) {
    const size_t need =
        gdr_chunk_fwd_workspace_size(num_seqs, total_tokens, H, d_k, d_v, chunk, dtype);
    if (need > (size_t)GDR_NOALLOC_SCRATCH_BYTES) return GDR_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != GDR_OK) return st;
    // need == 0 means unsupported sizes: gdr_chunk_fwd returns the matching status.
    return gdr_chunk_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k,
                         d_v, chunk, dtype, o, S_final, scratch, GDR_NOALLOC_SCRATCH_BYTES,
                         stream);
}
