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
// address of the current device's copy is looked up with cudaGetSymbolAddress
// on every call (a lookup, no allocation) and passed to the kernels as their
// workspace. Looking it up each time, rather than caching it per device
// ordinal, keeps a stale address from ever reaching a kernel after the device
// has been reset and the module reloaded elsewhere. The first call on a device
// also loads the library's module there, which is why that first call should
// come before any stream capture. Nothing here calls cudaMalloc, cudaFree or
// any allocating routine.
//
// Every call shares the one array and it keeps the previous call's contents.
// The kernels write every word of scratch they later read during the same
// call (the status word, the chunk plan and the per-chunk intermediates), so
// nothing has to be cleared between calls. Calls that overlap on the GPU (on
// different streams without ordering, or from several threads) race on the
// array and give wrong results; order them on one stream.
//
// The device-side checks of a call (a rejected cu_seqlens, a bounded wait that
// gave up) leave their status in the first word of the array, as they do in a
// caller's workspace; gdr_noalloc_read_device_status reads it back.
#include "internal.h"

static __device__ __align__(256) unsigned char g_gdr_noalloc_scratch[GDR_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.
static int noalloc_scratch(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gdr_noalloc_scratch) != cudaSuccess || !p) return GDR_ERR_CUDA;
    *out = p;
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

extern "C" int gdr_noalloc_read_device_status(int *status, gdr_stream_t stream) {
    if (!status) return GDR_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != GDR_OK) return st;
    int32_t word = 0;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    *status = word;
    return GDR_OK;
}
