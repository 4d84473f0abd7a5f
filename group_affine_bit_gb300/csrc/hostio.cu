// hostio.cu -- the host-buffer entry point's transfers as kernels.
//
// affqmm_run_host moves x from host memory to its device staging buffer and y
// back.  When the caller's host buffers are page-locked they are addressable
// from the GPU, and the two transfers run as small kernels chained to the
// projection by programmatic dependent launch instead of as copy-engine
// copies, which sit between kernels and keep each launch from overlapping the
// one before it:
//   * host_upload_kernel reads x from host memory at once (it depends on
//     nothing), then waits for the previous kernel in the stream (which may
//     still read the staging buffer) and stores x; the projection that follows
//     starts its weight copies meanwhile;
//   * host_download_kernel waits for the projection and writes y to host
//     memory.
// Both move 16-byte pieces when both addresses and the size allow it, else
// 2-byte values (the buffers hold bf16).
#include <cuda_runtime.h>

#include <cstdint>

#include "affqmm_internal.h"
#include "affqmm_tc.cuh"

namespace affqmm {
namespace {

constexpr int H_THREADS = 256;
constexpr int H_PER_THREAD = 4;  // pieces a thread holds between its loads and its stores

template <typename T>
__device__ __forceinline__ void move_pieces(const T* __restrict__ src, T* __restrict__ dst, size_t n, bool wait_first) {
    const size_t base = ((size_t)blockIdx.x * H_THREADS) * H_PER_THREAD + threadIdx.x;
    if (wait_first) pdl_wait();
    T v[H_PER_THREAD];
#pragma unroll
    for (int j = 0; j < H_PER_THREAD; ++j) {
        const size_t i = base + (size_t)j * H_THREADS;
        if (i < n) v[j] = src[i];
    }
    if (!wait_first) pdl_wait();
#pragma unroll
    for (int j = 0; j < H_PER_THREAD; ++j) {
        const size_t i = base + (size_t)j * H_THREADS;
        if (i < n) dst[i] = v[j];
    }
}

// x: host -> device staging buffer.  The loads come before the wait: they
// read only the caller's host buffer.
__global__ void __launch_bounds__(H_THREADS) host_upload_kernel(const void* src, void* dst, size_t bytes, int wide) {
    pdl_launch_dependents();
    if (wide)
        move_pieces(static_cast<const uint4*>(src), static_cast<uint4*>(dst), bytes / 16, false);
    else
        move_pieces(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), bytes / 2, false);
}

// y: device -> host, after the projection has written it.
__global__ void __launch_bounds__(H_THREADS) host_download_kernel(const void* src, void* dst, size_t bytes, int wide) {
    pdl_launch_dependents();
    if (wide)
        move_pieces(static_cast<const uint4*>(src), static_cast<uint4*>(dst), bytes / 16, true);
    else
        move_pieces(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), bytes / 2, true);
}

cudaError_t launch_move(bool upload, const void* src, void* dst, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return cudaSuccess;
    const bool wide = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15u) == 0;
    const size_t pieces = wide ? bytes / 16 : bytes / 2;
    const size_t per_block = (size_t)H_THREADS * H_PER_THREAD;
    const dim3 grid((unsigned)((pieces + per_block - 1) / per_block));
    if (upload) return launch_pdl(host_upload_kernel, grid, H_THREADS, 0, st, src, dst, bytes, wide ? 1 : 0);
    return launch_pdl(host_download_kernel, grid, H_THREADS, 0, st, src, dst, bytes, wide ? 1 : 0);
}

}  // namespace

cudaError_t launch_host_upload(const void* host_src, void* dev_dst, size_t bytes, cudaStream_t st) {
    return launch_move(true, host_src, dev_dst, bytes, st);
}

cudaError_t launch_host_download(const void* dev_src, void* host_dst, size_t bytes, cudaStream_t st) {
    return launch_move(false, dev_src, host_dst, bytes, st);
}

}  // namespace affqmm
