// pack.cu -- head vectors between their stored width and a padded width.
//
// The bf16 attention kernel reads 128-byte operand rows by TMA, which needs
// each head vector to start on a 16-byte boundary: 64 bf16 elements per head.
// For other head sizes (d_head 41 in the base-LM shape: 82-byte slices) the
// library copies q, k, v, the table and the biases once into 64-wide,
// zero-padded scratch vectors, runs the TMA kernel on them and copies the
// output's first d_head columns back.  HBM-bound elementwise passes, one
// thread per 16-byte chunk of the padded side.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace txl {
namespace {

constexpr int NT = 256;

constexpr int DPW = 64;     // the padded width (elements)

// dst[v][e] = e < d ? src[v][e] : 0, for v < nvec, e < 64.  One thread per
// 16-byte chunk of the output: the chunks of consecutive threads are
// consecutive in both buffers.
template <typename T>
__global__ void __launch_bounds__(NT)
pad_kernel(T *__restrict__ dst, const T *__restrict__ src, long nvec, int d)
{
    constexpr int E = 16 / sizeof(T);          // elements per chunk
    constexpr int CPV = DPW / E;               // chunks per padded vector
    const long n = nvec * CPV;
    for (long x = (long)blockIdx.x * NT + threadIdx.x; x < n; x += (long)gridDim.x * NT) {
        const long v = x / CPV;
        const int e0 = (int)(x % CPV) * E;
        T vals[E];
#pragma unroll
        for (int i = 0; i < E; ++i) vals[i] = e0 + i < d ? src[v * d + e0 + i] : T(0);
        reinterpret_cast<uint4 *>(dst)[x] = *reinterpret_cast<const uint4 *>(vals);
    }
}

// dst[v][e] = src[v][e] for e < d (src rows 64 wide), one 16-byte source chunk per thread
template <typename T>
__global__ void __launch_bounds__(NT)
unpad_kernel(T *__restrict__ dst, const T *__restrict__ src, long nvec, int d)
{
    constexpr int E = 16 / sizeof(T);
    constexpr int CPV = DPW / E;
    const long n = nvec * CPV;
    for (long x = (long)blockIdx.x * NT + threadIdx.x; x < n; x += (long)gridDim.x * NT) {
        const long v = x / CPV;
        const int e0 = (int)(x % CPV) * E;
        if (e0 >= d) continue;
        const uint4 raw = reinterpret_cast<const uint4 *>(src)[x];
        const T *vals = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int i = 0; i < E; ++i)
            if (e0 + i < d) dst[v * d + e0 + i] = vals[i];
    }
}

unsigned grid_for(long n)
{
    const long cap = (long)device_sm_count() * 8;
    const long want = (n + NT - 1) / NT;
    return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_pad_heads(void *dst, const void *src, long nvec, int d, int dp, int elem_size,
                             cudaStream_t s)
{
    if (nvec <= 0) return cudaSuccess;
    if (dp != DPW || d > DPW || ((uintptr_t)dst & 15)) return cudaErrorInvalidValue;
    if (elem_size == 4)
        pad_kernel<uint32_t><<<grid_for(nvec * (DPW / 4)), NT, 0, s>>>((uint32_t *)dst, (const uint32_t *)src, nvec, d);
    else
        pad_kernel<uint16_t><<<grid_for(nvec * (DPW / 8)), NT, 0, s>>>((uint16_t *)dst, (const uint16_t *)src, nvec, d);
    return cudaGetLastError();
}

cudaError_t launch_unpad_heads(void *dst, const void *src, long nvec, int d, int dp, int elem_size,
                               cudaStream_t s)
{
    if (nvec <= 0) return cudaSuccess;
    if (dp != DPW || d > DPW || ((uintptr_t)src & 15)) return cudaErrorInvalidValue;
    if (elem_size == 4)
        unpad_kernel<uint32_t><<<grid_for(nvec * (DPW / 4)), NT, 0, s>>>((uint32_t *)dst, (const uint32_t *)src, nvec, d);
    else
        unpad_kernel<uint16_t><<<grid_for(nvec * (DPW / 8)), NT, 0, s>>>((uint16_t *)dst, (const uint16_t *)src, nvec, d);
    return cudaGetLastError();
}

}  // namespace txl
