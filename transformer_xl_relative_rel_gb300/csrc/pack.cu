// pack.cu -- head vectors between their stored width and a padded width.
//
// The bf16 attention kernel reads 128-byte operand rows by TMA, which needs
// each head vector to start on a 16-byte boundary: 64 bf16 elements per head.
// For other head sizes (d_head 41 in the base-LM shape: 82-byte slices) the
// library copies q, k, v, the table and the biases once into 64-wide,
// zero-padded scratch vectors, runs the TMA kernel on them and copies the
// output's first d_head columns back.  HBM-bound elementwise passes: the six
// padding copies of a call in one launch (one thread per 16-byte chunk of the
// padded side), the copy back one thread per 16-byte chunk of the flat
// output (its elements gathered across row ends).
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

// Several pad jobs in one launch (q, k, v, the table and the two biases of
// a call): the jobs' 16-byte output chunks are numbered one after another and
// a thread finds its job from the running starts.
struct PadJobs {
    PadJob job[kMaxPadJobs];
    long start[kMaxPadJobs + 1];     // first chunk of each job; start[n] = total
    int n;
};

__global__ void __launch_bounds__(NT)
pad_many_kernel(const PadJobs jobs)
{
    const long total = jobs.start[jobs.n];
    for (long x = (long)blockIdx.x * NT + threadIdx.x; x < total; x += (long)gridDim.x * NT) {
        int j = 0;
        while (x >= jobs.start[j + 1]) ++j;
        const PadJob &jb = jobs.job[j];
        const long c = x - jobs.start[j];
        uint4 out;
        if (jb.elem_size == 4) {
            const long v = c / (DPW / 4);
            const int e0 = (int)(c % (DPW / 4)) * 4;
            const uint32_t *src = (const uint32_t *)jb.src + v * jb.d;
            uint32_t *o = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = e0 + i < jb.d ? src[e0 + i] : 0u;
        } else {
            const long v = c / (DPW / 8);
            const int e0 = (int)(c % (DPW / 8)) * 8;
            const uint16_t *src = (const uint16_t *)jb.src + v * jb.d;
            uint16_t *o = reinterpret_cast<uint16_t *>(&out);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = e0 + i < jb.d ? src[e0 + i] : (uint16_t)0;
        }
        reinterpret_cast<uint4 *>(jb.dst)[c] = out;
    }
}

// dst (flat, nvec*d bf16 elements) from the 64-wide src rows, one 16-byte
// chunk of the output per thread: its 8 elements gathered across the row
// boundaries they straddle (so every store is a full 16 bytes); the last
// nvec*d % 8 elements element by element.
__global__ void __launch_bounds__(NT)
unpad_flat_kernel(uint16_t *__restrict__ dst, const uint16_t *__restrict__ src, long nvec, int d)
{
    const long n = nvec * d, nch = n / 8;
    for (long x = (long)blockIdx.x * NT + threadIdx.x; x < nch; x += (long)gridDim.x * NT) {
        const long f0 = 8 * x;
        long v = f0 / d;
        int e = (int)(f0 - v * d);
        uint4 out;
        uint16_t *o = reinterpret_cast<uint16_t *>(&out);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i] = src[v * DPW + e];
            if (++e == d) {
                e = 0;
                ++v;
            }
        }
        reinterpret_cast<uint4 *>(dst)[x] = out;
    }
    if (blockIdx.x == 0 && (long)threadIdx.x < n - 8 * nch) {
        const long f = 8 * nch + threadIdx.x, v = f / d;
        dst[f] = src[v * DPW + (f - v * d)];
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

cudaError_t launch_pad_heads_many(const PadJob *jobs, int n, cudaStream_t s)
{
    if (n < 1 || n > kMaxPadJobs) return cudaErrorInvalidValue;
    PadJobs pj;
    pj.n = n;
    pj.start[0] = 0;
    for (int j = 0; j < n; ++j) {
        const PadJob &jb = jobs[j];
        if (jb.d > DPW || ((uintptr_t)jb.dst & 15) || (jb.elem_size != 2 && jb.elem_size != 4) || jb.nvec < 0)
            return cudaErrorInvalidValue;
        pj.job[j] = jb;
        pj.start[j + 1] = pj.start[j] + jb.nvec * (DPW * jb.elem_size / 16);
    }
    if (pj.start[n] == 0) return cudaSuccess;
    pad_many_kernel<<<grid_for(pj.start[n]), NT, 0, s>>>(pj);
    return cudaGetLastError();
}

cudaError_t launch_unpad_heads(void *dst, const void *src, long nvec, int d, int dp, int elem_size,
                               cudaStream_t s)
{
    if (nvec <= 0) return cudaSuccess;
    if (dp != DPW || d > DPW || ((uintptr_t)src & 15)) return cudaErrorInvalidValue;
    if (elem_size == 2 && ((uintptr_t)dst & 15) == 0) {
        unpad_flat_kernel<<<grid_for(nvec * d / 8 + 1), NT, 0, s>>>((uint16_t *)dst, (const uint16_t *)src, nvec, d);
        return cudaGetLastError();
    }
    if (elem_size == 4)
        unpad_kernel<uint32_t><<<grid_for(nvec * (DPW / 4)), NT, 0, s>>>((uint32_t *)dst, (const uint32_t *)src, nvec, d);
    else
        unpad_kernel<uint16_t><<<grid_for(nvec * (DPW / 8)), NT, 0, s>>>((uint16_t *)dst, (const uint16_t *)src, nvec, d);
    return cudaGetLastError();
}

}  // namespace txl
