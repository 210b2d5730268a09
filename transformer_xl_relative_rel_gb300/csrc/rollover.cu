// rollover.cu -- the per-layer memory rollover (Transformer-XL, Section 3.2).
//
// The next segment's memory is the newest M rows of [memory; current hidden
// states].  In the T-major layout [T][B][d_model] those rows (L..T-1) are one
// contiguous run of M*B*d_model elements, so the rollover is one flat copy.
// HBM-bound: each byte is read once and written once.  The copy moves 16-byte
// vectors with four independent loads in flight per thread; a grid of a few
// CTAs per SM strides over the buffer.  Misaligned heads/tails (possible when
// L*B*d_model is not a multiple of 8 bf16 elements) go through an element
// loop in the same launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace txl {
namespace {

constexpr int NT = 256;

// dst/src point at 16-byte aligned storage of n16 vectors; then `tail` bytes
// (< 16) follow, copied element-wise in units of `esz` bytes.
__global__ void __launch_bounds__(NT)
rollover_vec_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n16,
                    unsigned char *__restrict__ dst_tail, const unsigned char *__restrict__ src_tail,
                    int tail_bytes)
{
    const size_t stride = (size_t)gridDim.x * NT;
    size_t i = (size_t)blockIdx.x * NT + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i];
        const uint4 b = src[i + stride];
        const uint4 c = src[i + 2 * stride];
        const uint4 d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
    if (blockIdx.x == 0 && (int)threadIdx.x < tail_bytes) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

// fallback when the two pointers are not co-aligned to 16 bytes: element copy
template <typename E>
__global__ void __launch_bounds__(NT)
rollover_elem_kernel(E *__restrict__ dst, const E *__restrict__ src, size_t n)
{
    const size_t stride = (size_t)gridDim.x * NT;
    for (size_t i = (size_t)blockIdx.x * NT + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

int grid_for(size_t work_items)
{
    const int sms = device_sm_count();
    const size_t per_thread = 4;
    size_t blocks = (work_items + (size_t)NT * per_thread - 1) / ((size_t)NT * per_thread);
    const size_t cap = (size_t)sms * 8;     // 8 CTAs of 256 threads fill an SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

}  // namespace

cudaError_t launch_rollover(void *dst, const void *src, size_t bytes, int elem_size, cudaStream_t s)
{
    if (bytes == 0) return cudaSuccess;
    const uintptr_t d = (uintptr_t)dst, c = (uintptr_t)src;
    if ((d & 15) == 0 && (c & 15) == 0) {
        const size_t n16 = bytes / 16;
        const int tail = (int)(bytes % 16);
        rollover_vec_kernel<<<grid_for(n16 ? n16 : 1), NT, 0, s>>>(
            (uint4 *)dst, (const uint4 *)src, n16, (unsigned char *)dst + n16 * 16,
            (const unsigned char *)src + n16 * 16, tail);
    } else if (elem_size == 4 && (d & 3) == 0 && (c & 3) == 0) {
        rollover_elem_kernel<uint32_t><<<grid_for(bytes / 4), NT, 0, s>>>(
            (uint32_t *)dst, (const uint32_t *)src, bytes / 4);
    } else {
        rollover_elem_kernel<uint16_t><<<grid_for(bytes / 2), NT, 0, s>>>(
            (uint16_t *)dst, (const uint16_t *)src, bytes / 2);
    }
    return cudaGetLastError();
}

}  // namespace txl
