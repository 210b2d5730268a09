// project.cu -- the rest of a layer's attention inputs, written straight into
// the layout the attention kernels read (Transformer-XL, Section 3.3):
//
//   txl_project_heads: y[rows][heads][d_pad] = x[rows][d_in] . W[d_in][heads*d_head]
//     (the q / k / v projections W_q, W_kE, W_v of the extended context; with
//     rows = positions x batch of a T-major [T][B][d_model] buffer the result
//     is the T-major [T][B][H][d_pad] layout).  A plain GEMM: cuBLAS, one
//     strided batch over the heads; the padding columns d_head..d_pad-1 are
//     zeroed so that a padded head (d_pad a multiple of 8) can be read by TMA.
//   txl_rel_table: r[t][h][d] = sum_c R[T-1-t][c] W_kR[c][h*d_head + d], the
//     reversed projected table of Appendix B, with R the sinusoid encoding of
//     the relative distance (row p: sin / cos of p * 10000^(-2c/d_model)).
//     Computed once per layer (it does not depend on the batch or on the
//     segment); the sinusoid is evaluated in the kernel, fp32 accumulation.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "txl.h"

namespace txl {
namespace {

std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {nullptr};

// one cuBLAS handle per device, created on first use (released by txl_shutdown)
cublasStatus_t blas_handle(cublasHandle_t *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CUBLAS_STATUS_NOT_INITIALIZED;
    std::lock_guard<std::mutex> lock(g_blas_mu);
    if (!g_blas[dev]) {
        cublasStatus_t st = cublasCreate(&g_blas[dev]);
        if (st != CUBLAS_STATUS_SUCCESS) {
            g_blas[dev] = nullptr;
            return st;
        }
    }
    *out = g_blas[dev];
    return CUBLAS_STATUS_SUCCESS;
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16(x); }

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

constexpr int TB_T = 32;     // table rows per block
constexpr int TB_N = 64;     // output columns per block
constexpr int TB_K = 32;     // d_model slice staged per step

// r[t][h][d] for a 32-row x 64-column block; the sinusoid rows of the block
// are generated slice by slice in shared memory, W_kR slices are staged too.
template <typename T>
__global__ void __launch_bounds__(256)
rel_table_kernel(const T *__restrict__ w, T *__restrict__ out, int Tn, int d_model, int heads, int d_head,
                 int d_pad)
{
    __shared__ float rs[TB_T][TB_K + 1];
    __shared__ float ws[TB_K][TB_N + 1];
    const int t0 = blockIdx.x * TB_T, n0 = blockIdx.y * TB_N;
    const int ncols = heads * d_head;
    const int tid = threadIdx.x;
    const int tr = tid / 16, tc = tid % 16;    // each thread: rows tr, tr+16; columns tc + 16*c
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int k0 = 0; k0 < d_model; k0 += TB_K) {
        for (int x = tid; x < TB_T * TB_K; x += 256) {
            const int i = x / TB_K, c = k0 + x % TB_K;
            const int t = t0 + i;
            float val = 0.f;
            if (t < Tn && c < d_model) {
                const float p = (float)(Tn - 1 - t);                      // the row's distance
                const float freq = powf(10000.f, -(float)(c & ~1) / (float)d_model);
                val = (c & 1) ? cosf(p * freq) : sinf(p * freq);
            }
            rs[i][x % TB_K] = val;
        }
        for (int x = tid; x < TB_K * TB_N; x += 256) {
            const int kk = x / TB_N, n = n0 + x % TB_N, c = k0 + kk;
            ws[kk][x % TB_N] = (c < d_model && n < ncols) ? to_float(w[(long)c * ncols + n]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < TB_K; ++kk) {
            const float a0 = rs[tr][kk], a1 = rs[tr + 16][kk];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float b = ws[kk][tc + 16 * c];
                acc[0][c] += a0 * b;
                acc[1][c] += a1 * b;
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int t = t0 + tr + 16 * rr;
        if (t >= Tn) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = n0 + tc + 16 * c;
            if (n >= ncols) continue;
            const int h = n / d_head, d = n % d_head;
            out[((long)t * heads + h) * d_pad + d] = from_float<T>(acc[rr][c]);
        }
    }
}

bool al(const void *p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }

bool overlap_bytes(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

}  // namespace

void *blas_on_stream(cudaStream_t s)
{
    cublasHandle_t h = nullptr;
    if (blas_handle(&h) != CUBLAS_STATUS_SUCCESS || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return nullptr;
    return (void *)h;
}

cudaError_t blas_shutdown()
{
    std::lock_guard<std::mutex> lock(g_blas_mu);
    for (auto &h : g_blas) {
        if (h) cublasDestroy(h);
        h = nullptr;
    }
    return cudaSuccess;
}

}  // namespace txl

using namespace txl;

extern "C" {

txl_status txl_project_heads(const void *x, const void *w, void *out, int rows, int d_in, int heads,
                             int d_head, int d_pad, txl_dtype dtype, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (rows < 0 || d_in < 0 || heads < 0 || d_head < 1 || d_pad < d_head) return TXL_ERR_INVALID;
    if (rows == 0 || heads == 0) return TXL_OK;
    if (!x || !w || !out) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (!al(x, esz) || !al(w, esz) || !al(out, esz)) return TXL_ERR_INVALID;
    if ((long)heads * d_pad > INT32_MAX || (long)heads * d_head > INT32_MAX) return TXL_ERR_UNSUPPORTED;
    const size_t nout = (size_t)rows * heads * d_pad * esz;
    if (overlap_bytes(out, nout, x, (size_t)rows * d_in * esz) ||
        overlap_bytes(out, nout, w, (size_t)d_in * heads * d_head * esz))
        return TXL_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    if (d_in == 0) {   // empty contraction: zeros
        cudaError_t e = cudaMemsetAsync(out, 0, nout, s);
        return e == cudaSuccess ? TXL_OK : (note_cuda_error(e), TXL_ERR_CUDA);
    }
    cublasHandle_t h = nullptr;
    if (blas_handle(&h) != CUBLAS_STATUS_SUCCESS || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS)
        return TXL_ERR_CUDA;
    // column-major view: per head, y_h^T [d_head x rows] = W_h^T [d_head x d_in] . x^T [d_in x rows]
    const float one = 1.f, zero = 0.f;
    const cudaDataType_t ty = dtype == TXL_F32 ? CUDA_R_32F : CUDA_R_16BF;
    cublasStatus_t st = cublasGemmStridedBatchedEx(
        h, CUBLAS_OP_N, CUBLAS_OP_N, d_head, rows, d_in, &one, w, ty, heads * d_head, (long long)d_head, x, ty,
        d_in, 0LL, &zero, out, ty, heads * d_pad, (long long)d_pad, heads, CUBLAS_COMPUTE_32F,
        CUBLAS_GEMM_DEFAULT);
    if (st != CUBLAS_STATUS_SUCCESS) return TXL_ERR_CUDA;
    if (d_pad > d_head) {
        cudaError_t e = cudaMemset2DAsync((unsigned char *)out + (size_t)d_head * esz, (size_t)d_pad * esz, 0,
                                          (size_t)(d_pad - d_head) * esz, (size_t)rows * heads, s);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return TXL_ERR_CUDA;
        }
    }
    return TXL_OK;
}

txl_status txl_rel_table(const void *w_r, void *out, int klen, int d_model, int heads, int d_head, int d_pad,
                         txl_dtype dtype, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (klen < 0 || d_model < 0 || heads < 0 || d_head < 1 || d_pad < d_head) return TXL_ERR_INVALID;
    if (klen == 0 || heads == 0) return TXL_OK;
    if (!w_r || !out) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (!al(w_r, esz) || !al(out, esz)) return TXL_ERR_INVALID;
    const long ncols = (long)heads * d_head;
    if (ncols > INT32_MAX || (long)heads * d_pad > INT32_MAX || (klen + TB_T - 1) / TB_T > 65535 * 1024L)
        return TXL_ERR_UNSUPPORTED;
    const size_t nout = (size_t)klen * heads * d_pad * esz;
    if (overlap_bytes(out, nout, w_r, (size_t)d_model * ncols * esz)) return TXL_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (d_pad > d_head)
        e = cudaMemsetAsync(out, 0, nout, s);   // padding columns stay zero
    if (e == cudaSuccess) {
        dim3 grid((unsigned)((klen + TB_T - 1) / TB_T), (unsigned)((ncols + TB_N - 1) / TB_N));
        if (grid.y > 65535) return TXL_ERR_UNSUPPORTED;
        if (dtype == TXL_F32)
            rel_table_kernel<float><<<grid, 256, 0, s>>>((const float *)w_r, (float *)out, klen, d_model, heads,
                                                         d_head, d_pad);
        else
            rel_table_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16 *)w_r,
                                                                 (__nv_bfloat16 *)out, klen, d_model, heads,
                                                                 d_head, d_pad);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return TXL_ERR_CUDA;
    }
    return TXL_OK;
}

}  // extern "C"
