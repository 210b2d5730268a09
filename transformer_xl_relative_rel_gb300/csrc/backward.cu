// backward.cu -- gradients of one layer call of the relative attention
// (txl_rel_attn_bwd): the chain rule through the masked softmax and the
// four-term score of Transformer-XL, Section 3.3, for a given output gradient.
//
// Per (b, h), with qu = q + u, qv = q + v, P the softmax weights and A the
// unscaled score (Appendix B route: the position term of row i is the table
// product B~ = qv . r^T read at column L-1-i+j):
//     S    = (qu K^T + shift(qv r^T)) / sqrt(D),   P = masked softmax(S)
//     dP   = dO V^T,   dA = P * (dP - rowsum(P * dP)) / sqrt(D)
//     dV   = P^T dO,   dK = dA^T qu,   dQ = dA K + dB~ r
//     dr   = sum_b dB~^T qv,   du = sum_{b,i} (dA K)_i,   dv_bias = sum_{b,i} (dB~ r)_i
// where dB~ is dA moved into the table's column frame (row i shifted right by
// L-1-i: the inverse of the forward's left shift).
//
// Two routes, chosen per call:
//   - bf16, d_head 64, 16-byte aligned operands (run_bwd_fused): the
//     forward's output O and row log-sum-exp (the caller's saved ones, or the
//     forward kernel once more) feed the tcgen05 score kernel
//     (rel_attn_bwd_scores_kernel in attn_bf16.cu), which recomputes S and
//     the band per tile, forms dP = dO V^T in tensor memory and writes P, dA
//     and dB~ as bf16 matrices (delta = rowsum(dO * O) made in the kernel);
//     five launches of the tcgen05 contraction kernel below give dV, dK,
//     both halves of dQ and dr (dr per (b, h), summed over the batch by fp32
//     reductions), and one pass adds the halves of dQ and forms du, dv_bias
//     as its column sums;
//   - otherwise (fp32, other head sizes: run_bwd) the materialised form: the
//     score, P, dP and dA of every (b, h) are written to the caller's
//     workspace as [L][T] matrices, the eight plain contractions run on the
//     batched CUDA-core GEMM below (bf16 operands and fp32 accumulation on
//     the bf16 path; fp32 throughout on the fp32 path), and the kernels below
//     do the bias fold, the softmax, its gradient and both shifts, and the
//     batch / row reductions of dq, du, dv_bias and dr.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "sm100.cuh"
#include "txl.h"

namespace txl {

// bounded waits of the backward's contraction kernel that gave up (read by txl_check)
__device__ unsigned int g_bwd_err;

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16(x); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// qu = q + u and qv = q + v in q's layout [L][B][H][D]
template <typename T>
__global__ void bwd_fold_kernel(const T *__restrict__ q, const float *__restrict__ u,
                                const float *__restrict__ w, T *__restrict__ qu, T *__restrict__ qv, long n,
                                int H, int D)
{
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const int d = (int)(x % D), h = (int)((x / D) % H);
        const float qq = to_f(q[x]);
        qu[x] = from_f<T>(qq + u[h * D + d]);
        qv[x] = from_f<T>(qq + w[h * D + d]);
    }
}

// the table once per (b, h) so that every batched GEMM walks its operands
// with one stride: rrep[(b*H + h)*T + t][d] = r[t][h][d]
template <typename T>
__global__ void bwd_table_rep_kernel(const T *__restrict__ r, T *__restrict__ rrep, long n, int H, int D,
                                     int Tn)
{
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const int d = (int)(x % D), t = (int)((x / D) % Tn);
        const int h = (int)((x / ((long)D * Tn)) % H);
        rrep[x] = r[((long)t * H + h) * D + d];
    }
}

// The same two copies in 16-byte chunks (8 bf16 or 4 fp32 elements) when D
// is a multiple of the chunk.  A thread's chunk position within a row of
// heads (H * D / C chunks) advances by the grid stride modulo that row, so
// the loop needs one 32-bit division per chunk; with 16-byte aligned biases
// their elements come as float4 loads.
template <typename T, bool kB4>
__global__ void bwd_fold_vec_kernel(const T *__restrict__ q, const float *__restrict__ u,
                                    const float *__restrict__ w, T *__restrict__ qu, T *__restrict__ qv, long nch,
                                    int H, int D)
{
    constexpr int C = 16 / sizeof(T);
    const unsigned dc = (unsigned)(D / C), hdc = (unsigned)H * dc;
    const long x0 = (long)blockIdx.x * blockDim.x + threadIdx.x, stride = (long)gridDim.x * blockDim.x;
    unsigned y = (unsigned)(x0 % hdc);
    const unsigned ystep = (unsigned)(stride % hdc);
    for (long x = x0; x < nch; x += stride) {
        const unsigned h = y / dc;
        const int hd = (int)(h * D + (y - h * dc) * C);   // bias element of this chunk's first column
        const uint4 raw = reinterpret_cast<const uint4 *>(q)[x];
        const T *e = reinterpret_cast<const T *>(&raw);
        float ub[C], wb[C];
        if (kB4) {
#pragma unroll
            for (int c = 0; c < C; c += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(u + hd + c);
                const float4 b4 = *reinterpret_cast<const float4 *>(w + hd + c);
                ub[c] = a4.x, ub[c + 1] = a4.y, ub[c + 2] = a4.z, ub[c + 3] = a4.w;
                wb[c] = b4.x, wb[c + 1] = b4.y, wb[c + 2] = b4.z, wb[c + 3] = b4.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                ub[c] = u[hd + c];
                wb[c] = w[hd + c];
            }
        }
        uint4 a, b;
        T *ea = reinterpret_cast<T *>(&a), *eb = reinterpret_cast<T *>(&b);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float qq = to_f(e[c]);
            ea[c] = from_f<T>(qq + ub[c]);
            eb[c] = from_f<T>(qq + wb[c]);
        }
        reinterpret_cast<uint4 *>(qu)[x] = a;
        reinterpret_cast<uint4 *>(qv)[x] = b;
        y += ystep;
        if (y >= hdc) y -= hdc;
    }
}

// one launch of the chunked fold: float4 bias loads when both biases are
// 16-byte aligned
template <typename T>
void launch_fold_vec(const T *q, const float *u, const float *w, T *qu, T *qv, long nch, int H, int D, unsigned grid,
                     cudaStream_t s)
{
    if (((uintptr_t)u & 15) == 0 && ((uintptr_t)w & 15) == 0)
        bwd_fold_vec_kernel<T, true><<<grid, 256, 0, s>>>(q, u, w, qu, qv, nch, H, D);
    else
        bwd_fold_vec_kernel<T, false><<<grid, 256, 0, s>>>(q, u, w, qu, qv, nch, H, D);
}

template <typename T>
__global__ void bwd_table_rep_vec_kernel(const T *__restrict__ r, T *__restrict__ rrep, long nch, int H, int D,
                                         int Tn)
{
    const int dc = D / (16 / (int)sizeof(T));
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < nch; x += (long)gridDim.x * blockDim.x) {
        const int c = (int)(x % dc);
        const long tr = x / dc;                        // (b*H + h)*T + t
        const int t = (int)(tr % Tn), h = (int)((tr / Tn) % H);
        reinterpret_cast<uint4 *>(rrep)[x] = reinterpret_cast<const uint4 *>(r)[((long)t * H + h) * dc + c];
    }
}

// One warp per query row (b, h, i) (row = (b*H + h)*L + i): the score from
// the content product s (in place) and the table product bt read at column
// L-1-i+j, the masked softmax over keys 0..M+i, P written back to s (fp32,
// zeros where masked) and to pb in the GEMM operand type.
template <typename T>
__global__ void bwd_softmax_kernel(float *__restrict__ s, const float *__restrict__ bt, T *__restrict__ pb,
                                   long nrows, int L, int M, int Tn, float scale)
{
    const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const int i = (int)(row % L), last = M + i, sh = L - 1 - i;
    float *sr = s + row * Tn;
    const float *br = bt + row * Tn;
    T *pr = pb + row * Tn;
    float mx = -INFINITY;
    for (int j = lane; j <= last; j += 32) {
        const float a = (sr[j] + br[sh + j]) * scale;
        sr[j] = a;
        mx = fmaxf(mx, a);
    }
    mx = warp_max(mx);
    float z = 0.f;
    for (int j = lane; j <= last; j += 32) {
        const float e = expf(sr[j] - mx);
        sr[j] = e;
        z += e;
    }
    const float inv = 1.f / warp_sum(z);
    for (int j = lane; j < Tn; j += 32) {
        const float p = j <= last ? sr[j] * inv : 0.f;
        sr[j] = p;
        pr[j] = from_f<T>(p);
    }
}

// One warp per query row: dA = P (dP - sum_j P dP) / sqrt(D) over the visible
// keys (zero elsewhere) into da, and the same values moved to the table's
// column frame (column L-1-i+j; columns below L-1-i are zero) into db.
template <typename T>
__global__ void bwd_score_grad_kernel(const float *__restrict__ p, const float *__restrict__ dp,
                                      T *__restrict__ da, T *__restrict__ db, long nrows, int L, int M, int Tn,
                                      float scale)
{
    const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const int i = (int)(row % L), last = M + i, sh = L - 1 - i;
    const float *pr = p + row * Tn, *gr = dp + row * Tn;
    float delta = 0.f;
    for (int j = lane; j <= last; j += 32) delta += pr[j] * gr[j];
    delta = warp_sum(delta);
    T *dar = da + row * Tn, *dbr = db + row * Tn;
    for (int j = lane; j < Tn; j += 32) {
        dar[j] = from_f<T>(j <= last ? pr[j] * (gr[j] - delta) * scale : 0.f);
        const int jj = j - sh;   // the key whose pair has table column j
        dbr[j] = from_f<T>(jj >= 0 && jj <= last ? pr[jj] * (gr[jj] - delta) * scale : 0.f);
    }
}

// The same two steps with one 256-thread block per row and the row held in
// registers (NPT entries per thread, rows of up to 256*NPT keys): each input
// is read once and each output written once.
constexpr int RB = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red)
{
    v = is_max ? warp_max(v) : warp_sum(v);
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();                       // red is reused across calls
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float x = lane < (RB >> 5) ? red[lane] : (is_max ? -INFINITY : 0.f);
    return is_max ? warp_max(x) : warp_sum(x);
}

template <typename T, int NPT>
__global__ void __launch_bounds__(RB) bwd_softmax_row_kernel(float *__restrict__ s, const float *__restrict__ bt,
                                                             T *__restrict__ pb, int L, int M, int Tn, float scale)
{
    __shared__ float red[RB / 32];
    const long row = blockIdx.x;
    const int i = (int)(row % L), last = M + i, sh = L - 1 - i;
    float *sr = s + row * Tn;
    const float *br = bt + row * Tn;
    float x[NPT];
    float mx = -INFINITY;
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        const int j = threadIdx.x + RB * m;
        x[m] = j <= last ? (sr[j] + br[sh + j]) * scale : -INFINITY;
        mx = fmaxf(mx, x[m]);
    }
    mx = block_reduce(mx, true, red);
    float z = 0.f;
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        x[m] = expf(x[m] - mx);            // 0 for masked keys
        z += x[m];
    }
    const float inv = 1.f / block_reduce(z, false, red);
    T *pr = pb + row * Tn;
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        const int j = threadIdx.x + RB * m;
        if (j < Tn) {
            sr[j] = x[m] * inv;
            pr[j] = from_f<T>(x[m] * inv);
        }
    }
}

template <typename T, int NPT>
__global__ void __launch_bounds__(RB) bwd_score_grad_row_kernel(const float *__restrict__ p,
                                                                const float *__restrict__ dp, T *__restrict__ da,
                                                                T *__restrict__ db, int L, int M, int Tn,
                                                                float scale)
{
    __shared__ float red[RB / 32];
    __shared__ float row_da[RB * NPT];
    const long row = blockIdx.x;
    const int i = (int)(row % L), last = M + i, sh = L - 1 - i;
    const float *pr = p + row * Tn, *gr = dp + row * Tn;
    float pv[NPT], gv[NPT];
    float delta = 0.f;
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        const int j = threadIdx.x + RB * m;
        pv[m] = j <= last ? pr[j] : 0.f;
        gv[m] = j <= last ? gr[j] : 0.f;
        delta += pv[m] * gv[m];
    }
    delta = block_reduce(delta, false, red);
    T *dar = da + row * Tn, *dbr = db + row * Tn;
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        const int j = threadIdx.x + RB * m;
        const float a = pv[m] * (gv[m] - delta) * scale;   // 0 past the last key
        if (j < Tn) {
            row_da[j] = a;
            dar[j] = from_f<T>(a);
        }
    }
    __syncthreads();
    // table frame: column c holds the pair of key c - (L-1-i)
#pragma unroll
    for (int m = 0; m < NPT; ++m) {
        const int c = threadIdx.x + RB * m, jj = c - sh;
        if (c < Tn) dbr[c] = from_f<T>(jj >= 0 ? row_da[jj] : 0.f);
    }
}

// dq = dQ_content + dQ_position in the output type, and in the same pass the
// bias gradients: du[h][d] += the column sum over rows (i, b) of the content
// part, dw[h][d] likewise of the position part (du, dw zeroed before; either
// may be NULL).  Grid (row chunks, column slabs of blockDim.x); a thread owns
// one column of the [L*B][H*D] matrices and strides over the rows.
template <typename T>
__global__ void bwd_sum_bias_kernel(const float *__restrict__ a, const float *__restrict__ b, T *__restrict__ out,
                                    float *__restrict__ du, float *__restrict__ dw, long rows, int hd)
{
    const int c = blockIdx.y * blockDim.x + threadIdx.x;
    if (c >= hd) return;
    float su = 0.f, sw = 0.f;
    for (long rr = blockIdx.x; rr < rows; rr += gridDim.x) {
        const long x = rr * hd + c;
        const float va = a[x], vb = b[x];
        out[x] = from_f<T>(va + vb);
        su += va;
        sw += vb;
    }
    if (du) atomicAdd(du + c, su);
    if (dw) atomicAdd(dw + c, sw);
}

// bwd_sum_bias_kernel with du, dw zeroed first: about eight blocks of 256
// threads per SM over the column slabs, so that each thread streams a few
// dozen rows (enough loads in flight) and each column takes few atomics
template <typename T>
cudaError_t launch_sum_bias(const float *dqc, const float *dqp, T *dq, float *du, float *dw, long rows, int hd,
                            cudaStream_t s)
{
    cudaError_t e;
    if (du && (e = cudaMemsetAsync(du, 0, (size_t)hd * 4, s)) != cudaSuccess) return e;
    if (dw && (e = cudaMemsetAsync(dw, 0, (size_t)hd * 4, s)) != cudaSuccess) return e;
    const int slabs = (hd + 255) / 256;
    long chunks = 8L * device_sm_count() / slabs;
    if (chunks > rows) chunks = rows;
    if (chunks < 1) chunks = 1;
    bwd_sum_bias_kernel<T><<<dim3((unsigned)chunks, (unsigned)slabs), 256, 0, s>>>(dqc, dqp, dq, du, dw, rows, hd);
    return cudaGetLastError();
}

// dr[t][h][d] = sum_b part[(b*H + h)*T + t][d]
template <typename T>
__global__ void bwd_table_grad_kernel(const float *__restrict__ part, T *__restrict__ dr, int B, int H, int D,
                                      int Tn)
{
    const long n = (long)Tn * H * D;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const int d = (int)(x % D), h = (int)((x / D) % H), t = (int)(x / ((long)D * H));
        float acc = 0.f;
        for (int b = 0; b < B; ++b) acc += part[(((long)b * H + h) * Tn + t) * D + d];
        dr[x] = from_f<T>(acc);
    }
}

// Row-major C (m x n, ldc) = op(A) . op(B) for `batch` problems at the given
// element strides (sA, sB, sC between problems); ta: A is stored k x m (used
// transposed), tb: B is stored n x k.  A 64 x 64 block of C per CTA, K in
// slices of 16 staged in shared memory, 4 x 4 outputs per thread, fp32
// accumulation: the plain contractions of the materialised route (the fp32
// parity path and head sizes the tensor-core route does not take).
constexpr int SG_T = 64, SG_K = 16;

template <typename E, typename C>
__global__ void __launch_bounds__(256)
simt_gemm_kernel(bool ta, bool tb, int m, int n, int k, const E *__restrict__ A, long lda, long long sA,
                 const E *__restrict__ Bm, long ldb, long long sB, C *__restrict__ Cm, long ldc, long long sC)
{
    __shared__ float as[SG_K][SG_T + 1];
    __shared__ float bs[SG_K][SG_T + 1];
    const long z = blockIdx.z;
    const E *a = A + z * sA;
    const E *b = Bm + z * sB;
    C *c = Cm + z * sC;
    const int m0 = blockIdx.y * SG_T, n0 = blockIdx.x * SG_T;
    const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < k; k0 += SG_K) {
        for (int x = tid; x < SG_K * SG_T; x += 256) {
            // both tiles staged as [kk][row or column], element (row, k) read
            // along whichever index is contiguous in memory
            const int kk = ta ? x / SG_T : x % SG_K, mm = ta ? x % SG_T : x / SG_K;
            const int gm = m0 + mm, gk = k0 + kk;
            as[kk][mm] = (gm < m && gk < k) ? to_f(ta ? a[(long)gk * lda + gm] : a[(long)gm * lda + gk]) : 0.f;
            const int kb = tb ? x % SG_K : x / SG_T, nn = tb ? x / SG_K : x % SG_T;
            const int gn = n0 + nn, gkb = k0 + kb;
            bs[kb][nn] = (gn < n && gkb < k) ? to_f(tb ? b[(long)gn * ldb + gkb] : b[(long)gkb * ldb + gn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_K; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = as[kk][tr + 16 * i];
                bv[i] = bs[kk][tc + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] += av[i] * bv[j];
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + tr + 16 * i;
        if (gm >= m) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tc + 16 * j;
            if (gn < n) c[(long)gm * ldc + gn] = from_f<C>(acc[i][j]);
        }
    }
}

template <typename E, typename C>
bool gemm_rm(cudaStream_t s, bool ta, bool tb, int m, int n, int k, const void *A, long lda, long long sA,
             const void *Bm, long ldb, long long sB, void *Cm, long ldc, long long sC, int batch)
{
    const dim3 grid((unsigned)((n + SG_T - 1) / SG_T), (unsigned)((m + SG_T - 1) / SG_T), (unsigned)batch);
    if (grid.y > 65535 || grid.z > 65535) return false;
    simt_gemm_kernel<E, C><<<grid, 256, 0, s>>>(ta, tb, m, n, k, (const E *)A, lda, sA, (const E *)Bm, ldb, sB,
                                                (C *)Cm, ldc, sC);
    return cudaGetLastError() == cudaSuccess;
}

// =========================================================================
// The fused route's contractions on the tensor cores (bf16 operands, fp32
// accumulation in TMEM).  For each batch entry z and 128-row block of C:
//     C[z][m][0..63] = sum_p sum_k A_p[z](m, k) B_p[z](k, 0..63)
// over one or two operand pairs p (dQ's content and position halves could
// share a pass; each runs as its own pair here so that the bias gradients
// see them apart).  A is K-major (rows m of a matrix contiguous along k) or
// MN-major (the matrix stored with m contiguous, i.e. A^T row-major: P, dA
// and the table-frame dA used transposed); B is MN-major with 64 columns
// (rows k of 64 contiguous elements: dO, q+u, K, the table, q+v).  Both
// arrive by TMA with the 128-byte swizzle: a K-major A stage is 128 rows x
// 64 k; an MN-major A stage is two 64-row blocks of 64 k-rows, 8 KB apart
// (the descriptor's leading-dimension offset), a B stage is 64 k-rows.
// Warp 0 loads, warp 1 issues the MMAs (four K=16 steps per 64-wide stage),
// warps 4-7 take the accumulator (two 64-column buffers in TMEM) to global
// memory, a lane per row.  Four 24 KB stages, so that two CTAs share an SM
// (two independent load / MMA chains; 128 TMEM columns each).
constexpr int BG_M = 128, BG_K = 64, BG_ST = 4, BG_NT = 256;
constexpr uint64_t BG_WAIT_NS = 2000000000ull;

struct BgSmem {
    static constexpr uint32_t ASZ = BG_M * 128;        // 16 KB
    static constexpr uint32_t BSZ = BG_K * 128;        // 8 KB
    static constexpr uint32_t A = 0;
    static constexpr uint32_t B = A + BG_ST * ASZ;
    static constexpr uint32_t BARS = B + BG_ST * BSZ;
    static constexpr int FULL = 0, EMPTY = BG_ST, AFULL = 2 * BG_ST, AEMPTY = 2 * BG_ST + 2,
                         DONE = 2 * BG_ST + 4, NBAR = 2 * BG_ST + 5;
    static constexpr uint32_t MISC = BARS + NBAR * 8;
    static constexpr uint32_t TOTAL = MISC + 16 + 1024;
};

struct BgOperand {
    int rank;         // 3: coordinates (c0, c1, z') ; 4: (c0, c1, z / H, z % H)
    int zmod;         // rank 3: z' = z (0) or z % H (1)
};

struct BgParams {
    BgOperand a[2], b[2];
    int pairs, a_mn, ksteps[2];
    int M, nz, H, mtiles, tiles;
    void *out;
    long ostride;     // elements between output rows; batch entry z starts at z * 64
    int ofp32;        // output fp32 (else bf16)
    int oadd;         // fp32 reductions into out at column (z % H) * 64 (the batch sum of dr)
};

__device__ __forceinline__ void bg_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bg_load(uint32_t dst, const CUtensorMap *m, uint32_t bar, const BgOperand &o, int c0,
                                        int c1, int z, int H)
{
    if (o.rank == 4)
        sm100::tma_load_4d(dst, m, bar, c0, c1, z / H, z % H);
    else
        sm100::tma_load_3d(dst, m, bar, c0, c1, o.zmod ? z % H : z);
}

__global__ void __launch_bounds__(BG_NT, 2)
bwd_gemm_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1, const BgParams p)
{
    using namespace sm100;
    using S = BgSmem;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + S::BARS + 8u * (uint32_t)i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::MISC + 8);
    auto wait = [&](int i, uint32_t parity) -> bool {
        const uint32_t b = bar(i);
        if (mbar_try_wait(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            if (mbar_try_wait_sleep(b, parity, WAIT_SLEEP_NS)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > BG_WAIT_NS) {
                *abort = 1;
                atomicOr(&g_bwd_err, 1u);
                return false;
            }
        }
    };
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        *abort = 0;
        for (int x = 0; x < BG_ST; ++x) {
            mbar_init(bar(S::FULL + x), 1);
            mbar_init(bar(S::EMPTY + x), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(S::AFULL + x), 1);
            mbar_init(bar(S::AEMPTY + x), 128);
        }
        mbar_init(bar(S::DONE), 1);
        fence_mbar_init();
        prefetch_tmap(&ta0);
        prefetch_tmap(&tb0);
        if (p.pairs > 1) {
            prefetch_tmap(&ta1);
            prefetch_tmap(&tb1);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int G = gridDim.x;

    if (warp == 0) {
        // =================================================================== TMA producer
        if (lane == 0) {
            const uint32_t bytes = S::ASZ + S::BSZ;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.tiles; t += G) {
                const int z = t / p.mtiles, m0 = (t % p.mtiles) * BG_M;
                for (int q = 0; ok && q < p.pairs; ++q) {
                    const CUtensorMap *ma = q ? &ta1 : &ta0, *mb = q ? &tb1 : &tb0;
                    for (int ks = 0; ks < p.ksteps[q]; ++ks, ++it) {
                        const int s = it % BG_ST;
                        if (it >= BG_ST && !wait(S::EMPTY + s, ((it / BG_ST) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        const uint32_t da = sbase + S::A + s * S::ASZ, db = sbase + S::B + s * S::BSZ;
                        mbar_arrive_expect_tx(bar(S::FULL + s), bytes);
                        if (p.a_mn) {
                            // two 64-row blocks of the transposed matrix, 8 KB apart
                            bg_load(da, ma, bar(S::FULL + s), p.a[q], m0, ks * BG_K, z, p.H);
                            bg_load(da + 8192u, ma, bar(S::FULL + s), p.a[q], m0 + 64, ks * BG_K, z, p.H);
                        } else {
                            bg_load(da, ma, bar(S::FULL + s), p.a[q], ks * BG_K, m0, z, p.H);
                        }
                        bg_load(db, mb, bar(S::FULL + s), p.b[q], 0, ks * BG_K, z, p.H);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // =================================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(BG_M, 64, p.a_mn, 1);
            // K-major A: K steps of 32 bytes along the row; MN-major A and B:
            // K steps of 16 rows (2 KB), the A blocks 8 KB apart
            const uint64_t da0 = p.a_mn ? smem_desc_sw128(sbase + S::A, 8192, 1024)
                                        : smem_desc_sw128(sbase + S::A, 16, 1024);
            const uint64_t db0 = smem_desc_sw128(sbase + S::B, 16, 1024);
            const uint64_t astep = p.a_mn ? 128 : 2;
            int it = 0, lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.tiles; t += G, ++lt) {
                const int buf = lt & 1;
                if (lt >= 2 && !wait(S::AEMPTY + buf, ((lt >> 1) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)buf * 64u;
                bool first = true;
                for (int q = 0; ok && q < p.pairs; ++q) {
                    for (int ks = 0; ks < p.ksteps[q]; ++ks, ++it) {
                        const int s = it % BG_ST;
                        if (!wait(S::FULL + s, (it / BG_ST) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t da = da0 + ((uint64_t)(s * S::ASZ) >> 4);
                        const uint64_t db = db0 + ((uint64_t)(s * S::BSZ) >> 4);
#pragma unroll
                        for (int kk = 0; kk < BG_K / 16; ++kk) {
                            mma_bf16_ss(acc, da + astep * kk, db + 128 * kk, idesc, first ? 0u : 1u);
                            first = false;
                        }
                        mma_commit(bar(S::EMPTY + s));
                    }
                }
                if (ok) mma_commit(bar(S::AFULL + buf));
            }
            mma_commit(bar(S::DONE));
            wait(S::DONE, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // =================================================================== epilogue
        const int q = warp & 3;
        int lt = 0;
        for (int t = blockIdx.x; t < p.tiles; t += G, ++lt) {
            const int buf = lt & 1;
            const int z = t / p.mtiles, m0 = (t % p.mtiles) * BG_M;
            if (!wait(S::AFULL + buf, (lt >> 1) & 1)) break;
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 64u;
            float v[64];
            tmem_ld32(tacc, *reinterpret_cast<float(*)[32]>(v));
            tmem_ld32(tacc + 32u, *reinterpret_cast<float(*)[32]>(v + 32));
            tc_fence_before();
            bg_arrive(bar(S::AEMPTY + buf));
            const int row = m0 + 32 * q + lane;
            if (row < p.M && p.oadd) {
                // this batch entry's share of a sum over the batch: 16-byte
                // fp32 reductions (the order of the adds is not fixed)
                float *o = reinterpret_cast<float *>(p.out) + (long)row * p.ostride + (long)(z % p.H) * 64;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(o + 4 * j), "f"(v[4 * j]),
                                 "f"(v[4 * j + 1]), "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                                 : "memory");
            } else if (row < p.M) {
                const long off = (long)row * p.ostride + (long)z * 64;
                if (p.ofp32) {
                    float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + off);
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                } else {
                    uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + off);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 pk;
                        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * j + 0], v[8 * j + 1]);
                        __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * j + 2], v[8 * j + 3]);
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * j + 4], v[8 * j + 5]);
                        __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * j + 6], v[8 * j + 7]);
                        pk.x = *reinterpret_cast<uint32_t *>(&h0);
                        pk.y = *reinterpret_cast<uint32_t *>(&h1);
                        pk.z = *reinterpret_cast<uint32_t *>(&h2);
                        pk.w = *reinterpret_cast<uint32_t *>(&h3);
                        o[j] = pk;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// bf16 copy of an fp32 array, four elements per thread and step
__global__ void bwd_round_kernel(const float *__restrict__ src, __nv_bfloat16 *__restrict__ dst, long n4)
{
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (long)gridDim.x * blockDim.x) {
        const float4 f = reinterpret_cast<const float4 *>(src)[x];
        __nv_bfloat162 a = __floats2bfloat162_rn(f.x, f.y), b = __floats2bfloat162_rn(f.z, f.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        reinterpret_cast<uint2 *>(dst)[x] = u;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 bg_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// A bf16 tensor map with the 128-byte swizzle: dims / byte strides (of dims
// 1..rank-1) / box, innermost first.
bool bg_map(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box)
{
    auto enc = bg_encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_bwd_gemm(const CUtensorMap *ma, const CUtensorMap *mb, const BgParams &p0, cudaStream_t s)
{
    BgParams p = p0;
    p.mtiles = (p.M + BG_M - 1) / BG_M;
    const long tiles = (long)p.mtiles * p.nz;
    if (tiles > INT32_MAX) return cudaErrorNotSupported;
    p.tiles = (int)tiles;
    if (p.tiles == 0) return cudaSuccess;
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(opted.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(bwd_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BgSmem::TOTAL);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_relaxed);
    }
    const int grid = p.tiles < 2 * device_sm_count() ? p.tiles : 2 * device_sm_count();
    bwd_gemm_kernel<<<(unsigned)grid, BG_NT, BgSmem::TOTAL, s>>>(ma[0], mb[0], p.pairs > 1 ? ma[1] : ma[0],
                                                                  p.pairs > 1 ? mb[1] : mb[0], p);
    return cudaGetLastError();
}

struct Ws {
    size_t x1, x2, pb, da, db, qu, qv, rrep, dqc, dqp, drp, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

Ws layout(long B, long H, long D, long L, long M, size_t es)
{
    const long T = M + L;
    const size_t sq = (size_t)B * H * L * T;   // one [L][T] matrix per (b, h)
    Ws w;
    size_t o = 0;
    w.x1 = o;   o += up256(sq * 4);
    w.x2 = o;   o += up256(sq * 4);
    w.pb = o;   o += up256(sq * es);
    w.da = o;   o += up256(sq * es);
    w.db = o;   o += up256(sq * es);
    w.qu = o;   o += up256((size_t)L * B * H * D * es);
    w.qv = o;   o += up256((size_t)L * B * H * D * es);
    w.rrep = o; o += up256((size_t)B * H * T * D * es);
    w.dqc = o;  o += up256((size_t)L * B * H * D * 4);
    w.dqp = o;  o += up256((size_t)L * B * H * D * 4);
    w.drp = o;  o += up256((size_t)B * H * T * D * 4);
    w.total = o;
    return w;
}

// The fused path (bf16, D = 64): P, dA and dA in the table frame as bf16
// [B*H][L][TP] (TP = M+L rounded up to 128) written by the tcgen05 scores
// kernel, the forward's output and row log-sum-exp, delta, and the same
// GEMM operands and partial sums as the materialised path.
struct WsF {
    size_t pb, da, db, qu, qv, dqc, dqp, out, lse, split, dracc, total;
    long TP;
    int splits;
};

WsF layout_fused(long B, long H, long D, long L, long M)
{
    const long T = M + L;
    WsF w;
    w.TP = (T + 127) / 128 * 128;
    const size_t sq = (size_t)B * H * L * w.TP * 2;
    size_t o = 0;
    w.pb = o;    o += up256(sq);
    w.da = o;    o += up256(sq);
    w.db = o;    o += up256(sq);
    w.qu = o;    o += up256((size_t)L * B * H * D * 2);
    w.qv = o;    o += up256((size_t)L * B * H * D * 2);
    w.dqc = o;   o += up256((size_t)L * B * H * D * 4);
    w.dqp = o;   o += up256((size_t)L * B * H * D * 4);
    w.out = o;   o += up256((size_t)L * B * H * D * 2);
    w.lse = o;   o += up256((size_t)B * H * L * 4);
    AttnArgs a{};
    a.B = (int)B;
    a.H = (int)H;
    a.D = (int)D;
    a.L = (int)L;
    a.M = (int)M;
    w.splits = bf16_num_splits(a, device_sm_count());
    w.split = o; o += up256(w.splits > 1 ? bf16_scratch_bytes(a, w.splits) : 0);
    w.dracc = o; o += up256((size_t)T * H * D * 4);
    w.total = o;
    return w;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || !na || !nb) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

unsigned grid_for(long n, int threads)
{
    long g = (n + threads - 1) / threads;
    const long cap = (long)device_sm_count() * 16;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

template <typename E>
txl_status run_bwd(const void *q, const void *k, const void *v, const void *r, const float *u, const float *w,
                   const void *dout, int B, int M, int L, int H, int D, void *dq, void *dk, void *dv, void *dr,
                   float *du, float *dw, unsigned char *ws, const Ws &lay, cudaStream_t s, bool bf16)
{
    const long T = (long)M + L, BH = (long)B * H, nq = (long)L * BH * D, rows = BH * L;
    const long ld = BH * D;                 // row pitch of the [pos][B][H][D] tensors
    const float scale = 1.f / sqrtf((float)D);
    E *qu = (E *)(ws + lay.qu), *qv = (E *)(ws + lay.qv), *rrep = (E *)(ws + lay.rrep);
    E *pb = (E *)(ws + lay.pb), *dab = (E *)(ws + lay.da), *dbb = (E *)(ws + lay.db);
    float *x1 = (float *)(ws + lay.x1), *x2 = (float *)(ws + lay.x2);
    float *dqc = (float *)(ws + lay.dqc), *dqp = (float *)(ws + lay.dqp), *drp = (float *)(ws + lay.drp);
    (void)bf16;
    cudaError_t e = cudaSuccess;
    auto chk = [&]() {
        e = cudaGetLastError();
        return e == cudaSuccess;
    };
    if (D % (16 / (int)sizeof(E)) == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)r & 15) == 0) {
        const int C = 16 / (int)sizeof(E);
        launch_fold_vec<E>((const E *)q, u, w, qu, qv, nq / C, H, D, grid_for(nq / C, 256), s);
        if (!chk()) goto cuda_fail;
        bwd_table_rep_vec_kernel<E><<<grid_for(BH * T * D / C, 256), 256, 0, s>>>((const E *)r, rrep,
                                                                                BH * T * D / C, H, D, (int)T);
        if (!chk()) goto cuda_fail;
    } else {
        bwd_fold_kernel<E><<<grid_for(nq, 256), 256, 0, s>>>((const E *)q, u, w, qu, qv, nq, H, D);
        if (!chk()) goto cuda_fail;
        bwd_table_rep_kernel<E><<<grid_for(BH * T * D, 256), 256, 0, s>>>((const E *)r, rrep, BH * T * D, H, D,
                                                                         (int)T);
        if (!chk()) goto cuda_fail;
    }
    {
        const long long LT = (long long)L * T, TD = (long long)T * D;
        const int Ti = (int)T, nb = (int)BH;
        // content and table products, then the softmax
        if (!gemm_rm<E, float>(s, false, true, L, Ti, D, qu, ld, D, k, ld, D, x1, T, LT, nb) ||
            !gemm_rm<E, float>(s, false, true, L, Ti, D, qv, ld, D, rrep, D, TD, x2, T, LT, nb))
            return TXL_ERR_CUDA;
        if (T <= RB * 6)
            bwd_softmax_row_kernel<E, 6><<<(unsigned)rows, RB, 0, s>>>(x1, x2, pb, L, M, Ti, scale);
        else if (T <= RB * 16)
            bwd_softmax_row_kernel<E, 16><<<(unsigned)rows, RB, 0, s>>>(x1, x2, pb, L, M, Ti, scale);
        else
            bwd_softmax_kernel<E><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x1, x2, pb, rows, L, M, Ti, scale);
        if (!chk()) goto cuda_fail;
        // dP, then the score gradient in both frames
        if (!gemm_rm<E, float>(s, false, true, L, Ti, D, dout, ld, D, v, ld, D, x2, T, LT, nb)) return TXL_ERR_CUDA;
        if (T <= RB * 6)
            bwd_score_grad_row_kernel<E, 6><<<(unsigned)rows, RB, 0, s>>>(x1, x2, dab, dbb, L, M, Ti, scale);
        else if (T <= RB * 16)
            bwd_score_grad_row_kernel<E, 16><<<(unsigned)rows, RB, 0, s>>>(x1, x2, dab, dbb, L, M, Ti, scale);
        else
            bwd_score_grad_kernel<E><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x1, x2, dab, dbb, rows, L, M,
                                                                                Ti, scale);
        if (!chk()) goto cuda_fail;
        // dV = P^T dO, dK = dA^T qu, dQ = dA K + dB~ r, dr per (b, h) = dB~^T qv
        if (!gemm_rm<E, E>(s, true, false, Ti, D, L, pb, T, LT, dout, ld, D, dv, ld, D, nb) ||
            !gemm_rm<E, E>(s, true, false, Ti, D, L, dab, T, LT, qu, ld, D, dk, ld, D, nb) ||
            !gemm_rm<E, float>(s, false, false, L, D, Ti, dab, T, LT, k, ld, D, dqc, ld, D, nb) ||
            !gemm_rm<E, float>(s, false, false, L, D, Ti, dbb, T, LT, rrep, D, TD, dqp, ld, D, nb) ||
            !gemm_rm<E, float>(s, true, false, Ti, D, L, dbb, T, LT, qv, ld, D, drp, D, TD, nb))
            return TXL_ERR_CUDA;
    }
    if ((e = launch_sum_bias<E>(dqc, dqp, (E *)dq, du, dw, (long)L * B, H * D, s)) != cudaSuccess) goto cuda_fail;
    bwd_table_grad_kernel<E><<<grid_for(T * H * D, 256), 256, 0, s>>>(drp, (E *)dr, B, H, D, (int)T);
    if (!chk()) goto cuda_fail;
    return TXL_OK;
cuda_fail:
    note_cuda_error(e);
    return TXL_ERR_CUDA;
}

txl_status run_bwd_fused(const void *q, const void *k, const void *v, const void *r, const float *u,
                         const float *w, const void *dout, const void *out_saved, const float *lse_saved, int B,
                         int M, int L, int H, int D, void *dq, void *dk, void *dv, void *dr, float *du, float *dw,
                         unsigned char *ws, const WsF &lay, cudaStream_t s)
{
    typedef __nv_bfloat16 E;
    const long T = (long)M + L, BH = (long)B * H, nq = (long)L * BH * D, TP = lay.TP;
    E *qu = (E *)(ws + lay.qu), *qv = (E *)(ws + lay.qv);
    E *pb = (E *)(ws + lay.pb), *dab = (E *)(ws + lay.da), *dbb = (E *)(ws + lay.db), *outf = (E *)(ws + lay.out);
    float *lse = (float *)(ws + lay.lse);
    float *dqc = (float *)(ws + lay.dqc), *dqp = (float *)(ws + lay.dqp), *dracc = (float *)(ws + lay.dracc);
    cudaError_t e = cudaSuccess;
    auto chk = [&]() {
        e = cudaGetLastError();
        return e == cudaSuccess;
    };
    // the forward's output and row log-sum-exp: the caller's saved ones, or
    // the forward once more
    AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.r = r;
    a.u = u;
    a.w = w;
    a.out = outf;
    a.B = B;
    a.H = H;
    a.D = D;
    a.L = L;
    a.M = M;
    a.lse = lse;
    if (out_saved && lse_saved) {
        a.out = const_cast<void *>(out_saved);
        a.lse = const_cast<float *>(lse_saved);
        lse = a.lse;
    } else if ((e = launch_attn_bf16(a, lay.splits, lay.splits > 1 ? ws + lay.split : nullptr, s)) != cudaSuccess) {
        goto cuda_fail;
    }
    if ((e = launch_bwd_scores(a, dout, lse, pb, dab, dbb, TP, s)) != cudaSuccess) goto cuda_fail;
    // the GEMM operands q+u, q+v
    launch_fold_vec<E>((const E *)q, u, w, qu, qv, nq / 8, H, D, grid_for(nq / 8, 256), s);
    if (!chk()) goto cuda_fail;
    {
        // per (b, h): dV = P^T dO, dK = dA^T qu (rows j of the transposed
        // [L][TP] matrices), dQ's content half dA K (rows i); per (b, h) rows
        // i of the head-major table-frame dA~: dQ's position half dA~ r; per
        // head, over the head's (i, b) rows of dA~: dr = dA~^T qv (the batch
        // sum falls out of the contraction)
        const cuuint64_t e2 = 2, tp2 = (cuuint64_t)TP * e2, row2 = (cuuint64_t)BH * 64 * e2;
        CUtensorMap pmn, damn, dak, dbk, dbmn, mdo, mqu, mk, mr, mqv;
        const cuuint64_t d_mat[3] = {(cuuint64_t)TP, (cuuint64_t)L, (cuuint64_t)BH};
        const cuuint64_t s_mat[2] = {tp2, (cuuint64_t)L * tp2};
        const cuuint32_t box_mn[3] = {64, 64, 1}, box_k[3] = {64, 128, 1};
        const cuuint64_t d_db4[4] = {(cuuint64_t)TP, (cuuint64_t)L, (cuuint64_t)B, (cuuint64_t)H};
        const cuuint64_t s_db4[3] = {(cuuint64_t)B * tp2, tp2, (cuuint64_t)L * B * tp2};
        const cuuint32_t box_k4[4] = {64, 128, 1, 1};
        const cuuint32_t box_mn4[4] = {64, 64, 1, 1};
        const cuuint64_t d_q[3] = {64, (cuuint64_t)L, (cuuint64_t)BH}, s_q[2] = {row2, 64 * e2};
        const cuuint64_t d_k[3] = {64, (cuuint64_t)T, (cuuint64_t)BH};
        const cuuint64_t d_r[3] = {64, (cuuint64_t)T, (cuuint64_t)H}, s_r[2] = {(cuuint64_t)H * 64 * e2, 64 * e2};
        if (!bg_map(&pmn, 3, pb, d_mat, s_mat, box_mn) || !bg_map(&damn, 3, dab, d_mat, s_mat, box_mn) ||
            !bg_map(&dak, 3, dab, d_mat, s_mat, box_k) || !bg_map(&dbk, 4, dbb, d_db4, s_db4, box_k4) ||
            !bg_map(&dbmn, 4, dbb, d_db4, s_db4, box_mn4) || !bg_map(&mdo, 3, dout, d_q, s_q, box_mn) ||
            !bg_map(&mqu, 3, qu, d_q, s_q, box_mn) || !bg_map(&mk, 3, k, d_k, s_q, box_mn) ||
            !bg_map(&mr, 3, r, d_r, s_r, box_mn) || !bg_map(&mqv, 3, qv, d_q, s_q, box_mn))
            return TXL_ERR_CUDA;
        const BgOperand o3{3, 0}, o3h{3, 1}, o4{4, 0};
        auto run = [&](const CUtensorMap &a, const BgOperand &ao, const CUtensorMap &b, const BgOperand &bo, int a_mn,
                       long K, int M, int nz, void *outp, long ostride, int ofp32, int oadd = 0) {
            BgParams g{};
            g.a[0] = ao;
            g.b[0] = bo;
            g.pairs = 1;
            g.a_mn = a_mn;
            g.ksteps[0] = (int)((K + BG_K - 1) / BG_K);
            g.M = M;
            g.nz = nz;
            g.H = H;
            g.out = outp;
            g.ostride = ostride;
            g.ofp32 = ofp32;
            g.oadd = oadd;
            return launch_bwd_gemm(&a, &b, g, s);
        };
        const long ld64 = BH * 64;
        if ((e = run(pmn, o3, mdo, o3, 1, L, (int)T, (int)BH, dv, ld64, 0)) != cudaSuccess ||
            (e = run(damn, o3, mqu, o3, 1, L, (int)T, (int)BH, dk, ld64, 0)) != cudaSuccess ||
            (e = run(dak, o3, mk, o3, 0, T, L, (int)BH, dqc, ld64, 1)) != cudaSuccess ||
            (e = run(dbk, o4, mr, o3h, 0, T, L, (int)BH, dqp, ld64, 1)) != cudaSuccess ||
            (e = cudaMemsetAsync(dracc, 0, (size_t)T * H * 64 * 4, s)) != cudaSuccess ||
            (e = run(dbmn, o4, mqv, o3, 1, L, (int)T, (int)BH, dracc, (long)H * 64, 1, 1)) != cudaSuccess)
            goto cuda_fail;
        // dr (bf16) from its fp32 batch sum
        bwd_round_kernel<<<grid_for(T * H * 64 / 4, 256), 256, 0, s>>>(dracc, (E *)dr, T * H * 64 / 4);
        if (!chk()) goto cuda_fail;
    }
    // dq and the bias gradients in one pass over the two fp32 halves of dq
    if ((e = launch_sum_bias<E>(dqc, dqp, (E *)dq, du, dw, (long)L * B, H * D, s)) != cudaSuccess) goto cuda_fail;
    return TXL_OK;
cuda_fail:
    note_cuda_error(e);
    return TXL_ERR_CUDA;
}

bool fused_ok(int d_head, const void *const *ptrs, int n)
{
    if (d_head != 64) return false;
    for (int x = 0; x < n; ++x)
        if ((uintptr_t)ptrs[x] & 15) return false;
    return true;
}

txl_status check_sizes(int batch, int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (batch < 1 || mem_len < 0 || seg_len < 1 || heads < 1 || d_head < 1) return TXL_ERR_INVALID;
    if (d_head > 128) return TXL_ERR_UNSUPPORTED;
    const long T = (long)mem_len + seg_len;
    // GEMM dimensions and leading dimensions are int; batch counts index a grid dimension
    if (T > INT32_MAX || (long)batch * heads * d_head > INT32_MAX || (long)batch * heads > 65535)
        return TXL_ERR_UNSUPPORTED;
    return TXL_OK;
}

}  // namespace

cudaError_t read_and_clear_bwd_error(unsigned int *word, cudaStream_t s)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_bwd_err, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_bwd_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace txl

using namespace txl;

extern "C" {

txl_status txl_rel_attn_bwd_workspace(int batch, int mem_len, int seg_len, int heads, int d_head,
                                      txl_dtype dtype, size_t *bytes)
{
    if (!bytes) return TXL_ERR_INVALID;
    const txl_status st = check_sizes(batch, mem_len, seg_len, heads, d_head, dtype);
    if (st != TXL_OK) return st;
    size_t n = layout(batch, heads, d_head, seg_len, mem_len, dtype == TXL_F32 ? 4 : 2).total;
    if (dtype == TXL_BF16 && d_head == 64) {
        // the fused path when the operands are 16-byte aligned (else the materialised one)
        const size_t f = layout_fused(batch, heads, d_head, seg_len, mem_len).total;
        n = f > n ? f : n;
    }
    *bytes = n;
    return TXL_OK;
}

txl_status txl_rel_attn_bwd(const void *q, const void *k, const void *v, const void *r, const float *u_bias,
                            const float *v_bias, const void *dout, const void *out, const float *lse, int batch,
                            int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype, void *dq, void *dk,
                            void *dv, void *dr, float *du, float *dw, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    const txl_status st = check_sizes(batch, mem_len, seg_len, heads, d_head, dtype);
    if (st != TXL_OK) return st;
    if (!q || !k || !v || !r || !dout || !dq || !dk || !dv || !dr || !workspace) return TXL_ERR_INVALID;
    const size_t es = dtype == TXL_F32 ? 4 : 2;
    const Ws lay = layout(batch, heads, d_head, seg_len, mem_len, es);
    size_t need = lay.total;
    if (dtype == TXL_BF16 && d_head == 64) {
        const size_t f = layout_fused(batch, heads, d_head, seg_len, mem_len).total;
        need = f > need ? f : need;
    }
    if (workspace_bytes < need || ((uintptr_t)workspace & 255)) return TXL_ERR_INVALID;
    const void *ins[] = {q, k, v, r, dout, dq, dk, dv, dr};
    for (const void *x : ins)
        if ((uintptr_t)x % es) return TXL_ERR_INVALID;
    // the forward's saved output and row log-sum-exp come together or not at all
    if ((out == nullptr) != (lse == nullptr)) return TXL_ERR_INVALID;
    if (out && (((uintptr_t)out & 15) || ((uintptr_t)lse & 3))) return TXL_ERR_INVALID;
    if (((uintptr_t)u_bias & 3) || ((uintptr_t)v_bias & 3) || ((uintptr_t)du & 3) || ((uintptr_t)dw & 3))
        return TXL_ERR_INVALID;
    const long T = (long)mem_len + seg_len;
    const size_t nq = (size_t)seg_len * batch * heads * d_head * es, nk = (size_t)T * batch * heads * d_head * es;
    const size_t nr = (size_t)T * heads * d_head * es, nb = (size_t)heads * d_head * 4;
    // outputs must not overlap the inputs, each other or the workspace
    const void *outs[] = {dq, dk, dv, dr, du, dw};
    const size_t osz[] = {nq, nk, nk, nr, nb, nb};
    const size_t nl = (size_t)batch * heads * seg_len * 4;
    const void *rd[] = {q, k, v, r, dout, u_bias, v_bias, workspace, out, lse};
    const size_t rsz[] = {nq, nk, nk, nr, nq, nb, nb, need, nq, nl};
    for (int a = 0; a < 6; ++a) {
        for (int b = 0; b < 10; ++b)
            if (overlaps(outs[a], osz[a], rd[b], rsz[b])) return TXL_ERR_INVALID;
        for (int b = a + 1; b < 6; ++b)
            if (overlaps(outs[a], osz[a], outs[b], osz[b])) return TXL_ERR_INVALID;
    }
    for (int b = 0; b < 10; ++b)
        if (b != 7 && overlaps(workspace, need, rd[b], rsz[b])) return TXL_ERR_INVALID;
    // absent biases: the zero vector (their gradients are still reported when asked)
    const float *uu = u_bias, *ww = v_bias;
    if (!uu || !ww) {
        const float *z = nullptr;
        const cudaError_t ze = zero_bias((size_t)heads * d_head, &z);
        if (ze == cudaErrorNotSupported) return TXL_ERR_UNSUPPORTED;
        if (ze != cudaSuccess) {
            note_cuda_error(ze);
            return TXL_ERR_CUDA;
        }
        if (!uu) uu = z;
        if (!ww) ww = z;
    }
    cudaStream_t s = (cudaStream_t)stream;
    unsigned char *wsb = (unsigned char *)workspace;
    if (dtype == TXL_F32)
        return run_bwd<float>(q, k, v, r, uu, ww, dout, batch, mem_len, seg_len, heads, d_head, dq, dk, dv, dr, du,
                              dw, wsb, lay, s, false);
    // the tensor-core route reads its operands by TMA and writes dk, dv, dr
    // with 16-byte stores: every one of them 16-byte aligned
    const void *al[] = {q, k, v, r, dout, uu, ww, dk, dv, dr};
    if (fused_ok(d_head, al, 10))
        return run_bwd_fused(q, k, v, r, uu, ww, dout, out, lse, batch, mem_len, seg_len, heads, d_head, dq, dk, dv,
                             dr, du, dw, wsb, layout_fused(batch, heads, d_head, seg_len, mem_len), s);
    return run_bwd<__nv_bfloat16>(q, k, v, r, uu, ww, dout, batch, mem_len, seg_len, heads, d_head, dq, dk, dv, dr,
                                  du, dw, wsb, lay, s, true);
}

}  // extern "C"
