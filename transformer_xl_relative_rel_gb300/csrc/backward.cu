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
//     five strided-batched cuBLAS GEMMs give dV, dK, both halves of dQ and
//     dr (dr summed over the batch by the contraction itself), and one pass
//     adds the halves of dQ and forms du, dv_bias as its column sums;
//   - otherwise (fp32, other head sizes: run_bwd) the materialised form: the
//     score, P, dP and dA of every (b, h) are written to the caller's
//     workspace as [L][T] matrices, the eight plain contractions run as
//     strided-batched cuBLAS GEMMs (bf16 operands and fp32 accumulation on
//     the bf16 path; fp32 throughout on the fp32 path), and the kernels below
//     do the bias fold, the softmax, its gradient and both shifts, and the
//     batch / row reductions of dq, du, dv_bias and dr.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "txl.h"

namespace txl {
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
// is a multiple of the chunk: one index decomposition per chunk.
template <typename T>
__global__ void bwd_fold_vec_kernel(const T *__restrict__ q, const float *__restrict__ u,
                                    const float *__restrict__ w, T *__restrict__ qu, T *__restrict__ qv, long nch,
                                    int H, int D)
{
    constexpr int C = 16 / sizeof(T);
    const int dc = D / C;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < nch; x += (long)gridDim.x * blockDim.x) {
        const int d0 = (int)(x % dc) * C, h = (int)((x / dc) % H);
        const uint4 raw = reinterpret_cast<const uint4 *>(q)[x];
        const T *e = reinterpret_cast<const T *>(&raw);
        uint4 a, b;
        T *ea = reinterpret_cast<T *>(&a), *eb = reinterpret_cast<T *>(&b);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float qq = to_f(e[c]);
            ea[c] = from_f<T>(qq + u[h * D + d0 + c]);
            eb[c] = from_f<T>(qq + w[h * D + d0 + c]);
        }
        reinterpret_cast<uint4 *>(qu)[x] = a;
        reinterpret_cast<uint4 *>(qv)[x] = b;
    }
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
// element strides; ta: A is stored k x m (used transposed), tb: B is stored
// n x k.  cuBLAS sees the column-major transpose C^T = op(B)^T op(A)^T.
cublasStatus_t gemm_rm(cublasHandle_t hd, bool ta, bool tb, int m, int n, int k, const void *A, long lda,
                       long long sA, const void *Bm, long ldb, long long sB, void *C, long ldc, long long sC,
                       int batch, cudaDataType_t tab, cudaDataType_t tc)
{
    const float one = 1.f, zero = 0.f;
    return cublasGemmStridedBatchedEx(hd, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, n, m, k,
                                      &one, Bm, tab, (int)ldb, sB, A, tab, (int)lda, sA, &zero, C, tc, (int)ldc,
                                      sC, batch, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
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
    size_t pb, da, db, qu, qv, dqc, dqp, out, lse, split, total;
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
    const cudaDataType_t ty = bf16 ? CUDA_R_16BF : CUDA_R_32F;
    E *qu = (E *)(ws + lay.qu), *qv = (E *)(ws + lay.qv), *rrep = (E *)(ws + lay.rrep);
    E *pb = (E *)(ws + lay.pb), *dab = (E *)(ws + lay.da), *dbb = (E *)(ws + lay.db);
    float *x1 = (float *)(ws + lay.x1), *x2 = (float *)(ws + lay.x2);
    float *dqc = (float *)(ws + lay.dqc), *dqp = (float *)(ws + lay.dqp), *drp = (float *)(ws + lay.drp);
    cublasHandle_t hd = (cublasHandle_t)blas_on_stream(s);
    if (!hd) return TXL_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    auto chk = [&]() {
        e = cudaGetLastError();
        return e == cudaSuccess;
    };
    if (D % (16 / (int)sizeof(E)) == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)r & 15) == 0) {
        const int C = 16 / (int)sizeof(E);
        bwd_fold_vec_kernel<E><<<grid_for(nq / C, 256), 256, 0, s>>>((const E *)q, u, w, qu, qv, nq / C, H, D);
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
        if (gemm_rm(hd, false, true, L, Ti, D, qu, ld, D, k, ld, D, x1, T, LT, nb, ty, CUDA_R_32F) ||
            gemm_rm(hd, false, true, L, Ti, D, qv, ld, D, rrep, D, TD, x2, T, LT, nb, ty, CUDA_R_32F))
            return TXL_ERR_CUDA;
        if (T <= RB * 6)
            bwd_softmax_row_kernel<E, 6><<<(unsigned)rows, RB, 0, s>>>(x1, x2, pb, L, M, Ti, scale);
        else if (T <= RB * 16)
            bwd_softmax_row_kernel<E, 16><<<(unsigned)rows, RB, 0, s>>>(x1, x2, pb, L, M, Ti, scale);
        else
            bwd_softmax_kernel<E><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x1, x2, pb, rows, L, M, Ti, scale);
        if (!chk()) goto cuda_fail;
        // dP, then the score gradient in both frames
        if (gemm_rm(hd, false, true, L, Ti, D, dout, ld, D, v, ld, D, x2, T, LT, nb, ty, CUDA_R_32F))
            return TXL_ERR_CUDA;
        if (T <= RB * 6)
            bwd_score_grad_row_kernel<E, 6><<<(unsigned)rows, RB, 0, s>>>(x1, x2, dab, dbb, L, M, Ti, scale);
        else if (T <= RB * 16)
            bwd_score_grad_row_kernel<E, 16><<<(unsigned)rows, RB, 0, s>>>(x1, x2, dab, dbb, L, M, Ti, scale);
        else
            bwd_score_grad_kernel<E><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(x1, x2, dab, dbb, rows, L, M,
                                                                                Ti, scale);
        if (!chk()) goto cuda_fail;
        // dV = P^T dO, dK = dA^T qu, dQ = dA K + dB~ r, dr per (b, h) = dB~^T qv
        if (gemm_rm(hd, true, false, Ti, D, L, pb, T, LT, dout, ld, D, dv, ld, D, nb, ty, ty) ||
            gemm_rm(hd, true, false, Ti, D, L, dab, T, LT, qu, ld, D, dk, ld, D, nb, ty, ty) ||
            gemm_rm(hd, false, false, L, D, Ti, dab, T, LT, k, ld, D, dqc, ld, D, nb, ty, CUDA_R_32F) ||
            gemm_rm(hd, false, false, L, D, Ti, dbb, T, LT, rrep, D, TD, dqp, ld, D, nb, ty, CUDA_R_32F) ||
            gemm_rm(hd, true, false, Ti, D, L, dbb, T, LT, qv, ld, D, drp, D, TD, nb, ty, CUDA_R_32F))
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
    const long T = (long)M + L, BH = (long)B * H, nq = (long)L * BH * D, ld = BH * D, TP = lay.TP;
    E *qu = (E *)(ws + lay.qu), *qv = (E *)(ws + lay.qv);
    E *pb = (E *)(ws + lay.pb), *dab = (E *)(ws + lay.da), *dbb = (E *)(ws + lay.db), *outf = (E *)(ws + lay.out);
    float *lse = (float *)(ws + lay.lse);
    float *dqc = (float *)(ws + lay.dqc), *dqp = (float *)(ws + lay.dqp);
    cublasHandle_t hd = (cublasHandle_t)blas_on_stream(s);
    if (!hd) return TXL_ERR_CUDA;
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
    bwd_fold_vec_kernel<E><<<grid_for(nq / 8, 256), 256, 0, s>>>((const E *)q, u, w, qu, qv, nq / 8, H, D);
    if (!chk()) goto cuda_fail;
    {
        const long long LTP = (long long)L * TP, LBTP = (long long)L * B * TP;
        const int Ti = (int)T, nb = (int)BH, LB = L * B, HD = H * D;
        // per (b, h): dV = P^T dO, dK = dA^T qu, dQ (content) = dA K; per head
        // over the rows (i, b) of the head-major table-frame matrix dA~:
        // dQ (position) = dA~ r_h and dr_h = dA~^T qv, both straight into
        // their [.., H, D] layouts
        if (gemm_rm(hd, true, false, Ti, D, L, pb, TP, LTP, dout, ld, D, dv, ld, D, nb, CUDA_R_16BF, CUDA_R_16BF) ||
            gemm_rm(hd, true, false, Ti, D, L, dab, TP, LTP, qu, ld, D, dk, ld, D, nb, CUDA_R_16BF, CUDA_R_16BF) ||
            gemm_rm(hd, false, false, L, D, Ti, dab, TP, LTP, k, ld, D, dqc, ld, D, nb, CUDA_R_16BF, CUDA_R_32F) ||
            gemm_rm(hd, false, false, LB, D, Ti, dbb, TP, LBTP, r, HD, D, dqp, HD, D, H, CUDA_R_16BF, CUDA_R_32F) ||
            gemm_rm(hd, true, false, Ti, D, LB, dbb, TP, LBTP, qv, HD, D, dr, HD, D, H, CUDA_R_16BF, CUDA_R_16BF))
            return TXL_ERR_CUDA;
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
    // cuBLAS dimensions, leading dimensions and batch counts are int
    if (T > INT32_MAX || (long)batch * heads * d_head > INT32_MAX || (long)batch * heads > INT32_MAX)
        return TXL_ERR_UNSUPPORTED;
    return TXL_OK;
}

}  // namespace
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
    const void *al[] = {q, k, v, r, dout, uu, ww};
    if (fused_ok(d_head, al, 7))
        return run_bwd_fused(q, k, v, r, uu, ww, dout, out, lse, batch, mem_len, seg_len, heads, d_head, dq, dk, dv,
                             dr, du, dw, wsb, layout_fused(batch, heads, d_head, seg_len, mem_len), s);
    return run_bwd<__nv_bfloat16>(q, k, v, r, uu, ww, dout, batch, mem_len, seg_len, heads, d_head, dq, dk, dv, dr,
                                  du, dw, wsb, lay, s, true);
}

}  // extern "C"
