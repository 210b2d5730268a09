// attn_f32.cu -- float32 relative attention (the 1e-4 parity path).
//
// Transformer-XL, Section 3.3: s_ij = ((q_i+u).k_j + (q_i+v).W_kR R_{i-j}) / sqrt(D)
// over keys j <= M+i of the extended context, softmax over j, times v_j.
// Appendix B: the relative table arrives reversed (row t = W_kR R_{T-1-t}), so
// the pair (i, j) reads table row L-1-i+j.  For a block of query rows
// i0..i0+31 and key tile j0..j0+31 those rows form one contiguous window of 63
// rows, staged once in shared memory: the per-row left shift of Appendix B is
// just the index 31-(i-i0)+(j-j0) into that window.
//
// SIMT only (FFMA, no tensor cores: TF32 would miss 1e-4).  One CTA of 128
// threads per (32 query rows, b, h); 4 threads per query row.  Online softmax
// (running max and sum per row), so keys stream through shared memory once.
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"

namespace txl {
namespace {

constexpr int BR = 32;       // query rows per CTA
constexpr int BC = 32;       // keys per tile
constexpr int NT = 128;      // threads per CTA (4 per query row)
constexpr int RW = BR + BC - 1;  // relative-table rows per tile

template <int DMAX>
__global__ void __launch_bounds__(NT)
rel_attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                    const float *__restrict__ v, const float *__restrict__ r,
                    const float *__restrict__ u, const float *__restrict__ w,
                    float *__restrict__ out, int B, int H, int D, int L, int M, int kv_start, int scale_d)
{
    extern __shared__ float smem[];
    const int DP = D + 1;                 // odd pitch: rows land in distinct banks
    float *qu = smem;                     // [BR][DP]  q + u
    float *qv = qu + BR * DP;             // [BR][DP]  q + v
    float *ks = qv + BR * DP;             // [BC][DP]
    float *vs = ks + BC * DP;             // [BC][DP]
    float *rs = vs + BC * DP;             // [RW][DP]  table window
    float *ps = rs + RW * DP;             // [BR][BC+1] probabilities

    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int i0 = blockIdx.y * BR;
    const int T = M + L;
    const long rowstride = (long)B * H * D;      // between positions in q/k/v/out
    const long hoff = ((long)b * H + h) * D;
    const int rows_here = min(BR, L - i0);
    const float scale = 1.0f / sqrtf((float)scale_d);   // d_head (D may be a padded width)

    // stage q+u and q+v for the block (rows past L are zero)
    for (int x = tid; x < BR * D; x += NT) {
        const int rr = x / D, d = x % D;
        float qq = 0.f, uu = 0.f, ww = 0.f;
        if (rr < rows_here) {
            qq = q[(long)(i0 + rr) * rowstride + hoff + d];
            uu = u[h * D + d];
            ww = w[h * D + d];
        }
        qu[rr * DP + d] = qq + uu;
        qv[rr * DP + d] = qq + ww;
    }

    const int rr = tid >> 2;            // this thread's query row in the block
    const int cg = tid & 3;             // its column group
    const int i = i0 + rr;
    const bool row_ok = rr < rows_here;
    float m_run = -INFINITY, l_run = 0.f;
    float o[DMAX / 4];
#pragma unroll
    for (int e = 0; e < DMAX / 4; ++e) o[e] = 0.f;

    const int kend = min(T, M + i0 + rows_here);   // keys any row of the block sees
    for (int j0 = 0; j0 < kend; j0 += BC) {
        __syncthreads();   // previous tile fully consumed
        const int tbase = L - BR - i0 + j0;         // first table row of the window
        for (int x = tid; x < BC * D; x += NT) {
            const int c = x / D, d = x % D;
            const int j = j0 + c;
            float kk = 0.f, vv = 0.f;
            if (j < T) {
                // K, V may form a ring: key j at row (kv_start + j) mod T
                const int sj = j + kv_start < T ? j + kv_start : j + kv_start - T;
                kk = k[(long)sj * rowstride + hoff + d];
                vv = v[(long)sj * rowstride + hoff + d];
            }
            ks[c * DP + d] = kk;
            vs[c * DP + d] = vv;
        }
        for (int x = tid; x < RW * D; x += NT) {
            const int t = x / D, d = x % D;
            const int row = tbase + t;
            rs[t * DP + d] = (row >= 0 && row < T) ? r[((long)row * H + h) * D + d] : 0.f;
        }
        __syncthreads();

        // scores for columns c = cg + 4m
        float s[BC / 4];
#pragma unroll
        for (int m = 0; m < BC / 4; ++m) s[m] = 0.f;
        for (int d = 0; d < D; ++d) {
            const float a = qu[rr * DP + d];
            const float p = qv[rr * DP + d];
#pragma unroll
            for (int m = 0; m < BC / 4; ++m) {
                const int c = cg + 4 * m;
                s[m] = fmaf(a, ks[c * DP + d], s[m]);
                s[m] = fmaf(p, rs[(BR - 1 - rr + c) * DP + d], s[m]);
            }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int m = 0; m < BC / 4; ++m) {
            const int j = j0 + cg + 4 * m;
            const bool vis = row_ok && j <= M + i && j < T;
            s[m] = vis ? s[m] * scale : -INFINITY;
            tmax = fmaxf(tmax, s[m]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);
        const bool any = m_new != -INFINITY;
        const float alpha = any ? expf(m_run - m_new) : 1.f;
        float psum = 0.f;
#pragma unroll
        for (int m = 0; m < BC / 4; ++m) {
            const float p = (s[m] == -INFINITY) ? 0.f : expf(s[m] - m_new);
            ps[rr * (BC + 1) + cg + 4 * m] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l_run = l_run * alpha + psum;
        m_run = m_new;
        __syncwarp();
        // o(row, d = cg + 4e) = alpha * o + sum_c p(row, c) v(c, d)
#pragma unroll
        for (int e = 0; e < DMAX / 4; ++e) {
            const int d = cg + 4 * e;
            if (d < D) {
                float acc = o[e] * alpha;
#pragma unroll 8
                for (int c = 0; c < BC; ++c) acc = fmaf(ps[rr * (BC + 1) + c], vs[c * DP + d], acc);
                o[e] = acc;
            }
        }
    }
    if (row_ok) {
        const float inv = 1.0f / l_run;
#pragma unroll
        for (int e = 0; e < DMAX / 4; ++e) {
            const int d = cg + 4 * e;
            if (d < D) out[(long)i * rowstride + hoff + d] = o[e] * inv;
        }
    }
}

template <int DMAX>
cudaError_t launch(const AttnArgs &a, cudaStream_t s)
{
    const int DP = a.D + 1;
    const size_t smem = sizeof(float) * ((size_t)(2 * BR + 2 * BC + RW) * DP + BR * (BC + 1));
    cudaError_t e = cudaFuncSetAttribute(rel_attn_f32_kernel<DMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, (a.L + BR - 1) / BR);
    rel_attn_f32_kernel<DMAX><<<grid, NT, smem, s>>>(
        (const float *)a.q, (const float *)a.k, (const float *)a.v, (const float *)a.r, a.u, a.w,
        (float *)a.out, a.B, a.H, a.D, a.L, a.M, a.kv_start, a.scale_d ? a.scale_d : a.D);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs &a, cudaStream_t s)
{
    if (a.D <= 32) return launch<32>(a, s);
    if (a.D <= 64) return launch<64>(a, s);
    return launch<128>(a, s);
}

}  // namespace txl
