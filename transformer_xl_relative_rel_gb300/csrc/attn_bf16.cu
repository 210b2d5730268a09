// attn_bf16.cu -- fused bf16 relative attention on tcgen05 tensor cores.
//
// What is computed (Transformer-XL, Section 3.3, per-layer procedure):
//     s_ij = ((q_i+u).k_j + (q_i+v).Q_{L-1-i+j}) / sqrt(D),  j <= M+i,
//     out_i = softmax_j(s_ij) v_j,
// with Q the reversed projected table of Appendix B (row t = W_kR R_{T-1-t}).
//
// How (one CTA = 128 query rows of one (b, h), or one key-range split of them):
//   * q+u and q+v are formed once per CTA in fp32 and rounded to bf16 into two
//     shared-memory operand tiles (Section 3.3: u and v replace the per-query
//     position term of the absolute formulation).
//   * K, V and the table band are staged by TMA (one 4-D box each) in the
//     canonical no-swizzle K-major layout [d/8][rows][8].
//   * Content term: S = (q+u) K^T, one 128x128 tcgen05 MMA chain into TMEM.
//   * Position term, Appendix B: B~ = (q+v) Q_band^T over the 256 table rows
//     that the tile's pairs touch; the left shift of row i by L-1-i is pure
//     index arithmetic: row ii of the tile reads B~ column 127-ii+jj.  TMEM
//     loads are warp-uniform in the column, so each warp loads the 64-column
//     window its 32 rows need and every thread aligns its own row with a
//     5-stage register barrel shift by 31-lane.  The shifted matrix is never
//     materialised in memory.
//   * Mask j <= M+i, scale and online softmax in the log2 domain, one query
//     row per thread (row reductions stay inside the thread), P rounded to
//     bf16 into shared memory, O += P V as a tcgen05 MMA accumulating in TMEM,
//     O rescaled in TMEM when the running max grows.
//   * Epilogue: O / l to bf16 in global memory, or, when the keys are split
//     across CTAs (long memories), normalised partials plus their log-sum-exp
//     for the combine kernel below.
// Every mbarrier wait is bounded; on expiry the kernel records an error word
// (read by txl_check) and winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace txl {

__device__ unsigned int g_err_word;

namespace {
using namespace sm100;

constexpr int BM = 128;          // query rows per CTA (TMEM lanes)
constexpr int BN = 128;          // keys per tile
constexpr int RWIN = 256;        // table rows of a tile's band (BM+BN-1, rounded up)
constexpr int NT = 128;          // threads per CTA
constexpr uint32_t TM_S = 0;     // TMEM columns: S (fp32, then the scaled logits)
constexpr uint32_t TM_B = 128;   //               B~ band (256 columns)
constexpr uint32_t TM_O = 384;   //               O accumulator (DP <= 64 columns)
constexpr uint32_t TM_COLS = 512;
constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s per wait, then give up
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16 *q, *k, *v, *r;
    const float *u, *w;
    __nv_bfloat16 *out;
    float *part_o;      // [splits][B*H][L][DP] when splits > 1
    float *part_lse;    // [splits][B*H][L]
    int B, H, D, L, M, T;
    int nqt, splits;
    float sl2;          // log2(e) / sqrt(D)
};

template <int DP>
struct Smem {
    static constexpr uint32_t Q_BYTES = BM * DP * 2;
    static constexpr uint32_t K_BYTES = BN * DP * 2;
    static constexpr uint32_t R_BYTES = RWIN * DP * 2;
    static constexpr uint32_t P_BYTES = BM * BN * 2;
    static constexpr uint32_t QU = 0;
    static constexpr uint32_t QV = QU + Q_BYTES;
    static constexpr uint32_t KS = QV + Q_BYTES;
    static constexpr uint32_t VS = KS + K_BYTES;
    static constexpr uint32_t RS = VS + K_BYTES;
    static constexpr uint32_t PS = RS + R_BYTES;
    static constexpr uint32_t BARS = PS + P_BYTES;       // 6 mbarriers
    static constexpr uint32_t TMEM_HOLDER = BARS + 64;
    // at least 120 KB so that only one CTA fits on an SM: each CTA takes all
    // 512 TMEM columns
    static constexpr uint32_t USED = TMEM_HOLDER + 16;
    static constexpr uint32_t TOTAL = USED > 120 * 1024 ? USED : 120 * 1024;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void record_error(unsigned int code) { atomicOr(&g_err_word, code); }

// Cooperative (all 128 threads) load of `nrows` rows of D bf16 elements into
// the [d/8][nrows][8] layout, rows outside [0, limit) and columns >= D zero.
// Used when D is not a multiple of 8 (rows are then not 16-byte aligned and
// TMA cannot address them).
template <int DP>
__device__ __forceinline__ void load_rows_generic(unsigned char *dst, int nrows,
                                                  const __nv_bfloat16 *src, long row0_elems,
                                                  long row_stride, int first_row, int limit, int D)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int rr = warp; rr < nrows; rr += NT / 32) {
        const int row = first_row + rr;
        const bool ok = row >= 0 && row < limit;
        const __nv_bfloat16 *p = src + row0_elems + (long)row * row_stride;
#pragma unroll
        for (int d0 = 0; d0 < DP; d0 += 32) {
            const int d = d0 + lane;
            if (d < DP) {
                __nv_bfloat16 x = __float2bfloat16(0.f);
                if (ok && d < D) x = p[d];
                *reinterpret_cast<__nv_bfloat16 *>(dst + (d >> 3) * (nrows * 16) + rr * 16 +
                                                   (d & 7) * 2) = x;
            }
        }
    }
}

template <int DP, bool kTma>
__global__ void __launch_bounds__(NT, 1)
rel_attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_r, const Params p)
{
    using S = Smem<DP>;
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- which (b, h, query tile, key split) this CTA owns; late (heavier)
    // query tiles first so that the causal tail is not left for the last wave
    const int per_bh = p.nqt * p.splits;
    const int bh = blockIdx.x / per_bh;
    const int rem = blockIdx.x % per_bh;
    const int qt = p.nqt - 1 - rem / p.splits;
    const int split = rem % p.splits;
    const int b = bh / p.H, h = bh % p.H;
    const int i0 = qt * BM;
    const int rows_here = min(BM, p.L - i0);
    const int kend = min(p.T, p.M + i0 + rows_here);      // keys this tile can see
    const int ntile = (kend + BN - 1) / BN;
    const int t0 = (int)(((long)split * ntile) / p.splits);
    const int t1 = (int)(((long)(split + 1) * ntile) / p.splits);
    const int ii = tid;                                    // this thread's row = TMEM lane
    const int i = i0 + ii;
    const bool row_valid = ii < rows_here;
    const long qkv_row = (long)p.B * p.H * p.D;            // elements between positions
    const long head_off = ((long)b * p.H + h) * p.D;

    if (t0 >= t1) {   // an empty key split for this tile: neutral partials
        if (row_valid) {
            const long prow = ((long)split * p.B * p.H + bh) * p.L + i;
            p.part_lse[prow] = -INFINITY;
            for (int d = 0; d < DP; ++d) p.part_o[prow * DP + d] = 0.f;
        }
        return;
    }

    unsigned char *qu_s = smem + S::QU, *qv_s = smem + S::QV, *k_s = smem + S::KS;
    unsigned char *v_s = smem + S::VS, *r_s = smem + S::RS, *p_s = smem + S::PS;
    const uint32_t bar_kr = smem_u32(smem + S::BARS), bar_v = bar_kr + 8, bar_mma = bar_kr + 16;
    const uint32_t bar_pv = bar_kr + 24;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::TMEM_HOLDER);

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_kr, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_pv, 1);
        fence_mbar_init();
        if (kTma) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_r);
        }
    }
    // padding slice (D rounded up to 16 for the MMA K dimension) must be zero:
    // TMA never writes it, and 0 * (stale NaN) would poison the sums
    if (kTma && (p.D & 15)) {
        const int s0 = p.D >> 3;   // first padding slice
        for (int x = tid; x < BN * 4; x += NT) {
            reinterpret_cast<uint32_t *>(k_s + s0 * BN * 16)[x] = 0u;
            reinterpret_cast<uint32_t *>(v_s + s0 * BN * 16)[x] = 0u;
        }
        for (int x = tid; x < RWIN * 4; x += NT)
            reinterpret_cast<uint32_t *>(r_s + s0 * RWIN * 16)[x] = 0u;
    }

    // ---- q+u and q+v for this thread's row, rounded once to bf16
    {
        float qrow[DP];
#pragma unroll
        for (int d = 0; d < DP; ++d) qrow[d] = 0.f;
        if (row_valid) {
            const __nv_bfloat16 *qp = p.q + (long)i * qkv_row + head_off;
            if ((p.D & 7) == 0) {
#pragma unroll
                for (int d8 = 0; d8 < DP / 8; ++d8) {
                    if (d8 * 8 < p.D) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(qp + d8 * 8);
                        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
                        for (int z = 0; z < 8; ++z) qrow[d8 * 8 + z] = __bfloat162float(e[z]);
                    }
                }
            } else {
#pragma unroll
                for (int d = 0; d < DP; ++d)
                    if (d < p.D) qrow[d] = __bfloat162float(qp[d]);
            }
        }
        const float *up = p.u + h * p.D, *wp = p.w + h * p.D;
#pragma unroll
        for (int d8 = 0; d8 < DP / 8; ++d8) {
            uint32_t a[4], c[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int d = d8 * 8 + 2 * z;
                const bool in0 = row_valid && d < p.D, in1 = row_valid && d + 1 < p.D;
                const float u0 = in0 ? up[d] : 0.f, u1 = in1 ? up[d + 1] : 0.f;
                const float w0 = in0 ? wp[d] : 0.f, w1 = in1 ? wp[d + 1] : 0.f;
                a[z] = pack_bf16(qrow[d] + u0, qrow[d + 1] + u1);
                c[z] = pack_bf16(qrow[d] + w0, qrow[d + 1] + w1);
            }
            *reinterpret_cast<uint4 *>(qu_s + d8 * (BM * 16) + ii * 16) = make_uint4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<uint4 *>(qv_s + d8 * (BM * 16) + ii * 16) = make_uint4(c[0], c[1], c[2], c[3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);   // this warp's lanes

    const uint32_t kr_bytes = (uint32_t)(BN + RWIN) * (uint32_t)(p.D / 8) * 16u;
    const uint32_t v_bytes = (uint32_t)BN * (uint32_t)(p.D / 8) * 16u;
    const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
    const uint32_t idesc_b = idesc_bf16(BM, RWIN, 0, 0);
    const uint32_t idesc_o = idesc_bf16(BM, DP, 0, 1);   // V is MN-major (d contiguous)
    const uint32_t a_qu = smem_u32(qu_s), a_qv = smem_u32(qv_s), a_k = smem_u32(k_s);
    const uint32_t a_v = smem_u32(v_s), a_r = smem_u32(r_s), a_p = smem_u32(p_s);

    if (kTma && tid == 0) {
        const int j0 = t0 * BN, kb = p.L - BM - i0 + j0;
        mbar_arrive_expect_tx(bar_kr, kr_bytes);
        tma_load_4d(a_k, &tm_k, bar_kr, 0, j0, 0, bh);
        tma_load_4d(a_r, &tm_r, bar_kr, 0, kb, 0, h);
    }

    uint32_t ph_kr = 0, ph_v = 0, ph_mma = 0, ph_pv = 0;
    float m_run = -INFINITY, l_run = 0.f;
    bool fail = false;

    for (int t = t0; t < t1; ++t) {
        const int j0 = t * BN;
        const int kb = p.L - BM - i0 + j0;     // first table row of the band
        if (!kTma) {
            if (t > t0) {                       // previous P.V done: V and P free
                fail |= !mbar_wait(bar_pv, ph_pv, WAIT_NS);
                ph_pv ^= 1;
            }
            load_rows_generic<DP>(k_s, BN, p.k, head_off, qkv_row, j0, p.T, p.D);
            load_rows_generic<DP>(v_s, BN, p.v, head_off, qkv_row, j0, p.T, p.D);
            load_rows_generic<DP>(r_s, RWIN, p.r, (long)h * p.D, (long)p.H * p.D, kb, p.T, p.D);
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(fail)) break;
            tc_fence_after();
        }
        // ---- content and position MMAs (one thread issues)
        if (tid == 0) {
            bool ok = true;
            if (kTma) {
                ok = mbar_wait(bar_kr, ph_kr, WAIT_NS);
                ph_kr ^= 1;
            }
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < DP / 16; ++ks) {
                    mma_bf16_ss(tmem + TM_S, smem_desc(a_qu + ks * 2 * BM * 16, BM * 16, 128),
                                smem_desc(a_k + ks * 2 * BN * 16, BN * 16, 128), idesc_s, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < DP / 16; ++ks) {
                    mma_bf16_ss(tmem + TM_B, smem_desc(a_qv + ks * 2 * BM * 16, BM * 16, 128),
                                smem_desc(a_r + ks * 2 * RWIN * 16, RWIN * 16, 128), idesc_b, ks > 0);
                }
                mma_commit(bar_mma);
            } else {
                fail = true;
            }
        }
        __syncwarp();
        if (__syncthreads_or(fail)) break;
        fail |= !mbar_wait(bar_mma, ph_mma, WAIT_NS);
        ph_mma ^= 1;
        tc_fence_after();
        if (kTma && tid == 0 && !fail) {
            // the commit above also covers the previous P.V, so V is free
            mbar_arrive_expect_tx(bar_v, v_bytes);
            tma_load_4d(a_v, &tm_v, bar_v, 0, j0, 0, bh);
            if (t + 1 < t1) {   // K and the band are consumed: prefetch the next tile
                mbar_arrive_expect_tx(bar_kr, kr_bytes);
                tma_load_4d(a_k, &tm_k, bar_kr, 0, j0 + BN, 0, bh);
                tma_load_4d(a_r, &tm_r, bar_kr, 0, kb + BN, 0, h);
            }
        }
        __syncwarp();
        if (__syncthreads_or(fail)) break;

        // ---- pass 1: align the position term, add, mask, scale; keep in TMEM
        const int lim = row_valid ? (p.M + i - j0) : (p.T - 1 - j0);   // visible iff jj <= lim
        const int shift = 31 - lane;
        float tmax = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float s[32], a[64];
            const int base = 96 - 32 * warp + 32 * c;   // window of this warp's rows
            tmem_ld32(tlane + TM_S + 32 * c, s);
            tmem_ld32(tlane + TM_B + base, *reinterpret_cast<float(*)[32]>(&a[0]));
            tmem_ld32(tlane + TM_B + base + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
#pragma unroll
            for (int x = 0; x < 48; ++x) a[x] = (shift & 16) ? a[x + 16] : a[x];
#pragma unroll
            for (int x = 0; x < 40; ++x) a[x] = (shift & 8) ? a[x + 8] : a[x];
#pragma unroll
            for (int x = 0; x < 36; ++x) a[x] = (shift & 4) ? a[x + 4] : a[x];
#pragma unroll
            for (int x = 0; x < 34; ++x) a[x] = (shift & 2) ? a[x + 2] : a[x];
#pragma unroll
            for (int x = 0; x < 32; ++x) a[x] = (shift & 1) ? a[x + 1] : a[x];
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                float val = (s[x] + a[x]) * p.sl2;
                val = (32 * c + x <= lim) ? val : -INFINITY;
                tmax = fmaxf(tmax, val);
                s[x] = val;
            }
            tmem_st32(tlane + TM_S + 32 * c, s);
        }
        tmem_wait_st();

        // ---- pass 2: probabilities to shared memory (bf16), running sums
        const float m_new = fmaxf(m_run, tmax);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_use);
        float sum = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float x[32];
            tmem_ld32(tlane + TM_S + 32 * c, x);
            uint32_t pk[16];
#pragma unroll
            for (int y = 0; y < 16; ++y) {
                const float p0 = ex2(x[2 * y] - m_use), p1 = ex2(x[2 * y + 1] - m_use);
                sum += p0 + p1;
                pk[y] = pack_bf16(p0, p1);
            }
#pragma unroll
            for (int z = 0; z < 4; ++z)
                *reinterpret_cast<uint4 *>(p_s + (4 * c + z) * (BM * 16) + ii * 16) =
                    make_uint4(pk[4 * z], pk[4 * z + 1], pk[4 * z + 2], pk[4 * z + 3]);
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        // ---- rescale the accumulator when the running max moved
        if (t > t0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll
            for (int c = 0; c < DP / 16; ++c) {
                float o[16];
                tmem_ld16(tlane + TM_O + 16 * c, o);
#pragma unroll
                for (int x = 0; x < 16; ++x) o[x] *= alpha;
                tmem_st16(tlane + TM_O + 16 * c, o);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) break;

        // ---- O += P V
        if (tid == 0) {
            bool ok = true;
            if (kTma) {
                ok = mbar_wait(bar_v, ph_v, WAIT_NS);
                ph_v ^= 1;
            }
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    mma_bf16_ss(tmem + TM_O, smem_desc(a_p + kk * 2 * BM * 16, BM * 16, 128),
                                smem_desc(a_v + kk * 16 * 16, 128, BN * 16), idesc_o,
                                (t > t0 || kk > 0) ? 1u : 0u);
                }
                if (!kTma) mma_commit(bar_pv);
            } else {
                fail = true;
            }
        }
        __syncwarp();
    }

    // ---- wait for the last P.V, then the epilogue
    if (__syncthreads_or(fail)) {
        record_error(1u);
    } else {
        if (tid == 0) mma_commit(bar_mma);
        __syncwarp();
        if (!mbar_wait(bar_mma, ph_mma, WAIT_NS)) {
            record_error(2u);
            fail = true;
        }
        tc_fence_after();
    }
    if (!__syncthreads_or(fail)) {
        float o[DP];
#pragma unroll
        for (int c = 0; c < DP / 16; ++c) tmem_ld16(tlane + TM_O + 16 * c, *reinterpret_cast<float(*)[16]>(&o[16 * c]));
        if (row_valid) {
            if (p.splits == 1) {
                const float inv = 1.f / l_run;
                __nv_bfloat16 *op = p.out + (long)i * qkv_row + head_off;
                if ((p.D & 7) == 0) {
#pragma unroll
                    for (int d8 = 0; d8 < DP / 8; ++d8) {
                        if (d8 * 8 < p.D) {
                            uint4 pk;
                            pk.x = pack_bf16(o[d8 * 8 + 0] * inv, o[d8 * 8 + 1] * inv);
                            pk.y = pack_bf16(o[d8 * 8 + 2] * inv, o[d8 * 8 + 3] * inv);
                            pk.z = pack_bf16(o[d8 * 8 + 4] * inv, o[d8 * 8 + 5] * inv);
                            pk.w = pack_bf16(o[d8 * 8 + 6] * inv, o[d8 * 8 + 7] * inv);
                            *reinterpret_cast<uint4 *>(op + d8 * 8) = pk;
                        }
                    }
                } else {
#pragma unroll
                    for (int d = 0; d < DP; ++d)
                        if (d < p.D) op[d] = __float2bfloat16(o[d] * inv);
                }
            } else {
                const long prow = ((long)split * p.B * p.H + bh) * p.L + i;
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * DP);
#pragma unroll
                for (int d4 = 0; d4 < DP / 4; ++d4)
                    po[d4] = make_float4(o[4 * d4] * inv, o[4 * d4 + 1] * inv, o[4 * d4 + 2] * inv,
                                         o[4 * d4 + 3] * inv);
                p.part_lse[prow] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// Merge the key-split partials of one (b, h, i) row: weights 2^(lse_s - max).
__global__ void __launch_bounds__(64)
rel_attn_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                        __nv_bfloat16 *__restrict__ out, int splits, int B, int H, int L, int D,
                        int DP)
{
    const int row = blockIdx.x;           // over B*H*L
    const int bh = row / L, i = row % L;
    const int b = bh / H, h = bh % H;
    const long BHL = (long)B * H * L;
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_lse[s * BHL + (long)bh * L + i]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f, wsum = 0.f;
        for (int s = 0; s < splits; ++s) {
            const long prow = s * BHL + (long)bh * L + i;
            const float lse = part_lse[prow];
            const float wgt = (lse == -INFINITY) ? 0.f : exp2f(lse - mx);
            wsum += wgt;
            acc += wgt * part_o[prow * DP + d];
        }
        out[(((long)i * B + b) * H + h) * D + d] = __float2bfloat16(acc / wsum);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 4-D view {8, rows, D/8, groups} of a bf16 tensor whose rows are `row_stride`
// elements apart and whose groups (b*H+h or h) are D elements apart; the box
// {8, box_rows, D/8, 1} lands in shared memory as [d/8][box_rows][8].
bool make_map(CUtensorMap *m, const void *base, long rows, long row_stride, int D, long groups,
              int box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {8, (cuuint64_t)rows, (cuuint64_t)(D / 8), (cuuint64_t)groups};
    cuuint64_t strides[3] = {(cuuint64_t)row_stride * 2, 16, (cuuint64_t)D * 2};
    cuuint32_t box[4] = {8, (cuuint32_t)box_rows, (cuuint32_t)(D / 8), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int DP, bool kTma>
cudaError_t launch_t(const Params &p, const CUtensorMap &mk, const CUtensorMap &mv,
                     const CUtensorMap &mr, cudaStream_t s)
{
    const uint32_t smem = Smem<DP>::TOTAL;
    auto kern = rel_attn_bf16_kernel<DP, kTma>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long grid = (long)p.B * p.H * p.nqt * p.splits;
    kern<<<(unsigned)grid, NT, smem, s>>>(mk, mv, mr, p);
    return cudaGetLastError();
}

int dpad(int D) { return (D + 15) / 16 * 16; }

}  // namespace

int bf16_num_splits(const AttnArgs &a, int num_sms)
{
    const int nqt = (a.L + BM - 1) / BM;
    const long ctas = (long)a.B * a.H * nqt;
    const int ntile = (a.M + a.L + BN - 1) / BN;     // key tiles of the last query tile
    // choose the split count that minimises (waves x tiles per split), with a
    // small charge for the combine pass; 1 when the grid already fills the GPU
    double best = 1e30;
    int best_s = 1;
    for (int s = 1; s <= 16 && s <= ntile; ++s) {
        const long waves = (ctas * s + num_sms - 1) / num_sms;
        const int per = (ntile + s - 1) / s;
        const double cost = (double)waves * per + (s > 1 ? 1.0 : 0.0);
        if (cost < best - 1e-9) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

size_t bf16_scratch_bytes(const AttnArgs &a, int splits)
{
    const size_t rows = (size_t)splits * a.B * a.H * a.L;
    return rows * (size_t)dpad(a.D) * 4 + rows * 4 + 256;
}

cudaError_t launch_attn_bf16(const AttnArgs &a, int splits, void *scratch, cudaStream_t s)
{
    const int DP = dpad(a.D);
    if (DP > 64) return cudaErrorNotSupported;
    Params p;
    p.q = (const __nv_bfloat16 *)a.q;
    p.k = (const __nv_bfloat16 *)a.k;
    p.v = (const __nv_bfloat16 *)a.v;
    p.r = (const __nv_bfloat16 *)a.r;
    p.u = a.u;
    p.w = a.w;
    p.out = (__nv_bfloat16 *)a.out;
    p.B = a.B;
    p.H = a.H;
    p.D = a.D;
    p.L = a.L;
    p.M = a.M;
    p.T = a.M + a.L;
    p.nqt = (a.L + BM - 1) / BM;
    p.splits = splits;
    p.sl2 = LOG2E / sqrtf((float)a.D);
    p.part_o = nullptr;
    p.part_lse = nullptr;
    if (splits > 1) {
        const size_t rows = (size_t)splits * a.B * a.H * a.L;
        p.part_o = (float *)scratch;
        p.part_lse = (float *)((char *)scratch + rows * DP * 4);
    }
    CUtensorMap mk, mv, mr;
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
    memset(&mr, 0, sizeof(mr));
    const bool tma = (a.D % 8) == 0;
    if (tma) {
        const long bhn = (long)a.B * a.H;
        const long rs = bhn * a.D;
        if (!make_map(&mk, a.k, p.T, rs, a.D, bhn, BN) || !make_map(&mv, a.v, p.T, rs, a.D, bhn, BN) ||
            !make_map(&mr, a.r, p.T, (long)a.H * a.D, a.D, a.H, RWIN))
            return cudaErrorInvalidValue;
    }
    cudaError_t e;
    switch (DP) {
    case 16: e = tma ? launch_t<16, true>(p, mk, mv, mr, s) : launch_t<16, false>(p, mk, mv, mr, s); break;
    case 32: e = tma ? launch_t<32, true>(p, mk, mv, mr, s) : launch_t<32, false>(p, mk, mv, mr, s); break;
    case 48: e = tma ? launch_t<48, true>(p, mk, mv, mr, s) : launch_t<48, false>(p, mk, mv, mr, s); break;
    default: e = tma ? launch_t<64, true>(p, mk, mv, mr, s) : launch_t<64, false>(p, mk, mv, mr, s); break;
    }
    if (e != cudaSuccess || splits == 1) return e;
    rel_attn_combine_kernel<<<(unsigned)((long)a.B * a.H * a.L), 64, 0, s>>>(
        p.part_o, p.part_lse, p.out, splits, a.B, a.H, a.L, a.D, DP);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(unsigned int *word, cudaStream_t s)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_err_word, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace txl
