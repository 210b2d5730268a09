// project.cu -- the rest of a layer's attention inputs, written straight into
// the layout the attention kernels read (Transformer-XL, Section 3.3):
//
//   txl_project_heads: y[rows][heads][d_pad] = x[rows][d_in] . W^T with W the
//     paper's [heads*d_head][d_in] projection (q = h W_q^T, k = h~ W_kE^T,
//     v = h~ W_v^T); with rows = positions x batch of a T-major [T][B][d_model]
//     buffer the result is the T-major [T][B][H][d_pad] layout, padding
//     columns d_head..d_pad-1 exactly zero.  bf16: a persistent tcgen05 GEMM
//     (128 x up to 256 output tiles, fp32 accumulation in TMEM, operands
//     staged by TMA or, for rows TMA cannot address, by 4-byte cp.async, a
//     double-buffered accumulator so that a tile's epilogue overlaps the
//     next tile's MMAs, output by TMA store); fp32 and odd shapes: a tiled
//     CUDA-core kernel.
//   txl_rel_table: r[t][h][d] = sum_c R[T-1-t][c] W_kR[h*d_head + d][c], the
//     reversed projected table of Appendix B, with R the sinusoid encoding of
//     the relative distance (row p: sin / cos of p * 10000^(-2c/d_model)).
//     Computed once per layer (it does not depend on the batch or on the
//     segment); the sinusoid is evaluated in the kernel, fp32 accumulation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "sm100.cuh"
#include "txl.h"

namespace txl {

// bounded waits of the projection kernel that gave up (read by txl_check)
__device__ unsigned int g_gemm_err;

namespace {
using namespace sm100;

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

// =========================================================================
// tcgen05 projection GEMM (bf16 in, fp32 accumulation, bf16 out)
//
// D[m][c] = sum_k x[m][k] W[row(c)][k] over output columns c of the padded
// head layout: c = h*d_pad + d is W's row h*d_head + d when d < d_head, a
// zero row otherwise.  Both operands are K-major (rows of 64 K-elements =
// 128 bytes, the 128-byte swizzle), so the MMA is the plain A.B^T form.
// Roles (eight warps, one CTA per SM, persistent over 128 x bn tiles):
//   warp 0     TMA producer (one thread), or with warps 2 and 3 the
//              cp.async loaders when TMA cannot address the rows;
//   warp 1     one thread issues the MMAs (four K=16 steps per stage);
//   warps 4-7  epilogue: TMEM -> registers -> bf16 -> swizzled staging (two
//              buffers per warp) -> TMA store (32 rows x 64 columns per warp
//              and chunk).
// TMEM: two 256-column accumulators (tile i's epilogue overlaps tile i+1).
constexpr int GM = 128;           // output rows per tile (TMEM lanes)
constexpr int GK = 64;            // K elements per stage (one swizzled row)
constexpr int GNT = 256;          // threads
constexpr int GLOADERS = 96;      // cp.async loader threads (warps 0, 2, 3)
constexpr uint64_t GWAIT_NS = 2000000000ull;   // 2 s per wait, then give up

// Two shapes of the kernel: TMA operands with 256-wide tiles and four
// stages, one CTA per SM; cp.async operands (issue-bound loaders) with
// 128-wide tiles and two stages, two CTAs per SM so that one CTA's loaders
// run while the other's wait.
template <int BN_, int ST_>
struct GemmSmem {
    static constexpr int GBN = BN_;                           // widest output tile
    static constexpr int GST = ST_;                           // pipeline stages
    static constexpr uint32_t ASZ = GM * 128;                 // one stage of x: 16 KB
    static constexpr uint32_t BSZ = GBN * 128;                // one stage of W
    static constexpr uint32_t A = 0;
    static constexpr uint32_t B = A + GST * ASZ;
    static constexpr uint32_t OST = B + GST * BSZ;            // 4 epilogue warps x 2 x 4 KB staging
    static constexpr uint32_t BOFF = OST + 8 * 4096;          // W row offsets of a tile, per loader warp
    static constexpr uint32_t BARS = BOFF + 3 * 128 * 4;
    static constexpr int FULL = 0, EMPTY = GST, AFULL = 2 * GST, AEMPTY = 2 * GST + 2, DONE = 2 * GST + 4,
                         NBAR = 2 * GST + 5;
    static constexpr uint32_t MISC = BARS + NBAR * 8;          // tmem holder, abort flag
    static constexpr uint32_t TOTAL = MISC + 16 + 1024;        // + alignment of the base to 1024
};
using SmemTma = GemmSmem<256, 4>;
using SmemCpa = GemmSmem<128, 2>;
static_assert(SmemTma::TOTAL <= 232448 && 2 * (SmemCpa::TOTAL + 1024) <= 233472, "shared memory");

// Up to three products of the same x in one launch (q, k, v of a layer):
// segment s multiplies x by its own W and writes its own output, over the
// row blocks from seg_fb[s] on (seg_fb non-decreasing), output row = x row -
// seg_row0[s].  One segment is the plain y = x W^T.  When q's first row
// (seg_row0[2]) does not start a row block, q is not a nested segment but
// a band of its own after the others: qa_blocks 128-row blocks from x row
// seg_row0[2] on (nseg is then 2).  A launch can also take
// several such cells of one shape (the layer calls of one step that do not
// depend on each other), each with its own x, weights and outputs: tile t
// belongs to cell t / tiles_cell.
constexpr int GSEG = 3;
constexpr int GCELLS = 8;         // cells per launch of the grouped variant
struct GemmParams {
    const __nv_bfloat16 *x, *w;
    __nv_bfloat16 *out;
    int rows, d_in, heads, d_head, d_pad, n_out;
    int bn, tiles_n, tiles, ksteps;   // tiles_n: column tiles of one segment
    int tma_out;
    int nseg, row_blocks;
    int seg_fb[GSEG], seg_row0[GSEG];
    int qa_blocks;                    // row blocks of q's own band (0: none)
    int tiles_cell, ncell;            // tiles of one cell, cells in the launch
};
template <int NC>
struct GemmMapsN {
    CUtensorMap x[NC], w[NC][GSEG], o[NC][GSEG];
};
using GemmMaps = GemmMapsN<1>;

// Tile t of the launch: the row blocks fall into bands [seg_fb[b],
// seg_fb[b+1]) in which segments 0..b are active; within a row block the
// tiles run over the active segments' column tiles, so neighbouring CTAs
// read the same x rows.
struct GTile {
    int m0, seg, n0, cell;
};
template <int NC>
__host__ __device__ __forceinline__ GTile gemm_tile(const GemmParams &p, int t)
{
    int cell = 0;
    if (NC > 1) {
        cell = t / p.tiles_cell;
        t -= cell * p.tiles_cell;
    }
#pragma unroll
    for (int b = 0; b < GSEG; ++b) {   // unrolled: the fields are indexed by constants
        if (b >= p.nseg) break;
        const int end = b + 1 < p.nseg ? p.seg_fb[b + 1 < GSEG ? b + 1 : b] : p.row_blocks;
        const int per = (b + 1) * p.tiles_n;
        const int cnt = (end - p.seg_fb[b]) * per;
        if (t < cnt) {
            const int r = t % per;
            return {(p.seg_fb[b] + t / per) * GM, r / p.tiles_n, (r % p.tiles_n) * p.bn, cell};
        }
        t -= cnt;
    }
    if (t < p.qa_blocks * p.tiles_n)   // q's own band, its blocks from its first row
        return {p.seg_row0[2] + (t / p.tiles_n) * GM, 2, (t % p.tiles_n) * p.bn, cell};
    return {-1, 0, 0, cell};
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <bool kTmaIn, typename S, int kMinBlocks, int NC>
__global__ void __launch_bounds__(GNT, kMinBlocks)
project_gemm_kernel(const __grid_constant__ GemmMapsN<NC> maps, const GemmParams p)
{
    constexpr int GST = S::GST, GBN = S::GBN;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + S::BARS + 8u * (uint32_t)i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::MISC + 8);
    // bounded wait; gives up when another role has given up
    auto wait = [&](int i, uint32_t parity) -> bool {
        const uint32_t b = bar(i);
        if (mbar_try_wait(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            if (mbar_try_wait_sleep(b, parity, WAIT_SLEEP_NS)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > GWAIT_NS) {
                *abort = 1;
                atomicOr(&g_gemm_err, 1u);
                return false;
            }
        }
    };

    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 2 * GBN);
        tmem_relinquish();
    }
    if (tid == 0) {
        *abort = 0;
        for (int s = 0; s < GST; ++s) {
            mbar_init(bar(S::FULL + s), kTmaIn ? 1 : GLOADERS);
            mbar_init(bar(S::EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(S::AFULL + b), 1);
            mbar_init(bar(S::AEMPTY + b), 128);
        }
        mbar_init(bar(S::DONE), 1);
        fence_mbar_init();
        if (kTmaIn) {
            for (int c = 0; c < NC && c < p.ncell; ++c) {
                prefetch_tmap(&maps.x[c]);
                for (int sg = 0; sg < (p.qa_blocks ? 3 : p.nseg); ++sg) prefetch_tmap(&maps.w[c][sg]);
            }
        }
        if (p.tma_out)
            for (int c = 0; c < NC && c < p.ncell; ++c)
                for (int sg = 0; sg < (p.qa_blocks ? 3 : p.nseg); ++sg) prefetch_tmap(&maps.o[c][sg]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int G = gridDim.x;

    if (warp == 1) {
        // =================================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(GM, p.bn, 0, 0);
            const uint64_t da0 = smem_desc_sw128(sbase + S::A, 16, 1024);
            const uint64_t db0 = smem_desc_sw128(sbase + S::B, 16, 1024);
            int it = 0, lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.tiles; t += G, ++lt) {
                const int buf = lt & 1;
                // the accumulator was last read by the epilogue of tile lt-2
                if (lt >= 2 && !wait(S::AEMPTY + buf, ((lt >> 1) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(buf * GBN);
                for (int ks = 0; ks < p.ksteps; ++ks, ++it) {
                    const int s = it % GST;
                    if (!wait(S::FULL + s, (it / GST) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = da0 + ((uint64_t)(s * S::ASZ) >> 4), db = db0 + ((uint64_t)(s * S::BSZ) >> 4);
#pragma unroll
                    for (int k = 0; k < GK / 16; ++k)   // 32 bytes of the swizzled row per K step
                        mma_bf16_ss(acc, da + 2 * k, db + 2 * k, idesc, (ks > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar(S::EMPTY + s));
                }
                if (ok) mma_commit(bar(S::AFULL + buf));
            }
            // every MMA issued here has completed before the CTA winds down
            mma_commit(bar(S::DONE));
            wait(S::DONE, 0);
        }
        __syncwarp();
    } else if (warp == 0 || warp == 2 || warp == 3) {
        // =================================================================== operands
        if (kTmaIn) {
            if (warp == 0 && lane == 0) {
                const uint32_t bytes = (uint32_t)(GM * 128 + p.bn * 128);
                int it = 0;
                bool ok = true;
                for (int t = blockIdx.x; ok && t < p.tiles; t += G) {
                    const GTile tt = gemm_tile<NC>(p, t);
                    const int m0 = tt.m0, n0 = tt.n0;
                    const CUtensorMap *mw = &maps.w[tt.cell][tt.seg], *mx = &maps.x[tt.cell];
                    for (int ks = 0; ks < p.ksteps; ++ks, ++it) {
                        const int s = it % GST;
                        if (it >= GST && !wait(S::EMPTY + s, ((it / GST) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(S::FULL + s), bytes);
                        tma_load_2d(sbase + S::A + s * S::ASZ, mx, bar(S::FULL + s), ks * GK, m0);
                        // W viewed as [heads][d_head][d_in]: a box of bn / d_pad heads
                        // of d_pad rows each; rows d_head.. of a head are zero-filled
                        tma_load_3d(sbase + S::B + s * S::BSZ, mw, bar(S::FULL + s), ks * GK, 0, n0 / p.d_pad);
                    }
                }
            }
        } else {
            // 96 threads; warp wi (0..2) moves rows wi, wi+3, ... of both
            // operands, lane l the 4-byte word l of each row's 64 elements.
            // Per tile, each warp puts the element offsets of its W rows (-1:
            // a zero row) in a table of its own, so the stages do no index
            // division and the warps never wait on one another.
            const int wi = warp == 0 ? 0 : warp - 1;
            int *boff = reinterpret_cast<int *>(smem + S::BOFF) + wi * 128;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.tiles; t += G) {
                const GTile tt = gemm_tile<NC>(p, t);
                const int m0 = tt.m0, n0 = tt.n0;
                __syncwarp();                          // the previous tile's stages have read the table
                for (int j = lane; wi + 3 * j < p.bn; j += 32) {
                    const int col = n0 + wi + 3 * j, h = col / p.d_pad, d = col - h * p.d_pad;
                    boff[j] = (h < p.heads && d < p.d_head) ? (h * p.d_head + d) * p.d_in : -1;
                }
                __syncwarp();
                const long a_row0 = (long)(m0 + wi) * p.d_in;
                const long a_step = 3L * p.d_in;
                for (int ks = 0; ks < p.ksteps; ++ks, ++it) {
                    const int s = it % GST;
                    if (it >= GST && !wait(S::EMPTY + s, ((it / GST) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = sbase + S::A + s * S::ASZ, b_dst = sbase + S::B + s * S::BSZ;
                    const int kw = ks * GK + 2 * lane;
                    const bool kin = kw < p.d_in;      // d_in is even: the word is wholly in or out
                    const uint32_t cw = (uint32_t)(lane & 3) * 4u;     // byte within the 16-byte chunk
                    const uint32_t ch = (uint32_t)(lane >> 2);         // 16-byte chunk of the 128-byte row
                    const __nv_bfloat16 *ap = p.x + a_row0 + kw;
                    for (int r = wi; r < GM; r += 3, ap += a_step) {
                        const bool v = kin && m0 + r < p.rows;
                        cp_async4(a_dst + (uint32_t)r * 128u + ((ch ^ (uint32_t)(r & 7)) << 4) + cw, v ? ap : p.x, v);
                    }
                    for (int r = wi, j = 0; r < p.bn; r += 3, ++j) {
                        const int o = boff[j];
                        const bool v = kin && o >= 0;
                        cp_async4(b_dst + (uint32_t)r * 128u + ((ch ^ (uint32_t)(r & 7)) << 4) + cw,
                                  v ? p.w + o + kw : p.w, v);
                    }
                    cp_async_commit();
                    if (it > 0) {
                        // the previous stage's copies have landed: hand it to the MMA
                        cp_async_wait<1>();
                        fence_proxy_async_smem();
                        mbar_arrive(bar(S::FULL + (it - 1) % GST));
                    }
                }
            }
            cp_async_wait<0>();
            if (ok && it > 0) {
                fence_proxy_async_smem();
                mbar_arrive(bar(S::FULL + (it - 1) % GST));
            }
        }
    } else {
        // =================================================================== epilogue
        const int q = warp & 3;                      // TMEM lanes 32q .. 32q+31
        unsigned char *stg0 = smem + S::OST + (uint32_t)(warp - 4) * 8192u;
        const uint32_t stg0_a = sbase + S::OST + (uint32_t)(warp - 4) * 8192u;
        const int nch = (p.bn + 63) / 64;
        int lt = 0, nst = 0;                         // tiles, chunks stored (two staging buffers)
        for (int t = blockIdx.x; t < p.tiles; t += G, ++lt) {
            const int buf = lt & 1;
            const GTile tt = gemm_tile<NC>(p, t);
            const int m0 = tt.m0, n0 = tt.n0;
            const CUtensorMap *mo = &maps.o[tt.cell][tt.seg];
            const int orow = m0 - (tt.seg == 2 ? p.seg_row0[2] : tt.seg == 1 ? p.seg_row0[1] : p.seg_row0[0]) +
                             32 * q;   // this warp's first output row
            if (!wait(S::AFULL + buf, (lt >> 1) & 1)) break;
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * GBN);
            for (int c = 0; c < nch; ++c) {
                float v[64];
                tmem_ld32(tacc + 64u * c, *reinterpret_cast<float(*)[32]>(v));
                tmem_ld32(tacc + 64u * c + 32u, *reinterpret_cast<float(*)[32]>(v + 32));
                if (c == nch - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(S::AEMPTY + buf));   // the accumulator is free for tile lt+2
                }
                const int col0 = n0 + 64 * c;
                // padding columns come out exactly zero (whatever x holds)
                if (p.d_head != p.d_pad) {
                    int d = col0 % p.d_pad;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        if (d >= p.d_head) v[j] = 0.f;
                        if (++d == p.d_pad) d = 0;
                    }
                }
                if (p.tma_out) {
                    if (col0 >= p.n_out) continue;
                    unsigned char *stg = stg0 + (nst & 1) * 4096;
                    const uint32_t stg_a = stg0_a + (uint32_t)(nst & 1) * 4096u;
                    ++nst;
                    if (lane == 0) bulk_wait_read_1();   // the store before last has read this buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 pk;
                        pk.x = pack2_bf16(v[8 * j + 0], v[8 * j + 1]);
                        pk.y = pack2_bf16(v[8 * j + 2], v[8 * j + 3]);
                        pk.z = pack2_bf16(v[8 * j + 4], v[8 * j + 5]);
                        pk.w = pack2_bf16(v[8 * j + 6], v[8 * j + 7]);
                        *reinterpret_cast<uint4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = pk;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(mo, stg_a, col0, orow);   // rows / columns past the end are clipped
                        bulk_commit();
                    }
                } else {
                    const int row = m0 + 32 * q + lane;
                    if (row < p.rows) {
                        __nv_bfloat16 *o = p.out + (long)row * p.n_out;
                        for (int j = 0; j < 64; ++j)
                            if (col0 + j < p.n_out) o[col0 + j] = __float2bfloat16(v[j]);
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * GBN);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

// Encoded bf16 tensor maps with the 128-byte swizzle, cached by their
// arguments (an encode is a driver call that costs about a short launch).
struct GMap {
    int dev, rank;
    const void *base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    CUtensorMap map;
};
constexpr int GMAPS = 48;
std::mutex g_gmap_mu;
GMap g_gmaps[GMAPS];
int g_gmap_n = 0, g_gmap_next = 0;

bool gmap(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
          const cuuint32_t *box)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_gmap_mu);
    for (int i = 0; i < g_gmap_n; ++i) {
        const GMap &e = g_gmaps[i];
        bool same = e.dev == dev && e.rank == rank && e.base == base;
        for (int d = 0; same && d < rank; ++d) same = e.dims[d] == dims[d] && e.box[d] == box[d];
        for (int d = 0; same && d < rank - 1; ++d) same = e.strides[d] == strides[d];
        if (same) {
            *m = e.map;
            return true;
        }
    }
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    GMap &e = g_gmaps[g_gmap_next];
    e.dev = dev;
    e.rank = rank;
    e.base = base;
    for (int d = 0; d < 3; ++d) {
        e.dims[d] = d < rank ? dims[d] : 0;
        e.box[d] = d < rank ? box[d] : 0;
    }
    for (int d = 0; d < 2; ++d) e.strides[d] = d < rank - 1 ? strides[d] : 0;
    e.map = *m;
    g_gmap_next = (g_gmap_next + 1) % GMAPS;
    if (g_gmap_n < GMAPS) ++g_gmap_n;
    return true;
}

bool al(const void *p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }

template <bool kTmaIn, typename S, int kMinBlocks, int NC = 1>
cudaError_t launch_gemm_t(const GemmMapsN<NC> &maps, const GemmParams &p, cudaStream_t s)
{
    auto kern = project_gemm_kernel<kTmaIn, S, kMinBlocks, NC>;
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(opted.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::TOTAL);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_relaxed);
    }
    const long slots = (long)kMinBlocks * device_sm_count();
    const int grid = p.tiles < slots ? p.tiles : (int)slots;
    kern<<<(unsigned)grid, GNT, S::TOTAL, s>>>(maps, p);
    return cudaGetLastError();
}

// the shape fields of a launch and its single segment (y = x W^T, all rows)
void gemm_shape(GemmParams &p, int rows, int d_in, int heads, int d_head, int d_pad, int bn)
{
    p.rows = rows;
    p.d_in = d_in;
    p.heads = heads;
    p.d_head = d_head;
    p.d_pad = d_pad;
    p.n_out = heads * d_pad;
    p.bn = p.n_out >= bn ? bn : (p.n_out + 15) / 16 * 16;
    p.tiles_n = (p.n_out + p.bn - 1) / p.bn;
    p.ksteps = (d_in + GK - 1) / GK;
    p.row_blocks = (rows + GM - 1) / GM;
    p.nseg = 1;
    p.qa_blocks = 0;
    for (int sg = 0; sg < GSEG; ++sg) p.seg_fb[sg] = p.seg_row0[sg] = 0;
}

// q in the launch of k and v: a nested segment when its first row starts a
// row block (the three products then share x's row blocks), else a band of
// its own after k and v
void gemm_add_q(GemmParams &p, int q_row0)
{
    p.seg_row0[2] = q_row0;
    if (q_row0 % GM == 0) {
        p.nseg = 3;
        p.seg_fb[2] = q_row0 / GM;
    } else {
        p.nseg = 2;
        p.qa_blocks = (p.rows - q_row0 + GM - 1) / GM;
    }
}

// tiles of a launch: each band of row blocks times its active segments
bool gemm_count_tiles(GemmParams &p)
{
    long tiles = 0;
    for (int b = 0; b < p.nseg; ++b) {
        const int end = b + 1 < p.nseg ? p.seg_fb[b + 1] : p.row_blocks;
        tiles += (long)(end - p.seg_fb[b]) * (b + 1) * p.tiles_n;
    }
    tiles += (long)p.qa_blocks * p.tiles_n;
    if (tiles > INT32_MAX) return false;
    p.tiles = (int)tiles;
    p.tiles_cell = p.tiles;
    p.ncell = 1;
    return true;
}

// the tensor maps of one segment's W ([heads][d_head][d_in], a box of
// bn / d_pad whole heads of d_pad rows, rows d_head.. zero-filled) and
// output ([rows][n_out], 32-row x 64-column boxes)
bool gemm_wmap(CUtensorMap *m, const void *w, const GemmParams &p)
{
    const cuuint64_t dw[3] = {(cuuint64_t)p.d_in, (cuuint64_t)p.d_head, (cuuint64_t)p.heads};
    const cuuint64_t sw[2] = {(cuuint64_t)p.d_in * 2, (cuuint64_t)p.d_head * p.d_in * 2};
    const cuuint32_t bw[3] = {GK, (cuuint32_t)p.d_pad, (cuuint32_t)(p.bn / p.d_pad)};
    return gmap(m, 3, w, dw, sw, bw);
}
bool gemm_omap(CUtensorMap *m, void *out, int rows, const GemmParams &p)
{
    const cuuint64_t dO[2] = {(cuuint64_t)p.n_out, (cuuint64_t)rows}, sO[1] = {(cuuint64_t)p.n_out * 2};
    const cuuint32_t bO[2] = {64, 32};
    return gmap(m, 2, out, dO, sO, bO);
}
bool gemm_xmap(CUtensorMap *m, const void *x, const GemmParams &p)
{
    const cuuint64_t dx[2] = {(cuuint64_t)p.d_in, (cuuint64_t)p.rows}, sx[1] = {(cuuint64_t)p.d_in * 2};
    const cuuint32_t bx[2] = {GK, GM};
    return gmap(m, 2, x, dx, sx, bx);
}

// bf16 projection on the tensor cores: d_in even, x and w 4-byte aligned.
cudaError_t launch_project_gemm(const void *x, const void *w, void *out, int rows, int d_in, int heads, int d_head,
                                int d_pad, cudaStream_t s)
{
    GemmParams p;
    p.x = (const __nv_bfloat16 *)x;
    p.w = (const __nv_bfloat16 *)w;
    p.out = (__nv_bfloat16 *)out;
    // TMA addresses rows whose pitch is a multiple of 16 bytes; a W box holds
    // whole heads of d_pad rows
    const int bn_max = d_in % 8 == 0 && al(x, 16) && al(w, 16) ? SmemTma::GBN : SmemCpa::GBN;
    gemm_shape(p, rows, d_in, heads, d_head, d_pad, bn_max);
    const bool tma_in = bn_max == SmemTma::GBN && p.bn % d_pad == 0 && d_pad <= 256;
    p.tma_out = al(out, 16) && (p.n_out * 2) % 16 == 0;
    if (!tma_in && p.bn > SmemCpa::GBN) {   // TMA-able rows whose heads do not tile the box: 128-wide tiles
        p.bn = SmemCpa::GBN;
        p.tiles_n = (p.n_out + p.bn - 1) / p.bn;
    }
    if (!gemm_count_tiles(p)) return cudaErrorNotSupported;
    GemmMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (tma_in && (!gemm_xmap(&maps.x[0], x, p) || !gemm_wmap(&maps.w[0][0], w, p))) return cudaErrorInvalidValue;
    if (p.tma_out && !gemm_omap(&maps.o[0][0], out, rows, p)) return cudaErrorInvalidValue;
    return tma_in ? launch_gemm_t<true, SmemTma, 1>(maps, p, s) : launch_gemm_t<false, SmemCpa, 2>(maps, p, s);
}

// k = x W_k^T and v = x W_v^T over all rows and, when wq is given,
// q = x[q_row0..] W_q^T.  When every operand is TMA-addressable, the three
// come from one launch (q as a nested segment that shares x's row blocks
// when its first row starts a 128-row block, else as a band of its own);
// otherwise one launch per product.
cudaError_t launch_project_qkv(const void *x, int rows, int d_in, const void *wq, const void *wk, const void *wv,
                               void *q, void *k, void *v, int q_row0, int heads, int d_head, int d_pad,
                               cudaStream_t s)
{
    const bool with_q = wq != nullptr && rows > q_row0;
    const int n_out = heads * d_pad;
    GemmParams p;
    bool fused = d_in % 8 == 0 && al(x, 16) && al(wk, 16) && al(wv, 16) && al(k, 16) && al(v, 16) &&
                 (n_out * 2) % 16 == 0 && d_pad <= 256;
    if (fused) {
        gemm_shape(p, rows, d_in, heads, d_head, d_pad, SmemTma::GBN);
        fused = p.bn % d_pad == 0;
    }
    cudaError_t e = cudaSuccess;
    bool q_done = false;
    if (fused) {
        const bool q_in = with_q && al(wq, 16) && al(q, 16);
        p.x = (const __nv_bfloat16 *)x;
        p.w = (const __nv_bfloat16 *)wk;
        p.out = (__nv_bfloat16 *)k;
        p.tma_out = 1;
        p.nseg = 2;
        if (q_in) gemm_add_q(p, q_row0);
        if (!gemm_count_tiles(p)) return cudaErrorNotSupported;
        GemmMaps maps;
        memset(&maps, 0, sizeof(maps));
        if (!gemm_xmap(&maps.x[0], x, p) || !gemm_wmap(&maps.w[0][0], wk, p) || !gemm_wmap(&maps.w[0][1], wv, p) ||
            !gemm_omap(&maps.o[0][0], k, rows, p) || !gemm_omap(&maps.o[0][1], v, rows, p))
            return cudaErrorInvalidValue;
        if (q_in && (!gemm_wmap(&maps.w[0][2], wq, p) || !gemm_omap(&maps.o[0][2], q, rows - q_row0, p)))
            return cudaErrorInvalidValue;
        e = launch_gemm_t<true, SmemTma, 1>(maps, p, s);
        q_done = q_in;
    } else {
        e = launch_project_gemm(x, wk, k, rows, d_in, heads, d_head, d_pad, s);
        if (e == cudaSuccess) e = launch_project_gemm(x, wv, v, rows, d_in, heads, d_head, d_pad, s);
    }
    if (e == cudaSuccess && with_q && !q_done)
        e = launch_project_gemm((const __nv_bfloat16 *)x + (size_t)q_row0 * d_in, wq, q, rows - q_row0, d_in, heads,
                                d_head, d_pad, s);
    return e;
}

// Several layer calls' q, k, v projections of one shape in one launch
// (cells c = 0..n-1: k_c = x_c W_k,c^T, v_c = x_c W_v,c^T, q_c = x_c[q_row0..]
// W_q,c^T), when every operand is TMA-addressable; otherwise each cell as
// launch_project_qkv runs it.  Up to GCELLS cells per launch.
cudaError_t launch_project_qkv_cells(int n, const void *const *x, const void *const *wq, const void *const *wk,
                                     const void *const *wv, void *const *q, void *const *k, void *const *v,
                                     int rows, int d_in, int q_row0, int heads, int d_head, int d_pad, cudaStream_t s)
{
    const bool with_q = wq != nullptr && rows > q_row0;
    const int n_out = heads * d_pad;
    bool ok = d_in % 8 == 0 && (n_out * 2) % 16 == 0 && d_pad <= 256;
    for (int c = 0; ok && c < n; ++c) {
        ok = al(x[c], 16) && al(wk[c], 16) && al(wv[c], 16) && al(k[c], 16) && al(v[c], 16);
        if (with_q) ok = ok && al(wq[c], 16) && al(q[c], 16);
    }
    GemmParams p;
    if (ok) {
        gemm_shape(p, rows, d_in, heads, d_head, d_pad, SmemTma::GBN);
        ok = p.bn % d_pad == 0;
    }
    if (!ok || n < 2) {
        for (int c = 0; c < n; ++c) {
            const cudaError_t e = launch_project_qkv(x[c], rows, d_in, wq ? wq[c] : nullptr, wk[c], wv[c],
                                                     q ? q[c] : nullptr, k[c], v[c], q_row0, heads, d_head, d_pad, s);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    p.tma_out = 1;
    p.nseg = 2;
    if (with_q) gemm_add_q(p, q_row0);
    if (!gemm_count_tiles(p)) return cudaErrorNotSupported;
    const int per = p.tiles;
    for (int c0 = 0; c0 < n; c0 += GCELLS) {
        const int nc = n - c0 < GCELLS ? n - c0 : GCELLS;
        if ((long)per * nc > INT32_MAX) return cudaErrorNotSupported;
        p.x = (const __nv_bfloat16 *)x[c0];
        p.w = (const __nv_bfloat16 *)wk[c0];
        p.out = (__nv_bfloat16 *)k[c0];
        p.tiles_cell = per;
        p.tiles = per * nc;
        p.ncell = nc;
        GemmMapsN<GCELLS> maps;
        memset(&maps, 0, sizeof(maps));
        for (int c = 0; c < nc; ++c) {
            const int g = c0 + c;
            if (!gemm_xmap(&maps.x[c], x[g], p) || !gemm_wmap(&maps.w[c][0], wk[g], p) ||
                !gemm_wmap(&maps.w[c][1], wv[g], p) || !gemm_omap(&maps.o[c][0], k[g], rows, p) ||
                !gemm_omap(&maps.o[c][1], v[g], rows, p))
                return cudaErrorInvalidValue;
            if (with_q && (!gemm_wmap(&maps.w[c][2], wq[g], p) || !gemm_omap(&maps.o[c][2], q[g], rows - q_row0, p)))
                return cudaErrorInvalidValue;
        }
        const cudaError_t e = launch_gemm_t<true, SmemTma, 1, GCELLS>(maps, p, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// =========================================================================
// CUDA-core kernels (fp32, and bf16 shapes the tensor path does not take)
constexpr int TB_T = 32;     // rows per block
constexpr int TB_N = 64;     // output columns per block
constexpr int TB_K = 32;     // contraction slice staged per step

// y[m][c] = sum_k x[m][k] W[row(c)][k] for a 32-row x 64-column block of the
// padded output (c = h*d_pad + d, zero where d >= d_head)
template <typename T>
__global__ void __launch_bounds__(256)
project_simt_kernel(const T *__restrict__ x, const T *__restrict__ w, T *__restrict__ out, int rows, int d_in,
                    int heads, int d_head, int d_pad)
{
    __shared__ float xs[TB_T][TB_K + 1];
    __shared__ float ws[TB_K][TB_N + 1];
    const long m0 = (long)blockIdx.x * TB_T;
    const int n0 = blockIdx.y * TB_N;
    const int n_out = heads * d_pad;
    const int tid = threadIdx.x;
    const int tr = tid / 16, tc = tid % 16;    // rows tr, tr+16; columns tc + 16*c
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int k0 = 0; k0 < d_in; k0 += TB_K) {
        for (int i = tid; i < TB_T * TB_K; i += 256) {
            const long m = m0 + i / TB_K;
            const int k = k0 + i % TB_K;
            xs[i / TB_K][i % TB_K] = (m < rows && k < d_in) ? to_float(x[m * d_in + k]) : 0.f;
        }
        for (int i = tid; i < TB_K * TB_N; i += 256) {
            const int kk = i / TB_N, c = n0 + i % TB_N, k = k0 + kk;
            const int h = c / d_pad, d = c % d_pad;
            ws[kk][i % TB_N] = (k < d_in && c < n_out && d < d_head) ? to_float(w[((long)h * d_head + d) * d_in + k])
                                                                      : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < TB_K; ++kk) {
            const float a0 = xs[tr][kk], a1 = xs[tr + 16][kk];
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
        const long m = m0 + tr + 16 * rr;
        if (m >= rows) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = n0 + tc + 16 * c;
            if (n >= n_out) continue;
            out[m * n_out + n] = from_float<T>((n % d_pad) < d_head ? acc[rr][c] : 0.f);
        }
    }
}

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
            // W_kR in the paper's layout: row n (an output column), d_model inputs
            ws[kk][x % TB_N] = (c < d_model && n < ncols) ? to_float(w[(long)n * d_model + c]) : 0.f;
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

bool overlap_bytes(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

}  // namespace

cudaError_t read_and_clear_gemm_error(unsigned int *word, cudaStream_t s)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_gemm_err, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
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
    cudaError_t e;
    if (d_in == 0) {   // empty contraction: zeros
        e = cudaMemsetAsync(out, 0, nout, s);
    } else if (dtype == TXL_BF16 && d_in % 2 == 0 && al(x, 4) && al(w, 4) &&
               (long)heads * d_head * d_in <= INT32_MAX) {
        e = launch_project_gemm(x, w, out, rows, d_in, heads, d_head, d_pad, s);
    } else {
        const long n_out = (long)heads * d_pad;
        dim3 grid((unsigned)((rows + TB_T - 1) / TB_T), (unsigned)((n_out + TB_N - 1) / TB_N));
        if (grid.y > 65535) return TXL_ERR_UNSUPPORTED;
        if (dtype == TXL_F32)
            project_simt_kernel<float><<<grid, 256, 0, s>>>((const float *)x, (const float *)w, (float *)out, rows,
                                                            d_in, heads, d_head, d_pad);
        else
            project_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16 *)x,
                                                                    (const __nv_bfloat16 *)w, (__nv_bfloat16 *)out,
                                                                    rows, d_in, heads, d_head, d_pad);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return TXL_ERR_CUDA;
    }
    return TXL_OK;
}

txl_status txl_project_qkv(const void *x, int rows, int d_in, const void *w_q, const void *w_k, const void *w_v,
                           void *q, void *k, void *v, int q_row0, int heads, int d_head, int d_pad, txl_dtype dtype,
                           void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (rows < 0 || d_in < 0 || heads < 0 || d_head < 1 || d_pad < d_head) return TXL_ERR_INVALID;
    if ((w_q == nullptr) != (q == nullptr)) return TXL_ERR_INVALID;
    if (w_q && (q_row0 < 0 || q_row0 > rows)) return TXL_ERR_INVALID;
    if (rows == 0 || heads == 0) return TXL_OK;
    if (!x || !w_k || !w_v || !k || !v) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (!al(x, esz) || !al(w_k, esz) || !al(w_v, esz) || !al(k, esz) || !al(v, esz)) return TXL_ERR_INVALID;
    if (w_q && (!al(w_q, esz) || !al(q, esz))) return TXL_ERR_INVALID;
    if ((long)heads * d_pad > INT32_MAX || (long)heads * d_head > INT32_MAX) return TXL_ERR_UNSUPPORTED;
    // every output apart from x, the weights and the other outputs
    const size_t row_b = (size_t)heads * d_pad * esz, nw = (size_t)d_in * heads * d_head * esz;
    const size_t nx = (size_t)rows * d_in * esz, nkv = (size_t)rows * row_b;
    const size_t nq = w_q ? (size_t)(rows - q_row0) * row_b : 0;
    const void *outs[3] = {k, v, q};
    const size_t nout[3] = {nkv, nkv, nq};
    const void *ins[4] = {x, w_k, w_v, w_q};
    const size_t nin[4] = {nx, nw, nw, w_q ? nw : 0};
    for (int o = 0; o < 3; ++o) {
        if (nout[o] == 0) continue;
        for (int i = 0; i < 4; ++i)
            if (nin[i] && overlap_bytes(outs[o], nout[o], ins[i], nin[i])) return TXL_ERR_INVALID;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (nout[o2] && overlap_bytes(outs[o], nout[o], outs[o2], nout[o2])) return TXL_ERR_INVALID;
    }
    if (dtype == TXL_BF16 && d_in > 0 && d_in % 2 == 0 && al(x, 4) && al(w_k, 4) && al(w_v, 4) &&
        (!w_q || al(w_q, 4)) && (long)heads * d_head * d_in <= INT32_MAX) {
        const cudaError_t e = launch_project_qkv(x, rows, d_in, w_q, w_k, w_v, q, k, v, q_row0, heads, d_head,
                                                 d_pad, (cudaStream_t)stream);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return TXL_ERR_CUDA;
        }
        return TXL_OK;
    }
    // the three products one by one
    txl_status st = txl_project_heads(x, w_k, k, rows, d_in, heads, d_head, d_pad, dtype, stream);
    if (st == TXL_OK) st = txl_project_heads(x, w_v, v, rows, d_in, heads, d_head, d_pad, dtype, stream);
    if (st == TXL_OK && w_q && rows > q_row0)
        st = txl_project_heads((const unsigned char *)x + (size_t)q_row0 * d_in * esz, w_q, q, rows - q_row0, d_in,
                               heads, d_head, d_pad, dtype, stream);
    return st;
}

txl_status txl_project_qkv_cells(int cells, const void *const *x, const void *const *w_q, const void *const *w_k,
                                 const void *const *w_v, void *const *q, void *const *k, void *const *v, int rows,
                                 int d_in, int q_row0, int heads, int d_head, int d_pad, txl_dtype dtype, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (cells < 0 || rows < 0 || d_in < 0 || heads < 0 || d_head < 1 || d_pad < d_head) return TXL_ERR_INVALID;
    if ((w_q == nullptr) != (q == nullptr)) return TXL_ERR_INVALID;
    if (w_q && (q_row0 < 0 || q_row0 > rows)) return TXL_ERR_INVALID;
    if (cells == 0 || rows == 0 || heads == 0) return TXL_OK;
    if (!x || !w_k || !w_v || !k || !v) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if ((long)heads * d_pad > INT32_MAX || (long)heads * d_head > INT32_MAX) return TXL_ERR_UNSUPPORTED;
    const size_t row_b = (size_t)heads * d_pad * esz, nw = (size_t)d_in * heads * d_head * esz;
    const size_t nx = (size_t)rows * d_in * esz, nkv = (size_t)rows * row_b;
    const size_t nq = w_q ? (size_t)(rows - q_row0) * row_b : 0;
    for (int c = 0; c < cells; ++c) {
        if (!x[c] || !w_k[c] || !w_v[c] || !k[c] || !v[c]) return TXL_ERR_INVALID;
        if (w_q && (!w_q[c] || !q[c])) return TXL_ERR_INVALID;
        if (!al(x[c], esz) || !al(w_k[c], esz) || !al(w_v[c], esz) || !al(k[c], esz) || !al(v[c], esz))
            return TXL_ERR_INVALID;
        if (w_q && (!al(w_q[c], esz) || !al(q[c], esz))) return TXL_ERR_INVALID;
    }
    // every output apart from every input and every other output
    for (int c = 0; c < cells; ++c) {
        const void *outs[3] = {k[c], v[c], w_q ? q[c] : nullptr};
        const size_t nout[3] = {nkv, nkv, nq};
        for (int o = 0; o < 3; ++o) {
            if (!outs[o] || nout[o] == 0) continue;
            for (int c2 = 0; c2 < cells; ++c2) {
                const void *ins[4] = {x[c2], w_k[c2], w_v[c2], w_q ? w_q[c2] : nullptr};
                const size_t nin[4] = {nx, nw, nw, w_q ? nw : 0};
                for (int i = 0; i < 4; ++i)
                    if (ins[i] && nin[i] && overlap_bytes(outs[o], nout[o], ins[i], nin[i])) return TXL_ERR_INVALID;
                const void *outs2[3] = {k[c2], v[c2], w_q ? q[c2] : nullptr};
                for (int o2 = 0; o2 < 3; ++o2) {
                    if ((c2 == c && o2 == o) || !outs2[o2] || nout[o2] == 0) continue;
                    if (overlap_bytes(outs[o], nout[o], outs2[o2], nout[o2])) return TXL_ERR_INVALID;
                }
            }
        }
    }
    bool grouped = dtype == TXL_BF16 && d_in > 0 && d_in % 2 == 0 && (long)heads * d_head * d_in <= INT32_MAX;
    for (int c = 0; grouped && c < cells; ++c)
        grouped = al(x[c], 4) && al(w_k[c], 4) && al(w_v[c], 4) && (!w_q || al(w_q[c], 4));
    if (grouped) {
        const cudaError_t e = launch_project_qkv_cells(cells, x, w_q, w_k, w_v, q, k, v, rows, d_in, q_row0, heads,
                                                       d_head, d_pad, (cudaStream_t)stream);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return TXL_ERR_CUDA;
        }
        return TXL_OK;
    }
    for (int c = 0; c < cells; ++c) {
        const txl_status st = txl_project_qkv(x[c], rows, d_in, w_q ? w_q[c] : nullptr, w_k[c], w_v[c],
                                              w_q ? q[c] : nullptr, k[c], v[c], q_row0, heads, d_head, d_pad, dtype,
                                              stream);
        if (st != TXL_OK) return st;
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
