// attn_bf16.cu -- fused bf16 relative attention on tcgen05 tensor cores.
//
// What is computed (Transformer-XL, Section 3.3, per-layer procedure):
//     s_ij = ((q_i+u).k_j + (q_i+v).Q_{L-1-i+j}) / sqrt(D),  j <= M+i,
//     out_i = softmax_j(s_ij) v_j,
// with Q the reversed projected table of Appendix B (row t = W_kR R_{T-1-t}).
//
// One CTA owns 128 query rows of one (b, h) -- or one key-range split of them
// -- and walks its keys in tiles of 64.  Six warps with fixed roles:
//   warp 0    producer: TMA loads of K, V and one 64-row chunk of the table
//             per tile into a seven-stage shared-memory ring, 128-byte rows
//             with the 128-byte swizzle (threads' coalesced loads for head
//             sizes other than 64);
//   warp 1    S-MMA issuer (one thread): per tile, S = (q+u) K^T into one of
//             three TMEM S buffers and the next band chunk B~ = (q+v) Q_chunk^T
//             into a 4-slot TMEM ring, as far ahead as the buffers allow;
//   warp 6    P.V issuer (one thread): O += P V as each tile's P arrives
//             (two issuers, so neither kind of MMA waits on the other's
//             barrier).  q+u, q+v, K, the table and V come from shared
//             memory, P is a TMEM A operand;
//   warps 2-5 softmax, one query row per thread (TMEM lane = row): each tile
//             is two independent 32-key halves; each half reads its S part
//             and the band window it needs, aligns the band to the row
//             (Appendix B's left shift of row i by L-1-i, done as a register
//             barrel shift by 31-lane; three stages as selects on the ALU,
//             two as exact arithmetic selects on the FMA pipe), adds, masks
//             j <= M+i, and runs the online softmax in the log2 domain.  P
//             (bf16) goes back into the S buffer's TMEM columns for P.V.
// Appendix B's table product is formed once per 64-row chunk: tile n uses
// chunks n, n+1, n+2 of the band, and computes chunk n+2 itself, so the
// position term costs the same tensor work as the content term.  The MMAs of
// the next tiles run while the softmax of tile n runs (three S buffers).
// The running max used for the exponentials is raised only when a row's max
// grows by more than 8 (log2 units); O in TMEM is rescaled only then.
// The scale log2(e)/sqrt(D) is folded into q+u and q+v before rounding.
// Every mbarrier wait is bounded; on expiry the CTA records an error word
// (read by txl_check) and every role winds down.
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

constexpr int BM = 128;           // query rows per CTA (TMEM lanes)
constexpr int BN = 64;            // keys per tile; also table rows per band chunk
constexpr int NCHUNK = 4;         // TMEM band-chunk ring
constexpr int NSTAGE = 5;         // shared-memory ring of (K, V, table chunk) tiles
constexpr int NT = 384;           // 12 warps, see the role list above
constexpr uint32_t TM_S = 0;      // two S buffers (one per softmax set) of 64 columns
constexpr uint32_t TM_BAND = 128; // band ring, 4 x 64 columns
constexpr uint32_t TM_O = 384;    // two O accumulators (one per set), 64 columns each
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t REG_LOW = 96, REG_HIGH = 200;     // per-thread registers after the split
static_assert(128 * REG_LOW + 256 * REG_HIGH <= 65536 / NT / 8 * 8 * NT, "register split exceeds the launch");
constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s per wait, then give up
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;          // raise the exponent base only past 2^8

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

// Every operand tile in shared memory uses 128-byte rows with the 128-byte
// swizzle (element (row, k) at sw128_offset(row, k)); D <= 64 fits one row.
template <int DP>
struct Smem {
    static constexpr uint32_t TILE = BN * 128;             // one K, V or table chunk
    static constexpr uint32_t STAGE = 3 * TILE;             // K, V, chunk
    static constexpr uint32_t ST0 = 0;                      // NSTAGE stages
    static constexpr uint32_t QU = NSTAGE * STAGE;          // q+u, q+v: 128 rows of 128 bytes
    static constexpr uint32_t QV = QU + BM * 128;
    static constexpr uint32_t PB = QV + BM * 128;           // P (bf16): two buffers per set, 128 rows x 128 bytes
    static constexpr uint32_t PRE = PB;                     // table chunks 0, 1 (read before any P is written)
    static constexpr uint32_t XML = PB + 4 * BM * 128;      // epilogue: [128 rows] (m, l) of set 1
    static constexpr uint32_t BARS = XML + BM * 8;
    // barrier slots (8 bytes each): stage full / empty; per softmax set: S
    // full, S free (read by the softmax), P full, O done; per P buffer: P.V
    // done; epilogue exchange
    static constexpr int B_Q = 0, B_PRE = 1, B_FULL = 2, B_EMPTY = 2 + NSTAGE,
                         B_S = 2 + 2 * NSTAGE, B_SF = B_S + 2, B_P = B_SF + 2, B_PV = B_P + 2,
                         B_O = B_PV + 4, B_X = B_O + 2;
    static constexpr uint32_t MISC = BARS + 32 * 8;         // tmem holder, abort flag
    static constexpr uint32_t USED = MISC + 16;
    // + 1 KB to align the base to the 1024-byte swizzle atom; at least 120 KB
    // so that only one CTA fits on an SM: each CTA takes all 512 TMEM columns
    static constexpr uint32_t TOTAL = USED + 1024 > 120 * 1024 ? USED + 1024 : 120 * 1024;
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

// two fp32 -> packed fp16 pair (lo = a), round to nearest, saturated to +-65504
__device__ __forceinline__ uint32_t pack_f16_sat(float a, float b)
{
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// x0 += fp16 low half of h, x1 += fp16 high half (one fp32 rounding each)
__device__ __forceinline__ void add_f16x2_to(float &x0, float &x1, uint32_t h)
{
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "r"(h));
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// packed pairs of fp32 (Blackwell f32x2 arithmetic: one instruction, two lanes of work)
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ void record_error(unsigned int code) { atomicOr(&g_err_word, code); }

// A bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > WAIT_NS) {
            *abort = 1;
            record_error(1u);
            return false;
        }
    }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Warp-cooperative load of `nrows` rows of D bf16 elements into the 128-byte
// swizzled row layout, for head sizes TMA does not load (D != 64; D not a
// multiple of 8 also leaves rows that are not 16-byte aligned).  Each row is read as aligned
// 32-bit words, one per lane (coalesced); a row that starts in the middle of a
// word is realigned with a funnel shift from the next lane's word.  Rows
// outside [0, limit) are written as zeros; element D (the first padding
// element, when D is odd) is written as zero; later padding was zeroed once.
__device__ __forceinline__ void warp_load_rows(unsigned char *dst, int nrows, const __nv_bfloat16 *src,
                                               long row0_elems, long row_stride, int first_row,
                                               int limit, int D, int lane)
{
    const int npairs = (D + 1) >> 1;     // element pairs covering D (<= 32 for D <= 64)
    // 16 rows at a time: all their loads are issued before any is used
    for (int r0 = 0; r0 < nrows; r0 += 16) {
        uint32_t w[16];
        int odd[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int row = first_row + r0 + k;
            const bool ok = row >= 0 && row < limit;
            const long e0 = row0_elems + (long)row * row_stride;    // first element of the row
            odd[k] = (int)(e0 & 1);
            // lane l reads word l of the row (elements 2l-odd .. 2l+1-odd);
            // only the words that overlap the row are read
            const uint32_t *wbase = reinterpret_cast<const uint32_t *>(src + (e0 & ~1L));
            w[k] = (ok && lane <= ((odd[k] + D - 1) >> 1)) ? wbase[lane] : 0u;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t wn = __shfl_down_sync(0xffffffffu, w[k], 1);
            uint32_t pair = odd[k] ? __byte_perm(w[k], wn, 0x5432) : w[k];   // elements 2l, 2l+1
            if (2 * lane + 1 == D) pair &= 0xFFFFu;                            // padding element
            if (lane < npairs) *reinterpret_cast<uint32_t *>(dst + sw128_offset(r0 + k, 2 * lane)) = pair;
        }
    }
}

template <int DP, bool kTma>
__global__ void __launch_bounds__(NT, 1)
rel_attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_r, const Params p)
{
    using S = Smem<DP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
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
    const int N = t1 - t0;                                 // key tiles of this CTA
    const long qkv_row = (long)p.B * p.H * p.D;            // elements between positions
    const long head_off = ((long)b * p.H + h) * p.D;
    const int kb0 = p.L - BM - i0 + t0 * BN;              // first table row of chunk 0

    if (N <= 0) {   // an empty key split for this tile: neutral partials
        if (tid < rows_here) {
            const long prow = ((long)split * p.B * p.H + bh) * p.L + i0 + tid;
            p.part_lse[prow] = -INFINITY;
            for (int d = 0; d < DP; ++d) p.part_o[prow * DP + d] = 0.f;
        }
        return;
    }

    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + S::BARS + 8u * (uint32_t)i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::MISC + 8);
    // every lane of a warp waits; the warp continues only if all of them saw
    // the barrier (keeps the warp converged for its collective instructions)
    auto wwait = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_or_abort(bar(i), parity, abort)) != 0;
    };

    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        *abort = 0;
        mbar_init(bar(S::B_Q), 128);
        mbar_init(bar(S::B_PRE), kTma ? 1 : 32);
        for (int x = 0; x < NSTAGE; ++x) {
            mbar_init(bar(S::B_FULL + x), kTma ? 1 : 64);
            mbar_init(bar(S::B_EMPTY + x), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(S::B_S + x), 1);
            mbar_init(bar(S::B_SF + x), 128);
            mbar_init(bar(S::B_P + x), 128);
            mbar_init(bar(S::B_PV + 2 * x), 1);
            mbar_init(bar(S::B_PV + 2 * x + 1), 1);
            mbar_init(bar(S::B_O + x), 1);
        }
        mbar_init(bar(S::B_X), 128);
        fence_mbar_init();
        if (kTma) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_r);
        }
    }
    // the padding of D up to a multiple of 16 (the MMA K step) must be zero in
    // every operand buffer, and loads never write it: clear everything once
    if (p.D != DP) {
        for (uint32_t x = tid; x < S::XML / 16; x += NT)
            reinterpret_cast<uint4 *>(smem)[x] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // warpgroup 0 (producer, issuers) gives registers to the two softmax
    // warpgroups: 128 x 96 + 256 x 200 <= 384 x 168 (the launch allocation)
    if (warp < 4) {
        setmaxnreg_dec<REG_LOW>();
        if (warp == 0 || (warp == 3 && !kTma)) {
            // =============================================================== producer
            // (without TMA: warp 0 loads K and the table chunks, warp 3 loads V)
            const uint32_t tile_bytes = (uint32_t)BN * 128u;     // TMA only for D = 64
            // table chunks 0 and 1 for the first tile
            if (kTma) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_PRE), 2 * tile_bytes);
                    tma_load_3d(sbase + S::PRE, &tm_r, bar(S::B_PRE), 0, kb0, h);
                    tma_load_3d(sbase + S::PRE + S::TILE, &tm_r, bar(S::B_PRE), 0, kb0 + BN, h);
                }
            } else if (warp == 0) {
                warp_load_rows(smem + S::PRE, BN, p.r, (long)h * p.D, (long)p.H * p.D, kb0, p.T, p.D, lane);
                warp_load_rows(smem + S::PRE + S::TILE, BN, p.r, (long)h * p.D, (long)p.H * p.D, kb0 + BN,
                               p.T, p.D, lane);
                fence_proxy_async_smem();
                mbar_arrive(bar(S::B_PRE));
            }
            for (int n = 0; n < N; ++n) {
                const int st = n % NSTAGE;
                // the stage is free once the P.V of tile n-NSTAGE (its last reader) is done
                if (n >= NSTAGE && !wwait(S::B_EMPTY + st, ((n / NSTAGE) - 1) & 1)) break;
                const int j0 = (t0 + n) * BN;
                const int crow = kb0 + (n + 2) * BN;     // table chunk n+2
                const uint32_t dst = sbase + S::ST0 + st * S::STAGE;
                if (kTma) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar(S::B_FULL + st), 3 * tile_bytes);
                        tma_load_3d(dst, &tm_k, bar(S::B_FULL + st), 0, j0, bh);
                        tma_load_3d(dst + S::TILE, &tm_v, bar(S::B_FULL + st), 0, j0, bh);
                        tma_load_3d(dst + 2 * S::TILE, &tm_r, bar(S::B_FULL + st), 0, crow, h);
                    }
                } else {
                    unsigned char *d = smem + S::ST0 + st * S::STAGE;
                    if (warp == 0) {
                        warp_load_rows(d, BN, p.k, head_off, qkv_row, j0, p.T, p.D, lane);
                        warp_load_rows(d + 2 * S::TILE, BN, p.r, (long)h * p.D, (long)p.H * p.D, crow, p.T,
                                       p.D, lane);
                    } else {
                        warp_load_rows(d + S::TILE, BN, p.v, head_off, qkv_row, j0, p.T, p.D, lane);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(bar(S::B_FULL + st));
                }
            }
        } else if (warp == 1) {
            // =============================================================== S / band MMAs
            // one thread waits and issues (no warp-wide votes on this path: the
            // issuing lane shares its scheduler with two softmax warps)
            if (lane == 0) {
                const uint32_t idesc_64 = idesc_bf16(BM, BN, 0, 0);
                bool ok = wait_or_abort(bar(S::B_Q), 0, abort) && wait_or_abort(bar(S::B_PRE), 0, abort);
                tc_fence_after();
                // descriptors built once; the 14-bit start-address field (address / 16)
                // advances by 2 per 32-byte K step within a 128-byte swizzled row
                const uint64_t d_qu = smem_desc_sw128(sbase + S::QU, 16, 1024);
                const uint64_t d_qv = smem_desc_sw128(sbase + S::QV, 16, 1024);
                const uint64_t d_pre = smem_desc_sw128(sbase + S::PRE, 16, 1024);
                const uint64_t d_st0 = smem_desc_sw128(sbase + S::ST0, 16, 1024);
                constexpr uint64_t STAGE16 = S::STAGE >> 4, TILE16 = S::TILE >> 4;
                if (ok) {
                    for (int c = 0; c < 2; ++c) {   // band chunks 0 and 1
#pragma unroll
                        for (int ks = 0; ks < DP / 16; ++ks)
                            mma_bf16_ss(tmem + TM_BAND + 64 * c, d_qv + 2 * ks, d_pre + c * TILE16 + 2 * ks,
                                        idesc_64, ks > 0);
                    }
                }
                for (int n = 0; ok && n < N; ++n) {
                    const int sb = n & 1, st = n % NSTAGE;
                    // S buffer sb was last read by the softmax of tile n-2, and band
                    // slot (n+2) % 4 by the softmaxes of tiles n-4..n-2: wait for
                    // tile n-2 here (tile n-3 was waited one iteration earlier)
                    if (n >= 2) ok = wait_or_abort(bar(S::B_SF + sb), ((n - 2) >> 1) & 1, abort);
                    ok = ok && wait_or_abort(bar(S::B_FULL + st), (n / NSTAGE) & 1, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dk = d_st0 + st * STAGE16, dc = dk + 2 * TILE16;
                    const uint32_t ts = tmem + TM_S + 64 * sb;
                    const uint32_t tb = tmem + TM_BAND + 64 * (uint32_t)((n + 2) % NCHUNK);
#pragma unroll
                    for (int ks = 0; ks < DP / 16; ++ks) mma_bf16_ss(ts, d_qu + 2 * ks, dk + 2 * ks, idesc_64, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < DP / 16; ++ks) mma_bf16_ss(tb, d_qv + 2 * ks, dc + 2 * ks, idesc_64, ks > 0);
                    mma_commit(bar(S::B_S + sb));
                }
            }
            __syncwarp();
        } else if (warp == 2) {
            // =============================================================== P.V MMAs
            if (lane == 0) {
                const uint32_t idesc_o = idesc_bf16(BM, DP, 0, 1);   // V is MN-major (d contiguous)
                const uint64_t d_st0 = smem_desc_sw128(sbase + S::ST0, 16, 1024);
                const uint64_t d_p0 = smem_desc_sw128(sbase + S::PB, 16, 1024);
                constexpr uint64_t STAGE16 = S::STAGE >> 4, TILE16 = S::TILE >> 4, PB16 = (BM * 128) >> 4;
                for (int n = 0; n < N; ++n) {
                    const int sb = n & 1, st = n % NSTAGE;
                    if (!wait_or_abort(bar(S::B_P + sb), (n >> 1) & 1, abort)) break;
                    tc_fence_after();
                    const uint64_t dv = d_st0 + st * STAGE16 + TILE16;   // 16 keys = 2048 bytes of V
                    const int pbuf = 2 * sb + ((n >> 1) & 1);              // P buffer of tile n
                    const uint64_t dp = d_p0 + pbuf * PB16;                // 16 keys = 32 bytes of P
                    const uint32_t to = tmem + TM_O + 64 * sb;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_bf16_ss(to, dp + 2 * kk, dv + 128 * kk, idesc_o, (n >= 2 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(S::B_PV + pbuf));
                    mma_commit(bar(S::B_EMPTY + st));
                    if (n + 2 >= N) mma_commit(bar(S::B_O + sb));   // last tile of this set
                }
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<REG_HIGH>();
        // =============================================================== softmax
        // two sets of four warps; set k takes the key tiles n = k, k+2, k+4, ...
        // with its own S buffer and O accumulator, so the two warps that share
        // a scheduler work on different tiles and their ALU and MUFU phases
        // overlap; the two partial results are merged once at the end
        const int set = (warp - 4) >> 2;
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int ii = quarter * 32 + lane;        // this thread's query row
        const int i = i0 + ii;
        const bool row_valid = ii < rows_here;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t ts = tl + TM_S + 64 * set, tb0 = tl + TM_BAND, to = tl + TM_O + 64 * set;

        if (set == 0) {
            // q+u and q+v, scaled by log2(e)/sqrt(D), rounded once to bf16, into
            // shared memory as the A operands of the content and band MMAs
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
                uint32_t a4[4], c4[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const int d = d8 * 8 + 2 * z;
                    const bool in0 = row_valid && d < p.D, in1 = row_valid && d + 1 < p.D;
                    const float u0 = in0 ? up[d] : 0.f, u1 = in1 ? up[d + 1] : 0.f;
                    const float w0 = in0 ? wp[d] : 0.f, w1 = in1 ? wp[d + 1] : 0.f;
                    a4[z] = pack_bf16((qrow[d] + u0) * p.sl2, (qrow[d + 1] + u1) * p.sl2);
                    c4[z] = pack_bf16((qrow[d] + w0) * p.sl2, (qrow[d + 1] + w1) * p.sl2);
                }
                *reinterpret_cast<uint4 *>(smem + S::QU + sw128_offset(ii, 8 * d8)) =
                    make_uint4(a4[0], a4[1], a4[2], a4[3]);
                *reinterpret_cast<uint4 *>(smem + S::QV + sw128_offset(ii, 8 * d8)) =
                    make_uint4(c4[0], c4[1], c4[2], c4[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(S::B_Q));
        }

        const int shift = 31 - lane;
        // the tile's S (64 columns) and the 96-column band window its rows
        // need, in one batch of TMEM loads: the buffers are free right after
        auto load_tile = [&](int n, float (&x)[64], float (&a)[96]) {
            const int rel = 96 - 32 * quarter;            // window start in chunks n..n+2
            uint32_t c[3];
#pragma unroll
            for (int z = 0; z < 3; ++z) {
                const int rz = rel + 32 * z;
                c[z] = 64 * (uint32_t)((n + (rz >> 6)) % NCHUNK) + (rz & 63);
            }
            tmem_ld_5x32(ts, ts + 32, tb0 + c[0], tb0 + c[1], tb0 + c[2], x, a);
        };
        // scaled logits of the 64 keys: S plus the band aligned to this row
        // (Appendix B's left shift of row i by L-1-i: row ii reads band column
        // 127-ii+jj, a warp-uniform window start plus 31-lane), masked.  The
        // shift runs on the band rounded to fp16 pairs (11-bit significand,
        // saturated to the finite range): four select stages move whole
        // registers (shift / 2), one byte permute moves half a register
        // (shift & 1), then each fp16 is added to the fp32 content logit.
        const uint32_t odd_sel = (shift & 1) ? 0x5432u : 0x3210u;
        auto logits = [&](bool diag, int lim, float (&x)[64], float (&a)[96]) {
            uint32_t hb[48];
#pragma unroll
            for (int y = 0; y < 48; ++y) hb[y] = pack_f16_sat(a[2 * y], a[2 * y + 1]);
#pragma unroll
            for (int y = 0; y < 40; ++y) hb[y] = (shift & 16) ? hb[y + 8] : hb[y];
#pragma unroll
            for (int y = 0; y < 36; ++y) hb[y] = (shift & 8) ? hb[y + 4] : hb[y];
#pragma unroll
            for (int y = 0; y < 34; ++y) hb[y] = (shift & 4) ? hb[y + 2] : hb[y];
#pragma unroll
            for (int y = 0; y < 33; ++y) hb[y] = (shift & 2) ? hb[y + 1] : hb[y];
#pragma unroll
            for (int y = 0; y < 32; ++y) add_f16x2_to(x[2 * y], x[2 * y + 1], __byte_perm(hb[y], hb[y + 1], odd_sel));
            if (diag) {
#pragma unroll
                for (int y = 0; y < 64; ++y) x[y] = (y <= lim) ? x[y] : -INFINITY;
            }
        };
        auto rowmax32 = [&](const float *x) {
            float q1[11];
#pragma unroll
            for (int y = 0; y < 10; ++y) q1[y] = max3(x[3 * y], x[3 * y + 1], x[3 * y + 2]);
            q1[10] = fmaxf(x[30], x[31]);
            return max3(max3(q1[0], q1[1], q1[2]), max3(q1[3], q1[4], q1[5]),
                        max3(q1[6], q1[7], max3(q1[8], q1[9], q1[10])));
        };
        auto expo = [&](const float *x, float mu, float *pk) {
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int y = 0; y < 16; ++y) {
                const float p0 = ex2(x[2 * y] - mu), p1 = ex2(x[2 * y + 1] - mu);
                sacc[y & 3] += p0 + p1;
                pk[y] = __uint_as_float(pack_bf16(p0, p1));
            }
            return (sacc[0] + sacc[1]) + (sacc[2] + sacc[3]);
        };

        float m_used = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int n = set; n < N; n += 2) {
            const int j0 = (t0 + n) * BN;
            if (!wwait(S::B_S + set, (n >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the mask matters only where this warp's rows meet the diagonal
            const bool diag = j0 + BN - 1 > p.M + i0 + 32 * quarter;
            const int lim = row_valid ? (p.M + i - j0) : (p.T - 1 - j0);
            float x[64], a[96];
            load_tile(n, x, a);
            // S and the band window are in registers: the S buffer and the band
            // slot may be overwritten by the next MMAs from here on
            tc_fence_before();
            mbar_arrive(bar(S::B_SF + set));
            logits(diag, lim, x, a);
            const float *x0 = x, *x1 = x + 32;
            const float tmax = fmaxf(rowmax32(x0), rowmax32(x1));
            float alpha = 1.f;
            const bool raise = tmax > m_used + RESCALE_LOG2;   // also the first finite max
            if (raise) {
                alpha = ex2(m_used - tmax);                     // 0 when m_used = -inf
                m_used = tmax;
            }
            const float mu = (m_used == -INFINITY) ? 0.f : m_used;
            float pk[32];
            const float psum = expo(x0, mu, pk) + expo(x1, mu, pk + 16);
            l_run = l_run * alpha + psum;
            // P buffer b of this set was last read by the P.V of tile n-4
            const int b = (n >> 1) & 1;
            if (n >= 4 && !wwait(S::B_PV + 2 * set + b, ((n >> 2) - 1) & 1)) {
                ok = false;
                break;
            }
            if (n >= 2 && __any_sync(0xffffffffu, raise)) {
                // O holds the P.V of this set's earlier tiles: rescale it once the
                // last of them (tile n-2, the other buffer) is done
                if (!wwait(S::B_PV + 2 * set + (1 - b), ((n - 2) >> 2) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < DP / 16; ++c) {
                    float o[16];
                    tmem_ld16(to + 16 * c, o);
#pragma unroll
                    for (int y = 0; y < 16; ++y) o[y] *= alpha;
                    tmem_st16(to + 16 * c, o);
                }
                tmem_wait_st();
            }
            unsigned char *pb = smem + S::PB + (2 * set + b) * (BM * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(pb + sw128_offset(ii, 8 * c)) =
                    make_uint4(__float_as_uint(pk[4 * c]), __float_as_uint(pk[4 * c + 1]),
                               __float_as_uint(pk[4 * c + 2]), __float_as_uint(pk[4 * c + 3]));
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(S::B_P + set));
        }

        // ---- epilogue: merge the two sets' partial results of each row
        const bool has = set < N;                  // set 1 has no tile when N == 1
        if (ok && has) ok = wwait(S::B_O + set, 0);
        float o[DP];
#pragma unroll
        for (int d = 0; d < DP; ++d) o[d] = 0.f;
        if (ok && has) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < DP / 16; ++c) tmem_ld16(to + 16 * c, *reinterpret_cast<float(*)[16]>(&o[16 * c]));
        }
        // set 1 hands (m, l, O) to set 0 through the stage ring, once every
        // P.V of both sets (the ring's last readers) has completed
        float *xo = reinterpret_cast<float *>(smem + S::ST0);   // [128][64] O of set 1
        float *xml = reinterpret_cast<float *>(smem + S::XML);  // [128][2] (m, l) of set 1
        if (set == 1 && ok) ok = wwait(S::B_O + 0, 0);
        if (set == 1) {
#pragma unroll
            for (int d4 = 0; d4 < DP / 4; ++d4)
                reinterpret_cast<float4 *>(xo + ii * 64)[d4 ^ (ii & 7)] =   // swizzled: no bank conflicts
                    make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
            xml[2 * ii] = has ? m_used : -INFINITY;
            xml[2 * ii + 1] = has ? l_run : 0.f;
            mbar_arrive(bar(S::B_X));
        } else if (ok && wwait(S::B_X, 0)) {
            const float m1 = xml[2 * ii], l1 = xml[2 * ii + 1];
            const float mx = fmaxf(m_used, m1);
            const float w0 = (m_used == -INFINITY) ? 0.f : ex2(m_used - mx);
            const float w1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mx);
            const float l = l_run * w0 + l1 * w1;
#pragma unroll
            for (int d4 = 0; d4 < DP / 4; ++d4) {
                const float4 v1 = reinterpret_cast<const float4 *>(xo + ii * 64)[d4 ^ (ii & 7)];
                o[4 * d4] = o[4 * d4] * w0 + v1.x * w1;
                o[4 * d4 + 1] = o[4 * d4 + 1] * w0 + v1.y * w1;
                o[4 * d4 + 2] = o[4 * d4 + 2] * w0 + v1.z * w1;
                o[4 * d4 + 3] = o[4 * d4 + 3] * w0 + v1.w * w1;
            }
            l_run = l;
            m_used = mx;
            if (row_valid) {
                if (p.splits == 1) {
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    __nv_bfloat16 *op = p.out + (long)i * qkv_row + head_off;
                    if ((p.D & 7) == 0) {
#pragma unroll
                        for (int d8 = 0; d8 < DP / 8; ++d8) {
                            if (d8 * 8 < p.D) {
                                uint4 pk4;
                                pk4.x = pack_bf16(o[d8 * 8 + 0] * inv, o[d8 * 8 + 1] * inv);
                                pk4.y = pack_bf16(o[d8 * 8 + 2] * inv, o[d8 * 8 + 3] * inv);
                                pk4.z = pack_bf16(o[d8 * 8 + 4] * inv, o[d8 * 8 + 5] * inv);
                                pk4.w = pack_bf16(o[d8 * 8 + 6] * inv, o[d8 * 8 + 7] * inv);
                                *reinterpret_cast<uint4 *>(op + d8 * 8) = pk4;
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
                    // m_used is in log2 units of the scaled logits
                    p.part_lse[prow] = l_run > 0.f ? m_used + log2f(l_run) : -INFINITY;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

// 3-D view {64, rows, groups} of a bf16 tensor with D = 64 elements per row,
// rows `row_stride` elements apart and groups (b*H+h or h) 64 elements apart;
// the box {64, box_rows, 1} lands in shared memory as 128-byte rows with the
// 128-byte swizzle (the layout the MMA descriptors expect).
bool make_map(CUtensorMap *m, const void *base, long rows, long row_stride, long groups, int box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)groups};
    cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, 64 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
    // charge for the partials and the combine pass; 1 when the grid already
    // fills the GPU
    double best = 1e30;
    int best_s = 1;
    for (int s = 1; s <= 16 && s <= ntile; ++s) {
        const long waves = (ctas * s + num_sms - 1) / num_sms;
        const int per = (ntile + s - 1) / s;
        const double cost = (double)waves * (per + 2) + (s > 1 ? 2.0 : 0.0);
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
    const bool tma = a.D == 64;
    if (tma) {
        const long bhn = (long)a.B * a.H;
        const long rs = bhn * a.D;
        if (!make_map(&mk, a.k, p.T, rs, bhn, BN) || !make_map(&mv, a.v, p.T, rs, bhn, BN) ||
            !make_map(&mr, a.r, p.T, (long)a.H * a.D, a.H, BN))
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
