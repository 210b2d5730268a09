// attn_bf16.cu -- fused bf16 relative attention on tcgen05 tensor cores.
//
// What is computed (Transformer-XL, Section 3.3, per-layer procedure):
//     s_ij = ((q_i+u).k_j + (q_i+v).Q_{L-1-i+j}) / sqrt(D),  j <= M+i,
//     out_i = softmax_j(s_ij) v_j,
// with Q the reversed projected table of Appendix B (row t = W_kR R_{T-1-t}).
//
// Persistent: one CTA of twelve warps per SM walks work items (128 query
// rows of one (b, h), or one key-range split of them) heaviest first, and
// each item's keys in tiles of 128.  Roles:
//   warp 0     producer: TMA loads of K, V into a three-stage shared-memory
//              ring, of 128-row table chunks into a four-slot ring, and of
//              the next item's raw q rows and biases (for head sizes other
//              than 64: coalesced thread loads, warp 3 taking V);
//   warp 1     one thread issues, per tile, S = (q+u) K^T (N = 128) and the
//              tile's band window (q+v) [chunk n; chunk n+1]^T (256 columns)
//              into TMEM, their K steps interleaved;
//   warp 2     one thread issues O += P V with P read from TMEM, and the TMA
//              store of each finished output tile;
//   warps 4-11 softmax on the 16-lane TMEM shape: a warp owns 16 query rows;
//              lanes 0-15 take keys 0-63 of the tile, lanes 16-31 keys
//              64-127 of the same rows.  Each thread loads its 64 S columns
//              and the 80 band columns its row needs in one batch (S and the
//              band are then free for the next tile's MMAs), aligns the band
//              to the row (Appendix B's left shift of row i by L-1-i: a
//              barrel shift by 15 - (row mod 16) on fp16 pairs), adds it,
//              masks j <= M+i on diagonal tiles, exponentiates against the
//              row's running reference max and writes P (bf16) to TMEM.
// TMEM (512 columns): S 128, band window 256, P 64, O 64.  The band window
// costs twice the position term's pairs: a window of two 128-row chunks keeps
// each 16-row group's 80 columns contiguous for the load's fixed half-split
// offset.  The reference max is raised (and O in TMEM rescaled) on an item's
// first tile and when a row's sum passes 2^12.  The scale
// log2(e)/sqrt(D) is folded into q+u and q+v before rounding.  Every mbarrier
// wait is bounded; on expiry the CTA records an error word (read by
// txl_check) and every role winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "sm100.cuh"

namespace txl {

__device__ unsigned int g_err_word;

namespace {
using namespace sm100;

constexpr int BM = 128;           // query rows per CTA (TMEM lanes)
constexpr int BN = 128;           // keys per tile; also table rows per band chunk
constexpr int HN = BN / 2;        // keys per softmax thread and tile
constexpr int NSTAGE = 3;         // shared-memory ring of K, V tiles
constexpr int NCH = 4;            // shared-memory ring of 128-row table chunks
constexpr int NT = 384;           // 12 warps, see the role list above
constexpr uint32_t TM_S = 0;      // S of the current tile, 128 columns
constexpr uint32_t TM_BAND = 128; // the tile's band window: 256 table rows, 256 columns
constexpr uint32_t TM_P = 384;    // P (bf16 pairs), 64 columns
constexpr uint32_t TM_O = 448;    // O accumulator, up to 64 columns
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t REG_LOW = 96, REG_HIGH = 200;     // per-thread registers after the split
static_assert(128 * REG_LOW + 256 * REG_HIGH <= 65536 / NT / 8 * 8 * NT, "register split exceeds the launch");
constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s per wait, then give up
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float SUM_LIMIT = 4096.0f;          // raise the exponent base once a row sum passes 2^12

struct Params {
    const __nv_bfloat16 *q, *k, *v, *r;
    const float *u, *w;
    __nv_bfloat16 *out;
    // key-split partials when splits > 1: each split's normalised output in
    // bf16, laid out like the output over splits*B*H heads ([L][splits*B*H][DP],
    // head index split*B*H + bh), and its row log-sum-exp in log2 units,
    // [splits][B*H][L]
    __nv_bfloat16 *part_o;
    float *part_lse;
    float *lse;         // optional [B*H][L]: each row's log-sum-exp (natural log) of the scaled scores
    // backward scores only (the forward's output O comes in `out`): dO, the
    // outputs P and dA ([B*H][L][TP]) and dA in the table frame
    // ([H][L][B][TP]), 1/sqrt(d_head)
    const __nv_bfloat16 *dout;
    __nv_bfloat16 *p_out, *da_out, *db_out;
    long TP;
    float inv_sqrt_d;
    int B, H, D, L, M, T;
    int nqt, splits;
    int items;          // B*H*nqt*splits work items
    int streamk, sk_nt; // stream-K schedule (splits = 2 partial slots), key tiles per item
    int kv_start;       // K, V rows form a ring: key j at row (kv_start + j) mod T
    int ost;            // 1: output tiles written by TMA store (the output's tensor map)
    float sl2;          // log2(e) / sqrt(D)
    // the memory rollover copied by warp 3 of every CTA (its slice of
    // roll_n16 16-byte units), 0 units when not fused
    const uint4 *roll_src;
    uint4 *roll_dst;
    long roll_n16;
    // several calls of one shape in one launch (kernel instantiations with
    // NC > 1): ncell calls, each with its own tensor maps, biases and
    // rollover (roll_n16 units each); the fields above are the first call's
    int ncell;
    const float *cell_u[ATTN_CELLS], *cell_w[ATTN_CELLS];
    const uint4 *cell_roll_src[ATTN_CELLS];
    uint4 *cell_roll_dst[ATTN_CELLS];
};

// The tensor maps of a launch: per call K, V, the table, q and the output
// (NC calls), and the 8-row K, V boxes of a ring (one call only).
template <int NC>
struct AttnMaps {
    CUtensorMap k[NC], v[NC], r[NC], q[NC], o[NC];
    CUtensorMap k8, v8;
};

// Every operand tile in shared memory uses 128-byte rows with the 128-byte
// swizzle (element (row, k) at sw128_offset(row, k)); D <= 64 fits one row.
template <int DP>
struct Smem {
    static constexpr uint32_t TILE = BN * 128;             // 128 rows of 128 bytes: K, V or a table chunk
    static constexpr uint32_t KV = 2 * TILE;                // K and V of one key tile
    static constexpr uint32_t ST0 = 0;                      // NSTAGE K/V stages
    static constexpr uint32_t CH0 = NSTAGE * KV;            // NCH table chunks (a ring)
    static constexpr uint32_t QU = CH0 + NCH * TILE;        // q+u, q+v: 128 rows of 128 bytes
    static constexpr uint32_t QV = QU + BM * 128;
    static constexpr uint32_t QRAW = QV + BM * 128;         // raw q rows of the next item
    static constexpr uint32_t OST = QRAW + BM * 128;        // an item's output tile (bf16), for the TMA store
    static constexpr uint32_t UW = OST + BM * 128;          // the next item's u and v biases (fp32, 2 x 64)
    static constexpr uint32_t BARS = UW + 2 * 64 * 4;
    // barrier slots (8 bytes each): q+u/q+v ready, raw q ready, raw q read;
    // per K/V stage full / empty; per chunk slot full / empty; S full, S
    // free (loaded by the softmax), P full, P.V done; output tile written,
    // output buffer free
    static constexpr int B_Q = 0, B_QRAW = 1, B_QRF = 2, B_FULL = 3, B_EMPTY = 3 + NSTAGE,
                         B_CHF = 3 + 2 * NSTAGE, B_CHE = B_CHF + NCH, B_S = B_CHE + NCH, B_SF = B_S + 1,
                         B_P = B_SF + 1, B_PV = B_P + 1, B_OST = B_PV + 1, B_OFR = B_OST + 1;
    static_assert(B_OFR < 32, "barrier slots");
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

// packed pairs of fp32 (Blackwell f32x2 arithmetic: one instruction, two elements)
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
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ void record_error(unsigned int code) { atomicOr(&g_err_word, code); }

// A bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort,
                                              uint64_t limit_ns = WAIT_NS)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
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
                                               int limit, int D, int lane, int ring_start = 0)
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
            // a ring of `limit` rows stores logical row j at (ring_start + j) mod limit
            const int srow = row + ring_start < limit ? row + ring_start : row + ring_start - limit;
            const long e0 = row0_elems + (long)srow * row_stride;   // first element of the row
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

// One work item: 128 query rows of one (b, h) and one key-range split of
// them.  Items are numbered heaviest first (query tiles from the last one
// down; see make_item for launches of several calls); CTA c of G takes items
// c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the sorted list, so that every
// CTA gets a similar total of key tiles).
struct Item {
    int cell, bh, b, h, i0, rows_here, split, t0, N, kb0;
    int whole;          // the item's output is final (else a partial: key split or cut item)
    long head_off;
};

__device__ __forceinline__ Item make_item(const Params &p, int k)
{
    Item it;
    // The calls of a multi-call launch follow one another.  Inside a call the
    // query tiles go heaviest first in the last call and in every second call
    // before it, lightest first in the others, so that light items meet
    // light ones at the calls' boundaries and the CTAs' totals stay even;
    // a head's query tiles stay one level (B*H items) apart, so its keys and
    // values are still in L2 when the next one reads them.
    const int per_level = p.B * p.H * p.splits;           // one query tile level of one call
    const int nc = p.ncell > 1 ? p.ncell : 1;
    const int per_call = per_level * p.nqt;
    it.cell = k / per_call;
    const int kk = k % per_call;
    const bool heavy_first = ((nc - 1 - it.cell) & 1) == 0;
    const int qt = heavy_first ? p.nqt - 1 - kk / per_level : kk / per_level;
    const int rem = kk % per_level;
    it.bh = rem / p.splits;
    it.split = rem % p.splits;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    it.i0 = qt * BM;
    it.rows_here = min(BM, p.L - it.i0);
    const int kend = min(p.T, p.M + it.i0 + it.rows_here);   // keys these rows can see
    const int ntile = (kend + BN - 1) / BN;
    it.t0 = it.split * ntile / p.splits;                      // 32-bit: ntile * splits is small
    const int t1 = (it.split + 1) * ntile / p.splits;
    it.N = t1 - it.t0;
    // table row of (query i0+ii, key j0+jj) in tile n: kb0 + n*BN + 127 - ii + jj
    it.kb0 = p.L - BM - it.i0 + it.t0 * BN;
    it.head_off = ((long)it.b * p.H + it.h) * p.D;
    it.whole = p.splits == 1;
    return it;
}

// Stream-K schedule (one query tile per (b, h), at least as many (b, h) as
// CTAs): the B*H items' key tiles, numbered item by item, are cut into
// gridDim.x equal contiguous ranges, one per CTA.  An item inside one range
// is computed whole; an item cut by a range boundary (at most once, since a
// range holds at least one item's tiles) is computed in two parts, part 0
// from its first tile, part 1 to its last, each written as a partial and
// merged afterwards.  The j-th part or item of this CTA, or -1 past the end.
__device__ __forceinline__ int streamk_item(const Params &p, int j, Item &it)
{
    const long G = gridDim.x, c = blockIdx.x, nt = p.sk_nt;
    const long tt = (long)p.B * p.H * nt;
    const long s0 = c * tt / G, s1 = (c + 1) * tt / G;
    const long k = s0 / nt + j;
    if (s1 <= s0 || k * nt >= s1) return -1;
    it.cell = 0;
    const long a = (s0 > k * nt ? s0 : k * nt) - k * nt;
    const long e = (s1 < (k + 1) * nt ? s1 : (k + 1) * nt) - k * nt;
    it.bh = (int)k;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    it.i0 = 0;
    it.rows_here = min(BM, p.L);
    it.t0 = (int)a;
    it.N = (int)(e - a);
    it.split = a == 0 ? 0 : 1;
    it.whole = a == 0 && e == nt;
    it.kb0 = p.L - BM + it.t0 * BN;
    it.head_off = ((long)it.b * p.H + it.h) * p.D;
    return j;
}

// the j-th item of this CTA, or -1 past the end
__device__ __forceinline__ int item_of(const Params &p, int j)
{
    const int G = gridDim.x, c = blockIdx.x;
    const long k = (long)j * G + ((j & 1) ? (G - 1 - c) : c);
    return k < p.items ? (int)k : -1;
}

// the first item at position >= j with at least one key tile (-1 if none)
template <bool kSK>
__device__ __forceinline__ int next_busy(const Params &p, int j, Item &it)
{
    if (kSK) return streamk_item(p, j, it);
    for (;; ++j) {
        const int k = item_of(p, j);
        if (k < 0) return -1;
        it = make_item(p, k);
        if (it.N > 0) return j;
    }
}

// the call an item belongs to (always the first in one-call launches)
template <int NC>
__device__ __forceinline__ int cell_of(const Item &it)
{
    return NC == 1 ? 0 : it.cell;
}

template <int DP, bool kTma, bool kSK, int NC>
__global__ void __launch_bounds__(NT, 1)
rel_attn_bf16_kernel(const __grid_constant__ AttnMaps<NC> tm, const Params p)
{
    using S = Smem<DP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long qkv_row = (long)p.B * p.H * p.D;            // elements between positions

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
        mbar_init(bar(S::B_Q), 256);
        mbar_init(bar(S::B_QRAW), kTma ? 1 : 32);
        mbar_init(bar(S::B_QRF), 256);
        for (int x = 0; x < NSTAGE; ++x) {
            mbar_init(bar(S::B_FULL + x), kTma ? 1 : 64);
            mbar_init(bar(S::B_EMPTY + x), 1);
        }
        for (int x = 0; x < NCH; ++x) {
            mbar_init(bar(S::B_CHF + x), kTma ? 1 : 32);
            mbar_init(bar(S::B_CHE + x), 1);
        }
        mbar_init(bar(S::B_S), 1);
        mbar_init(bar(S::B_SF), 256);
        mbar_init(bar(S::B_P), 256);
        mbar_init(bar(S::B_PV), 1);
        mbar_init(bar(S::B_OST), 256);
        mbar_init(bar(S::B_OFR), 1);
        fence_mbar_init();
        if (kTma) {
            for (int c = 0; c < (NC == 1 ? 1 : p.ncell); ++c) {
                prefetch_tmap(&tm.k[c]);
                prefetch_tmap(&tm.v[c]);
                prefetch_tmap(&tm.r[c]);
                prefetch_tmap(&tm.q[c]);
                if (p.ost) prefetch_tmap(&tm.o[c]);
            }
            if (p.kv_start) {
                prefetch_tmap(&tm.k8);
                prefetch_tmap(&tm.v8);
            }
        }
    }
    // the padding of D up to a multiple of 16 (the MMA K step) must be zero in
    // every operand buffer, and loads never write it: clear everything once
    if (p.D != DP) {
        for (uint32_t x = tid; x < S::UW / 16; x += NT)
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
            // raw q rows (+ the head's u, v biases) of an item, for the
            // softmax warps to turn into the MMA operands q+u, q+v
            auto load_q = [&](const Item &it) {
                if (kTma) {
                    if (lane == 0) {
                        const int c = cell_of<NC>(it);
                        const float *u = NC == 1 ? p.u : p.cell_u[c], *w = NC == 1 ? p.w : p.cell_w[c];
                        mbar_arrive_expect_tx(bar(S::B_QRAW), S::TILE + 2 * 64 * 4);
                        tma_load_3d(sbase + S::QRAW, &tm.q[c], bar(S::B_QRAW), 0, it.i0, it.bh);
                        bulk_load(sbase + S::UW, u + it.h * p.D, 64 * 4, bar(S::B_QRAW));
                        bulk_load(sbase + S::UW + 256, w + it.h * p.D, 64 * 4, bar(S::B_QRAW));
                    }
                } else if (warp == 0) {
                    warp_load_rows(smem + S::QRAW, BM, p.q, it.head_off + (long)it.i0 * qkv_row, qkv_row, 0,
                                   it.rows_here, p.D, lane);
                    float *uw = reinterpret_cast<float *>(smem + S::UW);
                    for (int d = lane; d < 64; d += 32) {
                        uw[d] = d < p.D ? p.u[it.h * p.D + d] : 0.f;
                        uw[64 + d] = d < p.D ? p.w[it.h * p.D + d] : 0.f;
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(bar(S::B_QRAW));
                }
            };
            // table chunk number cg (global count) into ring slot cg % NCH,
            // once the S MMAs of its previous occupant are done (warp 0)
            auto load_chunk = [&](int cg, int row, int h, int c) {
                const int slot = cg % NCH;
                if (cg >= NCH && !wwait(S::B_CHE + slot, ((cg / NCH) - 1) & 1)) return false;
                if (kTma) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar(S::B_CHF + slot), S::TILE);
                        tma_load_3d(sbase + S::CH0 + slot * S::TILE, &tm.r[c], bar(S::B_CHF + slot), 0, row, h);
                    }
                } else {
                    warp_load_rows(smem + S::CH0 + slot * S::TILE, BN, p.r, (long)h * p.D, (long)p.H * p.D, row,
                                   p.T, p.D, lane);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(S::B_CHF + slot));
                }
                return true;
            };
            Item it;
            int j = next_busy<kSK>(p, 0, it);
            if (j >= 0) load_q(it);
            int g = 0, cg = 0, ni = 0;               // key tiles, table chunks, items so far
            bool ok = true;
            while (ok && j >= 0) {
                // chunk 0 of the item (its tile n reads chunks n and n+1)
                if (warp == 0 && !load_chunk(cg, it.kb0, it.h, cell_of<NC>(it))) break;
                ++cg;
                for (int n = 0; n < it.N; ++n, ++g) {
                    const int st = g % NSTAGE;
                    // the stage is free once the P.V of tile g-NSTAGE (its last reader) is done
                    if (g >= NSTAGE && !wwait(S::B_EMPTY + st, ((g / NSTAGE) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int j0 = (it.t0 + n) * BN;
                    const uint32_t dst = sbase + S::ST0 + st * S::KV;
                    if (kTma) {
                        if (lane == 0) {
                            // K, V rows may sit in a ring (key j at row (kv_start + j) mod T)
                            int s0 = p.kv_start + j0;
                            if (s0 >= p.T) s0 -= p.T;
                            mbar_arrive_expect_tx(bar(S::B_FULL + st), S::KV);
                            if (p.kv_start == 0 || s0 + BN <= p.T) {
                                // one box; in the plain layout rows past the last key
                                // are zero-filled
                                tma_load_3d(dst, &tm.k[cell_of<NC>(it)], bar(S::B_FULL + st), 0, s0, it.bh);
                                tma_load_3d(dst + S::TILE, &tm.v[cell_of<NC>(it)], bar(S::B_FULL + st), 0, s0, it.bh);
                            } else {
                                // the tile crosses the ring's end: sixteen 8-row boxes
                                // (one swizzle atom each, 1 KB apart in the stage), each
                                // from its own ring row; rows past the last key are
                                // other ring rows (finite, masked)
                                for (int m = 0; m < BN / 8; ++m) {
                                    const int sr = (s0 + 8 * m) % p.T;   // T may be below 128
                                    tma_load_3d(dst + 1024u * m, &tm.k8, bar(S::B_FULL + st), 0, sr, it.bh);
                                    tma_load_3d(dst + S::TILE + 1024u * m, &tm.v8, bar(S::B_FULL + st), 0, sr,
                                                it.bh);
                                }
                            }
                        }
                    } else {
                        unsigned char *d = smem + S::ST0 + st * S::KV;
                        if (warp == 0)
                            warp_load_rows(d, BN, p.k, it.head_off, qkv_row, j0, p.T, p.D, lane, p.kv_start);
                        else
                            warp_load_rows(d + S::TILE, BN, p.v, it.head_off, qkv_row, j0, p.T, p.D, lane,
                                           p.kv_start);
                        fence_proxy_async_smem();
                        mbar_arrive(bar(S::B_FULL + st));
                    }
                    // table chunk n+1
                    if (warp == 0 && !load_chunk(cg, it.kb0 + (n + 1) * BN, it.h, cell_of<NC>(it))) {
                        ok = false;
                        break;
                    }
                    ++cg;
                }
                if (!ok) break;
                // the next item's q rows, once this item's have been converted
                Item nx;
                const int jn = next_busy<kSK>(p, j + 1, nx);
                if (jn >= 0) {
                    if (!wwait(S::B_QRF, ni & 1)) break;
                    load_q(nx);
                }
                j = jn;
                it = nx;
                ++ni;
            }
        } else if (warp == 1) {
            // =============================================================== S / band MMAs
            // per tile: S = (q+u) K^T (N = 128) and the tile's band window
            // (q+v) [chunk n; chunk n+1]^T (N = 256) into TMEM.  One thread
            // waits and issues.
            if (lane == 0) {
                const uint32_t idesc_n = idesc_bf16(BM, BN, 0, 0);
                const uint32_t idesc_w = idesc_bf16(BM, 2 * BN, 0, 0);   // the band of two adjacent chunks
                // descriptors built once; the 14-bit start-address field (address / 16)
                // advances by 2 per 32-byte K step within a 128-byte swizzled row
                const uint64_t d_qu = smem_desc_sw128(sbase + S::QU, 16, 1024);
                const uint64_t d_qv = smem_desc_sw128(sbase + S::QV, 16, 1024);
                const uint64_t d_st0 = smem_desc_sw128(sbase + S::ST0, 16, 1024);
                const uint64_t d_ch0 = smem_desc_sw128(sbase + S::CH0, 16, 1024);
                constexpr uint64_t KV16 = S::KV >> 4, TILE16 = S::TILE >> 4;
                Item it;
                int g = 0, cg = 0, ni = 0;
                bool ok = true;
                for (int j = next_busy<kSK>(p, 0, it); ok && j >= 0; j = next_busy<kSK>(p, j + 1, it), ++ni) {
                    if (!wait_or_abort(bar(S::B_Q), ni & 1, abort)) break;     // q+u, q+v of the item
                    const int c0 = cg;
                    for (int n = 0; n < it.N; ++n, ++g) {
                        const int st = g % NSTAGE;
                        const int ca = c0 + n, cb = ca + 1, sa = ca % NCH, sb = cb % NCH;
                        // the S buffer and the band window were last read by the
                        // softmax loads of tile g-1
                        if (g >= 1) ok = wait_or_abort(bar(S::B_SF), (g - 1) & 1, abort);
                        ok = ok && wait_or_abort(bar(S::B_FULL + st), (g / NSTAGE) & 1, abort) &&
                             wait_or_abort(bar(S::B_CHF + sa), (ca / NCH) & 1, abort) &&
                             wait_or_abort(bar(S::B_CHF + sb), (cb / NCH) & 1, abort);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t dk = d_st0 + st * KV16, da = d_ch0 + sa * TILE16, db = d_ch0 + sb * TILE16;
                        // S and band K steps alternate (two accumulation chains
                        // in flight); when chunk n+1 sits in the slot after
                        // chunk n the band is one N = 256 MMA per K step
                        if (sb == sa + 1) {
#pragma unroll
                            for (int ks = 0; ks < DP / 16; ++ks) {
                                mma_bf16_ss(tmem + TM_S, d_qu + 2 * ks, dk + 2 * ks, idesc_n, ks > 0);
                                mma_bf16_ss(tmem + TM_BAND, d_qv + 2 * ks, da + 2 * ks, idesc_w, ks > 0);
                            }
                        } else {
#pragma unroll
                            for (int ks = 0; ks < DP / 16; ++ks) {
                                mma_bf16_ss(tmem + TM_S, d_qu + 2 * ks, dk + 2 * ks, idesc_n, ks > 0);
                                mma_bf16_ss(tmem + TM_BAND, d_qv + 2 * ks, da + 2 * ks, idesc_n, ks > 0);
                                mma_bf16_ss(tmem + TM_BAND + BN, d_qv + 2 * ks, db + 2 * ks, idesc_n, ks > 0);
                            }
                        }
                        mma_commit(bar(S::B_S));
                        mma_commit(bar(S::B_CHE + sa));                   // chunk n: read for the last time
                        if (n == it.N - 1) mma_commit(bar(S::B_CHE + sb));   // the item's last chunk
                    }
                    cg = c0 + it.N + 1;
                }
            }
            __syncwarp();
        } else if (kTma && warp == 3) {
            // =============================================================== memory rollover
            // Section 3.2's cache update of this layer, independent of the
            // attention: the CTA's contiguous slice of the flat copy,
            // sixteen 16-byte loads in flight per lane, streaming cache hints
            // (the data is used once; the layer's K, V and table stay in L2)
            // (each call's copy of a multi-call launch in turn)
            for (int c = 0; p.roll_n16 > 0 && c < (NC == 1 ? 1 : p.ncell); ++c) {
                const uint4 *src = NC == 1 ? p.roll_src : p.cell_roll_src[c];
                uint4 *dst = NC == 1 ? p.roll_dst : p.cell_roll_dst[c];
                const long G = gridDim.x, per = (p.roll_n16 + G - 1) / G;
                const long beg = (long)blockIdx.x * per;
                const long end = beg + per < p.roll_n16 ? beg + per : p.roll_n16;
                long x = beg + lane;
                for (; x + 15 * 32 < end; x += 16 * 32) {
                    uint4 t[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) t[u] = __ldcs(src + x + 32 * u);
#pragma unroll
                    for (int u = 0; u < 16; ++u) __stcs(dst + x + 32 * u, t[u]);
                }
                for (; x < end; x += 32) __stcs(dst + x, __ldcs(src + x));
            }
        } else if (warp == 2) {
            // =============================================================== P.V MMAs
            // This thread also writes the output tiles: the softmax threads
            // stage an item's O / l in shared memory during the next item's
            // first tile, before that tile's P, so the tile's P barrier shows
            // the stage complete.  The buffer is handed back (B_OFR) once the
            // store has read it; the CTA's last item signals on B_OST.
            if (lane == 0) {
                const uint32_t idesc_o = idesc_bf16(BM, DP, 0, 1);   // V is MN-major (d contiguous)
                const uint64_t d_st0 = smem_desc_sw128(sbase + S::ST0, 16, 1024);
                constexpr uint64_t KV16 = S::KV >> 4, TILE16 = S::TILE >> 4;
                const bool ost = kTma && p.ost;
                if (ost) mbar_arrive(bar(S::B_OFR));   // the buffer starts free
                bool in_flight = false;                // a store may still be reading the buffer
                Item it, prev;
                int g = 0;
                bool ok = true, have_prev = false;
                for (int j = next_busy<kSK>(p, 0, it); ok && j >= 0; j = next_busy<kSK>(p, j + 1, it)) {
                    for (int n = 0; n < it.N; ++n, ++g) {
                        const int st = g % NSTAGE;
                        if (in_flight) {
                            bulk_wait_read();
                            mbar_arrive(bar(S::B_OFR));
                            in_flight = false;
                        }
                        if (!wait_or_abort(bar(S::B_P), g & 1, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // under the stream-K schedule only whole items go
                        // through the staged tile (the output map is then the output)
                        if (ost && n == 0 && have_prev && (prev.whole || !kSK)) {
                            tma_store_3d(&tm.o[cell_of<NC>(prev)], sbase + S::OST, 0, prev.i0,
                                         (p.splits > 1 && !kSK) ? prev.split * p.B * p.H + prev.bh : prev.bh);
                            bulk_commit();
                            in_flight = true;
                        }
                        const uint64_t dv = d_st0 + st * KV16 + TILE16;   // 16 keys = 2048 bytes of V
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)   // P: 16 keys = 8 TMEM columns
                            mma_bf16_ts(tmem + TM_O, tmem + TM_P + 8 * kk, dv + 128 * kk, idesc_o,
                                        (n > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(bar(S::B_PV));
                        mma_commit(bar(S::B_EMPTY + st));
                    }
                    prev = it;
                    have_prev = true;
                }
                if (ok && ost && have_prev && (prev.whole || !kSK)) {
                    if (in_flight) {
                        bulk_wait_read();
                        mbar_arrive(bar(S::B_OFR));
                    }
                    if (wait_or_abort(bar(S::B_OST), 0, abort)) {
                        tma_store_3d(&tm.o[cell_of<NC>(prev)], sbase + S::OST, 0, prev.i0,
                                     (p.splits > 1 && !kSK) ? prev.split * p.B * p.H + prev.bh : prev.bh);
                        bulk_commit();
                    }
                }
                bulk_wait_all();   // the output stores are done
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<REG_HIGH>();
        // =============================================================== softmax
        // warp w owns 16 query rows (TMEM lanes lb..lb+15, lb = 32*quarter +
        // 16*rh) with the 16-lane TMEM shape: lanes 0-15 of the warp take keys
        // 0-63 of each tile, lanes 16-31 keys 64-127 of the same rows, so a
        // row's two halves meet in one warp (shuffles, no shared memory)
        const int quarter = warp & 3, rh = (warp - 4) >> 2;
        const int r16 = lane & 15, half = lane >> 4;
        const int lb = quarter * 32 + rh * 16;     // the warp's first row (TMEM lane)
        const int ii = lb + r16;                   // this thread's query row
        const uint32_t tl = tmem + ((uint32_t)lb << 16);
        // q+u and q+v of an item's row, scaled by log2(e)/sqrt(D) and rounded
        // once to bf16, from the raw rows into the MMA operand buffers (every
        // softmax thread: half of its own row, columns 8*DC*half ..; item
        // number ni)
        constexpr int DC = DP / 16;                // 8-column chunks per half row
        auto convert_q = [&](const Item &it, int ni) {
            if (!wwait(S::B_QRAW, ni & 1)) return false;
            const float4 *uw4 = reinterpret_cast<const float4 *>(smem + S::UW);
            const float keep = ii < it.rows_here ? 1.f : 0.f;   // rows past L: zero operands
            // every load first (the stores below could alias them as far as the
            // compiler knows), then the arithmetic and the stores
            uint4 raw[DC];
            float4 u4[2 * DC], w4[2 * DC];
#pragma unroll
            for (int c = 0; c < DC; ++c)
                raw[c] = *reinterpret_cast<const uint4 *>(smem + S::QRAW + sw128_offset(ii, 8 * (DC * half + c)));
#pragma unroll
            for (int d4 = 0; d4 < 2 * DC; ++d4) {
                u4[d4] = uw4[2 * DC * half + d4];
                w4[d4] = uw4[16 + 2 * DC * half + d4];
            }
            const float sk = p.sl2 * keep;
            const uint64_t sk2 = f2(sk, sk);
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const int d8 = DC * half + c;
                const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&raw[c]);
                const float *uu = reinterpret_cast<const float *>(&u4[2 * c]);
                const float *ww = reinterpret_cast<const float *>(&w4[2 * c]);
                uint32_t a4[4], c4[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    // (q + u) s as q s + (u s), on element pairs
                    const uint64_t q2 = f2(__bfloat162float(e[2 * z]), __bfloat162float(e[2 * z + 1]));
                    float a0, a1, b0, b1;
                    unf2(fma2(q2, sk2, mul2(f2(uu[2 * z], uu[2 * z + 1]), sk2)), a0, a1);
                    unf2(fma2(q2, sk2, mul2(f2(ww[2 * z], ww[2 * z + 1]), sk2)), b0, b1);
                    a4[z] = pack_bf16(a0, a1);
                    c4[z] = pack_bf16(b0, b1);
                }
                *reinterpret_cast<uint4 *>(smem + S::QU + sw128_offset(ii, 8 * d8)) =
                    make_uint4(a4[0], a4[1], a4[2], a4[3]);
                *reinterpret_cast<uint4 *>(smem + S::QV + sw128_offset(ii, 8 * d8)) =
                    make_uint4(c4[0], c4[1], c4[2], c4[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(S::B_Q));
            mbar_arrive(bar(S::B_QRF));
            return true;
        };

        // this thread's 64 S columns and the 80-column band window its row
        // needs: band column 127-ii+jj of the tile's 256-row window, a
        // warp-uniform start W0 (+64 for the key-half lanes 16-31) plus
        // 15-r16; one batch of five loads, the buffers free right after
        const int shift = 15 - r16;
        const int W0 = 112 - lb;
        auto load_tile = [&](float (&x)[64], float (&a)[80]) {
            const uint32_t ts = tl + TM_S, tb = tl + TM_BAND + (uint32_t)W0;
            tmem_ld_h_tile<HN>(ts, ts + 32, tb, tb + 32, tb + 64, x, a);
        };
        // the band aligned to this row and added to its 64 fp32 content
        // logits.  The shift runs on the band rounded to fp16 pairs (11-bit
        // significand, saturated to the finite range): three select stages
        // move whole registers (shift / 2) within a 40-register window, one
        // byte permute moves half a register (shift & 1), then each fp16 is
        // added to its fp32 logit.
        const uint32_t odd_sel = (shift & 1) ? 0x5432u : 0x3210u;
        auto band_all = [&](uint32_t *w, float *xb) {
#pragma unroll
            for (int y = 0; y < 36; ++y) w[y] = (shift & 8) ? w[y + 4] : w[y];
#pragma unroll
            for (int y = 0; y < 34; ++y) w[y] = (shift & 4) ? w[y + 2] : w[y];
#pragma unroll
            for (int y = 0; y < 33; ++y) w[y] = (shift & 2) ? w[y + 1] : w[y];
#pragma unroll
            for (int k = 0; k < 32; ++k) add_f16x2_to(xb[2 * k], xb[2 * k + 1], __byte_perm(w[k], w[k + 1], odd_sel));
        };
        // the same for 32 keys from a 24-register piece of the window (keys
        // 0-31: registers 0-23, keys 32-63: registers 16-39), so that the
        // exponentials of one piece can overlap the shifts of the other
        auto band_half = [&](const uint32_t *w0, float *xb) {
            uint32_t w[24];
#pragma unroll
            for (int y = 0; y < 24; ++y) w[y] = w0[y];
#pragma unroll
            for (int y = 0; y < 20; ++y) w[y] = (shift & 8) ? w[y + 4] : w[y];
#pragma unroll
            for (int y = 0; y < 18; ++y) w[y] = (shift & 4) ? w[y + 2] : w[y];
#pragma unroll
            for (int y = 0; y < 17; ++y) w[y] = (shift & 2) ? w[y + 1] : w[y];
#pragma unroll
            for (int k = 0; k < 16; ++k) add_f16x2_to(xb[2 * k], xb[2 * k + 1], __byte_perm(w[k], w[k + 1], odd_sel));
        };
        // keys past the row's causal limit (j > M+i) get -inf
        auto mask_block = [&](float *xb, int first, int lim) {
#pragma unroll
            for (int y = 0; y < 32; ++y) xb[y] = (first + y <= lim) ? xb[y] : -INFINITY;
        };
        auto rowmax32 = [&](const float *x) {
            float q1[11];
#pragma unroll
            for (int y = 0; y < 10; ++y) q1[y] = max3(x[3 * y], x[3 * y + 1], x[3 * y + 2]);
            q1[10] = fmaxf(x[30], x[31]);
            return max3(max3(q1[0], q1[1], q1[2]), max3(q1[3], q1[4], q1[5]),
                        max3(q1[6], q1[7], max3(q1[8], q1[9], q1[10])));
        };
        // 2^(x - mu) of 32 logits, packed to bf16 pairs; returns their sum.
        // The subtraction and the sum run on element pairs (f32x2).
        auto expo = [&](const float *x, float mu, float *pk) {
            const uint64_t mu2 = f2(mu, mu);
            uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
            for (int y = 0; y < 16; ++y) {
                float e0, e1;
                unf2(sub2(f2(x[2 * y], x[2 * y + 1]), mu2), e0, e1);
                const float p0 = ex2(e0), p1 = ex2(e1);
                acc[y & 1] = add2(acc[y & 1], f2(p0, p1));
                pk[y] = __uint_as_float(pack_bf16(p0, p1));
            }
            float s0, s1, s2, s3;
            unf2(acc[0], s0, s1);
            unf2(acc[1], s2, s3);
            return (s0 + s1) + (s2 + s3);
        };
        // the other half of this thread's row (lane ^ 16)
        auto partner = [&](float v) { return __shfl_xor_sync(0xffffffffu, v, 16); };

        constexpr int DH = DP / 2;                 // O columns of each key-half lane
        const uint32_t to = tl + TM_O;
        // an item's output: O / l for this thread's half of the columns
        struct Done {
            long head_off;
            int i0, rows_here, bh, split, whole;
            float m, l;
        };
        int n_out = 0;                             // items stored through the output buffer
        auto epilogue = [&](const Done &dn, int g_last, bool last) {
            if (!wwait(S::B_PV, g_last & 1)) return false;
            const float l = dn.l + partner(dn.l);
            tc_fence_after();
            float o[DH];
#pragma unroll
            for (int c = 0; c < DH / 8; ++c) tmem_ld_h8<DH>(to + 8 * c, o + 8 * c);
            tc_fence_before();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int d0 = DH * half;
            const int i = dn.i0 + ii;
            if (p.lse && dn.whole && half == 0 && ii < dn.rows_here)
                p.lse[(long)dn.bh * p.L + i] = l > 0.f ? (dn.m + log2f(l)) * LN2 : -INFINITY;
            if (!dn.whole && half == 0 && ii < dn.rows_here)   // m is in log2 units of the scaled logits
                p.part_lse[((long)dn.split * p.B * p.H + dn.bh) * p.L + i] = l > 0.f ? dn.m + log2f(l) : -INFINITY;
            if (kTma && p.ost && (dn.whole || !kSK)) {
                // the 128 x 64 tile (the output, or this split's partial)
                // goes through shared memory (the tensor map's swizzled
                // layout) and out by one TMA store, issued by the P.V thread;
                // rows past L are not written.  The buffer is free once the
                // previous item's store has read it.
                if (!wwait(S::B_OFR, n_out & 1)) return false;
#pragma unroll
                for (int c = 0; c < DH / 8; ++c) {
                    uint4 pk4;
                    pk4.x = pack_bf16(o[c * 8 + 0] * inv, o[c * 8 + 1] * inv);
                    pk4.y = pack_bf16(o[c * 8 + 2] * inv, o[c * 8 + 3] * inv);
                    pk4.z = pack_bf16(o[c * 8 + 4] * inv, o[c * 8 + 5] * inv);
                    pk4.w = pack_bf16(o[c * 8 + 6] * inv, o[c * 8 + 7] * inv);
                    *reinterpret_cast<uint4 *>(smem + S::OST + sw128_offset(ii, d0 + 8 * c)) = pk4;
                }
                fence_proxy_async_smem();
                if (last) mbar_arrive(bar(S::B_OST));   // no later P barrier shows it
                ++n_out;
                return true;
            }
            if (ii >= dn.rows_here) return true;
            if (dn.whole) {
                __nv_bfloat16 *op = p.out + (long)i * qkv_row + dn.head_off + d0;
                if ((p.D & 7) == 0) {
#pragma unroll
                    for (int d8 = 0; d8 < DH / 8; ++d8) {
                        if (d0 + d8 * 8 < p.D) {
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
                    for (int d = 0; d < DH; ++d)
                        if (d0 + d < p.D) op[d] = __float2bfloat16(o[d] * inv);
                }
            } else {
                // this split's partial row (bf16, 16-byte pieces: DH is a multiple of 8)
                const long BH = (long)p.B * p.H;
                __nv_bfloat16 *po = p.part_o + (((long)i * p.splits + dn.split) * BH + dn.bh) * DP + d0;
#pragma unroll
                for (int d8 = 0; d8 < DH / 8; ++d8) {
                    uint4 pk4;
                    pk4.x = pack_bf16(o[d8 * 8 + 0] * inv, o[d8 * 8 + 1] * inv);
                    pk4.y = pack_bf16(o[d8 * 8 + 2] * inv, o[d8 * 8 + 3] * inv);
                    pk4.z = pack_bf16(o[d8 * 8 + 4] * inv, o[d8 * 8 + 5] * inv);
                    pk4.w = pack_bf16(o[d8 * 8 + 6] * inv, o[d8 * 8 + 7] * inv);
                    *reinterpret_cast<uint4 *>(po + d8 * 8) = pk4;
                }
            }
            return true;
        };
        // items without key tiles (empty key splits) only get neutral partials
        auto neutral = [&](int jfrom, int jto) {
            if (kSK) return;                 // every part of the stream-K schedule has key tiles
            for (int q = jfrom; q < jto; ++q) {
                const int k = item_of(p, q);
                if (k < 0) break;
                const Item e = make_item(p, k);
                if (e.N <= 0 && half == 0 && ii < e.rows_here) {
                    const long BH = (long)p.B * p.H, ir = e.i0 + ii;
                    p.part_lse[((long)e.split * BH + e.bh) * p.L + ir] = -INFINITY;
                    __nv_bfloat16 *po = p.part_o + ((ir * p.splits + e.split) * BH + e.bh) * DP;
                    for (int d = 0; d < DP; ++d) po[d] = __float2bfloat16(0.f);
                }
            }
        };

        bool ok = true;
        Item it;
        int j = next_busy<kSK>(p, 0, it);
        if (j >= 0) ok = convert_q(it, 0);
        int g = 0, ni = 0;
        bool pending = false;                      // the previous item's output is still in O
        Done prev;
        neutral(0, j >= 0 ? j : 1 << 30);
        while (ok && j >= 0) {
            const int i = it.i0 + ii;
            const bool row_valid = ii < it.rows_here;
            Item nx;
            const int jn = next_busy<kSK>(p, j + 1, nx);
            float m_used = -INFINITY, l_run = 0.f;     // l_run: this thread's key half only
            for (int n = 0; n < it.N; ++n, ++g) {
                const int j0 = (it.t0 + n) * BN + HN * half;     // first key of this thread's half
                if (!wwait(S::B_S, g & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the item's last S MMAs have read q+u, q+v: the next item's
                // operands go in now, so that its first MMAs overlap the rest
                // of this item
                if (n == it.N - 1 && jn >= 0 && !convert_q(nx, ni + 1)) {
                    ok = false;
                    break;
                }
                // the mask matters only where the warp's rows meet the diagonal
                const bool diag = (it.t0 + n) * BN + BN - 1 > p.M + it.i0 + lb;
                const int lim = row_valid ? (p.M + i - j0) : (p.T - 1 - j0);
                float x[64], a[80];
                load_tile(x, a);
                tc_fence_before();
                mbar_arrive(bar(S::B_SF));
                uint32_t hb[40];
#pragma unroll
                for (int y = 0; y < 40; ++y) hb[y] = pack_f16_sat(a[2 * y], a[2 * y + 1]);
                // exponentials against the running reference max.  Once the
                // rows have a finite reference the tile runs straight
                // through: shift, add (on diagonal tiles the causal mask) and
                // exponentials of the two 32-key pieces.  The row's sum over
                // all 128 keys is then checked (the row's two lanes see the
                // same sum and the whole warp takes one branch): past
                // SUM_LIMIT, and on the first tile of an item, the reference
                // is first raised to the row's max.
                float pk[32], psum = 0.f, alpha = 1.f;
                bool raise = false, find_max;
                if (!__any_sync(0xffffffffu, m_used == -INFINITY)) {
                    band_half(hb, x);
                    if (diag) mask_block(x, 0, lim);
                    const float s0 = expo(x, m_used, pk);
                    band_half(hb + 16, x + 32);
                    if (diag) mask_block(x + 32, 32, lim);
                    const float s1 = expo(x + 32, m_used, pk + 16);
                    psum = s0 + s1;
                    find_max = __any_sync(0xffffffffu, !(psum + partner(psum) <= SUM_LIMIT));
                } else {
                    band_all(hb, x);
                    if (diag) {
                        mask_block(x, 0, lim);
                        mask_block(x + 32, 32, lim);
                    }
                    find_max = true;
                }
                if (find_max) {
                    float lmax = fmaxf(rowmax32(x), rowmax32(x + 32));
                    lmax = fmaxf(lmax, partner(lmax));
                    const float m_new = fmaxf(m_used, lmax);
                    if (m_new > m_used) {
                        alpha = ex2(m_used - m_new);      // 0 when m_used = -inf
                        m_used = m_new;
                        raise = true;
                    }
                    const float mu = (m_used == -INFINITY) ? 0.f : m_used;   // a row masked so far
                    psum = expo(x, mu, pk) + expo(x + 32, mu, pk + 16);
                }
                l_run = l_run * alpha + psum;
                if (n == 0) {
                    // the previous item's output leaves O before this item's
                    // first P.V overwrites it; its last P.V has long finished
                    if (pending && !epilogue(prev, g - 1, false)) {
                        ok = false;
                        break;
                    }
                    pending = false;
                } else if (!wwait(S::B_PV, (g - 1) & 1)) {
                    // P in TMEM and O are free once the P.V of tile g-1 is done
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (n >= 1 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
                    for (int c = 0; c < DH / 8; ++c) {
                        float o[8];
                        tmem_ld_h8<DH>(to + 8 * c, o);
#pragma unroll
                        for (int y = 0; y < 8; ++y) o[y] *= alpha;
                        tmem_st_h8<DH>(to + 8 * c, o);
                    }
                }
                tmem_st_h32<HN / 2>(tl + TM_P, *reinterpret_cast<float(*)[32]>(pk));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(S::B_P));
            }
            if (!ok) break;
            prev.head_off = it.head_off;
            prev.i0 = it.i0;
            prev.rows_here = it.rows_here;
            prev.bh = it.bh;
            prev.split = it.split;
            prev.whole = it.whole;
            prev.m = m_used;
            prev.l = l_run;
            pending = true;
            neutral(j + 1, jn >= 0 ? jn : 1 << 30);
            j = jn;
            it = nx;
            ++ni;
        }
        if (ok && pending) epilogue(prev, g - 1, true);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// ------------------------------------------------------------ backward scores
// The score side of the backward (txl_rel_attn_bwd, bf16, D = 64): for each
// 128-row block of one (b, h) and each 128-key tile, the tile's content and
// band products (as in the forward) and dP = dO V^T on the tensor cores, then
// per row P = 2^(s - lse) (the forward's log-sum-exp) and
// dA = P (dP - delta) / sqrt(D) (delta = rowsum(dO * O)); P and dA are written
// as bf16 [B*H][L][TP] matrices, and dA once more in the table's column
// frame (row i moved right by L-1-i: column c holds the pair of key
// c - (L-1-i)), the operands of the backward's plain contractions.
constexpr int BW_NSTAGE = 2;      // K/V stages
constexpr int BW_NCH = 3;         // table chunk slots
constexpr uint32_t TM_DP = 384;   // dP of the tile, 128 columns

struct BwdSmem {
    static constexpr uint32_t TILE = BN * 128;
    static constexpr uint32_t KV = 2 * TILE;
    static constexpr uint32_t QT = BM * 128;
    static constexpr uint32_t ST0 = 0;
    static constexpr uint32_t CH0 = BW_NSTAGE * KV;
    static constexpr uint32_t QU = CH0 + BW_NCH * TILE;
    static constexpr uint32_t QV = QU + QT;
    static constexpr uint32_t DO0 = QV + QT;                // two dO buffers (items alternate)
    static constexpr uint32_t QRAW = DO0 + 2 * QT;
    static constexpr uint32_t STG = QRAW + QT;              // per softmax warp: 16 rows of 256 bytes of dA
    static constexpr uint32_t UW = STG + 8 * 16 * 256;
    static constexpr uint32_t BARS = UW + 2 * 64 * 4;
    // q+u/q+v ready; raw q (+ u, v, the item's dO) ready, raw q read; per
    // K/V stage full / empty; per chunk slot full / empty; S, band, dP
    // full; S, band, dP free (loaded by the softmax)
    static constexpr int B_Q = 0, B_QRAW = 1, B_QRF = 2, B_FULL = 3, B_EMPTY = 3 + BW_NSTAGE,
                         B_CHF = 3 + 2 * BW_NSTAGE, B_CHE = B_CHF + BW_NCH, B_S = B_CHE + BW_NCH,
                         B_SF = B_S + 1;
    static_assert(B_SF < 32, "barrier slots");
    static constexpr uint32_t MISC = BARS + 32 * 8;
    static constexpr uint32_t USED = MISC + 16;
    static constexpr uint32_t TOTAL = USED + 1024;
};

__global__ void __launch_bounds__(NT, 1)
rel_attn_bwd_scores_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_do, const Params p)
{
    using S = BwdSmem;
    constexpr int DP = 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + S::BARS + 8u * (uint32_t)i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::MISC + 8);
    auto wwait = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_or_abort(bar(i), parity, abort)) != 0;
    };

    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        *abort = 0;
        mbar_init(bar(S::B_Q), 256);
        mbar_init(bar(S::B_QRAW), 1);
        mbar_init(bar(S::B_QRF), 256);
        for (int x = 0; x < BW_NSTAGE; ++x) {
            mbar_init(bar(S::B_FULL + x), 1);
            mbar_init(bar(S::B_EMPTY + x), 1);
        }
        for (int x = 0; x < BW_NCH; ++x) {
            mbar_init(bar(S::B_CHF + x), 1);
            mbar_init(bar(S::B_CHE + x), 1);
        }
        mbar_init(bar(S::B_S), 1);
        mbar_init(bar(S::B_SF), 256);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_r);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp < 4) {
        setmaxnreg_dec<REG_LOW>();
        if (warp == 0) {
            // =============================================================== producer
            // an item's raw q rows, its head's biases and its dO rows (into
            // the dO buffer of its parity)
            auto load_q = [&](const Item &it, int ni) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_QRAW), 2 * S::QT + 2 * 64 * 4);
                    tma_load_3d(sbase + S::QRAW, &tm_q, bar(S::B_QRAW), 0, it.i0, it.bh);
                    tma_load_3d(sbase + S::DO0 + (uint32_t)(ni & 1) * S::QT, &tm_do, bar(S::B_QRAW), 0, it.i0,
                                it.bh);
                    bulk_load(sbase + S::UW, p.u + it.h * p.D, 64 * 4, bar(S::B_QRAW));
                    bulk_load(sbase + S::UW + 256, p.w + it.h * p.D, 64 * 4, bar(S::B_QRAW));
                }
            };
            auto load_chunk = [&](int cg, int row, int h) {
                const int slot = cg % BW_NCH;
                if (cg >= BW_NCH && !wwait(S::B_CHE + slot, ((cg / BW_NCH) - 1) & 1)) return false;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_CHF + slot), S::TILE);
                    tma_load_3d(sbase + S::CH0 + slot * S::TILE, &tm_r, bar(S::B_CHF + slot), 0, row, h);
                }
                return true;
            };
            Item it;
            int j = next_busy<false>(p, 0, it);
            if (j >= 0) load_q(it, 0);
            int g = 0, cg = 0, ni = 0;
            bool ok = true;
            while (ok && j >= 0) {
                if (!load_chunk(cg, it.kb0, it.h)) break;
                ++cg;
                for (int n = 0; n < it.N; ++n, ++g) {
                    const int st = g % BW_NSTAGE;
                    if (g >= BW_NSTAGE && !wwait(S::B_EMPTY + st, ((g / BW_NSTAGE) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int j0 = (it.t0 + n) * BN;
                    const uint32_t dst = sbase + S::ST0 + st * S::KV;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar(S::B_FULL + st), S::KV);
                        tma_load_3d(dst, &tm_k, bar(S::B_FULL + st), 0, j0, it.bh);
                        tma_load_3d(dst + S::TILE, &tm_v, bar(S::B_FULL + st), 0, j0, it.bh);
                    }
                    if (!load_chunk(cg, it.kb0 + (n + 1) * BN, it.h)) {
                        ok = false;
                        break;
                    }
                    ++cg;
                }
                if (!ok) break;
                Item nx;
                const int jn = next_busy<false>(p, j + 1, nx);
                if (jn >= 0) {
                    if (!wwait(S::B_QRF, ni & 1)) break;
                    load_q(nx, ni + 1);
                }
                j = jn;
                it = nx;
                ++ni;
            }
        } else if (warp == 1) {
            // =============================================================== S, band, dP MMAs
            if (lane == 0) {
                const uint32_t idesc_n = idesc_bf16(BM, BN, 0, 0);
                const uint32_t idesc_w = idesc_bf16(BM, 2 * BN, 0, 0);
                const uint64_t d_qu = smem_desc_sw128(sbase + S::QU, 16, 1024);
                const uint64_t d_qv = smem_desc_sw128(sbase + S::QV, 16, 1024);
                const uint64_t d_do0 = smem_desc_sw128(sbase + S::DO0, 16, 1024);
                const uint64_t d_st0 = smem_desc_sw128(sbase + S::ST0, 16, 1024);
                const uint64_t d_ch0 = smem_desc_sw128(sbase + S::CH0, 16, 1024);
                constexpr uint64_t KV16 = S::KV >> 4, TILE16 = S::TILE >> 4, QT16 = S::QT >> 4;
                Item it;
                int g = 0, cg = 0, ni = 0;
                bool ok = true;
                for (int j = next_busy<false>(p, 0, it); ok && j >= 0; j = next_busy<false>(p, j + 1, it), ++ni) {
                    if (!wait_or_abort(bar(S::B_Q), ni & 1, abort)) break;
                    const uint64_t d_do = d_do0 + (uint64_t)(ni & 1) * QT16;
                    const int c0 = cg;
                    for (int n = 0; n < it.N; ++n, ++g) {
                        const int st = g % BW_NSTAGE;
                        const int ca = c0 + n, cb = ca + 1, sa = ca % BW_NCH, sb = cb % BW_NCH;
                        if (g >= 1) ok = wait_or_abort(bar(S::B_SF), (g - 1) & 1, abort);
                        ok = ok && wait_or_abort(bar(S::B_FULL + st), (g / BW_NSTAGE) & 1, abort) &&
                             wait_or_abort(bar(S::B_CHF + sa), (ca / BW_NCH) & 1, abort) &&
                             wait_or_abort(bar(S::B_CHF + sb), (cb / BW_NCH) & 1, abort);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t dk = d_st0 + st * KV16, dv = dk + TILE16;
                        const uint64_t da = d_ch0 + sa * TILE16, db = d_ch0 + sb * TILE16;
#pragma unroll
                        for (int ks = 0; ks < DP / 16; ++ks) {
                            mma_bf16_ss(tmem + TM_S, d_qu + 2 * ks, dk + 2 * ks, idesc_n, ks > 0);
                            if (sb == sa + 1) {
                                mma_bf16_ss(tmem + TM_BAND, d_qv + 2 * ks, da + 2 * ks, idesc_w, ks > 0);
                            } else {
                                mma_bf16_ss(tmem + TM_BAND, d_qv + 2 * ks, da + 2 * ks, idesc_n, ks > 0);
                                mma_bf16_ss(tmem + TM_BAND + BN, d_qv + 2 * ks, db + 2 * ks, idesc_n, ks > 0);
                            }
                            // dP = dO V^T: V rows are K-major for N = keys, like K
                            mma_bf16_ss(tmem + TM_DP, d_do + 2 * ks, dv + 2 * ks, idesc_n, ks > 0);
                        }
                        mma_commit(bar(S::B_S));
                        mma_commit(bar(S::B_EMPTY + st));
                        mma_commit(bar(S::B_CHE + sa));
                        if (n == it.N - 1) mma_commit(bar(S::B_CHE + sb));
                    }
                    cg = c0 + it.N + 1;
                }
            }
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<REG_HIGH>();
        // =============================================================== scores
        const int quarter = warp & 3, rh = (warp - 4) >> 2;
        const int r16 = lane & 15, half = lane >> 4;
        const int lb = quarter * 32 + rh * 16;
        const int ii = lb + r16;
        const uint32_t tl = tmem + ((uint32_t)lb << 16);
        constexpr int DC = DP / 16;
        auto convert_q = [&](const Item &it, int ni) {
            if (!wwait(S::B_QRAW, ni & 1)) return false;
            const float4 *uw4 = reinterpret_cast<const float4 *>(smem + S::UW);
            const float keep = ii < it.rows_here ? 1.f : 0.f;
            uint4 raw[DC];
            float4 u4[2 * DC], w4[2 * DC];
#pragma unroll
            for (int c = 0; c < DC; ++c)
                raw[c] = *reinterpret_cast<const uint4 *>(smem + S::QRAW + sw128_offset(ii, 8 * (DC * half + c)));
#pragma unroll
            for (int d4 = 0; d4 < 2 * DC; ++d4) {
                u4[d4] = uw4[2 * DC * half + d4];
                w4[d4] = uw4[16 + 2 * DC * half + d4];
            }
            const float sk = p.sl2 * keep;
            const uint64_t sk2 = f2(sk, sk);
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const int d8 = DC * half + c;
                const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&raw[c]);
                const float *uu = reinterpret_cast<const float *>(&u4[2 * c]);
                const float *ww = reinterpret_cast<const float *>(&w4[2 * c]);
                uint32_t a4[4], c4[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    // (q + u) s as q s + (u s), on element pairs
                    const uint64_t q2 = f2(__bfloat162float(e[2 * z]), __bfloat162float(e[2 * z + 1]));
                    float a0, a1, b0, b1;
                    unf2(fma2(q2, sk2, mul2(f2(uu[2 * z], uu[2 * z + 1]), sk2)), a0, a1);
                    unf2(fma2(q2, sk2, mul2(f2(ww[2 * z], ww[2 * z + 1]), sk2)), b0, b1);
                    a4[z] = pack_bf16(a0, a1);
                    c4[z] = pack_bf16(b0, b1);
                }
                *reinterpret_cast<uint4 *>(smem + S::QU + sw128_offset(ii, 8 * d8)) =
                    make_uint4(a4[0], a4[1], a4[2], a4[3]);
                *reinterpret_cast<uint4 *>(smem + S::QV + sw128_offset(ii, 8 * d8)) =
                    make_uint4(c4[0], c4[1], c4[2], c4[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(S::B_Q));
            mbar_arrive(bar(S::B_QRF));
            return true;
        };
        const int shift = 15 - r16;
        const int W0 = 112 - lb;
        const uint32_t odd_sel = (shift & 1) ? 0x5432u : 0x3210u;
        auto band_all = [&](uint32_t *w, float *xb) {
#pragma unroll
            for (int y = 0; y < 36; ++y) w[y] = (shift & 8) ? w[y + 4] : w[y];
#pragma unroll
            for (int y = 0; y < 34; ++y) w[y] = (shift & 4) ? w[y + 2] : w[y];
#pragma unroll
            for (int y = 0; y < 33; ++y) w[y] = (shift & 2) ? w[y + 1] : w[y];
#pragma unroll
            for (int k = 0; k < 32; ++k) add_f16x2_to(xb[2 * k], xb[2 * k + 1], __byte_perm(w[k], w[k + 1], odd_sel));
        };
        // dA of this warp's 16 rows staged for the table-frame copy: row r at
        // 256 bytes, 16-byte chunk c at position c ^ (r & 7) (conflict-free
        // both for the rows' chunk writes and the warp's column reads)
        unsigned char *stg = smem + S::STG + (uint32_t)(warp - 4) * 16 * 256;
        auto stg_off = [&](int r, int col) {   // byte offset of element col of row r
            return r * 256 + ((((col >> 3) ^ (r & 7)) & 15) << 4) + ((col & 7) << 1);
        };
        const long rowpitch = p.TP;
        bool ok = true;
        Item it;
        int j = next_busy<false>(p, 0, it);
        if (j >= 0) ok = convert_q(it, 0);
        int g = 0, ni = 0;
        while (ok && j >= 0) {
            const int i = it.i0 + ii;
            const bool row_valid = ii < it.rows_here;
            Item nx;
            const int jn = next_busy<false>(p, j + 1, nx);
            const long row = (long)it.bh * p.L + i;   // this thread's row of the [B*H][L] matrices
            const float lse = row_valid ? p.lse[row] * LOG2E : 0.f;   // log2 units of the scaled score
            // the table-frame matrix is head-major, [H][L][B][TP]: row (i, b) of
            // head h, so that one GEMM per head contracts over (i, b)
            auto db_row = [&](int ir) { return (((long)it.h * p.L + ir) * p.B + it.b) * rowpitch; };
            // delta = rowsum(dO * O): this thread's half of the row, dO from
            // the item's operand buffer (loaded with its q rows), O from the
            // forward's output
            float delta;
            {
                float acc = 0.f;
                if (row_valid) {
                    const unsigned char *dob = smem + S::DO0 + (uint32_t)(ni & 1) * S::QT;
                    const uint4 *op = reinterpret_cast<const uint4 *>(
                        p.out + ((long)i * p.B * p.H + it.bh) * DP + 32 * half);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 dv4 = *reinterpret_cast<const uint4 *>(dob + sw128_offset(ii, 32 * half + 8 * c));
                        const uint4 ov4 = op[c];
                        const __nv_bfloat16 *de = reinterpret_cast<const __nv_bfloat16 *>(&dv4);
                        const __nv_bfloat16 *oe = reinterpret_cast<const __nv_bfloat16 *>(&ov4);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc += __bfloat162float(de[e]) * __bfloat162float(oe[e]);
                    }
                }
                delta = acc + __shfl_xor_sync(0xffffffffu, acc, 16);
            }
            // keys past the item's last tile are masked for all its rows: P
            // and dA there are zeros (the columns up to the row pitch); and
            // the table frame of the rows before their first key (no key
            // lands there) is zero.  Each warp clears its 16 rows with
            // contiguous 16-byte stores.
            {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                const long c_end = (long)(it.t0 + it.N) * BN;
                for (int r = 0; r < 16; ++r) {
                    const int ir = it.i0 + lb + r;
                    if (ir >= p.L) break;
                    const long rr = ((long)it.bh * p.L + ir) * rowpitch;
                    for (long c = c_end + 8 * lane; c < rowpitch; c += 256) {
                        *reinterpret_cast<uint4 *>(p.p_out + rr + c) = z;
                        *reinterpret_cast<uint4 *>(p.da_out + rr + c) = z;
                    }
                    if (it.t0 == 0) {
                        const int pre = p.L - 1 - ir;                // table columns before key 0
                        const long dr0 = db_row(ir);
                        for (int c = 8 * lane; c < pre; c += 256) {
                            if (c + 8 <= pre)
                                *reinterpret_cast<uint4 *>(p.db_out + dr0 + c) = z;
                            else
                                for (int e = c; e < pre; ++e) p.db_out[dr0 + e] = __float2bfloat16(0.f);
                        }
                    }
                }
            }
            for (int n = 0; n < it.N; ++n, ++g) {
                const int jt = (it.t0 + n) * BN;                 // the tile's first key
                const int j0 = jt + HN * half;                    // first key of this thread's half
                if (!wwait(S::B_S, g & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (n == it.N - 1 && jn >= 0 && !convert_q(nx, ni + 1)) {
                    ok = false;
                    break;
                }
                const bool diag = jt + BN - 1 > p.M + it.i0 + lb;
                const int lim = row_valid ? (p.M + i - j0) : -1;   // rows past L: nothing visible
                float x[64];
                {
                    float a[80];
                    const uint32_t ts = tl + TM_S, tb = tl + TM_BAND + (uint32_t)W0;
                    tmem_ld_h_tile<HN>(ts, ts + 32, tb, tb + 32, tb + 64, x, a);
                    uint32_t hb[40];
#pragma unroll
                    for (int y = 0; y < 40; ++y) hb[y] = pack_f16_sat(a[2 * y], a[2 * y + 1]);
                    band_all(hb, x);
                }
                if (diag) {
#pragma unroll
                    for (int y = 0; y < 64; ++y) x[y] = (y <= lim) ? x[y] : -INFINITY;
                }
                // P from the forward's log-sum-exp (0 where masked); the
                // subtraction on element pairs
                {
                    const uint64_t lse2 = f2(lse, lse);
#pragma unroll
                    for (int y = 0; y < 32; ++y) {
                        float e0, e1;
                        unf2(sub2(f2(x[2 * y], x[2 * y + 1]), lse2), e0, e1);
                        x[2 * y] = ex2(e0);
                        x[2 * y + 1] = ex2(e1);
                    }
                }
                float dp[64];
                tmem_ld_h64<HN>(tl + TM_DP, tl + TM_DP + 32, dp);
                tc_fence_before();
                mbar_arrive(bar(S::B_SF));
                uint32_t pp[32], aa[32];   // this row's P and dA, bf16 pairs
                {
                    // dA = P (dP - delta) / sqrt(D) = P (dP c - delta c), c = 1/sqrt(D),
                    // on element pairs
                    const float c = p.inv_sqrt_d;
                    const uint64_t c2 = f2(c, c), ndc2 = f2(-delta * c, -delta * c);
#pragma unroll
                    for (int y = 0; y < 32; ++y) {
                        const uint64_t x2 = f2(x[2 * y], x[2 * y + 1]);
                        float a0, a1;
                        unf2(mul2(x2, fma2(f2(dp[2 * y], dp[2 * y + 1]), c2, ndc2)), a0, a1);
                        pp[y] = pack_bf16(x[2 * y], x[2 * y + 1]);
                        aa[y] = pack_bf16(a0, a1);
                    }
                }
                // P and dA go out through the warp's staging tile: a thread
                // stages its row's 64 values, then two rows per store
                // instruction leave as contiguous 256-byte runs
                auto stage = [&](const uint32_t *v) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(stg + stg_off(r16, 64 * half + 8 * c)) =
                            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                    __syncwarp();
                };
                auto write_rows = [&](__nv_bfloat16 *dstm) {
                    const int ch = lane & 15;
                    __nv_bfloat16 *base = dstm + ((long)it.bh * p.L + it.i0 + lb + (lane >> 4)) * rowpitch + jt + 8 * ch;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int r = 2 * k + (lane >> 4);
                        if (it.i0 + lb + r < p.L)
                            *reinterpret_cast<uint4 *>(base + (long)(2 * k) * rowpitch) =
                                *reinterpret_cast<const uint4 *>(stg + r * 256 + ((ch ^ (r & 7)) << 4));
                    }
                    __syncwarp();
                };
                stage(pp);
                write_rows(p.p_out);
                stage(aa);
                write_rows(p.da_out);
                // dA in the table frame from the same staged rows: row i's 128
                // values start at column L-1-i+jt.  Each lane takes staged
                // words lane and lane+32 (keys 2w, 2w+1); when that column is
                // odd the pairs are realigned with the neighbouring lane's
                // word (one element across), the two end elements on their own.
                {
                    const int x0 = lane >> 2, y0 = (lane & 3) << 2;     // word lane: 16-byte chunk, offset
                    for (int r = 0; r < 16; ++r) {
                        const int ir = it.i0 + lb + r;
                        if (ir >= p.L) break;
                        const unsigned char *srow = stg + r * 256;
                        const int sw = r & 7;
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(srow + ((x0 ^ sw) << 4) + y0);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(srow + (((x0 + 8) ^ sw) << 4) + y0);
                        const long c0 = (long)(p.L - 1 - ir) + jt;
                        const long room = rowpitch - c0;                   // columns left in the row
                        __nv_bfloat16 *dst = p.db_out + db_row(ir) + c0;
                        if ((c0 & 1) == 0) {
                            if (2 * lane + 1 < room) *reinterpret_cast<uint32_t *>(dst + 2 * lane) = w0;
                            if (2 * lane + 65 < room) *reinterpret_cast<uint32_t *>(dst + 2 * lane + 64) = w1;
                        } else {
                            // pair l = (element 2l-1, element 2l): high half of word l-1, low half of word l
                            const uint32_t up0 = __shfl_up_sync(0xffffffffu, w0, 1);
                            const uint32_t up1 = __shfl_up_sync(0xffffffffu, w1, 1);
                            const uint32_t w0_31 = __shfl_sync(0xffffffffu, w0, 31);
                            const uint32_t prev1 = lane == 0 ? w0_31 : up1;
                            if (lane > 0 && 2 * lane < room)
                                *reinterpret_cast<uint32_t *>(dst + 2 * lane - 1) = __byte_perm(up0, w0, 0x5432);
                            if (2 * lane + 64 < room)
                                *reinterpret_cast<uint32_t *>(dst + 2 * lane + 63) = __byte_perm(prev1, w1, 0x5432);
                            if (lane == 0 && room > 0)
                                reinterpret_cast<unsigned short *>(dst)[0] = (unsigned short)(w0 & 0xFFFFu);
                            if (lane == 31 && 127 < room)
                                reinterpret_cast<unsigned short *>(dst)[127] = (unsigned short)(w1 >> 16);
                        }
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            j = jn;
            it = nx;
            ++ni;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// Merge the key-split partials: one thread per output row (b, h, i) and
// 8-column chunk, rows numbered bh*L + i.  The row's weights 2^(lse_s - max)
// come from its splits' log-sum-exps (the same few words for the row's
// threads); each split's chunk is one 16-byte load, several in flight.
__global__ void __launch_bounds__(256)
rel_attn_combine_kernel(const __nv_bfloat16 *__restrict__ part_o, const float *__restrict__ part_lse,
                        __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out, int splits, int B, int H,
                        int L, int D, int DP, int sk_nt, int sk_grid)
{
    const int nch = DP / 8;
    const long BH = (long)B * H, BHL = BH * L;
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= BHL * nch) return;
    const long row = t / nch;
    const int c = (int)(t % nch);
    const int bh = (int)(row / L), i = (int)(row % L);
    if (sk_grid > 0) {
        // stream-K schedule: only items cut by a CTA's range boundary have
        // parts to merge (the attention kernel wrote the others); the item
        // is cut when its first and last key tiles fall in different ranges
        const long tt = BH * sk_nt, G = sk_grid;
        auto cta_of = [&](long x) {
            long cc = x * G / tt;
            while (cc + 1 < G && (cc + 1) * tt / G <= x) ++cc;
            while (cc > 0 && cc * tt / G > x) --cc;
            return cc;
        };
        if (cta_of((long)bh * sk_nt) == cta_of((long)(bh + 1) * sk_nt - 1)) return;
    }
    const int b = bh / H, h = bh % H;
    float mx = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) mx = fmaxf(mx, part_lse[sp * BHL + row]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
        const float ls = part_lse[sp * BHL + row];
        const float w = ls == -INFINITY ? 0.f : exp2f(ls - mx);
        wsum += w;
        const uint4 v = *reinterpret_cast<const uint4 *>(part_o + (((long)i * splits + sp) * BH + bh) * DP + 8 * c);
        const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int z = 0; z < 4; ++z) {
            const float2 f = __bfloat1622float2(e[z]);
            acc[2 * z] += w * f.x;
            acc[2 * z + 1] += w * f.y;
        }
    }
    if (lse_out && c == 0) lse_out[row] = wsum > 0.f ? (mx + log2f(wsum)) * LN2 : -INFINITY;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int d0 = 8 * c;
    if (d0 >= D) return;
    __nv_bfloat16 *op = out + (((long)i * B + b) * H + h) * D + d0;
    if (D % 8 == 0) {
        uint4 pk4;
        pk4.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        pk4.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        pk4.z = pack_bf16(acc[4] * inv, acc[5] * inv);
        pk4.w = pack_bf16(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4 *>(op) = pk4;
    } else {
#pragma unroll
        for (int z = 0; z < 8; ++z)
            if (d0 + z < D) op[z] = __float2bfloat16(acc[z] * inv);
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
bool encode_map(CUtensorMap *m, const void *base, long rows, long row_stride, long groups, int box_rows)
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

// Encoded maps of recent calls (a map holds only the address and the shape,
// so repeated calls on the same buffers reuse it: the encode is a driver call
// that costs about as much as a short launch).  A direct-mapped table: a
// key's slot is its hash; a new key takes the slot over.
struct MapEntry {
    bool used;
    int dev;
    const void *base;
    long rows, row_stride, groups;
    int box_rows;
    CUtensorMap map;
};
constexpr int MAP_CACHE = 1024;
std::mutex g_map_mu;
MapEntry g_maps[MAP_CACHE];

bool make_map(CUtensorMap *m, const void *base, long rows, long row_stride, long groups, int box_rows)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    uint64_t h = (uint64_t)(uintptr_t)base;
    for (uint64_t x : {(uint64_t)dev, (uint64_t)rows, (uint64_t)row_stride, (uint64_t)groups, (uint64_t)box_rows})
        h = (h ^ x) * 0x100000001b3ull;
    MapEntry &e = g_maps[(h ^ (h >> 29)) % MAP_CACHE];
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (e.used && e.dev == dev && e.base == base && e.rows == rows && e.row_stride == row_stride &&
        e.groups == groups && e.box_rows == box_rows) {
        *m = e.map;
        return true;
    }
    if (!encode_map(m, base, rows, row_stride, groups, box_rows)) return false;
    e.used = true;
    e.dev = dev;
    e.base = base;
    e.rows = rows;
    e.row_stride = row_stride;
    e.groups = groups;
    e.box_rows = box_rows;
    e.map = *m;
    return true;
}

template <int DP, bool kTma, bool kSK, int NC = 1>
cudaError_t launch_t(const Params &p, const AttnMaps<NC> &tm, cudaStream_t s)
{
    const uint32_t smem = Smem<DP>::TOTAL;
    auto kern = rel_attn_bf16_kernel<DP, kTma, kSK, NC>;
    // the shared-memory opt-in, once per device for this variant
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(opted.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_relaxed);
    }
    // persistent: one CTA per SM, each walks its share of the work items
    const int grid = p.items < device_sm_count() ? p.items : device_sm_count();
    kern<<<(unsigned)grid, NT, smem, s>>>(tm, p);
    return cudaGetLastError();
}

int dpad(int D) { return (D + 15) / 16 * 16; }

}  // namespace

namespace {
// The kernel's busiest CTA for a split count: the items of the static
// schedule (heaviest query tiles first, CTA c of G taking items c, 2G-1-c,
// 2G+c, ...) laid out exactly as the kernel does, in units of one key tile
// (~1.6 us of one SM), with one tile of fill per item (its first tile's max
// pass, the q conversion and the epilogue).
double busiest_cta(const AttnArgs &a, int num_sms, int s)
{
    const int nqt = (a.L + BM - 1) / BM;
    const long bh = (long)a.B * a.H;
    const long items = bh * nqt * s;
    const long G = items < num_sms ? items : num_sms;
    std::vector<double> load((size_t)G, 0.0);
    const long per_qt = bh * s;
    for (long k = 0; k < items; ++k) {
        const int qt = nqt - 1 - (int)(k / per_qt);
        const int split = (int)((k % per_qt) % s);
        const int i0 = qt * BM, rows = a.L - i0 < BM ? a.L - i0 : BM;
        const long kend = (long)a.M + a.L < (long)a.M + i0 + rows ? (long)a.M + a.L : (long)a.M + i0 + rows;
        const int ntile = (int)((kend + BN - 1) / BN);
        const int n = (split + 1) * ntile / s - split * ntile / s;
        if (n <= 0) continue;
        const long j = k / G, c = (j & 1) ? G - 1 - k % G : k % G;
        load[(size_t)c] += n + 1.0;
    }
    double mx = 0.0;
    for (double x : load) mx = x > mx ? x : mx;
    return mx;
}

struct SplitKey {
    int B, H, L, M, D, sms, s;
};
std::mutex g_split_mu;
SplitKey g_split_cache[64];
int g_split_count = 0, g_split_next = 0;
}  // namespace

int bf16_uniform_splits(const AttnArgs &a, int num_sms);

// The stream-K schedule applies to one query tile per (b, h) (L <= 128)
// with at least as many (b, h) as SMs, not a multiple of them: equal
// contiguous ranges of key tiles per CTA then cut each item at most once.
bool streamk_ok(const AttnArgs &a, int num_sms)
{
    const long bh = (long)a.B * a.H;
    return a.L <= BM && (a.D + 15) / 16 * 16 == 64 && bh >= num_sms && bh % num_sms != 0 && bh <= INT32_MAX;
}

// Whether a call the stream-K schedule can take runs under it: where the
// uniform model splits the shape (stream-K replaces the split: char_eval
// 93.3 -> 84.7 us), or where whole items would leave more than four fifths
// of the CTAs idle in the last round (H 16, L 128, M 1600: batch 10, 160
// items on 152 SMs, 48.6 us whole, 41.7 under stream-K; batch 12, 192
// items, 50.0 / 50.3; batch 16, 50.2 / 63.0 -- graph-replayed calls).
bool use_streamk(const AttnArgs &a, int num_sms)
{
    if (!streamk_ok(a, num_sms)) return false;
    if (bf16_uniform_splits(a, num_sms) > 1) return true;
    const long items = (long)a.B * a.H;                  // one query tile per (b, h)
    const long idle = (items + num_sms - 1) / num_sms * num_sms - items;
    return idle * 5 > (long)num_sms * 4;
}

int bf16_num_splits(const AttnArgs &a, int num_sms)
{
    return use_streamk(a, num_sms) ? 2 : bf16_uniform_splits(a, num_sms);
}

int bf16_uniform_splits(const AttnArgs &a, int num_sms)
{
    {
        std::lock_guard<std::mutex> lock(g_split_mu);
        for (int x = 0; x < g_split_count; ++x) {
            const SplitKey &k = g_split_cache[x];
            if (k.B == a.B && k.H == a.H && k.L == a.L && k.M == a.M && k.D == a.D && k.sms == num_sms) return k.s;
        }
    }
    // the busiest CTA (simulated schedule) plus, when split, what a split
    // was measured to cost on GB300: about 3 us (the merge launch) and
    // 1.25 us per MB of bf16 partials written and read back (fitted to the
    // best of 1-12 forced splits on char_eval and long-memory shapes)
    const int nqt = (a.L + BM - 1) / BM;
    const long bh = (long)a.B * a.H;
    int maxn = 1;
    for (int qt = 0; qt < nqt; ++qt) {
        const int i0 = qt * BM, rows = a.L - i0 < BM ? a.L - i0 : BM;
        const long kend = (long)a.M + i0 + rows;
        const int nt = (int)((kend + BN - 1) / BN);
        maxn = nt > maxn ? nt : maxn;
    }
    const double tile_us = 1.6;
    double best = 1e30;
    int best_s = 1;
    for (int s = 1; s <= 16 && s <= maxn; ++s) {
        double cost = busiest_cta(a, num_sms, s);
        if (s > 1) {
            const double bytes = 2.0 * s * (double)bh * a.L * (2.0 * dpad(a.D) + 4.0);
            cost += (3.0 + 1.25 * bytes / 1.0e6) / tile_us;
        }
        if (cost < best - 1e-9) {
            best = cost;
            best_s = s;
        }
    }
    std::lock_guard<std::mutex> lock(g_split_mu);
    g_split_cache[g_split_next] = SplitKey{a.B, a.H, a.L, a.M, a.D, num_sms, best_s};
    g_split_next = (g_split_next + 1) % 64;
    if (g_split_count < 64) ++g_split_count;
    return best_s;
}

size_t bf16_scratch_bytes(const AttnArgs &a, int splits)
{
    const size_t rows = (size_t)splits * a.B * a.H * a.L;
    return rows * (size_t)dpad(a.D) * 2 + rows * 4 + 256;
}

// Whether the forward launch also does the memory rollover (warp 3 of each
// CTA, otherwise idle under TMA): the pointers and size must allow 16-byte
// vectors, and a CTA's slice must take well under the attention's own time.
// One warp with sixteen 16-byte loads in flight moves about ROLL_GBS GB/s; a
// CTA's attention work is about TILE_US per 128 x 128 tile (its share of the
// launch's tiles, the per-item overhead counted as one tile).
bool roll_fuses(const AttnArgs &a, long items, int splits)
{
    constexpr double ROLL_GBS = 8.0, TILE_US = 1.6;
    if (((uintptr_t)a.roll_src & 15) || ((uintptr_t)a.roll_dst & 15) || (a.roll_bytes & 15)) return false;
    const long G = items < device_sm_count() ? items : device_sm_count();
    if (G <= 0) return false;
    const int nqt = (a.L + BM - 1) / BM;
    double tiles = 0.0;
    for (int qt = 0; qt < nqt; ++qt) {
        const long kend = (long)a.M + (long)qt * BM + (a.L - qt * BM < BM ? a.L - qt * BM : BM);
        tiles += (double)((kend + BN - 1) / BN) + splits;
    }
    tiles *= (double)a.B * a.H / (double)G;           // per CTA
    const double copy_us = (double)a.roll_bytes / (double)G / (ROLL_GBS * 1e3);
    return copy_us <= 0.5 * tiles * TILE_US;
}

cudaError_t launch_attn_bf16(const AttnArgs &a, int splits, void *scratch, cudaStream_t s)
{
    const int DP = dpad(a.D);
    if (DP > 64) return cudaErrorNotSupported;
    Params p;
    memset(&p, 0, sizeof(p));
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
    p.sl2 = LOG2E / sqrtf((float)(a.scale_d ? a.scale_d : a.D));
    p.part_o = nullptr;
    p.part_lse = nullptr;
    p.lse = a.lse;
    if (splits > 1) {
        const size_t rows = (size_t)splits * a.B * a.H * a.L;
        p.part_o = (__nv_bfloat16 *)scratch;
        p.part_lse = (float *)((char *)scratch + rows * DP * 2);
    }
    p.items = (int)((long)a.B * a.H * p.nqt * splits);
    // the stream-K schedule where it applies: the two partial slots are then
    // only the parts of items cut by a CTA's range
    p.streamk = splits == 2 && use_streamk(a, device_sm_count());
    p.sk_nt = (a.M + a.L + BN - 1) / BN;
    if (p.streamk) p.items = a.B * a.H;   // grid: one CTA per SM (B*H >= SMs)
    p.kv_start = a.kv_start;
    p.roll_src = nullptr;
    p.roll_dst = nullptr;
    p.roll_n16 = 0;
    p.ncell = 1;
    AttnMaps<1> tm;
    memset(&tm, 0, sizeof(tm));
    CUtensorMap &mk = tm.k[0], &mv = tm.v[0], &mr = tm.r[0], &mq = tm.q[0], &mo = tm.o[0], &mk8 = tm.k8,
                &mv8 = tm.v8;
    p.ost = 0;
    // TMA for D = 64 (128-byte rows); the biases then come by bulk copy,
    // which wants them 16-byte aligned.  A K/V ring whose start or length is
    // not a multiple of 8 rows is read by the thread loader (the 8-row boxes
    // of a wrapping tile must not straddle the ring's end).
    const bool ring_ok = a.kv_start == 0 || (a.kv_start % 8 == 0 && p.T % 8 == 0);
    const bool tma = a.D == 64 && ((uintptr_t)a.u & 15) == 0 && ((uintptr_t)a.w & 15) == 0 && ring_ok;
    if (tma) {
        const long bhn = (long)a.B * a.H;
        const long rs = bhn * a.D;
        if (!make_map(&mk, a.k, p.T, rs, bhn, BN) || !make_map(&mv, a.v, p.T, rs, bhn, BN) ||
            !make_map(&mr, a.r, p.T, (long)a.H * a.D, a.H, BN) || !make_map(&mq, a.q, a.L, rs, bhn, BM) ||
            !make_map(&mk8, a.k, p.T, rs, bhn, 8) || !make_map(&mv8, a.v, p.T, rs, bhn, 8))
            return cudaErrorInvalidValue;
        // the output (or with key splits, the bf16 partials laid out like it
        // over splits*B*H heads) by TMA store
        if ((splits == 1 || p.streamk) && ((uintptr_t)a.out & 15) == 0) {
            if (!make_map(&mo, a.out, a.L, rs, bhn, BM)) return cudaErrorInvalidValue;
            p.ost = 1;
        } else if (splits > 1 && !p.streamk) {
            if (!make_map(&mo, p.part_o, a.L, (long)splits * rs, (long)splits * bhn, BM)) return cudaErrorInvalidValue;
            p.ost = 1;
        }
        if (a.roll_bytes && roll_fuses(a, p.items, splits)) {
            p.roll_src = (const uint4 *)a.roll_src;
            p.roll_dst = (uint4 *)a.roll_dst;
            p.roll_n16 = (long)(a.roll_bytes / 16);
        }
    }
    cudaError_t e;
    switch (DP) {
    case 16: e = tma ? launch_t<16, true, false>(p, tm, s) : launch_t<16, false, false>(p, tm, s); break;
    case 32: e = tma ? launch_t<32, true, false>(p, tm, s) : launch_t<32, false, false>(p, tm, s); break;
    case 48: e = tma ? launch_t<48, true, false>(p, tm, s) : launch_t<48, false, false>(p, tm, s); break;
    default:
        if (p.streamk)
            e = tma ? launch_t<64, true, true>(p, tm, s) : launch_t<64, false, true>(p, tm, s);
        else
            e = tma ? launch_t<64, true, false>(p, tm, s) : launch_t<64, false, false>(p, tm, s);
        break;
    }
    if (e == cudaSuccess && splits > 1) {
        const long threads = (long)a.B * a.H * a.L * (DP / 8);
        const int sk_grid = p.streamk ? (p.items < device_sm_count() ? p.items : device_sm_count()) : 0;
        rel_attn_combine_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
            p.part_o, p.part_lse, p.out, a.lse, splits, a.B, a.H, a.L, a.D, DP, p.sk_nt, sk_grid);
        e = cudaGetLastError();
    }
    // a rollover the attention launch did not take: its own copy
    if (e == cudaSuccess && a.roll_bytes && p.roll_n16 == 0)
        e = launch_rollover(a.roll_dst, a.roll_src, a.roll_bytes, 2, s);
    return e;
}

cudaError_t launch_attn_bf16_cells(int n, const AttnArgs *a, cudaStream_t s)
{
    if (n < 2) return cudaErrorNotSupported;
    const AttnArgs &a0 = a[0];
    const int sms = device_sm_count();
    const int nqt = (a0.L + BM - 1) / BM;
    const long per_call = (long)a0.B * a0.H * nqt;
    auto al16 = [](const void *x) { return ((uintptr_t)x & 15) == 0; };
    // every call: the shape of the first, unsplit, TMA operands and output
    if (a0.D != 64 || a0.kv_start != 0 || a0.L < 1 || a0.B < 1 || a0.H < 1 || bf16_num_splits(a0, sms) != 1 ||
        per_call * ATTN_CELLS > INT32_MAX)
        return cudaErrorNotSupported;
    bool roll_in = a0.roll_bytes > 0 && roll_fuses(a0, per_call, 1);
    for (int c = 0; c < n; ++c) {
        const AttnArgs &x = a[c];
        if (x.B != a0.B || x.H != a0.H || x.D != a0.D || x.L != a0.L || x.M != a0.M || x.kv_start != 0 ||
            x.scale_d != a0.scale_d || x.lse || x.roll_bytes != a0.roll_bytes || !al16(x.u) || !al16(x.w) ||
            !al16(x.out))
            return cudaErrorNotSupported;
        if (x.roll_bytes && (!al16(x.roll_src) || !al16(x.roll_dst))) roll_in = false;
    }
    const int T = a0.M + a0.L;
    const long bhn = (long)a0.B * a0.H, rs = bhn * a0.D;
    for (int c0 = 0; c0 < n; c0 += ATTN_CELLS) {
        const int nc = n - c0 < ATTN_CELLS ? n - c0 : ATTN_CELLS;
        cudaError_t e;
        if (nc == 1) {
            AttnArgs x = a[c0];
            e = launch_attn_bf16(x, 1, nullptr, s);    // its rollover as that call decides
            if (e != cudaSuccess) return e;
            continue;
        }
        Params p;
        memset(&p, 0, sizeof(p));
        p.q = (const __nv_bfloat16 *)a[c0].q;
        p.k = (const __nv_bfloat16 *)a[c0].k;
        p.v = (const __nv_bfloat16 *)a[c0].v;
        p.r = (const __nv_bfloat16 *)a[c0].r;
        p.u = a[c0].u;
        p.w = a[c0].w;
        p.out = (__nv_bfloat16 *)a[c0].out;
        p.B = a0.B;
        p.H = a0.H;
        p.D = a0.D;
        p.L = a0.L;
        p.M = a0.M;
        p.T = T;
        p.nqt = nqt;
        p.splits = 1;
        p.sl2 = LOG2E / sqrtf((float)(a0.scale_d ? a0.scale_d : a0.D));
        p.sk_nt = (T + BN - 1) / BN;
        p.ncell = nc;
        p.items = (int)(per_call * nc);
        p.ost = 1;
        AttnMaps<ATTN_CELLS> tm;
        memset(&tm, 0, sizeof(tm));
        for (int c = 0; c < nc; ++c) {
            const AttnArgs &x = a[c0 + c];
            if (!make_map(&tm.k[c], x.k, T, rs, bhn, BN) || !make_map(&tm.v[c], x.v, T, rs, bhn, BN) ||
                !make_map(&tm.r[c], x.r, T, (long)a0.H * a0.D, a0.H, BN) ||
                !make_map(&tm.q[c], x.q, a0.L, rs, bhn, BM) || !make_map(&tm.o[c], x.out, a0.L, rs, bhn, BM))
                return cudaErrorInvalidValue;
            p.cell_u[c] = x.u;
            p.cell_w[c] = x.w;
            if (roll_in) {
                p.cell_roll_src[c] = (const uint4 *)x.roll_src;
                p.cell_roll_dst[c] = (uint4 *)x.roll_dst;
            }
        }
        if (roll_in) {
            p.roll_src = p.cell_roll_src[0];
            p.roll_dst = p.cell_roll_dst[0];
            p.roll_n16 = (long)(a0.roll_bytes / 16);
        }
        e = launch_t<64, true, false, ATTN_CELLS>(p, tm, s);
        if (e != cudaSuccess) return e;
        // rollovers the launch did not take: their own copies
        for (int c = 0; a0.roll_bytes && !roll_in && c < nc; ++c) {
            e = launch_rollover(a[c0 + c].roll_dst, a[c0 + c].roll_src, a0.roll_bytes, 2, s);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_bwd_scores(const AttnArgs &a, const void *dout, const float *lse, void *p_out, void *da_out,
                              void *db_out, long TP, cudaStream_t s)
{
    if (a.D != 64) return cudaErrorNotSupported;
    Params p;
    memset(&p, 0, sizeof(p));
    p.q = (const __nv_bfloat16 *)a.q;
    p.k = (const __nv_bfloat16 *)a.k;
    p.v = (const __nv_bfloat16 *)a.v;
    p.r = (const __nv_bfloat16 *)a.r;
    p.u = a.u;
    p.w = a.w;
    p.B = a.B;
    p.H = a.H;
    p.D = a.D;
    p.L = a.L;
    p.M = a.M;
    p.T = a.M + a.L;
    p.nqt = (a.L + BM - 1) / BM;
    p.splits = 1;
    p.ncell = 1;
    p.items = (int)((long)a.B * a.H * p.nqt);
    p.sl2 = LOG2E / sqrtf((float)a.D);
    p.lse = const_cast<float *>(lse);
    p.dout = (const __nv_bfloat16 *)dout;
    p.out = (__nv_bfloat16 *)a.out;   // the forward's output O (read: delta = rowsum(dO * O))
    p.p_out = (__nv_bfloat16 *)p_out;
    p.da_out = (__nv_bfloat16 *)da_out;
    p.db_out = (__nv_bfloat16 *)db_out;
    p.TP = TP;
    p.inv_sqrt_d = 1.f / sqrtf((float)a.D);
    const long bhn = (long)a.B * a.H, rs = bhn * a.D;
    CUtensorMap mk, mv, mr, mq, md;
    if (!make_map(&mk, a.k, p.T, rs, bhn, BN) || !make_map(&mv, a.v, p.T, rs, bhn, BN) ||
        !make_map(&mr, a.r, p.T, (long)a.H * a.D, a.H, BN) || !make_map(&mq, a.q, a.L, rs, bhn, BM) ||
        !make_map(&md, dout, a.L, rs, bhn, BM))
        return cudaErrorInvalidValue;
    const uint32_t smem = BwdSmem::TOTAL;
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(opted.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(rel_attn_bwd_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_relaxed);
    }
    const int grid = p.items < device_sm_count() ? p.items : device_sm_count();
    rel_attn_bwd_scores_kernel<<<(unsigned)grid, NT, smem, s>>>(mk, mv, mr, mq, md, p);
    return cudaGetLastError();
}

namespace {
// The failure path of the bounded waits, on its own: one warp waits on an
// mbarrier that nothing ever completes, through the same wait the kernels
// use but with the caller's limit.  The wait runs out, records the device
// error word exactly as a kernel's wait does, and the kernel returns; no
// copy, MMA or tensor memory is in flight, so nothing is left to drain.
__global__ void selftest_wait_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_or_abort(smem_u32(&bar), 0, &abort_flag, limit_ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
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
