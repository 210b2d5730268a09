// api.cu -- the C ABI of include/txl.h: argument checks, dispatch, scratch.
//
// Every argument error is found here, on the host, before anything is
// launched.  There is no CPU path: without a GPU the calls report
// TXL_ERR_CUDA.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>

#include "internal.h"
#include "txl.h"

namespace txl {

static thread_local int g_last_cuda_error = 0;

static txl_status cuda_fail(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    cudaGetLastError();   // clear the sticky-free error state of this thread
    return TXL_ERR_CUDA;
}

cudaError_t note_cuda_error(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    cudaGetLastError();
    return e;
}

int device_sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

// Library-owned scratch for split-key partial results and padded head copies:
// one buffer per (device, stream).  Calls on one stream run in order, so a
// stream's buffer is never used by two kernels at once, and calls on
// different streams never share one.  A buffer grows in stream order
// (cudaFreeAsync of the old one, cudaMallocAsync of the new one, both on that
// stream), so growing it waits for nothing on the host.
namespace {
struct Scratch {
    int dev = -1;
    cudaStream_t stream = nullptr;
    void *ptr = nullptr;
    size_t bytes = 0;
};
constexpr int kMaxScratch = 256;   // (device, stream) pairs served until txl_shutdown
std::mutex g_scratch_mu;
Scratch g_scratch[kMaxScratch];
int g_scratch_n = 0;

txl_status get_scratch(size_t bytes, cudaStream_t stream, void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    Scratch *s = nullptr;
    for (int x = 0; x < g_scratch_n; ++x)
        if (g_scratch[x].dev == dev && g_scratch[x].stream == stream) s = &g_scratch[x];
    if (!s) {
        if (g_scratch_n == kMaxScratch) return TXL_ERR_UNSUPPORTED;
        s = &g_scratch[g_scratch_n++];
        *s = Scratch{};
        s->dev = dev;
        s->stream = stream;
    }
    if (s->bytes < bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return cuda_fail(e);
        // growing the buffer allocates; a call made once outside capture first
        // sizes it, after which captured calls reuse it.
        if (cs != cudaStreamCaptureStatusNone) return TXL_ERR_UNSUPPORTED;
        if (s->ptr) {
            // earlier calls on this stream may still read it: freed in stream order
            e = cudaFreeAsync(s->ptr, stream);
            s->ptr = nullptr;
            s->bytes = 0;
            if (e != cudaSuccess) return cuda_fail(e);
        }
        const size_t want = bytes + bytes / 4;
        e = cudaMallocAsync(&s->ptr, want, stream);
        if (e != cudaSuccess) {
            s->ptr = nullptr;
            return cuda_fail(e);
        }
        s->bytes = want;
    }
    *out = s->ptr;
    return TXL_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

bool aligned(const void *p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }

// zeros standing in for an absent bias (Shaw et al.'s form has no u, v terms)
constexpr size_t kZeroBiasFloats = 1 << 16;
static __device__ __align__(256) float g_zero_bias[kZeroBiasFloats];
std::mutex g_zb_mu;
void *g_zb_addr[64] = {nullptr};

}  // namespace

cudaError_t zero_bias(size_t count, const float **out)
{
    if (count > kZeroBiasFloats) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(g_zb_mu);
    if (!g_zb_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_zero_bias);
        if (e != cudaSuccess) return e;
        g_zb_addr[dev] = p;
    }
    *out = (const float *)g_zb_addr[dev];
    return cudaSuccess;
}
}  // namespace txl

using namespace txl;

extern "C" {

// The argument checks of an attention call (no launch); TXL_OK also for an
// empty call (batch, seg_len or heads 0), whose pointers are not looked at.
static txl_status attn_checks(const void *q, const void *k, const void *v, const void *r, const float *u_bias,
                              const float *v_bias, int batch, int mem_len, int seg_len, int heads, int d_head,
                              int kv_start, txl_dtype dtype, const void *out, const float *lse)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (batch < 0 || mem_len < 0 || seg_len < 0 || heads < 0 || d_head < 1) return TXL_ERR_INVALID;
    if (batch == 0 || seg_len == 0 || heads == 0) return TXL_OK;
    if (kv_start < 0 || (long)kv_start >= (long)mem_len + seg_len) return TXL_ERR_INVALID;
    if (d_head > 128) return TXL_ERR_UNSUPPORTED;
    if (dtype == TXL_BF16 && d_head > 64) return TXL_ERR_UNSUPPORTED;
    if (!q || !k || !v || !r || !out) return TXL_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(r, 16) ||
        !aligned(out, 16) || !aligned(u_bias, 4) || !aligned(v_bias, 4))
        return TXL_ERR_INVALID;
    // sizes: every index is 64-bit in the kernels; keep byte counts in range
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    const size_t T = (size_t)mem_len + (size_t)seg_len;
    if (T > (size_t)INT32_MAX) return TXL_ERR_UNSUPPORTED;
    const size_t row = (size_t)batch * (size_t)heads * (size_t)d_head;
    const size_t nq = (size_t)seg_len * row * esz, nk = T * row * esz;
    const size_t nr = T * (size_t)heads * (size_t)d_head * esz;
    const size_t nb = (size_t)heads * (size_t)d_head * 4;
    if ((size_t)batch * (size_t)heads > (size_t)INT32_MAX || nk / esz / T != row)
        return TXL_ERR_UNSUPPORTED;
    if (overlaps(out, nq, q, nq) || overlaps(out, nq, k, nk) || overlaps(out, nq, v, nk) ||
        overlaps(out, nq, r, nr) || overlaps(out, nq, u_bias, nb) || overlaps(out, nq, v_bias, nb))
        return TXL_ERR_INVALID;
    if ((seg_len + 31) / 32 > 65535) return TXL_ERR_UNSUPPORTED;
    if (lse) {
        // the row log-sum-exp comes from the bf16 kernels
        if (dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
        const size_t nl = (size_t)batch * heads * seg_len * 4;
        if (!aligned(lse, 4) || overlaps(lse, nl, out, nq) || overlaps(lse, nl, q, nq) || overlaps(lse, nl, k, nk) ||
            overlaps(lse, nl, v, nk) || overlaps(lse, nl, r, nr))
            return TXL_ERR_INVALID;
    }
    return TXL_OK;
}

static txl_status rel_attn_common(const void *q, const void *k, const void *v, const void *r,
                                  const float *u_bias, const float *v_bias, int batch, int mem_len,
                                  int seg_len, int heads, int d_head, int kv_start, txl_dtype dtype,
                                  void *out, void *stream, int scale_d = 0, float *lse = nullptr,
                                  const void *roll_src = nullptr, void *roll_dst = nullptr, size_t roll_bytes = 0)
{
    const txl_status st = attn_checks(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head, kv_start,
                                      dtype, out, lse);
    if (st != TXL_OK) return st;
    if (batch == 0 || seg_len == 0 || heads == 0) return TXL_OK;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;

    // an absent bias drops its term (terms (a) + (b) only: Shaw et al.'s form)
    if (!u_bias || !v_bias) {
        const float *z = nullptr;
        const cudaError_t ze = zero_bias((size_t)heads * (size_t)d_head, &z);
        if (ze == cudaErrorNotSupported) return TXL_ERR_UNSUPPORTED;
        if (ze != cudaSuccess) return cuda_fail(ze);
        if (!u_bias) u_bias = z;
        if (!v_bias) v_bias = z;
    }
    AttnArgs a{q, k, v, r, u_bias, v_bias, out, batch, heads, d_head, seg_len, mem_len, kv_start, scale_d};
    a.lse = lse;
    a.roll_src = roll_src;
    a.roll_dst = roll_dst;
    a.roll_bytes = roll_bytes;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (dtype == TXL_F32) {
        e = launch_attn_f32(a, s);
        if (e == cudaSuccess && roll_bytes) e = launch_rollover(roll_dst, roll_src, roll_bytes, 4, s);
    } else if (a.D == 64) {
        const int splits = bf16_num_splits(a, device_sm_count());
        void *scratch = nullptr;
        if (splits > 1) {
            txl_status st = get_scratch(bf16_scratch_bytes(a, splits), s, &scratch);
            if (st != TXL_OK) return st;
        }
        e = launch_attn_bf16(a, splits, scratch, s);
    } else {
        // head vectors of another width: 64-wide zero-padded copies in the
        // scratch (rows TMA can read), the kernel on those, the output's first
        // D columns copied back
        constexpr int W = 64;
        const long nq = (long)seg_len * batch * heads, nk = (long)(mem_len + seg_len) * batch * heads;
        const long nr = (long)(mem_len + seg_len) * heads;
        auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
        const size_t bq = up((size_t)nq * W * 2), bk = up((size_t)nk * W * 2), br = up((size_t)nr * W * 2),
                     bb = up((size_t)heads * W * 4);
        AttnArgs ap = a;
        ap.D = W;
        ap.scale_d = a.scale_d ? a.scale_d : a.D;
        const int splits = bf16_num_splits(ap, device_sm_count());
        const size_t bs = splits > 1 ? up(bf16_scratch_bytes(ap, splits)) : 0;
        void *scratch = nullptr;
        txl_status st = get_scratch(2 * bq + 2 * bk + br + 2 * bb + bs, s, &scratch);
        if (st != TXL_OK) return st;
        unsigned char *base = (unsigned char *)scratch;
        void *qp = base, *op = base + bq, *kp = base + 2 * bq, *vp = base + 2 * bq + bk;
        void *rp = base + 2 * bq + 2 * bk;
        float *up_ = (float *)(base + 2 * bq + 2 * bk + br), *wp = (float *)(base + 2 * bq + 2 * bk + br + bb);
        void *sp = bs ? base + 2 * bq + 2 * bk + br + 2 * bb : nullptr;
        const PadJob jobs[6] = {{qp, a.q, nq, a.D, 2}, {kp, a.k, nk, a.D, 2}, {vp, a.v, nk, a.D, 2},
                                {rp, a.r, nr, a.D, 2}, {up_, a.u, heads, a.D, 4}, {wp, a.w, heads, a.D, 4}};
        e = launch_pad_heads_many(jobs, 6, s);
        ap.q = qp;
        ap.k = kp;
        ap.v = vp;
        ap.r = rp;
        ap.u = up_;
        ap.w = wp;
        ap.out = op;
        if (e == cudaSuccess) e = launch_attn_bf16(ap, splits, sp, s);
        if (e == cudaSuccess) e = launch_unpad_heads(a.out, op, nq, a.D, W, 2, s);
    }
    return e == cudaSuccess ? TXL_OK : cuda_fail(e);
}

txl_status txl_rel_attn_fwd(const void *q, const void *k, const void *v, const void *r,
                            const float *u_bias, const float *v_bias,
                            int batch, int mem_len, int seg_len, int heads, int d_head,
                            txl_dtype dtype, void *out, void *stream)
{
    return rel_attn_common(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head, 0,
                           dtype, out, stream);
}

txl_status txl_rel_attn_fwd_plan(int batch, int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype,
                                 int *splits, int *launches)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (!splits || !launches) return TXL_ERR_INVALID;
    if (batch < 0 || mem_len < 0 || seg_len < 0 || heads < 0 || d_head < 1) return TXL_ERR_INVALID;
    *splits = 1;
    *launches = 0;
    if (batch == 0 || seg_len == 0 || heads == 0) return TXL_OK;
    if (d_head > 128 || (dtype == TXL_BF16 && d_head > 64)) return TXL_ERR_UNSUPPORTED;
    if (dtype == TXL_F32) {
        *launches = 1;
        return TXL_OK;
    }
    AttnArgs a{};
    a.B = batch;
    a.H = heads;
    a.D = 64;                                     // other head sizes run on 64-wide padded copies
    a.L = seg_len;
    a.M = mem_len;
    a.scale_d = d_head;
    const int s = bf16_num_splits(a, device_sm_count());
    *splits = s;
    // the attention kernel, the split combine, and for head sizes other than
    // 64 the padding copies (one launch) and the output's copy back
    *launches = 1 + (s > 1 ? 1 : 0) + (d_head != 64 ? 2 : 0);
    return TXL_OK;
}

}  // extern "C"

// The rollover half of a txl_rel_attn_fwd_mem call: its checks, and the
// copy's source and size (0 bytes: nothing to roll).
static txl_status mem_checks(const void *q, const void *k, const void *v, const void *r, const float *u_bias,
                             const float *v_bias, int batch, int mem_len, int seg_len, int heads, int d_head,
                             txl_dtype dtype, const void *out, const void *mem_next, const void *ext_ctx,
                             int d_model, const void **src, size_t *nbytes)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (batch < 0 || mem_len < 0 || seg_len < 0 || heads < 0 || d_head < 1 || d_model < 0) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    *src = nullptr;
    *nbytes = 0;
    if (batch > 0 && mem_len > 0 && d_model > 0) {
        if (!mem_next || !ext_ctx) return TXL_ERR_INVALID;
        if (!aligned(mem_next, esz) || !aligned(ext_ctx, esz)) return TXL_ERR_INVALID;
        const size_t row = (size_t)batch * (size_t)d_model * esz;
        if (row / esz / (size_t)batch != (size_t)d_model) return TXL_ERR_UNSUPPORTED;
        const size_t T = (size_t)mem_len + (size_t)seg_len;
        const size_t n = (size_t)mem_len * row;
        if (overlaps(mem_next, n, ext_ctx, T * row)) return TXL_ERR_INVALID;
        // and the attention's: mem_next overlaps none of its buffers, ext_ctx not its output
        if (seg_len > 0 && heads > 0) {
            const size_t hrow = (size_t)batch * (size_t)heads * (size_t)d_head * esz;
            const size_t nq = (size_t)seg_len * hrow, nk = T * hrow, nr = T * (size_t)heads * d_head * esz;
            const size_t nb = (size_t)heads * d_head * 4;
            if (overlaps(mem_next, n, q, nq) || overlaps(mem_next, n, k, nk) || overlaps(mem_next, n, v, nk) ||
                overlaps(mem_next, n, r, nr) || overlaps(mem_next, n, out, nq) ||
                overlaps(mem_next, n, u_bias, nb) || overlaps(mem_next, n, v_bias, nb) ||
                overlaps(ext_ctx, T * row, out, nq))
                return TXL_ERR_INVALID;
        }
        *src = (const unsigned char *)ext_ctx + (size_t)seg_len * row;
        *nbytes = n;
    }
    return TXL_OK;
}

extern "C" {

txl_status txl_rel_attn_fwd_mem(const void *q, const void *k, const void *v, const void *r,
                                const float *u_bias, const float *v_bias, int batch, int mem_len,
                                int seg_len, int heads, int d_head, txl_dtype dtype, void *out,
                                void *mem_next, const void *ext_ctx, int d_model, void *stream)
{
    const void *src = nullptr;
    size_t nbytes = 0;
    const txl_status st = mem_checks(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head, dtype,
                                     out, mem_next, ext_ctx, d_model, &src, &nbytes);
    if (st != TXL_OK) return st;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (batch == 0 || seg_len == 0 || heads == 0) {
        // no attention work: the rollover alone
        if (!nbytes) return TXL_OK;
        const cudaError_t e = launch_rollover(mem_next, src, nbytes, (int)esz, (cudaStream_t)stream);
        return e == cudaSuccess ? TXL_OK : cuda_fail(e);
    }
    return rel_attn_common(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head, 0, dtype, out,
                           stream, 0, nullptr, src, nbytes ? mem_next : nullptr, nbytes);
}

txl_status txl_rel_attn_fwd_mem_cells(int cells, const void *const *q, const void *const *k, const void *const *v,
                                      const void *const *r, const float *const *u_bias,
                                      const float *const *v_bias, int batch, int mem_len, int seg_len, int heads,
                                      int d_head, txl_dtype dtype, void *const *out, void *const *mem_next,
                                      const void *const *ext_ctx, int d_model, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (cells < 0 || batch < 0 || mem_len < 0 || seg_len < 0 || heads < 0 || d_head < 1 || d_model < 0)
        return TXL_ERR_INVALID;
    if (cells == 0) return TXL_OK;
    const bool attend = batch > 0 && seg_len > 0 && heads > 0, roll = batch > 0 && mem_len > 0 && d_model > 0;
    if ((attend && (!q || !k || !v || !r || !out)) || (roll && (!mem_next || !ext_ctx))) return TXL_ERR_INVALID;
    auto at = [](const void *const *a, int c) { return a ? a[c] : nullptr; };
    auto atf = [](const float *const *a, int c) { return a ? a[c] : nullptr; };
    auto atw = [](void *const *a, int c) { return a ? a[c] : nullptr; };
    // every call as txl_rel_attn_fwd_mem checks it
    size_t nbytes = 0;
    for (int c = 0; c < cells; ++c) {
        const void *src = nullptr;
        txl_status st = mem_checks(at(q, c), at(k, c), at(v, c), at(r, c), atf(u_bias, c), atf(v_bias, c), batch,
                                   mem_len, seg_len, heads, d_head, dtype, at(out, c), at(mem_next, c),
                                   at(ext_ctx, c), d_model, &src, &nbytes);
        if (st == TXL_OK)
            st = attn_checks(at(q, c), at(k, c), at(v, c), at(r, c), atf(u_bias, c), atf(v_bias, c), batch, mem_len,
                             seg_len, heads, d_head, 0, dtype, at(out, c), nullptr);
        if (st != TXL_OK) return st;
    }
    // the calls are independent: what one writes (out, mem_next) meets
    // nothing another reads or writes
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    const size_t T = (size_t)mem_len + (size_t)seg_len;
    const size_t hrow = (size_t)batch * (size_t)heads * (size_t)d_head * esz;
    const size_t nq = attend ? (size_t)seg_len * hrow : 0, nk = attend ? T * hrow : 0;
    const size_t nr = attend ? T * (size_t)heads * d_head * esz : 0, nb = attend ? (size_t)heads * d_head * 4 : 0;
    const size_t next = roll ? T * (size_t)batch * (size_t)d_model * esz : 0;
    for (int c = 0; c < cells; ++c) {
        const void *wr[2] = {at(out, c), at(mem_next, c)};
        const size_t nw[2] = {nq, nbytes};
        for (int d = 0; d < cells; ++d) {
            if (d == c) continue;
            const void *bufs[9] = {at(q, d), at(k, d), at(v, d), at(r, d), atf(u_bias, d), atf(v_bias, d),
                                   at(out, d), at(mem_next, d), at(ext_ctx, d)};
            const size_t nbuf[9] = {nq, nk, nk, nr, nb, nb, nq, nbytes, next};
            for (int x = 0; x < 2; ++x)
                for (int y = 0; y < 9; ++y)
                    if (overlaps(wr[x], nw[x], bufs[y], nbuf[y])) return TXL_ERR_INVALID;
        }
    }
    // bf16 with 64-wide heads: the calls share launches
    if (attend && dtype == TXL_BF16 && d_head == 64 && cells >= 2) {
        const float *z = nullptr;
        bool zero_ok = true;
        for (int c = 0; c < cells && zero_ok; ++c)
            if (!atf(u_bias, c) || !atf(v_bias, c)) zero_ok = zero_bias((size_t)heads * d_head, &z) == cudaSuccess;
        if (zero_ok) {
            AttnArgs *args = new (std::nothrow) AttnArgs[cells];
            if (!args) return TXL_ERR_UNSUPPORTED;
            const size_t row = roll ? (size_t)batch * (size_t)d_model * esz : 0;
            for (int c = 0; c < cells; ++c) {
                AttnArgs &a = args[c];
                a = AttnArgs{q[c], k[c], v[c], r[c], atf(u_bias, c) ? u_bias[c] : z, atf(v_bias, c) ? v_bias[c] : z,
                             out[c], batch, heads, d_head, seg_len, mem_len, 0, 0};
                if (nbytes) {
                    a.roll_src = (const unsigned char *)ext_ctx[c] + (size_t)seg_len * row;
                    a.roll_dst = mem_next[c];
                    a.roll_bytes = nbytes;
                }
            }
            const cudaError_t e = launch_attn_bf16_cells(cells, args, (cudaStream_t)stream);
            delete[] args;
            if (e != cudaErrorNotSupported) return e == cudaSuccess ? TXL_OK : cuda_fail(e);
        }
    }
    for (int c = 0; c < cells; ++c) {
        const txl_status st = txl_rel_attn_fwd_mem(at(q, c), at(k, c), at(v, c), at(r, c), atf(u_bias, c),
                                                   atf(v_bias, c), batch, mem_len, seg_len, heads, d_head, dtype,
                                                   atw(out, c), atw(mem_next, c), at(ext_ctx, c), d_model, stream);
        if (st != TXL_OK) return st;
    }
    return TXL_OK;
}

txl_status txl_rel_attn_fwd_lse(const void *q, const void *k, const void *v, const void *r,
                                const float *u_bias, const float *v_bias, int batch, int mem_len, int seg_len,
                                int heads, int d_head, txl_dtype dtype, void *out, float *lse, void *stream)
{
    if (!lse && batch > 0 && seg_len > 0 && heads > 0) return TXL_ERR_INVALID;
    return rel_attn_common(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head, 0, dtype, out,
                           stream, 0, lse);
}

txl_status txl_rel_attn_fwd_padded(const void *q, const void *k, const void *v, const void *r,
                                   const float *u_bias, const float *v_bias, int batch, int mem_len,
                                   int seg_len, int heads, int d_head, int d_pad, txl_dtype dtype,
                                   void *out, void *stream)
{
    // every head vector is stored with d_pad elements, zeros past d_head: the
    // kernels run at width d_pad (the zeros add nothing) and scale by d_head
    if (d_head < 1 || d_pad < d_head) return TXL_ERR_INVALID;
    return rel_attn_common(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_pad, 0, dtype, out,
                           stream, d_head);
}

txl_status txl_rel_attn_fwd_ring(const void *q, const void *k, const void *v, const void *r,
                                 const float *u_bias, const float *v_bias, int batch, int mem_len,
                                 int seg_len, int heads, int d_head, int kv_start, txl_dtype dtype,
                                 void *out, void *stream)
{
    return rel_attn_common(q, k, v, r, u_bias, v_bias, batch, mem_len, seg_len, heads, d_head,
                           kv_start, dtype, out, stream);
}

txl_status txl_mem_update(void *mem_next, const void *ext_ctx, int batch, int mem_len,
                          int seg_len, int d_model, txl_dtype dtype, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (batch < 0 || mem_len < 0 || seg_len < 0 || d_model < 0) return TXL_ERR_INVALID;
    if (batch == 0 || mem_len == 0 || d_model == 0) return TXL_OK;
    if (!mem_next || !ext_ctx) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (!aligned(mem_next, esz) || !aligned(ext_ctx, esz)) return TXL_ERR_INVALID;
    const size_t row = (size_t)batch * (size_t)d_model * esz;
    const size_t T = (size_t)mem_len + (size_t)seg_len;
    if (row / esz / (size_t)batch != (size_t)d_model) return TXL_ERR_UNSUPPORTED;
    const size_t nbytes = (size_t)mem_len * row;
    if (overlaps(mem_next, nbytes, ext_ctx, T * row)) return TXL_ERR_INVALID;
    const void *src = (const unsigned char *)ext_ctx + (size_t)seg_len * row;
    cudaError_t e = launch_rollover(mem_next, src, nbytes, (int)esz, (cudaStream_t)stream);
    return e == cudaSuccess ? TXL_OK : cuda_fail(e);
}

txl_status txl_ring_append(void *ring, const void *rows, int ring_len, int n_rows, int row_elems,
                           int start, txl_dtype dtype, void *stream)
{
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (ring_len < 0 || n_rows < 0 || row_elems < 0 || n_rows > ring_len) return TXL_ERR_INVALID;
    if (n_rows == 0 || row_elems == 0) return TXL_OK;
    if (start < 0 || start >= ring_len) return TXL_ERR_INVALID;
    if (!ring || !rows) return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    if (!aligned(ring, esz) || !aligned(rows, esz)) return TXL_ERR_INVALID;
    const size_t row = (size_t)row_elems * esz;
    if (overlaps(ring, (size_t)ring_len * row, rows, (size_t)n_rows * row)) return TXL_ERR_INVALID;
    // rows [start, start + n) mod ring_len: one run up to the end, one from row 0
    const size_t first = (size_t)(ring_len - start) < (size_t)n_rows ? (size_t)(ring_len - start) : (size_t)n_rows;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_rollover((unsigned char *)ring + (size_t)start * row, rows, first * row, (int)esz, s);
    if (e == cudaSuccess && first < (size_t)n_rows)
        e = launch_rollover(ring, (const unsigned char *)rows + first * row, ((size_t)n_rows - first) * row,
                            (int)esz, s);
    return e == cudaSuccess ? TXL_OK : cuda_fail(e);
}

txl_status txl_selftest_wait(unsigned int limit_us, void *stream)
{
    if (limit_us < 1 || limit_us > 1000000) return TXL_ERR_INVALID;
    const cudaError_t e = launch_selftest_wait((uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
    return e == cudaSuccess ? TXL_OK : cuda_fail(e);
}

txl_status txl_check(void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0, gword = 0, bword = 0;
    e = read_and_clear_device_error(&word, s);
    if (e == cudaSuccess) e = read_and_clear_gemm_error(&gword, s);
    if (e == cudaSuccess) e = read_and_clear_bwd_error(&bword, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return (word | gword | bword) ? TXL_ERR_TIMEOUT : TXL_OK;
}

const char *txl_status_string(txl_status st)
{
    switch (st) {
    case TXL_OK: return "ok";
    case TXL_ERR_INVALID: return "invalid argument";
    case TXL_ERR_UNSUPPORTED: return "unsupported configuration";
    case TXL_ERR_CUDA: return "CUDA error";
    case TXL_ERR_TIMEOUT: return "in-kernel wait timed out";
    }
    return "unknown status";
}

int txl_last_cuda_error(void) { return g_last_cuda_error; }

int txl_version(void) { return 200; }   // 0.2.0: log-sum-exp, fused rollover, plan query; backward takes the saved forward

void txl_shutdown(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    bool synced = false;
    int kept = 0;
    for (int x = 0; x < g_scratch_n; ++x) {
        Scratch &s = g_scratch[x];
        if (s.dev != dev) {
            g_scratch[kept++] = s;
            continue;
        }
        if (s.ptr) {
            if (!synced) cudaDeviceSynchronize();   // every call that may read a buffer is done
            synced = true;
            cudaFree(s.ptr);
        }
    }
    g_scratch_n = kept;
    cudaGetLastError();
}

}  // extern "C"
