// noalloc.cu -- txl_rel_attn_fwd_noalloc: relative attention for callers that
// cannot allocate device memory.
//
// Some callers must not call cudaMalloc at all: code running inside a
// framework that owns every device allocation (a memory pool, or an arena
// sized once at start-up), real-time or embedded hosts that forbid
// allocation after initialisation, and processes whose device memory is
// already fully reserved.  The default entry point may allocate its split-key
// scratch on first use; this one never does.  Its scratch is the fixed array
// below, which lives as long as the library's device code is loaded on a GPU
// (TXL_NOALLOC_SCRATCH_BYTES per GPU, held until the process exits).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "txl.h"

namespace txl {
namespace {

constexpr size_t kNoallocBytes = TXL_NOALLOC_SCRATCH_BYTES;

// Partial results of the key-split path.  No slot needs to start at zero:
// every slot a call reads back was written earlier in that same call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

std::mutex g_na_mu;
void *g_na_addr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name only stands for the symbol, so the address is looked up once
// per device (with that device current) and cached.
txl_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return TXL_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) return TXL_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            note_cuda_error(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
            return TXL_ERR_CUDA;
        }
        g_na_addr[dev] = p;
    }
    *out = g_na_addr[dev];
    return TXL_OK;
}

bool na_aligned(const void *p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }

bool na_overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace txl

using namespace txl;

extern "C" txl_status txl_rel_attn_fwd_noalloc(const void *q, const void *k, const void *v,
                                               const void *r, const float *u_bias,
                                               const float *v_bias, int batch, int mem_len,
                                               int seg_len, int heads, int d_head, txl_dtype dtype,
                                               void *out, void *stream)
{
    // the same argument rules as txl_rel_attn_fwd
    if (dtype != TXL_F32 && dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (batch < 0 || mem_len < 0 || seg_len < 0 || heads < 0 || d_head < 1) return TXL_ERR_INVALID;
    if (batch == 0 || seg_len == 0 || heads == 0) return TXL_OK;
    if (d_head > 128) return TXL_ERR_UNSUPPORTED;
    if (dtype == TXL_BF16 && d_head > 64) return TXL_ERR_UNSUPPORTED;
    if (!q || !k || !v || !r || !out) return TXL_ERR_INVALID;
    if (!na_aligned(q, 16) || !na_aligned(k, 16) || !na_aligned(v, 16) || !na_aligned(r, 16) ||
        !na_aligned(out, 16) || !na_aligned(u_bias, 4) || !na_aligned(v_bias, 4))
        return TXL_ERR_INVALID;
    const size_t esz = dtype == TXL_F32 ? 4 : 2;
    const size_t T = (size_t)mem_len + (size_t)seg_len;
    if (T > (size_t)INT32_MAX) return TXL_ERR_UNSUPPORTED;
    const size_t row = (size_t)batch * (size_t)heads * (size_t)d_head;
    const size_t nq = (size_t)seg_len * row * esz, nk = T * row * esz;
    const size_t nr = T * (size_t)heads * (size_t)d_head * esz;
    const size_t nb = (size_t)heads * (size_t)d_head * 4;
    if ((size_t)batch * (size_t)heads > (size_t)INT32_MAX || nk / esz / T != row)
        return TXL_ERR_UNSUPPORTED;
    if (na_overlaps(out, nq, q, nq) || na_overlaps(out, nq, k, nk) || na_overlaps(out, nq, v, nk) ||
        na_overlaps(out, nq, r, nr) || na_overlaps(out, nq, u_bias, nb) ||
        na_overlaps(out, nq, v_bias, nb))
        return TXL_ERR_INVALID;
    if ((seg_len + 31) / 32 > 65535) return TXL_ERR_UNSUPPORTED;

    // an absent bias drops its term (Shaw et al.'s form); the zeros are a
    // fixed array too, so nothing is allocated here either
    if (!u_bias || !v_bias) {
        const float *z = nullptr;
        const cudaError_t ze = zero_bias((size_t)heads * (size_t)d_head, &z);
        if (ze == cudaErrorNotSupported) return TXL_ERR_UNSUPPORTED;
        if (ze != cudaSuccess) {
            note_cuda_error(ze);
            return TXL_ERR_CUDA;
        }
        if (!u_bias) u_bias = z;
        if (!v_bias) v_bias = z;
    }
    AttnArgs a{q, k, v, r, u_bias, v_bias, out, batch, heads, d_head, seg_len, mem_len};
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (dtype == TXL_F32) {
        e = launch_attn_f32(a, s);          // needs no scratch
    } else {
        const int splits = bf16_num_splits(a, device_sm_count());
        void *scratch = nullptr;
        if (splits > 1) {
            // too large for the fixed array: refuse before touching the GPU
            if (bf16_scratch_bytes(a, splits) > kNoallocBytes) return TXL_ERR_UNSUPPORTED;
            txl_status st = scratch_address(&scratch);
            if (st != TXL_OK) return st;
        }
        e = launch_attn_bf16(a, splits, scratch, s);
    }
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return TXL_ERR_CUDA;
    }
    return TXL_OK;
}
