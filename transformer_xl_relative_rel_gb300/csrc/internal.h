// internal.h -- launchers shared between the library's translation units.
// Not part of the public ABI (that is include/txl.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace txl {

struct AttnArgs {
    const void *q, *k, *v, *r;
    const float *u, *w;           // u and v biases, [H][D] float32
    void *out;
    int B, H, D, L, M;
    int kv_start = 0;             // K, V in a ring of M+L rows: key j at row (kv_start + j) mod (M+L)
    int scale_d = 0;              // d_head for the 1/sqrt(d_head) scale when D is a padded width (0: D)
    float *lse = nullptr;         // bf16 path, optional [B*H][L]: row log-sum-exp (natural log) of the scaled scores
    // optional memory rollover done by the same launch where that pays
    // (bf16 TMA path): roll_bytes bytes from roll_src to roll_dst; otherwise
    // the launcher issues the separate rollover copy after the attention
    const void *roll_src = nullptr;
    void *roll_dst = nullptr;
    size_t roll_bytes = 0;
};

// fp32 SIMT path (attn_f32.cu)
cudaError_t launch_attn_f32(const AttnArgs &a, cudaStream_t s);

// bf16 tcgen05 path (attn_bf16.cu).  `scratch` is device memory of at least
// bf16_scratch_bytes(a, splits) bytes (ignored when splits == 1).
int bf16_num_splits(const AttnArgs &a, int num_sms);
size_t bf16_scratch_bytes(const AttnArgs &a, int splits);
cudaError_t launch_attn_bf16(const AttnArgs &a, int splits, void *scratch, cudaStream_t s);
// Calls of one shape (bf16, D = 64, K and V not a ring, no row log-sum-exp)
// that each run unsplit with their output by TMA store: up to ATTN_CELLS of
// them per launch, items of all calls in one persistent schedule, each call's
// rollover (if any) in the same launch where it fuses, else after it.
// Returns cudaErrorNotSupported, having launched nothing, for calls that do
// not meet that (the caller then runs them one by one).
constexpr int ATTN_CELLS = 8;
cudaError_t launch_attn_bf16_cells(int n, const AttnArgs *a, cudaStream_t s);
// The score side of the backward (bf16, D = 64, 16-byte aligned operands):
// P and dA as bf16 [B*H][L][TP] and dA in the table frame as bf16
// [H][L][B][TP] (TP = M+L rounded up to 128), from the forward's output
// a.out and row log-sum-exp `lse` ([B*H][L]).
cudaError_t launch_bwd_scores(const AttnArgs &a, const void *dout, const float *lse, void *p_out, void *da_out,
                              void *db_out, long TP, cudaStream_t s);
// one warp's bounded wait on an mbarrier nothing completes, limit_ns long;
// records the device error word when it runs out (the failure path, tested)
cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s);
// reads and clears the device error word written by bounded waits (syncs on s)
cudaError_t read_and_clear_device_error(unsigned int *word, cudaStream_t s);

// memory rollover (rollover.cu): bit copy of `bytes` bytes
cudaError_t launch_rollover(void *dst, const void *src, size_t bytes, int elem_size,
                            cudaStream_t s);

// head vectors to / from a zero-padded width (pack.cu); elem_size 2 or 4
cudaError_t launch_pad_heads(void *dst, const void *src, long nvec, int d, int dp, int elem_size,
                             cudaStream_t s);
// several pad jobs (as launch_pad_heads, dp 64) in one launch
constexpr int kMaxPadJobs = 6;
struct PadJob {
    void *dst;
    const void *src;
    long nvec;
    int d, elem_size;
};
cudaError_t launch_pad_heads_many(const PadJob *jobs, int n, cudaStream_t s);
cudaError_t launch_unpad_heads(void *dst, const void *src, long nvec, int d, int dp, int elem_size,
                               cudaStream_t s);

int device_sm_count();

// Device address of `count` zero floats on the current device (a fixed array
// in the library), standing in for an absent u or v bias.  Returns
// cudaErrorNotSupported when count exceeds the array, or the CUDA error of
// the lookup.
cudaError_t zero_bias(size_t count, const float **out);

// the projection kernel's and the backward contraction kernel's error words
// (bounded waits that gave up), as above
cudaError_t read_and_clear_gemm_error(unsigned int *word, cudaStream_t s);
cudaError_t read_and_clear_bwd_error(unsigned int *word, cudaStream_t s);

// records `e` as the thread's last CUDA error (reported by txl_last_cuda_error)
// and clears the runtime's error state; returns e
cudaError_t note_cuda_error(cudaError_t e);

}  // namespace txl
