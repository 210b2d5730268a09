/*
 * txl.h -- C ABI of libtxl: Transformer-XL segment-level relative multi-head
 * attention and the per-layer memory rollover on one GB300 GPU (sm_103a).
 *
 * Every pointer argument named "device" is a CUDA device pointer owned by the
 * caller; the library never frees caller memory and keeps no pointer to it
 * after the call returns.  Calls are asynchronous on the given stream (a
 * cudaStream_t passed as void*, NULL = the legacy default stream): the library
 * never synchronises the device inside a compute call.  Argument errors are
 * detected on the host before any launch and nothing is launched then.
 *
 * Notation (Transformer-XL, Section 3.2 and Appendix B): B batch, H heads,
 * D head dimension, L segment length, M memory length, T = M + L the extended
 * context [memory (M rows, oldest first); current segment (L rows)].
 * Row-major layouts, D innermost:
 *     q, out : [L][B][H][D]      k, v : [T][B][H][D]
 *     r      : [T][H][D]  -- row t holds W_kR R_{T-1-t} (the reversed table Q
 *                            of Appendix B); shared by every sequence
 *     u_bias, v_bias : [H][D] float32 (the global biases u and v of
 *                            Section 3.3, one vector per head)
 */
#ifndef TXL_H_
#define TXL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TXL_OK = 0,
    TXL_ERR_INVALID = 1,     /* bad argument: NULL, negative size, misaligned, overlap */
    TXL_ERR_UNSUPPORTED = 2, /* valid but not built: d_head too large, unknown dtype */
    TXL_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (also: no GPU) */
    TXL_ERR_TIMEOUT = 4      /* a bounded in-kernel wait gave up (see txl_check) */
} txl_status;

typedef enum {
    TXL_F32 = 0,             /* float32 in, float32 accumulate, float32 out */
    TXL_BF16 = 1             /* bfloat16 in, float32 accumulate, bfloat16 out */
} txl_dtype;

/*
 * txl_rel_attn_fwd -- one layer of relative attention (Transformer-XL,
 * Section 3.3, the computing procedure; Appendix B, the linear-cost route).
 *
 * For every b < batch, h < heads and query position i < seg_len:
 *     s_ij = ((q_i + u).k_j + (q_i + v).r[T-1-(M+i-j)]) / sqrt(d_head)
 *                                          for key j = 0 .. M+i (causal)
 *     out_i = sum_j softmax_j(s_ij) v_j
 * where j indexes the extended context [memory; segment] and M+i-j is the
 * relative distance of the pair.
 *
 * q, k, v, r, out : device, dtype elements, layouts above; base addresses
 *                   16-byte aligned; out must not overlap any input.
 * u_bias, v_bias  : device, float32 [heads][d_head], 4-byte aligned; either
 *                   may be NULL, which drops its term: with both NULL the
 *                   score is terms (a) + (b) only, the form of Shaw et al.
 *                   the paper contrasts in Section 3.3 (r may then be any
 *                   table, e.g. a learned R^ in place of W_kR R).  NULL needs
 *                   heads*d_head <= 65536 (else TXL_ERR_UNSUPPORTED).
 * batch, heads, seg_len >= 0 (0 => nothing to do, TXL_OK, pointers unused);
 * mem_len >= 0; 1 <= d_head <= 128 for TXL_F32, 1 <= d_head <= 64 for
 * TXL_BF16 (larger: TXL_ERR_UNSUPPORTED).
 * stream          : cudaStream_t as void*.
 * Returns TXL_OK once the work is enqueued.  TXL_ERR_INVALID /
 * TXL_ERR_UNSUPPORTED before any launch; TXL_ERR_CUDA if a launch fails.
 * Long memories (few query tiles, many keys) split the keys across CTAs; the
 * partial results then live in a library-owned device scratch buffer.  bf16
 * heads with d_head != 64 also use it: q, k, v, r and the biases are copied
 * into 64-wide zero-padded vectors there (rows the TMA unit can read), and
 * the output's d_head columns are copied back.  There is one such buffer per
 * (device, stream handle): calls on different streams never share one and may
 * run concurrently.  A buffer is allocated on first need and grown in stream
 * order (cudaFreeAsync / cudaMallocAsync on that stream, no host-side wait),
 * so the first call of a larger size on a stream must not be made during
 * stream capture (it returns TXL_ERR_UNSUPPORTED there); later captured calls
 * reuse the buffer.  Buffers are keyed by the stream handle's value: destroy a
 * stream only after its calls have finished if a new stream may reuse the
 * handle.  At most 256 (device, stream) pairs are served (then
 * TXL_ERR_UNSUPPORTED); txl_shutdown() releases the current device's.
 */
txl_status txl_rel_attn_fwd(const void *q, const void *k, const void *v, const void *r,
                            const float *u_bias, const float *v_bias,
                            int batch, int mem_len, int seg_len, int heads, int d_head,
                            txl_dtype dtype, void *out, void *stream);

/*
 * txl_rel_attn_fwd_plan -- how txl_rel_attn_fwd runs a call of this shape:
 * the number of key-range splits (the keys of each query block divided over
 * that many CTAs, merged by a combine launch) and the number of kernel
 * launches it makes, for 16-byte aligned operands.  No GPU work; the split
 * choice is the one the call itself makes on the current device (a cost
 * model of the kernel's schedule, measured on GB300).
 *
 * splits, launches : host int outputs (NULL => TXL_ERR_INVALID).  A call with
 * nothing to do reports 1 split and 0 launches.  Same dtype and d_head limits
 * as txl_rel_attn_fwd.
 */
txl_status txl_rel_attn_fwd_plan(int batch, int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype,
                                 int *splits, int *launches);

/*
 * txl_rel_attn_fwd_lse -- txl_rel_attn_fwd that also stores, per query row,
 * the natural log of the softmax denominator (the log-sum-exp of the row's
 * visible scaled scores s_ij above):
 *     lse[(b*heads + h)*seg_len + i] = log sum_{j <= M+i} exp(s_ij)
 * so that P_ij = exp(s_ij - lse) recovers the weights without a second pass
 * over the keys.  txl_rel_attn_bwd takes out and lse back to skip its own
 * forward.
 *
 * lse : device float32 [batch][heads][seg_len], 4-byte aligned, must not
 *       overlap out or any input; required (NULL => TXL_ERR_INVALID unless
 *       there is nothing to do).
 * Only TXL_BF16 (else TXL_ERR_UNSUPPORTED).  Everything else, including the
 * result in out, as txl_rel_attn_fwd.
 */
txl_status txl_rel_attn_fwd_lse(const void *q, const void *k, const void *v, const void *r,
                                const float *u_bias, const float *v_bias, int batch, int mem_len,
                                int seg_len, int heads, int d_head, txl_dtype dtype, void *out,
                                float *lse, void *stream);

/*
 * txl_mem_update -- the per-layer memory rollover (Transformer-XL,
 * Section 3.2: a cache of the last M hidden states, possibly spanning several
 * segments, reused as extended context by the next segment).
 *
 * ext_ctx  : device, [M+L][batch][d_model] = [memory; current hidden states].
 * mem_next : device, at least [M][batch][d_model]; rows 0..M-1 receive the
 *            newest M rows of ext_ctx (rows L..M+L-1), oldest first -- i.e.
 *            the memory part of the next segment's extended context.  Must not
 *            overlap ext_ctx (use two buffers and swap them per segment).
 * Bit-exact copy of dtype elements.  mem_len == 0 or batch == 0 or
 * d_model == 0 => nothing to do.  Same error behaviour as above.
 */
txl_status txl_mem_update(void *mem_next, const void *ext_ctx, int batch, int mem_len,
                          int seg_len, int d_model, txl_dtype dtype, void *stream);

/*
 * txl_rel_attn_fwd_mem -- one layer's txl_rel_attn_fwd and txl_mem_update in
 * one call (Section 3.3's attention and Section 3.2's cache update of the
 * same layer, which do not depend on each other).  Where it pays, the
 * attention launch does the rollover copy as well (bf16, d_head = 64, the
 * tensor-memory path, 16-byte aligned ext_ctx + seg_len rows and mem_next,
 * M*batch*d_model*2 a multiple of 16, and a copy small against the
 * attention's own work); otherwise the rollover runs as its own launch right
 * after, on the same stream.  Results are exactly those of the two calls.
 *
 * Arguments as txl_rel_attn_fwd, plus mem_next, ext_ctx and d_model as
 * txl_mem_update (same batch, mem_len, seg_len and dtype).  mem_next must not
 * overlap ext_ctx or any buffer of the attention; ext_ctx must not overlap
 * out.  With nothing to attend (batch, seg_len or heads 0) only the rollover
 * runs; with nothing to roll (mem_len or d_model 0) mem_next and ext_ctx are
 * unused.  Same error behaviour as the two calls.
 */
txl_status txl_rel_attn_fwd_mem(const void *q, const void *k, const void *v, const void *r,
                                const float *u_bias, const float *v_bias, int batch, int mem_len,
                                int seg_len, int heads, int d_head, txl_dtype dtype, void *out,
                                void *mem_next, const void *ext_ctx, int d_model, void *stream);

/*
 * txl_rel_attn_fwd_mem_cells -- several independent txl_rel_attn_fwd_mem
 * calls of one shape (e.g. the layer calls of one step of a layer-by-segment
 * wavefront: different layers, different segments, none waiting for
 * another's result).  Call c takes q[c], k[c], v[c], r[c], u_bias[c],
 * v_bias[c], out[c], mem_next[c] and ext_ctx[c], each as
 * txl_rel_attn_fwd_mem takes it; batch, mem_len, seg_len, heads, d_head,
 * dtype and d_model are shared.  The results are exactly those of the calls
 * one after another.  With bf16 and d_head = 64, unsplit calls with TMA-
 * addressable operands share launches (up to 8 calls a launch, their work
 * items in one persistent schedule, each call's rollover inside where it
 * fuses); other shapes run call by call.
 *
 * cells           : number of calls, >= 0 (0: nothing).
 * q .. ext_ctx    : host arrays of `cells` device pointers.  u_bias, v_bias
 *                   may be NULL (no bias in any call) or hold NULL entries;
 *                   mem_next and ext_ctx may be NULL when there is nothing to
 *                   roll (batch, mem_len or d_model 0); the others are
 *                   required when there is attention work.
 * Errors: every call's txl_rel_attn_fwd_mem checks, plus TXL_ERR_INVALID
 * when one call's out or mem_next overlaps any buffer of another call.
 * Nothing is launched when an argument is rejected.
 */
txl_status txl_rel_attn_fwd_mem_cells(int cells, const void *const *q, const void *const *k,
                                      const void *const *v, const void *const *r,
                                      const float *const *u_bias, const float *const *v_bias, int batch,
                                      int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype,
                                      void *const *out, void *const *mem_next, const void *const *ext_ctx,
                                      int d_model, void *stream);

/*
 * txl_rel_attn_fwd_ring -- txl_rel_attn_fwd with k and v stored as a ring.
 * The extended context [memory; segment] of Section 3.2 slides forward by L
 * rows per segment; kept in a ring of M+L rows, a segment adds only its L new
 * rows (txl_ring_append) instead of moving the M memory rows.  The paper has
 * no counterpart to this storage order; the result is exactly that of
 * txl_rel_attn_fwd on the unrolled context.
 *
 * k, v     : device, [M+L][batch][heads][d_head]; the context's key j (j = 0
 *            is the oldest memory row, j = M+L-1 the segment's last row) is
 *            stored at row (kv_start + j) mod (M+L).
 * kv_start : 0 <= kv_start < M+L (0 gives txl_rel_attn_fwd's layout).
 * Everything else as txl_rel_attn_fwd.  With bf16 and d_head = 64 the rows
 * are read by TMA when kv_start and M+L are multiples of 8, by thread loads
 * otherwise (same result, slower).
 */
txl_status txl_rel_attn_fwd_ring(const void *q, const void *k, const void *v, const void *r,
                                 const float *u_bias, const float *v_bias, int batch, int mem_len,
                                 int seg_len, int heads, int d_head, int kv_start, txl_dtype dtype,
                                 void *out, void *stream);

/*
 * txl_rel_attn_fwd_padded -- txl_rel_attn_fwd on head vectors stored with
 * d_pad >= d_head elements each (zeros past d_head), the layout
 * txl_project_heads and txl_rel_table write.  q, k, v, r, out are
 * [..][heads][d_pad]; u_bias, v_bias [heads][d_pad] (or NULL).  The result
 * equals txl_rel_attn_fwd on the first d_head elements (scale 1/sqrt(d_head));
 * out's padding columns come out zero.  With bf16 and d_pad = 64 the rows are
 * read by TMA whatever d_head is (e.g. d_head 41 padded to 64).
 */
txl_status txl_rel_attn_fwd_padded(const void *q, const void *k, const void *v, const void *r,
                                   const float *u_bias, const float *v_bias, int batch, int mem_len,
                                   int seg_len, int heads, int d_head, int d_pad, txl_dtype dtype,
                                   void *out, void *stream);

/*
 * txl_project_heads -- the projections of Section 3.3's procedure
 * (q = h W_q^T, k = h~ W_kE^T, v = h~ W_v^T) into the attention's layout:
 *     y[rows][heads][d_pad] = x[rows][d_in] . W^T
 * with W in the paper's layout, [heads*d_head][d_in] (row h*d_head + d is
 * output column d of head h; also torch.nn.Linear's weight layout), and
 * padding columns d_head..d_pad-1 of every head exactly zero.  With
 * x = a T-major [positions][batch][d_model] buffer (rows = positions*batch)
 * the result is the T-major [positions][batch][heads][d_pad] layout.
 * bf16: the library's tcgen05 GEMM (fp32 accumulation, one rounding to
 * bf16), for d_in even and x, w 4-byte aligned (TMA operand loads when d_in
 * is a multiple of 8, x and w 16-byte aligned and d_pad divides 256; TMA
 * output stores when out is 16-byte aligned and heads*d_pad*2 a multiple of
 * 16); fp32 and other bf16 shapes: a CUDA-core kernel (fp32 accumulation).
 * x, w, out device, row-major, dtype elements; out must not overlap x or w.
 * d_pad >= d_head >= 1; d_in == 0 gives zeros.
 */
txl_status txl_project_heads(const void *x, const void *w, void *out, int rows, int d_in, int heads,
                             int d_head, int d_pad, txl_dtype dtype, void *stream);

/*
 * txl_project_qkv -- a layer's three projections of Section 3.3's procedure
 * from one extended context h~ = [memory; h] (x, [rows][d_in], rows =
 * positions x batch of a T-major buffer):
 *     k = x W_k^T and v = x W_v^T over all rows, and
 *     q = x[q_row0 ..] W_q^T over the last rows - q_row0 rows (the segment's
 *         own positions h: q_row0 = mem_len x batch),
 * each as txl_project_heads writes it ([..][heads][d_pad], padding zero).
 * w_q and q are both given or both NULL (then only k and v).  bf16 with
 * d_in a multiple of 8, every pointer 16-byte aligned, heads*d_pad*2 a
 * multiple of 16 and d_pad dividing 256: the three come from one launch of
 * the projection GEMM that reads x once for k and v (and for q too when
 * q_row0 is a multiple of 128; otherwise q's rows are a band of their own in
 * the same launch); other shapes are computed as by three txl_project_heads
 * calls.
 * Outputs must not overlap x, the weights or one another; 0 <= q_row0 <=
 * rows.  Results equal the separate txl_project_heads calls bit for bit.
 */
txl_status txl_project_qkv(const void *x, int rows, int d_in, const void *w_q, const void *w_k, const void *w_v,
                           void *q, void *k, void *v, int q_row0, int heads, int d_head, int d_pad, txl_dtype dtype,
                           void *stream);

/*
 * txl_project_qkv_cells -- txl_project_qkv for several layer calls of one
 * shape at once (cells c = 0 .. cells-1, e.g. the layer calls of a
 * recurrence that do not depend on each other): cell c projects x[c] with
 * w_q[c], w_k[c], w_v[c] into q[c], k[c], v[c] (rows, d_in, q_row0, heads,
 * d_head, d_pad shared).  x, w_*, q, k, v are host arrays of `cells` device
 * pointers (w_q and q both NULL, or both arrays with every entry set); no
 * output may overlap any input or any other output of any cell.  Where
 * txl_project_qkv would use one launch per cell, up to eight cells share a
 * launch; results equal the per-cell calls bit for bit.
 */
txl_status txl_project_qkv_cells(int cells, const void *const *x, const void *const *w_q, const void *const *w_k,
                                 const void *const *w_v, void *const *q, void *const *k, void *const *v, int rows,
                                 int d_in, int q_row0, int heads, int d_head, int d_pad, txl_dtype dtype,
                                 void *stream);

/*
 * txl_rel_table -- Appendix B's reversed projected table of one layer:
 * out[t][h][d] = sum_c R[klen-1-t][c] * W_kR[h*d_head + d][c] for t < klen,
 * R[p][2c] = sin(p * 10000^(-2c/d_model)), R[p][2c+1] = cos(the same angle)
 * (the sinusoid of the relative distance p, evaluated in fp32 on the device;
 * fp32 accumulation).  out [klen][heads][d_pad], padding zero; W_kR in the
 * paper's layout [heads*d_head][d_model].  Batch- and segment-independent:
 * once per layer.
 */
txl_status txl_rel_table(const void *w_r, void *out, int klen, int d_model, int heads, int d_head, int d_pad,
                         txl_dtype dtype, void *stream);

/*
 * txl_rel_attn_bwd -- gradients of one txl_rel_attn_fwd call for a given
 * output gradient dout (the chain rule through the masked softmax and the
 * four-term score of Section 3.3).  With P the softmax weights of query row
 * i, dA_ij = P_ij (dout_i.v_j - sum_l P_il dout_i.v_l) / sqrt(d_head) for the
 * visible keys j <= M+i and off = M+i-j:
 *     dq_i = sum_j dA_ij (k_j + r[T-1-off])    dk_j = sum_i dA_ij (q_i + u)
 *     dv_j = sum_i P_ij dout_i                 dr[T-1-off] += dA_ij (q_i + v)
 *     du   = sum_{b,i,j} dA_ij k_j             dw = sum_{b,i,j} dA_ij r[T-1-off]
 * (dr, du, dw summed over the batch).  Every input gets its gradient, the
 * memory rows 0..M-1 of k and v included: Section 3.2's stop-gradient acts
 * on the cached hidden states, while the keys and values projected from them
 * still carry gradient to the projections.
 *
 * q, k, v, r, dout : device, dtype, layouts as txl_rel_attn_fwd (dout like q).
 * u_bias, v_bias   : device float32 [heads][d_head] or NULL (zero bias).
 * out, lse         : the forward's output and row log-sum-exp as
 *                    txl_rel_attn_fwd_lse wrote them for these inputs (out
 *                    16-byte aligned, lse 4-byte aligned), or both NULL.
 *                    Given, they spare the backward its own forward pass;
 *                    the bf16 d_head = 64 path reads them, the others (which
 *                    recompute the scores in full) ignore them.  Exactly one
 *                    of them NULL => TXL_ERR_INVALID.
 * dq, dk, dv, dr   : device outputs, dtype, shaped like q, k, v, r.
 * du, dw           : device float32 [heads][d_head] outputs, or NULL (not
 *                    computed).  Outputs must not overlap each other, any
 *                    input or the workspace.
 * workspace        : device scratch of at least the bytes that
 *                    txl_rel_attn_bwd_workspace reports, 256-byte aligned,
 *                    owned by the caller.  bf16 with d_head = 64: P and dA
 *                    as bf16 plus dA in the table's frame (about 3 x 2 bytes
 *                    per (b, h, i, j) score entry); otherwise the score, P,
 *                    dP and dA of every head (about 3 x 4 + 3 x dtype bytes
 *                    per entry).
 * Limits: d_head <= 128 (else TXL_ERR_UNSUPPORTED).  Asynchronous on stream.
 * bf16: operands of the contractions in bf16 (q+u, q+v, P and dA rounded
 * once), fp32 accumulation, fp32 softmax; fp32: fp32 throughout.
 */
txl_status txl_rel_attn_bwd_workspace(int batch, int mem_len, int seg_len, int heads, int d_head,
                                      txl_dtype dtype, size_t *bytes);
txl_status txl_rel_attn_bwd(const void *q, const void *k, const void *v, const void *r, const float *u_bias,
                            const float *v_bias, const void *dout, const void *out, const float *lse, int batch,
                            int mem_len, int seg_len, int heads, int d_head, txl_dtype dtype, void *dq, void *dk,
                            void *dv, void *dr, float *du, float *dw, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * txl_ring_append -- write n_rows new rows into a ring of ring_len rows at
 * rows (start + i) mod ring_len, i = 0 .. n_rows-1 (the oldest rows of the
 * ring, for a ring kept as above: start = the current kv_start, after which
 * the next kv_start is (start + n_rows) mod ring_len).  Serves both the
 * cached hidden states of Section 3.2 and projected k / v rings.
 *
 * ring : device, [ring_len][row_elems] dtype elements.
 * rows : device, [n_rows][row_elems]; must not overlap ring.
 * 0 <= n_rows <= ring_len, 0 <= start < ring_len (unless nothing to do),
 * row_elems >= 0; element-aligned pointers.  Bit-exact copy (one or two
 * contiguous runs).  Same error behaviour as txl_mem_update.
 */
txl_status txl_ring_append(void *ring, const void *rows, int ring_len, int n_rows, int row_elems,
                           int start, txl_dtype dtype, void *stream);

/*
 * txl_rel_attn_fwd_noalloc -- txl_rel_attn_fwd for callers that may not
 * allocate device memory.  (No counterpart in the paper: this is a deployment
 * variant of the same computation.)
 *
 * Some callers cannot call cudaMalloc: code inside a framework that owns all
 * device memory through its own pool or a fixed arena, hosts that forbid
 * allocation once initialised, or processes whose device memory is already
 * fully reserved.  txl_rel_attn_fwd may allocate its split-key scratch on
 * first use; this entry point allocates nothing.  Its scratch is one fixed
 * array of TXL_NOALLOC_SCRATCH_BYTES inside the library's device code, held
 * on every GPU that loads that code until the process exits.
 *
 * Same arguments, layouts, results and error rules as txl_rel_attn_fwd, plus:
 *   - a call whose key split needs more than TXL_NOALLOC_SCRATCH_BYTES
 *     (splits * batch * heads * seg_len * (2 * ceil16(d_head) + 4) + 256
 *     bytes) returns TXL_ERR_UNSUPPORTED before touching the GPU;
 *   - the first call on a device that splits its keys looks up the array's
 *     device address (cudaGetSymbolAddress, with that device current); make
 *     that first call before any stream capture.  Under CUDA's default lazy
 *     module loading the array is reserved on a device when the library's
 *     device code is first loaded there, which can be as late as that lookup:
 *     a caller that reserves the rest of device memory afterwards should make
 *     one such call first (a long-memory shape, e.g. B 1, H 4, D 64,
 *     L 128, M 1600);
 *   - the cached address belongs to the device's primary context: a device
 *     reset (cudaDeviceReset) while the library is loaded is not supported;
 *   - every call shares the one array, and each call writes every part of it
 *     that it reads back, so nothing carries over between calls; but calls
 *     whose kernels overlap on the GPU (different streams, or concurrent
 *     host threads) race on it and must be serialised by the caller.
 */
#define TXL_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

txl_status txl_rel_attn_fwd_noalloc(const void *q, const void *k, const void *v, const void *r,
                                    const float *u_bias, const float *v_bias,
                                    int batch, int mem_len, int seg_len, int heads, int d_head,
                                    txl_dtype dtype, void *out, void *stream);

/*
 * txl_check -- synchronise `stream`, then report and clear the library's
 * device error word: TXL_ERR_TIMEOUT if an in-kernel bounded wait gave up
 * since the last check, TXL_ERR_CUDA if the stream reports an error, else
 * TXL_OK.
 */
txl_status txl_check(void *stream);

/*
 * txl_selftest_wait -- exercise the failure path of the kernels' bounded
 * waits without any fault: a one-warp kernel waits on an mbarrier that
 * nothing completes, through the same bounded wait the kernels use but
 * limited to limit_us microseconds (1 .. 1,000,000; else TXL_ERR_INVALID).
 * The wait runs out and records the device error word, so the next
 * txl_check(stream) returns TXL_ERR_TIMEOUT (and clears it); the context
 * stays usable.  No counterpart in the paper: a test hook of the library.
 */
txl_status txl_selftest_wait(unsigned int limit_us, void *stream);

/* Static description of a status code; never NULL. */
const char *txl_status_string(txl_status s);

/* Number of the most recent CUDA error seen by the library on this thread
 * (0 if none); pairs with TXL_ERR_CUDA. */
int txl_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int txl_version(void);

/* Free the library-owned scratch buffers of the current device (every
 * stream's).  Waits for the device to finish its work first (this is not a
 * compute call).  Safe to call more than once; later calls re-allocate on
 * demand. */
void txl_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* TXL_H_ */
