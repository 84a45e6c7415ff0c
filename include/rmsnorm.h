/*
 * rmsnorm.h -- C ABI of librmsnorm.so: Qwen3-style RMSNorm forward and
 * backward, the fused residual-add variant and the split-row forward for
 * decode-sized batches, as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Sources, cited by tag:
 *   [P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）"
 *        (iqiancheng.github.io, posts/triton-kernel-fusion-practice)
 *   [P2] the article on hand-writing 21 Triton kernels for decoding a 0.8B
 *        Qwen model (trdm.cn, news/483216; the extracted page has no title)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are row-major [M, H] (M rows of H features), owned by the
 *    caller, in device memory (or memory the device can address); dense
 *    (row stride H) except through the *_strided entry points, where each
 *    [M, H] tensor has its own row stride. The weight w has H entries. x, r,
 *    w, y, h, dy, dh_out and dx share one dtype (RMSNORM_F32, RMSNORM_BF16
 *    or RMSNORM_F16); rstd, dw and the workspace are always fp32.
 *  - Every pointer must be aligned to its element size. Rows whose start is
 *    16-byte aligned (aligned base pointer, H * element size and every row
 *    stride * element size multiples of 16) take the 128-bit vectorised
 *    kernels; anything else takes a scalar kernel with the same results up
 *    to fp32 summation order.
 *  - 1 <= H <= RMSNORM_MAX_H, 0 <= M. eps is a finite float >= 0 (a plain
 *    float, never a tensor: [P1 §5.6] gotcha table).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream). They allocate nothing, never synchronise and never copy
 *    to or from the host, so they can be recorded in a CUDA graph ([P2 §4.1,
 *    §4.3]: no allocation and no synchronisation inside the captured region).
 *  - Arguments are checked on the host before anything is launched; on error
 *    nothing is launched and no output is touched. A failed launch returns
 *    RMSNORM_ERR_CUDA (rmsnorm_last_cuda_error() gives the cudaError_t).
 *  - Results are deterministic: the same inputs on the same GPU model give the
 *    same bits on every run. No atomics are used ([P1 §5.4], [P1 §7.3]: a
 *    fixed reduction order instead of atomic adds; [P2 §3.3]).
 *  - Output buffers may coincide exactly with the input named in each entry
 *    point's comment (in-place use); any other overlap is rejected with
 *    RMSNORM_ERR_ALIAS.
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the row tensors and the weight ([P1 §4.2]: the forward
 * stores its result as fp16 or bf16; fp32 for reference runs). */
typedef enum { RMSNORM_F32 = 0, RMSNORM_BF16 = 1, RMSNORM_F16 = 2 } rmsnorm_dtype;

/* Return codes. */
typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_NULLPTR = -1,     /* a required pointer is NULL */
    RMSNORM_ERR_BAD_SHAPE = -2,   /* M < 0, H < 1, or M * H overflows */
    RMSNORM_ERR_BAD_DTYPE = -3,   /* dtype is not an rmsnorm_dtype */
    RMSNORM_ERR_BAD_EPS = -4,     /* eps is negative, NaN or infinite */
    RMSNORM_ERR_MISALIGNED = -5,  /* a pointer is not aligned to its element
                                     size (16 bytes for the workspace) */
    RMSNORM_ERR_WORKSPACE = -6,   /* workspace NULL or smaller than
                                     rmsnorm_bwd_workspace_bytes() */
    RMSNORM_ERR_UNSUPPORTED = -7, /* H > RMSNORM_MAX_H, or outside an entry point's limits */
    RMSNORM_ERR_CUDA = -8,        /* a CUDA runtime call failed */
    RMSNORM_ERR_ALIAS = -9,       /* buffers overlap in a way not allowed */
    RMSNORM_ERR_SCRATCH_LIMIT = -10, /* rmsnorm_bwd_static_scratch: the problem
                                       needs more scratch than the library's
                                       built-in RMSNORM_STATIC_SCRATCH_BYTES */
    RMSNORM_ERR_BAD_FLAGS = -11,  /* rmsnorm_bwd_ex: unknown flag bits */
    RMSNORM_ERR_BAD_STRIDE = -12  /* *_strided: a row stride below H, above
                                     2^31 - 1, or so large that the tensor's
                                     last element lies beyond 2^63 bytes */
} rmsnorm_status;

/* Largest feature count the kernels hold in registers ([P1 §7.1] puts the
 * whole-row-per-block limit near 16K features). */
#define RMSNORM_MAX_H 16384

/*
 * Forward ([P1 §4.1, §4.2]): for each row i,
 *   rstd_i = 1 / sqrt( (1/H) sum_j x_ij^2 + eps )
 *   y_ij   = round( x_ij * rstd_i * w_j )
 * summed and scaled in fp32, rounded once to the dtype (round-to-nearest-
 * even for bf16 and fp16; fp16 results beyond 65504 become infinite).
 *   x    [M,H] in, w [H] in, y [M,H] out (y may equal x: in place)
 *   rstd [M] fp32 out, or NULL when not wanted (the backward can recompute it)
 * M <= 64 rows take the split-row kernel ([P2 §3.2]): each row is spread over
 * a cluster of 2-8 CTAs whose fp32 partial sums of squares are combined in
 * rank order through distributed shared memory; larger M takes the row-wise
 * kernels (each row held in registers by a group of lanes).
 * M == 0 launches nothing.
 */
int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd,
                int64_t M, int64_t H, float eps, int dtype, void *stream);

/*
 * Backward ([P1 §5.3, §5.4]): with r_i = rstd_i and
 *   c_i   = (1/H) sum_j w_j dy_ij x_ij,
 *   dx_ij = round( r_i * (w_j dy_ij - x_ij r_i^2 c_i) )
 *   dw_j  = sum_i dy_ij x_ij r_i          (fp32, over all M rows)
 *   dy [M,H], x [M,H], w [H] in; dx [M,H] out (dx may equal dy: in place)
 *   rstd [M] fp32 in as saved by the forward, or NULL to recompute it from x
 *   dw [H] fp32 out (overwritten; all zeros when M == 0)
 *   workspace: caller-owned device scratch of at least
 *     rmsnorm_bwd_workspace_bytes(M, H, dtype) bytes, 16-byte aligned. It
 *     holds one fp32 partial dw row per CTA; a second kernel sums them in a
 *     fixed order. Its contents on entry do not matter; it must not be used
 *     by another call that overlaps on the GPU.
 */
int rmsnorm_bwd(const void *dy, const void *x, const void *w,
                const float *rstd, void *dx, float *dw, void *workspace,
                size_t workspace_bytes, int64_t M, int64_t H, float eps,
                int dtype, void *stream);

/*
 * Residual add fused with the forward ([P1 §1]: "residual + next RMSNorm"
 * across a block boundary; [P2 §2.1]: residual_add then rms_norm, with a
 * fused kernel planned):
 *   h_ij = round(x_ij + r_ij)   (fp32 add, one rounding to the dtype)
 *   then the forward above on the stored h: y, rstd.
 *   x, r [M,H] in; w [H] in; h [M,H] out (h may equal x or r: in place);
 *   y [M,H] out (must not overlap anything); rstd [M] out or NULL.
 * Same kernel choice as rmsnorm_fwd (split-row for M <= 64).
 */
int rmsnorm_residual_fwd(const void *x, const void *r, const void *w, void *h,
                         void *y, float *rstd, int64_t M, int64_t H, float eps,
                         int dtype, void *stream);

/*
 * Backward of the residual variant: the norm's backward at h, plus the
 * gradient dh_out that reaches h from the residual stream's other consumer
 * (NULL means zero). Because dh/dx = dh/dr = identity, the one output dx is
 * the gradient of both x and r:
 *   dx_ij = round( r_i (w_j dy_ij - h_ij r_i^2 c_i) + dh_out_ij )
 *   dw_j  = sum_i dy_ij h_ij r_i
 *   dy, h [M,H] in; dh_out [M,H] in or NULL; w [H] in; rstd [M] in or NULL;
 *   dx [M,H] out (dx may equal dy or dh_out); dw [H] out; workspace as for
 *   rmsnorm_bwd.
 */
int rmsnorm_residual_bwd(const void *dy, const void *dh_out, const void *h,
                         const void *w, const float *rstd, void *dx, float *dw,
                         void *workspace, size_t workspace_bytes, int64_t M,
                         int64_t H, float eps, int dtype, void *stream);

/*
 * Backward with options: the plain backward when dh_out is NULL, the
 * residual backward otherwise (x then holds h), with the same arguments,
 * results, aliasing and errors as rmsnorm_bwd / rmsnorm_residual_bwd, plus
 *   flags: 0, or RMSNORM_BWD_ACCUMULATE_DW to add this call's dw to the dw
 *   already in the buffer (gradient accumulation over micro-batches or over
 *   chunks of rows) instead of overwriting it. The addition follows the
 *   fixed-order sum of this call, so a sequence of calls in stream order is
 *   reproducible. Unknown bits give RMSNORM_ERR_BAD_FLAGS.
 */
#define RMSNORM_BWD_ACCUMULATE_DW 1
int rmsnorm_bwd_ex(const void *dy, const void *dh_out, const void *x,
                   const void *w, const float *rstd, void *dx, float *dw,
                   void *workspace, size_t workspace_bytes, int64_t M,
                   int64_t H, float eps, int dtype, int flags, void *stream);

/*
 * Strided rows ([P1 §4.2]: the forward kernel takes the row stride of its
 * input and of its output, so a row-major view with padded or interleaved
 * rows needs no copy). Each [M, H] tensor t is given with its row stride
 * ld_t in ELEMENTS (H <= ld_t <= 2^31 - 1): row i starts at t + i * ld_t.
 * ld_t == H is the dense layout of the entry points above, with identical
 * results; the results do not depend on the strides.
 *
 * Forward, plain or fused with the residual add: r and h both NULL gives
 * rmsnorm_fwd; both non-NULL gives rmsnorm_residual_fwd. The ld of a NULL
 * tensor is ignored.
 *   x [M,H] (ldx), r [M,H] (ldr) in; w [H] in;
 *   y [M,H] (ldy) out, h [M,H] (ldh) out; rstd [M] out or NULL.
 * Aliasing as for the dense calls, applied element by element: y (or h) may
 * be exactly x (same pointer and stride); two tensors that share memory but
 * touch disjoint columns of rows with the same stride (e.g. two column
 * windows of one [M, ld] buffer) do not overlap; anything else that shares
 * an element is RMSNORM_ERR_ALIAS.
 * Errors: those of rmsnorm_fwd / rmsnorm_residual_fwd; RMSNORM_ERR_NULLPTR
 * when only one of r and h is NULL; RMSNORM_ERR_BAD_STRIDE as defined above.
 * Kernel choice: as for the dense calls, except that the streamed kernels of
 * 128-wide rows (which copy blocks of consecutive rows) need every stride
 * equal to H, and the 256-bit forward needs every stride * element size to
 * be a multiple of 32.
 */
int rmsnorm_fwd_strided(const void *x, int64_t ldx, const void *r, int64_t ldr,
                        const void *w, void *y, int64_t ldy, void *h,
                        int64_t ldh, float *rstd, int64_t M, int64_t H,
                        float eps, int dtype, void *stream);

/*
 * Backward with strided rows: rmsnorm_bwd_ex with a row stride (in
 * elements, >= H) for dy, dh_out, x (h for the residual backward) and dx.
 *   dy [M,H] (lddy) in; dh_out [M,H] (lddh) in or NULL; x [M,H] (ldx) in;
 *   w [H] in; rstd [M] in or NULL; dx [M,H] (lddx) out; dw [H] fp32 out;
 *   workspace, flags: as for rmsnorm_bwd_ex (the workspace size does not
 *   depend on the strides).
 * Aliasing element by element as for rmsnorm_fwd_strided: dx may be exactly
 * dy or dh_out. Errors: those of rmsnorm_bwd_ex and RMSNORM_ERR_BAD_STRIDE.
 */
int rmsnorm_bwd_strided(const void *dy, int64_t lddy, const void *dh_out,
                        int64_t lddh, const void *x, int64_t ldx,
                        const void *w, const float *rstd, void *dx,
                        int64_t lddx, float *dw, void *workspace,
                        size_t workspace_bytes, int64_t M, int64_t H,
                        float eps, int dtype, int flags, void *stream);

/*
 * RMSNorm fused with the projection that follows it in decode ([P2 §2.1]:
 * rms_norm, then the q/k/v_proj or gate/up_proj GEMVs; §3.1: a [1, 896]
 * hidden state against the [1024, 896] q_proj weight, K split over several
 * programs; §6: fusing the chain is the next step). For each row i:
 *   (residual variant: h_ij = round(x_ij + r_ij), and the norm acts on h)
 *   rstd_i = 1 / sqrt( (1/H) sum_j x_ij^2 + eps )
 *   y_ij   = round( x_ij * rstd_i * w_j )            as rmsnorm_fwd stores it
 *   out_in = round( sum_k y_ik A_nk )                fp32 accumulation
 * i.e. the result of running the norm and then the GEMV on its stored
 * output, in one launch.
 *   x [M,H] in; r [M,H] in or NULL (plain norm); w [H] in;
 *   A [N,H] in, row-major (a linear layer's weight; stack q|k|v or gate|up
 *     rows to produce several projections in one call);
 *   out [M,N] out; h [M,H] out or NULL (residual variant only);
 *   y [M,H] out or NULL (the norm's output, when a caller needs it too);
 *   rstd [M] fp32 out or NULL. All dense row-major.
 * Limits (else RMSNORM_ERR_UNSUPPORTED): dtype RMSNORM_BF16 or RMSNORM_F16;
 *   M <= 64 (decode batches); H a multiple of 32 that one of the kernels
 *   holds in shared memory: the warp-level MMA kernels when
 *   ceil(M/16) * (16 * (2H + 64) + 2048) + 2H + 16 <= 227 KB (H <= 6720
 *   for M <= 16, 3424 for M <= 32, 2272 for M <= 48, 1664 for M <= 64),
 *   or above 8 rows a tcgen05 kernel: the one whose K is split over a
 *   cluster of up to 8 CTAs (with r: H <= 4608 for M <= 32, 4096 for
 *   M <= 48, 3584 for M <= 64; without r: 5120 for M <= 32) or the
 *   persistent one, whose K is split over a cluster of 1 to 8 CTAs
 *   (H <= 16384 for M <= 32, 11264 for M <= 48, 7168 for M <= 64).
 *   Calls only a tcgen05 kernel holds also return RMSNORM_ERR_UNSUPPORTED
 *   when a warp-level kernel is forced (rmsnorm_set_path_override) or the
 *   driver offers no tensor-map encoder;
 *   1 <= N < 2^30 (else RMSNORM_ERR_BAD_SHAPE).
 * Alignment: x, r, w, A, h, y 16-byte aligned (RMSNORM_ERR_MISALIGNED).
 * Aliasing: no output (out, h, y, rstd) may share a byte with an input or
 *   with another output (every CTA reads x while one writes h and y), else
 *   RMSNORM_ERR_ALIAS. h without r is RMSNORM_ERR_NULLPTR. M == 0 launches
 *   nothing. Deterministic (fixed-order fp32 sums, no atomics).
 * Performance: built for decode batches. Up to 8 rows the call is faster
 *   than the norm followed by a separate GEMM (measured on GB300 with the
 *   weights streaming from HBM). From 9 rows on it runs the product on the
 *   tensor cores (tcgen05): at 896 features with K split over a
 *   thread-block cluster, on rows of 2048 features or more in the
 *   persistent kernel. It stays correct and deterministic there; at 896
 *   features and 16 rows with 2048 outputs it is faster than the norm
 *   followed by a GEMM library call, elsewhere rmsnorm_fwd /
 *   rmsnorm_residual_fwd followed by a GEMM library call is faster (at 896
 *   features by some 0.4 to 2.5 us per call; at 4096 features and 6144 to
 *   24576 outputs the fused call takes 1.1 to 1.6 times as long at 16 and
 *   32 rows, 1.5 to 2.25 times at 48 and 64).
 * flags: 0, or RMSNORM_GEMV_STATIC_WEIGHTS: the caller guarantees that no
 *   work still in flight on the stream when this call is enqueued writes w
 *   or A (model weights during decoding). The kernel then fetches them while
 *   the preceding kernel is still running (it starts early through
 *   programmatic dependent launch), which takes their load latency off the
 *   critical path; x and r are always read only after the preceding work is
 *   complete. Breaking the guarantee gives results computed from stale
 *   weights. Unknown bits give RMSNORM_ERR_BAD_FLAGS.
 */
#define RMSNORM_GEMV_STATIC_WEIGHTS 1
int rmsnorm_gemv_fwd(const void *x, const void *r, const void *w,
                     const void *A, void *out, void *h, void *y, float *rstd,
                     int64_t M, int64_t H, int64_t N, float eps, int dtype,
                     int flags, void *stream);

/*
 * Double backward ([P1 §5.6]: an autograd wrapper implements it or refuses
 * it): given gradients gdx [M,H] arriving on the backward's dx and gdw [H]
 * (fp32) arriving on its dw, the gradients of
 *   L2 = sum_ij gdx_ij dx_ij + sum_j gdw_j dw_j
 * with respect to the backward's inputs dy, x and w, the backward being
 * that of rmsnorm_bwd ([P1 §5.3]) with r = rstd a function of x. Per row,
 * with c = (1/H) sum w dy x and A = sum gdx w dy, B = sum gdx x,
 * D = sum gdw dy x:
 *   ddy = r w gdx - (r^3 B / H) w x + r gdw x
 *   dx2 = (r^3 / H)(3 r^2 c B - A - D) x - (r^3 B / H) w dy - r^3 c gdx
 *         + r gdw dy
 *   dw2 = sum over rows of r gdx dy - (r^3 B / H) dy x        (fp32)
 *   dy, x [M,H] in; w [H] in; rstd [M] fp32 in (as the forward saved it) or
 *   NULL to recompute it; gdx [M,H] in or NULL (zero); gdw [H] fp32 in or
 *   NULL (zero), 16-byte aligned; ddy, dx2 [M,H] out; dw2 [H] fp32 out
 *   (overwritten; zeros when M == 0); workspace as for rmsnorm_bwd (at least
 *   rmsnorm_bwd_workspace_bytes(M, H, dtype) bytes).
 * For the residual variant pass h as x: dx2 is then the gradient on h, and
 * the gradient on dh_out is gdx itself (dx depends on dh_out as the
 * identity).
 * Aliasing: no output may share a byte with an input or another output
 * (RMSNORM_ERR_ALIAS). Errors otherwise as for rmsnorm_bwd. Deterministic.
 */
int rmsnorm_bwd_bwd(const void *dy, const void *x, const void *w,
                    const float *rstd, const void *gdx, const float *gdw,
                    void *ddy, void *dx2, float *dw2, void *workspace,
                    size_t workspace_bytes, int64_t M, int64_t H, float eps,
                    int dtype, void *stream);

/*
 * Bytes of workspace rmsnorm_bwd, rmsnorm_residual_bwd, rmsnorm_bwd_ex,
 * rmsnorm_bwd_strided and rmsnorm_bwd_bwd need for (M, H, dtype) on the
 * current CUDA device (one fp32 row of H per CTA of the backward grid; the
 * grid is sized from the device's SM count). Returns 0 on invalid arguments
 * or when no device is available.
 */
size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H, int dtype);

/* A static, human-readable name for a status code. */
const char *rmsnorm_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this library on the
 * calling thread (0 if none). */
int rmsnorm_last_cuda_error(void);

/*
 * Test hook: force the kernel family for later calls in this process.
 * 0 = automatic (default), 1 = row-wise vectorised, 2 = split-row (forward
 * only; the backward then takes row-wise), 3 = row-wise scalar, 4 = streamed
 * (rows staged through shared memory by bulk asynchronous copies; bf16 or
 * fp16 with H = 128 (dense rows only), 4096 or 5120; row-wise elsewhere).
 * For rmsnorm_gemv_fwd: 1 = the weight in registers, 6 = the weight by bulk
 * copies (the automatic choice up to 8 rows), 7 = the product on tcgen05
 * with K split over a cluster (the automatic choice above 8 rows where y is
 * too large for one CTA and a cluster of at most 8 CTAs fits its shared
 * memory; else as 6), 8 = the persistent product on tcgen05 with y held
 * whole by each CTA (the automatic choice above 8 rows where it fits: T x H
 * x 2 bytes of y, T = rows rounded up to 16, with a ring of the weight in
 * 227 KB; else as 6). Other values: automatic.
 * Forcing a vectorised family on rows that are not 16-byte aligned still
 * takes the scalar one. Not thread-safe against concurrent calls; intended
 * for tests only.
 */
void rmsnorm_set_path_override(int path);

/* Which kernel family the last call on this thread used: 1 row-wise
 * vectorised, 2 split-row, 3 row-wise scalar, 4 streamed, 5 to 8 the norm
 * fused with the GEMV (rmsnorm_gemv_fwd; 5: the weight in registers, which
 * override 1 forces; 6: the weight fed by bulk copies, automatic up to 8
 * rows; 7: the product on tcgen05 with K split over a cluster, automatic
 * above 8 rows on rows narrower than 2048 features; 8: the persistent
 * product on tcgen05, automatic above 8 rows on rows of 2048 features or
 * more; each also takes the rows only it holds), 0 none. */
int rmsnorm_last_path(void);

/*
 * Diagnostic (synchronous, not for the hot path): the number of bounded
 * waits on the current device that ran out of time (in the streamed kernels
 * a bulk copy that never completed, in the split-row forward a peer's sum
 * that never arrived, in the projection kernels a copy of the weight or a
 * peer's partial products; the affected rows are then left unwritten or
 * wrong and the results must not be used). *count receives the value;
 * reset != 0 also sets it back to zero. Every wait is bounded at about one
 * second, so a failed copy ends the kernel instead of hanging the GPU.
 */
int rmsnorm_wait_timeouts(unsigned int *count, int reset);

/*
 * Test hook for the bounded waits of the streamed kernels, process-wide, not
 * thread-safe against concurrent calls: later streamed launches make every
 * stage wait for extra_tx_bytes more than its copies deliver (so each wait
 * runs out) and give up after wait_limit_us microseconds (0 = the default of
 * about one second). The split-row forward's wait for its peers' sums, the
 * projection kernels' waits for the weight's copies and the double
 * backward's stage waits take the same hook. (0, 0) restores normal
 * operation. With a non-zero extra_tx_bytes the results of those calls are
 * left incomplete and rmsnorm_wait_timeouts counts the waits that ran out;
 * the kernels still end and the CUDA context stays usable.
 */
void rmsnorm_set_stream_test_fault(unsigned int extra_tx_bytes,
                                   unsigned int wait_limit_us);

/*
 * Test hook, process-wide, not thread-safe against concurrent calls: later
 * rmsnorm_gemv_fwd calls that run the persistent tcgen05 kernel (path 8)
 * split K over clusters of exactly cluster_size CTAs (1 to 8) instead of
 * the size the plan picks; where that size does not fit the call, the call
 * takes another kernel as it would if the persistent one did not fit. 0 (or
 * any value outside 1..8) restores the plan's choice. Results are the same
 * up to the order of the fp32 sums.
 */
void rmsnorm_set_gemv_cluster_test(int cluster_size);

/*
 * Backward that allocates nothing and needs no workspace from the caller.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc at all: plug-ins hosted by a runtime that owns
 * every byte of device memory and forbids its guests to allocate, and
 * latency-critical loops that cannot tolerate the device-wide
 * synchronisation cudaMalloc and cudaFree may imply.
 *
 * Same arguments, results and errors as rmsnorm_bwd without `workspace` and
 * `workspace_bytes`: the per-CTA partial dw rows go to a scratch array of
 * RMSNORM_STATIC_SCRATCH_BYTES that the library itself holds in device
 * memory (a file-scope __device__ array). Every GPU that loads the library
 * keeps that array until the process exits.
 *  - Size limit: a call whose rmsnorm_bwd_workspace_bytes(M, H, dtype)
 *    exceeds RMSNORM_STATIC_SCRATCH_BYTES is rejected with
 *    RMSNORM_ERR_SCRATCH_LIMIT before anything is launched (for H <= 16384
 *    on a 152-SM GB300 the need is at most about 10 MiB).
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress) with that device current; make that
 *    first call before any stream capture. The address is kept for that
 *    device's CUDA context: after cudaDeviceReset (a new context) the next
 *    call looks it up again, so make that call before any capture too.
 *  - Sharing: all calls, on every stream and thread, share the one array.
 *    Calls whose executions overlap on the GPU race on it and give wrong dw;
 *    serialise them (one stream, or events). Nothing in it needs clearing
 *    between calls: each call writes every partial row it later reads.
 */
#define RMSNORM_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
int rmsnorm_bwd_static_scratch(const void *dy, const void *x, const void *w,
                               const float *rstd, void *dx, float *dw,
                               int64_t M, int64_t H, float eps, int dtype,
                               void *stream);

/*
 * Test hook for rmsnorm_bwd_static_scratch, process-wide, not thread-safe
 * against concurrent calls: later calls treat the built-in array as holding
 * only min(bytes, RMSNORM_STATIC_SCRATCH_BYTES) bytes (0 restores the full
 * size). On a 152-SM GB300 no problem within RMSNORM_MAX_H needs the whole
 * array, so this is how the RMSNORM_ERR_SCRATCH_LIMIT refusal is exercised.
 */
void rmsnorm_set_static_scratch_test_limit(size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
