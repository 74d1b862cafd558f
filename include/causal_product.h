/*
 * causal_product.h -- C ABI of libcausal_product.so
 *
 * The causal dot product of causal linear attention, batched over
 * batch x heads.  For every (b, h), with q, k in R^{N x D} and v in R^{N x M}:
 *
 *     out_i = sum_{j <= i} (q_i . k_j) v_j  =  S_i^T q_i,
 *     S_i   = sum_{j <= i} k_j v_j^T        (a D x M running state).
 *
 * This is the prefix sum over the sequence that triton-lang/triton issue
 * #217 ("Dot Product Computes Wrong Values") sets out to batch-parallelise
 * (its opening comment names Algorithm 1 of "Transformers are RNNs"); the
 * loop listing in that issue adds the outer product of the key and value
 * rows to the state before reading the output out with the query, so row i
 * includes j = i.  No normaliser and no 1/sqrt(D) scale are applied.
 *
 * The backward pass (not printed on the pages; derived from the
 * definition with L = sum_i <g_i, out_i>) is
 *
 *     dq_i = sum_{j <= i} (g_i . v_j) k_j,
 *     dk_j = sum_{i >= j} (g_i . v_j) q_i,
 *     dv_j = sum_{i >= j} (q_i . k_j) g_i.
 *
 * Layout and ownership (every entry point):
 *   - q, k, grad_q, grad_k: contiguous row-major [B][H][N][D];
 *     v, out, grad_out, grad_v: contiguous row-major [B][H][N][M].
 *     All are DEVICE pointers owned by the caller, 16-byte aligned.
 *   - Outputs are written, never accumulated into, in the input dtype.
 *     Outputs must not alias inputs.
 *   - Accumulation and the running state are fp32 for both dtypes;
 *     bf16 outputs are rounded to nearest-even once, at the end.
 *   - All work is enqueued on `stream` (cudaStream_t; NULL = legacy default
 *     stream).  No entry point synchronises the host except
 *     causal_product_status().
 *   - `workspace` is device scratch of at least
 *     causal_product_workspace_size(...) bytes, owned by the caller, used
 *     only until the enqueued work completes; it holds the per-segment fp32
 *     state aggregates of the two-pass scan and a status word.  The status
 *     word is sticky: kernels only ever write an error code into it, and
 *     causal_product_status() reads and clears it.  Zero the first 256 bytes
 *     of a new workspace once before its first use.  Passing
 *     workspace = NULL makes the call allocate and free scratch itself
 *     with cudaMallocAsync / cudaFreeAsync on `stream`; its status word is
 *     then not observable.
 *   - Concurrent calls on different streams need separate workspaces.
 *
 * Supported shapes: B, H >= 1; N >= 0 (N = 0 returns CP_OK and enqueues
 * nothing); 1 <= D, M <= 256.  bf16 additionally needs D and M to be
 * multiples of 8 (16-byte rows for the tensor-memory-access engine); the
 * normaliser needs D a multiple of 8 for bf16 and fp16.
 *
 * Errors are reported before anything is enqueued (argument checks) or as
 * CP_ERR_CUDA for a failed launch.  A kernel that finds one of its internal
 * waits has not completed within about two seconds records
 * CP_ERR_TIMEOUT in the workspace status word and returns early (its
 * outputs are then undefined); causal_product_status() reads that word.
 */
#ifndef CAUSAL_PRODUCT_H_
#define CAUSAL_PRODUCT_H_

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden visibility; only these entry points are
 * exported. */
#if defined(__GNUC__)
#define CP_API __attribute__((visibility("default")))
#else
#define CP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_DTYPE_F32 = 0,  /* fp32 in/out; fp32 FMA arithmetic (no TF32 rounding) */
  CP_DTYPE_BF16 = 1, /* bf16 in/out; bf16 tensor-core products, fp32 accumulate */
  CP_DTYPE_F16 = 2   /* fp16 in/out; widened on load, fp32 FMA arithmetic (the fp32
                        path, CUDA cores), rounded to nearest-even once on store */
} cp_dtype_t;

/* Feature map applied to q and k before the product (causal linear
 * attention, "Transformers are RNNs": phi(x) = elu(x) + 1). */
typedef enum {
  CP_FEATURE_NONE = 0,  /* q, k used as given */
  CP_FEATURE_ELU1 = 1   /* phi(x) = x + 1 for x > 0, e^x otherwise */
} cp_feature_t;

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1,        /* null pointer, negative size, aliasing outputs */
  CP_ERR_UNSUPPORTED_SHAPE = 2,  /* D or M outside [1, 256], or not a multiple of 8 (bf16) */
  CP_ERR_UNSUPPORTED_DTYPE = 3,
  CP_ERR_MISALIGNED = 4,         /* a pointer is not 16-byte aligned */
  CP_ERR_WORKSPACE_TOO_SMALL = 5,
  CP_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed */
  CP_ERR_TIMEOUT = 7,            /* a kernel's bounded wait expired (status word) */
  CP_ERR_NO_DEVICE = 8,          /* no usable sm_103 device */
  CP_ERR_NOALLOC_LIMIT = 9       /* problem too large for causal_product_fwd_noalloc's scratch */
} cp_status_t;

/* Bytes of device workspace causal_product_fwd (backward = 0) or
 * causal_product_bwd (backward = 1) needs for this problem; always >= 256
 * (the status word), a multiple of 256.  Pure host computation.  Returns 0
 * for arguments the entry points would reject. */
CP_API size_t causal_product_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                            cp_dtype_t dtype, int backward);

/* Number of kernels one causal_product_fwd (backward = 0),
 * causal_product_bwd (backward = 1), causal_product_fwd_ckpt (backward = 2),
 * causal_product_bwd_ckpt (backward = 3) or causal_product_fwd_norm
 * (backward = 4) call launches for this problem,
 * with no carried state: 1 per unsplit scan, 3 per scan split into segments
 * (the segment sums, their prefix, the scan), 1 for a scan seeded from
 * precomputed states (dq from checkpoints; bf16 dk from dv's segment
 * prefixes), and 1 for the whole backward when bf16 with D, M <= 64 runs
 * unsplit on fewer problems than SMs.  With the environment variable
 * CP_SPLIT_SCAN=lookback (read at each call) a bf16 forward scan split into
 * segments runs as one launch instead of three when its grid fits the SMs
 * (each segment sums itself, publishes the sum, adds the sums before it in
 * scan order and scans; the same bits as the two passes), and is counted as
 * 1.  Pure host computation (the SM count of the current device, else 152).
 * Returns -1 for arguments the entry points would reject, 0 when N = 0. */
CP_API int causal_product_launch_count(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                       cp_dtype_t dtype, int backward);

/* Forward: out[b,h,i,:] = sum_{j<=i} (q[b,h,i,:] . k[b,h,j,:]) v[b,h,j,:].
 * `stream` is a cudaStream_t passed as void*. */
CP_API cp_status_t causal_product_fwd(const void* q, const void* k, const void* v, void* out,
                                      int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                      cp_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* Backward: given grad_out = dL/dout, writes grad_q, grad_k, grad_v (the
 * formulas in the header comment).  Three causal products: dq is the
 * forward product of (grad_out, v, k); dv and dk are reverse-order products
 * of (k, q, grad_out) and (v, grad_out, q). */
CP_API cp_status_t causal_product_bwd(const void* q, const void* k, const void* v, const void* grad_out,
                                      void* grad_q, void* grad_k, void* grad_v,
                                      int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                      cp_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* Forward and backward with checkpoints of the state.  The backward's dq is
 * the forward product of (grad_out, v, k), whose running state sum_j v_j k_j^T
 * is the transpose of the forward's S_i; causal_product_fwd_ckpt writes that
 * state at fixed row boundaries (every few 128-row tiles) into `ckpt`, so
 * causal_product_bwd_ckpt can split every dq scan into segments that start
 * from a checkpoint, with no pass of its own over k and v to find the
 * segments' starting states (a two-pass scan whose first pass the forward
 * has already done; the pages of triton-lang/triton issue #217 ask for the
 * prefix sum over the sequence to be parallel).
 *
 * causal_product_checkpoint_size returns the bytes of `ckpt` (fp32; layout
 * private to the library), a pure function of the shape and dtype; 0 means
 * no checkpoints are used for this problem (fp32 and fp16 inputs, short
 * sequences, or a backward that does not split dq), and then `ckpt` may be
 * NULL and the two calls are causal_product_fwd and causal_product_bwd.
 * Otherwise `ckpt` is a caller-owned device buffer of at least that many
 * bytes, 16-byte aligned, overlapping no other argument; the forward writes
 * it and the backward reads it, so pass the backward the buffer of the
 * forward on the same q, k, v (a stale or foreign buffer gives a wrong
 * grad_q, undetected).  All other arguments, errors and workspaces as
 * causal_product_fwd / causal_product_bwd; CP_ERR_WORKSPACE_TOO_SMALL if
 * ckpt_bytes is below the size.  No carried state in this mode. */
CP_API size_t causal_product_checkpoint_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                             int64_t M, cp_dtype_t dtype);
CP_API cp_status_t causal_product_fwd_ckpt(const void* q, const void* k, const void* v, void* out,
                                           float* ckpt, size_t ckpt_bytes, int64_t B, int64_t H,
                                           int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                                           void* workspace, size_t workspace_bytes, void* stream);
CP_API cp_status_t causal_product_bwd_ckpt(const void* q, const void* k, const void* v,
                                           const void* grad_out, const float* ckpt,
                                           size_t ckpt_bytes, void* grad_q, void* grad_k,
                                           void* grad_v, int64_t B, int64_t H, int64_t N,
                                           int64_t D, int64_t M, cp_dtype_t dtype,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* Forward with a carried state.  The recurrence of triton-lang/triton issue
 * #217 keeps its state across the sequence, and the Triton port there takes
 * that state as an argument; these entry points let a sequence be processed
 * in pieces (or continue from a cache) by handing the state on:
 *     S_i = S_0 + sum_{j<=i} k_j v_j^T,   out_i = S_i^T q_i,
 *     S_N = S_0 + sum_j k_j v_j^T.
 * state_in  [B,H,D,M] fp32, row-major (d, m): S_0; NULL means zero.
 * state_out [B,H,D,M] fp32: receives S_N; NULL means not written.
 * Both are device pointers, 16-byte aligned; state_out must not overlap any
 * other argument.  Everything else as causal_product_fwd, which is this call
 * with both states NULL.  With N = 0, state_out = state_in. */
CP_API cp_status_t causal_product_fwd_state(const void* q, const void* k, const void* v, void* out,
                                            const float* state_in, float* state_out,
                                            int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                            cp_dtype_t dtype, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* Backward of causal_product_fwd_state.  With L = sum_i <grad_out_i, out_i>
 * + <grad_state_out, S_N>:
 *     grad_q_i = S_i grad_out_i,                  (S_i includes S_0)
 *     R_j = grad_state_out + sum_{i>=j} q_i grad_out_i^T,
 *     grad_k_j = R_j v_j,   grad_v_j = R_j^T k_j,   grad_state_in = R_0.
 * state_in is the forward's S_0 (NULL: zero), grad_state_out = dL/dS_N
 * (NULL: zero), grad_state_in receives dL/dS_0 (NULL: not written); all
 * [B,H,D,M] fp32 device pointers, 16-byte aligned, outputs overlapping
 * nothing.  causal_product_bwd is this call with all three NULL.  With
 * N = 0, grad_state_in = grad_state_out. */
CP_API cp_status_t causal_product_bwd_state(const void* q, const void* k, const void* v,
                                            const void* grad_out, const float* state_in,
                                            const float* grad_state_out, void* grad_q,
                                            void* grad_k, void* grad_v, float* grad_state_in,
                                            int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                            cp_dtype_t dtype, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* One decoding step for every (b,h): the loop body of triton-lang/triton
 * issue #217 applied to one new row,
 *     S <- S + k v^T,   out = S^T q        (readout after the update),
 * i.e. causal_product_fwd_state with N = 1, updating the state in place.
 * q, k: [B,H,D], v, out: [B,H,M] in `dtype`; state: [B,H,D,M] fp32 (row d,
 * column m), read and written.  Device pointers, 16-byte aligned; out and
 * state overlap nothing.  fp32 arithmetic; out rounded to nearest-even for
 * bf16.  No workspace, no status word (nothing waits). */
CP_API cp_status_t causal_product_decode(const void* q, const void* k, const void* v, void* out,
                                         float* state, int64_t B, int64_t H, int64_t D, int64_t M,
                                         cp_dtype_t dtype, void* stream);

/* Normaliser of causal linear attention ("Transformers are RNNs", the
 * denominator of its causal attention; the pages of triton-lang/triton issue
 * #217 cite that paper for the recurrence but their loop leaves it out):
 *     z_i = q_i . sum_{j<=i} k_j,
 * the causal product with a value of 1 (M = 1, v_j = 1).  For every (b,h):
 * q, k [B,H,N,D] in `dtype` (same rules as causal_product_fwd: device
 * pointers, 16-byte aligned, D in [1, 256], bf16 needs D % 8 == 0);
 * z [B,H,N] fp32, written.  fp32 accumulation; sums run in a fixed order,
 * so results are bitwise reproducible.  Workspace as for the other entry
 * points, sized by causal_product_normalizer_workspace_size (nothing in
 * these kernels waits, so they never write the status word).  N = 0
 * enqueues nothing. */
CP_API size_t causal_product_normalizer_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                                       cp_dtype_t dtype);
CP_API cp_status_t causal_product_normalizer(const void* q, const void* k, float* z, int64_t B,
                                             int64_t H, int64_t N, int64_t D, cp_dtype_t dtype,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream);

/* The forward product and its normaliser in one call: out as
 * causal_product_fwd and z as causal_product_normalizer, from the same q, k
 * and v (the numerator and the denominator of causal linear attention,
 * "Transformers are RNNs", section 3.2 with the causal masking of section
 * 3.3).  z_i = q_i . sum_{j<=i} k_j is the product with a value of ones.
 *
 * bf16 problems whose forward is one launch with one 64-column box of q, k
 * and v (D, M <= 64, unsplit problems: causal_product_launch_count(...,
 * backward = 4) reports 1) compute z inside that launch.  The intra-tile
 * terms are the row sums of the masked fp32 q k^T tile, and the earlier
 * tiles' terms are q_i . (sum of their k) in fp32.  q, k and v are read
 * once.  Other shapes and dtypes run the product, then the normaliser
 * kernel.
 *
 * Arguments:
 *   q, k, v, out  as causal_product_fwd;
 *   z             [B,H,N] fp32, 16-byte aligned, overlapping no other
 *                 argument; written.
 * out is bitwise the output of causal_product_fwd on the same inputs.
 * Workspace: causal_product_fwd_norm_workspace_size (or null: allocated on
 * the stream).  Errors as causal_product_fwd and causal_product_normalizer;
 * N = 0 enqueues nothing. */
CP_API size_t causal_product_fwd_norm_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                                     int64_t M, cp_dtype_t dtype);
CP_API cp_status_t causal_product_fwd_norm(const void* q, const void* k, const void* v, void* out,
                                           float* z, int64_t B, int64_t H, int64_t N, int64_t D,
                                           int64_t M, cp_dtype_t dtype, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* Backward of causal_product_normalizer: with grad_z = dL/dz [B,H,N] fp32,
 *     grad_q_i = grad_z_i sum_{j<=i} k_j,
 *     grad_k_j = sum_{i>=j} grad_z_i q_i,
 * written in `dtype` ([B,H,N,D], overlapping nothing).  Two launches on
 * `stream`; same workspace size as the forward. */
CP_API cp_status_t causal_product_normalizer_bwd(const void* q, const void* k, const float* grad_z,
                                                 void* grad_q, void* grad_k, int64_t B, int64_t H,
                                                 int64_t N, int64_t D, cp_dtype_t dtype,
                                                 void* workspace, size_t workspace_bytes,
                                                 void* stream);

/* Forward with the feature map applied on load: out_i = sum_{j<=i}
 * (phi(q_i) . phi(k_j)) v_j for raw inputs q, k (the linear-attention
 * features phi(x) of "Transformers are RNNs"; the pages of
 * triton-lang/triton issue #217 feed the product such features).  phi is
 * computed inside the product kernels (on the tensor-core path, in shared
 * memory after the tile is loaded; bf16 operands are phi rounded to bf16), so
 * phi(q) and phi(k) are never written to memory.  Arguments, layout and
 * workspace as causal_product_fwd (its workspace size serves);
 * feature = CP_FEATURE_NONE is causal_product_fwd. */
CP_API cp_status_t causal_product_fwd_feature(const void* q, const void* k, const void* v,
                                              void* out, cp_feature_t feature, int64_t B,
                                              int64_t H, int64_t N, int64_t D, int64_t M,
                                              cp_dtype_t dtype, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* Backward of causal_product_fwd_feature: grad_q = phi'(q) * dL/dphi(q),
 * grad_k = phi'(k) * dL/dphi(k) (elementwise), grad_v as causal_product_bwd,
 * with phi'(x) = 1 for x > 0 and e^x otherwise.  bf16: three tensor-core
 * products on the raw rows (dq from (g, v, phi(k)), dv from the reverse
 * (phi(k), phi(q), g), dk from the reverse (v, g, phi(q))), phi applied to
 * the tiles in shared memory and phi' to each gradient element before its
 * store, so neither phi(q), phi(k) nor an unscaled gradient is written.
 * fp32 and fp16: phi(q) and phi(k) into the workspace, the product backward
 * on them, then the elementwise chain rule in place on grad_q and grad_k.
 * Workspace: at least causal_product_feature_workspace_size(..., backward =
 * 1) bytes (NULL: allocated and freed on `stream`). */
CP_API cp_status_t causal_product_bwd_feature(const void* q, const void* k, const void* v,
                                              const void* grad_out, void* grad_q, void* grad_k,
                                              void* grad_v, cp_feature_t feature, int64_t B,
                                              int64_t H, int64_t N, int64_t D, int64_t M,
                                              cp_dtype_t dtype, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* Workspace bytes of causal_product_fwd_feature (backward = 0, the same as
 * causal_product_fwd) or causal_product_bwd_feature (backward = 1: the
 * backward's workspace, plus phi(q) and phi(k) for fp32 and fp16); 0 for
 * rejected arguments. */
CP_API size_t causal_product_feature_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                                    int64_t M, cp_dtype_t dtype, int backward);

/* The normaliser of mapped features from raw inputs: z_i = phi(q_i) .
 * sum_{j<=i} phi(k_j) with phi applied inside the kernel, and its backward
 * with respect to the raw q, k (grad_q = phi'(q) * grad_z sum phi(k),
 * grad_k = phi'(k) * sum grad_z phi(q)), so that causal linear attention
 * from raw inputs, causal_product_fwd_feature(...) / z, never writes phi(q)
 * or phi(k) to memory.  Arguments as causal_product_normalizer /
 * causal_product_normalizer_bwd (same workspace size); feature =
 * CP_FEATURE_NONE is those calls.  A feature map needs rows of 16-byte
 * multiples (D % 8 == 0 for bf16 and fp16, D % 4 == 0 for fp32);
 * CP_ERR_UNSUPPORTED_SHAPE otherwise. */
CP_API cp_status_t causal_product_normalizer_feature(const void* q, const void* k, float* z,
                                                     cp_feature_t feature, int64_t B, int64_t H,
                                                     int64_t N, int64_t D, cp_dtype_t dtype,
                                                     void* workspace, size_t workspace_bytes,
                                                     void* stream);
CP_API cp_status_t causal_product_normalizer_bwd_feature(const void* q, const void* k,
                                                         const float* grad_z, void* grad_q,
                                                         void* grad_k, cp_feature_t feature,
                                                         int64_t B, int64_t H, int64_t N,
                                                         int64_t D, cp_dtype_t dtype,
                                                         void* workspace, size_t workspace_bytes,
                                                         void* stream);

/* Positive random features (the Performer feature map "FAVOR+"; the pages
 * of triton-lang/triton issue #217 offer the causal product as a drop-in for
 * the Performers code):
 *     phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D),   d = 0 .. D-1,
 *     out_i    = sum_{j<=i} (phi(xq_i) . phi(xk_j)) v_j,
 * from the raw rows xq, xk [B][H][N][R] and one projection W [D][R] (row d is
 * w_d) shared by every row and (b,h).  bf16 only: xq, xk, v, W, out (and the
 * gradients) are bf16 device pointers, 16-byte aligned; R in 8 .. 64 (a
 * multiple of 8), D in 64 .. 256 (a multiple of 64), M as for
 * causal_product_fwd.  The features are computed on the tensor cores (X W^T,
 * fp32 accumulation), exponentiated in fp32 and rounded to bf16 once.
 * causal_product_bwd_favor writes dL/dxq, dL/dxk (with respect to the raw
 * rows, W fixed: dL/dx = sum_d a_d phi_d (w_d - x), a = dL/dphi) and dL/dv.
 * Workspace: causal_product_favor_workspace_size(..., backward) bytes (NULL:
 * allocated on `stream`); it holds phi(xq), phi(xk) (and, backward, their
 * gradients).  CP_ERR_UNSUPPORTED_DTYPE for fp32/fp16,
 * CP_ERR_UNSUPPORTED_SHAPE for R or D out of range; otherwise errors as
 * causal_product_fwd.  N = 0 enqueues nothing. */
CP_API size_t causal_product_favor_workspace_size(int64_t B, int64_t H, int64_t N, int64_t R,
                                                  int64_t D, int64_t M, cp_dtype_t dtype,
                                                  int backward);
CP_API cp_status_t causal_product_fwd_favor(const void* xq, const void* xk, const void* v,
                                            const void* W, void* out, int64_t B, int64_t H,
                                            int64_t N, int64_t R, int64_t D, int64_t M,
                                            cp_dtype_t dtype, void* workspace,
                                            size_t workspace_bytes, void* stream);
CP_API cp_status_t causal_product_bwd_favor(const void* xq, const void* xk, const void* v,
                                            const void* W, const void* grad_out, void* grad_xq,
                                            void* grad_xk, void* grad_v, int64_t B, int64_t H,
                                            int64_t N, int64_t R, int64_t D, int64_t M,
                                            cp_dtype_t dtype, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* Size of the static device scratch array behind causal_product_fwd_noalloc. */
#define CP_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* Forward pass that allocates nothing: no cudaMalloc, no stream-ordered or
 * library allocation.  It is meant for callers that must not allocate device
 * memory themselves or through this library -- for example code running
 * inside a host framework that owns every device allocation (plugins of
 * inference runtimes with their own memory pools), or code that must not
 * call cudaMalloc because it may synchronise the device.  (The paper has no
 * counterpart of this entry point; it is a deployment convenience.)
 *
 * Same arguments, layout, ownership and result as causal_product_fwd, minus
 * the workspace: its scratch (status word and scan aggregates) lives in one
 * file-scope __device__ array of CP_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU loading the library holds until the process exits.  The first call on
 * a device, with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  Problems whose scratch would exceed the array return
 * CP_ERR_NOALLOC_LIMIT before enqueuing anything.  The array is shared by
 * every call and keeps the last call's contents; calls that overlap on the
 * GPU (different streams, no ordering between them) race on it.  Its first
 * bytes hold a status word shared by every call on the device: it starts
 * clear when the library's module is loaded, a kernel whose bounded wait runs
 * out writes CP_ERR_TIMEOUT into it (the outputs of that call are then
 * undefined), and it stays set until causal_product_noalloc_status reads it. */
CP_API cp_status_t causal_product_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                              int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                              cp_dtype_t dtype, void* stream);

/* Synchronises `stream`, then returns and clears the status word of the
 * static scratch array behind causal_product_fwd_noalloc on the current
 * device: CP_OK, CP_ERR_TIMEOUT if any call since the last read recorded a
 * timeout, or CP_ERR_CUDA if the stream reports an error.  Allocates
 * nothing.  (No counterpart in the paper; it completes the allocation-free
 * entry point, whose callers have no workspace to pass to
 * causal_product_status.) */
CP_API cp_status_t causal_product_noalloc_status(void* stream);

/* Self-test of the failure path (no counterpart on the pages): one block
 * waits on a barrier that nothing arrives at, gives up after `wait_ns`
 * nanoseconds (1 ns .. 1 s) and records CP_ERR_TIMEOUT in the status word of
 * `workspace` (at least 256 bytes, 16-byte aligned), exactly as a kernel
 * whose bounded wait runs out.  No fault, no trap; the context stays usable.
 * Read the result with causal_product_status. */
CP_API cp_status_t causal_product_selftest_timeout(void* workspace, uint64_t wait_ns,
                                                   void* stream);

/* Synchronises `stream`, then returns and clears the status word in
 * `workspace` (CP_OK or CP_ERR_TIMEOUT), or CP_ERR_CUDA if the stream
 * reports an error. */
CP_API cp_status_t causal_product_status(void* workspace, void* stream);

/* Static, human-readable name of a status code. */
CP_API const char* causal_product_error_string(cp_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* CAUSAL_PRODUCT_H_ */
