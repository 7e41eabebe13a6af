/*
 * libdiffattn: differential-attention head forward pass on NVIDIA GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The operation (source: "Differential Transformer", Ultralytics glossary,
 * section "How differential attention works"):
 *
 *   map1 = softmax_j(Q1 K1^T / sqrt(d))        per head, over keys j
 *   map2 = softmax_j(Q2 K2^T / sqrt(d))
 *   o    = (map1 - lambda_h * map2) V            V and o have 2d columns
 *
 * and, in the model the page describes, each head's output is normalised on
 * its own and then multiplied by (1 - lambda_init), where
 * lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)) for layer l.  This library
 * takes the normalisation as the RMS form over the 2d channels of one
 * (batch, head, token):
 *
 *   y[c] = o[c] / sqrt(mean_c(o^2) + eps) * w[h, c] * (1 - lambda_init)
 *
 * (headnorm = 1), or, with headnorm = 2, the mean-subtracting form the page
 * names (GroupNorm with one group per head, no bias):
 *
 *   y[c] = (o[c] - mean_c o) / sqrt(var_c(o) + eps) * w[h, c] * (1 - lambda_init)
 *
 * Conventions shared by every entry point:
 *   - All tensors are caller-owned, contiguous, row-major device buffers.
 *     The library allocates no device memory, never frees a caller buffer,
 *     and keeps no pointer after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL means the legacy default stream).  A DIFFATTN_OK return means the
 *     work was enqueued; kernel-side failures are reported through
 *     desc->status_dev (below).
 *   - Validation failures return before anything is launched.  A failed CUDA
 *     launch returns DIFFATTN_ERR_CUDA.  No C++ exception crosses the ABI.
 *   - Layout: q1, k1, q2, k2 are [B, H, N, d]; v and out are [B, H, N, 2d];
 *     lambda is float32 [H]; norm_w is float32 [H, 2d] or NULL (all ones).
 *   - Masking: causal = 1 means key j is visible to query i iff j <= i
 *     (square attention, same mask for both maps); causal = 0 means every
 *     key is visible.
 *   - The scale is 1/sqrt(d) with d the width of one query/key half, as in
 *     the page's worked example (d = 8, values of width 2d = 16).
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum diffattn_status {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer, bad dtype */
    DIFFATTN_ERR_UNSUPPORTED = 2, /* valid request outside the implemented domain */
    DIFFATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    DIFFATTN_ERR_TIMEOUT = 4,     /* written to status_dev by a kernel whose wait ran out */
    DIFFATTN_ERR_BOUNDS = 5       /* debug build only (compiled with DIFFATTN_DEBUG): a
                                     kernel's bounds check failed; status_dev holds
                                     5 | (site << 8) of the first failing check, and the
                                     checked access was skipped */
} diffattn_status;

typedef enum diffattn_dtype {
    DIFFATTN_BF16 = 0,    /* q/k/v/out bf16, fp32 accumulation */
    DIFFATTN_F32 = 1,     /* q/k/v/out fp32 throughout */
    DIFFATTN_E4M3_QK = 2  /* q1, k1, q2, k2 fp8 e4m3 (one byte each); v and out bf16;
                             fp32 accumulation (diffattn_fwd, d == 64 only) */
} diffattn_dtype;

/* Problem description shared by every entry point. */
typedef struct diffattn_desc {
    int64_t B;            /* batch size, >= 0 */
    int64_t H;            /* differential heads, >= 0 */
    int64_t N;            /* tokens: queries = keys (diffattn_fwd_kv: queries), >= 0 */
    int32_t d;            /* width of one query/key half; V and out have 2d columns */
    int32_t dtype;        /* diffattn_dtype of q1, k1, q2, k2, v and out */
    int32_t causal;       /* 1: key j visible to query i iff j <= i; 0: all visible */
    int32_t headnorm;     /* 0: raw o; 1: RMS head norm, w and (1 - lambda_init);
                             2: mean-subtracting head norm (the page's GroupNorm, one
                             group per head, no bias), w and (1 - lambda_init) */
    float eps;            /* RMS norm epsilon (inside the square root), >= 0 */
    float lambda_init;    /* the (1 - lambda_init) output scale uses this value */
    int32_t *status_dev;  /* optional device int32 (NULL = none).  Kernels never clear
                             it; a kernel whose internal pipeline wait exceeds its time
                             limit stores DIFFATTN_ERR_TIMEOUT there and returns early
                             (output then undefined).  The caller zeroes it and reads it
                             after synchronising. */
} diffattn_desc;

/*
 * diffattn_fwd — the full differential-attention head forward:
 *   out = headnorm ? RMSNorm_h((map1 - lambda_h map2) V) * w_h * (1 - lambda_init)
 *                  : (map1 - lambda_h map2) V
 * ("Differential Transformer", section "How differential attention works":
 * the two-map formula, values twice as wide as a query/key half, the per-head
 * normalisation and the (1 - lambda_init) scale.)
 *
 * Arguments: desc as above; q1, k1, q2, k2 device [B, H, N, d]; v device
 * [B, H, N, 2d]; lambda device float32 [H] (any finite value, not clamped);
 * norm_w device float32 [H, 2d] or NULL (ones; read when headnorm is 1 or 2);
 * out device [B, H, N, 2d] in desc->dtype, fully overwritten; stream a
 * cudaStream_t or NULL.
 *
 * Supported domain (anything else is DIFFATTN_ERR_UNSUPPORTED):
 *   - DIFFATTN_BF16: d == 64 (2d = 128) or d == 128 (2d = 256); any N >= 1
 *     (a ragged last tile is masked); B * H * ceil(N / 128) <= 2^31 - 1.  q1,
 *     k1, q2, k2, v must be 16-byte aligned (DIFFATTN_ERR_INVALID_ARG
 *     otherwise).  Runs a fused tcgen05/TMEM/TMA kernel (for d == 128 a
 *     two-pass one: row statistics, then a single normalised accumulator);
 *     needs an sm_103 device.  diffattn_fwd_strided takes both head widths;
 *     so does the key/value-cache entry (diffattn_fwd_kv, single pass), and
 *     so does training.
 *   - DIFFATTN_F32: 1 <= d <= 128, N <= 4096.  Plain CUDA-core kernel
 *     (accurate expf, fp32 accumulation).
 *   - DIFFATTN_E4M3_QK: d == 64, headnorm 0 or 1: the d == 64 kernel with the
 *     two Q K^T products on fp8 (e4m3) tensor-core MMAs; P V stays bf16.  The
 *     result is that of the same formula applied to the e4m3 input values
 *     (exactly representable, so only P and the output are rounded as in the
 *     bf16 path).  The page remarks that differential attention keeps its
 *     accuracy under low-bit quantisation; this is that input format.
 * B * H * N == 0 returns DIFFATTN_OK without launching anything.
 */
diffattn_status diffattn_fwd(const diffattn_desc *desc, const void *q1, const void *k1,
                             const void *q2, const void *k2, const void *v,
                             const float *lambda, const float *norm_w, void *out,
                             void *stream);

/* Element strides of one [B, H, rows, width] tensor whose rows (width
 * elements) are contiguous: element (b, h, i, c) sits at b*b + h*h + i*n + c. */
typedef struct diffattn_strides {
    int64_t b; /* batch stride */
    int64_t h; /* head stride */
    int64_t n; /* row (token) stride */
} diffattn_strides;

/*
 * diffattn_fwd_host — diffattn_fwd with its inputs and its output in host
 * memory: the call a host program makes when the tensors live on the CPU side.
 * Same computation, domain and errors as diffattn_fwd ("Differential
 * Transformer", "How differential attention works").
 *
 * Arguments as diffattn_fwd except: q1, k1, q2, k2, v (same shapes and dtypes)
 * and out_host ([B, H, N, 2d] in the output dtype) are HOST pointers;
 * page-locked memory keeps the copies asynchronous, pageable memory works with
 * the copies synchronising as cudaMemcpyAsync does.  lambda and norm_w stay
 * device pointers.  staging: a device buffer, 256-byte aligned, of at least
 * diffattn_fwd_host_staging_bytes(desc) bytes, owned by the caller; it holds
 * the five inputs and the output (each region rounded up to 256 bytes) and must
 * not be used by another call still in flight.  On `stream`, in order: one
 * host-to-device cudaMemcpyAsync per input, diffattn_fwd on the staged
 * tensors, one device-to-host cudaMemcpyAsync of the output; nothing is
 * allocated.  A NULL, misaligned or short staging buffer is
 * DIFFATTN_ERR_INVALID_ARG; a failed copy is DIFFATTN_ERR_CUDA.
 */
diffattn_status diffattn_fwd_host(const diffattn_desc *desc, const void *q1, const void *k1,
                                  const void *q2, const void *k2, const void *v,
                                  const float *lambda, const float *norm_w, void *out_host,
                                  void *staging, size_t staging_bytes, void *stream);

/* Bytes of the staging buffer diffattn_fwd_host needs for desc (host-only). */
diffattn_status diffattn_fwd_host_staging_bytes(const diffattn_desc *desc, size_t *bytes);

/*
 * diffattn_fwd_strided — diffattn_fwd with caller-given strides, so that
 * q1, k1, q2, k2, v and out may be views of other layouts (for example
 * [B, N, H, d] storage, strides {N*H*d, d, H*d}) without copies.  Same
 * computation and output values as diffattn_fwd on contiguous copies.
 *
 * strides[0..5] are those of q1, k1, q2, k2, v, out, in elements.  Rows must
 * be contiguous; every stride must be a positive multiple of 8 elements (16
 * bytes, the tensor-copy engine's rule) and below 2^39.  Domain: DIFFATTN_BF16,
 * d == 64 or d == 128, any N >= 1, headnorm 0, 1 or 2, 16-byte aligned bases,
 * an sm_103 device; anything else returns an error before launching.
 */
diffattn_status diffattn_fwd_strided(const diffattn_desc *desc, const void *q1, const void *k1,
                                     const void *q2, const void *k2, const void *v,
                                     const float *lambda, const float *norm_w, void *out,
                                     const diffattn_strides *strides, void *stream);

/*
 * diffattn_fwd_kv — the same forward for N queries against n_kv keys, with
 * the key range optionally split across CTAs ("split-KV").
 *
 * What it computes: exactly diffattn_fwd's formula ("Differential
 * Transformer", section "How differential attention works": each map is
 * ordinary softmax attention), with desc->N queries and n_kv keys/values per
 * head.  The queries are the LAST N positions of the sequence: query i sits at
 * position n_kv - N + i, so with causal = 1 it sees keys j <= n_kv - N + i
 * (a key/value cache: N = 1..16 is decoding, N = n_kv is diffattn_fwd).
 * Because each map is a softmax, its key range can be cut into pieces whose
 * partial states (unnormalised accumulator, running maximum, running sum)
 * merge exactly; with splits > 1 the fused kernel writes those states for
 * every (head, 128-query tile, key range) to `workspace` and a second kernel
 * merges them, forms map1 - lambda map2 and applies the head norm.  This
 * fills the GPU when B * H * ceil(N / 128) is small against the SM count.
 *
 * Arguments: q1, q2 device bf16 [B, H, N, d]; k1, k2 device bf16
 * [B, H, n_kv, d]; v device bf16 [B, H, n_kv, 2d]; out device bf16
 * [B, H, N, 2d], fully overwritten; lambda and norm_w as for diffattn_fwd;
 * d = 64, or d = 128 (which runs the two-pass d = 128 kernel over the whole
 * key range: splits 0 and 1 only).
 * With dtype DIFFATTN_E4M3_QK, q1, k1, q2, k2 are e4m3 (one byte each, same
 * shapes) and v, out stay bf16, as for diffattn_fwd.
 * splits: 0 lets the library choose (diffattn_fwd_kv_plan reports the
 * choice), 1 is the single-pass kernel (no workspace), 2..256 cut each row's
 * keys into that many ranges of ceil(ceil(n_kv / 128) / splits) 128-key tiles
 * (requests above ceil(n_kv / 128) are lowered to it).  workspace: device
 * buffer of at least the bytes diffattn_fwd_kv_plan reports, 16-byte aligned,
 * caller-owned scratch whose contents on entry do not matter; unused (may be
 * NULL) when the resolved split count is 1.  Two calls that share a workspace
 * must be ordered (same stream, or synchronised).
 *
 * Errors: DIFFATTN_ERR_INVALID_ARG for a negative n_kv, causal with
 * n_kv < N, n_kv = 0 with queries present, splits outside 0..256, a missing
 * or short workspace, or misaligned buffers; DIFFATTN_ERR_UNSUPPORTED unless
 * dtype is DIFFATTN_BF16 with d == 64, DIFFATTN_BF16 with d == 128 and splits
 * 0 or 1, or DIFFATTN_E4M3_QK with d == 64 and headnorm 0 or 1; and on a
 * non-sm_103 device.
 * B * H * N == 0 returns DIFFATTN_OK without launching anything.
 */
diffattn_status diffattn_fwd_kv(const diffattn_desc *desc, int64_t n_kv, const void *q1,
                                const void *k1, const void *q2, const void *k2,
                                const void *v, const float *lambda, const float *norm_w,
                                void *out, int splits, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * diffattn_fwd_kv_strided — diffattn_fwd_kv with caller-given strides, so that
 * a key/value cache kept in another layout (for example [B, n_kv, H, d]) is
 * read in place.  Same computation and output values as diffattn_fwd_kv on
 * contiguous copies.
 *
 * strides[0..5] are those of q1, k1, q2, k2, v, out, in elements, with the
 * rules of diffattn_fwd_strided (contiguous rows; every stride a positive
 * multiple of 8 elements and below 2^39).  Domain: DIFFATTN_BF16, d == 64 or
 * d == 128 (splits 0 or 1); other arguments, the workspace and the errors as
 * for diffattn_fwd_kv.
 */
diffattn_status diffattn_fwd_kv_strided(const diffattn_desc *desc, int64_t n_kv,
                                        const void *q1, const void *k1, const void *q2,
                                        const void *k2, const void *v, const float *lambda,
                                        const float *norm_w, void *out, int splits,
                                        void *workspace, size_t workspace_bytes,
                                        const diffattn_strides *strides, void *stream);

/*
 * diffattn_fwd_kv_plan — the split count diffattn_fwd_kv runs for this
 * request (splits = 0: the library's choice for the current device, from its
 * SM count and a per-CTA cost model) and the workspace bytes it needs (0 when
 * that count is 1).  Validates exactly as diffattn_fwd_kv does apart from
 * pointers; host-only apart from reading the device's SM count once.
 */
diffattn_status diffattn_fwd_kv_plan(const diffattn_desc *desc, int64_t n_kv, int splits,
                                     int *splits_out, size_t *workspace_bytes);

/*
 * Training: diffattn_fwd_train saves what the backward pass needs and
 * diffattn_bwd returns the gradients of sum(out * dy) with respect to q1, k1,
 * q2, k2, v, lambda and the norm weight.
 *
 * The pages define the forward only ("Differential Transformer", section "How
 * differential attention works"); the backward is its derivative by the
 * chain rule: with o_k = map_k V (k = 1, 2), o = o1 - lambda o2 and, with the
 * norm, y = o r g, r = 1/sqrt(mean(o^2) + eps), g = w (1 - lambda_init):
 *   do = r g dy - (r^3 / 2d) o sum_c(dy g o)  (do = dy without the norm;
 *        with the group form o is the centred row and do then loses its mean)
 *   dw = sum_rows dy o r (1 - lambda_init);  dlambda = -sum_rows do . o2
 *   dV = map1^T do - lambda map2^T do;  dW = do V^T
 *   dS_1 = P_1 * (dW - do.o1),  dS_2 = -lambda P_2 * (dW - do.o2)  (per row)
 *   dQ_k = dS_k K_k / sqrt(d),  dK_k = dS_k^T Q_k / sqrt(d)
 *
 * Domain: DIFFATTN_BF16, d == 64 or d == 128, square attention (N queries =
 * N keys), causal or not, headnorm 0, 1 or 2 (the group form: the page's
 * GroupNorm); an sm_103 device.  d == 128 runs its own kernels: the saving
 * forward is the d == 128 forward (the output with each map's log2-sum-exp
 * and the pre-norm o) and then one pass over the keys for map 2's output from
 * its saved statistics, and the backward two kinds of
 * work item (one computing dV from both maps, one computing one map's dK and
 * dQ), since the d == 64 kernel's tensor-memory layout does not fit 2d = 256.
 */

/* Bytes of the saved-activation buffer diffattn_fwd_train fills and of the
 * workspace diffattn_bwd needs (host-only). */
diffattn_status diffattn_train_sizes(const diffattn_desc *desc, size_t *saved_bytes,
                                     size_t *workspace_bytes);

/*
 * diffattn_fwd_train — diffattn_fwd (same arguments, same `out`, bitwise)
 * that also writes `saved` (caller-owned device buffer of at least
 * saved_bytes from diffattn_train_sizes, 16-byte aligned): each map's
 * normalised output o_k (fp32 [2][B*H][N][2d]; for d == 128 the first holds
 * o = o_1 - lambda o_2 before the norm instead of o_1) and log2-sum-exp
 * (fp32 [2][B*H][128 * ceil(N / 128)]; for d == 128 each region starts on a
 * 256-byte boundary).  Keep it unchanged until the matching diffattn_bwd has
 * run.
 */
diffattn_status diffattn_fwd_train(const diffattn_desc *desc, const void *q1, const void *k1,
                                   const void *q2, const void *k2, const void *v,
                                   const float *lambda, const float *norm_w, void *out,
                                   void *saved, size_t saved_bytes, void *stream);

/*
 * diffattn_bwd — gradients given the forward inputs, the same desc, lambda
 * and norm_w, the `saved` buffer of diffattn_fwd_train and dy (bf16
 * [B, H, N, 2d]).  Outputs (all device, overwritten): dq1, dk1, dq2, dk2
 * bf16 [B, H, N, d]; dv bf16 [B, H, N, 2d]; dlambda fp32 [H]; dnorm_w fp32
 * [H, 2d] (written when headnorm is 1 or 2; may be NULL to skip it).
 * workspace: caller-owned scratch of at least workspace_bytes from
 * diffattn_train_sizes, 256-byte aligned (its contents on entry do not
 * matter).  dq (and, for d == 64, dv) is summed over key tiles, dlambda and
 * dnorm_w over row blocks, with fp32 atomic adds, so their last bits can
 * differ between runs; dk (and, for d == 128, dv) is written once per key
 * tile and is deterministic.  Errors as for diffattn_fwd; DIFFATTN_ERR_INVALID_ARG also for a
 * missing or misaligned buffer or a short workspace.
 */
diffattn_status diffattn_bwd(const diffattn_desc *desc, const void *q1, const void *k1,
                             const void *q2, const void *k2, const void *v,
                             const float *lambda, const float *norm_w, const void *saved,
                             const void *dy, void *dq1, void *dk1, void *dq2, void *dk2,
                             void *dv, float *dlambda, float *dnorm_w, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * diffattn_fwd_train_strided — diffattn_fwd_train with caller-given strides
 * for q1, k1, q2, k2, v and out (strides[0..5], the rules of
 * diffattn_fwd_strided: contiguous rows, every stride a positive multiple of 8
 * elements and below 2^39).  `out` is bitwise that of diffattn_fwd_strided and
 * `saved` that of diffattn_fwd_train on contiguous copies; the saved buffer
 * itself is the library's contiguous layout.  Domain and errors as for
 * diffattn_fwd_train.
 */
diffattn_status diffattn_fwd_train_strided(const diffattn_desc *desc, const void *q1,
                                           const void *k1, const void *q2, const void *k2,
                                           const void *v, const float *lambda,
                                           const float *norm_w, void *out, void *saved,
                                           size_t saved_bytes,
                                           const diffattn_strides *strides, void *stream);

/*
 * diffattn_bwd_strided — diffattn_bwd with caller-given strides, so that the
 * inputs and the gradients may be views of other layouts (for example
 * [B, N, H, d] storage) without copies.  strides[0..10] are those of q1, k1,
 * q2, k2, v, dy, dq1, dk1, dq2, dk2, dv, in elements, with the rules of
 * diffattn_fwd_strided.  The same gradients as diffattn_bwd on contiguous
 * copies (dk bitwise; dq, dv, dlambda and dnorm_w up to the order of their
 * fp32 atomic sums).  Domain, workspace and errors as for diffattn_bwd.
 */
diffattn_status diffattn_bwd_strided(const diffattn_desc *desc, const void *q1, const void *k1,
                                     const void *q2, const void *k2, const void *v,
                                     const float *lambda, const float *norm_w,
                                     const void *saved, const void *dy, void *dq1, void *dk1,
                                     void *dq2, void *dk2, void *dv, float *dlambda,
                                     float *dnorm_w, void *workspace, size_t workspace_bytes,
                                     const diffattn_strides *strides, void *stream);

/* Size of the scratch area diffattn_fwd_kv_noalloc uses: 64 MiB. */
#define DIFFATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * diffattn_fwd_kv_noalloc — diffattn_fwd_kv without a caller workspace.
 * The pages have no counterpart to this entry point: it is a convenience of
 * this library for callers that cannot hand over scratch memory.
 *
 * Computes exactly what diffattn_fwd_kv computes, with the same arguments
 * apart from the workspace: the split-KV partial blocks go to a fixed
 * DIFFATTN_NOALLOC_SCRATCH_BYTES area that the library owns (a static device
 * array of its module; nothing is allocated).  Its device address is looked
 * up with cudaGetSymbolAddress on every call that needs it (after a context
 * reset the module may sit at another address, so none is kept between
 * calls); a failed lookup returns DIFFATTN_ERR_CUDA.  Nothing in the area has
 * to start at zero, so nothing is cleared.
 *
 * Errors: those of diffattn_fwd_kv and diffattn_fwd_kv_plan, plus
 * DIFFATTN_ERR_UNSUPPORTED when the planned workspace exceeds
 * DIFFATTN_NOALLOC_SCRATCH_BYTES (checked before anything is launched).
 *
 * Caveats: every call on a device shares the one scratch area, so calls
 * that overlap in time (different streams, or different host threads without
 * ordering) race on it and give undefined results; order them.  The first
 * call on each device performs the set-up (its symbol lookup can load the
 * module), so it must come before any CUDA stream capture that records this
 * entry point.
 */
diffattn_status diffattn_fwd_kv_noalloc(const diffattn_desc *desc, int64_t n_kv,
                                        const void *q1, const void *k1, const void *q2,
                                        const void *k2, const void *v, const float *lambda,
                                        const float *norm_w, void *out, int splits,
                                        void *stream);

/*
 * diffattn_headnorm — the per-head output normalisation on its own
 * ("Differential Transformer", section "How differential attention works":
 * each head's output normalised individually, then times (1 - lambda_init)):
 *   out[b,h,i,c] = x[b,h,i,c] / sqrt(mean_c x[b,h,i,:]^2 + eps) * w[h,c] * (1 - lambda_init)
 *
 * x is device float32 [B, H, N, 2d]; norm_w device float32 [H, 2d] or NULL;
 * out device [B, H, N, 2d] in desc->dtype (bf16 rounded to nearest even, or
 * fp32).  desc->headnorm = 2 selects the mean-subtracting form, 0 or 1 the RMS
 * form; desc->causal is ignored.  Supported: 1 <= d <= 128.
 */
diffattn_status diffattn_headnorm(const diffattn_desc *desc, const float *x,
                                  const float *norm_w, void *out, void *stream);

/*
 * diffattn_lambda_init — lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)), layers
 * numbered from 1 ("Differential Transformer", section "How differential
 * attention works": the initial value of lambda for layer l).  Host-only,
 * pure function, any int accepted.
 */
double diffattn_lambda_init(int layer);

/*
 * diffattn_selftest_wait — diagnostic with no counterpart on the pages: it
 * exercises the bounded pipeline wait every kernel here relies on (see
 * status_dev above) without faulting or hanging the device.  One warp waits
 * on an mbarrier that nothing ever arrives on, limited to timeout_ns; a second
 * warp waits on another such barrier with the kernels' full 2 s limit and
 * leaves as soon as the first raises the shared abort flag.
 * status_dev: device int32[3], written as {DIFFATTN_ERR_TIMEOUT if the wait
 * ran out and raised the flag (else 0), first wait in microseconds, second
 * wait in microseconds}.  timeout_ns in (0, 2e9].  Asynchronous on stream.
 */
diffattn_status diffattn_selftest_wait(int32_t *status_dev, int64_t timeout_ns, void *stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *diffattn_strerror(diffattn_status status);

/* Library version as 10000 * major + 100 * minor + patch. */
int diffattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
