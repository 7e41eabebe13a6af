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

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum diffattn_status {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer, bad dtype */
    DIFFATTN_ERR_UNSUPPORTED = 2, /* valid request outside the implemented domain */
    DIFFATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    DIFFATTN_ERR_TIMEOUT = 4      /* written to status_dev by a kernel whose wait ran out */
} diffattn_status;

typedef enum diffattn_dtype {
    DIFFATTN_BF16 = 0, /* q/k/v/out bf16, fp32 accumulation */
    DIFFATTN_F32 = 1   /* q/k/v/out fp32 throughout */
} diffattn_dtype;

/* Problem description shared by diffattn_fwd and diffattn_headnorm. */
typedef struct diffattn_desc {
    int64_t B;            /* batch size, >= 0 */
    int64_t H;            /* differential heads, >= 0 */
    int64_t N;            /* tokens (queries = keys), >= 0 */
    int32_t d;            /* width of one query/key half; V and out have 2d columns */
    int32_t dtype;        /* diffattn_dtype of q1, k1, q2, k2, v and out */
    int32_t causal;       /* 1: key j visible to query i iff j <= i; 0: all visible */
    int32_t headnorm;     /* 1: apply RMS head norm, w and (1 - lambda_init); 0: raw o */
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
 * norm_w device float32 [H, 2d] or NULL (ones; only read when headnorm = 1);
 * out device [B, H, N, 2d] in desc->dtype, fully overwritten; stream a
 * cudaStream_t or NULL.
 *
 * Supported domain (anything else is DIFFATTN_ERR_UNSUPPORTED):
 *   - DIFFATTN_BF16: d == 64 (2d = 128); any N >= 1 (a ragged last tile is
 *     masked); B * H * ceil(N / 128) <= 2^31 - 1.  q1, k1, q2, k2, v must be
 *     16-byte aligned (DIFFATTN_ERR_INVALID_ARG otherwise).  Runs the fused
 *     tcgen05/TMEM/TMA kernel; needs an sm_103 device.
 *   - DIFFATTN_F32: 1 <= d <= 128, N <= 4096.  Plain CUDA-core kernel
 *     (accurate expf, fp32 accumulation).
 * B * H * N == 0 returns DIFFATTN_OK without launching anything.
 */
diffattn_status diffattn_fwd(const diffattn_desc *desc, const void *q1, const void *k1,
                             const void *q2, const void *k2, const void *v,
                             const float *lambda, const float *norm_w, void *out,
                             void *stream);

/*
 * diffattn_headnorm — the per-head output normalisation on its own
 * ("Differential Transformer", section "How differential attention works":
 * each head's output normalised individually, then times (1 - lambda_init)):
 *   out[b,h,i,c] = x[b,h,i,c] / sqrt(mean_c x[b,h,i,:]^2 + eps) * w[h,c] * (1 - lambda_init)
 *
 * x is device float32 [B, H, N, 2d]; norm_w device float32 [H, 2d] or NULL;
 * out device [B, H, N, 2d] in desc->dtype (bf16 rounded to nearest even, or
 * fp32).  desc->causal and desc->headnorm are ignored.  Supported: 1 <= d <= 128.
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

/* Static, NUL-terminated description of a status code (never NULL). */
const char *diffattn_strerror(diffattn_status status);

/* Library version as 10000 * major + 100 * minor + patch. */
int diffattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
