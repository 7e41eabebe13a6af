// Launchers behind the C ABI.  Each takes an already validated descriptor and
// enqueues its kernel on `stream`; none allocates memory.
#pragma once

#include <cuda_runtime.h>

#include "../../include/diffattn.h"

namespace diffattn {

// Fused bf16 forward on tcgen05 / TMEM / TMA (d = 64).
diffattn_status launch_fwd_bf16_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, void *out,
                                      cudaStream_t stream);

// fp32 forward on CUDA cores (d <= 128, N <= 4096).
diffattn_status launch_fwd_f32(const diffattn_desc &desc, const float *q1, const float *k1,
                               const float *q2, const float *k2, const float *v,
                               const float *lambda, const float *norm_w, float *out,
                               cudaStream_t stream);

// Per-head RMS normalisation of an fp32 [B, H, N, 2d] tensor.
diffattn_status launch_headnorm(const diffattn_desc &desc, const float *x, const float *norm_w,
                                void *out, cudaStream_t stream);

constexpr int kF32MaxN = 4096;
constexpr int kF32MaxD = 128;

}  // namespace diffattn
