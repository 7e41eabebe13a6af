// Per-head RMS normalisation of an fp32 [B, H, N, 2d] tensor, times the
// per-head weight and (1 - lambda_init) ("Differential Transformer",
// Ultralytics glossary, section "How differential attention works": each
// head's output is normalised on its own, then scaled by (1 - lambda_init)).
//
// Memory-bound: one warp per row, lanes stride the row's 2d channels so each
// warp instruction touches one contiguous 128-byte segment; grid sized as a
// multiple of the SM count and grid-strided over rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace diffattn {
namespace {

constexpr int WARPS = 8;
constexpr int MAX_PER_LANE = 2 * kF32MaxD / 32;  // 8

template <bool kBf16Out>
__global__ void __launch_bounds__(WARPS * 32)
    diffattn_headnorm_kernel(const float *__restrict__ x, const float *__restrict__ w,
                             void *__restrict__ out, int64_t rows, int32_t N, int32_t H,
                             int32_t dv, float eps, float out_scale, int32_t centre) {
  const int lane = threadIdx.x % 32;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * WARPS;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * WARPS + threadIdx.x / 32; row < rows;
       row += warps_total) {
    const float *xr = x + row * dv;
    float v[MAX_PER_LANE];
    float sm = 0.f;
#pragma unroll
    for (int t = 0; t < MAX_PER_LANE; ++t) {
      const int c = lane + 32 * t;
      v[t] = c < dv ? __ldg(xr + c) : 0.f;
      sm += v[t];
    }
    if (centre) {  // mean-subtracting (group) form
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      const float mu = sm / static_cast<float>(dv);
#pragma unroll
      for (int t = 0; t < MAX_PER_LANE; ++t)
        if (lane + 32 * t < dv) v[t] -= mu;
    }
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < MAX_PER_LANE; ++t) ss = fmaf(v[t], v[t], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / static_cast<float>(dv) + eps) * out_scale;
    const int h = static_cast<int>((row / N) % H);
    const float *wr = w ? w + static_cast<int64_t>(h) * dv : nullptr;
#pragma unroll
    for (int t = 0; t < MAX_PER_LANE; ++t) {
      const int c = lane + 32 * t;
      if (c < dv) {
        const float y = v[t] * r * (wr ? __ldg(wr + c) : 1.f);
        if (kBf16Out)
          static_cast<__nv_bfloat16 *>(out)[row * dv + c] = __float2bfloat16_rn(y);
        else
          static_cast<float *>(out)[row * dv + c] = y;
      }
    }
  }
}

}  // namespace

diffattn_status launch_headnorm(const diffattn_desc &desc, const float *x, const float *norm_w,
                                void *out, cudaStream_t stream) {
  const int64_t rows = desc.B * desc.H * desc.N;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;
  const int64_t blocks_needed = (rows + WARPS - 1) / WARPS;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident blocks of 256 threads per SM
  const unsigned blocks = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
  const int dv = 2 * desc.d;
  const float out_scale = 1.0f - desc.lambda_init;
  if (desc.dtype == DIFFATTN_BF16)
    diffattn_headnorm_kernel<true><<<blocks, WARPS * 32, 0, stream>>>(
        x, norm_w, out, rows, static_cast<int32_t>(desc.N), static_cast<int32_t>(desc.H), dv,
        desc.eps, out_scale, desc.headnorm == 2 ? 1 : 0);
  else
    diffattn_headnorm_kernel<false><<<blocks, WARPS * 32, 0, stream>>>(
        x, norm_w, out, rows, static_cast<int32_t>(desc.N), static_cast<int32_t>(desc.H), dv,
        desc.eps, out_scale, desc.headnorm == 2 ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
