// fp32 differential-attention head forward on CUDA cores.
//
// For small problems (the glossary page's 6-token worked example, tiny
// shapes) where no tensor-core tile fits and fp32 accuracy is wanted.  The
// method ("Differential Transformer", Ultralytics glossary, section "How
// differential attention works"): out = (softmax(Q1 K1^T/sqrt(d)) -
// lambda softmax(Q2 K2^T/sqrt(d))) V, optionally followed by the per-head RMS
// normalisation, weight and (1 - lambda_init) scale.
//
// One warp per query row.  The row's logits for both maps are kept in shared
// memory (2 N floats per warp), the maxima and sums are warp reductions, and
// each lane then accumulates its own value columns.  Accurate expf.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace diffattn {
namespace {

constexpr int WARPS = 4;
constexpr int MAX_COLS_PER_LANE = 2 * kF32MaxD / 32;  // 8

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

struct F32Params {
  int64_t BH;
  int32_t H, N, d;
  int32_t causal, headnorm;
  float scale, eps, out_scale;
  const float *q1, *k1, *q2, *k2, *v, *lambda, *norm_w;
  float *out;
};

__global__ void __launch_bounds__(WARPS * 32) diffattn_fwd_f32_kernel(const F32Params p) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t bh = blockIdx.y;
  const int i = blockIdx.x * WARPS + warp;
  if (i >= p.N) return;  // no block-wide synchronisation below
  const int N = p.N, d = p.d, dv = 2 * d;
  float *l1 = sm + static_cast<size_t>(warp) * 2 * N;
  float *l2 = l1 + N;
  const float *q1 = p.q1 + (bh * N + i) * d;
  const float *q2 = p.q2 + (bh * N + i) * d;
  const float *k1 = p.k1 + bh * N * d;
  const float *k2 = p.k2 + bh * N * d;
  const float *v = p.v + bh * N * dv;
  const int n_vis = p.causal ? i + 1 : N;

  float m1 = -INFINITY, m2 = -INFINITY;
  for (int j = lane; j < n_vis; j += 32) {
    float s1 = 0.f, s2 = 0.f;
    for (int c = 0; c < d; ++c) {
      s1 = fmaf(q1[c], k1[static_cast<int64_t>(j) * d + c], s1);
      s2 = fmaf(q2[c], k2[static_cast<int64_t>(j) * d + c], s2);
    }
    s1 *= p.scale;
    s2 *= p.scale;
    l1[j] = s1;
    l2[j] = s2;
    m1 = fmaxf(m1, s1);
    m2 = fmaxf(m2, s2);
  }
  m1 = warp_max(m1);
  m2 = warp_max(m2);
  float z1 = 0.f, z2 = 0.f;
  for (int j = lane; j < n_vis; j += 32) {
    const float e1 = expf(l1[j] - m1), e2 = expf(l2[j] - m2);
    l1[j] = e1;
    l2[j] = e2;
    z1 += e1;
    z2 += e2;
  }
  z1 = warp_sum(z1);
  z2 = warp_sum(z2);
  __syncwarp();
  const float a1 = 1.f / z1;
  const float a2 = p.lambda[bh % p.H] / z2;

  float o[MAX_COLS_PER_LANE];
#pragma unroll
  for (int t = 0; t < MAX_COLS_PER_LANE; ++t) o[t] = 0.f;
  for (int j = 0; j < n_vis; ++j) {
    const float wgt = l1[j] * a1 - l2[j] * a2;
    const float *vj = v + static_cast<int64_t>(j) * dv;
#pragma unroll
    for (int t = 0; t < MAX_COLS_PER_LANE; ++t) {
      const int c = lane + 32 * t;
      if (c < dv) o[t] = fmaf(wgt, vj[c], o[t]);
    }
  }
  if (p.headnorm) {
    if (p.headnorm == 2) {  // mean-subtracting form: centre the row first
      float sm = 0.f;
#pragma unroll
      for (int t = 0; t < MAX_COLS_PER_LANE; ++t) sm += o[t];
      const float mu = warp_sum(sm) / static_cast<float>(dv);
#pragma unroll
      for (int t = 0; t < MAX_COLS_PER_LANE; ++t)
        if (lane + 32 * t < dv) o[t] -= mu;
    }
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < MAX_COLS_PER_LANE; ++t) ss += o[t] * o[t];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / static_cast<float>(dv) + p.eps) * p.out_scale;
    const float *w = p.norm_w ? p.norm_w + (bh % p.H) * dv : nullptr;
#pragma unroll
    for (int t = 0; t < MAX_COLS_PER_LANE; ++t) {
      const int c = lane + 32 * t;
      if (c < dv) o[t] *= r * (w ? w[c] : 1.f);
    }
  }
  float *out = p.out + (bh * N + i) * dv;
#pragma unroll
  for (int t = 0; t < MAX_COLS_PER_LANE; ++t) {
    const int c = lane + 32 * t;
    if (c < dv) out[c] = o[t];
  }
}

}  // namespace

diffattn_status launch_fwd_f32(const diffattn_desc &desc, const float *q1, const float *k1,
                               const float *q2, const float *k2, const float *v,
                               const float *lambda, const float *norm_w, float *out,
                               cudaStream_t stream) {
  const int64_t BH = desc.B * desc.H;
  if (BH > 65535) return DIFFATTN_ERR_UNSUPPORTED;
  F32Params p;
  p.BH = BH;
  p.H = static_cast<int32_t>(desc.H);
  p.N = static_cast<int32_t>(desc.N);
  p.d = desc.d;
  p.causal = desc.causal ? 1 : 0;
  p.headnorm = desc.headnorm;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc.d)));
  p.eps = desc.eps;
  p.out_scale = 1.0f - desc.lambda_init;
  p.q1 = q1; p.k1 = k1; p.q2 = q2; p.k2 = k2; p.v = v;
  p.lambda = lambda;
  p.norm_w = norm_w;
  p.out = out;
  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(desc.N) * WARPS;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(diffattn_fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;
  dim3 grid(static_cast<unsigned>((desc.N + WARPS - 1) / WARPS), static_cast<unsigned>(BH));
  diffattn_fwd_f32_kernel<<<grid, WARPS * 32, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
