// C ABI of libdiffattn: argument validation, dispatch and status codes.
// Every entry point is declared, with its contract, in include/diffattn.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace {

using namespace diffattn;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Fields shared by every entry point.
diffattn_status check_desc(const diffattn_desc *desc) {
  if (desc == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->B < 0 || desc->H < 0 || desc->N < 0 || desc->d <= 0) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->dtype != DIFFATTN_BF16 && desc->dtype != DIFFATTN_F32 &&
      desc->dtype != DIFFATTN_E4M3_QK)
    return DIFFATTN_ERR_INVALID_ARG;
  if (!(desc->eps >= 0.f) || !std::isfinite(desc->eps) || !std::isfinite(desc->lambda_init))
    return DIFFATTN_ERR_INVALID_ARG;
  if (desc->headnorm < 0 || desc->headnorm > 2) return DIFFATTN_ERR_INVALID_ARG;
  // B * H * N * 2d elements must be addressable with 64-bit offsets.
  const double elems = static_cast<double>(desc->B) * static_cast<double>(desc->H) *
                       static_cast<double>(desc->N) * 2.0 * static_cast<double>(desc->d);
  if (elems > 9.0e18) return DIFFATTN_ERR_INVALID_ARG;
  return DIFFATTN_OK;
}

// The bf16 kernel is built for sm_103a only.
// Per-device caches are atomics: host threads may call the library at once
// (two threads filling the same entry compute the same value).
diffattn_status check_sm103() {
  static std::atomic<int> cached[64];  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  int c = cached[dev].load(std::memory_order_acquire);
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    c = (major == 10 && minor == 3) ? 1 : 2;
    cached[dev].store(c, std::memory_order_release);
  }
  return c == 1 ? DIFFATTN_OK : DIFFATTN_ERR_UNSUPPORTED;
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_release);
  }
  return n;
}

// Strides (q1, k1, q2, k2, v, out for the forward entries; the backward's
// eleven): positive multiples of 8 elements (16 bytes, the tensor-copy rule)
// below 2^39.
diffattn_status check_strides(const diffattn_strides *strides, int count = 6) {
  for (int i = 0; i < count; ++i) {
    const int64_t s3[3] = {strides[i].b, strides[i].h, strides[i].n};
    for (int64_t x : s3)
      if (x <= 0 || (x & 7) != 0 || x >= (int64_t{1} << 39)) return DIFFATTN_ERR_INVALID_ARG;
  }
  return DIFFATTN_OK;
}

// Validation shared by diffattn_fwd_kv_plan and diffattn_fwd_kv; on success
// *splits_out is the split count that will run and *bytes the workspace it needs.
diffattn_status plan_kv(const diffattn_desc *desc, int64_t n_kv, int splits, int *splits_out,
                        size_t *bytes) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (n_kv < 0 || splits < 0 || splits > kMaxSplits) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->causal && n_kv < desc->N) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->dtype != DIFFATTN_BF16 && desc->dtype != DIFFATTN_E4M3_QK)
    return DIFFATTN_ERR_UNSUPPORTED;
  if (desc->d != 64 && !(desc->d == 128 && desc->dtype == DIFFATTN_BF16))
    return DIFFATTN_ERR_UNSUPPORTED;
  // d = 128 runs its two-pass kernel over the whole key range (no split-KV).
  if (desc->d == 128 && splits > 1) return DIFFATTN_ERR_UNSUPPORTED;
  if (desc->dtype == DIFFATTN_E4M3_QK && desc->headnorm == 2) return DIFFATTN_ERR_UNSUPPORTED;
  const int64_t BH = desc->B * desc->H;
  if (BH * desc->N == 0) {
    *splits_out = 1;
    *bytes = 0;
    return DIFFATTN_OK;
  }
  if (n_kv == 0) return DIFFATTN_ERR_INVALID_ARG;  // a softmax over no keys
  const int64_t n_qtiles = (desc->N + kTileRows - 1) / kTileRows;
  const int64_t n_ktiles = (n_kv + kTileKeys - 1) / kTileKeys;
  if (splits == 0 && desc->d == 128) splits = 1;
  if (splits == 0) {
    const int sms = sm_count();
    if (sms <= 0) return DIFFATTN_ERR_CUDA;
    splits = auto_splits(BH, desc->N, n_kv, desc->causal != 0, sms);
  }
  if (splits > n_ktiles) splits = static_cast<int>(n_ktiles);
  const double elems = static_cast<double>(BH) * static_cast<double>(n_qtiles) * splits *
                       static_cast<double>(kPartFloats);
  if (elems * 4.0 > 9.0e18) return DIFFATTN_ERR_UNSUPPORTED;
  *splits_out = splits;
  *bytes = splits > 1 ? static_cast<size_t>(BH * n_qtiles * splits * kPartFloats) * sizeof(float)
                      : 0;
  return DIFFATTN_OK;
}

}  // namespace

extern "C" {

namespace {
// The shapes and dtypes diffattn_fwd runs (desc already checked).
diffattn_status fwd_domain(const diffattn_desc &d) {
  if (d.dtype == DIFFATTN_BF16 || d.dtype == DIFFATTN_E4M3_QK) {
    if (d.d != 64 && d.d != 128) return DIFFATTN_ERR_UNSUPPORTED;
    if (d.dtype == DIFFATTN_E4M3_QK && (d.d != 64 || d.headnorm == 2))
      return DIFFATTN_ERR_UNSUPPORTED;
    return check_sm103();
  }
  if (d.d > kF32MaxD || d.N > kF32MaxN) return DIFFATTN_ERR_UNSUPPORTED;
  return DIFFATTN_OK;
}
}  // namespace

diffattn_status diffattn_fwd(const diffattn_desc *desc, const void *q1, const void *k1,
                             const void *q2, const void *k2, const void *v, const float *lambda,
                             const float *norm_w, void *out, void *stream) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out) return DIFFATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->dtype == DIFFATTN_BF16 || desc->dtype == DIFFATTN_E4M3_QK) {
    if (desc->d != 64 && desc->d != 128) return DIFFATTN_ERR_UNSUPPORTED;
    if (desc->dtype == DIFFATTN_E4M3_QK && (desc->d != 64 || desc->headnorm == 2))
      return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
        !aligned16(out))
      return DIFFATTN_ERR_INVALID_ARG;
    if ((st = check_sm103()) != DIFFATTN_OK) return st;
    if (desc->d == 128)
      return launch_fwd_d128_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out, s);
    return launch_fwd_bf16_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out, s, 1,
                                 nullptr);
  }
  if (desc->d > kF32MaxD || desc->N > kF32MaxN) return DIFFATTN_ERR_UNSUPPORTED;
  return launch_fwd_f32(*desc, static_cast<const float *>(q1), static_cast<const float *>(k1),
                        static_cast<const float *>(q2), static_cast<const float *>(k2),
                        static_cast<const float *>(v), lambda, norm_w, static_cast<float *>(out),
                        s);
}

namespace {
// Byte sizes of a forward's tensors: each q/k half, v and out.
struct FwdBytes {
  size_t qk, v, out;
};
FwdBytes fwd_bytes(const diffattn_desc &d) {
  const size_t n = static_cast<size_t>(d.B) * static_cast<size_t>(d.H) * static_cast<size_t>(d.N);
  const size_t wide = n * 2 * static_cast<size_t>(d.d);
  const size_t qk_elem = d.dtype == DIFFATTN_F32 ? 4 : d.dtype == DIFFATTN_E4M3_QK ? 1 : 2;
  const size_t vo_elem = d.dtype == DIFFATTN_F32 ? 4 : 2;
  return {n * static_cast<size_t>(d.d) * qk_elem, wide * vo_elem, wide * vo_elem};
}
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

diffattn_status diffattn_fwd_host_staging_bytes(const diffattn_desc *desc, size_t *bytes) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (bytes == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  const FwdBytes b = fwd_bytes(*desc);
  *bytes = 4 * round256(b.qk) + round256(b.v) + round256(b.out);
  return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_host(const diffattn_desc *desc, const void *q1, const void *k1,
                                  const void *q2, const void *k2, const void *v,
                                  const float *lambda, const float *norm_w, void *out_host,
                                  void *staging, size_t staging_bytes, void *stream) {
  size_t need = 0;
  diffattn_status st = diffattn_fwd_host_staging_bytes(desc, &need);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out_host) return DIFFATTN_ERR_INVALID_ARG;
  if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) & 255u) != 0 ||
      staging_bytes < need)
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = fwd_domain(*desc)) != DIFFATTN_OK) return st;  // before any copy is queued
  const FwdBytes b = fwd_bytes(*desc);
  uint8_t *base = static_cast<uint8_t *>(staging);
  uint8_t *dev[6];
  const size_t sizes[6] = {b.qk, b.qk, b.qk, b.qk, b.v, b.out};
  for (int i = 0; i < 6; ++i) {
    dev[i] = base;
    base += round256(sizes[i]);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *src[5] = {q1, k1, q2, k2, v};
  for (int i = 0; i < 5; ++i)
    if (cudaMemcpyAsync(dev[i], src[i], sizes[i], cudaMemcpyHostToDevice, s) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
  st = diffattn_fwd(desc, dev[0], dev[1], dev[2], dev[3], dev[4], lambda, norm_w, dev[5], stream);
  if (st != DIFFATTN_OK) return st;
  if (cudaMemcpyAsync(out_host, dev[5], b.out, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;
  return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_strided(const diffattn_desc *desc, const void *q1, const void *k1,
                                     const void *q2, const void *k2, const void *v,
                                     const float *lambda, const float *norm_w, void *out,
                                     const diffattn_strides *strides, void *stream) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (desc->dtype != DIFFATTN_BF16 || (desc->d != 64 && desc->d != 128))
    return DIFFATTN_ERR_UNSUPPORTED;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out || !strides)
    return DIFFATTN_ERR_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(out))
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = check_strides(strides)) != DIFFATTN_OK) return st;
  if (desc->B > INT32_MAX || desc->H > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  if (desc->d == 128)
    return launch_fwd_d128_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out,
                                 static_cast<cudaStream_t>(stream), strides);
  return launch_fwd_bf16_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out,
                               static_cast<cudaStream_t>(stream), 1, nullptr, nullptr, strides);
}

diffattn_status diffattn_fwd_kv_plan(const diffattn_desc *desc, int64_t n_kv, int splits,
                                     int *splits_out, size_t *workspace_bytes) {
  if (splits_out == nullptr || workspace_bytes == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  int sp = 1;
  size_t bytes = 0;
  const diffattn_status st = plan_kv(desc, n_kv, splits, &sp, &bytes);
  if (st != DIFFATTN_OK) return st;
  *splits_out = sp;
  *workspace_bytes = bytes;
  return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_kv(const diffattn_desc *desc, int64_t n_kv, const void *q1,
                                const void *k1, const void *q2, const void *k2, const void *v,
                                const float *lambda, const float *norm_w, void *out, int splits,
                                void *workspace, size_t workspace_bytes, void *stream) {
  int sp = 1;
  size_t need = 0;
  diffattn_status st = plan_kv(desc, n_kv, splits, &sp, &need);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out) return DIFFATTN_ERR_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(out))
    return DIFFATTN_ERR_INVALID_ARG;
  if (sp > 1 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need))
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->d == 128)
    return launch_fwd_d128_sm103(*desc, n_kv, q1, k1, q2, k2, v, lambda, norm_w, out, s);
  float *part = sp > 1 ? static_cast<float *>(workspace) : nullptr;
  st = launch_fwd_bf16_sm103(*desc, n_kv, q1, k1, q2, k2, v, lambda, norm_w, out, s, sp, part);
  if (st != DIFFATTN_OK || sp == 1) return st;
  return launch_splitkv_combine(*desc, n_kv, sp, part, lambda, norm_w, out, s);
}

diffattn_status diffattn_fwd_kv_strided(const diffattn_desc *desc, int64_t n_kv, const void *q1,
                                        const void *k1, const void *q2, const void *k2,
                                        const void *v, const float *lambda,
                                        const float *norm_w, void *out, int splits,
                                        void *workspace, size_t workspace_bytes,
                                        const diffattn_strides *strides, void *stream) {
  int sp = 1;
  size_t need = 0;
  diffattn_status st = plan_kv(desc, n_kv, splits, &sp, &need);
  if (st != DIFFATTN_OK) return st;
  if (desc->dtype != DIFFATTN_BF16) return DIFFATTN_ERR_UNSUPPORTED;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out || !strides)
    return DIFFATTN_ERR_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(out))
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = check_strides(strides)) != DIFFATTN_OK) return st;
  if (sp > 1 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need))
    return DIFFATTN_ERR_INVALID_ARG;
  if (desc->B > INT32_MAX || desc->H > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->d == 128)
    return launch_fwd_d128_sm103(*desc, n_kv, q1, k1, q2, k2, v, lambda, norm_w, out, s, strides);
  float *part = sp > 1 ? static_cast<float *>(workspace) : nullptr;
  st = launch_fwd_bf16_sm103(*desc, n_kv, q1, k1, q2, k2, v, lambda, norm_w, out, s, sp, part,
                             nullptr, strides);
  if (st != DIFFATTN_OK || sp == 1) return st;
  return launch_splitkv_combine(*desc, n_kv, sp, part, lambda, norm_w, out, s, &strides[5]);
}

diffattn_status diffattn_train_sizes(const diffattn_desc *desc, size_t *saved_bytes,
                                     size_t *workspace_bytes) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (saved_bytes == nullptr || workspace_bytes == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->dtype != DIFFATTN_BF16 || (desc->d != 64 && desc->d != 128))
    return DIFFATTN_ERR_UNSUPPORTED;
  const int64_t BH = desc->B * desc->H;
  if (desc->d == 128) {
    *saved_bytes = static_cast<size_t>(saved_bytes_d128(BH, desc->N));
    *workspace_bytes = static_cast<size_t>(bwd_workspace_bytes_d128(BH, desc->N));
    return DIFFATTN_OK;
  }
  *saved_bytes = static_cast<size_t>(saved_floats(BH, desc->N)) * sizeof(float);
  *workspace_bytes = static_cast<size_t>(bwd_workspace_floats(BH, desc->N)) * sizeof(float);
  return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_train(const diffattn_desc *desc, const void *q1, const void *k1,
                                   const void *q2, const void *k2, const void *v,
                                   const float *lambda, const float *norm_w, void *out,
                                   void *saved, size_t saved_bytes, void *stream) {
  size_t need = 0, ws = 0;
  diffattn_status st = diffattn_train_sizes(desc, &need, &ws);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out || !saved) return DIFFATTN_ERR_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(out) || !aligned16(saved) || saved_bytes < need)
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  if (desc->d == 128)
    return launch_fwd_train_d128(*desc, q1, k1, q2, k2, v, lambda, norm_w, out, saved,
                                 static_cast<cudaStream_t>(stream), nullptr);
  return launch_fwd_bf16_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out,
                               static_cast<cudaStream_t>(stream), 1, nullptr,
                               static_cast<float *>(saved));
}

namespace {

// diffattn_bwd and diffattn_bwd_strided (strides == nullptr: contiguous).
diffattn_status bwd_common(const diffattn_desc *desc, const void *q1, const void *k1,
                           const void *q2, const void *k2, const void *v, const float *lambda,
                           const float *norm_w, const void *saved, const void *dy, void *dq1,
                           void *dk1, void *dq2, void *dk2, void *dv, float *dlambda,
                           float *dnorm_w, void *workspace, size_t workspace_bytes,
                           const diffattn_strides *strides, void *stream) {
  size_t saved_need = 0, ws_need = 0;
  diffattn_status st = diffattn_train_sizes(desc, &saved_need, &ws_need);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  const void *ptrs[] = {q1, k1, q2, k2, v, saved, dy, dq1, dk1, dq2, dk2, dv, workspace};
  for (const void *q : ptrs)
    if (q == nullptr || !aligned16(q)) return DIFFATTN_ERR_INVALID_ARG;
  if (!lambda || !dlambda || workspace_bytes < ws_need) return DIFFATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DIFFATTN_ERR_INVALID_ARG;
  if (strides != nullptr && (st = check_strides(strides, kBwdStrides)) != DIFFATTN_OK) return st;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  if (desc->d == 128)
    return launch_bwd_d128_sm103(*desc, q1, k1, q2, k2, v, lambda, norm_w, saved, dy, dq1, dk1,
                                 dq2, dk2, dv, dlambda, dnorm_w, workspace,
                                 static_cast<cudaStream_t>(stream), strides);
  return launch_bwd_bf16_sm103(*desc, q1, k1, q2, k2, v, lambda, norm_w,
                               static_cast<const float *>(saved), dy, dq1, dk1, dq2, dk2, dv,
                               dlambda, dnorm_w, static_cast<float *>(workspace),
                               static_cast<cudaStream_t>(stream), strides);
}

}  // namespace

diffattn_status diffattn_bwd(const diffattn_desc *desc, const void *q1, const void *k1,
                             const void *q2, const void *k2, const void *v, const float *lambda,
                             const float *norm_w, const void *saved, const void *dy, void *dq1,
                             void *dk1, void *dq2, void *dk2, void *dv, float *dlambda,
                             float *dnorm_w, void *workspace, size_t workspace_bytes,
                             void *stream) {
  return bwd_common(desc, q1, k1, q2, k2, v, lambda, norm_w, saved, dy, dq1, dk1, dq2, dk2, dv,
                    dlambda, dnorm_w, workspace, workspace_bytes, nullptr, stream);
}

diffattn_status diffattn_bwd_strided(const diffattn_desc *desc, const void *q1, const void *k1,
                                     const void *q2, const void *k2, const void *v,
                                     const float *lambda, const float *norm_w,
                                     const void *saved, const void *dy, void *dq1, void *dk1,
                                     void *dq2, void *dk2, void *dv, float *dlambda,
                                     float *dnorm_w, void *workspace, size_t workspace_bytes,
                                     const diffattn_strides *strides, void *stream) {
  if (strides == nullptr) {
    const diffattn_status st = check_desc(desc);
    return st != DIFFATTN_OK ? st : DIFFATTN_ERR_INVALID_ARG;
  }
  return bwd_common(desc, q1, k1, q2, k2, v, lambda, norm_w, saved, dy, dq1, dk1, dq2, dk2, dv,
                    dlambda, dnorm_w, workspace, workspace_bytes, strides, stream);
}

diffattn_status diffattn_fwd_train_strided(const diffattn_desc *desc, const void *q1,
                                           const void *k1, const void *q2, const void *k2,
                                           const void *v, const float *lambda,
                                           const float *norm_w, void *out, void *saved,
                                           size_t saved_bytes, const diffattn_strides *strides,
                                           void *stream) {
  size_t need = 0, ws = 0;
  diffattn_status st = diffattn_train_sizes(desc, &need, &ws);
  if (st != DIFFATTN_OK) return st;
  if (strides == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!q1 || !k1 || !q2 || !k2 || !v || !lambda || !out || !saved) return DIFFATTN_ERR_INVALID_ARG;
  if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
      !aligned16(out) || !aligned16(saved) || saved_bytes < need)
    return DIFFATTN_ERR_INVALID_ARG;
  if ((st = check_strides(strides)) != DIFFATTN_OK) return st;
  if (desc->B > INT32_MAX || desc->H > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
  if ((st = check_sm103()) != DIFFATTN_OK) return st;
  if (desc->d == 128)
    return launch_fwd_train_d128(*desc, q1, k1, q2, k2, v, lambda, norm_w, out, saved,
                                 static_cast<cudaStream_t>(stream), strides);
  return launch_fwd_bf16_sm103(*desc, desc->N, q1, k1, q2, k2, v, lambda, norm_w, out,
                               static_cast<cudaStream_t>(stream), 1, nullptr,
                               static_cast<float *>(saved), strides);
}

diffattn_status diffattn_headnorm(const diffattn_desc *desc, const float *x, const float *norm_w,
                                  void *out, void *stream) {
  diffattn_status st = check_desc(desc);
  if (st != DIFFATTN_OK) return st;
  if (desc->B * desc->H * desc->N == 0) return DIFFATTN_OK;
  if (!x || !out) return DIFFATTN_ERR_INVALID_ARG;
  if (desc->d > kF32MaxD) return DIFFATTN_ERR_UNSUPPORTED;
  return launch_headnorm(*desc, x, norm_w, out, static_cast<cudaStream_t>(stream));
}

diffattn_status diffattn_selftest_wait(int32_t *status_dev, int64_t timeout_ns, void *stream) {
  if (status_dev == nullptr || timeout_ns <= 0 || timeout_ns > 2000000000) return DIFFATTN_ERR_INVALID_ARG;
  diffattn_status st = check_sm103();
  if (st != DIFFATTN_OK) return st;
  return launch_selftest_wait(status_dev, timeout_ns, static_cast<cudaStream_t>(stream));
}

double diffattn_lambda_init(int layer) {
  return 0.8 - 0.6 * std::exp(-0.3 * (static_cast<double>(layer) - 1.0));
}

const char *diffattn_strerror(diffattn_status status) {
  switch (status) {
    case DIFFATTN_OK: return "ok";
    case DIFFATTN_ERR_INVALID_ARG: return "invalid argument";
    case DIFFATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case DIFFATTN_ERR_CUDA: return "CUDA error";
    case DIFFATTN_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case DIFFATTN_ERR_BOUNDS: return "kernel bounds check failed (debug build)";
  }
  return "unknown status";
}

int diffattn_version(void) { return 100; }

}  // extern "C"
