// Launchers behind the C ABI.  Each takes an already validated descriptor and
// enqueues its kernel on `stream`; none allocates memory.
#pragma once

#include <cuda_runtime.h>

#include "../../include/diffattn.h"

namespace diffattn {

// Tile of the fused bf16 kernel: 128 query rows x 128 keys, d = 64, 2d = 128.
constexpr int kTileRows = 128;
constexpr int kTileKeys = 128;
constexpr int kValueCols = 128;

// Split-KV partial block of one (work item, split), fp32: per map, O
// column-major [kValueCols][kTileRows] as accumulated against the row's
// reference maximum, then the reference maxima [kTileRows] (log2 units) and
// the running sums [kTileRows].  Only real query rows are written.
constexpr int64_t kPartOffM = int64_t{kValueCols} * kTileRows;
constexpr int64_t kPartOffL = kPartOffM + kTileRows;
constexpr int64_t kPartMapFloats = kPartOffL + kTileRows;
constexpr int64_t kPartFloats = 2 * kPartMapFloats;
constexpr int kMaxSplits = 256;

// Fused bf16 forward on tcgen05 / TMEM / TMA (d = 64) of N queries against
// n_kv keys (causal: the queries are the last N positions).  splits == 1
// writes `out`; splits > 1 writes split-KV partial blocks to `part`, to be
// merged by launch_splitkv_combine.
diffattn_status launch_fwd_bf16_sm103(const diffattn_desc &desc, int64_t n_kv, const void *q1,
                                      const void *k1, const void *q2, const void *k2,
                                      const void *v, const float *lambda, const float *norm_w,
                                      void *out, cudaStream_t stream, int splits, float *part,
                                      float *save = nullptr,
                                      const diffattn_strides *strides = nullptr);

// Saved activations of diffattn_fwd_train (fp32): the two maps' normalised
// outputs [2][B*H][N][128], then their log2-sum-exp [2][B*H][n_pad] with
// n_pad = 128 * ceil(N / 128).
inline int64_t saved_floats(int64_t BH, int64_t N) {
  const int64_t n_pad = (N + kTileRows - 1) / kTileRows * kTileRows;
  return 2 * BH * N * kValueCols + 2 * BH * n_pad;
}

// Backward pass (bwd_bf16_sm103.cu): workspace size in floats, and the launch
// of its three kernels (preprocess, fused gradients, bf16 conversion).
int64_t bwd_workspace_floats(int64_t BH, int64_t N);
diffattn_status launch_bwd_bf16_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w,
                                      const float *saved, const void *dy, void *dq1, void *dk1,
                                      void *dq2, void *dk2, void *dv, float *dlambda,
                                      float *dnorm_w, float *workspace, cudaStream_t stream,
                                      const diffattn_strides *strides = nullptr);
// Element strides the strided backward takes: q1, k1, q2, k2, v, dy, dq1, dk1,
// dq2, dk2, dv.
constexpr int kBwdStrides = 11;

// Merge of the split-KV partial blocks: both maps' softmax states, then
// o = O1/l1 - lambda O2/l2, the optional head norm and the bf16 store (out
// with the given element strides, or contiguous).  If desc.status_dev holds a
// non-zero status when the partial kernel has finished (one of its CTAs gave
// up on a wait), every output element is NaN.
diffattn_status launch_splitkv_combine(const diffattn_desc &desc, int64_t n_kv, int splits,
                                       const float *part, const float *lambda,
                                       const float *norm_w, void *out, cudaStream_t stream,
                                       const diffattn_strides *out_strides = nullptr);

// Key tiles that query tile qt (of N queries against n_kv keys) sees: all of
// them, or under the causal mask those up to the one holding the position
// n_kv - N + 128 qt + 127 of its last row.
__host__ __device__ inline int64_t key_tiles_seen(int64_t qt, int64_t N, int64_t n_kv,
                                                  bool causal) {
  const int64_t n_ktiles = (n_kv + kTileKeys - 1) / kTileKeys;
  if (!causal) return n_ktiles;
  const int64_t t = ((n_kv - N) + qt * kTileRows + kTileRows - 1) / kTileKeys + 1;
  return t < n_ktiles ? t : n_ktiles;
}

// The split count the library picks when the caller asks for 0 (splitkv.cu).
int auto_splits(int64_t BH, int64_t N, int64_t n_kv, bool causal, int sm_count);

// Fused bf16 forward for d = 128 (value width 256): two passes per query tile
// (statistics, then one normalised accumulator) of N queries against n_kv
// keys (causal: the queries are the last N positions); [B, H, rows, width]
// with the element strides of q1, k1, q2, k2, v, out given (rows contiguous),
// or contiguous when strides is null.  Training: save_lse (fp32
// [2][BH][128 * n_qtiles]) receives each map's log2-sum-exp; o_save (fp32
// [BH][N][256]) each row's o = o_1 - lambda o_2 before the norm.
diffattn_status launch_fwd_d128_sm103(const diffattn_desc &desc, int64_t n_kv, const void *q1,
                                      const void *k1, const void *q2, const void *k2,
                                      const void *v, const float *lambda, const float *norm_w,
                                      void *out, cudaStream_t stream,
                                      const diffattn_strides *strides = nullptr,
                                      float *save_lse = nullptr, float *o_save = nullptr);

// Backward pass for d = 128 (bwd_d128_sm103.cu): saved-activation and workspace
// sizes in bytes, and the launch of its kernels (preprocess, the dV items, the
// dK / dQ items, dq conversion).  The saved buffer holds each map's normalised
// output o_k (bf16 [2][B*H][N][256]) and log2-sum-exp (fp32 [2][B*H][n_pad]).
int64_t saved_bytes_d128(int64_t BH, int64_t N);
int64_t bwd_workspace_bytes_d128(int64_t BH, int64_t N);
diffattn_status launch_fwd_train_d128(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, void *out,
                                      void *saved, cudaStream_t stream,
                                      const diffattn_strides *strides);
diffattn_status launch_bwd_d128_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, const void *saved,
                                      const void *dy, void *dq1, void *dk1, void *dq2, void *dk2,
                                      void *dv, float *dlambda, float *dnorm_w, void *workspace,
                                      cudaStream_t stream, const diffattn_strides *strides);

// Bounded-wait self-test (selftest.cu).
diffattn_status launch_selftest_wait(int32_t *status, int64_t timeout_ns, cudaStream_t stream);

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
