// Split-KV support for the fused bf16 forward: the merge of partial softmax
// states and the choice of the split count.
//
// Each map of the differential head ("Differential Transformer", section "How
// differential attention works") is ordinary softmax attention, so a row's
// keys can be cut into ranges processed independently.  Range s leaves, per
// map, an unnormalised accumulator O_s = sum_j 2^(x_j - m_s) v_j, its
// reference maximum m_s (log2 units) and sum l_s = sum_j 2^(x_j - m_s).  With
// M = max_s m_s and a_s = 2^(m_s - M):
//
//   softmax(x) V = (sum_s a_s O_s) / (sum_s a_s l_s)
//
// exactly (up to rounding).  The combine kernel forms that for both maps, then
// o = O1/l1 - lambda_h O2/l2, the optional RMS head norm, w[h] and
// (1 - lambda_init), and stores bf16, as the single-pass kernel's epilogue does.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <vector>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace diffattn {

// Split count for a launch of BH heads x ceil(N/128) query tiles against
// ceil(n_kv/128) key tiles on sm_count SMs, from a small model measured on
// GB300 (times in units of one 128-key tile step, about 1.3 us):
//   - a CTA costs kCtaCost (start-up, first loads, drain, epilogue, exit:
//     about 5 us) plus one unit per key tile;
//   - a key tile streams 64 KB, and HBM feeds about kStreamingCtas CTAs at
//     that rate, so with more CTAs resident each unit stretches in proportion;
//   - CTAs are taken in launch order by whichever SM frees first (heaviest
//     query tiles first, as the kernel numbers them);
//   - more than one split adds the combine kernel, kCombineCost.
// The smallest split count of least modelled time wins.  Split counts whose
// CTAs would exceed four waves are not considered.
int auto_splits(int64_t BH, int64_t N, int64_t n_kv, bool causal, int sm_count) {
  constexpr double kCtaCost = 4.0;
  constexpr double kCombineCost = 4.0;
  constexpr double kStreamingCtas = 129.0;
  const int64_t n_qtiles = (N + kTileRows - 1) / kTileRows;
  const int64_t n_ktiles = (n_kv + kTileKeys - 1) / kTileKeys;
  if (BH <= 0 || n_qtiles <= 0 || n_ktiles <= 1 || sm_count <= 0) return 1;
  const int64_t items = BH * n_qtiles;
  if (items >= sm_count) return 1;
  const int64_t max_splits = std::min<int64_t>({n_ktiles, kMaxSplits, 4 * sm_count / items});
  int best = 1;
  double best_cost = 0.0;
  std::vector<double> free_at;
  for (int64_t s = 1; s <= max_splits; ++s) {
    const int64_t st = (n_ktiles + s - 1) / s;
    if (s > 1 && (n_ktiles + st - 1) / st < s) continue;  // same ranges as a smaller s
    int64_t ctas = 0;
    for (int64_t qt = 0; qt < n_qtiles; ++qt)
      ctas += BH * ((key_tiles_seen(qt, N, n_kv, causal) + st - 1) / st);
    const double resident = static_cast<double>(std::min<int64_t>(ctas, sm_count));
    const double unit = std::max(1.0, resident / kStreamingCtas);
    // Min-heap of SM free times; CTAs in launch order (query tile from the
    // last, all heads, then the key ranges of each).
    free_at.assign(static_cast<size_t>(sm_count), 0.0);
    double makespan = 0.0;
    for (int64_t qt = n_qtiles - 1; qt >= 0; --qt) {
      const int64_t seen = key_tiles_seen(qt, N, n_kv, causal);
      for (int64_t b = 0; b < BH; ++b)
        for (int64_t lo = 0; lo < seen; lo += st) {
          const int64_t tiles = std::min(st, seen - lo);
          std::pop_heap(free_at.begin(), free_at.end(), std::greater<double>());
          const double end = free_at.back() + kCtaCost + unit * static_cast<double>(tiles);
          free_at.back() = end;
          std::push_heap(free_at.begin(), free_at.end(), std::greater<double>());
          makespan = std::max(makespan, end);
        }
    }
    const double cost = makespan + (s > 1 ? kCombineCost : 0.0);
    if (s == 1 || cost < best_cost) {
      best = static_cast<int>(s);
      best_cost = cost;
    }
  }
  return best;
}

namespace {

constexpr int kRowsPerBlock = 32;
constexpr int kColsPerThread = 8;
constexpr int kCombineWarps = kValueCols / kColsPerThread;  // 16
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kBlocksPerItem = kTileRows / kRowsPerBlock;
constexpr int kSplitBatch = 4;  // splits whose loads are in flight together

struct CombineParams {
  int64_t BH;
  int32_t H, N, n_qtiles, split_tiles, splits, headnorm;
  int64_t n_kv;
  int32_t causal;
  float eps, out_scale;
  const float *part;
  const float *lambda;
  const float *norm_w;
  __nv_bfloat16 *out;
  int64_t out_sb, out_sh, out_sn;  // element strides of out (batch, head, row)
  const int32_t *status;           // the call's status word, or null
};

// Running merge of one map's split states: (M, L, acc) absorbs (m, l, o).
// Factors are 1 when the maxima agree, so a row that saw no key in a range
// (m = -inf, l = 0, o = 0) merges as zeros instead of -inf - -inf.
__device__ __forceinline__ void merge_state(float &M, float &L, float (&acc)[kColsPerThread],
                                            float m, float l, const float (&o)[kColsPerThread]) {
  const float Mn = fmaxf(M, m);
  const float a_old = (M == Mn) ? 1.f : exp2f(M - Mn);
  const float a_new = (m == Mn) ? 1.f : exp2f(m - Mn);
  L = fmaf(L, a_old, l * a_new);
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) acc[c] = fmaf(acc[c], a_old, o[c] * a_new);
  M = Mn;
}

// Block (item, g): query rows 32g .. 32g+31 of the item's tile, lane = row;
// warp w: value columns 8w .. 8w+7.  A load of a partial block is a warp
// reading 32 consecutive rows of one column; the loads of kSplitBatch splits
// are issued before any of them is used.
__global__ void __launch_bounds__(kCombineThreads)
    diffattn_splitkv_combine_kernel(const CombineParams p) {
  __shared__ float ss_warp[kCombineWarps][32];
  const int64_t item = blockIdx.x / kBlocksPerItem;
  const int g = static_cast<int>(blockIdx.x % kBlocksPerItem);
  const int qt = p.n_qtiles - 1 - static_cast<int>(item / p.BH);  // same order as the partials
  const int64_t q_first = static_cast<int64_t>(qt) * kTileRows + g * kRowsPerBlock;
  if (q_first >= p.N) return;  // every row of this block is padding (uniform per block)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t bh = item % p.BH;
  const int h = static_cast<int>(bh % p.H);
  const int r = g * kRowsPerBlock + lane;
  const int64_t q = q_first + lane;
  const bool real = q < p.N;
  const int64_t seen = key_tiles_seen(qt, p.N, p.n_kv, p.causal != 0);
  const int used = static_cast<int>((seen + p.split_tiles - 1) / p.split_tiles);
  const float *blk0 = p.part + item * p.splits * kPartFloats;
  const int col0 = warp * kColsPerThread;
  // Inputs that do not come from the partial kernel are read before waiting
  // for it (this kernel may start while that one is still draining).
  const float lam = p.lambda[h];
  float wv[kColsPerThread];
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c)
    wv[c] = p.norm_w ? __ldg(p.norm_w + static_cast<int64_t>(h) * kValueCols + col0 + c) : 1.f;
  grid_dependency_wait();
  // A partial CTA that gave up on a wait has not written its block: rather
  // than merge stale scratch into a plausible-looking output, write NaN.
  const bool failed = p.status != nullptr && *reinterpret_cast<const volatile int32_t *>(p.status) != 0;

  float M1 = -INFINITY, L1 = 0.f, M2 = -INFINITY, L2 = 0.f;
  float acc1[kColsPerThread], acc2[kColsPerThread];
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) acc1[c] = acc2[c] = 0.f;
  if (real) {
    for (int s0 = 0; s0 < used; s0 += kSplitBatch) {
      float m[kSplitBatch][2], l[kSplitBatch][2], o[kSplitBatch][2][kColsPerThread];
#pragma unroll
      for (int u = 0; u < kSplitBatch; ++u) {
        const bool have = s0 + u < used;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float *b = blk0 + (s0 + u) * kPartFloats + k * kPartMapFloats;
          m[u][k] = have ? b[kPartOffM + r] : -INFINITY;
          l[u][k] = have ? b[kPartOffL + r] : 0.f;
#pragma unroll
          for (int c = 0; c < kColsPerThread; ++c)
            o[u][k][c] = have ? b[static_cast<int64_t>(col0 + c) * kTileRows + r] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kSplitBatch; ++u) {
        merge_state(M1, L1, acc1, m[u][0], l[u][0], o[u][0]);
        merge_state(M2, L2, acc2, m[u][1], l[u][1], o[u][1]);
      }
    }
  }
  const float c1 = real ? 1.f / L1 : 0.f;
  const float c2 = real ? -lam / L2 : 0.f;
  float ov[kColsPerThread];
  float ss = 0.f, sm = 0.f;
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) {
    ov[c] = fmaf(acc1[c], c1, acc2[c] * c2);
    sm += ov[c];
  }
  if (p.headnorm == 2) {  // mean-subtracting (group) form: centre the row first
    ss_warp[warp][lane] = sm;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) tot += ss_warp[w][lane];
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kColsPerThread; ++c) ov[c] -= tot * (1.f / kValueCols);
  }
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) ss = fmaf(ov[c], ov[c], ss);
  if (p.headnorm) {
    ss_warp[warp][lane] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) tot += ss_warp[w][lane];
    const float rr = rsqrtf(tot * (1.f / kValueCols) + p.eps) * p.out_scale;
#pragma unroll
    for (int c = 0; c < kColsPerThread; ++c) ov[c] *= rr * wv[c];
  }
  if (real && dbg_ok(q >= 0 && col0 + kColsPerThread <= kValueCols &&
                         item < p.BH * p.n_qtiles && used <= p.splits,
                     const_cast<int32_t *>(p.status), 30)) {
    __nv_bfloat162 x[kColsPerThread / 2];
#pragma unroll
    for (int c = 0; c < kColsPerThread / 2; ++c)
      x[c] = failed ? __floats2bfloat162_rn(NAN, NAN)
                    : __floats2bfloat162_rn(ov[2 * c], ov[2 * c + 1]);
    const int64_t b = bh / p.H;
    *reinterpret_cast<uint4 *>(p.out + b * p.out_sb + h * p.out_sh + q * p.out_sn + col0) =
        *reinterpret_cast<const uint4 *>(x);
  }
}

}  // namespace

diffattn_status launch_splitkv_combine(const diffattn_desc &desc, int64_t n_kv, int splits,
                                       const float *part, const float *lambda,
                                       const float *norm_w, void *out, cudaStream_t stream,
                                       const diffattn_strides *out_strides) {
  const int64_t BH = desc.B * desc.H;
  const int64_t n_qtiles = (desc.N + kTileRows - 1) / kTileRows;
  const int64_t n_ktiles = (n_kv + kTileKeys - 1) / kTileKeys;
  const int64_t blocks = BH * n_qtiles * kBlocksPerItem;
  if (splits < 2 || part == nullptr) return DIFFATTN_ERR_INVALID_ARG;
  if (blocks > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
  CombineParams p;
  p.BH = BH;
  p.H = static_cast<int32_t>(desc.H);
  p.N = static_cast<int32_t>(desc.N);
  p.n_qtiles = static_cast<int32_t>(n_qtiles);
  p.split_tiles = static_cast<int32_t>((n_ktiles + splits - 1) / splits);
  p.splits = splits;
  p.headnorm = desc.headnorm;
  p.n_kv = n_kv;
  p.causal = desc.causal ? 1 : 0;
  p.eps = desc.eps;
  p.out_scale = 1.0f - desc.lambda_init;
  p.part = part;
  p.lambda = lambda;
  p.norm_w = norm_w;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.out_sn = out_strides ? out_strides->n : kValueCols;
  p.out_sh = out_strides ? out_strides->h : desc.N * kValueCols;
  p.out_sb = out_strides ? out_strides->b : desc.H * desc.N * kValueCols;
  p.status = desc.status_dev;
  // Programmatic dependent launch: the kernel may be scheduled while the
  // partial kernel drains; it waits for that grid before reading `part`.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, diffattn_splitkv_combine_kernel, p) == cudaSuccess
             ? DIFFATTN_OK
             : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
