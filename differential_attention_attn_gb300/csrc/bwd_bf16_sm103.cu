// Backward pass of the differential-attention head on sm_103a.
//
// What it computes: the gradient of the head forward ("Differential
// Transformer", Ultralytics glossary, section "How differential attention
// works": map_k = softmax(Q_k K_k^T / sqrt(d)), o = (map1 - lambda map2) V,
// per-head RMS normalisation, times (1 - lambda_init)).  The pages give the
// forward only; the gradient is its derivative by the chain rule:
//
//   norm:    do = r g dy - (r^3 / 2d) o sum_c(dy g o),   r = rsqrt(mean o^2 + eps),
//            g = w (1 - lambda_init);  dw += dy o r (1 - lambda_init)
//   lambda:  dlambda = -sum_rows do . o2,  o_k = map_k V (normalised map outputs)
//   values:  dV = map1^T do - lambda map2^T do
//   maps:    dW = do V^T,  dS_k = c_k P_k * (dW - D_k),  D_k = do . o_k,
//            c_1 = 1, c_2 = -lambda
//   logits:  dQ_k = dS_k K_k / sqrt(d),  dK_k = dS_k^T Q_k / sqrt(d)
//
// Kernels:
//   1. diffattn_bwd_pre_kernel: one warp per row: do (bf16, for the tensor
//      cores), D_1 and D_2 from the bf16-rounded do, and per-head sums of
//      dlambda and dw (block reduction, one atomic per head and column).
//   2. diffattn_bwd_bf16_sm103_kernel: persistent, one CTA per SM walking
//      work items (128-key tile, head, map), heaviest first.  P is recomputed
//      from the forward's saved log2-sum-exp, with keys on the TMEM lanes
//      (S^T = K Q^T), so dV and dK accumulate in tensor memory over the query
//      tiles of an item; dQ of each query tile goes to an fp32 accumulator with
//      vector reductions.  TMEM (512 columns): S^T / P^T 0-127, dW^T 128-255,
//      dV 256-383, dK 384-447, dQ 448-511.  Inputs are read through 4-D tensor
//      maps ([B, H, N, width] views with any strides); a second instantiation
//      also writes dk through strides.
//   3. diffattn_bwd_finish_kernel: fp32 accumulators -> bf16 gradients (dq1,
//      dq2, dv; contiguous, or through strides in a second instantiation).
//
// Roles in kernel 2 (512 threads): warp 0 TMA producer; warp 1 TMEM
// allocator and MMA issuer (the converged warp, one elected lane issuing);
// warps 4-15 three warpgroups (thread = key row) sharing the P^T / dS^T work
// of each tile by 16-query chunks in three published steps, the one with
// fewer chunks also draining dQ (thread = query row).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include <cmath>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr int BK = 128;  // keys per CTA (TMEM lanes of S^T, dV, dK)
constexpr int BQ = 128;  // queries per tile
constexpr int HD = 64;
constexpr int DV = 128;
constexpr int NUM_THREADS = 512;

constexpr uint32_t TILE64 = 128 * HD * 2;            // one [128 x 64] bf16 box: 16 KB
constexpr uint32_t OFF_K = 0;                         // K_k [128 keys x 64]
constexpr uint32_t OFF_V = OFF_K + TILE64;            // V [128 keys x 128]: two boxes
constexpr uint32_t OFF_Q = OFF_V + 2 * TILE64;        // 2 stages of Q_k [128 x 64]
constexpr uint32_t OFF_DO = OFF_Q + 2 * TILE64;       // 2 stages of dO [128 x 128]
constexpr uint32_t OFF_DS = OFF_DO + 4 * TILE64;      // 2 buffers of dS^T [128 keys x 128 queries]
constexpr uint32_t DS_BYTES = 2 * TILE64;
constexpr uint32_t OFF_VEC = OFF_DS + 2 * DS_BYTES;   // 2 stages of (lse[128], D[128])
constexpr uint32_t VEC_BYTES = 2 * BQ * 4;
constexpr uint32_t OFF_CTRL = OFF_VEC + 2 * VEC_BYTES;

struct Ctrl {
  uint64_t kv_full;
  uint64_t kv_empty;
  uint64_t qd_full[2];
  uint64_t qd_empty[2];
  uint64_t s_full;
  uint64_t ds_ready[3];  // the three chunk steps of a tile
  uint64_t ds_free[2];
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t acc_done;
  uint64_t acc_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr uint32_t SMEM_BYTES = OFF_CTRL + sizeof(Ctrl) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(SMEM_BYTES + 1024 < (1u << 18), "descriptor start addresses must stay below 256 KB");

constexpr uint32_t TM_S = 0, TM_W = 128, TM_DV = 256, TM_DK = 384, TM_DQ = 448;
// Packed (2 bf16 per column) P^T and dS^T of 16-query chunk c.  P^T goes
// over the first half of the chunk's S^T columns; dS^T over the first half of
// its dW^T columns for chunks 0-5, and over the second half of its S^T columns
// for chunks 6 and 7, so that dW^T of the next tile can be written while
// chunks 6 and 7 are computed.  Either way a thread overwrites only columns of
// its own lane that it has already read.
__host__ __device__ constexpr uint32_t tm_p(int c) { return TM_S + 16 * c; }
__host__ __device__ constexpr uint32_t tm_ds(int c) {
  return c < 6 ? TM_W + 16 * c : TM_S + 16 * c + 8;
}
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr uint64_t DRAIN_TIMEOUT_NS = 200000000ull;

struct BwdParams {
  int64_t BH;
  int32_t H, N, n_qtiles, n_ktiles, causal;
  int64_t n_items;  // 2 * BH * n_ktiles
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  const float *lambda;
  const float *lse;   // [2][BH][n_pad] log2-sum-exp from the forward
  const float *dvec;  // [2][BH][n_pad] c_k D_k
  __nv_bfloat16 *dk1, *dk2;  // [B, H, N, 64] views
  int64_t dk_sb[2], dk_sh[2], dk_sn[2];  // their element strides (batch, head, row)
  float *dq_acc;             // [2][BH][N][64], zeroed
  float *dv_acc;             // [BH][N][128], zeroed
  int32_t *status;
};

// ---------------------------------------------------------------- PTX helpers
// Instruction descriptor, kind::f16, bf16 A and B, fp32 D; a_mn / b_mn select
// MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_ab(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Plain (non-tensor) bulk copy global -> shared, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > DRAIN_TIMEOUT_NS) return false;
  }
  return true;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled
// tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// TMEM loads of 16 columns without waiting, and a wait that passes the
// registers through (so no use is scheduled before it).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait16x4(uint32_t (&a)[16], uint32_t (&b)[16],
                                              uint32_t (&c)[16], uint32_t (&d)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]),
                 "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                 "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
  asm volatile("" : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]), "+r"(c[5]),
                    "+r"(c[6]), "+r"(c[7]), "+r"(c[8]), "+r"(c[9]), "+r"(c[10]), "+r"(c[11]),
                    "+r"(c[12]), "+r"(c[13]), "+r"(c[14]), "+r"(c[15]), "+r"(d[0]), "+r"(d[1]),
                    "+r"(d[2]), "+r"(d[3]), "+r"(d[4]), "+r"(d[5]), "+r"(d[6]), "+r"(d[7]),
                    "+r"(d[8]), "+r"(d[9]), "+r"(d[10]), "+r"(d[11]), "+r"(d[12]), "+r"(d[13]),
                    "+r"(d[14]), "+r"(d[15]) : : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// One chunk of a key row: P^T = 2^(S^T log2e/sqrt(d) - lse) and
// dS^T = P^T (c dW^T - c D); lse and c D are the tile's per-query vectors.
// kMasked: query column c0 + i is visible iff lo <= c0 + i < hi (and the key
// row is real); otherwise every column is visible.
template <bool kMasked, int W>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&x)[W], const uint32_t (&w)[W],
                                          const float *lse, const float *cd, int c0, float sl2,
                                          float coef, int lo, int hi, uint32_t (&pk)[W / 2],
                                          uint32_t (&dk)[W / 2]) {
  const float2 scale = make_float2(sl2, sl2), cc = make_float2(coef, coef);
#pragma unroll
  for (int c = 0; c < W; c += 4) {
    const float4 l4 = *reinterpret_cast<const float4 *>(lse + c0 + c);
    const float4 d4 = *reinterpret_cast<const float4 *>(cd + c0 + c);
#pragma unroll
    for (int h2 = 0; h2 < 4; h2 += 2) {
      const int i = c + h2;
      const float2 l2 = h2 ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
      const float2 d2 = h2 ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
      float2 e = __ffma2_rn(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), scale,
                            make_float2(-l2.x, -l2.y));
      float pa = ex2_approx(e.x), pb = ex2_approx(e.y);
      if (kMasked) {
        pa = (c0 + i >= lo && c0 + i < hi) ? pa : 0.f;
        pb = (c0 + i + 1 >= lo && c0 + i + 1 < hi) ? pb : 0.f;
      }
      const float2 t = __ffma2_rn(make_float2(__uint_as_float(w[i]), __uint_as_float(w[i + 1])),
                                  cc, make_float2(-d2.x, -d2.y));
      const float2 ds = __fmul2_rn(make_float2(pa, pb), t);
      pk[i / 2] = pack_bf16x2(pa, pb);
      dk[i / 2] = pack_bf16x2(ds.x, ds.y);
    }
  }
}

// One work item: a (128-key tile, head, map) of the backward.  Items are
// numbered heaviest first (under the causal mask key tile 0 sees every query
// tile): item j is key tile j / (2 BH), head (j / 2) % BH, map j % 2.
struct Item {
  int map, kt, h, k0, qt_first, n_q;
  int64_t bh;
};

__device__ __forceinline__ Item item_at(const BwdParams &p, int64_t j) {
  Item w;
  w.map = static_cast<int>(j & 1);
  w.kt = static_cast<int>((j >> 1) / p.BH);
  w.bh = (j >> 1) % p.BH;
  w.h = static_cast<int>(w.bh % p.H);
  w.k0 = w.kt * BK;
  w.qt_first = p.causal ? w.kt : 0;
  w.n_q = p.n_qtiles - w.qt_first;
  return w;
}

// The r-th item of this CTA: items are dealt to the persistent CTAs in rounds
// of gridDim.x, in alternating direction (so that the CTA that got the
// lightest item of one round gets the heaviest of the next).
__device__ __forceinline__ bool next_item(const BwdParams &p, int r, Item &w) {
  const int64_t G = gridDim.x;
  const int64_t c = (r & 1) ? (G - 1 - blockIdx.x) : blockIdx.x;
  const int64_t j = static_cast<int64_t>(r) * G + c;
  if (j >= p.n_items) return false;
  w = item_at(p, j);
  return true;
}

// ---------------------------------------------------------------- kernel 2
// Persistent: one CTA per SM walks its items; every role counts barrier
// phases by tile over all of its items (qd_*, s_full, ds_*, dq_*) or by item
// (kv_full, kv_empty, acc_done, acc_free).  kStridedDk: dk1 and dk2 are
// written through their strides (a separate instantiation: the 64-bit stride
// arithmetic costs the contiguous epilogue registers it does not have).
template <bool kStridedDk>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    diffattn_bwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tm_q1,
                                   const __grid_constant__ CUtensorMap tm_k1,
                                   const __grid_constant__ CUtensorMap tm_q2,
                                   const __grid_constant__ CUtensorMap tm_k2,
                                   const __grid_constant__ CUtensorMap tm_v,
                                   const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + OFF_CTRL);
  volatile int *abort_flag = &ctrl->abort;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t n_pad = static_cast<int64_t>(p.n_qtiles) * BQ;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->kv_full, 1);
    mbar_init(&ctrl->kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->qd_full[s], 1);
      mbar_init(&ctrl->qd_empty[s], 1);
    }
    mbar_init(&ctrl->s_full, 1);
    mbar_init(&ctrl->ds_ready[0], 384);
    mbar_init(&ctrl->ds_ready[1], 384);
    mbar_init(&ctrl->ds_ready[2], 256);
    mbar_init(&ctrl->ds_free[0], 1);
    mbar_init(&ctrl->ds_free[1], 1);
    mbar_init(&ctrl->dq_full, 1);
    mbar_init(&ctrl->dq_free, 128);
    mbar_init(&ctrl->acc_done, 1);
    mbar_init(&ctrl->acc_free, 384);
    mbar_init(&ctrl->drain, 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q1);
    tma_prefetch_desc(&tm_k1);
    tma_prefetch_desc(&tm_q2);
    tma_prefetch_desc(&tm_k2);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t issued[2] = {0, 0};
      uint32_t T = 0;  // tiles loaded so far, over all items
      int kv_issued = 0;
      Item w;
      bool ok = true;
      for (int r = 0; ok && next_item(p, r, w); ++r) {
        const CUtensorMap *tm_q = w.map ? &tm_q2 : &tm_q1;
        const CUtensorMap *tm_k = w.map ? &tm_k2 : &tm_k1;
        const float *lse_g = p.lse + (w.map * p.BH + w.bh) * n_pad;
        const float *dvec_g = p.dvec + (w.map * p.BH + w.bh) * n_pad;
        // batch index (b * H + h = bh < 2^31)
        const int wb = static_cast<int>(static_cast<uint32_t>(w.bh) / static_cast<uint32_t>(p.H));
        // K and V of the previous item are read until its last MMAs complete.
        if (r > 0 && !(ok = mbar_wait(&ctrl->kv_empty, (r - 1) & 1, abort_flag, WAIT_TIMEOUT_NS)))
          break;
        mbar_arrive_expect_tx(&ctrl->kv_full, 3 * TILE64);
        tma_load_4d(smem + OFF_K, tm_k, &ctrl->kv_full, 0, w.k0, w.h, wb);
        tma_load_4d(smem + OFF_V, &tm_v, &ctrl->kv_full, 0, w.k0, w.h, wb);
        tma_load_4d(smem + OFF_V + TILE64, &tm_v, &ctrl->kv_full, HD, w.k0, w.h, wb);
        kv_issued = r + 1;
        for (int it = 0; it < w.n_q; ++it, ++T) {
          const int s = T & 1;
          const uint32_t u = T >> 1;
          if (u > 0 && !(ok = mbar_wait(&ctrl->qd_empty[s], (u - 1) & 1, abort_flag,
                                        WAIT_TIMEOUT_NS)))
            break;
          const int q0 = (w.qt_first + it) * BQ;
          uint64_t *bar = &ctrl->qd_full[s];
          mbar_arrive_expect_tx(bar, 3 * TILE64 + VEC_BYTES);
          tma_load_4d(smem + OFF_Q + s * TILE64, tm_q, bar, 0, q0, w.h, wb);
          uint8_t *dst = smem + OFF_DO + s * 2 * TILE64;
          tma_load_4d(dst, &tm_do, bar, 0, q0, w.h, wb);
          tma_load_4d(dst + TILE64, &tm_do, bar, HD, q0, w.h, wb);
          float *vec = reinterpret_cast<float *>(smem + OFF_VEC + s * VEC_BYTES);
          bulk_g2s(vec, lse_g + q0, BQ * 4, bar);
          bulk_g2s(vec + BQ, dvec_g + q0, BQ * 4, bar);
          issued[s] = u + 1;
        }
      }
      // Loads still in flight land before the CTA exits.
      if (kv_issued > 0) drain_wait(&ctrl->kv_full, (kv_issued - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (issued[s] > 0) drain_wait(&ctrl->qd_full[s], (issued[s] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp walks the loop, so every operand is warp-uniform; one
    // elected lane issues each MMA and commit (the same lane throughout).
    constexpr uint32_t ID_S = idesc_ab(BK, BQ, false, false);   // S^T = K Q^T
    constexpr uint32_t ID_W = idesc_ab(BK, BQ, false, false);   // dW^T = V dO^T
    constexpr uint32_t ID_DV = idesc_ab(BK, DV, false, true);   // dV += P^T dO
    constexpr uint32_t ID_DK = idesc_ab(BK, HD, false, true);   // dK += dS^T Q
    constexpr uint32_t ID_DQ = idesc_ab(BQ, HD, true, true);    // dQ = dS K
    const uint32_t s_k = smem_u32(smem + OFF_K), s_v = smem_u32(smem + OFF_V);
    const uint32_t s_ds = smem_u32(smem + OFF_DS);
    // Every operand is a base tile plus a byte offset below 256 KB, so advancing
    // it adds offset >> 4 to the start-address field of the descriptor's low
    // word; all of them share the high word (stride offset 1024, version,
    // 128-byte swizzle).
    auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
    const uint32_t dhi = static_cast<uint32_t>(smem_desc_sw128(s_k, 16, 1024) >> 32);
    // K-major views (rows of 64 bf16): advance 32 bytes per 16 elements.
    const uint32_t d_k_kmaj = lo(smem_desc_sw128(s_k, 16, 1024));
    const uint32_t d_v_kmaj = lo(smem_desc_sw128(s_v, 16, 1024));
    // MN-major views (64-wide blocks TILE64 apart): advance 2048 bytes per 16 rows.
    const uint32_t d_k_mn = lo(smem_desc_sw128(s_k, TILE64, 1024));
    const uint32_t d_ds_mn = lo(smem_desc_sw128(s_ds, TILE64, 1024));
    auto stage_desc = [&](int st, bool k_major, bool is_do) {
      const uint32_t base = is_do ? smem_u32(smem + OFF_DO + st * 2 * TILE64)
                                  : smem_u32(smem + OFF_Q + st * TILE64);
      return lo(k_major ? smem_desc_sw128(base, 16, 1024) : smem_desc_sw128(base, TILE64, 1024));
    };
    // S^T = K Q^T (K = 64) and dW^T = V dO^T (K = 128: two 64-column boxes) of
    // the query tile held in stage st.
    auto issue_s = [&](int st) {
      const uint32_t d_q = stage_desc(st, true, false);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16_ss_lo_warp(tmem + TM_S, d_k_kmaj + 2 * kk, d_q + 2 * kk, dhi, ID_S, kk > 0);
    };
    auto issue_w = [&](int st) {
      const uint32_t d_do = stage_desc(st, true, true);
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * TILE64 + 32 * (kk & 3)) >> 4;
        umma_bf16_ss_lo_warp(tmem + TM_W, d_v_kmaj + off, d_do + off, dhi, ID_W, kk > 0);
      }
    };
    // The 16 queries of chunk c (the K slice of both products): dV += P^T dO,
    // A = packed P^T, B = dO MN-major; dK += dS^T Q, A = packed dS^T, B = Q
    // MN-major.  The packed operands sit at tm_p(c) and tm_ds(c).
    auto issue_dv_dk = [&](int st, int c, uint32_t acc) {
      const uint32_t off = (2048u * c) >> 4;
      umma_bf16_ts_lo_warp(tmem + TM_DV, tmem + tm_p(c), stage_desc(st, false, true) + off, dhi,
                           ID_DV, acc);
      umma_bf16_ts_lo_warp(tmem + TM_DK, tmem + tm_ds(c), stage_desc(st, false, false) + off,
                           dhi, ID_DK, acc);
    };
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, WAIT_TIMEOUT_NS));
    };
    // Order per query tile i of an item: dV_i and dK_i chunk by chunk as the
    // P^T / dS^T warps publish them (three steps).  Step 1 also means that
    // every dW^T_i column has been read and that the packed dS^T in the dW^T
    // columns is consumed by the MMAs issued so far, so dW^T of tile i+1
    // follows the chunks of step 1 while the warps compute step 2; S^T of tile
    // i+1 follows the chunks of step 2; then dQ_i, which runs while the warps
    // start on tile i+1.  The first tile of an item waits for the item's K
    // and V, which replace the previous item's once its last MMAs are done.
    bool ok = true;
    uint32_t T = 0;  // tiles processed so far, over all items
    Item w;
    for (int r = 0; ok && next_item(p, r, w); ++r) {
      if (!(ok = wait_all(&ctrl->kv_full, r & 1) && wait_all(&ctrl->qd_full[T & 1], (T >> 1) & 1)))
        break;
      tc_fence_after_sync();
      issue_w(T & 1);
      issue_s(T & 1);
      umma_commit_warp(&ctrl->s_full);
      // The item's first dV and dK MMAs overwrite the accumulators that the
      // previous item's epilogue reads.
      if (r > 0 && !(ok = wait_all(&ctrl->acc_free, (r - 1) & 1))) break;
      for (int it = 0; ok && it < w.n_q; ++it, ++T) {
        const int s = T & 1;  // Q / dO stage and dS^T buffer of tile T
        for (int step = 0; ok && step < 3; ++step) {
          if (!(ok = wait_all(&ctrl->ds_ready[step], T & 1))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int c = 3 * step + j;
            if (c < BQ / 16) issue_dv_dk(s, c, (it > 0 || c > 0) ? 1u : 0u);
          }
          if (it + 1 < w.n_q) {
            const int s1 = s ^ 1;
            if (step == 1) {
              if (!(ok = wait_all(&ctrl->qd_full[s1], ((T + 1) >> 1) & 1))) break;
              tc_fence_after_sync();
              issue_w(s1);
            } else if (step == 2) {
              issue_s(s1);
              umma_commit_warp(&ctrl->s_full);
            }
          }
        }
        if (!ok) break;
        umma_commit_warp(&ctrl->qd_empty[s]);  // the last reads of Q_i and dO_i
        // dQ = dS K: A = dS^T read MN-major (M = queries), B = K MN-major (K = keys).
        if (T > 0 && !(ok = wait_all(&ctrl->dq_free, (T - 1) & 1))) break;
        tc_fence_after_sync();
        const uint32_t d_ds = d_ds_mn + ((s * DS_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16_ss_lo_warp(tmem + TM_DQ, d_ds + 128 * kk, d_k_mn + 128 * kk, dhi, ID_DQ,
                               kk > 0);
        umma_commit_warp(&ctrl->dq_full);
        umma_commit_warp(&ctrl->ds_free[s]);
      }
      if (!ok) break;
      umma_commit_warp(&ctrl->acc_done);  // dV and dK of the item are complete
      umma_commit_warp(&ctrl->kv_empty);  // K and V of the item are no longer read
    }
    umma_commit_warp(&ctrl->drain);
    drain_wait(&ctrl->drain, 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- P^T, dS^T, dQ drain
    // Three warpgroups share the eight 16-query chunks of a tile in three
    // steps: in step t group g takes chunk 3t + g (step 2 has chunks 6 and 7,
    // for groups 0 and 1), and each step is published as soon as it is done so
    // that its dV and dK MMAs overlap the next step.  Chunk c leaves packed
    // P^T and dS^T at tm_p(c) and tm_ds(c), and dS^T in shared memory for dQ.
    // Step 1 is published only once the step-2 chunk's S^T and dW^T are in
    // registers.  Group 2, with one chunk fewer, drains dQ of the previous
    // tile (which may belong to the previous item) after its second step.
    // After an item's last tile, every group takes part in its dV / dK
    // epilogue.
    const int g = (warp - 4) / 4;
    const int kr = (warp % 4) * 32 + lane;  // key row (dQ: query row) = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_lane = tmem + lane_addr;
    const uint32_t t_s = t_lane + TM_S;
    const uint32_t t_w = t_lane + TM_W;
    const float sl2 = p.scale_log2;
    // dQ of tile t (query tile q0 of head bh, map `map`) into the fp32
    // accumulator (thread = query row).
    auto drain_dq = [&](uint32_t t, int map, int64_t bh, int q0) {
      bool okd = mbar_wait(&ctrl->dq_full, t & 1, abort_flag, WAIT_TIMEOUT_NS);
      okd = __all_sync(0xffffffffu, okd);
      if (!okd) return false;
      tc_fence_after_sync();
      uint32_t a[32], b[32];
      tmem_ld_x32_nowait(tmem + lane_addr + TM_DQ, a);
      tmem_ld_x32_nowait(tmem + lane_addr + TM_DQ + 32, b);
      tmem_ld_wait_x32(a);
      tmem_ld_wait_x32(b);
      tc_fence_before_sync();
      mbar_arrive(&ctrl->dq_free);
      // dQ rows, transposed across each 8-lane group so that every vector
      // reduction covers four 128-byte row segments (one row per lane made
      // each instruction touch 32 rows).
      float *dq_base = p.dq_acc + (map * p.BH + bh) * static_cast<int64_t>(p.N) * HD;
      const int row0 = q0 + (warp % 4) * 32 + (lane & ~7);  // the 8-lane group's first row
      float *col_base = dq_base + 4 * (lane & 7);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t(&src)[32] = half ? b : a;
        uint4 ch[8];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          ch[v] = make_uint4(__float_as_uint(__uint_as_float(src[4 * v]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 1]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 2]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 3]) * p.scale));
        transpose8_chunks(ch, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (row0 + j < p.N &&
              dbg_ok(row0 + j >= 0 && 32 * half + 4 * (lane & 7) + 4 <= HD, p.status, 40))
            red_add_v4(col_base + static_cast<int64_t>(row0 + j) * HD + 32 * half,
                       __uint_as_float(ch[j].x), __uint_as_float(ch[j].y),
                       __uint_as_float(ch[j].z), __uint_as_float(ch[j].w));
        }
      }
      return true;
    };
    // Packed P^T and dS^T in tensor memory and dS^T in shared memory visible
    // to the MMAs, then step `step` of this thread is published.
    auto publish = [&](int step) {
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&ctrl->ds_ready[step]);
    };
    bool ok = true;
    uint32_t T = 0;  // tiles processed so far, over all items
    int prev_map = 0, prev_q0 = 0;  // the previous tile, whose dQ group 2 drains
    int64_t prev_bh = 0;
    Item w;
    for (int r = 0; ok && next_item(p, r, w); ++r) {
      const float coef = w.map ? -p.lambda[w.h] : 1.f;
      const int kpos = w.k0 + kr;
      const bool key_ok = kpos < p.N;
      const bool key_tile_ragged = w.k0 + BK > p.N;
      for (int it = 0; it < w.n_q; ++it, ++T) {
        const int s = T & 1;
        const int q0 = (w.qt_first + it) * BQ;
        ok = mbar_wait(&ctrl->s_full, T & 1, abort_flag, WAIT_TIMEOUT_NS);
        // dS^T buffer s was last read by the dQ MMAs of tile T - 2.
        if (ok && T >= 2)
          ok = mbar_wait(&ctrl->ds_free[s], ((T >> 1) - 1) & 1, abort_flag, WAIT_TIMEOUT_NS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        uint8_t *ds_buf = smem + OFF_DS + s * DS_BYTES;
        const float *vec = reinterpret_cast<const float *>(smem + OFF_VEC + s * VEC_BYTES);
        const float *lse = vec;
        const float *cd = vec + BQ;
        // Query column c of the tile (query q0 + c) is visible iff lo <= c < hi.
        const int lo = p.causal ? (kpos - q0) : 0;
        const int hi = key_ok ? (p.N - q0) : 0;
        const bool masked = key_tile_ragged || q0 + BQ > p.N || (p.causal && q0 == w.k0);
        auto work = [&](const uint32_t (&x)[16], const uint32_t (&wv)[16], int c) {
          const int c0 = 16 * c;
          uint32_t pk[8], dk[8];
          if (masked)
            bwd_chunk<true, 16>(x, wv, lse, cd, c0, sl2, coef, lo, hi, pk, dk);
          else
            bwd_chunk<false, 16>(x, wv, lse, cd, c0, sl2, coef, lo, hi, pk, dk);
          tmem_st8(t_lane + tm_p(c), pk);
          tmem_st8(t_lane + tm_ds(c), dk);
          uint8_t *sub = ds_buf + (c >> 2) * TILE64;  // 64-query half of the dS^T tile
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint4 v4 = make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
            *reinterpret_cast<uint4 *>(sub + sw128(kr, (c & 3) * 2 + j)) = v4;
          }
        };
        // Loads of each step's chunk overlap the work on the one before.
        const int c_a = g, c_b = g + 3, c_c = g + 6;
        const bool third = c_c < BQ / 16;  // uniform per warp
        uint32_t xa[16], wa[16], xb[16], wb[16];
        tmem_ld16(t_s + 16 * c_a, xa);
        tmem_ld16(t_w + 16 * c_a, wa);
        tmem_ld16(t_s + 16 * c_b, xb);
        tmem_ld16(t_w + 16 * c_b, wb);
        tmem_wait16x4(xa, wa, xb, wb);
        work(xa, wa, c_a);
        publish(0);
        if (third) {
          tmem_ld16(t_s + 16 * c_c, xa);
          tmem_ld16(t_w + 16 * c_c, wa);
        }
        work(xb, wb, c_b);
        if (third) tmem_wait16x4(xa, wa, xb, wb);
        publish(1);
        if (third) {
          work(xa, wa, c_c);
          publish(2);
        } else if (T > 0 && !(ok = drain_dq(T - 1, prev_map, prev_bh, prev_q0))) {
          break;
        }
        prev_map = w.map;
        prev_bh = w.bh;
        prev_q0 = q0;
      }
      if (!ok) break;
      // ---------------------------------------------------------------- dV, dK out
      ok = mbar_wait(&ctrl->acc_done, r & 1, abort_flag, WAIT_TIMEOUT_NS);
      // Warp-uniform decision: the TMEM loads below are warp-collective.
      ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
      if (!ok) break;
      tc_fence_after_sync();
      // Every accumulator column this warp handles is read into registers
      // before the next item's MMAs may overwrite them: dV 32-column blocks
      // (group 0: blocks 0-1, group 1: block 2, group 2: block 3) and dK
      // 32-column halves (group 1: columns 0-31, group 2: columns 32-63).
      uint32_t va[32], vb[32];
      const int blk_a = g == 0 ? 0 : g + 1;
      tmem_ld_x32_nowait(tmem + lane_addr + TM_DV + 32 * blk_a, va);
      tmem_ld_x32_nowait(tmem + lane_addr + (g == 0 ? TM_DV + 32 : TM_DK + 32 * (g - 1)), vb);
      tmem_ld_wait_x32(va);
      tmem_ld_wait_x32(vb);
      tc_fence_before_sync();
      mbar_arrive(&ctrl->acc_free);
      // dV times c (both maps add into the fp32 accumulator), each 32-column
      // block transposed across 8-lane groups so that every vector reduction
      // covers four 128-byte row segments.
      const int krow0 = w.k0 + (warp % 4) * 32 + (lane & ~7);  // the 8-lane group's first key row
      float *dv_col = p.dv_acc + w.bh * static_cast<int64_t>(p.N) * DV + 4 * (lane & 7);
      auto store_dv = [&](const uint32_t (&v)[32], int bk) {
        uint4 ch[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          ch[q] = make_uint4(__float_as_uint(coef * __uint_as_float(v[4 * q])),
                             __float_as_uint(coef * __uint_as_float(v[4 * q + 1])),
                             __float_as_uint(coef * __uint_as_float(v[4 * q + 2])),
                             __float_as_uint(coef * __uint_as_float(v[4 * q + 3])));
        transpose8_chunks(ch, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (krow0 + j < p.N &&
              dbg_ok(krow0 + j >= 0 && 32 * bk + 4 * (lane & 7) + 4 <= DV, p.status, 41))
            red_add_v4(dv_col + static_cast<int64_t>(krow0 + j) * DV + 32 * bk,
                       __uint_as_float(ch[j].x), __uint_as_float(ch[j].y),
                       __uint_as_float(ch[j].z), __uint_as_float(ch[j].w));
        }
      };
      store_dv(va, blk_a);
      if (g == 0) store_dv(vb, 1);
      // dK (groups 1 and 2, 32 columns each), scaled by 1/sqrt(d), stored
      // once as bf16: packed, transposed across 4-lane groups, eight 64-byte
      // row segments per store instruction.
      if (g >= 1) {
        uint4 pkt[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 &pk = pkt[q];
          pk.x = pack_bf16x2(__uint_as_float(vb[8 * q + 0]) * p.scale,
                             __uint_as_float(vb[8 * q + 1]) * p.scale);
          pk.y = pack_bf16x2(__uint_as_float(vb[8 * q + 2]) * p.scale,
                             __uint_as_float(vb[8 * q + 3]) * p.scale);
          pk.z = pack_bf16x2(__uint_as_float(vb[8 * q + 4]) * p.scale,
                             __uint_as_float(vb[8 * q + 5]) * p.scale);
          pk.w = pack_bf16x2(__uint_as_float(vb[8 * q + 6]) * p.scale,
                             __uint_as_float(vb[8 * q + 7]) * p.scale);
        }
        transpose4_chunks(pkt, lane);
        const int krow4 = w.k0 + (warp % 4) * 32 + (lane & ~3);  // the 4-lane group's first key row
        const int dcol = 32 * (g - 1) + 8 * (lane & 3);
        __nv_bfloat16 *dk_col;
        int64_t sn;
        if (kStridedDk) {
          const uint32_t wb = static_cast<uint32_t>(w.bh) / static_cast<uint32_t>(p.H);
          const int64_t sb = w.map ? p.dk_sb[1] : p.dk_sb[0];
          const int64_t sh = w.map ? p.dk_sh[1] : p.dk_sh[0];
          sn = w.map ? p.dk_sn[1] : p.dk_sn[0];
          dk_col = (w.map ? p.dk2 : p.dk1) + wb * sb + w.h * sh + dcol;
        } else {
          sn = HD;
          dk_col = (w.map ? p.dk2 : p.dk1) + w.bh * static_cast<int64_t>(p.N) * HD + dcol;
        }
#pragma unroll
        for (int j2 = 0; j2 < 4; ++j2) {
          if (krow4 + j2 < p.N && dbg_ok(krow4 + j2 >= 0 && dcol + 8 <= HD, p.status, 42))
            *reinterpret_cast<uint4 *>(dk_col + (krow4 + j2) * sn) = pkt[j2];
        }
      }
    }
    // dQ of the last tile.
    if (ok && g == 2 && T > 0) drain_dq(T - 1, prev_map, prev_bh, prev_q0);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && p.status != nullptr)
    atomicExch(p.status, static_cast<int32_t>(DIFFATTN_ERR_TIMEOUT));
}

// ---------------------------------------------------------------- kernel 1
struct PreParams {
  int64_t BH;
  int32_t H, N, n_pad, headnorm;
  float eps, out_scale;  // out_scale = 1 - lambda_init
  const float *lambda, *norm_w;
  const __nv_bfloat16 *dy;  // [B, H, N, 128] view
  int64_t dy_sb, dy_sh, dy_sn;  // its element strides (batch, head, row)
  const float *o_n;         // [2][BH][N][128] normalised map outputs
  __nv_bfloat16 *dout;      // [BH][N][128]
  float *dvec;              // [2][BH][n_pad] c_k D_k
  float *dlambda;           // [H], zeroed
  float *dnorm_w;           // [H][128], zeroed
};

constexpr int PRE_WARPS = 8;
constexpr int PRE_ROWS = 64;  // rows per block

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Block (head bh, 64-row chunk); warp w takes rows w, w + 8, ...; lane = 4 columns.
__global__ void __launch_bounds__(PRE_WARPS * 32) diffattn_bwd_pre_kernel(const PreParams p) {
  __shared__ float red_w[PRE_WARPS][DV];
  __shared__ float red_l[PRE_WARPS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t bh = blockIdx.x;
  const int h = static_cast<int>(bh % p.H);
  const int c = 4 * lane;
  const float lam = p.lambda[h];
  float g[4] = {p.out_scale, p.out_scale, p.out_scale, p.out_scale};
  if (p.norm_w)
    for (int j = 0; j < 4; ++j) g[j] *= p.norm_w[h * DV + c + j];
  float acc_w[4] = {0.f, 0.f, 0.f, 0.f};
  float acc_l = 0.f;
  const int64_t plane = p.BH * static_cast<int64_t>(p.N) * DV;
  const __nv_bfloat16 *dy_bh = p.dy + (bh / p.H) * p.dy_sb + h * p.dy_sh;  // this head's dy
  for (int i = blockIdx.y * PRE_ROWS + warp; i < (blockIdx.y + 1) * PRE_ROWS; i += PRE_WARPS) {
    if (i >= p.n_pad) break;
    float d1 = 0.f, d2 = 0.f;
    if (i < p.N) {
      const int64_t row = (bh * p.N + i) * DV + c;
      const uint2 yb = *reinterpret_cast<const uint2 *>(dy_bh + i * p.dy_sn + c);
      const float2 y01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&yb.x));
      const float2 y23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&yb.y));
      const float dy[4] = {y01.x, y01.y, y23.x, y23.y};
      const float4 a = *reinterpret_cast<const float4 *>(p.o_n + row);
      const float4 b = *reinterpret_cast<const float4 *>(p.o_n + plane + row);
      const float o1[4] = {a.x, a.y, a.z, a.w}, o2[4] = {b.x, b.y, b.z, b.w};
      float o[4], dout[4];
      for (int j = 0; j < 4; ++j) o[j] = o1[j] - lam * o2[j];
      if (p.headnorm) {
        // The group form (headnorm = 2) normalises the centred row as the RMS
        // form normalises o; the centring's derivative then removes do's mean.
        if (p.headnorm == 2) {
          const float mu = warp_sum((o[0] + o[1]) + (o[2] + o[3])) * (1.f / DV);
          for (int j = 0; j < 4; ++j) o[j] -= mu;
        }
        float ms = 0.f, t = 0.f;
        for (int j = 0; j < 4; ++j) {
          ms = fmaf(o[j], o[j], ms);
          t = fmaf(dy[j] * g[j], o[j], t);
        }
        ms = warp_sum(ms) * (1.f / DV);
        t = warp_sum(t);
        const float r = rsqrtf(ms + p.eps);
        const float r3 = r * r * r * (1.f / DV);
        for (int j = 0; j < 4; ++j) {
          dout[j] = r * g[j] * dy[j] - r3 * o[j] * t;
          acc_w[j] = fmaf(dy[j] * o[j], r * p.out_scale, acc_w[j]);
        }
        if (p.headnorm == 2) {
          const float md = warp_sum((dout[0] + dout[1]) + (dout[2] + dout[3])) * (1.f / DV);
          for (int j = 0; j < 4; ++j) dout[j] -= md;
        }
      } else {
        for (int j = 0; j < 4; ++j) dout[j] = dy[j];
      }
      // dlambda uses do as computed; D_k the bf16 do the tensor cores see.
      float l2 = 0.f;
      __nv_bfloat162 b01 = __floats2bfloat162_rn(dout[0], dout[1]);
      __nv_bfloat162 b23 = __floats2bfloat162_rn(dout[2], dout[3]);
      const float2 r01 = __bfloat1622float2(b01), r23 = __bfloat1622float2(b23);
      const float dr[4] = {r01.x, r01.y, r23.x, r23.y};
      for (int j = 0; j < 4; ++j) {
        l2 = fmaf(dout[j], o2[j], l2);
        d1 = fmaf(dr[j], o1[j], d1);
        d2 = fmaf(dr[j], o2[j], d2);
      }
      uint2 ob;
      ob.x = *reinterpret_cast<uint32_t *>(&b01);
      ob.y = *reinterpret_cast<uint32_t *>(&b23);
      *reinterpret_cast<uint2 *>(p.dout + row) = ob;
      acc_l -= warp_sum(l2);
      d1 = warp_sum(d1);
      d2 = warp_sum(d2);
    }
    if (lane == 0 && dbg_ok(i < p.n_pad && bh < p.BH, nullptr, 43)) {  // c_k D_k: c_1 = 1, c_2 = -lambda
      p.dvec[bh * p.n_pad + i] = d1;
      p.dvec[(p.BH + bh) * p.n_pad + i] = -lam * d2;
    }
  }
  for (int j = 0; j < 4; ++j) red_w[warp][c + j] = acc_w[j];
  if (lane == 0) red_l[warp] = acc_l;
  __syncthreads();
  if (p.headnorm && p.dnorm_w != nullptr && threadIdx.x < DV) {
    float s = 0.f;
    for (int w = 0; w < PRE_WARPS; ++w) s += red_w[w][threadIdx.x];
    atomicAdd(p.dnorm_w + h * DV + threadIdx.x, s);
  }
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < PRE_WARPS; ++w) s += red_l[w];
    atomicAdd(p.dlambda + h, s);
  }
}

// ---------------------------------------------------------------- kernel 3
// fp32 accumulators -> bf16: dq_acc [2][BH][N][64] -> dq1, dq2; dv_acc -> dv.
// Each thread has FINISH_UNROLL 16-byte loads in flight before it stores (one
// at a time left the copy well short of the memory bandwidth).  kStrided: the
// three destinations are [B, H, N, width] views with the element strides in
// `fs` (dq1, dq2, dv), each 4-element group placed by its (batch, head, row).
constexpr int FINISH_UNROLL = 4;
struct FinishStrides {
  int64_t sb[3], sh[3], sn[3];
  int64_t H, N;
};
template <bool kStrided>
__global__ void diffattn_bwd_finish_kernel(const float *dq_acc, const float *dv_acc,
                                           __nv_bfloat16 *dq1, __nv_bfloat16 *dq2,
                                           __nv_bfloat16 *dv, int64_t n_q4, int64_t n_v4,
                                           const FinishStrides fs) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t total = 2 * n_q4 + n_v4;
  auto src_of = [&](int64_t i, int64_t &j) -> const float4 * {
    if (i < n_q4) { j = i; return reinterpret_cast<const float4 *>(dq_acc); }
    if (i < 2 * n_q4) { j = i - n_q4; return reinterpret_cast<const float4 *>(dq_acc + 4 * n_q4); }
    j = i - 2 * n_q4;
    return reinterpret_cast<const float4 *>(dv_acc);
  };
  for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; base < total;
       base += FINISH_UNROLL * stride) {
    float4 v[FINISH_UNROLL];
#pragma unroll
    for (int u = 0; u < FINISH_UNROLL; ++u) {
      const int64_t i = base + u * stride;
      int64_t j = 0;
      if (i < total) v[u] = src_of(i, j)[j];
    }
#pragma unroll
    for (int u = 0; u < FINISH_UNROLL; ++u) {
      const int64_t i = base + u * stride;
      if (i >= total) continue;
      __nv_bfloat16 *dst;
      int64_t j;
      int t;
      if (i < n_q4) { dst = dq1; j = i; t = 0; }
      else if (i < 2 * n_q4) { dst = dq2; j = i - n_q4; t = 1; }
      else { dst = dv; j = i - 2 * n_q4; t = 2; }
      uint2 o;
      o.x = pack_bf16x2(v[u].x, v[u].y);
      o.y = pack_bf16x2(v[u].z, v[u].w);
      if (kStrided) {
        const int64_t width4 = t == 2 ? DV / 4 : HD / 4;  // 4-element groups per row
        const int64_t row = j / width4, col = 4 * (j - row * width4);
        const int64_t bh = row / fs.N, n = row - bh * fs.N;
        const int64_t b = bh / fs.H, h = bh - b * fs.H;
        const int64_t sb = t == 0 ? fs.sb[0] : t == 1 ? fs.sb[1] : fs.sb[2];
        const int64_t sh = t == 0 ? fs.sh[0] : t == 1 ? fs.sh[1] : fs.sh[2];
        const int64_t sn = t == 0 ? fs.sn[0] : t == 1 ? fs.sn[1] : fs.sn[2];
        *reinterpret_cast<uint2 *>(dst + b * sb + h * sh + n * sn + col) = o;
      } else {
        reinterpret_cast<uint2 *>(dst)[j] = o;
      }
    }
  }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime (shared with the forward file's
// approach: looked up once, no link against the driver library).
using EncodeTiledFnB = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

// 4-D view {inner, rows, H, B} of a bf16 tensor with element strides st (rows
// contiguous); 128-row x 64-column boxes with 128-byte swizzle.
static CUresult encode_map_b(CUtensorMap *map, const void *base, uint64_t inner, uint64_t n,
                             uint64_t H, uint64_t B, const diffattn_strides &st) {
  static EncodeTiledFnB fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFnB>(ptr);
  }();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[4] = {inner, n, H, B};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int64_t bwd_workspace_floats(int64_t BH, int64_t N) {
  const int64_t n_pad = (N + BQ - 1) / BQ * BQ;
  // dO bf16 [BH][N][128] (as floats: half), D [2][BH][n_pad], dq_acc [2][BH][N][64],
  // dv_acc [BH][N][128]; each region rounded to 64 floats (256 bytes).
  auto r64 = [](int64_t x) { return (x + 63) / 64 * 64; };
  return r64(BH * N * DV / 2) + r64(2 * BH * n_pad) + r64(2 * BH * N * HD) + r64(BH * N * DV);
}

diffattn_status launch_bwd_bf16_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w,
                                      const float *saved, const void *dy, void *dq1, void *dk1,
                                      void *dq2, void *dk2, void *dv, float *dlambda,
                                      float *dnorm_w, float *workspace, cudaStream_t stream,
                                      const diffattn_strides *strides) {
  const int64_t BH = desc.B * desc.H, N = desc.N;
  // Element strides of q1, k1, q2, k2, v, dy, dq1, dk1, dq2, dk2, dv: given, or
  // contiguous [B, H, N, width].
  diffattn_strides st[kBwdStrides];
  for (int i = 0; i < kBwdStrides; ++i) {
    const int64_t width = (i == 4 || i == 5 || i == 10) ? DV : HD;
    st[i] = strides ? strides[i] : diffattn_strides{desc.H * N * width, N * width, width};
  }
  const int64_t n_qtiles = (N + BQ - 1) / BQ;
  const int64_t n_pad = n_qtiles * BQ;
  if (BH * n_qtiles * 2 > INT32_MAX || N > INT32_MAX / 2) return DIFFATTN_ERR_UNSUPPORTED;
  auto r64 = [](int64_t x) { return (x + 63) / 64 * 64; };
  float *ws = workspace;
  __nv_bfloat16 *dout = reinterpret_cast<__nv_bfloat16 *>(ws);
  ws += r64(BH * N * DV / 2);
  float *dvec = ws;
  ws += r64(2 * BH * n_pad);
  float *dq_acc = ws;
  ws += r64(2 * BH * N * HD);
  float *dv_acc = ws;
  const float *o_n = saved;
  const float *lse = saved + 2 * BH * N * DV;

  if (cudaMemsetAsync(dq_acc, 0, sizeof(float) * (2 * BH * N * HD), stream) != cudaSuccess ||
      cudaMemsetAsync(dv_acc, 0, sizeof(float) * (BH * N * DV), stream) != cudaSuccess ||
      cudaMemsetAsync(dlambda, 0, sizeof(float) * desc.H, stream) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;
  if (desc.headnorm && dnorm_w != nullptr &&
      cudaMemsetAsync(dnorm_w, 0, sizeof(float) * desc.H * DV, stream) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;

  // 1. do, D_1, D_2, dlambda, dw
  PreParams pp;
  pp.BH = BH;
  pp.H = static_cast<int32_t>(desc.H);
  pp.N = static_cast<int32_t>(N);
  pp.n_pad = static_cast<int32_t>(n_pad);
  pp.headnorm = desc.headnorm;  // 0, 1 (RMS) or 2 (group)
  pp.eps = desc.eps;
  pp.out_scale = 1.0f - desc.lambda_init;
  pp.lambda = lambda;
  pp.norm_w = norm_w;
  pp.dy = static_cast<const __nv_bfloat16 *>(dy);
  pp.dy_sb = st[5].b;
  pp.dy_sh = st[5].h;
  pp.dy_sn = st[5].n;
  pp.o_n = o_n;
  pp.dout = dout;
  pp.dvec = dvec;
  pp.dlambda = dlambda;
  pp.dnorm_w = desc.headnorm ? dnorm_w : nullptr;
  dim3 pre_grid(static_cast<unsigned>(BH), static_cast<unsigned>((n_pad + PRE_ROWS - 1) / PRE_ROWS));
  diffattn_bwd_pre_kernel<<<pre_grid, PRE_WARPS * 32, 0, stream>>>(pp);
  if (cudaGetLastError() != cudaSuccess) return DIFFATTN_ERR_CUDA;

  // 2. fused gradient kernel
  CUtensorMap maps[6];
  const void *bases[6] = {q1, k1, q2, k2, v, dout};
  const diffattn_strides dout_st{desc.H * N * DV, N * DV, DV};  // the workspace's dO
  for (int i = 0; i < 6; ++i) {
    const uint64_t inner = (i >= 4) ? DV : HD;
    if (encode_map_b(&maps[i], bases[i], inner, static_cast<uint64_t>(N),
                     static_cast<uint64_t>(desc.H), static_cast<uint64_t>(desc.B),
                     i == 5 ? dout_st : st[i]) != CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];  // per device (concurrent callers may both set)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(diffattn_bwd_bf16_sm103_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(diffattn_bwd_bf16_sm103_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  BwdParams p;
  p.BH = BH;
  p.H = static_cast<int32_t>(desc.H);
  p.N = static_cast<int32_t>(N);
  p.n_qtiles = static_cast<int32_t>(n_qtiles);
  p.n_ktiles = static_cast<int32_t>(n_qtiles);
  p.causal = desc.causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(HD)));
  p.lambda = lambda;
  p.lse = lse;
  p.dvec = dvec;
  p.dk1 = static_cast<__nv_bfloat16 *>(dk1);
  p.dk2 = static_cast<__nv_bfloat16 *>(dk2);
  for (int m = 0; m < 2; ++m) {  // dk1: strides[7], dk2: strides[9]
    p.dk_sb[m] = st[7 + 2 * m].b;
    p.dk_sh[m] = st[7 + 2 * m].h;
    p.dk_sn[m] = st[7 + 2 * m].n;
  }
  p.dq_acc = dq_acc;
  p.dv_acc = dv_acc;
  p.status = desc.status_dev;
  p.n_items = 2 * BH * n_qtiles;
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  dim3 grid(static_cast<unsigned>(std::min<int64_t>(p.n_items, sms)));
  if (strides != nullptr)
    diffattn_bwd_bf16_sm103_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  else
    diffattn_bwd_bf16_sm103_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  if (cudaGetLastError() != cudaSuccess) return DIFFATTN_ERR_CUDA;

  // 3. bf16 gradients
  const int64_t n_q4 = BH * N * HD / 4, n_v4 = BH * N * DV / 4;
  FinishStrides fs;
  const int dst_idx[3] = {6, 8, 10};  // dq1, dq2, dv
  for (int t = 0; t < 3; ++t) {
    fs.sb[t] = st[dst_idx[t]].b;
    fs.sh[t] = st[dst_idx[t]].h;
    fs.sn[t] = st[dst_idx[t]].n;
  }
  fs.H = desc.H;
  fs.N = N;
  if (strides != nullptr)
    diffattn_bwd_finish_kernel<true><<<4 * sms, 256, 0, stream>>>(
        dq_acc, dv_acc, static_cast<__nv_bfloat16 *>(dq1), static_cast<__nv_bfloat16 *>(dq2),
        static_cast<__nv_bfloat16 *>(dv), n_q4, n_v4, fs);
  else
    diffattn_bwd_finish_kernel<false><<<4 * sms, 256, 0, stream>>>(
        dq_acc, dv_acc, static_cast<__nv_bfloat16 *>(dq1), static_cast<__nv_bfloat16 *>(dq2),
        static_cast<__nv_bfloat16 *>(dv), n_q4, n_v4, fs);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
