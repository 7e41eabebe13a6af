// Training for query/key halves of width d = 128 (values 2d = 256 wide) on
// sm_103a: the saving forward and the backward pass.
//
// What it computes is the d = 64 training pair's ("Differential Transformer",
// Ultralytics glossary, section "How differential attention works": the page
// gives the forward; the gradient is its derivative by the chain rule):
//   dV = map1^T do - lambda map2^T do,  dW = do V^T,
//   dS_k = c_k P_k * (dW - D_k), D_k = do . o_k, c_1 = 1, c_2 = -lambda,
//   dQ_k = dS_k K_k / sqrt(d),  dK_k = dS_k^T Q_k / sqrt(d),
// with do, dlambda and dw from the head norm's chain rule as in the d = 64
// preprocess.
//
// The d = 64 gradient kernel keeps S^T, dW^T, dV, dK and dQ of one key tile in
// tensor memory at once (512 columns).  At d = 128 they would take 768 (dV
// alone is 256), so the work splits into two kinds of CTA, each with one key
// tile of one head:
//   dV items:     S1^T = K1 Q1^T, S2^T = K2 Q2^T, W^T = P1^T - lambda P2^T,
//                 dV += W^T dO                 (S1^T, S2^T, dV: 512 columns)
//   dK/dQ items:  one map: S^T = K Q^T, dW^T = V dO^T, dS^T, dK += dS^T Q,
//                 dQ = dS K (drained to an fp32 accumulator)   (512 columns)
// Both recompute P from the saved log2-sum-exp.  Each CTA streams its query
// tiles through one shared-memory stage (a second would not fit beside the
// K, V and dO tiles of this width), refilled piecewise as each operand is
// released: in dK/dQ items dO once dW^T is computed and each 64-query half of
// Q once that half's dK product is; in dV items Q once S^T is computed and dO
// once dV is.  Each query half of a tile (the softmax warps of one half) has
// its own barriers, so one half's products, and the next tile's S^T (and dW^T)
// of that half, run while the other half is still in its element loop.
//
// The saving forward runs the d = 128 forward (the output, also writing each
// map's log2-sum-exp and the row's o = o_1 - lambda o_2 before the norm), then
// map 2's output alone from its saved log2-sum-exp in one pass over the keys
// (diffattn_map_out_d128_kernel); the preprocess rebuilds o_1 = o + lambda o_2.
// Both are stored in fp32: dlambda = -sum do . o_2 cancels heavily once the head
// norm has made do nearly orthogonal to o, and bf16 map outputs put its error
// above 2 % of its size on ordinary inputs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <cmath>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr int BK = 128;   // keys per CTA (TMEM lanes)
constexpr int BQ = 128;   // queries per tile
constexpr int HD = 128;   // query/key half width d
constexpr int DV = 256;   // value width 2d
constexpr int NUM_THREADS = 384;  // producer, MMA issuer, 2 idle, 8 softmax warps
constexpr int SOFTMAX_THREADS = 256;
constexpr uint32_t BOX = 128 * 64 * 2;  // one [128 rows x 64 columns] bf16 box: 16 KB

// Shared memory (byte offsets), dV items: K1, K2 (two boxes each), Q1, Q2 (two
// boxes each), dO (four boxes), lse1 and lse2 of the tile's queries.
constexpr uint32_t V_OFF_K1 = 0, V_OFF_K2 = 2 * BOX, V_OFF_Q1 = 4 * BOX, V_OFF_Q2 = 6 * BOX;
constexpr uint32_t V_OFF_DO = 8 * BOX, V_OFF_VEC = 12 * BOX;
// dK/dQ items: K (two boxes), V (four), Q (two), dO (four), dS^T (two: queries
// 0-63 and 64-127 of each key row), lse and c D of the tile's queries.
constexpr uint32_t K_OFF_K = 0, K_OFF_V = 2 * BOX, K_OFF_Q = 6 * BOX, K_OFF_DO = 8 * BOX;
constexpr uint32_t K_OFF_DS = 12 * BOX, K_OFF_VEC = 14 * BOX;
constexpr uint32_t VEC_BYTES = 2 * BQ * 4;
// dV items load a tile's vectors with its queries, which are released while
// the previous tile's softmax may still read its own: two slots.
template <bool kDV>
constexpr int vec_slots() {
  return kDV ? 2 : 1;
}

struct Ctrl {
  uint64_t kv_full;   // the item's key (and value) tiles
  uint64_t q_full;    // dV items: the tile's queries and per-query vectors
  uint64_t q_empty;   // dV items: the tile's queries have been read (S1^T, S2^T)
  uint64_t do_full;   // the tile's dO
  uint64_t do_empty;  // the tile's dO has been read (dV items: dV; dK/dQ: dW^T)
  uint64_t q_half_full[2];   // dK/dQ items: query half h of Q and its vectors
  uint64_t q_half_empty[2];  // dK/dQ items: query half h of Q has been read (dK)
  uint64_t s_half[2];  // S^T (dK/dQ: and dW^T; dV: S1^T, S2^T) of the tile's query half h
  uint64_t p_half[2];  // query half h's packed operand is published (per thread)
  uint64_t acc_done;  // the item's dV or dK is complete
  uint64_t dq_full;   // dQ of the tile (dK/dQ items)
  uint64_t dq_free;   // dQ read out of tensor memory (per softmax thread)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <bool kDV>
constexpr uint32_t off_ctrl() {
  return (kDV ? V_OFF_VEC : K_OFF_VEC) + vec_slots<kDV>() * VEC_BYTES;
}
template <bool kDV>
constexpr uint32_t smem_bytes() {
  return off_ctrl<kDV>() + static_cast<uint32_t>(sizeof(Ctrl)) + 1024;  // + alignment slack
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448,
              "shared memory budget exceeded");
static_assert(smem_bytes<false>() + 1024 < (1u << 18), "descriptor start addresses below 256 KB");

// Tensor memory: dV items S1^T 0-127, S2^T 128-255, dV 256-511; dK/dQ items
// S^T 0-127, dW^T 128-255, dK 256-383, dQ 384-511.  A tile's packed operand
// (W^T or dS^T, two bf16 per column) goes over its own S^T columns: query
// pairs of queries 0-63 over columns 0-31, of queries 64-127 over 64-95, each
// thread writing only columns of its lane it has already read.
constexpr uint32_t TM_S = 0, TM_S2 = 128, TM_W = 128, TM_DV = 256, TM_DK = 256, TM_DQ = 384;
__host__ __device__ constexpr uint32_t tm_pack(int kk) {  // 16-query step kk of the packed operand
  return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4);
}

constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr uint64_t DRAIN_TIMEOUT_NS = 200000000ull;

struct Params {
  int64_t BH;
  int32_t H, N, n_qtiles, n_ktiles, causal;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  const float *lambda;
  const float *lse;   // [2][BH][n_pad] log2-sum-exp of the saving forward
  const float *dvec;  // [2][BH][n_pad] c_k D_k
  __nv_bfloat16 *dv;                 // dV items: [B, H, N, 256] view
  int64_t dv_sb, dv_sh, dv_sn;
  __nv_bfloat16 *dk1, *dk2;          // dK/dQ items: [B, H, N, 128] views
  int64_t dk_sb[2], dk_sh[2], dk_sn[2];
  float *dq_acc;                     // [2][BH][N][128], zeroed
  int32_t *status;
};

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
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
// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
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
__device__ __forceinline__ void tmem_wait16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]),
                 "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                 "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__host__ __device__ constexpr uint32_t idesc_ab(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Work items, heaviest first: under the causal mask key tile 0 sees every query
// tile.  dV items: (key tile, head); dK/dQ items: (key tile, head, map).
struct Item {
  int map, h, b, k0, qt_first, n_q;
  int64_t bh;
};
template <bool kDV>
__device__ __forceinline__ Item item_of(const Params &p, uint32_t j) {
  Item w;
  const uint32_t per_kt = static_cast<uint32_t>(p.BH) * (kDV ? 1u : 2u);
  const int kt = static_cast<int>(j / per_kt);
  const uint32_t rem = j % per_kt;
  w.map = kDV ? 0 : static_cast<int>(rem & 1u);
  const uint32_t bh32 = kDV ? rem : rem >> 1;
  w.bh = bh32;
  w.h = static_cast<int>(bh32 % static_cast<uint32_t>(p.H));
  w.b = static_cast<int>(bh32 / static_cast<uint32_t>(p.H));
  w.k0 = kt * BK;
  w.qt_first = p.causal ? kt : 0;
  w.n_q = p.n_qtiles - w.qt_first;
  return w;
}

template <bool kDV>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    diffattn_bwd_d128_sm103_kernel(const __grid_constant__ CUtensorMap tm_q1,
                                   const __grid_constant__ CUtensorMap tm_k1,
                                   const __grid_constant__ CUtensorMap tm_q2,
                                   const __grid_constant__ CUtensorMap tm_k2,
                                   const __grid_constant__ CUtensorMap tm_v,
                                   const __grid_constant__ CUtensorMap tm_do,
                                   const __grid_constant__ CUtensorMap tm_q1h,
                                   const __grid_constant__ CUtensorMap tm_q2h, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + off_ctrl<kDV>());
  volatile int *abort_flag = &ctrl->abort;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Item w = item_of<kDV>(p, blockIdx.x);
  const int64_t n_pad = static_cast<int64_t>(p.n_qtiles) * BQ;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->kv_full, 1);
    mbar_init(&ctrl->q_full, 1);
    mbar_init(&ctrl->q_empty, 1);
    mbar_init(&ctrl->do_full, 1);
    mbar_init(&ctrl->do_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&ctrl->q_half_full[h], 1);
      mbar_init(&ctrl->q_half_empty[h], 1);
      mbar_init(&ctrl->s_half[h], 1);
      mbar_init(&ctrl->p_half[h], SOFTMAX_THREADS / 2);
    }
    mbar_init(&ctrl->acc_done, 1);
    mbar_init(&ctrl->dq_full, 1);
    mbar_init(&ctrl->dq_free, SOFTMAX_THREADS);
    mbar_init(&ctrl->drain, 1);
    ctrl->abort = 0;
    fence_barrier_init();
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
      bool ok = true;
      if (kDV) {
        mbar_arrive_expect_tx(&ctrl->kv_full, 4 * BOX);
        for (int x = 0; x < 2; ++x) {
          tma_load_4d(smem + V_OFF_K1 + x * BOX, &tm_k1, &ctrl->kv_full, 64 * x, w.k0, w.h, w.b);
          tma_load_4d(smem + V_OFF_K2 + x * BOX, &tm_k2, &ctrl->kv_full, 64 * x, w.k0, w.h, w.b);
        }
      } else {
        mbar_arrive_expect_tx(&ctrl->kv_full, 6 * BOX);
        const CUtensorMap *tk = w.map ? &tm_k2 : &tm_k1;
        for (int x = 0; x < 2; ++x)
          tma_load_4d(smem + K_OFF_K + x * BOX, tk, &ctrl->kv_full, 64 * x, w.k0, w.h, w.b);
        for (int x = 0; x < 4; ++x)
          tma_load_4d(smem + K_OFF_V + x * BOX, &tm_v, &ctrl->kv_full, 64 * x, w.k0, w.h, w.b);
      }
      const float *lse_a = p.lse + (w.map * p.BH + w.bh) * n_pad;
      const float *lse_b = kDV ? p.lse + (p.BH + w.bh) * n_pad : p.dvec + (w.map * p.BH + w.bh) * n_pad;
      // Per tile: the queries (and vectors), then dO, each after the previous
      // tile released it; in dK/dQ items dO is released first, then each half of
      // the queries, so they go in that order.
      auto load_q = [&](int it) {
        const int q0 = (w.qt_first + it) * BQ;
        uint8_t *vec = smem + (kDV ? V_OFF_VEC : K_OFF_VEC) + (it % vec_slots<kDV>()) * VEC_BYTES;
        mbar_arrive_expect_tx(&ctrl->q_full, 4 * BOX + VEC_BYTES);
        for (int x = 0; x < 2; ++x) {
          tma_load_4d(smem + V_OFF_Q1 + x * BOX, &tm_q1, &ctrl->q_full, 64 * x, q0, w.h, w.b);
          tma_load_4d(smem + V_OFF_Q2 + x * BOX, &tm_q2, &ctrl->q_full, 64 * x, q0, w.h, w.b);
        }
        bulk_g2s(vec, lse_a + q0, BQ * 4, &ctrl->q_full);
        bulk_g2s(vec + BQ * 4, lse_b + q0, BQ * 4, &ctrl->q_full);
      };
      // dK/dQ items: rows 64 h .. 64 h + 63 of the tile's queries (64-row boxes,
      // the lower half of each 128-row box) and their vector entries.
      auto load_q_half = [&](int it, int h) {
        const int q0 = (w.qt_first + it) * BQ + 64 * h;
        uint64_t *bar = &ctrl->q_half_full[h];
        float *vec = reinterpret_cast<float *>(smem + K_OFF_VEC);
        mbar_arrive_expect_tx(bar, 2 * (BOX / 2) + 2 * 64 * 4);
        const CUtensorMap *tq = w.map ? &tm_q2h : &tm_q1h;
        for (int x = 0; x < 2; ++x)
          tma_load_4d(smem + K_OFF_Q + x * BOX + (BOX / 2) * h, tq, bar, 64 * x, q0, w.h, w.b);
        bulk_g2s(vec + 64 * h, lse_a + q0, 64 * 4, bar);
        bulk_g2s(vec + BQ + 64 * h, lse_b + q0, 64 * 4, bar);
      };
      auto load_do = [&](int it) {
        const int q0 = (w.qt_first + it) * BQ;
        mbar_arrive_expect_tx(&ctrl->do_full, 4 * BOX);
        for (int x = 0; x < 4; ++x)
          tma_load_4d(smem + (kDV ? V_OFF_DO : K_OFF_DO) + x * BOX, &tm_do, &ctrl->do_full,
                      64 * x, q0, w.h, w.b);
      };
      uint32_t issued_q = 0, issued_do = 0, issued_qh[2] = {0, 0};
      for (int it = 0; it < w.n_q; ++it) {
        const uint32_t par = static_cast<uint32_t>(it - 1) & 1u;
        if (kDV) {
          if (it > 0 && !(ok = mbar_wait(&ctrl->q_empty, par, abort_flag, WAIT_TIMEOUT_NS))) break;
          load_q(it);
          issued_q = it + 1;
          if (it > 0 && !(ok = mbar_wait(&ctrl->do_empty, par, abort_flag, WAIT_TIMEOUT_NS))) break;
          load_do(it);
          issued_do = it + 1;
        } else {
          if (it > 0 && !(ok = mbar_wait(&ctrl->do_empty, par, abort_flag, WAIT_TIMEOUT_NS))) break;
          load_do(it);
          issued_do = it + 1;
          for (int h = 0; ok && h < 2; ++h) {
            if (it > 0 &&
                !(ok = mbar_wait(&ctrl->q_half_empty[h], par, abort_flag, WAIT_TIMEOUT_NS)))
              break;
            load_q_half(it, h);
            issued_qh[h] = it + 1;
          }
          if (!ok) break;
        }
      }
      // Loads still in flight land before the CTA exits.
      drain_wait(&ctrl->kv_full, 0);
      if (issued_q > 0) drain_wait(&ctrl->q_full, (issued_q - 1) & 1);
      if (issued_do > 0) drain_wait(&ctrl->do_full, (issued_do - 1) & 1);
      for (int h = 0; h < 2; ++h)
        if (issued_qh[h] > 0) drain_wait(&ctrl->q_half_full[h], (issued_qh[h] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
    const uint32_t base = smem_u32(smem);
    const uint32_t dhi = static_cast<uint32_t>(smem_desc_sw128(base, 16, 1024) >> 32);
    auto kmaj = [&](uint32_t off) { return lo(smem_desc_sw128(base + off, 16, 1024)); };
    auto mnmaj = [&](uint32_t off) { return lo(smem_desc_sw128(base + off, BOX, 1024)); };
    // K-major operands of K = 128 or 256 columns in 64-column boxes: step kk
    // is box kk / 4, 32 bytes per 16 columns within it.
    auto kstep = [](int kk) { return static_cast<uint32_t>((kk >> 2) * BOX + 32 * (kk & 3)) >> 4; };
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return mbar_wait_warp(bar, parity, abort_flag, WAIT_TIMEOUT_NS);
    };
    constexpr uint32_t ID_S64 = idesc_ab(BK, 64, false, false);  // N = 64: one query half
    // dV items: S1^T and S2^T of query half h (queries 64 h ..).
    auto issue_s_half = [&](int h) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        umma_bf16_ss_lo_warp(tmem + TM_S + 64 * h, kmaj(V_OFF_K1) + kstep(kk),
                             kmaj(V_OFF_Q1 + 8192 * h) + kstep(kk), dhi, ID_S64, kk > 0);
        umma_bf16_ss_lo_warp(tmem + TM_S2 + 64 * h, kmaj(V_OFF_K2) + kstep(kk),
                             kmaj(V_OFF_Q2 + 8192 * h) + kstep(kk), dhi, ID_S64, kk > 0);
      }
    };
    // dK/dQ items: S^T = K Q^T and dW^T = V dO^T of query half h.
    auto issue_sk_half = [&](int h) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16_ss_lo_warp(tmem + TM_S + 64 * h, kmaj(K_OFF_K) + kstep(kk),
                             kmaj(K_OFF_Q + 8192 * h) + kstep(kk), dhi, ID_S64, kk > 0);
    };
    auto issue_dw_half = [&](int h) {
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk)
        umma_bf16_ss_lo_warp(tmem + TM_W + 64 * h, kmaj(K_OFF_V) + kstep(kk),
                             kmaj(K_OFF_DO + 8192 * h) + kstep(kk), dhi, ID_S64, kk > 0);
    };
    // dK/dQ items: the tile's dW^T and S^T of half h (dO for both halves is
    // already waited for), each half's S^T once that half of the queries landed.
    auto issue_k_front = [&](int it, int h) {
      issue_dw_half(h);
      if (h == 1) umma_commit_warp(&ctrl->do_empty);
      if (!wait_all(&ctrl->q_half_full[h], it & 1)) return false;
      tc_fence_after_sync();
      issue_sk_half(h);
      umma_commit_warp(&ctrl->s_half[h]);
      return true;
    };
    bool ok = wait_all(&ctrl->kv_full, 0);
    tc_fence_after_sync();
    if (ok) {  // the first tile's S^T (and dW^T)
      if (kDV) {
        if ((ok = wait_all(&ctrl->q_full, 0))) {
          tc_fence_after_sync();
          issue_s_half(0);
          umma_commit_warp(&ctrl->s_half[0]);
          issue_s_half(1);
          umma_commit_warp(&ctrl->s_half[1]);
          umma_commit_warp(&ctrl->q_empty);
        }
      } else if ((ok = wait_all(&ctrl->do_full, 0))) {
        tc_fence_after_sync();
        ok = issue_k_front(0, 0) && issue_k_front(0, 1);
      }
    }
    // Per query half h of tile `it`: the half's products, then the next tile's
    // S^T (and dW^T) of that half over the half's packed operand (MMAs run in
    // issue order), while the other half's warps are still busy.
    for (int it = 0; ok && it < w.n_q; ++it) {
      const bool more = it + 1 < w.n_q;
      if (kDV) {
        // dV += W^T dO over the half's queries: A packed in TMEM, B = dO read
        // MN-major (N = 256 in four 64-column blocks); 16 queries = 2048 bytes
        // of each block.
        constexpr uint32_t ID_DV = idesc_ab(BK, DV, false, true);
        for (int h = 0; h < 2; ++h) {
          if (!(ok = wait_all(&ctrl->p_half[h], it & 1))) break;
          tc_fence_after_sync();
          if (h == 0) {
            if (!(ok = wait_all(&ctrl->do_full, it & 1))) break;
            tc_fence_after_sync();
          }
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            umma_bf16_ts_lo_warp(tmem + TM_DV, tmem + TM_S + tm_pack(kk),
                                 mnmaj(V_OFF_DO) + ((2048u * kk) >> 4), dhi, ID_DV,
                                 (it > 0 || kk > 0) ? 1u : 0u);
          if (h == 1) umma_commit_warp(&ctrl->do_empty);
          if (more) {
            if (h == 0) {
              if (!(ok = wait_all(&ctrl->q_full, (it + 1) & 1))) break;
              tc_fence_after_sync();
            }
            issue_s_half(h);
            umma_commit_warp(&ctrl->s_half[h]);
            if (h == 1) umma_commit_warp(&ctrl->q_empty);
          }
        }
      } else {
        constexpr uint32_t ID_DK = idesc_ab(BK, HD, false, true);
        constexpr uint32_t ID_DQ = idesc_ab(BQ, HD, true, true);
        for (int h = 0; h < 2; ++h) {
          if (!(ok = wait_all(&ctrl->p_half[h], it & 1))) break;
          tc_fence_after_sync();
          // dK += dS^T Q over the half's queries: A packed in TMEM, B = Q
          // MN-major (N = 128: two blocks); then that half of Q is free.
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            umma_bf16_ts_lo_warp(tmem + TM_DK, tmem + TM_S + tm_pack(kk),
                                 mnmaj(K_OFF_Q) + ((2048u * kk) >> 4), dhi, ID_DK,
                                 (it > 0 || kk > 0) ? 1u : 0u);
          umma_commit_warp(&ctrl->q_half_empty[h]);
          if (h == 1) {
            // dQ = dS K: A = dS^T read MN-major (M = queries), B = K MN-major
            // (N = d); 16 keys = 2048 bytes of each block.  The previous tile's
            // dQ must have been read before this one overwrites it.
            if (it > 0 && !(ok = wait_all(&ctrl->dq_free, (it - 1) & 1))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16_ss_lo_warp(tmem + TM_DQ, mnmaj(K_OFF_DS) + ((2048u * kk) >> 4),
                                   mnmaj(K_OFF_K) + ((2048u * kk) >> 4), dhi, ID_DQ, kk > 0);
            umma_commit_warp(&ctrl->dq_full);
          }
          if (more) {
            if (h == 0) {
              if (!(ok = wait_all(&ctrl->do_full, (it + 1) & 1))) break;
              tc_fence_after_sync();
            }
            if (!(ok = issue_k_front(it + 1, h))) break;
          }
        }
      }
      if (!ok) break;
    }
    if (ok) umma_commit_warp(&ctrl->acc_done);
    umma_commit_warp(&ctrl->drain);
    drain_wait(&ctrl->drain, 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax warps
    // Warp 4 + 4 ch + q covers TMEM lane quarter q (key rows 32 q ..) and the
    // tile's queries 64 ch .. 64 ch + 63 in four 16-query chunks.
    const int sw = warp - 4;
    const int quarter = warp & 3, ch = sw >> 2;
    const int kr = quarter * 32 + lane;  // key row (dQ drain: query row) = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_lane = tmem + lane_addr;
    const float sl2 = p.scale_log2;
    const int kpos = w.k0 + kr;
    const bool key_ok = kpos < p.N;
    const float lam = p.lambda[w.h];
    const float coef = w.map ? -lam : 1.f;
    const float *vec0 = reinterpret_cast<const float *>(smem + (kDV ? V_OFF_VEC : K_OFF_VEC));
    // dQ of tile `t` (query tile q0) into the fp32 accumulator: this thread's
    // query row, 64 columns, transposed across 8-lane groups so that each vector
    // reduction covers four 128-byte row segments.
    auto drain_dq = [&](int t, int q0) {
      bool okd = mbar_wait(&ctrl->dq_full, t & 1, abort_flag, WAIT_TIMEOUT_NS);
      okd = __all_sync(0xffffffffu, okd);
      if (!okd) return false;
      tc_fence_after_sync();
      uint32_t a[32], b[32];
      tmem_ld_x32_nowait(t_lane + TM_DQ + 64 * ch, a);
      tmem_ld_x32_nowait(t_lane + TM_DQ + 64 * ch + 32, b);
      tmem_ld_wait_x32(a);
      tmem_ld_wait_x32(b);
      tc_fence_before_sync();
      mbar_arrive(&ctrl->dq_free);
      float *dq_base = p.dq_acc + (w.map * p.BH + w.bh) * static_cast<int64_t>(p.N) * HD;
      const int row0 = q0 + quarter * 32 + (lane & ~7);  // the 8-lane group's first row
      float *col_base = dq_base + 64 * ch + 4 * (lane & 7);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t(&src)[32] = half ? b : a;
        uint4 c8[8];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          c8[v] = make_uint4(__float_as_uint(__uint_as_float(src[4 * v]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 1]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 2]) * p.scale),
                             __float_as_uint(__uint_as_float(src[4 * v + 3]) * p.scale));
        transpose8_chunks(c8, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (row0 + j < p.N &&
              dbg_ok(row0 + j >= 0 && 64 * ch + 32 * half + 4 * (lane & 7) + 4 <= HD, p.status,
                     81))
            red_add_v4(col_base + static_cast<int64_t>(row0 + j) * HD + 32 * half,
                       __uint_as_float(c8[j].x), __uint_as_float(c8[j].y),
                       __uint_as_float(c8[j].z), __uint_as_float(c8[j].w));
        }
      }
      return true;
    };
    bool ok = true;
    int prev_q0 = 0;
    for (int it = 0; it < w.n_q; ++it) {
      const int q0 = (w.qt_first + it) * BQ;
      ok = mbar_wait(&ctrl->s_half[ch], it & 1, abort_flag, WAIT_TIMEOUT_NS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const float *vec = vec0 + (it % vec_slots<kDV>()) * (VEC_BYTES / 4);
      // Query column c of the tile (query q0 + c) is visible iff lo <= c < hi.
      const int lo = p.causal ? (kpos - q0) : 0;
      const int hi = key_ok ? (p.N - q0) : 0;
      const bool masked = (q0 + BQ > p.N) || !key_ok || (p.causal && q0 == w.k0);
      // 16 query columns c0 .. c0 + 15 of this thread's key row, packed to bf16
      // pairs; the mask is applied only on tiles that have masked columns.
      auto element_chunk = [&](auto mask_tag, const uint32_t(&x)[16], const uint32_t(&y)[16],
                               int c0, uint32_t(&pk)[8]) {
        constexpr bool kMask = decltype(mask_tag)::value;
        const float2 scale = make_float2(sl2, sl2);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 la4 = *reinterpret_cast<const float4 *>(vec + c0 + i);
          const float4 lb4 = *reinterpret_cast<const float4 *>(vec + BQ + c0 + i);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k = i + 2 * h;
            const float2 la = h ? make_float2(la4.z, la4.w) : make_float2(la4.x, la4.y);
            const float2 lb = h ? make_float2(lb4.z, lb4.w) : make_float2(lb4.x, lb4.y);
            const float2 sx = make_float2(__uint_as_float(x[k]), __uint_as_float(x[k + 1]));
            const float2 sy = make_float2(__uint_as_float(y[k]), __uint_as_float(y[k + 1]));
            float2 r;
            if (kDV) {
              // W^T = P1^T - lambda P2^T, each P from its map's log2-sum-exp.
              const float2 e1 = __ffma2_rn(sx, scale, make_float2(-la.x, -la.y));
              const float2 e2 = __ffma2_rn(sy, scale, make_float2(-lb.x, -lb.y));
              r = __ffma2_rn(make_float2(ex2_approx(e2.x), ex2_approx(e2.y)),
                             make_float2(-lam, -lam),
                             make_float2(ex2_approx(e1.x), ex2_approx(e1.y)));
            } else {
              // dS^T = P^T (c dW^T - c D).
              const float2 e = __ffma2_rn(sx, scale, make_float2(-la.x, -la.y));
              const float2 t = __ffma2_rn(sy, make_float2(coef, coef), make_float2(-lb.x, -lb.y));
              r = __fmul2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), t);
            }
            if (kMask) {
              const int q = c0 + k;
              r.x = (q >= lo && q < hi) ? r.x : 0.f;
              r.y = (q + 1 >= lo && q + 1 < hi) ? r.y : 0.f;
            }
            pk[k / 2] = pack_bf16x2(r.x, r.y);
          }
        }
      };
      uint32_t pks[4][8];  // the half's packed operand, kept for the shared-memory copy
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int c0 = 64 * ch + 16 * c;  // first query column of the chunk
        uint32_t x[16], y[16];
        tmem_ld16(t_lane + TM_S + c0, x);
        tmem_ld16(t_lane + (kDV ? TM_S2 : TM_W) + c0, y);
        tmem_wait16x2(x, y);
        if (masked)
          element_chunk(std::true_type{}, x, y, c0, pks[c]);
        else
          element_chunk(std::false_type{}, x, y, c0, pks[c]);
        // Packed over this thread's own, already read S^T columns.
        tmem_st8(t_lane + TM_S + 64 * ch + 8 * c, pks[c]);
      }
      tmem_st_wait();
      if (!kDV) {
        // dS^T rows in shared memory for dQ (this half's 64 queries of key row
        // kr), once the previous tile's dQ product has read the buffer: the
        // first half runs ahead of that product.
        if (it > 0) {
          ok = mbar_wait(&ctrl->dq_full, (it - 1) & 1, abort_flag, WAIT_TIMEOUT_NS);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        uint8_t *sub = smem + K_OFF_DS + ch * BOX;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4 *>(sub + sw128(kr, 2 * c + j)) =
                make_uint4(pks[c][4 * j], pks[c][4 * j + 1], pks[c][4 * j + 2], pks[c][4 * j + 3]);
        fence_proxy_async_smem();
      }
      tc_fence_before_sync();
      mbar_arrive(&ctrl->p_half[ch]);
      if (!kDV && it > 0 && !(ok = drain_dq(it - 1, prev_q0))) break;
      prev_q0 = q0;
    }
    if (!kDV && ok && w.n_q > 0) ok = drain_dq(w.n_q - 1, prev_q0);
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&ctrl->acc_done, 0, abort_flag, WAIT_TIMEOUT_NS);
    ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
    if (ok) {
      tc_fence_after_sync();
      const int64_t krow = kpos;
      if (kDV) {
        // This thread's key row, value columns 128 ch .. 128 ch + 127.
        __nv_bfloat16 *dst = p.dv + w.b * p.dv_sb + w.h * p.dv_sh + krow * p.dv_sn + 128 * ch;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32_nowait(t_lane + TM_DV + 128 * ch + c0, v);
          tmem_ld_wait_x32(v);
          if (key_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
              *reinterpret_cast<uint4 *>(dst + c0 + 8 * q) = o;
            }
          }
        }
      } else {
        // This thread's key row, d columns 64 ch .. 64 ch + 63, times 1/sqrt(d).
        const int m = w.map;
        __nv_bfloat16 *dst = (m ? p.dk2 : p.dk1) + w.b * (m ? p.dk_sb[1] : p.dk_sb[0]) +
                             w.h * (m ? p.dk_sh[1] : p.dk_sh[0]) +
                             krow * (m ? p.dk_sn[1] : p.dk_sn[0]) + 64 * ch;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32_nowait(t_lane + TM_DK + 64 * ch + c0, v);
          tmem_ld_wait_x32(v);
          if (key_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * q]) * p.scale,
                                __uint_as_float(v[8 * q + 1]) * p.scale);
              o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * p.scale,
                                __uint_as_float(v[8 * q + 3]) * p.scale);
              o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * p.scale,
                                __uint_as_float(v[8 * q + 5]) * p.scale);
              o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * p.scale,
                                __uint_as_float(v[8 * q + 7]) * p.scale);
              *reinterpret_cast<uint4 *>(dst + c0 + 8 * q) = o;
            }
          }
        }
      }
    }
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

// ---------------------------------------------------------------- preprocess
// One warp per row, lane = 8 value columns: do (bf16 for the tensor cores),
// c_k D_k = c_k bf16(do) . o_k, and per-head dlambda and dw (block reduction,
// one atomic per head and column).  The d = 64 preprocess with 256 columns.
struct PreParams {
  int64_t BH;
  int32_t H, N, n_pad, headnorm;
  float eps, out_scale;  // out_scale = 1 - lambda_init
  const float *lambda, *norm_w;
  const __nv_bfloat16 *dy;  // [B, H, N, 256] view
  int64_t dy_sb, dy_sh, dy_sn;
  const float *o_n;          // [2][BH][N][256]: o = o_1 - lambda o_2, then o_2
  __nv_bfloat16 *dout;       // [BH][N][256]
  float *dvec;               // [2][BH][n_pad] c_k D_k
  float *dlambda;            // [H], zeroed
  float *dnorm_w;            // [H][256], zeroed
};

constexpr int PRE_WARPS = 8;
constexpr int PRE_ROWS = 64;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16 *src, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(src);
  const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[j]));
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

__device__ __forceinline__ void load8_f32(const float *src, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(src);
  const float4 b = *reinterpret_cast<const float4 *>(src + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__global__ void __launch_bounds__(PRE_WARPS * 32) diffattn_bwd_pre_d128_kernel(const PreParams p) {
  __shared__ float red_w[PRE_WARPS][DV];
  __shared__ float red_l[PRE_WARPS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t bh = blockIdx.x;
  const int h = static_cast<int>(bh % p.H);
  const int c = 8 * lane;
  const float lam = p.lambda[h];
  float g[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = p.out_scale * (p.norm_w ? p.norm_w[h * DV + c + j] : 1.f);
  float acc_w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float acc_l = 0.f;
  const int64_t plane = p.BH * static_cast<int64_t>(p.N) * DV;
  const __nv_bfloat16 *dy_bh = p.dy + (bh / p.H) * p.dy_sb + h * p.dy_sh;
  for (int i = blockIdx.y * PRE_ROWS + warp; i < (blockIdx.y + 1) * PRE_ROWS; i += PRE_WARPS) {
    if (i >= p.n_pad) break;
    float d1 = 0.f, d2 = 0.f;
    if (i < p.N) {
      const int64_t row = (bh * p.N + i) * DV + c;
      float dy[8], o1[8], o2[8], o[8], dout[8];
      load8_bf16(dy_bh + i * p.dy_sn + c, dy);
      load8_f32(p.o_n + row, o);
      load8_f32(p.o_n + plane + row, o2);
#pragma unroll
      for (int j = 0; j < 8; ++j) o1[j] = fmaf(lam, o2[j], o[j]);
      if (p.headnorm) {
        if (p.headnorm == 2) {
          float sm = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) sm += o[j];
          const float mu = warp_sum(sm) * (1.f / DV);
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] -= mu;
        }
        float ms = 0.f, t = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          ms = fmaf(o[j], o[j], ms);
          t = fmaf(dy[j] * g[j], o[j], t);
        }
        ms = warp_sum(ms) * (1.f / DV);
        t = warp_sum(t);
        const float r = rsqrtf(ms + p.eps);
        const float r3 = r * r * r * (1.f / DV);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          dout[j] = r * g[j] * dy[j] - r3 * o[j] * t;
          acc_w[j] = fmaf(dy[j] * o[j], r * p.out_scale, acc_w[j]);
        }
        if (p.headnorm == 2) {
          float sd = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) sd += dout[j];
          const float md = warp_sum(sd) * (1.f / DV);
#pragma unroll
          for (int j = 0; j < 8; ++j) dout[j] -= md;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) dout[j] = dy[j];
      }
      // dlambda uses do as computed; D_k the bf16 do the tensor cores see.
      float l2 = 0.f;
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 bb = __floats2bfloat162_rn(dout[2 * j], dout[2 * j + 1]);
        pk[j] = *reinterpret_cast<const uint32_t *>(&bb);
        const float2 rr = __bfloat1622float2(bb);
        l2 = fmaf(dout[2 * j], o2[2 * j], fmaf(dout[2 * j + 1], o2[2 * j + 1], l2));
        d1 = fmaf(rr.x, o1[2 * j], fmaf(rr.y, o1[2 * j + 1], d1));
        d2 = fmaf(rr.x, o2[2 * j], fmaf(rr.y, o2[2 * j + 1], d2));
      }
      *reinterpret_cast<uint4 *>(p.dout + row) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      acc_l -= warp_sum(l2);
      d1 = warp_sum(d1);
      d2 = warp_sum(d2);
    }
    if (lane == 0) {  // c_k D_k: c_1 = 1, c_2 = -lambda
      p.dvec[bh * p.n_pad + i] = d1;
      p.dvec[(p.BH + bh) * p.n_pad + i] = -lam * d2;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red_w[warp][c + j] = acc_w[j];
  if (lane == 0) red_l[warp] = acc_l;
  __syncthreads();
  if (p.headnorm && p.dnorm_w != nullptr) {
    for (int col = threadIdx.x; col < DV; col += blockDim.x) {
      float s = 0.f;
      for (int w2 = 0; w2 < PRE_WARPS; ++w2) s += red_w[w2][col];
      atomicAdd(p.dnorm_w + h * DV + col, s);
    }
  }
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w2 = 0; w2 < PRE_WARPS; ++w2) s += red_l[w2];
    atomicAdd(p.dlambda + h, s);
  }
}

// ---------------------------------------------------------------- dq to bf16
// dq_acc [2][BH][N][128] -> dq1, dq2 ([B, H, N, 128] views), four columns per thread.
__global__ void diffattn_bwd_finish_d128_kernel(const float *dq_acc, __nv_bfloat16 *dq1,
                                                __nv_bfloat16 *dq2, int64_t BH, int64_t H,
                                                int64_t N, int64_t sb0, int64_t sh0, int64_t sn0,
                                                int64_t sb1, int64_t sh1, int64_t sn1) {
  const int64_t per_map = BH * N * (HD / 4);
  const int64_t total = 2 * per_map;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4 *>(dq_acc)[i];
    const int t = i >= per_map;
    const int64_t j = i - t * per_map;
    const int64_t row = j / (HD / 4), col = 4 * (j - row * (HD / 4));
    const int64_t bh = row / N, n = row - bh * N;
    const int64_t b = bh / H, h = bh - b * H;
    __nv_bfloat16 *dst = t ? dq2 + b * sb1 + h * sh1 + n * sn1 : dq1 + b * sb0 + h * sh0 + n * sn0;
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(dst + col) = o;
  }
}

using EncodeTiledFnD = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

// 4-D view {inner, rows, H, B} of a bf16 tensor with element strides st (rows
// contiguous); box_rows x 64-column boxes with 128-byte swizzle.
CUresult encode_map_d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t n, uint64_t H,
                      uint64_t B, const diffattn_strides &st, uint32_t box_rows) {
  static EncodeTiledFnD fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFnD>(ptr);
  }();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[4] = {inner, n, H, B};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}


// ---------------------------------------------------------------- map output from saved statistics
// o_k = map_k V of one map given its log2-sum-exp (the saving forward's second
// pass): o_k[q] = sum_j 2^(S[q, j] log2e / sqrt(d) - lse[q]) v_j.  One CTA per
// (128-query tile, head), heaviest tile first; queries on the TMEM lanes, S
// double-buffered (columns 0-255) so that the element work on key tile j
// overlaps S of tile j + 1 and P V of tile j - 1, O in columns 256-511; K and
// V double-buffered in shared memory.  Warps: producer, MMA issuer, 2 idle, 8
// element warps (warp 4 + 4 ch + q: lane quarter q, keys 64 ch .. of a tile).
// K is released once S has read it and V once P V has, so K of tile j + 2
// streams in while tile j's P V waits for its softmax.
constexpr uint32_t M_OFF_Q = 0, M_OFF_K = 2 * BOX, M_OFF_V = 6 * BOX, M_OFF_VEC = 14 * BOX;
constexpr uint32_t M_OFF_CTRL = M_OFF_VEC + BQ * 4;
constexpr uint32_t TM_O = 256;

struct MapCtrl {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];  // K of a key tile: released once S has read it
  uint64_t v_full[2], v_empty[2];  // V of a key tile: released once P V has read it
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t MAP_SMEM_BYTES = M_OFF_CTRL + static_cast<uint32_t>(sizeof(MapCtrl)) + 1024;
static_assert(MAP_SMEM_BYTES <= 232448, "shared memory budget exceeded");

struct MapParams {
  int64_t BH;
  int32_t H, N, n_qtiles, causal;
  float scale_log2;
  const float *lse;  // [BH][n_pad] this map's log2-sum-exp
  float *out;        // [BH][N][256] fp32
  int32_t *status;
};

__global__ void __launch_bounds__(384, 1)
    diffattn_map_out_d128_kernel(const __grid_constant__ CUtensorMap tm_q,
                                 const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v, const MapParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  MapCtrl *ctrl = reinterpret_cast<MapCtrl *>(smem + M_OFF_CTRL);
  volatile int *abort_flag = &ctrl->abort;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t n_bh = static_cast<uint32_t>(p.BH);
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x / n_bh);
  const uint32_t bh32 = blockIdx.x % n_bh;
  const int64_t bh = bh32;
  const int hh = static_cast<int>(bh32 % static_cast<uint32_t>(p.H));
  const int bb = static_cast<int>(bh32 / static_cast<uint32_t>(p.H));
  const int q0 = qt * BQ;
  const int n_kv = p.causal ? qt + 1 : p.n_qtiles;  // key tiles of 128 keys
  const int64_t n_pad = static_cast<int64_t>(p.n_qtiles) * BQ;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctrl->k_full[s], 1);
      mbar_init(&ctrl->k_empty[s], 1);
      mbar_init(&ctrl->v_full[s], 1);
      mbar_init(&ctrl->v_empty[s], 1);
      mbar_init(&ctrl->s_full[s], 1);
      mbar_init(&ctrl->p_ready[s], SOFTMAX_THREADS);
    }
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->drain, 1);
    ctrl->abort = 0;
    fence_barrier_init();
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
      int loaded = 0;  // key tiles whose loads were issued
      mbar_arrive_expect_tx(&ctrl->q_full, 2 * BOX + BQ * 4);
      for (int x = 0; x < 2; ++x)
        tma_load_4d(smem + M_OFF_Q + x * BOX, &tm_q, &ctrl->q_full, 64 * x, q0, hh, bb);
      bulk_g2s(smem + M_OFF_VEC, p.lse + bh * n_pad + q0, BQ * 4, &ctrl->q_full);
      int loaded_v = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t par = static_cast<uint32_t>((j >> 1) - 1) & 1u;
        if (j >= 2 && !mbar_wait(&ctrl->k_empty[s], par, abort_flag, WAIT_TIMEOUT_NS)) break;
        mbar_arrive_expect_tx(&ctrl->k_full[s], 2 * BOX);
        for (int x = 0; x < 2; ++x)
          tma_load_4d(smem + M_OFF_K + (2 * s + x) * BOX, &tm_k, &ctrl->k_full[s], 64 * x,
                      j * BK, hh, bb);
        loaded = j + 1;
        if (j >= 2 && !mbar_wait(&ctrl->v_empty[s], par, abort_flag, WAIT_TIMEOUT_NS)) break;
        mbar_arrive_expect_tx(&ctrl->v_full[s], 4 * BOX);
        for (int x = 0; x < 4; ++x)
          tma_load_4d(smem + M_OFF_V + (4 * s + x) * BOX, &tm_v, &ctrl->v_full[s], 64 * x,
                      j * BK, hh, bb);
        loaded_v = j + 1;
      }
      // Loads still in flight land before the CTA exits: the last tile issued
      // into each buffer (tile t completes phase t >> 1 of buffer t & 1).
      drain_wait(&ctrl->q_full, 0);
      for (int t = loaded - 2; t < loaded; ++t)
        if (t >= 0) drain_wait(&ctrl->k_full[t & 1], (t >> 1) & 1);
      for (int t = loaded_v - 2; t < loaded_v; ++t)
        if (t >= 0) drain_wait(&ctrl->v_full[t & 1], (t >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
    const uint32_t base = smem_u32(smem);
    const uint32_t dhi = static_cast<uint32_t>(smem_desc_sw128(base, 16, 1024) >> 32);
    auto kmaj = [&](uint32_t off) { return lo(smem_desc_sw128(base + off, 16, 1024)); };
    auto mnmaj = [&](uint32_t off) { return lo(smem_desc_sw128(base + off, BOX, 1024)); };
    auto kstep = [](int kk) { return static_cast<uint32_t>((kk >> 2) * BOX + 32 * (kk & 3)) >> 4; };
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return mbar_wait_warp(bar, parity, abort_flag, WAIT_TIMEOUT_NS);
    };
    constexpr uint32_t ID_S = idesc_ab(BQ, BK, false, false);   // S = Q K^T, both K-major
    constexpr uint32_t ID_PV = idesc_ab(BQ, DV, false, true);   // O += P V, V MN-major
    // S of key tile j into buffer j & 1, once K_j has landed.
    auto issue_s = [&](int j) {
      const int s = j & 1;
      if (!wait_all(&ctrl->k_full[s], (j >> 1) & 1)) return false;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16_ss_lo_warp(tmem + 128 * s, kmaj(M_OFF_Q) + kstep(kk),
                             kmaj(M_OFF_K + 2 * s * BOX) + kstep(kk), dhi, ID_S, kk > 0);
      umma_commit_warp(&ctrl->k_empty[s]);
      umma_commit_warp(&ctrl->s_full[s]);
      return true;
    };
    bool ok = wait_all(&ctrl->q_full, 0);
    tc_fence_after_sync();
    if (ok) ok = issue_s(0);
    if (ok && n_kv > 1) ok = issue_s(1);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1;
      if (!(ok = wait_all(&ctrl->p_ready[s], (j >> 1) & 1))) break;
      if (!(ok = wait_all(&ctrl->v_full[s], (j >> 1) & 1))) break;
      tc_fence_after_sync();
      // O += P V: A = packed P in TMEM over buffer s, B = V_j MN-major (N = 256
      // in four 64-column blocks); 16 keys = 2048 bytes of each block.
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        umma_bf16_ts_lo_warp(tmem + TM_O, tmem + 128 * s + tm_pack(kk),
                             mnmaj(M_OFF_V + 4 * s * BOX) + ((2048u * kk) >> 4), dhi, ID_PV,
                             (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit_warp(&ctrl->v_empty[s]);
      // S of tile j + 2 goes over this tile's packed P: MMAs run in issue order.
      if (j + 2 < n_kv && !(ok = issue_s(j + 2))) break;
    }
    if (ok) umma_commit_warp(&ctrl->o_done);
    umma_commit_warp(&ctrl->drain);
    drain_wait(&ctrl->drain, 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- element warps
    const int sw = warp - 4;
    const int quarter = warp & 3, ch = sw >> 2;
    const int r = quarter * 32 + lane;  // query row in the tile = TMEM lane
    const int qpos = q0 + r;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag, WAIT_TIMEOUT_NS);
    ok = __all_sync(0xffffffffu, ok);
    const float neg_lse = ok ? -reinterpret_cast<const float *>(smem + M_OFF_VEC)[r] : 0.f;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1;
      ok = mbar_wait(&ctrl->s_full[s], (j >> 1) & 1, abort_flag, WAIT_TIMEOUT_NS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int k0 = j * BK;
      // Key column c of the tile (key k0 + c) is visible iff c < hi.
      const int hi = min(p.N - k0, p.causal ? qpos - k0 + 1 : BK);
      const bool masked = (k0 + BK > p.N) || (p.causal && j == qt);
      const float2 scale = make_float2(sl2, sl2), nl2 = make_float2(neg_lse, neg_lse);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int c0 = 64 * ch + 16 * c;
        uint32_t x[16];
        tmem_ld16(t_lane + 128 * s + c0, x);
        tmem_wait16x2(x, x);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float2 e = __ffma2_rn(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])),
                                      scale, nl2);
          float pa = ex2_approx(e.x), pb = ex2_approx(e.y);
          if (masked) {
            pa = (c0 + i < hi) ? pa : 0.f;
            pb = (c0 + i + 1 < hi) ? pb : 0.f;
          }
          pk[i / 2] = pack_bf16x2(pa, pb);
        }
        // Packed over this thread's own, already read S columns.
        tmem_st8(t_lane + 128 * s + 64 * ch + 8 * c, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&ctrl->p_ready[s]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&ctrl->o_done, 0, abort_flag, WAIT_TIMEOUT_NS);
    ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
    if (ok) {
      tc_fence_after_sync();
      // This thread's query row, value columns 128 ch .. 128 ch + 127, stored
      // transposed across 8-lane groups (four 128-byte row segments per store).
      const int row0 = q0 + quarter * 32 + (lane & ~7);
      float *col_base = p.out + bh * static_cast<int64_t>(p.N) * DV + 128 * ch + 4 * (lane & 7);
#pragma unroll 1
      for (int c32 = 0; c32 < 128; c32 += 32) {
        uint32_t v[32];
        tmem_ld_x32_nowait(t_lane + TM_O + 128 * ch + c32, v);
        tmem_ld_wait_x32(v);
        uint4 c8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) c8[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        transpose8_chunks(c8, lane);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          if (row0 + jj < p.N &&
              dbg_ok(row0 + jj >= 0 && 128 * ch + c32 + 4 * (lane & 7) + 4 <= DV, p.status, 84))
            *reinterpret_cast<uint4 *>(col_base + static_cast<int64_t>(row0 + jj) * DV + c32) =
                c8[jj];
      }
    }
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

int64_t r256(int64_t bytes) { return (bytes + 255) / 256 * 256; }

}  // namespace

int64_t saved_bytes_d128(int64_t BH, int64_t N) {
  const int64_t n_pad = (N + BQ - 1) / BQ * BQ;
  return r256(2 * BH * N * DV * 4) + r256(2 * BH * n_pad * 4);
}

int64_t bwd_workspace_bytes_d128(int64_t BH, int64_t N) {
  const int64_t n_pad = (N + BQ - 1) / BQ * BQ;
  // dO bf16 [BH][N][256], c_k D_k [2][BH][n_pad], dq_acc [2][BH][N][128]
  return r256(BH * N * DV * 2) + r256(2 * BH * n_pad * 4) + r256(2 * BH * N * HD * 4);
}

diffattn_status launch_fwd_train_d128(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, void *out,
                                      void *saved, cudaStream_t stream,
                                      const diffattn_strides *strides) {
  const int64_t BH = desc.B * desc.H, N = desc.N;
  uint8_t *sv = static_cast<uint8_t *>(saved);
  float *o1 = reinterpret_cast<float *>(sv);
  float *o2 = o1 + BH * N * DV;
  float *lse = reinterpret_cast<float *>(sv + r256(2 * BH * N * DV * 4));
  // The output, each map's log2-sum-exp and the pre-norm o = o_1 - lambda o_2.
  diffattn_status st = launch_fwd_d128_sm103(desc, N, q1, k1, q2, k2, v, lambda, norm_w, out,
                                             stream, strides, lse, o1);
  if (st != DIFFATTN_OK) return st;
  // Map 2's output alone, from its saved log2-sum-exp: one pass over the keys.
  const int64_t n_qtiles = (N + BQ - 1) / BQ;
  if (BH * n_qtiles > INT32_MAX || desc.H > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
  const diffattn_strides cont64{desc.H * N * HD, N * HD, HD}, cont256{desc.H * N * DV, N * DV, DV};
  CUtensorMap maps[3];
  const void *bases[3] = {q2, k2, v};
  for (int i = 0; i < 3; ++i) {
    const diffattn_strides sti = strides ? strides[i == 2 ? 4 : 2 + i] : (i == 2 ? cont256 : cont64);
    if (encode_map_d(&maps[i], bases[i], i == 2 ? DV : HD, static_cast<uint64_t>(N),
                     static_cast<uint64_t>(desc.H), static_cast<uint64_t>(desc.B), sti, 128u) !=
        CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(diffattn_map_out_d128_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(MAP_SMEM_BYTES)) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  MapParams mp;
  mp.BH = BH;
  mp.H = static_cast<int32_t>(desc.H);
  mp.N = static_cast<int32_t>(N);
  mp.n_qtiles = static_cast<int32_t>(n_qtiles);
  mp.causal = desc.causal ? 1 : 0;
  mp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  mp.lse = lse + BH * n_qtiles * BQ;  // map 2's rows
  mp.out = o2;
  mp.status = desc.status_dev;
  diffattn_map_out_d128_kernel<<<static_cast<unsigned>(BH * n_qtiles), 384, MAP_SMEM_BYTES,
                                 stream>>>(maps[0], maps[1], maps[2], mp);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

diffattn_status launch_bwd_d128_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, const void *saved,
                                      const void *dy, void *dq1, void *dk1, void *dq2, void *dk2,
                                      void *dv, float *dlambda, float *dnorm_w, void *workspace,
                                      cudaStream_t stream, const diffattn_strides *strides) {
  const int64_t BH = desc.B * desc.H, N = desc.N;
  const int64_t n_qtiles = (N + BQ - 1) / BQ;
  const int64_t n_pad = n_qtiles * BQ;
  if (2 * BH * n_qtiles > INT32_MAX || N > INT32_MAX / 2 || desc.H > INT32_MAX)
    return DIFFATTN_ERR_UNSUPPORTED;
  // Element strides of q1, k1, q2, k2, v, dy, dq1, dk1, dq2, dk2, dv.
  diffattn_strides st[kBwdStrides];
  for (int i = 0; i < kBwdStrides; ++i) {
    const int64_t width = (i == 4 || i == 5 || i == 10) ? DV : HD;
    st[i] = strides ? strides[i] : diffattn_strides{desc.H * N * width, N * width, width};
  }
  const uint8_t *sv = static_cast<const uint8_t *>(saved);
  const float *o_n = reinterpret_cast<const float *>(sv);
  const float *lse = reinterpret_cast<const float *>(sv + r256(2 * BH * N * DV * 4));
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  __nv_bfloat16 *dout = reinterpret_cast<__nv_bfloat16 *>(ws);
  float *dvec = reinterpret_cast<float *>(ws + r256(BH * N * DV * 2));
  float *dq_acc = reinterpret_cast<float *>(ws + r256(BH * N * DV * 2) + r256(2 * BH * n_pad * 4));

  if (cudaMemsetAsync(dq_acc, 0, sizeof(float) * (2 * BH * N * HD), stream) != cudaSuccess ||
      cudaMemsetAsync(dlambda, 0, sizeof(float) * desc.H, stream) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;
  if (desc.headnorm && dnorm_w != nullptr &&
      cudaMemsetAsync(dnorm_w, 0, sizeof(float) * desc.H * DV, stream) != cudaSuccess)
    return DIFFATTN_ERR_CUDA;

  PreParams pp;
  pp.BH = BH;
  pp.H = static_cast<int32_t>(desc.H);
  pp.N = static_cast<int32_t>(N);
  pp.n_pad = static_cast<int32_t>(n_pad);
  pp.headnorm = desc.headnorm;
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
  diffattn_bwd_pre_d128_kernel<<<pre_grid, PRE_WARPS * 32, 0, stream>>>(pp);
  if (cudaGetLastError() != cudaSuccess) return DIFFATTN_ERR_CUDA;

  // q1, k1, q2, k2, v, dO in 128-row boxes; q1 and q2 again in 64-row boxes
  // (the dK/dQ items load each half of a query tile on its own).
  CUtensorMap maps[8];
  const void *bases[8] = {q1, k1, q2, k2, v, dout, q1, q2};
  const diffattn_strides dout_st{desc.H * N * DV, N * DV, DV};
  for (int i = 0; i < 8; ++i) {
    const uint64_t inner = (i == 4 || i == 5) ? DV : HD;
    const diffattn_strides &sti = i == 5 ? dout_st : i == 6 ? st[0] : i == 7 ? st[2] : st[i];
    if (encode_map_d(&maps[i], bases[i], inner, static_cast<uint64_t>(N),
                     static_cast<uint64_t>(desc.H), static_cast<uint64_t>(desc.B), sti,
                     i >= 6 ? 64u : 128u) != CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(diffattn_bwd_d128_sm103_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<true>())) != cudaSuccess ||
        cudaFuncSetAttribute(diffattn_bwd_d128_sm103_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<false>())) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  Params p;
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
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.dv_sb = st[10].b;
  p.dv_sh = st[10].h;
  p.dv_sn = st[10].n;
  p.dk1 = static_cast<__nv_bfloat16 *>(dk1);
  p.dk2 = static_cast<__nv_bfloat16 *>(dk2);
  for (int m = 0; m < 2; ++m) {  // dk1: strides[7], dk2: strides[9]
    p.dk_sb[m] = st[7 + 2 * m].b;
    p.dk_sh[m] = st[7 + 2 * m].h;
    p.dk_sn[m] = st[7 + 2 * m].n;
  }
  p.dq_acc = dq_acc;
  p.status = desc.status_dev;
  diffattn_bwd_d128_sm103_kernel<true>
      <<<static_cast<unsigned>(BH * n_qtiles), NUM_THREADS, smem_bytes<true>(), stream>>>(
          maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], p);
  if (cudaGetLastError() != cudaSuccess) return DIFFATTN_ERR_CUDA;
  diffattn_bwd_d128_sm103_kernel<false>
      <<<static_cast<unsigned>(2 * BH * n_qtiles), NUM_THREADS, smem_bytes<false>(), stream>>>(
          maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], p);
  if (cudaGetLastError() != cudaSuccess) return DIFFATTN_ERR_CUDA;
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  diffattn_bwd_finish_d128_kernel<<<4 * sms, 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16 *>(dq1), static_cast<__nv_bfloat16 *>(dq2), BH, desc.H,
      N, st[6].b, st[6].h, st[6].n, st[8].b, st[8].h, st[8].n);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
