// Fused differential-attention head forward for query/key halves of width
// d = 128 (values and output 2d = 256 wide), bf16 in / bf16 out, fp32
// accumulation, on sm_103a.
//
// The method is the one of the d = 64 kernel ("Differential Transformer",
// Ultralytics glossary, section "How differential attention works": two
// softmax maps, (map1 - lambda map2) V, per-head norm, (1 - lambda_init)).
// With 256 value columns, one fp32 accumulator per map (2 x 256 TMEM
// columns) would fill tensor memory, so this kernel makes two passes over the
// keys of a 128-row query tile and keeps a single accumulator:
//
//   pass 1, per 128-key tile:  S1 = Q1 K1^T, S2 = Q2 K2^T  (tcgen05, K = 128)
//            exact online row maxima m_k and sums l_k of 2^(S_k log2e/sqrt(d))
//   pass 2, per 128-key tile:  S1, S2 again;
//            P = 2^(x1 - m1) / l1 - lambda 2^(x2 - m2) / l2   (final weights)
//            O += P V   (one TS MMA per 16 keys, N = 256, P read from TMEM)
//
// Each map is an ordinary softmax, so after pass 1 the normalisers are final
// and pass 2 needs no rescaling: O is the raw output o directly.  The price is
// the second S and the second set of exponentials.  Tiles are 128 keys wide
// because an MMA with N = 64 takes nearly as long to issue as one with N = 128.
//
// Tensor memory (512 columns) changes layout between the passes:
//   pass 1: S1 / S2 double-buffered, buffer b at 256 b (S1) and 256 b + 128 (S2)
//   pass 2: S1 at 0, S2 at 128 (single), O at 256-511
// P of a pass-2 tile is written as packed bf16 over S1 (keys 0-63 at columns
// 0-31, keys 64-127 at 64-95, each over columns its writers have just read).
// Shared memory holds Q1, Q2 (64 KB) and two 64 KB halves: in pass 1 each
// half is a stage of K1, K2; in pass 2 half 0 holds K1, K2 and half 1 holds V,
// each released as soon as its MMA has read it.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer, warps 4-7 and 8-11 two warpgroups (thread = query row = TMEM
// lane).  Pass 1: group g keeps the statistics of map g + 1.  Pass 2: group g
// forms P for keys 64g .. 64g+63 of both maps.  Epilogue: group g normalises
// and stores output columns 128g .. 128g+127.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include <cmath>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per key tile
constexpr int HD = 128;   // query/key half width d
constexpr int DV = 256;   // value width 2d
constexpr int NUM_THREADS = 384;

constexpr uint32_t BOX = 128 * 64 * 2;   // one [128 rows x 64 columns] bf16 box: 16 KB
constexpr uint32_t OFF_Q1 = 0;           // two boxes
constexpr uint32_t OFF_Q2 = 2 * BOX;
constexpr uint32_t OFF_HALF = 4 * BOX;   // two halves of HALF_BYTES
constexpr uint32_t HALF_BYTES = 4 * BOX; // K1 + K2 (two boxes each), or V (four boxes)
constexpr uint32_t OFF_CTRL = OFF_HALF + 2 * HALF_BYTES;

struct Ctrl {
  uint64_t q_full;
  uint64_t kv_full[2];   // per shared-memory half
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t s_done[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float xch[6][BM];  // pass-1 statistics and epilogue partial sums
};

constexpr uint32_t SMEM_BYTES = OFF_CTRL + sizeof(Ctrl) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(SMEM_BYTES + 1024 < (1u << 18), "descriptor start addresses must stay below 256 KB");

// S_k (k = 0, 1) of tile t: pass 1 double-buffers, pass 2 has one buffer at 0.
__host__ __device__ constexpr uint32_t tm_s(int k, bool pass2, int t) {
  return (pass2 ? 0u : 256u * static_cast<uint32_t>(t & 1)) + 128u * static_cast<uint32_t>(k);
}
constexpr uint32_t TM_O = 256;

constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr uint64_t DRAIN_TIMEOUT_NS = 200000000ull;

struct Params {
  int64_t BH;
  int32_t H, N, n_qtiles, n_ktiles, causal, headnorm;
  int32_t N_kv;   // key/value rows per head
  int32_t q_off;  // sequence position of query row 0 (N_kv - N): causal alignment
  float scale_log2, eps, out_scale;
  const float *lambda;
  const float *norm_w;
  __nv_bfloat16 *out;
  int32_t *status;
  int64_t out_sb, out_sh, out_sn;  // element strides of `out` (rows of 256 contiguous)
  // Training: each map's log2-sum-exp m_k + log2 l_k per row (fp32
  // [2][BH][128 * n_qtiles]) when non-null.
  float *save_lse;
  // Training: the row's o = o_1 - lambda o_2 before the norm, fp32
  // (contiguous [BH][N][256]), when non-null.
  float *o_save;
};

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > DRAIN_TIMEOUT_NS) return false;
  }
  return true;
}

// kTrain: the saving forward's instantiation (save_lse, o_save); the plain
// forward's has neither path.
template <bool kTrain>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    diffattn_fwd_d128_sm103_kernel(const __grid_constant__ CUtensorMap tm_q1,
                                   const __grid_constant__ CUtensorMap tm_k1,
                                   const __grid_constant__ CUtensorMap tm_q2,
                                   const __grid_constant__ CUtensorMap tm_k2,
                                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + OFF_CTRL);
  volatile int *abort_flag = &ctrl->abort;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // Heaviest query tiles first (32-bit decode: the grid is below 2^31 CTAs).
  const uint32_t BH32 = static_cast<uint32_t>(p.BH), H32 = static_cast<uint32_t>(p.H);
  const uint32_t item = blockIdx.x;
  const int qt = p.n_qtiles - 1 - static_cast<int>(item / BH32);
  const uint32_t bh32 = item % BH32;
  const int64_t bh = bh32;
  const int h = static_cast<int>(bh32 % H32);
  const int b_idx = static_cast<int>(bh32 / H32);
  const int q0 = qt * BM;
  // Key tiles this query tile sees: all, or up to the one holding the position
  // of its last row (queries are the last N of N_kv positions).
  const int n_kv = p.causal ? min(p.n_ktiles, (p.q_off + q0 + BM - 1) / BN + 1) : p.n_ktiles;
  const int T = 2 * n_kv;  // tiles over both passes

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(&ctrl->kv_full[hf], 1);
      mbar_init(&ctrl->kv_empty[hf], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->s_full[b], 1);
      mbar_init(&ctrl->s_done[b], 256);
    }
    mbar_init(&ctrl->o_done, 1);
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
    // Shared-memory half hf is filled once per use: pass-1 tile t uses half
    // t & 1 (K1, K2); a pass-2 tile uses half 0 (K1, K2) and half 1 (V).
    if (lane == 0) {
      uint32_t uses[2] = {0, 0};
      mbar_arrive_expect_tx(&ctrl->q_full, 4 * BOX);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(smem + OFF_Q1 + c * BOX, &tm_q1, &ctrl->q_full, 64 * c, q0, h, b_idx);
        tma_load_4d(smem + OFF_Q2 + c * BOX, &tm_q2, &ctrl->q_full, 64 * c, q0, h, b_idx);
      }
      auto acquire = [&](int hf) {  // wait until half hf is free, then arm its barrier
        if (uses[hf] > 0 && !mbar_wait(&ctrl->kv_empty[hf], (uses[hf] - 1) & 1, abort_flag,
                                       WAIT_TIMEOUT_NS))
          return false;
        mbar_arrive_expect_tx(&ctrl->kv_full[hf], HALF_BYTES);
        ++uses[hf];
        return true;
      };
      bool ok = true;
      for (int t = 0; ok && t < T; ++t) {
        const bool pass2 = t >= n_kv;
        const int y = (pass2 ? t - n_kv : t) * BN;
        const int hk = pass2 ? 0 : (t & 1);
        if (!(ok = acquire(hk))) break;
        uint8_t *st = smem + OFF_HALF + hk * HALF_BYTES;
        for (int c = 0; c < 2; ++c) {
          tma_load_4d(st + c * BOX, &tm_k1, &ctrl->kv_full[hk], 64 * c, y, h, b_idx);
          tma_load_4d(st + (2 + c) * BOX, &tm_k2, &ctrl->kv_full[hk], 64 * c, y, h, b_idx);
        }
        if (pass2) {
          if (!(ok = acquire(1))) break;
          uint8_t *sv = smem + OFF_HALF + HALF_BYTES;
          for (int c = 0; c < 4; ++c)
            tma_load_4d(sv + c * BOX, &tm_v, &ctrl->kv_full[1], 64 * c, y, h, b_idx);
        }
      }
      drain_wait(&ctrl->q_full, 0);
      for (int hf = 0; hf < 2; ++hf)
        if (uses[hf] > 0) drain_wait(&ctrl->kv_full[hf], (uses[hf] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, true);
      const uint64_t dq[2] = {smem_desc_sw128(smem_u32(smem + OFF_Q1), 16, 1024),
                              smem_desc_sw128(smem_u32(smem + OFF_Q2), 16, 1024)};
      // K-major views of half hf: K1 at box 0-1, K2 at box 2-3.
      const uint64_t dh = smem_desc_sw128(smem_u32(smem + OFF_HALF), 16, 1024);
      // V [128 keys x 256 columns] in half 1 as four 64-column boxes (MN-major B).
      const uint64_t dvb = smem_desc_sw128(smem_u32(smem + OFF_HALF + HALF_BYTES), BOX, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      uint32_t uses[2] = {0, 0};  // consumed uses of each half
      // S_k of tile t from the K tiles in half hk (K = 128 as two 64-column boxes).
      auto issue_qk = [&](int t) {
        const bool pass2 = t >= n_kv;
        const int hk = pass2 ? 0 : (t & 1);
        if (!mbar_wait(&ctrl->kv_full[hk], uses[hk] & 1, abort_flag, WAIT_TIMEOUT_NS))
          return false;
        ++uses[hk];
        tc_fence_after_sync();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t d_tm = tmem + tm_s(k, pass2, t);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX + 32 * (kk & 3);
            umma_bf16_ss(d_tm, adv(dq[k], off),
                         adv(dh, hk * HALF_BYTES + 2 * k * BOX + off), IDESC_QK, kk > 0);
          }
        }
        umma_commit(&ctrl->s_full[t & 1]);
        umma_commit(&ctrl->kv_empty[hk]);  // K read once the S MMAs are done
        return true;
      };
      bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag, WAIT_TIMEOUT_NS);
      tc_fence_after_sync();
      // Pass 1 runs two tiles ahead (double-buffered S); pass 2 one tile ahead.
      if (ok) ok = issue_qk(0);
      if (ok && n_kv > 1) ok = issue_qk(1);
      for (int t = 0; ok && t < T; ++t) {
        const int b = t & 1;
        if (!(ok = mbar_wait(&ctrl->s_done[b], (t >> 1) & 1, abort_flag, WAIT_TIMEOUT_NS)))
          break;
        tc_fence_after_sync();
        if (t >= n_kv) {
          // O += P V: P packed over S1 (keys 0-63 at columns 0-31, 64-127 at
          // 64-95), V MN-major (16 keys = 2048 bytes per step), N = 256.
          if (!(ok = mbar_wait(&ctrl->kv_full[1], uses[1] & 1, abort_flag, WAIT_TIMEOUT_NS)))
            break;
          ++uses[1];
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t pcol = (kk < 4) ? 8 * kk : 64 + 8 * (kk - 4);
            umma_bf16_ts(tmem + TM_O, tmem + tm_s(0, true, t) + pcol, adv(dvb, 2048 * kk),
                         IDESC_PV, (t > n_kv || kk > 0) ? 1u : 0u);
          }
          umma_commit(&ctrl->kv_empty[1]);
        }
        // Next S: pass-1 tile t + 2 into this buffer, or (from the last pass-1
        // tile on) the next pass-2 tile, after PV of this one (in order).
        const int nxt = (t + 2 < n_kv) ? t + 2 : (t + 1 >= n_kv && t + 1 < T) ? t + 1 : -1;
        if (nxt >= 0 && !(ok = issue_qk(nxt))) break;
      }
      if (ok) umma_commit(&ctrl->o_done);
      umma_commit(&ctrl->drain);
      drain_wait(&ctrl->drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax groups
    const int g = (warp - 4) / 4;
    const int r = (warp % 4) * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const float sl2 = p.scale_log2;
    const int qpos = p.q_off + q0 + r;  // sequence position of this row
    float m = -INFINITY, l = 0.f;               // pass 1: statistics of map g + 1
    float m1 = 0.f, m2 = 0.f, c2 = 0.f;  // pass 2: log2-sum-exp of each map, lambda
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int b = t & 1;
      ok = mbar_wait(&ctrl->s_full[b], (t >> 1) & 1, abort_flag, WAIT_TIMEOUT_NS);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const bool pass2 = t >= n_kv;
      const int kv0 = (pass2 ? t - n_kv : t) * BN;
      // Key column c of the tile is visible to this row iff c <= lim.
      const int lim = p.causal ? (qpos - kv0) : (p.N_kv - 1 - kv0);
      const bool masked = __any_sync(0xffffffffu, lim < BN - 1);
      if (!pass2) {
        // Online statistics over four 32-column chunks.  As in the d = 64
        // kernel, exponentials are taken against the current reference m and a
        // chunk whose sum is at most 2^8 needs nothing else; otherwise its
        // maximum (from the registers) moves m first.  The buffer is released
        // as soon as the last chunk has been read.
        const uint32_t t_s = tmem + lane_addr + tm_s(g, false, t);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t a[32];
          tmem_ld_x32(t_s + c0, a);
          if (c0 == BN - 32) {
            tc_fence_before_sync();
            mbar_arrive(&ctrl->s_done[b]);
          }
          if (masked) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              a[i] = (c0 + i <= lim) ? a[i] : __float_as_uint(-INFINITY);
          }
          float2 acc = make_float2(0.f, 0.f);
          const float2 sc = make_float2(sl2, sl2), nm = make_float2(-m, -m);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float2 e = __ffma2_rn(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                                  sc, nm);
            e.x = ex2_approx(e.x);
            e.y = ex2_approx(e.y);
            acc = __fadd2_rn(acc, e);
          }
          const float sum = acc.x + acc.y;
          if (__any_sync(0xffffffffu, !(sum <= 256.f))) {
            // Exact: the chunk maximum, then the sum against max(m, chunk max).
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) mt = fmaxf(mt, __uint_as_float(a[i]));
            const float m_new = fmaxf(m, mt * sl2);
            if (m_new != -INFINITY) {
              float2 acc2 = make_float2(0.f, 0.f);
              const float2 nm2 = make_float2(-m_new, -m_new);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float2 e = __ffma2_rn(
                    make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])), sc, nm2);
                e.x = ex2_approx(e.x);
                e.y = ex2_approx(e.y);
                acc2 = __fadd2_rn(acc2, e);
              }
              l = l * ex2_approx(m - m_new) + (acc2.x + acc2.y);
              m = m_new;
            }
          } else {
            l += sum;
          }
        }
        if (t == n_kv - 1) {
          // Final statistics of both maps as log2-sum-exp per row.
          ctrl->xch[g][r] = m + __log2f(l);
          if (kTrain && p.save_lse != nullptr) {
            const int64_t n_pad = static_cast<int64_t>(p.n_qtiles) * BM;
            if (dbg_ok(q0 + r < n_pad, p.status, 80))
              p.save_lse[(g * p.BH + bh) * n_pad + q0 + r] = m + __log2f(l);
          }
          named_barrier_sync(1, 256);
          m1 = ctrl->xch[0][r];
          m2 = ctrl->xch[1][r];
          c2 = p.lambda[h];
        }
      } else {
        // Keys 64g .. 64g+63 of both maps in two 32-key chunks:
        // P = 2^(x1 - lse1) - lambda 2^(x2 - lse2), packed over S1.
        const float2 sc = make_float2(sl2, sl2);
        const float2 n1 = make_float2(-m1, -m1), n2 = make_float2(-m2, -m2);
        const float2 nl = make_float2(-c2, -c2);
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          const int kc = 64 * g + c0;  // first key column of the chunk
          uint32_t a[32], bb[32];
          tmem_ld_x32_nowait(tmem + lane_addr + tm_s(0, true, t) + kc, a);
          tmem_ld_x32_nowait(tmem + lane_addr + tm_s(1, true, t) + kc, bb);
          tmem_ld_wait_x32(a);
          tmem_ld_wait_x32(bb);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float2 e1 = __ffma2_rn(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                                   sc, n1);
            float2 e2 = __ffma2_rn(
                make_float2(__uint_as_float(bb[i]), __uint_as_float(bb[i + 1])), sc, n2);
            e1.x = ex2_approx(e1.x);
            e1.y = ex2_approx(e1.y);
            e2.x = ex2_approx(e2.x);
            e2.y = ex2_approx(e2.y);
            float2 pp = __ffma2_rn(e2, nl, e1);
            if (masked) {
              pp.x = (kc + i <= lim) ? pp.x : 0.f;
              pp.y = (kc + i + 1 <= lim) ? pp.y : 0.f;
            }
            pk[i / 2] = pack_bf16x2(pp.x, pp.y);
          }
          // Over S1 columns 64g + c0/2 .. +15: read in this or the previous chunk.
          tmem_st_x16(tmem + lane_addr + tm_s(0, true, t) + 64 * g + c0 / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&ctrl->s_done[b]);
      }
    }

    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&ctrl->o_done, 0, abort_flag, WAIT_TIMEOUT_NS);
    const bool failed = named_barrier_or(1, 256, !ok || *abort_flag != 0);
    if (!failed) {
      tc_fence_after_sync();
      // Columns 128g .. 128g+127 of o = O (already normalised per map).
      const uint32_t t_o = tmem + lane_addr + TM_O + 128 * g;
      float sm = 0.f, ss = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(t_o + c0, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float o = __uint_as_float(v[c]);
          sm += o;
          ss = fmaf(o, o, ss);
        }
      }
      float mu = 0.f, rr = 1.f;
      if (p.headnorm) {
        // Both groups' partial sums per row.  (Every thread read the pass-1
        // statistics in xch[0..3] before the barrier above, so they can go.)
        if (g == 0) {
          ctrl->xch[0][r] = sm;
          ctrl->xch[1][r] = ss;
        } else {
          ctrl->xch[2][r] = sm;
          ctrl->xch[3][r] = ss;
        }
        named_barrier_sync(1, 256);
        const float tsm = ctrl->xch[0][r] + ctrl->xch[2][r];
        const float tss = ctrl->xch[1][r] + ctrl->xch[3][r];
        if (p.headnorm == 2) {
          mu = tsm * (1.f / DV);
          rr = rsqrtf(fmaxf(tss * (1.f / DV) - mu * mu, 0.f) + p.eps) * p.out_scale;
        } else {
          rr = rsqrtf(tss * (1.f / DV) + p.eps) * p.out_scale;
        }
      }
      const float *w = (p.headnorm && p.norm_w) ? p.norm_w + static_cast<int64_t>(h) * DV + 128 * g
                                                : nullptr;
      // 64 columns at a time: packed to bf16, transposed across each 8-lane
      // group (rows) so that every store instruction writes four 128-byte row
      // segments instead of one 16-byte piece of 32 rows.
      const int row0 = q0 + (warp % 4) * 32 + (lane & ~7);  // the 8-lane group's first row
      __nv_bfloat16 *obase =
          p.out + b_idx * p.out_sb + h * p.out_sh + 128 * g + 8 * (lane & 7);
#pragma unroll 1
      for (int c64 = 0; c64 < 128; c64 += 64) {
        uint4 pkt[8];
#pragma unroll
        for (int c32 = 0; c32 < 64; c32 += 32) {
          uint32_t v[32];
          tmem_ld_x32(t_o + c64 + c32, v);  // warp-collective
          float y[32];
          if (w != nullptr) {  // uniform
#pragma unroll
            for (int c = 0; c < 32; ++c)
              y[c] = (__uint_as_float(v[c]) - mu) * rr * __ldg(w + c64 + c32 + c);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) y[c] = (__uint_as_float(v[c]) - mu) * rr;
          }
          if (kTrain && p.o_save != nullptr) {  // uniform: this thread's row, pre-norm
            if (q0 + r < p.N &&
                dbg_ok(q0 + r >= 0 && 128 * g + c64 + c32 + 32 <= DV, p.status, 52)) {
              float4 *dst = reinterpret_cast<float4 *>(
                  p.o_save + (bh * p.N + q0 + r) * static_cast<int64_t>(DV) + 128 * g + c64 +
                  c32);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 &pk = pkt[c32 / 8 + q];
            pk.x = pack_bf16x2(y[8 * q + 0], y[8 * q + 1]);
            pk.y = pack_bf16x2(y[8 * q + 2], y[8 * q + 3]);
            pk.z = pack_bf16x2(y[8 * q + 4], y[8 * q + 5]);
            pk.w = pack_bf16x2(y[8 * q + 6], y[8 * q + 7]);
          }
        }
        transpose8_chunks(pkt, lane);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (row0 + j < p.N && dbg_ok(row0 + j >= 0 && c64 + 8 * (lane & 7) + 8 <= DV, p.status, 50))
            *reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(row0 + j) * p.out_sn + c64) =
                pkt[j];
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

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 4-D view {width, N, H, B} of a bf16 tensor with element strides (sn, sh, sb)
// and contiguous rows; boxes of `rows` rows x 64 columns, 128-byte swizzle.
CUresult encode_map(CUtensorMap *map, const void *base, uint64_t width, uint64_t N, uint64_t H,
                    uint64_t B, uint32_t rows, const diffattn_strides &st) {
  static EncodeTiledFn fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[4] = {width, N, H, B};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  cuuint32_t box[4] = {64, rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

diffattn_status launch_fwd_d128_sm103(const diffattn_desc &desc, int64_t n_kv, const void *q1,
                                      const void *k1, const void *q2, const void *k2,
                                      const void *v, const float *lambda, const float *norm_w,
                                      void *out, cudaStream_t stream,
                                      const diffattn_strides *strides, float *save_lse,
                                      float *o_save) {
  const int64_t BH = desc.B * desc.H, N = desc.N;
  const int64_t n_qtiles = (N + BM - 1) / BM;
  const int64_t n_ktiles = (n_kv + BN - 1) / BN;
  if (BH * n_qtiles > INT32_MAX || N > INT32_MAX / 2 || n_kv > INT32_MAX / 2 ||
      desc.B > INT32_MAX || desc.H > INT32_MAX)
    return DIFFATTN_ERR_UNSUPPORTED;
  // Element strides of q1, k1, q2, k2, v, out: given, or contiguous [B, H, rows, width].
  diffattn_strides st[6];
  for (int i = 0; i < 6; ++i) {
    const int64_t width = (i >= 4) ? DV : HD;
    const int64_t rows = (i == 0 || i == 2 || i == 5) ? N : n_kv;
    st[i] = strides ? strides[i] : diffattn_strides{desc.H * rows * width, rows * width, width};
  }
  CUtensorMap maps[5];
  const void *bases[5] = {q1, k1, q2, k2, v};
  for (int i = 0; i < 5; ++i) {
    const uint64_t width = (i == 4) ? DV : HD;
    const uint32_t rows = 128;
    const int64_t n_rows = (i == 0 || i == 2) ? N : n_kv;
    if (encode_map(&maps[i], bases[i], width, static_cast<uint64_t>(n_rows),
                   static_cast<uint64_t>(desc.H), static_cast<uint64_t>(desc.B), rows, st[i]) !=
        CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];  // per device (concurrent callers may both set)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(diffattn_fwd_d128_sm103_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(diffattn_fwd_d128_sm103_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  Params p;
  p.BH = BH;
  p.H = static_cast<int32_t>(desc.H);
  p.N = static_cast<int32_t>(N);
  p.N_kv = static_cast<int32_t>(n_kv);
  p.q_off = static_cast<int32_t>(n_kv - N);
  p.n_qtiles = static_cast<int32_t>(n_qtiles);
  p.n_ktiles = static_cast<int32_t>(n_ktiles);
  p.causal = desc.causal ? 1 : 0;
  p.headnorm = desc.headnorm;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  p.eps = desc.eps;
  p.out_scale = 1.0f - desc.lambda_init;
  p.lambda = lambda;
  p.norm_w = norm_w;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.status = desc.status_dev;
  p.out_sb = st[5].b;
  p.out_sh = st[5].h;
  p.out_sn = st[5].n;
  p.save_lse = save_lse;
  p.o_save = o_save;
  dim3 grid(static_cast<unsigned>(BH * n_qtiles));
  if (save_lse != nullptr || o_save != nullptr)
    diffattn_fwd_d128_sm103_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else
    diffattn_fwd_d128_sm103_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
