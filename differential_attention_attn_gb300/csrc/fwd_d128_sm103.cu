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
//   pass 1, per 64-key tile:  S1 = Q1 K1^T, S2 = Q2 K2^T  (tcgen05, K = 128)
//            exact online row maxima m_k and sums l_k of 2^(S_k log2e/sqrt(d))
//   pass 2, per 64-key tile:  S1, S2 again;
//            P = 2^(x1 - m1) / l1 - lambda 2^(x2 - m2) / l2   (final weights)
//            O += P V   (one TS MMA, N = 256, P read from TMEM)
//
// Each map is an ordinary softmax, so after pass 1 the normalisers are final
// and pass 2 needs no rescaling: O is the raw output o directly.  The price is
// the second S and the second set of exponentials.
//
// Tensor memory (512 columns): S1 double-buffered at 0 and 64, S2 at 128 and
// 192 (64 fp32 columns each), O at 256-511.  P of tile j is written as packed
// bf16 over the S1 buffer of tile j (keys 0-31 at its columns 0-15, keys 32-63
// at 32-47, each over columns its writers have already read).
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer, warps 4-7 and 8-11 two warpgroups (thread = query row = TMEM
// lane).  Pass 1: group g keeps the statistics of map g + 1.  Pass 2: group g
// forms P for keys 32g .. 32g+31 of both maps.  Epilogue: group g normalises
// and stores output columns 128g .. 128g+127.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 64;    // keys per key tile
constexpr int HD = 128;   // query/key half width d
constexpr int DV = 256;   // value width 2d
constexpr int NUM_THREADS = 384;
constexpr int STAGES = 2;

constexpr uint32_t BOX_Q = BM * 64 * 2;  // [128 rows x 64 columns] bf16: 16 KB
constexpr uint32_t BOX_K = BN * 64 * 2;  // [64 rows x 64 columns] bf16: 8 KB
constexpr uint32_t OFF_Q1 = 0;           // two 64-column boxes
constexpr uint32_t OFF_Q2 = 2 * BOX_Q;
constexpr uint32_t OFF_ST = 4 * BOX_Q;
constexpr uint32_t ST_K1 = 0;            // two boxes
constexpr uint32_t ST_K2 = 2 * BOX_K;    // two boxes
constexpr uint32_t ST_V = 4 * BOX_K;     // four boxes (256 value columns)
constexpr uint32_t STAGE_BYTES = 8 * BOX_K;
constexpr uint32_t OFF_CTRL = OFF_ST + STAGES * STAGE_BYTES;

struct Ctrl {
  uint64_t q_full;
  uint64_t kv_full[STAGES];
  uint64_t kv_empty[STAGES];
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

__host__ __device__ constexpr uint32_t tm_s1(int b) { return 64u * b; }
__host__ __device__ constexpr uint32_t tm_s2(int b) { return 128u + 64u * b; }
constexpr uint32_t TM_O = 256;

constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr uint64_t DRAIN_TIMEOUT_NS = 200000000ull;

struct Params {
  int64_t BH;
  int32_t H, N, n_qtiles, n_ktiles, causal, headnorm;
  float scale_log2, eps, out_scale;
  const float *lambda;
  const float *norm_w;
  __nv_bfloat16 *out;
  int32_t *status;
};

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > DRAIN_TIMEOUT_NS) return false;
  }
  return true;
}

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
  // Key tiles this query tile sees: all, or up to the one holding its last row.
  const int n_kv = p.causal ? min(p.n_ktiles, (q0 + BM - 1) / BN + 1) : p.n_ktiles;
  const int T = 2 * n_kv;  // tiles over both passes

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->kv_full[s], 1);
      mbar_init(&ctrl->kv_empty[s], 1);
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
    if (lane == 0) {
      uint32_t issued[STAGES] = {0, 0};
      mbar_arrive_expect_tx(&ctrl->q_full, 4 * BOX_Q);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(smem + OFF_Q1 + c * BOX_Q, &tm_q1, &ctrl->q_full, 64 * c, q0, h, b_idx);
        tma_load_4d(smem + OFF_Q2 + c * BOX_Q, &tm_q2, &ctrl->q_full, 64 * c, q0, h, b_idx);
      }
      for (int t = 0; t < T; ++t) {
        const int s = t & 1;
        const uint32_t u = static_cast<uint32_t>(t >> 1);
        if (u > 0 && !mbar_wait(&ctrl->kv_empty[s], (u - 1) & 1, abort_flag, WAIT_TIMEOUT_NS))
          break;
        const bool pass2 = t >= n_kv;
        const int y = (pass2 ? t - n_kv : t) * BN;
        uint8_t *st = smem + OFF_ST + s * STAGE_BYTES;
        uint64_t *bar = &ctrl->kv_full[s];
        mbar_arrive_expect_tx(bar, (pass2 ? 8 : 4) * BOX_K);
        for (int c = 0; c < 2; ++c) {
          tma_load_4d(st + ST_K1 + c * BOX_K, &tm_k1, bar, 64 * c, y, h, b_idx);
          tma_load_4d(st + ST_K2 + c * BOX_K, &tm_k2, bar, 64 * c, y, h, b_idx);
        }
        if (pass2)
          for (int c = 0; c < 4; ++c)
            tma_load_4d(st + ST_V + c * BOX_K, &tm_v, bar, 64 * c, y, h, b_idx);
        issued[s] = u + 1;
      }
      drain_wait(&ctrl->q_full, 0);
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] > 0) drain_wait(&ctrl->kv_full[s], (issued[s] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, true);
      const uint64_t dq[2] = {smem_desc_sw128(smem_u32(smem + OFF_Q1), 16, 1024),
                              smem_desc_sw128(smem_u32(smem + OFF_Q2), 16, 1024)};
      const uint64_t dk[2] = {smem_desc_sw128(smem_u32(smem + OFF_ST + ST_K1), 16, 1024),
                              smem_desc_sw128(smem_u32(smem + OFF_ST + ST_K2), 16, 1024)};
      // V [64 keys x 256 columns] as four 64-column boxes BOX_K apart (MN-major B).
      const uint64_t dvb = smem_desc_sw128(smem_u32(smem + OFF_ST + ST_V), BOX_K, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      // S_k of tile t into buffer b: K = 128 as two 64-column boxes of Q and K.
      auto issue_qk = [&](int t) {
        const int s = t & 1, b = t & 1;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t d_tm = tmem + (k == 0 ? tm_s1(b) : tm_s2(b));
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * BOX_Q + 32 * (kk & 3);
            const uint32_t koff = s * STAGE_BYTES + (kk >> 2) * BOX_K + 32 * (kk & 3);
            umma_bf16_ss(d_tm, adv(dq[k], qoff), adv(dk[k], koff), IDESC_QK, kk > 0);
          }
        }
        umma_commit(&ctrl->s_full[b]);
        if (t < n_kv) umma_commit(&ctrl->kv_empty[s]);  // pass 1 reads only K
      };
      bool ok = mbar_wait(&ctrl->q_full, 0, abort_flag, WAIT_TIMEOUT_NS);
      tc_fence_after_sync();
      for (int t = 0; ok && t < 2 && t < T; ++t) {
        if (!(ok = mbar_wait(&ctrl->kv_full[t & 1], 0, abort_flag, WAIT_TIMEOUT_NS))) break;
        tc_fence_after_sync();
        issue_qk(t);
      }
      for (int t = 0; ok && t < T; ++t) {
        const int s = t & 1, b = t & 1;
        if (!(ok = mbar_wait(&ctrl->s_done[b], (t >> 1) & 1, abort_flag, WAIT_TIMEOUT_NS)))
          break;
        tc_fence_after_sync();
        if (t >= n_kv) {
          // O += P V: P packed over S1[b] (keys 0-31 at columns 0-15, 32-63 at
          // 32-47), V MN-major (16 keys = 2048 bytes per step), N = 256.
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t pcol = (kk < 2) ? 8 * kk : 32 + 8 * (kk - 2);
            umma_bf16_ts(tmem + TM_O, tmem + tm_s1(b) + pcol,
                         adv(dvb, s * STAGE_BYTES + 2048 * kk), IDESC_PV,
                         (t > n_kv || kk > 0) ? 1u : 0u);
          }
          umma_commit(&ctrl->kv_empty[s]);
        }
        if (t + 2 < T) {  // S of tile t+2 into buffer b, after PV of tile t (in order)
          if (!(ok = mbar_wait(&ctrl->kv_full[s], ((t + 2) >> 1) & 1, abort_flag,
                               WAIT_TIMEOUT_NS)))
            break;
          tc_fence_after_sync();
          issue_qk(t + 2);
        }
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
    const int qpos = q0 + r;
    float m = -INFINITY, l = 0.f;               // pass 1: statistics of map g + 1
    float m1 = 0.f, m2 = 0.f, c1 = 0.f, c2 = 0.f;  // pass 2: 2^(x - m_k) scaled by c_k
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
      const int lim = p.causal ? (qpos - kv0) : (p.N - 1 - kv0);
      const bool masked = __any_sync(0xffffffffu, lim < BN - 1);
      if (!pass2) {
        uint32_t a[32], bb[32];
        const uint32_t t_s = tmem + lane_addr + (g == 0 ? tm_s1(b) : tm_s2(b));
        tmem_ld_x32_nowait(t_s, a);
        tmem_ld_x32_nowait(t_s + 32, bb);
        tmem_ld_wait_x32(a);
        tmem_ld_wait_x32(bb);
        tc_fence_before_sync();
        mbar_arrive(&ctrl->s_done[b]);  // S read: the buffer may be refilled
        float x[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(a[i]) * sl2;
          x[32 + i] = __uint_as_float(bb[i]) * sl2;
        }
        if (masked) {
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = (i <= lim) ? x[i] : -INFINITY;
        }
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) mt = fmaxf(mt, x[i]);
        const float m_new = fmaxf(m, mt);
        if (m_new != -INFINITY) {
          float sum = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) sum += ex2_approx(x[i] - m_new);
          l = l * ex2_approx(m - m_new) + sum;
          m = m_new;
        }
        if (t == n_kv - 1) {
          // Final statistics of both maps for every row.
          ctrl->xch[2 * g][r] = m;
          ctrl->xch[2 * g + 1][r] = l;
          named_barrier_sync(1, 256);
          m1 = ctrl->xch[0][r];
          m2 = ctrl->xch[2][r];
          c1 = 1.f / ctrl->xch[1][r];
          c2 = p.lambda[h] / ctrl->xch[3][r];
        }
      } else {
        // Keys 32g .. 32g+31 of both maps: P = 2^(x1 - m1) / l1 - lambda 2^(x2 - m2) / l2.
        uint32_t a[32], bb[32];
        tmem_ld_x32_nowait(tmem + lane_addr + tm_s1(b) + 32 * g, a);
        tmem_ld_x32_nowait(tmem + lane_addr + tm_s2(b) + 32 * g, bb);
        tmem_ld_wait_x32(a);
        tmem_ld_wait_x32(bb);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float pa = ex2_approx(fmaf(__uint_as_float(a[i]), sl2, -m1)) * c1 -
                     ex2_approx(fmaf(__uint_as_float(bb[i]), sl2, -m2)) * c2;
          float pb = ex2_approx(fmaf(__uint_as_float(a[i + 1]), sl2, -m1)) * c1 -
                     ex2_approx(fmaf(__uint_as_float(bb[i + 1]), sl2, -m2)) * c2;
          if (masked) {
            pa = (32 * g + i <= lim) ? pa : 0.f;
            pb = (32 * g + i + 1 <= lim) ? pb : 0.f;
          }
          pk[i / 2] = pack_bf16x2(pa, pb);
        }
        // Over S1[b] columns 32g .. 32g+15, which this group has just read.
        tmem_st_x16(tmem + lane_addr + tm_s1(b) + 32 * g, pk);
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
      const bool real = qpos < p.N;
      const float *w = (p.headnorm && p.norm_w) ? p.norm_w + static_cast<int64_t>(h) * DV + 128 * g
                                                : nullptr;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + (bh * p.N + (real ? qpos : 0)) * DV +
                                             128 * g);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(t_o + c0, v);  // warp-collective: every lane loads, real rows store
        if (real) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float y[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int col = c0 + 8 * q + c;
              y[c] = (__uint_as_float(v[8 * q + c]) - mu) * rr * (w ? __ldg(w + col) : 1.f);
            }
            uint4 pkt;
            pkt.x = pack_bf16x2(y[0], y[1]);
            pkt.y = pack_bf16x2(y[2], y[3]);
            pkt.z = pack_bf16x2(y[4], y[5]);
            pkt.w = pack_bf16x2(y[6], y[7]);
            dst[c0 / 8 + q] = pkt;
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

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 4-D view {width, N, H, B} of a contiguous [B, H, N, width] bf16 tensor; boxes
// of `rows` rows x 64 columns, 128-byte swizzle.
CUresult encode_map(CUtensorMap *map, const void *base, uint64_t width, uint64_t N, uint64_t H,
                    uint64_t B, uint32_t rows) {
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
  cuuint64_t strides[3] = {width * 2, width * 2 * N, width * 2 * N * H};
  cuuint32_t box[4] = {64, rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

diffattn_status launch_fwd_d128_sm103(const diffattn_desc &desc, const void *q1, const void *k1,
                                      const void *q2, const void *k2, const void *v,
                                      const float *lambda, const float *norm_w, void *out,
                                      cudaStream_t stream) {
  const int64_t BH = desc.B * desc.H, N = desc.N;
  const int64_t n_qtiles = (N + BM - 1) / BM;
  const int64_t n_ktiles = (N + BN - 1) / BN;
  if (BH * n_qtiles > INT32_MAX || N > INT32_MAX / 2 || desc.B > INT32_MAX ||
      desc.H > INT32_MAX)
    return DIFFATTN_ERR_UNSUPPORTED;
  CUtensorMap maps[5];
  const void *bases[5] = {q1, k1, q2, k2, v};
  for (int i = 0; i < 5; ++i) {
    const uint64_t width = (i == 4) ? DV : HD;
    const uint32_t rows = (i == 0 || i == 2) ? BM : BN;
    if (encode_map(&maps[i], bases[i], width, static_cast<uint64_t>(N),
                   static_cast<uint64_t>(desc.H), static_cast<uint64_t>(desc.B), rows) !=
        CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(diffattn_fwd_d128_sm103_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    attr_set[dev] = true;
  }
  Params p;
  p.BH = BH;
  p.H = static_cast<int32_t>(desc.H);
  p.N = static_cast<int32_t>(N);
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
  dim3 grid(static_cast<unsigned>(BH * n_qtiles));
  diffattn_fwd_d128_sm103_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
