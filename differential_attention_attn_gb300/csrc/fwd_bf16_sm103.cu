// Fused differential-attention head forward, bf16 in / bf16 out, fp32
// accumulation, for sm_103a (GB300): TMA loads, tcgen05 MMAs with TMEM
// accumulators, two online softmax states per query row and a fused RMS
// head-norm epilogue.
//
// The method ("Differential Transformer", Ultralytics glossary, section "How
// differential attention works"): two softmax maps per head from two
// query/key halves, combined as (map1 - lambda map2) V with V twice as wide
// as a half; each head's output normalised on its own, then scaled by
// (1 - lambda_init).  The page notes that each map is ordinary softmax
// attention; that is what makes the flash-style online softmax below valid
// for each map separately.
//
// Work item: one (batch*head, 128-row query tile).  The single-pass grid is
// persistent (one CTA per SM at most), each CTA walking a fixed share of the
// items: the next item's Q load and first S MMAs overlap the current item's
// last P V products and epilogue, instead of a CTA exit, launch and prologue
// per item.  Per key tile of 128 keys:
//   S1 = Q1 K1^T, S2 = Q2 K2^T              tcgen05 SS MMAs into TMEM
//   P_k = exp2(S_k * log2(e)/sqrt(d) - m_k)  per map, thread-per-row softmax
//   O1 += P1 V, O2 += P2 V                   tcgen05 TS MMAs (P read from TMEM)
// and at the end o = O1/l1 - lambda O2/l2, then the RMS norm over the 128
// value channels, the weight, the (1 - lambda_init) scale and a bf16 store.
//
// One accumulator per map is needed: the two maps have independent running
// maxima and sums, so a single running (P1 - lambda P2) V cannot be
// renormalised exactly once the final sums are known.
//
// Warp roles (640 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator and MMA issuer (one elected lane of the warp)
//   warps 2-3   idle
//   warps 4-11  softmax of map 1, warps 12-19 softmax of map 2
// A softmax warp covers 16 query rows (TMEM lanes) of its warp's quarter, two
// threads per row: lanes 0-15 take keys 0-63 of each key tile, lanes 16-31
// keys 64-127 (the 16x32bx2 TMEM access shape).  The two threads of a row
// agree through warp shuffles, so a row's softmax state never waits on
// another warp, and each map's tile is spread over two warps per SM
// sub-partition.  The epilogue gives each of a row's four threads (two maps x
// two halves) 32 of its 128 value columns; 1/l and partial sums of squares
// are exchanged through shared memory.  Once every thread has read O1 and O2
// into registers they are released (o_free) to the next item's first P V.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S1: P1 as packed bf16, keys 0-63 over columns 0-31 and keys
//           64-127 over columns 64-95 (each half-row thread overwrites only
//           the S columns it has read)
//   [128,256) S2 (P2 likewise)   [256,384) O1   [384,512) O2
//
// MMA issue order per key tile j keeps the tensor pipe busy while the
// softmax of the other map runs:  S1_j, PV2_{j-1}, S2_j, PV1_j.  tcgen05 MMAs
// from one thread execute in order, so S_k of tile j+1 never overwrites P_k
// of tile j before PV_k of tile j has read it, and the commit that publishes
// S_k of tile j also certifies that PV_k of tile j-1 is complete (which the
// softmax needs before it rescales O_k).  Operand descriptors are built once
// and advanced by adding to their start-address field.
//
// Softmax (two threads per row, 64 key columns each per tile).  Each map
// keeps a reference maximum m (log2 units) per row and P = 2^(x - m), x = S
// log2(e) / sqrt(d).  In steady state a tile needs no maximum at all: the
// exponentials are computed against the current m, and since every P is at
// most its half row's sum, sums <= 2^16 certify the tile (P, O and the
// running sums then stay far from the fp32/bf16 range limits).  Otherwise
// (and on the first tile) the warp takes the exact path: the true maximum
// from S (still intact in TMEM, because P is held in registers until
// certified), m moved to that maximum plus a headroom whenever it is larger,
// a rescale of O_k and of the running sum, and the exponentials again.  The causal/ragged mask is
// compiled only into the tiles that need it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

constexpr int BM = 128;          // query rows per tile (TMEM lanes)
constexpr int BN = 128;          // keys per key tile
constexpr int HD = 64;           // query/key half width d
constexpr int DV = 2 * HD;       // value width 2d
constexpr int STAGES = 3;        // K/V pipeline depth
constexpr int NUM_THREADS = 640;
constexpr int SOFTMAX_THREADS = 512;    // warps 4-19
constexpr uint32_t REGS_LAUNCH = 96;    // 65536 / 640, rounded down to a multiple of 8
constexpr uint32_t REGS_CTRL = 64;      // per thread, warps 0-3 (loads, MMA issue)
constexpr uint32_t REGS_SOFTMAX = 104;  // per thread, warps 4-19 (softmax, epilogue)
constexpr float CERT_SUM = 65536.0f;    // half-row sums up to 2^16 certify a tile
// When the exact path sets the reference maximum it places it this far (log2
// units) above the tile's maximum: P then starts at most 2^-24 and later
// tiles may climb 24 + 16 units before the certificate fails again.  Only the
// scale of P, O and the sums changes (their relative precision does not); an
// entry more than about 100 units below the maximum flushes to zero, where
// its weight (below 2^-100 of the maximum's) is already far below rounding.
constexpr float M_HEADROOM = 24.0f;

constexpr uint32_t TILE_QK_BYTES = BM * HD * 2;     // 16 KB: one [128 x 64] bf16 tile
constexpr uint32_t TILE_V_BYTES = BN * DV * 2;      // 32 KB: two [128 x 64] column blocks
constexpr uint32_t OFF_Q1 = 0;
constexpr uint32_t OFF_Q2 = OFF_Q1 + TILE_QK_BYTES;
constexpr uint32_t OFF_STAGES = OFF_Q2 + TILE_QK_BYTES;
constexpr uint32_t STAGE_K1 = 0;
constexpr uint32_t STAGE_K2 = TILE_QK_BYTES;
constexpr uint32_t STAGE_V = 2 * TILE_QK_BYTES;
constexpr uint32_t STAGE_BYTES = 2 * TILE_QK_BYTES + TILE_V_BYTES;
constexpr uint32_t OFF_CTRL = OFF_STAGES + STAGES * STAGE_BYTES;

struct Ctrl {
  uint64_t q_full;
  uint64_t q_empty;   // the item's last Q K^T MMAs completed: Q may be replaced
  uint64_t k_full[STAGES];
  uint64_t v_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t o_free;    // the epilogue has read O1 and O2: the next item's P V may overwrite
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float xch[2 * BM];  // epilogue exchange of per-row values between the two maps
  alignas(16) float w_row[DV];  // the item's head-norm weights (staged for the epilogue)
};

constexpr uint32_t SMEM_BYTES = OFF_CTRL + sizeof(Ctrl) + 1024;  // + alignment slack
static_assert(offsetof(Ctrl, w_row) % 16 == 0 && OFF_CTRL % 16 == 0, "w_row is read as float4");
static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
static_assert(OFF_STAGES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "SW128 tiles need 1 KB alignment");
static_assert(SMEM_BYTES + 1024 < (1u << 18), "descriptor start addresses must stay below 256 KB");

constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_s(int k) { return 128u * k; }        // S_k / P_k
__host__ __device__ constexpr uint32_t tm_o(int k) { return 256u + 128u * k; }  // O_k

// Split-KV partial blocks (layout in internal.h).
constexpr int64_t PART_OFF_M = kPartOffM;
constexpr int64_t PART_OFF_L = kPartOffL;
constexpr int64_t PART_MAP_FLOATS = kPartMapFloats;
constexpr int64_t PART_FLOATS = kPartFloats;
static_assert(BM == kTileRows && BN == kTileKeys && DV == kValueCols, "tile shape");

constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr uint64_t DRAIN_TIMEOUT_NS = 200000000ull;   // 0.2 s to drain in-flight copies

struct Params {
  int64_t BH;
  int32_t H;
  int32_t N;          // query rows per head
  int32_t N_kv;       // key/value rows per head
  int32_t q_off;      // sequence position of query row 0 (N_kv - N): causal alignment
  int32_t n_qtiles;
  int32_t n_ktiles;
  uint32_t n_items;   // BH * n_qtiles
  int32_t causal;
  int32_t headnorm;
  float scale_log2;   // log2(e) / sqrt(d)
  float eps;
  float out_scale;    // 1 - lambda_init
  const float *lambda;
  const float *norm_w;
  __nv_bfloat16 *out;
  int32_t *status;
  // Split-KV partial mode (splits > 1): CTA blockIdx.x handles key tiles
  // [split * split_tiles, ...) of its query tile and writes unnormalised O_k,
  // reference maxima and running sums to `part` instead of the output.
  int32_t splits;
  int32_t split_tiles;
  float *part;
  // Saved activations for the backward pass (kSave): each map's normalised
  // output O_k / l_k as fp32 [2][B*H][N][128], and its log2-sum-exp
  // m_k + log2(l_k) as fp32 [2][B*H][n_pad], n_pad = 128 * n_qtiles.
  float *save_o;
  float *save_lse;
  // Element strides of `out` (batch, head, row); rows of 128 are contiguous.
  int64_t out_sb, out_sh, out_sn;
};

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > DRAIN_TIMEOUT_NS) return false;
  }
  return true;
}

// e4m3 operands (kind::f8f6f4): instruction descriptor with A and B both
// E4M3 (format code 0), fp32 D, K-major; and the shared-memory descriptor of
// a tile of 64-byte rows with 64-byte swizzle (layout code 4, 8-row groups
// 512 bytes apart).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>(1) << 16;
  desc |= static_cast<uint64_t>(512 >> 4) << 32;
  desc |= static_cast<uint64_t>(1) << 46;
  desc |= static_cast<uint64_t>(4) << 61;
  return desc;
}
// Issued by one elected lane of a converged warp (as umma_bf16_ss_lo_warp).
__device__ __forceinline__ void umma_e4m3_ss_warp(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 32-key chunk of a half row: mask (key key0 + i visible iff key0 + i <=
// lim), x = s * log2(e)/sqrt(d) - m, p = 2^x, accumulate the sum in four
// packed partial sums and pack p as bf16 pairs into pk[pk0 ..].
template <bool kMasked>
__device__ __forceinline__ void softmax_chunk_exp(const uint32_t (&x)[32], int key0, int pk0,
                                                  float m, float sl2, int lim, float2 (&acc)[4],
                                                  uint32_t (&pk)[BN / 4]) {
  const float2 scale = make_float2(sl2, sl2), negm = make_float2(-m, -m);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float a = __uint_as_float(x[i]), b = __uint_as_float(x[i + 1]);
    if (kMasked) {
      a = (key0 + i <= lim) ? a : -INFINITY;
      b = (key0 + i + 1 <= lim) ? b : -INFINITY;
    }
    float2 e = __ffma2_rn(make_float2(a, b), scale, negm);
    e.x = ex2_approx(e.x);
    e.y = ex2_approx(e.y);
    acc[(i / 2) % 4] = __fadd2_rn(acc[(i / 2) % 4], e);
    pk[pk0 + i / 2] = pack_bf16x2(e.x, e.y);
  }
}

// Exponentials of this thread's 64 keys of an S row (keys key0 .. key0 + 63,
// read through the two-threads-per-lane shape) against reference maximum m.
// Returns the half row's sum of the (unrounded) exponentials.
template <bool kMasked>
__device__ __forceinline__ float softmax_half_exp(uint32_t t_s, int key0, float m, float sl2,
                                                  int lim, uint32_t (&pk)[BN / 4]) {
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
  uint32_t a[32], b[32];
  tmem_ld16_x32_nowait(t_s, a);
  tmem_ld16_x32_nowait(t_s + 32, b);
  tmem_ld_wait_x32(a);
  tmem_ld_wait_x32(b);
  softmax_chunk_exp<kMasked>(a, key0, 0, m, sl2, lim, acc, pk);
  softmax_chunk_exp<kMasked>(b, key0 + 32, 16, m, sl2, lim, acc, pk);
  const float2 s01 = __fadd2_rn(acc[0], acc[1]), s23 = __fadd2_rn(acc[2], acc[3]);
  return (s01.x + s01.y) + (s23.x + s23.y);
}

// Maximum of this thread's 64 keys of an S row over the visible ones.
template <bool kMasked>
__device__ __forceinline__ float softmax_half_max(uint32_t t_s, int key0, int lim) {
  uint32_t a[32], b[32];
  tmem_ld16_x32_nowait(t_s, a);
  tmem_ld16_x32_nowait(t_s + 32, b);
  tmem_ld_wait_x32(a);
  tmem_ld_wait_x32(b);
  float v[64];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(a[i]);
    v[32 + i] = __uint_as_float(b[i]);
  }
  if (kMasked) {
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = (key0 + i <= lim) ? v[i] : -INFINITY;
  }
#pragma unroll
  for (int w = 32; w >= 1; w /= 2) {
#pragma unroll
    for (int i = 0; i < w; ++i) v[i] = fmaxf(v[i], v[i + w]);
  }
  return v[0];
}

// One work item: a (batch, head, 128-row query tile) and its key tiles.
struct Item {
  int q0;       // first query row
  int h, b;     // head, batch
  int64_t bh;   // b * H + h
  int kv_lo;    // first key tile (split-KV key range; 0 otherwise)
  int n_kv;     // key tiles to process
};

// The r-th work item of this CTA; false past the end.  The items are the
// (b*h, query tile) pairs, heaviest first: all heads' last query tiles, then the
// previous ones.  Single pass: the grid is persistent (at most one CTA per SM)
// and CTA c takes items c, 2G-1-c, 2G+c, 4G-1-c, ... of G, a deal whose
// direction alternates every round so that every CTA gets a similar mix of long
// and short items.  Split-KV: the CTA's single (query tile, key range),
// consecutive CTAs taking consecutive ranges of one query tile.  The decode uses
// 32-bit division (fewer than 2^31 items, checked at launch): a 64-bit one is a
// long software sequence.  The single-pass key range origin is a compile-time
// zero: a run-time origin measurably slows the loops.
template <bool kPartial>
__device__ __forceinline__ bool next_item(const Params &p, uint32_t r, Item &it) {
  uint32_t idx;
  int split = 0;
  if (kPartial) {
    if (r > 0) return false;
    idx = blockIdx.x / static_cast<uint32_t>(p.splits);
    split = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.splits));
  } else {
    const uint32_t G = gridDim.x, c = blockIdx.x;
    idx = r * G + ((r & 1) ? G - 1 - c : c);
    if (idx >= p.n_items) return false;
  }
  const uint32_t BH32 = static_cast<uint32_t>(p.BH), H32 = static_cast<uint32_t>(p.H);
  const int qt = p.n_qtiles - 1 - static_cast<int>(idx / BH32);
  const uint32_t bh = idx % BH32;
  it.h = static_cast<int>(bh % H32);
  it.b = static_cast<int>(bh / H32);
  it.bh = bh;
  it.q0 = qt * BM;
  const int n_all = static_cast<int>(key_tiles_seen(qt, p.N, p.N_kv, p.causal != 0));
  it.kv_lo = kPartial ? split * p.split_tiles : 0;
  it.n_kv = kPartial ? min(n_all, it.kv_lo + p.split_tiles) - it.kv_lo : n_all;
  return true;
}

// kPartial: split-KV partial mode (a key range per CTA, partial softmax
// states to p.part, no epilogue); otherwise the whole forward of a query tile.
// kSave (with !kPartial): also store the activations the backward pass needs.
// kGroup (with !kPartial): the head norm is the mean-subtracting form (with
// or without kSave).
// kFp8: q1, k1, q2, k2 are e4m3 (one byte per element, 64-byte
// rows with 64-byte swizzle in the same shared-memory slots); S is computed by
// kind::f8f6f4 MMAs, everything from P on is unchanged.
template <bool kPartial, bool kSave, bool kGroup, bool kFp8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    diffattn_fwd_bf16_sm103_kernel(const __grid_constant__ CUtensorMap tm_q1,
                                   const __grid_constant__ CUtensorMap tm_k1,
                                   const __grid_constant__ CUtensorMap tm_q2,
                                   const __grid_constant__ CUtensorMap tm_k2,
                                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + OFF_CTRL);
  volatile int *abort_flag = &ctrl->abort;
  constexpr uint32_t QK_LOAD_BYTES = kFp8 ? TILE_QK_BYTES / 2 : TILE_QK_BYTES;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // In split-KV mode the combine kernel launched behind this grid may be
  // scheduled once every CTA has started; it waits for this grid's completion
  // before reading the partial blocks.
  if (kPartial) grid_dependents_launch();

  // Split-KV partial mode: one (query tile, key range) per CTA, consecutive
  // CTAs taking consecutive key ranges of one query tile.  A CTA whose range is
  // empty (early causal query tiles see fewer key tiles than there are splits)
  // has nothing to do; the combine step skips it.
  if (kPartial) {
    const uint32_t item32 = blockIdx.x / static_cast<uint32_t>(p.splits);
    const int split = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.splits));
    const int qt = p.n_qtiles - 1 - static_cast<int>(item32 / static_cast<uint32_t>(p.BH));
    const int n_all = static_cast<int>(key_tiles_seen(qt, p.N, p.N_kv, p.causal != 0));
    if (min(n_all, (split + 1) * p.split_tiles) - split * p.split_tiles <= 0) return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctrl->q_full, 1);
    mbar_init(&ctrl->q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->k_full[s], 1);
      mbar_init(&ctrl->v_full[s], 1);
      mbar_init(&ctrl->kv_empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&ctrl->s_full[k], 1);
      mbar_init(&ctrl->p_ready[k], 8);  // one arrival per softmax warp of map k
    }
    mbar_init(&ctrl->o_done, 1);
    mbar_init(&ctrl->o_free, SOFTMAX_THREADS / 32);  // one arrival per softmax warp
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
    tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctrl->tmem_base;
  // Registers move from the load/MMA warpgroup to the four softmax warpgroups:
  // 128 x REGS_CTRL + 512 x REGS_SOFTMAX stays within the 640 x 96 of the launch.
  // (The e4m3 split-KV instantiation keeps the launch allocation.)
  static_assert(128 * REGS_CTRL + SOFTMAX_THREADS * REGS_SOFTMAX <= NUM_THREADS * REGS_LAUNCH,
                "register split");
  constexpr bool kSplitRegs = !(kFp8 && kPartial);

  // Every role walks the same sequence of work items (next_item) and counts
  // barrier phases by item (q_full, q_empty, o_done, o_free) or by key tile
  // over all items (k_full, v_full, kv_empty per stage; s_full, p_ready).
  if (warp < 4) {
    if (kSplitRegs) setmaxnreg_dec<REGS_CTRL>();  // warps 2 and 3 only give up registers
    if (warp == 0) {
      // ---------------------------------------------------------------- producer
      if (lane == 0) {
        uint32_t issued[STAGES];
        for (int s = 0; s < STAGES; ++s) issued[s] = 0;
        uint32_t q_loads = 0;
        uint32_t g = 0;  // key tiles loaded so far
        bool ok = true;
        Item it;
        for (uint32_t r = 0; ok && next_item<kPartial>(p, r, it); ++r) {
          // The previous item's Q is dead once its last Q K^T MMAs completed.
          if (r > 0 && !(ok = mbar_wait(&ctrl->q_empty, (r - 1) & 1, abort_flag, WAIT_TIMEOUT_NS)))
            break;
          if (!dbg_ok(it.q0 >= 0 && it.q0 < p.N && it.h >= 0 && it.h < p.H &&
                          it.bh >= 0 && it.bh < p.BH, p.status, 1))
            break;
          mbar_arrive_expect_tx(&ctrl->q_full, 2 * QK_LOAD_BYTES);
          tma_load_4d(smem + OFF_Q1, &tm_q1, &ctrl->q_full, 0, it.q0, it.h, it.b);
          tma_load_4d(smem + OFF_Q2, &tm_q2, &ctrl->q_full, 0, it.q0, it.h, it.b);
          q_loads = r + 1;
          for (int j = 0; j < it.n_kv; ++j, ++g) {
            const int s = static_cast<int>(g % STAGES);
            const uint32_t u = g / STAGES;
            if (u > 0 &&
                !(ok = mbar_wait(&ctrl->kv_empty[s], (u - 1) & 1, abort_flag, WAIT_TIMEOUT_NS)))
              break;
            uint8_t *st = smem + OFF_STAGES + s * STAGE_BYTES;
            const int32_t y = (it.kv_lo + j) * BN;
            if (!dbg_ok(s < STAGES && y >= 0 && y < p.n_ktiles * BN, p.status, 2)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&ctrl->k_full[s], 2 * QK_LOAD_BYTES);
            tma_load_4d(st + STAGE_K1, &tm_k1, &ctrl->k_full[s], 0, y, it.h, it.b);
            tma_load_4d(st + STAGE_K2, &tm_k2, &ctrl->k_full[s], 0, y, it.h, it.b);
            mbar_arrive_expect_tx(&ctrl->v_full[s], TILE_V_BYTES);
            tma_load_4d(st + STAGE_V, &tm_v, &ctrl->v_full[s], 0, y, it.h, it.b);
            tma_load_4d(st + STAGE_V + TILE_QK_BYTES, &tm_v, &ctrl->v_full[s], HD, y, it.h, it.b);
            issued[s] = u + 1;
          }
        }
        // Never leave with a copy in flight: wait (bounded) for every issued load.
        if (q_loads > 0) drain_wait(&ctrl->q_full, (q_loads - 1) & 1);
        for (int s = 0; s < STAGES; ++s) {
          if (issued[s] > 0) {
            drain_wait(&ctrl->k_full[s], (issued[s] - 1) & 1);
            drain_wait(&ctrl->v_full[s], (issued[s] - 1) & 1);
          }
        }
      }
      __syncwarp();  // the whole warp leaves together (the barriers below are warp-aligned)
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      // The whole warp walks the loop, so every operand is warp-uniform; one
      // elected lane issues each MMA and commit (the same lane throughout).
      {
        constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
        constexpr uint32_t IDESC_QK8 = idesc_e4m3_f32(BM, BN);
        constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, true);
        // Operand descriptors are built once.  Every operand is a base tile plus a
        // byte offset below 256 KB, so advancing it only adds offset >> 4 to the
        // 14-bit start-address field (no carry into the other fields).  All of
        // them share the high word (stride offset 1024, version, 128-byte
        // swizzle), so only their low words are kept.
        auto lo = [](uint64_t d) { return static_cast<uint32_t>(d); };
        const uint32_t dhi =
            static_cast<uint32_t>(smem_desc_sw128(smem_u32(smem + OFF_Q1), 16, 1024) >> 32);
        const uint32_t dq[2] = {lo(smem_desc_sw128(smem_u32(smem + OFF_Q1), 16, 1024)),
                                lo(smem_desc_sw128(smem_u32(smem + OFF_Q2), 16, 1024))};
        const uint32_t dk[2] = {
            lo(smem_desc_sw128(smem_u32(smem + OFF_STAGES + STAGE_K1), 16, 1024)),
            lo(smem_desc_sw128(smem_u32(smem + OFF_STAGES + STAGE_K2), 16, 1024))};
        const uint32_t dvb =
            lo(smem_desc_sw128(smem_u32(smem + OFF_STAGES + STAGE_V), TILE_QK_BYTES, 1024));
        auto qk = [&](int k, int s) {  // S_k = Q_k K_k^T, K from stage s; K slices of 32 bytes
          if (kFp8) {
            // e4m3 rows of 64 bytes, 64-byte swizzle (8-row atoms of 512 bytes); an
            // f8f6f4 MMA takes 32 elements (32 bytes) of K, so two cover d = 64.
            const uint64_t a = smem_desc_sw64(smem_u32(smem + (k ? OFF_Q2 : OFF_Q1)));
            const uint64_t b = smem_desc_sw64(smem_u32(smem + OFF_STAGES + s * STAGE_BYTES +
                                                       (k ? STAGE_K2 : STAGE_K1)));
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              umma_e4m3_ss_warp(tmem + tm_s(k), a + 2 * kk, b + 2 * kk, IDESC_QK8, kk > 0);
          } else {
            if (!dbg_ok(s < STAGES && tmem_cols_ok(tmem + tm_s(k), BN, tmem, TMEM_COLS), p.status,
                        3))
              return;
            const uint32_t a = dq[k], b = dk[k] + (static_cast<uint32_t>(s) * STAGE_BYTES >> 4);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
              umma_bf16_ss_lo_warp(tmem + tm_s(k), a + 2 * kk, b + 2 * kk, dhi, IDESC_QK, kk > 0);
          }
        };
        // O_k += P_k V; 16 keys = 2048 bytes of V.  P_k's keys 0-63 are packed over
        // S_k columns 0-31 and keys 64-127 over columns 64-95.
        auto pv = [&](int k, int s, bool accumulate) {
          if (!dbg_ok(s < STAGES && tmem_cols_ok(tmem + tm_o(k), DV, tmem, TMEM_COLS) &&
                          tmem_cols_ok(tmem + tm_s(k), BN, tmem, TMEM_COLS),
                      p.status, 4))
            return;
          const uint32_t b = dvb + (static_cast<uint32_t>(s) * STAGE_BYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_bf16_ts_lo_warp(tmem + tm_o(k), tmem + tm_s(k) + kk * 8 + (kk >= 4 ? 32 : 0),
                            b + 128 * kk, dhi, IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
        };
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
          return mbar_wait_warp(bar, parity, abort_flag, WAIT_TIMEOUT_NS);
        };
        bool ok = true;
        uint32_t g = 0;  // key tiles processed so far
        Item it;
        for (uint32_t r = 0; ok && next_item<kPartial>(p, r, it); ++r) {
          if (!(ok = wait_all(&ctrl->q_full, r & 1))) break;
          tc_fence_after_sync();
          for (int j = 0; j < it.n_kv; ++j, ++g) {
            const int s = static_cast<int>(g % STAGES);
            const uint32_t ph = (g / STAGES) & 1;
            if (!(ok = wait_all(&ctrl->k_full[s], ph))) break;
            tc_fence_after_sync();
            qk(0, s);
            umma_commit_warp(&ctrl->s_full[0]);
            if (j > 0) {
              if (!(ok = wait_all(&ctrl->p_ready[1], (g - 1) & 1)))
                break;
              tc_fence_after_sync();
              const int sp = static_cast<int>((g - 1) % STAGES);
              pv(1, sp, j - 1 > 0);
              umma_commit_warp(&ctrl->kv_empty[sp]);
            }
            qk(1, s);
            umma_commit_warp(&ctrl->s_full[1]);
            if (j == it.n_kv - 1) umma_commit_warp(&ctrl->q_empty);  // last use of this item's Q
            if (!(ok = wait_all(&ctrl->v_full[s], ph))) break;
            if (!(ok = wait_all(&ctrl->p_ready[0], g & 1))) break;
            // The first P V of an item overwrites O: the previous item's epilogue
            // must have read it.
            if (j == 0 && r > 0 &&
                !(ok = wait_all(&ctrl->o_free, (r - 1) & 1)))
              break;
            tc_fence_after_sync();
            pv(0, s, j > 0);
          }
          if (!ok) break;
          const uint32_t gl = g - 1;  // the item's last key tile
          if (!(ok = wait_all(&ctrl->p_ready[1], gl & 1))) break;
          tc_fence_after_sync();
          const int sl = static_cast<int>(gl % STAGES);
          pv(1, sl, it.n_kv > 1);
          umma_commit_warp(&ctrl->kv_empty[sl]);
          umma_commit_warp(&ctrl->o_done);
        }
        // Never free tensor memory under a running MMA: wait for all of them.
        umma_commit_warp(&ctrl->drain);
        drain_wait(&ctrl->drain, 0);
      }
      __syncwarp();  // the whole warp leaves together (the barriers below are warp-aligned)
    }
  } else {
    if (kSplitRegs) setmaxnreg_inc<REGS_SOFTMAX>();
    // ---------------------------------------------------------------- softmax
    const int sw = warp - 4;                     // softmax warp 0..15
    const int k = sw >> 3;                       // which map
    const int quarter = warp & 3;                // TMEM lane quarter of this warp
    const int hl = lane & 15;                    // row within the warp's 16
    const int hc = lane >> 4;                    // key half: keys 64 hc .. 64 hc + 63
    const int r = quarter * 32 + ((sw >> 2) & 1) * 16 + hl;  // query row = TMEM lane
    const int key0 = 64 * hc;
    const uint32_t lane_addr = static_cast<uint32_t>(r - hl) << 16;
    const uint32_t t_s = tmem + lane_addr + tm_s(k);
    const uint32_t t_o = tmem + lane_addr + tm_o(k);
    const float sl2 = p.scale_log2;
    float *xch = ctrl->xch;  // [2][BM]: per-row values of both maps
    uint32_t g = 0;  // key tiles processed so far
    for (uint32_t ri = 0;; ++ri) {
      Item it;
      if (!next_item<kPartial>(p, ri, it)) break;
      const int n_kv = it.n_kv;
      // Key column c of tile j is visible to this row iff c <= lim0 - 128 j.
      const int kv_first = kPartial ? it.kv_lo * BN : 0;
      const int lim0 = p.causal ? (p.q_off + it.q0 + r - kv_first) : (p.N_kv - 1 - kv_first);
      // The epilogue's per-head parameters, loaded now so that the key loop hides
      // their latency: lambda_h, and one head-norm weight per thread of the first
      // four softmax warps (weight (warp % 4) * 32 + lane).
      const float lam_h = kPartial ? 0.f : __ldg(p.lambda + it.h);
      const bool w_mine = !kPartial && p.norm_w != nullptr && sw < 4;
      const float w_pref =
          w_mine ? __ldg(p.norm_w + static_cast<int64_t>(it.h) * DV + quarter * 32 + lane) : 1.f;
      float m_run = -INFINITY;  // reference maximum (log2 units) used by the exponentials
      float l_run = 0.f;        // this half row's running sum of exp2(x - m_run)
      bool ok = true;
      for (int j = 0; j < n_kv; ++j, ++g) {
        ok = mbar_wait_warp(&ctrl->s_full[k], g & 1, abort_flag, WAIT_TIMEOUT_NS);
        if (!ok) break;
        tc_fence_after_sync();
        const int lim = lim0 - j * BN;
        const bool masked = __any_sync(0xffffffffu, lim < BN - 1);
        // This thread's S columns (two threads per lane: 64 apart) and its P.
        if (!dbg_ok_warp(tmem_range_ok(t_s, BN, tmem, TMEM_COLS, warp, 16) &&
                             tmem_range_ok(t_o, DV, tmem, TMEM_COLS, warp, 16),
                         p.status, 5)) {
          ok = false;
          break;
        }
        uint32_t pk[BN / 4];
        float tile_sum = 0.f;
        // Steady state: exponentials against the current reference maximum; a
        // half row's sum bounds each of its entries, so sums <= 2^16 certify the
        // tile and the maximum is never computed.  Otherwise (and on the first
        // tile) the exact path below recomputes the tile from S, which is still
        // intact in TMEM because P is only stored once certified.  Both threads of
        // a row are in this warp, so the warp-wide vote keeps them together.
        bool exact = (j == 0);
        if (!exact) {
          tile_sum = masked ? softmax_half_exp<true>(t_s, key0, m_run, sl2, lim, pk)
                            : softmax_half_exp<false>(t_s, key0, m_run, sl2, lim, pk);
          exact = __any_sync(0xffffffffu, !(tile_sum <= CERT_SUM));
        }
        if (exact) {
          float mt = masked ? softmax_half_max<true>(t_s, key0, lim)
                            : softmax_half_max<false>(t_s, key0, lim);
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the row's other half
          // A row can see no key at all in the first tile of a split key range
          // (mt = -inf); it then keeps m = -inf, its p are 0 and the next tile
          // rescales by 2^-inf = 0.
          const float m_new = fmaxf(m_run, mt * sl2 + M_HEADROOM);
          float alpha = 1.f;
          if (j == 0) {
            m_run = m_new;
          } else if (m_new > m_run) {  // move m whenever the tile exceeds it
            alpha = ex2_approx(m_run - m_new);
            m_run = m_new;
          }
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            // O_k of this row is complete up to tile j-1 (certified by s_full);
            // each thread rescales its 64 of the 128 columns.
#pragma unroll 1
            for (int c0 = 0; c0 < DV / 2; c0 += 32) {
              uint32_t o[32];
              tmem_ld16_x32(t_o + c0, o);
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const float2 v = __fmul2_rn(
                    make_float2(__uint_as_float(o[c]), __uint_as_float(o[c + 1])),
                    make_float2(alpha, alpha));
                o[c] = __float_as_uint(v.x);
                o[c + 1] = __float_as_uint(v.y);
              }
              tmem_st16_x32(t_o + c0, o);
            }
          }
          l_run *= alpha;
          const float m_use = m_run == -INFINITY ? 0.f : m_run;
          tile_sum = masked ? softmax_half_exp<true>(t_s, key0, m_use, sl2, lim, pk)
                            : softmax_half_exp<false>(t_s, key0, m_use, sl2, lim, pk);
        }
        l_run += tile_sum;
        // P_k as packed bf16 pairs over the first 32 of this thread's 64 S columns.
        tmem_st16_x32(t_s, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->p_ready[k]);
      }

      // -------------------------------------------------------------- epilogue
      if (ok) ok = mbar_wait_warp(&ctrl->o_done, ri & 1, abort_flag, WAIT_TIMEOUT_NS);
      const float l_row = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);  // both halves
      const float inv = 1.f / l_row;
      if (!dbg_ok(r >= 0 && r < BM && (!w_mine || quarter * 32 + lane < DV), p.status, 6))
        ok = false;
      if (!kPartial) {
        // Published by the barrier below.  Every thread finished reading the
        // previous item's exchange before this item's o_done could complete
        // (each thread's last P of this item follows its previous epilogue).
        if (hc == 0) xch[k * BM + r] = inv;
        if (w_mine) ctrl->w_row[quarter * 32 + lane] = w_pref;
      }
      // Every softmax warp takes the same branch: the barrier ORs every thread's view.
      if (named_barrier_or(1, SOFTMAX_THREADS, !ok || *abort_flag != 0)) break;
      tc_fence_after_sync();
      if (kPartial) {
        // Split-KV partial result of this map for real query rows: O_k column-major
        // (lanes 0-15 store 16 consecutive rows of a column, lanes 16-31 those of the
        // column 64 further), as accumulated against the reference maximum, then that
        // maximum and the running sum.
        float *blk = p.part + static_cast<int64_t>(blockIdx.x) * PART_FLOATS + k * PART_MAP_FLOATS;
        const bool real = dbg_ok(key0 + DV / 2 <= DV && r < BM, p.status, 7) && it.q0 + r < p.N;
#pragma unroll 1
        for (int c0 = 0; c0 < DV / 2; c0 += 32) {
          uint32_t v[32];
          tmem_ld16_x32(t_o + c0, v);
          if (real) {
#pragma unroll
            for (int c = 0; c < 32; ++c) blk[(key0 + c0 + c) * BM + r] = __uint_as_float(v[c]);
          }
        }
        if (real && hc == 0) {
          blk[PART_OFF_M + r] = m_run;
          blk[PART_OFF_L + r] = l_row;
        }
        continue;  // the only item of this CTA
      }
      if (kSave) {
        // This map's normalised output (this thread's 64 columns) and its
        // log2-sum-exp.  32 columns at a time, transposed across 8-lane groups
        // (8 rows of one key half) so that every store writes four 128-byte row
        // segments.
        const int64_t n_pad = static_cast<int64_t>(p.n_qtiles) * BM;
        if (hc == 0 && dbg_ok(it.q0 + r < n_pad && it.bh < p.BH, p.status, 8))
          p.save_lse[(k * p.BH + it.bh) * n_pad + it.q0 + r] = m_run + __log2f(l_row);
        const int row0 = it.q0 + r - (lane & 7);  // the 8-lane group's first row
        float *so = p.save_o + (k * p.BH + it.bh) * static_cast<int64_t>(p.N) * DV + key0 +
                    4 * (lane & 7);
#pragma unroll 1
        for (int c0 = 0; c0 < DV / 2; c0 += 32) {
          uint32_t v[32];
          tmem_ld16_x32(t_o + c0, v);  // warp-collective
          uint4 ch[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            ch[q] = make_uint4(__float_as_uint(__uint_as_float(v[4 * q]) * inv),
                               __float_as_uint(__uint_as_float(v[4 * q + 1]) * inv),
                               __float_as_uint(__uint_as_float(v[4 * q + 2]) * inv),
                               __float_as_uint(__uint_as_float(v[4 * q + 3]) * inv));
          transpose8_chunks(ch, lane);
#pragma unroll
          for (int jr = 0; jr < 8; ++jr) {
            if (row0 + jr < p.N &&
                dbg_ok(row0 + jr >= 0 && key0 + c0 + 4 * (lane & 7) + 4 <= DV, p.status, 9))
              *reinterpret_cast<uint4 *>(so + static_cast<int64_t>(row0 + jr) * DV + c0) = ch[jr];
          }
        }
      }
      const float inv1 = xch[r];
      const float c2 = lam_h * xch[BM + r];
      // This thread's 32 value columns: 64 hc + 32 k .. + 31, read from O1 and O2
      // through the two-threads-per-lane shape.
      const int col0 = key0 + 32 * k;
      if (!dbg_ok_warp(tmem_range_ok(tmem + lane_addr + tm_o(0) + 32 * k, 96, tmem, TMEM_COLS,
                                     warp, 16) &&
                           tmem_range_ok(tmem + lane_addr + tm_o(1) + 32 * k, 96, tmem,
                                         TMEM_COLS, warp, 16),
                       p.status, 10))
        break;
      float o[32];
      float ss = 0.f;
      {
        uint32_t o1r[32], o2r[32];
        tmem_ld16_x32_nowait(tmem + lane_addr + tm_o(0) + 32 * k, o1r);
        tmem_ld16_x32_nowait(tmem + lane_addr + tm_o(1) + 32 * k, o2r);
        tmem_ld_wait_x32(o1r);
        tmem_ld_wait_x32(o2r);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          o[c] = __uint_as_float(o1r[c]) * inv1 - __uint_as_float(o2r[c]) * c2;
          ss = fmaf(o[c], o[c], ss);
        }
      }
      // O1 and O2 are in registers: the next item's P V may overwrite them.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctrl->o_free);
      if (p.headnorm) {
        named_barrier_sync(1, SOFTMAX_THREADS);  // every thread has read the 1/l exchange
        if (kGroup) {  // mean-subtracting (group) form: centre the row first
          float sm = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) sm += o[c];
          sm += __shfl_xor_sync(0xffffffffu, sm, 16);
          if (hc == 0) xch[k * BM + r] = sm;
          named_barrier_sync(1, SOFTMAX_THREADS);
          const float mu = (xch[r] + xch[BM + r]) * (1.f / DV);
          named_barrier_sync(1, SOFTMAX_THREADS);  // every thread has read the sums
          ss = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            o[c] -= mu;
            ss = fmaf(o[c], o[c], ss);
          }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        if (hc == 0) xch[k * BM + r] = ss;
        named_barrier_sync(1, SOFTMAX_THREADS);
        const float tot = xch[r] + xch[BM + r];
        const float rr = rsqrtf(tot * (1.f / DV) + p.eps) * p.out_scale;
        if (p.norm_w != nullptr) {  // uniform: per-column weights from shared memory
          const float4 *w4 = reinterpret_cast<const float4 *>(ctrl->w_row + col0);
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 wv = w4[c / 4];
            o[c] *= rr * wv.x;
            o[c + 1] *= rr * wv.y;
            o[c + 2] *= rr * wv.z;
            o[c + 3] *= rr * wv.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] *= rr;
        }
      }
      // bf16 row chunks (4 x 16 bytes), transposed across each 4-lane group (4
      // rows of one key half) so that every store instruction writes eight
      // 64-byte row segments instead of one 16-byte piece of 32 rows.
      uint4 pkt[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        pkt[v].x = pack_bf16x2(o[8 * v + 0], o[8 * v + 1]);
        pkt[v].y = pack_bf16x2(o[8 * v + 2], o[8 * v + 3]);
        pkt[v].z = pack_bf16x2(o[8 * v + 4], o[8 * v + 5]);
        pkt[v].w = pack_bf16x2(o[8 * v + 6], o[8 * v + 7]);
      }
      transpose4_chunks(pkt, lane);
      const int row0 = it.q0 + r - (lane & 3);  // the 4-lane group's first row
      __nv_bfloat16 *obase = p.out + it.b * p.out_sb + it.h * p.out_sh + col0 + 8 * (lane & 3);
#pragma unroll
      for (int jr = 0; jr < 4; ++jr) {
        if (row0 + jr < p.N &&
            dbg_ok(row0 + jr >= 0 && col0 + 8 * (lane & 3) + 8 <= DV && it.b * p.H + it.h < p.BH,
                   p.status, 11))
          *reinterpret_cast<uint4 *>(obase + static_cast<int64_t>(row0 + jr) * p.out_sn) = pkt[jr];
      }
      // The next item writes xch and w_row only after its o_done, which needs
      // every thread's P of that item, so every thread has finished here.
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag && p.status != nullptr)
    atomicExch(p.status, static_cast<int32_t>(DIFFATTN_ERR_TIMEOUT));
}

// cuTensorMapEncodeTiled is a driver entry point; it is looked up through the
// runtime so that the library itself does not link against the driver.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 4-D view {inner, rows, H, B} of a bf16 tensor with element strides (sn, sh,
// sb) and contiguous rows; 128-row x 64-column boxes with 128-byte swizzle.
CUresult encode_tile_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t n,
                         uint64_t H, uint64_t B, const diffattn_strides &st, bool e4m3 = false) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  const uint64_t es = e4m3 ? 1 : 2;  // element bytes
  cuuint64_t dims[4] = {inner, n, H, B};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * es, static_cast<cuuint64_t>(st.h) * es,
                           static_cast<cuuint64_t>(st.b) * es};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                e4m3 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

diffattn_status launch_fwd_bf16_sm103(const diffattn_desc &desc, int64_t n_kv, const void *q1,
                                      const void *k1, const void *q2, const void *k2,
                                      const void *v, const float *lambda, const float *norm_w,
                                      void *out, cudaStream_t stream, int splits, float *part,
                                      float *save, const diffattn_strides *strides) {
  const int64_t BH = desc.B * desc.H;
  const int64_t N = desc.N;
  const int64_t n_qtiles = (N + BM - 1) / BM;
  const int64_t n_ktiles = (n_kv + BN - 1) / BN;
  const bool fp8 = desc.dtype == DIFFATTN_E4M3_QK;
  if (splits < 1 || (splits > 1 && part == nullptr) || (splits > 1 && save != nullptr))
    return DIFFATTN_ERR_INVALID_ARG;
  if (fp8 && (save != nullptr || desc.headnorm == 2)) return DIFFATTN_ERR_UNSUPPORTED;
  const int64_t split_tiles = (n_ktiles + splits - 1) / splits;
  if (BH * n_qtiles * splits > INT32_MAX || N > INT32_MAX / 2 || n_kv > INT32_MAX / 2 ||
      desc.H > INT32_MAX)
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
    const uint64_t inner = (i == 4) ? DV : HD;
    const uint64_t rows = (i == 0 || i == 2) ? N : n_kv;
    if (encode_tile_map(&maps[i], bases[i], inner, rows, static_cast<uint64_t>(desc.H),
                        static_cast<uint64_t>(desc.B), st[i], fp8 && i < 4) != CUDA_SUCCESS)
      return DIFFATTN_ERR_CUDA;
  }

  static std::atomic<bool> attr_set[64];  // per device (concurrent callers may both set)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DIFFATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DIFFATTN_ERR_UNSUPPORTED;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    auto *k0 = diffattn_fwd_bf16_sm103_kernel<false, false, false, false>;
    auto *k1 = diffattn_fwd_bf16_sm103_kernel<true, false, false, false>;
    auto *k2 = diffattn_fwd_bf16_sm103_kernel<false, true, false, false>;
    auto *k3 = diffattn_fwd_bf16_sm103_kernel<false, false, true, false>;
    auto *k4 = diffattn_fwd_bf16_sm103_kernel<false, false, false, true>;
    auto *k5 = diffattn_fwd_bf16_sm103_kernel<true, false, false, true>;
    auto *k6 = diffattn_fwd_bf16_sm103_kernel<false, true, true, false>;
    if (cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k5, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess ||
        cudaFuncSetAttribute(k6, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  p.n_items = static_cast<uint32_t>(BH * n_qtiles);
  p.causal = desc.causal ? 1 : 0;
  p.headnorm = desc.headnorm ? 1 : 0;  // the form is the kGroup instantiation
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  p.eps = desc.eps;
  p.out_scale = 1.0f - desc.lambda_init;
  p.lambda = lambda;
  p.norm_w = norm_w;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.status = desc.status_dev;
  p.splits = splits;
  p.split_tiles = static_cast<int32_t>(splits > 1 ? split_tiles : n_ktiles);
  p.part = splits > 1 ? part : nullptr;
  p.save_o = save;
  p.out_sb = st[5].b;
  p.out_sh = st[5].h;
  p.out_sn = st[5].n;
  p.save_lse = save ? save + 2 * BH * N * DV : nullptr;

  // Split-KV: one CTA per (query tile, key range).  Otherwise persistent: one
  // CTA per SM at most (one fits, by shared and tensor memory), each walking
  // its share of the items.
  static std::atomic<int> sm_cache[64];
  int sms = sm_cache[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DIFFATTN_ERR_CUDA;
    sm_cache[dev].store(sms, std::memory_order_release);
  }
  const int64_t items = BH * n_qtiles;
  if (items == 0) return DIFFATTN_OK;
  dim3 grid(static_cast<unsigned>(splits > 1 ? items * splits : std::min<int64_t>(items, sms)));
  if (fp8 && splits > 1)
    diffattn_fwd_bf16_sm103_kernel<true, false, false, true>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else if (fp8)
    diffattn_fwd_bf16_sm103_kernel<false, false, false, true>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else if (splits > 1)
    diffattn_fwd_bf16_sm103_kernel<true, false, false, false>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else if (save != nullptr && desc.headnorm == 2)
    diffattn_fwd_bf16_sm103_kernel<false, true, true, false>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else if (save != nullptr)
    diffattn_fwd_bf16_sm103_kernel<false, true, false, false>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else if (desc.headnorm == 2)
    diffattn_fwd_bf16_sm103_kernel<false, false, true, false>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  else
    diffattn_fwd_bf16_sm103_kernel<false, false, false, false>
        <<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  return cudaGetLastError() == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace diffattn
