// attn_fwd.cu — softmax attention forward on tcgen05 tensor cores.
//
// Computes, per (b, h), O = softmax(s * q_hat k_hat^T) v and the natural-log
// row log-sum-exp, streaming over 128-key tiles with an online softmax so the
// N x N score matrix never leaves the SM (re-diffusion README, "attention
// fix" section: the materialised B x 12 x 1101 x 1101 scores were the memory
// wall; the same [B, H, N, d] Q/K/V layout goes through a fused kernel).
//
// Work unit: 256 query rows of one (b, h) as two 128-row tiles A and B,
// streaming all key/value tiles of that head.  The kernel is persistent: one
// CTA per SM walks the units u = blockIdx.x, blockIdx.x + gridDim.x, ...
// with the K/V ring, the Q buffers (two at d = 64) and every barrier phase
// running on across units, so the next unit's Q load and first score
// products overlap the current unit's last tiles and its epilogue.  Roles:
//
//   warp 8      TMA producer: per unit its Q tiles, then K_0, V_0, K_1, V_1,
//               ... into a ring of 128 x d bf16 slots (128-byte swizzle).
//   warps 9-10  MMA issuers, one thread per query tile (A: warp 9, B: warp
//               10): S_X = Q_X K_j^T into TMEM and O_X += P_X V_j.  Two
//               issuers keep the tensor pipe fed while either one waits on a
//               barrier (a single issuer's waits and commits between MMA
//               groups leave the pipe idle).  A ring slot is released once
//               both issuers have committed their last MMA that reads it.
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: one thread
//               per query row (TMEM lane), 128 scores per key tile; running
//               max kept in the log2 domain and O in TMEM rescaled only when
//               the max grows by more than 2^8 (the probabilities stay <= 256,
//               exact in fp32 and well inside bf16 range).  P is written back
//               into TMEM as packed bf16 over the first 64 columns of the
//               tile's own S buffer, and the PV MMA reads its A operand from
//               there (no shared-memory round trip).
//
// TMEM (512 columns): S_A / P_A [0,128), S_B / P_B [128,256), O_A
// [256,256+d), O_B [256+d, 256+2d).  S_X(j+1) overwrites P_X(j) only after
// PV_X(j) was issued (tcgen05 MMAs of one thread run in issue order).  Rows
// past N in the last query tile read zeros (TMA fill) and are not stored;
// key columns past N in the last key tile are masked to -inf.
#include <cuda_bf16.h>

#include "jattn_internal.h"
#include "sm103_ptx.cuh"

namespace jattn {
namespace {

constexpr int kFwdThreads = 384;  // 8 softmax warps, producer, 2 MMA issuers, accumulator zeroing
// Registers per thread (setmaxnreg): softmax 208, the other warpgroup 88.
// Each SM sub-partition holds two softmax warps and one other (warp w on
// w % 4), and an increase draws only on the registers its three warps were
// launched with, so 2 x 208 + 88 must equal 3 x the launch count (168).  The
// launcher refuses any build whose register count differs.
constexpr int kRegLaunchFwd = 168, kRegSoftmax = 208, kRegOtherFwd = 88;
static_assert(2 * kRegSoftmax + kRegOtherFwd == 3 * kRegLaunchFwd, "forward register split");
static_assert(kRegSoftmax >= kRegLaunchFwd && kRegOtherFwd <= kRegLaunchFwd, "setmaxnreg direction");
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  static constexpr int kQTileBytes = kTileM * D * 2;
  static constexpr int kSlotBytes = kTileN * D * 2;
  static constexpr int kSlots = (D == 64) ? 8 : 5;
  // Q buffers (two query tiles each): two at d = 64, so the next unit's Q
  // loads while the current unit runs.
  static constexpr int kQBufs = (D == 64) ? 2 : 1;
  static constexpr int kOffQ = 0;  // + buf * 2 * kQTileBytes + x * kQTileBytes
  static constexpr int kOffRing = kOffQ + kQBufs * 2 * kQTileBytes;
  // d = 64: the normalised O tiles are staged (128-byte swizzle) and leave
  // with one TMA store per query tile; d = 128 has no room and stores rows.
  static constexpr bool kStageO = (D == 64);
  static constexpr int kOffStage = kOffRing + kSlots * kSlotBytes;  // + x * kQTileBytes
  static constexpr int kTileBytes = kOffStage + (kStageO ? 2 * kQTileBytes : 0);
  static constexpr int kDynSmem = kTileBytes + 1024;  // + alignment slack
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
  // d = 64: S_A, S_B, O_A, O_B and two packed-bf16 P buffers fill the 512
  // TMEM columns exactly, so P gets its own columns and S(j+1) can be issued
  // ahead of PV(j).  d = 128: P is written over the consumed S columns.
  static constexpr bool kSepP = (D == 64);
  static constexpr uint32_t kColS = 0;              // + 128 x
  static constexpr uint32_t kColO = 256;            // + D x
  static constexpr uint32_t kColP = kSepP ? 384 : 0;  // + 64 x (d = 64), + 128 x (aliased)
  static constexpr uint32_t kPStride = kSepP ? 64 : 128;
};

struct FwdBars {
  uint64_t full[8];
  uint64_t empty[8];  // kSlots <= 8
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t pv_done[2];
  uint64_t s_free[2];  // d = 64: the softmax has the scores in registers
  uint64_t drain[2];
  uint64_t epi[2];  // d = 64: the query tile's O rows are staged (one arrival per warp)
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Units: 256 query rows (tiles A and B) of one segment of one head.  Per
// head the units run over the segments' 256-row blocks in order; CTA c takes
// u = c, c + gridDim.x, ...  A unit streams its segment's key tiles.  Key
// tiles, ring slots and every per-tile barrier are counted on across units.
struct FwdUnit {
  int bh;      // head
  int q0;      // first query row (tile A) in the head
  int kvb;     // the segment's first row
  int end;     // one past its last row
  int nkv;     // its 128-key tiles
  bool has_b;  // tile B has rows
};

// The [B, H, N, d] layout: one segment [0, N) per head, decoded without the
// segment table.
struct FwdWorkUniform {
  int upc;    // 256-row blocks per head
  int units;  // heads * upc
  int nkv;    // 128-key tiles per head
  struct {
    int rows;
  } seg;
  __device__ __forceinline__ FwdUnit unit(int u) const {
    FwdUnit r;
    r.bh = u / upc;
    r.q0 = (u - r.bh * upc) * 2 * kTileM;
    r.kvb = 0;
    r.end = seg.rows;
    r.nkv = nkv;
    r.has_b = r.q0 + kTileM < r.end;
    return r;
  }
};

// Packed variable-length layout: segments from the table.
struct FwdWork {
  int upc;    // units per head
  int units;  // heads * upc
  SegTable seg;
  int uf[kMaxSegments + 1];  // units before each segment (256-row blocks)
  __device__ __forceinline__ FwdUnit unit(int u) const {
    FwdUnit r;
    r.bh = u / upc;
    const int k = u - r.bh * upc;
    int lo = 0, hi = seg.n;  // uf[lo] <= k < uf[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (uf[mid] <= k) lo = mid;
      else hi = mid;
    }
    r.kvb = seg.cu[lo];
    r.end = seg.cu[lo + 1];
    r.q0 = r.kvb + (k - uf[lo]) * 2 * kTileM;
    r.nkv = (r.end - r.kvb + kTileN - 1) / kTileN;
    r.has_b = r.q0 + kTileM < r.end;
    return r;
  }
};

// Warp 11 (training pair): zeroes the backward's fp32 dQ accumulator rows of
// this CTA's units, with HBM bandwidth the forward leaves idle, then counts
// the CTA as done (release increment).  The backward's preparation skips its
// own zeroing when the count equals this launch's grid size, and the
// norm backward resets the count.  (Pacing the writes by the producer's unit
// progress instead of writing them at once measured slower: 336.0 against
// 338.8 us per training step at 512 px.)
template <int D, class W>
__device__ void fwd_zero_dq(const W& w, float* dq, uint32_t* count, int lane) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int u = blockIdx.x; u < w.units; u += gridDim.x) {
    const FwdUnit un = w.unit(u);
    const int r1 = min(un.q0 + 2 * kTileM, un.end);
    uint4* base = reinterpret_cast<uint4*>(dq + (static_cast<size_t>(un.bh) * w.seg.rows + un.q0) * D);
    const int n = (r1 - un.q0) * (D / 4);
    for (int i = lane; i < n; i += 32) base[i] = z;
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(count, 1u);
  }
}

template <int D, class W>
__device__ void fwd_producer(const CUtensorMap* map_q, const CUtensorMap* map_k, const CUtensorMap* map_v,
                             uint8_t* sm, FwdBars& bars, const W& w, uint32_t* dev_err) {
  using C = FwdCfg<D>;
  tma_prefetch_desc(map_q);
  tma_prefetch_desc(map_k);
  tma_prefetch_desc(map_v);
  volatile int* ab = &bars.abort;
  int issued = 0, q_issued = 0;
  bool ok = true;
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const FwdUnit un = w.unit(u);
    const int bh = un.bh, q0 = un.q0;
    const bool hasB = un.has_b;
    const int per_unit = 2 * un.nkv;
    const int b = ui % C::kQBufs;
    if (ui >= C::kQBufs && !(ok = mbar_wait(&bars.q_empty[b], ((ui / C::kQBufs) - 1) & 1, ab, dev_err))) break;
    mbar_arrive_expect_tx(&bars.q_full[b], (hasB ? 2u : 1u) * C::kQTileBytes);
    for (int x = 0; x < (hasB ? 2 : 1); ++x)
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d(sm + C::kOffQ + (b * 2 + x) * C::kQTileBytes + blk * 16384, map_q, &bars.q_full[b], blk * 64,
                    q0 + x * 128, bh);
    ++q_issued;
    for (int i = 0; i < per_unit; ++i, ++issued) {
      const int slot = issued % C::kSlots;
      if (issued >= C::kSlots && !(ok = mbar_wait(&bars.empty[slot], ((issued / C::kSlots) - 1) & 1, ab, dev_err)))
        break;
      mbar_arrive_expect_tx(&bars.full[slot], C::kSlotBytes);
      const CUtensorMap* m = (i & 1) ? map_v : map_k;
      const int kv0 = un.kvb + (i >> 1) * kTileN;
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d(sm + C::kOffRing + slot * C::kSlotBytes + blk * 16384, m, &bars.full[slot], blk * 64, kv0, bh);
    }
  }
  if (*ab) {
    // Aborted: let the copies already in flight land before the CTA exits.
    for (int t = (q_issued > C::kQBufs ? q_issued - C::kQBufs : 0); t < q_issued; ++t)
      mbar_wait_drain(&bars.q_full[t % C::kQBufs], (t / C::kQBufs) & 1);
    for (int t = (issued > C::kSlots ? issued - C::kSlots : 0); t < issued; ++t)
      mbar_wait_drain(&bars.full[t % C::kSlots], (t / C::kSlots) & 1);
  }
}

// S = Q K^T: both operands K-major 128 x d tiles; base descriptors are built
// once and advanced by (byte offset >> 4) per 16-wide K step.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
  using C = FwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
    umma_bf16_ss(tmem_s, q_desc + off, k_desc + off, C::kIdescS, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V with P read from TMEM (16 keys = 8 packed columns per MMA) and
// V a 128-key x d slot stored key-rows x d (MN-major B operand).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, bool accumulate) {
  using C = FwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < kTileN / 16; ++kk) {
    umma_bf16_ts(tmem_o, tmem_p + kk * 8, v_desc + static_cast<uint64_t>((kk * 2048) >> 4), C::kIdescO,
                 (accumulate || kk > 0) ? 1u : 0u);
  }
}

// MMA issue for query tile slot x (A: x = 0, B: x = 1).  Both issuers read
// the same K/V slots; a slot's empty barrier and a Q buffer's empty barrier
// count one commit per issuer, so the B issuer walks and releases them also
// for units whose tile B has no rows.
template <int D, class W>
__device__ void fwd_mma(uint8_t* sm, FwdBars& bars, uint32_t tmem, int x, const W& w, uint32_t* dev_err) {
  using C = FwdCfg<D>;
  const uint32_t ring = smem_u32(sm + C::kOffRing);
  const uint32_t tS = tmem + C::kColS + x * 128;
  const uint32_t tO = tmem + C::kColO + x * D;
  const uint32_t tP = tmem + C::kColP + x * C::kPStride;
  auto slot_of = [](int i) { return i % C::kSlots; };
  auto phase_of = [](int i) { return (uint32_t)((i / C::kSlots) & 1); };
  auto k_desc = [=](int i) { return sdesc_sw128(ring + slot_of(i) * C::kSlotBytes, 16, 1024); };
  auto v_desc = [=](int i) { return sdesc_sw128(ring + slot_of(i) * C::kSlotBytes, 16384, 1024); };
  volatile int* ab = &bars.abort;
  int jx = 0;  // key tiles this issuer has processed (its barrier phases)
  int gb = 0;  // ring items of the previous units
  // d = 64: the next unit's first score product is issued in place of the
  // last tile's S(j+1), so that it is ready when the softmax finishes the
  // unit's epilogue.
  bool s0_issued = false;
  bool ok = true;
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const int b = ui % C::kQBufs;
    const FwdUnit uo = w.unit(u);
    const int nkv = uo.nkv;
    const int g0 = gb;  // first ring item of the unit
    gb += 2 * nkv;
    if (x == 1 && !uo.has_b) {
      // No tile B in this unit: only release the unit's slots and Q buffer.
      for (int i = 0; ok && i < 2 * nkv; ++i) {
        if (!(ok = mbar_wait(&bars.full[slot_of(g0 + i)], phase_of(g0 + i), ab, dev_err))) break;
        umma_commit(&bars.empty[slot_of(g0 + i)]);
      }
      if (ok) umma_commit(&bars.q_empty[b]);
      continue;
    }
    const uint64_t q_desc = sdesc_sw128(smem_u32(sm + C::kOffQ + (b * 2 + x) * C::kQTileBytes), 16, 1024);
    if (!s0_issued) {
      if (!(ok = mbar_wait(&bars.q_full[b], (ui / C::kQBufs) & 1, ab, dev_err))) break;
      if (!(ok = mbar_wait(&bars.full[slot_of(g0)], phase_of(g0), ab, dev_err))) break;
      // S_X of the unit's first key tile once the softmax holds the previous
      // tile's scores (d = 128: P over S was read by the PV issued before).
      if (C::kSepP && jx > 0 && !(ok = mbar_wait(&bars.s_free[x], (jx - 1) & 1, ab, dev_err))) break;
      tc_fence_after();
      issue_qk<D>(tS, q_desc, k_desc(g0));
      umma_commit(&bars.s_full[x]);
      umma_commit(&bars.empty[slot_of(g0)]);
    }
    s0_issued = false;
    // The next unit, if this issuer computes a tile of it (tile B may be
    // absent): its first score product goes out early (d = 64).
    const int un = u + static_cast<int>(gridDim.x);
    const bool early_next = C::kSepP && un < w.units && (x == 0 || w.unit(un).has_b);
    const int bn = (ui + 1) % C::kQBufs, g0n = g0 + 2 * nkv;
    for (int j = 0; ok && j < nkv; ++j) {
      const int jt = jx + j;
      const int iv = g0 + 2 * j + 1, ik = g0 + 2 * j + 2;
      const bool more = j + 1 < nkv;
      if (!(ok = mbar_wait(&bars.full[slot_of(iv)], phase_of(iv), ab, dev_err))) break;
      if (more && !(ok = mbar_wait(&bars.full[slot_of(ik)], phase_of(ik), ab, dev_err))) break;
      if (C::kSepP) {
        // S_X(j+1) as soon as the softmax holds S_X(j) in registers, so it is
        // computed during this tile's exponentials; then PV_X(j) from the
        // separate P columns once P_X(j) is written.
        if (more) {
          if (!(ok = mbar_wait(&bars.s_free[x], jt & 1, ab, dev_err))) break;
          tc_fence_after();
          issue_qk<D>(tS, q_desc, k_desc(ik));
          umma_commit(&bars.s_full[x]);
        } else if (early_next) {
          if (!(ok = mbar_wait(&bars.q_full[bn], ((ui + 1) / C::kQBufs) & 1, ab, dev_err))) break;
          if (!(ok = mbar_wait(&bars.full[slot_of(g0n)], phase_of(g0n), ab, dev_err))) break;
          if (!(ok = mbar_wait(&bars.s_free[x], jt & 1, ab, dev_err))) break;
          tc_fence_after();
          const uint64_t q_desc_n =
              sdesc_sw128(smem_u32(sm + C::kOffQ + (bn * 2 + x) * C::kQTileBytes), 16, 1024);
          issue_qk<D>(tS, q_desc_n, k_desc(g0n));
          umma_commit(&bars.s_full[x]);
          umma_commit(&bars.empty[slot_of(g0n)]);
          s0_issued = true;
        }
        if (!(ok = mbar_wait(&bars.p_full[x], jt & 1, ab, dev_err))) break;
        tc_fence_after();
        issue_pv<D>(tO, tP, v_desc(iv), j > 0);
        umma_commit(&bars.pv_done[x]);
      } else {
        // P lives in the S columns: PV_X(j) must be issued before S_X(j+1).
        if (!(ok = mbar_wait(&bars.p_full[x], jt & 1, ab, dev_err))) break;
        tc_fence_after();
        issue_pv<D>(tO, tP, v_desc(iv), j > 0);
        umma_commit(&bars.pv_done[x]);
        if (more) {
          issue_qk<D>(tS, q_desc, k_desc(ik));
          umma_commit(&bars.s_full[x]);
        }
      }
      if (j == nkv - 1) {
        umma_commit(&bars.o_done[x]);
        umma_commit(&bars.q_empty[b]);
      }
      umma_commit(&bars.empty[slot_of(iv)]);
      if (more) umma_commit(&bars.empty[slot_of(ik)]);
    }
    jx += nkv;
  }
  // Every MMA this thread issued has completed once this barrier flips.
  umma_commit(&bars.drain[x]);
  mbar_wait_drain(&bars.drain[x], 0);
}

// Softmax / epilogue of one 128-row query tile (x = 0: tile A, 1: tile B).
template <int D, class W>
__device__ void fwd_softmax(uint8_t* sm, FwdBars& bars, uint32_t tmem, int x, const W& w, float scale_log2,
                            const CUtensorMap* map_o, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                            uint32_t* dev_err) {
  using C = FwdCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS + x * 128;
  const uint32_t tO = tmem + lane_base + C::kColO + x * D;
  const uint32_t tP = tmem + lane_base + C::kColP + x * C::kPStride;
  volatile int* ab = &bars.abort;
  const size_t rows = static_cast<size_t>(w.seg.rows);
  int jx = 0;       // key tiles processed by this query-tile slot (barrier phases)
  uint32_t uc = 0;  // units processed by this slot (o_done phases)
  uint32_t us = 0;  // tiles stored through the staging buffer (epi phases)
  bool ok = true;
  for (int u = blockIdx.x; ok && u < w.units; u += gridDim.x) {
  const FwdUnit un = w.unit(u);
  if (x == 1 && !un.has_b) continue;
  // Per-unit values, so that the tile loop keeps few of them live.
  const int nkv = un.nkv;
  const int qt0 = un.q0 + x * 128;  // the tile's first row
  const int n = qt0 + row;
  const int nvalid_last = un.end - (un.kvb + (nkv - 1) * kTileN);  // keys of the last key tile
  const bool live = n < un.end;
  // The staged tile store writes whole 128-row tiles, clipped only at the
  // head's last row: a tile that runs past its segment into the next one
  // stores rows instead.
  const bool tile_store = C::kStageO && (qt0 + 128 <= un.end || un.end == w.seg.rows);
  const size_t orow = static_cast<size_t>(un.bh) * rows + (live ? n : 0);  // the row's index in O / LSE
  const int bh = un.bh;
  float m_ref = -INFINITY;
  float l = 0.f;
  for (int j = 0; j < nkv; ++j) {
    const int jt = jx + j;
    ok = mbar_wait(&bars.s_full[x], jt & 1, ab, dev_err);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    // The whole 128-score row in registers: four loads, one wait.
    uint32_t s[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
    tmem_wait_ld();
    if (C::kSepP) {  // the S columns may be overwritten by S(j+1) now
      tc_fence_before();
      mbar_arrive(&bars.s_free[x]);
    }
    const int nvalid = j + 1 < nkv ? kTileN : nvalid_last;
    if (nvalid < kTileN) {  // only the ragged last key tile needs the mask
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c * 32 + e >= nvalid) s[c][e] = __float_as_uint(-INFINITY);
    }
    // Row max as eight independent partial maxima (short dependency chains).
    float mp[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mp[a] = fmaxf(__uint_as_float(s[a >> 1][(a & 1) * 16]), __uint_as_float(s[a >> 1][(a & 1) * 16 + 1]));
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int e = 2; e < 16; e += 2)
        mp[a] = fmax3(mp[a], __uint_as_float(s[a >> 1][(a & 1) * 16 + e]), __uint_as_float(s[a >> 1][(a & 1) * 16 + e + 1]));
    const float mt = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
    const float m_tile = mt * scale_log2;
    const float m_new = (m_tile > m_ref + kRescaleThreshold) ? m_tile : m_ref;
    const bool need = (m_new != m_ref) && (j > 0);
    const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
    l *= alpha;
    m_ref = m_new;
    const float neg_m = -m_ref;
    // Probabilities and row sum; P (bf16 pairs, 16 packed columns per 32
    // scores) into TMEM.  x = s * scale_log2 - m and the row sum in packed
    // f32x2 arithmetic (two scores per instruction), 2^x on the MUFU unit;
    // masked keys of the ragged last tile give exact zeros.
    const uint64_t scale2 = f2_make(scale_log2, scale_log2);
    const uint64_t negm2 = f2_make(neg_m, neg_m);
    uint64_t l2[8];  // partial row sums: two per 32-column chunk
    // The whole packed P row is formed in registers before the P columns
    // are touched, so the wait for PV(j-1) to release them comes after the
    // exponentials instead of stalling ahead of them.
    uint32_t packed[4][16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      l2[2 * c] = f2_make(0.f, 0.f);
      l2[2 * c + 1] = f2_make(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        float x0, x1;
        f2_split(f2_fma(f2_make(__uint_as_float(s[c][2 * h]), __uint_as_float(s[c][2 * h + 1])), scale2, negm2), x0,
                 x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        l2[2 * c + (h & 1)] = f2_add(l2[2 * c + (h & 1)], f2_make(p0, p1));
        packed[c][h] = pack_bf16x2(p0, p1);
      }
    }
    if (C::kSepP && jt > 0) {
      // PV(jt-1) must be done with the P columns and with O (rescale below).
      ok = mbar_wait(&bars.pv_done[x], (jt - 1) & 1, ab, dev_err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_st16(tP + c * 16, packed[c]);
    {
      float la, lb;
      f2_split(f2_add(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])),
                      f2_add(f2_add(l2[4], l2[5]), f2_add(l2[6], l2[7]))),
               la, lb);
      l += la + lb;
    }
    // Rescale O (after P, when the score registers are free); PV(j) waits for
    // this tile's p_full, so O is not being accumulated meanwhile.
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(tO + c * 32, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars.p_full[x]);
  }
  if (!ok) return;
  ok = mbar_wait(&bars.o_done[x], uc & 1, ab, dev_err);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return;
  tc_fence_after();
  const float inv_l = 1.f / l;
  if (tile_store) {
    // O rows into the query tile's staging tile (128-byte swizzle: 16-byte
    // chunk c of row r at c ^ (r & 7)), then one TMA store of the tile; rows
    // past N fall outside the tensor and are not written.
    const uint32_t stage = smem_u32(sm + C::kOffStage + x * C::kQTileBytes);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t chunk = static_cast<uint32_t>(c * 4 + g) ^ static_cast<uint32_t>(row & 7);
        st_shared_v4(stage + row * 128 + (chunk << 4),
                     pack_bf16x2(__uint_as_float(o[g * 8 + 0]) * inv_l, __uint_as_float(o[g * 8 + 1]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[g * 8 + 2]) * inv_l, __uint_as_float(o[g * 8 + 3]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[g * 8 + 4]) * inv_l, __uint_as_float(o[g * 8 + 5]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[g * 8 + 6]) * inv_l, __uint_as_float(o[g * 8 + 7]) * inv_l));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.epi[x]);
    if (row == 0) {
      // Every row is staged; the store has read the tile before this thread
      // goes on (the next unit's rows reuse it only after this tile's
      // p_full, which counts this thread).
      if (mbar_wait(&bars.epi[x], us & 1, ab, dev_err)) {
        tma_store_3d(map_o, sm + C::kOffStage + x * C::kQTileBytes, 0, qt0, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
    ++us;
  } else {
    uint4* orow_p = reinterpret_cast<uint4*>(out + orow * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_wait_ld();
      if (live) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w4;
          w4.x = pack_bf16x2(__uint_as_float(o[g * 8 + 0]) * inv_l, __uint_as_float(o[g * 8 + 1]) * inv_l);
          w4.y = pack_bf16x2(__uint_as_float(o[g * 8 + 2]) * inv_l, __uint_as_float(o[g * 8 + 3]) * inv_l);
          w4.z = pack_bf16x2(__uint_as_float(o[g * 8 + 4]) * inv_l, __uint_as_float(o[g * 8 + 5]) * inv_l);
          w4.w = pack_bf16x2(__uint_as_float(o[g * 8 + 6]) * inv_l, __uint_as_float(o[g * 8 + 7]) * inv_l);
          orow_p[c * 4 + g] = w4;
        }
      }
    }
  }
  if (live) lse[orow] = (m_ref + lg2_approx(l)) * kLn2;
  jx += nkv;
  ++uc;
  }
  if (C::kStageO && row == 0) bulk_wait_group0();
}

template <int D, class W>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                    const __grid_constant__ W w, float scale_log2,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* dq_zero, uint32_t* zero_count,
                    uint32_t* dev_err) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBars bars;
  uint8_t* sm = align1024(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 2);  // one commit per MMA issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.q_full[b], 1);
      mbar_init(&bars.q_empty[b], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.p_full[x], 128);
      mbar_init(&bars.o_done[x], 1);
      mbar_init(&bars.pv_done[x], 1);
      mbar_init(&bars.s_free[x], 128);
      mbar_init(&bars.drain[x], 1);
      mbar_init(&bars.epi[x], 4);
    }
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  griddep_wait();  // the previous grid's writes (q_hat, k_hat) are visible from here on
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp >= 8) {
    setmaxnreg_dec<kRegOtherFwd>();
    if (warp == 8) {
      if (lane == 0) fwd_producer<D>(&map_q, &map_k, &map_v, sm, bars, w, dev_err);
    } else if (warp == 11) {
      if (dq_zero) fwd_zero_dq<D>(w, dq_zero, zero_count, lane);
    } else {
      if (lane == 0) fwd_mma<D>(sm, bars, tmem, warp - 9, w, dev_err);
    }
  } else {
    setmaxnreg_inc<kRegSoftmax>();
    fwd_softmax<D>(sm, bars, tmem, warp >> 2, w, scale_log2, &map_o, out, lse, dev_err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, class W>
cudaError_t launch_fwd_w(const W& w, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const AttnShape& s, uint16_t* out, float* lse, float* dq_zero, uint32_t* zero_count,
                         uint32_t* dev_err, cudaStream_t st) {
  using C = FwdCfg<D>;
  static_assert(C::kDynSmem + static_cast<int>(sizeof(FwdBars)) <= 232448, "shared memory budget");
  auto kernel = attn_fwd_kernel<D, W>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split is valid only for the register count it was sized
  // for; any other build is refused rather than launched.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kRegLaunchFwd) return cudaErrorInvalidConfiguration;
  const int sms = device_sm_count();
  const int grid = w.units < sms ? w.units : sms;
  const float scale_log2 = s.scale * 1.4426950408889634f;
  CUtensorMap mo;  // the output, for the staged tile stores (d = 64)
  if (!encode_bhnd_map(&mo, out, s.BH, s.N, D)) return cudaErrorInvalidValue;
  return launch_pdl(kernel, dim3(grid), dim3(kFwdThreads), C::kDynSmem, st, mq, mk, mv, mo, w, scale_log2,
                    reinterpret_cast<__nv_bfloat16*>(out), lse, dq_zero, zero_count, dev_err);
}

// Work units (256 query rows of one head's segment) of a launch.
int fwd_units(const AttnShape& s) {
  int upc = 0;
  for (int i = 0; i < s.seg.n; ++i) upc += (s.seg.cu[i + 1] - s.seg.cu[i] + 2 * kTileM - 1) / (2 * kTileM);
  return s.BH * upc;
}

template <int D>
cudaError_t launch_fwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const AttnShape& s,
                         uint16_t* out, float* lse, float* dq_zero, uint32_t* zero_count, uint32_t* dev_err,
                         cudaStream_t st) {
  if (s.seg.n == 1) {
    FwdWorkUniform w;
    w.seg.rows = s.seg.rows;
    w.upc = (s.seg.rows + 2 * kTileM - 1) / (2 * kTileM);
    w.nkv = (s.seg.rows + kTileN - 1) / kTileN;
    w.units = s.BH * w.upc;
    return launch_fwd_w<D>(w, mq, mk, mv, s, out, lse, dq_zero, zero_count, dev_err, st);
  }
  FwdWork w;
  w.seg = s.seg;
  w.uf[0] = 0;
  for (int i = 0; i < s.seg.n; ++i)
    w.uf[i + 1] = w.uf[i] + (s.seg.cu[i + 1] - s.seg.cu[i] + 2 * kTileM - 1) / (2 * kTileM);
  w.upc = w.uf[s.seg.n];
  w.units = s.BH * w.upc;
  return launch_fwd_w<D>(w, mq, mk, mv, s, out, lse, dq_zero, zero_count, dev_err, st);
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const AttnShape& s, uint16_t* out, float* lse, uint32_t* dev_err, cudaStream_t st,
                            float* dq_zero, uint32_t* zero_count) {
  if (s.d == 64) return launch_fwd_d<64>(map_q, map_k, map_v, s, out, lse, dq_zero, zero_count, dev_err, st);
  if (s.d == 128) return launch_fwd_d<128>(map_q, map_k, map_v, s, out, lse, dq_zero, zero_count, dev_err, st);
  return cudaErrorInvalidValue;
}

int attn_fwd_grid(const AttnShape& s) {
  const int units = fwd_units(s);
  const int sms = device_sm_count();
  return units < sms ? units : sms;
}

}  // namespace jattn
