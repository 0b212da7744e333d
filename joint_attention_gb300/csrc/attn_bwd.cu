// attn_bwd.cu — softmax attention backward on tcgen05 tensor cores.
//
// Gradient of L = sum(dO * O) with O = softmax(s q_hat k_hat^T) V, P never
// stored: it is recomputed from the forward's log-sum-exp (the re-diffusion
// README's "attention fix" section: the fused kernels keep the N x N matrix
// out of memory in the backward too).  Per key tile j and query tile i:
//
//   S^T  = K_j Q_i^T            P^T  = exp(s S^T - LSE_i)      (per column)
//   dP^T = V_j dO_i^T           dS^T = P^T * (dP^T - D_i),  D = rowsum(dO*O)
//   dV_j += P^T dO_i            dK_j += dS^T Q_i              (TMEM accumulators)
//   dQ_i += dS K_j              (TMA fp32 reduce-add into a global accumulator)
//
// Work unit: one 128-key tile j of one segment of one head (a (b, h) of the
// [B, H, N, d] layout, or one sequence of a packed variable-length call),
// streaming every query tile of that segment.  The kernel is persistent: one
// CTA per SM walks the units u = blockIdx.x, blockIdx.x + gridDim.x, ...
// with every barrier phase running on across units, so the next unit's K/V
// load and first S / dP products overlap the current unit's last tiles and
// its epilogue.
// 640 threads (five warpgroups; setmaxnreg splits the registers per role,
// see the budgets below):
//
//   warps 0-3   compute group 0: query columns 0-63 of each tile;
//   warps 4-7   compute group 1: query columns 64-127.  One thread per key
//               row (TMEM lane).  P^T is written into TMEM as packed bf16
//               (A operand of the dV MMA).  dS^T goes to shared memory in
//               the MMA's swizzled layout (read MN-major as the A operand of
//               dQ) and, d = 64, into TMEM over the group's own dP^T columns
//               as the A operand of dK (d = 128: dK reads the shared tile).
//   warps 8-11  dQ drain, one thread per query row: dQ_i from TMEM into
//               swizzled 128 x 32 fp32 staging tiles, each added into the
//               global accumulator by one TMA tensor reduce (d = 128: two of
//               the four tiles over the query tile's finished Q stage);
//               d = 128, also the unit epilogue.
//   warps 12-15 d = 64 unit epilogue, one thread per key row: dv, and the
//               K-RMSNorm backward of dK (dk and the unit's dgk partial),
//               built in the unit's own K/V buffer once the MMAs are done
//               with it; the TMEM accumulators are released as soon as they
//               are read.
//   warp 16     TMA producer: K_j, V_j per unit (double-buffered for d = 64);
//               per query tile Q_i and dO_i through rings, with the tile's
//               softmax statistics (a bf16 chunk for the MMAs).
//   warps 17-19 MMA issuers (d = 64): recompute (S, dK, dP), dV, and dQ;
//               d = 128 uses warp 17 alone.
//
// d = 64: TMEM (512 columns) S^T [0,128), dP^T [128,256) (then dS^T),
// dV [256,320), dK [320,384), dQ [384,448), P^T [448,512) (packed bf16).
// S(i+1) is computed as soon as the compute groups hold S^T(i) in registers
// (s_free); dP(i+1) once dK(i) has read dS^T(i) out of the dP^T columns;
// P^T(i+1) is written only after dV(i) has read P^T(i).  The statistics
// enter as one more K = 16 step of the S^T and dP^T products, so TMEM holds
// S^T - LSE / scale and dP^T - D.
//
// d = 128: TMEM S^T/P^T [0,128), dP^T [128,256), dV [256,384), dK [384,512),
// dQ over the dP^T columns; one issuer in the order dV(i), dK(i), dQ(i),
// S(i+1), dP(i+1), with dP(i+1) waiting for dQ(i) to be out of TMEM.
#include <cuda_bf16.h>

#include <type_traits>

#include "jattn_internal.h"
#include "sm103_ptx.cuh"

namespace jattn {
namespace {

constexpr int kBwdThreads = 640;  // 5 warpgroups
// Warp roles: 0-7 compute (two groups), 8-11 dQ drain, 12-15 epilogue
// (d = 64), 16 TMA, 17-19 MMA issuers.  Registers per thread (setmaxnreg):
// d = 64: compute 120, drain 88, epilogue 104, TMA / issuers 48;
// 256 x 120 + 128 x (88 + 104 + 48) = 61440, the 640 x 96 the block launches
// with (112 / 88 / 112 / 56 spills nothing but runs slower: the compute
// warps want the registers).  d = 128: compute 128, drain + epilogue 104,
// the idle warps 12-15 24, TMA / issuer 96 (their launch count, no
// setmaxnreg); 256 x 128 + 128 x (104 + 24 + 96) = 61440.  The issuers spill
// below 96.
// setmaxnreg budgets.  An increase must not be below, a decrease not above,
// the count the kernel launches with, and the sum must fit the launch's
// registers (640 x that count); the launcher checks both against the
// compiled kernel before every launch.
constexpr int kRegCompute64 = 120, kRegDrain64 = 88, kRegEpi64 = 104, kRegMma64 = 48;
constexpr int kRegCompute128 = 128, kRegDrain128 = 104, kRegIdle128 = 24, kRegMma128 = 96;
// The split uses the whole launch allocation (640 x 96): the kernel must launch
// with exactly 96 registers per thread.
constexpr int kRegLaunchMin = 96, kRegLaunchMax = 96;
// Each SM sub-partition holds one warp of every warpgroup (warp w on w % 4),
// and setmaxnreg.inc draws only on the registers its five warps were launched
// with (5 x 32 x 96): a warp's increase that the decreases on its own
// sub-partition do not cover waits forever.  So the five warps of every
// sub-partition must fit the launch allocation of five warps.
constexpr int kSubPartRegs = 5 * 32 * kRegLaunchMin;
static_assert(32 * (2 * kRegCompute64 + kRegDrain64 + kRegEpi64 + kRegMma64) <= kSubPartRegs,
              "d = 64 register split exceeds a sub-partition's launch allocation");
static_assert(32 * (2 * kRegCompute128 + kRegDrain128 + kRegIdle128 + kRegMma128) <= kSubPartRegs,
              "d = 128 register split exceeds a sub-partition's launch allocation");
static_assert(256 * kRegCompute64 + 128 * (kRegDrain64 + kRegEpi64 + kRegMma64) <= kBwdThreads * kRegLaunchMin,
              "d = 64 register split exceeds the launch allocation");
static_assert(256 * kRegCompute128 + 128 * (kRegDrain128 + kRegIdle128 + kRegMma128) <= kBwdThreads * kRegLaunchMin,
              "d = 128 register split exceeds the launch allocation");
static_assert(kRegEpi64 >= kRegLaunchMax && kRegMma64 <= kRegLaunchMin && kRegDrain128 >= kRegLaunchMax && kRegIdle128 <= kRegLaunchMin &&
                  kRegMma128 <= kRegLaunchMin &&
                  kRegDrain64 <= kRegLaunchMin && kRegCompute64 >= kRegLaunchMax && kRegCompute128 >= kRegLaunchMax,
              "setmaxnreg direction");
constexpr int kWarpEpi = 12;
constexpr int kWarpTma = 16;
constexpr int kWarpMma0 = 17;  // recompute issuer (d = 128: the only one)
constexpr int kWarpMma1 = 18;  // dV issuer
constexpr int kWarpMma2 = 19;  // dQ issuer
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128 x d bf16 tile
  static constexpr int kQStages = (D == 64) ? 3 : 2;
  static constexpr int kDOStages = (D == 64) ? 2 : 1;
  static constexpr int kDSBufs = 1;
  // K/V buffers: two let the next unit's keys load during the current unit.
  static constexpr int kKVBufs = (D == 64) ? 2 : 1;
  // d = 64: three MMA issuers (S, dK, dP; dV; dQ) and
  // P^T in its own TMEM columns.  d = 128: one issuer, P^T over S^T.
  static constexpr bool kSplitIssuers = (D == 64);
  // The softmax statistics enter through the tensor cores.  Each query tile
  // brings a 16-column bf16 chunk B of its rows' -LSE / scale and -D, each
  // split into three bf16 terms (columns 0-2 and 3-5), and one more K = 16
  // step of the S^T and dP^T products with a constant A chunk (ones in
  // columns 0-2, resp. 3-5, of every key row) gives S^T - LSE / scale and
  // dP^T - D directly in TMEM.  The compute warps then read no per-query
  // values from shared memory.
  static constexpr int kStatsChunk = 128 * 16 * 2;             // 128 rows x 16 bf16, 32-byte swizzle
  // The constant A chunks repeat one 8-row atom (256 bytes) with a zero atom
  // stride, so each takes 256 bytes.
  static constexpr int kConstAtom = 256;
  // dQ staging: 128 x 32 fp32 tiles (128-byte rows, 128-byte swizzle), each
  // reduced into the accumulator by one TMA tensor reduce; d = 64 has two of
  // its own, d = 128 one (two more lie over the query tile's Q stage).
  static constexpr int kDQStageBytes = (D == 64) ? 2 * 128 * 128 : 128 * 128;
  static constexpr int kOffKV = 0;                            // + buf * 2 * kTile: K, then V
  static constexpr int kOffQ = kKVBufs * 2 * kTile;           // + stage * kTile
  static constexpr int kOffDO = kOffQ + kQStages * kTile;     // + stage * kTile
  static constexpr int kOffDS = kOffDO + kDOStages * kTile;   // + buf * 32 KB (128 x 128 bf16)
  static constexpr int kOffStats = kOffDS + kDSBufs * 128 * 128 * 2;          // + stage * kStatsChunk
  static constexpr int kOffConst = kOffStats + kQStages * kStatsChunk;  // S, then dP
  static constexpr int kOffDQ = kOffConst + 1024;
  static constexpr int kTileBytes = kOffDQ + kDQStageBytes;
  static constexpr int kDynSmem = kTileBytes + 1024;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 128;
  static constexpr uint32_t kColP = (D == 64) ? 448 : 0;  // P^T (packed bf16)
  static constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV (A in TMEM), dK
  static constexpr uint32_t kIdescMM = idesc_bf16_f32(128, D, true, true);      // dQ
  static __device__ __forceinline__ int off_k(int b) { return kOffKV + b * 2 * kTile; }
  static __device__ __forceinline__ int off_v(int b) { return kOffKV + b * 2 * kTile + kTile; }
};

// Units: one 128-key tile of one segment of one head.  Per head the units
// run over the segments' 128-row tiles in order (unit index k within the
// head is the segment's first padded row / 128 plus the key tile j); CTA c
// takes u = c, c + gridDim.x, ...  Each unit visits every query tile of its
// own segment.  Query tiles are counted on across units (t runs over all
// query tiles of the CTA's units), and every ring / handshake barrier takes
// its phase from that count.
// dQ accumulation order.  kDqArrival: every key tile's contribution is a
// bulk reduce-add into a zeroed accumulator, in whatever order they land (the
// default; dq and dgq repeat to rounding).  kDqRotated / kDqAscending: the
// deterministic mode, a fixed order per query tile (see bwd_drain64).
enum : int { kDqArrival = 0, kDqRotated = 1, kDqAscending = 2 };

struct BwdUnit {
  int bh;     // head
  int j;      // key tile within the segment
  int nkt;    // 128-row tiles of the segment (key tiles == query tiles)
  int row0;   // the segment's first row in the head
  int end;    // one past its last row
  int prow0;  // its first row in the padded per-head scratch
  int ord;    // dQ order: kDqArrival, kDqRotated or kDqAscending
  // The i-th query tile visited: except in the ascending order, the key tiles
  // of one segment (which run side by side on neighbouring CTAs) start at
  // different query tiles, so that their dQ contributions go to different
  // rows at any one time.
  __device__ __forceinline__ int query_tile(int i) const {
    if (ord == kDqAscending) return i;
    const int q = i + j;
    return q < nkt ? q : q - nkt;
  }
  // Ordered modes: contributions to that query tile's accumulator made before
  // this one.
  __device__ __forceinline__ int rank(int i) const { return ord == kDqAscending ? j : i; }
  __device__ __forceinline__ int kv0() const { return row0 + 128 * j; }  // first key row
};

// The [B, H, N, d] layout: one segment [0, N) per head, decoded without the
// segment table.
struct BwdWorkUniform {
  int upc;    // 128-row tiles per head
  int units;  // heads * upc
  int ord;    // dQ order
  struct {
    int rows, prows;
  } seg;
  __device__ __forceinline__ BwdUnit unit(int u) const {
    BwdUnit r;
    r.bh = u / upc;
    r.j = u - r.bh * upc;
    r.nkt = upc;
    r.row0 = 0;
    r.end = seg.rows;
    r.prow0 = 0;
    r.ord = ord;
    return r;
  }
};

// Packed variable-length layout: segments from the table.
struct BwdWork {
  int upc;    // units per head (padded rows per head / 128)
  int units;  // heads * upc
  int ord;    // dQ order
  SegTable seg;
  __device__ __forceinline__ BwdUnit unit(int u) const {
    BwdUnit r;
    r.bh = u / upc;
    const int k = u - r.bh * upc;
    int lo = 0, hi = seg.n;  // seg.pcu[lo] <= 128 k < seg.pcu[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg.pcu[mid] <= 128 * k) lo = mid;
      else hi = mid;
    }
    r.j = k - seg.pcu[lo] / 128;
    r.nkt = (seg.pcu[lo + 1] - seg.pcu[lo]) / 128;
    r.row0 = seg.cu[lo];
    r.end = seg.cu[lo + 1];
    r.prow0 = seg.pcu[lo];
    r.ord = ord;
    return r;
  }
};

struct BwdBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t kv_mmadone[2];  // d = 64: the unit's MMAs are done with K/V buffer b
  uint64_t q_full[3], q_empty[3];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, dp_full;
  uint64_t p_ready, ds_ready;
  uint64_t ds_free[2];
  uint64_t dq_full, dq_free;
  uint64_t acc_full;                // a unit's dV / dK accumulators are final
  uint64_t acc_free_v, acc_free_k;  // ... and have been read out of TMEM
  uint64_t s_free;
  uint64_t dv_done;
  uint64_t epi;
  uint64_t drain_sync;  // the dQ drain threads' staging handshakes
  uint64_t kraw_full;   // d = 64: the unit's raw k tile has landed (epilogue)
  uint64_t drain[3];
  uint32_t tmem_base;
  int abort;
  __align__(16) float gk[128];  // K-RMSNorm gain (d entries)
  __align__(16) float wsum[4][128];  // unit epilogue: per-warp dgk column sums
  float dgk_cta[128];               // this CTA's dgk partial, summed over its units in unit order
};

__device__ __forceinline__ uint8_t* align1024b(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int D, class W>
__device__ void bwd_producer(const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                             const CUtensorMap* mdo, const CUtensorMap* mstats, uint8_t* sm, BwdBars& bars,
                             const W& w, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  tma_prefetch_desc(mq);
  tma_prefetch_desc(mk);
  tma_prefetch_desc(mv);
  tma_prefetch_desc(mdo);
  tma_prefetch_desc(mstats);
  volatile int* ab = &bars.abort;
  int nkv_issued = 0, nq_issued = 0, ndo_issued = 0;
  bool ok = true;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const BwdUnit un = w.unit(u);
    const int bh = un.bh, kv0 = un.kv0();
    const int b = ui % C::kKVBufs;
    if (ui >= C::kKVBufs && !(ok = mbar_wait(&bars.kv_empty[b], ((ui / C::kKVBufs) - 1) & 1, ab, dev_err))) break;
    mbar_arrive_expect_tx(&bars.kv_full[b], 2u * C::kTile);
    for (int blk = 0; blk < D / 64; ++blk) {
      tma_load_3d(sm + C::off_k(b) + blk * 16384, mk, &bars.kv_full[b], blk * 64, kv0, bh);
      tma_load_3d(sm + C::off_v(b) + blk * 16384, mv, &bars.kv_full[b], blk * 64, kv0, bh);
    }
    ++nkv_issued;
    for (int i = 0; i < un.nkt; ++i) {
      const int t = tb + i;
      const int qs = t % C::kQStages;
      if (t >= C::kQStages && !(ok = mbar_wait(&bars.q_empty[qs], ((t / C::kQStages) - 1) & 1, ab, dev_err))) break;
      const int qi = un.query_tile(i);
      mbar_arrive_expect_tx(&bars.q_full[qs], C::kTile + C::kStatsChunk);
      tma_load_3d(sm + C::kOffStats + qs * C::kStatsChunk, mstats, &bars.q_full[qs], 0, un.prow0 + qi * 128, bh);
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d(sm + C::kOffQ + qs * C::kTile + blk * 16384, mq, &bars.q_full[qs], blk * 64, un.row0 + qi * 128,
                    bh);
      ++nq_issued;
      const int ds = t % C::kDOStages;
      if (t >= C::kDOStages && !(ok = mbar_wait(&bars.do_empty[ds], ((t / C::kDOStages) - 1) & 1, ab, dev_err)))
        break;
      mbar_arrive_expect_tx(&bars.do_full[ds], C::kTile);
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d(sm + C::kOffDO + ds * C::kTile + blk * 16384, mdo, &bars.do_full[ds], blk * 64,
                    un.row0 + qi * 128, bh);
      ++ndo_issued;
    }
    tb += un.nkt;
  }
  if (*ab) {
    // Aborted: let the copies already in flight land before the CTA exits.
    for (int t = (nkv_issued > C::kKVBufs ? nkv_issued - C::kKVBufs : 0); t < nkv_issued; ++t)
      mbar_wait_drain(&bars.kv_full[t % C::kKVBufs], (t / C::kKVBufs) & 1);
    for (int t = (nq_issued > C::kQStages ? nq_issued - C::kQStages : 0); t < nq_issued; ++t)
      mbar_wait_drain(&bars.q_full[t % C::kQStages], (t / C::kQStages) & 1);
    for (int t = (ndo_issued > C::kDOStages ? ndo_issued - C::kDOStages : 0); t < ndo_issued; ++t)
      mbar_wait_drain(&bars.do_full[t % C::kDOStages], (t / C::kDOStages) & 1);
  }
}

// The MMA helpers take base shared-memory descriptors built once by the MMA
// thread and advance them by (byte offset >> 4) per 16-wide K step.
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t byte_off) { return desc + (byte_off >> 4); }

// D[tmem] = A * B^T with A, B K-major 128 x d tiles (d/16 MMAs of K = 16).
template <int D>
__device__ __forceinline__ void mma_kk(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
    umma_bf16_ss(tmem_d, dadd(a, off), dadd(b, off), idesc, kk > 0 ? 1u : 0u);
  }
}

// dV (+)= P^T dO: A = P^T from TMEM over the S^T columns (queries 0-63
// packed in columns [0,32), queries 64-127 in [64,96)), B = dO tile stored
// query-rows x d (MN-major).
template <int D>
__device__ __forceinline__ void mma_dv(uint32_t tmem_d, uint32_t tmem_p, uint64_t b, bool accumulate) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t acol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
    umma_bf16_ts(tmem_d, tmem_p + acol, dadd(b, kk * 2048), C::kIdescKM, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// dV (+)= P^T dO with P^T in its own 64 TMEM columns (queries 16kk..16kk+15
// packed at columns 8kk..8kk+7), B = dO tile stored query-rows x d.
template <int D>
__device__ __forceinline__ void mma_dv_sep(uint32_t tmem_d, uint32_t tmem_p, uint64_t b, bool accumulate) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16_ts(tmem_d, tmem_p + kk * 8, dadd(b, kk * 2048), C::kIdescKM, (accumulate || kk > 0) ? 1u : 0u);
}

// dK (+)= dS^T Q: A = dS^T (K-major over queries), B = Q tile stored
// query-rows x d (MN-major).
template <int D>
__device__ __forceinline__ void mma_dk(uint32_t tmem_d, uint64_t a, uint64_t b, bool accumulate) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
    umma_bf16_ss(tmem_d, dadd(a, aoff), dadd(b, kk * 2048), C::kIdescKM, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// dK (+)= dS^T Q with dS^T in TMEM over the dP^T columns (queries 0-63
// packed in columns [0,32), queries 64-127 in [64,96)), B = Q tile stored
// query-rows x d (MN-major).
template <int D>
__device__ __forceinline__ void mma_dk_ts(uint32_t tmem_d, uint32_t tmem_ds, uint64_t b, bool accumulate) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t acol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
    umma_bf16_ts(tmem_d, tmem_ds + acol, dadd(b, kk * 2048), C::kIdescKM, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// dQ = dS K: A = dS read from the dS^T tile (MN-major), B = K tile stored
// key-rows x d (MN-major); K = 128 keys.
template <int D>
__device__ __forceinline__ void mma_dq(uint32_t tmem_d, uint64_t a, uint64_t b) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    umma_bf16_ss(tmem_d, dadd(a, kk * 2048), dadd(b, kk * 2048), C::kIdescMM, kk > 0 ? 1u : 0u);
  }
}

// Three-issuer backward (d = 64).  Recompute issuer: S(t) = K Q_t^T - LSE /
// scale once the compute groups hold S(t-1) in registers, then dK(t-1) once
// dS^T(t-1) is in TMEM, then dP(t) = V dO_t^T - D (the statistics by one
// more K step of S and dP, from the query stage's statistics chunk).
// Gradient issuer: dV(t) from P^T in TMEM.  dQ issuer: dQ(t) from the dS^T
// tile in shared memory.  A dO stage is released by commits from its two
// readers (dP, dV), a K/V buffer by the unit's last dP and last dQ, a Q stage
// by its last reader (dK), the dS^T tile by dQ, and a unit's accumulators are
// final once both the dV and the dK issuer have committed.
template <int D, class W>
__device__ void bwd_mma_recompute(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w,
                                  uint32_t* dev_err) {
  using C = BwdCfg<D>;
  volatile int* ab = &bars.abort;
  auto kQ = [=](int t) { return sdesc_sw128(smem_u32(sm + C::kOffQ + (t % C::kQStages) * C::kTile), 16, 1024); };
  auto mQ = [=](int t) { return sdesc_sw128(smem_u32(sm + C::kOffQ + (t % C::kQStages) * C::kTile), 16384, 1024); };
  auto kDO = [=](int t) { return sdesc_sw128(smem_u32(sm + C::kOffDO + (t % C::kDOStages) * C::kTile), 16, 1024); };
  auto kSt = [=](int t) {
    return sdesc_sw32_kmajor(smem_u32(sm + C::kOffStats + (t % C::kQStages) * C::kStatsChunk), 256u);
  };
  const uint64_t kOnesS = sdesc_sw32_kmajor(smem_u32(sm + C::kOffConst), 0u);
  const uint64_t kOnesD = sdesc_sw32_kmajor(smem_u32(sm + C::kOffConst + C::kConstAtom), 0u);
  // dK(t) is issued one tile late, between S(t+1) and dP(t+1): it reads
  // dS^T(t) out of the dP^T columns, which dP(t+1) then overwrites, and MMAs
  // issued by one thread execute in issue order.
  int pend_t = -1, pend_ui = 0;
  bool pend_first = false, pend_last = false;
  auto issue_dk = [&]() -> bool {
    if (!mbar_wait(&bars.ds_ready, pend_t & 1, ab, dev_err)) return false;
    // The previous unit's dK has been read out of TMEM.
    if (pend_first && pend_ui > 0 && !mbar_wait(&bars.acc_free_k, (pend_ui - 1) & 1, ab, dev_err)) return false;
    tc_fence_after();
    mma_dk_ts<D>(tmem + C::kColDK, tmem + C::kColDP, mQ(pend_t), !pend_first);
    umma_commit(&bars.q_empty[pend_t % C::kQStages]);  // the stage's last reader
    if (pend_last) umma_commit(&bars.acc_full);
    return true;
  };
  bool ok = true;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const int nkt = w.unit(u).nkt;
    const int b = ui % C::kKVBufs;
    if (!(ok = mbar_wait(&bars.kv_full[b], (ui / C::kKVBufs) & 1, ab, dev_err))) break;
    const uint64_t kK = sdesc_sw128(smem_u32(sm + C::off_k(b)), 16, 1024);
    const uint64_t kV = sdesc_sw128(smem_u32(sm + C::off_v(b)), 16, 1024);
    for (int i = 0; i < nkt; ++i) {
      const int t = tb + i;
      if (t > 0 && !(ok = mbar_wait(&bars.s_free, (t - 1) & 1, ab, dev_err))) break;
      if (!(ok = mbar_wait(&bars.q_full[t % C::kQStages], (t / C::kQStages) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_kk<D>(tmem + C::kColS, kK, kQ(t), C::kIdescSS);
      umma_bf16_ss(tmem + C::kColS, kOnesS, kSt(t), C::kIdescSS, 1u);
      umma_commit(&bars.s_full);
      if (pend_t >= 0 && !(ok = issue_dk())) break;
      if (!(ok = mbar_wait(&bars.do_full[t % C::kDOStages], (t / C::kDOStages) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_kk<D>(tmem + C::kColDP, kV, kDO(t), C::kIdescSS);
      umma_bf16_ss(tmem + C::kColDP, kOnesD, kSt(t), C::kIdescSS, 1u);
      umma_commit(&bars.dp_full);
      umma_commit(&bars.do_empty[t % C::kDOStages]);
      pend_t = t;
      pend_ui = ui;
      pend_first = (i == 0);
      pend_last = (i == nkt - 1);
    }
    tb += nkt;
    if (ok) umma_commit(&bars.kv_mmadone[b]);
  }
  if (ok && pend_t >= 0) issue_dk();
  umma_commit(&bars.drain[0]);
  mbar_wait_drain(&bars.drain[0], 0);
}

// Gradient issuer (d = 64): dV(t) += P^T(t) dO_t once P^T(t) is in TMEM.
template <int D, class W>
__device__ void bwd_mma_gradients(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w,
                                  uint32_t* dev_err) {
  using C = BwdCfg<D>;
  volatile int* ab = &bars.abort;
  auto mDO = [=](int t) {
    return sdesc_sw128(smem_u32(sm + C::kOffDO + (t % C::kDOStages) * C::kTile), 16384, 1024);
  };
  bool ok = true;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const int nkt = w.unit(u).nkt;
    for (int i = 0; i < nkt; ++i) {
      const int t = tb + i;
      if (!(ok = mbar_wait(&bars.p_ready, t & 1, ab, dev_err))) break;
      if (!(ok = mbar_wait(&bars.do_full[t % C::kDOStages], (t / C::kDOStages) & 1, ab, dev_err))) break;
      // The previous unit's dV has been read out of TMEM.
      if (i == 0 && ui > 0 && !(ok = mbar_wait(&bars.acc_free_v, (ui - 1) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_dv_sep<D>(tmem + C::kColDV, tmem + C::kColP, mDO(t), i > 0);
      umma_commit(&bars.dv_done);
      umma_commit(&bars.do_empty[t % C::kDOStages]);
    }
    tb += nkt;
    if (ok) umma_commit(&bars.acc_full);
  }
  umma_commit(&bars.drain[1]);
  mbar_wait_drain(&bars.drain[1], 0);
}

// dQ issuer (d = 64): dQ(t) = dS(t) K once dS^T(t) is in shared memory and
// dQ(t-1) has been drained from its TMEM columns.
template <int D, class W>
__device__ void bwd_mma_dq(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  volatile int* ab = &bars.abort;
  const uint64_t mDS = sdesc_sw128(smem_u32(sm + C::kOffDS), 16384, 1024);
  bool ok = true;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const int nkt = w.unit(u).nkt;
    const int b = ui % C::kKVBufs;
    if (!(ok = mbar_wait(&bars.kv_full[b], (ui / C::kKVBufs) & 1, ab, dev_err))) break;
    const uint64_t mK = sdesc_sw128(smem_u32(sm + C::off_k(b)), 16384, 1024);
    for (int i = 0; i < nkt; ++i) {
      const int t = tb + i;
      if (!(ok = mbar_wait(&bars.ds_ready, t & 1, ab, dev_err))) break;
      if (t > 0 && !(ok = mbar_wait(&bars.dq_free, (t - 1) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_dq<D>(tmem + C::kColDQ, mDS, mK);
      umma_commit(&bars.dq_full);
      umma_commit(&bars.ds_free[0]);
    }
    tb += nkt;
    if (ok) umma_commit(&bars.kv_mmadone[b]);
  }
  umma_commit(&bars.drain[2]);
  mbar_wait_drain(&bars.drain[2], 0);
}

// Single-issuer backward (d = 128), per unit: S(0), dP(0), then per tile
// dV(i), S(i+1), dK(i), dQ(i) (into the dP^T columns), dP(i+1) once dQ(i) is
// drained.
template <int D, class W>
__device__ void bwd_mma(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  volatile int* ab = &bars.abort;
  auto qaddr = [=](int t) { return smem_u32(sm + C::kOffQ + (t % C::kQStages) * C::kTile); };
  auto doaddr = [=](int t) { return smem_u32(sm + C::kOffDO + (t % C::kDOStages) * C::kTile); };
  auto dsaddr = [=](int t) { return smem_u32(sm + C::kOffDS + (t % C::kDSBufs) * (128 * 128 * 2)); };
  auto kQ = [=](int t) { return sdesc_sw128(qaddr(t), 16, 1024); };
  auto mQ = [=](int t) { return sdesc_sw128(qaddr(t), 16384, 1024); };
  auto kDO = [=](int t) { return sdesc_sw128(doaddr(t), 16, 1024); };
  auto mDO = [=](int t) { return sdesc_sw128(doaddr(t), 16384, 1024); };
  auto kDS = [=](int t) { return sdesc_sw128(dsaddr(t), 16, 1024); };
  auto mDS = [=](int t) { return sdesc_sw128(dsaddr(t), 16384, 1024); };
  auto q_ph = [](int t) { return static_cast<uint32_t>((t / C::kQStages) & 1); };
  auto do_ph = [](int t) { return static_cast<uint32_t>((t / C::kDOStages) & 1); };
  auto kSt = [=](int t) {
    return sdesc_sw32_kmajor(smem_u32(sm + C::kOffStats + (t % C::kQStages) * C::kStatsChunk), 256u);
  };
  const uint64_t kOnesS = sdesc_sw32_kmajor(smem_u32(sm + C::kOffConst), 0u);
  const uint64_t kOnesD = sdesc_sw32_kmajor(smem_u32(sm + C::kOffConst + C::kConstAtom), 0u);

  bool ok = true;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const int nkt = w.unit(u).nkt;
    const int b = ui % C::kKVBufs;
    const int t0 = tb;
    tb += nkt;
    if (!(ok = mbar_wait(&bars.kv_full[b], (ui / C::kKVBufs) & 1, ab, dev_err))) break;
    const uint32_t aK = smem_u32(sm + C::off_k(b)), aV = smem_u32(sm + C::off_v(b));
    const uint64_t kK = sdesc_sw128(aK, 16, 1024), kV = sdesc_sw128(aV, 16, 1024);
    const uint64_t mK = sdesc_sw128(aK, 16384, 1024);
    if (!(ok = mbar_wait(&bars.q_full[t0 % C::kQStages], q_ph(t0), ab, dev_err))) break;
    tc_fence_after();
    mma_kk<D>(tmem + C::kColS, kK, kQ(t0), C::kIdescSS);
    umma_bf16_ss(tmem + C::kColS, kOnesS, kSt(t0), C::kIdescSS, 1u);
    umma_commit(&bars.s_full);
    // dP(t0) lands where the previous unit's last dQ was drained from.
    if (t0 > 0 && !(ok = mbar_wait(&bars.dq_free, (t0 - 1) & 1, ab, dev_err))) break;
    if (!(ok = mbar_wait(&bars.do_full[t0 % C::kDOStages], do_ph(t0), ab, dev_err))) break;
    tc_fence_after();
    mma_kk<D>(tmem + C::kColDP, kV, kDO(t0), C::kIdescSS);
    umma_bf16_ss(tmem + C::kColDP, kOnesD, kSt(t0), C::kIdescSS, 1u);
    umma_commit(&bars.dp_full);
    for (int i = 0; i < nkt; ++i) {
      const int t = t0 + i;
      // dV(t): needs P^T(t) in TMEM (and the previous unit's dV read out).
      if (!(ok = mbar_wait(&bars.p_ready, t & 1, ab, dev_err))) break;
      if (i == 0 && ui > 0 && !(ok = mbar_wait(&bars.acc_free_v, (ui - 1) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_dv<D>(tmem + C::kColDV, tmem + C::kColS, mDO(t), i > 0);
      umma_commit(&bars.do_empty[t % C::kDOStages]);
      // dK(t): needs dS^T(t) in shared memory (compute is then done with dP(t)).
      if (!(ok = mbar_wait(&bars.ds_ready, t & 1, ab, dev_err))) break;
      if (i == 0 && ui > 0 && !(ok = mbar_wait(&bars.acc_free_k, (ui - 1) & 1, ab, dev_err))) break;
      tc_fence_after();
      mma_dk<D>(tmem + C::kColDK, kDS(t), mQ(t), i > 0);
      umma_commit(&bars.q_empty[t % C::kQStages]);
      // dQ(t) lands in the dP^T columns (dP(t) already consumed); the drain
      // of dQ(t-1) from those columns finished before dP(t) was issued.
      mma_dq<D>(tmem + C::kColDQ, mDS(t), mK);
      umma_commit(&bars.dq_full);
      umma_commit(&bars.ds_free[t % C::kDSBufs]);
      if (i + 1 < nkt) {
        // S(t+1): overwrites the S^T/P^T columns behind dV(t); issued after
        // dK(t) and dQ(t), which lead to dP(t+1) through the dQ drain (the
        // compute groups need S(t+1) no sooner than dP(t+1)).
        if (!(ok = mbar_wait(&bars.q_full[(t + 1) % C::kQStages], q_ph(t + 1), ab, dev_err))) break;
        tc_fence_after();
        mma_kk<D>(tmem + C::kColS, kK, kQ(t + 1), C::kIdescSS);
        umma_bf16_ss(tmem + C::kColS, kOnesS, kSt(t + 1), C::kIdescSS, 1u);
        umma_commit(&bars.s_full);
        if (!(ok = mbar_wait(&bars.dq_free, t & 1, ab, dev_err))) break;
        if (!(ok = mbar_wait(&bars.do_full[(t + 1) % C::kDOStages], do_ph(t + 1), ab, dev_err))) break;
        tc_fence_after();
        mma_kk<D>(tmem + C::kColDP, kV, kDO(t + 1), C::kIdescSS);
        umma_bf16_ss(tmem + C::kColDP, kOnesD, kSt(t + 1), C::kIdescSS, 1u);
        umma_commit(&bars.dp_full);
      }
    }
    if (ok) {
      umma_commit(&bars.acc_full);
      umma_commit(&bars.kv_empty[b]);
    }
  }
  // Every MMA issued above has completed once this barrier flips.
  umma_commit(&bars.drain[0]);
  mbar_wait_drain(&bars.drain[0], 0);
}

// Key-row threads of one compute group (query columns 64g .. 64g+63).
template <int D, class W>
__device__ void bwd_compute(uint8_t* sm, BwdBars& bars, uint32_t tmem, int g, const W& w, float scale,
                            uint32_t* dev_err) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kr = (warp & 3) * 32 + lane;  // key row in the tile == TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS + 64 * g;   // this group's S^T columns
  // P^T: own 32 packed columns (d = 64) or over the group's S^T columns
  const uint32_t tP = C::kSplitIssuers ? tmem + lane_base + C::kColP + 32 * g : tS;
  const uint32_t tDP = tmem + lane_base + C::kColDP + 64 * g;
  const uint32_t swz = static_cast<uint32_t>(kr & 7);
  const uint64_t sc2 = f2_make(scale * kLog2e, scale * kLog2e);
  volatile int* ab = &bars.abort;

  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; u < w.units; u += gridDim.x, ++ui) {
    const BwdUnit un = w.unit(u);
    const bool key_live = un.kv0() + kr < un.end;
    const int t0 = tb;
    tb += un.nkt;
    for (int i = 0; i < un.nkt; ++i) {
      const int t = t0 + i;
      bool ok = mbar_wait(&bars.s_full, t & 1, ab, dev_err);
      if (!__all_sync(0xffffffffu, ok)) return;
      tc_fence_after();
      // P^T = exp2(s log2e S^T - LSE log2e), packed bf16 pairs into TMEM
      // (chunk c -> 16 packed columns at 16c).  Key rows past N get P = 0.
      // TMEM holds S^T - LSE / scale (the statistics step), so only the
      // product by s log2e remains.
      uint32_t pp[32];
      // Both 32-column chunks of this group's S^T in flight at once.
      uint32_t sall[2][32];
      tmem_ld32(tS, sall[0]);
      tmem_ld32(tS + 32, sall[1]);
      tmem_wait_ld();
      if (C::kSplitIssuers) {  // S^T is in registers: S(t+1) may overwrite it
        tc_fence_before();
        mbar_arrive(&bars.s_free);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t(&s)[32] = sall[c];
        if (key_live) {  // warp-uniform except in a head's last key tile
          const uint64_t zero2 = f2_make(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float x0, x1, x2, x3;
            f2_split(f2_fma(f2_make(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sc2, zero2), x0, x1);
            f2_split(f2_fma(f2_make(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])), sc2, zero2), x2, x3);
            pp[(c * 32 + e) / 2] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
            pp[(c * 32 + e) / 2 + 1] = pack_bf16x2(ex2_approx(x2), ex2_approx(x3));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) pp[(c * 32 + e) / 2] = 0u;
        }
      }
      if (C::kSplitIssuers && t > 0) {
        // dV(t-1) must be done reading P^T(t-1) before it is overwritten;
        // waited for after all the exponentials, so that they overlap dV(t-1).
        ok = mbar_wait(&bars.dv_done, (t - 1) & 1, ab, dev_err);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_st16(tP + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pp[c * 16]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars.p_ready);

      ok = mbar_wait(&bars.dp_full, t & 1, ab, dev_err);
      if (!__all_sync(0xffffffffu, ok)) return;
      tc_fence_after();
      const uint32_t ds_row = smem_u32(sm + C::kOffDS + (t % C::kDSBufs) * (128 * 128 * 2)) + g * 16384 + kr * 128;
      uint32_t dsw[2][16];
      {
        uint32_t dpall[2][32];
        tmem_ld32(tDP, dpall[0]);
        tmem_ld32(tDP + 32, dpall[1]);
        tmem_wait_ld();
        // dS = P * bf16(dP - D), dP - D from TMEM: one pack, one bf16x2 product
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            dsw[c][e / 2] = bf16x2_mul(pp[(c * 32 + e) / 2], pack_bf16x2(__uint_as_float(dpall[c][e]),
                                                                          __uint_as_float(dpall[c][e + 1])));
          // d = 64: dS^T(t) also goes over this group's dP^T(t) columns
          // (packed like P^T), where dK(t) reads it; dP(t+1) is issued once
          // dK(t) is done.
          if (C::kSplitIssuers) tmem_st16(tDP + c * 16, dsw[c]);
        }
      }
      // The shared dS^T tile is free once the previous tile's readers are
      // done with it: waited for after the arithmetic, which overlaps them.
      if (t >= C::kDSBufs) {
        ok = mbar_wait(&bars.ds_free[t % C::kDSBufs], ((t / C::kDSBufs) - 1) & 1, ab, dev_err);
        if (!__all_sync(0xffffffffu, ok)) return;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          st_shared_v4(ds_row + ((static_cast<uint32_t>((c * 32 + e) >> 3) ^ swz) << 4), dsw[c][e / 2],
                       dsw[c][e / 2 + 1], dsw[c][e / 2 + 2], dsw[c][e / 2 + 3]);
      if (C::kSplitIssuers) tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bars.ds_ready);
    }
  }
}

// d = 64, warps 8-11 (one thread per query row): per query tile, dQ_t out of
// TMEM into registers and its columns released, then into the two staging
// halves (columns 0-31 and 32-63, 128-byte rows with 16-byte chunks XOR-ed
// by row % 8, so that the row-per-thread writes are free of bank conflicts),
// each added into the fp32 accumulator by one TMA tensor reduce issued by
// thread 0.  Rows past the tensor's end are clipped by the TMA unit; rows of
// the tile that belong to the next segment receive exact zeros (their
// probabilities are 0).  Thread 0 waits for the previous tile's reduces to
// have read the staging before the halves are rewritten.
// Ordered modes: thread 0 also waits, before the tile's reduces, until the
// contributions of lower rank to the query tile are complete (its counter),
// and announces its own once they are complete (at the next tile, or at once
// for a unit's last).  In the [B, H, N, d] layout (whose tiles end at the
// tensor's end) the rank-0 contribution is a TMA store, so that the
// accumulator needs no zeroing beforehand.  (Arrival order keeps the zeroed
// accumulator: a first-store there would make later contributions wait for
// the store's completion, which queues behind the reduces already in flight
// and stalled the drain by microseconds.)
template <int D, bool kOrd, class W>
__device__ void bwd_drain64(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w, const CUtensorMap* mdq,
                            uint32_t* __restrict__ counters, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  static_assert(D == 64, "tiled dQ drain serves d = 64");
  constexpr bool kFirstStore = kOrd && std::is_same<W, BwdWorkUniform>::value;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r128 = (warp & 3) * 32 + lane;  // query row == TMEM lane
  const bool leader = r128 == 0;
  const uint32_t tQ = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kColDQ;
  uint8_t* stage = sm + C::kOffDQ;
  const uint32_t srow = smem_u32(stage) + static_cast<uint32_t>(r128 * 128);
  const uint32_t swz = static_cast<uint32_t>(r128 & 7);
  volatile int* ab = &bars.abort;
  if (leader) tma_prefetch_desc(mdq);
  uint32_t uses = 0;
  // Bounded barrier among the 128 drain threads.
  auto drain_sync = [&]() -> bool {
    mbar_arrive(&bars.drain_sync);
    const bool okb = mbar_wait(&bars.drain_sync, (uses++) & 1, ab, dev_err);
    return __all_sync(0xffffffffu, okb) && !*ab;
  };
  // Thread 0, ordered modes: the counter to announce on once its
  // contribution is complete.
  uint32_t* pend = nullptr;
  auto complete_previous = [&]() {
    if (!pend) return;
    bulk_wait_group0();
    fence_proxy_async_global();
    red_release_gpu_add(pend, 1u);
    pend = nullptr;
  };
  bool ok = true;
  const int tiles_per_head = w.seg.prows / 128;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x; ok && u < w.units; u += gridDim.x) {
    const BwdUnit un = w.unit(u);
    const int t0 = tb;
    tb += un.nkt;
    for (int i = 0; i < un.nkt; ++i) {
      const int t = t0 + i;
      const int qt = un.query_tile(i), rank = un.rank(i);
      uint32_t* cnt = counters + static_cast<size_t>(un.bh) * tiles_per_head + un.prow0 / 128 + qt;
      // Ordered modes: the counter read ahead (its latency overlaps the wait for dQ).
      const uint32_t seen = kOrd && leader && rank > 0 ? ld_acquire_gpu(cnt) : 0u;
      const bool store = kFirstStore && rank == 0;
      ok = mbar_wait(&bars.dq_full, t & 1, ab, dev_err);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      uint32_t a[D];
      tmem_ld32(tQ, *reinterpret_cast<uint32_t(*)[32]>(a));
      tmem_ld32(tQ + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars.dq_free);
      if (leader) {
        if constexpr (kOrd) {
          complete_previous();
          if (rank > 0 && seen < static_cast<uint32_t>(rank)) gwait_geq(cnt, static_cast<uint32_t>(rank), ab, dev_err);
          fence_proxy_async_global();  // the lower ranks' sums before this tile's reduces
        }
        bulk_wait_group_read0();  // the previous tile's reduces have read the staging
      }
      if (!(ok = drain_sync())) break;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int e = h * 32 + 4 * c;
          st_shared_v4(srow + h * 16384 + ((static_cast<uint32_t>(c) ^ swz) << 4), a[e], a[e + 1], a[e + 2], a[e + 3]);
        }
      fence_proxy_async_smem();
      if (!(ok = drain_sync())) break;
      if (leader) {
        const int row = un.row0 + qt * 128;
        if (store) {
          tma_store_3d(mdq, stage, 0, row, un.bh);
          tma_store_3d(mdq, stage + 16384, 32, row, un.bh);
        } else {
          tma_reduce_add_3d(mdq, stage, 0, row, un.bh);
          tma_reduce_add_3d(mdq, stage + 16384, 32, row, un.bh);
        }
        bulk_commit_group();
        if constexpr (kOrd) {
          if (rank != un.nkt - 1) {
            pend = cnt;
            if (i == un.nkt - 1) complete_previous();
          }
        }
      }
    }
  }
  if (leader) {
    if (ok) complete_previous();
    bulk_wait_group0();
  }
}

// d = 128, warps 8-11 (one thread per query row, then per key row).
// Per query tile: dQ_t out of TMEM in four 32-column quarters, staged as
// 128 x 32 fp32 tiles with the 128-byte swizzle (16-byte chunk c of row r at
// c ^ (r % 8), so that the row-per-thread writes are free of bank conflicts)
// and added into the fp32 accumulator by TMA tensor reduces issued by
// thread 0.  One staging tile (H0) is the drain's own; two more (H1, H2) lie
// over the query tile's Q stage, which its last reader dK(t) is done with
// once dQ(t) is complete and which the producer reloads only after the
// reduces have read it (the stage's q_empty also counts thread 0's arrival,
// and their reduces are issued first); the first and fourth quarters wait
// in registers until H0 is free.  All four quarters are out of TMEM before
// dq_free, so that dP(t+1), which lands in those columns, never waits for
// the reduces.  Rows past the tensor's end are clipped by the TMA unit;
// rows of the tile that belong to the next segment receive exact zeros
// (their probabilities are 0).
// Ordered modes, as in bwd_drain64: thread 0 waits, before the tile's first
// reduce, until the contributions of lower rank to the query tile are
// complete (its counter), and announces its own once it is complete (at the
// next tile, or at once for a unit's last); in the [B, H, N, d] layout the
// rank-0 contribution is a TMA store.
// Per unit, once its accumulators are final (one thread per key row):
//   dv = bf16(dV acc);
//   dk_hat = scale * dK acc; u = g * dk_hat; dk = r u - (r^3/d) k sum(u k);
//   dgk partial = column sums over the tile's rows of dk_hat * k * r: a
//   fixed-order reduce-scatter within each warp, then a fixed-order sum of
//   the four warps.
template <int D, bool kOrd, class W>
__device__ void bwd_drain128(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w, float scale,
                             const CUtensorMap* mdq, uint32_t* __restrict__ counters,
                             const __nv_bfloat16* __restrict__ k_raw, const float* __restrict__ rk,
                             __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                             float* __restrict__ dgk_part, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  static_assert(D == 128, "the d = 64 drain is bwd_drain64");
  constexpr bool kFirstStore = kOrd && std::is_same<W, BwdWorkUniform>::value;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r128 = (warp & 3) * 32 + lane;  // TMEM lane: query row (dQ) or key row (dV, dK)
  const bool leader = r128 == 0;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tQ = tmem + lane_base + C::kColDQ;
  const uint32_t tDK = tmem + lane_base + C::kColDK;
  uint8_t* h0 = sm + C::kOffDQ;
  const uint32_t rowoff = static_cast<uint32_t>(r128 * 128);
  const uint32_t swz = static_cast<uint32_t>(r128 & 7);
  auto stage32 = [&](uint8_t* tile, const uint32_t (&a)[32]) {
    const uint32_t base = smem_u32(tile) + rowoff;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      st_shared_v4(base + ((static_cast<uint32_t>(c) ^ swz) << 4), a[4 * c], a[4 * c + 1], a[4 * c + 2],
                   a[4 * c + 3]);
  };
  volatile int* ab = &bars.abort;
  if (leader) tma_prefetch_desc(mdq);
  uint32_t uses = 0, epi_uses = 0;
  // Bounded barriers among the 128 drain threads.
  auto drain_sync = [&]() -> bool {
    mbar_arrive(&bars.drain_sync);
    const bool okb = mbar_wait(&bars.drain_sync, (uses++) & 1, ab, dev_err);
    return __all_sync(0xffffffffu, okb) && !*ab;
  };
  auto epi_sync = [&]() -> bool {
    mbar_arrive(&bars.epi);
    const bool okb = mbar_wait(&bars.epi, (epi_uses++) & 1, ab, dev_err);
    return __all_sync(0xffffffffu, okb);
  };
  // Thread 0, ordered modes: the counter to announce on once its
  // contribution is complete.
  uint32_t* pend = nullptr;
  auto complete_previous = [&]() {
    if (!pend) return;
    bulk_wait_group0();
    fence_proxy_async_global();
    red_release_gpu_add(pend, 1u);
    pend = nullptr;
  };
  bool ok = true;
  const size_t rows = static_cast<size_t>(w.seg.rows);
  const int tiles_per_head = w.seg.prows / 128;
  int tb = 0;  // query tiles of the previous units
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const BwdUnit un = w.unit(u);
    const int bh = un.bh;
    const int t0 = tb;
    tb += un.nkt;
    for (int i = 0; i < un.nkt; ++i) {
      const int t = t0 + i;
      const int qt = un.query_tile(i), rank = un.rank(i);
      uint32_t* cnt = counters + static_cast<size_t>(bh) * tiles_per_head + un.prow0 / 128 + qt;
      // Ordered modes: the counter read ahead (its latency overlaps the wait for dQ).
      const uint32_t seen = kOrd && leader && rank > 0 ? ld_acquire_gpu(cnt) : 0u;
      const bool store = kFirstStore && rank == 0;
      const int row = un.row0 + qt * 128;
      // H1 / H2: the query tile's Q stage, which its last reader dK(t) is
      // done with once dQ(t) is complete.
      uint8_t* h1 = sm + C::kOffQ + (t % C::kQStages) * C::kTile;
      uint8_t* h2 = h1 + 16384;
      ok = mbar_wait(&bars.dq_full, t & 1, ab, dev_err);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      // Columns 32-95 into H1 / H2, whose reduces go first: the producer
      // reloads the Q stage once they have been read.
      uint32_t a[32];
      tmem_ld32(tQ + 32, a);
      tmem_wait_ld();
      stage32(h1, a);
      tmem_ld32(tQ + 64, a);
      tmem_wait_ld();
      stage32(h2, a);
      fence_proxy_async_smem();
      if constexpr (kOrd) {
        if (leader) {
          complete_previous();
          if (rank > 0 && seen < static_cast<uint32_t>(rank)) gwait_geq(cnt, static_cast<uint32_t>(rank), ab, dev_err);
          fence_proxy_async_global();  // the lower ranks' sums before this tile's reduces
        }
      }
      if (!(ok = drain_sync())) break;
      if (leader) {
        if (store) {
          tma_store_3d(mdq, h1, 32, row, bh);
          tma_store_3d(mdq, h2, 64, row, bh);
        } else {
          tma_reduce_add_3d(mdq, h1, 32, row, bh);
          tma_reduce_add_3d(mdq, h2, 64, row, bh);
        }
        bulk_commit_group();
      }
      // Columns 0-31 and 96-127 into registers; then dQ's columns are free.
      uint32_t b[32];
      tmem_ld32(tQ, a);
      tmem_ld32(tQ + 96, b);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars.dq_free);
      // H0 is free once the previous tile's reduces from it have read it
      // (every group but this tile's first).
      if (leader) bulk_wait_group_read<1>();
      if (!(ok = drain_sync())) break;
      stage32(h0, a);
      fence_proxy_async_smem();
      if (!(ok = drain_sync())) break;
      if (leader) {
        if (store) tma_store_3d(mdq, h0, 0, row, bh);
        else tma_reduce_add_3d(mdq, h0, 0, row, bh);
        bulk_commit_group();
        bulk_wait_group_read<1>();                        // H1 and H2 have been read
        mbar_arrive(&bars.q_empty[t % C::kQStages]);  // the producer may reload the Q stage
        bulk_wait_group_read0();        // ... and H0
      }
      if (!(ok = drain_sync())) break;
      stage32(h0, b);
      fence_proxy_async_smem();
      if (!(ok = drain_sync())) break;
      if (leader) {
        if (store) tma_store_3d(mdq, h0, 96, row, bh);
        else tma_reduce_add_3d(mdq, h0, 96, row, bh);
        bulk_commit_group();
        if constexpr (kOrd) {
          if (rank != un.nkt - 1) {
            pend = cnt;
            if (i == un.nkt - 1) complete_previous();
          }
        }
      }
    }
    if (!ok) break;

    // ---- unit epilogue ----
    ok = mbar_wait(&bars.acc_full, ui & 1, ab, dev_err);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    tc_fence_after();
    const int n = un.kv0() + r128;  // key row of this thread
    const bool key_live = n < un.end;
    const size_t row_off = (static_cast<size_t>(bh) * rows + (key_live ? n : 0)) * D;
    const float r = key_live ? rk[static_cast<size_t>(bh) * rows + n] : 0.f;
    const uint4* krow = reinterpret_cast<const uint4*>(k_raw + row_off);
    uint4* dvrow = reinterpret_cast<uint4*>(dv + row_off);
    uint4* dkrow = reinterpret_cast<uint4*>(dk + row_off);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tmem + lane_base + C::kColDV + c * 32, a);
      tmem_wait_ld();
      if (c == D / 32 - 1) {
        tc_fence_before();
        mbar_arrive(&bars.acc_free_v);
      }
      if (key_live) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 o;
          o.x = pack_bf16x2(__uint_as_float(a[q * 8 + 0]), __uint_as_float(a[q * 8 + 1]));
          o.y = pack_bf16x2(__uint_as_float(a[q * 8 + 2]), __uint_as_float(a[q * 8 + 3]));
          o.z = pack_bf16x2(__uint_as_float(a[q * 8 + 4]), __uint_as_float(a[q * 8 + 5]));
          o.w = pack_bf16x2(__uint_as_float(a[q * 8 + 6]), __uint_as_float(a[q * 8 + 7]));
          dvrow[c * 4 + q] = o;
        }
      }
    }
    // The gain, 8 columns at a time (two 16-byte broadcasts).
    auto gain8 = [&](int col, float (&g)[8]) {
      const float4 g0 = *reinterpret_cast<const float4*>(&bars.gk[col]);
      const float4 g1 = *reinterpret_cast<const float4*>(&bars.gk[col + 4]);
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
      g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    };
    // Pass 1 over the dK accumulator: dot = sum_c g_c dk_hat_c k_c (packed
    // f32x2 arithmetic: even and odd columns in two partial sums).
    uint64_t dot2 = f2_make(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tDK + c * 32, a);
      tmem_wait_ld();
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 kw = key_live ? krow[c * 4 + c8] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kx[4] = {kw.x, kw.y, kw.z, kw.w};
        float g[8];
        gain8(c * 32 + c8 * 8, g);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = c8 * 8 + 2 * h;
          const uint64_t ga = f2_mul(f2_make(g[2 * h], g[2 * h + 1]),
                                     f2_make(__uint_as_float(a[e]), __uint_as_float(a[e + 1])));
          dot2 = f2_fma(ga, f2_make(__uint_as_float(kx[h] << 16), __uint_as_float(kx[h] & 0xFFFF0000u)), dot2);
        }
      }
    }
    float dot0, dot1;
    f2_split(dot2, dot0, dot1);
    const float coef = r * r * r * (1.f / D) * scale * (dot0 + dot1);
    const float rs = r * scale;
    const uint64_t rs2 = f2_make(rs, rs), ncoef2 = f2_make(-coef, -coef);
    // Pass 2, per 32-column chunk: dk = r g dk_hat - coef k, and the chunk's
    // dgk terms dk_hat k r summed over the warp's 32 rows by a reduce-scatter
    // (lane L ends with column 32 c + L).
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tDK + c * 32, a);
      tmem_wait_ld();
      if (c == D / 32 - 1) {
        tc_fence_before();
        mbar_arrive(&bars.acc_free_k);
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 kw = key_live ? krow[c * 4 + c8] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kx[4] = {kw.x, kw.y, kw.z, kw.w};
        float y[8], g[8];
        gain8(c * 32 + c8 * 8, g);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = c8 * 8 + 2 * h;
          // Key rows past the segment have r = 0 and k = 0, so their terms vanish.
          const uint64_t x2 = f2_make(__uint_as_float(kx[h] << 16), __uint_as_float(kx[h] & 0xFFFF0000u));
          const uint64_t a2 = key_live ? f2_make(__uint_as_float(a[e]), __uint_as_float(a[e + 1])) : f2_make(0.f, 0.f);
          float p0, p1;
          f2_split(f2_fma(f2_mul(rs2, f2_make(g[2 * h], g[2 * h + 1])), a2, f2_mul(ncoef2, x2)), y[2 * h], y[2 * h + 1]);
          f2_split(f2_mul(f2_mul(a2, x2), rs2), p0, p1);
          a[e] = __float_as_uint(p0);
          a[e + 1] = __float_as_uint(p1);
        }
        if (key_live) {
          uint4 o;
          o.x = pack_bf16x2(y[0], y[1]);
          o.y = pack_bf16x2(y[2], y[3]);
          o.z = pack_bf16x2(y[4], y[5]);
          o.w = pack_bf16x2(y[6], y[7]);
          dkrow[c * 4 + c8] = o;
        }
      }
#pragma unroll
      for (int m = 16, half = 16; m >= 1; m >>= 1, half >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = __uint_as_float(upper ? a[j] : a[j + half]);
          const float keep = __uint_as_float(upper ? a[j + half] : a[j]);
          a[j] = __float_as_uint(keep + __shfl_xor_sync(0xffffffffu, send, m));
        }
      }
      bars.wsum[warp & 3][c * 32 + lane] = __uint_as_float(a[0]);
    }
    if (!(ok = epi_sync())) break;  // the warp sums are complete
    bars.dgk_cta[r128] += ((bars.wsum[0][r128] + bars.wsum[1][r128]) + bars.wsum[2][r128]) + bars.wsum[3][r128];
    if (!(ok = epi_sync())) break;  // ... and read before the next unit rewrites them
  }
  if (leader) {
    if (ok) complete_previous();
    bulk_wait_group0();
  }
  dgk_part[static_cast<size_t>(blockIdx.x) * D + r128] = bars.dgk_cta[r128];
}

// d = 64 epilogue warps (warps 12-15, one thread per key row): per unit,
// once its last dK product is done, dv = bf16(dV acc) and the K-RMSNorm
// backward of dK (dk_hat = scale * acc; u = g * dk_hat; dk = r u - (r^3/d) k
// sum(u k); the unit's dgk partial = column sums of dk_hat * k * r).  The
// tiles are built in the unit's own K/V buffer, which the MMAs have finished
// with (kv_mmadone) and which the producer reloads only after this releases
// it (kv_empty), so that k, dk and dv move with contiguous 512-byte warp
// accesses and no other role waits on this work except through the TMEM
// accumulators, released as soon as they are read.
template <int D, class W>
__device__ void bwd_epilogue_warps(uint8_t* sm, BwdBars& bars, uint32_t tmem, const W& w, float scale,
                                   const CUtensorMap* mkraw, const CUtensorMap* mdk, const CUtensorMap* mdv,
                                   const float* __restrict__ rk,
                                   __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                                   float* __restrict__ dgk_part, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  static_assert(D == 64, "the epilogue warps serve d = 64");
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r128 = (warp & 3) * 32 + lane;  // key row == TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tDK = tmem + lane_base + C::kColDK;
  auto chunk_addr = [](uint32_t tile, int row, int c) {
    return tile + static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
  };
  volatile int* ab = &bars.abort;
  uint32_t epi_uses = 0;
  uint32_t kraw_issued = 0, kraw_done = 0;  // thread 0 issues the raw k tile loads
  if (r128 == 0) {
    tma_prefetch_desc(mkraw);
    tma_prefetch_desc(mdk);
    tma_prefetch_desc(mdv);
  }
  // Bounded barrier among the 128 epilogue threads.
  auto epi_sync = [&]() -> bool {
    mbar_arrive(&bars.epi);
    const bool okb = mbar_wait(&bars.epi, (epi_uses++) & 1, ab, dev_err);
    return __all_sync(0xffffffffu, okb);
  };
  bool ok = true;
  const size_t rows = static_cast<size_t>(w.seg.rows);
  for (int u = blockIdx.x, ui = 0; ok && u < w.units; u += gridDim.x, ++ui) {
    const BwdUnit un = w.unit(u);
    const int bh = un.bh, kv0 = un.kv0();
    const int b = ui % C::kKVBufs;
    const int n = kv0 + r128;
    const bool key_live = n < un.end;
    const int live_rows = un.end - kv0 < 128 ? un.end - kv0 : 128;
    const size_t tile_off = (static_cast<size_t>(bh) * rows + kv0) * D;
    const float r = key_live ? rk[static_cast<size_t>(bh) * rows + n] : 0.f;
    const uint32_t tile_k = smem_u32(sm + C::off_k(b));  // k, then dk
    const uint32_t tile_v = smem_u32(sm + C::off_v(b));  // dv

    ok = mbar_wait(&bars.acc_full, ui & 1, ab, dev_err);
    // ... and the unit's MMAs are done with its K/V buffer.
    if (ok) ok = mbar_wait(&bars.kv_mmadone[b], (ui / C::kKVBufs) & 1, ab, dev_err);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    tc_fence_after();
    // The raw k tile into the unit's K buffer by TMA (the MMAs are done with
    // it), in the same 128-byte swizzled layout the tile had.  Rows past the
    // segment (zero-filled past the tensor's end, the next sequence's rows in
    // a packed call) have r = 0 and zero dK, so they contribute nothing.
    if (r128 == 0) {
      mbar_arrive_expect_tx(&bars.kraw_full, C::kTile);
      tma_load_3d(sm + C::off_k(b), mkraw, &bars.kraw_full, 0, kv0, bh);
      ++kraw_issued;
    }
    // dV out of TMEM into the dv tile (bf16), its columns released.
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tmem + lane_base + C::kColDV + c * 32, a);
      tmem_wait_ld();
      if (c == D / 32 - 1) {
        tc_fence_before();
        mbar_arrive(&bars.acc_free_v);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(chunk_addr(tile_v, r128, c * 4 + q),
                     pack_bf16x2(__uint_as_float(a[q * 8 + 0]), __uint_as_float(a[q * 8 + 1])),
                     pack_bf16x2(__uint_as_float(a[q * 8 + 2]), __uint_as_float(a[q * 8 + 3])),
                     pack_bf16x2(__uint_as_float(a[q * 8 + 4]), __uint_as_float(a[q * 8 + 5])),
                     pack_bf16x2(__uint_as_float(a[q * 8 + 6]), __uint_as_float(a[q * 8 + 7])));
    }
    // dK out of TMEM into registers and its columns released at once: the
    // next unit's first dK product (and through it the next dP product)
    // waits for this read only.
    uint32_t dkr[D];
    tmem_ld32(tDK, *reinterpret_cast<uint32_t(*)[32]>(dkr));
    tmem_ld32(tDK + 32, *reinterpret_cast<uint32_t(*)[32]>(dkr + 32));
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars.acc_free_k);
    ok = mbar_wait(&bars.kraw_full, ui & 1, ab, dev_err);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    ++kraw_done;
    // Pass 1: dot = sum_c g_c dk_hat_c k_c over this thread's row.
    // The gain is read 8 columns at a time (two 16-byte broadcasts).
    auto gain8 = [&](int col, float (&g)[8]) {
      const float4 g0 = *reinterpret_cast<const float4*>(&bars.gk[col]);
      const float4 g1 = *reinterpret_cast<const float4*>(&bars.gk[col + 4]);
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
      g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    };
    // (packed f32x2 arithmetic: even and odd columns in two partial sums)
    uint64_t dot2 = f2_make(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 kw = ld_shared_v4(chunk_addr(tile_k, r128, c * 4 + q));
        const uint32_t kx[4] = {kw.x, kw.y, kw.z, kw.w};
        float g[8];
        gain8(c * 32 + q * 8, g);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = c * 32 + q * 8 + 2 * h;
          const uint64_t ga = f2_mul(f2_make(g[2 * h], g[2 * h + 1]),
                                     f2_make(__uint_as_float(dkr[e]), __uint_as_float(dkr[e + 1])));
          dot2 = f2_fma(ga, f2_make(__uint_as_float(kx[h] << 16), __uint_as_float(kx[h] & 0xFFFF0000u)), dot2);
        }
      }
    }
    float dot0, dot1;
    f2_split(dot2, dot0, dot1);
    const float coef = r * r * r * (1.f / D) * scale * (dot0 + dot1);
    // Key rows past the segment have r = 0 and k = 0, so their terms vanish.
    const float rs = r * scale;
    const uint64_t rs2 = f2_make(rs, rs), ncoef2 = f2_make(-coef, -coef);
    // Pass 2, per 32-column chunk: dk = r g dk_hat - coef k over the k row
    // (in place), and the chunk's dgk terms dk_hat k r summed over the warp's
    // 32 rows by a reduce-scatter (lane L ends with column 32c + L).
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      // The chunk's dK values are dead once read: the dgk terms replace them.
      uint32_t(&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(dkr + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t addr = chunk_addr(tile_k, r128, c * 4 + q);
        const uint4 kw = ld_shared_v4(addr);
        const uint32_t kx[4] = {kw.x, kw.y, kw.z, kw.w};
        uint32_t o[4];
        float g[8];
        gain8(c * 32 + q * 8, g);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = q * 8 + 2 * h;
          const uint64_t x2 = f2_make(__uint_as_float(kx[h] << 16), __uint_as_float(kx[h] & 0xFFFF0000u));
          const uint64_t a2 = f2_make(__uint_as_float(a[e]), __uint_as_float(a[e + 1]));
          float y0, y1, p0, p1;
          f2_split(f2_fma(f2_mul(rs2, f2_make(g[2 * h], g[2 * h + 1])), a2, f2_mul(ncoef2, x2)), y0, y1);
          o[h] = pack_bf16x2(y0, y1);
          f2_split(f2_mul(f2_mul(a2, x2), rs2), p0, p1);
          a[e] = __float_as_uint(p0);
          a[e + 1] = __float_as_uint(p1);
        }
        st_shared_v4(addr, o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int m = 16, half = 16; m >= 1; m >>= 1, half >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = __uint_as_float(upper ? a[j] : a[j + half]);
          const float keep = __uint_as_float(upper ? a[j + half] : a[j]);
          a[j] = __float_as_uint(keep + __shfl_xor_sync(0xffffffffu, send, m));
        }
      }
      bars.wsum[warp & 3][c * 32 + lane] = __uint_as_float(a[0]);
    }
    fence_proxy_async_smem();  // the dk / dv tiles, for the TMA stores
    if (!(ok = epi_sync())) break;  // dk tile, dv tile and warp sums complete
    if (r128 < D)
      bars.dgk_cta[r128] += ((bars.wsum[0][r128] + bars.wsum[1][r128]) + bars.wsum[2][r128]) + bars.wsum[3][r128];
    if (live_rows == 128 || un.end == w.seg.rows) {
      // The tiles out by TMA (rows past the tensor's end are clipped).
      if (r128 == 0) {
        tma_store_3d(mdk, sm + C::off_k(b), 0, kv0, bh);
        tma_store_3d(mdv, sm + C::off_v(b), 0, kv0, bh);
        bulk_commit_group();
        bulk_wait_group_read0();  // read out of the K/V buffer
      }
    } else {
      // A segment's last tile in a packed call: the live rows only, 32
      // consecutive 16-byte chunks per warp access.
      uint4* dkdst = reinterpret_cast<uint4*>(dk + tile_off);
      uint4* dvdst = reinterpret_cast<uint4*>(dv + tile_off);
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int q = it * 128 + r128;
        if ((q >> 3) < live_rows) {
          dkdst[q] = ld_shared_v4(chunk_addr(tile_k, q >> 3, q & 7));
          dvdst[q] = ld_shared_v4(chunk_addr(tile_v, q >> 3, q & 7));
        }
      }
    }
    // The K/V buffer goes back to the producer: every thread orders its
    // generic-proxy accesses before the next TMA fill, then one releases it.
    fence_proxy_async_smem();
    if (!(ok = epi_sync())) break;  // tiles read (and wsum free)
    if (r128 == 0) mbar_arrive(&bars.kv_empty[b]);
  }
  if (r128 == 0) {
    // Aborted: a raw k tile load still in flight lands before the CTA exits.
    if (kraw_issued > kraw_done) mbar_wait_drain(&bars.kraw_full, kraw_done & 1);
    bulk_wait_group0();  // the dk / dv stores are complete
  }
  if (r128 < D) dgk_part[static_cast<size_t>(blockIdx.x) * D + r128] = bars.dgk_cta[r128];
}

template <int D, class W, bool kOrd>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_stats, const __grid_constant__ CUtensorMap map_dq,
                    const __grid_constant__ CUtensorMap map_kraw, const __grid_constant__ CUtensorMap map_dk,
                    const __grid_constant__ CUtensorMap map_dv, const __grid_constant__ W w, float scale,
                    const __nv_bfloat16* __restrict__ k_raw,
                    const float* __restrict__ rk, const float* __restrict__ gk, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, float* __restrict__ dqacc, uint32_t* __restrict__ counters,
                    float* __restrict__ dgk_part, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) BwdBars bars;
  uint8_t* sm = align1024b(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    // With three issuers a Q / dO stage, the dS^T tile and a K/V buffer are
    // each released by commits from their two readers.
    const uint32_t n_rel = C::kSplitIssuers ? 2u : 1u;
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars.q_full[s], 1);
      // Released after its last product (dK); d = 128 also by the drain,
      // whose reduces read two staging tiles over the stage.
      mbar_init(&bars.q_empty[s], D == 128 ? 2 : 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);  // d = 64: the epilogue; d = 128: the issuer
      mbar_init(&bars.kv_mmadone[s], n_rel);  // d = 64: the recompute and the dQ issuers
      mbar_init(&bars.do_full[s], 1);
      mbar_init(&bars.do_empty[s], n_rel);
      mbar_init(&bars.ds_free[s], 1);  // the dQ product (d = 64: dK reads dS^T from TMEM)
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_ready, 256);
    mbar_init(&bars.ds_ready, 256);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_free, 128);
    mbar_init(&bars.acc_full, n_rel);  // d = 64: the dV and the dK issuers
    mbar_init(&bars.acc_free_v, 128);
    mbar_init(&bars.acc_free_k, 128);
    mbar_init(&bars.s_free, 256);
    mbar_init(&bars.dv_done, 1);
    mbar_init(&bars.epi, 128);
    mbar_init(&bars.drain_sync, 128);
    mbar_init(&bars.kraw_full, 1);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    mbar_init(&bars.drain[2], 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma0) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  {
    // The constant A chunks of the statistics K step: key rows of ones in
    // columns 0-2 (S^T) and 3-5 (dP^T), zeros elsewhere, in the 32-byte
    // swizzled K-major layout (16-byte half h of row r at r * 32 + 16 (h ^ bit
    // 2 of r)); one 8-row atom each, which the descriptor repeats.
    for (int i = threadIdx.x; i < 2 * 8 * 2; i += blockDim.x) {
      const int which = i >> 4, r = (i >> 1) & 7, h = i & 1;
      const uint32_t one = 0x3F80u;  // bf16 1.0
      uint32_t w0 = 0u, w1 = 0u, w2 = 0u;
      if (h == 0) {
        if (which == 0) {
          w0 = one | (one << 16);
          w1 = one;
        } else {
          w1 = one << 16;
          w2 = one | (one << 16);
        }
      }
      st_shared_v4(smem_u32(sm + C::kOffConst + which * C::kConstAtom + r * 32 + ((h ^ ((r >> 2) & 1)) << 4)), w0, w1,
                   w2, 0u);
    }
    fence_proxy_async_smem();  // visible to the tensor cores
  }

  griddep_wait();  // the previous grid's writes (q_hat, k_hat, statistics chunks, zeroed dQ) are visible
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    bars.gk[c] = gk[c];
    bars.dgk_cta[c] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp < 8) {
    setmaxnreg_inc<D == 64 ? kRegCompute64 : kRegCompute128>();
    bwd_compute<D>(sm, bars, tmem, warp >> 2, w, scale, dev_err);
  } else if constexpr (D == 64) {
    if (warp < kWarpEpi) setmaxnreg_dec<kRegDrain64>();
    else if (warp < kWarpTma) setmaxnreg_inc<kRegEpi64>();
    else setmaxnreg_dec<kRegMma64>();
    if (warp < kWarpEpi) {
      bwd_drain64<D, kOrd>(sm, bars, tmem, w, &map_dq, counters, dev_err);
    } else if (warp < kWarpTma) {
      bwd_epilogue_warps<D>(sm, bars, tmem, w, scale, &map_kraw, &map_dk, &map_dv, rk, dk, dv, dgk_part, dev_err);
    } else if (warp == kWarpTma) {
      if (lane == 0)
        bwd_producer<D>(&map_q, &map_k, &map_v, &map_do, &map_stats, sm, bars, w, dev_err);
    } else if (warp == kWarpMma0) {
      if (lane == 0) bwd_mma_recompute<D>(sm, bars, tmem, w, dev_err);
    } else if (warp == kWarpMma1) {
      if (lane == 0) bwd_mma_gradients<D>(sm, bars, tmem, w, dev_err);
    } else if (warp == kWarpMma2) {
      if (lane == 0) bwd_mma_dq<D>(sm, bars, tmem, w, dev_err);
    }
  } else {
    // d = 128: each role's setmaxnreg heads its own branch, so that the
    // compiler sizes the role's code for the count it sets; the TMA / issuer
    // warps keep their launch count.
    static_assert(kRegMma128 == kRegLaunchMin, "d = 128: the TMA / issuer warps keep their launch count");
    if (warp < kWarpEpi) {
      setmaxnreg_inc<kRegDrain128>();
      bwd_drain128<D, kOrd>(sm, bars, tmem, w, scale, &map_dq, counters, k_raw, rk, dk, dv, dgk_part, dev_err);
    } else if (warp < kWarpTma) {
      setmaxnreg_dec<kRegIdle128>();
    } else if (warp == kWarpTma) {
      if (lane == 0)
        bwd_producer<D>(&map_q, &map_k, &map_v, &map_do, &map_stats, sm, bars, w, dev_err);
    } else if (warp == kWarpMma0) {
      if (lane == 0) bwd_mma<D>(sm, bars, tmem, w, dev_err);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kOrd, class W>
cudaError_t launch_bwd_w(const W& w, int grid, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mstats, const CUtensorMap& mdq,
                         const CUtensorMap& mkraw, const CUtensorMap& mdk, const CUtensorMap& mdv, const AttnShape& s,
                         const uint16_t* k_raw, const float* rk, const float* gk, uint16_t* dk, uint16_t* dv,
                         float* dqacc, uint32_t* counters, float* dgk_part, uint32_t* dev_err, cudaStream_t st) {
  using C = BwdCfg<D>;
  static_assert(C::kDynSmem + static_cast<int>(sizeof(BwdBars)) <= 232448, "shared memory budget");
  auto kernel = attn_bwd_kernel<D, W, kOrd>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split is valid only for the register count it was sized
  // for; any other build is refused rather than launched.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kRegLaunchMin || fa.numRegs > kRegLaunchMax) return cudaErrorInvalidConfiguration;
  return launch_pdl(kernel, dim3(grid), dim3(kBwdThreads), C::kDynSmem, st, mq, mk, mv, mdo, mstats, mdq, mkraw, mdk, mdv, w, s.scale,
                    reinterpret_cast<const __nv_bfloat16*>(k_raw), rk, gk,
                    reinterpret_cast<__nv_bfloat16*>(dk), reinterpret_cast<__nv_bfloat16*>(dv), dqacc, counters,
                    dgk_part, dev_err);
}

// The dQ order and grid of a launch.  Arrival order unless the deterministic
// mode is on; then the rotated order when every segment's key tiles fit on
// the grid at once (the waits between CTAs cannot then form a cycle), else
// the ascending order, which no wait can deadlock.  For the [B, H, N, d]
// layout in rotated order the grid is cut to a multiple of the key tiles per
// head when that takes no more rounds, so that no head's units straddle two
// rounds.
struct BwdPlan {
  int ord;
  int grid;
};
BwdPlan bwd_plan(const AttnShape& s) {
  const int sms = device_sm_count();
  const int units = s.BH * (s.seg.prows / 128);
  BwdPlan p;
  p.grid = units < sms ? units : sms;
  p.ord = kDqArrival;
  if (!s.deterministic) return p;
  int max_nkt = 0;
  for (int i = 0; i < s.seg.n; ++i) {
    const int nkt = (s.seg.pcu[i + 1] - s.seg.pcu[i]) / 128;
    max_nkt = nkt > max_nkt ? nkt : max_nkt;
  }
  p.ord = max_nkt <= p.grid ? kDqRotated : kDqAscending;
  if (p.ord == kDqRotated && s.seg.n == 1) {
    const int g2 = (p.grid / max_nkt) * max_nkt;
    const int rounds = (units + p.grid - 1) / p.grid, rounds2 = (units + g2 - 1) / g2;
    if (g2 > 0 && rounds2 == rounds) p.grid = g2;
  }
  return p;
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mstats, const CUtensorMap& mdq, const AttnShape& s,
                         const uint16_t* k_raw, const float* rk, const float* gk, uint16_t* dk,
                         uint16_t* dv, float* dqacc, uint32_t* counters, float* dgk_part, uint32_t* dev_err,
                         cudaStream_t st) {
  // d = 64: the epilogue loads raw k tiles and stores dk / dv tiles by TMA.
  CUtensorMap mkraw = mq, mdk = mq, mdv = mq;
  if (D == 64 && (!encode_bhnd_map(&mkraw, k_raw, s.BH, s.N, s.d) || !encode_bhnd_map(&mdk, dk, s.BH, s.N, s.d) ||
                  !encode_bhnd_map(&mdv, dv, s.BH, s.N, s.d)))
    return cudaErrorInvalidValue;
  const BwdPlan plan = bwd_plan(s);
  if (s.seg.n == 1) {
    BwdWorkUniform w;
    w.seg.rows = s.seg.rows;
    w.seg.prows = s.seg.prows;
    w.upc = s.seg.prows / 128;
    w.units = s.BH * w.upc;
    w.ord = plan.ord;
    if (plan.ord == kDqArrival)
      return launch_bwd_w<D, false>(w, plan.grid, mq, mk, mv, mdo, mstats, mdq, mkraw, mdk, mdv, s, k_raw, rk, gk, dk, dv,
                                    dqacc, counters, dgk_part, dev_err, st);
    return launch_bwd_w<D, true>(w, plan.grid, mq, mk, mv, mdo, mstats, mdq, mkraw, mdk, mdv, s, k_raw, rk, gk, dk, dv,
                                 dqacc, counters, dgk_part, dev_err, st);
  }
  BwdWork w;
  w.seg = s.seg;
  w.upc = s.seg.prows / 128;
  w.units = s.BH * w.upc;
  w.ord = plan.ord;
  if (plan.ord == kDqArrival)
    return launch_bwd_w<D, false>(w, plan.grid, mq, mk, mv, mdo, mstats, mdq, mkraw, mdk, mdv, s, k_raw, rk, gk, dk, dv,
                                  dqacc, counters, dgk_part, dev_err, st);
  return launch_bwd_w<D, true>(w, plan.grid, mq, mk, mv, mdo, mstats, mdq, mkraw, mdk, mdv, s, k_raw, rk, gk, dk, dv, dqacc,
                               counters, dgk_part, dev_err, st);
}

}  // namespace

// One dgk partial per CTA.
int attn_bwd_dgk_parts(const AttnShape& s) { return bwd_plan(s).grid; }

int attn_bwd_counter_words(const AttnShape& s) { return s.deterministic ? s.BH * (s.seg.prows / 128) : 0; }

cudaError_t launch_attn_bwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, const CUtensorMap& map_stats, const CUtensorMap& map_dq,
                            const AttnShape& s, const uint16_t* k_raw, const float* rk, const float* gk,
                            uint16_t* dk, uint16_t* dv, float* dqacc, uint32_t* counters, float* dgk_part,
                            uint32_t* dev_err, cudaStream_t st) {
  if (s.d == 64)
    return launch_bwd_d<64>(map_q, map_k, map_v, map_do, map_stats, map_dq, s, k_raw, rk, gk, dk, dv, dqacc,
                            counters, dgk_part, dev_err, st);
  if (s.d == 128)
    return launch_bwd_d<128>(map_q, map_k, map_v, map_do, map_stats, map_dq, s, k_raw, rk, gk, dk, dv, dqacc,
                             counters, dgk_part, dev_err, st);
  return cudaErrorInvalidValue;
}

}  // namespace jattn
