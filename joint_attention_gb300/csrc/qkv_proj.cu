// qkv_proj.cu — the QKV projections of the two token streams with QK-RMSNorm
// in their epilogue, on tcgen05 tensor cores.
//
// The MM-DiT block projects each stream's tokens to Q, K and V with that
// stream's own weights, concatenates the caption and image streams along the
// token axis, normalises Q and K (RMSNorm over the head dim, one learned gain
// vector each) and runs one attention over the joint sequence (re-diffusion
// README, "architecture flowchart"; "design notes" table, row "QK norm").
// One launch covers both streams:
//
//   Y = bf16(X W^T + bias)      X: [B * N_s, C] tokens, W: [3 H d, C] (q heads, k heads, v heads)
//   q, k, v = Y by heads, into the joint [B, H, N, d] layout at the stream's
//             rows row0 .. row0 + N_s - 1 of every batch item
//   q_hat = bf16(gq * q * r(q)), k_hat likewise, r(x) = (mean x^2 + eps)^(-1/2)
//
// with q_hat / k_hat correctly rounded as in the norm kernels (the bf16 value
// nearest the exact real product), and r(q), r(k) kept: exactly what the
// training forward keeps for the backward, so the attention forward starts
// from q_hat / k_hat with no normalisation pass of its own.
//
// Tiles: 128 token rows x 256 output columns per accumulator, K in steps of
// 64; persistent, one CTA per SM, the image stream's tiles then the caption
// stream's.
//   warp 8      TMA producer: the X tile (128 x 64) and the W tile (256 x 64)
//               of each K step, 128-byte swizzle, through a 4-stage ring.
//   warp 9      MMA issuer: 4 MMAs (M 128, N 256, K 16) per K step into one of
//               two TMEM accumulators (256 columns each), so that a tile's
//               epilogue overlaps the next tile's products.
//   warps 0-7   epilogue, one thread per token row (TMEM lane): warps w and
//               w + 4 share the lanes of warp w % 4 and take columns 0-127 and
//               128-255 of the tile (two heads of d = 64, or one of d = 128).
//               Per head: d fp32 values out of TMEM, + bias, rounded to bf16
//               (the projection's output) and stored to q / k / v; for q and
//               k the row's RMSNorm from those bf16 values, and q_hat / k_hat
//               and r stored too.  Each thread writes whole head rows with
//               16-byte stores.
// Heads past 3 H in the last column tile, and token rows past the stream's
// end in its last row tile, read the TMA's zero fill and are not stored.
//
// Correct rounding: the per-thread sum of the d squares is a balanced tree
// (at most 7 roundings per term, within the 8 that the rounding window of the
// norm kernels allows for), and elements in the bf16-midpoint window are
// re-rounded from a double-float r.
#include <cuda_bf16.h>

#include "jattn_internal.h"
#include "sm103_ptx.cuh"
#include "bf16_round.cuh"

namespace jattn {
namespace {

constexpr int kQkvThreads = 320;
constexpr int kQkvStages = 4;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kBTile = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kQkvDynSmem = kQkvStages * kStageBytes + 1024;
constexpr int kWarpProd = 8, kWarpIssue = 9;
constexpr int kEpiThreads = 256;

struct QkvBars {
  uint64_t full[kQkvStages], empty[kQkvStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  __align__(16) float gq[128];
  __align__(16) float gk[128];
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t byte_off) { return desc + (byte_off >> 4); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The rare path, taken by the whole warp for each of its rows that has an
// element near a bf16 midpoint (owner: the lane holding the row): each lane
// takes D / 32 of the row's values (words lane, lane + 32, ... of the owner's
// packed yb), their squares (exact) summed by error-free additions and a
// butterfly over the warp (every lane ends with the same double-float sum),
// then re-rounds its elements that the owner's fp32 path put near a
// midpoint, storing them again over the owner's hat row.
template <int D>
__device__ __forceinline__ void fix_hat_rows(unsigned todo, const uint32_t (&yb)[D / 2], float r, size_t hrow,
                                             uint16_t* hat_base, const float* g, int lane) {
  constexpr int kW = D / 64;  // packed words per lane
  while (todo) {
    const int owner = __ffs(todo) - 1;
    todo &= todo - 1;
    uint32_t mine[kW];
#pragma unroll
    for (int i = 0; i < D / 2; ++i) {
      const uint32_t t = __shfl_sync(0xffffffffu, yb[i], owner);
      if ((i & 31) == lane) mine[i >> 5] = t;
    }
    const float ro = __shfl_sync(0xffffffffu, r, owner);
    const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(hrow), owner);
    const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(hrow >> 32), owner);
    uint16_t* hat = hat_base + ((static_cast<size_t>(hi) << 32) | lo) * D;
    float s = 0.f, c = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      float t, e;
      two_sum(s, __fmul_rn(bf_lo(mine[w]), bf_lo(mine[w])), t, e);
      c = __fadd_rn(c, e);
      two_sum(t, __fmul_rn(bf_hi(mine[w]), bf_hi(mine[w])), s, e);
      c = __fadd_rn(c, e);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s, off), c2 = __shfl_xor_sync(0xffffffffu, c, off);
      float t, e;
      two_sum(s, s2, t, e);
      s = t;
      c = __fadd_rn(__fadd_rn(c, c2), e);
    }
    fast_two_sum(s, c, s, c);
    float rh, rl;
    rsqrt_mean_eps_df(s, c, 1.f / D, rh, rl);
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int e0 = 2 * (lane + 32 * w);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x = j ? bf_hi(mine[w]) : bf_lo(mine[w]);
        if (near_bf16_midpoint(__fmul_rn(__fmul_rn(g[e0 + j], x), ro))) {
          const float z = round_bf16_df(g[e0 + j], x, rh, rl);
          hat[e0 + j] = static_cast<uint16_t>(pack_bf16x2(z, 0.f) & 0xFFFFu);
        }
      }
    }
  }
}

struct QkvStream {
  int M;       // token rows (B * N_s)
  int N_s;     // tokens per batch item
  int row0;    // the stream's first row in the joint sequence
  int tile0;   // its first tile
  const float* bias;  // [3 H d] or null
};

struct QkvParams {
  QkvStream s[2];     // 0: image stream, 1: caption stream
  int H, C, N;        // heads, model width (K of the product), joint sequence length
  int n_tiles;        // column tiles: ceil(3 H d / 256)
  int tiles;          // all tiles of both streams
  uint16_t* out[3];   // q, k, v: [B, H, N, d]
  uint16_t* hat[2];   // q_hat, k_hat
  float* r[2];        // rq, rk: [B, H, N]
};

// One head of one token row: D accumulator columns at taddr.  row is head
// 0's row index (b H N + n); the head's is row + h N.
template <int D>
__device__ __forceinline__ void qkv_emit_head(uint32_t taddr, int ocol, bool live, size_t row, const QkvParams& p,
                                              const float* bias, const QkvBars& bars) {
  const int hd = p.H * D;
  const int which = ocol / hd;  // 0 q, 1 k, 2 v
  const size_t hrow = row + static_cast<size_t>((ocol - which * hd) / D) * p.N;
  // Y = bf16(acc + bias), 64 columns at a time (packed pairs).
  uint32_t yb[D / 2];
#pragma unroll
  for (int h64 = 0; h64 < D / 64; ++h64) {
    uint32_t acc[2][32];
    tmem_ld32(taddr + h64 * 64, acc[0]);
    tmem_ld32(taddr + h64 * 64 + 32, acc[1]);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
      float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bias) bv = *reinterpret_cast<const float4*>(bias + ocol + h64 * 64 + e);
      const uint32_t* a = &acc[e / 32][e % 32];
      yb[h64 * 32 + e / 2] = pack_bf16x2(__uint_as_float(a[0]) + bv.x, __uint_as_float(a[1]) + bv.y);
      yb[h64 * 32 + e / 2 + 1] = pack_bf16x2(__uint_as_float(a[2]) + bv.z, __uint_as_float(a[3]) + bv.w);
    }
  }
  if (live) {
    uint4* dst = reinterpret_cast<uint4*>(p.out[which] + hrow * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(yb[4 * c], yb[4 * c + 1], yb[4 * c + 2], yb[4 * c + 3]);
  }
  if (which == 2) return;

  const float* g = which == 0 ? bars.gq : bars.gk;
  bool near = false;
  float r = 0.f;
  if (live) {
    // Sum of the squares of the bf16 values: a balanced tree over exact squares.
    float sq[D / 2];
#pragma unroll
    for (int i = 0; i < D / 2; ++i)
      sq[i] = __fadd_rn(__fmul_rn(bf_lo(yb[i]), bf_lo(yb[i])), __fmul_rn(bf_hi(yb[i]), bf_hi(yb[i])));
#pragma unroll
    for (int w = D / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) sq[i] = __fadd_rn(sq[i], sq[i + w]);
    r = rsqrtf(__fadd_rn(__fmul_rn(sq[0], 1.f / D), kEps));
    uint32_t hb[D / 2];
#pragma unroll
    for (int e = 0; e < D; e += 2) {
      const float z0 = __fmul_rn(__fmul_rn(g[e], bf_lo(yb[e / 2])), r);
      const float z1 = __fmul_rn(__fmul_rn(g[e + 1], bf_hi(yb[e / 2])), r);
      near |= near_bf16_midpoint(z0) | near_bf16_midpoint(z1);
      hb[e / 2] = pack_bf16x2(z0, z1);
    }
    uint4* hdst = reinterpret_cast<uint4*>(p.hat[which] + hrow * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) hdst[c] = make_uint4(hb[4 * c], hb[4 * c + 1], hb[4 * c + 2], hb[4 * c + 3]);
    p.r[which][hrow] = r;
  }
  const unsigned todo = __ballot_sync(0xffffffffu, near);
  if (todo) fix_hat_rows<D>(todo, yb, r, hrow, p.hat[which], g, threadIdx.x % 32);
}

template <int D>
__global__ void __launch_bounds__(kQkvThreads, 1)
    qkv_norm_kernel(const __grid_constant__ CUtensorMap map_x0, const __grid_constant__ CUtensorMap map_w0,
                    const __grid_constant__ CUtensorMap map_x1, const __grid_constant__ CUtensorMap map_w1,
                    const __grid_constant__ QkvParams p, const float* __restrict__ gq, const float* __restrict__ gk,
                    uint32_t* dev_err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) QkvBars bars;
  uint8_t* sm = align1024(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* ab = &bars.abort;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQkvStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.acc_full[b], 1);
      mbar_init(&bars.acc_empty[b], kEpiThreads);
    }
    mbar_init(&bars.mma_done, 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpIssue) {
    tmem_alloc(&bars.tmem_base, 2 * kBN);
    tmem_relinquish();
  }
  griddep_wait();  // the previous grid's writes are visible from here on
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    bars.gq[i] = gq[i];
    bars.gk[i] = gk[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const int ksteps = (p.C + kBK - 1) / kBK;

  if (warp == kWarpProd) {
    if (lane == 0) {
      tma_prefetch_desc(&map_x0);
      tma_prefetch_desc(&map_w0);
      tma_prefetch_desc(&map_x1);
      tma_prefetch_desc(&map_w1);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        const int si = t >= p.s[1].tile0 ? 1 : 0;
        const int tl = t - p.s[si].tile0;
        const int mt = tl / p.n_tiles, nt = tl - mt * p.n_tiles;
        const CUtensorMap* mx = si ? &map_x1 : &map_x0;
        const CUtensorMap* mw = si ? &map_w1 : &map_w0;
        for (int kb = 0; kb < ksteps; ++kb) {
          const int s = it % kQkvStages;
          if (it >= kQkvStages && !(ok = mbar_wait(&bars.empty[s], ((it / kQkvStages) - 1) & 1, ab, dev_err)))
            break;
          uint8_t* st = sm + s * kStageBytes;
          mbar_arrive_expect_tx(&bars.full[s], kStageBytes);
          tma_load_2d(st, mx, &bars.full[s], kb * kBK, mt * kBM);
          tma_load_2d(st + kATile, mw, &bars.full[s], kb * kBK, nt * kBN);
          ++it;
        }
      }
      if (*ab) {  // aborted: the copies in flight land before the CTA exits
        for (int i = (it > kQkvStages ? it - kQkvStages : 0); i < it; ++i)
          mbar_wait_drain(&bars.full[i % kQkvStages], (i / kQkvStages) & 1);
      }
    }
  } else if (warp == kWarpIssue) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x, ++lt) {
        const int abuf = lt & 1;
        if (lt >= 2 && !(ok = mbar_wait(&bars.acc_empty[abuf], ((lt >> 1) - 1) & 1, ab, dev_err))) break;
        tc_fence_after();
        const uint32_t acc = tmem + abuf * kBN;
        for (int kb = 0; kb < ksteps; ++kb, ++it) {
          const int s = it % kQkvStages;
          if (!(ok = mbar_wait(&bars.full[s], (it / kQkvStages) & 1, ab, dev_err))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(sm + s * kStageBytes);
          const uint64_t a = sdesc_sw128(st, 16, 1024), b = sdesc_sw128(st + kATile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_ss(acc, desc_add(a, kk * 32), desc_add(b, kk * 32), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars.empty[s]);
        }
        if (ok) umma_commit(&bars.acc_full[abuf]);
      }
      // Every MMA this thread issued has completed once this barrier flips.
      umma_commit(&bars.mma_done);
      mbar_wait_drain(&bars.mma_done, 0);
    }
  } else {
    const int lg = warp & 3, half = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(lg * 32) << 16;
    const int hd3 = 3 * p.H * D;
    int lt = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++lt) {
      const int abuf = lt & 1;
      const bool ok = mbar_wait(&bars.acc_full[abuf], (lt >> 1) & 1, ab, dev_err);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int si = t >= p.s[1].tile0 ? 1 : 0;
      const QkvStream& S = p.s[si];
      const int tl = t - S.tile0;
      const int mt = tl / p.n_tiles, nt = tl - mt * p.n_tiles;
      const int m = mt * kBM + lg * 32 + lane;
      const bool live = m < S.M;
      const int bi = live ? m / S.N_s : 0;
      const int n = live ? S.row0 + (m - bi * S.N_s) : 0;
      const size_t row = static_cast<size_t>(bi) * p.H * p.N + n;
#pragma unroll
      for (int j = 0; j < 128 / D; ++j) {
        const int tcol = half * 128 + j * D;  // the head's first column in the tile
        const int ocol = nt * kBN + tcol;     // ... in Y
        if (ocol < hd3)
          qkv_emit_head<D>(tmem + lane_base + abuf * kBN + tcol, ocol, live, row, p, S.bias, bars);
      }
      tc_fence_before();
      mbar_arrive(&bars.acc_empty[abuf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIssue) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

}  // namespace

cudaError_t launch_qkv_norm(const CUtensorMap (&maps)[4], const QkvLaunch& a, uint32_t* dev_err, cudaStream_t st) {
  QkvParams p;
  p.H = a.H;
  p.C = a.C;
  p.N = a.N;
  p.n_tiles = (3 * a.H * a.d + kBN - 1) / kBN;
  int tile0 = 0;
  for (int i = 0; i < 2; ++i) {
    p.s[i].M = a.M[i];
    p.s[i].N_s = a.N_s[i];
    p.s[i].row0 = a.row0[i];
    p.s[i].tile0 = tile0;
    p.s[i].bias = a.bias[i];
    tile0 += ((a.M[i] + kBM - 1) / kBM) * p.n_tiles;
  }
  p.tiles = tile0;
  for (int i = 0; i < 3; ++i) p.out[i] = a.out[i];
  for (int i = 0; i < 2; ++i) {
    p.hat[i] = a.hat[i];
    p.r[i] = a.r[i];
  }
  if (p.tiles == 0) return cudaSuccess;
  auto kernel = a.d == 64 ? qkv_norm_kernel<64> : qkv_norm_kernel<128>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkvDynSmem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int grid = p.tiles < sms ? p.tiles : sms;
  return launch_pdl(kernel, dim3(grid), dim3(kQkvThreads), kQkvDynSmem, st, maps[0], maps[1], maps[2], maps[3], p,
                    a.gq, a.gk, dev_err);
}

}  // namespace jattn
