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
//   dQ_i += dS K_j              (fp32 atomics into a global accumulator)
//
// One CTA owns one 128-key tile of one (b, h) and streams every query tile
// of the head through a small ring:
//
//   warp 8      TMA producer: K_j, V_j once; then (Q_i, dO_i) per query tile.
//   warp 9      MMA issuer (one thread): the five MMAs above.
//   warps 0-3   one thread per key row: P^T and dS^T (bf16, written to shared
//               memory in the MMA's swizzled layout); at the end the dV / dK
//               epilogue, which also applies the K-RMSNorm backward to its
//               own rows (dk, and this CTA's partial of dgk).
//   warps 4-7   one thread per query row: drain dQ_i from TMEM into the fp32
//               accumulator.
//
// The dS^T tile in shared memory serves two MMAs: as a K-major A operand
// (dK = dS^T Q) and, read the other way, as an MN-major A operand
// (dQ = dS K).
//
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dV [256,256+d),
// dK [256+d,256+2d), dQ [384,448) for d = 64; for d = 128 dQ reuses the dP^T
// columns, so dP^T of the next query tile waits for dQ to be drained.
#include <cuda_bf16.h>

#include "jattn_internal.h"
#include "sm103_ptx.cuh"

namespace jattn {
namespace {

constexpr int kBwdThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128 x d bf16 tile
  static constexpr int kStages = (D == 64) ? 2 : 1;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffQ = 2 * kTile;                    // + stage * kTile
  static constexpr int kOffDO = kOffQ + kStages * kTile;     // + stage * kTile
  static constexpr int kOffP = kOffDO + kStages * kTile;     // 128 x 128 bf16
  static constexpr int kOffDS = kOffP + 128 * 128 * 2;       // 128 x 128 bf16
  static constexpr int kTileBytes = kOffDS + 128 * 128 * 2;
  static constexpr int kDynSmem = kTileBytes + 1024;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 128;
  static constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV, dK
  static constexpr uint32_t kIdescMM = idesc_bf16_f32(128, D, true, true);      // dQ
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full, s_free;
  uint64_t dp_full, dp_free;
  uint64_t p_ready, ds_ready;
  uint64_t dq_full, dq_free;
  uint64_t kv_done;
  uint64_t epi;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  // Per ring stage: the query tile's LSE in the log2 domain (+inf past N)
  // and D (0 past N), copied in with the tile from padded scratch rows.
  __align__(16) float lse2[2][128];
  __align__(16) float delta[2][128];
};

__device__ __forceinline__ uint8_t* align1024b(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int D>
__device__ void bwd_producer(const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                             const CUtensorMap* mdo, uint8_t* sm, BwdBars& bars, int bh, int kv0, int nq,
                             const float* lse2_pad, const float* delta_pad, int n_pad, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  tma_prefetch_desc(mq);
  tma_prefetch_desc(mk);
  tma_prefetch_desc(mv);
  tma_prefetch_desc(mdo);
  mbar_arrive_expect_tx(&bars.kv_full, 2u * C::kTile);
  for (int blk = 0; blk < D / 64; ++blk) {
    tma_load_3d(sm + C::kOffK + blk * 16384, mk, &bars.kv_full, blk * 64, kv0, bh);
    tma_load_3d(sm + C::kOffV + blk * 16384, mv, &bars.kv_full, blk * 64, kv0, bh);
  }
  int i = 0;
  for (; i < nq; ++i) {
    const int st = i % C::kStages;
    if (i >= C::kStages) {
      if (!mbar_wait(&bars.q_empty[st], ((i / C::kStages) - 1) & 1, &bars.abort, dev_err)) break;
    }
    mbar_arrive_expect_tx(&bars.q_full[st], 2u * C::kTile + 1024u);
    const size_t prow = static_cast<size_t>(bh) * n_pad + static_cast<size_t>(i) * 128;
    bulk_load(bars.lse2[st], lse2_pad + prow, 512, &bars.q_full[st]);
    bulk_load(bars.delta[st], delta_pad + prow, 512, &bars.q_full[st]);
    for (int blk = 0; blk < D / 64; ++blk) {
      tma_load_3d(sm + C::kOffQ + st * C::kTile + blk * 16384, mq, &bars.q_full[st], blk * 64, i * 128, bh);
      tma_load_3d(sm + C::kOffDO + st * C::kTile + blk * 16384, mdo, &bars.q_full[st], blk * 64, i * 128, bh);
    }
  }
  if (i < nq) {
    mbar_wait_drain(&bars.kv_full, 0);
    for (int s = 0; s < C::kStages; ++s) {
      int last = -1;
      for (int t = i - 1; t >= 0 && t >= i - C::kStages; --t)
        if (t % C::kStages == s) { last = t; break; }
      if (last >= 0) mbar_wait_drain(&bars.q_full[s], (last / C::kStages) & 1);
    }
  }
}

// D[tmem] = A * B^T with A, B K-major 128 x d tiles (d/16 MMAs of K = 16).
template <int D>
__device__ __forceinline__ void mma_kk(uint32_t tmem_d, uint32_t a, uint32_t b, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
    umma_bf16_ss(tmem_d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A * B with A a K-major 128 x 128 bf16 tile (K = 128 queries)
// and B a 128 x d tile stored K-rows x d (MN-major).
template <int D>
__device__ __forceinline__ void mma_km(uint32_t tmem_d, uint32_t a, uint32_t b, uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
    umma_bf16_ss(tmem_d, sdesc_sw128(a + aoff, 16, 1024), sdesc_sw128(b + kk * 2048, 16384, 1024), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
  }
}

// D[tmem] = A * B with A given transposed (stored K-rows x M, MN-major) and
// B stored K-rows x d (MN-major); K = 128 keys.
template <int D>
__device__ __forceinline__ void mma_mm(uint32_t tmem_d, uint32_t a, uint32_t b, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    umma_bf16_ss(tmem_d, sdesc_sw128(a + kk * 2048, 16384, 1024), sdesc_sw128(b + kk * 2048, 16384, 1024), idesc,
                 kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ void bwd_mma(uint8_t* sm, BwdBars& bars, uint32_t tmem, int nq, uint32_t* dev_err) {
  using C = BwdCfg<D>;
  const uint32_t aK = smem_u32(sm + C::kOffK), aV = smem_u32(sm + C::kOffV);
  const uint32_t aP = smem_u32(sm + C::kOffP), aDS = smem_u32(sm + C::kOffDS);
  volatile int* ab = &bars.abort;
  bool ok = mbar_wait(&bars.kv_full, 0, ab, dev_err);
  for (int i = 0; ok && i < nq; ++i) {
    const int st = i % C::kStages;
    const uint32_t aQ = smem_u32(sm + C::kOffQ + st * C::kTile);
    const uint32_t aDO = smem_u32(sm + C::kOffDO + st * C::kTile);
    if (!(ok = mbar_wait(&bars.q_full[st], (i / C::kStages) & 1, ab, dev_err))) break;
    if (i > 0 && !(ok = mbar_wait(&bars.s_free, (i - 1) & 1, ab, dev_err))) break;
    tc_fence_after();
    mma_kk<D>(tmem + C::kColS, aK, aQ, C::kIdescSS);
    umma_commit(&bars.s_full);
    if (i > 0) {
      if (!(ok = mbar_wait(&bars.dp_free, (i - 1) & 1, ab, dev_err))) break;
      if (D == 128 && !(ok = mbar_wait(&bars.dq_free, (i - 1) & 1, ab, dev_err))) break;
    }
    tc_fence_after();
    mma_kk<D>(tmem + C::kColDP, aV, aDO, C::kIdescSS);
    umma_commit(&bars.dp_full);
    if (!(ok = mbar_wait(&bars.p_ready, i & 1, ab, dev_err))) break;
    tc_fence_after();
    mma_km<D>(tmem + C::kColDV, aP, aDO, C::kIdescKM, i > 0);
    if (!(ok = mbar_wait(&bars.ds_ready, i & 1, ab, dev_err))) break;
    tc_fence_after();
    mma_km<D>(tmem + C::kColDK, aDS, aQ, C::kIdescKM, i > 0);
    if (D == 64 && i > 0 && !(ok = mbar_wait(&bars.dq_free, (i - 1) & 1, ab, dev_err))) break;
    tc_fence_after();
    mma_mm<D>(tmem + C::kColDQ, aDS, aK, C::kIdescMM);
    umma_commit(&bars.dq_full);
    umma_commit(&bars.q_empty[st]);
  }
  if (ok) umma_commit(&bars.kv_done);
  umma_commit(&bars.drain);
  mbar_wait_drain(&bars.drain, 0);
}

// Key-row threads: P^T / dS^T per query tile, then the dV / dK epilogue.
template <int D>
__device__ void bwd_compute(uint8_t* sm, BwdBars& bars, uint32_t tmem, int bh, int kv0, int N, int nq,
                            float scale, const __nv_bfloat16* __restrict__ k_raw, const float* __restrict__ rk,
                            const float* __restrict__ gk, __nv_bfloat16* __restrict__ dk,
                            __nv_bfloat16* __restrict__ dv, float* __restrict__ dgk_part, int part_index,
                            uint32_t* dev_err) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kr = warp * 32 + lane;  // key row in the tile == TMEM lane
  const int n = kv0 + kr;
  const bool key_live = n < N;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS;
  const uint32_t tDP = tmem + lane_base + C::kColDP;
  const uint32_t p_row = smem_u32(sm + C::kOffP) + kr * 128;
  const uint32_t ds_row = smem_u32(sm + C::kOffDS) + kr * 128;
  const uint32_t swz = static_cast<uint32_t>(kr & 7);
  const float scale_log2 = scale * kLog2e;
  volatile int* ab = &bars.abort;
  bool ok = true;

  for (int i = 0; i < nq; ++i) {
    const int st = i % C::kStages;
    ok = mbar_wait(&bars.s_full, i & 1, ab, dev_err);
    // The stage's LSE / D arrived with the query tile (already complete).
    if (ok) ok = mbar_wait(&bars.q_full[st], (i / C::kStages) & 1, ab, dev_err);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    tc_fence_after();
    // P^T row as packed bf16 pairs: the exact operand of the dV MMA, and the
    // factor reused for dS below.
    uint32_t pp[64];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t s[32];
      tmem_ld32(tS + c * 32, s);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(&bars.lse2[st][c * 32 + e]);
        const float p0 = ex2_approx(fmaf(__uint_as_float(s[e + 0]), scale_log2, -l4.x));
        const float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), scale_log2, -l4.y));
        const float p2 = ex2_approx(fmaf(__uint_as_float(s[e + 2]), scale_log2, -l4.z));
        const float p3 = ex2_approx(fmaf(__uint_as_float(s[e + 3]), scale_log2, -l4.w));
        pp[(c * 32 + e) / 2] = key_live ? pack_bf16x2(p0, p1) : 0u;
        pp[(c * 32 + e) / 2 + 1] = key_live ? pack_bf16x2(p2, p3) : 0u;
      }
    }
    tc_fence_before();
    mbar_arrive(&bars.s_free);
    // P^T / dS^T buffers are free once the previous tile's dV/dK/dQ MMAs ran.
    if (i > 0) {
      ok = mbar_wait(&bars.dq_full, (i - 1) & 1, ab, dev_err);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
    }
#pragma unroll
    for (int col = 0; col < 128; col += 8) {
      const uint32_t off = (col >> 6) * 16384 + ((((col & 63) >> 3) ^ swz) << 4);
      st_shared_v4(p_row + off, pp[col / 2], pp[col / 2 + 1], pp[col / 2 + 2], pp[col / 2 + 3]);
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars.p_ready);

    ok = mbar_wait(&bars.dp_full, i & 1, ab, dev_err);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t dpv[32];
      tmem_ld32(tDP + c * 32, dpv);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        const int col = c * 32 + e;
        const float4 d0 = *reinterpret_cast<const float4*>(&bars.delta[st][col]);
        const float4 d1 = *reinterpret_cast<const float4*>(&bars.delta[st][col + 4]);
        const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint32_t pw = pp[col / 2 + h];
          const float pa = __uint_as_float(pw << 16), pb = __uint_as_float(pw & 0xFFFF0000u);
          const float ds0 = pa * (__uint_as_float(dpv[e + 2 * h]) - dd[2 * h]);
          const float ds1 = pb * (__uint_as_float(dpv[e + 2 * h + 1]) - dd[2 * h + 1]);
          w[h] = pack_bf16x2(ds0, ds1);
        }
        const uint32_t off = (col >> 6) * 16384 + ((((col & 63) >> 3) ^ swz) << 4);
        st_shared_v4(ds_row + off, w[0], w[1], w[2], w[3]);
      }
    }
    tc_fence_before();
    mbar_arrive(&bars.dp_free);
    fence_proxy_async_smem();
    mbar_arrive(&bars.ds_ready);
  }
  if (!ok) return;

  // ---- epilogue: dV, and dK through the K-RMSNorm backward ----------------
  ok = mbar_wait(&bars.kv_done, 0, ab, dev_err);
  if (!(ok = __all_sync(0xffffffffu, ok))) return;
  tc_fence_after();
  const size_t row_off = (static_cast<size_t>(bh) * N + (key_live ? n : 0)) * D;
  {
    uint4* dvrow = reinterpret_cast<uint4*>(dv + row_off);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tmem + lane_base + C::kColDV + c * 32, a);
      tmem_wait_ld();
      if (key_live) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(a[g * 8 + 0]), __uint_as_float(a[g * 8 + 1]));
          w.y = pack_bf16x2(__uint_as_float(a[g * 8 + 2]), __uint_as_float(a[g * 8 + 3]));
          w.z = pack_bf16x2(__uint_as_float(a[g * 8 + 4]), __uint_as_float(a[g * 8 + 5]));
          w.w = pack_bf16x2(__uint_as_float(a[g * 8 + 6]), __uint_as_float(a[g * 8 + 7]));
          dvrow[c * 4 + g] = w;
        }
      }
    }
  }
  // dk_hat = scale * acc; u = g * dk_hat; dk = r u - (r^3/d) k sum(u k);
  // dgk partial = sum over this tile's rows of dk_hat * k * r.  Two passes
  // over the TMEM row (the dot product first), 32 columns at a time.
  const float r = key_live ? rk[static_cast<size_t>(bh) * N + n] : 0.f;
  const uint4* krow = reinterpret_cast<const uint4*>(k_raw + row_off);
  const uint32_t tDK = tmem + lane_base + C::kColDK;
  float dot = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(tDK + c * 32, a);
    tmem_wait_ld();
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      const uint4 w = key_live ? krow[c * 4 + c8] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int e = c8 * 8 + 2 * h, col = c * 32 + e;
        dot = fmaf(gk[col] * __uint_as_float(a[e]) * scale, __uint_as_float(u[h] << 16), dot);
        dot = fmaf(gk[col + 1] * __uint_as_float(a[e + 1]) * scale, __uint_as_float(u[h] & 0xFFFF0000u), dot);
      }
    }
  }
  const float coef = r * r * r * (1.f / D) * dot;
  // Per-row dgk contributions go to shared memory (reusing the query-tile
  // ring and the P^T / dS^T tiles, all idle now) for a fixed-order column sum.
  float* red = reinterpret_cast<float*>(sm + C::kOffQ);
  static_assert(128 * (D + 4) * 4 <= C::kTileBytes - C::kOffQ, "dgk reduction buffer");
  constexpr int kRedStride = D + 4;
  uint4* dkrow = reinterpret_cast<uint4*>(dk + row_off);
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(tDK + c * 32, a);
    tmem_wait_ld();
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      const uint4 w = key_live ? krow[c * 4 + c8] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      float y[8], gpart[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int e = c8 * 8 + 2 * h, col = c * 32 + e;
        const float x0 = __uint_as_float(u[h] << 16), x1 = __uint_as_float(u[h] & 0xFFFF0000u);
        const float dk0 = key_live ? __uint_as_float(a[e]) * scale : 0.f;
        const float dk1 = key_live ? __uint_as_float(a[e + 1]) * scale : 0.f;
        y[2 * h] = r * gk[col] * dk0 - coef * x0;
        y[2 * h + 1] = r * gk[col + 1] * dk1 - coef * x1;
        gpart[2 * h] = dk0 * x0 * r;
        gpart[2 * h + 1] = dk1 * x1 * r;
      }
      if (key_live) {
        uint4 o;
        o.x = pack_bf16x2(y[0], y[1]);
        o.y = pack_bf16x2(y[2], y[3]);
        o.z = pack_bf16x2(y[4], y[5]);
        o.w = pack_bf16x2(y[6], y[7]);
        dkrow[c * 4 + c8] = o;
      }
      float4* dst = reinterpret_cast<float4*>(red + kr * kRedStride + c * 32 + c8 * 8);
      dst[0] = make_float4(gpart[0], gpart[1], gpart[2], gpart[3]);
      dst[1] = make_float4(gpart[4], gpart[5], gpart[6], gpart[7]);
    }
  }
  // Bounded barrier among the 128 key-row threads.
  mbar_arrive(&bars.epi);
  ok = mbar_wait(&bars.epi, 0, ab, dev_err);
  if (!ok) return;
  if (kr < D) {
    float s = 0.f;
    for (int t = 0; t < 128; ++t) s += red[t * kRedStride + kr];
    dgk_part[static_cast<size_t>(part_index) * D + kr] = s;
  }
}

// Query-row threads: move dQ_i from TMEM into the fp32 accumulator.
template <int D>
__device__ void bwd_dq_drain(BwdBars& bars, uint32_t tmem, int bh, int N, int nq, float* __restrict__ dqacc,
                             uint32_t* dev_err) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int qr = (warp & 3) * 32 + lane;
  const uint32_t tQ = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kColDQ;
  volatile int* ab = &bars.abort;
  for (int i = 0; i < nq; ++i) {
    bool ok = mbar_wait(&bars.dq_full, i & 1, ab, dev_err);
    if (!__all_sync(0xffffffffu, ok)) return;
    tc_fence_after();
    const int qrow = i * 128 + qr;
    float4* dst = reinterpret_cast<float4*>(dqacc + (static_cast<size_t>(bh) * N + (qrow < N ? qrow : 0)) * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tQ + c * 32, a);
      tmem_wait_ld();
      if (c == D / 32 - 1) {
        tc_fence_before();
        mbar_arrive(&bars.dq_free);
      }
      if (qrow < N) {
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          atomicAdd(dst + c * 8 + c4, make_float4(__uint_as_float(a[4 * c4]), __uint_as_float(a[4 * c4 + 1]),
                                                  __uint_as_float(a[4 * c4 + 2]), __uint_as_float(a[4 * c4 + 3])));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do, int N,
                    float scale, const float* __restrict__ lse2_pad, const float* __restrict__ delta_pad,
                    int n_pad, const __nv_bfloat16* __restrict__ k_raw, const float* __restrict__ rk,
                    const float* __restrict__ gk, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                    float* __restrict__ dqacc, float* __restrict__ dgk_part, uint32_t* dev_err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) BwdBars bars;
  uint8_t* sm = align1024b(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.x, bh = blockIdx.y;
  const int kv0 = j * 128;
  const int nq = (N + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, 128);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_free, 128);
    mbar_init(&bars.p_ready, 128);
    mbar_init(&bars.ds_ready, 128);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_free, 128);
    mbar_init(&bars.kv_done, 1);
    mbar_init(&bars.epi, 128);
    mbar_init(&bars.drain, 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 8) {
    if (lane == 0) bwd_producer<D>(&map_q, &map_k, &map_v, &map_do, sm, bars, bh, kv0, nq, lse2_pad, delta_pad, n_pad,
                                   dev_err);
  } else if (warp == 9) {
    if (lane == 0) bwd_mma<D>(sm, bars, tmem, nq, dev_err);
  } else if (warp < 4) {
    bwd_compute<D>(sm, bars, tmem, bh, kv0, N, nq, scale, k_raw, rk, gk, dk, dv, dgk_part,
                   bh * gridDim.x + j, dev_err);
  } else {
    bwd_dq_drain<D>(bars, tmem, bh, N, nq, dqacc, dev_err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const AttnShape& s, const float* lse2_pad,
                         const float* delta_pad, const uint16_t* k_raw, const float* rk, const float* gk, uint16_t* dk, uint16_t* dv,
                         float* dqacc, float* dgk_part, uint32_t* dev_err, cudaStream_t st) {
  using C = BwdCfg<D>;
  static_assert(C::kDynSmem + static_cast<int>(sizeof(BwdBars)) <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.N + 127) / 128, s.BH);
  attn_bwd_kernel<D><<<grid, kBwdThreads, C::kDynSmem, st>>>(
      mq, mk, mv, mdo, s.N, s.scale, lse2_pad, delta_pad, ((s.N + 127) / 128) * 128, reinterpret_cast<const __nv_bfloat16*>(k_raw), rk, gk,
      reinterpret_cast<__nv_bfloat16*>(dk), reinterpret_cast<__nv_bfloat16*>(dv), dqacc, dgk_part, dev_err);
  return cudaGetLastError();
}

}  // namespace

int attn_bwd_dgk_parts(const AttnShape& s) { return s.BH * ((s.N + 127) / 128); }

cudaError_t launch_attn_bwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, const AttnShape& s, const float* lse2_pad,
                            const float* delta_pad, const uint16_t* k_raw, const float* rk, const float* gk,
                            uint16_t* dk, uint16_t* dv, float* dqacc, float* dgk_part, uint32_t* dev_err,
                            cudaStream_t st) {
  if (s.d == 64)
    return launch_bwd_d<64>(map_q, map_k, map_v, map_do, s, lse2_pad, delta_pad, k_raw, rk, gk, dk, dv, dqacc, dgk_part,
                            dev_err, st);
  if (s.d == 128)
    return launch_bwd_d<128>(map_q, map_k, map_v, map_do, s, lse2_pad, delta_pad, k_raw, rk, gk, dk, dv, dqacc, dgk_part,
                             dev_err, st);
  return cudaErrorInvalidValue;
}

}  // namespace jattn
