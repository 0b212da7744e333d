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
//               of each K step, 128-byte swizzle, through a 3-stage ring.
//   warp 9      MMA issuer: 4 MMAs (M 128, N 256, K 16) per K step into one of
//               two TMEM accumulators (256 columns each), so that a tile's
//               epilogue overlaps the next tile's products.
//   warps 0-7   epilogue, one thread per token row (TMEM lane): warps w and
//               w + 4 share the lanes of warp w % 4 and take columns 0-127 and
//               128-255 of the tile (two heads of d = 64, or one of d = 128).
//               Per head: d fp32 values out of TMEM, + bias (the warp's
//               slice, copied to shared memory while the products run),
//               rounded to bf16 (the projection's output) for q / k / v; for
//               q and k the row's RMSNorm from those bf16 values, q_hat /
//               k_hat and r.  Rows are staged in shared memory and written
//               out as whole 128-byte lines, four rows per store instruction.
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

constexpr int kQkvStages = 3;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kBTile = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kStageRowBytes = 128;                 // 64 bf16 columns of one token row
constexpr int kStagingBytes = 32 * kStageRowBytes;  // per epilogue warp: its 32 rows of 64 columns
constexpr uint32_t kDeadRow = 0xFFFFFFFFu;

// Eight epilogue warps (warps w and w + 4 take the TMEM lanes of warp w % 4
// and columns 0-127 / 128-255 of the tile: two heads of d = 64, or one of
// d = 128), then the TMA producer and the MMA issuer.  Each epilogue warp
// stages its rows in shared memory: at d = 64 raw rows and q_hat / k_hat rows
// in two buffers, at d = 128 one buffer used for each 64-column half.
template <int D>
struct QkvCfg {
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kWarpProd = kEpiWarps, kWarpIssue = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kBuffers = D == 64 ? 2 : 1;
  static constexpr int kStaging = kBuffers * kStagingBytes;
  static constexpr int kBiasBytes = 128 * 4;  // per epilogue warp: the bias of its 128 columns
  static constexpr int kOffStaging = kQkvStages * kStageBytes;
  static constexpr int kOffBias = kOffStaging + kEpiWarps * kStaging;
  static constexpr int kDynSmem = kOffBias + kEpiWarps * kBiasBytes + 1024;
};

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
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  const uint4 v = ld_shared_v4(addr);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// Staging of a warp's 32 token rows of 64 bf16 columns (128 bytes each) in
// shared memory: row i at i * 128, its 16-byte chunk c at slot c ^ (i % 8),
// so that a row written by one lane and a chunk column read across 8 lanes
// both touch every bank once.
__device__ __forceinline__ uint32_t staged(uint32_t buf, int row, int chunk) {
  return buf + row * kStageRowBytes + ((chunk ^ (row & 7)) << 4);
}
// This lane's row: w[0..31] (packed pairs).
__device__ __forceinline__ void stage_row(uint32_t buf, const uint32_t* w, int lane) {
#pragma unroll
  for (int c = 0; c < 8; ++c) st_shared_v4(staged(buf, lane, c), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}
// Writes the 32 staged rows out, four whole rows (four 128-byte lines) per
// store instruction: lanes 8 j' .. 8 j' + 7 take row 4 j + j', one chunk
// each.  rows[j]: the global row index (b H + h) N + n of staged row
// 4 j + lane / 8 for head 0 (kDeadRow: past the stream's end); head_rows =
// h N; col: the first column (0, or 64 within a d = 128 head row).
template <int D>
__device__ __forceinline__ void store_rows(uint32_t buf, uint16_t* base, const uint32_t (&rows)[8],
                                           uint32_t head_rows, int col, int lane) {
  const int ch = lane & 7;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 val = ld_shared_v4(staged(buf, 4 * j + (lane >> 3), ch));
    if (rows[j] != kDeadRow)
      *reinterpret_cast<uint4*>(base + (static_cast<size_t>(rows[j]) + head_rows) * D + col + ch * 8) = val;
  }
}

// The double-float sum of squares of a row spread over the warp, the same
// on every lane: each lane's own error-free sum (s, c), then a butterfly of
// error-free additions (symmetric, so every lane forms the same values).
__device__ __forceinline__ void warp_sum_df(float& s, float& c) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off), c2 = __shfl_xor_sync(0xffffffffu, c, off);
    float t, e;
    two_sum(s, s2, t, e);
    s = t;
    c = __fadd_rn(__fadd_rn(c, c2), e);
  }
  fast_two_sum(s, c, s, c);
}
__device__ __forceinline__ void add_sq_df(uint32_t w, float& s, float& c) {
  float t, e;
  two_sum(s, __fmul_rn(bf_lo(w), bf_lo(w)), t, e);
  c = __fadd_rn(c, e);
  two_sum(t, __fmul_rn(bf_hi(w), bf_hi(w)), s, e);
  c = __fadd_rn(c, e);
}

// The rare path.  The warp takes each of its rows that has an element near
// a bf16 midpoint (owner: the lane holding the row) together: each lane
// takes D / 32 of the row's values, their squares (exact) are summed by
// error-free additions over the warp, and each lane re-rounds its elements
// that the owner's fp32 path put near a midpoint, from the double-float r.
//
// d = 64 (fix_staged_rows): the row's raw values come from the raw staging
// buffer and each lane writes its word of the row (two elements, re-rounded
// where needed) over the staged q_hat / k_hat row, before that is written
// out.
__device__ __forceinline__ void fix_staged_rows(unsigned todo, uint32_t raw, uint32_t hat, float r, const float* g,
                                                int lane) {
  while (todo) {
    const int o = __ffs(todo) - 1;
    todo &= todo - 1;
    // Word `lane` of row o: elements 2 lane, 2 lane + 1 (chunk lane / 4).
    const uint32_t off = (lane & 3) * 4;
    const uint32_t w = ld_shared_u32(staged(raw, o, lane >> 2) + off);
    const float ro = __shfl_sync(0xffffffffu, r, o);
    float s = 0.f, c = 0.f;
    add_sq_df(w, s, c);
    warp_sum_df(s, c);
    float rh, rl;
    rsqrt_mean_eps_df(s, c, 1.f / 64, rh, rl);
    float f[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int e = 2 * lane + j;
      const float x = j ? bf_hi(w) : bf_lo(w);
      const float z = __fmul_rn(__fmul_rn(g[e], x), ro);
      f[j] = near_bf16_midpoint(z) ? round_bf16_df(g[e], x, rh, rl) : z;
    }
    st_shared_u32(staged(hat, o, lane >> 2) + off, pack_bf16x2(f[0], f[1]));
  }
}
// d = 128 (fix_stored_rows): the row's raw values come from the owner's
// registers (yb, by shuffles) and the corrected elements are stored again
// over the owner's q_hat / k_hat row, which is already written.
__device__ __forceinline__ void fix_stored_rows(unsigned todo, const uint32_t (&yb)[64], float r, size_t hrow,
                                                uint16_t* hat_base, const float* g, int lane) {
  while (todo) {
    const int o = __ffs(todo) - 1;
    todo &= todo - 1;
    uint32_t mine[2];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const uint32_t t = __shfl_sync(0xffffffffu, yb[i], o);
      if ((i & 31) == lane) mine[i >> 5] = t;
    }
    const float ro = __shfl_sync(0xffffffffu, r, o);
    const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(hrow), o);
    const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(hrow >> 32), o);
    uint16_t* hat = hat_base + ((static_cast<size_t>(hi) << 32) | lo) * 128;
    float s = 0.f, c = 0.f;
    add_sq_df(mine[0], s, c);
    add_sq_df(mine[1], s, c);
    warp_sum_df(s, c);
    float rh, rl;
    rsqrt_mean_eps_df(s, c, 1.f / 128, rh, rl);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
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

// TMA maps over the five outputs ([B H, N, d] bf16, box 64 columns x 32 rows,
// 128-byte swizzle: the staging buffers' layout), for warps whose 32 rows lie
// in one batch item.
struct QkvOutMaps {
  CUtensorMap out[3];  // q, k, v
  CUtensorMap hat[2];  // q_hat, k_hat
};
__device__ __forceinline__ void tma_store_3d_s(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Field selection by a runtime index through selects: indexing the kernel's
// parameter arrays with a runtime value would copy them to local memory.
__device__ __forceinline__ uint16_t* out_of(const QkvParams& p, int which) {
  return which == 0 ? p.out[0] : which == 1 ? p.out[1] : p.out[2];
}
__device__ __forceinline__ uint16_t* hat_of(const QkvParams& p, int which) { return which == 0 ? p.hat[0] : p.hat[1]; }
__device__ __forceinline__ float* r_of(const QkvParams& p, int which) { return which == 0 ? p.r[0] : p.r[1]; }
__device__ __forceinline__ const CUtensorMap* out_map(const QkvOutMaps& m, int which) {
  return which == 0 ? &m.out[0] : which == 1 ? &m.out[1] : &m.out[2];
}
__device__ __forceinline__ const CUtensorMap* hat_map(const QkvOutMaps& m, int which) {
  return which == 0 ? &m.hat[0] : &m.hat[1];
}

// Where a warp's 32 staged rows go: one TMA tile store when they are 32
// consecutive rows of one head (contig; n0 and bh0 = b H of the first row),
// else the row-by-row stores of store_rows.
struct RowsOut {
  bool contig;
  int n0, bh0;
};
template <int D>
__device__ __forceinline__ void emit_rows(uint32_t buf, const CUtensorMap* map, uint16_t* base, const RowsOut& ro,
                                          const uint32_t (&rows)[8], uint32_t head_rows, int h, int col, int lane) {
  if (ro.contig) {
    fence_proxy_async_smem();  // this lane's staged writes, to the TMA unit
    __syncwarp();
    if (lane == 0) {
      tma_store_3d_s(map, buf, col, ro.n0, ro.bh0 + h);
      bulk_commit_group();
    }
  } else {
    __syncwarp();
    store_rows<D>(buf, base, rows, head_rows, col, lane);
  }
}
// Before a staging buffer is written again: the TMA stores have read it.
__device__ __forceinline__ void staging_free(int lane) {
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
}
__device__ __forceinline__ QkvStream stream_of(const QkvParams& p, int si) {
  QkvStream s;
  s.M = si ? p.s[1].M : p.s[0].M;
  s.N_s = si ? p.s[1].N_s : p.s[0].N_s;
  s.row0 = si ? p.s[1].row0 : p.s[0].row0;
  s.tile0 = si ? p.s[1].tile0 : p.s[0].tile0;
  s.bias = si ? p.s[1].bias : p.s[0].bias;
  return s;
}

// r of one row from its bf16 values (packed pairs; exact squares): a
// balanced tree, built block by block (16 values, then across the D / 16
// blocks) so that few partial sums are live at once.
template <int D>
__device__ __forceinline__ float row_rsqrt(const uint32_t (&yb)[D / 2]) {
  float blk[D / 16];
#pragma unroll
  for (int b = 0; b < D / 16; ++b) {
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t u = yb[b * 8 + i];
      t[i] = __fadd_rn(__fmul_rn(bf_lo(u), bf_lo(u)), __fmul_rn(bf_hi(u), bf_hi(u)));
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = __fadd_rn(t[i], t[i + w]);
    blk[b] = t[0];
  }
#pragma unroll
  for (int w = D / 32; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) blk[i] = __fadd_rn(blk[i], blk[i + w]);
  return rsqrtf(__fadd_rn(__fmul_rn(blk[0], 1.f / D), kEps));
}

// 64 columns of this lane's q_hat / k_hat row, (g x) r per element, staged
// 16 bytes at a time into its row of the staging buffer; `near` collects the
// elements within the midpoint window.
__device__ __forceinline__ void stage_hat_row(uint32_t buf, const uint32_t* y, uint32_t g, float r, bool& near,
                                              int lane) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    // The gains through ordered shared loads: loaded chunk by chunk, not all
    // at once ahead of the loop.
    const float4 ga = ld_shared_f4(g + c * 32), gb = ld_shared_f4(g + c * 32 + 16);
    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t yv = y[4 * c + i];
      const float z0 = __fmul_rn(__fmul_rn(gv[2 * i], bf_lo(yv)), r);
      const float z1 = __fmul_rn(__fmul_rn(gv[2 * i + 1], bf_hi(yv)), r);
      near |= near_bf16_midpoint(z0) | near_bf16_midpoint(z1);
      w[i] = pack_bf16x2(z0, z1);
    }
    st_shared_v4(staged(buf, lane, c), w[0], w[1], w[2], w[3]);
  }
}

// One head of the warp's 32 token rows: D accumulator columns at taddr
// (this lane's row).  row: head 0's row index (b H N + n) of this lane; the
// head's is row + h N.  bias: this head's D bias values in shared memory.
template <int D>
__device__ __forceinline__ void qkv_emit_head(uint32_t taddr, int ocol, bool live, size_t row,
                                              const uint32_t (&rows)[8], const RowsOut& ro, uint32_t stg,
                                              uint32_t bias, const QkvParams& p, const QkvOutMaps& om,
                                              const QkvBars& bars, int lane) {
  const int hd = p.H * D;
  const int which = ocol / hd;  // 0 q, 1 k, 2 v
  const int h = (ocol - which * hd) / D;
  const uint32_t head_rows = static_cast<uint32_t>(h) * static_cast<uint32_t>(p.N);
  const size_t hrow = row + head_rows;
  const uint32_t raw = stg;
  // Y = bf16(acc + bias), 32 columns at a time (packed pairs).
  uint32_t yb[D / 2];
#pragma unroll
  for (int c32 = 0; c32 < D / 32; ++c32) {
    uint32_t acc[32];
    tmem_ld32(taddr + c32 * 32, acc);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 bv = ld_shared_f4(bias + (c32 * 32 + e) * 4);
      yb[c32 * 16 + e / 2] = pack_bf16x2(__uint_as_float(acc[e]) + bv.x, __uint_as_float(acc[e + 1]) + bv.y);
      yb[c32 * 16 + e / 2 + 1] = pack_bf16x2(__uint_as_float(acc[e + 2]) + bv.z, __uint_as_float(acc[e + 3]) + bv.w);
    }
  }
  const float* g = which == 0 ? bars.gq : bars.gk;
  if constexpr (D == 64) {
    const uint32_t hat = raw + kStagingBytes;
    staging_free(lane);
    stage_row(raw, yb, lane);
    if (which == 2) {
      emit_rows<D>(raw, out_map(om, which), out_of(p, which), ro, rows, head_rows, h, 0, lane);
      __syncwarp();
      return;
    }
    const float r = row_rsqrt<D>(yb);
    bool near = false;
    stage_hat_row(hat, yb, smem_u32(g), r, near, lane);
    const unsigned todo = __ballot_sync(0xffffffffu, near && live);
    __syncwarp();
    if (todo) {
      fix_staged_rows(todo, raw, hat, r, g, lane);
      __syncwarp();
    }
    emit_rows<D>(raw, out_map(om, which), out_of(p, which), ro, rows, head_rows, h, 0, lane);
    emit_rows<D>(hat, hat_map(om, which), hat_of(p, which), ro, rows, head_rows, h, 0, lane);
    if (live) r_of(p, which)[hrow] = r;
    __syncwarp();
  } else {
    // d = 128: each 64-column half through the raw staging buffer.
#pragma unroll
    for (int h64 = 0; h64 < 2; ++h64) {
      staging_free(lane);
      stage_row(raw, yb + h64 * 32, lane);
      emit_rows<D>(raw, out_map(om, which), out_of(p, which), ro, rows, head_rows, h, h64 * 64, lane);
      __syncwarp();
    }
    if (which == 2) return;
    const float r = row_rsqrt<D>(yb);
    bool near = false;
#pragma unroll
    for (int h64 = 0; h64 < 2; ++h64) {
      staging_free(lane);
      stage_hat_row(raw, yb + h64 * 32, smem_u32(g + h64 * 64), r, near, lane);
      emit_rows<D>(raw, hat_map(om, which), hat_of(p, which), ro, rows, head_rows, h, h64 * 64, lane);
      __syncwarp();
    }
    // The row re-rounding below stores over these rows: the tile stores first.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
    if (live) r_of(p, which)[hrow] = r;
    const unsigned todo = __ballot_sync(0xffffffffu, near && live);
    if (todo) fix_stored_rows(todo, *reinterpret_cast<const uint32_t(*)[64]>(yb), r, hrow, hat_of(p, which), g, lane);
  }
}

template <int D>
__global__ void __launch_bounds__(QkvCfg<D>::kThreads, 1)
    qkv_norm_kernel(const __grid_constant__ CUtensorMap map_x0, const __grid_constant__ CUtensorMap map_w0,
                    const __grid_constant__ CUtensorMap map_x1, const __grid_constant__ CUtensorMap map_w1,
                    const __grid_constant__ QkvOutMaps om, const __grid_constant__ QkvParams p,
                    const float* __restrict__ gq, const float* __restrict__ gk, uint32_t* dev_err) {
  using Cfg = QkvCfg<D>;
  constexpr int kWarpProd = Cfg::kWarpProd, kWarpIssue = Cfg::kWarpIssue;
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
      mbar_init(&bars.acc_empty[b], Cfg::kEpiThreads);
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
        const int tl = t - (si ? p.s[1].tile0 : p.s[0].tile0);
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
    // Warp w: the TMEM lanes of warp w % 4, and columns 128 (w / 4) .. + 127 of the tile.
    const int lg = warp & 3, wcol = (warp >> 2) * 128;
    const uint32_t stg = smem_u32(sm + Cfg::kOffStaging + warp * Cfg::kStaging);
    const uint32_t bias_w = smem_u32(sm + Cfg::kOffBias + warp * Cfg::kBiasBytes);
    const uint32_t lane_base = static_cast<uint32_t>(lg * 32) << 16;
    const int hd3 = 3 * p.H * D;
    int lt = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++lt) {
      const int abuf = lt & 1;
      const int si = t >= p.s[1].tile0 ? 1 : 0;
      const QkvStream S = stream_of(p, si);
      const int tl = t - S.tile0;
      const int mt = tl / p.n_tiles, nt = tl - mt * p.n_tiles;
      const int col0 = nt * kBN + wcol;  // the warp's first column in Y
      // The bias of the warp's 128 columns (zero past 3 H d, or without a
      // bias) into its shared slice, while the products are still running.
      float4 bq = make_float4(0.f, 0.f, 0.f, 0.f);
      if (S.bias && col0 + lane * 4 < hd3) bq = __ldg(reinterpret_cast<const float4*>(S.bias + col0) + lane);
      __syncwarp();  // the previous tile's reads of the slice are done
      st_shared_v4(bias_w + lane * 16, __float_as_uint(bq.x), __float_as_uint(bq.y), __float_as_uint(bq.z),
                   __float_as_uint(bq.w));
      const bool ok = mbar_wait(&bars.acc_full[abuf], (lt >> 1) & 1, ab, dev_err);
      if (!__all_sync(0xffffffffu, ok)) break;
      __syncwarp();
      tc_fence_after();
      const int m = mt * kBM + lg * 32 + lane;
      const bool live = m < S.M;
      const int bi = live ? m / S.N_s : 0;
      const int n = live ? S.row0 + (m - bi * S.N_s) : 0;
      const size_t row = static_cast<size_t>(bi) * p.H * p.N + n;  // < B H N < 2^31 / d
      const uint32_t row32 = live ? static_cast<uint32_t>(row) : kDeadRow;
      uint32_t rows[8];  // the rows this lane writes out in store_rows
#pragma unroll
      for (int j = 0; j < 8; ++j) rows[j] = __shfl_sync(0xffffffffu, row32, 4 * j + (lane >> 3));
      RowsOut ro;
      {
        const uint32_t first = __shfl_sync(0xffffffffu, row32, 0), last = __shfl_sync(0xffffffffu, row32, 31);
        ro.contig = first != kDeadRow && last != kDeadRow && last - first == 31u;
        ro.n0 = __shfl_sync(0xffffffffu, n, 0);
        ro.bh0 = __shfl_sync(0xffffffffu, bi, 0) * p.H;
      }
#pragma unroll
      for (int j = 0; j < 128 / D; ++j) {
        const int ocol = col0 + j * D;  // the head's first column in Y
        if (ocol < hd3)
          qkv_emit_head<D>(tmem + lane_base + abuf * kBN + wcol + j * D, ocol, live, row, rows, ro, stg,
                           bias_w + j * D * 4, p, om, bars, lane);
      }
      tc_fence_before();
      mbar_arrive(&bars.acc_empty[abuf]);
    }
    if (lane == 0) bulk_wait_group0();  // this warp's tile stores are complete
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIssue) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

}  // namespace

cudaError_t launch_qkv_norm(const CUtensorMap (&maps)[4], const CUtensorMap (&out_maps)[5], const QkvLaunch& a,
                            uint32_t* dev_err, cudaStream_t st) {
  QkvOutMaps om;
  for (int i = 0; i < 3; ++i) om.out[i] = out_maps[i];
  for (int i = 0; i < 2; ++i) om.hat[i] = out_maps[3 + i];
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
  const int sms = device_sm_count();
  const int grid = p.tiles < sms ? p.tiles : sms;
  auto go = [&](auto kernel, int threads, int smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(grid), dim3(threads), smem, st, maps[0], maps[1], maps[2], maps[3], om, p, a.gq,
                      a.gk, dev_err);
  };
  if (a.d == 64) return go(qkv_norm_kernel<64>, QkvCfg<64>::kThreads, QkvCfg<64>::kDynSmem);
  return go(qkv_norm_kernel<128>, QkvCfg<128>::kThreads, QkvCfg<128>::kDynSmem);
}

}  // namespace jattn
