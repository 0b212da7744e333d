// norm_kernels.cu — the HBM-bound steps around the attention kernels.
//
// QK-RMSNorm (re-diffusion README, "design notes" table, row "QK norm":
// RMSNorm on Q and K): per row of d values,
//     r = (mean_c x_c^2 + eps)^(-1/2),   x_hat = g * x * r  (rounded to bf16)
// and its gradient with u = g * dx_hat:
//     dx = r * u - (r^3 / d) * x * sum_c(u_c x_c),   dg = sum_rows dx_hat * x * r.
//
// Row layout: every row is d contiguous values, d/8 threads per row, each
// thread holding one 16-byte chunk (8 bf16) so global accesses are fully
// coalesced 16-byte vectors; the row reduction is a shuffle within the
// d/8-lane group.  The streaming kernels hold no shared memory and meet no
// block barrier: every thread loads its next rows while it transforms the
// current ones (register double buffering), and grids fill every SM.
#include <atomic>

#include <cuda_bf16.h>

#include "jattn_internal.h"
#include "sm103_ptx.cuh"
#include "bf16_round.cuh"

namespace jattn {
namespace {


__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}
// Sum over the TPR lanes that share a row (TPR = d/8 = 8 or 16).
template <int TPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct F8 {
  float v[8];
};

// (rh, rl) = (mean of the row's squares + eps)^(-1/2) as a double-float.
// Every lane of the warp calls it (row reduction by shuffles).
template <int TPR>
__device__ __forceinline__ void rsqrt_mean_sq_df(const float (&x)[8], float& rh, float& rl) {
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float t, e;
    two_sum(s, __fmul_rn(x[i], x[i]), t, e);
    s = t;
    c = __fadd_rn(c, e);
  }
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
    float t, e;
    two_sum(s, s2, t, e);
    fast_two_sum(t, __fadd_rn(__fadd_rn(c, c2), e), s, c);
  }
  rsqrt_mean_eps_df(s, c, 1.f / (TPR * 8), rh, rl);
}

// The rare path, kept out of line so that the streaming loops keep their
// registers: re-rounds the near-midpoint elements of y (all lanes call it).
template <int TPR>
__device__ __noinline__ F8 rerround_near_midpoints(const uint4 w, const F8 g, F8 y) {
  float x[8];
  unpack8(w, x);
  float rh, rl;
  rsqrt_mean_sq_df<TPR>(x, rh, rl);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (near_bf16_midpoint(y.v[i])) y.v[i] = round_bf16_df(g.v[i], x[i], rh, rl);
  return y;
}

// Normalises one 8-element chunk of a row; returns r through *r_out.  All
// lanes of the warp call it together (row shuffles).
template <int TPR>
__device__ __forceinline__ uint4 norm_chunk(const uint4 w, const float (&g)[8], float* r_out) {
  float x[8];
  unpack8(w, x);
  uint64_t s2 = f2_mul(f2_make(x[0], x[1]), f2_make(x[0], x[1]));
#pragma unroll
  for (int i = 2; i < 8; i += 2) s2 = f2_fma(f2_make(x[i], x[i + 1]), f2_make(x[i], x[i + 1]), s2);
  float sa, sb;
  f2_split(s2, sa, sb);
  const float ss = row_sum<TPR>(sa + sb);
  const float r = rsqrtf(ss * (1.f / (TPR * 8)) + kEps);
  const uint64_t r2 = f2_make(r, r);
  F8 y;
  bool near = false;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    f2_split(f2_mul(f2_mul(f2_make(g[i], g[i + 1]), f2_make(x[i], x[i + 1])), r2), y.v[i], y.v[i + 1]);
    near |= near_bf16_midpoint(y.v[i]) | near_bf16_midpoint(y.v[i + 1]);
  }
  if (__any_sync(0xffffffffu, near)) {
    F8 gg;
#pragma unroll
    for (int i = 0; i < 8; ++i) gg.v[i] = g[i];
    y = rerround_near_midpoints<TPR>(w, gg, y);
  }
  *r_out = r;
  return pack8(y.v);
}

// --- streaming kernels -------------------------------------------------------
constexpr int kNormThreads = 256;
// The dq kernel runs one 1024-thread block per SM: few dgq partials, and
// 1024 / d threads per column for their final sum.
constexpr int kQBwdThreads = 1024;

// q, k -> q_hat, k_hat (bf16), and 1/rms of every row into rq, rk unless
// they are null.  Rows [0, rows) are q rows, [rows, 2 rows) k rows; each
// thread takes kU rows per pass and loads the next pass's rows before it
// transforms the current ones.
template <int D>
__global__ void __launch_bounds__(kNormThreads) qk_norm_fwd_kernel(const uint4* __restrict__ q,
                                                                   const uint4* __restrict__ k,
                                                                   const float* __restrict__ gq,
                                                                   const float* __restrict__ gk,
                                                                   uint4* __restrict__ qhat,
                                                                   uint4* __restrict__ khat, float* __restrict__ rq,
                                                                   float* __restrict__ rk, int64_t rows) {
  constexpr int TPR = D / 8;
  constexpr int RPB = kNormThreads / TPR;  // rows per block and pass slot
  constexpr int kU = 2;
  const int sub = threadIdx.x % TPR;
  griddep_launch_dependents();
  griddep_wait();
  float g_q[8], g_k[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    g_q[i] = gq[sub * 8 + i];
    g_k[i] = gk[sub * 8 + i];
  }
  const int64_t total = 2 * rows;
  const int64_t span = static_cast<int64_t>(RPB) * kU;
  const int64_t step = static_cast<int64_t>(gridDim.x) * span;
  auto load = [&](int64_t b, uint4 (&w)[kU]) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t rr = b + u * RPB + threadIdx.x / TPR;
      w[u] = rr < total ? (rr >= rows ? k[(rr - rows) * TPR + sub] : q[rr * TPR + sub]) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int64_t base = static_cast<int64_t>(blockIdx.x) * span;
  uint4 cur[kU];
  load(base, cur);
  // The loop bound is block-uniform so every lane reaches the row shuffles.
  for (; base < total; base += step) {
    uint4 nxt[kU];
    load(base + step, nxt);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t rr = base + u * RPB + threadIdx.x / TPR;
      const bool is_k = rr >= rows;
      float r;
      const uint4 y = norm_chunk<TPR>(cur[u], is_k ? g_k : g_q, &r);
      if (rr < total) {
        (is_k ? khat[(rr - rows) * TPR + sub] : qhat[rr * TPR + sub]) = y;
        if (rq && sub == 0) (is_k ? rk[rr - rows] : rq[rr]) = r;
      }
      cur[u] = nxt[u];
    }
  }
}

// Backward preparation, one pass over the padded rows (bh, p) of the heads'
// segment-padded layout: a padded row of a segment's first len rows is the
// segment's row t, for which it writes q_hat, k_hat, 1/rms of q and k,
// D = rowsum(dout * out), minus LSE in the log2 domain and a zeroed fp32 dq
// accumulator row; pad rows get -LSE = -inf and D = 0 so the attention
// backward sees zero probabilities.  Each thread loads its next row while it
// transforms the current one.
// x as three bf16 terms (bit patterns), each the round-to-nearest of what
// the previous ones leave (each remainder is exact in fp32): their sum is
// within 2^-24 |x| of x.
__device__ __forceinline__ void split3_bf16(float x, uint32_t (&h)[3]) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    h[i] = __bfloat16_as_ushort(b);
    x -= __bfloat162float(b);
  }
}

// Division of n < 2^31 by a fixed d >= 1 through a multiply-high: with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, n / d =
// (mulhi(n, m) + n) >> l (the round-up method for invariant divisors, as in
// Hacker's Delight, ch. 10); mulhi(n, m) + n < 2^32 for n < 2^31.
struct DivU31 {
  uint32_t m, l;
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> l; }
};
DivU31 make_div_u31(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  DivU31 r;
  r.l = l;
  r.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1);
  return r;
}

template <int D, bool kNorm>
__global__ void __launch_bounds__(kNormThreads) bwd_prep_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ k, const float* __restrict__ gq,
    const float* __restrict__ gk, const uint4* __restrict__ out, const uint4* __restrict__ dout,
    const float* __restrict__ lse, uint4* __restrict__ qhat, uint4* __restrict__ khat, float* __restrict__ rq,
    float* __restrict__ rk, uint4* __restrict__ stats,
    float inv_scale, float4* __restrict__ dqacc, unsigned int* __restrict__ tickets, int n_tickets,
    const __grid_constant__ SegTable seg, int64_t padded_rows, DivU31 div_prows, const uint32_t* zero_count,
    uint32_t zeroed_by) {
  griddep_launch_dependents();
  griddep_wait();
  // The accumulator is already zero when every CTA of the training forward
  // counted its share.
  if (dqacc && zero_count && *zero_count == zeroed_by) dqacc = nullptr;
  for (int i = blockIdx.x * kNormThreads + threadIdx.x; i < n_tickets; i += gridDim.x * kNormThreads)
    tickets[i] = 0u;
  constexpr int TPR = D / 8;
  constexpr int RPB = kNormThreads / TPR;
  const int sub = threadIdx.x % TPR;
  float g_q[8], g_k[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    g_q[i] = gq[sub * 8 + i];
    g_k[i] = gk[sub * 8 + i];
  }
  struct Row {
    uint4 q, k, o, d;
    float lse;
  };
  // Padded rows number below 2^31 (B H N d < 2^31), so the head index comes
  // from a 32-bit multiply-high division.
  auto locate = [&](int64_t b, int64_t& prow, int64_t& row, bool& in_range, bool& valid) {
    prow = b + threadIdx.x / TPR;
    in_range = prow < padded_rows;
    const uint32_t p32 = in_range ? static_cast<uint32_t>(prow) : 0u;
    const uint32_t bh = div_prows.div(p32);
    const int p = static_cast<int>(p32 - bh * static_cast<uint32_t>(seg.prows));
    int lo = 0, hi = seg.n;  // seg.pcu[lo] <= p < seg.pcu[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg.pcu[mid] <= p) lo = mid;
      else hi = mid;
    }
    const int t = seg.cu[lo] + (p - seg.pcu[lo]);
    valid = in_range && t < seg.cu[lo + 1];
    row = static_cast<int64_t>(bh) * seg.rows + t;
  };
  auto load = [&](int64_t b, Row& w) {
    int64_t prow, row;
    bool in_range, valid;
    locate(b, prow, row, in_range, valid);
    const int64_t idx = (valid ? row : 0) * TPR + sub;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    w.q = kNorm && valid ? q[idx] : zero;
    w.k = kNorm && valid ? k[idx] : zero;
    w.o = valid ? out[idx] : zero;
    w.d = valid ? dout[idx] : zero;
    w.lse = (valid && sub == 0) ? lse[row] : 0.f;
  };
  const int64_t step = static_cast<int64_t>(gridDim.x) * RPB;
  int64_t base = static_cast<int64_t>(blockIdx.x) * RPB;
  Row cur;
  load(base, cur);
  for (; base < padded_rows; base += step) {
    Row nxt;
    load(base + step, nxt);
    int64_t prow, row;
    bool in_range, valid;
    locate(base, prow, row, in_range, valid);
    float r1 = 0.f, r2 = 0.f;
    uint4 yq = make_uint4(0u, 0u, 0u, 0u), yk = yq;
    if constexpr (kNorm) {
      yq = norm_chunk<TPR>(cur.q, g_q, &r1);
      yk = norm_chunk<TPR>(cur.k, g_k, &r2);
    }
    float o[8], dd[8];
    unpack8(cur.o, o);
    unpack8(cur.d, dd);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) dot = fmaf(o[i], dd[i], dot);
    dot = row_sum<TPR>(dot);
    if (in_range) {
      // Two 16-byte halves per row: the split statistics, then zeros.
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (sub == 0) {
        uint32_t l[3], dd3[3];
        split3_bf16(valid ? -cur.lse * inv_scale : -1e30f, l);
        split3_bf16(valid ? -dot : 0.f, dd3);
        v = make_uint4(l[0] | (l[1] << 16), l[2] | (dd3[0] << 16), dd3[1] | (dd3[2] << 16), 0u);
      }
      if (sub < 2) stats[prow * 2 + sub] = v;
      if (valid) {
        const int64_t idx = row * TPR + sub;
        if constexpr (kNorm) {
          qhat[idx] = yq;
          khat[idx] = yk;
        }
        if (dqacc) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          dqacc[idx * 2] = z;
          dqacc[idx * 2 + 1] = z;
        }
        if (kNorm && sub == 0) {
          rq[row] = r1;
          rk[row] = r2;
        }
      }
    }
    cur = nxt;
  }
}

// dq from the fp32 accumulator of dS k_hat (times `scale`), and the gain
// gradients.  Each block writes its dgq partial to partial[blockIdx.x][d];
// the last block to finish (an atomic ticket, zeroed by the backward
// preparation) then sums every block's dgq partial and the attention
// backward's nk dgk partials, each in index order, into dgq and dgk.  The
// grid size is fixed, so the reduction order is fixed.  Each thread loads its
// next row while it transforms the current one.
template <int D>
__global__ void __launch_bounds__(kQBwdThreads) q_norm_bwd_kernel(const float4* __restrict__ dqacc,
                                                                  const uint4* __restrict__ q,
                                                                  const float* __restrict__ rq,
                                                                  const float* __restrict__ gq, float scale,
                                                                  uint4* __restrict__ dq,
                                                                  float* __restrict__ partial, int64_t rows,
                                                                  const float* __restrict__ part_k, int nk,
                                                                  unsigned int* __restrict__ ticket,
                                                                  float* __restrict__ dgq, float* __restrict__ dgk,
                                                                  uint32_t* zero_count) {
  constexpr int TPR = D / 8;
  constexpr int RPB = kQBwdThreads / TPR;
  const int sub = threadIdx.x % TPR;
  griddep_launch_dependents();
  griddep_wait();
  if (zero_count && blockIdx.x == 0 && threadIdx.x == 0) *zero_count = 0u;
  float g[8], acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    g[i] = gq[sub * 8 + i];
    acc[i] = 0.f;
  }
  struct Row {
    float4 a, b;
    uint4 x;
    float r;
  };
  auto load = [&](int64_t b, Row& w) {
    const int64_t row = b + threadIdx.x / TPR;
    const bool valid = row < rows;
    const int64_t idx = (valid ? row : 0) * TPR + sub;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    w.a = valid ? dqacc[idx * 2] : z4;
    w.b = valid ? dqacc[idx * 2 + 1] : z4;
    w.x = valid ? q[idx] : make_uint4(0u, 0u, 0u, 0u);
    w.r = valid ? rq[row] : 0.f;
  };
  const int64_t step = static_cast<int64_t>(gridDim.x) * RPB;
  int64_t base = static_cast<int64_t>(blockIdx.x) * RPB;
  Row cur;
  load(base, cur);
  for (; base < rows; base += step) {
    Row nxt;
    load(base + step, nxt);
    const int64_t row = base + threadIdx.x / TPR;
    const float dh[8] = {cur.a.x * scale, cur.a.y * scale, cur.a.z * scale, cur.a.w * scale,
                         cur.b.x * scale, cur.b.y * scale, cur.b.z * scale, cur.b.w * scale};
    float x[8];
    unpack8(cur.x, x);
    const float r = cur.r;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) dot = fmaf(g[i] * dh[i], x[i], dot);
    dot = row_sum<TPR>(dot);
    const float c = r * r * r * (1.f / D) * dot;
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[i] = r * g[i] * dh[i] - c * x[i];
      acc[i] = fmaf(dh[i], x[i] * r, acc[i]);  // rows past the end are zero
    }
    if (row < rows) dq[row * TPR + sub] = pack8(y);
    cur = nxt;
  }
  // Block reduction of acc over the RPB row slots, in a fixed order: kSplit
  // threads per column each add the slots w = sl (mod kSplit) in slot order,
  // then one thread per column adds the kSplit slices in slice order.
  constexpr int kSplit = kQBwdThreads / D;
  static_assert(RPB % kSplit == 0, "slots per slice");
  __shared__ float red[RPB][D];
  __shared__ float comb[2][kSplit][D];
  const int slot = threadIdx.x / TPR;
#pragma unroll
  for (int i = 0; i < 8; ++i) red[slot][sub * 8 + i] = acc[i];
  __syncthreads();
  const int c = threadIdx.x % D, sl = threadIdx.x / D;
  {
    float t = 0.f;
#pragma unroll
    for (int w = sl; w < RPB; w += kSplit) t += red[w][c];
    comb[0][sl][c] = t;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kSplit; ++i) t += comb[0][i][c];
    partial[static_cast<size_t>(blockIdx.x) * D + c] = t;
  }
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // kSplit threads per column, each summing the partial rows p = sl (mod
  // kSplit) in order, the dgq and dgk rows of a chunk loaded together; the
  // slices are then added in slice order.
  constexpr int kChunk = 12;
  const int nq = static_cast<int>(gridDim.x);
  const int n = nq > nk ? nq : nk;
  float sq = 0.f, sk = 0.f;
  for (int p0 = sl; p0 < n; p0 += kChunk * kSplit) {
    float vq[kChunk], vk[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int p = p0 + i * kSplit;
      vq[i] = p < nq ? __ldcg(&partial[static_cast<size_t>(p) * D + c]) : 0.f;
      vk[i] = p < nk ? __ldcg(&part_k[static_cast<size_t>(p) * D + c]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      sq += vq[i];
      sk += vk[i];
    }
  }
  comb[0][sl][c] = sq;
  comb[1][sl][c] = sk;
  __syncthreads();
  if (threadIdx.x < D) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int i = 0; i < kSplit; ++i) {
      a += comb[0][i][c];
      b += comb[1][i][c];
    }
    dgq[c] = a;
    dgk[c] = b;
  }
}

std::atomic<int> g_sm_limit{0};

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  const int lim = g_sm_limit.load(std::memory_order_relaxed);
  return lim > 0 && lim < n ? lim : n;
}

// As many 256-thread blocks as fit on every SM (from the kernel's
// registers), no more than the rows need.
template <class Kernel>
int row_grid(Kernel kernel, int64_t rows, int d) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kNormThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t rpb = kNormThreads / (d / 8);
  const int64_t need = (rows + rpb - 1) / rpb;
  const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace

int device_sm_count() { return sm_count(); }

void set_sm_limit(int n) { g_sm_limit.store(n > 0 ? n : 0, std::memory_order_relaxed); }

int q_norm_bwd_parts(int d) {
  int per_sm = 1;
  const cudaError_t e = d == 128 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q_norm_bwd_kernel<128>,
                                                                                   kQBwdThreads, 0)
                                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q_norm_bwd_kernel<64>,
                                                                                   kQBwdThreads, 0);
  if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  return sm_count() * per_sm;
}

cudaError_t launch_qk_norm_fwd(const uint16_t* q, const uint16_t* k, const float* gq, const float* gk,
                               uint16_t* qhat, uint16_t* khat, float* rq, float* rk, int64_t rows, int d,
                               uint32_t* dev_err, cudaStream_t st) {
  (void)dev_err;
  auto* a = reinterpret_cast<const uint4*>(q);
  auto* b = reinterpret_cast<const uint4*>(k);
  auto kernel = d == 64 ? qk_norm_fwd_kernel<64> : qk_norm_fwd_kernel<128>;
  return launch_pdl(kernel, dim3(row_grid(kernel, 2 * rows, d)), dim3(kNormThreads), 0, st, a, b, gq, gk,
                    reinterpret_cast<uint4*>(qhat), reinterpret_cast<uint4*>(khat), rq, rk, rows);
}

cudaError_t launch_bwd_prep(const uint16_t* q, const uint16_t* k, const float* gq, const float* gk,
                            const uint16_t* out, const uint16_t* dout, const float* lse, uint16_t* qhat,
                            uint16_t* khat, float* rq, float* rk, uint16_t* stats,
                            float inv_scale, float* dqacc, unsigned int* tickets, int n_tickets, int BH,
                            const SegTable& seg, int d, uint32_t* dev_err, cudaStream_t st,
                            const uint32_t* zero_count, uint32_t zeroed_by) {
  (void)dev_err;
  const int64_t padded_rows = static_cast<int64_t>(BH) * seg.prows;
  auto u4 = [](const uint16_t* p) { return reinterpret_cast<const uint4*>(p); };
  // q_hat / k_hat / rq / rk saved by a training forward: only the statistics.
  const bool norm = qhat != nullptr;
  auto kernel = d == 64 ? (norm ? bwd_prep_kernel<64, true> : bwd_prep_kernel<64, false>)
                        : (norm ? bwd_prep_kernel<128, true> : bwd_prep_kernel<128, false>);
  return launch_pdl(kernel, dim3(row_grid(kernel, padded_rows, d)), dim3(kNormThreads), 0, st, u4(q), u4(k), gq,
                    gk, u4(out), u4(dout), lse, reinterpret_cast<uint4*>(qhat), reinterpret_cast<uint4*>(khat), rq,
                    rk, reinterpret_cast<uint4*>(stats), inv_scale, reinterpret_cast<float4*>(dqacc),
                    tickets, n_tickets, seg, padded_rows, make_div_u31(static_cast<uint32_t>(seg.prows)), zero_count,
                    zeroed_by);
}

cudaError_t launch_q_norm_bwd(const float* dqacc, const uint16_t* q, const float* rq, const float* gq, float scale,
                              uint16_t* dq, float* dgq_part, int nparts, int64_t rows, const float* dgk_part, int nk,
                              unsigned int* ticket, float* dgq, float* dgk, int d, uint32_t* dev_err,
                              cudaStream_t st, uint32_t* zero_count) {
  (void)dev_err;
  auto* a = reinterpret_cast<const float4*>(dqacc);
  auto* x = reinterpret_cast<const uint4*>(q);
  auto* y = reinterpret_cast<uint4*>(dq);
  // Every one of the nparts blocks writes its partial (zeros if it has no row).
  return launch_pdl(d == 64 ? q_norm_bwd_kernel<64> : q_norm_bwd_kernel<128>, dim3(nparts), dim3(kQBwdThreads), 0,
                    st, a, x, rq, gq, scale, y, dgq_part, rows, dgk_part, nk, ticket, dgq, dgk, zero_count);
}

}  // namespace jattn
