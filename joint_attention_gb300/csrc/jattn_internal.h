// jattn_internal.h — declarations shared by the libjattn translation units
// (kernel launchers and their parameter blocks).  Host-side only; no torch.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace jattn {

// Launches kernel<<<grid, block, smem, st>>>(args...) with programmatic
// stream serialisation, so that its launch and prologue overlap the tail of
// the previous kernel on the stream (the kernel waits on griddepcontrol.wait
// before reading its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Tile sizes of the tensor-core kernels: 128 query rows per tile (the
// tcgen05 M = 128 accumulator, one row per TMEM lane), 128 keys per tile.
constexpr int kTileM = 128;
constexpr int kTileN = 128;

// Rows of every head split into segments that attend only within
// themselves.  A [B, H, N, d] call is B*H heads of one segment [0, N); a
// packed variable-length call is H heads of T = sum of the sequence lengths
// rows with one segment per sequence.  Segment s holds the head's rows
// [cu[s], cu[s+1]); in the 128-row-padded per-head scratch (-LSE log2 e and
// D for the attention backward) it starts at pcu[s], so pcu[s+1] - pcu[s] is
// 128 times the segment's number of 128-row tiles.
constexpr int kMaxSegments = 256;
struct SegTable {
  int n;      // segments per head (1 .. kMaxSegments)
  int rows;   // rows per head
  int prows;  // padded rows per head (pcu[n])
  int cu[kMaxSegments + 1];
  int pcu[kMaxSegments + 1];
};
// Fills t from n + 1 row offsets (cu[0] = 0, strictly increasing); false if
// they are not valid or n is out of range.
bool make_seg_table(SegTable* t, const int* cu, int n);
// One segment of N rows (the [B, H, N, d] layout).
void make_uniform_seg_table(SegTable* t, int N);

// --- norm / elementwise kernels (HBM-bound) ---------------------------------
// The streaming norm kernels take the per-launch device error word: their
// bounded waits on the bulk-copy ring report a timeout through it.
// rq / rk (1/rms of every q / k row) are written unless null.
cudaError_t launch_qk_norm_fwd(const uint16_t* q, const uint16_t* k, const float* gq, const float* gk,
                               uint16_t* qhat, uint16_t* khat, float* rq, float* rk, int64_t rows, int d,
                               uint32_t* dev_err, cudaStream_t st);
// Rows are the BH heads' seg.rows rows.  The softmax statistics are written
// in the per-head padded layout (segment s from seg.pcu[s], 128-row
// multiples): `stats` gets 16 bf16 per row, -LSE * inv_scale and -D each as
// three bf16 terms whose sum rounds to the fp32 value (columns 0-2 and 3-5;
// pad rows -1e30 and 0), zeros after.  The
// dq accumulator rows are zeroed unless dqacc is null (the deterministic
// backward stores its first contribution); the first n_tickets words of
// `tickets` are zeroed.  With qhat null (q_hat, k_hat, rq and rk saved by a
// training forward) only the statistics, the zeroing and the tickets are
// done, and q, k, qhat, khat, rq, rk are not accessed.  With zero_count
// non-null, the zeroing is skipped when *zero_count == zeroed_by (a training
// forward's CTAs zeroed the accumulator and counted themselves there).
cudaError_t launch_bwd_prep(const uint16_t* q, const uint16_t* k, const float* gq, const float* gk,
                            const uint16_t* out, const uint16_t* dout, const float* lse, uint16_t* qhat,
                            uint16_t* khat, float* rq, float* rk, uint16_t* stats,
                            float inv_scale, float* dqacc, unsigned int* tickets, int n_tickets, int BH,
                            const SegTable& seg, int d, uint32_t* dev_err, cudaStream_t st,
                            const uint32_t* zero_count = nullptr, uint32_t zeroed_by = 0);
// nparts = q_norm_bwd_parts() CTAs, each writing one d-vector of dgq
// partials; the last one (by *ticket, zeroed by the backward preparation)
// sums them and the nk dgk partials into dgq and dgk.  zero_count (or null)
// is reset to 0: the accumulator it vouched for is no longer zero.
cudaError_t launch_q_norm_bwd(const float* dqacc, const uint16_t* q, const float* rq, const float* gq, float scale,
                              uint16_t* dq, float* dgq_part, int nparts, int64_t rows, const float* dgk_part, int nk,
                              unsigned int* ticket, float* dgq, float* dgk, int d, uint32_t* dev_err,
                              cudaStream_t st, uint32_t* zero_count = nullptr);
int q_norm_bwd_parts(int d);
// Streaming multiprocessors of the current device (cached after the first
// call), or the limit set by set_sm_limit if that is lower: the number of
// CTAs the persistent kernels launch.
int device_sm_count();
void set_sm_limit(int n);  // n <= 0: no limit

// --- tensor-core attention kernels ------------------------------------------
struct AttnShape {
  int BH;        // heads (B*H, or H for a packed variable-length call)
  int N;         // rows per head
  int d;
  float scale;   // 1/sqrt(d)
  SegTable seg;  // the heads' segments (one segment [0, N) for the [B, H, N, d] layout)
  bool deterministic = false;  // backward: fixed dQ accumulation order
};

// dq_zero / zero_count (training pair, else null): the backward's fp32 dQ
// accumulator ([BH, rows, d]) to zero, and the word each CTA increments once
// its share is zeroed (attn_fwd_grid(s) increments in all).
cudaError_t launch_attn_fwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const AttnShape& s, uint16_t* out, float* lse, uint32_t* dev_err, cudaStream_t st,
                            float* dq_zero = nullptr, uint32_t* zero_count = nullptr);
int attn_fwd_grid(const AttnShape& s);

// map_stats: a TMA map over the bf16 statistics chunks (encode_stats_map);
// map_dq one over the fp32 dQ accumulator (encode_dq_map).  The accumulator must be zeroed unless
// attn_bwd_dq_stores_first(s).
cudaError_t launch_attn_bwd(const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, const CUtensorMap& map_stats, const CUtensorMap& map_dq,
                            const AttnShape& s, const uint16_t* k_raw, const float* rk, const float* gk, uint16_t* dk, uint16_t* dv,
                            float* dqacc, uint32_t* counters, float* dgk_part, uint32_t* dev_err, cudaStream_t st);
// Whether the first dQ contribution to each query tile is stored rather than
// added, so that the accumulator needs no zeroing: the deterministic mode in
// the [B, H, N, d] layout (one segment), whose 128-row tiles end at the
// tensor's end.
inline bool attn_bwd_dq_stores_first(const AttnShape& s) { return s.deterministic && s.seg.n == 1; }
// CTAs of the backward launch (one dgk partial each), and the counter words
// it needs zeroed (deterministic mode: one per query tile; else 0).
int attn_bwd_dgk_parts(const AttnShape& s);
int attn_bwd_counter_words(const AttnShape& s);

// --- QKV projection with the QK-RMSNorm epilogue ---------------------------
// Stream 0 is the image stream, stream 1 the caption stream; maps holds the
// TMA maps of x0, w0, x1, w1 (encode_rows_map: x with 128-row boxes, w with
// 256-row boxes).  A stream with M = 0 rows launches no tiles (its maps are
// then any valid map).
struct QkvLaunch {
  int H, C, N, d;
  int M[2];     // token rows B * N_s
  int N_s[2];   // tokens per batch item
  int row0[2];  // first row in the joint sequence
  const float* bias[2];  // [3 H d] fp32 or null
  const float *gq, *gk;
  uint16_t* out[3];  // q, k, v
  uint16_t* hat[2];  // q_hat, k_hat
  float* r[2];       // rq, rk
};
// out_maps: q, k, v, q_hat, k_hat as encode_bhnd_map_rows(..., 32) maps.
cudaError_t launch_qkv_norm(const CUtensorMap (&maps)[4], const CUtensorMap (&out_maps)[5], const QkvLaunch& a,
                            uint32_t* dev_err, cudaStream_t st);
// A 2-D TMA map over a row-major [rows, cols] bf16 matrix with a
// (64, box_rows) box and 128-byte swizzle (cols * 2 a multiple of 16).
bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows);

// Encodes a 3-D TMA map over a [BH, N, d] bf16 tensor with a (64, 128, 1)
// box and 128-byte swizzle.  Returns false if the driver rejects it.
bool encode_bhnd_map(CUtensorMap* map, const void* base, int BH, int N, int d);
// The same with a (64, box_rows, 1) box.
bool encode_bhnd_map_rows(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);
// A 3-D TMA map over [BH, prows, 16] bf16 statistics chunks with a
// (16, 128, 1) box and 32-byte swizzle.
bool encode_stats_map(CUtensorMap* map, const void* base, int BH, int prows);
// A 3-D TMA map over a [BH, rows, 64] fp32 accumulator with a (32, 128, 1)
// box and 128-byte swizzle.
bool encode_dq_map(CUtensorMap* map, const void* base, int BH, int rows, int d);

}  // namespace jattn
