// jattn_api.cu — the C ABI of libjattn (declared in include/jattn.h):
// argument validation, per-call scratch, TMA tensor maps and the launch
// sequence of the forward and backward passes.
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "jattn.h"
#include "jattn_internal.h"
#include "sm103_ptx.cuh"

namespace jattn {
namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;

// Device error word written by the kernels' bounded waits (one per device).
__device__ uint32_t g_dev_err;

// Backward mode set by jattn_set_deterministic (applies to later calls).
std::atomic<int> g_deterministic{0};

// Text of the last failure seen by an entry point on this thread.
thread_local char g_last_msg[256] = "no error";

int fail(int status, const char* where, cudaError_t e = cudaSuccess) {
  if (e != cudaSuccess)
    snprintf(g_last_msg, sizeof(g_last_msg), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  else
    snprintf(g_last_msg, sizeof(g_last_msg), "%s", where);
  return status;
}

uint32_t* dev_err_ptr() {
  static uint32_t* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ---------------------------------------------------------------------------
// Kernel timing: CUDA event pairs around each launch while enabled.
// ---------------------------------------------------------------------------
struct Prof {
  std::mutex mu;
  bool on = false;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  long long launches[JATTN_KERNEL_COUNT] = {0};
  double ms[JATTN_KERNEL_COUNT] = {0};

  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
};
Prof& prof() {
  static Prof p;
  return p;
}

// Brackets one launch; a no-op unless timing is enabled.
class Timed {
 public:
  Timed(int kind, cudaStream_t st) : kind_(kind), st_(st) {
    Prof& p = prof();
    std::lock_guard<std::mutex> lock(p.mu);
    if (!p.on) return;
    a_ = p.get();
    b_ = p.get();
    if (a_ && b_) cudaEventRecord(a_, st_);
  }
  ~Timed() {
    if (!a_ || !b_) return;
    cudaEventRecord(b_, st_);
    Prof& p = prof();
    std::lock_guard<std::mutex> lock(p.mu);
    p.pending.push_back({kind_, a_, b_});
  }

 private:
  int kind_;
  cudaStream_t st_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

struct Range {
  uintptr_t lo, hi;
};
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range range_of(const void* p, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + bytes};
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
  int B, H, N, d, BH;  // BH heads of N rows each (packed variable-length: H heads of T rows)
  size_t rows;         // BH * N
  size_t elems;        // BH * N * d
  SegTable seg;        // the heads' segments
};

int check_shape(int B, int H, int N_img, int N_txt, int d, Shape* s) {
  if (B <= 0 || H <= 0 || d <= 0 || N_img < 0 || N_txt < 0) return JATTN_ERR_INVALID_ARG;
  const int64_t N = static_cast<int64_t>(N_img) + N_txt;
  if (N < 1) return JATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return JATTN_ERR_UNSUPPORTED;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > 65535) return JATTN_ERR_INVALID_ARG;  // grid y extent
  const int64_t elems = BH * N * d;
  if (elems >= (int64_t{1} << 31)) return JATTN_ERR_INVALID_ARG;
  s->B = B;
  s->H = H;
  s->N = static_cast<int>(N);
  s->d = d;
  s->BH = static_cast<int>(BH);
  s->rows = static_cast<size_t>(BH * N);
  s->elems = static_cast<size_t>(elems);
  make_uniform_seg_table(&s->seg, s->N);
  return JATTN_OK;
}

// Packed variable-length layout: H heads of T = cu[n] rows, one segment per
// sequence.  cu is a host array of n + 1 row offsets.
int check_shape_varlen(const int* cu, int n, int H, int d, Shape* s) {
  if (!cu || n < 1 || H <= 0 || d <= 0) return JATTN_ERR_INVALID_ARG;
  if (n > kMaxSegments) return JATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return JATTN_ERR_UNSUPPORTED;
  if (H > 65535) return JATTN_ERR_INVALID_ARG;
  if (!make_seg_table(&s->seg, cu, n)) return JATTN_ERR_INVALID_ARG;
  const int64_t T = s->seg.rows;
  const int64_t elems = static_cast<int64_t>(H) * T * d;
  if (elems >= (int64_t{1} << 31) || static_cast<int64_t>(H) * s->seg.prows >= (int64_t{1} << 31))
    return JATTN_ERR_INVALID_ARG;
  s->B = 1;
  s->H = H;
  s->N = static_cast<int>(T);
  s->d = d;
  s->BH = H;
  s->rows = static_cast<size_t>(H) * T;
  s->elems = static_cast<size_t>(elems);
  return JATTN_OK;
}

// Bump allocator over one stream-ordered allocation.
struct Carve {
  uint8_t* base = nullptr;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = reinterpret_cast<T*>(base + off);
    off += count * sizeof(T);
    return p;
  }
};

size_t fwd_scratch_bytes(const Shape& s) { return 2 * (s.elems * 2 + 256) + 256; }

// The activations a training forward keeps for its backward, at 256-byte
// aligned offsets of one caller buffer: q_hat, k_hat (bf16, q's shape), then
// 1/rms of every q and k row (fp32); then the backward's fp32 dQ accumulator
// (q's shape), which the forward zeroes with bandwidth it leaves idle, and the
// word that counts the forward CTAs that have zeroed their share.
struct SavedLayout {
  size_t qhat, khat, rq, rk, dq, zero_count, total;
};
SavedLayout saved_layout(const Shape& s) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SavedLayout l;
  l.qhat = 0;
  l.khat = up(s.elems * 2);
  l.rq = l.khat + up(s.elems * 2);
  l.rk = l.rq + up(s.rows * 4);
  l.dq = l.rk + up(s.rows * 4);
  l.zero_count = l.dq + up(s.elems * 4);
  l.total = l.zero_count + 256;
  return l;
}

size_t bwd_scratch_bytes(const Shape& s, int nparts_q, int nparts_k, int counter_words, bool saved) {
  size_t b = 0;
  if (!saved) {
    b += 2 * (s.elems * 2 + 256);  // q_hat, k_hat
    b += 2 * (s.rows * 4 + 256);   // rq, rk
    b += s.elems * 4 + 256;        // dq accumulator
  }
  b += static_cast<size_t>(s.BH) * s.seg.prows * 32 + 256;  // statistics chunks
  b += (static_cast<size_t>(nparts_q) + nparts_k) * s.d * 4 + 512; // dg partials
  b += 4 * (1 + static_cast<size_t>(counter_words)) + 256;      // dg ticket, dQ order counters
  return b + 256;
}

}  // namespace

bool make_seg_table(SegTable* t, const int* cu, int n) {
  if (!t || !cu || n < 1 || n > kMaxSegments || cu[0] != 0) return false;
  t->n = n;
  t->cu[0] = 0;
  t->pcu[0] = 0;
  for (int i = 0; i < n; ++i) {
    if (cu[i + 1] <= cu[i]) return false;  // every segment has a row
    const int64_t padded = t->pcu[i] + (static_cast<int64_t>(cu[i + 1] - cu[i]) + 127) / 128 * 128;
    if (padded >= (int64_t{1} << 31)) return false;
    t->cu[i + 1] = cu[i + 1];
    t->pcu[i + 1] = static_cast<int>(padded);
  }
  t->rows = cu[n];
  t->prows = t->pcu[n];
  return true;
}

void make_uniform_seg_table(SegTable* t, int N) {
  const int cu[2] = {0, N};
  make_seg_table(t, cu, 1);
}

bool encode_bhnd_map(CUtensorMap* map, const void* base, int BH, int N, int d) {
  return encode_bhnd_map_rows(map, base, BH, N, d, 128);
}

bool encode_bhnd_map_rows(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_dq_map(CUtensorMap* map, const void* base, int BH, int rows, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(rows) * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_stats_map(CUtensorMap* map, const void* base, int BH, int prows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {16, static_cast<cuuint64_t>(prows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {32, static_cast<cuuint64_t>(prows) * 32};
  cuuint32_t box[3] = {16, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace jattn

using namespace jattn;

namespace jattn {
namespace {

// The fixed scratch of jattn_fwd_noalloc (see include/jattn.h): one array per
// device, looked up once per device and then shared by every call.
static __device__ __align__(256) uint8_t g_noalloc_scratch[JATTN_NOALLOC_SCRATCH_BYTES];

uint8_t* noalloc_scratch_ptr() {
  static uint8_t* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      fail(JATTN_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch)", e);
      return nullptr;
    }
    ptrs[dev] = static_cast<uint8_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace jattn

extern "C" int jattn_fwd_noalloc(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                                 const float* gk, int B, int H, int N_img, int N_txt, int d, jattn_bf16* out,
                                 float* lse, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  const void* ptrs[] = {q, k, v, gq, gk, out, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JATTN_ERR_MISALIGNED;
  const size_t tb = s.elems * 2;
  const Range ins[] = {range_of(q, tb), range_of(k, tb), range_of(v, tb), range_of(gq, s.d * 4),
                       range_of(gk, s.d * 4)};
  const Range outs[] = {range_of(out, tb), range_of(lse, s.rows * 4)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlaps(o, i)) return JATTN_ERR_ALIAS;
  if (overlaps(outs[0], outs[1])) return JATTN_ERR_ALIAS;
  const size_t part = (tb + 255) & ~static_cast<size_t>(255);
  if (2 * part > JATTN_NOALLOC_SCRATCH_BYTES) return JATTN_ERR_SCRATCH_LIMIT;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word", cudaGetLastError());
  uint8_t* scratch = noalloc_scratch_ptr();
  if (!scratch) return JATTN_ERR_CUDA;
  uint16_t* qhat = reinterpret_cast<uint16_t*>(scratch);
  uint16_t* khat = reinterpret_cast<uint16_t*>(scratch + part);
  cudaError_t ce;
  {
    Timed t(JATTN_KERNEL_QK_NORM_FWD, st);
    ce = launch_qk_norm_fwd(q, k, gq, gk, qhat, khat, nullptr, nullptr, static_cast<int64_t>(s.rows), s.d, err, st);
  }
  if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "qk_norm_fwd launch", ce);
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, qhat, s.BH, s.N, s.d) || !encode_bhnd_map(&mk, khat, s.BH, s.N, s.d) ||
      !encode_bhnd_map(&mv, v, s.BH, s.N, s.d))
    return fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  AttnShape as{s.BH, s.N, s.d, 1.0f / sqrtf(static_cast<float>(s.d)), s.seg};
  Timed t(JATTN_KERNEL_ATTN_FWD, st);
  ce = launch_attn_fwd(mq, mk, mv, as, out, lse, err, st);
  if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "attn_fwd launch", ce);
  return JATTN_OK;
}

namespace {

// The forward for a validated shape (either layout); with `saved` non-null
// (a training forward) q_hat, k_hat and the rows' 1/rms go there instead of
// into scratch.
int fwd_body(const Shape& s, const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
             const float* gk, jattn_bf16* out, float* lse, void* saved, void* stream) {
  const void* ptrs[] = {q, k, v, gq, gk, out, lse, saved};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JATTN_ERR_MISALIGNED;
  const size_t tb = s.elems * 2;
  const SavedLayout sl = saved_layout(s);
  const Range ins[] = {range_of(q, tb), range_of(k, tb), range_of(v, tb), range_of(gq, s.d * 4),
                       range_of(gk, s.d * 4)};
  const Range outs[] = {range_of(out, tb), range_of(lse, s.rows * 4), range_of(saved, saved ? sl.total : 0)};
  for (size_t a = 0; a < sizeof(outs) / sizeof(outs[0]); ++a) {
    for (const Range& i : ins)
      if (overlaps(outs[a], i)) return JATTN_ERR_ALIAS;
    for (size_t b = a + 1; b < sizeof(outs) / sizeof(outs[0]); ++b)
      if (overlaps(outs[a], outs[b])) return JATTN_ERR_ALIAS;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word", cudaGetLastError());
  Carve cv;
  uint16_t *qhat, *khat;
  float *rq = nullptr, *rk = nullptr;
  cudaError_t ce;
  if (saved) {
    uint8_t* base = static_cast<uint8_t*>(saved);
    qhat = reinterpret_cast<uint16_t*>(base + sl.qhat);
    khat = reinterpret_cast<uint16_t*>(base + sl.khat);
    rq = reinterpret_cast<float*>(base + sl.rq);
    rk = reinterpret_cast<float*>(base + sl.rk);
  } else {
    ce = cudaMallocAsync(reinterpret_cast<void**>(&cv.base), fwd_scratch_bytes(s), st);
    if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "cudaMallocAsync", ce);
    qhat = cv.take<uint16_t>(s.elems);
    khat = cv.take<uint16_t>(s.elems);
  }
  int status = JATTN_OK;
  CUtensorMap mq, mk, mv;
  {
    Timed t(JATTN_KERNEL_QK_NORM_FWD, st);
    ce = launch_qk_norm_fwd(q, k, gq, gk, qhat, khat, rq, rk, static_cast<int64_t>(s.rows), s.d, err, st);
  }
  if (ce != cudaSuccess) {
    status = fail(JATTN_ERR_CUDA, "qk_norm_fwd launch", ce);
  } else if (!encode_bhnd_map(&mq, qhat, s.BH, s.N, s.d) || !encode_bhnd_map(&mk, khat, s.BH, s.N, s.d) ||
             !encode_bhnd_map(&mv, v, s.BH, s.N, s.d)) {
    status = fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  } else {
    AttnShape as{s.BH, s.N, s.d, 1.0f / sqrtf(static_cast<float>(s.d)), s.seg};
    Timed t(JATTN_KERNEL_ATTN_FWD, st);
    uint8_t* base = static_cast<uint8_t*>(saved);
    ce = launch_attn_fwd(mq, mk, mv, as, out, lse, err, st, saved ? reinterpret_cast<float*>(base + sl.dq) : nullptr,
                         saved ? reinterpret_cast<uint32_t*>(base + sl.zero_count) : nullptr);
    if (ce != cudaSuccess) status = fail(JATTN_ERR_CUDA, "attn_fwd launch", ce);
  }
  if (cv.base) {
    ce = cudaFreeAsync(cv.base, st);
    if (ce != cudaSuccess) status = fail(JATTN_ERR_CUDA, "cudaFreeAsync", ce);
  }
  return status;
}

}  // namespace

extern "C" int jattn_fwd(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                         const float* gk, int B, int H, int N_img, int N_txt, int d, jattn_bf16* out, float* lse,
                         void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  return fwd_body(s, q, k, v, gq, gk, out, lse, nullptr, stream);
}

extern "C" int jattn_fwd_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                                const float* gk, const int* cu_seqlens, int n_seqs, int H, int d, jattn_bf16* out,
                                float* lse, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape_varlen(cu_seqlens, n_seqs, H, d, &s);
  if (rc != JATTN_OK) return rc;
  return fwd_body(s, q, k, v, gq, gk, out, lse, nullptr, stream);
}

namespace {

// The backward for a validated shape (either layout); with `saved` non-null
// q_hat, k_hat and the rows' 1/rms come from a training forward instead of
// being recomputed.
int bwd_body(const Shape& s, const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
             const float* gk, const jattn_bf16* out, const float* lse, const jattn_bf16* dout, void* saved,
             jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq, float* dgk, void* stream) {
  const void* ptrs[] = {q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JATTN_ERR_MISALIGNED;
  const size_t tb = s.elems * 2;
  const size_t gb = static_cast<size_t>(s.d) * 4;
  const SavedLayout sl = saved_layout(s);
  const Range ins[] = {range_of(q, tb),  range_of(k, tb),   range_of(v, tb),           range_of(gq, gb),
                       range_of(gk, gb), range_of(out, tb), range_of(lse, s.rows * 4), range_of(dout, tb),
                       range_of(saved, saved ? sl.total : 0)};
  const Range outs[] = {range_of(dq, tb), range_of(dk, tb), range_of(dv, tb), range_of(dgq, gb), range_of(dgk, gb)};
  for (size_t a = 0; a < sizeof(outs) / sizeof(outs[0]); ++a) {
    for (const Range& i : ins)
      if (overlaps(outs[a], i)) return JATTN_ERR_ALIAS;
    for (size_t b = a + 1; b < sizeof(outs) / sizeof(outs[0]); ++b)
      if (overlaps(outs[a], outs[b])) return JATTN_ERR_ALIAS;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word", cudaGetLastError());
  AttnShape as{s.BH, s.N, s.d, 1.0f / sqrtf(static_cast<float>(s.d)), s.seg};
  const int nparts_q = q_norm_bwd_parts(s.d);
  as.deterministic = g_deterministic.load(std::memory_order_relaxed) != 0;
  const int nparts_k = attn_bwd_dgk_parts(as);
  const int counter_words = attn_bwd_counter_words(as);
  Carve cv;
  cudaError_t ce = cudaMallocAsync(reinterpret_cast<void**>(&cv.base),
                                   bwd_scratch_bytes(s, nparts_q, nparts_k, counter_words, saved != nullptr), st);
  if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "cudaMallocAsync", ce);
  uint16_t *qhat, *khat;
  float *rq, *rk, *dqacc;
  uint32_t* zero_count = nullptr;
  if (saved) {
    uint8_t* base = static_cast<uint8_t*>(saved);
    qhat = reinterpret_cast<uint16_t*>(base + sl.qhat);
    khat = reinterpret_cast<uint16_t*>(base + sl.khat);
    rq = reinterpret_cast<float*>(base + sl.rq);
    rk = reinterpret_cast<float*>(base + sl.rk);
    dqacc = reinterpret_cast<float*>(base + sl.dq);
    zero_count = reinterpret_cast<uint32_t*>(base + sl.zero_count);
  } else {
    qhat = cv.take<uint16_t>(s.elems);
    khat = cv.take<uint16_t>(s.elems);
    rq = cv.take<float>(s.rows);
    rk = cv.take<float>(s.rows);
    dqacc = cv.take<float>(s.elems);
  }
  uint16_t* stats = cv.take<uint16_t>(static_cast<size_t>(s.BH) * s.seg.prows * 16);
  float* dgq_part = cv.take<float>(static_cast<size_t>(nparts_q) * s.d);
  float* dgk_part = cv.take<float>(static_cast<size_t>(nparts_k) * s.d);
  // The gain-gradient ticket, then (deterministic mode) one dQ order counter
  // per query tile; the preparation zeroes them all.
  unsigned int* dg_ticket = cv.take<unsigned int>(1 + static_cast<size_t>(counter_words));

  int status = JATTN_OK;
  CUtensorMap mq, mk, mv, mdo, mstats, mdqacc;
  {
    Timed t(JATTN_KERNEL_BWD_PREP, st);
    // Saved activations: the preparation computes only the statistics.
    ce = launch_bwd_prep(q, k, gq, gk, out, dout, lse, saved ? nullptr : qhat, khat, rq, rk, stats,
                         sqrtf(static_cast<float>(s.d)), attn_bwd_dq_stores_first(as) ? nullptr : dqacc, dg_ticket,
                         1 + counter_words, s.BH, s.seg, s.d, err, st, zero_count,
                         static_cast<uint32_t>(attn_fwd_grid(as)));
  }
  if (ce != cudaSuccess) {
    status = fail(JATTN_ERR_CUDA, "bwd_prep launch", ce);
  } else if (!encode_bhnd_map(&mq, qhat, s.BH, s.N, s.d) || !encode_bhnd_map(&mk, khat, s.BH, s.N, s.d) ||
             !encode_bhnd_map(&mv, v, s.BH, s.N, s.d) || !encode_bhnd_map(&mdo, dout, s.BH, s.N, s.d) ||
             !encode_stats_map(&mstats, stats, s.BH, s.seg.prows) ||
             !encode_dq_map(&mdqacc, dqacc, s.BH, s.seg.rows, s.d)) {
    status = fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  } else {
    const char* stage = "attn_bwd launch";
    {
      Timed t(JATTN_KERNEL_ATTN_BWD, st);
      ce = launch_attn_bwd(mq, mk, mv, mdo, mstats, mdqacc, as, k, rk, gk, dk, dv, dqacc, dg_ticket + 1, dgk_part, err,
                           st);
    }
    if (ce == cudaSuccess) {
      stage = "q_norm_bwd launch";
      Timed t(JATTN_KERNEL_Q_NORM_BWD, st);
      ce = launch_q_norm_bwd(dqacc, q, rq, gq, as.scale, dq, dgq_part, nparts_q, static_cast<int64_t>(s.rows),
                             dgk_part, nparts_k, dg_ticket, dgq, dgk, s.d, err, st, zero_count);
    }
    if (ce != cudaSuccess) status = fail(JATTN_ERR_CUDA, stage, ce);
  }
  ce = cudaFreeAsync(cv.base, st);
  if (ce != cudaSuccess) status = fail(JATTN_ERR_CUDA, "cudaFreeAsync", ce);
  return status;
}

}  // namespace

extern "C" int jattn_bwd(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                         const float* gk, const jattn_bf16* out, const float* lse, const jattn_bf16* dout,
                         jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq, float* dgk, int B, int H,
                         int N_img, int N_txt, int d, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !dout || !dq || !dk || !dv || !dgq || !dgk)
    return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  return bwd_body(s, q, k, v, gq, gk, out, lse, dout, nullptr, dq, dk, dv, dgq, dgk, stream);
}

extern "C" int jattn_bwd_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                                const float* gk, const jattn_bf16* out, const float* lse, const jattn_bf16* dout,
                                jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq, float* dgk,
                                const int* cu_seqlens, int n_seqs, int H, int d, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !dout || !dq || !dk || !dv || !dgq || !dgk)
    return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape_varlen(cu_seqlens, n_seqs, H, d, &s);
  if (rc != JATTN_OK) return rc;
  return bwd_body(s, q, k, v, gq, gk, out, lse, dout, nullptr, dq, dk, dv, dgq, dgk, stream);
}

extern "C" size_t jattn_saved_bytes(int B, int H, int N_img, int N_txt, int d) {
  Shape s;
  if (check_shape(B, H, N_img, N_txt, d, &s) != JATTN_OK) return 0;
  return saved_layout(s).total;
}

extern "C" size_t jattn_saved_bytes_varlen(const int* cu_seqlens, int n_seqs, int H, int d) {
  Shape s;
  if (check_shape_varlen(cu_seqlens, n_seqs, H, d, &s) != JATTN_OK) return 0;
  return saved_layout(s).total;
}

extern "C" int jattn_fwd_train(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                               const float* gk, int B, int H, int N_img, int N_txt, int d, jattn_bf16* out,
                               float* lse, void* saved, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !saved) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  return fwd_body(s, q, k, v, gq, gk, out, lse, saved, stream);
}

extern "C" int jattn_fwd_train_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                                      const float* gk, const int* cu_seqlens, int n_seqs, int H, int d,
                                      jattn_bf16* out, float* lse, void* saved, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !saved) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape_varlen(cu_seqlens, n_seqs, H, d, &s);
  if (rc != JATTN_OK) return rc;
  return fwd_body(s, q, k, v, gq, gk, out, lse, saved, stream);
}

extern "C" int jattn_bwd_train(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                               const float* gk, const jattn_bf16* out, const float* lse, const jattn_bf16* dout,
                               void* saved, jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq,
                               float* dgk, int B, int H, int N_img, int N_txt, int d, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !dout || !saved || !dq || !dk || !dv || !dgq || !dgk)
    return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  return bwd_body(s, q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk, stream);
}

extern "C" int jattn_bwd_train_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v,
                                      const float* gq, const float* gk, const jattn_bf16* out, const float* lse,
                                      const jattn_bf16* dout, void* saved, jattn_bf16* dq, jattn_bf16* dk,
                                      jattn_bf16* dv, float* dgq, float* dgk, const int* cu_seqlens, int n_seqs,
                                      int H, int d, void* stream) {
  if (!q || !k || !v || !gq || !gk || !out || !lse || !dout || !saved || !dq || !dk || !dv || !dgq || !dgk)
    return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape_varlen(cu_seqlens, n_seqs, H, d, &s);
  if (rc != JATTN_OK) return rc;
  return bwd_body(s, q, k, v, gq, gk, out, lse, dout, saved, dq, dk, dv, dgq, dgk, stream);
}

extern "C" int jattn_qkv_norm(const jattn_bf16* x_img, const jattn_bf16* w_img, const float* b_img,
                              const jattn_bf16* x_txt, const jattn_bf16* w_txt, const float* b_txt, const float* gq,
                              const float* gk, int B, int H, int N_img, int N_txt, int d, int C, jattn_bf16* q,
                              jattn_bf16* k, jattn_bf16* v, void* saved, void* stream) {
  if (!gq || !gk || !q || !k || !v || !saved) return JATTN_ERR_INVALID_ARG;
  if ((N_img > 0 && (!x_img || !w_img)) || (N_txt > 0 && (!x_txt || !w_txt))) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  if (C <= 0) return JATTN_ERR_INVALID_ARG;
  if (C % 8 != 0) return JATTN_ERR_UNSUPPORTED;  // TMA row stride: a multiple of 16 bytes
  const int64_t ycols = 3 * static_cast<int64_t>(H) * d;
  if (ycols * C >= (int64_t{1} << 31) || static_cast<int64_t>(B) * N_img * C >= (int64_t{1} << 31) ||
      static_cast<int64_t>(B) * N_txt * C >= (int64_t{1} << 31))
    return JATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk, q, k, v, saved};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JATTN_ERR_MISALIGNED;
  const size_t tb = s.elems * 2;
  const SavedLayout sl = saved_layout(s);
  const size_t xb_img = static_cast<size_t>(B) * N_img * C * 2, xb_txt = static_cast<size_t>(B) * N_txt * C * 2;
  const size_t wb = static_cast<size_t>(ycols) * C * 2, bb = static_cast<size_t>(ycols) * 4;
  const Range ins[] = {range_of(x_img, N_img ? xb_img : 0), range_of(w_img, N_img ? wb : 0),
                       range_of(b_img, N_img && b_img ? bb : 0), range_of(x_txt, N_txt ? xb_txt : 0),
                       range_of(w_txt, N_txt ? wb : 0), range_of(b_txt, N_txt && b_txt ? bb : 0),
                       range_of(gq, d * 4), range_of(gk, d * 4)};
  const Range outs[] = {range_of(q, tb), range_of(k, tb), range_of(v, tb), range_of(saved, sl.total)};
  for (size_t a = 0; a < sizeof(outs) / sizeof(outs[0]); ++a) {
    for (const Range& i : ins)
      if (overlaps(outs[a], i)) return JATTN_ERR_ALIAS;
    for (size_t b = a + 1; b < sizeof(outs) / sizeof(outs[0]); ++b)
      if (overlaps(outs[a], outs[b])) return JATTN_ERR_ALIAS;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word", cudaGetLastError());
  uint8_t* base = static_cast<uint8_t*>(saved);
  QkvLaunch a;
  a.H = H;
  a.C = C;
  a.N = s.N;
  a.d = d;
  // Stream 0: the image rows (after the caption rows); stream 1: the caption rows.
  a.M[0] = B * N_img;
  a.N_s[0] = N_img;
  a.row0[0] = N_txt;
  a.bias[0] = b_img;
  a.M[1] = B * N_txt;
  a.N_s[1] = N_txt;
  a.row0[1] = 0;
  a.bias[1] = b_txt;
  a.gq = gq;
  a.gk = gk;
  a.out[0] = q;
  a.out[1] = k;
  a.out[2] = v;
  a.hat[0] = reinterpret_cast<uint16_t*>(base + sl.qhat);
  a.hat[1] = reinterpret_cast<uint16_t*>(base + sl.khat);
  a.r[0] = reinterpret_cast<float*>(base + sl.rq);
  a.r[1] = reinterpret_cast<float*>(base + sl.rk);
  CUtensorMap maps[4];
  const jattn_bf16* xs[2] = {N_img ? x_img : x_txt, N_txt ? x_txt : x_img};
  const jattn_bf16* ws[2] = {N_img ? w_img : w_txt, N_txt ? w_txt : w_img};
  const int64_t ms[2] = {N_img ? a.M[0] : a.M[1], N_txt ? a.M[1] : a.M[0]};
  for (int i = 0; i < 2; ++i)
    if (!encode_rows_map(&maps[2 * i], xs[i], ms[i], C, 128) || !encode_rows_map(&maps[2 * i + 1], ws[i], ycols, C, 256))
      return fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  CUtensorMap out_maps[5];
  const void* outs_p[5] = {q, k, v, a.hat[0], a.hat[1]};
  for (int i = 0; i < 5; ++i)
    if (!encode_bhnd_map_rows(&out_maps[i], outs_p[i], s.BH, s.N, d, 32)) return fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  cudaError_t ce;
  {
    Timed t(JATTN_KERNEL_QKV_NORM, st);
    ce = launch_qkv_norm(maps, out_maps, a, err, st);
  }
  if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "qkv_norm launch", ce);
  return JATTN_OK;
}

extern "C" int jattn_fwd_saved(const jattn_bf16* v, int B, int H, int N_img, int N_txt, int d, jattn_bf16* out,
                               float* lse, void* saved, void* stream) {
  if (!v || !out || !lse || !saved) return JATTN_ERR_INVALID_ARG;
  Shape s;
  int rc = check_shape(B, H, N_img, N_txt, d, &s);
  if (rc != JATTN_OK) return rc;
  const void* ptrs[] = {v, out, lse, saved};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JATTN_ERR_MISALIGNED;
  const size_t tb = s.elems * 2;
  const SavedLayout sl = saved_layout(s);
  const Range ins[] = {range_of(v, tb), range_of(saved, sl.total)};
  const Range outs[] = {range_of(out, tb), range_of(lse, s.rows * 4)};
  for (size_t a = 0; a < sizeof(outs) / sizeof(outs[0]); ++a) {
    for (const Range& i : ins)
      if (overlaps(outs[a], i)) return JATTN_ERR_ALIAS;
    for (size_t b = a + 1; b < sizeof(outs) / sizeof(outs[0]); ++b)
      if (overlaps(outs[a], outs[b])) return JATTN_ERR_ALIAS;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word", cudaGetLastError());
  uint8_t* base = static_cast<uint8_t*>(saved);
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd_map(&mq, base + sl.qhat, s.BH, s.N, s.d) || !encode_bhnd_map(&mk, base + sl.khat, s.BH, s.N, s.d) ||
      !encode_bhnd_map(&mv, v, s.BH, s.N, s.d))
    return fail(JATTN_ERR_CUDA, "cuTensorMapEncodeTiled");
  AttnShape as{s.BH, s.N, s.d, 1.0f / sqrtf(static_cast<float>(s.d)), s.seg};
  cudaError_t ce;
  {
    Timed t(JATTN_KERNEL_ATTN_FWD, st);
    ce = launch_attn_fwd(mq, mk, mv, as, out, lse, err, st, reinterpret_cast<float*>(base + sl.dq),
                         reinterpret_cast<uint32_t*>(base + sl.zero_count));
  }
  if (ce != cudaSuccess) return fail(JATTN_ERR_CUDA, "attn_fwd launch", ce);
  return JATTN_OK;
}

namespace jattn {

// One thread waits on an mbarrier that nothing arrives at, through the same
// bounded wait the attention kernels use: it gives up after kWaitLimitNs and
// records DEV_ERR_WAIT_TIMEOUT, and the kernel returns.
__global__ void selftest_wait_kernel(uint32_t* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0u, &abort_flag, dev_err);
}

}  // namespace jattn

extern "C" int jattn_selftest_wait_timeout(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = dev_err_ptr();
  if (!err) return fail(JATTN_ERR_CUDA, "device error word");
  jattn::selftest_wait_kernel<<<1, 32, 0, st>>>(err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(JATTN_ERR_CUDA, "selftest_wait_kernel launch", e);
  return JATTN_OK;
}

extern "C" int jattn_last_device_error(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return JATTN_ERR_CUDA;
  uint32_t* p = dev_err_ptr();
  if (!p) return JATTN_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return JATTN_ERR_CUDA;
  if (v == 0) return JATTN_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return JATTN_ERR_CUDA;
  return (v & DEV_ERR_WAIT_TIMEOUT) ? JATTN_ERR_TIMEOUT : JATTN_ERR_CUDA;
}

extern "C" int jattn_profile_enable(int on) {
  Prof& p = prof();
  std::lock_guard<std::mutex> lock(p.mu);
  p.on = on != 0;
  return JATTN_OK;
}

extern "C" int jattn_profile_reset(void) {
  Prof& p = prof();
  std::lock_guard<std::mutex> lock(p.mu);
  int status = JATTN_OK;
  for (auto& r : p.pending) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) status = JATTN_ERR_CUDA;
    p.pool.push_back(r.a);
    p.pool.push_back(r.b);
  }
  p.pending.clear();
  for (int i = 0; i < JATTN_KERNEL_COUNT; ++i) {
    p.launches[i] = 0;
    p.ms[i] = 0;
  }
  return status;
}

extern "C" int jattn_profile_read(int kind, int* launches, double* total_ms) {
  if (kind < 0 || kind >= JATTN_KERNEL_COUNT || !launches || !total_ms) return JATTN_ERR_INVALID_ARG;
  Prof& p = prof();
  std::lock_guard<std::mutex> lock(p.mu);
  int status = JATTN_OK;
  for (auto& r : p.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      status = JATTN_ERR_CUDA;
    } else {
      p.launches[r.kind] += 1;
      p.ms[r.kind] += ms;
    }
    p.pool.push_back(r.a);
    p.pool.push_back(r.b);
  }
  p.pending.clear();
  *launches = static_cast<int>(p.launches[kind]);
  *total_ms = p.ms[kind];
  return status;
}

extern "C" int jattn_set_deterministic(int on) {
  g_deterministic.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
  return JATTN_OK;
}

extern "C" int jattn_set_sm_limit(int max_sms) {
  if (max_sms < 0) return JATTN_ERR_INVALID_ARG;
  set_sm_limit(max_sms);
  return JATTN_OK;
}

extern "C" const char* jattn_kernel_name(int kind) {
  switch (kind) {
    case JATTN_KERNEL_QK_NORM_FWD: return "qk_norm_fwd";
    case JATTN_KERNEL_ATTN_FWD: return "attn_fwd";
    case JATTN_KERNEL_BWD_PREP: return "bwd_prep";
    case JATTN_KERNEL_ATTN_BWD: return "attn_bwd";
    case JATTN_KERNEL_Q_NORM_BWD: return "q_norm_bwd";
    case JATTN_KERNEL_QKV_NORM: return "qkv_norm";
    default: return "unknown";
  }
}

extern "C" const char* jattn_status_string(int status) {
  switch (status) {
    case JATTN_OK: return "ok";
    case JATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive or overflowing size)";
    case JATTN_ERR_UNSUPPORTED:
      return "unsupported size (d must be 64 or 128; jattn_qkv_norm: C a multiple of 8)";
    case JATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case JATTN_ERR_ALIAS: return "an output buffer overlaps another buffer";
    case JATTN_ERR_CUDA: return "CUDA launch or allocation failed";
    case JATTN_ERR_TIMEOUT: return "device-side bounded wait timed out";
    case JATTN_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed no-alloc array holds";
    default: return "unknown status";
  }
}

extern "C" int jattn_version(void) { return kVersion; }

extern "C" const char* jattn_last_error_message(void) { return g_last_msg; }
