/*
 * jattn.h — C ABI of libjattn: MM-DiT joint self-attention with QK-RMSNorm,
 * forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (re-diffusion README — "architecture flowchart": inside each
 * DiT layer the caption-stream and image-stream Q/K/V are concatenated as
 * [c; x] and one multi-head self-attention runs over the joint sequence;
 * "design notes" table, row "QK norm": RMSNorm on Q and on K; "attention fix"
 * section: scaled-dot-product attention over the same [B, H, N, d] Q/K/V
 * layout, without materialising the B x H x N x N score matrix):
 *
 *   r(x)   = (mean_c x_c^2 + eps)^(-1/2),  eps = 1e-6          (per row)
 *   q_hat  = bf16(gq * q * r(q)),  k_hat = bf16(gk * k * r(k))
 *   S      = q_hat k_hat^T / sqrt(d)                           (per b, h)
 *   LSE_i  = ln sum_j exp(S_ij),   O = exp(S - LSE) V
 *
 * Layout.  q, k, v, out, dout, dq, dk, dv are contiguous row-major
 * [B, H, N, d] bfloat16 (stored as uint16_t bit patterns), N = N_txt + N_img
 * with the N_txt caption rows first, then the N_img image rows.  lse is
 * [B, H, N] float32, natural log.  gq, gk, dgq, dgk are [d] float32, one gain
 * vector shared by all heads.  No mask, dropout or causality: N_txt and N_img
 * only define N and the row order.
 *
 * Pointers.  Every array pointer is a DEVICE pointer (CUDA global memory),
 * 16-byte aligned.  `stream` is a cudaStream_t passed as void* (NULL = the
 * legacy default stream); all work is enqueued on it and the call returns
 * without synchronising.  The caller owns every buffer.  The library
 * allocates its scratch memory per call, stream-ordered on `stream`
 * (cudaMallocAsync / cudaFreeAsync), and keeps no state between calls.
 *
 * Errors.  Every entry point returns a jattn_status and never aborts or
 * prints.  Arguments are validated before anything is enqueued; a non-OK
 * status from validation means nothing ran.  JATTN_ERR_CUDA reports a failed
 * launch or allocation.  The kernels' internal waits are bounded: a wait
 * that gives up ends the kernel early and jattn_last_device_error() then
 * reports it (it synchronises `stream`).  Asynchronous faults surface, as
 * usual in CUDA, at the caller's next synchronisation.
 */
#ifndef JATTN_H
#define JATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t jattn_bf16; /* bfloat16 bit pattern */

typedef enum {
  JATTN_OK = 0,
  JATTN_ERR_INVALID_ARG = 1, /* null pointer, B/H/d <= 0, N_img/N_txt < 0, N < 1, size overflow */
  JATTN_ERR_UNSUPPORTED = 2, /* d not in {64, 128}; jattn_qkv_norm: C not a multiple of 8 */
  JATTN_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  JATTN_ERR_ALIAS = 4,       /* an output buffer overlaps an input or another output */
  JATTN_ERR_CUDA = 5,        /* a CUDA launch or allocation failed */
  JATTN_ERR_TIMEOUT = 6,     /* a device-side bounded wait gave up (reported by jattn_last_device_error) */
  JATTN_ERR_SCRATCH_LIMIT = 7 /* jattn_fwd_noalloc: the problem needs more scratch than its fixed array holds */
} jattn_status;

/*
 * Forward.  Computes out = softmax(q_hat k_hat^T / sqrt(d)) v and lse (the
 * natural-log row log-sum-exp of the scaled scores) for every (b, h).
 *   q, k, v : [B, H, N, d] bf16, read only.
 *   gq, gk  : [d] float32 RMSNorm gains for q and k, read only.
 *   B, H    : batch size and heads (>= 1).
 *   N_img   : image-token rows, N_txt: caption-token rows (>= 0 each,
 *             N = N_img + N_txt >= 1).
 *   d       : head dimension, 64 or 128.
 *   out     : [B, H, N, d] bf16, overwritten.
 *   lse     : [B, H, N] float32, overwritten.
 * Limits: B*H*N*d < 2^31.
 */
int jattn_fwd(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
              int B, int H, int N_img, int N_txt, int d, jattn_bf16* out, float* lse, void* stream);

/*
 * Backward.  Given the forward's inputs, its outputs (out, lse) and the
 * upstream gradient dout, computes the gradients of L = sum(dout * out):
 *   dq, dk, dv : [B, H, N, d] bf16, overwritten.
 *   dgq, dgk   : [d] float32, overwritten (summed over all b, h, n).
 * The bf16 rounding of q_hat/k_hat is treated as the identity.  The
 * normalised q_hat/k_hat are recomputed from q, k (nothing is cached from
 * the forward call; jattn_fwd_train / jattn_bwd_train below keep them).  dk, dv and dgk are always summed in a fixed order and
 * repeat bit for bit.  dq is accumulated in float32 across key tiles: by
 * default with reduce-adds in arrival order, so that dq and dgq (a sum over
 * dq's accumulator) may differ in the last bits between runs; with
 * jattn_set_deterministic(1), in a fixed order, so that all five gradients
 * repeat bit for bit (on the same GPU model and CTA cap).
 */
int jattn_bwd(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
              const jattn_bf16* out, const float* lse, const jattn_bf16* dout, jattn_bf16* dq, jattn_bf16* dk,
              jattn_bf16* dv, float* dgq, float* dgk, int B, int H, int N_img, int N_txt, int d, void* stream);

/*
 * Packed variable-length forward and backward: one call over sequences of
 * different lengths, each attending only within itself.  This is for batches
 * that mix resolutions, for example images from different aspect-ratio buckets
 * with their captions.  The re-diffusion README's training-data paragraph
 * describes the aspect-bucketed export, and its roadmap lists multi-resolution
 * training.
 *   Layout: [H, T, d] bf16 with T = cu_seqlens[n_seqs].  Head h holds T rows,
 *           and sequence s is rows cu_seqlens[s] .. cu_seqlens[s+1]-1 of every
 *           head.  This is the [B, H, N, d] layout with B = 1 and the
 *           sequences concatenated along N; each sequence lists its caption
 *           rows and image rows in any order.
 *   cu_seqlens: HOST array of n_seqs + 1 ints, cu_seqlens[0] = 0, strictly
 *           increasing (every sequence has at least one row); read during
 *           the call only.
 *   n_seqs: 1 .. JATTN_MAX_SEQS.
 *   lse   : [H, T] float32.
 *   The other arguments and every status are those of jattn_fwd / jattn_bwd.
 *   An invalid cu_seqlens gives JATTN_ERR_INVALID_ARG; n_seqs above
 *   JATTN_MAX_SEQS gives JATTN_ERR_UNSUPPORTED.  H*T*d < 2^31.
 * dgq and dgk sum over every sequence, head and row.
 */
#define JATTN_MAX_SEQS 256
int jattn_fwd_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
                     const int* cu_seqlens, int n_seqs, int H, int d, jattn_bf16* out, float* lse, void* stream);
int jattn_bwd_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
                     const jattn_bf16* out, const float* lse, const jattn_bf16* dout, jattn_bf16* dq, jattn_bf16* dk,
                     jattn_bf16* dv, float* dgq, float* dgk, const int* cu_seqlens, int n_seqs, int H, int d,
                     void* stream);

/*
 * Training pair: a forward that keeps the normalised q_hat, k_hat and the
 * rows' 1/rms r(q), r(k) in a caller buffer `saved`, and a backward that
 * reads them there instead of recomputing them (the autograd practice of
 * saving an op's activations for its backward).  Results are those of
 * jattn_fwd / jattn_bwd with the same arguments, bit for bit where those
 * repeat bit for bit.
 *   saved : DEVICE buffer of jattn_saved_bytes(...) bytes (16-byte aligned),
 *           written by the forward and used by the backward, which must be
 *           given the same q, k, gq, gk and shape; its layout is private.
 *           It may not overlap any other argument.  It also holds the
 *           backward's fp32 dQ accumulator, which the forward zeroes while it
 *           runs (with HBM bandwidth its attention kernel leaves idle) so
 *           that the backward need not; a backward that finds it not zeroed
 *           by a forward since the last backward (a second backward on the
 *           same buffer, or a buffer no forward has filled) zeroes it itself,
 *           so any number of backward calls per forward stay correct.
 *           Size: 2 B*H*N*d*2 + B*H*N*d*4 + 2 B*H*N*4 bytes plus alignment.
 * jattn_saved_bytes returns 0 for a shape the calls would reject.  The other
 * arguments and every status are those of jattn_fwd / jattn_bwd (and of
 * their varlen forms); a null `saved` gives JATTN_ERR_INVALID_ARG.
 */
size_t jattn_saved_bytes(int B, int H, int N_img, int N_txt, int d);
size_t jattn_saved_bytes_varlen(const int* cu_seqlens, int n_seqs, int H, int d);
int jattn_fwd_train(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
                    int B, int H, int N_img, int N_txt, int d, jattn_bf16* out, float* lse, void* saved,
                    void* stream);
int jattn_bwd_train(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
                    const jattn_bf16* out, const float* lse, const jattn_bf16* dout, void* saved,
                    jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq, float* dgk, int B, int H, int N_img,
                    int N_txt, int d, void* stream);
int jattn_fwd_train_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                           const float* gk, const int* cu_seqlens, int n_seqs, int H, int d, jattn_bf16* out,
                           float* lse, void* saved, void* stream);
int jattn_bwd_train_varlen(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq,
                           const float* gk, const jattn_bf16* out, const float* lse, const jattn_bf16* dout,
                           void* saved, jattn_bf16* dq, jattn_bf16* dk, jattn_bf16* dv, float* dgq, float* dgk,
                           const int* cu_seqlens, int n_seqs, int H, int d, void* stream);

/*
 * QKV projection with QK-RMSNorm in its epilogue (re-diffusion README,
 * "architecture flowchart": each stream's tokens are projected to Q, K, V
 * with that stream's own weights, the streams are concatenated along the
 * token axis and Q, K are RMS-normalised before the attention; "design notes"
 * table, row "QK norm").  One call computes, for both streams,
 *
 *   Y = bf16(X W^T + b)           fp32 accumulation, bias added in fp32,
 *                                 then one rounding to bf16
 *   q, k, v = the Y columns of each head, written into the joint layout
 *   q_hat, k_hat, 1/rms of every q and k row, as jattn_fwd_train keeps them
 *
 * so that jattn_fwd_saved can start the attention from q_hat / k_hat and
 * jattn_bwd_train can run the backward, with no normalisation pass of their
 * own.  Results are those of projecting, then calling jattn_fwd_train on the
 * projected q, k, v: q_hat, k_hat bit for bit (both correctly rounded), the
 * 1/rms values to fp32 rounding.
 *   x_img  : [B, N_img, C] bf16 image-stream tokens (rows N_txt .. N - 1)
 *   w_img  : [3 H d, C] bf16 image-stream weight, row-major like a linear
 *            layer's weight: rows h d .. h d + d - 1 give head h of q, rows
 *            H d + h d .. of k, rows 2 H d + h d .. of v
 *   b_img  : [3 H d] float32 bias, or NULL for none
 *   x_txt, w_txt, b_txt : the caption stream's, likewise (rows 0 .. N_txt - 1);
 *            a stream with no rows may pass NULL tokens and weight
 *   gq, gk : [d] float32 gains
 *   C      : model width, a multiple of 8 (else JATTN_ERR_UNSUPPORTED)
 *   q, k, v: [B, H, N, d] outputs (the layout above)
 *   saved  : jattn_saved_bytes(B, H, N_img, N_txt, d) bytes, written as a
 *            training forward writes it
 * Every pointer is a 16-byte aligned DEVICE pointer; outputs may not overlap
 * inputs or each other (JATTN_ERR_ALIAS).  The [B, H, N, d] layout only (no
 * varlen form).  Sizes: 3 H d C, B N_img C and B N_txt C below 2^31.
 *
 * jattn_fwd_saved is the attention forward of a training pair whose q_hat /
 * k_hat are already in `saved` (from jattn_qkv_norm, or from jattn_fwd_train
 * with the same shape): out and lse as jattn_fwd computes them from the q, k
 * that gave those q_hat / k_hat.  It launches the attention kernel only (which
 * also zeroes the buffer's dQ accumulator, as jattn_fwd_train does).
 */
int jattn_qkv_norm(const jattn_bf16* x_img, const jattn_bf16* w_img, const float* b_img, const jattn_bf16* x_txt,
                   const jattn_bf16* w_txt, const float* b_txt, const float* gq, const float* gk, int B, int H,
                   int N_img, int N_txt, int d, int C, jattn_bf16* q, jattn_bf16* k, jattn_bf16* v, void* saved,
                   void* stream);
int jattn_fwd_saved(const jattn_bf16* v, int B, int H, int N_img, int N_txt, int d, jattn_bf16* out, float* lse,
                    void* saved, void* stream);

/*
 * Forward without any device allocation.  (No counterpart on the pages: an
 * integration entry point.)  Same arguments, layout and results as jattn_fwd,
 * but the scratch it needs (the normalised q_hat and k_hat, 2 * 2 * B*H*N*d
 * bytes, each part 256-byte aligned) lives in one fixed file-scope device
 * array of JATTN_NOALLOC_SCRATCH_BYTES (64 MiB) instead of a per-call
 * cudaMallocAsync.  It calls no cudaMalloc / cudaFree / allocating library
 * routine.
 *
 * Who needs it: callers that cannot let a library allocate device memory, such
 * as a serving process that reserves nearly all of HBM for its own pool up
 * front (a library allocation would then fail mid-step), or a launch sequence
 * that must never block on or recover from an allocator call.
 *
 * Rules:
 *  - Problems needing more than the array (B*H*N*d > 16,777,216 = 2^24 at these
 *    alignments, e.g. the 768 px / d = 128 workload) return
 *    JATTN_ERR_SCRATCH_LIMIT before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture.
 *  - Every call, on any stream, shares the one array, which keeps the last
 *    call's contents.  Nothing in it needs clearing (the norm kernel writes
 *    every element it is later read back from), but calls that overlap on the
 *    GPU (for example on two streams at once) race on it: serialise them.
 *  - Every GPU that loads this library holds the array until the process
 *    exits.
 */
#define JATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int jattn_fwd_noalloc(const jattn_bf16* q, const jattn_bf16* k, const jattn_bf16* v, const float* gq, const float* gk,
                      int B, int H, int N_img, int N_txt, int d, jattn_bf16* out, float* lse, void* stream);

/*
 * Synchronises `stream` and returns JATTN_ERR_TIMEOUT if any kernel launched
 * by this library on the current device since the previous call gave up a
 * bounded wait, JATTN_ERR_CUDA if the synchronisation itself failed, else
 * JATTN_OK.  Clears the recorded device error.
 */
int jattn_last_device_error(void* stream);

/*
 * Self-test of the bounded-wait path (no counterpart on the pages: failure
 * detection).  Enqueues on `stream` a one-thread kernel that waits on an
 * mbarrier nothing ever arrives at.  The wait is the one every attention
 * kernel uses: it gives up after its limit (about 1 s), records the device
 * error and returns, so the context stays usable.  The next
 * jattn_last_device_error(stream) then returns JATTN_ERR_TIMEOUT.  Returns
 * JATTN_OK, or JATTN_ERR_CUDA if the launch failed.
 */
int jattn_selftest_wait_timeout(void* stream);

/*
 * Kernel timing (off by default; no counterpart on the pages: measurement
 * support).  While enabled, every kernel launch made by the library
 * on the calling thread's device is bracketed by two CUDA events recorded on
 * the caller's stream.  jattn_profile_read synchronises on those events and
 * adds, for one kernel kind, the number of launches and their summed
 * event-to-event milliseconds since the last jattn_profile_reset.
 */
typedef enum {
  JATTN_KERNEL_QK_NORM_FWD = 0,  /* RMSNorm of q and k (forward) */
  JATTN_KERNEL_ATTN_FWD = 1,     /* tensor-core attention forward */
  JATTN_KERNEL_BWD_PREP = 2,     /* norm recompute + rowsum(dO*O) + dq accumulator clear */
  JATTN_KERNEL_ATTN_BWD = 3,     /* tensor-core attention backward (+ K-norm backward) */
  JATTN_KERNEL_Q_NORM_BWD = 4,   /* Q-norm backward from the dq accumulator, and the gain gradients */
  JATTN_KERNEL_QKV_NORM = 5,     /* QKV projection of both streams with the QK-RMSNorm epilogue */
  JATTN_KERNEL_COUNT = 6
} jattn_kernel_kind;

int jattn_profile_enable(int on);
int jattn_profile_reset(void);
int jattn_profile_read(int kind, int* launches, double* total_ms);
const char* jattn_kernel_name(int kind);

/*
 * Deterministic backward (off by default; no counterpart on the pages).
 * With on != 0, later jattn_bwd / jattn_bwd_varlen calls from any thread add
 * the key tiles' contributions to each query tile's float32 dq accumulator in
 * a fixed order (the first is stored, each later one is added only after the
 * one before it has completed), so that dq and dgq repeat bit for bit.  The
 * order costs time: contributions wait on one another across CTAs (bounded
 * waits: a stalled wait ends the kernel and jattn_last_device_error reports
 * JATTN_ERR_TIMEOUT).  Every CTA of the launch must be able to run at the
 * same time as the others (see jattn_set_sm_limit).  Returns JATTN_OK.
 */
int jattn_set_deterministic(int on);

/*
 * Caps the number of CTAs the persistent attention kernels launch, and so the
 * SMs they occupy, at max_sms (0 = every SM of the device, the default); for
 * sharing the GPU with concurrent work, and for exercising the kernels' work
 * schedules on small problems.  It applies to later calls from any thread.
 * In the deterministic mode the backward picks its dQ order from it.  A cap
 * above the SMs the process may use (for example under an MPS thread limit)
 * can make the deterministic backward's cross-CTA waits give up
 * (JATTN_ERR_TIMEOUT).  Returns JATTN_ERR_INVALID_ARG for a negative cap.
 * (No counterpart on the pages.)
 */
int jattn_set_sm_limit(int max_sms);

/* Static description of a status code (never NULL). */
const char* jattn_status_string(int status);

/* Human-readable detail of the last failing CUDA call or driver step seen
 * by an entry point on the calling thread (never NULL). */
const char* jattn_last_error_message(void);

/* Library version, major*10000 + minor*100 + patch. */
int jattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* JATTN_H */
