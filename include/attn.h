/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The operation ("[GPU] Deep Learning for HPC", bkkhyunn.github.io
 * hardware/pytorch_for_HPC, section "Flash Attention"): scores S = Q K^T,
 * a softmax over each row of S, then O = softmax(S) V, computed as one fused,
 * tiled kernel so the N x N score matrix never reaches device memory.  The
 * argument list follows the FlashAttention-2 Triton forward shown on
 * null-ptr.tistory.com (category "development", the `_fwd_kernel` post):
 * Q, K, V, Out, Lse, softmax_scale, batch, nheads, IS_CAUSAL.  That kernel's
 * TMP scratch has no counterpart: the running row statistics stay on chip.
 *
 * For every batch b, head h and query row i:
 *   s_ij   = scale * sum_d Q[b,h,i,d] K[b,h,j,d]       (j <= i when causal)
 *   O[b,h,i,:] = sum_j softmax_j(s_ij) V[b,h,j,:]
 *   LSE[b,h,i] = log(sum_j exp(s_ij))                  (natural log)
 * The softmax is evaluated tile by tile with a running maximum and running
 * sum (exp2-based on the device); accumulation is fp32, O is rounded once to
 * bf16 (nearest even), LSE is fp32.
 *
 * All entry points are host functions.  They allocate no device memory per
 * call, never synchronise the device except attn_last_status, and are safe
 * to call from several host threads.
 */
#ifndef ATTN_FWD_GB300_ATTN_H
#define ATTN_FWD_GB300_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned/overlapping pointer, bad size or scale */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request this library does not implement (head dim, lengths, device) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed (launch, tensor map, ...) */
  ATTN_ERR_TIMEOUT = 4      /* a kernel pipeline wait exceeded its bound and the kernel gave up */
} attn_status_t;

/*
 * attn_fwd -- enqueue the fused forward on `stream` and return.
 *
 * q, k, v : device pointers, bf16, [B, H, N, D] contiguous row-major (D
 *           innermost), 16-byte aligned.  Read only.
 * o       : device pointer, bf16, [B, H, N, D] contiguous, 16-byte aligned.
 *           Written.  Must not overlap q, k, v or lse.
 * lse     : device pointer, fp32, [B, H, N] contiguous, 4-byte aligned.
 *           Written.  Must not overlap q, k, v or o.
 * B, H, N : batch, heads, sequence length (queries = keys = N).  Any N >= 1
 *           (a ragged last tile is masked).  B, H or N equal to 0 is an empty
 *           problem: ATTN_OK, nothing launched, and the pointers (which may
 *           then be null) are not examined.
 * D       : head dimension, a multiple of 8 up to 256 (others:
 *           ATTN_ERR_UNSUPPORTED).  Below 64, 128 or 256 the computation runs
 *           at that width with zero padding (the padding is never read from or
 *           written to memory).
 * causal  : nonzero -> key j is visible to query i only when j <= i.
 * scale   : softmax scale applied to the logits, finite and > 0 (usually
 *           1/sqrt(D)).
 * stream  : a cudaStream_t (0 = legacy default stream).
 *
 * The caller owns every buffer.  Argument errors return synchronously with
 * nothing launched: ATTN_ERR_INVALID_ARG, or ATTN_ERR_UNSUPPORTED for a head
 * dimension that is not a multiple of 8 up to 256, or a device that is not
 * sm_103.  A failed
 * launch returns ATTN_ERR_CUDA.  A kernel that hits a pipeline timeout does
 * not trap: it records ATTN_ERR_TIMEOUT in a device status word that
 * attn_last_status reports; its outputs are then unspecified.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t N, int64_t D, int causal, float scale,
                       void* stream);

/*
 * attn_fwd_qk -- attn_fwd for queries and keys of different lengths.
 *
 * q, o : [B, H, Nq, D] bf16;  k, v : [B, H, Nk, D] bf16;  lse : [B, H, Nq] fp32.
 * Same pointer rules, layouts and errors as attn_fwd.  With `causal`, the mask
 * is aligned at the bottom-right corner of the Nq x Nk score matrix: key j is
 * visible to query i iff j <= i + (Nk - Nq), i.e. the queries are the last Nq
 * positions of a sequence whose first Nk positions have keys (a query block
 * appended to a key/value cache); for Nq = Nk this is attn_fwd's mask.  The
 * pages give only an IS_CAUSAL flag for the Triton forward (null-ptr.tistory.com
 * "development", the `_fwd_kernel` post); the alignment is this library's
 * reading.  Requests in which some query sees no key -- Nk = 0 with Nq > 0, or
 * causal with Nq > Nk -- return ATTN_ERR_UNSUPPORTED.  Nq = 0 (or B or H = 0)
 * is an empty problem: ATTN_OK, nothing launched.
 */
attn_status_t attn_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                          int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal,
                          float scale, void* stream);

/*
 * attn_fwd_ld -- attn_fwd_qk for tensors whose rows are padded: every row of q,
 * k, v and o starts `ld` elements after the previous one, i.e. [B, H, N, ld]
 * buffers of which the first D columns are the data.  This takes any head
 * dimension 1 <= D <= 256, including those that are not multiples of 8, which
 * contiguous rows cannot carry (the tensor copies need 16-byte row strides).
 * The FlashAttention-2 Triton forward shown on the pages takes per-tensor
 * strides for the same purpose (null-ptr.tistory.com "development", the
 * `_fwd_kernel` post: stride_qm, stride_kn, ...).
 *
 * The kernels use the first D8 = roundup8(D) columns of every row (the tensor
 * copies move whole 16-byte groups): columns D..D8-1 of q, k, v must hold
 * zeros (they add nothing then) and the same columns of o receive zeros;
 * columns D8..ld-1 are never read or written.  ld must be a multiple of 8 and
 * at least D8 (else ATTN_ERR_INVALID_ARG).  lse stays [B, H, Nq] contiguous.
 * Sizes, pointer rules, masks and errors otherwise as attn_fwd_qk, with byte
 * extents B*H*N*ld*2.
 */
attn_status_t attn_fwd_ld(const void* q, const void* k, const void* v, void* o, float* lse,
                          int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int64_t ld,
                          int causal, float scale, void* stream);

/*
 * attn_fwd_from_host -- attn_fwd_qk for inputs and outputs in host memory.
 *
 * q_host, k_host, v_host : host (or device) pointers, the layouts of attn_fwd_qk's
 *           q, k, v.  Read.
 * o_host, lse_host : host (or device) pointers, the layouts of o and lse.  Written.
 * q, k, v, o, lse : device buffers of the full sizes with attn_fwd_qk's rules
 *           (alignment, no overlap); owned by the caller, used as the staging
 *           area (q, k, v receive the inputs; o, lse hold the results).
 * Other arguments as attn_fwd_qk (Nq = Nk for the square problem).
 *
 * The work is enqueued behind everything already on `stream` and the call
 * returns; synchronising `stream` waits for all of it, host outputs included.
 * The heads are processed in up to 8 chunks: the host-to-device copy of one
 * chunk, the kernel on the previous one and the device-to-host copy of the one
 * before overlap (two copy streams and a set of events, created once per device
 * and reused; this is the GB300 counterpart of the pages' advice to keep the
 * copy engines and the SMs busy at the same time, "GPUの爆発的な性能向上",
 * ja.news.hada.io topic 14783, section "アドレス生成とTMA").  Host buffers
 * should be pinned (page-locked) for the copies to run asynchronously; pageable
 * ones give the same results with less overlap.  The host buffers must stay
 * valid until the work completes.  Results are bit-identical to attn_fwd_qk on
 * the same device inputs.  Errors: the argument checks of attn_fwd_qk run before
 * anything is enqueued (plus ATTN_ERR_INVALID_ARG for a null host pointer); a
 * failed copy or launch returns ATTN_ERR_CUDA, with earlier chunks possibly
 * enqueued; timeouts through attn_last_status.  Calls from several host threads
 * are serialised while they enqueue.
 */
attn_status_t attn_fwd_from_host(const void* q_host, const void* k_host, const void* v_host,
                                 void* o_host, float* lse_host, void* q, void* k, void* v, void* o,
                                 float* lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                                 int64_t D, int causal, float scale, void* stream);

/* Size in bytes of the device array that attn_fwd_from_host_static stages through. */
#define ATTN_STATIC_STAGING_BYTES (64u << 20)

/*
 * attn_fwd_from_host_static -- attn_fwd_from_host without caller-owned device
 * buffers, for callers that hold host data and a stream but cannot allocate
 * device memory.  The pages have no counterpart: their forward always runs on
 * tensors that already sit in device memory.
 *
 * q_host, k_host, v_host, o_host, lse_host : as attn_fwd_from_host (host, or
 *           device, pointers in attn_fwd_qk's layouts; the first three read,
 *           the last two written).  Other arguments as attn_fwd_qk.
 *
 * Staging: Q, K, V, O and LSE are placed one after another, each on a 256-byte
 * boundary, in one device array of ATTN_STATIC_STAGING_BYTES (64 MiB) that is
 * part of this library's device code.  No device memory is allocated or freed
 * by the call.  The array exists on every device that has loaded the library's
 * device code, is shared by every call on that device and keeps the last
 * call's inputs and results; nothing in it needs to start at zero (each call
 * writes, before its kernel, every byte that kernel reads).
 *
 * Ordering: three host-to-device copies, the kernel and two device-to-host
 * copies are enqueued on `stream` behind the work already there, and the call
 * returns; synchronising `stream` waits for all of it.  Calls whose work can
 * overlap on the device (on different streams, or from several host threads
 * without ordering) race on the shared array and give undefined results; order
 * them on one stream.  The first call on a device looks up the array's device
 * address (and may load the library's device code); make that first call before
 * any stream capture begins.  Host buffers should be pinned for the copies to
 * be asynchronous and must stay valid until the work completes.
 *
 * Errors: attn_fwd_qk's argument rules (ATTN_ERR_INVALID_ARG for a null host
 * pointer in a non-empty problem); ATTN_ERR_UNSUPPORTED when the staged bytes
 * (2 B*H*(2 Nq + 2 Nk) D plus 4 B*H*Nq, with each part rounded up to 256) exceed
 * ATTN_STATIC_STAGING_BYTES -- use attn_fwd_from_host with buffers of one's own
 * then; ATTN_ERR_CUDA for a failed copy, launch or address lookup (work enqueued
 * before the failure stays enqueued); timeouts through attn_last_status.
 * Results are bit-identical to attn_fwd_qk on the same inputs.
 */
attn_status_t attn_fwd_from_host_static(const void* q_host, const void* k_host, const void* v_host,
                                        void* o_host, float* lse_host, int64_t B, int64_t H,
                                        int64_t Nq, int64_t Nk, int64_t D, int causal, float scale,
                                        void* stream);

/*
 * attn_bwd -- enqueue the backward of attn_fwd on `stream`: the gradients of
 * sum(dO * O) with respect to Q, K and V.
 *
 * q, k, v : the forward's inputs; o, lse : its outputs (bf16 [B,H,N,D], fp32
 * [B,H,N]); dout : the upstream gradient dO, bf16 [B,H,N,D].  All read only.
 * dq, dk, dv : bf16 [B,H,N,D], written.  delta : fp32 [B,H,N], written:
 * D_i = sum_d dO_id O_id, which the chain rule through the softmax needs
 * (ds_ij = p_ij (dp_ij - D_i)); returned so that no scratch memory is needed.
 * Outputs must not overlap each other or any input.  Same sizes, alignment
 * (16 bytes for bf16 tensors, 4 for fp32) and scale rules as attn_fwd; head
 * dims a multiple of 8 up to 256, like attn_fwd (ATTN_ERR_UNSUPPORTED
 * otherwise; 136..256 run on the D = 256 kernels, zero-padded).  The pages
 * call the backward an order of magnitude harder than the forward
 * ("GPUの爆発的な性能向上", ja.news.hada.io topic 14783) without a formula;
 * the math is the chain rule written out in oracle/attn_oracle_bwd.c and the
 * kernels' header comment.  Two kernels are enqueued (dQ and D first, then dK
 * and dV); errors as attn_fwd, timeouts through attn_last_status.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, float* delta, int64_t B,
                       int64_t H, int64_t N, int64_t D, int causal, float scale, void* stream);

/*
 * attn_bwd_qk -- attn_bwd for queries and keys of different lengths, the
 * backward of attn_fwd_qk: q, o, dout, dq [B,H,Nq,D]; k, v, dk, dv [B,H,Nk,D];
 * lse, delta [B,H,Nq].  Causal alignment and the unsupported cases (some query
 * without a key; also Nq = 0 with Nk > 0) as attn_fwd_qk.
 */
attn_status_t attn_bwd_qk(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          float* delta, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                          int causal, float scale, void* stream);

/*
 * attn_bwd_ld -- attn_bwd_qk for row-padded tensors: q, k, v, o, dout, dq, dk,
 * dv all with rows `ld` elements apart, any head dimension 1 <= D <= 256; lse
 * and delta contiguous [B, H, Nq].  As for attn_fwd_ld, the first roundup8(D)
 * columns are used: columns D.. of that group must be zero in the inputs (as
 * attn_fwd_ld leaves them in o) and receive zeros in dq, dk, dv; columns
 * beyond it are never read or written.  Errors as attn_fwd_ld.
 */
attn_status_t attn_bwd_ld(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          float* delta, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                          int64_t ld, int causal, float scale, void* stream);

/*
 * attn_last_status -- report and clear the status word of the current device:
 * ATTN_OK, or ATTN_ERR_TIMEOUT if some kernel of this library gave up on a
 * pipeline wait since the word was last cleared; ATTN_ERR_CUDA if the status
 * read or the synchronisation failed.
 *
 * The read is enqueued on `stream` (behind the work already there) as one
 * atomic read-and-clear on the device, and the call then synchronises
 * `stream`.  The word is device-wide, not per stream: a timeout of a kernel on
 * any stream is reported once, to the first call that reads the word after the
 * kernel recorded it, and is never lost when several streams or threads call
 * this at the same time.
 */
attn_status_t attn_last_status(void* stream);

/*
 * attn_set_tuning -- process-wide overrides of the launcher's own choices, for
 * tuning and testing.  0 in an argument restores the automatic choice.
 *
 * unit              : how query tiles form work units: 1 = one tile (of 128
 *                     rows) per unit; 2 = two tiles of one head sharing every
 *                     K/V tile; 3 = key split, one tile whose key tiles are
 *                     shared out between the CTA's two softmax warpgroups and
 *                     merged at the end (head dims up to 64; above, 3 means 1);
 *                     4 = one tile per unit on the short-unit kernel, two CTAs
 *                     per SM each with half of its resources (head dims up to
 *                     64, where it ignores `grid`; above, 4 means 1).
 *                     Head dims above 128 always run one tile per unit.
 * grid              : 1 = one CTA per unit; 2 = persistent (one CTA per SM,
 *                     each walking many units).  Head dims above 128 always
 *                     run one CTA per unit.
 * pipe_chunks       : 1..32, chunks of heads in attn_fwd_from_host.
 * wait_limit_cycles : bound of every pipeline wait in SM cycles (default 2^32,
 *                     about 2 s); a lower bound turns a stalled pipeline into
 *                     ATTN_ERR_TIMEOUT sooner.
 *
 * An out-of-range value returns ATTN_ERR_INVALID_ARG and changes nothing.
 * Calls that start after this returns use the new values; any thread may call it.
 * The results of attn_fwd do not depend on these choices beyond fp32 rounding
 * order (each setting is tested against the same oracle).
 */
attn_status_t attn_set_tuning(int unit, int grid, int pipe_chunks, int64_t wait_limit_cycles);

/*
 * attn_fwd_kernel_name -- the kernel instance attn_fwd_qk would launch for a
 * problem of these sizes on the current device with the current tuning, e.g.
 * "attn_fwd_sm103<128,full,persistent,2 tiles/unit>" or
 * "attn_fwd_short_sm103<causal>" (for diagnostics, benchmarks and profiles).
 * The string lives in thread-local storage until this thread's next call.
 * NULL for sizes attn_fwd_qk would reject (non-positive, D > 256, too large)
 * or when the device cannot be prepared.
 */
const char* attn_fwd_kernel_name(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * attn_fwd_flops -- algorithmic FLOPs of one attn_fwd call:
 * 4 * B * H * N^2 * D, halved when causal (exp and softmax not counted).
 */
double attn_fwd_flops(int64_t B, int64_t H, int64_t N, int64_t D, int causal);

/*
 * attn_fwd_qk_flops -- algorithmic FLOPs of one attn_fwd_qk call: 4 * B * H * D
 * times the visible (query, key) pairs, Nq * Nk, or Nq * (Nk - Nq) + Nq^2 / 2
 * when causal (equal to attn_fwd_flops when Nq = Nk).
 */
double attn_fwd_qk_flops(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal);

/*
 * attn_bwd_qk_flops -- algorithmic FLOPs of one attn_bwd_qk call: the five
 * products S = Q K^T, dP = dO V^T, dV, dK and dQ, i.e. 2.5 times
 * attn_fwd_qk_flops (the kernels recompute S and dP once more).
 */
double attn_bwd_qk_flops(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal);

/*
 * attn_based_fwd -- enqueue the Based linear-attention forward on `stream`.
 *
 * The pages name this kernel ("GPU의 폭발적인 성능 향상", news.hada.io topic
 * 14783, section "ThunderKittens": a Based linear-attention forward, 215
 * TFLOP/s on an H100) without a formula; the definition is the published
 * Based layer (Arora et al., 2024): causal linear attention with the
 * second-order Taylor kernel of exp.  For every batch b, head h and row i:
 *   s_ij = scale * sum_f Q[b,h,i,f] K[b,h,j,f]            (j <= i)
 *   a_ij = 1 + s_ij + s_ij^2 / 2
 *   Z[b,h,i] = sum_{j<=i} a_ij
 *   Y[b,h,i,:] = sum_{j<=i} a_ij V[b,h,j,:] / Z[b,h,i]
 * evaluated chunk by chunk (128 tokens) with a running state of the feature
 * map phi(k) v^T; accumulation is fp32, the weights, features and state enter
 * the tensor-core products in bf16, Y is rounded once to bf16, Z is fp32.
 *
 * q, k : device, bf16 [B, H, N, F] contiguous (F innermost), 16-byte aligned.
 * v    : device, bf16 [B, H, N, D] contiguous, 16-byte aligned.
 * y    : device, bf16 [B, H, N, D], written; z : device, fp32 [B, H, N], written.
 *        Neither may overlap any input or the other.
 * F    : feature dimension, 8 or 16 (others ATTN_ERR_UNSUPPORTED; Based uses 16).
 * D    : value head dimension, a multiple of 8 up to 64 (others ATTN_ERR_UNSUPPORTED).
 * N    : any length >= 1 (a ragged last chunk is zero padded); B, H or N = 0 is
 *        an empty problem (ATTN_OK, nothing launched, pointers not examined).
 * scale: finite and > 0 (usually 1/sqrt(F)).
 * Ownership, asynchrony and errors as attn_fwd (timeouts through attn_last_status).
 */
attn_status_t attn_based_fwd(const void* q, const void* k, const void* v, void* y, float* z, int64_t B,
                             int64_t H, int64_t N, int64_t F, int64_t D, float scale, void* stream);

/*
 * attn_based_fwd_flops -- FLOPs of the linear (running-state) form of one
 * attn_based_fwd call: per token 4 * Fs * (D + 1) (state update and readout),
 * Fs = 1 + F + F (F + 1) / 2 features of the symmetric Taylor map.
 */
double attn_based_fwd_flops(int64_t B, int64_t H, int64_t N, int64_t F, int64_t D);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_GB300_ATTN_H */
