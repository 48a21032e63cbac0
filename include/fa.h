/*
 * fa.h -- C ABI of the exact-attention library (libfa.so), GB300 / sm_103a.
 *
 * The library computes exact scaled dot-product attention
 *     O = softmax(scale * Q K^T) V
 * tile by tile with the online-softmax recurrence, never materialising the
 * N x N score or probability matrix, and saves the per-row log-sum-exp
 *     L_i = m_i + ln l_i
 * for the backward pass, which recomputes the probabilities from Q, K and L.
 *
 * Sources of each operation (page title and section):
 *   - problem statement, S = QK^T/sqrt(d), P = softmax(S), O = PV:
 *     "research-attention" tutorial, section 01 equations;
 *   - running state (m, l, u) and its merge with alpha = exp(m - m'):
 *     same tutorial, section 02;
 *   - saved statistic L = m + log(l) and rebuilding P = exp(s - L):
 *     same tutorial, section 04;
 *   - tiled forward loop and the final division O_i / l_i:
 *     "Flash Attention 原理与实现", section "Forward 的 Tiling 策略";
 *   - backward by recomputation, dV = P^T dO, dP = dO V^T, dS from the
 *     softmax gradient, dQ = dS K, dK = dS^T Q: same blog, section
 *     "Backward 的 Tiling 策略"; dQ is gathered across key blocks by local
 *     accumulation (one of the two ways item 3 of "实际实现中的注意事项"
 *     names) rather than by atomic adds.
 *
 * Conventions shared by every entry point
 *   Layout     Q, K, V, O, dO, dQ, dK, dV are contiguous [B][H][N][d] arrays
 *              of the entry point's element type (bf16 for fa_fwd/fa_bwd,
 *              float for the _f32 twins); lse is a contiguous [B][H][N] float
 *              array holding the natural-log log-sum-exp of the scaled scores.
 *              Q and K/V share the sequence length N.
 *   Mask       causal != 0 lets query i see keys j <= i; causal == 0 lets
 *              every query see all N keys.
 *   Scale      any finite float; callers usually pass 1/sqrt(d). dQ and dK
 *              are the true derivatives and therefore carry the factor scale.
 *   Memory     every pointer is a DEVICE pointer owned by the caller. The
 *              library never allocates, frees or synchronises; all work is
 *              enqueued on `stream` (0 = legacy default stream) and returns
 *              immediately.
 *   Errors     argument errors return a non-zero fa_status and launch
 *              nothing. FA_ERR_LAUNCH reports a CUDA launch error (the CUDA
 *              error is left for cudaGetLastError-style inspection via
 *              fa_last_cuda_error). A kernel that gives up on an internal
 *              wait (it never traps) records FA_ERR_TIMEOUT in a device
 *              status word read by fa_device_status.
 *   Supported  bf16 and f16: d in {64, 96, 128} (the forward also takes
 *              d = 256; the backward returns FA_ERR_UNSUPPORTED for it),
 *              N >= 1 (ragged tails are masked), every pointer 16-byte
 *              aligned.
 *              f32: 1 <= d <= 128, N >= 1, every pointer 4-byte aligned.
 *              B, H >= 1; B*H*N*d must be below 2^40 elements; d above
 *              256 (128 for f32) is FA_ERR_SHAPE.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,        /* a required pointer is NULL */
  FA_ERR_SHAPE = 2,       /* B, H, N or d out of range, or sizes overflow */
  FA_ERR_UNSUPPORTED = 3, /* valid shape this build has no kernel for */
  FA_ERR_ALIGN = 4,       /* pointer not aligned as required */
  FA_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than fa_bwd_workspace_size */
  FA_ERR_LAUNCH = 6,      /* a CUDA launch or tensor-map call failed */
  FA_ERR_TIMEOUT = 7,     /* a kernel gave up waiting on a pipeline barrier */
  FA_ERR_ARCH = 8,        /* current device is not sm_103 */
  FA_ERR_ARG = 9,         /* other invalid argument (non-finite scale, dtype) */
  FA_ERR_CHECK = 10       /* only in a library built with FA_CHECKED: a kernel's
                             own check rejected a TMA coordinate or address, a
                             bulk-copy address or size, or a TMEM address, and
                             skipped that access; the results are not valid */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1, FA_F16 = 2 } fa_dtype;

/*
 * Forward, bf16 in / bf16 out.
 *   q, k, v  [B][H][N][d] bf16, read only.
 *   o        [B][H][N][d] bf16, written: O = softmax(scale*QK^T) V.
 *   lse      [B][H][N] float, written: L_i = ln sum_j exp(scale q_i.k_j).
 * Arithmetic: bf16 operands, fp32 accumulation; probabilities are rounded to
 * bf16 before the P.V product.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int N, int d, float scale, int causal,
           fa_stream_t stream);

/*
 * Backward, bf16 in / bf16 out, for upstream gradient dO.
 *   q, k, v, o, dO   [B][H][N][d] bf16, read only (o as written by fa_fwd).
 *   lse              [B][H][N] float from fa_fwd, read only.
 *   dq, dk, dv       [B][H][N][d] bf16, written.
 *   workspace        device scratch of at least
 *                    fa_bwd_workspace_size(B, H, N, d, FA_BF16) bytes, 256-byte
 *                    aligned, owned by the caller; holds the per-row terms
 *                    -L*log2(e) and D_i = sum_c dO_ic O_ic, padded to whole
 *                    128-row tiles (8 bytes per padded row). Its contents on
 *                    entry are ignored.
 * Three kernels run on `stream`: the row terms; a pass over key blocks that
 * forms dK and dV; a pass over query tiles that forms dQ. Both passes
 * recompute S and dP, so no partial sums go through global memory and the
 * result does not depend on scheduling.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o,
           const float *lse, const void *dO, void *dq, void *dk, void *dv,
           int B, int H, int N, int d, float scale, int causal,
           void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* Forward and backward with IEEE half (f16) tensors: same kernels, arguments,
 * layout, workspace and errors as fa_fwd / fa_bwd with f16 in place of bf16;
 * P and dS are rounded to f16 before their products. fp16 inputs are the
 * blog's own setting (its pitfalls items on FP16 training and overflow). */
int fa_fwd_f16(const void *q, const void *k, const void *v, void *o, float *lse,
               int B, int H, int N, int d, float scale, int causal,
               fa_stream_t stream);
int fa_bwd_f16(const void *q, const void *k, const void *v, const void *o,
               const float *lse, const void *dO, void *dq, void *dk, void *dv,
               int B, int H, int N, int d, float scale, int causal,
               void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Forward and backward with Nq query rows against Nk key/value rows per head
 * (decode and chunked-prefill shapes; the blog's setting is a 64K-token
 * inference service, and the tutorial's section 06 lists query and key
 * lengths as separate parameters). Q, O, dO, dQ are [B][H][Nq][d]; K, V, dK,
 * dV are [B][H][Nk][d]; lse is [B][H][Nq]. dtype is FA_BF16 or FA_F16
 * (FA_F32 returns FA_ERR_UNSUPPORTED). With causal != 0 the mask is aligned
 * at the bottom right: query i sees key j iff j <= i + (Nk - Nq), so the
 * queries act as the last Nq rows of the square problem; that requires
 * Nk >= Nq (else FA_ERR_SHAPE). The backward's workspace is
 * fa_bwd_workspace_size(B, H, Nq, d, dtype) bytes. Everything else is as for
 * fa_fwd / fa_bwd; fa_fwd(...) is fa_fwd_kv(..., N, N, ..., FA_BF16, ...).
 */
int fa_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int H, int Nq, int Nk, int d, float scale, int causal,
              int dtype, fa_stream_t stream);
int fa_bwd_kv(const void *q, const void *k, const void *v, const void *o,
              const float *lse, const void *dO, void *dq, void *dk, void *dv,
              int B, int H, int Nq, int Nk, int d, float scale, int causal,
              int dtype, void *workspace, size_t workspace_bytes,
              fa_stream_t stream);

/*
 * Forward and backward with dropout on the attention probabilities. The
 * tutorial page "research-attention" keeps dropout out of its plain
 * definition (section 01) and asks that its probability and its
 * forward/backward scope stay fixed across a comparison (section 06); the
 * pages give no placement and no random-number generator, so both are fixed
 * here:
 *   Pd = P o Z / (1 - p'),  O = Pd V,  lse = the undropped log-sum-exp;
 *   backward with the same Z: dV = Pd^T dO, dP = (dO V^T) o Z / (1 - p'),
 *   dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 * Z_ij (query i, key j, head index h = head_base + b*H + head) is 1 iff
 * byte (j mod 4) of word (i mod 4) of Philox4x32-10 (Salmon et al., SC 2011)
 * with counter (j/4, i/4, h, offset) and key (seed low word, seed high word)
 * is >= t,
 * t = round(256 p_drop) capped at 255, and p' = t / 256. The same
 * (p_drop, seed, offset, head_base) must be passed to both calls. head_base
 * places the call's heads in a larger problem: a batch computed in pieces of
 * heads (or sharded over GPUs) draws the same mask as one call on all of it
 * when each piece passes the index of its first head. Arguments, layouts
 * and errors are as for fa_fwd_kv / fa_bwd_kv; p_drop outside [0, 1) or NaN
 * is FA_ERR_ARG. p_drop = 0 gives the plain results.
 */
int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o,
                   float *lse, int B, int H, int Nq, int Nk, int d,
                   float scale, int causal, int dtype, float p_drop,
                   unsigned long long seed, unsigned int offset,
                   unsigned int head_base, fa_stream_t stream);
int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dO, void *dq, void *dk,
                   void *dv, int B, int H, int Nq, int Nk, int d, float scale,
                   int causal, int dtype, float p_drop,
                   unsigned long long seed, unsigned int offset,
                   unsigned int head_base, void *workspace,
                   size_t workspace_bytes, fa_stream_t stream);

/*
 * Workspace of fa_bwd_dropout in which its two passes share the keep bits:
 * fa_bwd_workspace_size(B, H, Nq, d, dtype) plus fa_dropout_mask_size(B, H,
 * Nq, Nk) bytes (0 unless B, H, Nq, Nk >= 1, d is 64, 96 or 128 and dtype
 * is FA_BF16 or FA_F16). Given at least this many bytes, fa_bwd_dropout's
 * dK/dV pass writes the keep bits it draws into the rest of the workspace
 * (the saved-bits layout below) and its dQ pass reads them there instead of
 * drawing them again; with less (but at least fa_bwd_workspace_size bytes)
 * both passes draw them. The results are the same, bit for bit; the larger
 * workspace trades that memory for about a fifth of the dQ pass's time.
 */
size_t fa_bwd_dropout_workspace_size(int B, int H, int Nq, int Nk, int d,
                                     int dtype);

/*
 * Dropout with saved keep bits: the same method, results and arguments as
 * fa_fwd_dropout / fa_bwd_dropout, but the forward also writes every keep
 * bit it draws into `mask`, and the backward reads them from there instead
 * of drawing them again with Philox4x32-10 (which costs each backward pass
 * about as much as the forward's drawing). The trade is memory: one bit per
 * (query, key) pair, fa_dropout_mask_size(B, H, Nq, Nk) bytes, e.g. 512 MiB
 * for B 8, H 32, Nq = Nk = 4096.
 *   mask    device memory owned by the caller, 16-byte aligned, at least
 *           fa_dropout_mask_size(...) bytes (FA_ERR_NULL / FA_ERR_ALIGN /
 *           FA_ERR_WORKSPACE otherwise). Layout: for head bh = b*H + h (the
 *           call's own heads), query tile qt < ceil(Nq/128) and key tile
 *           kt < ceil(Nk/128), a 2048-byte block at byte offset
 *           ((bh * ceil(Nq/128) + qt) * ceil(Nk/128) + kt) * 2048 of 512
 *           32-bit words, word-major: bit 8 (b mod 4) + floor(b / 4) of
 *           word w * 128 + r (b = 0..31) = the keep bit of query 128 qt + r
 *           and key 128 kt + 32 w + b (the Philox mask of fa_fwd_dropout
 *           with the given seed, offset and head_base). Byte i of a word
 *           thus holds keys i, i + 4, ..., i + 28 of its 32, one bit per
 *           4-key Philox group.
 *           Blocks of tiles the causal mask hides entirely, and bits past Nq
 *           or Nk, are left unspecified.
 *   backward  takes the forward's p_drop and the mask it wrote (no seed:
 *           the bits are given); its results equal fa_bwd_dropout's with the
 *           forward's seed, offset and head_base, bit for bit.
 */
size_t fa_dropout_mask_size(int B, int H, int Nq, int Nk);
int fa_fwd_dropout_mask(const void *q, const void *k, const void *v, void *o,
                        float *lse, int B, int H, int Nq, int Nk, int d,
                        float scale, int causal, int dtype, float p_drop,
                        unsigned long long seed, unsigned int offset,
                        unsigned int head_base, void *mask, size_t mask_bytes,
                        fa_stream_t stream);
int fa_bwd_dropout_mask(const void *q, const void *k, const void *v,
                        const void *o, const float *lse, const void *dO,
                        void *dq, void *dk, void *dv, int B, int H, int Nq,
                        int Nk, int d, float scale, int causal, int dtype,
                        float p_drop, const void *mask, size_t mask_bytes,
                        void *workspace, size_t workspace_bytes,
                        fa_stream_t stream);

/* Forward with float tensors (all fp32 arithmetic, exact expf). Same
 * arguments and layout as fa_fwd with float element type. */
int fa_fwd_f32(const float *q, const float *k, const float *v, float *o,
               float *lse, int B, int H, int N, int d, float scale, int causal,
               fa_stream_t stream);

/* Backward with float tensors. dk and dv are accumulated with fp32 atomics
 * after being cleared on `stream`. workspace as for fa_bwd (dtype FA_F32). */
int fa_bwd_f32(const float *q, const float *k, const float *v, const float *o,
               const float *lse, const float *dO, float *dq, float *dk,
               float *dv, int B, int H, int N, int d, float scale, int causal,
               void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* Bytes of workspace fa_bwd / fa_bwd_f16 / fa_bwd_f32 need for this shape (0
 * on invalid shape). dtype is an fa_dtype. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, int dtype);

/* Static description of a status code; never NULL. */
const char *fa_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this library on the
 * calling host thread (0 if none). */
int fa_last_cuda_error(void);

/* Reads and clears the device status word that kernels set when they give up
 * on a wait (FA_OK or FA_ERR_TIMEOUT). Synchronises the current device. */
int fa_device_status(void);

/*
 * The same status, without synchronising: enqueues on `stream` a copy of the
 * current device's status word into *dst, then clears the word. dst is device
 * memory or page-locked host memory (cudaHostAlloc, torch pin_memory); it
 * holds FA_OK or FA_ERR_TIMEOUT once the stream has reached the copy. The
 * word is one per device, shared by every stream and host thread: a timeout
 * recorded by any earlier kernel of this library on the device shows up in
 * the next read. Returns FA_ERR_NULL / FA_ERR_ALIGN (dst not 4-byte aligned)
 * or FA_ERR_LAUNCH if the copy cannot be enqueued.
 */
int fa_status_async(int *dst, fa_stream_t stream);

/*
 * Device address of the current device's status word, for callers that read
 * it from their own stream-ordered work (their kernels, a captured graph).
 * The library's kernels write FA_ERR_TIMEOUT there and nothing else; clear it
 * by writing 0.
 */
int fa_status_word(int **dev_ptr);

/* Number of kernels the most recent successful fa_* call on this host thread
 * enqueued. */
int fa_last_launch_count(void);

/*
 * Per-kernel timing for benchmarks (no counterpart on the pages; it only
 * measures). `events` holds 2*n_pairs cudaEvent_t handles created by the
 * caller with timing enabled. After this call, every tensor-core kernel that
 * fa_fwd / fa_bwd launch on this host thread is bracketed by the next free
 * pair: events[2i] is recorded on the call's stream just before the kernel
 * and events[2i+1] just after it. fa_fwd uses one pair (the forward kernel),
 * fa_bwd two (the dK/dV pass, then the dQ pass); once all n_pairs are used,
 * nothing more is recorded. Pass NULL / 0 to switch it off. Returns
 * FA_ERR_ARG for n_pairs < -1, and the number of pairs used so far when
 * called with n_pairs == -1 (events ignored).
 */
int fa_set_kernel_timing(void **events, int n_pairs);

/*
 * fa_bwd_static_scratch -- the bf16 backward pass for callers that cannot
 * allocate device memory (no counterpart on the pages; the method is the
 * same as fa_bwd's, only the scratch memory differs).
 *
 * Who needs it: code that runs under a host framework which reserves the
 * GPU's memory up front in its own pool and allows no other cudaMalloc, a
 * plug-in whose fixed calling convention has no slot for a workspace, or a
 * latency-bound path that may not allocate after start-up (cudaMalloc can
 * synchronise the device).
 *
 * Arguments, layout and results are those of fa_bwd without the workspace
 * pair. Instead of a caller buffer the pass uses one static device array of
 * FA_STATIC_SCRATCH_BYTES that this library holds on every GPU that loads it,
 * until the process exits; the call itself allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).
 *   Limit   returns FA_ERR_WORKSPACE, launching nothing, when
 *           fa_bwd_workspace_size(B, H, N, d, FA_BF16) exceeds
 *           FA_STATIC_SCRATCH_BYTES, i.e. past about 2M padded query rows
 *           (B*H*128*ceil(N/128) > 2,097,152).
 *   Set-up  the first call on a device looks up the array's device address
 *           (cudaGetSymbolAddress); make that first call before any stream
 *           capture.
 *   Sharing every call on a device uses the same array, which keeps the last
 *           call's contents; the pass rewrites every byte it reads before
 *           reading it. Calls whose kernels overlap on the GPU (different
 *           streams, or host threads, with no ordering between them) race on
 *           the array and give wrong gradients: order them.
 *   Reset   the looked-up address belongs to the device's current context;
 *           after cudaDeviceReset the next call (on the new context) looks it
 *           up again, so that call, too, should come before any capture.
 */
#define FA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

int fa_bwd_static_scratch(const void *q, const void *k, const void *v,
                          const void *o, const float *lse, const void *dO,
                          void *dq, void *dk, void *dv, int B, int H, int N,
                          int d, float scale, int causal, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
