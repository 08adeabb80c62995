/*
 * fa.h -- exact fused attention for NVIDIA GB300 (sm_103a): the C ABI.
 *
 * Computes, for every batch b and head h,
 *
 *     O = softmax(scale * Q K^T + mask) V
 *
 * tile by tile with a running row maximum and normaliser (online softmax) and
 * a rescaled output accumulator, so the N x N score and probability matrices
 * never reach device memory.  The forward saves O and one logsumexp per row;
 * the backward recomputes scores and probabilities tile by tile from Q, K, V
 * and that logsumexp.
 *
 * Sources (cited by page title and passage):
 *   [T] blog.teqners.com, "13% more FLOPs, 5.7x faster: how FlashAttention's
 *       online softmax keeps the N x N matrix out of HBM"
 *   [L] lensaml.com, "FlashAttention" explainer
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout   q, k, v, o, dout, dq, dk, dv: contiguous [B, H, N, d] bf16
 *           (row-major; element (b,h,i,c) at ((b*H + h)*N + i)*d + c).
 *           lse: contiguous [B, H, N] fp32.
 *  Sizes    B >= 1, H >= 1, N >= 1, d in {64, 128}; B*H*N*d < 2^31 elements
 *           per tensor; B*H < 2^31.
 *  scale    any finite value (typically 1/sqrt(d); 0 gives uniform
 *           attention, a negative value is allowed); applied to Q K^T
 *           before the mask.
 *  causal   0: every key is visible.  1: key j is visible to query i iff
 *           j <= i (square, top-left aligned).  No other mask is supported.
 *  Pointers device pointers, 16-byte aligned; all memory is owned by the
 *           caller; the library allocates no device memory on these paths.
 *           Outputs must not overlap inputs or each other.
 *  Streams  every call is asynchronous on `stream` (0 = legacy default);
 *           argument validation is synchronous and leaves no CUDA error set.
 *  Numbers  bf16 operands, fp32 accumulation and softmax; P (and dS in the
 *           backward) rounded to bf16 before the second contraction; outputs
 *           rounded to nearest even.  Results equal standard attention up to
 *           rounding ([L] Step 6 and FAQ); the backward's dQ is summed with
 *           fp32 atomics, so its last bits depend on arrival order.
 *  Errors   a non-zero fa_status_t.  Nothing is launched when validation
 *           fails.  A kernel that gives up waiting records
 *           FA_ERR_DEVICE_TIMEOUT (FA_ERR_INTERNAL if it finds its shared
 *           memory misaligned) in a device status word that
 *           fa_get_device_status() reads and clears.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, scale, causal */
  FA_ERR_UNSUPPORTED = 2,     /* d not in {64, 128}, or device is not sm_103 */
  FA_ERR_WORKSPACE = 3,       /* workspace missing or smaller than required */
  FA_ERR_CUDA = 4,            /* a CUDA runtime/driver call or launch failed */
  FA_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up on a bounded wait */
  FA_ERR_INTERNAL = 6         /* a kernel found an internal layout assumption violated */
} fa_status_t;

/*
 * Forward pass.  [T] "FlashAttention's move: rescale the output, too";
 * [L] Step 3 "Tiling" and Step 4 "Online Softmax".
 *
 *   q, k, v  in   [B, H, N, d] bf16
 *   o        out  [B, H, N, d] bf16, O = softmax(scale * Q K^T + mask) V
 *   lse      out  [B, H, N] fp32, natural-log logsumexp of each scaled,
 *                 masked score row (m + ln l of the running statistics,
 *                 [T] "The backward pass: recompute instead of read")
 *
 * One persistent kernel launch.  Returns FA_OK or an error above.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, cudaStream_t stream);

/*
 * Forward with FP8 queries and keys.  [L] "Key ideas": FlashAttention-3 adds
 * FP8.  Q and K arrive as E4M3 codes (OCP FP8: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest 448),
 * each tensor with one descale factor: the real value of an element is its
 * decoded code times the factor.  S = Q K^T runs on the tensor cores in E4M3
 * with fp32 accumulation (every product of two E4M3 values is exact in
 * fp32); P and V stay bf16.
 *
 *   q8, k8    in   [B, H, N, d] E4M3 codes, one byte each, d = 128
 *   v         in   [B, H, N, d] bf16
 *   o, lse    out  as fa_fwd, for the scores scale * q_descale * k_descale *
 *                  (decoded Q)(decoded K)^T
 *   q_descale, k_descale  finite, >= 0 (and scale >= 0 here)
 *
 * One persistent kernel launch.  A NaN code makes the rows it reaches NaN.
 * Errors as fa_fwd, plus FA_ERR_UNSUPPORTED for d != 128 and
 * FA_ERR_INVALID_ARG for a negative or non-finite descale, a negative scale,
 * or a non-finite product of the three.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, float q_descale, float k_descale, int causal, cudaStream_t stream);

/*
 * Split-KV forward for decoding.  [L] FAQ "Does FlashAttention help during
 * LLM decoding?": a decode step has one query (or a few) per sequence, the
 * cost is reading the key/value cache, and Flash-Decoding spreads that read
 * over many thread blocks.  Each split (a run of 128-key tiles of one head)
 * computes its own softmax partial; the partials are merged with the
 * online-softmax rescale ([T] "Softmax is the anti-tiling operation").
 *
 *   q         in   [B, H, Nq, d] bf16, 1 <= Nq <= 8: the last Nq positions
 *   k, v      in   [B, H, Nk, d] bf16, the whole cache (Nk >= 1)
 *   o         out  [B, H, Nq, d] bf16
 *   lse       out  [B, H, Nq] fp32, natural-log logsumexp of each row
 *   causal    key j is visible to query i iff j <= i + (Nk - Nq)
 *             (bottom-right; needs Nq <= Nk); 0 = every key
 *   num_splits  splits per head; 0 picks as many as fill the SMs with one
 *             CTA each; never more than the 128-key tiles of the cache
 *   workspace  fa_fwd_splitkv_workspace_size() bytes, 256-byte aligned,
 *             owned by the caller (may be NULL when that size is 0)
 *
 * One launch when a head has one split, or when a head's splits fit one
 * thread-block cluster that the device can co-schedule for every head (the
 * cluster merges in shared memory); else two (splits, then the merge).
 * Errors: FA_ERR_UNSUPPORTED for Nq > 8 or d not in {64, 128};
 * FA_ERR_INVALID_ARG for non-positive sizes, causal with Nq > Nk, a negative
 * num_splits or misaligned pointers; FA_ERR_WORKSPACE for a missing or
 * short workspace.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, int num_splits, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/*
 * Workspace bytes fa_fwd_splitkv needs for these sizes (with the current
 * device's SM count when num_splits is 0): the fp32 partial outputs and
 * partial logsumexps of the splits.  0 when one split per head suffices or
 * the splits merge inside a cluster, or when the sizes are invalid
 * (fa_fwd_splitkv then reports the error).
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: an fp32 dQ
 * accumulator [B, H, N, d] and the row terms D = rowsum(dO * O) [B, H, N],
 * each 256-byte aligned.  Returns 0 when the sizes are invalid.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass.  [T] "The backward pass: recompute instead of read": scores
 * and probabilities are rebuilt tile by tile from q, k, v and lse; nothing of
 * size N x N is read or written.  Gradients of L = sum(O * dO):
 *
 *   q, k, v, o, dout  in   [B, H, N, d] bf16 (o and lse from fa_fwd)
 *   lse               in   [B, H, N] fp32
 *   dq, dk, dv        out  [B, H, N, d] bf16
 *   workspace         scratch of at least fa_bwd_workspace_size() bytes,
 *                     256-byte aligned, owned by the caller; its contents on
 *                     entry do not matter and are undefined on return.
 *
 * Three launches on `stream`: preprocess (D, zero dQ accumulator), the fused
 * dK/dV/dQ kernel, and the dQ conversion.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
           size_t workspace_bytes, cudaStream_t stream);

/*
 * Forward and backward with dropout on the attention probabilities.  [T] "The
 * backward pass: recompute instead of read": the forward keeps only the
 * dropout generator state and the backward regenerates the mask from it.
 *
 *   p_drop  probability of dropping a probability, 0 <= p_drop < 1
 *   seed    64-bit key of the counter-based generator (Philox4x32-10)
 *   offset  fourth counter word (e.g. a step count, for a fresh mask)
 *
 * Element (b, h, query i, key j) is kept iff word (j mod 4) of
 * Philox4x32-10(counter = (j / 4, i, b H + h, offset), key = seed) is at
 * least round(p_drop 2^32); O = (P o M / (1 - p_drop)) V, lse is that of the
 * undropped softmax.  fa_bwd_dropout takes the same p_drop, seed and offset
 * and fa_bwd's other arguments and workspace, and returns the gradients of
 * that forward.  Errors as fa_fwd / fa_bwd, plus FA_ERR_INVALID_ARG for
 * p_drop outside [0, 1).
 */
int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, int causal, float p_drop, unsigned long long seed, unsigned int offset,
                   cudaStream_t stream);
int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, float p_drop,
                   unsigned long long seed, unsigned int offset, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/*
 * Deterministic backward (bitwise the same on every run): the same arguments,
 * workspace and results as fa_bwd, without any reduction between CTAs.
 * [L] Step 3 and [T] "The backward pass: recompute instead of read": the
 * gradients are rebuilt tile by tile in the two loop orders, key tiles outer
 * for dK and dV (as in fa_bwd, minus dQ) and query tiles outer for dQ, which
 * accumulates in tensor memory in a fixed order and is written once.  Three
 * launches on `stream`: preprocess (D and lse * log2 e), the dK / dV kernel,
 * the dQ kernel.  Slower than fa_bwd (S and P are rebuilt twice).
 */
int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The three launches of fa_bwd as separate calls, for callers that schedule
 * or time them individually.  Running them in this order on one stream with
 * one workspace is exactly fa_bwd; arguments mean the same as there.
 *
 *   fa_bwd_preprocess  reads o, dout, lse; writes the row terms
 *                      D = rowsum(dO * O) and lse * log2(e) into the
 *                      workspace and zeroes its fp32 dQ accumulator.
 *   fa_bwd_dkdv        the fused recompute kernel: writes dk and dv and adds
 *                      every dQ partial into the workspace accumulator.
 *   fa_bwd_dq_convert  dq = scale * accumulator, rounded to bf16.
 */
int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);
int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv, int B, int H,
                int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                cudaStream_t stream);
int fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale, const void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/*
 * Size of the library-owned scratch fa_bwd_noalloc uses: 64 MiB, held on every
 * GPU that loads the library until the process exits.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Backward pass without a caller-supplied workspace.  The pages have no
 * counterpart: this serves callers that cannot allocate device memory (code
 * running where cudaMalloc is forbidden or unwanted, such as inside an
 * allocator hook or a plug-in that must not touch the process's memory pool).
 * Arguments and results are those of fa_bwd; the workspace is a file-scope
 * device array of FA_NOALLOC_SCRATCH_BYTES owned by the library, and nothing
 * is allocated or freed by the call.
 *
 *   Limit     exactly fa_bwd_workspace_size(B, H, N, d) <=
 *             FA_NOALLOC_SCRATCH_BYTES, where that size is
 *             round256(4 B H N d) + 2 round256(4 B H Npad) bytes, Npad = N
 *             rounded up to a multiple of 128 (for example B = 2, H = 8,
 *             N = 8064, d = 128 fits with 16 KiB to spare; N = 8065 does
 *             not).  Larger problems return FA_ERR_WORKSPACE without
 *             launching anything; invalid arguments are reported first, with
 *             fa_bwd's codes.
 *   Set-up    the first call in each CUDA context looks up the scratch's
 *             device address (cudaGetSymbolAddress) with that context and
 *             its device current, and caches it by the context's unique ID
 *             (another context, or a primary context created again after a
 *             reset, looks it up anew); make that first call before any
 *             stream capture.
 *   Sharing   every call on a device uses the same scratch, which keeps the
 *             last call's contents (the call itself clears what must start at
 *             zero).  Calls that overlap on the GPU (different streams, no
 *             ordering between them) race on it and give wrong results.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                   int causal, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: FA_OK, or FA_ERR_DEVICE_TIMEOUT if any kernel of this
 * library gave up on a bounded wait since the last call (FA_ERR_INTERNAL for
 * a violated layout assumption); FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int fa_get_device_status(cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
