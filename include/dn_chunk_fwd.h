/*
 * dn_chunk_fwd.h -- C ABI of the chunkwise gated delta rule forward for GB300.
 *
 * Sources (web pages on the method, cited by title and section):
 *   [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现"
 *   [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么"
 *
 * Operation ([CGDR] §1 recurrence, evaluated per chunk as in [CGDR] §3 and
 * [WY] §2.4): for every sequence n and value head h (query/key head
 * h / (Nv/Nk), [CGDR] §1), starting from S = h0[n,h] (or 0),
 *
 *     S_t = e^{g_t} S_{t-1} + beta_t k_t (v_t - k_t^T e^{g_t} S_{t-1})^T
 *     o_t = scale * S_t^T q_t
 *
 * and ht[n,h] = S after the sequence's last token.  The state is decayed
 * before the delta read ("forget first, then write", [CGDR] §1); o_t reads
 * the state after token t's own write.  The library computes it per 64-token
 * chunk: gate prefix sum, WY matrix and T = (I - A)^-1 by forward
 * substitution, W and U, the cross-chunk state pass and the causal output.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, owned by the caller, row-major
 *     and contiguous, 16-byte aligned.  The library keeps no reference to
 *     them after the call and allocates no device memory: scratch space the
 *     computation needs is a caller-owned workspace (see
 *     dn_chunk_fwd_workspace_bytes).
 *   - Calls are asynchronous and ordered on `stream` (NULL = legacy default
 *     stream).  Outputs are valid once the stream reaches the call.
 *   - Errors are returned as a dn_status, never thrown or aborted.  Argument
 *     errors are found on the host before anything is launched; nothing is
 *     written then.  A launch failure returns DN_ERR_CUDA.  Errors found on
 *     the device (a bounded wait that ran out, a malformed cu_seqlens) are
 *     recorded in a per-device status word and reported by dn_check().
 */
#ifndef DN_CHUNK_FWD_H
#define DN_CHUNK_FWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *dn_stream_t;

typedef enum {
    DN_OK = 0,
    DN_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or combination */
    DN_ERR_UNSUPPORTED = 2,  /* valid per the method but not built here (e.g. chunk != 64) */
    DN_ERR_CUDA = 3,         /* the CUDA runtime reported an error */
    DN_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out (dn_check) */
    DN_ERR_DEVICE_ARG = 5    /* the device found a malformed cu_seqlens (dn_check) */
} dn_status;

/*
 * Option bits (the `flags` argument of the forward entry points; other bits
 * are rejected with DN_ERR_INVALID_ARG).
 *   DN_QK_L2NORM  the kernels replace every query and key row (one token,
 *                 one head, length dk) by x / max(||x||_2, 1e-12) before
 *                 using it, in fp32, without writing the normalised rows
 *                 anywhere ([WY] §5 use_qk_l2norm_in_kernel: the same
 *                 normalisation the pages' tests apply to k beforehand,
 *                 [WY] §6, done inside the kernels to save memory).
 */
#define DN_QK_L2NORM 1u

/* Element type of q, k, v and o (one dtype for all four, as in [WY] §5). */
typedef enum {
    DN_BF16 = 0,
    DN_F32 = 1
} dn_dtype;

/*
 * dn_chunk_fwd -- forward pass of the chunkwise gated delta rule.
 *
 * Arguments (all shapes row-major; "tokens" = B*T, flattened over the batch):
 *   q, k        [B, T, Nk, dk]  dtype       queries, keys ([CGDR] §1 table)
 *   v           [B, T, Nv, dv]  dtype       values
 *   beta        [B, T, Nv]      float32     write strength beta_t
 *   g           [B, T, Nv]      float32     log-domain decay g_t; NULL means
 *                                           g = 0 (plain DeltaNet, [WY] §1)
 *   h0          [N, Nv, dk, dv] float32     initial state; NULL means zero
 *   cu_seqlens  [N+1]           int64       packed sequence offsets
 *                                           ([WY] §5 varlen); NULL means N = B
 *                                           sequences of length T.  Non-NULL
 *                                           requires B == 1.  Must be
 *                                           non-decreasing with cu[0] = 0 and
 *                                           cu[N] <= T (checked on the device:
 *                                           a bad sequence is skipped and
 *                                           dn_check returns DN_ERR_DEVICE_ARG).
 *   n_seqs      N; must equal B when cu_seqlens is NULL.  N = 0 is a no-op.
 *   B, T        batch and tokens per batch row; T may be 0.
 *   Nk, Nv      key/value head counts; Nv % Nk == 0 (GQA, nvPerNk = Nv/Nk).
 *   dk, dv      head dims, each one of 16, 32, 64, 128, 256.
 *   dtype       DN_BF16 or DN_F32.  With DN_F32 every product is computed in
 *               fp32 on CUDA cores (no TF32), and dk must be <= 128.
 *   scale       multiplies q in the output; scale <= 0 selects 1/sqrt(dk).
 *   flags       0 or DN_QK_L2NORM (q and k rows normalised in the kernels).
 *   chunk       chunk length C: 16, 32 or 64 ([WY] §5 chunk_size; the result
 *               is the same up to rounding, [WY] §6).  The tensor-core path
 *               takes all three (a chunk fills the first C rows of its 64-row
 *               tiles, so a step costs about the same at every C and C = 64
 *               is the fastest); other values: DN_ERR_UNSUPPORTED.
 *   o           [B, T, Nv, dv]  dtype       output, written for every token of
 *                                           every sequence (rounded to nearest
 *                                           even from fp32 for DN_BF16).
 *   ht          [N, Nv, dk, dv] float32     final state; NULL: not written.
 *   workspace   device scratch of at least dn_chunk_fwd_workspace_bytes()
 *               bytes for these sizes, 16-byte aligned, owned by the caller
 *               and not touched by anyone else until the stream has passed
 *               the call.  May be NULL when that size is 0.  Its contents on
 *               entry do not matter; on exit they are unspecified.
 *   workspace_bytes  its size in bytes.
 *   stream      CUDA stream for the launch.
 *
 * Returns DN_OK once the work is enqueued; DN_ERR_INVALID_ARG also when the
 * workspace is missing, misaligned or too small.  The tensor-core path
 * (bf16, dk = 128 or 256, dv a multiple of 128) launches two kernels per
 * call: the per-chunk WY inverse T and causal scores of every chunk in
 * parallel ([WY] §2.3-§2.4), then the sequential state scan and output
 * ([CGDR] §3.2-§3.3).  Other shapes launch one CUDA-core kernel; for DN_BF16 its
 * state products (K S, Q S, the state update) are TF32 tensor-core tiles with
 * fp32 accumulation, within the bf16 bound.
 *
 * Why a workspace.  The per-chunk work that needs no state (the inverse T,
 * the scores P) runs for all chunks at once in the first kernel; only the
 * scan is sequential.  The two kernels hand over three bf16 matrices per
 * chunk and value head through the workspace (mostly through L2 between the
 * two launches).  A single kernel that formed T beside the scan put that
 * work back on the scan's serial path and measured slower (158 against about
 * 120 us per forward at B = 4, H = 16, T = 2048, d = 128).  So the call takes
 * the caller's workspace instead of allocating one (dn_chunk_fwd_noalloc
 * below uses a fixed array of the library instead), plus the flags and chunk
 * arguments of the options it implements.
 */
dn_status dn_chunk_fwd(const void *q, const void *k, const void *v,
                       const float *beta, const float *g, const float *h0,
                       const int64_t *cu_seqlens, int n_seqs,
                       int B, int T, int Nk, int Nv, int dk, int dv,
                       dn_dtype dtype, float scale, unsigned flags, int chunk,
                       void *o, float *ht, void *workspace, size_t workspace_bytes,
                       dn_stream_t stream);

/*
 * dn_chunk_fwd_workspace_bytes -- bytes of workspace dn_chunk_fwd needs for
 * these sizes (same meaning as there).  For the tensor-core path it is
 * (floor(B*T / C) + n_seqs) * Nv * S (C the chunk length): one slot of S
 * bytes per chunk and value head holding bf16 matrices of the chunk --
 * T diag(beta e^G) (64 x 64; for dk = 256 instead -W = -T diag(beta e^G) K,
 * 64 x 256) and T diag(beta) (64 x 64) of its WY representation ([WY] §2.4)
 * and its causal score matrix tril(scale QK^T . D) (64 x 64, [CGDR] §3.2) --
 * then the chunk's 64 key and 64 query inverse norms (fp32; written only
 * with DN_QK_L2NORM).  S = 25088 for dk = 128 and 49664 for dk = 256.  The
 * size does
 * not depend on the flags.  Returns 0 when no workspace is
 * needed, and for sizes dn_chunk_fwd would reject.  Host-only; no CUDA call.
 */
size_t dn_chunk_fwd_workspace_bytes(int n_seqs, int B, int T, int Nk, int Nv, int dk, int dv,
                                    dn_dtype dtype, int chunk);

/*
 * dn_recurrent_fwd -- the same forward evaluated token by token ("fused
 * recurrent", "flash linear attention" notes, Attention section: the
 * recurrent mode the RetNet layer there picks for query lengths up to 64).
 * It suits decoding (T = 1 with h0 in and ht out) and short prompts.
 *
 * Arguments as for dn_chunk_fwd (flags included) without chunk and
 * workspace; any dtype and
 * dk, dv in {16, 32, 64, 128, 256} (fp32 included up to 256).  Per token,
 * in fp32: S <- e^{g_t} S; d = beta_t (v_t - S^T k_t); S <- S + k_t d^T;
 * o_t = scale S^T q_t ([CGDR] §1).  One CUDA-core kernel launch per call; it
 * allocates nothing and needs no workspace.  Errors as for dn_chunk_fwd.
 */
dn_status dn_recurrent_fwd(const void *q, const void *k, const void *v,
                           const float *beta, const float *g, const float *h0,
                           const int64_t *cu_seqlens, int n_seqs,
                           int B, int T, int Nk, int Nv, int dk, int dv,
                           dn_dtype dtype, float scale, unsigned flags,
                           void *o, float *ht, dn_stream_t stream);

/*
 * dn_chunk_fwd_noalloc -- dn_chunk_fwd for callers that cannot allocate
 * device memory where they call it (for example a plugin host whose execute
 * path may not allocate because the host owns every device buffer, or a
 * runtime that committed all device memory to its own pool, where cudaMalloc
 * would fail or stall the device).  The paper has no counterpart: this is a
 * packaging variant of the same computation, not a step of the method.
 *
 * Same arguments and results as dn_chunk_fwd, without a workspace: the
 * scratch space lives in one fixed device array of this library,
 * DN_NOALLOC_SCRATCH_BYTES long.  The call allocates nothing itself.
 *   - Arguments are checked exactly as dn_chunk_fwd checks them, first: a
 *     bad argument gives DN_ERR_INVALID_ARG (or DN_ERR_UNSUPPORTED for a
 *     shape no kernel takes) whatever the sizes.
 *   - Then sizes whose dn_chunk_fwd_workspace_bytes() exceeds
 *     DN_NOALLOC_SCRATCH_BYTES are rejected with DN_ERR_UNSUPPORTED before
 *     anything is launched.
 *   - The first call with a given device current looks up the array's device
 *     address there.  Under CUDA's default lazy module loading that lookup
 *     also loads this part of the library onto the GPU, which is when the
 *     GPU reserves the array: the first call can therefore fail with
 *     DN_ERR_CUDA if device memory is already exhausted.  Make that first
 *     call at set-up time, before committing the rest of the device memory
 *     and before any stream capture on that device; later calls reserve
 *     nothing, and the array is held until the process exits.
 *   - Every call uses the same array; its contents on entry do not matter.
 *     Calls whose kernels can overlap on one GPU (other streams, other host
 *     threads) race on it; calls ordered in one stream do not.
 */
#define DN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

dn_status dn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                               const float *beta, const float *g, const float *h0,
                               const int64_t *cu_seqlens, int n_seqs,
                               int B, int T, int Nk, int Nv, int dk, int dv,
                               dn_dtype dtype, float scale, unsigned flags, int chunk,
                               void *o, float *ht, dn_stream_t stream);

/*
 * dn_chunk_bwd -- gradient of dn_chunk_fwd ([WY] §3.4: the backward
 * recomputes each chunk's WY quantities and walks the chunks in reverse; it
 * gives dq, dk, dv, dbeta and dh0, and the gated form dg).
 *
 * For the loss l = sum(d_o . o) + sum(d_ht . ht) of the forward with the same
 * inputs, writes the gradients of l:
 *   d_q, d_k   [B, T, Nk, dk]  float32   (summed over the Nv/Nk value heads
 *                                          that read each key head)
 *   d_v        [B, T, Nv, dv]  float32
 *   d_beta     [B, T, Nv]      float32
 *   d_g        [B, T, Nv]      float32 or NULL (not computed); with g NULL it
 *                                          is the gradient at g = 0
 *   d_h0       [N, Nv, dk, dv] float32 or NULL; with h0 NULL it is the
 *                                          gradient at h0 = 0
 * from
 *   d_o        [B, T, Nv, dv]  dtype     gradient of o (required)
 *   d_ht       [N, Nv, dk, dv] float32   gradient of ht; NULL means zero.
 * The other arguments are those of dn_chunk_fwd (the chunk length is 64).
 * The reverse walk is fp32 arithmetic on CUDA cores.  The chunk-start states
 * it reads come from a forward pass with no output: for bf16 with dk = 128
 * and dv a multiple of 128, the tensor-core forward (bf16 MMA operands, fp32
 * state), as the [WY] §3.4 backward recomputes them with the forward
 * kernels; otherwise the fp32 CUDA-core forward.  dk must be at most 128
 * (DN_ERR_UNSUPPORTED otherwise).  With DN_QK_L2NORM the forward it
 * differentiates normalises q and k in the kernels, and d_q, d_k are the
 * gradients of the raw rows (through the normalisation; a fourth launch maps
 * them row by row).  Rows of tokens outside every sequence are 0 in d_q,
 * d_k, d_beta and d_g and not written in d_v.  The sums over value tiles and
 * value heads use fp32 atomic adds, so the last bits of d_q, d_k, d_beta
 * and d_g may differ from run to run.
 *
 * workspace: at least dn_chunk_bwd_workspace_bytes() bytes, 16-byte
 * aligned, owned by the caller (it holds the fp32 state at the start of every
 * 64-token chunk, then, on the tensor-core forward, that forward's
 * workspace).  Launches a zero fill, the forward (one or two launches,
 * saving those states) and the backward kernel.  Errors as for dn_chunk_fwd.
 */
dn_status dn_chunk_bwd(const void *q, const void *k, const void *v,
                       const float *beta, const float *g, const float *h0,
                       const int64_t *cu_seqlens, int n_seqs,
                       int B, int T, int Nk, int Nv, int dk, int dv,
                       dn_dtype dtype, float scale, unsigned flags,
                       const void *d_o, const float *d_ht,
                       float *d_q, float *d_k, float *d_v, float *d_beta, float *d_g,
                       float *d_h0, void *workspace, size_t workspace_bytes,
                       dn_stream_t stream);

/*
 * dn_chunk_bwd_workspace_bytes -- bytes of workspace dn_chunk_bwd needs:
 * (floor(B*T / 64) + n_seqs) * Nv * dk * dv * 4 (one fp32 state per chunk and
 * value head), plus, where the backward's forward pass runs on the tensor
 * cores (bf16, dk = 128, dv a multiple of 128), dn_chunk_fwd_workspace_bytes()
 * of the same sizes at chunk 64 and (floor(B*T / 64) + n_seqs) * Nv * 49152:
 * three fp32 64 x 64 matrices per chunk and value head (-(K K^T . D), the
 * scores P and the WY inverse T), which that forward pass keeps so that the
 * reverse walk need not form them again for every value tile.  0 for sizes
 * dn_chunk_bwd would reject.  Host-only.
 */
size_t dn_chunk_bwd_workspace_bytes(int n_seqs, int B, int T, int Nk, int Nv, int dk, int dv,
                                    dn_dtype dtype);

/*
 * dn_check -- wait for `stream`, then read and clear the device status word
 * of the current device.  Returns DN_ERR_TIMEOUT or DN_ERR_DEVICE_ARG if a
 * kernel of this library recorded one since the last check, DN_ERR_CUDA if
 * the stream reports an error, else DN_OK.
 */
dn_status dn_check(dn_stream_t stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char *dn_status_str(dn_status status);

/*
 * dn_last_kernel -- name of the kernel(s) the last successful call of a
 * compute entry point on this host thread launched ("" before any call).
 * Static storage.
 */
const char *dn_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* DN_CHUNK_FWD_H */
