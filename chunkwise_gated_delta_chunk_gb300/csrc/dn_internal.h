// Internal declarations shared by the C-ABI front end and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dn_chunk_fwd.h"

namespace dn {

constexpr int kChunk = 64;  // C: tokens per chunk of the tensor-core path; tile size of both paths

// Bits of the per-device status word (see dn_check in the public header).
constexpr unsigned kStatusTimeout = 1u;   // a bounded mbarrier wait ran out
constexpr unsigned kStatusBadSeq = 2u;    // cu_seqlens out of order / out of range

// Option bits of Params::flags (the public DN_ flags of the same value).
constexpr unsigned kQkL2Norm = 1u;        // q and k rows divided by max(||x||_2, 1e-12)

// Limit of every bounded mbarrier wait of the tensor-core kernels.  A build
// for the failure-path test (-DDN_TEST_STALL) shortens it, so that a wait
// that runs out costs milliseconds, not seconds.
#ifdef DN_TEST_STALL
constexpr unsigned long long kWaitLimitNs = 2000000ull;     // 2 ms
#else
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
#endif

// Params::test_stall in a -DDN_TEST_STALL build: the call makes one wait run
// out on purpose (1: the scan kernel's first stage never completes; 2: the
// first item of one WY worker expects more TMA bytes than arrive).  Always 0
// in the library's own build, which contains none of this code.
constexpr unsigned kStallScan = 1u, kStallWy = 2u;

struct Params {
    const void *q, *k, *v;     // [tokens, Nk, dk], [tokens, Nk, dk], [tokens, Nv, dv]
    const float *beta, *g;     // [tokens, Nv]; g may be null
    const float *h0;           // [N, Nv, dk, dv] or null
    const int64_t *cu;         // [N+1] or null
    void *o;                   // [tokens, Nv, dv]
    float *ht;                 // [N, Nv, dk, dv] or null
    int N, B, T, Nk, Nv, dk, dv;
    long long tokens;          // B*T
    float scale;
    unsigned *status;          // per-device status word
    void *ws;                  // workspace: nslots x Nv slots of T' | T'' | P (tensor-core path)
    long long nslots;          // floor(tokens / C) + N
    int chunk;                 // chunk length: 64 (both paths) or 16 / 32 (CUDA-core path)
    unsigned flags;            // kQkL2Norm
    unsigned test_stall;       // 0, or kStallScan / kStallWy in a -DDN_TEST_STALL build
    // backward (dn_chunk_bwd) only; null elsewhere
    float *hs;                 // [Nv][nslots][dk][dv]: state before each 64-token chunk (slot t0/64 + n)
    const void *dout;          // [tokens, Nv, dv] gradient of o (dtype of q)
    const float *dht;          // [N, Nv, dk, dv] gradient of ht or null
    float *dq, *dkk, *dvv;     // [tokens, Nk, dk], [tokens, Nk, dk], [tokens, Nv, dv]
    float *dbeta, *dg;         // [tokens, Nv]; dg may be null
    float *dh0;                // [N, Nv, dk, dv] or null
    // [Nv][nslots][3][64][64] fp32 per chunk: -(K K^T . D) (strictly lower),
    // P (lower) and T = (I - A)^-1, written by the WY kernel in the backward's
    // forward pass (dk = 128 tensor-core path) for the reverse walk; else null
    float *wyx;
};

// CUDA-core kernel: any supported shape.  `bf16` selects bf16 q/k/v/o, else
// fp32.  `tf32` (bf16 only): the state products as TF32 tensor-core tiles;
// otherwise every product is an fp32 FMA.  Returns the launch error.
cudaError_t simt_launch(const Params &p, bool bf16, bool tf32, cudaStream_t stream, const char **name);
size_t simt_smem_bytes(int dk, bool bf16);

// Backward: zero the accumulated gradients, rerun the CUDA-core forward
// saving each chunk's start state in p.hs (p.o and p.ht null), then walk the
// chunks in reverse.  dk <= 128.
cudaError_t bwd_launch(const Params &p, bool bf16, cudaStream_t stream, const char **name);
size_t bwd_smem_bytes(int dk, bool bf16, bool mma);  // mma: the tensor-core instantiation

// Host checks of dn_chunk_fwd's arguments other than the workspace, in the
// order that entry point applies them: DN_ERR_INVALID_ARG for arguments that
// are wrong whatever is built, then DN_ERR_UNSUPPORTED for valid shapes no
// kernel takes; DN_OK otherwise.  Touches no device state.
dn_status chunk_fwd_check_args(const void *q, const void *k, const void *v, const float *beta,
                               const float *g, const float *h0, const int64_t *cu_seqlens, int n_seqs,
                               int B, int T, int Nk, int Nv, int dk, int dv, dn_dtype dtype,
                               float scale, unsigned flags, int chunk, const void *o, const float *ht);

// Token-serial kernel (decode / short sequences): any supported shape.
cudaError_t recurrent_launch(const Params &p, bool bf16, cudaStream_t stream, const char **name);

}  // namespace dn
