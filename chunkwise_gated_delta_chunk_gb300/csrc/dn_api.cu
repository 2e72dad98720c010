// C-ABI front end: argument validation, kernel selection and launch.
//
// Everything here runs on the host.  Validation happens before any CUDA call,
// so argument errors return without touching the device.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "dn_chunk_fwd.h"
#include "dn_internal.h"
#include "dn_tc.h"

#define DN_EXPORT extern "C" __attribute__((visibility("default")))

// Per-device status word: kernels OR error bits into it; dn_check reads and
// clears it.  Module-scope device memory, so no allocation is ever needed.
__device__ unsigned g_dn_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];

thread_local const char *t_last_kernel = "";

#ifdef DN_TEST_STALL
// The failure-path test build's hook: the next dn_chunk_fwd call on this
// thread makes one bounded wait run out (kStallScan / kStallWy).
thread_local unsigned t_test_stall = 0;
#endif

// Device address of g_dn_status on the current device (looked up once per
// device; the lookup is a host call that allocates nothing).
cudaError_t status_ptr(unsigned **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_dn_status);
        if (err != cudaSuccess) return err;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_status_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }

bool flags_ok(unsigned flags) { return (flags & ~DN_QK_L2NORM) == 0; }
static_assert(DN_QK_L2NORM == dn::kQkL2Norm, "public and internal flag bits agree");

// Bytes of workspace the call with these sizes needs (0: none).  The
// tensor-core path keeps T' | T'' of every chunk there between its two kernels.
bool chunk_ok(int chunk) { return chunk == 16 || chunk == 32 || chunk == dn::kChunk; }

// The tensor-core path takes bf16, dk = 128 or 256 and dv a multiple of 128,
// at every chunk length; everything else runs on the CUDA-core kernel.
bool use_tc(long long tokens, int dk, int dv, dn_dtype dtype, int chunk) {
    return tokens > 0 && dn::tc_supported(dk, dv, dtype == DN_BF16, chunk);
}

size_t workspace_bytes(long long tokens, int n_seqs, int Nv, int dk, int dv, dn_dtype dtype, int chunk) {
    if (!use_tc(tokens, dk, dv, dtype, chunk)) return 0;
    return dn::tc_workspace_bytes(tokens, n_seqs, Nv, dk, chunk);
}

}  // namespace

DN_EXPORT size_t dn_chunk_fwd_workspace_bytes(int n_seqs, int B, int T, int Nk, int Nv, int dk, int dv,
                                              dn_dtype dtype, int chunk) {
    if (n_seqs <= 0 || B < 0 || T < 0 || Nk <= 0 || Nv <= 0 || !chunk_ok(chunk)) return 0;
    return workspace_bytes((long long)B * T, n_seqs, Nv, dk, dv, dtype, chunk);
}

namespace dn {

// Checks of dn_chunk_fwd's arguments other than the workspace (also run by
// dn_chunk_fwd_noalloc before it looks at sizes).  DN_OK: the call can run.
dn_status chunk_fwd_check_args(const void *q, const void *k, const void *v, const float *beta,
                               const float *g, const float *h0, const int64_t *cu_seqlens, int n_seqs,
                               int B, int T, int Nk, int Nv, int dk, int dv, dn_dtype dtype,
                               float scale, unsigned flags, int chunk, const void *o, const float *ht) {
    // ---- arguments that are wrong whatever is built ----------------------
    if (dtype != DN_BF16 && dtype != DN_F32) return DN_ERR_INVALID_ARG;
    if (n_seqs < 0 || B < 0 || T < 0 || Nk <= 0 || Nv <= 0 || dk <= 0 || dv <= 0)
        return DN_ERR_INVALID_ARG;
    if (Nv % Nk != 0) return DN_ERR_INVALID_ARG;
    if (cu_seqlens ? B != 1 : n_seqs != B) return DN_ERR_INVALID_ARG;
    if (isnan(scale) || isinf(scale)) return DN_ERR_INVALID_ARG;
    if (!flags_ok(flags)) return DN_ERR_INVALID_ARG;
    if (chunk <= 0) return DN_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    if (tokens > 0 && (!q || !k || !v || !beta || !o)) return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, g, h0, cu_seqlens, o, ht};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return DN_ERR_INVALID_ARG;
    // ---- valid, but not built --------------------------------------------
    if (!chunk_ok(chunk)) return DN_ERR_UNSUPPORTED;
    if (!dim_ok(dk) || !dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (dtype == DN_F32 && dk > 128) return DN_ERR_UNSUPPORTED;
    return DN_OK;
}

}  // namespace dn

DN_EXPORT dn_status dn_chunk_fwd(const void *q, const void *k, const void *v,
                                 const float *beta, const float *g, const float *h0,
                                 const int64_t *cu_seqlens, int n_seqs,
                                 int B, int T, int Nk, int Nv, int dk, int dv,
                                 dn_dtype dtype, float scale, unsigned flags, int chunk,
                                 void *o, float *ht, void *workspace, size_t workspace_bytes_,
                                 dn_stream_t stream) {
    const dn_status args = dn::chunk_fwd_check_args(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv,
                                                    dk, dv, dtype, scale, flags, chunk, o, ht);
    if (args != DN_OK) return args;
    if (n_seqs == 0) return DN_OK;
    const long long tokens = (long long)B * T;
    const size_t ws_need = workspace_bytes(tokens, n_seqs, Nv, dk, dv, dtype, chunk);
    if (ws_need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes_ < ws_need))
        return DN_ERR_INVALID_ARG;

    dn::Params p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.cu = cu_seqlens;
    p.o = o; p.ht = ht;
    p.N = n_seqs; p.B = B; p.T = T; p.Nk = Nk; p.Nv = Nv; p.dk = dk; p.dv = dv;
    p.tokens = tokens;
    p.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)dk);
    p.ws = workspace;
    p.nslots = tokens / chunk + n_seqs;
    p.chunk = chunk;
    p.flags = flags;
#ifdef DN_TEST_STALL
    p.test_stall = t_test_stall;
    t_test_stall = 0;
#endif
    if (status_ptr(&p.status) != cudaSuccess) return DN_ERR_CUDA;

    const char *name = "";
    const bool bf16 = dtype == DN_BF16;
    cudaError_t err;
    if (use_tc(tokens, dk, dv, dtype, chunk))
        err = dn::tc_launch(p, (cudaStream_t)stream, &name);
    else
        err = dn::simt_launch(p, bf16, bf16, (cudaStream_t)stream, &name);
    if (err != cudaSuccess) return DN_ERR_CUDA;
    t_last_kernel = name;
    return DN_OK;
}

DN_EXPORT dn_status dn_recurrent_fwd(const void *q, const void *k, const void *v,
                                     const float *beta, const float *g, const float *h0,
                                     const int64_t *cu_seqlens, int n_seqs,
                                     int B, int T, int Nk, int Nv, int dk, int dv,
                                     dn_dtype dtype, float scale, unsigned flags,
                                     void *o, float *ht, dn_stream_t stream) {
    if (dtype != DN_BF16 && dtype != DN_F32) return DN_ERR_INVALID_ARG;
    if (n_seqs < 0 || B < 0 || T < 0 || Nk <= 0 || Nv <= 0 || dk <= 0 || dv <= 0)
        return DN_ERR_INVALID_ARG;
    if (Nv % Nk != 0) return DN_ERR_INVALID_ARG;
    if (cu_seqlens ? B != 1 : n_seqs != B) return DN_ERR_INVALID_ARG;
    if (isnan(scale) || isinf(scale)) return DN_ERR_INVALID_ARG;
    if (!flags_ok(flags)) return DN_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    if (tokens > 0 && (!q || !k || !v || !beta || !o)) return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, g, h0, cu_seqlens, o, ht};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return DN_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (n_seqs == 0) return DN_OK;

    dn::Params p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.cu = cu_seqlens;
    p.o = o; p.ht = ht;
    p.N = n_seqs; p.B = B; p.T = T; p.Nk = Nk; p.Nv = Nv; p.dk = dk; p.dv = dv;
    p.tokens = tokens;
    p.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)dk);
    p.flags = flags;
    if (status_ptr(&p.status) != cudaSuccess) return DN_ERR_CUDA;
    const char *name = "";
    if (dn::recurrent_launch(p, dtype == DN_BF16, (cudaStream_t)stream, &name) != cudaSuccess) return DN_ERR_CUDA;
    t_last_kernel = name;
    return DN_OK;
}

namespace {

// Sizes the backward takes: dk <= 128 (its shared-memory tiles), dv any.
bool bwd_dims_ok(int dk, int dv) { return dim_ok(dk) && dk <= 128 && dim_ok(dv); }

// The backward keeps the fp32 state every 64-token chunk starts from; where
// the forward runs on the tensor cores, that forward's WY slots follow.
size_t bwd_states_bytes(long long tokens, int n_seqs, int Nv, int dk, int dv) {
    return (size_t)(tokens / dn::kChunk + n_seqs) * (size_t)Nv * (size_t)dk * (size_t)dv * 4u;
}

// Where the backward's forward pass runs on the tensor cores, its WY slots
// follow the states, then the fp32 matrices that WY kernel also keeps for the
// reverse walk (Params::wyx): three 64 x 64 per chunk and value head.
size_t bwd_wyx_bytes(long long tokens, int n_seqs, int Nv) {
    return (size_t)(tokens / dn::kChunk + n_seqs) * (size_t)Nv * 3u * 64u * 64u * 4u;
}

size_t bwd_workspace_bytes(long long tokens, int n_seqs, int Nv, int dk, int dv, dn_dtype dtype) {
    size_t b = bwd_states_bytes(tokens, n_seqs, Nv, dk, dv);
    if (use_tc(tokens, dk, dv, dtype, dn::kChunk))
        b += dn::tc_workspace_bytes(tokens, n_seqs, Nv, dk, dn::kChunk) + bwd_wyx_bytes(tokens, n_seqs, Nv);
    return b;
}

}  // namespace

DN_EXPORT size_t dn_chunk_bwd_workspace_bytes(int n_seqs, int B, int T, int Nk, int Nv, int dk, int dv,
                                              dn_dtype dtype) {
    if (n_seqs <= 0 || B < 0 || T < 0 || Nk <= 0 || Nv <= 0) return 0;
    if (dtype != DN_BF16 && dtype != DN_F32) return 0;
    if (!bwd_dims_ok(dk, dv)) return 0;
    return bwd_workspace_bytes((long long)B * T, n_seqs, Nv, dk, dv, dtype);
}

DN_EXPORT dn_status dn_chunk_bwd(const void *q, const void *k, const void *v,
                                 const float *beta, const float *g, const float *h0,
                                 const int64_t *cu_seqlens, int n_seqs,
                                 int B, int T, int Nk, int Nv, int dk, int dv,
                                 dn_dtype dtype, float scale, unsigned flags,
                                 const void *d_o, const float *d_ht,
                                 float *d_q, float *d_k, float *d_v, float *d_beta, float *d_g,
                                 float *d_h0, void *workspace, size_t workspace_bytes_,
                                 dn_stream_t stream) {
    if (dtype != DN_BF16 && dtype != DN_F32) return DN_ERR_INVALID_ARG;
    if (n_seqs < 0 || B < 0 || T < 0 || Nk <= 0 || Nv <= 0 || dk <= 0 || dv <= 0)
        return DN_ERR_INVALID_ARG;
    if (Nv % Nk != 0) return DN_ERR_INVALID_ARG;
    if (cu_seqlens ? B != 1 : n_seqs != B) return DN_ERR_INVALID_ARG;
    if (isnan(scale) || isinf(scale)) return DN_ERR_INVALID_ARG;
    if (!flags_ok(flags)) return DN_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    if (tokens > 0 && (!q || !k || !v || !beta || !d_o || !d_q || !d_k || !d_v || !d_beta))
        return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, g, h0, cu_seqlens, d_o, d_ht, d_q, d_k, d_v, d_beta, d_g, d_h0};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return DN_ERR_INVALID_ARG;
    if (!bwd_dims_ok(dk, dv)) return DN_ERR_UNSUPPORTED;
    if (n_seqs == 0) return DN_OK;
    const size_t ws_need = bwd_workspace_bytes(tokens, n_seqs, Nv, dk, dv, dtype);
    if (!workspace || !aligned16(workspace) || workspace_bytes_ < ws_need) return DN_ERR_INVALID_ARG;

    dn::Params p{};
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.cu = cu_seqlens;
    p.N = n_seqs; p.B = B; p.T = T; p.Nk = Nk; p.Nv = Nv; p.dk = dk; p.dv = dv;
    p.tokens = tokens;
    p.scale = scale > 0.0f ? scale : 1.0f / sqrtf((float)dk);
    p.nslots = tokens / dn::kChunk + n_seqs;
    p.chunk = dn::kChunk;
    p.flags = flags;
    p.hs = static_cast<float *>(workspace);
    if (use_tc(tokens, dk, dv, dtype, dn::kChunk)) {
        p.ws = static_cast<uint8_t *>(workspace) + bwd_states_bytes(tokens, n_seqs, Nv, dk, dv);
        p.wyx = reinterpret_cast<float *>(static_cast<uint8_t *>(p.ws) +
                                          dn::tc_workspace_bytes(tokens, n_seqs, Nv, dk, dn::kChunk));
    }
    p.dout = d_o; p.dht = d_ht;
    p.dq = d_q; p.dkk = d_k; p.dvv = d_v; p.dbeta = d_beta; p.dg = d_g; p.dh0 = d_h0;
    if (status_ptr(&p.status) != cudaSuccess) return DN_ERR_CUDA;
    const char *name = "";
    if (dn::bwd_launch(p, dtype == DN_BF16, (cudaStream_t)stream, &name) != cudaSuccess) return DN_ERR_CUDA;
    t_last_kernel = name;
    return DN_OK;
}

DN_EXPORT dn_status dn_check(dn_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DN_ERR_CUDA;
    unsigned *dptr = nullptr;
    if (status_ptr(&dptr) != cudaSuccess) return DN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, dptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DN_ERR_CUDA;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpy(dptr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return DN_ERR_CUDA;
    }
    if (word & dn::kStatusTimeout) return DN_ERR_TIMEOUT;
    if (word & dn::kStatusBadSeq) return DN_ERR_DEVICE_ARG;
    return DN_OK;
}

DN_EXPORT const char *dn_status_str(dn_status status) {
    switch (status) {
        case DN_OK: return "DN_OK";
        case DN_ERR_INVALID_ARG: return "DN_ERR_INVALID_ARG";
        case DN_ERR_UNSUPPORTED: return "DN_ERR_UNSUPPORTED";
        case DN_ERR_CUDA: return "DN_ERR_CUDA";
        case DN_ERR_TIMEOUT: return "DN_ERR_TIMEOUT";
        case DN_ERR_DEVICE_ARG: return "DN_ERR_DEVICE_ARG";
    }
    return "DN_ERR_UNKNOWN";
}

DN_EXPORT const char *dn_last_kernel(void) { return t_last_kernel; }

#ifdef DN_TEST_STALL
// Exported only by the failure-path test build (-DDN_TEST_STALL), never by
// the library's own build: arm a stall for the next dn_chunk_fwd call.
DN_EXPORT void dn_test_stall_next(unsigned mode) { t_test_stall = mode; }
#endif
