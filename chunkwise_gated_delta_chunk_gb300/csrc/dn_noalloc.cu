// dn_chunk_fwd_noalloc: the forward with its scratch space in a fixed device
// array of this library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run the forward.  Examples are plugin-style hosts whose execute path is
// forbidden to allocate (the host owns every device buffer and hands out only
// inputs and outputs), and runtimes that reserved all device memory for their
// own pool up front, where a cudaMalloc would fail or would synchronize the
// device in the middle of a latency-critical path.  Such a caller passes its
// inputs and outputs only; the T' | T'' slots the tensor-core path keeps
// between its two kernels live in g_noalloc_scratch below.
//
// The array is kNoAllocScratchBytes (64 MiB) of device memory.  The device
// copy of this file's module is made when the module is first used on a GPU:
// with CUDA's default lazy module loading that is the first
// dn_chunk_fwd_noalloc call on that GPU (its symbol lookup), which therefore
// reserves the 64 MiB and can fail with DN_ERR_CUDA if the device memory is
// already taken.  Callers make one call at set-up time, before they commit
// the rest of the device memory; later calls reserve nothing more, and the
// array is held until the process exits.
// Nothing in it has to start at zero: every slot a call reads was written by
// the same call.  All calls share it, so two calls whose kernels overlap on
// the GPU (different streams, or different host threads on one device) race
// on it; calls in one stream are ordered and safe.
#include <mutex>

#include "dn_chunk_fwd.h"
#include "dn_internal.h"

#define DN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)DN_NOALLOC_SCRATCH_BYTES;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call made with that device current (a host query; it allocates
// nothing).
cudaError_t scratch_ptr(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

DN_EXPORT dn_status dn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                         const float *beta, const float *g, const float *h0,
                                         const int64_t *cu_seqlens, int n_seqs,
                                         int B, int T, int Nk, int Nv, int dk, int dv,
                                         dn_dtype dtype, float scale, unsigned flags, int chunk,
                                         void *o, float *ht, dn_stream_t stream) {
    // the same argument checks as dn_chunk_fwd first, so a bad argument is
    // reported as such whatever the sizes
    const dn_status args = dn::chunk_fwd_check_args(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv,
                                                    dk, dv, dtype, scale, flags, chunk, o, ht);
    if (args != DN_OK) return args;
    const size_t need = dn_chunk_fwd_workspace_bytes(n_seqs, B, T, Nk, Nv, dk, dv, dtype, chunk);
    if (need > kNoAllocScratchBytes) return DN_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (need > 0 && scratch_ptr(&ws) != cudaSuccess) return DN_ERR_CUDA;
    return dn_chunk_fwd(q, k, v, beta, g, h0, cu_seqlens, n_seqs, B, T, Nk, Nv, dk, dv, dtype, scale,
                        flags, chunk, o, ht, ws, need > 0 ? kNoAllocScratchBytes : 0, stream);
}
