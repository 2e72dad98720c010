// WY kernel of the chunkwise gated delta rule forward (bf16 q/k, dk = 128):
// for every chunk of every (sequence, value head), the lower-triangular
// inverse T = (I - A)^-1 of the chunk's WY representation and the chunk's
// causal score matrix, written to the workspace as the three bf16 MMA
// operands T' = T diag(beta e^G) and T'' = T diag(beta) (which give
// W = T' K and U = T'' V) and P = tril(scale QK^T . D).
//
// Sources: [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现"
//                 §2.3 (A = -tril(diag(beta) K K^T, -1), T = (I - A)^-1 by
//                 forward substitution), §2.4 (W = T diag(beta) K, U = T diag(beta) V,
//                 intra-chunk output through tril(Q K^T));
//          [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.2 (gated form:
//                 A_ij and P_ij carry e^{G_i - G_j}, W carries e^{G}).
//
// Every chunk is independent, so this kernel runs all of them in parallel
// ahead of the sequential scan kernel, which then only reads T', T'' and P.
// 128-thread CTAs (one worker of dn_wy_item.cuh each), 36 KB of shared
// memory and 64 TMEM columns each, 6 per SM, as many as fit on the GPU at
// once; each loops over (64-token tile, value head) items, so the TMEM
// allocation and barrier setup are paid once per CTA, not per item.  Per item:
//   1. TMA brings the chunk's K and Q (64 x 128 bf16 each, as two
//      128-byte-swizzled column halves); warp 0 computes the gate scalars;
//   2. one tcgen05 MMA chain computes [K; Q] K^T into tensor memory: lanes
//      0-63 hold K K^T, lanes 64-127 hold Q K^T;
//   3. warps 0-1 turn their rows into A_ij = -beta_i e^{G_i - G_j} (K K^T)_ij
//      (j < i) in shared memory, fp32; warps 2-3 turn theirs into
//      P_ij = scale e^{G_i - G_j} (Q K^T)_ij (j <= i), bf16;
//   4. the four warps invert I - A (blocked, below: fp32 forward substitution
//      on the diagonal blocks, TF32 tensor-core products for the rest);
//   5. T' and T'' are scaled and rounded to bf16; each thread stores its rows
//      of the three images straight from registers into the chunk's slot.
// Waits are bounded: a wait that runs out records kStatusTimeout in the status
// word, the CTA skips the rest and drains its own TMA / MMA work before it
// frees its tensor memory.
#include <atomic>

#include "dn_wy_item.cuh"

namespace dn {
namespace {

// QKN: in-kernel q / k normalisation (kQkL2Norm); a template parameter so
// that the plain instantiation carries none of its registers.  CTAs per SM:
// dk = 128: 6 (80 registers x 128 threads x 6 fit the register file, 36 KB
// of shared memory each); dk = 256: 3 (67 KB of shared memory each).
template <int DKW>
constexpr int wy_ctas_per_sm() { return DKW == 128 ? 6 : 3; }

// BWD (dk = 128, the backward's forward pass): also keep the fp32 rows of
// -(K K^T . D), P and T in Params::wyx for the backward's reverse walk.
// SUB: chunks of 16 or 32 tokens, several per 64-token tile (never with BWD,
// whose forward pass runs 64-token chunks).
template <int DKW, bool QKN, bool BWD, bool SUB>
__global__ void __launch_bounds__(wy::NT, wy_ctas_per_sm<DKW>())
wy_fwd(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
       const __grid_constant__ Params p) {
    using Y = wy::Lay<DKW>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (base - raw);
    wy::Group g{base, gb, 0u, 1u, (int)threadIdx.x, 0u};
    wy::group_init<DKW>(g);
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(base + Y::OFF_BAR + 16, Y::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    g.tm = *reinterpret_cast<volatile uint32_t *>(gb + Y::OFF_BAR + 16);

    // items, one per (64-token tile, value head) (< 2^31, checked at launch),
    // in steps of the grid; each item's gates are loaded during the item before
    const unsigned items = (unsigned)(wy::tile_count(p) * p.Nv), nv = (unsigned)p.Nv;
    ChunkGates gates{0.f, 0.f, 0.f, 0.f};
    if (threadIdx.x < 32 && blockIdx.x < items)
        gates = wy::item_gates(p, blockIdx.x / nv, (int)(blockIdx.x % nv), threadIdx.x);
    for (unsigned it = blockIdx.x; it < items; it += gridDim.x) {
        const unsigned nx = it + gridDim.x;
        const wy::ItemLoc loc = wy::locate(p, it / nv);
        if (!wy::item<DKW, QKN, BWD, SUB>(g, &mK, &mQ, p, it / nv, (int)(it % nv), loc, gates,
                                nx < items ? (long long)(nx / nv) : -1, (int)(nx % nv)))
            break;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(g.tm, Y::TM_COLS);
    }
    // the scan kernel may start: it reads this grid's slots only after
    // waiting for its completion
    ptx::grid_dep_launch();
}

template <int DKW>
cudaError_t wy_launch_dk(const Params &p, const CUtensorMap &mK, const CUtensorMap &mQ, cudaStream_t stream,
                         unsigned items) {
    const uint32_t smem = wy::Lay<DKW>::GROUP_BYTES + 1024;
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    const bool bwd = DKW == 128 && p.wyx != nullptr;
    const bool sub = p.chunk < kChunk;
    if (bwd && sub) return cudaErrorInvalidValue;
    const void *kern = qkn ? (bwd ? (const void *)wy_fwd<DKW, true, DKW == 128, false>
                                  : (sub ? (const void *)wy_fwd<DKW, true, false, true> : (const void *)wy_fwd<DKW, true, false, false>))
                           : (bwd ? (const void *)wy_fwd<DKW, false, DKW == 128, false>
                                  : (sub ? (const void *)wy_fwd<DKW, false, false, true> : (const void *)wy_fwd<DKW, false, false, false>));
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    // one resident wave of CTAs (per device, head size and instantiation,
    // looked up once); on 2048 items (B = 4, H = 16, T = 2048, dk = 128) it
    // measured 1.5 us faster per forward than one CTA per item
    static std::atomic<int> wave_cache[64][4];  // 0: not looked up yet (calls may come from several threads)
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    const int ci = 2 * (int)qkn + (int)bwd;
    int wave = (dev >= 0 && dev < 64) ? wave_cache[dev][ci].load(std::memory_order_relaxed) : 0;
    if (wave <= 0) {
        // CTAs per SM: the launch bound, or fewer if shared memory runs out
        // (the occupancy query reports fewer under the default carveout)
        int sms = 0, smem_sm = 0, reserved = 0;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return err;
        if ((err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
            return err;
        int per_sm = smem_sm / (int)(smem + (uint32_t)reserved);
        if (per_sm > wy_ctas_per_sm<DKW>()) per_sm = wy_ctas_per_sm<DKW>();
        wave = sms * (per_sm > 0 ? per_sm : 1);
        if (dev >= 0 && dev < 64) wave_cache[dev][ci].store(wave, std::memory_order_relaxed);
    }
    const unsigned grid = items < (unsigned)wave ? items : (unsigned)wave;
    void *args[] = {const_cast<CUtensorMap *>(&mK), const_cast<CUtensorMap *>(&mQ), const_cast<Params *>(&p)};
    if ((err = cudaLaunchKernel(kern, dim3(grid), dim3(wy::NT), args, smem, stream)) != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t wy_launch(const Params &p, const CUtensorMap &mK, const CUtensorMap &mQ, cudaStream_t stream) {
    const long long items = wy::tile_count(p) * p.Nv;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (p.dk == 128) return wy_launch_dk<128>(p, mK, mQ, stream, (unsigned)items);
    if (p.dk == 256) return wy_launch_dk<256>(p, mK, mQ, stream, (unsigned)items);
    return cudaErrorInvalidValue;
}

}  // namespace dn
