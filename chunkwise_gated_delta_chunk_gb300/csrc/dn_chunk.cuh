// Per-chunk pieces shared by the WY kernel (T of every chunk) and the scan
// kernel: sequence bounds, the workspace slot of a chunk and the gate scalars.
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1 (gate
//          prefix sum G and the decay matrix D_ij = e^{G_i - G_j});
//          [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §2.4.
#pragma once

#include "dn_internal.h"
#include "dn_order.cuh"

namespace dn {

// Scalars of one chunk (floats within a scalar block): G, beta, beta e^G,
// e^{G_L - G} (zero past the chunk's length), scale e^G, the decay factors
// e^{G_i - G_0} and e^{G_0 - G_j}, alpha = e^{G_L}, L, and whether the factors
// may be used (the chunk's log-gate span is at most kSpanMax).
constexpr int SC_G = 0, SC_BETA = 64, SC_BEG = 128, SC_DEC = 192, SC_OSC = 256, SC_AF = 320,
              SC_BF = 384, SC_ALPHA = 448, SC_L = 449, SC_FACT = 450;
constexpr int SCAL_FLOATS = 512;
constexpr float kSpanMax = 80.f;

// One workspace slot of the tensor-core path holds a chunk's per-chunk
// operands for one value head, each a bf16 matrix stored as the
// 128-byte-swizzled image the MMAs read (row i at 128 i, 16-byte chunk c at
// (c ^ (i & 7)) * 16):
//   dk = 128: T' = T diag(beta e^G) (64 x 64), then T'' and P;
//   dk = 256: -W = -T' K (64 x 256, as four 64-column quarters of 8 KB),
//             then T'' and P;
// with T'' = T diag(beta) and P = tril(scale QK^T . D) (64 x 64 each); then,
// with kQkL2Norm, the fp32 factors 1 / max(||k_i||, 1e-12) and
// 1 / max(||q_i||, 1e-12) of the chunk's 64 rows (the WY kernel folds them
// into T', W and P; the scan kernel folds them into its per-token factors).
constexpr uint32_t kImageBytes = 8192;
__host__ __device__ constexpr uint32_t slot_tu_off(int dk) { return dk == 256 ? 32768u : kImageBytes; }
__host__ __device__ constexpr uint32_t slot_p_off(int dk) { return slot_tu_off(dk) + kImageBytes; }
__host__ __device__ constexpr uint32_t slot_norm_off(int dk) { return slot_p_off(dk) + kImageBytes; }
__host__ __device__ constexpr uint32_t slot_bytes(int dk) { return slot_norm_off(dk) + 2 * 64 * 4; }
constexpr uint32_t kSlotNormOff = slot_norm_off(128);  // 64 key factors, then 64 query factors
constexpr uint32_t kSlotBytes = slot_bytes(128);

__device__ __forceinline__ long long seq_bos(const Params &p, int n) {
    return p.cu ? p.cu[n] : (long long)n * p.T;
}

__device__ __forceinline__ long long seq_eos(const Params &p, int n) {
    return p.cu ? p.cu[n + 1] : (long long)(n + 1) * p.T;
}

// Workspace slot of the chunk that starts at token t0 of sequence n, for
// chunks of `chunk` tokens.  With non-decreasing offsets, floor(t0 / chunk) + n
// is one-to-one over every chunk of every sequence and stays below
// floor(tokens / chunk) + N.
// (chunk is a power of two on every path that has slots.)
__device__ __forceinline__ long long wy_slot(long long t0, int n, int chunk) { return (t0 >> (__ffs(chunk) - 1)) + n; }

// Gate scalars of one chunk, per lane (tokens lane and lane + 32).
struct ChunkScalars {
    float ga, gb, ba, bb;      // G and beta of the lane's two tokens
    float GL, G0, span;        // G at the last token and at the first, max - min of G
    float ka, kb, qa, qb;      // inverse key / query norms of the two tokens (1: no normalisation)
    int L;
};

// The raw gates and betas of a chunk's tokens lane and lane + 32 (one warp),
// loaded ahead of their use.  Tokens past L get beta = 0 and g = 0, so they
// write nothing and decay nothing.
struct ChunkGates {
    float ga, gb, ba, bb;
};

__device__ __forceinline__ ChunkGates chunk_gates_load(const Params &p, int h, long long t0, int L, int lane) {
    ChunkGates r{0.f, 0.f, 0.f, 0.f};
    if (lane < L) {
        r.ba = p.beta[(t0 + lane) * p.Nv + h];
        if (p.g) r.ga = p.g[(t0 + lane) * p.Nv + h];
    }
    if (lane + 32 < L) {
        r.bb = p.beta[(t0 + lane + 32) * p.Nv + h];
        if (p.g) r.gb = p.g[(t0 + lane + 32) * p.Nv + h];
    }
    return r;
}

// Prefix-sums the gates of the chunk [t0, t0 + L) (one warp).
__device__ __forceinline__ ChunkScalars chunk_scalars_from(const ChunkGates &in, int L, int lane) {
    ChunkScalars r;
    float ga = in.ga, gb = in.gb;
    const float ba = in.ba, bb = in.bb;
    // inclusive prefix sums G_i = g_0 + ... + g_i
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ta = __shfl_up_sync(0xffffffffu, ga, off);
        const float tb = __shfl_up_sync(0xffffffffu, gb, off);
        if (lane >= off) {
            ga += ta;
            gb += tb;
        }
    }
    gb += __shfl_sync(0xffffffffu, ga, 31);
    const float GLa = __shfl_sync(0xffffffffu, ga, (L - 1) & 31);
    const float GLb = __shfl_sync(0xffffffffu, gb, (L - 1) & 31);
    r.GL = (L - 1) < 32 ? GLa : GLb;
    r.G0 = __shfl_sync(0xffffffffu, ga, 0);
    float gmax = fmaxf(ga, gb), gmin = fminf(ga, gb);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
        gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, off));
    }
    r.span = gmax - gmin;
    r.ga = ga;
    r.gb = gb;
    r.ba = ba;
    r.bb = bb;
    r.ka = r.kb = r.qa = r.qb = 1.f;
    r.L = L;
    return r;
}

// The chunk's inverse key and query norms from the factors in its workspace
// slot (written by the WY kernel), for the lane's two tokens.
__device__ __forceinline__ void chunk_norms_load(ChunkScalars &r, const uint8_t *norms, int lane) {
    const float *f = reinterpret_cast<const float *>(norms);
    r.ka = f[lane];
    r.kb = f[lane + 32];
    r.qa = f[64 + lane];
    r.qb = f[64 + lane + 32];
}

// Writes the scalar block of a chunk (see the SC_ offsets) into `sc`.  The
// inverse norms, where set, ride on e^{G_L - G_i} (which multiplies k_i's
// contribution to the state) and on scale e^{G_i} (which multiplies q_i).
__device__ __forceinline__ void chunk_scalars_store(const Params &p, const ChunkScalars &r, float *sc, int lane) {
    const int ia = lane, ib = lane + 32;
    sc[SC_G + ia] = r.ga;
    sc[SC_G + ib] = r.gb;
    sc[SC_BETA + ia] = r.ba;
    sc[SC_BETA + ib] = r.bb;
    sc[SC_BEG + ia] = r.ba * __expf(r.ga);
    sc[SC_BEG + ib] = r.bb * __expf(r.gb);
    sc[SC_DEC + ia] = ia < r.L ? __expf(r.GL - r.ga) * r.ka : 0.f;
    sc[SC_DEC + ib] = ib < r.L ? __expf(r.GL - r.gb) * r.kb : 0.f;
    sc[SC_OSC + ia] = p.scale * __expf(r.ga) * r.qa;
    sc[SC_OSC + ib] = p.scale * __expf(r.gb) * r.qb;
    // e^{G_i - G_j} = e^{G_i - G_0} e^{G_0 - G_j} is safe when the chunk's
    // log-gate span is small enough that neither factor leaves fp32 range
    sc[SC_AF + ia] = __expf(r.ga - r.G0);
    sc[SC_AF + ib] = __expf(r.gb - r.G0);
    sc[SC_BF + ia] = __expf(r.G0 - r.ga);
    sc[SC_BF + ib] = __expf(r.G0 - r.gb);
    if (lane == 0) {
        sc[SC_ALPHA] = __expf(r.GL);
        sc[SC_L] = __int_as_float(r.L);
        sc[SC_FACT] = (r.span <= kSpanMax) ? 1.f : 0.f;
    }
}

// The scan kernels keep the state in tensor memory unscaled: acc_s holds
// S_c / A_c, where A_c is the product of the decays alpha = e^{G_L} of the
// chunks since the last renormalisation.  A chunk whose decay keeps
// alpha_c A_c within [2^-40, 2^40] needs no pass over acc_s: A_{c+1} =
// alpha_c A_c, and v~ is divided by A_{c+1} before DS accumulates it (the
// factor rides on e^{G_L - G_i}).  Otherwise (strong decay, or alpha = 0) the
// chunk renormalises: acc_s is scaled by alpha_c A_c before DS(c) and
// A_{c+1} = 1.  The bf16 image of the state is A_c acc_s and ht =
// A acc_s, so every product sees S itself.  The loader tracks A; the scalar
// block of chunk c then also holds:
constexpr int SC_A = 452;   // A_c
constexpr int SC_RN = 453;  // 1: renormalise before DS(c)
constexpr int SC_RS = 454;  // alpha_c A_c, the renormalising scale
constexpr int SC_AN = 455;  // A_{c+1}
static_assert(SC_A > SC_FACT && SC_AN < SCAL_FLOATS, "free scalar slots");
constexpr float kAMin = 0x1p-40f, kAMax = 0x1p40f;

struct ChunkDecay {
    float A, rs, an;
    bool rn;
};

// The decay bookkeeping of a chunk whose G at its last token is GL, entered
// with A = A_c (every lane computes the same).
__device__ __forceinline__ ChunkDecay chunk_decay(float GL, float A) {
    ChunkDecay d;
    d.A = A;
    d.rs = __expf(GL) * A;
    d.rn = !(d.rs >= kAMin && d.rs <= kAMax);
    d.an = d.rn ? 1.f : d.rs;
    return d;
}

__device__ __forceinline__ void chunk_decay_store(float *sc, const ChunkDecay &d) {
    sc[SC_A] = d.A;
    sc[SC_RN] = d.rn ? 1.f : 0.f;
    sc[SC_RS] = d.rs;
    sc[SC_AN] = d.an;
}

// Loads and prefix-sums the gates of the chunk [t0, t0 + L) of value head h
// (one warp).
__device__ __forceinline__ ChunkScalars chunk_scalars_load(const Params &p, int h, long long t0, int L, int lane) {
    return chunk_scalars_from(chunk_gates_load(p, h, t0, L, lane), L, lane);
}

// Gate scalars of the chunk [t0, t0 + L) of value head h, computed by one
// warp into `sc`.
__device__ __forceinline__ void chunk_scalars(const Params &p, int h, long long t0, int L, float *sc,
                                              int lane) {
    chunk_scalars_store(p, chunk_scalars_load(p, h, t0, L, lane), sc, lane);
}

}  // namespace dn
