// Tensor-core (tcgen05 / TMEM / TMA) kernel of the chunkwise gated delta rule
// forward, bf16 q/k/v/o, dk = 128, 128 value columns per CTA.
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.3;
//          [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §2.3-§3.4.
//
// One persistent CTA per (sequence, value head, 128-column value tile) walks
// the sequence's 64-token chunks in order.  The fp32 state lives in tensor
// memory, transposed (lane = value column v, column = key index d), for the
// whole sequence.  Every contraction is a tcgen05 MMA with M = 128:
//
//   KQ  [K;Q] K^T        -> KK^T and QK^T        (a2, a6)
//   W   K^T T'^T         -> W^T, T' = T diag(beta e^G)          (a4)
//   U   V^T T''^T        -> U^T, T'' = T diag(beta)             (a4)
//   VN  U^T - S^T W^T    -> v_new^T (S^T as a bf16 TMEM operand) (a5)
//   O   S^T Q^T          -> inter-chunk output                   (a6)
//   DS  S^T += v~^T K    -> state update, v~ = e^{G_L-G} v_new   (a5)
//   PV  v_new^T P^T      -> intra-chunk output, P = tril(QK^T.D) (a6)
//
// Warp roles (14 warps; warp w reaches TMEM lanes 32 (w % 4) .. +31, so each
// group of four consecutive warps covers all 128 lanes):
//   0      loader: TMA for the K, Q, V tiles of a chunk and the gate scalars
//          (prefix sum G, e^G, decays) computed with warp shuffles;
//   1      chain MMA issuer (one thread: VN, O, DS, PV) and TMEM owner;
//   2-5    prep: A and P from KK^T / QK^T, T = (I - A)^-1 (16x16 diagonal
//          blocks by forward substitution, then block rows with TF32 mma.sync),
//          T' and T'', then W^T from TMEM to a bf16 operand.  One of its
//          threads issues the prep MMAs (KQ of the next chunk as soon as this
//          chunk's is read, W and U once T is ready), so the prep runs ahead
//          of the state scan;
//   6-9    state: v_new and v~ operands, the fp32 state update, ht;
//   10-13  output: o = scale e^{G} (S^T Q^T) + P v_new, stored as bf16.
//
// Every wait is bounded: after kTimeoutNs a CTA records kStatusTimeout in the
// status word, raises a shared abort flag so the other roles stop too, drains
// its own outstanding TMA and MMA work and frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "dn_internal.h"
#include "dn_tc.h"
#include "dn_tmap.h"
#include "tc_ptx.cuh"

// Optional per-chunk event trace of CTA 0 (SM clock), compiled in only with
// -DDN_TRACE for profiling builds; the default build contains no trace code.
#ifdef DN_TRACE
__device__ unsigned long long g_dn_trace[14][1024][16];
#define DN_TRACE_EV(ev, c)                                                    \
    do {                                                                      \
        if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (c) < 1024)         \
            g_dn_trace[threadIdx.x >> 5][(c)][(ev)] = clock64();              \
    } while (0)
extern "C" __attribute__((visibility("default"))) int dn_trace_dump(void *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_dn_trace, sizeof(g_dn_trace));
}
#else
#define DN_TRACE_EV(ev, c) \
    do {                   \
    } while (0)
#endif

namespace dn {
namespace {

using namespace ptx;

constexpr int C = kChunk;      // 64
constexpr int DK = 128;
constexpr int BVT = 128;       // value columns per CTA
constexpr int NS = 3;          // pipeline stages of K/Q/V tiles
constexpr int NTHREADS = 448;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s

// ---- shared memory map (offsets from a 1024-byte aligned base) -------------
constexpr uint32_t STAGE_BYTES = 49152;  // K0 Q0 K1 Q1 V0 V1, 8 KB each
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_P = OFF_STAGE + NS * STAGE_BYTES;  // 2 x 8 KB (double buffered)
constexpr uint32_t OFF_TP = OFF_P + 2 * 8192;              // T'  8 KB
constexpr uint32_t OFF_TPP = OFF_TP + 8192;                // T'' 8 KB
constexpr uint32_t OFF_WT = OFF_TPP + 8192;                // -W^T 16 KB
constexpr int LDA = 68;                                    // fp32 row stride of A / T
constexpr uint32_t OFF_A = OFF_WT + 16384;                 // 64 x 68 fp32
constexpr int SCAL_FLOATS = 512;
constexpr uint32_t OFF_SCAL = OFF_A + 64 * LDA * 4;        // NS x 2048 B
constexpr uint32_t OFF_BAR = OFF_SCAL + NS * SCAL_FLOATS * 4;
constexpr int NBARS = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;         // TMEM base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;          // alignment slack

static_assert(OFF_P % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_TPP % 1024 == 0 && OFF_WT % 1024 == 0,
              "MMA operands need 1024-byte aligned swizzle atoms");
static_assert(SMEM_ALLOC <= 232448, "exceeds the 227 KB of shared memory per CTA");

// Scalars of one chunk (floats within a stage's scalar block): G, beta,
// beta e^G, e^{G_L - G}, scale e^G, the decay factors e^{G_i - G_0} and
// e^{G_0 - G_j}, alpha = e^{G_L}, L, and whether the factors may be used
// (the chunk's log-gate span is at most kSpanMax).
constexpr int SC_G = 0, SC_BETA = 64, SC_BEG = 128, SC_DEC = 192, SC_OSC = 256, SC_AF = 320,
              SC_BF = 384, SC_ALPHA = 448, SC_L = 449, SC_FACT = 450;
constexpr float kSpanMax = 80.f;

// Barrier indices.
enum {
    B_FULL = 0,                 // NS: TMA bytes + loader scalars
    B_EMPTY = B_FULL + NS,      // NS: every reader of the stage is done
    B_KQ_FULL = B_EMPTY + NS,   // KK^T / QK^T of a chunk in acc_kq
    B_WU_FULL,                  // W^T in acc_w and U^T in acc_v
    B_WSM_FULL,                 // -W^T bf16 operand in shared memory
    B_S_FULL,
    B_V_FULL,
    B_VSM_FULL,
    B_D_FULL,
    B_O_EMPTY,
    B_DRAIN,
    B_DRAIN2,
    B_COUNT
};
static_assert(B_COUNT <= NBARS, "barrier space");

// Tensor memory columns (fp32 accumulators; SB holds bf16 pairs).
constexpr uint32_t TM_KQ = 0, TM_W = 64, TM_V = 128, TM_S = 192, TM_SB = 320, TM_O = 384,
                   TM_P = 448, TM_COLS = 512;

// Instruction descriptors.
constexpr uint32_t ID_KQ = idesc_bf16(128, 64, 0, 0);   // A, B K-major
constexpr uint32_t ID_W = idesc_bf16(128, 64, 1, 0);    // A MN-major (K^T), B K-major
constexpr uint32_t ID_U = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_VN = idesc_bf16(128, 64, 0, 1);   // A TMEM, B MN-major (-W^T rows d)
constexpr uint32_t ID_O = idesc_bf16(128, 64, 0, 0);    // A TMEM, B K-major (Q rows)
constexpr uint32_t ID_DS = idesc_bf16(128, 128, 0, 1);  // A TMEM, B MN-major (K rows)
constexpr uint32_t ID_PV = idesc_bf16(128, 64, 0, 0);   // A TMEM, B K-major (P rows)

struct Ctx {
    uint32_t base;     // shared address of the aligned base
    uint8_t *gbase;    // generic pointer to the same
    volatile int *abort_flag;
    unsigned *status;
};

__device__ __forceinline__ uint32_t bar(const Ctx &x, int i) { return x.base + OFF_BAR + 8u * i; }
__device__ __forceinline__ float *scal(const Ctx &x, int s) {
    return reinterpret_cast<float *>(x.gbase + OFF_SCAL + s * SCAL_FLOATS * 4);
}

// Bounded wait.  Returns false once the CTA is aborting.
__device__ __noinline__ bool wait_slow(const Ctx &x, uint32_t b, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
#ifdef DN_WAIT_HINT
        if (mbar_try_wait_sleep(b, parity, DN_WAIT_HINT)) return true;
#else
        if (mbar_try_wait(b, parity)) return true;
#endif
        if ((it & 31u) == 0) {
            if (*x.abort_flag) return false;
            if (globaltimer() - t0 > kTimeoutNs) {
                *x.abort_flag = 1;
                atomicOr(x.status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait(const Ctx &x, uint32_t b, uint32_t parity) {
    if (mbar_try_wait(b, parity)) return true;
    return wait_slow(x, b, parity);
}

// Wait that ignores the abort flag (used while draining); bounded by time.
__device__ __noinline__ void wait_drain(uint32_t b, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(b, parity))
        if (globaltimer() - t0 > kTimeoutNs) return;
}

// Warp-uniform wait: every lane gets the same answer, so lanes never diverge
// around the .sync.aligned tcgen05 instructions and warp syncs that follow.
__device__ __forceinline__ bool wwait(const Ctx &x, uint32_t b, uint32_t parity) {
    const bool ok = wait(x, b, parity);
    return __all_sync(0xffffffffu, ok);
}

// OR of `pred` over the `n` threads of named barrier `id` (also a barrier).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16);
}

__device__ __forceinline__ void warp_arrive(uint32_t b) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(b);
}

struct Unit {
    long long bos, eos;
    int n, h, hk, v0, nc;
};

__device__ __forceinline__ Unit unit_of(const Params &p) {
    Unit u;
    const int nvt = p.dv / BVT;
    const int idx = blockIdx.x;
    const int vt = idx % nvt;
    u.h = (idx / nvt) % p.Nv;
    u.n = idx / (nvt * p.Nv);
    u.hk = u.h / (p.Nv / p.Nk);
    u.v0 = vt * BVT;
    if (p.cu) {
        u.bos = p.cu[u.n];
        u.eos = p.cu[u.n + 1];
        if (u.bos < 0 || u.eos < u.bos || u.eos > p.tokens) {
            if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeq);
            u.bos = u.eos = 0;
        }
    } else {
        u.bos = (long long)u.n * p.T;
        u.eos = u.bos + p.T;
    }
    u.nc = (int)((u.eos - u.bos + C - 1) / C);
    return u;
}

// ---------------------------------------------------------------------------
// Loader warp: TMA tiles + gate scalars of each chunk.
// ---------------------------------------------------------------------------
__device__ void loader_role(const Ctx x, const Params &p, const Unit u, const CUtensorMap *mK,
                            const CUtensorMap *mQ, const CUtensorMap *mV, int &armed_last) {
    const int lane = threadIdx.x & 31;
    armed_last = -1;
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        if (!wwait(x, bar(x, B_EMPTY + s), ((c / NS) & 1) ^ 1)) return;
        DN_TRACE_EV(0, c);
        const long long t0 = u.bos + (long long)c * C;
        const int L = (int)min((long long)C, u.eos - t0);
        const uint32_t st = x.base + OFF_STAGE + s * STAGE_BYTES;
        if (lane == 0) {
            const uint32_t fb = bar(x, B_FULL + s);
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            const int tt = (int)t0;
            tma_load_3d(st + 0, mK, fb, 0, u.hk, tt);
            tma_load_3d(st + 8192, mQ, fb, 0, u.hk, tt);
            tma_load_3d(st + 16384, mK, fb, 64, u.hk, tt);
            tma_load_3d(st + 24576, mQ, fb, 64, u.hk, tt);
            tma_load_3d(st + 32768, mV, fb, u.v0, u.h, tt);
            tma_load_3d(st + 40960, mV, fb, u.v0 + 64, u.h, tt);
        }
        armed_last = c;
        // gate scalars: lane owns tokens lane and lane + 32 of the chunk
        float ga = 0.f, gb = 0.f, ba = 0.f, bb = 0.f;
        if (lane < L) {
            ba = p.beta[(t0 + lane) * p.Nv + u.h];
            if (p.g) ga = p.g[(t0 + lane) * p.Nv + u.h];
        }
        if (lane + 32 < L) {
            bb = p.beta[(t0 + lane + 32) * p.Nv + u.h];
            if (p.g) gb = p.g[(t0 + lane + 32) * p.Nv + u.h];
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float ta = __shfl_up_sync(0xffffffffu, ga, off);
            const float tb = __shfl_up_sync(0xffffffffu, gb, off);
            if (lane >= off) { ga += ta; gb += tb; }
        }
        gb += __shfl_sync(0xffffffffu, ga, 31);
        const float GLa = __shfl_sync(0xffffffffu, ga, (L - 1) & 31);
        const float GLb = __shfl_sync(0xffffffffu, gb, (L - 1) & 31);
        const float GL = (L - 1) < 32 ? GLa : GLb;
        // e^{G_i - G_j} = e^{G_i - G_0} e^{G_0 - G_j} is safe when the chunk's
        // log-gate span is small enough that neither factor leaves fp32 range
        const float G0 = __shfl_sync(0xffffffffu, ga, 0);
        float gmax = fmaxf(ga, gb), gmin = fminf(ga, gb);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
            gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, off));
        }
        float *sc = scal(x, s);
        const int ia = lane, ib = lane + 32;
        sc[SC_G + ia] = ga;
        sc[SC_G + ib] = gb;
        sc[SC_BETA + ia] = ba;
        sc[SC_BETA + ib] = bb;
        sc[SC_BEG + ia] = ba * __expf(ga);
        sc[SC_BEG + ib] = bb * __expf(gb);
        sc[SC_DEC + ia] = ia < L ? __expf(GL - ga) : 0.f;
        sc[SC_DEC + ib] = ib < L ? __expf(GL - gb) : 0.f;
        sc[SC_OSC + ia] = p.scale * __expf(ga);
        sc[SC_OSC + ib] = p.scale * __expf(gb);
        sc[SC_AF + ia] = __expf(ga - G0);
        sc[SC_AF + ib] = __expf(gb - G0);
        sc[SC_BF + ia] = __expf(G0 - ga);
        sc[SC_BF + ib] = __expf(G0 - gb);
        if (lane == 0) {
            sc[SC_ALPHA] = __expf(GL);
            sc[SC_L] = __int_as_float(L);
            sc[SC_FACT] = (gmax - gmin <= kSpanMax) ? 1.f : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(x, B_FULL + s));
        DN_TRACE_EV(1, c);
    }
}

// ---------------------------------------------------------------------------
// MMA issue helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void issue_kq(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a = st + kb * 16384 + kk * 32;
            mma_ss(tm + TM_KQ, sdesc(a, 16, 1024), sdesc(a, 16, 1024), ID_KQ, (kb | kk) != 0);
        }
}

__device__ __forceinline__ void issue_w(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + TM_W, sdesc(st + kk * 2048, 16384, 1024), sdesc(x.base + OFF_TP + kk * 32, 16, 1024),
               ID_W, kk != 0);
}

__device__ __forceinline__ void issue_u(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES + 32768;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + TM_V, sdesc(st + kk * 2048, 8192, 1024), sdesc(x.base + OFF_TPP + kk * 32, 16, 1024),
               ID_U, kk != 0);
}

// ---------------------------------------------------------------------------
// Chain MMA issuer (one thread): the state-dependent contractions only.
// ---------------------------------------------------------------------------
__device__ void mma_role(const Ctx x, const Unit u, uint32_t tm) {
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const uint32_t st = x.base + OFF_STAGE + s * STAGE_BYTES;
        const uint32_t par = c & 1;
        // v_new^T = U^T + S^T (-W^T)   (U^T was written into acc_v by the prep)
        if (!wait(x, bar(x, B_WSM_FULL), par)) break;
        if (!wait(x, bar(x, B_S_FULL), par)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_ts(tm + TM_V, tm + TM_SB + kk * 8, sdesc(x.base + OFF_WT + kk * 2048, 8192, 1024), ID_VN, 1);
        mma_commit(bar(x, B_V_FULL));
        DN_TRACE_EV(0, c);
        // inter-chunk output S^T Q^T
        if (!wait(x, bar(x, B_O_EMPTY), par ^ 1)) break;
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ts(tm + TM_O, tm + TM_SB + kb * 32 + kk * 8,
                       sdesc(st + 8192 + kb * 16384 + kk * 32, 16, 1024), ID_O, (kb | kk) != 0);
        // state update and intra-chunk output
        if (!wait(x, bar(x, B_VSM_FULL), par)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_S, tm + TM_V + 32 + kk * 8, sdesc(st + kk * 2048, 16384, 1024), ID_DS, 1);
        const uint32_t pbuf = x.base + OFF_P + (c & 1) * 8192;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_P, tm + TM_V + kk * 8, sdesc(pbuf + kk * 32, 16, 1024), ID_PV, kk != 0);
        mma_commit(bar(x, B_D_FULL));
        mma_commit(bar(x, B_EMPTY + s));
        DN_TRACE_EV(3, c);
    }
    // every MMA issued by this thread completes before tensor memory is freed
    mma_commit(bar(x, B_DRAIN));
    wait_drain(bar(x, B_DRAIN), 0);
}

// ---------------------------------------------------------------------------
// Prep warpgroup: A, P, T = (I - A)^-1, T', T'', and the prep MMAs (KQ of the
// next chunk, W and U of this one), so the prep runs ahead of the state scan.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t to_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- 16 x 16 block helpers for the solve (fp32 blocks, TF32 mma.sync) -------
// acc (16 x 8 tile, columns n0..n0+7 of the product) += Ab (16 x 16) Bb (16 x 16).
__device__ __forceinline__ void tile_mma(float (&acc)[4], const float *Ab, int lda, const float *Bb,
                                         int ldb, int n0, int g, int t) {
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4], b[2];
        a[0] = to_tf32(Ab[g * lda + 8 * kk + t]);
        a[1] = to_tf32(Ab[(g + 8) * lda + 8 * kk + t]);
        a[2] = to_tf32(Ab[g * lda + 8 * kk + t + 4]);
        a[3] = to_tf32(Ab[(g + 8) * lda + 8 * kk + t + 4]);
        b[0] = to_tf32(Bb[(8 * kk + t) * ldb + n0 + g]);
        b[1] = to_tf32(Bb[(8 * kk + t + 4) * ldb + n0 + g]);
        mma_tf32(acc, a, b);
    }
}

// Same with A = Ab + Ab2 (two blocks of the same layout).
__device__ __forceinline__ void tile_mma_sum(float (&acc)[4], const float *Ab, const float *Ab2, int lda,
                                             const float *Bb, int ldb, int n0, int g, int t) {
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4], b[2];
        a[0] = to_tf32(Ab[g * lda + 8 * kk + t] + Ab2[g * lda + 8 * kk + t]);
        a[1] = to_tf32(Ab[(g + 8) * lda + 8 * kk + t] + Ab2[(g + 8) * lda + 8 * kk + t]);
        a[2] = to_tf32(Ab[g * lda + 8 * kk + t + 4] + Ab2[g * lda + 8 * kk + t + 4]);
        a[3] = to_tf32(Ab[(g + 8) * lda + 8 * kk + t + 4] + Ab2[(g + 8) * lda + 8 * kk + t + 4]);
        b[0] = to_tf32(Bb[(8 * kk + t) * ldb + n0 + g]);
        b[1] = to_tf32(Bb[(8 * kk + t + 4) * ldb + n0 + g]);
        mma_tf32(acc, a, b);
    }
}

__device__ __forceinline__ void tile_load(float (&acc)[4], const float *Cb, int ldc, int n0, int g, int t) {
    acc[0] = Cb[g * ldc + n0 + 2 * t];
    acc[1] = Cb[g * ldc + n0 + 2 * t + 1];
    acc[2] = Cb[(g + 8) * ldc + n0 + 2 * t];
    acc[3] = Cb[(g + 8) * ldc + n0 + 2 * t + 1];
}

__device__ __forceinline__ void tile_store(float *Cb, int ldc, int n0, const float (&acc)[4], int g, int t) {
    Cb[g * ldc + n0 + 2 * t] = acc[0];
    Cb[g * ldc + n0 + 2 * t + 1] = acc[1];
    Cb[(g + 8) * ldc + n0 + 2 * t] = acc[2];
    Cb[(g + 8) * ldc + n0 + 2 * t + 1] = acc[3];
}

// Scratch blocks of the solve (fp32, row stride SLD) in the T'/T'' buffer,
// which is free while T is being computed.
constexpr int SLD = 20, SBLK = 16 * SLD;
enum { XN10, XN20, XN21, XN30, XN31, XN32, XP20, XS31, XS30 };

// In-place T = (I - A)^-1 for the 64 x 64 strictly lower A in sA (row stride
// LDA); 128 threads.  With A_D the four 16 x 16 diagonal blocks and A_O the
// rest, I - A = (I - A_D)(I - N) with N = (I - A_D)^-1 A_O strictly block
// lower, so N^4 = 0 and
//     T = (I + N + N^2 + N^3) T_D,   T_D = (I - A_D)^-1,   N_ij = T_ii A_ij.
// The diagonal blocks are inverted by forward substitution in fp32 (warp pw
// owns block pw, lane l the column l % 16); the products are TF32 tensor-core
// tiles accumulated in fp32, in four barrier-separated phases.
__device__ void solve_T(float *sA, float *scr, int pw, int lane, int c) {
    {
        // x = column `col` of (I - A_bb)^-1:  x_r = [r == col] + sum_{m < r} A[r][m] x_m.
        // Rows of the block are read as float4 (one broadcast wavefront per
        // four elements); four partial sums shorten the dependency chain.
        const int col = lane & 15, o = 16 * pw;
        float xv[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float4 *ar = reinterpret_cast<const float4 *>(sA + (o + r) * LDA + o);
            float p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q4 = 0; q4 < (r + 3) / 4; ++q4) {
                const float4 a = ar[q4];
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q4 + e < r) p4[e] = fmaf(av[e], xv[4 * q4 + e], p4[e]);
            }
            xv[r] = (p4[0] + p4[1]) + (p4[2] + p4[3]) + ((r == col) ? 1.f : 0.f);
        }
        __syncwarp();
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) sA[(o + r) * LDA + o + col] = xv[r];
        }
    }
    named_bar_sync(1, 128);
    DN_TRACE_EV(3, c);
    const int g = lane >> 2, t = lane & 3;
    auto blkA = [&](int i, int j) { return sA + 16 * i * LDA + 16 * j; };
    auto blkX = [&](int k) { return scr + k * SBLK; };
    // phase 1: N_ij = T_ii A_ij, six blocks x two column halves
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const int task = pw + 4 * q, b = task >> 1, n0 = 8 * (task & 1);
        const int bi = (b == 0) ? 1 : (b < 3 ? 2 : 3);
        const int bj = (b == 0) ? 0 : (b < 3 ? b - 1 : b - 3);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(acc, blkA(bi, bi), LDA, blkA(bi, bj), LDA, n0, g, t);
        tile_store(blkX(b), SLD, n0, acc, g, t);
    }
    named_bar_sync(1, 128);
    // phase 2: P20 = N21 N10, S31 = N31 + N32 N21, S30 = N30 + N31 N10 + N32 N20
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int task = pw + 4 * q;
        if (task < 6) {
            const int n0 = 8 * (task & 1);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (task < 2) {
                tile_mma(acc, blkX(XN21), SLD, blkX(XN10), SLD, n0, g, t);
                tile_store(blkX(XP20), SLD, n0, acc, g, t);
            } else if (task < 4) {
                tile_load(acc, blkX(XN31), SLD, n0, g, t);
                tile_mma(acc, blkX(XN32), SLD, blkX(XN21), SLD, n0, g, t);
                tile_store(blkX(XS31), SLD, n0, acc, g, t);
            } else {
                tile_load(acc, blkX(XN30), SLD, n0, g, t);
                tile_mma(acc, blkX(XN31), SLD, blkX(XN10), SLD, n0, g, t);
                tile_mma(acc, blkX(XN32), SLD, blkX(XN20), SLD, n0, g, t);
                tile_store(blkX(XS30), SLD, n0, acc, g, t);
            }
        }
    }
    named_bar_sync(1, 128);
    // phase 3: S30 += N32 P20, and T_ij = S_ij T_jj for every block but (3,0)
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const int task = pw + 4 * q, n0 = 8 * (task & 1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        switch (task >> 1) {
            case 0:
                tile_load(acc, blkX(XS30), SLD, n0, g, t);
                tile_mma(acc, blkX(XN32), SLD, blkX(XP20), SLD, n0, g, t);
                tile_store(blkX(XS30), SLD, n0, acc, g, t);
                break;
            case 1:
                tile_mma(acc, blkX(XN10), SLD, blkA(0, 0), LDA, n0, g, t);
                tile_store(blkA(1, 0), LDA, n0, acc, g, t);
                break;
            case 2:
                tile_mma(acc, blkX(XN21), SLD, blkA(1, 1), LDA, n0, g, t);
                tile_store(blkA(2, 1), LDA, n0, acc, g, t);
                break;
            case 3:
                tile_mma(acc, blkX(XN32), SLD, blkA(2, 2), LDA, n0, g, t);
                tile_store(blkA(3, 2), LDA, n0, acc, g, t);
                break;
            case 4:
                tile_mma(acc, blkX(XS31), SLD, blkA(1, 1), LDA, n0, g, t);
                tile_store(blkA(3, 1), LDA, n0, acc, g, t);
                break;
            default:
                tile_mma_sum(acc, blkX(XN20), blkX(XP20), SLD, blkA(0, 0), LDA, n0, g, t);
                tile_store(blkA(2, 0), LDA, n0, acc, g, t);
                break;
        }
    }
    named_bar_sync(1, 128);
    DN_TRACE_EV(14, c);
    // phase 4: T30 = S30 T00
    if (pw < 2) {
        const int n0 = 8 * pw;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(acc, blkX(XS30), SLD, blkA(0, 0), LDA, n0, g, t);
        tile_store(blkA(3, 0), LDA, n0, acc, g, t);
    }
    named_bar_sync(1, 128);
}

__device__ void prep_role(const Ctx x, const Unit u, uint32_t tm, float scale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pw = warp - 2;                  // 0..3: diagonal block of the solve
    const int row = 32 * (warp & 3) + lane;   // TMEM lane this thread reads
    const bool leader = (pw == 0 && lane == 0);
    float *sA = reinterpret_cast<float *>(x.gbase + OFF_A);
    float *scr = reinterpret_cast<float *>(x.gbase + OFF_TP);  // solve scratch
    const uint32_t lb = lane_base(tm, warp);
    const int i = row & 63;       // row of KK^T (TMEM lanes 0-63) or QK^T (64-127)
    const bool rowA = row < 64;   // KK^T rows -> A (j < i), QK^T rows -> P (j <= i)
    const int ib = i >> 4;
    const int jmax = rowA ? i - 1 : i;
    bool ok = true;
    if (u.nc > 0 && leader) {
        ok = wait(x, bar(x, B_FULL + 0), 0);
        tc_fence_after();
        issue_kq(x, tm, 0);
        mma_commit(bar(x, B_KQ_FULL));
    }
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const uint32_t par = c & 1;
        // A failed wait leaves `ok` false but the chunk body still runs to its
        // end (on garbage), so all four warps meet every named barrier; the
        // group then leaves together.
        ok = ok && wwait(x, bar(x, B_KQ_FULL), par);
        DN_TRACE_EV(0, c);
        tc_fence_after();
        uint32_t r0[32];
        DN_TRACE_EV(8, c);
        ok = ok && wwait(x, bar(x, B_FULL + s), (c / NS) & 1);
        DN_TRACE_EV(9, c);
        const float *sc = scal(x, s);
        const float Gi = sc[SC_G + i], ai = sc[SC_AF + i];
        const bool fact = sc[SC_FACT] != 0.f;  // uniform over the chunk
        const float rs = rowA ? -sc[SC_BETA + i] : scale;
        const uint32_t pb = x.base + OFF_P + (c & 1) * 8192;
        float *arow = sA + i * LDA;
        // D_ij = e^{G_i - G_j} for j <= jmax, else 0: the product of the two
        // per-chunk factors when the chunk's log-gate span allows it, else
        // one exponential per element.
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
            if ((jb & 1) == 0) {  // columns 32 (jb/2) .. +31 of this row
                tmem_ld32(lb + TM_KQ + 16 * jb, r0);
                tmem_wait_ld_dep(r0);
            }
            float dcy[16];
            if (jb > ib) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) dcy[jj] = 0.f;
            } else if (fact) {
                const float4 *b4 = reinterpret_cast<const float4 *>(sc + SC_BF + 16 * jb);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 bb = b4[q4];
                    const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 16 * jb + 4 * q4 + e;
                        dcy[4 * q4 + e] = j <= jmax ? ai * bv[e] : 0.f;
                    }
                }
            } else {
                const float4 *g4 = reinterpret_cast<const float4 *>(sc + SC_G + 16 * jb);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 gg = g4[q4];
                    const float gv[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 16 * jb + 4 * q4 + e;
                        dcy[4 * q4 + e] = __expf(j <= jmax ? Gi - gv[e] : -INFINITY);
                    }
                }
            }
            float val[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int j = 16 * jb + jj;
                val[jj] = rs * dcy[jj] * __uint_as_float(r0[j & 31]);
            }
            if (rowA) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4 *>(arow + 16 * jb + 4 * q4) =
                        make_float4(val[4 * q4], val[4 * q4 + 1], val[4 * q4 + 2], val[4 * q4 + 3]);
            } else {
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8)
                    st_shared_v4(pb + sw128(i, 2 * jb + h8), pack_bf16(val[8 * h8], val[8 * h8 + 1]),
                                 pack_bf16(val[8 * h8 + 2], val[8 * h8 + 3]),
                                 pack_bf16(val[8 * h8 + 4], val[8 * h8 + 5]),
                                 pack_bf16(val[8 * h8 + 6], val[8 * h8 + 7]));
            }
            DN_TRACE_EV(10 + jb, c);
        }
        DN_TRACE_EV(1, c);
        // acc_kq is read by all four warps: the next chunk's KK^T/QK^T may go
        tc_fence_before();
        named_bar_sync(1, 128);
        tc_fence_after();
        DN_TRACE_EV(2, c);
        if (leader && c + 1 < u.nc) {
            ok = ok && wait(x, bar(x, B_FULL + (c + 1) % NS), ((c + 1) / NS) & 1);
            tc_fence_after();
            issue_kq(x, tm, c + 1);
            mma_commit(bar(x, B_KQ_FULL));
        }
        solve_T(sA, scr, pw, lane, c);
        DN_TRACE_EV(4, c);
        // T' = T diag(beta e^G) (KK^T-row threads), T'' = T diag(beta) (others)
        {
            const float *trow = sA + i * LDA;
            const float *cs = sc + (rowA ? SC_BEG : SC_BETA);
            const uint32_t dst = x.base + (rowA ? OFF_TP : OFF_TPP);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float tv[32];
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 a = *reinterpret_cast<const float4 *>(trow + 32 * hf + 4 * q4);
                    const float4 cc = *reinterpret_cast<const float4 *>(cs + 32 * hf + 4 * q4);
                    tv[4 * q4] = a.x * cc.x;
                    tv[4 * q4 + 1] = a.y * cc.y;
                    tv[4 * q4 + 2] = a.z * cc.z;
                    tv[4 * q4 + 3] = a.w * cc.w;
                }
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    st_shared_v4(dst + sw128(i, 4 * hf + ch), pack_bf16(tv[8 * ch], tv[8 * ch + 1]),
                                 pack_bf16(tv[8 * ch + 2], tv[8 * ch + 3]),
                                 pack_bf16(tv[8 * ch + 4], tv[8 * ch + 5]),
                                 pack_bf16(tv[8 * ch + 6], tv[8 * ch + 7]));
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        DN_TRACE_EV(5, c);
        // W^T and U^T of this chunk.  U^T overwrites acc_v, whose previous
        // contents (the chunk before's v_new operands) the chain MMAs read:
        // wait for them.
        if (leader) {
            if (c > 0) ok = ok && wait(x, bar(x, B_D_FULL), (c - 1) & 1);
            tc_fence_after();
            issue_w(x, tm, c);
            issue_u(x, tm, c);
            mma_commit(bar(x, B_WU_FULL));
        }
        warp_arrive(bar(x, B_EMPTY + s));  // done with this chunk's scalars
        ok = ok && wwait(x, bar(x, B_WU_FULL), par);
        DN_TRACE_EV(6, c);
        tc_fence_after();
        {
            // -W^T bf16 operand, row d = this thread's TMEM lane
            const uint32_t dst = x.base + OFF_WT;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                tmem_ld32(lb + TM_W + 32 * hf, r0);
                tmem_wait_ld_dep(r0);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(-__uint_as_float(r0[8 * ch + 2 * e]), -__uint_as_float(r0[8 * ch + 2 * e + 1]));
                    st_shared_v4(dst + sw128(row, 4 * hf + ch), w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_proxy_async_smem();
        warp_arrive(bar(x, B_WSM_FULL));
        DN_TRACE_EV(7, c);
        if (bar_red_or(1, 128, !ok || *x.abort_flag)) break;
    }
    if (leader) {  // prep MMAs complete before tensor memory is freed
        mma_commit(bar(x, B_DRAIN2));
        wait_drain(bar(x, B_DRAIN2), 0);
    }
}

// ---------------------------------------------------------------------------
// State warpgroup: v_new operands, fp32 state, ht.
// ---------------------------------------------------------------------------
__device__ void state_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);  // value column = TMEM lane
    const uint32_t lb = lane_base(tm, warp);
    const size_t sbase = ((size_t)u.n * p.Nv + u.h) * DK * p.dv + u.v0 + v;
    const int dv = p.dv;
    uint32_t r[32], pk[16];

    if (u.nc == 0) {  // empty sequence: ht = h0
        if (p.ht)
            for (int d = 0; d < DK; ++d) p.ht[sbase + (size_t)d * dv] = p.h0 ? p.h0[sbase + (size_t)d * dv] : 0.f;
        return;
    }
    // initial state: acc_s = alpha_0 h0^T, SB = bf16(h0^T)
    if (!wwait(x, bar(x, B_FULL + 0), 0)) return;
    {
        const float alpha = scal(x, 0)[SC_ALPHA];
        for (int blk = 0; blk < 4; ++blk) {
            float f[32];
            const float *hp = p.h0 ? p.h0 + sbase + (size_t)(32 * blk) * dv : nullptr;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                f[k] = hp ? *hp : 0.f;
                if (hp) hp += dv;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(f[2 * k], f[2 * k + 1]);
            tmem_st16(lb + TM_SB + 16 * blk, pk);
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(alpha * f[k]);
            tmem_st32(lb + TM_S + 32 * blk, r);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(x, B_S_FULL));
    }
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const uint32_t par = c & 1;
        // ---- v_new^T and v~^T operands --------------------------------
        // acc_v columns j = 0..63 (fp32) become v_new^T packed in columns
        // 0..31 and v~^T packed in columns 32..63; a column is rewritten only
        // after it has been read.
        if (!wwait(x, bar(x, B_V_FULL), par)) return;
        DN_TRACE_EV(0, c);
        tc_fence_after();
        {
            // quarter qq holds j = 16 qq .. 16 qq + 15 in columns 16 qq ..;
            // v_new^T pairs go to columns 8 qq .., v~^T pairs to 32 + 8 qq ..
            // (each destination column has been read before it is written).
            const float4 *dec4 = reinterpret_cast<const float4 *>(scal(x, s) + SC_DEC);
            uint32_t q16[16], pv8[8], t8[3][8];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                tmem_ld16(lb + TM_V + 16 * qq, q16);
                tmem_wait_ld_dep16(q16);
                uint32_t tq[8];
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 dd = dec4[4 * qq + k4];
                    const float a0 = __uint_as_float(q16[4 * k4]), a1 = __uint_as_float(q16[4 * k4 + 1]);
                    const float a2 = __uint_as_float(q16[4 * k4 + 2]), a3 = __uint_as_float(q16[4 * k4 + 3]);
                    pv8[2 * k4] = pack_bf16(a0, a1);
                    pv8[2 * k4 + 1] = pack_bf16(a2, a3);
                    tq[2 * k4] = pack_bf16(a0 * dd.x, a1 * dd.y);
                    tq[2 * k4 + 1] = pack_bf16(a2 * dd.z, a3 * dd.w);
                }
                tmem_st8(lb + TM_V + 8 * qq, pv8);
                if (qq < 2) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) t8[qq][k] = tq[k];
                } else if (qq == 2) {
                    tmem_st8(lb + TM_V + 32, t8[0]);
                    tmem_st8(lb + TM_V + 40, t8[1]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) t8[2][k] = tq[k];
                } else {
                    tmem_st8(lb + TM_V + 48, t8[2]);
                    tmem_st8(lb + TM_V + 56, tq);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(x, B_VSM_FULL));
            DN_TRACE_EV(1, c);
            warp_arrive(bar(x, B_EMPTY + s));
        }
        // ---- state: S_in(c+1) operand, then pre-scale by alpha(c+1) ------
        if (!wwait(x, bar(x, B_D_FULL), par)) return;
        DN_TRACE_EV(2, c);
        tc_fence_after();
        const bool last = (c + 1 == u.nc);
        for (int blk = 0; blk < 4; ++blk) {
            tmem_ld32(lb + TM_S + 32 * blk, r);
            tmem_wait_ld_dep(r);
            if (!last) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    pk[k] = pack_bf16(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
                tmem_st16(lb + TM_SB + 16 * blk, pk);
            } else if (p.ht) {
                float *hp = p.ht + sbase + (size_t)(32 * blk) * dv;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    *hp = __uint_as_float(r[k]);
                    hp += dv;
                }
            }
        }
        if (last) break;
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(x, B_S_FULL));
        DN_TRACE_EV(3, c);
        const int s1 = (c + 1) % NS;
        if (!wwait(x, bar(x, B_FULL + s1), ((c + 1) / NS) & 1)) return;
        const float alpha = scal(x, s1)[SC_ALPHA];
        for (int blk = 0; blk < 4; ++blk) {
            tmem_ld32(lb + TM_S + 32 * blk, r);
            tmem_wait_ld_dep(r);
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(alpha * __uint_as_float(r[k]));
            tmem_st32(lb + TM_S + 32 * blk, r);
        }
        tmem_wait_st();  // ordered before the next v~ arrive (fence there)
        DN_TRACE_EV(4, c);
    }
}

// ---------------------------------------------------------------------------
// Output warpgroup: o = scale e^{G_i} (S^T Q^T)[v][i] + (v_new^T P^T)[v][i].
// ---------------------------------------------------------------------------
__device__ void output_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);  // value column = TMEM lane
    const uint32_t lb = lane_base(tm, warp);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    const long long rs = (long long)p.Nv * p.dv;
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const uint32_t par = c & 1;
        if (!wwait(x, bar(x, B_D_FULL), par)) return;
        if (!wwait(x, bar(x, B_FULL + s), (c / NS) & 1)) return;
        DN_TRACE_EV(0, c);
        tc_fence_after();
        const float *sc = scal(x, s);
        const int L = __float_as_int(sc[SC_L]);
        const long long t0 = u.bos + (long long)c * C;
        __nv_bfloat16 *op = o + (t0 * p.Nv + u.h) * (long long)p.dv + u.v0 + v;
        // combine both halves into packed bf16 pairs first, release the
        // accumulators, then store
        uint32_t ra[16], qa[16], ob[32];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            tmem_ld16(lb + TM_O + 16 * qq, ra);
            tmem_wait_ld_dep16(ra);
            tmem_ld16(lb + TM_P + 16 * qq, qa);
            tmem_wait_ld_dep16(qa);
            const float4 *osc4 = reinterpret_cast<const float4 *>(sc + SC_OSC + 16 * qq);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 os = osc4[k4];
                ob[8 * qq + 2 * k4] =
                    pack_bf16(fmaf(os.x, __uint_as_float(ra[4 * k4]), __uint_as_float(qa[4 * k4])),
                              fmaf(os.y, __uint_as_float(ra[4 * k4 + 1]), __uint_as_float(qa[4 * k4 + 1])));
                ob[8 * qq + 2 * k4 + 1] =
                    pack_bf16(fmaf(os.z, __uint_as_float(ra[4 * k4 + 2]), __uint_as_float(qa[4 * k4 + 2])),
                              fmaf(os.w, __uint_as_float(ra[4 * k4 + 3]), __uint_as_float(qa[4 * k4 + 3])));
            }
        }
        tc_fence_before();
        warp_arrive(bar(x, B_O_EMPTY));
        // rows i < L of column v; bf16 pair k holds rows 2k (low) and 2k + 1
        uint16_t *po = reinterpret_cast<uint16_t *>(op);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (2 * k < L) po[(2 * k) * rs] = (uint16_t)(ob[k] & 0xffffu);
            if (2 * k + 1 < L) po[(2 * k + 1) * rs] = (uint16_t)(ob[k] >> 16);
        }
        warp_arrive(bar(x, B_EMPTY + s));
        DN_TRACE_EV(1, c);
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
tc_fwd(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
       const __grid_constant__ CUtensorMap mV, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Ctx x;
    x.base = (raw + 1023u) & ~1023u;
    x.gbase = smem_raw + (x.base - raw);
    x.abort_flag = reinterpret_cast<volatile int *>(x.gbase + OFF_MISC + 4);
    x.status = p.status;
    const int warp = threadIdx.x >> 5;
    const Unit u = unit_of(p);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(x, B_FULL + s), 2);
            mbar_init(bar(x, B_EMPTY + s), 13);
        }
        mbar_init(bar(x, B_KQ_FULL), 1);
        mbar_init(bar(x, B_WU_FULL), 1);
        mbar_init(bar(x, B_WSM_FULL), 4);
        mbar_init(bar(x, B_S_FULL), 4);
        mbar_init(bar(x, B_V_FULL), 1);
        mbar_init(bar(x, B_VSM_FULL), 4);
        mbar_init(bar(x, B_D_FULL), 1);
        mbar_init(bar(x, B_O_EMPTY), 4);
        mbar_init(bar(x, B_DRAIN), 1);
        mbar_init(bar(x, B_DRAIN2), 1);
        *x.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(x.base + OFF_MISC, TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        prefetch_tmap(&mK);
        prefetch_tmap(&mQ);
        prefetch_tmap(&mV);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *reinterpret_cast<volatile uint32_t *>(x.gbase + OFF_MISC);

    if (warp == 0) {
        int armed_last = -1;
        loader_role(x, p, u, &mK, &mQ, &mV, armed_last);
        // drain: the last NS armed stages must have landed before exit
        if ((threadIdx.x & 31) == 0)
            for (int c = armed_last - NS + 1; c <= armed_last; ++c)
                if (c >= 0) wait_drain(bar(x, B_FULL + c % NS), (c / NS) & 1);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0 && u.nc > 0) mma_role(x, u, tm);
        __syncwarp();
    } else if (warp < 6) {
        prep_role(x, u, tm, p.scale);
    } else if (warp < 10) {
        state_role(x, p, u, tm);
    } else {
        output_role(x, p, u, tm);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tm, TM_COLS);
}

}  // namespace

bool tc_supported(int dk, int dv, bool bf16) { return bf16 && dk == DK && dv % BVT == 0; }

cudaError_t tc_launch(const Params &p, cudaStream_t stream, const char **name) {
    CUtensorMap mK, mQ, mV;
    const uint64_t tokens = (uint64_t)p.tokens;
    if (!make_tmap_rows_heads_d(&mK, p.k, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mQ, p.q, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mV, p.v, tokens, p.Nv, p.dv, 64, C))
        return cudaErrorInvalidValue;
    const long long grid = (long long)p.N * p.Nv * (p.dv / BVT);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(tc_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (err != cudaSuccess) return err;
    tc_fwd<<<(unsigned)grid, NTHREADS, SMEM_ALLOC, stream>>>(mK, mQ, mV, p);
    *name = "tc_fwd";
    return cudaGetLastError();
}

}  // namespace dn
