// One WY work item of the chunkwise gated delta rule forward (bf16 q/k,
// dk = 128 or 256): for one 64-token tile and value head, the lower-triangular
// inverse T = (I - A)^-1 of each chunk's WY representation and each chunk's
// causal score matrix, written to the chunk's workspace slot as the three
// bf16 MMA operands T' = T diag(beta e^G) and T'' = T diag(beta) (which give
// W = T' K and U = T'' V) and P = tril(scale QK^T . D).  A tile holds one
// chunk of 64 tokens, or two of 32 or four of 16: A and P are then block
// diagonal (each chunk's own block), the solve gives each chunk's T in its
// block, and each chunk's rows go to its own slot.
//
// Sources: [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现"
//                 §2.3 (A = -tril(diag(beta) K K^T, -1), T = (I - A)^-1 by
//                 forward substitution), §2.4 (W = T diag(beta) K, U = T diag(beta) V,
//                 intra-chunk output through tril(Q K^T));
//          [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.2 (gated form:
//                 A_ij and P_ij carry e^{G_i - G_j}, W carries e^{G}).
//
// A worker is a group of 128 threads (four consecutive warps, so warp w of
// the group reaches TMEM lanes 32 w .. 32 w + 31) with its own 36 KB of
// shared memory, 64 TMEM columns, two mbarriers and one named barrier; the
// WY kernel runs one worker per CTA.  Per item:
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
// word and the item reports failure after draining its own TMA / MMA work.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "dn_chunk.cuh"
#include "dn_internal.h"
#include "dn_tc.h"
#include "tc_ptx.cuh"

namespace dn {
namespace wy {
namespace {

using namespace ptx;

constexpr int C = kChunk;  // 64
constexpr int NT = 128;
constexpr uint64_t kTimeoutNs = kWaitLimitNs;

// Shared memory of a worker (offsets from a 1024-byte aligned base): the K
// and Q tiles as 64-column quarters K0 Q0 K1 Q1 .. (8 KB each, so that K_q
// and Q_q form the 128 rows of one MMA operand), then the gate scalars, the
// inverse norms and the barriers.  Once the [K; Q] K^T MMA has read the tiles,
// A / T (fp32, row stride LDA, 16-row block rows RS floats apart) and the
// solve scratch (groups of three 16 x 16 blocks, XRS floats apart) reuse
// them: for dk = 128 the whole tile region, for dk = 256 only the Q quarters,
// since the K tile is read again by the W MMA.  For dk = 256 the bf16 T'
// image that MMA reads then takes the first Q quarter (OFF_TPI).
constexpr int LDA = 68;              // fp32 row stride of A / T
constexpr int SLD = 20, SBLK = 16 * SLD;  // scratch blocks: fp32, row stride SLD
template <int DKW>
struct Lay {
    static_assert(DKW == 128 || DKW == 256, "key head size");
    static constexpr uint32_t TILE_BYTES = 2u * 64u * DKW * 2u;
    static constexpr uint32_t OFF_A = DKW == 128 ? 0u : 8192u;
    static constexpr int RS = DKW == 128 ? 16 * LDA : 4096;
    static constexpr uint32_t OFF_SCR = DKW == 128 ? 64u * LDA * 4u : 8192u + 16u * LDA * 4u;
    static constexpr int XRS = DKW == 128 ? 3 * SBLK : 4096;
    static constexpr uint32_t OFF_TPI = 8192;
    static constexpr uint32_t OFF_SC = TILE_BYTES;
    static constexpr uint32_t OFF_NRM = OFF_SC + SCAL_FLOATS * 4;  // 64 inverse key norms, 64 inverse query norms
    static constexpr uint32_t OFF_BAR = OFF_NRM + 512;
    static constexpr uint32_t SMEM_USED = OFF_BAR + 40;             // 2 mbarriers, TMEM base, flag, 2 W mbarriers
    static constexpr uint32_t GROUP_BYTES = (SMEM_USED + 1023u) & ~1023u;  // one worker's region
    // [K; Q] K^T in columns 0-63; for dk = 256, then W, one 128-column half
    // of d at a time
    static constexpr uint32_t TM_COLS = DKW == 128 ? 64 : 128;
};
static_assert(kImageBytes == 8192 && slot_norm_off(128) == 3 * kImageBytes &&
                  slot_norm_off(256) == 32768 + 2 * kImageBytes,
              "slot = T' or -W | T'' | P | norms");

constexpr uint32_t ID_KQ = idesc_bf16(128, 64, 0, 0);  // A, B K-major
constexpr uint32_t ID_WK = idesc_bf16(128, 128, 0, 1); // A K-major (T' rows), B MN-major (K rows)

__device__ bool wait_bounded(uint32_t b, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(b, parity))
        if (globaltimer() - t0 > kTimeoutNs) return false;
    return true;
}

// ---- 16 x 16 block helpers for the solve (fp32 blocks, TF32 mma.sync) -------
// A 16 x 8 output tile (columns n0..n0+7 of the product) per warp, in the
// m16n8k8 fragment layout: lane l = 4 g + t holds rows g and g + 8, columns
// 2 t and 2 t + 1.  Products run on the tensor cores with TF32 operands
// (rounded to nearest) and fp32 accumulation.
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

// acc += Ab (16 x 16) Bb[:, n0 .. n0 + 7]
__device__ __forceinline__ void tile_mma(float (&acc)[4], const float *Ab, int lda, const float *Bb, int ldb,
                                         int n0, int lane) {
    const int g = lane >> 2, t = lane & 3;
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
                                             const float *Bb, int ldb, int n0, int lane) {
    const int g = lane >> 2, t = lane & 3;
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

__device__ __forceinline__ void tile_load(float (&acc)[4], const float *Cb, int ldc, int n0, int lane) {
    const int g = lane >> 2, t = lane & 3;
    acc[0] = Cb[g * ldc + n0 + 2 * t];
    acc[1] = Cb[g * ldc + n0 + 2 * t + 1];
    acc[2] = Cb[(g + 8) * ldc + n0 + 2 * t];
    acc[3] = Cb[(g + 8) * ldc + n0 + 2 * t + 1];
}

__device__ __forceinline__ void tile_store(float *Cb, int ldc, int n0, const float (&acc)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    Cb[g * ldc + n0 + 2 * t] = acc[0];
    Cb[g * ldc + n0 + 2 * t + 1] = acc[1];
    Cb[(g + 8) * ldc + n0 + 2 * t] = acc[2];
    Cb[(g + 8) * ldc + n0 + 2 * t + 1] = acc[3];
}

// Scratch blocks of the solve.
enum { XN10, XN20, XN21, XN30, XN31, XN32, XP20, XS31, XS30, XCOUNT };
static_assert(Lay<128>::OFF_SCR + XCOUNT * SBLK * 4 <= Lay<128>::OFF_SC, "the solve scratch fits in the tiles");
static_assert(16 * LDA * 4 + 3 * SBLK * 4 <= 8192 && (XCOUNT + 2) / 3 <= 3,
              "dk = 256: 16 rows of A / T and three scratch blocks fit in each of Q0-Q2");

// In-place T = (I - A)^-1 for the 64 x 64 strictly lower A at sA (row stride
// LDA, block row b at sA + b RS); scratch block k at scr + (k / 3) XRS +
// (k % 3) SBLK; 128 threads.  With A_D the four 16 x 16 diagonal blocks and A_O the
// rest, I - A = (I - A_D)(I - N) with N = (I - A_D)^-1 A_O strictly block
// lower, so N^4 = 0 and
//     T = (I + N + N^2 + N^3) T_D,   T_D = (I - A_D)^-1,   N_ij = T_ii A_ij.
// The diagonal blocks are inverted by forward substitution in fp32 (warp pw
// owns block pw, lane l the column l % 16); the block products are TF32
// tensor-core tiles with fp32 accumulation, in four barrier-separated phases.
template <int RS, int XRS>
__device__ __forceinline__ void solve_T(float *sA, float *scr, int pw, int lane, uint32_t bid) {
    {
        // x = column `col` of (I - A_bb)^-1:  x_r = [r == col] + sum_{m < r} A[r][m] x_m.
        // Rows of the block are read as float4 (one broadcast wavefront per
        // four elements); four partial sums shorten the dependency chain.
        const int col = lane & 15, o = 16 * pw;
        float xv[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float4 *ar = reinterpret_cast<const float4 *>(sA + pw * RS + r * LDA + o);
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
            for (int r = 0; r < 16; ++r) sA[pw * RS + r * LDA + o + col] = xv[r];
        }
    }
    named_bar_sync(bid, 128);
    auto blkA = [&](int i, int j) { return sA + i * RS + 16 * j; };
    auto blkX = [&](int k) { return scr + (k / 3) * XRS + (k % 3) * SBLK; };
    // phase 1: N_ij = T_ii A_ij, six blocks x two column halves (3 per warp)
    {
        float acc[3][4];
        float *dst[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int task = pw + 4 * q, b = task >> 1, n0 = 8 * (task & 1);
            const int bi = (b == 0) ? 1 : (b < 3 ? 2 : 3);
            const int bj = (b == 0) ? 0 : (b < 3 ? b - 1 : b - 3);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;
            tile_mma(acc[q], blkA(bi, bi), LDA, blkA(bi, bj), LDA, n0, lane);
            dst[q] = blkX(b) + n0;
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) tile_store(dst[q], SLD, 0, acc[q], lane);
    }
    named_bar_sync(bid, 128);
    // phase 2: P20 = N21 N10, S31 = N31 + N32 N21, S30 = N30 + N31 N10 + N32 N20
    {
        float acc[2][4];
        float *dst[2];
        bool live[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int task = pw + 4 * q, n0 = 8 * (task & 1);
            live[q] = task < 6;
            const int kind = task >> 1;  // 0: P20, 1: S31, 2: S30
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;
            if (live[q]) {
                if (kind == 1) tile_load(acc[q], blkX(XN31), SLD, n0, lane);
                if (kind == 2) tile_load(acc[q], blkX(XN30), SLD, n0, lane);
                const float *A0 = blkX(kind == 0 ? XN21 : (kind == 1 ? XN32 : XN31));
                const float *B0 = blkX(kind == 0 ? XN10 : (kind == 1 ? XN21 : XN10));
                tile_mma(acc[q], A0, SLD, B0, SLD, n0, lane);
                if (kind == 2) tile_mma(acc[q], blkX(XN32), SLD, blkX(XN20), SLD, n0, lane);
            }
            dst[q] = blkX(kind == 0 ? XP20 : (kind == 1 ? XS31 : XS30)) + n0;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (live[q]) tile_store(dst[q], SLD, 0, acc[q], lane);
    }
    named_bar_sync(bid, 128);
    // phase 3: S30 += N32 P20, and T_ij = S_ij T_jj for every block but (3,0)
    {
        float acc[3][4];
        float *dst[3];
        int ldd[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int task = pw + 4 * q, n0 = 8 * (task & 1), kind = task >> 1;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;
            if (kind == 0) {
                tile_load(acc[q], blkX(XS30), SLD, n0, lane);
                tile_mma(acc[q], blkX(XN32), SLD, blkX(XP20), SLD, n0, lane);
                dst[q] = blkX(XS30) + n0;
                ldd[q] = SLD;
            } else if (kind == 5) {
                tile_mma_sum(acc[q], blkX(XN20), blkX(XP20), SLD, blkA(0, 0), LDA, n0, lane);
                dst[q] = blkA(2, 0) + n0;
                ldd[q] = LDA;
            } else {
                // kind 1: T10 = N10 T00, 2: T21 = N21 T11, 3: T32 = N32 T22, 4: T31 = S31 T11
                const int xa = kind == 1 ? XN10 : (kind == 2 ? XN21 : (kind == 3 ? XN32 : XS31));
                const int dj = kind == 1 ? 0 : (kind == 3 ? 2 : 1);
                const int di = kind == 1 ? 1 : (kind == 2 ? 2 : 3);
                tile_mma(acc[q], blkX(xa), SLD, blkA(dj, dj), LDA, n0, lane);
                dst[q] = blkA(di, dj) + n0;
                ldd[q] = LDA;
            }
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) tile_store(dst[q], ldd[q], 0, acc[q], lane);
    }
    named_bar_sync(bid, 128);
    // phase 4: T30 = S30 T00
    if (pw < 2) {
        const int n0 = 8 * pw;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma(acc, blkX(XS30), SLD, blkA(0, 0), LDA, n0, lane);
        tile_store(blkA(3, 0), LDA, n0, acc, lane);
    }
    named_bar_sync(bid, 128);
}


// Row i of a 64 x 64 bf16 image (32 values in two halves of packed pairs)
// straight to global memory, in the 128-byte-swizzled layout.
__device__ __forceinline__ void store_image_row(uint8_t *img, int i, int hf, const uint32_t (&pk)[16]) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const int cc = 4 * hf + ch;
        *reinterpret_cast<uint4 *>(img + i * 128 + ((cc ^ (i & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    }
}


// Tiles of several chunks (ch = 16 or 32 tokens).  Tile row i's chunk owns
// the tile columns from i & ~(ch - 1), all within column half
// (i & ~(ch - 1)) / 32.  From that half's packed words pk (columns 2k, 2k + 1
// of the half), in place: the first half of row i mod ch of the chunk's own
// image (the chunk's ch columns, then zeros).
__device__ __forceinline__ void sub_row_words(uint32_t (&pk)[16], int i, int ch) {
    if (ch == 16) {
        const bool hi = ((i >> 4) & 1) != 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) pk[k] = hi ? pk[8 + k] : pk[k];
#pragma unroll
        for (int k = 8; k < 16; ++k) pk[k] = 0u;
    }
}

// Row r of a chunk's image (first half w, second half zero) and the zero rows
// r + ch, r + 2 ch, ... below the chunk's ch rows.
__device__ __forceinline__ void store_sub_rows(uint8_t *img, int r, int ch, const uint32_t (&w)[16]) {
    uint32_t z[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) z[k] = 0u;
    store_image_row(img, r, 0, w);
    store_image_row(img, r, 1, z);
    for (int rr = r + ch; rr < C; rr += ch) {
        store_image_row(img, rr, 0, z);
        store_image_row(img, rr, 1, z);
    }
}

// One worker: its shared-memory region, TMEM columns and named barrier.
struct Group {
    uint32_t base;  // shared address of the worker's 1024-aligned region
    uint8_t *gb;    // generic pointer to the same
    uint32_t tm;    // first of the worker's TM_COLS tensor-memory columns
    uint32_t bid;   // named barrier of the worker's NT threads
    int tid;        // thread index within the worker, 0 .. NT - 1
    uint32_t it;    // items run so far (mbarrier phases)
};

// Barrier setup of a worker (its thread 0); the caller synchronises after.
template <int DKW>
__device__ __forceinline__ void group_init(const Group &g) {
    if (g.tid == 0) {
        mbar_init(g.base + Lay<DKW>::OFF_BAR, 1);
        mbar_init(g.base + Lay<DKW>::OFF_BAR + 8, 1);
        mbar_init(g.base + Lay<DKW>::OFF_BAR + 24, 1);
        mbar_init(g.base + Lay<DKW>::OFF_BAR + 32, 1);
        fence_barrier_init();
    }
}

// Where work tile `tile` lies: sequence n, first token t0 and length L (at
// most 64).  A tile is 64 tokens of one sequence (tiles numbered like the
// slots of 64-token chunks, t0 / 64 + n): one chunk of 64 tokens, or two of
// 32 or four of 16, each with its own workspace slot.  valid is false for a
// tile number no tokens map to and for a malformed sequence (which the scan
// kernel reports).
struct ItemLoc {
    long long t0;
    int n, L;
    bool valid;
};

__device__ __forceinline__ ItemLoc locate(const Params &p, long long tile) {
    ItemLoc r{0, 0, 0, false};
    int lo = 0, hi = p.N - 1;  // largest n with wy_slot(bos_n, n, 64) <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (wy_slot(seq_bos(p, mid), mid, C) <= tile) lo = mid; else hi = mid - 1;
    }
    const long long bos = seq_bos(p, lo), eos = seq_eos(p, lo);
    if (bos < 0 || eos < bos || eos > p.tokens) return r;
    const long long c = tile - wy_slot(bos, lo, C);
    const long long t0 = bos + c * C;
    if (c < 0 || t0 >= eos) return r;
    r.t0 = t0;
    r.n = lo;
    r.L = (int)min((long long)C, eos - t0);
    r.valid = true;
    return r;
}

// Number of work tiles (a bound: tile numbers no tokens map to are skipped).
__host__ __device__ inline long long tile_count(const Params &p) { return p.tokens / C + p.N; }

// Warp 0, tiles of several chunks (ch = 16 or 32 tokens each): the scalars
// the WY item reads (SC_G, SC_BETA, SC_BEG, SC_AF, SC_BF, SC_FACT) with the
// gate prefix sums restarting at every chunk, so that G_i, and e^{G_i - G_0}
// with G_0 that of the chunk's first token, are each chunk's own.
__device__ __forceinline__ void sub_chunk_scalars_store(const ChunkGates &in, int ch, float *sc, int lane) {
    float ga = in.ga, gb = in.gb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ta = __shfl_up_sync(0xffffffffu, ga, off);
        const float tb = __shfl_up_sync(0xffffffffu, gb, off);
        if (lane >= off && (lane ^ (lane - off)) < ch) {  // the same chunk
            ga += ta;
            gb += tb;
        }
    }
    const int first = lane & ~(ch - 1);
    const float g0a = __shfl_sync(0xffffffffu, ga, first), g0b = __shfl_sync(0xffffffffu, gb, first);
    float mxa = ga, mna = ga, mxb = gb, mnb = gb;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float xa = __shfl_xor_sync(0xffffffffu, mxa, off), na = __shfl_xor_sync(0xffffffffu, mna, off);
        const float xb = __shfl_xor_sync(0xffffffffu, mxb, off), nb = __shfl_xor_sync(0xffffffffu, mnb, off);
        if (off < ch) {  // partners within the same chunk
            mxa = fmaxf(mxa, xa);
            mna = fminf(mna, na);
            mxb = fmaxf(mxb, xb);
            mnb = fminf(mnb, nb);
        }
    }
    const bool fact = __all_sync(0xffffffffu, mxa - mna <= kSpanMax && mxb - mnb <= kSpanMax);
    const int ia = lane, ib = lane + 32;
    sc[SC_G + ia] = ga;
    sc[SC_G + ib] = gb;
    sc[SC_BETA + ia] = in.ba;
    sc[SC_BETA + ib] = in.bb;
    sc[SC_BEG + ia] = in.ba * __expf(ga);
    sc[SC_BEG + ib] = in.bb * __expf(gb);
    sc[SC_AF + ia] = __expf(ga - g0a);
    sc[SC_AF + ib] = __expf(gb - g0b);
    sc[SC_BF + ia] = __expf(g0a - ga);
    sc[SC_BF + ib] = __expf(g0b - gb);
    if (lane == 0) sc[SC_FACT] = fact ? 1.f : 0.f;
}

// Warp 0: the gates of the tokens of tile `tile`, value head h (zero where no
// tokens map to the tile).
__device__ __forceinline__ ChunkGates item_gates(const Params &p, long long tile, int h, int lane) {
    const ItemLoc l = locate(p, tile);
    if (!l.valid) return ChunkGates{0.f, 0.f, 0.f, 0.f};
    return chunk_gates_load(p, h, l.t0, l.L, lane);
}

// dk = 256: -W = -T' K as the bf16 K-major image the scan kernel reads (four
// 64-column quarters of 64 rows x 128 B, swizzled like the other images), in
// two 128-column halves of d.  Each half is one MMA chain with M = 128: A is
// the T' image at OFF_TPI (written by threads 0-63 just before) followed by
// 64 rows the result ignores, B the K tile quarters read MN-major; TMEM lane
// i < 64 then holds row i of W.  Returns false when a wait ran out.
// Threads 0-63 store row i of -W as row `row` of the image at `img` (null:
// none), and zero rows row + rs, row + 2 rs, ... below it.
template <int DKW>
__device__ bool w_step(Group &g, const Params &p, uint8_t *img, int row, int rs, uint32_t par) {
    using Y = Lay<DKW>;
    volatile int *okf = reinterpret_cast<volatile int *>(g.gb + Y::OFF_BAR + 20);
    const int warp = g.tid >> 5, i = g.tid;
    fence_proxy_async_smem();  // the T' image is read through the async proxy
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const uint32_t b_w = g.base + Y::OFF_BAR + 24 + 8 * hh;
        tc_fence_before();
        named_bar_sync(g.bid, NT);  // T' written / the previous half read
        if (g.tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss(g.tm, sdesc(g.base + Y::OFF_TPI + kk * 32, 16, 1024),
                       sdesc(g.base + 32768 * hh + kk * 2048, 16384, 1024), ID_WK, kk != 0);
            mma_commit(b_w);
            if (!wait_bounded(b_w, par)) {
                wait_bounded(b_w, par);  // drain: the MMA still reads shared memory
                *okf = 0;
                atomicOr(p.status, kStatusTimeout);
            }
        }
        tc_fence_before();
        named_bar_sync(g.bid, NT);
        tc_fence_after();
        if (*okf == 0) return false;
        if (warp < 2) {
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {  // 32 columns of d at a time
                uint32_t r[32], pk[16];
                tmem_ld32(g.tm + ((uint32_t)(32 * warp) << 16) + 32 * cb, r);
                tmem_wait_ld_dep(r);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    pk[k] = pack_bf16(-__uint_as_float(r[2 * k]), -__uint_as_float(r[2 * k + 1]));
                // d = 128 hh + 32 cb + 8 ch + e: quarter 2 hh + cb / 2, 16-byte chunk 4 (cb & 1) + ch
                if (!img) continue;
                uint8_t *qb = img + 8192 * (2 * hh + (cb >> 1));
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4 *>(qb + row * 128 + (((4 * (cb & 1) + ch) ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                for (int rr = row + rs; rr < C; rr += rs)
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
                        *reinterpret_cast<uint4 *>(qb + rr * 128 + (((4 * (cb & 1) + ch) ^ (rr & 7)) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    return true;
}

// The item of workspace slot `slot` and value head h, located at `loc`.
// Warp 0 enters with the item's gates in `gates` (loaded ahead) and leaves
// with those of the worker's next item (slot next_slot < 0: none; value head
// next_h), whose loads then overlap the rest of this item.  Returns false
// when a wait ran out (the worker must stop).
//
// dk = 256 adds a step 6: the bf16 T' image goes to shared memory, MMAs
// compute W = T' K into tensor memory (two 128-column halves of d), and
// threads 0-63 store row i of -W to the slot, so that the scan kernel needs
// neither T' nor tensor memory for W.
template <int DKW, bool QKN, bool BWD, bool SUB>
__device__ bool item(Group &g, const CUtensorMap *mK, const CUtensorMap *mQ, const Params &p, long long slot,
                     int h, const ItemLoc &loc, ChunkGates &gates, long long next_slot, int next_h) {
    using Y = Lay<DKW>;
    constexpr int NQ = DKW / 64;  // 64-column quarters of a K / Q row
    const int warp = g.tid >> 5, lane = g.tid & 31;
    const uint32_t b_tma = g.base + Y::OFF_BAR, b_mma = g.base + Y::OFF_BAR + 8;
    volatile int *okf = reinterpret_cast<volatile int *>(g.gb + Y::OFF_BAR + 20);
    float *sc = reinterpret_cast<float *>(g.gb + Y::OFF_SC);
    float *sA = reinterpret_cast<float *>(g.gb + Y::OFF_A);
    float *scr = reinterpret_cast<float *>(g.gb + Y::OFF_SCR);
    auto arow = [&](int i) { return sA + (i >> 4) * Y::RS + (i & 15) * LDA; };  // row i of A / T
    if (!loc.valid) {
        if (warp == 0 && next_slot >= 0) gates = item_gates(p, next_slot, next_h, lane);
        return true;
    }
    const long long t0 = loc.t0;
    const int L = loc.L;
    const int hk = h / (p.Nv / p.Nk);
    const uint32_t par = g.it & 1;
    ++g.it;
    // chunks of ch tokens: one per tile (ch = 64, its slot `slot`) or several
    // (ch = 16, 32), each with its own slot; img is the single chunk's slot
    const int ch = SUB ? p.chunk : C;
    constexpr bool sub = SUB;
    uint8_t *img = static_cast<uint8_t *>(p.ws) + ((size_t)h * p.nslots + slot) * slot_bytes(DKW);
    // sub: the slot of the chunk that holds tile row i (null past the tile's tokens)
    auto sub_img = [&](int i) -> uint8_t * {
        const int c0 = i & ~(ch - 1);
        if (c0 >= L) return nullptr;
        const long long s2 = wy_slot(t0 + c0, loc.n, ch);
        return static_cast<uint8_t *>(p.ws) + ((size_t)h * p.nslots + (size_t)s2) * slot_bytes(DKW);
    };

    if (warp == 0) {
        if (lane == 0) {
            *okf = 1;
            uint32_t tx = Y::TILE_BYTES;
#ifdef DN_TEST_STALL
            // failure-path test: the first item of worker 0 expects 16 bytes
            // more than its copies bring, so its wait runs out after the
            // copies have landed
            if (p.test_stall == kStallWy && blockIdx.x == 0 && g.it == 1) tx += 16;
#endif
            mbar_arrive_expect_tx(b_tma, tx);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                tma_load_3d(g.base + 16384 * q, mK, b_tma, 64 * q, hk, (int)t0);
                tma_load_3d(g.base + 16384 * q + 8192, mQ, b_tma, 64 * q, hk, (int)t0);
            }
        }
        if (sub)
            sub_chunk_scalars_store(gates, ch, sc, lane);
        else
            chunk_scalars_store(p, chunk_scalars_from(gates, L, lane), sc, lane);
        // the next item's gates: their loads run under this item's work
        if (next_slot >= 0) gates = item_gates(p, next_slot, next_h, lane);
        __syncwarp();
        if (lane == 0) {
            bool ok = wait_bounded(b_tma, par);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < NQ; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t a = g.base + kb * 16384 + kk * 32;
                        mma_ss(g.tm, sdesc(a, 16, 1024), sdesc(a, 16, 1024), ID_KQ, (kb | kk) != 0);
                    }
                mma_commit(b_mma);
                ok = wait_bounded(b_mma, par);
                if (!ok) wait_bounded(b_mma, par);  // drain: the MMA still reads shared memory
            } else {
                wait_bounded(b_tma, par);  // drain: the copy may still land
            }
            if (!ok) {
                *okf = 0;
                atomicOr(p.status, kStatusTimeout);
            }
        }
    }
    tc_fence_before();
    named_bar_sync(g.bid, NT);
    tc_fence_after();
    if (*okf == 0) return false;

    float *nrm = reinterpret_cast<float *>(g.gb + Y::OFF_NRM);
    constexpr bool qkn = QKN;
    if (qkn) {
        // 1 / max(||x||, 1e-12) of key row i (threads 0-63) or query row
        // i (64-127), from the quarters of the tile.  The sum of squares
        // does not depend on the order of the row's 16-byte chunks, so the
        // swizzle is ignored; each lane starts at chunk (i & 7) so that
        // eight lanes of a phase hit eight bank groups.
        const int i = g.tid & 63;
        const uint8_t *row = g.gb + (g.tid < 64 ? 0 : 8192) + i * 128;
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int hb = 0; hb < NQ; ++hb)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 w = *reinterpret_cast<const uint4 *>(row + hb * 16384 + (((cc + i) & 7) << 4));
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(wv[e] << 16), hi = __uint_as_float(wv[e] & 0xffff0000u);
                    ss0 = fmaf(lo, lo, ss0);
                    ss1 = fmaf(hi, hi, ss1);
                }
            }
        const float rn = rsqrtf(fmaxf(ss0 + ss1, 1e-24f));
        nrm[g.tid] = rn;
        if (!sub) {
            reinterpret_cast<float *>(img + slot_norm_off(DKW))[g.tid] = rn;
        } else if (uint8_t *im = sub_img(i)) {
            // row i mod ch of its chunk's slot; 1 in the rows past the chunk
            float *nf = reinterpret_cast<float *>(im + slot_norm_off(DKW)) + (g.tid < 64 ? 0 : 64);
            nf[i & (ch - 1)] = rn;
            for (int rr = (i & (ch - 1)) + ch; rr < C; rr += ch) nf[rr] = 1.f;
        }
        // T' = T diag(beta e^G / ||k||)
        if (g.tid < 64) sc[SC_BEG + i] *= rn;
        named_bar_sync(g.bid, NT);
    }

    {
        // row i of K K^T (warps 0-1) or of Q K^T (warps 2-3) = TMEM lane
        const int row = g.tid, i = row & 63;
        const bool rowA = row < 64;
        const float Gi = sc[SC_G + i];
        // A_ij = -beta_i e^{G_i - G_j} (K K^T)_ij for j < i;
        // P_ij = scale e^{G_i - G_j} (Q K^T)_ij for j <= i
        // with kQkL2Norm: times 1/||k_i|| or 1/||q_i||, and 1/||k_j|| per column
        // (BWD: the rows of A are formed without beta_i, as -(K K^T . D),
        // which the backward keeps; A_ij = beta_i times that)
        const float ri = (rowA ? (BWD ? -1.f : -sc[SC_BETA + i]) : p.scale) * (qkn ? nrm[row] : 1.f);
        const float ai = ri * sc[SC_AF + i];
        const bool live = i < loc.L;  // BWD: rows past the chunk are stored as zero
        float *wx = BWD ? p.wyx + ((size_t)h * p.nslots + (size_t)slot) * 3 * 4096 + (rowA ? 0 : 4096) + i * 64
                        : nullptr;
        const int jmax = rowA ? i - 1 : i;
        const int jmin = i & ~(ch - 1);        // the first row of row i's chunk
        const bool fact = sc[SC_FACT] != 0.f;  // uniform over the tile
        uint32_t r[32];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            tmem_ld32(g.tm + ((uint32_t)(32 * warp) << 16) + 32 * hf, r);
            // D_ij = e^{G_i - G_j}: the product of the two per-chunk
            // factors when the chunk's log-gate span allows it, else one
            // exponential
            float dcy[32];
            if (fact) {
                const float4 *b4 = reinterpret_cast<const float4 *>(sc + SC_BF + 32 * hf);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 bb = b4[q4];
                    dcy[4 * q4] = ai * bb.x;
                    dcy[4 * q4 + 1] = ai * bb.y;
                    dcy[4 * q4 + 2] = ai * bb.z;
                    dcy[4 * q4 + 3] = ai * bb.w;
                }
            } else {
                const float4 *g4 = reinterpret_cast<const float4 *>(sc + SC_G + 32 * hf);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 gg = g4[q4];
                    const int j = 32 * hf + 4 * q4;
                    dcy[4 * q4] = ri * __expf(j <= jmax && j >= jmin ? Gi - gg.x : -INFINITY);
                    dcy[4 * q4 + 1] = ri * __expf(j + 1 <= jmax && j + 1 >= jmin ? Gi - gg.y : -INFINITY);
                    dcy[4 * q4 + 2] = ri * __expf(j + 2 <= jmax && j + 2 >= jmin ? Gi - gg.z : -INFINITY);
                    dcy[4 * q4 + 3] = ri * __expf(j + 3 <= jmax && j + 3 >= jmin ? Gi - gg.w : -INFINITY);
                }
            }
            if (qkn) {
                const float4 *n4 = reinterpret_cast<const float4 *>(nrm + 32 * hf);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 nn = n4[q4];
                    dcy[4 * q4] *= nn.x;
                    dcy[4 * q4 + 1] *= nn.y;
                    dcy[4 * q4 + 2] *= nn.z;
                    dcy[4 * q4 + 3] *= nn.w;
                }
            }
            tmem_wait_ld_dep(r);
            float val[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = 32 * hf + jj;
                val[jj] = (j <= jmax && j >= jmin) ? dcy[jj] * __uint_as_float(r[jj]) : 0.f;
            }
            if (BWD) {
                // -(K K^T . D) or P row i, fp32, for the backward
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    *reinterpret_cast<float4 *>(wx + 32 * hf + 4 * q4) =
                        live ? make_float4(val[4 * q4], val[4 * q4 + 1], val[4 * q4 + 2], val[4 * q4 + 3])
                             : make_float4(0.f, 0.f, 0.f, 0.f);
                if (rowA) {
                    const float bi = sc[SC_BETA + i];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) val[jj] *= bi;
                }
            }
            if (rowA) {
                float *ar = arow(i);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    *reinterpret_cast<float4 *>(ar + 32 * hf + 4 * q4) =
                        make_float4(val[4 * q4], val[4 * q4 + 1], val[4 * q4 + 2], val[4 * q4 + 3]);
            } else {
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(val[2 * k], val[2 * k + 1]);
                if (!sub) {
                    store_image_row(img + slot_p_off(DKW), i, hf, pk);
                } else if (hf == (i >> 5)) {  // the half that holds row i's chunk
                    if (uint8_t *im = sub_img(i)) {
                        sub_row_words(pk, i, ch);
                        store_sub_rows(im + slot_p_off(DKW), i & (ch - 1), ch, pk);
                    }
                }
            }
        }
    }
    tc_fence_before();
    named_bar_sync(g.bid, NT);
    solve_T<Y::RS, Y::XRS>(sA, scr, warp, lane, g.bid);
    {
        // T' = T diag(beta e^G) (threads 0-63), T'' = T diag(beta) (64-127)
        const int i = g.tid & 63;
        const bool tp = g.tid < 64;
        const float *trow = arow(i);
        const float *cs = sc + (tp ? SC_BEG : SC_BETA);
        if (BWD) {
            // T, fp32, for the backward (rows past the chunk: the identity's,
            // as A is zero there), copied from shared memory by all 128
            // threads: each warp stores two whole 256-byte rows at a time
            float *wt = p.wyx + ((size_t)h * p.nslots + (size_t)slot) * 3 * 4096 + 8192;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int idx = g.tid + 128 * it, rr = idx >> 4, q4 = idx & 15;
                *reinterpret_cast<float4 *>(wt + rr * 64 + 4 * q4) = *reinterpret_cast<const float4 *>(arow(rr) + 4 * q4);
            }
        }
        uint32_t pk[2][16];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 a = *reinterpret_cast<const float4 *>(trow + 32 * hf + 4 * q4);
                const float4 cc = *reinterpret_cast<const float4 *>(cs + 32 * hf + 4 * q4);
                pk[hf][2 * q4] = pack_bf16(a.x * cc.x, a.y * cc.y);
                pk[hf][2 * q4 + 1] = pack_bf16(a.z * cc.z, a.w * cc.w);
            }
            if (DKW == 128 || !tp) {
                if (!sub) {
                    store_image_row(img + (tp ? 0 : slot_tu_off(DKW)), i, hf, pk[hf]);
                } else if (hf == (i >> 5)) {  // the half that holds row i's chunk
                    if (uint8_t *im = sub_img(i)) {
                        uint32_t w[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) w[k] = pk[hf][k];
                        sub_row_words(w, i, ch);
                        store_sub_rows(im + (tp ? 0 : slot_tu_off(DKW)), i & (ch - 1), ch, w);
                    }
                }
            }
        }
        if (DKW == 256) {
            // T' into shared memory once every row of T has been read
            named_bar_sync(g.bid, NT);
            if (tp) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
                        st_shared_v4(g.base + Y::OFF_TPI + sw128(i, 4 * hf + ch), pk[hf][4 * ch], pk[hf][4 * ch + 1],
                                     pk[hf][4 * ch + 2], pk[hf][4 * ch + 3]);
            }
        }
    }
    if (DKW == 256) {
        // row i of -W goes to row i mod ch of its chunk's slot (threads 0-63)
        uint8_t *wimg = sub ? sub_img(g.tid & 63) : img;
        if (!w_step<DKW>(g, p, wimg, sub ? (g.tid & (ch - 1)) : g.tid, sub ? ch : C, par)) return false;
    }
    // A / T and the scratch are read; the next item's TMA rewrites them
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_sync(g.bid, NT);
    tc_fence_after();
    return true;
}

}  // namespace
}  // namespace wy
}  // namespace dn
