// Pieces shared by the CUDA-core forward and backward kernels: the padded
// shared-memory copies of a chunk's K and Q rows, vector loads from them, and
// the chunk's two score matrices K K^T and Q K^T.
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1 (K K^T in A),
//          §3.2 (Q K^T in the intra-chunk output).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "dn_internal.h"

namespace dn {
namespace simt {

constexpr int C = kChunk;  // 64 rows per chunk tile

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Row stride (elements) of the shared K / Q copies: rows start on 16-byte
// boundaries, and consecutive rows are 4 banks apart, so the eight rows an
// mma.sync fragment load touches (and eight lanes reading 16-byte pieces of
// consecutive rows) hit different banks.
template <typename Tin>
__host__ __device__ constexpr int kq_ld(int dk) { return sizeof(Tin) == 2 ? dk + 8 : dk + 4; }

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Elements d .. d+3 of a shared row as fp32 (d a multiple of 4).
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// Copy L rows of a [tokens, H, d] tensor (head hh, tokens from t0) into a
// padded shared tile, zero-filling rows L..C-1 (the padding columns are never
// read).
template <typename Tin, int NT>
__device__ __forceinline__ void load_rows(Tin *dst, const Tin *src, long long t0, int L, int H, int hh,
                                          int d, int tid) {
    constexpr int VEC = 16 / sizeof(Tin);
    const int ld = kq_ld<Tin>(d);
    const int per_row = d / VEC;
    for (int idx = tid; idx < L * per_row; idx += NT) {
        const int i = idx / per_row, cv = idx - i * per_row;
        *reinterpret_cast<uint4 *>(dst + i * ld + cv * VEC) =
            *reinterpret_cast<const uint4 *>(src + ((t0 + i) * H + hh) * (long long)d + cv * VEC);
    }
    for (int idx = L * ld + tid; idx < C * ld; idx += NT) dst[idx] = Tin(0.0f);
}

// The same rows as load_rows, as asynchronous copies (cp.async, 16 bytes
// each) that land while the caller does other work; cp_async_wait_all() then
// a barrier before the rows are read.  Rows past L are zeroed with stores.
template <typename Tin, int NT>
__device__ __forceinline__ void load_rows_async(Tin *dst, const Tin *src, long long t0, int L, int H, int hh,
                                                int d, int tid) {
    constexpr int VEC = 16 / sizeof(Tin);
    const int ld = kq_ld<Tin>(d);
    const int per_row = d / VEC;
    for (int idx = tid; idx < L * per_row; idx += NT) {
        const int i = idx / per_row, cv = idx - i * per_row;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(dst + i * ld + cv * VEC)),
                     "l"(src + ((t0 + i) * H + hh) * (long long)d + cv * VEC)
                     : "memory");
    }
    for (int idx = L * ld + tid; idx < C * ld; idx += NT) dst[idx] = Tin(0.0f);
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// bf16 m16n8k16 tensor-core product with fp32 accumulation: d += a b.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// The chunk's (K K^T)_ij and (Q K^T)_ij, handed to epi(i, j, kk, qk) for every
// (i, j) of the 64 x 64 grid: computed where j <= i (up to the 8-column tile
// that holds the diagonal) and i < L, zero elsewhere.  Rows past the chunk's
// length L are zero in the tiles, so skipping them changes nothing.  bf16:
// tensor-core tiles (the products of bf16 values are exact in fp32,
// accumulation is fp32); one warp per (16-row, 8-column) tile pair.
template <int NT, typename Epi>
__device__ __forceinline__ void kq_products(const __nv_bfloat16 *sK, const __nv_bfloat16 *sQ, int ld, int dk,
                                            int L, int tid, Epi epi) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    // 20 tiles hold the lower triangle: 16-row tile mt pairs with 8-column
    // tiles 0 .. 2 mt + 1; the row tiles below L come first in this order
    for (int pidx = warp; pidx < 20; pidx += NT / 32) {
        const int mt = pidx < 2 ? 0 : (pidx < 6 ? 1 : (pidx < 12 ? 2 : 3));
        const int nt = pidx - (mt == 0 ? 0 : (mt == 1 ? 2 : (mt == 2 ? 6 : 12)));
        const int r0 = 16 * mt + g, j0 = 8 * nt + g;
        float ck[4] = {0.f, 0.f, 0.f, 0.f}, cq[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; 16 * mt < L && k0 < dk; k0 += 16) {
            const int kc = k0 + 2 * t;
            uint32_t a[4], aq[4], b[2];
            a[0] = *reinterpret_cast<const uint32_t *>(sK + r0 * ld + kc);
            a[1] = *reinterpret_cast<const uint32_t *>(sK + (r0 + 8) * ld + kc);
            a[2] = *reinterpret_cast<const uint32_t *>(sK + r0 * ld + kc + 8);
            a[3] = *reinterpret_cast<const uint32_t *>(sK + (r0 + 8) * ld + kc + 8);
            aq[0] = *reinterpret_cast<const uint32_t *>(sQ + r0 * ld + kc);
            aq[1] = *reinterpret_cast<const uint32_t *>(sQ + (r0 + 8) * ld + kc);
            aq[2] = *reinterpret_cast<const uint32_t *>(sQ + r0 * ld + kc + 8);
            aq[3] = *reinterpret_cast<const uint32_t *>(sQ + (r0 + 8) * ld + kc + 8);
            b[0] = *reinterpret_cast<const uint32_t *>(sK + j0 * ld + kc);
            b[1] = *reinterpret_cast<const uint32_t *>(sK + j0 * ld + kc + 8);
            mma_bf16(ck, a, b);
            mma_bf16(cq, aq, b);
        }
        const int i0 = 16 * mt + g, jj = 8 * nt + 2 * t;
        epi(i0, jj, ck[0], cq[0]);
        epi(i0, jj + 1, ck[1], cq[1]);
        epi(i0 + 8, jj, ck[2], cq[2]);
        epi(i0 + 8, jj + 1, ck[3], cq[3]);
    }
    // the 12 tiles above them are zero
    for (int e = tid; e < 12 * 128; e += NT) {
        const int tile = e >> 7, r = (e & 127) >> 3, cc = e & 7;
        const int mt = tile < 6 ? 0 : (tile < 10 ? 1 : 2);
        const int nt = (mt == 0 ? 2 + tile : (mt == 1 ? 4 + tile - 6 : 6 + tile - 10));
        epi(16 * mt + r, 8 * nt + cc, 0.f, 0.f);
    }
}

// fp32: one (i, j) pair per thread and step, fp32 FMAs over d.
template <int NT, typename Epi>
__device__ __forceinline__ void kq_products(const float *sK, const float *sQ, int ld, int dk, int L, int tid,
                                            Epi epi) {
    for (int idx = tid; idx < C * C; idx += NT) {
        const int i = idx >> 6, j = idx & 63;
        float kk = 0.f, qk = 0.f;
        if (j <= i && i < L) {
            const float *ki = sK + i * ld, *kj = sK + j * ld, *qi = sQ + i * ld;
            for (int d = 0; d < dk; d += 4) {
                const float4 a = ld4(ki + d), b = ld4(kj + d), q = ld4(qi + d);
                kk = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, kk))));
                qk = fmaf(q.x, b.x, fmaf(q.y, b.y, fmaf(q.z, b.z, fmaf(q.w, b.w, qk))));
            }
        }
        epi(i, j, kk, qk);
    }
}

}  // namespace simt
}  // namespace dn

namespace dn {
namespace simt {

// T = (I - A)^-1 of the chunk's 64 x 64 strictly lower A, in fp32 on CUDA
// cores, blocked over 16 x 16 blocks (all NT threads call it; it synchronises
// with __syncthreads):
//   A_im = rs[i] * sA[i * lda + m] (rs null: 1), zero on and above the diagonal;
//   T_D = the inverses of the four diagonal blocks I - A_bb (forward
//   substitution, one column per thread), N = T_D A_O (A_O: the blocks below
//   the diagonal), N^4 = 0, and
//       T = (I + N + N^2 + N^3) T_D,
//   i.e. T10 = N10 T00, T21 = N21 T11, T32 = N32 T22,
//        T20 = (N20 + N21 N10) T00, T31 = (N31 + N32 N21) T11,
//        T30 = (N30 + N31 N10 + N32 N20 + N32 N21 N10) T00.
// sT (row stride ldt) gets T, zero above the diagonal; scr holds 3 x 256
// floats of scratch.  Rows and columns past the chunk's length L have A = 0
// and so come out as the identity's; with L <= 32 only T10 = N10 T00 is
// formed off the diagonal (the other blocks are zero).
template <int NT>
__device__ __forceinline__ void solve_T_blocked(const float *sA, int lda, const float *rs, float *sT, int ldt,
                                                float *scr, int L, int tid) {
    static_assert(NT >= 96, "enough threads for the block rows");
    auto A = [&](int i, int m) { return (rs ? rs[i] : 1.0f) * sA[i * lda + m]; };
    auto Tb = [&](int bi, int bj) { return sT + 16 * bi * ldt + 16 * bj; };
    // phase 0: diagonal blocks (threads 0-63: block t / 16, column t % 16);
    // the others zero the blocks above the diagonal
    if (tid < 64) {
        const int b = tid >> 4, col = tid & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == col) ? 1.0f : 0.0f;
#pragma unroll
            for (int m = 0; m < r; ++m) s = fmaf(A(o + r, o + m), x[m], s);
            x[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * ldt + o + col] = x[r];
    } else {
        for (int e = tid - 64; e < 6 * 256; e += NT - 64) {
            const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
            // upper blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            Tb(bi, bj)[r * ldt + c] = 0.0f;
        }
    }
    __syncthreads();
    if (L <= 32) {  // (uniform) two diagonal blocks at most
        if (tid < 16) {
            // N10 = T11 A10, then T10 = N10 T00
            const int r = tid;
            float n[16], out[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) n[c] = 0.0f;
            for (int k = 0; k <= r; ++k) {
                const float t = Tb(1, 1)[r * ldt + k];
#pragma unroll
                for (int c = 0; c < 16; ++c) n[c] = fmaf(t, A(16 + k, c), n[c]);
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k)
#pragma unroll
                for (int c = 0; c <= k; ++c) out[c] = fmaf(n[k], Tb(0, 0)[k * ldt + c], out[c]);
#pragma unroll
            for (int c = 0; c < 16; ++c) Tb(1, 0)[r * ldt + c] = out[c];
        } else {
            for (int e = tid - 16; e < 5 * 256; e += NT - 16) {
                const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
                // lower blocks (2,0) (2,1) (3,0) (3,1) (3,2)
                const int bi = blk < 2 ? 2 : 3;
                const int bj = blk < 2 ? blk : blk - 2;
                Tb(bi, bj)[r * ldt + c] = 0.0f;
            }
        }
        __syncthreads();
        return;
    }
    // phase 1: N_ij = T_ii A_ij into block (i, j) of sT
    if (tid < 96) {
        const int task = tid >> 4, r = tid & 15;
        const int bi = task == 0 ? 1 : (task < 3 ? 2 : 3);
        const int bj = task == 0 ? 0 : (task < 3 ? task - 1 : task - 3);
        const float *Tii = Tb(bi, bi);
        float out[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) out[c] = 0.0f;
        for (int k = 0; k <= r; ++k) {
            const float t = Tii[r * ldt + k];
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = fmaf(t, A(16 * bi + k, 16 * bj + c), out[c]);
        }
        float *dst = Tb(bi, bj) + r * ldt;
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = out[c];
    }
    __syncthreads();
    // phase 2: P20 = N21 N10, S31 = N31 + N32 N21, S30 = N30 + N31 N10 + N32 N20
    if (tid < 48) {
        const int task = tid >> 4, r = tid & 15;
        float out[16];
        auto mul_add = [&](const float *X, const float *Y) {  // out += X[r, :] Y
            for (int k = 0; k < 16; ++k) {
                const float xv = X[r * ldt + k];
#pragma unroll
                for (int c = 0; c < 16; ++c) out[c] = fmaf(xv, Y[k * ldt + c], out[c]);
            }
        };
        if (task == 0) {
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = 0.0f;
            mul_add(Tb(2, 1), Tb(1, 0));
        } else if (task == 1) {
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = Tb(3, 1)[r * ldt + c];
            mul_add(Tb(3, 2), Tb(2, 1));
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = Tb(3, 0)[r * ldt + c];
            mul_add(Tb(3, 1), Tb(1, 0));
            mul_add(Tb(3, 2), Tb(2, 0));
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) scr[task * 256 + r * 16 + c] = out[c];
    }
    __syncthreads();
    // phase 3: S30 += N32 P20; T31 = S31 T11; T20 = (N20 + P20) T00;
    // T10 = N10 T00; T21 = N21 T11 (a thread reads its own row of an
    // in-place block before it writes it, and no one else reads that row)
    if (tid < 80) {
        const int task = tid >> 4, r = tid & 15;
        float x[16], out[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) out[c] = 0.0f;
        if (task == 0) {
#pragma unroll
            for (int c = 0; c < 16; ++c) out[c] = scr[2 * 256 + r * 16 + c];
            for (int k = 0; k < 16; ++k) {
                const float xv = Tb(3, 2)[r * ldt + k];
#pragma unroll
                for (int c = 0; c < 16; ++c) out[c] = fmaf(xv, scr[k * 16 + c], out[c]);
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) scr[2 * 256 + r * 16 + c] = out[c];
        } else {
            // X T_jj with X = S31 (task 1), N20 + P20 (2), N10 (3), N21 (4)
            const int bi = task == 1 ? 3 : (task == 2 ? 2 : (task == 3 ? 1 : 2));
            const int bj = task == 1 ? 1 : (task == 2 ? 0 : (task == 3 ? 0 : 1));
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                x[k] = task == 1 ? scr[256 + r * 16 + k] : Tb(bi, bj)[r * ldt + k];
                if (task == 2) x[k] += scr[r * 16 + k];
            }
            const float *Tjj = Tb(bj, bj);
#pragma unroll
            for (int k = 0; k < 16; ++k)
#pragma unroll
                for (int c = 0; c <= k; ++c) out[c] = fmaf(x[k], Tjj[k * ldt + c], out[c]);
            float *dst = Tb(bi, bj) + r * ldt;
#pragma unroll
            for (int c = 0; c < 16; ++c) dst[c] = out[c];
        }
    }
    __syncthreads();
    // phase 4: T30 = S30 T00; T32 = N32 T22 (in place)
    if (tid < 32) {
        const int task = tid >> 4, r = tid & 15;
        float x[16], out[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            x[k] = task == 0 ? scr[2 * 256 + r * 16 + k] : Tb(3, 2)[r * ldt + k];
            out[k] = 0.0f;
        }
        const float *Tjj = task == 0 ? Tb(0, 0) : Tb(2, 2);
#pragma unroll
        for (int k = 0; k < 16; ++k)
#pragma unroll
            for (int c = 0; c <= k; ++c) out[c] = fmaf(x[k], Tjj[k * ldt + c], out[c]);
        float *dst = Tb(3, task == 0 ? 0 : 2) + r * ldt;
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = out[c];
    }
    __syncthreads();
}

}  // namespace simt
}  // namespace dn
