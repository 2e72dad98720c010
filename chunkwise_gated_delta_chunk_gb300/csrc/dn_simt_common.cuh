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
// that holds the diagonal), zero elsewhere.  Rows past the chunk's length are
// zero in the tiles and so give zero.  bf16: tensor-core tiles (the products
// of bf16 values are exact in fp32, accumulation is fp32); one warp per
// (16-row, 8-column) tile pair.
template <int NT, typename Epi>
__device__ __forceinline__ void kq_products(const __nv_bfloat16 *sK, const __nv_bfloat16 *sQ, int ld, int dk,
                                            int tid, Epi epi) {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    // 20 tiles hold the lower triangle: 16-row tile mt pairs with 8-column tiles 0 .. 2 mt + 1
    for (int pidx = warp; pidx < 20; pidx += NT / 32) {
        const int mt = pidx < 2 ? 0 : (pidx < 6 ? 1 : (pidx < 12 ? 2 : 3));
        const int nt = pidx - (mt == 0 ? 0 : (mt == 1 ? 2 : (mt == 2 ? 6 : 12)));
        const int r0 = 16 * mt + g, j0 = 8 * nt + g;
        float ck[4] = {0.f, 0.f, 0.f, 0.f}, cq[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < dk; k0 += 16) {
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
__device__ __forceinline__ void kq_products(const float *sK, const float *sQ, int ld, int dk, int tid, Epi epi) {
    for (int idx = tid; idx < C * C; idx += NT) {
        const int i = idx >> 6, j = idx & 63;
        float kk = 0.f, qk = 0.f;
        if (j <= i) {
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
