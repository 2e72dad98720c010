// Backward of the chunkwise gated delta rule forward (CUDA cores, fp32 arithmetic).
//
// Sources: [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现"
//                 §3.4 (the backward recomputes the chunk's WY quantities
//                 and walks the chunks in reverse for dS; gradients dq, dk,
//                 dv, dbeta, dh0), §2.3-§2.4 (the chunk form it differentiates);
//          [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.3 (gated chunk form).
//
// The pages print no backward formula.  This kernel applies the chain rule
// to the chunk form the forward kernels evaluate.  For one chunk (L tokens,
// rows past L zero), with S the state it starts from and G the in-chunk
// gate prefix sum,
//     A   = -diag(beta) (K K^T . D)  (strictly lower),  D_ij = e^{G_i - G_j}
//     T   = (I - A)^-1
//     U   = V - diag(e^G) K S,   R = diag(beta) U,   Vn = T R     (v_new)
//     P   = scale (Q K^T . D)    (lower, diagonal included)
//     O   = scale diag(e^G) Q S + P Vn
//     S'  = e^{G_L} S + K^T diag(dec) Vn,   dec_i = e^{G_L - G_i}
// and, given dO and dS' (the gradient of the state the chunk hands on):
//     dVn = diag(dec) K dS' + P^T dO
//     dR  = T^T dVn,   dv = diag(beta) dR
//     dA  = dR Vn^T  (strictly lower; = T^T (dVn R^T) T^T),   dP = dO Vn^T (lower)
//     dS  = e^{G_L} dS' + scale Q^T diag(e^G) dO - K^T diag(beta e^G) dR
//     dq_i = scale e^{G_i} S dO_i + sum_j scale D_ij dP_ij k_j
//     dk_i = dec_i dS' Vn_i - beta_i e^{G_i} S dR_i + sum_j (M_ij + M_ji) k_j
//            + sum_j scale D_ji dP_ji q_j,     M_ij = -beta_i D_ij dA_ij
//     dbeta_i = dR_i . U_i + sum_j dA_ij (-(k_i . k_j) D_ij)
//     dG_i = e^{G_i} (scale (Q S)_i . dO_i - beta_i (K S)_i . dR_i)
//            + sum_j E_ij - sum_j E_ji - e_i
//            + [i = L-1] (sum_j e_j + e^{G_L} <S, dS'>),
//     E_ij = dA_ij A_ij + dP_ij P_ij,   e_i = dec_i (K dS')_i . Vn_i
// and dg is the reverse prefix sum of dG over the chunk (G_i = sum_{j<=i} g_j).
//
// One CTA per (sequence, value head, 32-column value tile), as in the
// CUDA-core forward.  The chunk-start states come from a forward pass at
// chunk 64 that saves them: the tensor-core forward where it applies (bf16,
// dk = 128, dv a multiple of 128; its states carry the bf16 rounding of its
// MMA operands, like the pages' backward, which recomputes them with the
// forward kernels), else the CUDA-core forward in fp32.  Every quantity above that sums over
// value columns (dq, dk, dbeta, dg, and dA, dP through them) is linear in the
// tile's columns, so each CTA adds its share to zero-initialised fp32 outputs
// with atomics; dv and dh0 belong to one tile and are stored directly.
#include <cuda_bf16.h>
#include <math.h>

#include "dn_internal.h"
#include "dn_order.cuh"
#include "dn_simt_common.cuh"
#include "dn_tc.h"

namespace dn {
namespace {

using simt::kq_ld;
using simt::ld4;
using simt::to_f;
using simt::align16;

constexpr int C = kChunk;    // 64
constexpr int BV = 32;       // value columns per CTA
constexpr int NT = 256;      // 8 warps
// Row strides of the C x C matrices (LDC) and of the C x BV tiles (LDV).
// FMA code: C + 1 and BV + 1 (conflict-free row-per-lane reads).  Tensor-core
// code: 4 mod 32, so that a fragment's 8 rows x 4 columns hit 32 banks.
template <bool MMA>
struct Strides {
    static constexpr int LDC = MMA ? C + 4 : C + 1;
    static constexpr int LDV = MMA ? BV + 4 : BV + 1;
};

// Row stride (floats) of the transposed state tiles S^T, dS^T ([BV][dk]):
// 16-byte rows, consecutive rows 4 banks apart.
__host__ __device__ inline int st_ld(int dk) { return dk + 4; }

struct Layout {
    size_t k, q, k2, q2, s, ds, m0, m1, m2, u, dO, ks, vn, dv, kds, stg, sc, end;
};

// Per-row scalars (C floats each) at Layout::sc.
enum { R_G, R_EG, R_DEC, R_BETA, R_QSDO, R_DBU, R_DGAM, R_E, R_ROWE, R_DBA, R_RK, R_RQ, R_COLE, R_COUNT };

template <typename Tin, bool MMA>
__host__ __device__ inline Layout layout(int dk) {
    constexpr int LDC = Strides<MMA>::LDC, LDV = Strides<MMA>::LDV;
    Layout L{};
    size_t off = 0;
    const size_t kq = align16(size_t(C) * kq_ld<Tin>(dk) * sizeof(Tin));
    L.k = off; off += kq;
    L.q = off; off += kq;
    // tensor-core path: second K / Q buffers, filled one chunk ahead
    L.k2 = off; off += MMA ? kq : 0;
    L.q2 = off; off += MMA ? kq : 0;
    L.s = off; off += align16(size_t(BV) * st_ld(dk) * 4);
    L.ds = off; off += align16(size_t(BV) * st_ld(dk) * 4);
    L.m0 = off; off += align16(size_t(C) * LDC * 4);
    L.m1 = off; off += align16(size_t(C) * LDC * 4);
    L.m2 = off; off += align16(size_t(C) * LDC * 4);
    L.u = off; off += align16(size_t(C) * LDV * 4);
    L.dO = off; off += align16(size_t(C) * LDV * 4);
    L.ks = off; off += align16(size_t(C) * LDV * 4);
    L.vn = off; off += align16(size_t(C) * LDV * 4);
    L.dv = off; off += align16(size_t(C) * LDV * 4);
    L.kds = off; off += align16(size_t(C) * LDV * 4);
    // tensor-core path: the next chunk's V and dO tiles (raw) and its beta and
    // g, copied in while this chunk is worked on
    L.stg = off; off += MMA ? align16(2 * size_t(C) * BV * sizeof(Tin) + 2 * size_t(C) * 4) : 0;
    L.sc = off; off += size_t(R_COUNT) * C * 4 + 64;  // + G_L, block partial sums
    L.end = off;
    return L;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// ---- TF32 tensor-core tiles for the products of the reverse walk ------------
// Used where the chunk-start states come from the tensor-core forward (bf16,
// dk = 128, dv a multiple of 128): every product of a phase below is one
// m16n8k8 mma.sync chain with fp32 accumulation; fp32 operands are rounded to
// TF32 (bf16 inputs are exact in it).  Fragments, lane = 4 g + t:
//   A (16 x 8, m x k): a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B (8 x 8,  k x n): b0 (t, g), b1 (t + 4, g)
//   C (16 x 8, m x n): c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1)
namespace tf32 {
__device__ __forceinline__ uint32_t cvt(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
// a bf16 value is exact in tf32: its bits, widened
__device__ __forceinline__ uint32_t bf(__nv_bfloat16 x) { return (uint32_t)__bfloat16_as_ushort(x) << 16; }
__device__ __forceinline__ float f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// sum over the four lanes t of a fragment row (lanes 4 g .. 4 g + 3)
__device__ __forceinline__ float row_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v + __shfl_xor_sync(0xffffffffu, v, 2);
}
// sum over the eight lanes g of a fragment column pair (lanes t, t + 4, ..)
__device__ __forceinline__ float col_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    return v + __shfl_xor_sync(0xffffffffu, v, 16);
}
}  // namespace tf32

// Asynchronous global -> shared copies (no register staging).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every committed group but the latest one has landed
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// The tensor-core phases (their own strides).
namespace tcp {
constexpr int LDC = Strides<true>::LDC, LDV = Strides<true>::LDV;

// The chunk's shared-memory operands, as the tensor-core phases see them.
struct BwdChunk {
    const __nv_bfloat16 *K, *Q;          // [C][ldkq]
    float *St, *dSt;                     // [BV][SLD]
    float *M0, *M1, *M2;                 // [C][LDC]
    float *U, *dO, *KS, *Vn, *dV, *KdS;  // [C][LDV]
    const float *G, *EG, *Dec, *Beta, *RK, *RQ;
    float *QSdO, *DBU, *DGam, *E, *RowE, *DBA, *ColE;
    int ldkq, SLD, L;
    float scale;
};

// K S, Q S, K dS' (M = 64 rows i, N = 32 columns, K = dk = 128) and from
// them KS, KdS, U = V - e^G KS and the row sums (Q S . dO) into QSdO
// (zeroed before).  Warp w: row tile w % 4, column tiles 2 (w / 4) + {0, 1}.
__device__ __forceinline__ void mma_ks(const BwdChunk &s, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3, nh = warp >> 2;
    const int r0 = 16 * (warp & 3) + g;
    float aks[2][4] = {}, aqs[2][4] = {}, akd[2][4] = {};
#pragma unroll 4
    for (int ks = 0; ks < 16; ++ks) {
        const int d = 8 * ks + t;
        const uint32_t k0 = tf32::bf(s.K[r0 * s.ldkq + d]), k1 = tf32::bf(s.K[(r0 + 8) * s.ldkq + d]),
                       k2 = tf32::bf(s.K[r0 * s.ldkq + d + 4]), k3 = tf32::bf(s.K[(r0 + 8) * s.ldkq + d + 4]);
        const uint32_t q0 = tf32::bf(s.Q[r0 * s.ldkq + d]), q1 = tf32::bf(s.Q[(r0 + 8) * s.ldkq + d]),
                       q2 = tf32::bf(s.Q[r0 * s.ldkq + d + 4]), q3 = tf32::bf(s.Q[(r0 + 8) * s.ldkq + d + 4]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int cc = 16 * nh + 8 * n + g;
            const uint32_t sb0 = tf32::cvt(s.St[cc * s.SLD + d]), sb1 = tf32::cvt(s.St[cc * s.SLD + d + 4]);
            const uint32_t db0 = tf32::cvt(s.dSt[cc * s.SLD + d]), db1 = tf32::cvt(s.dSt[cc * s.SLD + d + 4]);
            tf32::mma(aks[n], k0, k1, k2, k3, sb0, sb1);
            tf32::mma(aqs[n], q0, q1, q2, q3, sb0, sb1);
            tf32::mma(akd[n], k0, k1, k2, k3, db0, db1);
        }
    }
    float qd[2] = {0.0f, 0.0f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r0 + 8 * (e >> 1), cc = 16 * nh + 8 * n + 2 * t + (e & 1);
            const float rk = s.RK[i], ksv = rk * aks[n][e];
            s.KS[i * LDV + cc] = ksv;
            s.KdS[i * LDV + cc] = rk * akd[n][e];
            s.U[i * LDV + cc] = i < s.L ? s.U[i * LDV + cc] - s.EG[i] * ksv : 0.0f;
            qd[e >> 1] = fmaf(s.RQ[i] * aqs[n][e], s.dO[i * LDV + cc], qd[e >> 1]);
        }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const float v = tf32::row_sum(qd[hf]);
        if (t == 0) atomicAdd(s.QSdO + r0 + 8 * hf, v);
    }
}

// Vn = T diag(beta) U (T lower triangular: column tiles up to the diagonal).
__device__ __forceinline__ void mma_vn(const BwdChunk &s, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3, nh = warp >> 2, mt = warp & 3;
    const int r0 = 16 * mt + g;
    float acc[2][4] = {};
    for (int ks = 0; ks < 2 * mt + 2; ++ks) {
        const int j = 8 * ks + t;
        const uint32_t a0 = tf32::cvt(s.M1[r0 * LDC + j]), a1 = tf32::cvt(s.M1[(r0 + 8) * LDC + j]),
                       a2 = tf32::cvt(s.M1[r0 * LDC + j + 4]), a3 = tf32::cvt(s.M1[(r0 + 8) * LDC + j + 4]);
        const float bj0 = s.Beta[j], bj1 = s.Beta[j + 4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int cc = 16 * nh + 8 * n + g;
            tf32::mma(acc[n], a0, a1, a2, a3, tf32::cvt(bj0 * s.U[j * LDV + cc]),
                      tf32::cvt(bj1 * s.U[(j + 4) * LDV + cc]));
        }
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r0 + 8 * (e >> 1), cc = 16 * nh + 8 * n + 2 * t + (e & 1);
            s.Vn[i * LDV + cc] = i < s.L ? acc[n][e] : 0.0f;
        }
}

// dVn = diag(dec) KdS + P^T dO (P lower: row tiles from the diagonal down)
// and e_i = dec_i (KdS_i . Vn_i) into E (zeroed before).
__device__ __forceinline__ void mma_dvn(const BwdChunk &s, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3, nh = warp >> 2, mt = warp & 3;
    const int r0 = 16 * mt + g;
    float acc[2][4];
    float part[2] = {0.0f, 0.0f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r0 + 8 * (e >> 1), cc = 16 * nh + 8 * n + 2 * t + (e & 1);
            const float kd = s.KdS[i * LDV + cc];
            acc[n][e] = s.Dec[i] * kd;
            part[e >> 1] = fmaf(kd, s.Vn[i * LDV + cc], part[e >> 1]);
        }
    for (int ks = 2 * mt; ks < 8; ++ks) {
        const int j = 8 * ks + t;
        const uint32_t a0 = tf32::cvt(s.M2[j * LDC + r0]), a1 = tf32::cvt(s.M2[j * LDC + r0 + 8]),
                       a2 = tf32::cvt(s.M2[(j + 4) * LDC + r0]), a3 = tf32::cvt(s.M2[(j + 4) * LDC + r0 + 8]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int cc = 16 * nh + 8 * n + g;
            tf32::mma(acc[n], a0, a1, a2, a3, tf32::cvt(s.dO[j * LDV + cc]), tf32::cvt(s.dO[(j + 4) * LDV + cc]));
        }
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r0 + 8 * (e >> 1), cc = 16 * nh + 8 * n + 2 * t + (e & 1);
            s.dV[i * LDV + cc] = i < s.L ? acc[n][e] : 0.0f;
        }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const float v = tf32::row_sum(part[hf]);
        if (t == 0) atomicAdd(s.E + r0 + 8 * hf, s.Dec[r0 + 8 * hf] * v);
    }
}

// dR = T^T dVn, written over dVn (every warp reads dVn before any writes);
// dv = diag(beta) dR to global memory; row sums dR . U into DBU (zeroed
// before) and -beta (dR . KS) into DGam (holding scale (Q S . dO) before).
// Called by every thread of the CTA (it holds a barrier).  dv0: dv of the
// chunk's first row at the tile's first column; rows dvs apart.
__device__ __forceinline__ void mma_dr(const BwdChunk &s, int warp, int lane, float *dv0, long long dvs) {
    const int g = lane >> 2, t = lane & 3, nh = warp >> 2, mt = warp & 3;
    const int r0 = 16 * mt + g;
    float acc[2][4] = {};
    for (int ks = 2 * mt; ks < 8; ++ks) {
        const int j = 8 * ks + t;
        const uint32_t a0 = tf32::cvt(s.M1[j * LDC + r0]), a1 = tf32::cvt(s.M1[j * LDC + r0 + 8]),
                       a2 = tf32::cvt(s.M1[(j + 4) * LDC + r0]), a3 = tf32::cvt(s.M1[(j + 4) * LDC + r0 + 8]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int cc = 16 * nh + 8 * n + g;
            tf32::mma(acc[n], a0, a1, a2, a3, tf32::cvt(s.dV[j * LDV + cc]), tf32::cvt(s.dV[(j + 4) * LDV + cc]));
        }
    }
    __syncthreads();  // every warp has read dVn
    float bu[2] = {0.0f, 0.0f}, bk[2] = {0.0f, 0.0f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = r0 + 8 * hf, cc = 16 * nh + 8 * n + 2 * t;
            const float d0 = i < s.L ? acc[n][2 * hf] : 0.0f, d1 = i < s.L ? acc[n][2 * hf + 1] : 0.0f;
            s.dV[i * LDV + cc] = d0;
            s.dV[i * LDV + cc + 1] = d1;
            if (i < s.L)
                *reinterpret_cast<float2 *>(dv0 + i * dvs + cc) = make_float2(s.Beta[i] * d0, s.Beta[i] * d1);
            bu[hf] = fmaf(d0, s.U[i * LDV + cc], fmaf(d1, s.U[i * LDV + cc + 1], bu[hf]));
            bk[hf] = fmaf(d0, s.KS[i * LDV + cc], fmaf(d1, s.KS[i * LDV + cc + 1], bk[hf]));
        }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const float u = tf32::row_sum(bu[hf]), k = tf32::row_sum(bk[hf]);
        if (t == 0) {
            const int i = r0 + 8 * hf;
            atomicAdd(s.DBU + i, u);
            atomicAdd(s.DGam + i, -s.Beta[i] * k);
        }
    }
}

// Of the tile (mt, nt) of the lower band (nt <= 2 mt + 1) numbered k in
// row-tile order: k = mt (mt + 1) + nt.
__device__ __forceinline__ int band_mt(int k) { return k < 2 ? 0 : (k < 6 ? 1 : (k < 12 ? 2 : 3)); }

// dA = dR Vn^T, dP = dO Vn^T over the band of 16 x 8 tiles that holds j <= i
// (20 tiles, M = 64, N = 64, K = 32), then per element (j <= i < L)
//   M_ij = -beta_i D_ij dA_ij,  WP_ij = scale D_ij dP_ij,
//   E_ij = beta_i dA_ij A'_ij + dP_ij P_ij   (A' = -(K K^T . D), dA_ii = 0)
// over M0, M1, M2 within the band, with row sums of E into RowE, column
// sums of E into ColE and row sums of dA . A' into DBA (all zeroed before).
__device__ __forceinline__ void mma_e(const BwdChunk &s, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3;
    for (int k = warp; k < 20; k += 8) {
        const int mt = band_mt(k), nt = k - mt * (mt + 1);
        const int r0 = 16 * mt + g, jb = 8 * nt + g;
        float da[4] = {}, dp[4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int cc = 8 * ks + t;
            const uint32_t b0 = tf32::cvt(s.Vn[jb * LDV + cc]), b1 = tf32::cvt(s.Vn[jb * LDV + cc + 4]);
            tf32::mma(da, tf32::cvt(s.dV[r0 * LDV + cc]), tf32::cvt(s.dV[(r0 + 8) * LDV + cc]),
                      tf32::cvt(s.dV[r0 * LDV + cc + 4]), tf32::cvt(s.dV[(r0 + 8) * LDV + cc + 4]), b0, b1);
            tf32::mma(dp, tf32::cvt(s.dO[r0 * LDV + cc]), tf32::cvt(s.dO[(r0 + 8) * LDV + cc]),
                      tf32::cvt(s.dO[r0 * LDV + cc + 4]), tf32::cvt(s.dO[(r0 + 8) * LDV + cc + 4]), b0, b1);
        }
        float rowe[2] = {0.0f, 0.0f}, dba[2] = {0.0f, 0.0f}, cole[2] = {0.0f, 0.0f};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r0 + 8 * (e >> 1), j = 8 * nt + 2 * t + (e & 1);
            float m = 0.0f, wp = 0.0f, ee = 0.0f;
            if (i < s.L && j <= i) {
                const float dav = j == i ? 0.0f : da[e];
                const float ap = s.M0[i * LDC + j], pp = s.M2[i * LDC + j];
                const float D = expf(s.G[i] - s.G[j]);
                ee = dav * s.Beta[i] * ap + dp[e] * pp;
                dba[e >> 1] = fmaf(dav, ap, dba[e >> 1]);
                m = -s.Beta[i] * D * dav;
                wp = s.scale * D * dp[e];
                rowe[e >> 1] += ee;
                cole[e & 1] += ee;
            }
            s.M0[i * LDC + j] = m;
            s.M1[i * LDC + j] = wp;
            s.M2[i * LDC + j] = ee;
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float re = tf32::row_sum(rowe[hf]), db = tf32::row_sum(dba[hf]);
            if (t == 0) {
                atomicAdd(s.RowE + r0 + 8 * hf, re);
                atomicAdd(s.DBA + r0 + 8 * hf, db);
            }
            const float ce = tf32::col_sum(cole[hf]);
            if (g == 0) atomicAdd(s.ColE + 8 * nt + 2 * t + hf, ce);
        }
    }
    // (right of the band, j > i: M0 and M2 hold the zeros of -(K K^T . D)
    // and P, M1 those of T, as the later phases need)
}

// dq, dk of the chunk's rows (M = 64 rows i, N = dk = 128 columns d):
//   dq_i = scale e^{G_i} S dO_i + sum_j WP_ij rk_j k_j
//   dk_i = dec_i dS' Vn_i - beta_i e^{G_i} S dR_i + sum_j (M_ij + M_ji) rk_j k_j
//          + sum_j WP_ji rq_j q_j
// added into dq0 / dk0 (the chunk's first row, rows dqs apart) with fp32
// atomics.  Warp w: row tile w % 4, columns 64 (w / 4) .. + 63.
__device__ __forceinline__ void mma_dqdk(const BwdChunk &s, int warp, int lane, float *dq0, float *dk0,
                                         long long dqs) {
    const int g = lane >> 2, t = lane & 3, mt = warp & 3, nq = warp >> 2;
    const int i0 = 16 * mt + g, i1 = i0 + 8;
    float gq[8][4] = {}, gk[8][4] = {};
    {
        const float fq0 = s.scale * s.EG[i0], fq1 = s.scale * s.EG[i1];
        const float fd0 = s.Dec[i0], fd1 = s.Dec[i1];
        const float fr0 = -s.Beta[i0] * s.EG[i0], fr1 = -s.Beta[i1] * s.EG[i1];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int cc = 8 * ks + t;
            const uint32_t o0 = tf32::cvt(fq0 * s.dO[i0 * LDV + cc]), o1 = tf32::cvt(fq1 * s.dO[i1 * LDV + cc]),
                           o2 = tf32::cvt(fq0 * s.dO[i0 * LDV + cc + 4]), o3 = tf32::cvt(fq1 * s.dO[i1 * LDV + cc + 4]);
            const uint32_t v0 = tf32::cvt(fd0 * s.Vn[i0 * LDV + cc]), v1 = tf32::cvt(fd1 * s.Vn[i1 * LDV + cc]),
                           v2 = tf32::cvt(fd0 * s.Vn[i0 * LDV + cc + 4]), v3 = tf32::cvt(fd1 * s.Vn[i1 * LDV + cc + 4]);
            const uint32_t r0 = tf32::cvt(fr0 * s.dV[i0 * LDV + cc]), r1 = tf32::cvt(fr1 * s.dV[i1 * LDV + cc]),
                           r2 = tf32::cvt(fr0 * s.dV[i0 * LDV + cc + 4]), r3 = tf32::cvt(fr1 * s.dV[i1 * LDV + cc + 4]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int d = 64 * nq + 8 * nt + g;
                const uint32_t sb0 = tf32::cvt(s.St[cc * s.SLD + d]), sb1 = tf32::cvt(s.St[(cc + 4) * s.SLD + d]);
                const uint32_t db0 = tf32::cvt(s.dSt[cc * s.SLD + d]), db1 = tf32::cvt(s.dSt[(cc + 4) * s.SLD + d]);
                tf32::mma(gq[nt], o0, o1, o2, o3, sb0, sb1);
                tf32::mma(gk[nt], v0, v1, v2, v3, db0, db1);
                tf32::mma(gk[nt], r0, r1, r2, r3, sb0, sb1);
            }
        }
    }
    for (int ks = 0; ks < 8; ++ks) {
        const int j = 8 * ks + t;
        const float rk0 = s.RK[j], rk1 = s.RK[j + 4], rq0 = s.RQ[j], rq1 = s.RQ[j + 4];
        const bool lower = ks <= 2 * mt + 1, upper = ks >= 2 * mt;  // WP_ij, WP_ji can be nonzero
        const uint32_t w0 = tf32::cvt(rk0 * s.M1[i0 * LDC + j]), w1 = tf32::cvt(rk0 * s.M1[i1 * LDC + j]),
                       w2 = tf32::cvt(rk1 * s.M1[i0 * LDC + j + 4]), w3 = tf32::cvt(rk1 * s.M1[i1 * LDC + j + 4]);
        const uint32_t m0 = tf32::cvt(rk0 * (s.M0[i0 * LDC + j] + s.M0[j * LDC + i0])),
                       m1 = tf32::cvt(rk0 * (s.M0[i1 * LDC + j] + s.M0[j * LDC + i1])),
                       m2 = tf32::cvt(rk1 * (s.M0[i0 * LDC + j + 4] + s.M0[(j + 4) * LDC + i0])),
                       m3 = tf32::cvt(rk1 * (s.M0[i1 * LDC + j + 4] + s.M0[(j + 4) * LDC + i1]));
        const uint32_t x0 = tf32::cvt(rq0 * s.M1[j * LDC + i0]), x1 = tf32::cvt(rq0 * s.M1[j * LDC + i1]),
                       x2 = tf32::cvt(rq1 * s.M1[(j + 4) * LDC + i0]), x3 = tf32::cvt(rq1 * s.M1[(j + 4) * LDC + i1]);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int d = 64 * nq + 8 * nt + g;
            const uint32_t kb0 = tf32::bf(s.K[j * s.ldkq + d]), kb1 = tf32::bf(s.K[(j + 4) * s.ldkq + d]);
            if (lower) tf32::mma(gq[nt], w0, w1, w2, w3, kb0, kb1);
            tf32::mma(gk[nt], m0, m1, m2, m3, kb0, kb1);
            if (upper) tf32::mma(gk[nt], x0, x1, x2, x3, tf32::bf(s.Q[j * s.ldkq + d]), tf32::bf(s.Q[(j + 4) * s.ldkq + d]));
        }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int i = hf ? i1 : i0;
            if (i >= s.L) continue;
            const int d = 64 * nq + 8 * nt + 2 * t;
            atomicAdd(reinterpret_cast<float2 *>(dq0 + i * dqs + d), make_float2(gq[nt][2 * hf], gq[nt][2 * hf + 1]));
            atomicAdd(reinterpret_cast<float2 *>(dk0 + i * dqs + d), make_float2(gk[nt][2 * hf], gk[nt][2 * hf + 1]));
        }
}

// dS = e^{G_L} dS' + scale Q^T diag(e^G) dO - K^T diag(beta e^G) dR, in
// place over dS'^T (M = dk = 128 rows d, N = 32 columns, K = the chunk's
// rows).  Warp w: rows 16 w .. 16 w + 15, every column.
__device__ __forceinline__ void mma_ds(const BwdChunk &s, int warp, int lane, float eGL) {
    const int g = lane >> 2, t = lane & 3;
    const int d0 = 16 * warp + g, d1 = d0 + 8;
    float acc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        const int cc = 8 * n + 2 * t;
        acc[n][0] = eGL * s.dSt[cc * s.SLD + d0];
        acc[n][1] = eGL * s.dSt[(cc + 1) * s.SLD + d0];
        acc[n][2] = eGL * s.dSt[cc * s.SLD + d1];
        acc[n][3] = eGL * s.dSt[(cc + 1) * s.SLD + d1];
    }
    const int kend = (s.L + 7) >> 3;
    for (int ks = 0; ks < kend; ++ks) {
        const int i = 8 * ks + t;
        const float fq0 = s.scale * s.EG[i] * s.RQ[i], fq1 = s.scale * s.EG[i + 4] * s.RQ[i + 4];
        const float fk0 = -s.Beta[i] * s.EG[i] * s.RK[i], fk1 = -s.Beta[i + 4] * s.EG[i + 4] * s.RK[i + 4];
        const uint32_t q0 = tf32::cvt(fq0 * tf32::f(s.Q[i * s.ldkq + d0])),
                       q1 = tf32::cvt(fq0 * tf32::f(s.Q[i * s.ldkq + d1])),
                       q2 = tf32::cvt(fq1 * tf32::f(s.Q[(i + 4) * s.ldkq + d0])),
                       q3 = tf32::cvt(fq1 * tf32::f(s.Q[(i + 4) * s.ldkq + d1]));
        const uint32_t k0 = tf32::cvt(fk0 * tf32::f(s.K[i * s.ldkq + d0])),
                       k1 = tf32::cvt(fk0 * tf32::f(s.K[i * s.ldkq + d1])),
                       k2 = tf32::cvt(fk1 * tf32::f(s.K[(i + 4) * s.ldkq + d0])),
                       k3 = tf32::cvt(fk1 * tf32::f(s.K[(i + 4) * s.ldkq + d1]));
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int cc = 8 * n + g;
            tf32::mma(acc[n], q0, q1, q2, q3, tf32::cvt(s.dO[i * LDV + cc]), tf32::cvt(s.dO[(i + 4) * LDV + cc]));
            tf32::mma(acc[n], k0, k1, k2, k3, tf32::cvt(s.dV[i * LDV + cc]), tf32::cvt(s.dV[(i + 4) * LDV + cc]));
        }
    }
#pragma unroll
    for (int n = 0; n < 4; ++n) {
        const int cc = 8 * n + 2 * t;
        s.dSt[cc * s.SLD + d0] = acc[n][0];
        s.dSt[(cc + 1) * s.SLD + d0] = acc[n][1];
        s.dSt[cc * s.SLD + d1] = acc[n][2];
        s.dSt[(cc + 1) * s.SLD + d1] = acc[n][3];
    }
}

}  // namespace tcp

// MMA: the products run as TF32 tensor-core tiles (bf16 inputs, dk = 128,
// dv a multiple of BV; the states come from the tensor-core forward); else
// as fp32 FMAs.
template <typename Tin, bool MMA>
__global__ void __launch_bounds__(NT) simt_bwd(Params p) {
    constexpr int LDC = Strides<MMA>::LDC, LDV = Strides<MMA>::LDV;
    extern __shared__ __align__(16) unsigned char smem[];
    // the tensor-core path runs dk = 128 only (bwd_launch): a constant there,
    // so that the index arithmetic on it needs no division
    const int dk = MMA ? 128 : p.dk, dv = p.dv, Nk = p.Nk, Nv = p.Nv;
    const int nvt = (dv + BV - 1) / BV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vt = blockIdx.x % nvt;
    const int h = (blockIdx.x / nvt) % Nv;
    const int n = seq_of_rank(p, blockIdx.x / (nvt * Nv), lane);  // longest sequences first
    const int hk = h / (Nv / Nk);
    const int v0 = vt * BV;
    const int bvw = min(BV, dv - v0);
    const int c = lane;  // value column of the C x BV tiles in the row-per-warp loops
    const int SLD = st_ld(dk);

    const Layout lay = layout<Tin, MMA>(dk);
    // K / Q buffers (two on the tensor-core path: chunk ci in buffer ci & 1)
    Tin *const sK0 = reinterpret_cast<Tin *>(smem + lay.k), *const sK1 = reinterpret_cast<Tin *>(smem + lay.k2);
    Tin *const sQ0 = reinterpret_cast<Tin *>(smem + lay.q), *const sQ1 = reinterpret_cast<Tin *>(smem + lay.q2);
    Tin *sK = sK0;
    Tin *sQ = sQ0;
    float *sSt = reinterpret_cast<float *>(smem + lay.s);    // [BV][SLD]: S^T, S = state the chunk starts from
    float *sdSt = reinterpret_cast<float *>(smem + lay.ds);  // [BV][SLD]: dS'^T, gradient of the state it hands on
    float *sM0 = reinterpret_cast<float *>(smem + lay.m0);   // -(K K^T . D), then M
    float *sM1 = reinterpret_cast<float *>(smem + lay.m1);   // T, then scale D . dP
    float *sM2 = reinterpret_cast<float *>(smem + lay.m2);   // P, then E
    float *sU = reinterpret_cast<float *>(smem + lay.u);     // V, then U
    float *sdO = reinterpret_cast<float *>(smem + lay.dO);
    float *sKS = reinterpret_cast<float *>(smem + lay.ks);
    float *sVn = reinterpret_cast<float *>(smem + lay.vn);
    float *sdV = reinterpret_cast<float *>(smem + lay.dv);   // dVn, then dR
    float *sKdS = reinterpret_cast<float *>(smem + lay.kds);
    float *sc = reinterpret_cast<float *>(smem + lay.sc);
    // staged V, dO (C x BV, raw) and beta, g (C) of the chunk to come
    Tin *const sVst = reinterpret_cast<Tin *>(smem + lay.stg);
    Tin *const sdOst = sVst + C * BV;
    float *const sBst = reinterpret_cast<float *>(sdOst + C * BV);
    float *const sGst = sBst + C;
    float *sG = sc + R_G * C, *sEG = sc + R_EG * C, *sDec = sc + R_DEC * C, *sBeta = sc + R_BETA * C;
    float *sQSdO = sc + R_QSDO * C, *sDBU = sc + R_DBU * C, *sDGam = sc + R_DGAM * C;
    float *sE = sc + R_E * C, *sRowE = sc + R_ROWE * C, *sDBA = sc + R_DBA * C;
    // inverse key / query norms of the chunk's rows (1 without kQkL2Norm):
    // every product below that reads a k or q row takes the row's factor, so
    // the gradients the CTA adds up are those of the normalised rows
    float *sRK = sc + R_RK * C, *sRQ = sc + R_RQ * C;
    float *sColE = sc + R_COLE * C;  // column sums of E (tensor-core path)
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    float *sGL = sc + R_COUNT * C;      // [0]: G_L
    float *sRed = sGL + 4;              // [8]: per-warp partial <S, dS'>
    const int ldkq = kq_ld<Tin>(dk);
    tcp::BwdChunk bc{reinterpret_cast<const __nv_bfloat16 *>(sK), reinterpret_cast<const __nv_bfloat16 *>(sQ),
                sSt, sdSt, sM0, sM1, sM2, sU, sdO, sKS, sVn, sdV, sKdS,
                sG, sEG, sDec, sBeta, sRK, sRQ, sQSdO, sDBU, sDGam, sE, sRowE, sDBA, sColE,
                ldkq, SLD, 0, p.scale};

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dout = static_cast<const Tin *>(p.dout);

    long long bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        if (bos < 0 || eos < bos || eos > p.tokens) {
            if (tid == 0) atomicOr(p.status, kStatusBadSeq);
            bos = eos = 0;
        }
    } else {
        bos = (long long)n * p.T;
        eos = bos + p.T;
    }

    // dS' of the last chunk = dht (or 0)
    const size_t sbase = ((size_t)n * Nv + h) * dk * dv;
    for (int idx = tid; idx < dk * BV; idx += NT) {
        const int d = idx / BV, cc = idx - d * BV;
        sdSt[cc * SLD + d] = (p.dht && cc < bvw) ? p.dht[sbase + (size_t)d * dv + v0 + cc] : 0.0f;
    }

    const long long nch = (eos - bos + C - 1) / C;
    // asynchronous copies of chunk cj's K and Q rows (rows past its length
    // zeroed) and of the state it starts from
    auto load_kq = [&](long long cj, Tin *dK, Tin *dQ) {
        constexpr int VEC = 16 / sizeof(Tin);
        const long long tj = bos + cj * C;
        const int Lj = (eos - tj) < C ? (int)(eos - tj) : C;
        const int per_row = dk / VEC;
        for (int idx = tid; idx < Lj * per_row; idx += NT) {
            const int i = idx / per_row, cv = idx - i * per_row;
            const long long go = ((tj + i) * Nk + hk) * (long long)dk + cv * VEC;
            cp_async16(dK + i * ldkq + cv * VEC, k + go);
            cp_async16(dQ + i * ldkq + cv * VEC, q + go);
        }
        for (int idx = Lj * ldkq + tid; idx < C * ldkq; idx += NT) dK[idx] = dQ[idx] = Tin(0.0f);
    };
    auto load_hs = [&](long long cj) {
        const long long tj = bos + cj * C;
        const float *hs = p.hs + ((size_t)h * p.nslots + (size_t)(tj / C + n)) * dk * dv + v0;
        for (int idx = tid; idx < dk * BV; idx += NT) {
            const int d = idx / BV, cc = idx - d * BV;
            if (cc < bvw)
                cp_async4(sSt + cc * SLD + d, hs + (size_t)d * dv + cc);
            else
                sSt[cc * SLD + d] = 0.0f;
        }
    };
    // tensor-core path (bf16, dv a multiple of 128, so every tile is BV
    // columns wide): chunk cj's V and dO rows, beta and g into the staging
    // buffer (rows past its length are not read)
    auto stage_vdo = [&](long long cj) {
        const long long tj = bos + cj * C;
        const int Lj = (eos - tj) < C ? (int)(eos - tj) : C;
        constexpr int PARTS = BV * sizeof(Tin) / 16;  // 16-byte pieces of a tile row
        for (int idx = tid; idx < Lj * PARTS; idx += NT) {
            const int i = idx / PARTS, part = idx - i * PARTS;
            const long long off = ((tj + i) * Nv + h) * (long long)dv + v0 + part * (16 / sizeof(Tin));
            cp_async16(sVst + i * BV + part * (16 / sizeof(Tin)), v + off);
            cp_async16(sdOst + i * BV + part * (16 / sizeof(Tin)), dout + off);
        }
        if (tid < Lj) {
            cp_async4(sBst + tid, p.beta + (tj + tid) * Nv + h);
            if (p.g) cp_async4(sGst + tid, p.g + (tj + tid) * Nv + h);
        }
    };
    if (MMA && nch > 0) {
        load_kq(nch - 1, ((nch - 1) & 1) ? sK1 : sK0, ((nch - 1) & 1) ? sQ1 : sQ0);
        load_hs(nch - 1);
        stage_vdo(nch - 1);
        cp_async_commit();
    }
    for (long long ci = nch - 1; ci >= 0; --ci) {
        const long long t0 = bos + ci * C;
        const int pc = (int)(nch - 1 - ci);  // position in the walk (phase stamps)
        (void)pc;
        const int L = (eos - t0) < C ? (int)(eos - t0) : C;
        __syncthreads();  // the previous (later) chunk is done with every buffer

        // ---- load --------------------------------------------------------
        // K, Q rows and the state: asynchronous copies, in flight while V and
        // dO are converted.  On the tensor-core path this chunk's were issued
        // one chunk ahead (K, Q) and during the previous chunk's dS update
        // (the state); the next chunk's K and Q go out now.
        if constexpr (MMA) {
            // the chunk's -(K K^T . D), P and T, which the forward pass's WY
            // kernel kept (Params::wyx): in flight until they are needed
            const float *wx = p.wyx + ((size_t)h * p.nslots + (size_t)(t0 / C + n)) * 3 * 4096;
            for (int idx = tid; idx < 3 * 64 * 16; idx += NT) {
                const int mtx = idx >> 10, rr = (idx >> 4) & 63, c4 = idx & 15;
                float *dst = (mtx == 0 ? sM0 : (mtx == 1 ? sM2 : sM1)) + rr * LDC + 4 * c4;
                cp_async16(dst, wx + mtx * 4096 + rr * 64 + 4 * c4);
            }
            cp_async_commit();
            sK = (ci & 1) ? sK1 : sK0;
            sQ = (ci & 1) ? sQ1 : sQ0;
            bc.K = reinterpret_cast<const __nv_bfloat16 *>(sK);
            bc.Q = reinterpret_cast<const __nv_bfloat16 *>(sQ);
            if (ci > 0) {
                load_kq(ci - 1, (ci & 1) ? sK0 : sK1, (ci & 1) ? sQ0 : sQ1);
                cp_async_commit();
            }
        } else {
            load_kq(ci, sK, sQ);
            load_hs(ci);
        }
        if (MMA && ci > 0)
            cp_async_wait_prev2();  // not the matrices above, nor the next chunk's K, Q
        else if (MMA)
            cp_async_wait_prev();
        else
            cp_async_wait_all();
        if constexpr (MMA) {
            // V, dO, beta and g were staged while the chunk before was worked on
            __syncthreads();
            for (int idx = tid; idx < C * BV; idx += NT) {
                const int i = idx / BV, cc = idx - i * BV;
                const bool in = i < L;
                sU[i * LDV + cc] = in ? to_f(sVst[i * BV + cc]) : 0.0f;
                sdO[i * LDV + cc] = in ? to_f(sdOst[i * BV + cc]) : 0.0f;
            }
            if (tid < C) {
                sBeta[tid] = tid < L ? sBst[tid] : 0.0f;
                sG[tid] = (tid < L && p.g) ? sGst[tid] : 0.0f;
                // row sums the tensor-core phases add into
                sQSdO[tid] = sE[tid] = sRowE[tid] = sDBA[tid] = sDBU[tid] = sColE[tid] = 0.0f;
            }
        } else {
            for (int idx = tid; idx < C * BV; idx += NT) {
                const int i = idx / BV, cc = idx - i * BV;
                const bool in = i < L && cc < bvw;
                const long long off = ((t0 + i) * Nv + h) * (long long)dv + v0 + cc;
                sU[i * LDV + cc] = in ? to_f(v[off]) : 0.0f;
                sdO[i * LDV + cc] = in ? to_f(dout[off]) : 0.0f;
            }
            if (tid < C) {
                sBeta[tid] = tid < L ? p.beta[(t0 + tid) * Nv + h] : 0.0f;
                sG[tid] = (tid < L && p.g) ? p.g[(t0 + tid) * Nv + h] : 0.0f;
            }
        }
        bc.L = L;
        __syncthreads();
        // the staging buffer is free: the chunk before this one (next in the walk)
        if (MMA && ci > 0) {
            stage_vdo(ci - 1);
            cp_async_commit();
        }

        // ---- gate prefix sum (warp 0); <S, dS'> partials (every warp) ----
        if (warp == 0) {
            float a = sG[lane], b = sG[lane + 32];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float ta = __shfl_up_sync(0xffffffffu, a, off);
                const float tb = __shfl_up_sync(0xffffffffu, b, off);
                if (lane >= off) { a += ta; b += tb; }
            }
            b += __shfl_sync(0xffffffffu, a, 31);
            const float ga = __shfl_sync(0xffffffffu, a, (L - 1) & 31);
            const float gb = __shfl_sync(0xffffffffu, b, (L - 1) & 31);
            const float GL = (L - 1) < 32 ? ga : gb;
            sG[lane] = a;
            sG[lane + 32] = b;
            sEG[lane] = lane < L ? expf(a) : 0.0f;
            sEG[lane + 32] = lane + 32 < L ? expf(b) : 0.0f;
            sDec[lane] = lane < L ? expf(GL - a) : 0.0f;
            sDec[lane + 32] = lane + 32 < L ? expf(GL - b) : 0.0f;
            if (lane == 0) sGL[0] = GL;
        } else {
            for (int rr = warp - 1; rr < 2 * C; rr += 7) {
                const int i = rr & (C - 1);
                float ss = 0.0f;
                if (qkn) {
                    const Tin *x = (rr < C ? sK : sQ) + i * ldkq;
                    for (int d = lane; d < dk; d += 32) {
                        const float f = to_f(x[d]);
                        ss = fmaf(f, f, ss);
                    }
                    ss = warp_sum(ss);
                }
                if (lane == 0) (rr < C ? sRK : sRQ)[i] = qkn ? rsqrtf(fmaxf(ss, 1e-24f)) : 1.0f;
            }
        }
        {
            float part = 0.0f;
            for (int idx = tid; idx < dk * BV; idx += NT) {
                const int cc = idx / dk, d = idx - cc * dk;
                part = fmaf(sSt[cc * SLD + d], sdSt[cc * SLD + d], part);
            }
            part = warp_sum(part);
            if (lane == 0) sRed[warp] = part;
        }
        __syncthreads();

        if constexpr (MMA) {
            // -(K K^T . D), P and T have landed (not the next chunk's K, Q
            // and staged V, dO)
            if (ci > 0)
                cp_async_wait_prev2();
            else
                cp_async_wait_all();
            __syncthreads();
        } else {
            // ---- -(K K^T . D) (strictly lower) and P (lower) --------------
            simt::kq_products<NT>(sK, sQ, ldkq, dk, L, tid, [&](int i, int j, float kk, float qk) {
                float a = 0.0f, pv = 0.0f;
                if (i < L && j <= i) {
                    const float D = expf(sG[i] - sG[j]) * sRK[j];
                    if (j < i) a = -kk * D * sRK[i];
                    pv = p.scale * qk * D * sRQ[i];
                }
                sM0[i * LDC + j] = a;
                sM2[i * LDC + j] = pv;
            });
            __syncthreads();

            // ---- T = (I - A)^-1, A_im = beta_i sM0_im (blocked; sVn,
            // written later, is its scratch) ---------------------------------
            simt::solve_T_blocked<NT>(sM0, LDC, sBeta, sM1, LDC, sVn, L, tid);
        }
        // ---- K S, Q S (.dO), K dS'; U = V - e^G K S ------------------------
        // thread: rows i0, i0 + 1; columns cg + 8 x (x < 4)
        if constexpr (MMA) {
            tcp::mma_ks(bc, warp, lane);
        } else {
            const int i0 = 2 * (tid >> 3), cg = tid & 7;
            float ks[2][4], qs[2][4], kd[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) ks[r][x] = qs[r][x] = kd[r][x] = 0.0f;
            for (int d = 0; d < dk; d += 4) {
                float4 kr[2], qr[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    kr[r] = ld4(sK + (i0 + r) * ldkq + d);
                    qr[r] = ld4(sQ + (i0 + r) * ldkq + d);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(sSt + (cg + 8 * x) * SLD + d);
                    const float4 d4 = *reinterpret_cast<const float4 *>(sdSt + (cg + 8 * x) * SLD + d);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        ks[r][x] = fmaf(kr[r].x, s4.x, fmaf(kr[r].y, s4.y, fmaf(kr[r].z, s4.z, fmaf(kr[r].w, s4.w, ks[r][x]))));
                        qs[r][x] = fmaf(qr[r].x, s4.x, fmaf(qr[r].y, s4.y, fmaf(qr[r].z, s4.z, fmaf(qr[r].w, s4.w, qs[r][x]))));
                        kd[r][x] = fmaf(kr[r].x, d4.x, fmaf(kr[r].y, d4.y, fmaf(kr[r].z, d4.z, fmaf(kr[r].w, d4.w, kd[r][x]))));
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = i0 + r;
                const float rk = sRK[i], rq = sRQ[i];
                float qd = 0.0f;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int cc = cg + 8 * x;
                    const float ksv = rk * ks[r][x];
                    sKS[i * LDV + cc] = ksv;
                    sKdS[i * LDV + cc] = rk * kd[r][x];
                    sU[i * LDV + cc] = i < L ? sU[i * LDV + cc] - sEG[i] * ksv : 0.0f;
                    qd = fmaf(rq * qs[r][x], sdO[i * LDV + cc], qd);
                }
                // the eight threads of a row pair are lanes 8 m .. 8 m + 7
                qd += __shfl_xor_sync(0xffffffffu, qd, 1);
                qd += __shfl_xor_sync(0xffffffffu, qd, 2);
                qd += __shfl_xor_sync(0xffffffffu, qd, 4);
                if (cg == 0) sQSdO[i] = qd;
            }
        }
        __syncthreads();

        // ---- Vn = T diag(beta) U ------------------------------------------
        if constexpr (MMA) {
            if (tid < C) sDGam[tid] = p.scale * sQSdO[tid];  // dR's row sums are added to it
            tcp::mma_vn(bc, warp, lane);
        } else {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
            for (int j = 0; j < L; ++j) {
                const float rj = sBeta[j] * sU[j * LDV + c];
#pragma unroll
                for (int r = 0; r < 8; ++r) acc[r] = fmaf(sM1[(warp + 8 * r) * LDC + j], rj, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                sVn[i * LDV + c] = i < L ? acc[r] : 0.0f;
            }
        }
        __syncthreads();

        // ---- dVn = diag(dec) K dS' + P^T dO; e_i --------------------------
        if constexpr (MMA) {
            tcp::mma_dvn(bc, warp, lane);
        } else {
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                float acc = sDec[i] * sKdS[i * LDV + c];
                for (int j = i; j < L; ++j) acc = fmaf(sM2[j * LDC + i], sdO[j * LDV + c], acc);
                sdV[i * LDV + c] = i < L ? acc : 0.0f;
                const float e = warp_sum(sKdS[i * LDV + c] * sVn[i * LDV + c]);
                if (lane == 0) sE[i] = sDec[i] * e;
            }
        }
        __syncthreads();

        // ---- dR = T^T dVn; dv = diag(beta) dR ------------------------------
        if constexpr (MMA) {
            tcp::mma_dr(bc, warp, lane, p.dvv + (t0 * Nv + h) * (long long)dv + v0, (long long)Nv * dv);
        } else {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
            for (int j = 0; j < L; ++j) {
                const float dvj = sdV[j * LDV + c];
#pragma unroll
                for (int r = 0; r < 8; ++r) acc[r] = fmaf(sM1[j * LDC + warp + 8 * r], dvj, acc[r]);
            }
            __syncthreads();  // every thread has read dVn
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                const float dr = i < L ? acc[r] : 0.0f;
                sdV[i * LDV + c] = dr;
                if (i < L && c < bvw) p.dvv[((t0 + i) * Nv + h) * (long long)dv + v0 + c] = sBeta[i] * dr;
                const float bu = warp_sum(dr * sU[i * LDV + c]);
                const float bk = warp_sum(dr * sKS[i * LDV + c]);
                if (lane == 0) {
                    sDBU[i] = bu;
                    sDGam[i] = p.scale * sQSdO[i] - sBeta[i] * bk;
                }
            }
        }
        __syncthreads();

        // ---- dA, dP and E (row i per warp, columns j = lane, lane + 32) ----
        if constexpr (MMA) {
            tcp::mma_e(bc, warp, lane);
        } else {
#pragma unroll 1
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                float rowE = 0.0f, dba = 0.0f;
#pragma unroll
                for (int hj = 0; hj < 2; ++hj) {
                    const int j = lane + 32 * hj;
                    float m = 0.0f, wp = 0.0f, e = 0.0f;
                    if (i < L && j <= i) {
                        float da = 0.0f, dp = 0.0f;
#pragma unroll 8
                        for (int cc = 0; cc < BV; ++cc) {
                            const float vnj = sVn[j * LDV + cc];
                            da = fmaf(sdV[i * LDV + cc], vnj, da);
                            dp = fmaf(sdO[i * LDV + cc], vnj, dp);
                        }
                        if (j == i) da = 0.0f;
                        const float ap = sM0[i * LDC + j];   // -(k_i.k_j) D_ij
                        const float pp = sM2[i * LDC + j];   // P_ij
                        const float D = expf(sG[i] - sG[j]);
                        e = da * sBeta[i] * ap + dp * pp;
                        dba = fmaf(da, ap, dba);
                        m = -sBeta[i] * D * da;
                        wp = p.scale * D * dp;
                    }
                    rowE += e;
                    sM0[i * LDC + j] = m;
                    sM1[i * LDC + j] = wp;
                    sM2[i * LDC + j] = e;
                }
                rowE = warp_sum(rowE);
                dba = warp_sum(dba);
                if (lane == 0) {
                    sRowE[i] = rowE;
                    sDBA[i] = dba;
                }
            }
        }
        __syncthreads();

        // ---- warp 0: dbeta, dG and dg ------------------------------------
        if (warp == 0) {
            float dG[2], db[2];
            float esum = 0.0f;
#pragma unroll
            for (int hj = 0; hj < 2; ++hj) {
                const int i = lane + 32 * hj;
                float colE = 0.0f;
                if constexpr (MMA)
                    colE = sColE[i];
                else
                    for (int i2 = i; i2 < L; ++i2) colE += sM2[i2 * LDC + i];
                dG[hj] = i < L ? sEG[i] * sDGam[i] + sRowE[i] - colE - sE[i] : 0.0f;
                db[hj] = sDBU[i] + sDBA[i];
                esum += i < L ? sE[i] : 0.0f;
            }
            esum = warp_sum(esum);
            float red = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) red += sRed[w];
            const float extra = esum + expf(sGL[0]) * red;
            if (lane == ((L - 1) & 31)) {
                if ((L - 1) >> 5) dG[1] += extra; else dG[0] += extra;
            }
            // dg_t = sum_{i >= t} dG_i: suffix sums over the 64 rows
            float a = dG[0], b = dG[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float ta = __shfl_down_sync(0xffffffffu, a, off);
                const float tb = __shfl_down_sync(0xffffffffu, b, off);
                if (lane + off < 32) { a += ta; b += tb; }
            }
            a += __shfl_sync(0xffffffffu, b, 0);
#pragma unroll
            for (int hj = 0; hj < 2; ++hj) {
                const int i = lane + 32 * hj;
                if (i < L) {
                    atomicAdd(p.dbeta + (t0 + i) * Nv + h, db[hj]);
                    if (p.dg) atomicAdd(p.dg + (t0 + i) * Nv + h, hj ? b : a);
                }
            }
        }
        // ---- dq, dk: 4-row x 8-column register tiles ----------------------
        //   dq_i = scale e^{G_i} S dO_i + sum_j WP_ij k_j
        //   dk_i = dec_i dS' Vn_i - beta_i e^{G_i} S dR_i
        //          + sum_j (M_ij + M_ji) k_j + sum_j WP_ji q_j
        if constexpr (MMA) {
            tcp::mma_dqdk(bc, warp, lane, p.dq + (t0 * Nk + hk) * (long long)dk, p.dkk + (t0 * Nk + hk) * (long long)dk,
                     (long long)Nk * dk);
        } else {
            const int ndg = dk >> 3;
            for (int tile = tid; tile < 16 * ndg; tile += NT) {
                const int i0 = 4 * (tile / ndg), d0 = 8 * (tile % ndg);
                if (i0 >= L) continue;
                float gq[4][8], gk[4][8];
                {
                    float a1[4][8], a2[4][8], a3[4][8];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int x = 0; x < 8; ++x) a1[r][x] = a2[r][x] = a3[r][x] = 0.0f;
                    for (int cc = 0; cc < BV; ++cc) {
                        const float4 s0 = *reinterpret_cast<const float4 *>(sSt + cc * SLD + d0);
                        const float4 s1 = *reinterpret_cast<const float4 *>(sSt + cc * SLD + d0 + 4);
                        const float4 t0v = *reinterpret_cast<const float4 *>(sdSt + cc * SLD + d0);
                        const float4 t1v = *reinterpret_cast<const float4 *>(sdSt + cc * SLD + d0 + 4);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float o = sdO[(i0 + r) * LDV + cc], vn = sVn[(i0 + r) * LDV + cc],
                                        dr = sdV[(i0 + r) * LDV + cc];
                            const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                            const float tv[8] = {t0v.x, t0v.y, t0v.z, t0v.w, t1v.x, t1v.y, t1v.z, t1v.w};
#pragma unroll
                            for (int x = 0; x < 8; ++x) {
                                a1[r][x] = fmaf(o, sv[x], a1[r][x]);
                                a2[r][x] = fmaf(vn, tv[x], a2[r][x]);
                                a3[r][x] = fmaf(dr, sv[x], a3[r][x]);
                            }
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int i = i0 + r;
                        const float fq = p.scale * sEG[i], fd = sDec[i], fr = sBeta[i] * sEG[i];
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            gq[r][x] = fq * a1[r][x];
                            gk[r][x] = fd * a2[r][x] - fr * a3[r][x];
                        }
                    }
                }
                for (int j = 0; j < L; ++j) {
                    const float4 k0v = ld4(sK + j * ldkq + d0), k1v = ld4(sK + j * ldkq + d0 + 4);
                    const float4 q0v = ld4(sQ + j * ldkq + d0), q1v = ld4(sQ + j * ldkq + d0 + 4);
                    const float kv[8] = {k0v.x, k0v.y, k0v.z, k0v.w, k1v.x, k1v.y, k1v.z, k1v.w};
                    const float qv[8] = {q0v.x, q0v.y, q0v.z, q0v.w, q1v.x, q1v.y, q1v.z, q1v.w};
                    const float rkj = sRK[j], rqj = sRQ[j];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int i = i0 + r;
                        const float wq = rkj * sM1[i * LDC + j];                       // WP_ij (0 for j > i)
                        const float mk = rkj * (sM0[i * LDC + j] + sM0[j * LDC + i]);  // M_ij + M_ji
                        const float wt = rqj * sM1[j * LDC + i];                       // WP_ji (0 for j < i)
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            gq[r][x] = fmaf(wq, kv[x], gq[r][x]);
                            gk[r][x] = fmaf(mk, kv[x], fmaf(wt, qv[x], gk[r][x]));
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = i0 + r;
                    if (i >= L) continue;
                    float *pq = p.dq + ((t0 + i) * Nk + hk) * (long long)dk + d0;
                    float *pk = p.dkk + ((t0 + i) * Nk + hk) * (long long)dk + d0;
                    atomicAdd(reinterpret_cast<float4 *>(pq), make_float4(gq[r][0], gq[r][1], gq[r][2], gq[r][3]));
                    atomicAdd(reinterpret_cast<float4 *>(pq + 4), make_float4(gq[r][4], gq[r][5], gq[r][6], gq[r][7]));
                    atomicAdd(reinterpret_cast<float4 *>(pk), make_float4(gk[r][0], gk[r][1], gk[r][2], gk[r][3]));
                    atomicAdd(reinterpret_cast<float4 *>(pk + 4), make_float4(gk[r][4], gk[r][5], gk[r][6], gk[r][7]));
                }
            }
        }
        __syncthreads();

        // ---- dS = e^{G_L} dS' + scale Q^T diag(e^G) dO - K^T diag(beta e^G) dR
        // thread: columns 2 cp, 2 cp + 1; rows d0 .. d0 + 7 of dS
        if constexpr (MMA) {
            // S^T is free until the next chunk's K S: its state goes out now
            if (ci > 0) {
                load_hs(ci - 1);
                cp_async_commit();
            }
            tcp::mma_ds(bc, warp, lane, expf(sGL[0]));
        } else {
            const float eGL = expf(sGL[0]);
            const int ndg = dk >> 3;
            for (int tile = tid; tile < 16 * ndg; tile += NT) {
                const int c0 = 2 * (tile / ndg), d0 = 8 * (tile % ndg);
                float acc[2][8];
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    const float4 a = *reinterpret_cast<const float4 *>(sdSt + (c0 + y) * SLD + d0);
                    const float4 b = *reinterpret_cast<const float4 *>(sdSt + (c0 + y) * SLD + d0 + 4);
                    acc[y][0] = eGL * a.x; acc[y][1] = eGL * a.y; acc[y][2] = eGL * a.z; acc[y][3] = eGL * a.w;
                    acc[y][4] = eGL * b.x; acc[y][5] = eGL * b.y; acc[y][6] = eGL * b.z; acc[y][7] = eGL * b.w;
                }
                for (int i = 0; i < L; ++i) {
                    const float fq = p.scale * sEG[i] * sRQ[i], fk = -sBeta[i] * sEG[i] * sRK[i];
                    const float4 q0v = ld4(sQ + i * ldkq + d0), q1v = ld4(sQ + i * ldkq + d0 + 4);
                    const float4 k0v = ld4(sK + i * ldkq + d0), k1v = ld4(sK + i * ldkq + d0 + 4);
                    const float qv[8] = {q0v.x, q0v.y, q0v.z, q0v.w, q1v.x, q1v.y, q1v.z, q1v.w};
                    const float kv[8] = {k0v.x, k0v.y, k0v.z, k0v.w, k1v.x, k1v.y, k1v.z, k1v.w};
#pragma unroll
                    for (int y = 0; y < 2; ++y) {
                        const float a = fq * sdO[i * LDV + c0 + y], b = fk * sdV[i * LDV + c0 + y];
#pragma unroll
                        for (int x = 0; x < 8; ++x) acc[y][x] = fmaf(a, qv[x], fmaf(b, kv[x], acc[y][x]));
                    }
                }
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    *reinterpret_cast<float4 *>(sdSt + (c0 + y) * SLD + d0) =
                        make_float4(acc[y][0], acc[y][1], acc[y][2], acc[y][3]);
                    *reinterpret_cast<float4 *>(sdSt + (c0 + y) * SLD + d0 + 4) =
                        make_float4(acc[y][4], acc[y][5], acc[y][6], acc[y][7]);
                }
            }
        }
    }

    __syncthreads();
    if (p.dh0) {
        for (int idx = tid; idx < dk * BV; idx += NT) {
            const int d = idx / BV, cc = idx - d * BV;
            if (cc < bvw) p.dh0[sbase + (size_t)d * dv + v0 + cc] = sdSt[cc * SLD + d];
        }
    }
}

// With kQkL2Norm the backward kernel's dq and dk are the gradients of the
// normalised rows y = x r, r = 1 / max(||x||, 1e-12).  This maps each row
// back: dx = r (dy - y (y . dy)) where ||x|| > 1e-12, else dx = r dy (the
// divisor is the constant 1e-12 there).  One warp per row; rows of q, then k.
template <typename Tin>
__global__ void l2norm_bwd_rows(const Tin *q, const Tin *k, float *dq, float *dk, long long rows, int d) {
    const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= 2 * rows) return;
    const bool isq = wid < rows;
    const long long row = isq ? wid : wid - rows;
    const Tin *x = (isq ? q : k) + row * d;
    float *g = (isq ? dq : dk) + row * d;
    float xv[8], gv[8];  // d <= 256
    float ss = 0.0f, xg = 0.0f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int e = lane + 32 * m;
        xv[m] = e < d ? to_f(x[e]) : 0.0f;
        gv[m] = e < d ? g[e] : 0.0f;
        ss = fmaf(xv[m], xv[m], ss);
        xg = fmaf(xv[m], gv[m], xg);
    }
    ss = warp_sum(ss);
    xg = warp_sum(xg);
    const bool big = ss > 1e-24f;
    const float r = rsqrtf(fmaxf(ss, 1e-24f));
    // y . dy = r (x . dy);  r (dy - y (y . dy)) = r dy - r^3 (x . dy) x
    const float c = big ? r * r * r * xg : 0.0f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int e = lane + 32 * m;
        if (e < d) g[e] = r * gv[m] - c * xv[m];
    }
}

// Zero-fills up to four fp32 buffers in one launch (null pointers skipped).
struct ZeroArgs {
    float *ptr[4];
    long long n[4];
};

__global__ void fill_zero(ZeroArgs z) {
    const long long stride = (long long)gridDim.x * blockDim.x;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (!z.ptr[b]) continue;
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < z.n[b]; i += stride)
            z.ptr[b][i] = 0.0f;
    }
}

}  // namespace

size_t bwd_smem_bytes(int dk, bool bf16, bool mma) {
    return bf16 ? (mma ? layout<__nv_bfloat16, true>(dk).end : layout<__nv_bfloat16, false>(dk).end)
                : layout<float, false>(dk).end;
}

cudaError_t bwd_launch(const Params &p, bool bf16, cudaStream_t stream, const char **name) {
    const int nvt = (p.dv + BV - 1) / BV;
    const long long grid = (long long)p.N * p.Nv * nvt;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t err;
    {
        const ZeroArgs z{{p.dq, p.dkk, p.dbeta, p.dg},
                         {p.tokens * p.Nk * p.dk, p.tokens * p.Nk * p.dk, p.tokens * p.Nv, p.tokens * p.Nv}};
        const long long most = p.tokens * p.Nk * p.dk;
        long long blocks = (most + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        if (blocks < 1) blocks = 1;
        fill_zero<<<(unsigned)blocks, 256, 0, stream>>>(z);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    // forward pass at chunk 64 with no output, saving the chunk-start states:
    // the tensor-core forward where it applies (its WY slots in p.ws), else
    // the CUDA-core one
    Params f = p;
    f.o = nullptr;
    f.ht = nullptr;
    f.chunk = kChunk;
    const bool tc = p.tokens > 0 && p.dk == 128 && tc_supported(p.dk, p.dv, bf16, kChunk);
    if (tc && !p.ws) return cudaErrorInvalidValue;
    const char *fname = "";
    if ((err = tc ? tc_launch(f, stream, &fname) : simt_launch(f, bf16, false, stream, &fname)) != cudaSuccess) return err;
    const size_t smem = bwd_smem_bytes(p.dk, bf16, tc);
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    const long long rows = p.tokens * p.Nk;  // q (and k) rows
    const unsigned nblk = (unsigned)((2 * rows * 32 + 255) / 256);
    if (bf16) {
        // the tensor-core products where the states come from the
        // tensor-core forward (dk = 128, dv a multiple of 128)
        auto kern = tc ? simt_bwd<__nv_bfloat16, true> : simt_bwd<__nv_bfloat16, false>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<(unsigned)grid, NT, smem, stream>>>(p);
        if (qkn && rows > 0)
            l2norm_bwd_rows<__nv_bfloat16><<<nblk, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k), p.dq, p.dkk, rows,
                p.dk);
        if (tc)
            *name = qkn ? "fill_zero+wy_fwd+tc_fwd+simt_bwd<bf16,tf32>+l2norm_bwd_rows<bf16>"
                        : "fill_zero+wy_fwd+tc_fwd+simt_bwd<bf16,tf32>";
        else
            *name = qkn ? "fill_zero+simt_fwd<bf16>+simt_bwd<bf16>+l2norm_bwd_rows<bf16>"
                        : "fill_zero+simt_fwd<bf16>+simt_bwd<bf16>";
    } else {
        err = cudaFuncSetAttribute(simt_bwd<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_bwd<float, false><<<(unsigned)grid, NT, smem, stream>>>(p);
        if (qkn && rows > 0)
            l2norm_bwd_rows<float><<<nblk, 256, 0, stream>>>(static_cast<const float *>(p.q),
                                                             static_cast<const float *>(p.k), p.dq, p.dkk, rows, p.dk);
        *name = qkn ? "fill_zero+simt_fwd<f32>+simt_bwd<f32>+l2norm_bwd_rows<f32>"
                    : "fill_zero+simt_fwd<f32>+simt_bwd<f32>";
    }
    return cudaGetLastError();
}

}  // namespace dn
