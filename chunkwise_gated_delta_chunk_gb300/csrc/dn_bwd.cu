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
#include "dn_simt_common.cuh"
#include "dn_tc.h"

#ifdef DN_TRACE
__device__ unsigned long long g_bwd_ph[64][16];
extern "C" __attribute__((visibility("default"))) int dn_trace_dump_bwd(void *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_bwd_ph, sizeof(g_bwd_ph));
}
#endif

namespace dn {
namespace {

using simt::kq_ld;
using simt::ld4;
using simt::to_f;
using simt::align16;

constexpr int C = kChunk;    // 64
constexpr int BV = 32;       // value columns per CTA
constexpr int NT = 256;      // 8 warps
constexpr int LDC = C + 1;   // row stride of the C x C matrices
constexpr int LDV = BV + 1;  // row stride of the C x BV tiles (conflict-free row-per-lane reads)

// Row stride (floats) of the transposed state tiles S^T, dS^T ([BV][dk]):
// 16-byte rows, consecutive rows 4 banks apart.
__host__ __device__ inline int st_ld(int dk) { return dk + 4; }

struct Layout {
    size_t k, q, s, ds, m0, m1, m2, u, dO, ks, vn, dv, kds, sc, end;
};

// Per-row scalars (C floats each) at Layout::sc.
enum { R_G, R_EG, R_DEC, R_BETA, R_QSDO, R_DBU, R_DGAM, R_E, R_ROWE, R_DBA, R_RK, R_RQ, R_COUNT };

template <typename Tin>
__host__ __device__ inline Layout layout(int dk) {
    Layout L{};
    size_t off = 0;
    const size_t kq = align16(size_t(C) * kq_ld<Tin>(dk) * sizeof(Tin));
    L.k = off; off += kq;
    L.q = off; off += kq;
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
    L.sc = off; off += size_t(R_COUNT) * C * 4 + 64;  // + G_L, block partial sums
    L.end = off;
    return L;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <typename Tin>
__global__ void __launch_bounds__(NT) simt_bwd(Params p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int dk = p.dk, dv = p.dv, Nk = p.Nk, Nv = p.Nv;
    const int nvt = (dv + BV - 1) / BV;
    const int vt = blockIdx.x % nvt;
    const int h = (blockIdx.x / nvt) % Nv;
    const int n = blockIdx.x / (nvt * Nv);
    const int hk = h / (Nv / Nk);
    const int v0 = vt * BV;
    const int bvw = min(BV, dv - v0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = lane;  // value column of the C x BV tiles in the row-per-warp loops
    const int SLD = st_ld(dk);

    const Layout lay = layout<Tin>(dk);
    Tin *sK = reinterpret_cast<Tin *>(smem + lay.k);
    Tin *sQ = reinterpret_cast<Tin *>(smem + lay.q);
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
    float *sG = sc + R_G * C, *sEG = sc + R_EG * C, *sDec = sc + R_DEC * C, *sBeta = sc + R_BETA * C;
    float *sQSdO = sc + R_QSDO * C, *sDBU = sc + R_DBU * C, *sDGam = sc + R_DGAM * C;
    float *sE = sc + R_E * C, *sRowE = sc + R_ROWE * C, *sDBA = sc + R_DBA * C;
    // inverse key / query norms of the chunk's rows (1 without kQkL2Norm):
    // every product below that reads a k or q row takes the row's factor, so
    // the gradients the CTA adds up are those of the normalised rows
    float *sRK = sc + R_RK * C, *sRQ = sc + R_RQ * C;
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    float *sGL = sc + R_COUNT * C;      // [0]: G_L
    float *sRed = sGL + 4;              // [8]: per-warp partial <S, dS'>
    const int ldkq = kq_ld<Tin>(dk);

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
    for (long long ci = nch - 1; ci >= 0; --ci) {
        const long long t0 = bos + ci * C;
        const int pc = (int)(nch - 1 - ci);  // position in the walk (phase stamps)
        (void)pc;
        const int L = (eos - t0) < C ? (int)(eos - t0) : C;
        __syncthreads();  // the previous (later) chunk is done with every buffer

        DN_PHASE(g_bwd_ph, pc, 0);
        // ---- load --------------------------------------------------------
        simt::load_rows<Tin, NT>(sK, k, t0, L, Nk, hk, dk, tid);
        simt::load_rows<Tin, NT>(sQ, q, t0, L, Nk, hk, dk, tid);
        for (int idx = tid; idx < C * BV; idx += NT) {
            const int i = idx / BV, cc = idx - i * BV;
            const bool in = i < L && cc < bvw;
            const long long off = ((t0 + i) * Nv + h) * (long long)dv + v0 + cc;
            sU[i * LDV + cc] = in ? to_f(v[off]) : 0.0f;
            sdO[i * LDV + cc] = in ? to_f(dout[off]) : 0.0f;
        }
        {
            const float *hs = p.hs + ((size_t)h * p.nslots + (size_t)(t0 / C + n)) * dk * dv + v0;
            for (int idx = tid; idx < dk * BV; idx += NT) {
                const int d = idx / BV, cc = idx - d * BV;
                sSt[cc * SLD + d] = cc < bvw ? hs[(size_t)d * dv + cc] : 0.0f;
            }
        }
        if (tid < C) {
            sBeta[tid] = tid < L ? p.beta[(t0 + tid) * Nv + h] : 0.0f;
            sG[tid] = (tid < L && p.g) ? p.g[(t0 + tid) * Nv + h] : 0.0f;
        }
        __syncthreads();

        DN_PHASE(g_bwd_ph, pc, 1);
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

        DN_PHASE(g_bwd_ph, pc, 2);
        // ---- -(K K^T . D) (strictly lower) and P (lower) ------------------
        simt::kq_products<NT>(sK, sQ, ldkq, dk, tid, [&](int i, int j, float kk, float qk) {
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

        DN_PHASE(g_bwd_ph, pc, 3);
        // ---- T = (I - A)^-1, A_im = beta_i sM0_im (blocked; sVn, written
        // later, is its scratch) ---------------------------------------------
        simt::solve_T_blocked<NT>(sM0, LDC, sBeta, sM1, LDC, sVn, L, tid);
        DN_PHASE(g_bwd_ph, pc, 4);
        // ---- K S, Q S (.dO), K dS'; U = V - e^G K S ------------------------
        // thread: rows i0, i0 + 1; columns cg + 8 x (x < 4)
        {
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

        DN_PHASE(g_bwd_ph, pc, 5);
        // ---- Vn = T diag(beta) U ------------------------------------------
        {
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

        DN_PHASE(g_bwd_ph, pc, 6);
        // ---- dVn = diag(dec) K dS' + P^T dO; e_i --------------------------
        {
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

        DN_PHASE(g_bwd_ph, pc, 7);
        // ---- dR = T^T dVn; dv = diag(beta) dR ------------------------------
        {
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

        DN_PHASE(g_bwd_ph, pc, 8);
        // ---- dA, dP and E (row i per warp, columns j = lane, lane + 32) ----
        {
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

        DN_PHASE(g_bwd_ph, pc, 9);
        // ---- warp 0: dbeta, dG and dg ------------------------------------
        if (warp == 0) {
            float dG[2], db[2];
            float esum = 0.0f;
#pragma unroll
            for (int hj = 0; hj < 2; ++hj) {
                const int i = lane + 32 * hj;
                float colE = 0.0f;
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
        {
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

        DN_PHASE(g_bwd_ph, pc, 10);
        // ---- dS = e^{G_L} dS' + scale Q^T diag(e^G) dO - K^T diag(beta e^G) dR
        // thread: columns 2 cp, 2 cp + 1; rows d0 .. d0 + 7 of dS
        {
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
        DN_PHASE(g_bwd_ph, pc, 11);
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

size_t bwd_smem_bytes(int dk, bool bf16) {
    return bf16 ? layout<__nv_bfloat16>(dk).end : layout<float>(dk).end;
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
    const bool tc = p.tokens > 0 && tc_supported(p.dk, p.dv, bf16);
    if (tc && !p.ws) return cudaErrorInvalidValue;
    const char *fname = "";
    if ((err = tc ? tc_launch(f, stream, &fname) : simt_launch(f, bf16, stream, &fname)) != cudaSuccess) return err;
    const size_t smem = bwd_smem_bytes(p.dk, bf16);
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    const long long rows = p.tokens * p.Nk;  // q (and k) rows
    const unsigned nblk = (unsigned)((2 * rows * 32 + 255) / 256);
    if (bf16) {
        err = cudaFuncSetAttribute(simt_bwd<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_bwd<__nv_bfloat16><<<(unsigned)grid, NT, smem, stream>>>(p);
        if (qkn && rows > 0)
            l2norm_bwd_rows<__nv_bfloat16><<<nblk, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k), p.dq, p.dkk, rows,
                p.dk);
        if (tc)
            *name = qkn ? "fill_zero+wy_fwd+tc_fwd+simt_bwd<bf16>+l2norm_bwd_rows<bf16>"
                        : "fill_zero+wy_fwd+tc_fwd+simt_bwd<bf16>";
        else
            *name = qkn ? "fill_zero+simt_fwd<bf16>+simt_bwd<bf16>+l2norm_bwd_rows<bf16>"
                        : "fill_zero+simt_fwd<bf16>+simt_bwd<bf16>";
    } else {
        err = cudaFuncSetAttribute(simt_bwd<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_bwd<float><<<(unsigned)grid, NT, smem, stream>>>(p);
        if (qkn && rows > 0)
            l2norm_bwd_rows<float><<<nblk, 256, 0, stream>>>(static_cast<const float *>(p.q),
                                                             static_cast<const float *>(p.k), p.dq, p.dkk, rows, p.dk);
        *name = qkn ? "fill_zero+simt_fwd<f32>+simt_bwd<f32>+l2norm_bwd_rows<f32>"
                    : "fill_zero+simt_fwd<f32>+simt_bwd<f32>";
    }
    return cudaGetLastError();
}

}  // namespace dn
