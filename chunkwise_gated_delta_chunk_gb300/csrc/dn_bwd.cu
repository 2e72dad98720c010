// Backward of the chunkwise gated delta rule forward (CUDA cores, fp32).
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
// CUDA-core forward.  The chunk-start states come from a forward pass of that
// kernel (saved per 64-token chunk).  Every quantity above that sums over
// value columns (dq, dk, dbeta, dg, and dA, dP through them) is linear in the
// tile's columns, so each CTA adds its share to zero-initialised fp32 outputs
// with atomics; dv and dh0 belong to one tile and are stored directly.
#include <cuda_bf16.h>
#include <math.h>

#include "dn_internal.h"

namespace dn {
namespace {

constexpr int C = kChunk;  // 64
constexpr int BV = 32;     // value columns per CTA
constexpr int NT = 256;    // 8 warps
constexpr int LDC = C + 1; // row stride of the C x C matrices
constexpr int LDV = BV + 1;  // row stride of the C x BV and dk x BV tiles (conflict-free row-per-lane reads)

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename Tin>
__host__ __device__ constexpr int kq_ld(int dk) { return sizeof(Tin) == 2 ? dk + 2 : dk + 1; }

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

struct Layout {
    size_t k, q, s, ds, m0, m1, m2, u, dO, ks, vn, dv, kds, sc, end;
};

// Per-row scalars (C floats each) at Layout::sc.
enum { R_G, R_EG, R_DEC, R_BETA, R_QSDO, R_DBU, R_DGAM, R_E, R_ROWE, R_DBA, R_COUNT };

template <typename Tin>
__host__ __device__ inline Layout layout(int dk) {
    Layout L{};
    size_t off = 0;
    const size_t kq = align16(size_t(C) * kq_ld<Tin>(dk) * sizeof(Tin));
    L.k = off; off += kq;
    L.q = off; off += kq;
    L.s = off; off += align16(size_t(dk) * LDV * 4);
    L.ds = off; off += align16(size_t(dk) * LDV * 4);
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

template <typename Tin>
__device__ __forceinline__ void load_rows(Tin *dst, const Tin *src, long long t0, int L, int H, int hh,
                                          int d, int tid) {
    constexpr int VEC = 16 / sizeof(Tin);
    const int ld = kq_ld<Tin>(d);
    const int per_row = d / VEC;
    for (int idx = tid; idx < L * per_row; idx += NT) {
        const int i = idx / per_row, cv = idx - i * per_row;
        const uint4 w = *reinterpret_cast<const uint4 *>(src + ((t0 + i) * H + hh) * (long long)d + cv * VEC);
        const Tin *e = reinterpret_cast<const Tin *>(&w);
#pragma unroll
        for (int x = 0; x < VEC; ++x) dst[i * ld + cv * VEC + x] = e[x];
    }
    for (int idx = L * ld + tid; idx < C * ld; idx += NT) dst[idx] = Tin(0.0f);
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
    const int c = lane;  // value column of the C x BV tiles

    const Layout lay = layout<Tin>(dk);
    Tin *sK = reinterpret_cast<Tin *>(smem + lay.k);
    Tin *sQ = reinterpret_cast<Tin *>(smem + lay.q);
    float *sS = reinterpret_cast<float *>(smem + lay.s);     // [dk][LDV] state the chunk starts from
    float *sdS = reinterpret_cast<float *>(smem + lay.ds);   // [dk][LDV] gradient of the state it hands on
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
        sdS[d * LDV + cc] = (p.dht && cc < bvw) ? p.dht[sbase + (size_t)d * dv + v0 + cc] : 0.0f;
    }

    const long long nch = (eos - bos + C - 1) / C;
    for (long long ci = nch - 1; ci >= 0; --ci) {
        const long long t0 = bos + ci * C;
        const int L = (eos - t0) < C ? (int)(eos - t0) : C;
        __syncthreads();  // the previous (later) chunk is done with every buffer

        // ---- load --------------------------------------------------------
        load_rows<Tin>(sK, k, t0, L, Nk, hk, dk, tid);
        load_rows<Tin>(sQ, q, t0, L, Nk, hk, dk, tid);
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
                sS[d * LDV + cc] = cc < bvw ? hs[(size_t)d * dv + cc] : 0.0f;
            }
        }
        if (tid < C) {
            sBeta[tid] = tid < L ? p.beta[(t0 + tid) * Nv + h] : 0.0f;
            sG[tid] = (tid < L && p.g) ? p.g[(t0 + tid) * Nv + h] : 0.0f;
        }
        __syncthreads();

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
        }
        {
            float part = 0.0f;
            for (int idx = tid; idx < dk * BV; idx += NT) {
                const int d = idx / BV, cc = idx - d * BV;
                part = fmaf(sS[d * LDV + cc], sdS[d * LDV + cc], part);
            }
            part = warp_sum(part);
            if (lane == 0) sRed[warp] = part;
        }
        __syncthreads();

        // ---- -(K K^T . D) (strictly lower) and P (lower) ------------------
        for (int idx = tid; idx < C * C; idx += NT) {
            const int i = idx >> 6, j = idx & 63;
            float a = 0.0f, pv = 0.0f;
            if (i < L && j <= i) {
                const Tin *ki = sK + i * ldkq, *kj = sK + j * ldkq, *qi = sQ + i * ldkq;
                float skk = 0.0f, sqk = 0.0f;
                for (int d = 0; d < dk; ++d) {
                    const float kjd = to_f(kj[d]);
                    skk = fmaf(to_f(ki[d]), kjd, skk);
                    sqk = fmaf(to_f(qi[d]), kjd, sqk);
                }
                const float dec = expf(sG[i] - sG[j]);
                if (j < i) a = -skk * dec;
                pv = p.scale * sqk * dec;
            }
            sM0[i * LDC + j] = a;
            sM2[i * LDC + j] = pv;
        }
        __syncthreads();

        // ---- T = (I - A)^-1, A_im = beta_i sM0_im; column j by 4 lanes ----
        {
            const int j = tid >> 2, pl = tid & 3;
            for (int i = pl; i < C; i += 4) sM1[i * LDC + j] = (i == j) ? 1.0f : 0.0f;
            __syncwarp();
            for (int i = 1; i < L; ++i) {
                float part = 0.0f;
                if (i > j) {
                    for (int m = j + pl; m < i; m += 4) part = fmaf(sM0[i * LDC + m], sM1[m * LDC + j], part);
                }
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (i > j && ((i - j) & 3) == pl) sM1[i * LDC + j] = sBeta[i] * part;
            }
        }
        // ---- K S, Q S (.dO), K dS'; U = V - e^G K S ------------------------
        {
            float ks[8], qs[8], kd[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) { ks[r] = 0.0f; qs[r] = 0.0f; kd[r] = 0.0f; }
            for (int d = 0; d < dk; ++d) {
                const float s = sS[d * LDV + c], ds = sdS[d * LDV + c];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int i = warp + 8 * r;
                    const float kv = to_f(sK[i * ldkq + d]);
                    ks[r] = fmaf(kv, s, ks[r]);
                    kd[r] = fmaf(kv, ds, kd[r]);
                    qs[r] = fmaf(to_f(sQ[i * ldkq + d]), s, qs[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                sKS[i * LDV + c] = ks[r];
                sKdS[i * LDV + c] = kd[r];
                sU[i * LDV + c] = i < L ? sU[i * LDV + c] - sEG[i] * ks[r] : 0.0f;
                const float qd = warp_sum(qs[r] * sdO[i * LDV + c]);
                if (lane == 0) sQSdO[i] = qd;
            }
        }
        __syncthreads();

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

        // ---- warp 0: dbeta, dG and dg; warps 1-7: dq, dk ------------------
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
            if (lane == ((L - 1) & 31)) dG[(L - 1) >> 5] += extra;
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
        } else {
            // rows i = (warp - 1) + 7 m, columns d = lane + 32 x
            for (int i = warp - 1; i < L; i += 7) {
                const float eg = sEG[i], dec = sDec[i], bi = sBeta[i];
                for (int d = lane; d < dk; d += 32) {
                    float sdo = 0.0f, sdr = 0.0f, dsv = 0.0f;
#pragma unroll 8
                    for (int cc = 0; cc < BV; ++cc) {
                        const float s = sS[d * LDV + cc];
                        sdo = fmaf(s, sdO[i * LDV + cc], sdo);
                        sdr = fmaf(s, sdV[i * LDV + cc], sdr);
                        dsv = fmaf(sdS[d * LDV + cc], sVn[i * LDV + cc], dsv);
                    }
                    float gq = p.scale * eg * sdo;
                    float gk = dec * dsv - bi * eg * sdr;
                    for (int j = 0; j <= i; ++j) {
                        const float kj = to_f(sK[j * ldkq + d]);
                        gq = fmaf(sM1[i * LDC + j], kj, gq);   // scale D_ij dP_ij k_j
                        gk = fmaf(sM0[i * LDC + j], kj, gk);   // M_ij k_j (j < i; M_ii = 0)
                    }
                    for (int j = i; j < L; ++j) {
                        gk = fmaf(sM0[j * LDC + i], to_f(sK[j * ldkq + d]), gk);  // M_ji k_j
                        gk = fmaf(sM1[j * LDC + i], to_f(sQ[j * ldkq + d]), gk);  // scale D_ji dP_ji q_j
                    }
                    atomicAdd(p.dq + ((t0 + i) * Nk + hk) * (long long)dk + d, gq);
                    atomicAdd(p.dkk + ((t0 + i) * Nk + hk) * (long long)dk + d, gk);
                }
            }
        }
        __syncthreads();

        // ---- dS = e^{G_L} dS' + scale Q^T diag(e^G) dO - K^T diag(beta e^G) dR
        {
            const float eGL = expf(sGL[0]);
            for (int d = warp; d < dk; d += 8) {
                float acc = eGL * sdS[d * LDV + c];
                for (int i = 0; i < L; ++i) {
                    const float eg = sEG[i];
                    acc = fmaf(p.scale * eg * to_f(sQ[i * ldkq + d]), sdO[i * LDV + c], acc);
                    acc = fmaf(-sBeta[i] * eg * to_f(sK[i * ldkq + d]), sdV[i * LDV + c], acc);
                }
                sdS[d * LDV + c] = acc;
            }
        }
    }

    __syncthreads();
    if (p.dh0) {
        for (int idx = tid; idx < dk * BV; idx += NT) {
            const int d = idx / BV, cc = idx - d * BV;
            if (cc < bvw) p.dh0[sbase + (size_t)d * dv + v0 + cc] = sdS[d * LDV + cc];
        }
    }
}

__global__ void fill_zero(float *p, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        p[i] = 0.0f;
}

cudaError_t zero(float *ptr, long long n, cudaStream_t stream) {
    if (!ptr || n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    fill_zero<<<(unsigned)blocks, 256, 0, stream>>>(ptr, n);
    return cudaGetLastError();
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
    if ((err = zero(p.dq, p.tokens * p.Nk * p.dk, stream)) != cudaSuccess) return err;
    if ((err = zero(p.dkk, p.tokens * p.Nk * p.dk, stream)) != cudaSuccess) return err;
    if ((err = zero(p.dbeta, p.tokens * p.Nv, stream)) != cudaSuccess) return err;
    if ((err = zero(p.dg, p.tokens * p.Nv, stream)) != cudaSuccess) return err;
    // forward pass at chunk 64, saving the chunk-start states
    Params f = p;
    f.o = nullptr;
    f.ht = nullptr;
    f.chunk = kChunk;
    const char *fname = "";
    if ((err = simt_launch(f, bf16, stream, &fname)) != cudaSuccess) return err;
    const size_t smem = bwd_smem_bytes(p.dk, bf16);
    if (bf16) {
        err = cudaFuncSetAttribute(simt_bwd<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_bwd<__nv_bfloat16><<<(unsigned)grid, NT, smem, stream>>>(p);
        *name = "fill_zero+simt_fwd<bf16>+simt_bwd<bf16>";
    } else {
        err = cudaFuncSetAttribute(simt_bwd<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_bwd<float><<<(unsigned)grid, NT, smem, stream>>>(p);
        *name = "fill_zero+simt_fwd<f32>+simt_bwd<f32>";
    }
    return cudaGetLastError();
}

}  // namespace dn
