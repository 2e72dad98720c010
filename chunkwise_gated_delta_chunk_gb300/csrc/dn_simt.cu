// CUDA-core kernel of the chunkwise gated delta rule forward: every shape
// the tensor-core scan does not take (fp32 inputs, chunks of 16 or 32 tokens,
// d other than 128).
//
// Two kinds of instantiation.  simt_fwd<T, false>: every product an fp32
// FMA, for fp32 inputs (whose tolerance leaves no room for reduced-precision
// products) and the backward's state pass.  simt_fwd<bf16, true>: K S, Q S
// and the state update as TF32 tensor-core tiles (mma.sync, fp32
// accumulation), within the bf16 bound.  K K^T and Q K^T of bf16 inputs are
// bf16 tensor-core tiles in both (products of bf16 values are exact in fp32).
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.3;
//          [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §2.3-§2.4.
//
// One CTA owns one (sequence, value head, 32-column value tile) and walks the
// sequence's chunks in order, keeping its fp32 state tile S[dk][32] in shared
// memory.  Chunks are p.chunk = 16, 32 or 64 tokens long; every chunk uses
// 64-row tiles whose rows past its length L are zero.  Per chunk:
//   a1  G = inclusive prefix sum of g (warp scan), e^{G_i}, e^{G_L - G_i}
//   a2  A_ij = -beta_i (k_i.k_j) e^{G_i-G_j} (j < i),
//       P_ij = scale (q_i.k_j) e^{G_i-G_j} (j <= i)
//   a3  T = (I - A)^-1: the diagonal 16 x 16 blocks by forward substitution,
//       the rest from block products (dn_simt_common.cuh)
//   a4+a5  v_new = U - W S_in = T diag(beta) (V - diag(e^G) K S_in)
//       (the same product as T diag(beta) V - T diag(beta e^G) K S_in, grouped
//        so that W = T diag(beta e^G) K is never formed: K S_in is 64 x 32,
//        cheaper than the 64 x dk matrix W on CUDA cores)
//   a6  o = scale e^{G} (Q S_in) + P v_new
//   a5  S_out = e^{G_L} S_in + sum_i e^{G_L-G_i} k_i v_new_i^T
// With kQkL2Norm every product that reads a row k_i or q_i also takes the
// row's factor 1 / max(||x||, 1e-12), computed in a1; the rows in shared
// memory stay as loaded.
#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "dn_internal.h"
#include "dn_order.cuh"
#include "dn_simt_common.cuh"

namespace dn {
namespace {

using simt::align16;
using simt::kq_ld;
using simt::to_f;

constexpr int C = kChunk;
constexpr int BV = 32;   // value columns per CTA
constexpr int NT = 256;  // threads per CTA (8 warps)
constexpr int LDC = C + 4;   // row stride of the C x C matrices (16-byte rows)

// Row stride (floats) of the transposed state tile S^T ([BV][dk]): 16-byte
// rows, consecutive rows 4 banks apart.
__host__ __device__ inline int st_ld(int dk) { return dk + 4; }

__device__ __forceinline__ void put(float *p, float x) { *p = x; }
__device__ __forceinline__ void put(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

struct Layout {
    size_t k, q, s, a, t, p, v, r, vn, oi, g, eg, dec, beta, rk, rq, end;
};

template <typename Tin>
__host__ __device__ inline Layout layout(int dk) {
    Layout L{};
    size_t off = 0;
    const size_t kq = align16(size_t(C) * kq_ld<Tin>(dk) * sizeof(Tin));
    L.k = off; off += kq;
    L.q = off; off += kq;
    L.s = off; off += align16(size_t(BV) * st_ld(dk) * 4);
    L.a = off; off += align16(size_t(C) * LDC * 4);
    L.t = off; off += align16(size_t(C) * LDC * 4);
    L.p = off; off += align16(size_t(C) * LDC * 4);
    L.v = off; off += size_t(C) * BV * 4;
    L.r = off; off += size_t(C) * BV * 4;
    L.vn = off; off += size_t(C) * BV * 4;
    L.oi = off; off += size_t(C) * BV * 4;
    L.g = off; off += C * 4;
    L.eg = off; off += C * 4;
    L.dec = off; off += C * 4;
    L.beta = off; off += C * 4;
    off += 16;  // G_L and spare
    L.rk = off; off += C * 4;
    L.rq = off; off += C * 4;
    L.end = off;
    return L;
}

// TF32 tensor-core tiles (m16n8k8 mma.sync, fp32 accumulation) for the
// state products of bf16 inputs; fp32 operands are rounded to TF32, bf16
// inputs are exact in it.  Fragments, lane = 4 g + t: A (16 x 8) a0 (g, t),
// a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4); B (8 x 8, k x n) b0 (t, g),
// b1 (t + 4, g); C (16 x 8) c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t),
// c3 (g + 8, 2t + 1).
namespace mmat {
__device__ __forceinline__ uint32_t cvt(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
__device__ __forceinline__ uint32_t bf(__nv_bfloat16 x) { return (uint32_t)__bfloat16_as_ushort(x) << 16; }
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
}  // namespace mmat

// MMA: the state products (K S, Q S and the state update) as TF32
// tensor-core tiles; used by the forward for bf16 inputs (its bf16 parity
// bound).  Without it every product is an fp32 FMA (the fp32 configuration
// and the backward's state pass).
template <typename Tin, bool MMA>
__global__ void __launch_bounds__(NT) simt_fwd(Params p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int dk = p.dk, dv = p.dv, Nk = p.Nk, Nv = p.Nv;
    const int nvt = (dv + BV - 1) / BV;
    const int unit = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vt = unit % nvt;
    const int h = (unit / nvt) % Nv;
    const int n = seq_of_rank(p, unit / (nvt * Nv), lane);  // longest sequences first
    const int hk = h / (Nv / Nk);
    const int v0 = vt * BV;
    const int bvw = min(BV, dv - v0);

    const Layout lay = layout<Tin>(dk);
    Tin *sK = reinterpret_cast<Tin *>(smem + lay.k);
    Tin *sQ = reinterpret_cast<Tin *>(smem + lay.q);
    float *sSt = reinterpret_cast<float *>(smem + lay.s);  // [BV][SLD]: S^T
    float *sA = reinterpret_cast<float *>(smem + lay.a);
    float *sT = reinterpret_cast<float *>(smem + lay.t);
    float *sP = reinterpret_cast<float *>(smem + lay.p);
    float *sV = reinterpret_cast<float *>(smem + lay.v);
    float *sR = reinterpret_cast<float *>(smem + lay.r);
    float *sVn = reinterpret_cast<float *>(smem + lay.vn);
    float *sOi = reinterpret_cast<float *>(smem + lay.oi);  // scale e^G (Q S_in), the inter-chunk output
    float *sG = reinterpret_cast<float *>(smem + lay.g);
    float *sEG = reinterpret_cast<float *>(smem + lay.eg);
    float *sDec = reinterpret_cast<float *>(smem + lay.dec);
    float *sBeta = reinterpret_cast<float *>(smem + lay.beta);
    float *sGL = reinterpret_cast<float *>(smem + lay.beta + C * 4);
    float *sRK = reinterpret_cast<float *>(smem + lay.rk);  // inverse key norms (1 without kQkL2Norm)
    float *sRQ = reinterpret_cast<float *>(smem + lay.rq);  // inverse query norms
    const bool qkn = (p.flags & kQkL2Norm) != 0;
    const int ldkq = kq_ld<Tin>(dk);

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);
    const bool want_o = o != nullptr;  // the backward's forward pass needs only the states
    const int SLD = st_ld(dk);

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

    // S <- h0 tile (or 0)
    const size_t sbase = ((size_t)n * Nv + h) * dk * dv;
    for (int idx = tid; idx < dk * BV; idx += NT) {
        const int d = idx / BV, c = idx - d * BV;
        sSt[c * SLD + d] = (p.h0 && c < bvw) ? p.h0[sbase + (size_t)d * dv + v0 + c] : 0.0f;
    }

    const int CH = p.chunk;  // 16, 32 or 64 (<= C)
    int ci = -1;  // chunk index (phase stamps of profiling builds)
    (void)ci;
    for (long long t0 = bos; t0 < eos; t0 += CH) {
        ++ci;
        const int L = (eos - t0) < CH ? (int)(eos - t0) : CH;
        __syncthreads();  // previous chunk fully consumed

        // backward's forward pass: keep the state this chunk starts from
        if (p.hs) {
            float *dst = p.hs + ((size_t)h * p.nslots + (size_t)(t0 / C + n)) * dk * dv + v0;
            for (int idx = tid; idx < dk * BV; idx += NT) {
                const int d = idx / BV, c = idx - d * BV;
                if (c < bvw) dst[(size_t)d * dv + c] = sSt[c * SLD + d];
            }
        }

        // ---- load the chunk (K and Q rows asynchronously, beside V) --------
        simt::load_rows_async<Tin, NT>(sK, k, t0, L, Nk, hk, dk, tid);
        simt::load_rows_async<Tin, NT>(sQ, q, t0, L, Nk, hk, dk, tid);
        for (int idx = tid; idx < C * BV; idx += NT) {
            const int i = idx / BV, c = idx - i * BV;
            sV[idx] = (i < L && c < bvw) ? to_f(v[((t0 + i) * Nv + h) * (long long)dv + v0 + c]) : 0.0f;
        }
        if (tid < C) {
            sBeta[tid] = tid < L ? p.beta[(t0 + tid) * Nv + h] : 0.0f;
            sG[tid] = (tid < L && p.g) ? p.g[(t0 + tid) * Nv + h] : 0.0f;
        }
        simt::cp_async_wait_all();
        __syncthreads();

        // ---- a1: gate prefix sum ----------------------------------------
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
            // warps 1-7: 1 / max(||x||, 1e-12) of every key and query row
            for (int rr = warp - 1; rr < 2 * C; rr += 7) {
                const int i = rr & (C - 1);
                float ss = 0.0f;
                if (qkn) {
                    const Tin *x = (rr < C ? sK : sQ) + i * ldkq;
                    for (int d = lane; d < dk; d += 32) {
                        const float f = to_f(x[d]);
                        ss = fmaf(f, f, ss);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                }
                if (lane == 0) (rr < C ? sRK : sRQ)[i] = qkn ? rsqrtf(fmaxf(ss, 1e-24f)) : 1.0f;
            }
        }
        __syncthreads();

        // ---- a2: A (strictly lower) and P (lower incl. diagonal) ---------
        simt::kq_products<NT>(sK, sQ, ldkq, dk, L, tid, [&](int i, int j, float kk, float qk) {
            float a = 0.0f, pv = 0.0f;
            if (i < L && j <= i) {
                const float dec = expf(sG[i] - sG[j]) * sRK[j];
                if (j < i) a = -sBeta[i] * sRK[i] * dec * kk;
                pv = p.scale * sRQ[i] * dec * qk;
            }
            sA[i * LDC + j] = a;
            sP[i * LDC + j] = pv;
        });
        __syncthreads();

        // ---- a3: T = (I - A)^-1, blocked over 16 x 16 blocks ----------------
        // (sVn, written only in a5, is the solve's scratch)
        simt::solve_T_blocked<NT>(sA, LDC, nullptr, sT, LDC, sVn, L, tid);

        // ---- a4/a5: R = diag(beta)(V - diag(e^G) K S_in); also Q S_in -----
        // thread: RP rows from i0; columns cg + 8 x (x < 4).  RP = 2 covers
        // 64 rows, RP = 1 the first 32 (enough for chunks of up to 32 tokens)
        auto ks_qs = [&](auto rows) {
            constexpr int RP = decltype(rows)::value;
            const int i0 = RP * (tid >> 3), cg = tid & 7;
            float ks[RP][4], qs[RP][4];
#pragma unroll
            for (int r = 0; r < RP; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) ks[r][x] = qs[r][x] = 0.0f;
            for (int d = 0; d < dk; d += 4) {
                float4 kr[RP], qr[RP];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    kr[r] = simt::ld4(sK + (i0 + r) * ldkq + d);
                    if (want_o) qr[r] = simt::ld4(sQ + (i0 + r) * ldkq + d);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(sSt + (cg + 8 * x) * SLD + d);
#pragma unroll
                    for (int r = 0; r < RP; ++r) {
                        ks[r][x] = fmaf(kr[r].x, s4.x, fmaf(kr[r].y, s4.y, fmaf(kr[r].z, s4.z, fmaf(kr[r].w, s4.w, ks[r][x]))));
                        if (want_o)
                            qs[r][x] = fmaf(qr[r].x, s4.x, fmaf(qr[r].y, s4.y, fmaf(qr[r].z, s4.z, fmaf(qr[r].w, s4.w, qs[r][x]))));
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const int i = i0 + r;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int cc = cg + 8 * x;
                    sR[i * BV + cc] = i < L ? sBeta[i] * (sV[i * BV + cc] - sEG[i] * sRK[i] * ks[r][x]) : 0.0f;
                    sOi[i * BV + cc] = p.scale * sEG[i] * sRQ[i] * qs[r][x];
                }
            }
        };
        if constexpr (MMA) {
            // 16 x 8 tiles of K S and Q S over the chunk's row tiles: warp w
            // takes column tile w % 4 and row tiles w / 4, w / 4 + 2 (below
            // L), loading each S^T fragment once for both
            const int g = lane >> 2, t = lane & 3, nt = warp & 3;
            const int mtiles = (L + 15) >> 4, m0 = warp >> 2;
            const int cb = 8 * nt + g;
            float ks[2][4] = {}, qs[2][4] = {};
            for (int d = t; d < dk; d += 8) {
                const uint32_t b0 = mmat::cvt(sSt[cb * SLD + d]), b1 = mmat::cvt(sSt[cb * SLD + d + 4]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int mt = m0 + 2 * j;
                    if (mt >= mtiles) break;
                    const int r0 = 16 * mt + g;
                    mmat::mma(ks[j], mmat::bf(sK[r0 * ldkq + d]), mmat::bf(sK[(r0 + 8) * ldkq + d]),
                              mmat::bf(sK[r0 * ldkq + d + 4]), mmat::bf(sK[(r0 + 8) * ldkq + d + 4]), b0, b1);
                    if (want_o)
                        mmat::mma(qs[j], mmat::bf(sQ[r0 * ldkq + d]), mmat::bf(sQ[(r0 + 8) * ldkq + d]),
                                  mmat::bf(sQ[r0 * ldkq + d + 4]), mmat::bf(sQ[(r0 + 8) * ldkq + d + 4]), b0, b1);
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int mt = m0 + 2 * j;
                if (mt >= mtiles) break;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 16 * mt + g + 8 * (e >> 1), cc = 8 * nt + 2 * t + (e & 1);
                    sR[i * BV + cc] = i < L ? sBeta[i] * (sV[i * BV + cc] - sEG[i] * sRK[i] * ks[j][e]) : 0.0f;
                    sOi[i * BV + cc] = p.scale * sEG[i] * sRQ[i] * qs[j][e];
                }
            }
        } else if (L <= 32) {
            ks_qs(std::integral_constant<int, 1>{});
        } else {
            ks_qs(std::integral_constant<int, 2>{});
        }
        __syncthreads();

        // ---- a5: v_new = T R (row i per warp, lane = column) ---------------
        const int c = lane;
        {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
            for (int j = 0; j < L; j += 4) {
                float rj[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) rj[x] = sR[(j + x) * BV + c];  // rows past L are zero
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(sT + (warp + 8 * r) * LDC + j);
                    acc[r] = fmaf(t4.x, rj[0], fmaf(t4.y, rj[1], fmaf(t4.z, rj[2], fmaf(t4.w, rj[3], acc[r]))));
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                sVn[i * BV + c] = i < L ? acc[r] : 0.0f;
            }
        }
        __syncthreads();

        // ---- a6: o = scale e^G (Q S_in) + P v_new ------------------------
        if (want_o) {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = sOi[(warp + 8 * r) * BV + c];
            for (int j = 0; j < L; j += 4) {
                float vj[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) vj[x] = sVn[(j + x) * BV + c];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float4 p4 = *reinterpret_cast<const float4 *>(sP + (warp + 8 * r) * LDC + j);
                    acc[r] = fmaf(p4.x, vj[0], fmaf(p4.y, vj[1], fmaf(p4.z, vj[2], fmaf(p4.w, vj[3], acc[r]))));
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = warp + 8 * r;
                if (i < L && c < bvw) put(o + ((t0 + i) * Nv + h) * (long long)dv + v0 + c, acc[r]);
            }
        }

        // ---- a5: S_out = e^{G_L} S_in + sum_i e^{G_L-G_i} k_i v_new_i^T ----
        // thread: columns 2 cp, 2 cp + 1; rows d0 .. d0 + 7 of S
        if constexpr (MMA) {
            // S^T[c][d] += sum_i (dec_i rk_i v_new[i][c]) k_i[d]: 16 x 8 tiles
            // of (value column, key index) over the chunk's rows
            // warp w: value-column tile w % 2, key-index tiles w / 2 + 4 j;
            // each A fragment (v_new rows) is built once for all of them
            const int g = lane >> 2, t = lane & 3;
            const float eGL = expf(sGL[0]);
            const int kend = (L + 7) >> 3;
            const int c0 = 16 * (warp & 1) + g, n0 = warp >> 1, ntn = dk >> 3;
            float acc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int nt = n0 + 4 * j;
                if (nt >= ntn) break;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[j][e] = eGL * sSt[(c0 + 8 * (e >> 1)) * SLD + 8 * nt + 2 * t + (e & 1)];
            }
            for (int kk = 0; kk < kend; ++kk) {
                const int i = 8 * kk + t;
                const float f0 = sDec[i] * sRK[i], f1 = sDec[i + 4] * sRK[i + 4];
                const uint32_t a0 = mmat::cvt(f0 * sVn[i * BV + c0]), a1 = mmat::cvt(f0 * sVn[i * BV + c0 + 8]),
                               a2 = mmat::cvt(f1 * sVn[(i + 4) * BV + c0]), a3 = mmat::cvt(f1 * sVn[(i + 4) * BV + c0 + 8]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int nt = n0 + 4 * j;
                    if (nt >= ntn) break;
                    const int dn = 8 * nt + g;
                    mmat::mma(acc[j], a0, a1, a2, a3, mmat::bf(sK[i * ldkq + dn]), mmat::bf(sK[(i + 4) * ldkq + dn]));
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int nt = n0 + 4 * j;
                if (nt >= ntn) break;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    sSt[(c0 + 8 * (e >> 1)) * SLD + 8 * nt + 2 * t + (e & 1)] = acc[j][e];
            }
        } else {
            const float eGL = expf(sGL[0]);
            const int ndg = dk >> 3;
            for (int tile = tid; tile < 16 * ndg; tile += NT) {
                const int c0 = 2 * (tile / ndg), d0 = 8 * (tile % ndg);
                float acc[2][8];
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    const float4 a = *reinterpret_cast<const float4 *>(sSt + (c0 + y) * SLD + d0);
                    const float4 b = *reinterpret_cast<const float4 *>(sSt + (c0 + y) * SLD + d0 + 4);
                    acc[y][0] = eGL * a.x; acc[y][1] = eGL * a.y; acc[y][2] = eGL * a.z; acc[y][3] = eGL * a.w;
                    acc[y][4] = eGL * b.x; acc[y][5] = eGL * b.y; acc[y][6] = eGL * b.z; acc[y][7] = eGL * b.w;
                }
                for (int i = 0; i < L; ++i) {
                    const float f = sDec[i] * sRK[i];
                    const float4 k0v = simt::ld4(sK + i * ldkq + d0), k1v = simt::ld4(sK + i * ldkq + d0 + 4);
                    const float kv[8] = {k0v.x, k0v.y, k0v.z, k0v.w, k1v.x, k1v.y, k1v.z, k1v.w};
#pragma unroll
                    for (int y = 0; y < 2; ++y) {
                        const float w = f * sVn[i * BV + c0 + y];
#pragma unroll
                        for (int x = 0; x < 8; ++x) acc[y][x] = fmaf(w, kv[x], acc[y][x]);
                    }
                }
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    *reinterpret_cast<float4 *>(sSt + (c0 + y) * SLD + d0) =
                        make_float4(acc[y][0], acc[y][1], acc[y][2], acc[y][3]);
                    *reinterpret_cast<float4 *>(sSt + (c0 + y) * SLD + d0 + 4) =
                        make_float4(acc[y][4], acc[y][5], acc[y][6], acc[y][7]);
                }
            }
        }
    }

    __syncthreads();
    if (p.ht) {
        for (int idx = tid; idx < dk * BV; idx += NT) {
            const int d = idx / BV, c = idx - d * BV;
            if (c < bvw) p.ht[sbase + (size_t)d * dv + v0 + c] = sSt[c * SLD + d];
        }
    }
}

}  // namespace

size_t simt_smem_bytes(int dk, bool bf16) {
    return bf16 ? layout<__nv_bfloat16>(dk).end : layout<float>(dk).end;
}

cudaError_t simt_launch(const Params &p, bool bf16, bool tf32, cudaStream_t stream, const char **name) {
    const int nvt = (p.dv + BV - 1) / BV;
    const long long grid = (long long)p.N * p.Nv * nvt;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = simt_smem_bytes(p.dk, bf16);
    cudaError_t err;
    if (bf16) {
        auto kern = tf32 ? simt_fwd<__nv_bfloat16, true> : simt_fwd<__nv_bfloat16, false>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<(unsigned)grid, NT, smem, stream>>>(p);
        *name = tf32 ? "simt_fwd<bf16,tf32>" : "simt_fwd<bf16>";
    } else {
        err = cudaFuncSetAttribute(simt_fwd<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        simt_fwd<float, false><<<(unsigned)grid, NT, smem, stream>>>(p);
        *name = "simt_fwd<f32>";
    }
    return cudaGetLastError();
}

}  // namespace dn
