// Token-serial ("fused recurrent") forward of the gated delta rule, for
// decoding and short sequences.
//
// Sources: "flash linear attention" (fla notes), Attention: the fused
//          recurrent forward walks the tokens of one sequence and head in
//          order, adds each token's key-value outer product to the state and
//          reads the output from the updated state; the RetNet layer there
//          uses it when the query length is at most 64.
//          [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §1: the gated
//          delta update, decay first ("forget first, then write").
//
// Per token t of a sequence, for one value head h (key head h / (Nv / Nk)):
//     S   <- e^{g_t} S
//     d   <- beta_t (v_t - S^T k_t)
//     S   <- S + k_t d^T
//     o_t <- scale S^T q_t
// in fp32, the same recurrence the chunk form evaluates blockwise.  With
// kQkL2Norm, k_t and q_t enter divided by max(||x||, 1e-12): the two factors
// ride on the dot products and on d, and the rows in shared memory stay as
// loaded.
//
// One 128-thread CTA per (sequence, value head, 32-column value tile).  The
// fp32 state tile S[dk][32] lives in registers: lane c owns value column
// v0 + c, warp w owns key rows [w dk/4, (w+1) dk/4).  The two dot products
// over d per token are split over the four warps and summed through shared
// memory (three barriers per token).  The state is read once (h0) and
// written once (ht), so a decode step is bound by those two transfers.
#include <cuda_bf16.h>
#include <math.h>

#include "dn_internal.h"

namespace dn {
namespace {

constexpr int RT = 128;  // threads per CTA
constexpr int RBV = 32;  // value columns per CTA

__device__ __forceinline__ float ld_f(const float *p, long long i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16 *p, long long i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_o(float *p, long long i, float x) { p[i] = x; }
__device__ __forceinline__ void st_o(__nv_bfloat16 *p, long long i, float x) { p[i] = __float2bfloat16_rn(x); }

template <typename Tin, int DK>
__global__ void __launch_bounds__(RT) rec_fwd(Params p) {
    constexpr int DPT = DK / 4;  // key rows per thread
    __shared__ float sk[DK], sq[DK];
    __shared__ float red[2][4][RBV];

    const int c = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nvt = (p.dv + RBV - 1) / RBV;
    const int vt = blockIdx.x % nvt;
    const int h = (blockIdx.x / nvt) % p.Nv;
    const int n = blockIdx.x / (nvt * p.Nv);
    const int hk = h / (p.Nv / p.Nk);
    const int v0 = vt * RBV;
    const bool col = v0 + c < p.dv;
    const int d0 = w * DPT;

    long long bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        if (bos < 0 || eos < bos || eos > p.tokens) {
            if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeq);
            bos = eos = 0;
        }
    } else {
        bos = (long long)n * p.T;
        eos = bos + p.T;
    }

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);

    // S <- h0 tile (or 0); row d of the tile is 32 consecutive floats
    float S[DPT];
    const size_t sbase = ((size_t)n * p.Nv + h) * DK * p.dv + v0 + c;
#pragma unroll
    for (int i = 0; i < DPT; ++i) S[i] = (p.h0 && col) ? p.h0[sbase + (size_t)(d0 + i) * p.dv] : 0.f;

    for (long long t = bos; t < eos; ++t) {
        // the token's k and q, shared by the CTA
        const long long kq = (t * p.Nk + hk) * (long long)DK;
        for (int d = threadIdx.x; d < DK; d += RT) {
            sk[d] = ld_f(k, kq + d);
            sq[d] = ld_f(q, kq + d);
        }
        const float beta = p.beta[t * p.Nv + h];
        const float decay = p.g ? __expf(p.g[t * p.Nv + h]) : 1.f;
        const float vc = col ? ld_f(v, (t * p.Nv + h) * (long long)p.dv + v0 + c) : 0.f;
        __syncthreads();
        // inverse norms of k_t and q_t (every warp computes both, in the same order)
        float nk = 1.f, nq = 1.f;
        if (p.flags & kQkL2Norm) {
            float a = 0.f, b = 0.f;
            for (int d = c; d < DK; d += 32) {
                a = fmaf(sk[d], sk[d], a);
                b = fmaf(sq[d], sq[d], b);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                b += __shfl_xor_sync(0xffffffffu, b, off);
            }
            nk = rsqrtf(fmaxf(a, 1e-24f));
            nq = rsqrtf(fmaxf(b, 1e-24f));
        }
        // S <- e^g S; this warp's share of (S^T k)_c
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            S[i] *= decay;
            part = fmaf(S[i], sk[d0 + i], part);
        }
        red[0][w][c] = part;
        __syncthreads();
        const float skc = nk * ((red[0][0][c] + red[0][1][c]) + (red[0][2][c] + red[0][3][c]));
        const float delta = beta * (vc - skc) * nk;  // k^ d = k (d / ||k||)
        // S <- S + k d^T; this warp's share of (S^T q)_c
        float op = 0.f;
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
            S[i] = fmaf(sk[d0 + i], delta, S[i]);
            op = fmaf(S[i], sq[d0 + i], op);
        }
        red[1][w][c] = op;
        __syncthreads();
        if (w == 0 && col)
            st_o(o, (t * p.Nv + h) * (long long)p.dv + v0 + c,
                 p.scale * nq * ((red[1][0][c] + red[1][1][c]) + (red[1][2][c] + red[1][3][c])));
    }
    if (p.ht && col) {
#pragma unroll
        for (int i = 0; i < DPT; ++i) p.ht[sbase + (size_t)(d0 + i) * p.dv] = S[i];
    }
}

template <typename Tin>
cudaError_t launch_dk(const Params &p, unsigned grid, cudaStream_t stream) {
    switch (p.dk) {
        case 16: rec_fwd<Tin, 16><<<grid, RT, 0, stream>>>(p); break;
        case 32: rec_fwd<Tin, 32><<<grid, RT, 0, stream>>>(p); break;
        case 64: rec_fwd<Tin, 64><<<grid, RT, 0, stream>>>(p); break;
        case 128: rec_fwd<Tin, 128><<<grid, RT, 0, stream>>>(p); break;
        case 256: rec_fwd<Tin, 256><<<grid, RT, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t recurrent_launch(const Params &p, bool bf16, cudaStream_t stream, const char **name) {
    const int nvt = (p.dv + RBV - 1) / RBV;
    const long long grid = (long long)p.N * p.Nv * nvt;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    *name = bf16 ? "rec_fwd<bf16>" : "rec_fwd<f32>";
    return bf16 ? launch_dk<__nv_bfloat16>(p, (unsigned)grid, stream) : launch_dk<float>(p, (unsigned)grid, stream);
}

}  // namespace dn
