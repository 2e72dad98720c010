// Tensor-core (tcgen05 / TMEM / TMA) scan kernel of the chunkwise gated delta
// rule forward, bf16 q/k/v/o, dk = 128, 128 value columns per CTA.
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.3;
//          [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §2.3-§3.4.
//
// The WY kernel (dn_wy.cu) has already written T' = T diag(beta e^G),
// T'' = T diag(beta) and P = tril(scale QK^T . D) of every chunk to the
// workspace.  One persistent CTA per (sequence, value head, 128-column value
// tile; after a placement lead of CTAs that exit at once, see tc_launch) then
// walks the sequence's 64-token chunks in order.  The fp32 state
// lives in tensor memory, transposed (lane = value column v, column = key
// index d), for the whole sequence.  Every contraction is a tcgen05 MMA with
// M = 128:
//
//   W   K^T T'^T         -> W^T                                   (a4)
//   U   V^T T''^T        -> U^T                                   (a4)
//   VN  U^T - S^T W^T    -> v_new^T (S^T as a bf16 TMEM operand)  (a5)
//   DS  S^T += v~^T K    -> state update, v~ = e^{G_L-G} v_new    (a5)
//   O   S^T Q~^T         -> inter-chunk output, Q~ = diag(scale e^G) Q  (a6)
//   PV  += v_new^T P^T   -> intra-chunk output, same accumulator   (a6)
//
// With in-kernel q / k normalisation (kQkL2Norm) the K and Q tiles stay as
// loaded: T' and P already carry the inverse norms, and the loader folds the
// per-token factors 1/||k_i|| into v~ and 1/||q_i|| into Q~.
//
// Warp roles (15 warps; warp w reaches TMEM lanes 32 (w % 4) .. +31, so each
// group of four consecutive warps covers all 128 lanes):
//   0      loader: TMA for the K, Q, V tiles of a chunk, bulk copies of the
//          chunk's T', T'' and P into three two-deep rings, and the gate
//          scalars (prefix sum G, e^G, decays) computed with warp shuffles;
//   1      chain MMA issuer (one thread: U, VN, DS) and TMEM owner;
//   2-5    prep: one thread issues W of the next chunk as soon as its tiles
//          and T' have landed; the warpgroup turns W^T into the bf16 -W^T
//          operand, running ahead of the state scan, then scales the chunk's
//          Q rows by scale e^G in place for O;
//   6-9    state: v_new and v~ operands; key blocks 0-1 of the state passes;
//   10-13  output: key blocks 2-3 of each state pass (the S^T operand or
//          ht); then reads o = scale e^{G} (S^T Q^T) + P v_new, transposes
//          it through shared memory, stores bf16 rows;
//   14     output MMA issuer (one thread: O, PV).
//
// acc_s holds the state divided by a running product of the chunk decays
// (chunk_decay in dn_chunk.cuh), so a chunk's decay needs no pass over the
// state: the state passes multiply by the product where they read it out.
//
// With Params::hs set (the backward's state pass, no o) the state passes also
// store the fp32 state each chunk starts from, and o is not written.
//
// Every wait is bounded: after kTimeoutNs a CTA records kStatusTimeout in the
// status word, raises a shared abort flag so the other roles stop too, drains
// its own outstanding copies and MMA work and frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "dn_chunk.cuh"
#include "dn_internal.h"
#include "dn_tc.h"
#include "dn_tmap.h"
#include "tc_ptx.cuh"
#include "dn_tc_sync.cuh"

namespace dn {
namespace {

using namespace ptx;
using namespace tcs;

constexpr int C = kChunk;      // 64
constexpr int DK = 128;
constexpr int BVT = 128;       // value columns per CTA
constexpr int NS = 3;          // pipeline stages of K/Q/V tiles
constexpr int NTHREADS = 480;
constexpr int kLeadCtas = 12;  // placement lead of the scan grid (tc_launch)

// ---- shared memory map (offsets from a 1024-byte aligned base) -------------
constexpr uint32_t STAGE_BYTES = 49152;  // K0 Q0 K1 Q1 V0 V1, 8 KB each
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_TP = OFF_STAGE + NS * STAGE_BYTES;  // T'  ring, 2 x 8 KB
constexpr uint32_t OFF_TU = OFF_TP + 2 * 8192;              // T'' ring, 2 x 8 KB
constexpr uint32_t OFF_PR = OFF_TU + 2 * 8192;              // P   ring, 2 x 8 KB
constexpr uint32_t OFF_WT = OFF_PR + 2 * 8192;              // -W^T 16 KB
constexpr uint32_t OFF_SCAL = OFF_WT + 16384;               // NS x 2048 B
constexpr uint32_t OFF_OST = OFF_SCAL + NS * SCAL_FLOATS * 4;  // output staging, 32 x 256 B
constexpr uint32_t OFF_BAR = OFF_OST + 8192;
constexpr int NBARS = 34;
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;          // TMEM base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;           // alignment slack

static_assert(OFF_TP % 1024 == 0 && OFF_TU % 1024 == 0 && OFF_PR % 1024 == 0 && OFF_WT % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
static_assert(SMEM_ALLOC <= 232448, "exceeds the 227 KB of shared memory per CTA");

// Barrier indices.
enum {
    B_FULL = 0,                 // NS: TMA bytes + loader scalars
    B_EMPTY = B_FULL + NS,      // NS: every reader of the stage is done
    B_QS = B_EMPTY + NS,        // NS: the stage's Q rows scaled by scale e^G (prep)
    B_TPF = B_QS + NS,          // 2: T' landed    (ring r's full barriers at B_TPF + 4 r)
    B_TUF = B_TPF + 4,          // 2: T'' landed
    B_PF = B_TUF + 4,           // 2: P landed
    B_WF = B_PF + 2,            // W^T in acc_w
    B_WSM_FULL,                 // -W^T bf16 operand in shared memory
    B_S_FULL,
    B_V_FULL,
    B_VSM_FULL,
    B_S_UPD,                    // DS of the chunk (and every earlier MMA) done
    B_D_FULL,                   // every MMA of the chunk done
    B_O_EMPTY,
    B_DRAIN,
    B_DRAIN2,
    B_DRAIN3,                   // the output issuer's own MMAs
    B_KF,                       // NS: the stage's K tiles (W reads them before the rest lands)
    B_COUNT = B_KF + NS
};
static_assert(B_COUNT <= NBARS, "barrier space");

// Tensor memory columns (fp32 accumulators; SB holds bf16 pairs).
// TM_V: two 64-column buffers (chunk parity); TM_SB: two 64-column buffers
// (bf16 S^T at the start of chunk c in buffer c & 1); TM_O: O and PV of a chunk.
constexpr uint32_t TM_W = 0, TM_V = 64, TM_S = 192, TM_SB = 320, TM_O = 448, TM_COLS = 512;

// Instruction descriptors.
constexpr uint32_t ID_W = idesc_bf16(128, 64, 1, 0);    // A MN-major (K^T), B K-major
constexpr uint32_t ID_U = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_VN = idesc_bf16(128, 64, 0, 1);   // A TMEM, B MN-major (-W^T rows d)
constexpr uint32_t ID_O = idesc_bf16(128, 64, 0, 0);    // A TMEM, B K-major (Q rows)
constexpr uint32_t ID_DS = idesc_bf16(128, 128, 0, 1);  // A TMEM, B MN-major (K rows)
constexpr uint32_t ID_PV = idesc_bf16(128, 64, 0, 0);   // A TMEM, B K-major (P rows)

__device__ __forceinline__ uint32_t bar(const Ctx &x, int i) { return x.base + OFF_BAR + 8u * i; }
__device__ __forceinline__ float *scal(const Ctx &x, int s) {
    return reinterpret_cast<float *>(x.gbase + OFF_SCAL + s * SCAL_FLOATS * 4);
}

struct Unit {
    long long bos, eos;
    int n, h, hk, v0, nc;
};

// Units of a launch: one per (sequence, value head, value-column tile).
__device__ __forceinline__ unsigned unit_count(const Params &p) {
    return (unsigned)p.N * (unsigned)p.Nv * (unsigned)(p.dv / BVT);
}

// Rank of this CTA's sequence in the launch order (its unit index over
// Nv x value tiles); the grid's first gridDim.x - unit_count(p) CTAs are the
// placement lead (see tc_launch) and have none.
__device__ __forceinline__ int unit_rank(const Params &p) {
    const int idx = (int)(blockIdx.x - (gridDim.x - unit_count(p)));
    return idx / ((p.dv / BVT) * p.Nv);
}

// The unit of this CTA, whose sequence is n (seq_of_rank of unit_rank).
__device__ __forceinline__ Unit unit_of(const Params &p, int n) {
    Unit u;
    const int nvt = p.dv / BVT;
    const int idx = (int)(blockIdx.x - (gridDim.x - unit_count(p)));
    const int vt = idx % nvt;
    u.h = (idx / nvt) % p.Nv;
    u.n = n;
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
    u.nc = (int)((u.eos - u.bos + p.chunk - 1) / p.chunk);
    return u;
}

// Bulk copy of ring r (0: T', 1: T'', 2: P) of chunk c into buffer c & 1
// (one thread; the buffer must be free).
__device__ __forceinline__ void load_ring(const Ctx &x, const Params &p, const Unit &u, int r, int c) {
    const long long t0 = u.bos + (long long)c * p.chunk;
    const uint8_t *slot = static_cast<const uint8_t *>(p.ws) +
                          ((size_t)u.h * p.nslots + (size_t)wy_slot(t0, u.n, p.chunk)) * kSlotBytes + 8192 * r;
    const uint32_t fb = bar(x, B_TPF + 4 * r + (c & 1));
    mbar_arrive_expect_tx(fb, 8192);
    bulk_load(x.base + OFF_TP + r * 16384 + (c & 1) * 8192, slot, 8192, fb);
}

// ---------------------------------------------------------------------------
// Loader warp: TMA tiles and gate scalars of each chunk, and the first two
// chunks' T', T'' and P images (later ones are fetched by their readers as
// soon as a ring buffer frees up).  armed is the last chunk whose stage was
// armed.
//
// The kernel is launched as a programmatic dependent of the WY kernel, so
// it can start while that kernel's last CTAs finish: the first stage's
// copies (q, k, v: inputs) go out first, and the workspace slots are read
// only after grid_dep_wait, here and in the two other threads that refill
// the rings.
// ---------------------------------------------------------------------------
template <bool QKN>
__device__ void loader_role(const Ctx x, const Params &p, const Unit u, const CUtensorMap *mK,
                            const CUtensorMap *mQ, const CUtensorMap *mV, int &armed) {
    const int lane = threadIdx.x & 31;
    armed = -1;
    float A = 1.f;  // running decay product A_c (chunk_decay), the same in every lane
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const long long t0 = u.bos + (long long)c * p.chunk;
        const int L = (int)min((long long)p.chunk, u.eos - t0);
        // the stage's copies: once every reader of its previous chunk is done
        auto arm = [&]() -> bool {
            if (!wwait(x, bar(x, B_EMPTY + s), ((c / NS) & 1) ^ 1)) return false;
            const uint32_t st = x.base + OFF_STAGE + s * STAGE_BYTES;
            if (lane == 0) {
                const uint32_t fb = bar(x, B_FULL + s), kb = bar(x, B_KF + s);
                mbar_arrive_expect_tx(kb, 16384);
                mbar_arrive_expect_tx(fb, STAGE_BYTES - 16384);
                const int tt = (int)t0;
                tma_load_3d(st + 0, mK, kb, 0, u.hk, tt);
                tma_load_3d(st + 16384, mK, kb, 64, u.hk, tt);
                tma_load_3d(st + 8192, mQ, fb, 0, u.hk, tt);
                tma_load_3d(st + 24576, mQ, fb, 64, u.hk, tt);
                tma_load_3d(st + 32768, mV, fb, u.v0, u.h, tt);
                tma_load_3d(st + 40960, mV, fb, u.v0 + 64, u.h, tt);
            }
            armed = c;
            return true;
        };
        // the WY kernel's slots of the first two chunks, once that kernel
        // has completed (issued even when arming failed: their readers drain
        // them)
        auto rings = [&]() {
            grid_dep_wait();
            if (lane == 0)
                for (int c2 = 0; c2 < min(u.nc, 2); ++c2)
                    for (int r = 0; r < 3; ++r) load_ring(x, p, u, r, c2);
        };
        constexpr bool qkn = QKN;
        // the first NS stages are free from the start: their copies go out
        // before the gates are loaded
        if (c < NS) {
            const bool ok = arm();
            // with normalisation chunk 0's scalars need its slot (the norms)
            if (c == 0 && (qkn || !ok)) rings();
            if (!ok) return;
        }
        // the gates (and the WY kernel's inverse q / k norms) come from
        // global memory while the stage is still in use
        ChunkScalars cs = chunk_scalars_load(p, u.h, t0, L, lane);
        if (qkn)
            chunk_norms_load(cs, static_cast<const uint8_t *>(p.ws) +
                                     ((size_t)u.h * p.nslots + (size_t)wy_slot(t0, u.n, p.chunk)) * kSlotBytes +
                                     kSlotNormOff,
                             lane);
        const ChunkDecay dec = chunk_decay(cs.GL, A);
        A = dec.an;
        cs.ka /= dec.an;  // rides on e^{G_L - G_i}: v~ / A_{c+1}
        cs.kb /= dec.an;
        if (c >= NS && !arm()) return;
        chunk_scalars_store(p, cs, scal(x, s), lane);
        if (lane == 0) chunk_decay_store(scal(x, s), dec);
        __syncwarp();
#ifdef DN_TEST_STALL
        // failure-path test: the first stage's second arrival never comes, so
        // every wait on it runs out (its TMA bytes still land)
        const bool skip = p.test_stall == kStallScan && c == 0;
#else
        const bool skip = false;
#endif
        if (lane == 0 && !skip) mbar_arrive(bar(x, B_FULL + s));
        // without normalisation chunk 0's stage (tiles and scalars) is out
        // before the wait for the WY kernel, so that the initial state and
        // everything else that needs no slot can proceed
        if (c == 0 && !qkn) rings();
    }
}

// ---------------------------------------------------------------------------
// MMA issue helpers.
// ---------------------------------------------------------------------------
// W^T = K^T T'^T of chunk c into acc_w.
__device__ __forceinline__ void issue_w(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES;
    const uint32_t tp = x.base + OFF_TP + (c & 1) * 8192;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + TM_W, sdesc(st + kk * 2048, 16384, 1024), sdesc(tp + kk * 32, 16, 1024), ID_W, kk != 0);
}

// U^T = V^T T''^T of chunk c into acc_v[c & 1].
__device__ __forceinline__ void issue_u(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES + 32768;
    const uint32_t tpp = x.base + OFF_TU + (c & 1) * 8192;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss(tm + TM_V + 64 * (c & 1), sdesc(st + kk * 2048, 8192, 1024), sdesc(tpp + kk * 32, 16, 1024), ID_U,
               kk != 0);
}

// O^T = S^T Q~^T (inter-chunk output, Q~ = diag(scale e^G) Q) of chunk c into acc_o.
__device__ __forceinline__ void issue_o(const Ctx &x, uint32_t tm, int c) {
    const uint32_t st = x.base + OFF_STAGE + (c % NS) * STAGE_BYTES;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_O, tm + TM_SB + 64 * (c & 1) + kb * 32 + kk * 8,
                   sdesc(st + 8192 + kb * 16384 + kk * 32, 16, 1024), ID_O, (kb | kk) != 0);
}

// ---------------------------------------------------------------------------
// Chain MMA issuer (one thread): the MMAs on the serial chain of the scan,
//   VN(c); DS(c); U(c+1).
// Issuing a tcgen05 MMA holds the issuing thread for tens of cycles, so O(c)
// and PV(c), which are off the chain, have their own issuer thread (warp
// 14); they enter the in-order tensor pipe after DS(c) and run while the
// state is converted.  This thread also refills the
// T'' and P rings as their buffers free up (W and the T' ring belong to the
// prep warpgroup).
// ---------------------------------------------------------------------------
// (ring 0, T': the W MMA reads only the stage's K tiles)
__device__ __forceinline__ bool wait_tiles(const Ctx &x, int c, int ring) {
    return wait(x, bar(x, (ring == 0 ? B_KF : B_FULL) + c % NS), (c / NS) & 1) &&
           wait(x, bar(x, B_TPF + 4 * ring + (c & 1)), (c >> 1) & 1);
}

__device__ void mma_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    int loaded[3];  // last chunk whose T'' / P copy was issued (index 1, 2)
    loaded[1] = loaded[2] = min(u.nc, 2) - 1;
    grid_dep_wait();  // this thread refills the T'' and P rings from the workspace
    int c = 0;
    if (wait_tiles(x, 0, 1)) {
        tc_fence_after();
        issue_u(x, tm, 0);
    } else {
        c = u.nc;
    }
    for (; c < u.nc; ++c) {
        const int s = c % NS, t = c & 1;
        const uint32_t st = x.base + OFF_STAGE + s * STAGE_BYTES;
        const uint32_t par = c & 1;
        const uint32_t av = tm + TM_V + 64 * t;  // acc_v of this chunk
        // v_new^T = U^T + S^T (-W^T), accumulated onto U^T (issued before by
        // this thread, so in order)
        if (!wait(x, bar(x, B_WSM_FULL), par)) break;
        if (!wait(x, bar(x, B_S_FULL), par)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_ts(av, tm + TM_SB + 64 * t + kk * 8, sdesc(x.base + OFF_WT + kk * 2048, 8192, 1024), ID_VN, 1);
        mma_commit(bar(x, B_V_FULL));
        // U of the next chunk into the other acc_v buffer, whose last readers
        // (DS / PV of chunk c - 1) are done; PV of c - 1 also freed the P
        // buffer of chunk c + 1
        if (c > 0) {
            if (!wait(x, bar(x, B_D_FULL), (c - 1) & 1)) break;
            if (c + 1 < u.nc) {
                load_ring(x, p, u, 2, c + 1);
                loaded[2] = c + 1;
            }
        }
        // state update (VSM also means VN, hence U, of this chunk is done:
        // its T'' buffer takes chunk c + 2's)
        if (!wait(x, bar(x, B_VSM_FULL), par)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_S, av + 32 + kk * 8, sdesc(st + kk * 2048, 16384, 1024), ID_DS, 1);
        mma_commit(bar(x, B_S_UPD));
        // U of the next chunk, behind DS in the tensor pipe: issued while
        // v_new was converted it slowed that conversion more than it gains
        if (c + 1 < u.nc) {
            if (!wait_tiles(x, c + 1, 1)) break;
            tc_fence_after();
            issue_u(x, tm, c + 1);
        }
        if (c + 2 < u.nc) {
            load_ring(x, p, u, 1, c + 2);
            loaded[1] = c + 2;
        }
    }
    // every MMA issued by this thread completes before tensor memory is
    // freed, and the last ring copies it issued land before shared memory
    // goes
    mma_commit(bar(x, B_DRAIN));
    wait_drain(bar(x, B_DRAIN), 0);
    for (int r = 1; r < 3; ++r)
        for (int k = max(loaded[r] - 1, 0); k <= loaded[r]; ++k)
            wait_drain(bar(x, B_TPF + 4 * r + (k & 1)), (k >> 1) & 1);
}

// ---------------------------------------------------------------------------
// The fp32 state acc_s (TMEM lane = value column, 128 columns = key index d)
// is handled in 32-column blocks: blocks 0-1 by the state warpgroup, blocks
// 2-3 by the output warpgroup, which is otherwise idle in the window after
// DS.  Halving each pass halves the S^T conversion on the scan's serial
// chain.  `lb` is the thread's TMEM lane base; `hb` its element of h0 / ht at
// key index 0 (row stride dv).
// ---------------------------------------------------------------------------
// The initial state, key blocks b0 and b0 + 1: f = the lane's h0 rows (zero
// without h0), then SB[0] = bf16(h0^T) (and, with hsd, the fp32 state chunk 0
// starts from), and once chunk 0's scalars are out acc_s = s0 h0^T, with s0 =
// alpha_0 when chunk 0 renormalises and 1 otherwise (chunk_decay: A_0 = 1).
// The loads go out before the wait for the scalars, so that their latency
// overlaps the first stage's copies.
// Column of this lane's value column v in the saved state of chunk c (row
// d = 0, rows dv apart), or null when the states are not saved (HS: the
// backward's state pass).
template <bool HS>
__device__ __forceinline__ float *hs_col(const Params &p, const Unit &u, int c, int v) {
    if (!HS) return nullptr;
    const long long slot = wy_slot(u.bos + (long long)c * p.chunk, u.n, p.chunk);
    return p.hs + ((size_t)u.h * p.nslots + (size_t)slot) * DK * p.dv + u.v0 + v;
}

__device__ __forceinline__ void state_init_load(const Params &p, size_t hb, int b0, float (&f)[2][32]) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float *hp = p.h0 ? p.h0 + hb + (size_t)(32 * (b0 + e)) * p.dv : nullptr;
#pragma unroll
        for (int k = 0; k < 32; ++k) f[e][k] = hp ? hp[(size_t)k * p.dv] : 0.f;
    }
}

__device__ __forceinline__ void state_init_sb(const Params &p, uint32_t lb, int b0, const float (&f)[2][32],
                                              float *hsd) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int blk = b0 + e;
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(f[e][2 * k], f[e][2 * k + 1]);
        tmem_st16(lb + TM_SB + 16 * blk, pk);
        if (hsd) {
            float *dp = hsd + (size_t)(32 * blk) * p.dv;
#pragma unroll
            for (int k = 0; k < 32; ++k) dp[(size_t)k * p.dv] = f[e][k];
        }
    }
}

__device__ __forceinline__ void state_init_s(uint32_t lb, int b0, float s0, const float (&f)[2][32]) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        uint32_t r[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(s0 * f[e][k]);
        tmem_st32(lb + TM_S + 32 * (b0 + e), r);
    }
}

// The last chunk's ht = a acc_s, key blocks b0 and b0 + 1 (out of line: run once).
__device__ __noinline__ void state_write_ht(const Params &p, uint32_t lb, size_t hb, int b0, float a) {
    if (!p.ht) return;
    for (int e = 0; e < 2; ++e) {
        uint32_t r[32];
        tmem_ld32(lb + TM_S + 32 * (b0 + e), r);
        tmem_wait_ld_dep(r);
        float *hp = p.ht + hb + (size_t)(32 * (b0 + e)) * p.dv;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            *hp = a * __uint_as_float(r[k]);
            hp += p.dv;
        }
    }
}

// After DS(c), key blocks b0 and b0 + 1: SB[(c+1) & 1] = bf16(a acc_s) with
// a = A_{c+1} (and, with hsd, the fp32 state chunk c + 1 starts from); or for
// the last chunk ht = a acc_s with a = A_{nc} (chunk_decay), out of line.
// Both TMEM loads are in flight before the one wait.
__device__ __forceinline__ void state_convert_blocks(const Params &p, uint32_t lb, size_t hb, int c, bool last,
                                                     int b0, float *hsd, float a) {
    if (last) {
        state_write_ht(p, lb, hb, b0, a);
        return;
    }
    uint32_t r[2][32];
    tmem_ld32(lb + TM_S + 32 * b0, r[0]);
    tmem_ld32(lb + TM_S + 32 * (b0 + 1), r[1]);
    tmem_wait_ld_dep(r[0]);
    tmem_ld_dep(r[1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int blk = b0 + e;
        if (!last) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = pack_bf16(a * __uint_as_float(r[e][2 * k]), a * __uint_as_float(r[e][2 * k + 1]));
            tmem_st16(lb + TM_SB + 64 * ((c + 1) & 1) + 16 * blk, pk);
            if (hsd) {
                float *dp = hsd + (size_t)(32 * blk) * p.dv;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    *dp = a * __uint_as_float(r[e][k]);
                    dp += p.dv;
                }
            }
        }
    }
}

// A renormalising chunk c + 1 (chunk_decay): acc_s *= rs = alpha_{c+1}
// A_{c+1} before DS(c+1), key blocks b0 and b0 + 1.
__device__ __noinline__ void state_renorm_blocks(uint32_t lb, float rs, int b0) {
    uint32_t r[2][32];
    tmem_ld32(lb + TM_S + 32 * b0, r[0]);
    tmem_ld32(lb + TM_S + 32 * (b0 + 1), r[1]);
    tmem_wait_ld_dep(r[0]);
    tmem_ld_dep(r[1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[e][k] = __float_as_uint(rs * __uint_as_float(r[e][k]));
        tmem_st32(lb + TM_S + 32 * (b0 + e), r[e]);
    }
}

// ---------------------------------------------------------------------------
// Output warpgroup: o[i][v] = (S^T Q~^T + v_new^T P^T)[v][i] for value column
// v = this thread's TMEM lane, chunk by chunk once O and PV are done.
// ---------------------------------------------------------------------------
template <bool HS>
__device__ void output_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);
    const int tid = threadIdx.x - 320;  // 0..127 in the output warpgroup
    const uint32_t lb = lane_base(tm, warp);
    const uint32_t buf = x.base + OFF_OST;
    const uint8_t *gbuf = x.gbase + OFF_OST;
    const long long rstride = (long long)p.Nv * p.dv * 2;  // bytes between tokens
    const size_t hb = ((size_t)u.n * p.Nv + u.h) * DK * p.dv + u.v0 + v;  // h0 / ht of this lane
    if (u.nc > 0) {
        // blocks 2-3 of the initial state; then acc_s is ready for DS(0)
        float f[2][32];
        state_init_load(p, hb, 2, f);
        state_init_sb(p, lb, 2, f, hs_col<HS>(p, u, 0, v));
        if (!bar_red_or(2, 128, !wwait(x, bar(x, B_FULL + 0), 0))) {
            const float *s0 = scal(x, 0);
            state_init_s(lb, 2, s0[SC_RN] != 0.f ? s0[SC_RS] : 1.f, f);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(x, B_S_FULL));
            warp_arrive(bar(x, B_VSM_FULL));
        }
    }
    for (int c = 0; c < u.nc; ++c) {
        // Every exit is taken by the whole warpgroup together (bar_red_or), so
        // no warp is left waiting at one of its named barriers.
        // Blocks 2-3 of the state: the S^T operand of chunk c + 1 (or ht);
        // acc_s is then ready for DS(c+1) (VSM_FULL).
        const bool last = c + 1 == u.nc;
        const int s1 = (c + 1) % NS;
        if (!last && bar_red_or(2, 128, !wwait(x, bar(x, B_FULL + s1), ((c + 1) / NS) & 1))) break;
        const float *sn = scal(x, last ? c % NS : s1);
        if (bar_red_or(2, 128, !wwait(x, bar(x, B_S_UPD), c & 1))) break;
        tc_fence_after();
        state_convert_blocks(p, lb, hb, c, last, 2, last ? nullptr : hs_col<HS>(p, u, c + 1, v),
                             last ? sn[SC_AN] : sn[SC_A]);
        if (!last && sn[SC_RN] != 0.f) state_renorm_blocks(lb, sn[SC_RS], 2);
        if (!last) {
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(x, B_S_FULL));
            warp_arrive(bar(x, B_VSM_FULL));
        }
        if (bar_red_or(2, 128, !wwait(x, bar(x, B_D_FULL), c & 1))) break;
        tc_fence_after();
        const long long t0 = u.bos + (long long)c * p.chunk;
        const int L = (int)min((long long)p.chunk, u.eos - t0);
        // the chunk's output column v as packed bf16 pairs (tokens 2k, 2k + 1)
        // (with no o, as in the backward's state pass, only the hand-off)
        uint32_t ob[32];
        if (!HS) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t ra[32];
                tmem_ld32(lb + TM_O + 32 * hf, ra);
                tmem_wait_ld_dep(ra);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    ob[16 * hf + k] = pack_bf16(__uint_as_float(ra[2 * k]), __uint_as_float(ra[2 * k + 1]));
            }
        }
        tc_fence_before();
        warp_arrive(bar(x, B_O_EMPTY));
        if (HS) continue;
        // transpose through shared memory, 32 tokens x 128 value columns
        // (256-byte rows) at a time, then 16-byte stores of whole rows i < L
        // (loops here and in the prep warpgroup are left rolled where they
        // are off the chain: the scan measured faster with a smaller
        // instruction footprint)
        uint8_t *obase = static_cast<uint8_t *>(p.o) + ((t0 * p.Nv + u.h) * (long long)p.dv + u.v0) * 2;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t w = hf ? ob[16 + k] : ob[k];
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(buf + (2 * k) * 256 + 2 * v),
                             "h"((uint16_t)(w & 0xffffu)));
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(buf + (2 * k + 1) * 256 + 2 * v),
                             "h"((uint16_t)(w >> 16)));
            }
            named_bar_sync(2, 128);
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int idx = tid + 128 * it, r = idx >> 4, ch = idx & 15;
                const int i = 32 * hf + r;
                const uint4 val = *reinterpret_cast<const uint4 *>(gbuf + r * 256 + ch * 16);
                if (i < L) *reinterpret_cast<uint4 *>(obase + i * rstride + ch * 16) = val;
            }
            named_bar_sync(2, 128);
        }
    }
}

// ---------------------------------------------------------------------------
// Output MMA issuer (warp 14, one thread): O(c) = S_in(c)^T Q~^T and
// PV(c) = v_new(c)^T P(c)^T into acc_o.  S_UPD(c): DS(c) is done, so these
// follow it in the tensor pipe and run while the state is converted (VSM(c),
// hence v_new^T(c), was ready before DS(c) was issued).  O_EMPTY: acc_o of
// chunk c - 1 has been read.  Issuing holds the issuing thread for tens of
// cycles per MMA, which is why neither the chain thread nor a thread of a
// converting warpgroup does it.
// ---------------------------------------------------------------------------
__device__ void out_mma_role(const Ctx x, const Unit u, uint32_t tm) {
    bool issued = false;
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS, t = c & 1;
        if (!(wait(x, bar(x, B_S_UPD), c & 1) && wait(x, bar(x, B_O_EMPTY), (c & 1) ^ 1) &&
              wait(x, bar(x, B_QS + s), (c / NS) & 1) && wait(x, bar(x, B_PF + t), (c >> 1) & 1)))
            break;
        tc_fence_after();
        issue_o(x, tm, c);
        const uint32_t av = tm + TM_V + 64 * t;
        const uint32_t pbuf = x.base + OFF_PR + t * 8192;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ts(tm + TM_O, av + kk * 8, sdesc(pbuf + kk * 32, 16, 1024), ID_PV, 1);
        mma_commit(bar(x, B_D_FULL));
        mma_commit(bar(x, B_EMPTY + s));  // the last reader of the stage
        issued = true;
    }
    // every MMA this thread issued completes before tensor memory is freed
    if (issued) {
        mma_commit(bar(x, B_DRAIN3));
        wait_drain(bar(x, B_DRAIN3), 0);
    }
}

// ---------------------------------------------------------------------------
// Prep warpgroup: W^T of each chunk (acc_w) into the bf16 -W^T operand of VN.
// One thread issues W of the next chunk as soon as this chunk's operand is
// out, and refills the T' ring.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool issue_w_mma(const Ctx &x, uint32_t tm, int c) {
    const bool ok = wait_tiles(x, c, 0);
    if (ok) {
        tc_fence_after();
        issue_w(x, tm, c);
        mma_commit(bar(x, B_WF));
    }
    return ok;
}

// Q row i *= scale e^{G_i} in place (bf16) for chunk c, so that O and PV
// share one accumulator: o_i = S^T (scale e^{G_i} q_i) + sum_j P_ij v_new_j.
// 128 threads; each step of a warp covers 512 contiguous bytes (4 rows x 8
// chunks of 16 B), free of bank conflicts; the swizzle only permutes chunks
// within a row.  Returns false if the stage did not arrive.
__device__ __forceinline__ bool scale_q(const Ctx &x, int c) {
    const int s = c % NS;
    if (!wwait(x, bar(x, B_FULL + s), (c / NS) & 1)) return false;
    const float *sc = scal(x, s);
    const int tid = threadIdx.x - 64;
#pragma unroll 2
    for (int it = 0; it < 8; ++it) {
        const int k = tid + 128 * it, half = k >> 9, r = (k >> 3) & 63, ch = k & 7;
        const float f = sc[SC_OSC + r];
        uint4 *qp = reinterpret_cast<uint4 *>(x.gbase + OFF_STAGE + s * STAGE_BYTES + 8192 + 16384 * half + 128 * r +
                                              16 * ch);
        const uint4 q = *qp;
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
            w[e] = pack_bf16(lo * f, hi * f);
        }
        *qp = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    warp_arrive(bar(x, B_QS + s));
    return true;
}

__device__ void prep_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const bool leader = warp == 2 && (threadIdx.x & 31) == 0;
    const int row = 32 * (warp & 3) + (threadIdx.x & 31);  // TMEM lane = key index d
    const uint32_t lb = lane_base(tm, warp);
    int loaded = min(u.nc, 2) - 1;  // last chunk whose T' copy was issued
    bool lok = true;                // the leader's own waits
    if (leader) grid_dep_wait();    // it refills the T' ring from the workspace
    if (leader && u.nc > 0) lok = issue_w_mma(x, tm, 0);
    for (int c = 0; c < u.nc; ++c) {
        if (!wwait(x, bar(x, B_WF), c & 1) || !__all_sync(0xffffffffu, lok)) break;
        // W of chunk c is done with its T' buffer: it takes chunk c + 2's
        if (leader && c + 2 < u.nc) {
            load_ring(x, p, u, 0, c + 2);
            loaded = c + 2;
        }
        // the -W^T buffer is free once the chain's VN of the chunk before has
        // completed
        if (c > 0 && !wwait(x, bar(x, B_V_FULL), (c - 1) & 1)) break;
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(lb + TM_W, r0);
        tmem_ld32(lb + TM_W + 32, r1);
        tmem_wait_ld_dep(r0);
        tmem_wait_ld_dep(r1);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 8 * ch + 2 * e;
                    w[e] = pack_bf16(-__uint_as_float(hf ? r1[k] : r0[k]), -__uint_as_float(hf ? r1[k + 1] : r0[k + 1]));
                }
                st_shared_v4(x.base + OFF_WT + sw128(row, 4 * hf + ch), w[0], w[1], w[2], w[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(x, B_WSM_FULL));
        // the next chunk's W, once all four warps have read acc_w (their
        // WSM arrivals)
        if (leader && c + 1 < u.nc) lok = wait(x, bar(x, B_WSM_FULL), c & 1) && issue_w_mma(x, tm, c + 1);
        // this chunk's Q rows, which only O(c) reads (after DS(c)): off the
        // path from the stage's arrival to -W^T
        if (!scale_q(x, c)) break;
    }
    if (leader) {
        // W completes before tensor memory is freed; the last T' copies it
        // issued land before shared memory goes
        mma_commit(bar(x, B_DRAIN2));
        wait_drain(bar(x, B_DRAIN2), 0);
        for (int k = max(loaded - 1, 0); k <= loaded; ++k) wait_drain(bar(x, B_TPF + (k & 1)), (k >> 1) & 1);
    }
}

// ---------------------------------------------------------------------------
// State warpgroup: v_new operands, fp32 state, ht.
// ---------------------------------------------------------------------------
template <bool HS>
__device__ void state_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);  // value column = TMEM lane
    const uint32_t lb = lane_base(tm, warp);
    const size_t sbase = ((size_t)u.n * p.Nv + u.h) * DK * p.dv + u.v0 + v;
    const int dv = p.dv;

    if (u.nc == 0) {  // empty sequence: ht = h0
        if (p.ht)
            for (int d = 0; d < DK; ++d) p.ht[sbase + (size_t)d * dv] = p.h0 ? p.h0[sbase + (size_t)d * dv] : 0.f;
        return;
    }
    // initial state: acc_s = s0 h0^T, SB = bf16(h0^T) (blocks 0-1 here,
    // 2-3 in the output warpgroup)
    {
        float f[2][32];
        state_init_load(p, sbase, 0, f);
        state_init_sb(p, lb, 0, f, hs_col<HS>(p, u, 0, v));
        if (!wwait(x, bar(x, B_FULL + 0), 0)) return;
        const float *s0 = scal(x, 0);
        state_init_s(lb, 0, s0[SC_RN] != 0.f ? s0[SC_RS] : 1.f, f);
    }
    tmem_wait_st();
    tc_fence_before();
    warp_arrive(bar(x, B_S_FULL));
    for (int c = 0; c < u.nc; ++c) {
        const int s = c % NS;
        const uint32_t par = c & 1;
        // ---- v_new^T and v~^T operands --------------------------------
        // acc_v columns j = 0..63 (fp32) become v_new^T packed in columns
        // 0..31 and v~^T packed in columns 32..63; a column is rewritten only
        // after it has been read.
        if (!wwait(x, bar(x, B_V_FULL), par)) return;
        // O(c - 1), the last reader of the bf16 S^T buffer this chunk's state
        // pass rewrites, comes from the output issuer: wait for its commit.
        // (D_FULL(c) needs this warpgroup's VSM(c), so the barrier is at most
        // one phase ahead here.)
        if (c > 0 && !wwait(x, bar(x, B_D_FULL), (c - 1) & 1)) return;
        tc_fence_after();
        {
            const float4 *dec4 = reinterpret_cast<const float4 *>(scal(x, s) + SC_DEC);
            const uint32_t lbv = lb + TM_V + 64 * (c & 1);
            uint32_t r[32], tvh[16];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                tmem_ld32(lbv + 32 * hf, r);
                tmem_wait_ld_dep(r);
                if (hf == 1) tmem_st16(lbv + 32, tvh);  // columns 32-47 are loaded now
                uint32_t pv[16], tv[16];
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 dd = dec4[8 * hf + k4];
                    const float a0 = __uint_as_float(r[4 * k4]), a1 = __uint_as_float(r[4 * k4 + 1]);
                    const float a2 = __uint_as_float(r[4 * k4 + 2]), a3 = __uint_as_float(r[4 * k4 + 3]);
                    pv[2 * k4] = pack_bf16(a0, a1);
                    pv[2 * k4 + 1] = pack_bf16(a2, a3);
                    tv[2 * k4] = pack_bf16(a0 * dd.x, a1 * dd.y);
                    tv[2 * k4 + 1] = pack_bf16(a2 * dd.z, a3 * dd.w);
                }
                tmem_st16(lbv + 16 * hf, pv);
                if (hf == 0) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) tvh[k] = tv[k];
                } else {
                    tmem_st16(lbv + 48, tv);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(x, B_VSM_FULL));
        }
        warp_arrive(bar(x, B_EMPTY + s));  // done with this chunk's scalars
        // ---- state: S_in(c+1) operand (blocks 0-1) -----------------------
        const bool last = (c + 1 == u.nc);
        const int s1 = (c + 1) % NS;
        if (!last && !wwait(x, bar(x, B_FULL + s1), ((c + 1) / NS) & 1)) return;
        const float *sn = scal(x, last ? s : s1);
        if (!wwait(x, bar(x, B_S_UPD), par)) return;
        tc_fence_after();
        state_convert_blocks(p, lb, sbase, c, last, 0, last ? nullptr : hs_col<HS>(p, u, c + 1, v),
                             last ? sn[SC_AN] : sn[SC_A]);
        if (last) break;
        if (sn[SC_RN] != 0.f) state_renorm_blocks(lb, sn[SC_RS], 0);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(x, B_S_FULL));
    }
}

// ---------------------------------------------------------------------------
// Output warpgroup: o = scale e^{G_i} (S^T Q^T)[v][i] + (v_new^T P^T)[v][i].
// ---------------------------------------------------------------------------
// HS: the backward's state pass (p.hs set, no o); QKN: in-kernel q / k
// normalisation.  Template parameters, so that the forward's instance
// carries neither path's code.
template <bool HS, bool QKN>
__global__ void __maxnreg__(128)
tc_fwd(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
       const __grid_constant__ CUtensorMap mV, const __grid_constant__ Params p) {
    if (blockIdx.x + unit_count(p) < gridDim.x) return;  // placement lead: no unit
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Ctx x;
    x.base = (raw + 1023u) & ~1023u;
    x.gbase = smem_raw + (x.base - raw);
    x.abort_flag = reinterpret_cast<volatile int *>(x.gbase + OFF_MISC + 4);
    x.status = p.status;
    const int warp = threadIdx.x >> 5;
    const Unit u = unit_of(p, seq_of_rank(p, unit_rank(p), threadIdx.x & 31));

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(x, B_FULL + s), 2);
            mbar_init(bar(x, B_KF + s), 1);
            mbar_init(bar(x, B_EMPTY + s), 5);
            mbar_init(bar(x, B_QS + s), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(x, B_TPF + b), 1);
            mbar_init(bar(x, B_TUF + b), 1);
            mbar_init(bar(x, B_PF + b), 1);
        }
        mbar_init(bar(x, B_WF), 1);
        mbar_init(bar(x, B_WSM_FULL), 4);
        mbar_init(bar(x, B_S_FULL), 8);    // state and output warpgroups, half the state each
        mbar_init(bar(x, B_V_FULL), 1);
        mbar_init(bar(x, B_VSM_FULL), 8);  // state (v_new^T, v~^T) and output (acc_s scaled)
        mbar_init(bar(x, B_S_UPD), 1);
        mbar_init(bar(x, B_D_FULL), 1);
        mbar_init(bar(x, B_O_EMPTY), 4);
        mbar_init(bar(x, B_DRAIN), 1);
        mbar_init(bar(x, B_DRAIN2), 1);
        mbar_init(bar(x, B_DRAIN3), 1);
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
        int armed = -1;
        loader_role<QKN>(x, p, u, &mK, &mQ, &mV, armed);
        // drain: the last NS armed stages must have landed before exit (the
        // ring copies are drained by the roles that issued them)
        if ((threadIdx.x & 31) == 0)
            for (int c = armed - NS + 1; c <= armed; ++c)
                if (c >= 0) {
                    wait_drain(bar(x, B_FULL + c % NS), (c / NS) & 1);
                    wait_drain(bar(x, B_KF + c % NS), (c / NS) & 1);
                }
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0 && u.nc > 0) mma_role(x, p, u, tm);
        __syncwarp();
    } else if (warp < 6) {
        prep_role(x, p, u, tm);
    } else if (warp < 10) {
        state_role<HS>(x, p, u, tm);
    } else if (warp < 14) {
        output_role<HS>(x, p, u, tm);
    } else {
        if ((threadIdx.x & 31) == 0) out_mma_role(x, u, tm);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tm, TM_COLS);
}

}  // namespace

bool tc_supported(int dk, int dv, bool bf16, int chunk) {
    return bf16 && (dk == DK || dk == 256) && dv % BVT == 0 && (chunk == 16 || chunk == 32 || chunk == C);
}

size_t tc_workspace_bytes(long long tokens, int N, int Nv, int dk, int chunk) {
    if (tokens <= 0 || N <= 0 || chunk <= 0) return 0;
    return (size_t)(tokens / chunk + N) * (size_t)Nv * slot_bytes(dk);
}

cudaError_t tc_launch(const Params &p, cudaStream_t stream, const char **name) {
    if (p.dk == 256) return tc_wide_launch(p, stream, name);
    CUtensorMap mK, mQ, mV;
    const uint64_t tokens = (uint64_t)p.tokens;
    if (!make_tmap_rows_heads_d(&mK, p.k, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mQ, p.q, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mV, p.v, tokens, p.Nv, p.dv, 64, C))
        return cudaErrorInvalidValue;
    const long long grid = (long long)p.N * p.Nv * (p.dv / BVT);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    // T', T'' and P of every chunk first (all chunks in parallel), then the scan
    cudaError_t err = wy_launch(p, mK, mQ, stream);
    if (err != cudaSuccess) return err;
    // the backward's state pass saves the states and writes no o; the
    // forward writes o
    const bool hs = p.hs != nullptr, qkn = (p.flags & kQkL2Norm) != 0;
    if (hs != (p.o == nullptr)) return cudaErrorInvalidValue;
    const void *kern = hs ? (qkn ? (const void *)tc_fwd<true, true> : (const void *)tc_fwd<true, false>)
                          : (qkn ? (const void *)tc_fwd<false, true> : (const void *)tc_fwd<false, false>);
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (err != cudaSuccess) return err;
    // Placement lead.  One scan CTA fills an SM (its shared memory), and the
    // block scheduler hands a grid's first CTAs to the same SMs every launch:
    // on GB300 the first 12 go to four SMs of the second die and to the first
    // TPC of four GPCs, where a scan CTA measured up to 10 % slower than on
    // the SMs filled next (82-86 against 74-77 us on B = 4, H = 16, T = 2048).
    // The scan lasts as long as its slowest CTA, so when the grid leaves room
    // on the GPU it leads with kLeadCtas CTAs that exit at once and the units
    // go to the CTAs after them (A/B of two builds on one GPU: 118.7 against
    // 122.2 us per forward).  Results do not depend on where a unit runs.
    static std::atomic<int> sms_cache[64];  // 0: not looked up yet (calls may come from several threads)
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    int sms = (dev >= 0 && dev < 64) ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
    if (sms <= 0) {
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
    }
    const long long lead = (grid + kLeadCtas <= sms) ? kLeadCtas : 0;
    // a programmatic dependent of the WY kernel: its launch and its CTAs'
    // set-up, h0 loads and first tile copies overlap the end of that kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid + lead));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<CUtensorMap *>(&mK), const_cast<CUtensorMap *>(&mQ), const_cast<CUtensorMap *>(&mV),
                    const_cast<Params *>(&p)};
    if ((err = cudaLaunchKernelExC(&cfg, kern, args)) != cudaSuccess) return err;
    *name = "wy_fwd+tc_fwd";
    return cudaGetLastError();
}

}  // namespace dn
