// Tensor-core (tcgen05 / TMEM / TMA) scan kernel of the chunkwise gated delta
// rule forward for wide key heads: bf16 q/k/v/o, dk = 256, 128 value columns
// per CTA.
//
// Sources: [CGDR] "01 · 数学原理:ChunkGatedDeltaRule 在算什么" §3.1-§3.3;
//          [WY]   "flash-linear-attention 中 DeltaNet 的分块并行化WY 表示推导与 Triton 内核实现" §2.3-§3.4.
//
// The fp32 state of one (sequence, value head, 128-column value tile) is
// 128 x 256 floats: transposed in tensor memory (lane = value column v,
// column = key index d) it takes 256 of the SM's 512 columns, and its bf16
// image (the A operand of VN and O) another 128.  That leaves no room for W,
// so the WY kernel (dn_wy.cu) forms -W = -T' K per chunk and writes it to the
// workspace beside T'' and P.  One persistent CTA per unit walks the
// sequence's chunks in order; every contraction is a tcgen05 MMA with
// M = 128, and VN and O, which share their A operand, run as one:
//
//   U    [V^T T''^T | 0]            -> [acc_v | acc_o] = [U^T | 0]       (a4)
//   VNO  += S^T [-W^T | Q~^T]       -> [v_new^T | inter-chunk output]    (a5, a6)
//   DS   acc_s += v~^T K            -> state update, v~ = e^{G_L-G} v_new (a5)
//   PV   acc_o += v_new^T P^T       -> intra-chunk output                (a6)
//
// with Q~ = diag(scale e^G) Q.  acc_v (64 columns) and acc_o (64) are
// adjacent, so U and VNO are N = 128 MMAs on the same accumulator: U's B
// operand is T'' followed by 64 zero rows, VNO's is -W followed by Q~, which
// is why each buffer of the -W and Q tiles interleaves their 64-column
// quarters (W0 Q0 W1 Q1 ..).  U and VNO are ordered by the tensor pipe (same
// accumulator and shape); every other dependency between MMAs goes through a
// commit and an mbarrier.
//
// Shared memory holds two chunks' interleaved -W / Q tiles (2 x 64 KB) and
// one chunk's K (32 KB), V (16 KB), T'' and P (8 KB each): every buffer has
// its own full / empty mbarriers, and its loader refills it as soon as its
// last reader (an MMA, through a commit) releases it.
//
// Warp roles (15 warps):
//   0      loader: gate scalars (two-deep ring, gates fetched a chunk ahead),
//          TMA for K and V, bulk copies of T'' and P;
//   1      MMA issuer (one thread: U, VNO, DS, PV) and TMEM owner;
//   2-5    prep: Q rows scaled by scale e^G in place (a chunk ahead); key
//          blocks 0-3 of each state pass;
//   6-9    state: v_new / v~ operands from acc_v; key blocks 4-7;
//   10-13  output: o from acc_o (released at once, since the next U writes
//          it), transposed through shared memory and stored as 16-byte bf16
//          rows;
//   14     loader of the -W / Q tiles (one thread), up to two chunks ahead.
// A state pass turns acc_s into the next chunk's bf16 image (or ht after the
// last chunk).  acc_s holds the state divided by a running product of the
// chunk decays, so the decay of each chunk needs no pass over it (see
// chunk_decay in dn_chunk.cuh).
//
// Every wait is bounded (dn_tc_sync.cuh): a wait that runs out records
// kStatusTimeout, raises the CTA's abort flag, and every role drains its own
// outstanding copies and MMAs before tensor memory is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "dn_chunk.cuh"
#include "dn_internal.h"
#include "dn_tc.h"
#include "dn_tc_sync.cuh"
#include "dn_tmap.h"
#include "tc_ptx.cuh"

namespace dn {
namespace {

using namespace ptx;
using namespace tcs;

constexpr int C = kChunk;  // 64-row tiles
constexpr int DK = 256;
constexpr int BVT = 128;  // value columns per CTA
constexpr int NTHREADS = 480;
constexpr uint32_t SLOT = slot_bytes(DK);

// ---- shared memory map (offsets from a 1024-byte aligned base) -------------
constexpr uint32_t QW_BYTES = 65536;               // one buffer: W0 Q0 W1 Q1 W2 Q2 W3 Q3, 8 KB each
constexpr uint32_t OFF_QW = 0;                     // 2 buffers
constexpr uint32_t OFF_K = OFF_QW + 2 * QW_BYTES;  // K: 4 quarters of 64 columns, 8 KB each
constexpr uint32_t OFF_V = OFF_K + 32768;          // V: 2 halves of 64 value columns
constexpr uint32_t OFF_TU = OFF_V + 16384;         // T''
constexpr uint32_t OFF_ZERO = OFF_TU + 8192;       // 64 zero rows: U's B operand continues here
constexpr uint32_t OFF_PR = OFF_ZERO + 8192;       // P
constexpr uint32_t OFF_SCAL = OFF_PR + 8192;       // 2 x SCAL_FLOATS floats
constexpr uint32_t OFF_OST = OFF_SCAL + 2 * SCAL_FLOATS * 4;  // output staging, 32 x 256 B
constexpr uint32_t OFF_BAR = OFF_OST + 8192;
constexpr int NBARS = 40;
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;  // TMEM base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // alignment slack

static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_TU % 1024 == 0 && OFF_ZERO == OFF_TU + 8192 &&
                  OFF_PR % 1024 == 0,
              "swizzled operands need 1024-byte alignment");
static_assert(SMEM_ALLOC <= 232448, "exceeds the 227 KB of shared memory per CTA");
static_assert(SLOT % 16 == 0 && slot_tu_off(DK) == 32768, "slot = -W | T'' | P | norms");

// Barrier indices.  Buffer barriers: FULL = copy landed (tx bytes + the
// loader's arrive), EMPTY = last reader done (an MMA commit).  Two-deep
// buffers have one of each per buffer (chunk c uses buffer c & 1).
enum {
    B_KF = 0, B_KE,
    B_WF, B_QF = B_WF + 2, B_QWE = B_QF + 2,  // 2 each
    B_VF = B_QWE + 2, B_VE,
    B_TUF, B_TUE,
    B_PF, B_PE,
    B_SCF, B_SCE = B_SCF + 2,   // 2 each: scalars landed (loader) / read (8 warps)
    B_QS = B_SCE + 2,           // 2: Q of the buffer's chunk scaled (prep)
    B_S_FULL = B_QS + 2,        // bf16 S^T image of the chunk written (8 warps)
    B_VN,                       // VNO(c) done (commit)
    B_VSM,                      // v_new / v~ operands (state) + the state pass before the chunk (12 warps)
    B_S_UPD,                    // DS(c), and every MMA before it, done (commit)
    B_D_FULL,                   // PV(c) done: acc_o complete, acc_v free (commit)
    B_O_EMPTY,                  // acc_o read (output)
    B_DRAIN,
    B_COUNT
};
static_assert(B_COUNT <= NBARS, "barrier space");

// Tensor memory columns: acc_v and acc_o adjacent, one N = 128 accumulator
// for U and VNO.
constexpr uint32_t TM_S = 0, TM_SB = 256, TM_V = 384, TM_O = 448, TM_COLS = 512;
static_assert(TM_O == TM_V + 64, "acc_o follows acc_v");

// Instruction descriptors.
constexpr uint32_t ID_U = idesc_bf16(128, 128, 1, 0);    // A MN-major (V^T), B K-major ([T''; 0] rows)
constexpr uint32_t ID_VNO = idesc_bf16(128, 128, 0, 0);  // A TMEM, B K-major ([-W; Q~] rows)
constexpr uint32_t ID_DS = idesc_bf16(128, 256, 0, 1);   // A TMEM, B MN-major (K rows)
constexpr uint32_t ID_PV = idesc_bf16(128, 64, 0, 0);    // A TMEM, B K-major (P rows)

// Key blocks (32 columns of acc_s) of each state pass, per warpgroup.
constexpr int kPrepB0 = 0, kStateB0 = 4, kPassNB = 4;



__device__ __forceinline__ uint32_t bar(const Ctx &x, int i) { return x.base + OFF_BAR + 8u * i; }
__device__ __forceinline__ float *scal(const Ctx &x, int c) {
    return reinterpret_cast<float *>(x.gbase + OFF_SCAL + (c & 1) * SCAL_FLOATS * 4);
}

struct Unit {
    long long bos, eos;
    int n, h, hk, v0, nc;
};

// The unit of this CTA: one per (sequence, value head, value-column tile).
__device__ __forceinline__ Unit unit_of(const Params &p) {
    Unit u;
    const int nvt = p.dv / BVT;
    const int idx = (int)blockIdx.x;
    const int vt = idx % nvt;
    u.h = (idx / nvt) % p.Nv;
    u.n = seq_of_rank(p, idx / (nvt * p.Nv), threadIdx.x & 31);  // longest sequences first
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

__device__ __forceinline__ const uint8_t *slot_of(const Params &p, const Unit &u, int c) {
    const long long t0 = u.bos + (long long)c * p.chunk;
    return static_cast<const uint8_t *>(p.ws) + ((size_t)u.h * p.nslots + (size_t)wy_slot(t0, u.n, p.chunk)) * SLOT;
}

// ---------------------------------------------------------------------------
// Loaders.  Warp 0: per chunk the gate scalars (whole warp), then (lane 0)
// the single-buffered copies in the order their buffers free up in the
// previous chunk: V and T'' (after U), K (after DS), P (after PV).  Warp 14
// (one thread): the -W and Q tiles of each chunk into its two-deep buffer,
// as soon as VNO of the chunk two back has released it.  last[] records the
// last chunk loaded into each buffer kind, for the drain at exit.  The kernel
// is launched as a programmatic dependent of the WY kernel, so it may start
// while that kernel's last CTAs finish: copies of the inputs (V, K, Q) go out
// at once, the slots' -W, T'', P and norms only after grid_dep_wait.
// ---------------------------------------------------------------------------
enum { LV, LTU, LK, LP, LQW, LCOUNT };

__device__ bool load_chunk(const Ctx &x, const Unit &u, int c, long long t0, const uint8_t *slot,
                           const CUtensorMap *mK, const CUtensorMap *mV, int (&last)[LCOUNT]) {
    const int tt = (int)t0;
    const uint32_t p1 = (c & 1) ^ 1;  // free-wait parity of a single buffer
    if (!wait(x, bar(x, B_VE), p1)) return false;
    mbar_arrive_expect_tx(bar(x, B_VF), 16384);
    tma_load_3d(x.base + OFF_V, mV, bar(x, B_VF), u.v0, u.h, tt);
    tma_load_3d(x.base + OFF_V + 8192, mV, bar(x, B_VF), u.v0 + 64, u.h, tt);
    last[LV] = c;
    // the WY kernel's slots only once that kernel has completed (the scan
    // is its programmatic dependent)
    if (c == 0) grid_dep_wait();
    if (!wait(x, bar(x, B_TUE), p1)) return false;
    mbar_arrive_expect_tx(bar(x, B_TUF), kImageBytes);
    bulk_load(x.base + OFF_TU, slot + slot_tu_off(DK), kImageBytes, bar(x, B_TUF));
    last[LTU] = c;
    if (!wait(x, bar(x, B_KE), p1)) return false;
    mbar_arrive_expect_tx(bar(x, B_KF), 32768);
#pragma unroll
    for (int q = 0; q < 4; ++q) tma_load_3d(x.base + OFF_K + 8192 * q, mK, bar(x, B_KF), 64 * q, u.hk, tt);
    last[LK] = c;
    if (!wait(x, bar(x, B_PE), p1)) return false;
    mbar_arrive_expect_tx(bar(x, B_PF), kImageBytes);
    bulk_load(x.base + OFF_PR, slot + slot_p_off(DK), kImageBytes, bar(x, B_PF));
    last[LP] = c;
    return true;
}

// The raw gates of chunk c and, with kQkL2Norm, its inverse key / query
// norms from the WY kernel's slot, for the lane's two tokens.
struct ChunkInputs {
    ChunkGates gates;
    float ka, kb, qa, qb;
};

template <bool QKN>
__device__ __forceinline__ ChunkInputs chunk_inputs_load(const Params &p, const Unit &u, int c, int lane) {
    ChunkInputs r;
    const long long t0 = u.bos + (long long)c * p.chunk;
    r.gates = chunk_gates_load(p, u.h, t0, (int)min((long long)p.chunk, u.eos - t0), lane);
    r.ka = r.kb = r.qa = r.qb = 1.f;
    if (QKN) {
        const float *f = reinterpret_cast<const float *>(slot_of(p, u, c) + slot_norm_off(DK));
        r.ka = f[lane];
        r.kb = f[lane + 32];
        r.qa = f[64 + lane];
        r.qb = f[64 + lane + 32];
    }
    return r;
}

template <bool QKN>
__device__ void loader_role(const Ctx x, const Params &p, const Unit u, const CUtensorMap *mK,
                            const CUtensorMap *mV, int (&last)[LCOUNT]) {
    const int lane = threadIdx.x & 31;
    // each chunk's gates (and norms) are loaded one iteration ahead, so that
    // their latency hides under the previous chunk's waits
    ChunkInputs next{};
    if (QKN) grid_dep_wait();  // the norms come from the slots
    if (u.nc > 0) next = chunk_inputs_load<QKN>(p, u, 0, lane);
    float A = 1.f;  // A_c, the same in every lane
    for (int c = 0; c < u.nc; ++c) {
        const long long t0 = u.bos + (long long)c * p.chunk;
        const int L = (int)min((long long)p.chunk, u.eos - t0);
        const ChunkInputs in = next;
        if (c + 1 < u.nc) next = chunk_inputs_load<QKN>(p, u, c + 1, lane);
        ChunkScalars cs = chunk_scalars_from(in.gates, L, lane);
        const ChunkDecay dec = chunk_decay(cs.GL, A);
        const float inv_an = 1.f / dec.an;
        cs.ka = in.ka * inv_an;  // rides on e^{G_L - G_i}: v~ / A_{c+1}
        cs.kb = in.kb * inv_an;
        cs.qa = in.qa;
        cs.qb = in.qb;
        if (!wwait(x, bar(x, B_SCE + (c & 1)), ((c >> 1) & 1) ^ 1)) return;
        float *sc = scal(x, c);
        chunk_scalars_store(p, cs, sc, lane);
        if (lane == 0) chunk_decay_store(sc, dec);
        A = dec.an;
        __syncwarp();
        bool ok = true;
        if (lane == 0) {
#ifdef DN_TEST_STALL
            // failure-path test: the first chunk's scalars are never
            // announced, so every wait on them runs out (the copies land)
            if (!(p.test_stall == kStallScan && c == 0))
#endif
                mbar_arrive(bar(x, B_SCF + (c & 1)));
            ok = load_chunk(x, u, c, t0, slot_of(p, u, c), mK, mV, last);
        }
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) return;
    }
}

// One thread: -W (four 8 KB quarters, bulk copies from the slot) and Q (TMA)
// of chunk c into the odd and even 8 KB slots of buffer c & 1.
__device__ void qw_loader_role(const Ctx x, const Params &p, const Unit u, const CUtensorMap *mQ,
                               int (&last)[LCOUNT]) {
    for (int c = 0; c < u.nc; ++c) {
        const int b = c & 1;
        if (!wait(x, bar(x, B_QWE + b), ((c >> 1) & 1) ^ 1)) return;
        const uint32_t buf = x.base + OFF_QW + QW_BYTES * b;
        const uint8_t *slot = slot_of(p, u, c);
        mbar_arrive_expect_tx(bar(x, B_QF + b), 32768);
        const int tt = (int)(u.bos + (long long)c * p.chunk);
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_load_3d(buf + 16384 * q + 8192, mQ, bar(x, B_QF + b), 64 * q, u.hk, tt);
        if (c == 0) grid_dep_wait();  // -W comes from the WY kernel's slots
        mbar_arrive_expect_tx(bar(x, B_WF + b), 32768);
#pragma unroll
        for (int q = 0; q < 4; ++q) bulk_load(buf + 16384 * q, slot + 8192 * q, 8192, bar(x, B_WF + b));
        last[LQW] = c;
    }
}

// Waits (ignoring the abort flag) for the last copies into each buffer to
// land, so none writes shared memory after the CTA has left (lane 0 of the
// loader warps).
__device__ void loader_drain(const Ctx &x, const int (&last)[LCOUNT], bool qw) {
    if (!qw) {
        const int single[4][2] = {{LV, B_VF}, {LTU, B_TUF}, {LK, B_KF}, {LP, B_PF}};
        for (int i = 0; i < 4; ++i)
            if (last[single[i][0]] >= 0) wait_drain(bar(x, single[i][1]), last[single[i][0]] & 1);
        return;
    }
    for (int k = last[LQW] - 1; k <= last[LQW]; ++k)
        if (k >= 0) {
            wait_drain(bar(x, B_WF + (k & 1)), (k >> 1) & 1);
            wait_drain(bar(x, B_QF + (k & 1)), (k >> 1) & 1);
        }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread): per chunk U, VNO, DS, PV, in that order.  Each
// buffer is released by a commit after its last reading MMA.
// ---------------------------------------------------------------------------
__device__ void mma_role(const Ctx x, const Unit u, uint32_t tm) {
    for (int c = 0; c < u.nc; ++c) {
        const int b = c & 1;
        const uint32_t par = c & 1, par2 = (c >> 1) & 1;
        // U(c) into [acc_v | acc_o]: acc_v is free once PV(c - 1) is done,
        // acc_o once the output warpgroup has read it
        if (c > 0 && !(wait(x, bar(x, B_D_FULL), par ^ 1) && wait(x, bar(x, B_O_EMPTY), par ^ 1))) break;
        if (!(wait(x, bar(x, B_VF), par) && wait(x, bar(x, B_TUF), par))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ss(tm + TM_V, sdesc(x.base + OFF_V + kk * 2048, 8192, 1024), sdesc(x.base + OFF_TU + kk * 32, 16, 1024),
                   ID_U, kk != 0);
        mma_commit(bar(x, B_VE));
        mma_commit(bar(x, B_TUE));
        // VNO(c): [acc_v | acc_o] += S^T [-W^T | Q~^T]
        if (!(wait(x, bar(x, B_WF + b), par2) && wait(x, bar(x, B_QS + b), par2) &&
              wait(x, bar(x, B_S_FULL), par)))
            break;
        tc_fence_after();
        const uint32_t qw = x.base + OFF_QW + QW_BYTES * b;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_ts(tm + TM_V, tm + TM_SB + kk * 8, sdesc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), ID_VNO, 1);
        mma_commit(bar(x, B_VN));
        mma_commit(bar(x, B_QWE + b));
        // DS(c): acc_s (scaled by alpha(c)) += v~^T K
        if (!(wait(x, bar(x, B_VSM), par) && wait(x, bar(x, B_KF), par))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_S, tm + TM_V + 32 + kk * 8, sdesc(x.base + OFF_K + kk * 2048, 8192, 1024), ID_DS, 1);
        mma_commit(bar(x, B_S_UPD));
        mma_commit(bar(x, B_KE));
        // PV(c): acc_o += v_new^T P^T
        if (!wait(x, bar(x, B_PF), par)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts(tm + TM_O, tm + TM_V + kk * 8, sdesc(x.base + OFF_PR + kk * 32, 16, 1024), ID_PV, 1);
        mma_commit(bar(x, B_D_FULL));
        mma_commit(bar(x, B_PE));
    }
    // every MMA issued completes before tensor memory is freed
    mma_commit(bar(x, B_DRAIN));
    wait_drain(bar(x, B_DRAIN), 0);
}

// ---------------------------------------------------------------------------
// State passes.  The fp32 state acc_s (TMEM lane = value column v, column =
// key index d) is handled in 32-column key blocks, NB consecutive blocks from
// b0 per warpgroup; `lb` is the thread's TMEM lane base, `hb` its element of
// h0 / ht at key index 0 (rows dv apart).
// ---------------------------------------------------------------------------
// acc_s = alpha_0 h0^T and the bf16 image = bf16(h0^T).
template <int NB>
__device__ __forceinline__ void state_init(const Params &p, uint32_t lb, size_t hb, float alpha, int b0) {
#pragma unroll 1
    for (int blk = b0; blk < b0 + NB; ++blk) {
        float f[32];
        const float *hp = p.h0 ? p.h0 + hb + (size_t)(32 * blk) * p.dv : nullptr;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            f[k] = hp ? *hp : 0.f;
            if (hp) hp += p.dv;
        }
        uint32_t pk[16], r[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(f[2 * k], f[2 * k + 1]);
        tmem_st16(lb + TM_SB + 16 * blk, pk);
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(alpha * f[k]);
        tmem_st32(lb + TM_S + 32 * blk, r);
    }
}

// Hand-off after TMEM stores: the stores are complete and ordered before the
// MMAs that the arrival releases.
__device__ __forceinline__ void st_arrive(uint32_t b) {
    tmem_wait_st();
    tc_fence_before();
    warp_arrive(b);
}

// ht = a acc_s for key blocks [b0, b0 + kPassNB) (out of line: run once).
__device__ __noinline__ void state_pass_ht(const Params &p, uint32_t lb, size_t hb, int b0, float a) {
    if (!p.ht) return;
    for (int e = 0; e < kPassNB; ++e) {
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

// After DS(c), key blocks [b0, b0 + kPassNB), two at a time: the bf16
// image of S_{c+1} = A_{c+1} acc_s (then S_FULL, which VNO(c + 1) waits
// for), and for a renormalising chunk c + 1 acc_s *= alpha_{c+1} A_{c+1}
// (before VSM, which DS(c + 1) waits for); after the last chunk, ht =
// A_{c+1} acc_s.  sn: the scalars of chunk c + 1 (those of chunk c after the
// last chunk).
__device__ __forceinline__ void state_pass(const Ctx &x, const Params &p, uint32_t lb, size_t hb, bool last,
                                           int b0, const float *sn) {
    const float a = last ? sn[SC_AN] : sn[SC_A];
    if (last) {
        state_pass_ht(p, lb, hb, b0, a);
        return;
    }
    const bool rn = !last && sn[SC_RN] != 0.f;
    const float rs = sn[SC_RS];
#pragma unroll 1
    for (int e0 = 0; e0 < kPassNB; e0 += 2) {
        uint32_t r[2][32];
        tmem_ld32(lb + TM_S + 32 * (b0 + e0), r[0]);
        tmem_ld32(lb + TM_S + 32 * (b0 + e0 + 1), r[1]);
        tmem_wait_ld_dep(r[0]);
        tmem_ld_dep(r[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int blk = b0 + e0 + e;
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = pack_bf16(a * __uint_as_float(r[e][2 * k]), a * __uint_as_float(r[e][2 * k + 1]));
            tmem_st16(lb + TM_SB + 16 * blk, pk);
            if (rn) {
#pragma unroll
                for (int k = 0; k < 32; ++k) r[e][k] = __float_as_uint(rs * __uint_as_float(r[e][k]));
                tmem_st32(lb + TM_S + 32 * blk, r[e]);
            }
        }
    }
    st_arrive(bar(x, B_S_FULL));
    warp_arrive(bar(x, B_VSM));
}

// ---------------------------------------------------------------------------
// Prep warpgroup: Q rows scaled in place a chunk ahead, key blocks 0-2 of
// the state.
// ---------------------------------------------------------------------------
// Q row i *= scale e^{G_i} (bf16) for chunk c, so that O and PV share one
// accumulator: o_i = S^T (scale e^{G_i} q_i) + sum_j P_ij v_new_j.  Each step
// of a warp covers 512 contiguous bytes (4 rows x 8 chunks of 16 B), free of
// bank conflicts; the swizzle only permutes chunks within a row.  Returns
// false if a wait ran out.
__device__ __forceinline__ bool scale_q(const Ctx &x, int c) {
    const int b = c & 1;
    if (!wwait(x, bar(x, B_QF + b), (c >> 1) & 1) || !wwait(x, bar(x, B_SCF + b), (c >> 1) & 1)) return false;
    const float *sc = scal(x, c);
    const int tid = threadIdx.x - 64;
    uint8_t *qt = x.gbase + OFF_QW + QW_BYTES * b + 8192;  // quarter q at qt + 16384 q
#pragma unroll 4
    for (int it = 0; it < 16; ++it) {
        const int k = tid + 128 * it, quarter = k >> 9, r = (k >> 3) & 63, ch = k & 7;
        const float f = sc[SC_OSC + r];
        uint4 *qp = reinterpret_cast<uint4 *>(qt + 16384 * quarter + 128 * r + 16 * ch);
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
    warp_arrive(bar(x, B_QS + b));
    return true;
}

__device__ void prep_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);
    const uint32_t lb = lane_base(tm, warp);
    const size_t hb = ((size_t)u.n * p.Nv + u.h) * DK * p.dv + u.v0 + v;
    if (u.nc == 0 || !scale_q(x, 0)) return;
    state_init<kPassNB>(p, lb, hb, scal(x, 0)[SC_RN] != 0.f ? scal(x, 0)[SC_RS] : 1.f, kPrepB0);
    st_arrive(bar(x, B_S_FULL));
    warp_arrive(bar(x, B_VSM));
    warp_arrive(bar(x, B_SCE + 0));
    for (int c = 0; c < u.nc; ++c) {
        const bool last = c + 1 == u.nc;
        // Q~ of the next chunk, which VNO(c + 1) reads, while this chunk's
        // VNO and DS run
        if (!last && !scale_q(x, c + 1)) return;
        if (!wwait(x, bar(x, B_S_UPD), c & 1)) return;
        tc_fence_after();
        state_pass(x, p, lb, hb, last, kPrepB0, scal(x, last ? c : c + 1));
        if (last) break;
        warp_arrive(bar(x, B_SCE + ((c + 1) & 1)));
    }
}

// ---------------------------------------------------------------------------
// State warpgroup: v_new / v~ operands of each chunk, key blocks 3-5.
// ---------------------------------------------------------------------------
__device__ void state_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);  // value column = TMEM lane
    const uint32_t lb = lane_base(tm, warp);
    const size_t hb = ((size_t)u.n * p.Nv + u.h) * DK * p.dv + u.v0 + v;
    if (u.nc == 0) {  // empty sequence: ht = h0
        if (p.ht)
            for (int d = 0; d < DK; ++d) p.ht[hb + (size_t)d * p.dv] = p.h0 ? p.h0[hb + (size_t)d * p.dv] : 0.f;
        return;
    }
    if (!wwait(x, bar(x, B_SCF + 0), 0)) return;
    state_init<kPassNB>(p, lb, hb, scal(x, 0)[SC_RN] != 0.f ? scal(x, 0)[SC_RS] : 1.f, kStateB0);
    st_arrive(bar(x, B_S_FULL));
    warp_arrive(bar(x, B_VSM));
    for (int c = 0; c < u.nc; ++c) {
        // ---- v_new^T and v~^T operands --------------------------------
        // acc_v columns j = 0..63 (fp32) become v_new^T packed in columns
        // 0..31 and v~^T packed in columns 32..63; a column is rewritten only
        // after it has been read.
        if (!wwait(x, bar(x, B_VN), c & 1)) return;
        tc_fence_after();
        {
            const float4 *dec4 = reinterpret_cast<const float4 *>(scal(x, c) + SC_DEC);
            const uint32_t lbv = lb + TM_V;
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
            st_arrive(bar(x, B_VSM));
        }
        warp_arrive(bar(x, B_SCE + (c & 1)));  // done with this chunk's scalars
        // ---- state: the next chunk's bf16 image (key blocks 4-7) ---------
        const bool last = c + 1 == u.nc;
        if (!last && !wwait(x, bar(x, B_SCF + ((c + 1) & 1)), ((c + 1) >> 1) & 1)) return;
        if (!wwait(x, bar(x, B_S_UPD), c & 1)) return;
        tc_fence_after();
        state_pass(x, p, lb, hb, last, kStateB0, scal(x, last ? c : c + 1));
        if (last) break;
    }
}

// ---------------------------------------------------------------------------
// Output warpgroup: o[i][v] = (S^T Q~^T + v_new^T P^T)[v][i] for value column
// v = this thread's TMEM lane, chunk by chunk once PV is done.  acc_o is read
// and released first (it is the next chunk's U accumulator too), then
// transposed through shared memory and stored.  Every exit is taken by the
// whole warpgroup together (bar_red_or), so no warp is left waiting at one of
// its named barriers.
// ---------------------------------------------------------------------------
__device__ void output_role(const Ctx x, const Params &p, const Unit u, uint32_t tm) {
    const int warp = threadIdx.x >> 5;
    const int v = 32 * (warp & 3) + (threadIdx.x & 31);
    const int tid = threadIdx.x - 320;  // 0..127 in the output warpgroup
    const uint32_t lb = lane_base(tm, warp);
    const uint32_t buf = x.base + OFF_OST;
    const uint8_t *gbuf = x.gbase + OFF_OST;
    const long long rstride = (long long)p.Nv * p.dv * 2;  // bytes between tokens
    for (int c = 0; c < u.nc; ++c) {
        if (bar_red_or(2, 128, !wwait(x, bar(x, B_D_FULL), c & 1))) break;
        tc_fence_after();
        // the chunk's output column v as packed bf16 pairs (tokens 2k, 2k + 1)
        uint32_t ob[32];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t ra[32];
            tmem_ld32(lb + TM_O + 32 * hf, ra);
            tmem_wait_ld_dep(ra);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                ob[16 * hf + k] = pack_bf16(__uint_as_float(ra[2 * k]), __uint_as_float(ra[2 * k + 1]));
        }
        tc_fence_before();
        warp_arrive(bar(x, B_O_EMPTY));
        // transpose through shared memory, 32 tokens x 128 value columns
        // (256-byte rows) at a time, then 16-byte stores of whole rows i < L
        // (a rolled loop: the scan measured faster with a smaller
        // instruction footprint)
        const long long t0 = u.bos + (long long)c * p.chunk;
        const int L = (int)min((long long)p.chunk, u.eos - t0);
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
// QKN: in-kernel q / k normalisation (a template parameter, so that the plain
// instance carries none of its code).
template <bool QKN>
__global__ void __launch_bounds__(NTHREADS, 1)
tc_wide_fwd(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
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
        const int ones[] = {B_KF, B_KE, B_WF, B_WF + 1, B_QF, B_QF + 1, B_QWE, B_QWE + 1, B_VF, B_VE,
                            B_TUF, B_TUE, B_PF, B_PE, B_SCF, B_SCF + 1, B_VN, B_S_UPD, B_D_FULL, B_DRAIN};
        for (int b : ones) mbar_init(bar(x, b), 1);
        mbar_init(bar(x, B_SCE), 8);      // prep and state warpgroups
        mbar_init(bar(x, B_SCE + 1), 8);
        mbar_init(bar(x, B_QS), 4);
        mbar_init(bar(x, B_QS + 1), 4);
        mbar_init(bar(x, B_S_FULL), 8);   // prep and state warpgroups, half the state each
        mbar_init(bar(x, B_VSM), 12);     // the same eight (state pass) + state (v_new, v~)
        mbar_init(bar(x, B_O_EMPTY), 4);
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
    // the 64 zero rows of U's B operand
    for (int i = threadIdx.x; i < 8192 / 16; i += NTHREADS)
        *reinterpret_cast<uint4 *>(x.gbase + OFF_ZERO + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *reinterpret_cast<volatile uint32_t *>(x.gbase + OFF_MISC);

    if (warp == 0 || warp == 14) {
        int last[LCOUNT];
        for (int i = 0; i < LCOUNT; ++i) last[i] = -1;
        if (warp == 0)
            loader_role<QKN>(x, p, u, &mK, &mV, last);
        else if ((threadIdx.x & 31) == 0)
            qw_loader_role(x, p, u, &mQ, last);
        if ((threadIdx.x & 31) == 0) loader_drain(x, last, warp == 14);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0 && u.nc > 0) mma_role(x, u, tm);
        __syncwarp();
    } else if (warp < 6) {
        prep_role(x, p, u, tm);
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

cudaError_t tc_wide_launch(const Params &p, cudaStream_t stream, const char **name) {
    CUtensorMap mK, mQ, mV;
    const uint64_t tokens = (uint64_t)p.tokens;
    if (!make_tmap_rows_heads_d(&mK, p.k, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mQ, p.q, tokens, p.Nk, DK, 64, C) ||
        !make_tmap_rows_heads_d(&mV, p.v, tokens, p.Nv, p.dv, 64, C))
        return cudaErrorInvalidValue;
    const long long grid = (long long)p.N * p.Nv * (p.dv / BVT);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    // -W, T'' and P of every chunk first (all chunks in parallel), then the scan
    cudaError_t err = wy_launch(p, mK, mQ, stream);
    if (err != cudaSuccess) return err;
    const void *kern = (p.flags & kQkL2Norm) ? (const void *)tc_wide_fwd<true> : (const void *)tc_wide_fwd<false>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (err != cudaSuccess) return err;
    // a programmatic dependent of the WY kernel (its loaders wait for that
    // kernel before they read the slots)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
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
    *name = "wy_fwd+tc_wide_fwd";
    return cudaGetLastError();
}

}  // namespace dn
