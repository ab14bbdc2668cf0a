// kernel_bwd_tc.cu -- the attention backward on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA-fed shared memory): a dQ kernel and
// a dK/dV kernel (further down).
//
// dQ[q] = scale * sum_k dS[q,k] K[k],  dS = P (dP - Dq),  P = exp2(S c - LSE_2),
// S = Q K^T, dP = dO V^T over each row's legal keys (the derivative of the
// forward definition; Dq = rowsum(dO * O) is computed here for the CTA's rows
// and written for the dK/dV kernel that follows, or read from memory).  The
// structure is the dQ kernel of "Accelerating PyTorch on AMD GPUs with
// FlyDSL", section on FMHA through AOTriton: its three products match the
// forward's (S like the forward's S, dP likewise, dQ += dS K like O += P V),
// and the K tile is staged once and read in both orientations -- K-major as
// the B operand of S, MN-major as the B operand of dQ.
//
// A CTA owns 128 query rows of one head (TMEM lane = row) and walks their
// legal keys 64 at a time:
//   warp 4 (one thread): TMA loads of the Q and dO tiles, of O's tile (into
//     the last ring slot(s), which take K/V tiles once Dq is computed) and a
//     ring of K/V tiles;
//   warps 5 and 7 (one thread each): S_b = Q K^T and dP_b = dO V^T into TMEM
//     buffer b = tile mod 3, once the dQ products of tile - 3 have released
//     S_b;
//   warp 6 (one thread): once the elementwise warps have turned a tile into
//     dS, dQ += dS K with dS read from TMEM (it overwrites S_b);
//   warps 0-3: first Dq of their row from the dO and O tiles; per tile, P
//     and dS from S_b and dP_b in registers, dS stored to TMEM as 16-bit
//     pairs; at the end dQ out of TMEM, scaled, to memory.
// The three buffers let the tensor core compute the S and dP of the next two
// tiles while the elementwise warps work on tile j and its dQ products wait
// for them (two buffers: 1.78 ms for the backward step, three: 1.73 ms).
// TMEM: S0 S1 S2 | dP0 dP1 dP2 | dQ, all 512 columns at D = 128.
// Every mbarrier wait is bounded; a wait that runs out records a status and
// raises an abort flag, and the CTA drains its copies and frees TMEM.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_softmax.cuh"

namespace attn {
namespace {

using namespace sm100;
using tcfwd::f2pack;
using tcfwd::f2unpack;
using tcfwd::ffma2;
using tcfwd::fadd2;
using tcfwd::fmul2;

constexpr int kRowsT = 128;  // query rows per CTA (MMA M)
constexpr int kKeysT = 64;   // keys per tile (N of S and dP, contraction of dQ)
constexpr int kStagesT = 4;  // K/V ring depth
constexpr int kSBufT = 3;    // S / dP buffers in TMEM
constexpr int kThreadsQ = 256;  // dQ: warps 0-3 elementwise, 4 TMA, 5 S, 6 dQ, 7 dP MMAs
constexpr int kLoadWarpT = 4;
constexpr int kMmaWarpT = 5;  // S MMAs; owns the TMEM allocation
constexpr int kDqWarpT = 6;
constexpr int kDpWarpT = 7;
constexpr int kStatusTimeoutBwdTc = 0x301;

struct DqArgs {
    BwdParams bp;
    int nqt;            // 128-row query tiles per (sequence, head)
    float c2;           // scale * log2(e)
    uint32_t idesc_s;   // M128 N64, both operands K-major
    uint32_t idesc_dq;  // M128 N=D, B MN-major
    // 0: Dq of each row from bp.delta; 1: computed here, rowsum(dO * O) with
    // dO from the staged tile; 2: as 1, and written to bp.delta for a dK/dV
    // launch that follows
    int self_delta;
};

template <int D, int DV> struct DqLayout {
    static constexpr int QCH = kRowsT * 128;  // one 64-column chunk of a 128-row tile
    static constexpr int KCH = kKeysT * 128;  // one 64-column chunk of a 64-key tile
    static constexpr int QTILE = (D / 64) * QCH;
    static constexpr int OTILE = (DV / 64) * QCH;
    static constexpr int KTILE = (D / 64) * KCH;
    static constexpr int VTILE = (DV / 64) * KCH;
    static constexpr int STAGE = KTILE + VTILE;
    static constexpr int Q_OFF = 0;
    static constexpr int DO_OFF = QTILE;
    static constexpr int KV_OFF = QTILE + OTILE;
    static constexpr int BAR_OFF = KV_OFF + kStagesT * STAGE;
    static constexpr int SMEM = 1024 + BAR_OFF + 256;
    // O's tile (for Dq = rowsum(dO * O) computed in the kernel) is staged in
    // the last O_STAGES ring slots before their first K / V tile
    static constexpr int O_STAGES = (OTILE + STAGE - 1) / STAGE;
    static constexpr int O_OFF = KV_OFF + (kStagesT - O_STAGES) * STAGE;
    static_assert(O_STAGES < kStagesT, "O tile in the ring");
    // TMEM columns: S_0 .. S_{kSBufT-1} | dP_0 .. | dQ
    static constexpr int S_COL = 0, DP_COL = kSBufT * kKeysT, DQ_COL = 2 * kSBufT * kKeysT;
    static_assert(DQ_COL + D <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// barrier slots (8 bytes each)
enum : int {
    T_QD_FULL = 0,
    T_S_FULL = 1,                   // [kSBufT]
    T_DS_READY = 1 + kSBufT,        // [kSBufT]
    T_DQ_FULL = 1 + 2 * kSBufT,
    T_TEARDOWN = 2 + 2 * kSBufT,    // one commit from each of the three MMA-issuing warps
    T_S_EMPTY = 3 + 2 * kSBufT,     // [kSBufT]: the dQ MMAs that read dS out of S_b have completed
    T_KV_FULL = 3 + 3 * kSBufT,     // [kStagesT] full, then [kStagesT] empty
    T_O_FULL = T_KV_FULL + 2 * kStagesT,  // O's tile has landed
    T_O_FREE = T_O_FULL + 1,        // Dq is computed: O's ring slots may take K / V
    T_NBARS = T_O_FREE + 1,
};

__device__ __forceinline__ float ex2f(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}

template <typename T> __device__ __forceinline__ uint32_t pack16(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack16<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack16<__half>(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// a + the dot product of two 16-bit pairs, in fp32
template <typename T> __device__ __forceinline__ float dot2_acc(uint32_t x, uint32_t y, float a);
template <>
__device__ __forceinline__ float dot2_acc<__nv_bfloat16>(uint32_t x, uint32_t y, float a) {
    a = fmaf(__uint_as_float(x << 16), __uint_as_float(y << 16), a);
    return fmaf(__uint_as_float(x & 0xffff0000u), __uint_as_float(y & 0xffff0000u), a);
}
template <> __device__ __forceinline__ float dot2_acc<__half>(uint32_t x, uint32_t y, float a) {
    const float2 fx = __half22float2(*reinterpret_cast<const __half2 *>(&x));
    const float2 fy = __half22float2(*reinterpret_cast<const __half2 *>(&y));
    return fmaf(fx.y, fy.y, fmaf(fx.x, fy.x, a));
}

__device__ __forceinline__ bool warp_wait_t(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort_flag, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void raise_abort_t(volatile int *abort_flag, int *status) {
    *abort_flag = 1;
    report_status(status, kStatusTimeoutBwdTc);
}

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreadsQ, 1)
    bwd_dq_tc_kernel(const __grid_constant__ DqArgs a, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmOut) {
    using L = DqLayout<D, DV>;
    extern __shared__ uint8_t smem_t[];
    // a dK/dV launch that depends on this one (programmatic) may be scheduled
    // once every CTA has started: it sets up on the SMs the last ones free and
    // waits for this grid's Dq before reading it
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const BwdParams &bp = a.bp;
    const AttnParams &p = bp.f;
    const uint64_t wl = p.wait_ns;  // limit of every wait but the drains

    // work: (query tile rank, sequence, head); the last query tiles see the
    // most keys and start first
    const int nbh = p.B * p.Hq;
    const int rank = blockIdx.x / nbh;
    const int b = (blockIdx.x % nbh) / p.Hq, h = (blockIdx.x % nbh) % p.Hq;
    const int kvh = h / p.G;
    const SeqInfo si = seq_info(p, b);
    const bool padded = p.cu_q == nullptr;
    const int q0 = (a.nqt - 1 - rank) * kRowsT;
    const int qcap = padded ? p.Q : si.Qb;  // rows this CTA may write
    if (q0 >= qcap) return;                 // uniform: before any barrier

    const uint32_t raw = smem_addr(smem_t);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_t + (base - raw);
    const uint32_t bars = base + L::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::BAR_OFF + 8 * T_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto kv_full = [&](int s) { return bar(T_KV_FULL + s); };
    auto kv_empty = [&](int s) { return bar(T_KV_FULL + kStagesT + s); };
    auto stage = [&](int s) { return base + L::KV_OFF + (uint32_t)s * L::STAGE; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // legal keys of the CTA's rows: the union of the rows' ranges, which grow
    // with the row
    const int qlast = min(q0 + kRowsT, si.Qb) - 1;
    int klo = 0, khi = 0;
    if (qlast >= q0) {
        int a0, a1;
        legal_range(q0, si.Qb, si.Kb, p.window, p.mask, klo, a0);
        legal_range(qlast, si.Qb, si.Kb, p.window, p.mask, a1, khi);
    }
    const int tfirst = klo / kKeysT * kKeysT;
    const int ntiles = khi > klo ? (khi - tfirst + kKeysT - 1) / kKeysT : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(T_QD_FULL), 1);
        for (int i = 0; i < kSBufT; ++i) {
            mbar_init(bar(T_S_FULL + i), 2);  // S and dP commits
            mbar_init(bar(T_DS_READY + i), 128);
            mbar_init(bar(T_S_EMPTY + i), 1);
        }
        mbar_init(bar(T_DQ_FULL), 1);
        mbar_init(bar(T_TEARDOWN), 3);
        mbar_init(bar(T_O_FULL), 1);
        mbar_init(bar(T_O_FREE), 128);
        for (int s = 0; s < kStagesT; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarpT) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kLoadWarpT && lane == 0 && ntiles > 0) {
        // the tensor maps' descriptors on their way while the CTA sets up
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if (a.self_delta) tma_prefetch_desc(&tmOut);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kLoadWarpT) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0 && ntiles > 0) {
            const int qrow = (padded ? 0 : (int)si.q_off) + q0;
            const int krow = padded ? 0 : (int)si.k_off;
            const int bc = padded ? b : 0;
            bool ok = true;
            uint32_t armed = 0, armed_ph = 0;
            mbar_arrive_expect_tx(bar(T_QD_FULL), L::QTILE + L::OTILE);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(base + L::Q_OFF + c * L::QCH, &tmQ, bar(T_QD_FULL), c * 64, h, qrow, bc);
            for (int c = 0; c < DV / 64; ++c)
                tma_load_4d(base + L::DO_OFF + c * L::QCH, &tmO, bar(T_QD_FULL), c * 64, h, qrow, bc);
            if (a.self_delta) {
                mbar_arrive_expect_tx(bar(T_O_FULL), L::OTILE);
                for (int c = 0; c < DV / 64; ++c)
                    tma_load_4d(base + L::O_OFF + c * L::QCH, &tmOut, bar(T_O_FULL), c * 64, h, qrow,
                                bc);
            }
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % kStagesT;
                const uint32_t ph = (uint32_t)(j / kStagesT) & 1u;
                // the first K / V tile of a slot O's tile occupies waits for Dq
                if (a.self_delta && j == kStagesT - L::O_STAGES &&
                    !mbar_wait(bar(T_O_FREE), 0, abort_flag, wl)) {
                    raise_abort_t(abort_flag, p.status);
                    ok = false;
                    break;
                }
                if (!mbar_wait(kv_empty(s), ph ^ 1u, abort_flag, wl)) {
                    raise_abort_t(abort_flag, p.status);
                    ok = false;
                    break;
                }
                const int kr = krow + tfirst + j * kKeysT;
                mbar_arrive_expect_tx(kv_full(s), L::STAGE);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(stage(s) + c * L::KCH, &tmK, kv_full(s), c * 64, kvh, kr, bc);
                for (int c = 0; c < DV / 64; ++c)
                    tma_load_4d(stage(s) + L::KTILE + c * L::KCH, &tmV, kv_full(s), c * 64, kvh,
                                kr, bc);
                armed |= 1u << s;
                armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
            }
            (void)ok;
            // drain: every copy issued has landed before the CTA exits (these
            // waits ignore the abort flag: the copies always land)
            mbar_wait_drain(bar(T_QD_FULL), 0);
            if (a.self_delta) mbar_wait_drain(bar(T_O_FULL), 0);
            for (int s = 0; s < kStagesT; ++s)
                if (armed & (1u << s)) mbar_wait_drain(kv_full(s), (armed_ph >> s) & 1u);
        }
    } else if (warp == kMmaWarpT || warp == kDpWarpT) {
        // ------------------------------------------- S and dP MMA issuers
        // Three issuing warps, one thread each (S, dP, dQ): one thread issuing
        // the sixteen N = 64 products of S and dP took ~1550 cycles a tile at
        // ~100 cycles an issue, three times their tensor time, and a second
        // thread had already taken the dQ products off it; a warp-wide wait per
        // tile costs more than the wait of one thread.
        if (lane == 0) {
            const bool is_s = warp == kMmaWarpT;
            bool ok = ntiles == 0 || mbar_wait(bar(T_QD_FULL), 0, abort_flag, wl);
            const uint64_t ad = sw128_desc(base + (is_s ? L::Q_OFF : L::DO_OFF), 16, 1024);
            for (int j = 0; j < ntiles && ok; ++j) {
                const int s = j % kStagesT, bf = j % kSBufT;
                if (!mbar_wait(kv_full(s), (uint32_t)(j / kStagesT) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                // S_bf and dP_bf were last read for tile j - kSBufT: dP by the
                // elementwise warps, S (as dS) by its dQ MMAs, which have completed
                if (j >= kSBufT && !mbar_wait(bar(T_S_EMPTY + bf),
                                              (uint32_t)(j / kSBufT - 1) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (is_s) {
                    const uint64_t kd = sw128_desc(stage(s), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + L::S_COL + bf * kKeysT,
                               ad + (((kk / 4) * L::QCH + (kk % 4) * 32) >> 4),
                               kd + (((kk / 4) * L::KCH + (kk % 4) * 32) >> 4), a.idesc_s, kk > 0);
                } else {
                    const uint64_t vd = sw128_desc(stage(s) + L::KTILE, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < DV / 16; ++kk)
                        mma_ss(tmem + L::DP_COL + bf * kKeysT,
                               ad + (((kk / 4) * L::QCH + (kk % 4) * 32) >> 4),
                               vd + (((kk / 4) * L::KCH + (kk % 4) * 32) >> 4), a.idesc_s, kk > 0);
                }
                mma_commit(bar(T_S_FULL + bf));
            }
            if (!ok) raise_abort_t(abort_flag, p.status);
            // every MMA issued completes before TMEM is released
            mma_commit(bar(T_TEARDOWN));
            mbar_wait_drain(bar(T_TEARDOWN), 0);  // ignores the abort flag
        }
        __syncwarp();
    } else if (warp == kDqWarpT) {
        // ----------------------------------------------------- dQ MMA issuer
        if (lane == 0) {
            bool ok = true;
            const uint32_t dq_tm = tmem + L::DQ_COL;
            for (int jj = 0; jj < ntiles && ok; ++jj) {
                const int bf = jj % kSBufT, s = jj % kStagesT;
                if (!mbar_wait(bar(T_DS_READY + bf), (uint32_t)(jj / kSBufT) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Keys past the last one in use (last tile only) are left out 16
                // at a time; the K rows of the last 16-key step past it may hold
                // anything (NaN included), so they are zeroed: 0 * K must stay 0.
                // S of this tile has completed (the elementwise warps read it).
                const int nvalid = min(kKeysT, khi - (tfirst + jj * kKeysT));
                const int ksteps = (nvalid + 15) / 16;
                const int nzero = ksteps * 16 - nvalid;
                if (nzero > 0) {
                    uint8_t *kt = gbase + (stage(s) - base) + nvalid * 128;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        for (int i = 0; i < nzero * 8; ++i)
                            *reinterpret_cast<uint4 *>(kt + c * L::KCH + i * 16) =
                                make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
                // K as the MN-major B operand: 64-column chunks L::KCH apart
                const uint64_t kmn = sw128_desc(stage(s), L::KCH, 1024);
#pragma unroll
                for (int kk = 0; kk < kKeysT / 16; ++kk)
                    if (kk < ksteps)
                        mma_ts(dq_tm, tmem + L::S_COL + bf * kKeysT + kk * 8,
                               kmn + ((kk * 2048) >> 4), a.idesc_dq, (jj > 0 || kk > 0) ? 1u : 0u);
                mma_commit(kv_empty(s));
                mma_commit(bar(T_S_EMPTY + bf));
                if (jj == ntiles - 1) mma_commit(bar(T_DQ_FULL));
            }
            if (!ok) raise_abort_t(abort_flag, p.status);
            // every MMA issued completes before TMEM is released
            mma_commit(bar(T_TEARDOWN));
            mbar_wait_drain(bar(T_TEARDOWN), 0);  // ignores the abort flag
        }
        __syncwarp();
    } else {
        // ------------------------------------------- elementwise warps, epilogue
        const int r = warp * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int qpos = q0 + r;
        const bool valid = qpos < si.Qb;
        int lo = 0, hi = 0;
        if (valid) legal_range(qpos, si.Qb, si.Kb, p.window, p.mask, lo, hi);
        const long long row = (si.q_off + qpos) * p.Hq + h;
        float lse2 = 0.f, dl = 0.f;
        if (hi > lo) lse2 = p.lse[row] * kLog2e;
        bool ok = true;
        if (a.self_delta) {
            // Dq = rowsum(dO * O) of this row from the staged dO and O tiles (from
            // memory when the CTA has no key tile and so stages nothing); rows
            // past the sequence's queries: none
            float acc = 0.f;
            auto dot = [&](const uint4 &x, const uint4 &y) {
                acc = dot2_acc<T>(x.x, y.x, acc);
                acc = dot2_acc<T>(x.y, y.y, acc);
                acc = dot2_acc<T>(x.z, y.z, acc);
                acc = dot2_acc<T>(x.w, y.w, acc);
            };
            if (ntiles > 0) {
                ok = warp_wait_t(bar(T_QD_FULL), 0, abort_flag, wl) &&
                     warp_wait_t(bar(T_O_FULL), 0, abort_flag, wl);
                if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
                if (valid && ok) {
#pragma unroll
                    for (int i = 0; i < DV / 8; ++i) {
                        // 128-byte swizzled rows, 64 columns a chunk
                        const int off = (i / 8) * L::QCH + r * 128 + (((i % 8) ^ (r & 7)) << 4);
                        dot(*reinterpret_cast<const uint4 *>(gbase + L::O_OFF + off),
                            *reinterpret_cast<const uint4 *>(gbase + L::DO_OFF + off));
                    }
                }
                mbar_arrive(bar(T_O_FREE));
            } else if (valid) {
                const T *orow = static_cast<const T *>(p.o) + row * (long long)p.Dv;
                const T *grow = static_cast<const T *>(bp.dout) + row * (long long)p.Dv;
                for (int i = 0; i * 8 < p.Dv; ++i)
                    dot(*reinterpret_cast<const uint4 *>(orow + i * 8),
                        *reinterpret_cast<const uint4 *>(grow + i * 8));
            }
            if (a.self_delta == 2 && valid && ok) bp.delta[row] = acc;
            dl = acc;
        } else if (hi > lo) {
            dl = bp.delta[row];
        }
        for (int j = 0; j < ntiles && ok; ++j) {
            const int bf = j % kSBufT;
            if (!warp_wait_t(bar(T_S_FULL + bf), (uint32_t)(j / kSBufT) & 1u, abort_flag, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + L::S_COL + bf * kKeysT;
            const uint32_t tP = tmem + lane_off + L::DP_COL + bf * kKeysT;
            uint32_t sv[2][32], pv[2][32];
            tmem_ld32(tS, sv[0]);
            tmem_ld32(tS + 32, sv[1]);
            tmem_ld32(tP, pv[0]);
            tmem_ld32(tP + 32, pv[1]);
            tmem_ld_wait();
            const int k0 = tfirst + j * kKeysT;
            // bit i of keep[hf]: key k0 + 32 hf + i lies in the row's [lo, hi).
            // Tested against a compile-time bit below: a per-key comparison
            // there compiled to branches and cost ~3x the rest of the step.
            uint32_t keep[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int a0 = min(max(lo - k0 - hf * 32, 0), 32);
                const int b0 = min(max(hi - k0 - hf * 32, 0), 32);
                const uint32_t below_b = b0 >= 32 ? 0xffffffffu : (1u << b0) - 1u;
                const uint32_t below_a = a0 >= 32 ? 0xffffffffu : (1u << a0) - 1u;
                keep[hf] = below_b & ~below_a;
            }
            // pairs of keys share packed f32x2 arithmetic; warps whose rows all
            // see the whole tile skip the test
            const bool all_in = __all_sync(0xffffffffu, (keep[0] & keep[1]) == 0xffffffffu);
            const uint64_t c2 = f2pack(a.c2, a.c2), nl2 = f2pack(-lse2, -lse2),
                           nd2 = f2pack(-dl, -dl);
            uint32_t pk[32];
            auto body = [&](auto masked) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const uint64_t x2 = ffma2(
                            f2pack(__uint_as_float(sv[hf][i]), __uint_as_float(sv[hf][i + 1])), c2, nl2);
                        float x0, x1;
                        f2unpack(x2, x0, x1);
                        const uint64_t y2 = fmul2(
                            fadd2(f2pack(__uint_as_float(pv[hf][i]), __uint_as_float(pv[hf][i + 1])), nd2),
                            f2pack(ex2f(x0), ex2f(x1)));
                        float d0, d1;
                        f2unpack(y2, d0, d1);
                        if (decltype(masked)::value) {
                            d0 = ((keep[hf] >> i) & 1u) ? d0 : 0.f;
                            d1 = ((keep[hf] >> (i + 1)) & 1u) ? d1 : 0.f;
                        }
                        pk[hf * 16 + i / 2] = pack16<T>(d0, d1);
                    }
            };
            if (all_in)
                body(std::false_type{});
            else
                body(std::true_type{});
            tmem_st32(tS, pk);  // dS over the first half of S_bf
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(T_DS_READY + bf));
        }
        if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
        // epilogue: dQ * scale to memory (zeros where no key contributed)
        const bool writes = qpos < qcap;
        if (ok && ntiles > 0) {
            ok = warp_wait_t(bar(T_DQ_FULL), 0, abort_flag, wl);
            if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
            tc_fence_after();
        }
        T *dqg = static_cast<T *>(bp.dq);
        const int Dr = p.D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            if (ok && ntiles > 0) {
                tmem_ld32(tmem + lane_off + L::DQ_COL + c * 32, v);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
            if (writes) {
                // 16-byte stores (D is a multiple of 16, so rows are 32-byte aligned)
                T *dst = dqg + row * Dr + c * 32;
                auto f = [&](int i) { return valid ? __uint_as_float(v[i]) * p.scale : 0.f; };
#pragma unroll
                for (int i = 0; i < 32; i += 8)
                    if (c * 32 + i < Dr)
                        *reinterpret_cast<uint4 *>(dst + i) =
                            make_uint4(pack16<T>(f(i), f(i + 1)), pack16<T>(f(i + 2), f(i + 3)),
                                       pack16<T>(f(i + 4), f(i + 5)), pack16<T>(f(i + 6), f(i + 7)));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpT) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// dK / dV.  A CTA owns 128 keys of one (sequence, KV head) -- TMEM lane = key
// -- with K and V resident in shared memory, and streams the rows that attend
// to them: 128 rows a tile of the flattened (query position, head-in-group)
// space, all heads of the group, one TMA box {64 columns, G heads, 128 / G
// positions} per 64 columns (the forward loop transposed, keys resident and
// rows streamed, as the FlyDSL page describes its dK/dV kernel).  Per tile:
//   S^T = K Q^T and dP^T = V dO^T into TMEM (M = 128 keys, N = 128 rows);
//   two elementwise warpgroups, one per 64-row half, turn S^T into P^T as
//   soon as S^T is in (while dP^T is still computed), then dP^T into dS^T,
//   16-bit pairs over the first halves of their columns;
//   dV += P^T dO for a half as soon as its P^T is in, dK += dS^T Q once its
//   dS^T is, with dO and Q read MN-major from the same row tile.
// At N = 128 every product takes 64 tensor cycles an MMA; 64-row tiles made
// S^T and dP^T N = 64 products, bound by shared-memory operand reads and by
// issue.  Two threads issue the products (S^T and dP^T in warp 9, dV and dK
// in warp 10).  S^T and dP^T are single-buffered: the next tile's S^T waits
// for this tile's dV products to complete (they read P^T over S^T), its dP^T
// for the dK products (dS^T over dP^T).
// TMEM: S^T | dP^T | dV | dK.  Per-row LSE, Dq and legal key range ride with
// each row tile (written by the loader warp, published by the tile's full
// barrier).
constexpr int kKeysK = 128;     // keys per CTA (MMA M)
constexpr int kRowsK = 128;     // rows per tile (N of S^T and dP^T, contraction of dV and dK)
constexpr int kHalfK = 64;      // rows per elementwise warpgroup
constexpr int kStagesK = 2;     // row-tile ring
// warps 0-7 elementwise (two warpgroups), 8 TMA, 9 S^T / dP^T MMAs, 10 dV / dK
// MMAs, 11 idle
constexpr int kThreadsK = 384;
constexpr int kLoadWarpK = 8;
constexpr int kMmaWarpK = 9;
constexpr int kAccWarpK = 10;
// Three warps share each SM sub-partition, so a thread may hold 168 registers
// at launch; the elementwise warps keep 64 fp32 P values across the wait for
// dP^T and take more from the loader, MMA and idle warps (whole warpgroups).
constexpr uint32_t kRegsLaunchK = 168;
constexpr uint32_t kRegsElemK = 208;
constexpr uint32_t kRegsOtherK = 80;
static_assert(256 * kRegsElemK + 128 * kRegsOtherK <= kThreadsK * kRegsLaunchK, "register split");
static_assert(2 * kRegsElemK + kRegsOtherK <= 512, "register split per sub-partition");

template <int D, int DV> struct KvLayout {
    static constexpr int KCH = kKeysK * 128;  // a 64-column chunk of the 128-key tile
    static constexpr int RCH = kRowsK * 128;  // a 64-column chunk of a 128-row tile
    static constexpr int KTILE = (D / 64) * KCH;
    static constexpr int VTILE = (DV / 64) * KCH;
    static constexpr int QTILE = (D / 64) * RCH;
    static constexpr int OTILE = (DV / 64) * RCH;
    static constexpr int STAGE = QTILE + OTILE;
    static constexpr int STATS = kRowsK * 16;  // per row: LSE (log2 units), Dq, lo, hi
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = KTILE;
    static constexpr int R_OFF = KTILE + VTILE;
    static constexpr int ST_OFF = R_OFF + kStagesK * STAGE;
    static constexpr int FLAG_OFF = ST_OFF + kStagesK * STATS;  // [kStagesK] ints: interior tile
    static constexpr int BAR_OFF = FLAG_OFF + 64;
    static constexpr int SMEM = 1024 + BAR_OFF + 256;
    static constexpr int ST_COL = 0, DPT_COL = 128, DV_COL = 256, DK_COL = 256 + DV;
    static_assert(DK_COL + D <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

enum : int {
    K_KV_FULL = 0,
    K_S_FULL = 1,     // S^T of the tile has completed
    K_DP_FULL = 2,    // dP^T of the tile has completed
    K_P_READY = 3,    // [2] by half: its P^T is in TMEM
    K_DS_READY = 5,   // [2] by half: its dS^T is in TMEM
    K_ACC_FULL = 7,
    K_TEARDOWN = 8,
    K_ROW_FULL = 9,   // [kStagesK] full, then [kStagesK] empty
    K_DV_DONE = 9 + 2 * kStagesK,  // the tile's dV products have completed (P^T read)
    K_DK_DONE = 10 + 2 * kStagesK, // the tile's dK products have completed (dS^T read)
    K_ROWS_READY = 11 + 2 * kStagesK,  // a tile's rows past the queries are zeroed
    K_NBARS = 12 + 2 * kStagesK,
};

struct KvArgs {
    BwdParams bp;
    int nkt;           // 128-key tiles per (sequence, KV head)
    int gsz;           // (sequence, KV head) pairs per group of the launch order
    float c2;          // scale * log2(e)
    uint32_t idesc_s;  // M128 N128, both K-major
    uint32_t idesc_v;  // M128 N=DV, B MN-major
    uint32_t idesc_k;  // M128 N=D, B MN-major
};

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreadsK, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ KvArgs a, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
    using L = KvLayout<D, DV>;
    extern __shared__ uint8_t smem_k[];
    const BwdParams &bp = a.bp;
    const AttnParams &p = bp.f;
    const uint64_t wl = p.wait_ns;  // limit of every wait but the drains
    const int G = p.G;
    const int PP = kRowsK / G;  // query positions per row tile

    // Launch order: groups of gsz (sequence, KV head) pairs, and within a group
    // key tile rank first (the first keys are seen by the most rows, so the
    // longest CTAs start first).  A group's Q / dO rows come to about L2's
    // size; ordered by rank alone, the rows of every pair stream at once
    // (4096^2 backward: 1.90 -> 1.84 ms with two groups; six smaller groups
    // were slower, their long first-rank CTAs starting late).
    const int nbh = p.B * p.Hkv;
    const int ngrp = (nbh + a.gsz - 1) / a.gsz;
    const int grp = min((int)(blockIdx.x / ((unsigned)a.nkt * a.gsz)), ngrp - 1);
    const int gsize = grp == ngrp - 1 ? nbh - grp * a.gsz : a.gsz;
    const int rem = (int)blockIdx.x - grp * a.nkt * a.gsz;
    const int rank = rem / gsize;
    const int bh = grp * a.gsz + rem % gsize;
    const int b = bh / p.Hkv, kvh = bh % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool padded = p.cu_q == nullptr;
    const int k0 = rank * kKeysK;
    const int kcap = padded ? p.K : si.Kb;  // keys this CTA may write
    if (k0 >= kcap) return;                 // uniform: before any barrier

    const uint32_t raw = smem_addr(smem_k);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_k + (base - raw);
    const uint32_t bars = base + L::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::BAR_OFF + 8 * K_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto row_full = [&](int s) { return bar(K_ROW_FULL + s); };
    auto row_empty = [&](int s) { return bar(K_ROW_FULL + kStagesK + s); };
    auto rstage = [&](int s) { return base + L::R_OFF + (uint32_t)s * L::STAGE; };
    // [stage][4][kRowsK]: -LSE (log2 units), -Dq, lo, hi
    float *stats = reinterpret_cast<float *>(gbase + L::ST_OFF);
    int *flags = reinterpret_cast<int *>(gbase + L::FLAG_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the query positions that attend to any of the CTA's keys: an interval
    int qf = 0, qe = 0;
    if (k0 < si.Kb) rows_for_keys(k0, min(k0 + kKeysK, si.Kb), si.Qb, si.Kb, p.window, p.mask, qf, qe);
    const int ntiles = qe > qf ? (qe - qf + PP - 1) / PP : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(K_KV_FULL), 1);
        mbar_init(bar(K_S_FULL), 1);
        mbar_init(bar(K_DP_FULL), 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(K_P_READY + h), 128);
            mbar_init(bar(K_DS_READY + h), 128);
        }
        mbar_init(bar(K_ACC_FULL), 1);
        mbar_init(bar(K_TEARDOWN), 2);  // one commit from each MMA-issuing thread
        mbar_init(bar(K_DV_DONE), 1);
        mbar_init(bar(K_DK_DONE), 1);
        mbar_init(bar(K_ROWS_READY), 1);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(row_full(s), 1);
            mbar_init(row_empty(s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarpK) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kLoadWarpK && lane == 0 && ntiles > 0) {
        // the tensor maps' descriptors on their way while the CTA sets up
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kLoadWarpK) regs_decrease<kRegsOtherK>();
    if (warp == kLoadWarpK) {
        // ------------------------------------------------ TMA producer + row stats
        const int qrow = padded ? 0 : (int)si.q_off;
        const int krow = padded ? 0 : (int)si.k_off;
        const int bc = padded ? b : 0;
        bool ok = true;
        uint32_t armed = 0, armed_ph = 0;
        if (ntiles > 0 && lane == 0) {
            mbar_arrive_expect_tx(bar(K_KV_FULL), L::KTILE + L::VTILE);
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(base + L::K_OFF + c * L::KCH, &tmK, bar(K_KV_FULL), c * 64, kvh,
                            krow + k0, bc);
            for (int c = 0; c < DV / 64; ++c)
                tma_load_4d(base + L::V_OFF + c * L::KCH, &tmV, bar(K_KV_FULL), c * 64, kvh,
                            krow + k0, bc);
        }
        // The rows of tile t + kStagesK are prefetched into L2 when tile t is
        // loaded, and each tile's row statistics (global LSE and Dq loads) are
        // gathered before waiting for its stage: the stage is free only once
        // the previous occupant's products have completed, and a load started
        // then from DRAM stalled the MMA threads.
        auto prefetch_rows = [&](int tt) {
            const int r0 = qrow + qf + tt * PP;
            for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_4d(&tmQ, c * 64, kvh * G, r0, bc);
            for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_4d(&tmO, c * 64, kvh * G, r0, bc);
        };
        if (lane == 0)
            for (int tt = 0; tt < kStagesK && tt < ntiles; ++tt) prefetch_rows(tt);
        // launched as a programmatic dependent of the dQ kernel (which writes
        // Dq): Dq is complete and visible once this returns (a no-op otherwise)
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        for (int t = 0; t < ntiles && ok; ++t) {
            const int s = t % kStagesK;
            const uint32_t ph = (uint32_t)(t / kStagesK) & 1u;
            // per-row statistics of the tile, four rows a lane
            float nl2[kRowsK / 32], ndl[kRowsK / 32];
            int rlo[kRowsK / 32], rhi[kRowsK / 32];
            bool inner = true;
#pragma unroll
            for (int e = 0; e < kRowsK / 32; ++e) {
                const int i = lane + 32 * e;  // row of the tile = smem row
                const int pos = qf + t * PP + i / G;
                const int hh = kvh * G + i % G;
                int lo = 0, hi = 0;
                if (pos < si.Qb) legal_range(pos, si.Qb, si.Kb, p.window, p.mask, lo, hi);
                float l2 = 0.f, dl = 0.f;
                if (hi > lo) {
                    const long long row = (si.q_off + pos) * p.Hq + hh;
                    l2 = p.lse[row] * kLog2e;
                    dl = bp.delta[row];
                }
                nl2[e] = -l2;  // stored negated: one packed FMA / add a pair of rows
                ndl[e] = -dl;
                rlo[e] = lo;
                rhi[e] = hi;
                inner = inner && lo <= k0 && hi >= k0 + kKeysK;
            }
            inner = __all_sync(0xffffffffu, inner);
            ok = warp_wait_t(row_empty(s), ph ^ 1u, abort_flag, wl);
            if (!ok) break;
            float *st = stats + s * 4 * kRowsK;
#pragma unroll
            for (int e = 0; e < kRowsK / 32; ++e) {
                const int i = lane + 32 * e;
                st[i] = nl2[e];
                st[kRowsK + i] = ndl[e];
                reinterpret_cast<int *>(st)[2 * kRowsK + i] = rlo[e];
                reinterpret_cast<int *>(st)[3 * kRowsK + i] = rhi[e];
            }
            if (lane == 0) flags[s] = inner ? 1 : 0;
            __syncwarp();
            if (lane == 0) {
                const int r0 = qrow + qf + t * PP;
                mbar_arrive_expect_tx(row_full(s), L::STAGE);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(rstage(s) + c * L::RCH, &tmQ, row_full(s), c * 64, kvh * G, r0, bc);
                for (int c = 0; c < DV / 64; ++c)
                    tma_load_4d(rstage(s) + L::QTILE + c * L::RCH, &tmO, row_full(s), c * 64,
                                kvh * G, r0, bc);
                armed |= 1u << s;
                armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
                if (t + kStagesK < ntiles) prefetch_rows(t + kStagesK);
            }
        }
        if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
        if (lane == 0) {
            // drain: every copy issued has landed before the CTA exits (these
            // waits ignore the abort flag: the copies always land)
            if (ntiles > 0) mbar_wait_drain(bar(K_KV_FULL), 0);
            for (int s = 0; s < kStagesK; ++s)
                if (armed & (1u << s)) mbar_wait_drain(row_full(s), (armed_ph >> s) & 1u);
        }
    } else if (warp == kMmaWarpK) {
        // ---------------------------------------------- S^T / dP^T MMA issuer
        // Two issuing threads (S^T and dP^T here, dV and dK in warp 10): one
        // thread issuing the 32 products of a tile spent more cycles issuing
        // than the tensor core spent on them.  S^T and dP^T overwrite the
        // previous tile's P^T / dS^T, so they wait for its dV / dK products to
        // complete (the other thread's commits).  A warp-wide wait costs more
        // than the wait of one thread.
        if (lane == 0) {
            bool ok = ntiles == 0 || mbar_wait(bar(K_KV_FULL), 0, abort_flag, wl);
            const uint64_t kd = sw128_desc(base + L::K_OFF, 16, 1024);
            const uint64_t vd = sw128_desc(base + L::V_OFF, 16, 1024);
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t % kStagesK;
                const uint32_t tp = (uint32_t)t & 1u;  // parity of this tile's phases
                if (!mbar_wait(row_full(s), (uint32_t)(t / kStagesK) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                if (t > 0 && !mbar_wait(bar(K_DV_DONE), tp ^ 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t qd = sw128_desc(rstage(s), 16, 1024);
                const uint64_t od = sw128_desc(rstage(s) + L::QTILE, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + L::ST_COL, kd + (((kk / 4) * L::KCH + (kk % 4) * 32) >> 4),
                           qd + (((kk / 4) * L::RCH + (kk % 4) * 32) >> 4), a.idesc_s, kk > 0);
                mma_commit(bar(K_S_FULL));
                if (t > 0 && !mbar_wait(bar(K_DK_DONE), tp ^ 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DV / 16; ++kk)
                    mma_ss(tmem + L::DPT_COL, vd + (((kk / 4) * L::KCH + (kk % 4) * 32) >> 4),
                           od + (((kk / 4) * L::RCH + (kk % 4) * 32) >> 4), a.idesc_s, kk > 0);
                mma_commit(bar(K_DP_FULL));
                // rows of the tile past the sequence's queries may hold anything
                // (NaN included): their P and dS are 0, and their Q and dO rows
                // are zeroed so that 0 * row stays 0 -- once S^T and dP^T, which
                // read them, have completed, and before the dV / dK products
                // (the other thread waits for K_ROWS_READY on such tiles)
                const int pos0 = qf + t * PP;
                const int nreal = min(kRowsK, max(0, (si.Qb - pos0) * G));
                if (nreal < kRowsK) {
                    if (!mbar_wait(bar(K_DP_FULL), tp, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    uint8_t *rt = gbase + (rstage(s) - base);
                    const int nzero = kRowsK - nreal;
                    for (int c = 0; c < D / 64 + DV / 64; ++c)
                        for (int i = 0; i < nzero * 8; ++i)
                            *reinterpret_cast<uint4 *>(rt + c * L::RCH + nreal * 128 + i * 16) =
                                make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(K_ROWS_READY));
                }
            }
            if (!ok) raise_abort_t(abort_flag, p.status);
            mma_commit(bar(K_TEARDOWN));
            mbar_wait_drain(bar(K_TEARDOWN), 0);  // ignores the abort flag
        }
        __syncwarp();
    } else if (warp == kAccWarpK) {
        // --------------------------------------------------- dV / dK MMA issuer
        if (lane == 0) {
            bool ok = true;
            uint32_t nz = 0;  // tiles with zeroed rows so far (K_ROWS_READY phases)
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t % kStagesK;
                const uint32_t tp = (uint32_t)t & 1u;
                if (!mbar_wait(row_full(s), (uint32_t)(t / kStagesK) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                const int pos0 = qf + t * PP;
                const int nreal = min(kRowsK, max(0, (si.Qb - pos0) * G));
                if (nreal < kRowsK) {
                    if (!mbar_wait(bar(K_ROWS_READY), nz & 1u, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    ++nz;
                }
                // dV += P^T dO, half by half as the warpgroups deliver P^T
                const uint64_t omn = sw128_desc(rstage(s) + L::QTILE, L::RCH, 1024);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!mbar_wait(bar(K_P_READY + h), tp, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kHalfK / 16; ++kk)
                        mma_ts(tmem + L::DV_COL, tmem + L::ST_COL + h * kHalfK + kk * 8,
                               omn + (((h * kHalfK + kk * 16) * 128) >> 4), a.idesc_v,
                               (t > 0 || h > 0 || kk > 0) ? 1u : 0u);
                }
                if (!ok) break;
                mma_commit(bar(K_DV_DONE));
                // dK += dS^T Q, likewise
                const uint64_t qmn = sw128_desc(rstage(s), L::RCH, 1024);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!mbar_wait(bar(K_DS_READY + h), tp, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kHalfK / 16; ++kk)
                        mma_ts(tmem + L::DK_COL, tmem + L::DPT_COL + h * kHalfK + kk * 8,
                               qmn + (((h * kHalfK + kk * 16) * 128) >> 4), a.idesc_k,
                               (t > 0 || h > 0 || kk > 0) ? 1u : 0u);
                }
                if (!ok) break;
                mma_commit(bar(K_DK_DONE));
                // the stage's S^T / dP^T products completed before its dS^T was
                // written, so this commit covers every read of the stage
                mma_commit(row_empty(s));
                if (t == ntiles - 1) mma_commit(bar(K_ACC_FULL));
            }
            if (!ok) raise_abort_t(abort_flag, p.status);
            mma_commit(bar(K_TEARDOWN));
            mbar_wait_drain(bar(K_TEARDOWN), 0);  // ignores the abort flag
        }
        __syncwarp();
    } else if (warp < kLoadWarpK) {
        // ------------------------------------------- elementwise warps, epilogue
        regs_increase<kRegsElemK>();
        const int hg = warp >> 2;  // warpgroup = half of the tile's rows
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key of the CTA = TMEM lane
        const int key = k0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + L::ST_COL + hg * kHalfK;
        const uint32_t tP = tmem + lane_off + L::DPT_COL + hg * kHalfK;
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int s = t % kStagesK;
            const uint32_t tp = (uint32_t)t & 1u;
            if (!warp_wait_t(bar(K_S_FULL), tp, abort_flag, wl)) {
                ok = false;
                break;
            }
            // the tile's row statistics: published with its row_full phase (the
            // stage is not refilled before this tile's dV / dK MMAs, which wait
            // for both warpgroups)
            if (!warp_wait_t(row_full(s), (uint32_t)(t / kStagesK) & 1u, abort_flag, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *st = stats + s * 4 * kRowsK + hg * kHalfK;
            const int *sti = reinterpret_cast<const int *>(stats + s * 4 * kRowsK) + hg * kHalfK;
            // Rows that may not see this key give P = dS = 0.  Interior tiles
            // (every row sees every key of the CTA; the flag is the same for
            // every thread) take a path without the test; elsewhere bit `row`
            // of keep[row / 32], built once a tile, is tested against
            // compile-time bits (a per-key || / && compiled to branches, ~3x
            // the step's cost).  Pairs of rows share packed f32x2 arithmetic:
            // with eight elementwise warps the step is bound by issue.
            const bool inner = flags[s] != 0;
            uint32_t keep[2] = {0xffffffffu, 0xffffffffu};
            if (!inner) {
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    uint32_t m = 0;
#pragma unroll 8
                    for (int i = 0; i < 32; ++i) {
                        const int row = w * 32 + i;
                        const bool in = (key >= sti[2 * kRowsK + row]) & (key < sti[3 * kRowsK + row]);
                        m |= (in ? 1u : 0u) << i;
                    }
                    keep[w] = m;
                }
            }
            const uint64_t c2 = f2pack(a.c2, a.c2);
            float pr[kHalfK];
            // P^T: 2^(S c - LSE), then 16-bit pairs over the first half of this
            // half's S^T columns
            auto p_phase = [&](auto masked) {
#pragma unroll
                for (int c = 0; c < kHalfK / 32; ++c) {
                    uint32_t sv[32];
                    tmem_ld32(tS + c * 32, sv);
                    tmem_ld_wait();
                    const float4 *l4 = reinterpret_cast<const float4 *>(st + c * 32);
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 nl = l4[i4];  // -LSE of four rows
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int i = 4 * i4 + 2 * h2;
                            const uint64_t x2 = ffma2(
                                f2pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2,
                                h2 == 0 ? f2pack(nl.x, nl.y) : f2pack(nl.z, nl.w));
                            float x0, x1;
                            f2unpack(x2, x0, x1);
                            float e0 = ex2f(x0), e1 = ex2f(x1);
                            if (decltype(masked)::value) {
                                e0 = ((keep[c] >> i) & 1u) ? e0 : 0.f;
                                e1 = ((keep[c] >> (i + 1)) & 1u) ? e1 : 0.f;
                            }
                            pr[c * 32 + i] = e0;
                            pr[c * 32 + i + 1] = e1;
                            sv[i / 2] = pack16<T>(e0, e1);  // over the consumed sv[i / 2]
                        }
                    }
                    tmem_st16(tS + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(sv));
                }
            };
            // dS^T: P (dP - Dq), likewise over dP^T
            auto ds_phase = [&](auto masked) {
#pragma unroll
                for (int c = 0; c < kHalfK / 32; ++c) {
                    uint32_t pv[32];
                    tmem_ld32(tP + c * 32, pv);
                    tmem_ld_wait();
                    const float4 *d4 = reinterpret_cast<const float4 *>(st + kRowsK + c * 32);
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 nd = d4[i4];  // -Dq of four rows
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int i = 4 * i4 + 2 * h2;
                            const uint64_t y2 = fmul2(
                                fadd2(f2pack(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])),
                                      h2 == 0 ? f2pack(nd.x, nd.y) : f2pack(nd.z, nd.w)),
                                f2pack(pr[c * 32 + i], pr[c * 32 + i + 1]));
                            float d0, d1;
                            f2unpack(y2, d0, d1);
                            if (decltype(masked)::value) {
                                d0 = ((keep[c] >> i) & 1u) ? d0 : 0.f;
                                d1 = ((keep[c] >> (i + 1)) & 1u) ? d1 : 0.f;
                            }
                            pv[i / 2] = pack16<T>(d0, d1);  // over the consumed pv[i / 2]
                        }
                    }
                    tmem_st16(tP + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(pv));
                }
            };
            if (inner)
                p_phase(std::false_type{});
            else
                p_phase(std::true_type{});
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(K_P_READY + hg));
            if (!warp_wait_t(bar(K_DP_FULL), tp, abort_flag, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (inner)
                ds_phase(std::false_type{});
            else
                ds_phase(std::true_type{});
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(K_DS_READY + hg));
        }
        if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
        // epilogue: warpgroup 0 writes dV, warpgroup 1 dK * scale (zeros for
        // keys no row sees)
        if (ok && ntiles > 0) {
            ok = warp_wait_t(bar(K_ACC_FULL), 0, abort_flag, wl);
            if (!ok && lane == 0) raise_abort_t(abort_flag, p.status);
            tc_fence_after();
        }
        const bool writes = key < kcap;
        const bool has = ok && ntiles > 0;
        const long long krow = (si.k_off + key) * p.Hkv + kvh;
        const int W = hg == 0 ? p.Dv : p.D;
        const int WT = hg == 0 ? DV : D;
        const float sc = hg == 0 ? 1.f : p.scale;
        T *dst = static_cast<T *>(hg == 0 ? bp.dv : bp.dk) + krow * W;
        const uint32_t col0 = hg == 0 ? L::DV_COL : L::DK_COL;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c * 32 < WT) {
                uint32_t v[32];
                if (has) {
                    tmem_ld32(tmem + lane_off + col0 + c * 32, v);
                    tmem_ld_wait();
                }
                if (writes) {
                    auto f = [&](int i) { return has ? __uint_as_float(v[i]) * sc : 0.f; };
#pragma unroll
                    for (int i = 0; i < 32; i += 8)
                        if (c * 32 + i < W)
                            *reinterpret_cast<uint4 *>(dst + c * 32 + i) = make_uint4(
                                pack16<T>(f(i), f(i + 1)), pack16<T>(f(i + 2), f(i + 3)),
                                pack16<T>(f(i + 4), f(i + 5)), pack16<T>(f(i + 6), f(i + 7)));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpK) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T, int D, int DV>
int launch_kv_t(const BwdParams &bp, bool bf16, cudaStream_t stream, bool pdl) {
    using L = KvLayout<D, DV>;
    const AttnParams &p = bp.f;
    KvArgs a;
    a.bp = bp;
    a.nkt = (p.K + kKeysK - 1) / kKeysK;
    {
        // rows of one (sequence, KV head) pair: Q and dO of its G heads
        const long long qlen = p.cu_q ? (p.Tq + p.B - 1) / p.B : p.Q;
        const long long pair_bytes = qlen * p.G * (long long)(p.D + p.Dv) * 2;
        // groups of about equal size, each group's rows within the budget
        const long long budget = 128ll << 20;
        const long long nbh = (long long)p.B * p.Hkv;
        const long long ngrp = std::max(1ll, (nbh * pair_bytes + budget - 1) / budget);
        a.gsz = (int)std::max(1ll, (nbh + ngrp - 1) / ngrp);
    }
    a.c2 = p.scale * kLog2e;
    a.idesc_s = idesc_f16(bf16, kKeysK, kRowsK, false, false);
    a.idesc_v = idesc_f16(bf16, kKeysK, DV, true, false);
    a.idesc_k = idesc_f16(bf16, kKeysK, D, true, false);
    const long long grid = (long long)a.nkt * p.B * p.Hkv;
    if (grid == 0) return 0;
    if (grid >= (1LL << 31)) {
        set_error("tcgen05 dK/dV: %lld blocks exceed one launch", grid);
        return 2;
    }
    const bool padded = p.cu_q == nullptr;
    const uint64_t qrows = padded ? (uint64_t)p.Q : (uint64_t)p.Tq;
    const uint64_t krows = padded ? (uint64_t)p.K : (uint64_t)p.Tk;
    const uint64_t nb = padded ? (uint64_t)p.B : 1;
    const uint32_t pp = (uint32_t)(kRowsK / p.G);
    CUtensorMap tq, to, tk, tv;
    int rc = make_tma_map_4d(&tq, p.q, bf16, (uint64_t)p.D, p.Hq, qrows, nb, (uint32_t)p.G, pp);
    if (!rc) rc = make_tma_map_4d(&to, bp.dout, bf16, (uint64_t)p.Dv, p.Hq, qrows, nb, (uint32_t)p.G, pp);
    if (!rc) rc = make_tma_map_4d(&tk, p.k, bf16, (uint64_t)p.D, p.Hkv, krows, nb, 1, kKeysK);
    if (!rc) rc = make_tma_map_4d(&tv, p.v, bf16, (uint64_t)p.Dv, p.Hkv, krows, nb, 1, kKeysK);
    if (rc) return rc;
    auto kern = bwd_dkdv_tc_kernel<T, D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("tcgen05 dK/dV: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsK);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, a, tq, to, tk, tv);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 dK/dV launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_kv_dtype(const BwdParams &bp, bool bf16, cudaStream_t stream, bool pdl) {
    const bool d128 = bp.f.D > 64, dv128 = bp.f.Dv > 64;
    if (d128 && dv128) return launch_kv_t<T, 128, 128>(bp, bf16, stream, pdl);
    if (!d128 && !dv128) return launch_kv_t<T, 64, 64>(bp, bf16, stream, pdl);
    if (d128) return launch_kv_t<T, 128, 64>(bp, bf16, stream, pdl);
    return launch_kv_t<T, 64, 128>(bp, bf16, stream, pdl);
}

template <typename T, int D, int DV>
int launch_t(const BwdParams &bp, bool bf16, cudaStream_t stream, int self_delta) {
    using L = DqLayout<D, DV>;
    const AttnParams &p = bp.f;
    DqArgs a;
    a.bp = bp;
    a.self_delta = self_delta;
    a.nqt = (p.Q + kRowsT - 1) / kRowsT;
    a.c2 = p.scale * kLog2e;
    a.idesc_s = idesc_f16(bf16, kRowsT, kKeysT, false, false);
    a.idesc_dq = idesc_f16(bf16, kRowsT, D, true, false);
    const long long grid = (long long)a.nqt * p.B * p.Hq;
    if (grid == 0) return 0;
    if (grid >= (1LL << 31)) {
        set_error("tcgen05 dQ: %lld blocks exceed one launch", grid);
        return 2;
    }
    const bool padded = p.cu_q == nullptr;
    const uint64_t qrows = padded ? (uint64_t)p.Q : (uint64_t)p.Tq;
    const uint64_t krows = padded ? (uint64_t)p.K : (uint64_t)p.Tk;
    const uint64_t nb = padded ? (uint64_t)p.B : 1;
    CUtensorMap tq, to, tk, tv, tout;
    int rc = make_tma_map_4d(&tq, p.q, bf16, (uint64_t)p.D, p.Hq, qrows, nb, 1, kRowsT);
    if (!rc) rc = make_tma_map_4d(&to, bp.dout, bf16, (uint64_t)p.Dv, p.Hq, qrows, nb, 1, kRowsT);
    if (!rc && self_delta)
        rc = make_tma_map_4d(&tout, p.o, bf16, (uint64_t)p.Dv, p.Hq, qrows, nb, 1, kRowsT);
    else
        tout = tq;  // never read
    if (!rc && krows > 0) {
        rc = make_tma_map_4d(&tk, p.k, bf16, (uint64_t)p.D, p.Hkv, krows, nb, 1, kKeysT);
        if (!rc) rc = make_tma_map_4d(&tv, p.v, bf16, (uint64_t)p.Dv, p.Hkv, krows, nb, 1, kKeysT);
    } else {
        tk = tq;  // never read: no CTA has a key tile
        tv = tq;
    }
    if (rc) return rc;
    auto kern = bwd_dq_tc_kernel<T, D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("tcgen05 dQ: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    kern<<<(unsigned)grid, kThreadsQ, L::SMEM, stream>>>(a, tq, to, tk, tv, tout);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 dQ launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_dtype(const BwdParams &bp, bool bf16, cudaStream_t stream, int self_delta) {
    const bool d128 = bp.f.D > 64, dv128 = bp.f.Dv > 64;
    if (d128 && dv128) return launch_t<T, 128, 128>(bp, bf16, stream, self_delta);
    if (!d128 && !dv128) return launch_t<T, 64, 64>(bp, bf16, stream, self_delta);
    if (d128) return launch_t<T, 128, 64>(bp, bf16, stream, self_delta);
    return launch_t<T, 64, 128>(bp, bf16, stream, self_delta);
}

}  // namespace

bool bwd_dq_tc_supported(const AttnParams &p, int dtype) {
    if (dtype != 1 && dtype != 2) return false;
    if (p.D < 64 || p.D > 128 || p.D % 16 || p.Dv < 64 || p.Dv > 128 || p.Dv % 16) return false;
    if (p.block_table != nullptr) return false;
    const long long rows = p.cu_q ? p.Tq : (long long)p.Q;
    const long long keys = p.cu_q ? p.Tk : (long long)p.K;
    return rows < (1LL << 31) && keys < (1LL << 31);
}

bool bwd_dkdv_tc_supported(const AttnParams &p, int dtype) {
    // the rows of a tile are (position, head) pairs of one KV group: 128 / G positions
    return bwd_dq_tc_supported(p, dtype) && p.G >= 1 && p.G <= kRowsK && kRowsK % p.G == 0;
}

int launch_bwd_dkdv_tc(const BwdParams &bp, int dtype, cudaStream_t stream, bool after_dq) {
    if (dtype == 2) return launch_kv_dtype<__nv_bfloat16>(bp, true, stream, after_dq);
    return launch_kv_dtype<__half>(bp, false, stream, after_dq);
}

int launch_bwd_dq_tc(const BwdParams &bp, int dtype, cudaStream_t stream, int self_delta) {
    if (dtype == 2) return launch_dtype<__nv_bfloat16>(bp, true, stream, self_delta);
    return launch_dtype<__half>(bp, false, stream, self_delta);
}

}  // namespace attn
