// kernel_prefill_wide_tc.cu -- bf16 / fp16 causal GQA prefill on tcgen05 for
// head widths above 128 (up to 256), sm_103a.
//
// The same online-softmax program as kernel_prefill_tc.cu ("Attention
// execution mapping" (LuisaCompute), sections 1-2), laid out for wide heads.
// A 128-row Q tile of width 256 is 64 KB of shared memory and its O
// accumulator 256 TMEM columns, so a CTA holds one Q tile per work unit
// instead of two:
//
// * TMEM (512 columns): S0 | S1 | O.  S is double-buffered: while the softmax
//   warpgroup works on S(j), the tensor core computes S(j+1) into the other
//   buffer (and O += P(j-1) V(j-1)), so the softmax steps follow one another
//   without waiting for the MMA chain.  S(j+2) reuses S(j)'s buffer: it is
//   issued after PV(j) by the same thread (tcgen05.mma executes in order).
// * Shared memory: the Q tile, a ring of two 64 KB elements (a whole K or V
//   tile of 128 keys), a 16 KB epilogue staging box.  The TMA warp loads K one
//   tile ahead of V -- K0, K1, V0, K2, V1, K3, V2, ... -- which is the order
//   the MMA warp consumes them in (S0, S1, PV0, S2, PV1, S3, ...), so two
//   elements suffice: V(j) is loaded once S(j) has freed its element, K(j+2)
//   once S(j+1) has freed its.
// * Warp roles: warps 0-3 the softmax (TMEM lane = row = thread), warps 4-7
//   the epilogue (O out of TMEM, normalised, TMA stores), warp 8 issues the
//   MMAs, warp 9 the TMA loads; warps 10-11 idle.
// * The FlyDSL page ("Accelerating PyTorch on AMD GPUs with FlyDSL", section
//   on FMHA through AOTriton, figure 13) stages wide K / V through LDS in
//   halves of the head dimension; here a whole 256-wide tile fits one ring
//   element, and the split that matters is in time: S of one tile against
//   the softmax and PV of the previous one.
// Every mbarrier wait is bounded as in kernel_prefill_tc.cu.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_softmax.cuh"
#include "wide_common.cuh"

namespace attn {
namespace {

using namespace sm100;
using namespace tcfwd;
using namespace tcwide;

constexpr int kBM = 128;  // rows per Q tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;  // warps 4-7
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kRegsSoftmax = 192;
constexpr uint32_t kRegsEpi = 152;
constexpr uint32_t kRegsOther = 152;
constexpr uint32_t kRegsLaunch = 168;  // 65536 / 384, rounded down to a multiple of 8
static_assert(128 * (kRegsSoftmax + kRegsEpi + kRegsOther) <= kThreads * kRegsLaunch,
              "register split");
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 128 bytes (64 columns)
constexpr int kNE = 2;                        // ring elements
constexpr int kPrefetchTiles = 3;

struct WideArgs {
    AttnParams p;
    int Gp;            // heads packed into the rows of a Q tile
    int QP;            // query positions per Q tile (kBM / Gp)
    int nsub;          // head subgroups per KV head
    int nqblk;         // query blocks (QP positions) per sequence
    uint32_t per;      // units per query block: B * Hkv * nsub
    uint32_t hs;       // Hkv * nsub
    long long nunits;
    float c_scale;     // |scale| * log2(e)
    uint32_t idesc_s;  // S = Q K^T (M 128, N 128)
    uint32_t idesc_o;  // O += P V (M 128, N DV)
};

template <int D, int DV> struct WideLayout {
    static constexpr int QTILE = kBM * D * 2;
    static constexpr int KTILE = kBN * D * 2;
    static constexpr int VTILE = kBN * DV * 2;
    static constexpr int ELEM = KTILE > VTILE ? KTILE : VTILE;
    static constexpr int STG_BYTES = kBM * 128;           // 64 columns of the Q tile
    static constexpr int STATS_BYTES = 2 * kBM * 4;       // 1 / l per row, by unit parity
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = QTILE;
    static constexpr int STG_OFF = KV_OFF + kNE * ELEM;
    static constexpr int STATS_OFF = STG_OFF + STG_BYTES;
    static constexpr int BAR_OFF = STATS_OFF + STATS_BYTES;
    static constexpr int SMEM = 1024 + BAR_OFF + 256;
    static constexpr int O_COL = 256;  // TMEM: S0 [0, 128), S1 [128, 256), O [256, 256 + DV)
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(O_COL + DV <= 512, "TMEM budget");
};

enum : int {
    W_Q_FULL = 0,
    W_Q_EMPTY = 1,
    W_S_FULL = 2,     // [2] by S buffer
    W_P_READY = 4,    // [2]
    W_O_FULL = 6,
    W_O_EMPTY = 7,
    W_STATS = 8,      // [2] by unit parity
    W_TEARDOWN = 10,
    W_KV_FULL = 11,   // [kNE]
    W_KV_EMPTY = 13,  // [kNE]
    W_PV_DONE = 15,   // one phase per tile: its PV has completed
    W_NBARS = 16,
};

__device__ __forceinline__ QTileUnit wide_unit(const WideArgs &a, long long u64) {
    return qtile_unit(a.p, a.per, a.hs, a.nsub, a.Gp, a.QP, a.nqblk, (uint32_t)u64);
}

// Ring positions (relative to the unit's first element) of K_j and V_j in
// the load order K0, K1, V0, K2, V1, K3, V2, ..., V_{n-2}, V_{n-1}.
__device__ __forceinline__ uint32_t pos_k(int j) { return j == 0 ? 0u : (uint32_t)(2 * j - 1); }
__device__ __forceinline__ uint32_t pos_v(int j, int n) {
    return j + 1 < n ? (uint32_t)(2 * j + 2) : (uint32_t)(2 * n - 1);
}

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_tc_kernel(const __grid_constant__ WideArgs a,
                           const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO) {
    using L = WideLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t q_smem = base + L::Q_OFF;
    const uint32_t kv_smem = base + L::KV_OFF;
    const uint32_t bars = base + L::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::BAR_OFF + 8 * W_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *unit_desc = reinterpret_cast<int *>(tmem_slot + 2);  // [2 parities][4]

    const AttnParams &p = a.p;
    const uint64_t wl = p.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool padded = p.cu_q == nullptr;

    if (threadIdx.x == 0) {
        mbar_init(bar(W_Q_FULL), 1);
        mbar_init(bar(W_Q_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(W_S_FULL + i), 1);
            mbar_init(bar(W_P_READY + i), 128);
            mbar_init(bar(W_STATS + i), 128);
        }
        mbar_init(bar(W_O_FULL), 1);
        mbar_init(bar(W_O_EMPTY), 128);
        mbar_init(bar(W_TEARDOWN), 1);
        mbar_init(bar(W_PV_DONE), 1);
        for (int e = 0; e < kNE; ++e) {
            mbar_init(bar(W_KV_FULL + e), 1);
            mbar_init(bar(W_KV_EMPTY + e), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto kv_full = [&](int e) { return bar(W_KV_FULL + e); };
    auto kv_empty = [&](int e) { return bar(W_KV_EMPTY + e); };
    auto elem = [&](int e) { return kv_smem + (uint32_t)e * L::ELEM; };

    if (warp >= kMmaWarp) {
        regs_decrease<kRegsOther>();
        if (warp == kLoadWarp) {
            // --------------------------------------------------------- TMA producer
            if (lane == 0) {
                uint32_t kv_it = 0, q_ph = 0;
                int last_q_parity = -1;
                uint32_t armed = 0, armed_parity = 0;
                bool ok = true;
                for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
                    const long long u = snake(rnd, blockIdx.x, gridDim.x);
                    if (u >= a.nunits) continue;
                    const QTileUnit x = wide_unit(a, u);
                    if (x.n_kv == 0) continue;
                    const int qrow = (padded ? 0 : (int)x.si.q_off) + x.q0;
                    const int krow = padded ? 0 : (int)x.si.k_off;
                    const int bc = padded ? x.b : 0;
                    if (!mbar_wait(bar(W_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                        ok = false;
                        break;
                    }
                    int *d = unit_desc + q_ph * 4;
                    d[0] = x.n_kv;
                    d[1] = x.kv_start;
                    d[2] = x.hi_unit;
                    mbar_arrive_expect_tx(bar(W_Q_FULL), L::QTILE);
                    last_q_parity = (int)q_ph;
                    q_ph ^= 1u;
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(q_smem + c * kChunkBytes, &tmQ, bar(W_Q_FULL), c * 64, x.h0,
                                    qrow, bc);
                    auto prefetch_kv = [&](int jj) {
                        const int kr = krow + x.kv_start + jj * kBN;
                        for (int c = 0; c < D / 64; ++c)
                            tma_prefetch_l2_4d(&tmK, c * 64, x.kvh, kr, bc);
                        for (int c = 0; c < DV / 64; ++c)
                            tma_prefetch_l2_4d(&tmV, c * 64, x.kvh, kr, bc);
                    };
                    for (int jj = 1; jj < kPrefetchTiles && jj < x.n_kv; ++jj) prefetch_kv(jj);
                    // one ring element: K_j (which == 0) or V_j (which == 1)
                    auto emit = [&](int j, int which) -> bool {
                        const uint32_t it = kv_it++;
                        const int e = (int)(it % kNE);
                        const uint32_t ph = (it / kNE) & 1u;
                        if (!mbar_wait(kv_empty(e), ph ^ 1u, abort_flag, wl)) {
                            raise_abort(abort_flag, p.status, kStatusTimeoutKvEmpty);
                            return false;
                        }
                        const int kr = krow + x.kv_start + j * kBN;
                        if (which == 0) {
                            mbar_arrive_expect_tx(kv_full(e), L::KTILE);
                            for (int c = 0; c < D / 64; ++c)
                                tma_load_4d(elem(e) + c * kChunkBytes, &tmK, kv_full(e), c * 64,
                                            x.kvh, kr, bc);
                        } else {
                            mbar_arrive_expect_tx(kv_full(e), L::VTILE);
                            for (int c = 0; c < DV / 64; ++c)
                                tma_load_4d(elem(e) + c * kChunkBytes, &tmV, kv_full(e), c * 64,
                                            x.kvh, kr, bc);
                        }
                        armed |= 1u << e;
                        armed_parity = (armed_parity & ~(1u << e)) | (ph << e);
                        return true;
                    };
                    ok = emit(0, 0);
                    if (ok && x.n_kv > 1) ok = emit(1, 0);
                    for (int j = 0; j < x.n_kv && ok; ++j) {
                        if (j + kPrefetchTiles < x.n_kv) prefetch_kv(j + kPrefetchTiles);
                        ok = emit(j, 1);
                        if (ok && j + 2 < x.n_kv) ok = emit(j + 2, 0);
                    }
                }
                if (ok) {  // end marker, once the last Q tile has been consumed
                    if (mbar_wait(bar(W_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        unit_desc[q_ph * 4] = 0;
                        mbar_arrive(bar(W_Q_FULL));
                        last_q_parity = -1;
                    } else {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                    }
                }
                // drain: the copies always land, so these ignore the abort flag
                if (last_q_parity >= 0) mbar_wait_drain(bar(W_Q_FULL), (uint32_t)last_q_parity);
                for (int e = 0; e < kNE; ++e)
                    if (armed & (1u << e)) mbar_wait_drain(kv_full(e), (armed_parity >> e) & 1u);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            uint32_t kv_it = 0, q_ph = 0, o_ph = 0;
            uint32_t gt = 0;  // tiles issued so far, all units: S buffer gt & 1
            uint32_t p_par = 0;  // bit b: parity of P_READY[b]'s next phase
            bool ok = true;
            const uint64_t qd = sw128_desc(q_smem, 16, 1024);
            const uint32_t o_tm = tmem + (uint32_t)L::O_COL;
            while (ok) {
                if (!warp_wait(bar(W_Q_FULL), q_ph, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                const volatile int *d = unit_desc + q_ph * 4;
                q_ph ^= 1u;
                const int n = d[0], kv_start = d[1], hi_unit = d[2];
                if (n == 0) break;  // end marker
                const uint32_t kb = kv_it, g0 = gt;
                auto wait_elem = [&](uint32_t pos) -> bool {
                    const uint32_t it = kb + pos;
                    return warp_wait(kv_full((int)(it % kNE)), (it / kNE) & 1u, abort_flag, wl);
                };
                // S(j) = Q K_j^T into buffer (g0 + j) & 1, then release K_j
                auto issue_s = [&](int j) -> bool {
                    const uint32_t it = kb + pos_k(j);
                    if (!wait_elem(pos_k(j))) return false;
                    tc_fence_after();
                    if (lane == 0) {
                        const int e = (int)(it % kNE);
                        const uint64_t kd = sw128_desc(elem(e), 16, 1024);
                        const int nvalid = min(kBN, hi_unit - (kv_start + j * kBN));
                        const uint32_t ncols = (uint32_t)((nvalid + 15) & ~15);
                        const uint32_t idesc = (a.idesc_s & ~(0x3Fu << 17)) | ((ncols >> 3) << 17);
                        const uint32_t s_tm = tmem + ((g0 + (uint32_t)j) & 1u) * 128u;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4;
                            mma_ss(s_tm, qd + off, kd + off, idesc, kk > 0);
                        }
                        mma_commit(bar(W_S_FULL + (int)((g0 + (uint32_t)j) & 1u)));
                        mma_commit(kv_empty(e));
                        if (j == n - 1) mma_commit(bar(W_Q_EMPTY));
                    }
                    __syncwarp();
                    return true;
                };
                if (!issue_s(0) || (n > 1 && !issue_s(1))) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < n && ok; ++j) {
                    const uint32_t itv = kb + pos_v(j, n);
                    const int ev = (int)(itv % kNE);
                    // keys past the last one in use (last tile only) are left out
                    // 16 at a time; the V rows of the last 16-key step past it are
                    // zeroed (they may hold NaN) so that 0 * V stays 0
                    const int nvalid = min(kBN, hi_unit - (kv_start + j * kBN));
                    const int ksteps = (nvalid + 15) / 16;
                    const int nzero = ksteps * 16 - nvalid;
                    if (!wait_elem(pos_v(j, n))) {
                        ok = false;
                        break;
                    }
                    if (nzero > 0) {
                        uint8_t *vt = gbase + (elem(ev) - base) + nvalid * 128;
#pragma unroll
                        for (int c = 0; c < DV / 64; ++c)
                            for (int i = lane; i < nzero * 8; i += 32)
                                *reinterpret_cast<uint4 *>(vt + c * kChunkBytes + i * 16) =
                                    make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (j == 0) {  // the epilogue has read the previous unit's O
                        if (!warp_wait(bar(W_O_EMPTY), o_ph ^ 1u, abort_flag, wl)) {
                            ok = false;
                            break;
                        }
                        o_ph ^= 1u;
                    }
                    const uint32_t sb = (g0 + (uint32_t)j) & 1u;
                    if (!warp_wait(bar(W_P_READY + (int)sb), (p_par >> sb) & 1u, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    p_par ^= 1u << sb;
                    tc_fence_after();
                    if (lane == 0) {
                        // O (+)= P_j V_j: P from TMEM over S_j, V MN-major (64-column
                        // chunks kChunkBytes apart), N = DV
                        const uint64_t vd = sw128_desc(elem(ev), kChunkBytes, 1024);
                        const uint32_t s_tm = tmem + sb * 128u;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            if (kk < ksteps)
                                mma_ts(o_tm, s_tm + kk * 8, vd + (kk * 2048 >> 4), a.idesc_o,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(kv_empty(ev));
                        mma_commit(bar(W_PV_DONE));
                    }
                    __syncwarp();
                    // S(j + 2) reuses S_j's buffer: issued after PV(j)
                    if (j + 2 < n && !issue_s(j + 2)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                if (lane == 0) mma_commit(bar(W_O_FULL));
                __syncwarp();
                kv_it += 2u * (uint32_t)n;
                gt += (uint32_t)n;
            }
            if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutMma);
            if (lane == 0) {  // every MMA issued completes before TMEM is freed
                mma_commit(bar(W_TEARDOWN));
                mbar_wait_drain(bar(W_TEARDOWN), 0);
            }
            __syncwarp();
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------- softmax
        regs_increase<kRegsSoftmax>();
        const int r = warp * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tO = tmem + lane_off + (uint32_t)L::O_COL;
        const float c = a.c_scale;
        uint32_t gt = 0, s_par = 0, nunit = 0;  // s_par bit b: S_FULL[b]'s next parity
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        float *inv_l = reinterpret_cast<float *>(gbase + L::STATS_OFF);
        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            const QTileUnit x = wide_unit(a, u);
            const int qpos = x.q0 + r / a.Gp;
            const int head = x.h0 + r % a.Gp;
            const bool valid = qpos < x.si.Qb;
            const bool writes = padded ? qpos < p.Q : valid;
            int lo = 0, hi = 0;
            if (valid) legal_range(qpos, x.si.Qb, x.si.Kb, p.window, p.mask, lo, hi);
            const long long orow = (x.si.q_off + qpos) * p.Hq + head;
            if (x.n_kv == 0) {  // nothing to attend: +0 and -inf
                if (writes) {
                    uint4 *dst = reinterpret_cast<uint4 *>(og + orow * p.Dv);
                    for (int i = 0; i < p.Dv * 2 / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[orow] = -INFINITY;
                }
                continue;
            }
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < x.n_kv && ok; ++j) {
                const uint32_t sb = gt & 1u;
                ++gt;
                if (!warp_wait(bar(W_S_FULL + (int)sb), (s_par >> sb) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                s_par ^= 1u << sb;
                tc_fence_after();
                const uint32_t tS = tmem + lane_off + sb * 128u;
                const int k0 = x.kv_start + j * kBN;
                const bool interior = x.all_valid && k0 >= x.lo_last && k0 + kBN <= x.hi_first;
                // a rescale first waits for PV(j - 1): its phase of W_PV_DONE
                if (!softmax_tile<T, DV>(tS, tO, k0, interior, lo, hi, c, m_run, l_run,
                                         bar(W_PV_DONE), (gt - 2u) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(bar(W_P_READY + (int)sb));
            }
            if (!ok) break;
            const bool has = valid && l_run > 0.f;
            if (writes && p.lse) p.lse[orow] = has ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
            inv_l[(nunit & 1u) * kBM + r] = has ? 1.f / l_run : 0.f;
            mbar_arrive(bar(W_STATS + (int)(nunit & 1u)));
            ++nunit;
        }
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutSoftmax);
    } else {
        // ------------------------------------------------------------ epilogue
        regs_decrease<kRegsEpi>();
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const bool leader = warp == kEpiWarp0 && lane == 0;
        uint32_t o_ph = 0, st_par = 0, nunit = 0;  // st_par bit b: STATS[b]'s next parity
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        const float *inv_l = reinterpret_cast<const float *>(gbase + L::STATS_OFF);
        uint8_t *stg = gbase + L::STG_OFF;
        const uint32_t stg_s = base + L::STG_OFF;
        const uint32_t tO = tmem + lane_off + (uint32_t)L::O_COL;
        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            const QTileUnit x = wide_unit(a, u);
            if (x.n_kv == 0) continue;  // the softmax warps wrote those rows
            const int b = (int)(nunit & 1u);
            ++nunit;
            const bool got = warp_wait(bar(W_O_FULL), o_ph, abort_flag, wl) &&
                             warp_wait(bar(W_STATS + b), (st_par >> b) & 1u, abort_flag, wl);
            // the four warps go on or give up together (named barriers below)
            if (!bar_red_and(2, 128, got)) {
                ok = false;
                break;
            }
            o_ph ^= 1u;
            st_par ^= 1u << b;
            tc_fence_after();
            const float inv = inv_l[b * kBM + r];
            const bool by_tma = padded || x.q0 + a.QP <= x.si.Qb;
#pragma unroll
            for (int cp = 0; cp < DV / 64; ++cp) {
                if (leader) bulk_wait_read0();
                named_bar_sync(1, 128);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ov[32];
                    tmem_ld32(tO + cp * 64 + h * 32, ov);
                    tmem_ld_wait();
                    if (cp == DV / 64 - 1 && h == 1) {  // O is read: free it
                        tc_fence_before();
                        mbar_arrive(bar(W_O_EMPTY));
                    }
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = 8 * c4 + 2 * i;
                            w[i] = pack2<T>(inv > 0.f ? __uint_as_float(ov[e]) * inv : 0.f,
                                            inv > 0.f ? __uint_as_float(ov[e + 1]) * inv : 0.f);
                        }
                        const int ch = 4 * h + c4;
                        *reinterpret_cast<uint4 *>(stg + r * 128 + ((ch ^ (r & 7)) << 4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                if (by_tma) {
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    if (leader) {
                        const int qrow = (padded ? 0 : (int)x.si.q_off) + x.q0;
                        tma_store_4d(&tmO, stg_s, cp * 64, x.h0, qrow, padded ? x.b : 0);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int e = i * 32 + lane;
                        const int rr = quarter * 32 + (e >> 3), ch = e & 7;
                        const int qp = x.q0 + rr / a.Gp;
                        if (qp < x.si.Qb && cp * 64 + ch * 8 < p.Dv) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
                            const long long orr = (x.si.q_off + qp) * p.Hq + x.h0 + rr % a.Gp;
                            *reinterpret_cast<uint4 *>(og + orr * p.Dv + cp * 64 + ch * 8) = v;
                        }
                    }
                }
            }
        }
        if (leader) bulk_wait0();
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutEpilogue);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int wide_pack_factor(int G) {
    int gp = 1;
    while (gp < 16 && G % (gp * 2) == 0) gp *= 2;
    return gp;
}

template <typename T, int D, int DV>
int launch_wide_t(const AttnParams &p, bool bf16, cudaStream_t stream) {
    using L = WideLayout<D, DV>;
    WideArgs a;
    a.p = p;
    a.Gp = wide_pack_factor(p.G);
    a.QP = kBM / a.Gp;
    a.nsub = p.G / a.Gp;
    a.nqblk = (p.Q + a.QP - 1) / a.QP;
    a.nunits = (long long)a.nqblk * p.B * p.Hkv * a.nsub;
    a.per = (uint32_t)((long long)p.B * p.Hkv * a.nsub);
    a.hs = (uint32_t)(p.Hkv * a.nsub);
    const float sc = p.scale == 0.f ? 1e-30f : fabsf(p.scale);
    a.c_scale = sc * kLog2e;
    a.idesc_s = idesc_f16(bf16, kBM, kBN, false, p.scale < 0.f);
    a.idesc_o = idesc_f16(bf16, kBM, DV, true, false);
    if (a.nunits == 0) return 0;
    const bool padded = p.cu_q == nullptr;
    const uint64_t qrows = padded ? (uint64_t)p.Q : (uint64_t)p.Tq;
    const uint64_t krows = padded ? (uint64_t)p.K : (uint64_t)p.Tk;
    const uint64_t nb = padded ? (uint64_t)p.B : 1;
    CUtensorMap tq, tk, tv, to;
    int rc = make_tma_map_4d(&tq, p.q, bf16, (uint64_t)p.D, p.Hq, qrows, nb, a.Gp, a.QP);
    if (!rc) rc = make_tma_map_4d(&to, p.o, bf16, (uint64_t)p.Dv, p.Hq, qrows, nb, a.Gp, a.QP);
    if (rc) return rc;
    if (krows > 0) {
        rc = make_tma_map_4d(&tk, p.k, bf16, (uint64_t)p.D, p.Hkv, krows, nb, 1, kBN);
        if (!rc) rc = make_tma_map_4d(&tv, p.v, bf16, (uint64_t)p.Dv, p.Hkv, krows, nb, 1, kBN);
        if (rc) return rc;
    } else {
        tk = tq;  // never read: every unit has no key
        tv = tq;
    }
    auto kern = prefill_wide_tc_kernel<T, D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("wide prefill kernel: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    const int nsm = sm_count(dev);
    const long long grid = a.nunits < nsm ? a.nunits : nsm;
    kern<<<(unsigned)grid, kThreads, L::SMEM, stream>>>(a, tq, tk, tv, to);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("wide prefill kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_wide_dtype(const AttnParams &p, bool bf16, cudaStream_t stream) {
    const bool d256 = p.D > 128, dv256 = p.Dv > 128;
    if (d256 && dv256) return launch_wide_t<T, 256, 256>(p, bf16, stream);
    if (d256) return launch_wide_t<T, 256, 128>(p, bf16, stream);
    return launch_wide_t<T, 128, 256>(p, bf16, stream);
}

}  // namespace

bool prefill_wide_tc_supported(const AttnParams &p, int dtype) {
    if (p.D > 256 || p.Dv > 256) return prefill_wide512_tc_supported(p, dtype);
    if (dtype != 1 && dtype != 2) return false;
    if (p.D < 64 || p.D > 256 || p.D % 16 || p.Dv < 64 || p.Dv > 256 || p.Dv % 16) return false;
    if (p.D <= 128 && p.Dv <= 128) return false;  // the two-tile kernel's widths
    if (p.Q < 1 || p.block_table != nullptr || p.mask_bits != nullptr) return false;
    const long long rows = p.cu_q ? p.Tq : (long long)p.Q;
    const long long keys = p.cu_q ? p.Tk : (long long)p.K;
    const int gp = wide_pack_factor(p.G), qp = kBM / gp;
    const long long nunits = (long long)((p.Q + qp - 1) / qp) * p.B * p.Hkv * (p.G / gp);
    return rows < (1LL << 31) && keys < (1LL << 31) && nunits < (1LL << 31);
}

int launch_prefill_wide_tc(const AttnParams &p, int dtype, cudaStream_t stream) {
    if (p.D > 256 || p.Dv > 256) return launch_prefill_wide512_tc(p, dtype, stream);
    if (dtype == 2) return launch_wide_dtype<__nv_bfloat16>(p, true, stream);
    return launch_wide_dtype<__half>(p, false, stream);
}

}  // namespace attn
