// kernel_prefill_wide512_tc.cu -- bf16 / fp16 causal GQA prefill on tcgen05
// for head widths above 256 (up to 512), sm_103a.
//
// The same online-softmax program as the other tcgen05 forward kernels
// ("Attention execution mapping" (LuisaCompute), sections 1-2).  At width 512
// a 128-row Q tile is 128 KB of shared memory, a 128-key K tile another
// 128 KB, and O for 128 rows needs all 512 TMEM columns, so:
//
// * The output columns are split in halves of 256.  Each half of a Q tile
//   is a work unit of its own, on its own CTA: both halves compute the same
//   scores and softmax (the same inputs, the same code, so the same m and l)
//   and each accumulates O for its 256 columns.  The FlyDSL page
//   ("Accelerating PyTorch on AMD GPUs with FlyDSL", FMHA through AOTriton,
//   figure 13) splits its 512-wide O between waves the same way; here the
//   split is between CTAs, and the two halves of a Q tile are adjacent units
//   of the serpentine order, so they run at the same time and read K / V
//   through L2 once.
// * TMEM (512 columns): S0 | S1 | O-half.  S is double-buffered as in the
//   256-wide kernel: S(j + 1) is computed while the softmax works on S(j).
// * Shared memory: the Q tile (8 chunks of 64 columns x 128 rows, 128 KB)
//   and a ring of three 32 KB slots.  K streams through the ring two
//   64-column chunks (x 128 keys) a slot, so S(j) is the sum of eight chunk
//   products over four slots; V 64 keys x the half's 256 columns a slot (four
//   64-column boxes, 8 KB apart), so that every PV product still runs at
//   N = 256.  The TMA warp fills the slots in the order the MMA warp drains
//   them: K0, K1, V0, K2, V1, ..., V(n-1).  O leaves through direct 16-byte
//   stores from the epilogue warps (no staging box, to leave the ring its
//   room).
// * Warp roles: warps 0-3 the softmax (TMEM lane = row = thread), warps 4-7
//   the epilogue, warp 8 issues the MMAs (one thread: at this width the MMAs
//   are small against the cost of a warp-wide wait per slot, and clock
//   stamps showed the issuing warp, not the copies or the tensor core,
//   setting the pace), warp 9 the TMA loads.
// Every mbarrier wait is bounded as in the other tcgen05 kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

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
constexpr int kKC = 2;      // 64-column K chunks per ring slot
constexpr int kVKeys = 64;  // keys per V ring slot
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
constexpr uint32_t kVBoxBytes = kVKeys * 128;  // kVKeys keys x 64 columns
constexpr uint32_t kSlotBytes = kKC * kChunkBytes;
constexpr int kSlots = 3;
static_assert(4 * kVBoxBytes <= kSlotBytes, "a V slot holds four 64-column boxes");
constexpr int kMaxChunks = 8;  // 64-column chunks of a 512-wide Q tile
constexpr int kOCols = 256;    // O columns of a half

constexpr int Q_OFF = 0;
constexpr int RING_OFF = kMaxChunks * (int)kChunkBytes;
constexpr int STATS_OFF = RING_OFF + kSlots * (int)kSlotBytes;
constexpr int BAR_OFF = STATS_OFF + 2 * kBM * 4;
constexpr int SMEM = 1024 + BAR_OFF + 256;
constexpr int O_COL = 256;  // TMEM: S0 [0, 128), S1 [128, 256), O [256, 512)
static_assert(SMEM <= 227 * 1024, "shared memory budget");

enum : int {
    X_Q_FULL = 0,
    X_Q_EMPTY = 1,
    X_S_FULL = 2,   // [2] by S buffer
    X_P_READY = 4,  // [2]
    X_O_FULL = 6,
    X_O_EMPTY = 7,
    X_STATS = 8,  // [2] by unit parity
    X_TEARDOWN = 10,
    X_PV_DONE = 11,  // one phase per tile: its PV has completed
    X_FULL = 12,               // [kSlots]
    X_EMPTY = 12 + kSlots,     // [kSlots]
    X_NBARS = 12 + 2 * kSlots,
};
static_assert(8 * X_NBARS + 4 + 4 + 32 <= 256, "barrier area");

struct W512Args {
    AttnParams p;
    int Gp;            // heads packed into the rows of a Q tile
    int QP;            // query positions per Q tile (kBM / Gp)
    int nsub;          // head subgroups per KV head
    int nqblk;         // query blocks (QP positions) per sequence
    uint32_t per;      // Q tiles per query block: B * Hkv * nsub
    uint32_t hs;       // Hkv * nsub
    int nh;            // output halves (1 or 2): units = Q tiles x nh
    int dc;            // 64-column chunks of D
    long long nunits;
    float c_scale;       // |scale| * log2(e)
    uint32_t idesc_s;    // S = Q K^T (M 128, N 128)
    uint32_t idesc_o[2];  // O += P V (M 128, N = the half's columns)
    int vbox[2];          // 64-column V boxes of each half
    int ocols[2];         // output columns of each half
};

__device__ __forceinline__ QTileUnit unit_of(const W512Args &a, long long u, int &half) {
    const uint32_t uu = (uint32_t)u;
    const uint32_t t = a.nh == 2 ? uu >> 1 : uu;
    half = a.nh == 2 ? (int)(uu & 1u) : 0;
    return qtile_unit(a.p, a.per, a.hs, a.nsub, a.Gp, a.QP, a.nqblk, t);
}

__device__ __forceinline__ int tile_keys(int hi_unit, int kv_start, int j) {
    return min(kBN, hi_unit - (kv_start + j * kBN));
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide512_tc_kernel(const __grid_constant__ W512Args a,
                              const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t q_smem = base + Q_OFF;
    const uint32_t ring = base + RING_OFF;
    const uint32_t bars = base + BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + BAR_OFF + 8 * X_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *unit_desc = reinterpret_cast<int *>(tmem_slot + 2);  // [2 parities][4]

    const AttnParams &p = a.p;
    const uint64_t wl = p.wait_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool padded = p.cu_q == nullptr;

    if (threadIdx.x == 0) {
        mbar_init(bar(X_Q_FULL), 1);
        mbar_init(bar(X_Q_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(X_S_FULL + i), 1);
            mbar_init(bar(X_P_READY + i), 128);
            mbar_init(bar(X_STATS + i), 128);
        }
        mbar_init(bar(X_O_FULL), 1);
        mbar_init(bar(X_O_EMPTY), 128);
        mbar_init(bar(X_TEARDOWN), 1);
        mbar_init(bar(X_PV_DONE), 1);
        for (int e = 0; e < kSlots; ++e) {
            mbar_init(bar(X_FULL + e), 1);
            mbar_init(bar(X_EMPTY + e), 1);
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto full = [&](int s) { return bar(X_FULL + s); };
    auto empty = [&](int s) { return bar(X_EMPTY + s); };
    auto slot = [&](int s) { return ring + (uint32_t)s * kSlotBytes; };

    if (warp >= kMmaWarp) {
        regs_decrease<kRegsOther>();
        if (warp == kLoadWarp) {
            // --------------------------------------------------------- TMA producer
            if (lane == 0) {
                uint32_t it = 0, q_ph = 0;
                int last_q_parity = -1;
                uint32_t armed = 0, armed_parity = 0;
                bool ok = true;
                // the next ring slot, once the MMAs that read it have completed
                auto take = [&](int &s) -> bool {
                    const uint32_t i = it++;
                    s = (int)(i % kSlots);
                    const uint32_t ph = (i / kSlots) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, wl)) {
                        raise_abort(abort_flag, p.status, kStatusTimeoutKvEmpty);
                        return false;
                    }
                    armed |= 1u << s;
                    armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                    return true;
                };
                for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
                    const long long u = snake(rnd, blockIdx.x, gridDim.x);
                    if (u >= a.nunits) continue;
                    int half;
                    const QTileUnit x = unit_of(a, u, half);
                    if (x.n_kv == 0) continue;
                    const int qrow = (padded ? 0 : (int)x.si.q_off) + x.q0;
                    const int krow = padded ? 0 : (int)x.si.k_off;
                    const int bc = padded ? x.b : 0;
                    const int vcol = half * kOCols, nbox = a.vbox[half];
                    if (!mbar_wait(bar(X_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                        ok = false;
                        break;
                    }
                    int *d = unit_desc + q_ph * 4;
                    d[0] = x.n_kv;
                    d[1] = x.kv_start;
                    d[2] = x.hi_unit;
                    d[3] = half;
                    mbar_arrive_expect_tx(bar(X_Q_FULL), (uint32_t)a.dc * kChunkBytes);
                    last_q_parity = (int)q_ph;
                    q_ph ^= 1u;
                    for (int c = 0; c < a.dc; ++c)
                        tma_load_4d(q_smem + c * kChunkBytes, &tmQ, bar(X_Q_FULL), c * 64, x.h0,
                                    qrow, bc);
                    auto load_k = [&](int j) -> bool {
                        const int kr = krow + x.kv_start + j * kBN;
                        for (int c0 = 0; c0 < a.dc; c0 += kKC) {
                            const int nc = min(kKC, a.dc - c0);
                            int s;
                            if (!take(s)) return false;
                            mbar_arrive_expect_tx(full(s), (uint32_t)nc * kChunkBytes);
                            for (int cc = 0; cc < nc; ++cc)
                                tma_load_4d(slot(s) + cc * kChunkBytes, &tmK, full(s),
                                            (c0 + cc) * 64, x.kvh, kr, bc);
                        }
                        return true;
                    };
                    auto load_v = [&](int j) -> bool {
                        const int kr = krow + x.kv_start + j * kBN;
                        const int nvc = (tile_keys(x.hi_unit, x.kv_start, j) + kVKeys - 1) / kVKeys;
                        for (int c = 0; c < nvc; ++c) {
                            int s;
                            if (!take(s)) return false;
                            mbar_arrive_expect_tx(full(s), (uint32_t)nbox * kVBoxBytes);
                            for (int bx = 0; bx < nbox; ++bx)
                                tma_load_4d(slot(s) + bx * kVBoxBytes, &tmV, full(s),
                                            vcol + bx * 64, x.kvh, kr + c * kVKeys, bc);
                        }
                        return true;
                    };
                    ok = load_k(0);
                    if (ok && x.n_kv > 1) ok = load_k(1);
                    for (int j = 0; j < x.n_kv && ok; ++j) {
                        ok = load_v(j);
                        if (ok && j + 2 < x.n_kv) ok = load_k(j + 2);
                    }
                }
                if (ok) {  // end marker, once the last Q tile has been consumed
                    if (mbar_wait(bar(X_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        unit_desc[q_ph * 4] = 0;
                        mbar_arrive(bar(X_Q_FULL));
                        last_q_parity = -1;
                    } else {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                    }
                }
                // drain: the copies always land, so these ignore the abort flag
                if (last_q_parity >= 0) mbar_wait_drain(bar(X_Q_FULL), (uint32_t)last_q_parity);
                for (int s = 0; s < kSlots; ++s)
                    if (armed & (1u << s)) mbar_wait_drain(full(s), (armed_parity >> s) & 1u);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // One thread runs the whole loop: it waits, issues and commits
            // (per-slot warp-wide waits and reconvergence cost more than the
            // MMAs of a slot take to issue).
            if (lane == 0) {
                uint32_t it = 0, q_ph = 0, o_ph = 0;
                uint32_t gt = 0;     // tiles issued so far, all units: S buffer gt & 1
                uint32_t p_par = 0;  // bit b: parity of P_READY[b]'s next phase
                bool ok = true;
                const uint64_t qd = sw128_desc(q_smem, 16, 1024);
                const uint32_t o_tm = tmem + (uint32_t)O_COL;
                // the next ring slot, once its copy has landed
                auto take = [&](int &s) -> bool {
                    const uint32_t i = it++;
                    s = (int)(i % kSlots);
                    return mbar_wait(full(s), (i / kSlots) & 1u, abort_flag, wl);
                };
                while (ok) {
                    if (!mbar_wait(bar(X_Q_FULL), q_ph, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    const volatile int *d = unit_desc + q_ph * 4;
                    q_ph ^= 1u;
                    const int n = d[0], kv_start = d[1], hi_unit = d[2], half = d[3];
                    if (n == 0) break;  // end marker
                    const uint32_t g0 = gt;
                    const uint32_t idesc_o = a.idesc_o[half];
                    const int nbox = a.vbox[half];
                    // S(j) = Q K_j^T into buffer (g0 + j) & 1, kKC 64-column chunks
                    // of K a ring slot
                    auto issue_s = [&](int j) -> bool {
                        const int nvalid = tile_keys(hi_unit, kv_start, j);
                        const uint32_t ncols = (uint32_t)((nvalid + 15) & ~15);
                        const uint32_t idesc =
                            (a.idesc_s & ~(0x3Fu << 17)) | ((ncols >> 3) << 17);
                        const uint32_t sb = (g0 + (uint32_t)j) & 1u;
                        const uint32_t s_tm = tmem + sb * 128u;
                        for (int c0 = 0; c0 < a.dc; c0 += kKC) {
                            int s;
                            if (!take(s)) return false;
                            tc_fence_after();
                            const uint64_t kd = sw128_desc(slot(s), 16, 1024);
#pragma unroll
                            for (int cc = 0; cc < kKC; ++cc) {
                                if (c0 + cc < a.dc) {
                                    const uint64_t qc = qd + (((c0 + cc) * kChunkBytes) >> 4);
                                    const uint64_t kc = kd + ((cc * kChunkBytes) >> 4);
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        mma_ss(s_tm, qc + ((kk * 32) >> 4), kc + ((kk * 32) >> 4),
                                               idesc, (c0 + cc > 0 || kk > 0) ? 1u : 0u);
                                }
                            }
                            mma_commit(empty(s));
                        }
                        mma_commit(bar(X_S_FULL + (int)sb));
                        if (j == n - 1) mma_commit(bar(X_Q_EMPTY));
                        return true;
                    };
                    if (!issue_s(0) || (n > 1 && !issue_s(1))) {
                        ok = false;
                        break;
                    }
                    for (int j = 0; j < n && ok; ++j) {
                        // keys past the last one in use (last tile only) are left out
                        // 16 at a time; the V rows of the last 16-key step past it
                        // are zeroed (they may hold NaN) so that 0 * V stays 0
                        const int nvalid = tile_keys(hi_unit, kv_start, j);
                        const int ksteps = (nvalid + 15) / 16;
                        const int nvc = (nvalid + kVKeys - 1) / kVKeys;
                        if (j == 0) {  // the epilogue has read the previous unit's O
                            if (!mbar_wait(bar(X_O_EMPTY), o_ph ^ 1u, abort_flag, wl)) {
                                ok = false;
                                break;
                            }
                            o_ph ^= 1u;
                        }
                        const uint32_t sb = (g0 + (uint32_t)j) & 1u;
                        if (!mbar_wait(bar(X_P_READY + (int)sb), (p_par >> sb) & 1u, abort_flag,
                                       wl)) {
                            ok = false;
                            break;
                        }
                        p_par ^= 1u << sb;
                        const uint32_t s_tm = tmem + sb * 128u;
                        for (int c = 0; c < nvc && ok; ++c) {
                            int s;
                            if (!take(s)) {
                                ok = false;
                                break;
                            }
                            // rows [nvalid, 16 * ksteps) of the tile, local to this slot
                            const int z0 = nvalid - c * kVKeys, z1 = ksteps * 16 - c * kVKeys;
                            if (z0 < z1 && z0 < kVKeys) {
                                uint8_t *vt = gbase + (slot(s) - base);
                                const int nz = (min(z1, kVKeys) - z0) * 8;  // 16 B units a box
                                for (int bx = 0; bx < nbox; ++bx)
                                    for (int i = 0; i < nz; ++i)
                                        *reinterpret_cast<uint4 *>(vt + bx * kVBoxBytes +
                                                                   z0 * 128 + i * 16) =
                                            make_uint4(0, 0, 0, 0);
                                fence_proxy_async_smem();
                            }
                            tc_fence_after();
                            // O (+)= P V over kVKeys keys: P from TMEM over S, V MN-major
                            // (64-column boxes kVBoxBytes apart), N = the half's columns
                            const uint64_t vd = sw128_desc(slot(s), kVBoxBytes, 1024);
#pragma unroll
                            for (int h = 0; h < kVKeys / 16; ++h) {
                                const int kk = c * (kVKeys / 16) + h;
                                if (kk < ksteps)
                                    mma_ts(o_tm, s_tm + kk * 8, vd + ((h * 2048) >> 4), idesc_o,
                                           (j > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_commit(empty(s));
                        }
                        if (!ok) break;
                        mma_commit(bar(X_PV_DONE));
                        // S(j + 2) reuses S_j's buffer: issued after PV(j)
                        if (j + 2 < n && !issue_s(j + 2)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    mma_commit(bar(X_O_FULL));
                    gt += (uint32_t)n;
                }
                if (!ok) raise_abort(abort_flag, p.status, kStatusTimeoutMma);
                // every MMA issued completes before TMEM is freed
                mma_commit(bar(X_TEARDOWN));
                mbar_wait_drain(bar(X_TEARDOWN), 0);
            }
            __syncwarp();
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------- softmax
        regs_increase<kRegsSoftmax>();
        const int r = warp * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tO = tmem + lane_off + (uint32_t)O_COL;
        const float c = a.c_scale;
        uint32_t gt = 0, s_par = 0, nunit = 0;  // s_par bit b: S_FULL[b]'s next parity
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        float *inv_l = reinterpret_cast<float *>(gbase + STATS_OFF);
        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            int half;
            const QTileUnit x = unit_of(a, u, half);
            const int qpos = x.q0 + r / a.Gp;
            const int head = x.h0 + r % a.Gp;
            const bool valid = qpos < x.si.Qb;
            const bool writes = padded ? qpos < p.Q : valid;
            int lo = 0, hi = 0;
            if (valid) legal_range(qpos, x.si.Qb, x.si.Kb, p.window, p.mask, lo, hi);
            const long long orow = (x.si.q_off + qpos) * p.Hq + head;
            if (x.n_kv == 0) {  // nothing to attend: +0 and -inf (LSE from half 0)
                if (writes) {
                    uint4 *dst = reinterpret_cast<uint4 *>(og + orow * p.Dv + half * kOCols);
                    for (int i = 0; i < a.ocols[half] * 2 / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (p.lse && half == 0) p.lse[orow] = -INFINITY;
                }
                continue;
            }
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < x.n_kv && ok; ++j) {
                const uint32_t sb = gt & 1u;
                ++gt;
                if (!warp_wait(bar(X_S_FULL + (int)sb), (s_par >> sb) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                s_par ^= 1u << sb;
                tc_fence_after();
                const uint32_t tS = tmem + lane_off + sb * 128u;
                const int k0 = x.kv_start + j * kBN;
                const bool interior = x.all_valid && k0 >= x.lo_last && k0 + kBN <= x.hi_first;
                // a rescale first waits for PV(j - 1): its phase of X_PV_DONE
                if (!softmax_tile<T, kOCols>(tS, tO, k0, interior, lo, hi, c, m_run, l_run,
                                             bar(X_PV_DONE), (gt - 2u) & 1u, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(bar(X_P_READY + (int)sb));
            }
            if (!ok) break;
            const bool has = valid && l_run > 0.f;
            if (writes && p.lse && half == 0)
                p.lse[orow] = has ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
            inv_l[(nunit & 1u) * kBM + r] = has ? 1.f / l_run : 0.f;
            mbar_arrive(bar(X_STATS + (int)(nunit & 1u)));
            ++nunit;
        }
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutSoftmax);
    } else {
        // ------------------------------------------------------------ epilogue
        regs_decrease<kRegsEpi>();
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t o_ph = 0, st_par = 0, nunit = 0;  // st_par bit b: STATS[b]'s next parity
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        const float *inv_l = reinterpret_cast<const float *>(gbase + STATS_OFF);
        const uint32_t tO = tmem + lane_off + (uint32_t)O_COL;
        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            int half;
            const QTileUnit x = unit_of(a, u, half);
            if (x.n_kv == 0) continue;  // the softmax warps wrote those rows
            const int b = (int)(nunit & 1u);
            ++nunit;
            const bool got = warp_wait(bar(X_O_FULL), o_ph, abort_flag, wl) &&
                             warp_wait(bar(X_STATS + b), (st_par >> b) & 1u, abort_flag, wl);
            if (!got) {
                ok = false;
                break;
            }
            o_ph ^= 1u;
            st_par ^= 1u << b;
            tc_fence_after();
            const float inv = inv_l[b * kBM + r];
            const int qpos = x.q0 + r / a.Gp;
            const bool writes = padded ? qpos < p.Q : qpos < x.si.Qb;
            const long long orow = (x.si.q_off + qpos) * p.Hq + x.h0 + r % a.Gp;
            T *dst = og + orow * p.Dv + half * kOCols;
            const int ncol = a.ocols[half];
            const int nld = (ncol + 31) / 32;
            for (int cc = 0; cc < nld; ++cc) {
                uint32_t ov[32];
                tmem_ld32(tO + cc * 32, ov);
                tmem_ld_wait();
                if (cc == nld - 1) {  // O is read: free it
                    tc_fence_before();
                    mbar_arrive(bar(X_O_EMPTY));
                }
                if (writes) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        if (cc * 32 + c4 * 8 < ncol) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int e = 8 * c4 + 2 * i;
                                w[i] = pack2<T>(inv > 0.f ? __uint_as_float(ov[e]) * inv : 0.f,
                                                inv > 0.f ? __uint_as_float(ov[e + 1]) * inv : 0.f);
                            }
                            *reinterpret_cast<uint4 *>(dst + cc * 32 + c4 * 8) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutEpilogue);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int pack_factor512(int G) {
    int gp = 1;
    while (gp < 16 && G % (gp * 2) == 0) gp *= 2;
    return gp;
}

template <typename T>
int launch_t(const AttnParams &p, bool bf16, cudaStream_t stream) {
    W512Args a;
    a.p = p;
    a.Gp = pack_factor512(p.G);
    a.QP = kBM / a.Gp;
    a.nsub = p.G / a.Gp;
    a.nqblk = (p.Q + a.QP - 1) / a.QP;
    a.nh = p.Dv > kOCols ? 2 : 1;
    a.dc = (p.D + 63) / 64;
    a.nunits = (long long)a.nqblk * p.B * p.Hkv * a.nsub * a.nh;
    a.per = (uint32_t)((long long)p.B * p.Hkv * a.nsub);
    a.hs = (uint32_t)(p.Hkv * a.nsub);
    const float sc = p.scale == 0.f ? 1e-30f : fabsf(p.scale);
    a.c_scale = sc * kLog2e;
    a.idesc_s = idesc_f16(bf16, kBM, kBN, false, p.scale < 0.f);
    for (int h = 0; h < 2; ++h) {
        const int w = h < a.nh ? (p.Dv - h * kOCols < kOCols ? p.Dv - h * kOCols : kOCols) : 16;
        a.ocols[h] = w;
        a.vbox[h] = (w + 63) / 64;
        a.idesc_o[h] = idesc_f16(bf16, kBM, w, true, false);  // w: a multiple of 16
    }
    if (a.nunits == 0) return 0;
    const bool padded = p.cu_q == nullptr;
    const uint64_t qrows = padded ? (uint64_t)p.Q : (uint64_t)p.Tq;
    const uint64_t krows = padded ? (uint64_t)p.K : (uint64_t)p.Tk;
    const uint64_t nb = padded ? (uint64_t)p.B : 1;
    CUtensorMap tq, tk, tv;
    int rc = make_tma_map_4d(&tq, p.q, bf16, (uint64_t)p.D, p.Hq, qrows, nb, a.Gp, a.QP);
    if (rc) return rc;
    if (krows > 0) {
        rc = make_tma_map_4d(&tk, p.k, bf16, (uint64_t)p.D, p.Hkv, krows, nb, 1, kBN);
        if (!rc) rc = make_tma_map_4d(&tv, p.v, bf16, (uint64_t)p.Dv, p.Hkv, krows, nb, 1, kVKeys);
        if (rc) return rc;
    } else {
        tk = tq;  // never read: every unit has no key
        tv = tq;
    }
    auto kern = prefill_wide512_tc_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) {
        set_error("512-wide prefill kernel: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    const int nsm = sm_count(dev);
    const long long grid = a.nunits < nsm ? a.nunits : nsm;
    kern<<<(unsigned)grid, kThreads, SMEM, stream>>>(a, tq, tk, tv);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("512-wide prefill kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

}  // namespace

bool prefill_wide512_tc_supported(const AttnParams &p, int dtype) {
    if (dtype != 1 && dtype != 2) return false;
    if (p.D < 64 || p.D > 512 || p.D % 16 || p.Dv < 64 || p.Dv > 512 || p.Dv % 16) return false;
    if (p.D <= 256 && p.Dv <= 256) return false;  // the 256-wide kernel's widths
    if (p.Q < 1 || p.block_table != nullptr || p.mask_bits != nullptr) return false;
    const long long rows = p.cu_q ? p.Tq : (long long)p.Q;
    const long long keys = p.cu_q ? p.Tk : (long long)p.K;
    const int gp = pack_factor512(p.G), qp = kBM / gp;
    const long long nunits =
        (long long)((p.Q + qp - 1) / qp) * p.B * p.Hkv * (p.G / gp) * (p.Dv > kOCols ? 2 : 1);
    return rows < (1LL << 31) && keys < (1LL << 31) && nunits < (1LL << 31);
}

int launch_prefill_wide512_tc(const AttnParams &p, int dtype, cudaStream_t stream) {
    if (dtype == 2) return launch_t<__nv_bfloat16>(p, true, stream);
    return launch_t<__half>(p, false, stream);
}

}  // namespace attn
