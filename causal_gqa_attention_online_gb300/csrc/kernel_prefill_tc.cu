// kernel_prefill_tc.cu -- bf16 / fp16 causal GQA prefill on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-fed shared memory), sm_103a.
//
// What it computes is the online-softmax program of "Attention execution
// mapping" (LuisaCompute), sections 1-2: per KV block QK^T -> mask -> max ->
// exp -> sum -> alpha-rescale -> PV, with the row max / row sum / accumulator
// carried across blocks.  How it runs it is GB300-specific:
//
// * Persistent CTAs, one per SM, walk work units (sequence, KV head, head
//   subgroup, query block) in longest-first order (bottom-right causal: the
//   last query blocks see the most keys), in rounds that alternate direction
//   across the CTAs so that the total work per CTA evens out.
// * A unit holds two Q tiles of 128 rows.  The rows of a tile are
//   (query position, head) pairs with up to 16 heads of one KV group packed
//   together, so every K/V tile brought in by TMA serves all of those heads
//   (the cross-head KV reuse of the same page, section 5).
// * Warp roles: warps 0-3 and 4-7 are the softmax warpgroups of Q tile 0 and
//   Q tile 1 (TMEM lane = row = thread); warps 8 and 9 issue the tcgen05.mma
//   of Q tile 0 and Q tile 1 (one thread each: a single issuing thread leaves
//   the tensor core idle whenever it waits on a dependency, two keep it fed);
//   warp 10 issues TMA loads from one thread; warp 11 idles; warps 12-15
//   are the epilogue warpgroup, which takes each finished O_t out of TMEM,
//   normalises it by the row sums the softmax warpgroup handed over through
//   shared memory, frees O_t for the next unit as soon as it is read, and
//   writes it out with TMA stores -- so the softmax warpgroups go straight on
//   to the next unit and the tensor core to its first PV.
// * TMEM (512 columns): S0 | S1 | O0 | O1.  S_t = Q_t K^T accumulates in fp32;
//   the softmax writes P_t as bf16/fp16 pairs over the first half of S_t and
//   the PV MMA reads P_t straight from TMEM (A operand in TMEM, V from shared
//   memory as an MN-major operand).  While one warpgroup runs its softmax the
//   tensor core works on the other tile (the dual-pipeline idea of the FlyDSL
//   FMHA forward on the "Accelerating PyTorch on AMD GPUs with FlyDSL" page,
//   rebuilt around TMEM and an MMA-issuing warp).
// * K/V tiles stream through a ring of shared-memory stages with
//   full/empty mbarriers; Q tiles are reloaded per unit.
// * The O rescale by alpha = exp2(m_old - m_new) is skipped unless the row
//   max grows by more than 2^8: the stale max is kept and the final
//   normalisation uses the same reference, so the result is unchanged.
// * Every mbarrier wait is bounded; a wait that runs out records a status,
//   raises an abort flag, and the CTA drains its copies and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_softmax.cuh"

namespace attn {
namespace {

using namespace sm100;
using namespace tcfwd;

constexpr int kBM = 128;  // rows per Q tile (MMA M)
constexpr int kBN = 128;  // keys per KV tile
// Four warpgroups: two softmax warpgroups, one for the MMA warps, the TMA
// warp and an idle warp, and the epilogue warpgroup.  Launched at 128
// registers a thread (512 x 128 = 65536, the whole register file); the
// softmax warpgroups take 192 and the other two give back down to 64:
// 256 x 192 + 256 x 64 = 65536, and per SM sub-partition (one warp of each
// warpgroup) 2 x 192 + 2 x 64 = 512 register slots a lane.
constexpr int kThreads = 512;
constexpr int kMmaWarp0 = 8;  // issues the MMAs of Q tile 0; owns the TMEM allocation
constexpr int kMmaWarp1 = 9;  // issues the MMAs of Q tile 1
constexpr int kLoadWarp = 10;
constexpr int kEpiWarp0 = 12;  // warps 12-15: epilogue
constexpr uint32_t kRegsLaunch = 65536 / kThreads;
constexpr uint32_t kRegsSoftmax = 192;
constexpr uint32_t kRegsOther = 56;  // MMA, TMA and idle warps
constexpr uint32_t kRegsEpi = 72;    // epilogue warpgroup
static_assert(256 * kRegsSoftmax + 128 * (kRegsOther + kRegsEpi) <= kThreads * kRegsLaunch,
              "register split");
static_assert(2 * kRegsSoftmax + kRegsOther + kRegsEpi <= 512, "register split per sub-partition");
constexpr uint32_t kChunkBytes = 128 * 128;       // one 128-row x 128-byte swizzled chunk
constexpr int kPrefetchTiles = 4;                 // K/V tiles pulled into L2 ahead of use
// Where the two softmax warpgroups take turns: 0 = never, 1 = the whole
// softmax of a tile (the turn passes when P is stored), 2 = only its exp
// phase, 3 = the whole softmax, the turn passing as soon as the exps of the
// tile are issued (the P store wait and arrival overlap the next group).
constexpr int kTurnMode = 1;

struct PrefillArgs {
    AttnParams p;
    int Gp;            // heads packed into the rows of a Q tile
    int QP;            // query positions per Q tile (kBM / Gp)
    int nsub;          // head subgroups per KV head (G / Gp)
    int nqblk;         // query blocks (2 * QP positions) per sequence
    uint32_t per;      // units per query block: B * Hkv * nsub
    uint32_t hs;       // Hkv * nsub
    long long nunits;  // < 2^31
    float c_scale;     // |scale| * log2(e)  (> 0)
    uint32_t idesc_s;  // S = Q K^T
    uint32_t idesc_o;  // O += P V
    // Ragged problems: the unit indices ordered by their KV tile count, most
    // first (written by unit_order_kernel); null: the natural order, which is
    // longest-first already when every sequence has the same lengths.
    const int *order;
    // Arbitrary mask: live[row * live_tiles + T] is 0 when no row of the unit
    // may attend to a key of 128-key tile T (a dead tile: neither loaded nor
    // multiplied), 2 when every real row may attend to all of its keys (the
    // mask bits need not be read), 1 otherwise (written by mask_summary_kernel);
    // a row is one (sequence, query block) when the mask is shared by all
    // heads, else one unit (its natural index).
    const uint8_t *live;
    int live_tiles;   // ceil(K / 128)
    int live_shared;  // 1: the mask is shared by all heads
};

template <int D, int DV> struct Layout {
    static constexpr int QTILE = kBM * D * 2;
    static constexpr int KTILE = kBN * D * 2;
    static constexpr int VTILE = kBN * DV * 2;
    static constexpr int STAGE = KTILE > VTILE ? KTILE : VTILE;
    static constexpr int BUDGET = 227 * 1024;  // opt-in shared memory per block
    static constexpr int STG_BYTES = kBM * 128;  // epilogue staging: 64 columns of a Q tile
    static constexpr int STATS_BYTES = 2 * 2 * kBM * 4;  // 1 / l per row: [unit parity][tile]
    static constexpr int NS_FIT = (BUDGET - 2 * QTILE - STG_BYTES - STATS_BYTES - 1024 - 512) / STAGE;
    static constexpr int NS = NS_FIT > 8 ? 8 : NS_FIT;
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = 2 * QTILE;
    static constexpr int STG_OFF = KV_OFF + NS * STAGE;
    static constexpr int STATS_OFF = STG_OFF + STG_BYTES;
    static constexpr int BAR_OFF = STATS_OFF + STATS_BYTES;
    static constexpr int SMEM = 1024 + BAR_OFF + 512;  // + alignment slack
    static constexpr int O_COL = 256;                  // TMEM columns: S0 S1 | O0 O1
    static_assert(NS >= 2, "K/V ring needs two stages");
    static_assert(O_COL + 2 * DV <= 512, "TMEM budget");
};

// Barrier slots (8 bytes each) after the K/V ring.
enum : int {
    B_Q_FULL = 0,
    B_Q_EMPTY = 1,
    B_S_FULL = 2,    // [2]
    B_P_READY = 4,   // [2]
    B_O_FULL = 6,    // [2]
    B_O_EMPTY = 8,   // [2]
    B_TEARDOWN = 10,  // [2]
    B_TURN = 12,      // [2] softmax group t has issued the exps of its tile
    B_STATS = 14,     // [2 tiles][2 unit parities]: the 1 / l of tile t's rows are in
                      // shared memory.  One barrier per unit parity, so that none runs
                      // more than one phase ahead of the epilogue (a unit's stats can
                      // only be written once the epilogue has freed O of the unit two
                      // back)
    B_KV_FULL = 18,   // [NS] kv_full, [NS] kv_empty, [NS] v_tail: the zeroed tail V
                      // tile of a ring slot, handed from MMA warp 0 to MMA warp 1
                      // (a slot is refilled only after both warps released it, so
                      // its v_tail barrier is never more than one phase ahead)
};

struct UnitInfo {
    int b, kvh, h0, q0;  // first head of the packed subgroup, first query position
    SeqInfo si;
    int n_kv;            // KV tiles
    int kv_start;        // first key of tile 0
    int lo_last, hi_first;  // interior test: all rows legal on [lo_last, hi_first)
    int hi_unit;         // one past the last key any row uses
    bool all_valid;      // every row of both tiles holds a real query
    uint32_t u;          // natural unit index
};

// Kernel modes: 0 the plain layouts, 1 paged K/V, 2 an arbitrary mask.
template <int MODE>
__device__ __forceinline__ UnitInfo unit_info(const PrefillArgs &a, long long u64) {
    const AttnParams &p = a.p;
    // 32-bit index arithmetic (the unit count is below 2^31)
    const uint32_t u = a.order != nullptr ? (uint32_t)__ldg(a.order + u64) : (uint32_t)u64;
    const uint32_t qi = u / a.per, rest = u - qi * a.per;
    const uint32_t b = rest / a.hs, r2 = rest - b * a.hs;
    const uint32_t kvh = r2 / (uint32_t)a.nsub, sub = r2 - kvh * (uint32_t)a.nsub;
    const int qblk = a.nqblk - 1 - (int)qi;
    UnitInfo x;
    x.u = u;
    x.b = (int)b;
    x.kvh = (int)kvh;
    x.h0 = x.kvh * p.G + (int)sub * a.Gp;
    x.q0 = qblk * 2 * a.QP;
    x.si = seq_info(p, x.b);
    x.n_kv = 0;
    x.kv_start = 0;
    x.lo_last = INT_MAX;
    x.hi_first = INT_MIN;
    x.hi_unit = 0;
    x.all_valid = false;
    if (x.q0 >= x.si.Qb) return x;
    const int q_last = min(x.q0 + 2 * a.QP, x.si.Qb) - 1;
    int lo_f, hi_f, lo_l, hi_l;
    legal_range(x.q0, x.si.Qb, x.si.Kb, p.window, p.mask, lo_f, hi_f);
    legal_range(q_last, x.si.Qb, x.si.Kb, p.window, p.mask, lo_l, hi_l);
    if (hi_l <= lo_f) return x;
    // paged K/V and an arbitrary mask: tiles start on 128-key boundaries, so
    // that each lies in one page, or covers four whole words of a mask row
    // (the keys before lo_f are masked)
    x.kv_start = MODE != 0 ? (lo_f & ~(kBN - 1)) : lo_f;
    x.hi_unit = hi_l;
    x.n_kv = (hi_l - x.kv_start + kBN - 1) / kBN;
    x.lo_last = lo_l;
    x.hi_first = hi_f;
    x.all_valid = x.q0 + 2 * a.QP <= x.si.Qb;
    return x;
}

// Unit processed by CTA c in round r: rounds alternate direction over the
// longest-first unit order (c, then G-1-c, ...), so every CTA gets a mix of
// long and short units (a plain stride leaves CTA 0 with the longest of every
// round).
__device__ __forceinline__ long long snake_unit(long long r, int c, int G) {
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// Arbitrary mask: the live flags of the unit's tiles (tile j of the unit is
// entry j), and how many are live (*last: the last live one).
__device__ __forceinline__ const uint8_t *live_row(const PrefillArgs &a, const UnitInfo &x) {
    const long long row =
        a.live_shared ? (long long)x.b * a.nqblk + x.q0 / (2 * a.QP) : (long long)x.u;
    return a.live + row * a.live_tiles + x.kv_start / kBN;
}
__device__ __forceinline__ int count_live(const uint8_t *lv, int n_kv, int *last) {
    int n = 0;
    *last = -1;
    for (int j = 0; j < n_kv; ++j)
        if (lv[j] != 0) {
            ++n;
            *last = j;
        }
    return n;
}

// D, DV: the tile widths (64 or 128 columns); the real head dims p.D <= D and
// p.Dv <= DV are multiples of 16, the rest of the tile columns zero-filled.
// MODE: 0 the plain layouts; 1 K / V tiles found through the block table; 2 an
// arbitrary mask (dead tiles skipped, live ones masked bit by bit).  Separate
// instances, so that the plain one carries none of the others' code.
template <typename T, int D, int DV, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmO) {
    using L = Layout<D, DV>;
    constexpr int NS = L::NS;
    constexpr bool PAGED = MODE == 1;
    constexpr bool MASKED = MODE == 2;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzle atoms
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t q_smem = base + L::Q_OFF;
    const uint32_t kv_smem = base + L::KV_OFF;
    const uint32_t bars = base + L::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::BAR_OFF + 8 * (B_KV_FULL + 3 * NS));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // per Q load, for the MMA warps: {KV tiles, first key, end of keys in use}
    // of the unit (two slots by load parity; KV tiles 0 = no more units)
    int *unit_desc = reinterpret_cast<int *>(tmem_slot + 2);

    const AttnParams &p = a.p;
    const uint64_t wl = p.wait_ns;  // limit of every wait but the drains
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_EMPTY), 2);  // one commit from each MMA warp
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_S_FULL + t), 1);
            mbar_init(bar(B_P_READY + t), 128);
            mbar_init(bar(B_O_FULL + t), 1);
            mbar_init(bar(B_O_EMPTY + t), 128);
            mbar_init(bar(B_TURN + t), 128);
            mbar_init(bar(B_STATS + 2 * t), 128);
            mbar_init(bar(B_STATS + 2 * t + 1), 128);
        }
        mbar_init(bar(B_TEARDOWN), 1);
        mbar_init(bar(B_TEARDOWN + 1), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_FULL + NS + s), 2);  // kv_empty: one commit per MMA warp
            mbar_init(bar(B_KV_FULL + 2 * NS + s), 1);  // v_tail
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp0) {
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
    // launched as a programmatic dependent of unit_order_kernel: the unit
    // order is complete and visible once this returns
    if (a.order != nullptr || a.live != nullptr) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    auto kv_full = [&](int s) { return bar(B_KV_FULL + s); };
    auto kv_empty = [&](int s) { return bar(B_KV_FULL + NS + s); };
    auto v_tail = [&](int s) { return bar(B_KV_FULL + 2 * NS + s); };
    auto stage = [&](int s) { return kv_smem + (uint32_t)s * L::STAGE; };
    const bool padded = p.cu_q == nullptr;

    if (warp >= 8 && warp < kEpiWarp0) {
        // the setmaxnreg of each role dominates that role's code, so that the
        // compiler allocates the role's registers against its own limit
        regs_decrease<kRegsOther>();
        if (warp == kLoadWarp) {
            // ------------------------------------------------------ TMA producer
            if (lane == 0) {
                uint32_t kv_it = 0, q_ph = 0;
                int last_q_parity = -1;
                uint32_t armed = 0, armed_parity = 0;  // per ring slot: loaded at least once, last parity
                bool ok = true;
                for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
                    const long long u = snake_unit(rnd, blockIdx.x, gridDim.x);
                    if (u >= a.nunits) continue;
                    const UnitInfo x = unit_info<MODE>(a, u);
                    if (x.n_kv == 0) continue;
                    // an arbitrary mask: only the live tiles are loaded and multiplied;
                    // the MMA warps see n_use tiles and a first key placed so that
                    // the last one they process starts at the last live tile
                    const uint8_t *lv = MASKED ? live_row(a, x) : nullptr;
                    int n_use = x.n_kv, j_last = x.n_kv - 1;
                    if (MASKED) {
                        n_use = count_live(lv, x.n_kv, &j_last);
                        if (n_use == 0) continue;
                    }
                    const int qrow = (padded ? 0 : (int)x.si.q_off) + x.q0;
                    const int krow = padded ? 0 : (int)x.si.k_off;
                    const int bc = padded ? x.b : 0;
                    // K/V tile coordinates: (row, batch) of key k0 of the unit's sequence
                    const int kbc = PAGED ? 0 : bc;
                    auto kv_coord = [&](int k0) -> int {
                        return PAGED ? (int)kv_row(p, x.si, x.b, k0) : krow + k0;
                    };
                    if (!mbar_wait(bar(B_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                        ok = false;
                        break;
                    }
                    int *d = unit_desc + q_ph * 4;  // slot by the parity of this Q_FULL phase
                    d[0] = n_use;
                    d[1] = x.kv_start + (j_last - (n_use - 1)) * kBN;
                    d[2] = x.hi_unit;
                    mbar_arrive_expect_tx(bar(B_Q_FULL), 2 * L::QTILE);
                    last_q_parity = (int)q_ph;
                    q_ph ^= 1u;
                    for (int t = 0; t < 2; ++t)
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(q_smem + t * L::QTILE + c * kChunkBytes, &tmQ, bar(B_Q_FULL),
                                        c * 64, x.h0, qrow + t * a.QP, bc);
                    // L2 prefetch: the first K/V tiles of this unit and the next unit's Q
                    auto prefetch_kv = [&](int jj) {
                        const int kk0 = x.kv_start + jj * kBN;
                        const int kr = kv_coord(kk0);
                        for (int c = 0; c < D / 64; ++c)
                            tma_prefetch_l2_4d(&tmK, c * 64, x.kvh, kr, kbc);
                        for (int c = 0; c < DV / 64; ++c)
                            tma_prefetch_l2_4d(&tmV, c * 64, x.kvh, kr, kbc);
                    };
                    for (int jj = 1; jj < kPrefetchTiles && jj < x.n_kv; ++jj)
                        if (!MASKED || lv[jj] != 0) prefetch_kv(jj);
                    const long long un = snake_unit(rnd + 1, blockIdx.x, gridDim.x);
                    if (un < a.nunits) {
                        const UnitInfo nx = unit_info<MODE>(a, un);
                        if (nx.n_kv > 0) {
                            const int nq = (padded ? 0 : (int)nx.si.q_off) + nx.q0;
                            const int nbc = padded ? nx.b : 0;
                            for (int t = 0; t < 2; ++t)
                                for (int c = 0; c < D / 64; ++c)
                                    tma_prefetch_l2_4d(&tmQ, c * 64, nx.h0, nq + t * a.QP, nbc);
                        }
                    }
                    for (int j = 0; j < x.n_kv && ok; ++j) {
                        if (MASKED && lv[j] == 0) continue;
                        const int kr = kv_coord(x.kv_start + j * kBN);
                        if (j + kPrefetchTiles < x.n_kv && (!MASKED || lv[j + kPrefetchTiles] != 0))
                            prefetch_kv(j + kPrefetchTiles);
#pragma unroll
                        for (int which = 0; which < 2; ++which) {
                            const uint32_t it = kv_it++;
                            const int s = (int)(it % NS);
                            const uint32_t ph = (it / NS) & 1u;
                            if (!mbar_wait(kv_empty(s), ph ^ 1u, abort_flag, wl)) {
                                raise_abort(abort_flag, p.status, kStatusTimeoutKvEmpty);
                                ok = false;
                                break;
                            }
                            if (which == 0) {
                                mbar_arrive_expect_tx(kv_full(s), L::KTILE);
                                for (int c = 0; c < D / 64; ++c)
                                    tma_load_4d(stage(s) + c * kChunkBytes, &tmK, kv_full(s), c * 64,
                                                x.kvh, kr, kbc);
                            } else {
                                mbar_arrive_expect_tx(kv_full(s), L::VTILE);
                                for (int c = 0; c < DV / 64; ++c)
                                    tma_load_4d(stage(s) + c * kChunkBytes, &tmV, kv_full(s), c * 64,
                                                x.kvh, kr, kbc);
                            }
                            armed |= 1u << s;
                            armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                        }
                    }
                }
                // End marker for the MMA warps, once the last Q tile has been
                // consumed (so no Q load is left in flight either).
                if (ok) {
                    if (mbar_wait(bar(B_Q_EMPTY), q_ph ^ 1u, abort_flag, wl)) {
                        unit_desc[q_ph * 4] = 0;
                        mbar_arrive(bar(B_Q_FULL));
                        last_q_parity = -1;
                    } else {
                        raise_abort(abort_flag, p.status, kStatusTimeoutQ);
                    }
                }
                // Drain: every copy this thread issued has landed before the CTA exits.
                // (these waits ignore the abort flag: the copies always land)
                if (last_q_parity >= 0) mbar_wait_drain(bar(B_Q_FULL), (uint32_t)last_q_parity);
                for (int s = 0; s < NS; ++s)
                    if (armed & (1u << s)) mbar_wait_drain(kv_full(s), (armed_parity >> s) & 1u);
            }
        } else if (warp == kMmaWarp0 || warp == kMmaWarp1) {
            // -------------------------------------- MMA issuers, one per Q tile
            // Each warp runs the chain S_t(j) -> [softmax_t] -> PV_t(j) -> S_t(j+1)
            // of its own tile; two issuing warps keep the tensor core fed while
            // either one waits.  P_t aliases S_t in TMEM, so S_t(j+1) is issued
            // after PV_t(j) by the same thread (tcgen05.mma executes in order).
            // Only the wait for P_t(j) is left between the softmax and the two
            // MMA batches: V_j, K_{j+1} and O_t's release are waited for while
            // the softmax still runs (each mbarrier wait costs a few hundred
            // cycles here even when its phase is long complete: 494 -> 421 us
            // on the 4096^2 bf16 prefill).
            const int t = warp - kMmaWarp0;
            uint32_t kv_it = 0, q_ph = 0, p_ph = 0, oe_ph = 0;
            uint32_t vt_ph = 0;  // per ring slot: parity of its next v_tail phase (bit s)
            bool ok = true;
            const uint32_t s_tm = tmem + (uint32_t)t * 128u;
            const uint32_t o_tm = tmem + (uint32_t)(L::O_COL + t * DV);
            const uint64_t qd = sw128_desc(q_smem + t * L::QTILE, 16, 1024);
            // The units come from the TMA warp with each Q tile: no index
            // arithmetic on this warp's path from one unit to the next.
            while (ok) {
                if (!warp_wait(bar(B_Q_FULL), q_ph, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                const volatile int *d = unit_desc + q_ph * 4;
                q_ph ^= 1u;
                struct {
                    int n_kv, kv_start, hi_unit;
                } x;
                x.n_kv = d[0];
                x.kv_start = d[1];
                x.hi_unit = d[2];
                if (x.n_kv == 0) break;  // end marker
                const uint32_t kb = kv_it;

                // S_t(j) = Q_t K_j^T into TMEM (K_j has landed), then release K_j
                auto issue_s = [&](int j) {
                    const uint32_t it = kb + 2u * (uint32_t)j;
                    const int kslot = (int)(it % NS);
                    tc_fence_after();
                    if (lane == 0) {
                        // the start-address field is the low 14 bits (address >> 4)
                        const uint64_t kd = sw128_desc(stage(kslot), 16, 1024);
                        // the last tile computes only the key columns in use (rounded
                        // up to 16); the softmax masks the stale columns past them
                        const int nvalid = min(kBN, x.hi_unit - (x.kv_start + j * kBN));
                        const uint32_t ncols = (uint32_t)((nvalid + 15) & ~15);
                        const uint32_t idesc =
                            (a.idesc_s & ~(0x3Fu << 17)) | ((ncols >> 3) << 17);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4;
                            mma_ss(s_tm, qd + off, kd + off, idesc, kk > 0);
                        }
                        mma_commit(bar(B_S_FULL + t));
                        mma_commit(kv_empty(kslot));
                        if (j == x.n_kv - 1) mma_commit(bar(B_Q_EMPTY));
                    }
                    __syncwarp();
                };
                auto wait_k = [&](int j) -> bool {
                    const uint32_t it = kb + 2u * (uint32_t)j;
                    return warp_wait(kv_full((int)(it % NS)), (it / NS) & 1u, abort_flag, wl);
                };

                if (!wait_k(0)) {
                    ok = false;
                    break;
                }
                issue_s(0);
                for (int jj = 0; jj < x.n_kv && ok; ++jj) {
                    // Everything PV_t(jj) and S_t(jj + 1) need apart from P_t(jj) is
                    // waited for first, while the softmax still runs: V_jj (zeroed
                    // past the unit's last key), K_{jj+1}, and for the first tile the
                    // previous unit's O_t read out by the epilogue.
                    const uint32_t it = kb + 2u * (uint32_t)jj + 1u;
                    const int vslot = (int)(it % NS);
                    // Keys past the last one any row of the unit uses (only in the
                    // last tile) are left out 16 at a time; the V rows of the
                    // last 16-key step that lie past it may hold anything (NaN
                    // included), so they are zeroed to keep 0 * V at 0.
                    const int nvalid = min(kBN, x.hi_unit - (x.kv_start + jj * kBN));
                    const int ksteps = (nvalid + 15) / 16;
                    const int nzero = ksteps * 16 - nvalid;
                    if (t == 0 || nzero == 0) {
                        if (!warp_wait(kv_full(vslot), (it / NS) & 1u, abort_flag, wl)) {
                            ok = false;
                            break;
                        }
                    }
                    if (nzero > 0) {
                        if (t == 0) {
                            // zero the rows (whole 128-byte rows: the swizzle does not
                            // matter), then hand the tile to the other MMA warp
                            uint8_t *vt = gbase + (stage(vslot) - base) + nvalid * 128;
#pragma unroll
                            for (int c = 0; c < DV / 64; ++c)
                                for (int i = lane; i < nzero * 8; i += 32)
                                    *reinterpret_cast<uint4 *>(vt + c * kChunkBytes + i * 16) =
                                        make_uint4(0, 0, 0, 0);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(v_tail(vslot));
                        } else {
                            if (!warp_wait(v_tail(vslot), (vt_ph >> vslot) & 1u, abort_flag, wl)) {
                                ok = false;
                                break;
                            }
                            vt_ph ^= 1u << vslot;
                        }
                    }
                    const bool more = jj + 1 < x.n_kv;
                    if (more && !wait_k(jj + 1)) {
                        ok = false;
                        break;
                    }
                    if (jj == 0) {  // the previous unit's epilogue has read O_t
                        if (!warp_wait(bar(B_O_EMPTY + t), oe_ph ^ 1u, abort_flag, wl)) {
                            ok = false;
                            break;
                        }
                        oe_ph ^= 1u;
                    }
                    if (!warp_wait(bar(B_P_READY + t), p_ph, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    p_ph ^= 1u;
                    // O_t (+)= P_t V_jj, then release V_jj
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t vd = sw128_desc(stage(vslot), kChunkBytes, 1024);
                        // unrolled with a guard: a loop with a run-time trip count
                        // issues markedly slower
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            if (kk < ksteps)
                                mma_ts(o_tm, s_tm + kk * 8, vd + (kk * 2048 >> 4), a.idesc_o,
                                       (jj > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(kv_empty(vslot));
                    }
                    __syncwarp();
                    // S_t(jj + 1) overwrites P_t(jj): issued after PV_t(jj) by the same
                    // thread (tcgen05.mma executes in order)
                    if (more) issue_s(jj + 1);
                }
                if (!ok) break;
                if (lane == 0) mma_commit(bar(B_O_FULL + t));
                __syncwarp();
                kv_it += 2u * (uint32_t)x.n_kv;
            }
            if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutMma);
            // all MMAs issued by this warp complete before TMEM is released
            // (also after an abort: this wait ignores the abort flag)
            if (lane == 0) {
                mma_commit(bar(B_TEARDOWN + t));
                mbar_wait_drain(bar(B_TEARDOWN + t), 0);
            }
            __syncwarp();
        }
    } else if (warp < 8) {
        // ------------------------------------------------- softmax warpgroups
        regs_increase<kRegsSoftmax>();
        const int t = warp >> 2;                 // Q tile of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;       // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)(t * 128);
        const uint32_t tO = tmem + lane_off + (uint32_t)(L::O_COL + t * DV);
        const float c = a.c_scale;
        uint32_t s_ph = 0;
        uint32_t ntile = 0;  // tiles this warpgroup has processed (all units)
        uint32_t nunit = 0;  // units with keys this warpgroup has processed
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        float *inv_l = reinterpret_cast<float *>(gbase + L::STATS_OFF);

        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake_unit(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            const UnitInfo x = unit_info<MODE>(a, u);
            const int qpos = x.q0 + t * a.QP + r / a.Gp;
            const int head = x.h0 + r % a.Gp;
            const bool valid = qpos < x.si.Qb;
            const bool writes = padded ? qpos < p.Q : valid;
            int lo = 0, hi = 0;
            if (valid) legal_range(qpos, x.si.Qb, x.si.Kb, p.window, p.mask, lo, hi);
            const long long orow = (x.si.q_off + qpos) * p.Hq + head;
            const uint8_t *lv = nullptr;
            int n_use = x.n_kv;
            const uint32_t *mrow = nullptr;  // arbitrary mask: this row's words
            if (MASKED && x.n_kv > 0) {
                int j_last;
                lv = live_row(a, x);
                n_use = count_live(lv, x.n_kv, &j_last);
                if (valid) mrow = mask_row(p, x.b, head, qpos);
            }

            if (n_use == 0) {  // nothing to attend: +0 and -inf
                if (writes) {
                    uint4 *dst = reinterpret_cast<uint4 *>(og + orow * p.Dv);
                    for (int i = 0; i < p.Dv * 2 / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[orow] = -INFINITY;
                }
                continue;
            }

            float m_run = -INFINITY, l_run = 0.f;
            // One KV tile of this warpgroup's softmax.
            auto tile_step = [&](int j, bool interior) -> bool {
                // an arbitrary mask: this row's 128 bits of the tile (k0 is a multiple
                // of 128, the row a multiple of four words), fetched before the waits
                uint4 mw = make_uint4(~0u, ~0u, ~0u, ~0u);
                if (MASKED && lv[j] != 2) {
                    mw = make_uint4(0u, 0u, 0u, 0u);
                    if (mrow != nullptr)
                        mw = __ldg(reinterpret_cast<const uint4 *>(mrow + (x.kv_start + j * kBN) / 32));
                }
                // The two warpgroups take turns (tile k of group 0, tile k of
                // group 1, tile k+1 of group 0, ...): while one runs its softmax
                // the tensor core works on the other's tile.  Left free, the two
                // drift into step and then both wait on the tensor core together.
                // Each p_ready barrier is thus never more than one phase ahead
                // of the group that waits on it.
                auto take_turn = [&]() -> bool {
                    const int tb = kTurnMode == 3 ? B_TURN : B_P_READY;
                    bool w = true;
                    if (t == 1)
                        w = warp_wait(bar(tb + 0), ntile & 1u, abort_flag, wl);
                    else if (ntile > 0)
                        w = warp_wait(bar(tb + 1), (ntile - 1) & 1u, abort_flag, wl);
                    ++ntile;
                    return w;
                };
                if ((kTurnMode == 1 || kTurnMode == 3) && !take_turn()) return false;
                if (!warp_wait(bar(B_S_FULL + t), s_ph, abort_flag, wl)) return false;
                s_ph ^= 1u;
                tc_fence_after();
                if (!interior) {
                    // A tile that crosses the causal diagonal, the window edge or the
                    // end of the keys: keys outside [lo, hi) are set to -inf in TMEM
                    // (which also keeps NaN from padding out) before the softmax
                    // below reads S, so that there is one copy of that code for all
                    // tiles.  Per 32-key chunk: the row's legal keys as a bit mask;
                    // a chunk that every row of the warp keeps whole is left alone.
                    const int k0 = x.kv_start + j * kBN;
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        const int a0 = min(max(lo - k0 - cc * 32, 0), 32);
                        const int b0 = min(max(hi - k0 - cc * 32, 0), 32);
                        const uint32_t below_b = b0 >= 32 ? 0xffffffffu : (1u << b0) - 1u;
                        const uint32_t below_a = a0 >= 32 ? 0xffffffffu : (1u << a0) - 1u;
                        uint32_t keep = below_b & ~below_a;
                        if (MASKED) keep &= cc == 0 ? mw.x : cc == 1 ? mw.y : cc == 2 ? mw.z : mw.w;
                        if (__all_sync(0xffffffffu, keep == 0xffffffffu)) continue;
                        uint32_t v[32];
                        tmem_ld32(tS + cc * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = ((keep >> i) & 1u) ? v[i] : 0xff800000u;
                        tmem_st32(tS + cc * 32, v);
                    }
                    tmem_st_wait();
                }
                uint32_t sr[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
                tmem_ld_wait();
                // row max: eight independent chains of 3-input max
                float mc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mc[i] = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        mc[i & 7] = fmax3(mc[i & 7], __uint_as_float(sr[cc][2 * i]),
                                          __uint_as_float(sr[cc][2 * i + 1]));
                const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]),
                                       fmaxf(mc[6], mc[7]));
                const float m_tile = mx * c;
                float alpha = 1.f;
                bool rescale = false;
                if (m_run == -INFINITY) {
                    m_run = m_tile;  // first keys of this row (or still none)
                } else if (m_tile > m_run + 8.f) {
                    alpha = ex2(m_run - m_tile);
                    m_run = m_tile;
                    rescale = true;
                }
                const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
                if (__any_sync(0xffffffffu, rescale)) {
                    // O_t holds every PV up to tile j-1 (the commit that signalled
                    // S_t(j) was issued after them) and none of tile j yet
#pragma unroll
                    for (int cc = 0; cc < DV / 16; ++cc) {
                        uint32_t ov[16];
                        tmem_ld16(tO + cc * 16, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st16(tO + cc * 16, ov);
                    }
                }
                if (kTurnMode == 2 && !take_turn()) return false;
                // p = 2^(s*c - m) two keys at a time: one packed FMA, two MUFU
                // exps, one packed add into the row sum, one pack to P
                const uint64_t c2 = f2pack(c, c), nm2 = f2pack(neg_m, neg_m);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    // P columns [32*half, 32*half + 32) hold keys [64*half, 64*half + 64)
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 2 * half; cc < 2 * half + 2; ++cc)
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint64_t x2 = ffma2(
                                f2pack(__uint_as_float(sr[cc][2 * i]), __uint_as_float(sr[cc][2 * i + 1])),
                                c2, nm2);
                            float x0, x1;
                            f2unpack(x2, x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            acc2[i & 3] = fadd2(acc2[i & 3], f2pack(p0, p1));
                            pk[(cc & 1) * 16 + i] = pack2<T>(p0, p1);
                        }
                    tmem_st32(tS + 32 * half, pk);
                }
                if (kTurnMode == 3) mbar_arrive(bar(B_TURN + t));
                float sa[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) f2unpack(acc2[i], sa[2 * i], sa[2 * i + 1]);
                const float sum = ((sa[0] + sa[1]) + (sa[2] + sa[3])) + ((sa[4] + sa[5]) + (sa[6] + sa[7]));
                l_run = l_run * alpha + sum;
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(B_P_READY + t));
                return true;
            };
            for (int j = 0; j < x.n_kv && ok; ++j) {
                if (MASKED && lv[j] == 0) continue;  // a dead tile: not computed
                const int k0 = x.kv_start + j * kBN;
                // (a live tile every row may attend to whole is masked as unmasked)
                const bool interior = (!MASKED || lv[j] == 2) && x.all_valid && k0 >= x.lo_last &&
                                      k0 + kBN <= x.hi_first;
                ok = tile_step(j, interior);
            }
            if (!ok) break;

            // LSE here; 1 / l (0 for a row without keys) to the epilogue warpgroup
            const bool has = valid && l_run > 0.f;
            if (writes && p.lse) p.lse[orow] = has ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
            inv_l[(nunit & 1u) * 2 * kBM + t * kBM + r] = has ? 1.f / l_run : 0.f;
            mbar_arrive(bar(B_STATS + 2 * t + (int)(nunit & 1u)));
            ++nunit;
        }
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutSoftmax);
    } else {
        // ------------------------------------------------ epilogue warpgroup
        // Per unit, tile 0 then tile 1: wait for O_t and the rows' 1 / l, read
        // O_t out of TMEM 64 columns at a time into a staging tile (the TMA
        // box layout: 128 rows of 128 bytes, 16-byte chunks XOR-swizzled by the
        // row's low 3 bits), free O_t once the last columns are read, and store
        // each staged box with one TMA store.  The next unit's first PV into
        // O_t waits only for the TMEM reads.  A tile whose rows run into the
        // next sequence of a packed batch goes out row by row instead.
        regs_decrease<kRegsEpi>();
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const bool leader = warp == kEpiWarp0 && lane == 0;  // issues the TMA stores
        uint32_t o_ph = 0;   // bit t: parity of O_t's next phase
        uint32_t st_ph = 0;  // bit 2t+b: parity of stats barrier (t, b)
        uint32_t nunit = 0;
        bool ok = true;
        T *og = static_cast<T *>(p.o);
        const float *inv_l = reinterpret_cast<const float *>(gbase + L::STATS_OFF);
        uint8_t *stg = gbase + L::STG_OFF;
        const uint32_t stg_s = base + L::STG_OFF;

        for (long long rnd = 0; rnd * gridDim.x < a.nunits && ok; ++rnd) {
            const long long u = snake_unit(rnd, blockIdx.x, gridDim.x);
            if (u >= a.nunits) continue;
            const UnitInfo x = unit_info<MODE>(a, u);
            if (x.n_kv == 0) continue;  // the softmax warpgroups wrote those rows
            if (MASKED) {
                int j_last;
                if (count_live(live_row(a, x), x.n_kv, &j_last) == 0) continue;  // likewise
            }
            const int b = (int)(nunit & 1u);
            ++nunit;
            for (int t = 0; t < 2; ++t) {
                const int sb = 2 * t + b;
                const bool got = warp_wait(bar(B_O_FULL + t), (o_ph >> t) & 1u, abort_flag, wl) &&
                                 warp_wait(bar(B_STATS + sb), (st_ph >> sb) & 1u, abort_flag, wl);
                // The four warps go on or give up together: a warp that went on
                // alone would wait forever at the named barriers below.
                if (!bar_red_and(2, 128, got)) {
                    ok = false;
                    break;
                }
                o_ph ^= 1u << t;
                st_ph ^= 1u << sb;
                tc_fence_after();
                const float inv = inv_l[b * 2 * kBM + t * kBM + r];
                const int qt0 = x.q0 + t * a.QP;  // first query position of the tile
                // padded rows past Q fall outside the tensor map and are dropped
                // by the TMA store; rows in [Qb, Q) are written as zeros
                const bool by_tma = padded || qt0 + a.QP <= x.si.Qb;
                const uint32_t tO = tmem + lane_off + (uint32_t)(L::O_COL + t * DV);
#pragma unroll
                for (int cp = 0; cp < DV / 64; ++cp) {
                    if (leader) bulk_wait_read0();  // the staging tile is free again
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t ov[32];
                        tmem_ld32(tO + cp * 64 + h * 32, ov);
                        tmem_ld_wait();
                        if (cp == DV / 64 - 1 && h == 1) {  // O_t is read: free it
                            tc_fence_before();
                            mbar_arrive(bar(B_O_EMPTY + t));
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
                            const int qrow = (padded ? 0 : (int)x.si.q_off) + qt0;
                            tma_store_4d(&tmO, stg_s, cp * 64, x.h0, qrow, padded ? x.b : 0);
                            bulk_commit();
                        }
                    } else {
                        // this warp's 32 rows, 16 bytes a lane per step
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int e = i * 32 + lane;
                            const int rr = quarter * 32 + (e >> 3), ch = e & 7;
                            const int qp = qt0 + rr / a.Gp;
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
        }
        if (leader) bulk_wait0();
        if (!ok && lane == 0) raise_abort(abort_flag, p.status, kStatusTimeoutEpilogue);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Longest-first order of the units of a ragged problem (one block): a
// counting sort of the unit indices by KV tile count, descending, so that the
// persistent CTAs' alternating rounds deal the long units out first and the
// short ones even out the ends (the natural order is longest-first only when
// all sequences have the same lengths).  Units in the same bin keep no fixed
// order; each unit still writes only its own rows, so the result does not
// depend on it.
constexpr int kOrderThreads = 1024;
constexpr int kOrderBins = 2048;  // tile counts at or above the last bin share it

template <int MODE>
__global__ void __launch_bounds__(kOrderThreads) unit_order_kernel(const PrefillArgs a,
                                                                   int *order) {
    __shared__ int hist[kOrderBins];
    __shared__ int warp_sum[kOrderThreads / 32];
    // the prefill grid (a programmatic dependent launch) may be scheduled now:
    // its blocks set up and then wait in griddepcontrol.wait for this order
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = (int)a.nunits;
    auto bin_of = [&](int u) {
        const UnitInfo x = unit_info<MODE>(a, u);  // a.order is null here
        int c = x.n_kv;
        if (MODE == 2 && c > 0) {  // an arbitrary mask: the live tiles only
            int j_last;
            c = count_live(live_row(a, x), c, &j_last);
        }
        return kOrderBins - 1 - min(c, kOrderBins - 1);  // bin 0: the most tiles
    };
    for (int i = tid; i < kOrderBins; i += kOrderThreads) hist[i] = 0;
    __syncthreads();
    for (int u = tid; u < n; u += kOrderThreads) atomicAdd(&hist[bin_of(u)], 1);
    __syncthreads();
    // exclusive scan of the histogram: two bins a thread, then warps, then block
    constexpr int PER = kOrderBins / kOrderThreads;
    int v[PER], local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        v[i] = hist[tid * PER + i];
        local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sum[lane] = w;  // inclusive
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? warp_sum[warp - 1] : 0);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        hist[tid * PER + i] = run;
        run += v[i];
    }
    __syncthreads();
    for (int u = tid; u < n; u += kOrderThreads) order[atomicAdd(&hist[bin_of(u)], 1)] = u;
}

// Arbitrary mask: which 128-key tiles have a key some row of a unit may attend
// to.  One warp per (summary row, tile): a summary row is one (sequence, query
// block) when the mask is shared by all heads (its rows are the block's query
// positions) and one unit otherwise (the block's positions x the unit's
// heads); each lane ORs the tile's four words of its rows.  Rows past the
// sequence's queries are not read.
constexpr int kSummaryWarps = 8;

template <int MODE>
__global__ void __launch_bounds__(kSummaryWarps * 32) mask_summary_kernel(const PrefillArgs a,
                                                                          uint8_t *live) {
    // the next launch (a programmatic dependent) may set up meanwhile
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const AttnParams &p = a.p;
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * kSummaryWarps + (threadIdx.x >> 5);
    const long long nrow = a.live_shared ? (long long)p.B * a.nqblk : a.nunits;
    if (w >= nrow * a.live_tiles) return;
    const long long row = w / a.live_tiles;
    const int tile = (int)(w - row * a.live_tiles);
    int b, q0, h0, nh;
    if (a.live_shared) {
        b = (int)(row / a.nqblk);
        q0 = (int)(row - (long long)b * a.nqblk) * 2 * a.QP;
        h0 = 0;
        nh = 1;
    } else {
        const UnitInfo x = unit_info<MODE>(a, row);  // a.order is null here
        b = x.b;
        q0 = x.q0;
        h0 = x.h0;
        nh = a.Gp;
    }
    const int Qb = seq_info(p, b).Qb;
    uint32_t any = 0, all = 0xffffffffu;
    for (int r = lane; r < 2 * a.QP * nh; r += 32) {
        const int pos = q0 + r / nh;
        if (pos >= Qb) continue;
        const uint4 m = __ldg(reinterpret_cast<const uint4 *>(mask_row(p, b, h0 + r % nh, pos)) + tile);
        any |= m.x | m.y | m.z | m.w;
        all &= m.x & m.y & m.z & m.w;
    }
    const bool some = __any_sync(0xffffffffu, any != 0);
    const bool full = __all_sync(0xffffffffu, all == 0xffffffffu);
    if (lane == 0) live[w] = some ? (full ? 2 : 1) : 0;
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 4-D map over [d3][d2][d1][d0] (d0 innermost) with a {64, b1, b2, 1} box and
// 128-byte swizzle.
int make_map(CUtensorMap *map, const void *ptr, CUtensorMapDataType dt, uint64_t d0, uint64_t d1,
             uint64_t d2, uint64_t d3, uint32_t b1, uint32_t b2) {
    auto fn = encode_fn();
    if (fn == nullptr) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return 3;
    }
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    const cuuint32_t box[4] = {64, b1, b2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, dt, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
        return 3;
    }
    return 0;
}

int pack_factor(int G) {
    int gp = 1;
    while (gp < 16 && G % (gp * 2) == 0) gp *= 2;
    return gp;
}

template <typename T, int D, int DV>
int launch_t(const AttnParams &p, bool bf16, cudaStream_t stream, int *order_ws,
             uint8_t *live_ws) {
    using L = Layout<D, DV>;
    PrefillArgs a;
    a.p = p;
    a.order = nullptr;
    a.live = nullptr;
    a.live_tiles = (p.K + kBN - 1) / kBN;
    a.live_shared = p.mask_heads == 1 ? 1 : 0;
    a.Gp = pack_factor(p.G);
    a.QP = kBM / a.Gp;
    a.nsub = p.G / a.Gp;
    a.nqblk = (p.Q + 2 * a.QP - 1) / (2 * a.QP);
    a.nunits = (long long)a.nqblk * p.B * p.Hkv * a.nsub;
    a.per = (uint32_t)((long long)p.B * p.Hkv * a.nsub);
    a.hs = (uint32_t)(p.Hkv * a.nsub);
    const float sc = p.scale == 0.f ? 1e-30f : fabsf(p.scale);
    a.c_scale = sc * kLog2e;
    a.idesc_s = idesc_f16(bf16, kBM, kBN, false, p.scale < 0.f);
    a.idesc_o = idesc_f16(bf16, kBM, DV, true, false);
    if (a.nunits == 0) return 0;

    const CUtensorMapDataType dt =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool padded = p.cu_q == nullptr;
    const uint64_t qrows = padded ? (uint64_t)p.Q : (uint64_t)p.Tq;
    const bool paged = p.block_table != nullptr;
    const uint64_t krows = (padded && !paged) ? (uint64_t)p.K : (uint64_t)p.Tk;
    const uint64_t nb = padded ? (uint64_t)p.B : 1;
    const uint64_t nbk = (padded && !paged) ? (uint64_t)p.B : 1;
    CUtensorMap tq, tk, tv, to;
    // maps over the real head dims: the columns up to the padded D / DV of the
    // tiles are zero-filled by the loads (so they add nothing to S or O) and
    // dropped by the O stores
    int rc = make_map(&tq, p.q, dt, (uint64_t)p.D, p.Hq, qrows, nb, a.Gp, a.QP);
    if (rc) return rc;
    rc = make_map(&to, p.o, dt, (uint64_t)p.Dv, p.Hq, qrows, nb, a.Gp, a.QP);
    if (rc) return rc;
    if (krows > 0) {
        rc = make_map(&tk, p.k, dt, (uint64_t)p.D, p.Hkv, krows, nbk, 1, kBN);
        if (rc) return rc;
        rc = make_map(&tv, p.v, dt, (uint64_t)p.Dv, p.Hkv, krows, nbk, 1, kBN);
        if (rc) return rc;
    } else {
        tk = tq;  // never read: every unit has no key
        tv = tq;
    }
    const bool masked = p.mask_bits != nullptr;
    cudaError_t e;
    if (masked) {
        if (live_ws == nullptr) {
            set_error("prefill kernel: the masked launch needs its tile workspace");
            return 1;
        }
        const long long nrow = a.live_shared ? (long long)p.B * a.nqblk : a.nunits;
        const long long warps = nrow * a.live_tiles;
        const long long blocks = (warps + kSummaryWarps - 1) / kSummaryWarps;
        if (blocks >= (1LL << 31)) {
            set_error("prefill kernel: too many mask tiles");
            return 2;
        }
        mask_summary_kernel<2><<<(unsigned)blocks, kSummaryWarps * 32, 0, stream>>>(a, live_ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error("mask summary kernel launch: %s", cudaGetErrorString(e));
            return 3;
        }
        count_launch();
        a.live = live_ws;
    }
    if (order_ws != nullptr) {
        auto ok = masked ? unit_order_kernel<2> : paged ? unit_order_kernel<1> : unit_order_kernel<0>;
        ok<<<1, kOrderThreads, 0, stream>>>(a, order_ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error("unit order kernel launch: %s", cudaGetErrorString(e));
            return 3;
        }
        count_launch();
        a.order = order_ws;
    }
    auto kern = masked ? prefill_tc_kernel<T, D, DV, 2>
                       : paged ? prefill_tc_kernel<T, D, DV, 1> : prefill_tc_kernel<T, D, DV, 0>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("prefill kernel: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    const int nsm = sm_count(dev);
    const long long grid = a.nunits < nsm ? a.nunits : nsm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // after the order / mask summary kernel: overlap their run
    cfg.numAttrs = (a.order != nullptr || a.live != nullptr) ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, a, tq, tk, tv, to);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("prefill kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_dtype(const AttnParams &p, bool bf16, cudaStream_t stream, int *order_ws,
                 uint8_t *live_ws) {
    // tiles padded to 64 or 128 columns
    const bool d128 = p.D > 64, dv128 = p.Dv > 64;
    if (d128 && dv128) return launch_t<T, 128, 128>(p, bf16, stream, order_ws, live_ws);
    if (!d128 && !dv128) return launch_t<T, 64, 64>(p, bf16, stream, order_ws, live_ws);
    if (d128) return launch_t<T, 128, 64>(p, bf16, stream, order_ws, live_ws);
    return launch_t<T, 64, 128>(p, bf16, stream, order_ws, live_ws);
}

long long unit_count(const AttnParams &p) {
    const int gp = pack_factor(p.G), qp = kBM / gp;
    return (long long)((p.Q + 2 * qp - 1) / (2 * qp)) * p.B * p.Hkv * (p.G / gp);
}

}  // namespace

bool prefill_tc_supported(const AttnParams &p, int dtype) {
    if (dtype != 1 && dtype != 2) return false;
    // head dims: multiples of 16 in [64, 128] (tiles padded to 64 or 128 columns)
    if (p.D < 64 || p.D > 128 || p.D % 16 || p.Dv < 64 || p.Dv > 128 || p.Dv % 16) return false;
    if (p.Q < 1) return false;
    const long long rows = p.cu_q ? p.Tq : (long long)p.Q;
    const long long keys = (p.cu_q || p.block_table) ? p.Tk : (long long)p.K;
    // paged K/V: a 128-key tile must lie in one page
    if (p.block_table && p.page_size % kBN != 0) return false;
    // an arbitrary mask: padded layout, contiguous K/V
    if (p.mask_bits && (p.block_table || p.cu_q)) return false;
    // work units are indexed in 32 bits
    return rows < (1LL << 31) && keys < (1LL << 31) && unit_count(p) < (1LL << 31);
}

long long prefill_tc_order_len(const AttnParams &p) {
    // ragged problems (packed, or padded with per-sequence lengths, or an
    // arbitrary mask) of a size the one-block sort handles in a few microseconds
    const bool ragged = p.cu_q != nullptr || p.seqlens_q != nullptr || p.seqlens_k != nullptr ||
                        p.mask_bits != nullptr;
    const long long n = unit_count(p);
    return (ragged && n > 1 && n <= (1LL << 16)) ? n : 0;
}

long long prefill_tc_live_len(const AttnParams &p) {
    if (p.mask_bits == nullptr) return 0;
    const int gp = pack_factor(p.G), qp = kBM / gp;
    const long long nqblk = (p.Q + 2 * qp - 1) / (2 * qp);
    const long long rows = p.mask_heads == 1 ? (long long)p.B * nqblk : unit_count(p);
    return rows * ((p.K + kBN - 1) / kBN);
}

int make_tma_map_4d(CUtensorMap *map, const void *ptr, bool bf16, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t d3, uint32_t b1, uint32_t b2) {
    return make_map(map, ptr,
                    bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, d0,
                    d1, d2, d3, b1, b2);
}

int launch_prefill_tc(const AttnParams &p, int dtype, cudaStream_t stream, int *order_ws,
                      uint8_t *live_ws) {
    if (dtype == 2) return launch_dtype<__nv_bfloat16>(p, true, stream, order_ws, live_ws);
    return launch_dtype<__half>(p, false, stream, order_ws, live_ws);
}

}  // namespace attn
