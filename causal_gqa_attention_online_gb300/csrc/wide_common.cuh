// wide_common.cuh -- pieces shared by the one-Q-tile tcgen05 forward kernels
// for wide heads (kernel_prefill_wide_tc.cu: widths up to 256;
// kernel_prefill_wide512_tc.cu: up to 512): the work-unit decode, the
// serpentine unit order, and one softmax step over a 128-key S tile in TMEM.
//
// The step is the online softmax of "Attention execution mapping"
// (LuisaCompute), sections 1-2: keys outside the row's legal range [lo, hi)
// to -inf, the tile max, the conditional rescale of the running sum and of O
// (only when the max grows by more than 2^8, the reference max is kept
// otherwise), P = 2^(c S - m) packed to 16 bits over S for the PV product,
// and the row sum.
#pragma once

#include <climits>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tc_softmax.cuh"

namespace attn {
namespace tcwide {

using namespace sm100;
using namespace tcfwd;

// One work unit: a 128-row Q tile (Gp heads of a KV group x QP positions)
// against the legal keys of its rows, walked in 128-key tiles.
struct QTileUnit {
    int b, kvh, h0, q0;
    SeqInfo si;
    int n_kv, kv_start, lo_last, hi_first, hi_unit;
    bool all_valid;
};

// Unit u of per = B * Hkv * nsub units per query block, hs = Hkv * nsub;
// query blocks are taken from the last (longest) to the first.
__device__ __forceinline__ QTileUnit qtile_unit(const AttnParams &p, uint32_t per, uint32_t hs,
                                                int nsub, int Gp, int QP, int nqblk,
                                                uint32_t u) {
    const uint32_t qi = u / per, rest = u - qi * per;
    const uint32_t b = rest / hs, r2 = rest - b * hs;
    const uint32_t kvh = r2 / (uint32_t)nsub, sub = r2 - kvh * (uint32_t)nsub;
    const int qblk = nqblk - 1 - (int)qi;
    QTileUnit x;
    x.b = (int)b;
    x.kvh = (int)kvh;
    x.h0 = x.kvh * p.G + (int)sub * Gp;
    x.q0 = qblk * QP;
    x.si = seq_info(p, x.b);
    x.n_kv = 0;
    x.kv_start = 0;
    x.lo_last = INT_MAX;
    x.hi_first = INT_MIN;
    x.hi_unit = 0;
    x.all_valid = false;
    if (x.q0 >= x.si.Qb) return x;
    const int q_last = min(x.q0 + QP, x.si.Qb) - 1;
    int lo_f, hi_f, lo_l, hi_l;
    legal_range(x.q0, x.si.Qb, x.si.Kb, p.window, p.mask, lo_f, hi_f);
    legal_range(q_last, x.si.Qb, x.si.Kb, p.window, p.mask, lo_l, hi_l);
    if (hi_l <= lo_f) return x;
    x.kv_start = lo_f;
    x.hi_unit = hi_l;
    x.n_kv = (hi_l - lo_f + 127) / 128;
    x.lo_last = lo_l;
    x.hi_first = hi_f;
    x.all_valid = x.q0 + QP <= x.si.Qb;
    return x;
}

// Round r of a persistent grid of G CTAs: CTA c takes unit r*G + c on even
// rounds and r*G + G-1-c on odd ones, so every CTA's total stays balanced
// while the units shrink.
__device__ __forceinline__ long long snake(long long r, int c, int G) {
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// One softmax step of the row held by this thread (TMEM lane = row) over
// the S tile at tS (128 fp32 columns; keys k0 .. k0 + 127).  Updates m_run
// (log2 domain) and l_run, rescales the OCOLS columns of O at tO when the
// max grows by more than 2^8 (first waiting for the previous tile's PV
// through pv_bar / pv_parity), and leaves P (16-bit) over the first 64
// columns of S.  Returns false when a bounded wait gave up.
template <typename T, int OCOLS>
__device__ __forceinline__ bool softmax_tile(uint32_t tS, uint32_t tO, int k0, bool interior,
                                             int lo, int hi, float c, float &m_run,
                                             float &l_run, uint32_t pv_bar, uint32_t pv_parity,
                                             volatile int *abort_flag, uint64_t wl) {
    if (!interior) {
        // keys outside [lo, hi) of this row to -inf in TMEM, 32 at a time
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            const int a0 = min(max(lo - k0 - cc * 32, 0), 32);
            const int b0 = min(max(hi - k0 - cc * 32, 0), 32);
            const uint32_t below_b = b0 >= 32 ? 0xffffffffu : (1u << b0) - 1u;
            const uint32_t below_a = a0 >= 32 ? 0xffffffffu : (1u << a0) - 1u;
            const uint32_t keep = below_b & ~below_a;
            if (__all_sync(0xffffffffu, keep == 0xffffffffu)) continue;
            uint32_t v[32];
            tmem_ld32(tS + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = ((keep >> i) & 1u) ? v[i] : 0xff800000u;
            tmem_st32(tS + cc * 32, v);
        }
        tmem_st_wait();
    }
    uint32_t sr[4][32];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
    tmem_ld_wait();
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
        m_run = m_tile;
    } else if (m_tile > m_run + 8.f) {
        alpha = ex2(m_run - m_tile);
        m_run = m_tile;
        rescale = true;
    }
    const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
    if (__any_sync(0xffffffffu, rescale)) {
        // S(j) was issued before PV(j - 1), so O may still be taking PV(j - 1):
        // wait for that tile's phase of the PV barrier (PV(j) is issued only
        // after this step, so the barrier cannot be two phases ahead).  The
        // first tile of a unit sets the reference max without a rescale.
        if (!warp_wait(pv_bar, pv_parity, abort_flag, wl)) return false;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < OCOLS / 16; ++cc) {
            uint32_t ov[16];
            tmem_ld16(tO + cc * 16, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st16(tO + cc * 16, ov);
        }
    }
    const uint64_t c2 = f2pack(c, c), nm2 = f2pack(neg_m, neg_m);
    uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int cc = 2 * half; cc < 2 * half + 2; ++cc)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint64_t x2 = ffma2(f2pack(__uint_as_float(sr[cc][2 * i]),
                                                 __uint_as_float(sr[cc][2 * i + 1])),
                                          c2, nm2);
                float x0, x1;
                f2unpack(x2, x0, x1);
                const float p0 = ex2(x0), p1 = ex2(x1);
                acc2[i & 3] = fadd2(acc2[i & 3], f2pack(p0, p1));
                pk[(cc & 1) * 16 + i] = pack2<T>(p0, p1);
            }
        tmem_st32(tS + 32 * half, pk);
    }
    float sa[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2unpack(acc2[i], sa[2 * i], sa[2 * i + 1]);
    const float sum = ((sa[0] + sa[1]) + (sa[2] + sa[3])) + ((sa[4] + sa[5]) + (sa[6] + sa[7]));
    l_run = l_run * alpha + sum;
    tmem_st_wait();
    return true;
}

}  // namespace tcwide
}  // namespace attn
