// kernel_fwd_mma.cu -- warp-level tensor-core (mma.sync m16n8k16) forward for
// bf16 / fp16 head widths the tcgen05 prefill kernel does not take (D or Dv
// above 128, up to 512).
//
// The same recurrence as the other forward kernels ("Attention execution
// mapping" (LuisaCompute), sections 1-2: per KV tile QK -> mask -> max ->
// exp -> sum -> alpha-rescale -> PV, row max / row sum / accumulator carried
// across tiles), in registers:
//   * a block owns 64 consecutive rows of the flattened (query position,
//     head-in-group) space of one (sequence, KV head), 16 rows per warp, so
//     every K/V tile it stages serves all heads of the group (section 5,
//     cross-head KV reuse);
//   * K/V tiles are double-buffered in shared memory by cp.async (16-byte
//     chunks into an XOR-swizzled layout, rows past the keys zero-filled
//     without a read); Q stays staged for the whole block;
//   * S = Q K^T and O += P V are m16n8k16 MMAs with fp32 accumulation; the S
//     accumulator of two adjacent 8-key tiles is the A operand of a 16-key
//     step of PV (P packed to the storage type), and each row's max and sum
//     are reduced over the 4 lanes that hold it;
//   * masks are applied only on tiles some row of the warp does not see whole.
// Rows are ordered so that the blocks with the most keys start first.
#include <climits>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using sm100::named_bar_sync;
__device__ __forceinline__ void sm_bar_sync(int id, int n) { named_bar_sync(id, n); }

constexpr int kRowsF = 64;  // flattened rows per block (16 per warp)

template <int DW, int DVW> struct FwdTile {
    // keys per K/V tile: two stages of K and V plus Q fit two blocks an SM
    static constexpr int KEYS = (DW > 128 || DVW > 128) ? 32 : 64;
    static constexpr int KB = DW * 2, VB = DVW * 2;  // bytes per staged row
    static constexpr int SMEM = kRowsF * KB + 2 * KEYS * (KB + VB);
};

template <typename T, int DW, int DVW>
__global__ void __launch_bounds__(128) fwd_mma_kernel(const AttnParams p) {
    using L = FwdTile<DW, DVW>;
    constexpr int KEYS = L::KEYS, KB = L::KB, VB = L::VB;
    constexpr int NT = KEYS / 8;  // 8-key n-tiles of S per warp
    extern __shared__ __align__(128) uint8_t smem_f[];
    uint8_t *qs = smem_f;                 // [kRowsF][KB]
    uint8_t *ks = qs + kRowsF * KB;       // [2][KEYS][KB]
    uint8_t *vs = ks + 2 * KEYS * KB;     // [2][KEYS][VB]

    const int nbh = p.B * p.Hkv;
    const int rank = blockIdx.x / nbh, ntiles_q = gridDim.x / nbh;
    const int b = (blockIdx.x % nbh) / p.Hkv, kvh = (blockIdx.x % nbh) % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (ntiles_q - 1 - rank) * kRowsF;  // the last rows see the most keys
    if (r0 >= ncap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v);
    auto row_of = [&](int r) { return (si.q_off + r / G) * p.Hq + kvh * G + r % G; };

    for (int c = tid; c < kRowsF * (DW / 8); c += 128) {
        const int i = c / (DW / 8), ch = c % (DW / 8), r = r0 + i;
        const bool ok = r < nvalid && ch * 8 < D;
        cp_async16(smem_u32(qs + swz(i, ch, KB)), ok ? qg + row_of(r) * D + ch * 8 : qg,
                   ok ? 16 : 0);
    }
    // this thread's two rows: 16 * warp + g and + 8
    int lo[2], hi[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 16 * warp + g + 8 * hh;
        lo[hh] = hi[hh] = 0;
        if (r < nvalid) legal_range(r / G, si.Qb, si.Kb, p.window, p.mask, lo[hh], hi[hh]);
    }
    int klo = 0, khi = 0;
    if (nvalid > r0) {
        int a, c;
        legal_range(r0 / G, si.Qb, si.Kb, p.window, p.mask, klo, c);
        legal_range((min(r0 + kRowsF, nvalid) - 1) / G, si.Qb, si.Kb, p.window, p.mask, a, khi);
    }
    const int tfirst = klo / KEYS * KEYS;
    const int ntiles = khi > klo ? (khi - tfirst + KEYS - 1) / KEYS : 0;
    auto load_kv = [&](int i, int buf) {
        const int kt0 = tfirst + i * KEYS;
        for (int c = tid; c < KEYS * (DW / 8); c += 128) {
            const int r = c / (DW / 8), ch = c % (DW / 8), key = kt0 + r;
            const bool ok = key < si.Kb && ch * 8 < D;
            const T *src = ok ? kg + (kv_row(p, si, b, key) * p.Hkv + kvh) * (long long)D + ch * 8
                              : kg;
            cp_async16(smem_u32(ks + buf * KEYS * KB + swz(r, ch, KB)), src, ok ? 16 : 0);
        }
        for (int c = tid; c < KEYS * (DVW / 8); c += 128) {
            const int r = c / (DVW / 8), ch = c % (DVW / 8), key = kt0 + r;
            const bool ok = key < si.Kb && ch * 8 < Dv;
            const T *src =
                ok ? vg + (kv_row(p, si, b, key) * p.Hkv + kvh) * (long long)Dv + ch * 8 : vg;
            cp_async16(smem_u32(vs + buf * KEYS * VB + swz(r, ch, VB)), src, ok ? 16 : 0);
        }
    };
    if (ntiles > 0) load_kv(0, 0);
    cp_async_commit();

    float o[DVW / 8][4];
#pragma unroll
    for (int j = 0; j < DVW / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            load_kv(i + 1, (i + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint8_t *kb = ks + (i & 1) * KEYS * KB;
        const uint8_t *vb = vs + (i & 1) * KEYS * VB;
        const int kt0 = tfirst + i * KEYS;
        // S = Q K^T: this warp's 16 rows x KEYS keys
        float s[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DW / 16; ++kk) {
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(qs + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), KB)));
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t bk[4];
                ldmatrix_x4(bk, smem_u32(kb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                  2 * kk + ((lane >> 3) & 1), KB)));
                MmaOp<T>::run(s[2 * np], a, bk[0], bk[1]);
                MmaOp<T>::run(s[2 * np + 1], a, bk[2], bk[3]);
            }
        }
        // scores in log2 units, then the mask (only where some row of the
        // warp does not see the whole tile)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[j][c] *= p.scale_log2;
        const bool inner = __all_sync(0xffffffffu, lo[0] <= kt0 && lo[1] <= kt0 &&
                                                       hi[0] >= kt0 + KEYS && hi[1] >= kt0 + KEYS);
        if (!inner) {
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int hh = c >> 1, key = kt0 + 8 * j + 2 * t + (c & 1);
                    if (key < lo[hh] || key >= hi[hh]) s[j][c] = -INFINITY;
                }
        }
        // online max / exp2 / sum per row (a row lives in the 4 lanes of a quad)
        float alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float mx = m[hh];
#pragma unroll
            for (int j = 0; j < NT; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * hh], s[j][2 * hh + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            // a row with no legal key so far keeps a finite reference
            const float ref = mx == -INFINITY ? 0.f : mx;
            alpha[hh] = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - ref);
            m[hh] = mx;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = exp2f(s[j][2 * hh + e] - ref);
                    s[j][2 * hh + e] = pv;
                    sum += pv;
                }
            l[hh] = l[hh] * alpha[hh] + sum;  // quad-partial; reduced at the end
        }
#pragma unroll
        for (int j = 0; j < DVW / 8; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
        }
        // O += P V, contracting over the tile's keys 16 at a time
#pragma unroll
        for (int kk = 0; kk < KEYS / 16; ++kk) {
            uint32_t a[4];
            a[0] = MmaOp<T>::pack(s[2 * kk][0], s[2 * kk][1]);
            a[1] = MmaOp<T>::pack(s[2 * kk][2], s[2 * kk][3]);
            a[2] = MmaOp<T>::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = MmaOp<T>::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int trow = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int np = 0; np < DVW / 16; ++np) {
                uint32_t bb[4];
                ldmatrix_x4_trans(bb, smem_u32(vb + swz(trow, 2 * np + (lane >> 4), VB)));
                MmaOp<T>::run(o[2 * np], a, bb[0], bb[1]);
                MmaOp<T>::run(o[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        __syncthreads();  // buffer i & 1 is reloaded by the next iteration's prefetch
    }
    cp_async_wait<0>();

    // epilogue: O / l and LSE = (m + log2 l) * ln 2 (m in log2 units); rows
    // without a legal key and padded rows get O = +0 and LSE = -inf
    T *og = static_cast<T *>(p.o);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float sum = l[hh];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        const int r = r0 + 16 * warp + g + 8 * hh;
        if (r >= ncap) continue;
        const long long row = row_of(r);
        const bool has = r < nvalid && sum > 0.f;
        const float inv = has ? 1.f / sum : 0.f;
#pragma unroll
        for (int j = 0; j < DVW / 8; ++j) {
            const int d = 8 * j + 2 * t;
            if (d < Dv)
                *reinterpret_cast<uint32_t *>(og + row * Dv + d) =
                    MmaOp<T>::pack(o[j][2 * hh] * inv, o[j][2 * hh + 1] * inv);
        }
        if (t == 0 && p.lse != nullptr)
            p.lse[row] = has ? (m[hh] + log2f(sum)) * kLn2 : -INFINITY;
    }
}

// Wide heads (D or Dv above 256, up to 512): one 16 x 512 fp32 accumulator
// per warp would not fit in registers, so warps work in pairs on the same 16
// rows, each accumulating half of the output columns -- the across-wave split
// of the wide-head body in "Accelerating PyTorch on AMD GPUs with FlyDSL"
// (section on FMHA through AOTriton, figure 13), where both waves compute
// the same scores.  Here the score contraction is split too.  Warp w (< 4) and warp w + 4 each contract half of the head width
// for S (columns [0, DW/2) and [DW/2, DW)), swap their partial scores
// through shared memory behind a 64-thread named barrier and add them (in
// the same order, so both hold the same bits), run the same online softmax,
// and accumulate half of the O columns each ([0, DVW/2) and [DVW/2, DVW)).
constexpr int kWideKeys = 32;

template <int DW, int DVW> struct WideTile {
    static constexpr int KB = DW * 2, VB = DVW * 2;
    static constexpr int SMEM = kRowsF * KB + 2 * kWideKeys * (KB + VB) + 8 * 16 * 32 * 4;
};

template <typename T, int DW, int DVW>
__global__ void __launch_bounds__(256, 1) fwd_mma_wide_kernel(const AttnParams p) {
    using L = WideTile<DW, DVW>;
    constexpr int KEYS = kWideKeys, KB = L::KB, VB = L::VB;
    constexpr int NT = KEYS / 8;
    constexpr int DH = DW / 2, DVH = DVW / 2;  // each warp's share of D and Dv
    extern __shared__ __align__(128) uint8_t smem_w[];
    uint8_t *qs = smem_w;                  // [kRowsF][KB]
    uint8_t *ks = qs + kRowsF * KB;        // [2][KEYS][KB]
    uint8_t *vs = ks + 2 * KEYS * KB;      // [2][KEYS][VB]
    float *xs = reinterpret_cast<float *>(vs + 2 * KEYS * VB);  // [8 warps][16][32] partial S

    const int nbh = p.B * p.Hkv;
    const int rank = blockIdx.x / nbh, ntiles_q = gridDim.x / nbh;
    const int b = (blockIdx.x % nbh) / p.Hkv, kvh = (blockIdx.x % nbh) % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (ntiles_q - 1 - rank) * kRowsF;
    if (r0 >= ncap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int pr = warp & 3, half = warp >> 2;  // row group, half of the width
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v);
    auto row_of = [&](int r) { return (si.q_off + r / G) * p.Hq + kvh * G + r % G; };

    for (int c = tid; c < kRowsF * (DW / 8); c += 256) {
        const int i = c / (DW / 8), ch = c % (DW / 8), r = r0 + i;
        const bool ok = r < nvalid && ch * 8 < D;
        cp_async16(smem_u32(qs + swz(i, ch, KB)), ok ? qg + row_of(r) * D + ch * 8 : qg,
                   ok ? 16 : 0);
    }
    int lo[2], hi[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 16 * pr + g + 8 * hh;
        lo[hh] = hi[hh] = 0;
        if (r < nvalid) legal_range(r / G, si.Qb, si.Kb, p.window, p.mask, lo[hh], hi[hh]);
    }
    int klo = 0, khi = 0;
    if (nvalid > r0) {
        int a, c;
        legal_range(r0 / G, si.Qb, si.Kb, p.window, p.mask, klo, c);
        legal_range((min(r0 + kRowsF, nvalid) - 1) / G, si.Qb, si.Kb, p.window, p.mask, a, khi);
    }
    const int tfirst = klo / KEYS * KEYS;
    const int ntiles = khi > klo ? (khi - tfirst + KEYS - 1) / KEYS : 0;
    auto load_kv = [&](int i, int buf) {
        const int kt0 = tfirst + i * KEYS;
        for (int c = tid; c < KEYS * (DW / 8); c += 256) {
            const int r = c / (DW / 8), ch = c % (DW / 8), key = kt0 + r;
            const bool ok = key < si.Kb && ch * 8 < D;
            const T *src = ok ? kg + (kv_row(p, si, b, key) * p.Hkv + kvh) * (long long)D + ch * 8
                              : kg;
            cp_async16(smem_u32(ks + buf * KEYS * KB + swz(r, ch, KB)), src, ok ? 16 : 0);
        }
        for (int c = tid; c < KEYS * (DVW / 8); c += 256) {
            const int r = c / (DVW / 8), ch = c % (DVW / 8), key = kt0 + r;
            const bool ok = key < si.Kb && ch * 8 < Dv;
            const T *src =
                ok ? vg + (kv_row(p, si, b, key) * p.Hkv + kvh) * (long long)Dv + ch * 8 : vg;
            cp_async16(smem_u32(vs + buf * KEYS * VB + swz(r, ch, VB)), src, ok ? 16 : 0);
        }
    };
    if (ntiles > 0) load_kv(0, 0);
    cp_async_commit();

    float o[DVH / 8][4];
#pragma unroll
    for (int j = 0; j < DVH / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float *xmine = xs + warp * 16 * 32, *xother = xs + (warp ^ 4) * 16 * 32;

    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            load_kv(i + 1, (i + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint8_t *kb = ks + (i & 1) * KEYS * KB;
        const uint8_t *vb = vs + (i & 1) * KEYS * VB;
        const int kt0 = tfirst + i * KEYS;
        // this warp's half of S = Q K^T (16 rows x KEYS keys)
        float s[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
            const int ck = half * (DH / 8) + 2 * kk;  // 16-byte chunk of this k-step
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(qs + swz(16 * pr + (lane & 15), ck + (lane >> 4), KB)));
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t bk[4];
                ldmatrix_x4(bk, smem_u32(kb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                  ck + ((lane >> 3) & 1), KB)));
                MmaOp<T>::run(s[2 * np], a, bk[0], bk[1]);
                MmaOp<T>::run(s[2 * np + 1], a, bk[2], bk[3]);
            }
        }
        // swap partials with the pair's other warp; both add lower half first
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) xmine[(j * 4 + c) * 32 + lane] = s[j][c];
        sm_bar_sync(1 + pr, 64);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float other = xother[(j * 4 + c) * 32 + lane];
                s[j][c] = (half == 0 ? s[j][c] + other : other + s[j][c]) * p.scale_log2;
            }
        const bool inner = __all_sync(0xffffffffu, lo[0] <= kt0 && lo[1] <= kt0 &&
                                                       hi[0] >= kt0 + KEYS && hi[1] >= kt0 + KEYS);
        if (!inner) {
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int hh = c >> 1, key = kt0 + 8 * j + 2 * t + (c & 1);
                    if (key < lo[hh] || key >= hi[hh]) s[j][c] = -INFINITY;
                }
        }
        float alpha[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float mx = m[hh];
#pragma unroll
            for (int j = 0; j < NT; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * hh], s[j][2 * hh + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float ref = mx == -INFINITY ? 0.f : mx;
            alpha[hh] = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - ref);
            m[hh] = mx;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = exp2f(s[j][2 * hh + e] - ref);
                    s[j][2 * hh + e] = pv;
                    sum += pv;
                }
            l[hh] = l[hh] * alpha[hh] + sum;
        }
#pragma unroll
        for (int j = 0; j < DVH / 8; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
        }
        // this warp's half of O += P V
#pragma unroll
        for (int kk = 0; kk < KEYS / 16; ++kk) {
            uint32_t a[4];
            a[0] = MmaOp<T>::pack(s[2 * kk][0], s[2 * kk][1]);
            a[1] = MmaOp<T>::pack(s[2 * kk][2], s[2 * kk][3]);
            a[2] = MmaOp<T>::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = MmaOp<T>::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int trow = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int np = 0; np < DVH / 16; ++np) {
                uint32_t bb[4];
                ldmatrix_x4_trans(bb, smem_u32(vb + swz(trow, half * (DVH / 8) + 2 * np +
                                                                  (lane >> 4), VB)));
                MmaOp<T>::run(o[2 * np], a, bb[0], bb[1]);
                MmaOp<T>::run(o[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    T *og = static_cast<T *>(p.o);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float sum = l[hh];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        const int r = r0 + 16 * pr + g + 8 * hh;
        if (r >= ncap) continue;
        const long long row = row_of(r);
        const bool has = r < nvalid && sum > 0.f;
        const float inv = has ? 1.f / sum : 0.f;
#pragma unroll
        for (int j = 0; j < DVH / 8; ++j) {
            const int d = half * DVH + 8 * j + 2 * t;
            if (d < Dv)
                *reinterpret_cast<uint32_t *>(og + row * Dv + d) =
                    MmaOp<T>::pack(o[j][2 * hh] * inv, o[j][2 * hh + 1] * inv);
        }
        if (half == 0 && t == 0 && p.lse != nullptr)
            p.lse[row] = has ? (m[hh] + log2f(sum)) * kLn2 : -INFINITY;
    }
}

template <typename T, int DW, int DVW>
int launch_wide_t(const AttnParams &p, cudaStream_t stream) {
    using L = WideTile<DW, DVW>;
    const long long qtiles = ((long long)p.Q * p.G + kRowsF - 1) / kRowsF;
    const long long grid = qtiles * p.B * p.Hkv;
    if (grid >= (1LL << 31)) {
        set_error("mma forward: %lld blocks exceed one launch", grid);
        return 2;
    }
    auto kern = fwd_mma_wide_kernel<T, DW, DVW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("mma forward (wide): cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    kern<<<(unsigned)grid, 256, L::SMEM, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("mma forward (wide) launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_wide(const AttnParams &p, cudaStream_t stream) {
    // widths padded to 128 / 256 / 512 (each warp's half is at least 64
    // wide); one of D, Dv is above 256 here
    if (p.D <= 128) return launch_wide_t<T, 128, 512>(p, stream);
    if (p.D <= 256) return launch_wide_t<T, 256, 512>(p, stream);
    if (p.Dv <= 128) return launch_wide_t<T, 512, 128>(p, stream);
    if (p.Dv <= 256) return launch_wide_t<T, 512, 256>(p, stream);
    return launch_wide_t<T, 512, 512>(p, stream);
}

template <typename T, int DW, int DVW>
int launch_t(const AttnParams &p, cudaStream_t stream) {
    using L = FwdTile<DW, DVW>;
    const long long qtiles = ((long long)p.Q * p.G + kRowsF - 1) / kRowsF;
    const long long grid = qtiles * p.B * p.Hkv;
    if (grid >= (1LL << 31)) {
        set_error("mma forward: %lld blocks exceed one launch", grid);
        return 2;
    }
    auto kern = fwd_mma_kernel<T, DW, DVW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) {
        set_error("mma forward: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    kern<<<(unsigned)grid, 128, L::SMEM, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("mma forward launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T, int DW>
int launch_dv(const AttnParams &p, cudaStream_t stream) {
    if (p.Dv <= 64) return launch_t<T, DW, 64>(p, stream);
    if (p.Dv <= 128) return launch_t<T, DW, 128>(p, stream);
    return launch_t<T, DW, 256>(p, stream);
}

template <typename T>
int launch_dtype(const AttnParams &p, cudaStream_t stream) {
    if (p.D <= 64) return launch_dv<T, 64>(p, stream);
    if (p.D <= 128) return launch_dv<T, 128>(p, stream);
    return launch_dv<T, 256>(p, stream);
}

}  // namespace

bool fwd_mma_supported(const AttnParams &p, int dtype) {
    return dtype != 0 && p.D % 8 == 0 && p.Dv % 8 == 0 && p.D <= 512 && p.Dv <= 512;
}

int launch_fwd_mma(const AttnParams &p, int dtype, cudaStream_t stream) {
    if (p.D > 256 || p.Dv > 256)
        return dtype == 1 ? launch_wide<__half>(p, stream) : launch_wide<__nv_bfloat16>(p, stream);
    return dtype == 1 ? launch_dtype<__half>(p, stream) : launch_dtype<__nv_bfloat16>(p, stream);
}

}  // namespace attn
