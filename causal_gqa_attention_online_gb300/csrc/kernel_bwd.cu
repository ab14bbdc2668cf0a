// kernel_bwd.cu -- backward of the attention: dQ, dK, dV from dO, the
// forward's O and LSE, recomputing the probabilities.
//
// "Accelerating PyTorch on AMD GPUs with FlyDSL", section on FMHA through
// AOTriton, describes the backward's structure (separate dQ and dK/dV
// kernels, dK/dV as the forward loop transposed with K and V resident and Q
// and dO streamed, dQ's products matching the forward's) but prints no
// arithmetic.  The arithmetic is the derivative of the forward definition
// (O = softmax(scale Q K^T + mask) V with the row LSE kept), per legal (row, key):
//
//     P   = exp(scale q.k - LSE)          (recomputed, no stored P)
//     Dq  = sum_j dO[j] O[j]              (one number per row: bwd_delta_kernel,
//                                          or the tcgen05 dQ kernel for its rows)
//     dP  = dO . v
//     dS  = P (dP - Dq)
//     dQ  = scale sum_k dS k      dK = scale sum_rows dS q      dV = sum_rows P dO
//
// where a KV head's dK / dV sum over all query heads of its group.  Two
// kernels share the recomputation and never write to the same element, so
// there are no atomics and the result does not depend on scheduling:
//   * dK/dV: a block owns a tile of keys of one (sequence, KV head) and walks
//     the rows (all heads of the group) that attend to any of its keys;
//   * dQ: a block owns a tile of flattened (query position, head-in-group)
//     rows and walks the union of their legal keys.
// Each comes as an mma.sync m16n8k16 kernel for bf16 / fp16 (fp32
// accumulation; P and dS rounded to the storage type as MMA operands) and a
// CUDA-core fp32 kernel for fp32 and for head widths the former does not take.
#include <algorithm>
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

// A 1-D grid of (tile, sequence x KV head) blocks, ordered tile rank first:
// every (sequence, KV head)'s rank-0 tile, then every rank-1 tile, ...  The
// kernels give rank 0 to their longest tile, so the long blocks start first
// and the short ones fill the tail of the launch.
__device__ __forceinline__ void block_tile(const AttnParams &p, int &rank, int &ntiles, int &b,
                                           int &kvh) {
    const int nbh = p.B * p.Hkv;
    rank = blockIdx.x / nbh;
    ntiles = gridDim.x / nbh;
    const int bh = blockIdx.x % nbh;
    b = bh / p.Hkv;
    kvh = bh % p.Hkv;
}

// Legal key range of flattened row r of (sequence si, KV head); rows past the
// sequence get the empty range [0, 0).
__device__ __forceinline__ void row_range(const AttnParams &p, const SeqInfo &si, int r,
                                          int &lo, int &hi) {
    lo = hi = 0;
    if (r < si.Qb * p.G) legal_range(r / p.G, si.Qb, si.Kb, p.window, p.mask, lo, hi);
}

// ---------------------------------------------------------------------------
// Dq = rowsum(dO * O), one warp per (token, head) row.

// Dq = rowsum(dO * O), one float a row.  A warp covers kDeltaRows rows: a
// row is split over L lanes of 16-byte loads (L = Dv / 8 rounded up to a power
// of two, at most 32), 32 / L rows a pass, and every load of the warp is
// issued before any arithmetic, so enough bytes are in flight to run at the
// HBM rate (one 256-byte row a warp left it at half of it).
constexpr int kDeltaRows = 8;     // rows per warp
constexpr int kDeltaWarps = 8;    // warps per block

template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BwdParams bp, long long rows) {
    const int lane = threadIdx.x & 31;
    const long long row0 = ((long long)blockIdx.x * kDeltaWarps + (threadIdx.x >> 5)) * kDeltaRows;
    if (row0 >= rows) return;
    const int Dv = bp.f.Dv;
    const T *ob = static_cast<const T *>(bp.f.o);
    const T *gb = static_cast<const T *>(bp.dout);
    constexpr int kVec = 16 / sizeof(T);
    const int nchunk = Dv / kVec;
    if (Dv % kVec == 0 && nchunk <= 32) {
        int L = 1;
        while (L < nchunk) L *= 2;
        const int rpp = 32 / L;  // rows a pass
        const int sub = lane / L, c = lane % L;
        const bool active = c < nchunk;
        constexpr int kMaxPass = kDeltaRows;  // L = 1 .. 32: passes = 8 / rpp <= 8
        uint4 ov[kMaxPass], gv[kMaxPass];
        const int npass = (kDeltaRows + rpp - 1) / rpp;
#pragma unroll
        for (int ps = 0; ps < kMaxPass; ++ps) {
            ov[ps] = gv[ps] = make_uint4(0, 0, 0, 0);
            const long long row = row0 + (long long)ps * rpp + sub;
            if (ps < npass && active && ps * rpp + sub < kDeltaRows && row < rows) {
                ov[ps] = *reinterpret_cast<const uint4 *>(ob + row * Dv + c * kVec);
                gv[ps] = *reinterpret_cast<const uint4 *>(gb + row * Dv + c * kVec);
            }
        }
#pragma unroll
        for (int ps = 0; ps < kMaxPass; ++ps) {
            if (ps >= npass) break;  // uniform
            const T *oe = reinterpret_cast<const T *>(&ov[ps]);
            const T *ge = reinterpret_cast<const T *>(&gv[ps]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc += to_f32(oe[e]) * to_f32(ge[e]);
            for (int off = L / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const long long row = row0 + (long long)ps * rpp + sub;
            if (c == 0 && ps * rpp + sub < kDeltaRows && row < rows) bp.delta[row] = acc;
        }
    } else {
        for (int r = 0; r < kDeltaRows; ++r) {
            const long long row = row0 + r;
            if (row >= rows) break;
            float acc = 0.f;
            for (int j = lane; j < Dv; j += 32)
                acc += to_f32(ob[row * Dv + j]) * to_f32(gb[row * Dv + j]);
            acc = warp_sum(acc);
            if (lane == 0) bp.delta[row] = acc;
        }
    }
}

// ---------------------------------------------------------------------------
// CUDA-core kernels (fp32 math; any storage type, D, Dv <= 256)

constexpr int kGRows = 32;  // dQ: flattened rows per block (8 per warp)
constexpr int kGTK = 32;    // keys per tile (one per lane)

// dQ.  DL = output columns per lane (D <= 32 * DL).
template <typename T, int DL>
__global__ void __launch_bounds__(128) bwd_dq_generic(const BwdParams bp) {
    extern __shared__ __align__(128) uint8_t smem_b[];
    float *smem = reinterpret_cast<float *>(smem_b);
    const AttnParams &p = bp.f;
    const int D = p.D, Dv = p.Dv, G = p.G;
    const int Dp = D | 1, Dvp = Dv | 1;  // odd pitches: lane-per-key reads hit distinct banks
    float *qs = smem;                // [kGRows][D]
    float *dos = qs + kGRows * D;    // [kGRows][Dv]
    float *ks = dos + kGRows * Dv;   // [kGTK][Dp]
    float *vs = ks + kGTK * Dp;      // [kGTK][Dvp]

    int rank, ntiles, b, kvh;
    block_tile(p, rank, ntiles, b, kvh);
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (ntiles - 1 - rank) * kGRows;  // the last rows see the most keys
    if (r0 >= ncap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v), *dog = static_cast<const T *>(bp.dout);

    for (int i = tid; i < kGRows * D; i += blockDim.x) {
        const int r = r0 + i / D;
        float x = 0.f;
        if (r < nvalid)
            x = to_f32(qg[((si.q_off + r / G) * p.Hq + kvh * G + r % G) * (long long)D + i % D]);
        qs[i] = x;
    }
    for (int i = tid; i < kGRows * Dv; i += blockDim.x) {
        const int r = r0 + i / Dv;
        float x = 0.f;
        if (r < nvalid)
            x = to_f32(dog[((si.q_off + r / G) * p.Hq + kvh * G + r % G) * (long long)Dv + i % Dv]);
        dos[i] = x;
    }
    constexpr int kRPW = kGRows / 4;
    int lo[kRPW], hi[kRPW];
    float lse2[kRPW], del[kRPW], acc[kRPW][DL];
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        const int r = r0 + warp * kRPW + i;
        row_range(p, si, r, lo[i], hi[i]);
        lse2[i] = 0.f;
        del[i] = 0.f;
        if (hi[i] > lo[i]) {
            const long long row = (si.q_off + r / G) * p.Hq + kvh * G + r % G;
            lse2[i] = p.lse[row] * kLog2e;
            del[i] = bp.delta[row];
        }
#pragma unroll
        for (int m = 0; m < DL; ++m) acc[i][m] = 0.f;
    }
    // union of the block's legal keys (ranges grow with the row)
    int klo = 0, khi = 0;
    if (nvalid > r0) {
        int a, c;
        legal_range(r0 / G, si.Qb, si.Kb, p.window, p.mask, klo, c);
        legal_range((min(r0 + kGRows, nvalid) - 1) / G, si.Qb, si.Kb, p.window, p.mask, a, khi);
    }
    for (int t0 = klo / kGTK * kGTK; t0 < khi; t0 += kGTK) {
        __syncthreads();
        for (int i = tid; i < kGTK * D; i += blockDim.x) {
            const int key = t0 + i / D;
            ks[(i / D) * Dp + i % D] =
                key < si.Kb ? to_f32(kg[((si.k_off + key) * p.Hkv + kvh) * (long long)D + i % D])
                            : 0.f;
        }
        for (int i = tid; i < kGTK * Dv; i += blockDim.x) {
            const int key = t0 + i / Dv;
            vs[(i / Dv) * Dvp + i % Dv] =
                key < si.Kb ? to_f32(vg[((si.k_off + key) * p.Hkv + kvh) * (long long)Dv + i % Dv])
                            : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kRPW; ++i) {
            if (hi[i] <= lo[i] || hi[i] <= t0 || lo[i] >= t0 + kGTK) continue;  // warp-uniform
            const float *qr = qs + (warp * kRPW + i) * D;
            const float *dr = dos + (warp * kRPW + i) * Dv;
            float s = 0.f, dp = 0.f;
            for (int d = 0; d < D; ++d) s += qr[d] * ks[lane * Dp + d];
            for (int j = 0; j < Dv; ++j) dp += dr[j] * vs[lane * Dvp + j];
            const int key = t0 + lane;
            const bool ok = key >= lo[i] && key < hi[i];
            const float pr = ok ? exp2f(s * p.scale_log2 - lse2[i]) : 0.f;
            const float ds = pr * (dp - del[i]);
            for (int jj = 0; jj < kGTK; ++jj) {
                const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
                for (int m = 0; m < DL; ++m) {
                    const int d = lane + 32 * m;
                    if (d < D) acc[i][m] += dsj * ks[jj * Dp + d];
                }
            }
        }
    }
    T *dqg = static_cast<T *>(bp.dq);
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        const int r = r0 + warp * kRPW + i;
        if (r >= ncap) continue;
        const long long row = (si.q_off + r / G) * p.Hq + kvh * G + r % G;
#pragma unroll
        for (int m = 0; m < DL; ++m) {
            const int d = lane + 32 * m;
            if (d < D) dqg[row * D + d] = from_f32<T>(r < nvalid ? acc[i][m] * p.scale : 0.f);
        }
    }
}

// dK / dV.  A block owns kGTK keys (one per lane); warp w accumulates the
// columns d = w + 4m (m < DL) of dK and dV for every key.  Rows are taken
// four at a time, one per warp, through shared memory.
template <typename T, int DL>
__global__ void __launch_bounds__(128) bwd_dkdv_generic(const BwdParams bp) {
    extern __shared__ __align__(128) uint8_t smem_b[];
    float *smem = reinterpret_cast<float *>(smem_b);
    const AttnParams &p = bp.f;
    const int D = p.D, Dv = p.Dv, G = p.G;
    const int Dp = D | 1, Dvp = Dv | 1;
    float *ks = smem;               // [kGTK][Dp]
    float *vs = ks + kGTK * Dp;     // [kGTK][Dvp]
    float *qr = vs + kGTK * Dvp;    // [4][D]
    float *dr = qr + 4 * D;         // [4][Dv]
    float *pw = dr + 4 * Dv;        // [4][kGTK]
    float *dsw = pw + 4 * kGTK;     // [4][kGTK]

    int rank, ntiles, b, kvh;
    block_tile(p, rank, ntiles, b, kvh);
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int kcap = packed ? si.Kb : p.K;
    const int k0 = rank * kGTK;  // the first keys are seen by the most rows
    if (k0 >= kcap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v), *dog = static_cast<const T *>(bp.dout);

    for (int i = tid; i < kGTK * D; i += blockDim.x) {
        const int key = k0 + i / D;
        ks[(i / D) * Dp + i % D] =
            key < si.Kb ? to_f32(kg[((si.k_off + key) * p.Hkv + kvh) * (long long)D + i % D]) : 0.f;
    }
    for (int i = tid; i < kGTK * Dv; i += blockDim.x) {
        const int key = k0 + i / Dv;
        vs[(i / Dv) * Dvp + i % Dv] =
            key < si.Kb ? to_f32(vg[((si.k_off + key) * p.Hkv + kvh) * (long long)Dv + i % Dv])
                        : 0.f;
    }
    float acck[DL], accv[DL];
#pragma unroll
    for (int m = 0; m < DL; ++m) acck[m] = accv[m] = 0.f;
    int rf = 0, re = 0;
    if (k0 < si.Kb) {
        int qf, qe;
        rows_for_keys(k0, min(k0 + kGTK, si.Kb), si.Qb, si.Kb, p.window, p.mask, qf, qe);
        if (qe > qf) {
            rf = qf * G;
            re = qe * G;
        }
    }
    for (int base = rf; base < re; base += 4) {
        __syncthreads();  // the previous rows' readers are done (and K / V staged)
        const int r = base + warp;
        int lo, hi;
        row_range(p, si, r < re ? r : INT_MAX, lo, hi);
        const long long row = (si.q_off + r / G) * p.Hq + kvh * G + r % G;
        const bool has = r < re && hi > lo;
        for (int d = lane; d < D; d += 32)
            qr[warp * D + d] = has ? to_f32(qg[row * D + d]) : 0.f;
        for (int j = lane; j < Dv; j += 32)
            dr[warp * Dv + j] = has ? to_f32(dog[row * Dv + j]) : 0.f;
        __syncwarp();
        float pr = 0.f, ds = 0.f;
        if (has) {
            float s = 0.f, dp = 0.f;
            for (int d = 0; d < D; ++d) s += qr[warp * D + d] * ks[lane * Dp + d];
            for (int j = 0; j < Dv; ++j) dp += dr[warp * Dv + j] * vs[lane * Dvp + j];
            const int key = k0 + lane;
            if (key >= lo && key < hi) {
                pr = exp2f(s * p.scale_log2 - p.lse[row] * kLog2e);
                ds = pr * (dp - bp.delta[row]);
            }
        }
        pw[warp * kGTK + lane] = pr;
        dsw[warp * kGTK + lane] = ds;
        __syncthreads();
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
            const float pv = pw[w2 * kGTK + lane], dsv = dsw[w2 * kGTK + lane];
#pragma unroll
            for (int m = 0; m < DL; ++m) {
                const int d = warp + 4 * m;
                if (d < D) acck[m] += dsv * qr[w2 * D + d];
                if (d < Dv) accv[m] += pv * dr[w2 * Dv + d];
            }
        }
    }
    const int key = k0 + lane;
    if (key < kcap) {
        T *dkg = static_cast<T *>(bp.dk), *dvg = static_cast<T *>(bp.dv);
        const long long krow = (si.k_off + key) * p.Hkv + kvh;
#pragma unroll
        for (int m = 0; m < DL; ++m) {
            const int d = warp + 4 * m;
            if (d < D) dkg[krow * D + d] = from_f32<T>(acck[m] * p.scale);
            if (d < Dv) dvg[krow * Dv + d] = from_f32<T>(accv[m]);
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor-core kernels (bf16 / fp16; D, Dv multiples of 8 up to 128, staged
// in 64- or 128-column tiles whose unused columns are zero-filled).
//
// Tiles live in shared memory as rows of 16-byte chunks, XOR-swizzled by the
// row (swz), and are read with ldmatrix: plain for operands whose contraction
// index runs along the stored row, transposed (.trans) otherwise.  An MMA's
// fp32 accumulator for two adjacent 8-column tiles has exactly the register
// layout of the A operand of a 16-deep contraction, so P and dS go from one
// product to the next through registers (pack to the storage type).

constexpr int kMKeys = 64;   // dK/dV: keys per block (16 per warp)
constexpr int kMRows = 32;   // dK/dV: rows per step
constexpr int kMStages = 3;  // dK/dV: row-tile ring depth
constexpr int kQRows = 64;   // dQ: rows per block (16 per warp)
constexpr int kQKeys = 64;   // dQ: keys per step

// Copies `nrows` rows of W columns into swizzled shared memory with
// cp.async; src(r) gives the global address of row r, or nullptr for a row
// of zeros.  Columns at or past `cols` are zero-filled.  Zero-filled chunks
// read nothing; they are given `base` (a valid address) all the same.
template <typename T, int W, int NT = 128, typename Src>
__device__ __forceinline__ void stage_rows(uint8_t *dst, int nrows, int cols, int tid,
                                           const T *base, Src src) {
    constexpr int kChunks = W / 8;
    for (int c = tid; c < nrows * kChunks; c += NT) {
        const int r = c / kChunks, ch = c % kChunks;
        const T *g = src(r);
        const bool ok = g != nullptr && ch * 8 < cols;
        cp_async16(smem_u32(dst + swz(r, ch, W * 2)), ok ? g + ch * 8 : base, ok ? 16 : 0);
    }
}

// dK / dV.  A block owns kMKeys keys of one (sequence, KV head) and walks,
// kMRows at a time, the flattened rows of the group that attend to them.
// Warps come in pairs over the same 16 keys, each pair splitting the work of
// a step in two halves of equal MMA count:
//   P warp  (w < 4):  S^T = K Q^T,  P^T = exp2(S^T scale_log2 - LSE_2),  dV += P^T dO
//   dS warp (w >= 4): dP^T = V dO^T, dS^T = P^T (dP^T - Dq),            dK += dS^T Q
// P^T goes from one to the other through shared memory in the MMA
// accumulator layout (both warps' fragments map lane / register to the same
// (key, row)), behind a 64-thread named barrier per pair.  Each warp keeps one
// 16 x 128 fp32 accumulator, so two blocks of eight warps fit an SM.
template <typename T, int DW, int DVW>
__global__ void __launch_bounds__(256, 2) bwd_dkdv_mma(const BwdParams bp) {
    constexpr int NT = 256;
    extern __shared__ __align__(128) uint8_t smem_b[];
    uint8_t *smem = smem_b;
    const AttnParams &p = bp.f;
    constexpr int KB = DW * 2, VB = DVW * 2;  // bytes per staged row
    uint8_t *ks = smem;                        // [kMKeys][KB]
    uint8_t *vs = ks + kMKeys * KB;            // [kMKeys][VB]
    uint8_t *qs = vs + kMKeys * VB;                   // [kMStages][kMRows][KB]
    uint8_t *dos = qs + kMStages * kMRows * KB;       // [kMStages][kMRows][VB]
    float *pbuf = reinterpret_cast<float *>(dos + kMStages * kMRows * VB);  // [4][16][32]
    float *lse_s = pbuf + 4 * 16 * 32;                // [kMStages][kMRows]
    float *del_s = lse_s + kMStages * kMRows;         // [kMStages][kMRows]
    int *lo_s = reinterpret_cast<int *>(del_s + kMStages * kMRows);
    int *hi_s = lo_s + kMStages * kMRows;
    int *flag_s = hi_s + kMStages * kMRows;          // [kMStages]: step needs no mask

    int rank, ntiles, b, kvh;
    block_tile(p, rank, ntiles, b, kvh);
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int kcap = packed ? si.Kb : p.K;
    const int k0 = rank * kMKeys;  // the first keys are seen by the most rows
    if (k0 >= kcap) return;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const bool pwarp = warp < 4;
    const int kw = 16 * (warp & 3);  // this pair's first key in the tile
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v), *dog = static_cast<const T *>(bp.dout);

    stage_rows<T, DW, NT>(ks, kMKeys, D, tid, kg, [&](int r) -> const T * {
        const int key = k0 + r;
        return key < si.Kb ? kg + ((si.k_off + key) * p.Hkv + kvh) * (long long)D : nullptr;
    });
    stage_rows<T, DVW, NT>(vs, kMKeys, Dv, tid, vg, [&](int r) -> const T * {
        const int key = k0 + r;
        return key < si.Kb ? vg + ((si.k_off + key) * p.Hkv + kvh) * (long long)Dv : nullptr;
    });
    int rf = 0, re = 0;
    if (k0 < si.Kb) {
        int qf, qe;
        rows_for_keys(k0, min(k0 + kMKeys, si.Kb), si.Qb, si.Kb, p.window, p.mask, qf, qe);
        if (qe > qf) {
            rf = qf * G;
            re = qe * G;
        }
    }
    const int nsteps = (re - rf + kMRows - 1) / kMRows;

    // Row r of a tile is copied by the threads tid / kCh == r (mod NT / kCh),
    // one 16-byte chunk each; a thread finds its rows' addresses once a step.
    constexpr int kChQ = DW / 8, kChO = DVW / 8;
    auto row_of = [&](int r) { return (si.q_off + r / G) * p.Hq + kvh * G + r % G; };
    auto load_rows = [&](int step, int buf) {
        const int rb = rf + step * kMRows;
        uint8_t *qd = qs + buf * kMRows * KB;
        uint8_t *od = dos + buf * kMRows * VB;
        if constexpr (kChQ == kChO) {
#pragma unroll
            for (int i = tid / kChQ; i < kMRows; i += NT / kChQ) {
                const int r = rb + i, ch = tid % kChQ;
                const long long row = r < re ? row_of(r) : 0;
                const bool okq = r < re && ch * 8 < D, oko = r < re && ch * 8 < Dv;
                cp_async16(smem_u32(qd + swz(i, ch, KB)), okq ? qg + row * D + ch * 8 : qg,
                           okq ? 16 : 0);
                cp_async16(smem_u32(od + swz(i, ch, VB)), oko ? dog + row * Dv + ch * 8 : dog,
                           oko ? 16 : 0);
            }
        } else {
#pragma unroll
            for (int i = tid / kChQ; i < kMRows; i += NT / kChQ) {
                const int r = rb + i, ch = tid % kChQ;
                const bool ok = r < re && ch * 8 < D;
                cp_async16(smem_u32(qd + swz(i, ch, KB)), ok ? qg + row_of(r) * D + ch * 8 : qg,
                           ok ? 16 : 0);
            }
#pragma unroll
            for (int i = tid / kChO; i < kMRows; i += NT / kChO) {
                const int r = rb + i, ch = tid % kChO;
                const bool ok = r < re && ch * 8 < Dv;
                cp_async16(smem_u32(od + swz(i, ch, VB)),
                           ok ? dog + row_of(r) * Dv + ch * 8 : dog, ok ? 16 : 0);
            }
        }
        if (tid < kMRows) {
            // LSE and Dq travel with the tile (no thread waits on them here);
            // rows without a legal key read nothing and are masked by [lo, hi)
            const int r = rb + tid;
            int lo = 0, hi = 0;
            if (r < re) row_range(p, si, r, lo, hi);
            const bool ok = hi > lo;
            const long long row = ok ? row_of(r) : 0;
            cp_async4(smem_u32(lse_s + buf * kMRows + tid), p.lse + row, ok ? 4 : 0);
            cp_async4(smem_u32(del_s + buf * kMRows + tid), bp.delta + row, ok ? 4 : 0);
            lo_s[buf * kMRows + tid] = lo;
            hi_s[buf * kMRows + tid] = hi;
            // the step needs no mask when every row sees all of the tile's keys
            const bool inner = lo <= k0 && hi >= k0 + kMKeys;
            const unsigned all = __ballot_sync(0xffffffffu, inner);
            if (tid == 0) flag_s[buf] = all == 0xffffffffu;
        }
    };

    // a ring of three row tiles: the tile loaded during step i was last read
    // in step i - 1, which every thread has left at step i's barrier
    if (nsteps > 0) load_rows(0, 0);
    cp_async_commit();
    if (nsteps > 1) load_rows(1, 1);
    cp_async_commit();

    // P warps accumulate dV (DVW columns), dS warps dK (DW columns)
    constexpr int kAcc = (DW > DVW ? DW : DVW) / 8;
    float acc[kAcc][4];
#pragma unroll
    for (int j = 0; j < kAcc; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float *pmine = pbuf + (warp & 3) * 16 * 32;

    for (int step = 0; step < nsteps; ++step) {
        cp_async_wait<1>();  // step's tile has landed (step + 1's may be in flight)
        __syncthreads();
        if (step + 2 < nsteps) load_rows(step + 2, (step + 2) % kMStages);
        cp_async_commit();
        const int buf = step % kMStages;
        const uint8_t *qb = qs + buf * kMRows * KB;
        const uint8_t *db = dos + buf * kMRows * VB;
        // S^T = K Q^T (P warps) or dP^T = V dO^T (dS warps): 16 keys x 32 rows
        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        if (pwarp) {
#pragma unroll
            for (int kk = 0; kk < DW / 16; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(a, smem_u32(ks + swz(kw + (lane & 15), 2 * kk + (lane >> 4), KB)));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bq[4];
                    ldmatrix_x4(bq, smem_u32(qb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                      2 * kk + ((lane >> 3) & 1), KB)));
                    MmaOp<T>::run(s[2 * np], a, bq[0], bq[1]);
                    MmaOp<T>::run(s[2 * np + 1], a, bq[2], bq[3]);
                }
            }
            const bool inner = flag_s[buf] != 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int rl = buf * kMRows + 8 * j + 2 * t + cc;
                    const float l2 = lse_s[rl] * kLog2e;
                    int lo = INT_MIN, hi = INT_MAX;
                    if (!inner) {
                        lo = lo_s[rl];
                        hi = hi_s[rl];
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int c = 2 * hh + cc;
                        const int key = k0 + kw + g + 8 * hh;
                        s[j][c] = key >= lo && key < hi ? exp2f(s[j][c] * p.scale_log2 - l2) : 0.f;
                        pmine[(j * 4 + c) * 32 + lane] = s[j][c];
                    }
                }
            sm100::named_bar_arrive(1 + (warp & 3), 64);
        } else {
#pragma unroll
            for (int kk = 0; kk < DVW / 16; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(a, smem_u32(vs + swz(kw + (lane & 15), 2 * kk + (lane >> 4), VB)));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bq[4];
                    ldmatrix_x4(bq, smem_u32(db + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                      2 * kk + ((lane >> 3) & 1), VB)));
                    MmaOp<T>::run(s[2 * np], a, bq[0], bq[1]);
                    MmaOp<T>::run(s[2 * np + 1], a, bq[2], bq[3]);
                }
            }
            sm100::named_bar_sync(1 + (warp & 3), 64);  // the partner's P^T is in pmine
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int rl = buf * kMRows + 8 * j + 2 * t + (c & 1);
                    s[j][c] = pmine[(j * 4 + c) * 32 + lane] * (s[j][c] - del_s[rl]);
                }
        }
        // dV += P^T dO (P warps) or dK += dS^T Q (dS warps), over the 32 rows
        const uint8_t *bsrc = pwarp ? db : qb;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint32_t pa[4];
            pa[0] = MmaOp<T>::pack(s[2 * m][0], s[2 * m][1]);
            pa[1] = MmaOp<T>::pack(s[2 * m][2], s[2 * m][3]);
            pa[2] = MmaOp<T>::pack(s[2 * m + 1][0], s[2 * m + 1][1]);
            pa[3] = MmaOp<T>::pack(s[2 * m + 1][2], s[2 * m + 1][3]);
            const int trow = 16 * m + (lane & 7) + (((lane >> 3) & 1) << 3);
            if (pwarp) {
#pragma unroll
                for (int np = 0; np < DVW / 16; ++np) {
                    uint32_t bb[4];
                    ldmatrix_x4_trans(bb, smem_u32(bsrc + swz(trow, 2 * np + (lane >> 4), VB)));
                    MmaOp<T>::run(acc[2 * np], pa, bb[0], bb[1]);
                    MmaOp<T>::run(acc[2 * np + 1], pa, bb[2], bb[3]);
                }
            } else {
#pragma unroll
                for (int np = 0; np < DW / 16; ++np) {
                    uint32_t bb[4];
                    ldmatrix_x4_trans(bb, smem_u32(bsrc + swz(trow, 2 * np + (lane >> 4), KB)));
                    MmaOp<T>::run(acc[2 * np], pa, bb[0], bb[1]);
                    MmaOp<T>::run(acc[2 * np + 1], pa, bb[2], bb[3]);
                }
            }
        }
    }
    cp_async_wait<0>();

    // keys past the sequence (padded layout) come out as zeros: P = dS = 0 there
    T *dst = static_cast<T *>(pwarp ? bp.dv : bp.dk);
    const int width = pwarp ? Dv : D;
    const float sc = pwarp ? 1.f : p.scale;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int key = k0 + kw + g + 8 * hh;
        if (key >= kcap) continue;
        const long long krow = (si.k_off + key) * p.Hkv + kvh;
#pragma unroll
        for (int j = 0; j < kAcc; ++j) {
            const int d = 8 * j + 2 * t;
            if (d < width)
                *reinterpret_cast<uint32_t *>(dst + krow * width + d) =
                    MmaOp<T>::pack(acc[j][2 * hh] * sc, acc[j][2 * hh + 1] * sc);
        }
    }
}

template <typename T, int DW, int DVW>
__global__ void __launch_bounds__(128) bwd_dq_mma(const BwdParams bp) {
    extern __shared__ __align__(128) uint8_t smem_b[];
    uint8_t *smem = smem_b;
    const AttnParams &p = bp.f;
    constexpr int KB = DW * 2, VB = DVW * 2;
    uint8_t *qs = smem;                     // [kQRows][KB]
    uint8_t *dos = qs + kQRows * KB;        // [kQRows][VB]
    uint8_t *ks = dos + kQRows * VB;        // [2][kQKeys][KB]
    uint8_t *vs = ks + 2 * kQKeys * KB;     // [2][kQKeys][VB]

    int rank, ntiles_q, b, kvh;
    block_tile(p, rank, ntiles_q, b, kvh);
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (ntiles_q - 1 - rank) * kQRows;  // the last rows see the most keys
    if (r0 >= ncap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v), *dog = static_cast<const T *>(bp.dout);
    auto row_of = [&](int r) { return (si.q_off + r / G) * p.Hq + kvh * G + r % G; };

    stage_rows<T, DW>(qs, kQRows, D, tid, qg, [&](int i) -> const T * {
        const int r = r0 + i;
        return r < nvalid ? qg + row_of(r) * D : nullptr;
    });
    stage_rows<T, DVW>(dos, kQRows, Dv, tid, dog, [&](int i) -> const T * {
        const int r = r0 + i;
        return r < nvalid ? dog + row_of(r) * Dv : nullptr;
    });
    // this thread's two rows: 16 * warp + g and + 8
    int lo[2], hi[2];
    float l2[2], dl[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 16 * warp + g + 8 * hh;
        row_range(p, si, r, lo[hh], hi[hh]);
        l2[hh] = dl[hh] = 0.f;
        if (hi[hh] > lo[hh]) {
            l2[hh] = p.lse[row_of(r)] * kLog2e;
            dl[hh] = bp.delta[row_of(r)];
        }
    }
    int klo = 0, khi = 0;
    if (nvalid > r0) {
        int a, c;
        legal_range(r0 / G, si.Qb, si.Kb, p.window, p.mask, klo, c);
        legal_range((min(r0 + kQRows, nvalid) - 1) / G, si.Qb, si.Kb, p.window, p.mask, a, khi);
    }
    const int tfirst = klo / kQKeys * kQKeys;
    const int ntiles = khi > klo ? (khi - tfirst + kQKeys - 1) / kQKeys : 0;
    auto load_kv = [&](int i, int buf) {
        const int kt0 = tfirst + i * kQKeys;
        stage_rows<T, DW>(ks + buf * kQKeys * KB, kQKeys, D, tid, kg, [&](int r) -> const T * {
            const int key = kt0 + r;
            return key < si.Kb ? kg + ((si.k_off + key) * p.Hkv + kvh) * (long long)D : nullptr;
        });
        stage_rows<T, DVW>(vs + buf * kQKeys * VB, kQKeys, Dv, tid, vg, [&](int r) -> const T * {
            const int key = kt0 + r;
            return key < si.Kb ? vg + ((si.k_off + key) * p.Hkv + kvh) * (long long)Dv : nullptr;
        });
    };
    if (ntiles > 0) load_kv(0, 0);
    cp_async_commit();

    float dq[DW / 8][4];
#pragma unroll
    for (int j = 0; j < DW / 8; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = 0.f;

    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            load_kv(i + 1, (i + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int buf = i & 1;
        const uint8_t *kb = ks + buf * kQKeys * KB;
        const uint8_t *vb = vs + buf * kQKeys * VB;
        const int kt0 = tfirst + i * kQKeys;
        // S = Q K^T and dP = dO V^T for this warp's 16 rows x 64 keys
        float s[8][4], dp[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[j][c] = dp[j][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < (DW > DVW ? DW : DVW) / 16; ++kk) {
            if (kk < DW / 16) {
                uint32_t a[4];
                ldmatrix_x4(a, smem_u32(qs + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), KB)));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t bk[4];
                    ldmatrix_x4(bk, smem_u32(kb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                      2 * kk + ((lane >> 3) & 1), KB)));
                    MmaOp<T>::run(s[2 * np], a, bk[0], bk[1]);
                    MmaOp<T>::run(s[2 * np + 1], a, bk[2], bk[3]);
                }
            }
            if (kk < DVW / 16) {
                uint32_t a[4];
                ldmatrix_x4(a, smem_u32(dos + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), VB)));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t bv[4];
                    ldmatrix_x4(bv, smem_u32(vb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                      2 * kk + ((lane >> 3) & 1), VB)));
                    MmaOp<T>::run(dp[2 * np], a, bv[0], bv[1]);
                    MmaOp<T>::run(dp[2 * np + 1], a, bv[2], bv[3]);
                }
            }
        }
        // dS (in s); no mask where all of the warp's rows see the whole tile
        const bool inner = __all_sync(0xffffffffu, lo[0] <= kt0 && lo[1] <= kt0 &&
                                                       hi[0] >= kt0 + kQKeys &&
                                                       hi[1] >= kt0 + kQKeys);
        if (inner) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int hh = c >> 1;
                    s[j][c] = exp2f(s[j][c] * p.scale_log2 - l2[hh]) * (dp[j][c] - dl[hh]);
                }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int hh = c >> 1;
                    const int key = kt0 + 8 * j + 2 * t + (c & 1);
                    const bool ok = key >= lo[hh] && key < hi[hh];
                    const float pr = ok ? exp2f(s[j][c] * p.scale_log2 - l2[hh]) : 0.f;
                    s[j][c] = pr * (dp[j][c] - dl[hh]);
                }
        }
        // dQ += dS K, contracting over the 64 keys
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t a[4];
            a[0] = MmaOp<T>::pack(s[2 * m][0], s[2 * m][1]);
            a[1] = MmaOp<T>::pack(s[2 * m][2], s[2 * m][3]);
            a[2] = MmaOp<T>::pack(s[2 * m + 1][0], s[2 * m + 1][1]);
            a[3] = MmaOp<T>::pack(s[2 * m + 1][2], s[2 * m + 1][3]);
            const int trow = 16 * m + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int np = 0; np < DW / 16; ++np) {
                uint32_t bb[4];
                ldmatrix_x4_trans(bb, smem_u32(kb + swz(trow, 2 * np + (lane >> 4), KB)));
                MmaOp<T>::run(dq[2 * np], a, bb[0], bb[1]);
                MmaOp<T>::run(dq[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    T *dqg = static_cast<T *>(bp.dq);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 16 * warp + g + 8 * hh;
        if (r >= ncap) continue;
        const long long row = row_of(r);
        const float sc = r < nvalid ? p.scale : 0.f;
#pragma unroll
        for (int j = 0; j < DW / 8; ++j) {
            const int d = 8 * j + 2 * t;
            if (d < D)
                *reinterpret_cast<uint32_t *>(dqg + row * D + d) =
                    MmaOp<T>::pack(dq[j][2 * hh] * sc, dq[j][2 * hh + 1] * sc);
        }
    }
}

// ---------------------------------------------------------------------------
// launchers

template <typename... Args>
int launch_k(void (*kern)(Args...), dim3 grid, int block, size_t smem, cudaStream_t stream,
             const char *name, Args... args) {
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            set_error("%s: cudaFuncSetAttribute: %s", name, cudaGetErrorString(e));
            return 3;
        }
    }
    kern<<<grid, block, smem, stream>>>(args...);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s launch: %s", name, cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

// A 1-D grid of tiles x (sequence, KV head) blocks must stay below 2^31.
bool grid_fits(long long tiles, unsigned bh) {
    if (tiles * (long long)bh < (1LL << 31)) return true;
    set_error("backward: %lld tiles x %u (sequence, KV head) pairs exceed one launch", tiles, bh);
    return false;
}

int pow2_at_least(int x, int lo) {
    int v = lo;
    while (v < x) v *= 2;
    return v;
}

template <typename T, int DL>
int launch_generic_bwd_t(const BwdParams &bp, cudaStream_t stream) {
    const AttnParams &p = bp.f;
    const int D = p.D, Dv = p.Dv;
    const unsigned y = (unsigned)p.B * p.Hkv;
    const size_t s_dkdv = sizeof(float) * ((size_t)kGTK * ((D | 1) + (Dv | 1)) + 4 * (D + Dv) +
                                           8 * kGTK);
    const long long ktiles = ((long long)p.K + kGTK - 1) / kGTK;
    if (!grid_fits(ktiles, y) || !grid_fits(((long long)p.Q * p.G + kGRows - 1) / kGRows, y))
        return 2;
    int rc = 0;
    if (ktiles > 0) {
        rc = launch_k(bwd_dkdv_generic<T, DL>, dim3((unsigned)(ktiles * y)), 128, s_dkdv, stream,
                      "bwd_dkdv_generic", bp);
        if (rc) return rc;
    }
    const size_t s_dq = sizeof(float) * ((size_t)kGRows * (D + Dv) + (size_t)kGTK * ((D | 1) + (Dv | 1)));
    const long long qtiles = ((long long)p.Q * p.G + kGRows - 1) / kGRows;
    constexpr int DQL = DL / 8;  // D <= 4 * DL = 32 * DQL
    return launch_k(bwd_dq_generic<T, DQL>, dim3((unsigned)(qtiles * y)), 128, s_dq, stream,
                    "bwd_dq_generic", bp);
}

template <typename T>
int launch_generic_bwd(const BwdParams &bp, cudaStream_t stream) {
    const int w = pow2_at_least((std::max)(bp.f.D, bp.f.Dv), 32);  // 32 .. 256
    switch (w) {
        case 32: return launch_generic_bwd_t<T, 8>(bp, stream);
        case 64: return launch_generic_bwd_t<T, 16>(bp, stream);
        case 128: return launch_generic_bwd_t<T, 32>(bp, stream);
        default: return launch_generic_bwd_t<T, 64>(bp, stream);
    }
}

template <typename T>
int launch_delta(const BwdParams &bp, cudaStream_t stream);

template <typename T, int DW, int DVW>
int launch_mma_bwd_t(const BwdParams &bp, bool tc_dq, cudaStream_t stream) {
    const AttnParams &p = bp.f;
    const unsigned y = (unsigned)p.B * p.Hkv;
    const long long ktiles = ((long long)p.K + kMKeys - 1) / kMKeys;
    if (!grid_fits(ktiles, y) || !grid_fits(((long long)p.Q * p.G + kQRows - 1) / kQRows, y))
        return 2;
    int rc = 0;
    const int dt = std::is_same<T, __half>::value ? 1 : 2;
    if (ktiles > 0 && tc_dq && bwd_dkdv_tc_supported(p, dt)) {
        // The dQ kernel computes Dq = rowsum(dO * O) of its rows itself (from
        // the dO tile it stages anyway and O's tile, staged in ring slots before
        // their first K / V tile) and writes it; the dK/dV kernel, launched as
        // its programmatic dependent, sets up on the SMs the dQ kernel's last
        // CTAs free and waits for that grid before reading Dq.  No Dq launch.
        rc = launch_bwd_dq_tc(bp, dt, stream, 2);
        if (rc) return rc;
        return launch_bwd_dkdv_tc(bp, dt, stream, true);
    }
    rc = launch_delta<T>(bp, stream);
    if (rc) return rc;
    if (ktiles > 0) {
        const size_t s = (size_t)kMKeys * 2 * (DW + DVW) +
                         (size_t)kMStages * kMRows * (2 * (DW + DVW) + 16) + 4 * 16 * 32 * 4 +
                         kMStages * 4;
        rc = launch_k(bwd_dkdv_mma<T, DW, DVW>, dim3((unsigned)(ktiles * y)), 256, s, stream,
                      "bwd_dkdv_mma", bp);
        if (rc) return rc;
    }
    if (tc_dq) return launch_bwd_dq_tc(bp, dt, stream, 0);
    const size_t s = (size_t)kQRows * 2 * (DW + DVW) + (size_t)2 * kQKeys * 2 * (DW + DVW);
    const long long qtiles = ((long long)p.Q * p.G + kQRows - 1) / kQRows;
    return launch_k(bwd_dq_mma<T, DW, DVW>, dim3((unsigned)(qtiles * y)), 128, s, stream,
                    "bwd_dq_mma", bp);
}

template <typename T>
int launch_mma_bwd(const BwdParams &bp, bool tc_dq, cudaStream_t stream) {
    const bool wd = bp.f.D > 64, wv = bp.f.Dv > 64;
    if (wd && wv) return launch_mma_bwd_t<T, 128, 128>(bp, tc_dq, stream);
    if (wd) return launch_mma_bwd_t<T, 128, 64>(bp, tc_dq, stream);
    if (wv) return launch_mma_bwd_t<T, 64, 128>(bp, tc_dq, stream);
    return launch_mma_bwd_t<T, 64, 64>(bp, tc_dq, stream);
}

template <typename T>
int launch_delta(const BwdParams &bp, cudaStream_t stream) {
    const long long rows = bp.f.Tq * bp.f.Hq;
    const long long per_block = (long long)kDeltaWarps * kDeltaRows;
    return launch_k(bwd_delta_kernel<T>, dim3((unsigned)((rows + per_block - 1) / per_block)), 256,
                    0, stream, "bwd_delta", bp, rows);
}

template <typename T>
int launch_bwd_t(const BwdParams &bp, int mode, cudaStream_t stream) {
    if constexpr (!std::is_same<T, float>::value) {
        if (mode != 0) return launch_mma_bwd<T>(bp, mode == 2, stream);
    }
    const int rc = launch_delta<T>(bp, stream);
    if (rc) return rc;
    return launch_generic_bwd<T>(bp, stream);
}

}  // namespace

bool bwd_mma_supported(const AttnParams &p, int dtype) {
    return dtype != 0 && p.D % 8 == 0 && p.Dv % 8 == 0 && p.D <= 128 && p.Dv <= 128;
}

int launch_bwd(const BwdParams &bp, int dtype, int mode, cudaStream_t stream) {
    if (bp.f.Tq * bp.f.Hq == 0) return 0;
    switch (dtype) {
        case 0: return launch_bwd_t<float>(bp, 0, stream);
        case 1: return launch_bwd_t<__half>(bp, mode, stream);
        default: return launch_bwd_t<__nv_bfloat16>(bp, mode, stream);
    }
}

}  // namespace attn
