// kernel_bwd.cu -- backward of the attention: dQ, dK, dV from dO, the
// forward's O and LSE, recomputing the probabilities.
//
// The pages give the forward only ("Online softmax" / "FlashAttention"
// passages: O = softmax(scale Q K^T + mask) V with the row LSE kept).  The
// backward is the derivative of that definition, per legal (row, key):
//
//     P   = exp(scale q.k - LSE)          (recomputed, no stored P)
//     Dq  = sum_j dO[j] O[j]              (one number per row: bwd_delta_kernel)
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

namespace attn {
namespace {

// Query positions [qf, qe) of a sequence that have a legal key in [k0, k1)
// (k0 < k1 <= Kb); empty when qe <= qf.  The causal masks' ranges
// [lo(qi), hi(qi)) both grow with qi, so the set is an interval.
__device__ __forceinline__ void rows_for_keys(int k0, int k1, int Qb, int Kb, int window,
                                              int mask, int &qf, int &qe) {
    if (mask == 2) {
        qf = 0;
        qe = Qb;
        return;
    }
    const int off = mask == 1 ? 0 : Kb - Qb;  // diagonal key of row qi is qi + off
    qf = max(0, k0 - off);                     // hi(qi) > k0  <=>  qi + off >= k0
    qe = Qb;
    if (window > 0) qe = min(Qb, k1 + window - 1 - off);  // lo(qi) < k1
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

template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BwdParams bp, long long rows) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int Dv = bp.f.Dv;
    const T *o = static_cast<const T *>(bp.f.o) + row * Dv;
    const T *g = static_cast<const T *>(bp.dout) + row * Dv;
    float acc = 0.f;
    constexpr int kVec = 16 / sizeof(T);
    if (Dv % kVec == 0) {
        for (int j = lane * kVec; j < Dv; j += 32 * kVec) {
            const uint4 ov = *reinterpret_cast<const uint4 *>(o + j);
            const uint4 gv = *reinterpret_cast<const uint4 *>(g + j);
            const T *oe = reinterpret_cast<const T *>(&ov);
            const T *ge = reinterpret_cast<const T *>(&gv);
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc += to_f32(oe[e]) * to_f32(ge[e]);
        }
    } else {
        for (int j = lane; j < Dv; j += 32) acc += to_f32(o[j]) * to_f32(g[j]);
    }
    acc = warp_sum(acc);
    if (lane == 0) bp.delta[row] = acc;
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

    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (gridDim.x - 1 - blockIdx.x) * kGRows;  // longest rows first
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

    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int kcap = packed ? si.Kb : p.K;
    const int k0 = blockIdx.x * kGTK;
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
constexpr int kQRows = 64;   // dQ: rows per block (16 per warp)
constexpr int kQKeys = 64;   // dQ: keys per step

// Copies `nrows` rows of W columns into swizzled shared memory with
// cp.async; src(r) gives the global address of row r, or nullptr for a row
// of zeros.  Columns at or past `cols` are zero-filled.  Zero-filled chunks
// read nothing; they are given `base` (a valid address) all the same.
template <typename T, int W, typename Src>
__device__ __forceinline__ void stage_rows(uint8_t *dst, int nrows, int cols, int tid,
                                           const T *base, Src src) {
    constexpr int kChunks = W / 8;
    for (int c = tid; c < nrows * kChunks; c += 128) {
        const int r = c / kChunks, ch = c % kChunks;
        const T *g = src(r);
        const bool ok = g != nullptr && ch * 8 < cols;
        cp_async16(smem_u32(dst + swz(r, ch, W * 2)), ok ? g + ch * 8 : base, ok ? 16 : 0);
    }
}

template <typename T, int DW, int DVW>
__global__ void __launch_bounds__(128) bwd_dkdv_mma(const BwdParams bp) {
    extern __shared__ __align__(128) uint8_t smem_b[];
    uint8_t *smem = smem_b;
    const AttnParams &p = bp.f;
    constexpr int KB = DW * 2, VB = DVW * 2;  // bytes per staged row
    uint8_t *ks = smem;                        // [kMKeys][KB]
    uint8_t *vs = ks + kMKeys * KB;            // [kMKeys][VB]
    uint8_t *qs = vs + kMKeys * VB;            // [2][kMRows][KB]
    uint8_t *dos = qs + 2 * kMRows * KB;       // [2][kMRows][VB]
    float *lse_s = reinterpret_cast<float *>(dos + 2 * kMRows * VB);  // [2][kMRows], log2 units
    float *del_s = lse_s + 2 * kMRows;                                 // [2][kMRows]
    int *lo_s = reinterpret_cast<int *>(del_s + 2 * kMRows);           // [2][kMRows]
    int *hi_s = lo_s + 2 * kMRows;                                     // [2][kMRows]

    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int kcap = packed ? si.Kb : p.K;
    const int k0 = blockIdx.x * kMKeys;
    if (k0 >= kcap) return;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const T *qg = static_cast<const T *>(p.q), *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v), *dog = static_cast<const T *>(bp.dout);

    stage_rows<T, DW>(ks, kMKeys, D, tid, kg, [&](int r) -> const T * {
        const int key = k0 + r;
        return key < si.Kb ? kg + ((si.k_off + key) * p.Hkv + kvh) * (long long)D : nullptr;
    });
    stage_rows<T, DVW>(vs, kMKeys, Dv, tid, vg, [&](int r) -> const T * {
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

    auto load_rows = [&](int step, int buf) {
        const int rb = rf + step * kMRows;
        auto row_of = [&](int r) { return (si.q_off + r / G) * p.Hq + kvh * G + r % G; };
        stage_rows<T, DW>(qs + buf * kMRows * KB, kMRows, D, tid, qg, [&](int i) -> const T * {
            const int r = rb + i;
            return r < re ? qg + row_of(r) * D : nullptr;
        });
        stage_rows<T, DVW>(dos + buf * kMRows * VB, kMRows, Dv, tid, dog, [&](int i) -> const T * {
            const int r = rb + i;
            return r < re ? dog + row_of(r) * Dv : nullptr;
        });
        if (tid < kMRows) {
            const int r = rb + tid;
            int lo = 0, hi = 0;
            float l2 = 0.f, dl = 0.f;
            if (r < re) {
                row_range(p, si, r, lo, hi);
                if (hi > lo) {
                    l2 = p.lse[row_of(r)] * kLog2e;
                    dl = bp.delta[row_of(r)];
                }
            }
            lse_s[buf * kMRows + tid] = l2;
            del_s[buf * kMRows + tid] = dl;
            lo_s[buf * kMRows + tid] = lo;
            hi_s[buf * kMRows + tid] = hi;
        }
    };

    if (nsteps > 0) load_rows(0, 0);
    cp_async_commit();

    float dk[DW / 8][4], dv[DVW / 8][4];
#pragma unroll
    for (int j = 0; j < DW / 8; ++j) dk[j][0] = dk[j][1] = dk[j][2] = dk[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < DVW / 8; ++j) dv[j][0] = dv[j][1] = dv[j][2] = dv[j][3] = 0.f;

    for (int step = 0; step < nsteps; ++step) {
        if (step + 1 < nsteps) {
            load_rows(step + 1, (step + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int buf = step & 1;
        const uint8_t *qb = qs + buf * kMRows * KB;
        const uint8_t *db = dos + buf * kMRows * VB;
        // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x 32 rows
        float s[4][4], dp[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[j][c] = dp[j][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DW / 16; ++kk) {
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(ks + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), KB)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bq[4];
                ldmatrix_x4(bq, smem_u32(qb + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                  2 * kk + ((lane >> 3) & 1), KB)));
                MmaOp<T>::run(s[2 * np], a, bq[0], bq[1]);
                MmaOp<T>::run(s[2 * np + 1], a, bq[2], bq[3]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < DVW / 16; ++kk) {
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(vs + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), VB)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bq[4];
                ldmatrix_x4(bq, smem_u32(db + swz(16 * np + (lane & 7) + ((lane >> 4) << 3),
                                                  2 * kk + ((lane >> 3) & 1), VB)));
                MmaOp<T>::run(dp[2 * np], a, bq[0], bq[1]);
                MmaOp<T>::run(dp[2 * np + 1], a, bq[2], bq[3]);
            }
        }
        // P^T (in s) and dS^T (in dp)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = k0 + 16 * warp + g + 8 * (c >> 1);
                const int rl = buf * kMRows + 8 * j + 2 * t + (c & 1);
                const bool ok = key >= lo_s[rl] && key < hi_s[rl];
                const float pr = ok ? exp2f(s[j][c] * p.scale_log2 - lse_s[rl]) : 0.f;
                s[j][c] = pr;
                dp[j][c] = pr * (dp[j][c] - del_s[rl]);
            }
        // dV += P^T dO and dK += dS^T Q, contracting over the 32 rows
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint32_t pa[4], da[4];
            pa[0] = MmaOp<T>::pack(s[2 * m][0], s[2 * m][1]);
            pa[1] = MmaOp<T>::pack(s[2 * m][2], s[2 * m][3]);
            pa[2] = MmaOp<T>::pack(s[2 * m + 1][0], s[2 * m + 1][1]);
            pa[3] = MmaOp<T>::pack(s[2 * m + 1][2], s[2 * m + 1][3]);
            da[0] = MmaOp<T>::pack(dp[2 * m][0], dp[2 * m][1]);
            da[1] = MmaOp<T>::pack(dp[2 * m][2], dp[2 * m][3]);
            da[2] = MmaOp<T>::pack(dp[2 * m + 1][0], dp[2 * m + 1][1]);
            da[3] = MmaOp<T>::pack(dp[2 * m + 1][2], dp[2 * m + 1][3]);
            const int trow = 16 * m + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int np = 0; np < DVW / 16; ++np) {
                uint32_t bb[4];
                ldmatrix_x4_trans(bb, smem_u32(db + swz(trow, 2 * np + (lane >> 4), VB)));
                MmaOp<T>::run(dv[2 * np], pa, bb[0], bb[1]);
                MmaOp<T>::run(dv[2 * np + 1], pa, bb[2], bb[3]);
            }
#pragma unroll
            for (int np = 0; np < DW / 16; ++np) {
                uint32_t bb[4];
                ldmatrix_x4_trans(bb, smem_u32(qb + swz(trow, 2 * np + (lane >> 4), KB)));
                MmaOp<T>::run(dk[2 * np], da, bb[0], bb[1]);
                MmaOp<T>::run(dk[2 * np + 1], da, bb[2], bb[3]);
            }
        }
        __syncthreads();  // buffer `buf` is reloaded by the next step's prefetch
    }
    cp_async_wait<0>();

    // keys past the sequence (padded layout) come out as zeros: P = dS = 0 there
    T *dkg = static_cast<T *>(bp.dk), *dvg = static_cast<T *>(bp.dv);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int key = k0 + 16 * warp + g + 8 * hh;
        if (key >= kcap) continue;
        const long long krow = (si.k_off + key) * p.Hkv + kvh;
#pragma unroll
        for (int j = 0; j < DW / 8; ++j) {
            const int d = 8 * j + 2 * t;
            if (d < D)
                *reinterpret_cast<uint32_t *>(dkg + krow * D + d) = MmaOp<T>::pack(
                    dk[j][2 * hh] * p.scale, dk[j][2 * hh + 1] * p.scale);
        }
#pragma unroll
        for (int j = 0; j < DVW / 8; ++j) {
            const int d = 8 * j + 2 * t;
            if (d < Dv)
                *reinterpret_cast<uint32_t *>(dvg + krow * Dv + d) =
                    MmaOp<T>::pack(dv[j][2 * hh], dv[j][2 * hh + 1]);
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

    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int G = p.G, D = p.D, Dv = p.Dv;
    const int nvalid = si.Qb * G;
    const int ncap = (packed ? si.Qb : p.Q) * G;
    const int r0 = (gridDim.x - 1 - blockIdx.x) * kQRows;  // longest rows first
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
        for (int kk = 0; kk < DW / 16; ++kk) {
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
#pragma unroll
        for (int kk = 0; kk < DVW / 16; ++kk) {
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
        // dS (in s)
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
    int rc = 0;
    if (ktiles > 0) {
        rc = launch_k(bwd_dkdv_generic<T, DL>, dim3((unsigned)ktiles, y), 128, s_dkdv, stream,
                      "bwd_dkdv_generic", bp);
        if (rc) return rc;
    }
    const size_t s_dq = sizeof(float) * ((size_t)kGRows * (D + Dv) + (size_t)kGTK * ((D | 1) + (Dv | 1)));
    const long long qtiles = ((long long)p.Q * p.G + kGRows - 1) / kGRows;
    constexpr int DQL = DL / 8;  // D <= 4 * DL = 32 * DQL
    return launch_k(bwd_dq_generic<T, DQL>, dim3((unsigned)qtiles, y), 128, s_dq, stream,
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

template <typename T, int DW, int DVW>
int launch_mma_bwd_t(const BwdParams &bp, cudaStream_t stream) {
    const AttnParams &p = bp.f;
    const unsigned y = (unsigned)p.B * p.Hkv;
    const long long ktiles = ((long long)p.K + kMKeys - 1) / kMKeys;
    int rc = 0;
    if (ktiles > 0) {
        const size_t s = (size_t)kMKeys * 2 * (DW + DVW) + (size_t)2 * kMRows * 2 * (DW + DVW) +
                         16 * kMRows * 4;
        rc = launch_k(bwd_dkdv_mma<T, DW, DVW>, dim3((unsigned)ktiles, y), 128, s, stream,
                      "bwd_dkdv_mma", bp);
        if (rc) return rc;
    }
    const size_t s = (size_t)kQRows * 2 * (DW + DVW) + (size_t)2 * kQKeys * 2 * (DW + DVW);
    const long long qtiles = ((long long)p.Q * p.G + kQRows - 1) / kQRows;
    return launch_k(bwd_dq_mma<T, DW, DVW>, dim3((unsigned)qtiles, y), 128, s, stream,
                    "bwd_dq_mma", bp);
}

template <typename T>
int launch_mma_bwd(const BwdParams &bp, cudaStream_t stream) {
    const bool wd = bp.f.D > 64, wv = bp.f.Dv > 64;
    if (wd && wv) return launch_mma_bwd_t<T, 128, 128>(bp, stream);
    if (wd) return launch_mma_bwd_t<T, 128, 64>(bp, stream);
    if (wv) return launch_mma_bwd_t<T, 64, 128>(bp, stream);
    return launch_mma_bwd_t<T, 64, 64>(bp, stream);
}

template <typename T>
int launch_bwd_t(const BwdParams &bp, bool mma, cudaStream_t stream) {
    const long long rows = bp.f.Tq * bp.f.Hq;
    int rc = launch_k(bwd_delta_kernel<T>, dim3((unsigned)((rows + 7) / 8)), 256, 0, stream,
                      "bwd_delta", bp, rows);
    if (rc) return rc;
    if constexpr (!std::is_same<T, float>::value) {
        if (mma) return launch_mma_bwd<T>(bp, stream);
    }
    return launch_generic_bwd<T>(bp, stream);
}

}  // namespace

bool bwd_mma_supported(const AttnParams &p, int dtype) {
    return dtype != 0 && p.D % 8 == 0 && p.Dv % 8 == 0 && p.D <= 128 && p.Dv <= 128;
}

int launch_bwd(const BwdParams &bp, int dtype, bool mma, cudaStream_t stream) {
    if (bp.f.Tq * bp.f.Hq == 0) return 0;
    switch (dtype) {
        case 0: return launch_bwd_t<float>(bp, false, stream);
        case 1: return launch_bwd_t<__half>(bp, mma, stream);
        default: return launch_bwd_t<__nv_bfloat16>(bp, mma, stream);
    }
}

}  // namespace attn
