// kernel_decode.cu -- split-KV tensor-core decode for bf16 / fp16.
//
// Decode has one (or a few) query rows per sequence and head, so the matrix
// atoms cannot be filled along the query axis ("Attention execution mapping",
// LuisaCompute, section 4: a Q=1 contraction does not match an 8-multiple
// matrix atom).  This kernel swaps the operands instead: keys run along M and
// the G query heads of a KV group (times the query rows, at most 16) along N,
//
//     S^T[key, row]  = K[key, :] . Q[row, :]          (M = 16 keys per warp)
//     O^T[dv, row]  += V^T[dv, key] . P^T[key, row]   (M = 16 value columns)
//
// with mma.sync m16n8k16 (fp32 accumulate).  The S^T accumulator is turned
// into the B operand of the second product with movmatrix (an 8x8 transpose
// in registers), and every thread's softmax columns are exactly the columns
// of O^T it owns, so the online rescale needs no data exchange.
//
// The kernel is bound by HBM bandwidth (about 4 FLOP per byte of K/V), so the
// tensor-core choice only has to keep the ALUs out of the way; the design
// work is in streaming K/V: a 3-stage ring of 64-key tiles, each brought in by
// TMA -- one thread, one 64-row box per 64 columns, one mbarrier a stage --
// in the 128-byte swizzle that keeps ldmatrix conflict-free.  A tile starts on
// a 64-key boundary, so with paged K/V it is one page and one table read.  V
// rows past the block's last key are zeroed in shared memory (their P is 0,
// and 0 * NaN must not reach O).  Pages of fewer than 64 rows take a cp.async
// path instead (16-byte copies, a table read per row).  TMA moved the batched
// decode from 5.66 to 5.79 TB/s and the paged one from 4.63 to 5.72 TB/s:
// the per-thread copies and per-tile address work had kept fewer bytes in
// flight than the scattered pages needed.  One K/V tile serves all query heads
// of the group ("Attention execution mapping", section 5, cross-head KV
// reuse).
//
// Work unit: (sequence, KV head, split of the key axis).  Each of the 4 warps
// runs its own online softmax over 16 keys of every tile; the warps' states
// are merged through shared memory at the end, and rows spanning several
// splits are merged by the combine kernel (the legal (max, sum, acc) merge of
// section 5).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

constexpr int kTK = 64;      // keys per tile (4 warps x 16)
constexpr int kStages = 3;
constexpr int kThreads = 128;

// How K / V tiles come in.  kLoadTma: one thread issues TMA copies of 64-row
// boxes (one per 64 columns) onto the stage's mbarrier -- the contiguous layout,
// and paged K / V with pages of at least 64 rows (a 64-key tile is then one
// page).  kLoadAsync / kLoadAsyncPaged: every thread issues 16-byte cp.async
// copies, the latter finding each row through the block table (pages of fewer
// than 64 rows).
enum : int { kLoadAsync = 0, kLoadAsyncPaged = 1, kLoadTma = 2 };

// Byte offset of 16-byte chunk c of row r in a TMA-loaded tile: 64-column
// boxes of 64 rows x 128 bytes, 8 KB apart, in the 128-byte swizzle (chunk
// c % 8 of a row stored at c % 8 ^ r % 8), which keeps ldmatrix free of bank
// conflicts.
__device__ __forceinline__ int swz_box(int r, int c) {
    return (c >> 3) * (kTK * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <typename T, int D, int DV, int NT, int LOAD>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
    constexpr bool PAGED = LOAD == kLoadAsyncPaged;
    constexpr bool TMA = LOAD == kLoadTma;
    constexpr int R = NT * 8;               // query rows of a (sequence, KV head)
    constexpr int KROW = D * 2, VROW = DV * 2;
    constexpr int KTILE = kTK * KROW, VTILE = kTK * VROW;
    constexpr int STAGE = KTILE + VTILE;
    constexpr int OPITCH = DV + 4;          // fp32 merge buffer row pitch
    static_assert(4 * R * OPITCH * 4 + 8 * 4 * R * 4 <= kStages * STAGE, "merge buffer");
    extern __shared__ __align__(128) uint8_t smem[];

    const int split = blockIdx.x;
    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int G = p.G;
    const int nrows = (packed ? si.Qb : p.Q) * G;  // rows this unit writes (<= R)
    const int nvalid = si.Qb * G;

    // Block-uniform: key range of this split and whether it owns any row.
    int lo_min = INT_MAX, hi_max = 0;
    bool mine = false;
    for (int r = 0; r < nrows; ++r) {
        int lo = 0, hi = 0;
        if (r < nvalid) legal_range(r / G, si.Qb, si.Kb, p.window, p.mask, lo, hi);
        const SplitSpan sp = split_span(lo, hi, p.split_len);
        if (sp.direct ? sp.first == split : (split >= sp.first && split <= sp.last)) mine = true;
        if (hi > lo) {
            lo_min = min(lo_min, lo);
            hi_max = max(hi_max, hi);
        }
    }
    // let the combine grid (a programmatic dependent launch) be scheduled
    // while this grid's last blocks run; it waits for our completion itself
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    if (!mine) return;
    // TMA tiles start on a 64-key boundary, so a tile is one page of a paged
    // layout; the keys this adds before the first legal one are masked
    const int kbeg0 = max(lo_min, split * p.split_len);
    const int kbeg = TMA ? (kbeg0 & ~(kTK - 1)) : kbeg0;
    const int kend = min(hi_max, (split + 1) * p.split_len);
    const int ntiles = kend > kbeg ? (kend - kbeg + kTK - 1) / kTK : 0;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const T *qg = static_cast<const T *>(p.q);
    const T *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t fbar = sbase + kStages * STAGE;  // TMA: one full barrier a stage
    if (TMA) {
        if (tid == 0) {
            for (int s = 0; s < kStages; ++s) sm100::mbar_init(fbar + 8u * s, 1);
            sm100::fence_mbar_init();
        }
        __syncthreads();
    }

    // Q^T fragments (B operand of S^T = K Q^T): column n = query row g.
    uint32_t qf[D / 16][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int row = nt * 8 + g;
        const T *qrow = nullptr;
        if (row < nvalid) {
            const int qi = row / G, h = kvh * G + row % G;
            qrow = qg + ((si.q_off + qi) * p.Hq + h) * (long long)D;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][nt][0] = qrow ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 2 * tig) : 0u;
            qf[kk][nt][1] =
                qrow ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + 2 * tig) : 0u;
        }
    }

    // Legal keys of the two rows (per n-tile) this thread's columns hold.
    int rlo[NT][2], rhi[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = nt * 8 + 2 * tig + e;
            int lo = 0, hi = 0;
            if (row < nvalid) legal_range(row / G, si.Qb, si.Kb, p.window, p.mask, lo, hi);
            rlo[nt][e] = max(lo, kbeg);
            rhi[nt][e] = min(hi, kend);
        }

    uint32_t armed = 0, armed_ph = 0;  // TMA: stages with a copy in flight, its phase
    auto load_tile = [&](int t) {
        const int key0 = kbeg + t * kTK;
        const uint32_t st = sbase + (t % kStages) * STAGE;
        if constexpr (TMA) {
            if (tid == 0) {
                const int row = (int)kv_row(p, si, b, key0);
                const uint32_t fb = fbar + 8u * (t % kStages);
                sm100::mbar_arrive_expect_tx(fb, KTILE + VTILE);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    sm100::tma_load_4d(st + c * kTK * 128, &tmK, fb, c * 64, kvh, row, 0);
#pragma unroll
                for (int c = 0; c < DV / 64; ++c)
                    sm100::tma_load_4d(st + KTILE + c * kTK * 128, &tmV, fb, c * 64, kvh, row, 0);
                armed |= 1u << (t % kStages);
                armed_ph = (armed_ph & ~(1u << (t % kStages))) |
                           (((uint32_t)(t / kStages) & 1u) << (t % kStages));
            }
            return;
        }
        constexpr int CK = D / 8, CV = DV / 8;
        // paged: a tile that starts on a 64-key boundary lies in one page when
        // pages hold at least 64 rows (one table read); otherwise a read per
        // row.  Only keys below kend are looked up.
        long long tile_base = si.k_off + key0;
        const bool one_page = !PAGED || (p.page_size >= kTK && (key0 & (kTK - 1)) == 0);
        if (PAGED && one_page) tile_base = kv_row(p, si, b, key0);
        auto row_of = [&](int key) -> long long {
            return one_page ? tile_base + (key - key0) : kv_row(p, si, b, key);
        };
#pragma unroll
        for (int i = tid; i < kTK * CK; i += kThreads) {
            const int row = i / CK, c = i % CK, key = key0 + row;
            const bool ok = key < kend;
            const T *src = ok ? kg + (row_of(key) * p.Hkv + kvh) * (long long)D + c * 8 : kg;
            cp_async16(st + swz(row, c, KROW), src, ok ? 16 : 0);
        }
#pragma unroll
        for (int i = tid; i < kTK * CV; i += kThreads) {
            const int row = i / CV, c = i % CV, key = key0 + row;
            const bool ok = key < kend;
            const T *src = ok ? vg + (row_of(key) * p.Hkv + kvh) * (long long)DV + c * 8 : vg;
            cp_async16(st + KTILE + swz(row, c, VROW), src, ok ? 16 : 0);
        }
    };

    float m[NT][2], l[NT][2];
    float oacc[DV / 16][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < DV / 16; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) oacc[mt][nt][j] = 0.f;
    }

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < ntiles) load_tile(s);
        if (!TMA) cp_async_commit();
    }

    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
        if constexpr (TMA) {
            // tile t has landed (a bounded wait: a copy that never lands records
            // a status, and the block stops with its outputs unwritten)
            const bool got = sm100::mbar_wait_drain(fbar + 8u * (t % kStages),
                                             (uint32_t)(t / kStages) & 1u, p.wait_ns);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            armed &= ~(1u << (t % kStages));
            // V rows past the split's last key may hold anything (NaN included):
            // their P is 0, and 0 * NaN must not reach O
            const int nreal = kend - (kbeg + t * kTK);
            if (nreal < kTK) {
                uint8_t *vt = smem + (t % kStages) * STAGE + KTILE;
                const int nz = (kTK - nreal) * 8;  // 16-byte chunks a box
                for (int i = tid; i < nz * (DV / 64); i += kThreads) {
                    const int bx = i / nz, j = i % nz;
                    *reinterpret_cast<uint4 *>(vt + bx * kTK * 128 + nreal * 128 + j * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                sm100::fence_proxy_async_smem();
            }
            __syncthreads();  // tile t visible to all; tile t-1's stage is free
            if (t + kStages - 1 < ntiles) load_tile(t + kStages - 1);
        } else {
            cp_async_wait<kStages - 2>();
            __syncthreads();  // tile t visible to all; tile t-1's stage is free
            if (t + kStages - 1 < ntiles) load_tile(t + kStages - 1);
            cp_async_commit();
        }

        const uint32_t ks = sbase + (t % kStages) * STAGE;
        const uint32_t vs = ks + KTILE;
        const int kw0 = warp * 16;
        const int key_a = kbeg + t * kTK + kw0 + g, key_b = key_a + 8;

        // S^T = K Q^T for this warp's 16 keys
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) sacc[nt][j] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            const int row = kw0 + (lane & 15);
            ldmatrix_x4(a, ks + (TMA ? swz_box(row, kk * 2 + (lane >> 4))
                                     : swz(row, kk * 2 + (lane >> 4), KROW)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) MmaOp<T>::run(sacc[nt], a, qf[kk][nt][0], qf[kk][nt][1]);
        }

        // mask, online max / exp2 / sum, rescale, P^T -> B fragments
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool la = key_a >= rlo[nt][e] && key_a < rhi[nt][e];
                const bool lb = key_b >= rlo[nt][e] && key_b < rhi[nt][e];
                const float s0 = la ? sacc[nt][e] * p.scale_log2 : -INFINITY;
                const float s1 = lb ? sacc[nt][2 + e] * p.scale_log2 : -INFINITY;
                float mx = fmaxf(s0, s1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mnew = fmaxf(m[nt][e], mx);
                const float mref = mnew == -INFINITY ? 0.f : mnew;  // no key yet: keep zeros
                const float alpha = exp2f(m[nt][e] - mref);
                const float p0 = exp2f(s0 - mref), p1 = exp2f(s1 - mref);
                l[nt][e] = l[nt][e] * alpha + p0 + p1;
                m[nt][e] = mnew;
#pragma unroll
                for (int mt = 0; mt < DV / 16; ++mt) {
                    oacc[mt][nt][e] *= alpha;
                    oacc[mt][nt][2 + e] *= alpha;
                }
                pv[e] = p0;
                pv[2 + e] = p1;
            }
            pb[nt][0] = movmatrix_trans(MmaOp<T>::pack(pv[0], pv[1]));
            pb[nt][1] = movmatrix_trans(MmaOp<T>::pack(pv[2], pv[3]));
        }

        // O^T += V^T P^T
#pragma unroll
        for (int mt = 0; mt < DV / 16; ++mt) {
            uint32_t a[4];
            const int mi = lane >> 3;
            const int key = kw0 + (mi >> 1) * 8 + (lane & 7);
            ldmatrix_x4_trans(a, vs + (TMA ? swz_box(key, mt * 2 + (mi & 1))
                                           : swz(key, mt * 2 + (mi & 1), VROW)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) MmaOp<T>::run(oacc[mt][nt], a, pb[nt][0], pb[nt][1]);
        }
    }
    if (TMA && !ok) {
        // copies still in flight land before the block exits (a wait that
        // ignores the abort: they always land); the outputs stay unwritten
        if (tid == 0) {
            report_status(p.status, kStatusTimeoutDecode);
            for (int s2 = 0; s2 < kStages; ++s2)
                if (armed & (1u << s2)) sm100::mbar_wait_drain(fbar + 8u * s2, (armed_ph >> s2) & 1u);
        }
        return;
    }
    if (!TMA) cp_async_wait<0>();
    __syncthreads();  // ring drained: reuse it as the merge buffer

    // Merge the four warps' states: buffer [warp][row][dv] + per-warp (m, l).
    float *obuf = reinterpret_cast<float *>(smem);
    float *mbuf = obuf + 4 * R * OPITCH;   // [warp][row]
    float *lbuf = mbuf + 4 * R;            // [warp][row]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float ls = l[nt][e];
            ls += __shfl_xor_sync(0xffffffffu, ls, 4);
            ls += __shfl_xor_sync(0xffffffffu, ls, 8);
            ls += __shfl_xor_sync(0xffffffffu, ls, 16);
            const int row = nt * 8 + 2 * tig + e;
            if (g == 0) {
                mbuf[warp * R + row] = m[nt][e];
                lbuf[warp * R + row] = ls;
            }
#pragma unroll
            for (int mt = 0; mt < DV / 16; ++mt) {
                obuf[(warp * R + row) * OPITCH + mt * 16 + g] = oacc[mt][nt][e];
                obuf[(warp * R + row) * OPITCH + mt * 16 + g + 8] = oacc[mt][nt][2 + e];
            }
        }
    __syncthreads();

    T *og = static_cast<T *>(p.o);
    constexpr int C4 = DV / 4;
    for (int idx = tid; idx < nrows * C4; idx += kThreads) {
        const int row = idx / C4, c = (idx % C4) * 4;
        int lo = 0, hi = 0;
        if (row < nvalid) legal_range(row / G, si.Qb, si.Kb, p.window, p.mask, lo, hi);
        const SplitSpan sp = split_span(lo, hi, p.split_len);
        const bool direct = sp.direct;
        if (direct ? sp.first != split : (split < sp.first || split > sp.last)) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mbuf[w * R + row]);
        float L = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float f = exp2f(mbuf[w * R + row] - M);
                L += f * lbuf[w * R + row];
                const float *src = obuf + (w * R + row) * OPITCH + c;
#pragma unroll
                for (int j = 0; j < 4; ++j) o4[j] = fmaf(f, src[j], o4[j]);
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        const int qi = row / G, h = kvh * G + row % G;
        if (direct) {
            T *dst = og + ((si.q_off + qi) * p.Hq + h) * (long long)DV + c;
            T v4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v4[j] = from_f32<T>(o4[j] * inv);
            *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(v4);
            if (c == 0 && p.lse) p.lse[(si.q_off + qi) * p.Hq + h] = lse;
        } else {
            const long long prow = (((long long)split * p.B + b) * p.Q + qi) * p.Hq + h;
            *reinterpret_cast<float4 *>(p.part_o + prow * DV + c) =
                make_float4(o4[0] * inv, o4[1] * inv, o4[2] * inv, o4[3] * inv);
            if (c == 0) p.part_lse[prow] = lse;
        }
    }
}

template <typename T, int D, int DV, int NT>
int launch_decode_t(const AttnParams &p, cudaStream_t stream) {
    constexpr int smem = kStages * kTK * (D + DV) * 2 + 64;  // ring + TMA barriers
    // K / V by TMA as flat [rows][Hkv][D] arrays (rows: B * K padded, Tk
    // packed, the page pool when paged); cp.async where pages hold fewer
    // than 64 rows or a tensor map cannot be made
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    const long long rows = p.block_table ? (long long)p.num_pages * p.page_size
                                         : (p.cu_q ? p.Tk : (long long)p.B * p.K);
    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    bool tma = (!p.block_table || p.page_size >= kTK) && rows > 0 && rows < (1LL << 31);
    if (tma) {
        tma = make_tma_map_4d(&tk, p.k, bf16, (uint64_t)D, p.Hkv, (uint64_t)rows, 1, 1, kTK) == 0 &&
              make_tma_map_4d(&tv, p.v, bf16, (uint64_t)DV, p.Hkv, (uint64_t)rows, 1, 1, kTK) == 0;
        if (!tma) clear_error();
    }
    auto kern = tma ? decode_kernel<T, D, DV, NT, kLoadTma>
                    : (p.block_table ? decode_kernel<T, D, DV, NT, kLoadAsyncPaged>
                                     : decode_kernel<T, D, DV, NT, kLoadAsync>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) {
        set_error("decode kernel: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    dim3 grid((unsigned)p.nsplit, (unsigned)(p.B * p.Hkv));
    kern<<<grid, kThreads, smem, stream>>>(p, tk, tv);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("decode kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T, int D, int DV>
int launch_decode_nt(const AttnParams &p, cudaStream_t stream) {
    return p.Q * p.G <= 8 ? launch_decode_t<T, D, DV, 1>(p, stream)
                          : launch_decode_t<T, D, DV, 2>(p, stream);
}

template <typename T>
int launch_decode_dims(const AttnParams &p, cudaStream_t stream) {
    if (p.D == 128 && p.Dv == 128) return launch_decode_nt<T, 128, 128>(p, stream);
    if (p.D == 256 && p.Dv == 256) return launch_decode_nt<T, 256, 256>(p, stream);
    if (p.D == 64 && p.Dv == 64) return launch_decode_nt<T, 64, 64>(p, stream);
    if (p.D == 128 && p.Dv == 64) return launch_decode_nt<T, 128, 64>(p, stream);
    return launch_decode_nt<T, 64, 128>(p, stream);
}

}  // namespace

bool decode_supported(const AttnParams &p, int dtype) {
    if (dtype != 1 && dtype != 2) return false;
    // head dims 64 / 128 in any pair, or 256 / 256 (one block an SM: 192 KB of ring)
    const bool small = (p.D == 64 || p.D == 128) && (p.Dv == 64 || p.Dv == 128);
    if (!small && !(p.D == 256 && p.Dv == 256)) return false;
    if ((long long)p.Q * p.G > 16 || p.Q < 1) return false;
    return (long long)p.B * p.Hkv <= 65535;
}

int decode_split_len(const AttnParams &p, int nsm) {
    // Small splits balance sequences of very different lengths; fewer, longer
    // splits when the (sequence, KV head) units already fill the SMs.
    if (nsm < 1) nsm = 1;  // a failed device query must not divide by zero
    const long long units = (long long)p.B * p.Hkv;
    long long len = ((long long)p.K * units + 4LL * nsm - 1) / (4LL * nsm);
    len = (len + kTK - 1) / kTK * kTK;
    if (len < 128) len = 128;
    if (len > 1024) len = 1024;
    return (int)len;
}

int launch_decode(const AttnParams &p, int dtype, cudaStream_t stream) {
    if (p.nsplit > 0x7fffffff / 2) {
        set_error("decode kernel: too many splits");
        return 2;
    }
    if (dtype == 2) return launch_decode_dims<__nv_bfloat16>(p, stream);
    return launch_decode_dims<__half>(p, stream);
}

}  // namespace attn
