// kernel_generic.cu -- CUDA-core online-softmax attention forward (any storage
// dtype, head widths up to 512) and the split-KV combine kernels.
//
// This is the fp32 path ("Accelerating PyTorch on AMD GPUs with FlyDSL",
// section on FMHA through AOTriton: that attention kernel family has no FP32
// variant, so fp32 needs its own kernel) and the fallback for bf16/fp16 head
// widths the tensor-core kernels do not take.  It follows the phase graph of
// "Attention execution mapping" (LuisaCompute), section 2: per KV tile,
// QK -> mask -> max -> exp -> sum -> alpha-rescale -> PV, with the row max,
// row sum and accumulator carried across tiles (section 1).
//
// Work decomposition: a block owns 32 consecutive rows of the flattened
// (query position, head-in-group) space of one (sequence, KV head), so every
// K/V tile it stages serves all query heads of the group; it walks the union
// of its rows' legal key ranges in tiles of 32 keys (one key per lane for QK,
// output columns spread over lanes for PV).  Blocks may also own one split
// of the key axis (split-KV), writing normalised partials and their LSE for
// the combine kernel (the legal (max, sum, acc) merge of section 5).
#include <climits>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"

namespace attn {
namespace {

constexpr int kRows = 32;            // flattened rows per block
constexpr int kTK = 32;              // keys per tile (one per lane)
constexpr int kWarps = 8;
constexpr int kRPW = kRows / kWarps;  // rows per warp

template <typename T, int DVL>
__global__ void __launch_bounds__(kWarps * 32, 1) generic_fwd_kernel(const AttnParams p) {
    extern __shared__ float smem[];
    const int D = p.D, Dv = p.Dv, G = p.G;
    const int Dp = D | 1;  // odd row pitch: lane-per-key reads hit distinct banks
    float *qs = smem;                // [kRows][D], pre-scaled by scale*log2(e)
    float *ks = qs + kRows * D;      // [kTK][Dp]
    float *vs = ks + kTK * Dp;       // [kTK][Dv]

    const int b = blockIdx.y / p.Hkv, kvh = blockIdx.y % p.Hkv;
    const int split = blockIdx.z;
    const SeqInfo si = seq_info(p, b);
    const bool packed = p.cu_q != nullptr;
    const int r0 = blockIdx.x * kRows;
    const int nvalid = si.Qb * G;                    // rows holding real queries
    const int ncap = (packed ? si.Qb : p.Q) * G;     // rows this block must write
    if (r0 >= ncap) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *qg = static_cast<const T *>(p.q);
    const T *kg = static_cast<const T *>(p.k);
    const T *vg = static_cast<const T *>(p.v);

    // fp32: every element of a tile is copied by cp.async, so a thread has
    // all of its loads in flight at once (the kernel is latency-bound on
    // small problems); other storage types convert through registers
    constexpr bool kAsync = std::is_same<T, float>::value;
    // a warp per row, lanes along the row
    for (int rr = warp; rr < kRows; rr += kWarps) {
        const int r = r0 + rr;
        const bool ok = r < nvalid;
        const T *src = ok ? qg + ((si.q_off + r / G) * p.Hq + kvh * G + r % G) * (long long)D : qg;
        for (int d = lane; d < D; d += 32) {
            if constexpr (kAsync) {
                cp_async4(smem_u32(qs + rr * D + d), ok ? src + d : qg, ok ? 4 : 0);
            } else {
                qs[rr * D + d] = ok ? to_f32(src[d]) * p.scale_log2 : 0.f;
            }
        }
    }
    if constexpr (kAsync) {
        cp_async_commit();
        cp_async_wait<0>();
        for (int rr = warp; rr < kRows; rr += kWarps)  // this thread's own copies
            for (int d = lane; d < D; d += 32) qs[rr * D + d] *= p.scale_log2;
    }

    // Key range of the block: legal ranges are monotone in the query index.
    int key_lo = 0, key_hi = 0;
    if (r0 < nvalid) {
        int lo_a, hi_a, lo_b, hi_b;
        legal_range(r0 / G, si.Qb, si.Kb, p.window, p.mask, lo_a, hi_a);
        legal_range((min(r0 + kRows, nvalid) - 1) / G, si.Qb, si.Kb, p.window, p.mask, lo_b, hi_b);
        key_lo = lo_a;
        key_hi = hi_b;
    }
    const int s_lo = split * p.split_len;
    key_lo = max(key_lo, s_lo);
    key_hi = min(key_hi, s_lo + p.split_len);

    float m[kRPW], l[kRPW], acc[kRPW][DVL];
    int rlo[kRPW], rhi[kRPW];
    SplitSpan span[kRPW];
    const uint32_t *mrow[kRPW];  // arbitrary mask rows (null: no mask or no real query)
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        const int r = r0 + warp + kWarps * i;
        rlo[i] = 0;
        rhi[i] = 0;
        mrow[i] = nullptr;
        if (r < nvalid) {
            legal_range(r / G, si.Qb, si.Kb, p.window, p.mask, rlo[i], rhi[i]);
            if (p.mask_bits != nullptr) mrow[i] = mask_row(p, b, kvh * G + r % G, r / G);
        }
        span[i] = split_span(rlo[i], rhi[i], p.split_len);
        rlo[i] = max(rlo[i], key_lo);
        rhi[i] = min(rhi[i], key_hi);
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < DVL; ++c) acc[i][c] = 0.f;
    }

    for (int t0 = key_lo; t0 < key_hi; t0 += kTK) {
        __syncthreads();  // previous tile consumed; q staged
        // a warp per key row (one row lookup), lanes along the row
        for (int j = warp; j < kTK; j += kWarps) {
            const int key = t0 + j;
            const bool ok = key < key_hi;
            const long long row = ok ? kv_row(p, si, b, key) * p.Hkv + kvh : 0;
            const T *ksrc = kg + row * D, *vsrc = vg + row * Dv;
            for (int d = lane; d < D; d += 32) {
                if constexpr (kAsync) {
                    cp_async4(smem_u32(ks + j * Dp + d), ok ? ksrc + d : kg, ok ? 4 : 0);
                } else {
                    ks[j * Dp + d] = ok ? to_f32(ksrc[d]) : 0.f;
                }
            }
            for (int c = lane; c < Dv; c += 32) {
                if constexpr (kAsync) {
                    cp_async4(smem_u32(vs + j * Dv + c), ok ? vsrc + c : vg, ok ? 4 : 0);
                } else {
                    vs[j * Dv + c] = ok ? to_f32(vsrc[c]) : 0.f;
                }
            }
        }
        if constexpr (kAsync) {
            cp_async_commit();
            cp_async_wait<0>();
        }
        __syncthreads();
        // The warp's kRPW rows go together (the kernel is latency-bound on
        // small problems): each K element a lane reads feeds kRPW independent
        // dot products, and each V element kRPW accumulators.  Rows whose
        // legal keys miss the tile see only masked scores (p = 0, alpha = 1).
        bool any = false;
#pragma unroll
        for (int i = 0; i < kRPW; ++i)
            any |= rhi[i] > rlo[i] && rhi[i] > t0 && rlo[i] < t0 + kTK;
        if (!any) continue;  // warp-uniform
        const int key = t0 + lane;
        float s[kRPW];
#pragma unroll
        for (int i = 0; i < kRPW; ++i) s[i] = 0.f;
        {
            const float *kr = ks + lane * Dp;
            const float *qw = qs + warp * D;  // row warp + kWarps * i starts at i * kWarps * D
#pragma unroll 4
            for (int d = 0; d < D; ++d) {
                const float kd = kr[d];
#pragma unroll
                for (int i = 0; i < kRPW; ++i) s[i] = fmaf(qw[i * kWarps * D + d], kd, s[i]);
            }
        }
        float pj[kRPW];
#pragma unroll
        for (int i = 0; i < kRPW; ++i) {
            bool legal = key >= rlo[i] && key < rhi[i];
            // (a key in the row's range is below Kb <= K: its word is in the row)
            if (legal && mrow[i] != nullptr) legal = (__ldg(mrow[i] + (key >> 5)) >> (key & 31)) & 1u;
            const float si = legal ? s[i] : -INFINITY;
            const float mnew = fmaxf(m[i], warp_max(si));
            // a row with no legal key so far keeps a finite reference: p = 0
            const float ref = mnew == -INFINITY ? 0.f : mnew;
            pj[i] = exp2f(si - ref);
            const float alpha = exp2f(m[i] - ref);
            l[i] = l[i] * alpha + warp_sum(pj[i]);
#pragma unroll
            for (int c = 0; c < DVL; ++c) acc[i][c] *= alpha;
            m[i] = mnew;
        }
        for (int j = 0; j < kTK; ++j) {
            const float *vr = vs + j * Dv;
            float vv[DVL];
#pragma unroll
            for (int c = 0; c < DVL; ++c) {
                const int col = lane + 32 * c;
                vv[c] = col < Dv ? vr[col] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kRPW; ++i) {
                const float pb = __shfl_sync(0xffffffffu, pj[i], j);
#pragma unroll
                for (int c = 0; c < DVL; ++c) acc[i][c] = fmaf(pb, vv[c], acc[i][c]);
            }
        }
    }

    T *og = static_cast<T *>(p.o);
#pragma unroll
    for (int i = 0; i < kRPW; ++i) {
        const int r = r0 + warp + kWarps * i;
        if (r >= ncap) continue;
        const int qi = r / G, h = kvh * G + r % G;
        // padded rows (r >= nvalid) and empty rows are direct with first == 0
        if (span[i].direct ? split != span[i].first
                           : (split < span[i].first || split > span[i].last))
            continue;
        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
        const float lse = l[i] > 0.f ? (m[i] + __log2f(l[i])) * kLn2 : -INFINITY;
        if (span[i].direct) {
            T *orow = og + ((si.q_off + qi) * p.Hq + h) * (long long)Dv;
#pragma unroll
            for (int c = 0; c < DVL; ++c) {
                const int col = lane + 32 * c;
                if (col < Dv) orow[col] = from_f32<T>(acc[i][c] * inv);
            }
            if (lane == 0 && p.lse) p.lse[(si.q_off + qi) * p.Hq + h] = lse;
        } else {
            const long long prow = (((long long)split * p.B + b) * p.Q + qi) * p.Hq + h;
            float *po = p.part_o + prow * Dv;
#pragma unroll
            for (int c = 0; c < DVL; ++c) {
                const int col = lane + 32 * c;
                if (col < Dv) po[col] = acc[i][c] * inv;
            }
            if (lane == 0) p.part_lse[prow] = lse;
        }
    }
}

// One warp per output row: merge nsplit normalised partials by their LSE.
// Lane s holds the weight of split s (of each group of 32 splits), so every
// weight is computed once; the column loop then issues independent loads.
template <typename T>
__device__ __forceinline__ void combine_one_row(const float *o_parts, const float *lse_parts,
                                                long long part_stride_rows, long long prow,
                                                int nsplit, int Dv, T *orow, float *lse_out,
                                                int lane) {
    float mx = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) mx = fmaxf(mx, lse_parts[s * part_stride_rows + prow]);
    mx = warp_max(mx);
    if (mx == -INFINITY) {
        for (int c = lane; c < Dv; c += 32) orow[c] = from_f32<T>(0.f);
        if (lane == 0 && lse_out) *lse_out = -INFINITY;
        return;
    }
    float wsum = 0.f;
    for (int s = lane; s < nsplit; s += 32)
        wsum += exp2f((lse_parts[s * part_stride_rows + prow] - mx) * kLog2e);
    wsum = warp_sum(wsum);
    const float inv = 1.f / wsum;
    if ((Dv & 3) == 0 && Dv <= 128 && nsplit <= 16) {
        // common case: one 4-column block per lane, every split's partial
        // loaded before any is used (16 independent loads in flight a lane)
        const int c = lane * 4;
        const bool act = c < Dv;
        const float wl = lane < nsplit
            ? exp2f((lse_parts[lane * part_stride_rows + prow] - mx) * kLog2e) : 0.f;
        float4 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = (act && j < nsplit)
                ? *reinterpret_cast<const float4 *>(o_parts + (j * part_stride_rows + prow) * Dv + c)
                : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float w = __shfl_sync(0xffffffffu, wl, j);
            a.x = fmaf(w, v[j].x, a.x);
            a.y = fmaf(w, v[j].y, a.y);
            a.z = fmaf(w, v[j].z, a.z);
            a.w = fmaf(w, v[j].w, a.w);
        }
        if (act) {
            orow[c] = from_f32<T>(a.x * inv);
            orow[c + 1] = from_f32<T>(a.y * inv);
            orow[c + 2] = from_f32<T>(a.z * inv);
            orow[c + 3] = from_f32<T>(a.w * inv);
        }
    } else if ((Dv & 3) == 0) {
        // uniform trip count: every lane takes part in the shuffles
        for (int c0 = 0; c0 < Dv; c0 += 128) {
            const int c = c0 + lane * 4;
            const bool act = c < Dv;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < nsplit; s0 += 32) {
                const int sl = s0 + lane;
                const float wl =
                    sl < nsplit ? exp2f((lse_parts[sl * part_stride_rows + prow] - mx) * kLog2e) : 0.f;
                const int n = min(32, nsplit - s0);
#pragma unroll 4
                for (int j = 0; j < n; ++j) {
                    const float w = __shfl_sync(0xffffffffu, wl, j);
                    const float4 v = act ? *reinterpret_cast<const float4 *>(
                                               o_parts + ((s0 + j) * part_stride_rows + prow) * Dv + c)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    a.x = fmaf(w, v.x, a.x);
                    a.y = fmaf(w, v.y, a.y);
                    a.z = fmaf(w, v.z, a.z);
                    a.w = fmaf(w, v.w, a.w);
                }
            }
            if (act) {
                orow[c] = from_f32<T>(a.x * inv);
                orow[c + 1] = from_f32<T>(a.y * inv);
                orow[c + 2] = from_f32<T>(a.z * inv);
                orow[c + 3] = from_f32<T>(a.w * inv);
            }
        }
    } else {
        for (int c = lane; c < Dv; c += 32) {
            float a = 0.f;
            for (int s = 0; s < nsplit; ++s) {
                const float w = exp2f((lse_parts[s * part_stride_rows + prow] - mx) * kLog2e);
                a = fmaf(w, o_parts[(s * part_stride_rows + prow) * Dv + c], a);
            }
            orow[c] = from_f32<T>(a * inv);
        }
    }
    if (lane == 0 && lse_out) *lse_out = mx + __logf(wsum);
}

template <typename T>
__global__ void __launch_bounds__(128) combine_rows_kernel(const AttnParams p) {
    // launched as a programmatic dependent of the forward kernel: wait here
    // until that grid has completed and its partials are visible
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= (long long)p.B * p.Q * p.Hq) return;
    const int h = (int)(row % p.Hq);
    const int qi = (int)((row / p.Hq) % p.Q);
    const int b = (int)(row / ((long long)p.Hq * p.Q));
    const SeqInfo si = seq_info(p, b);
    T *orow = static_cast<T *>(p.o) + ((si.q_off + qi) * p.Hq + h) * (long long)p.Dv;
    float *lse_out = p.lse ? p.lse + (si.q_off + qi) * p.Hq + h : nullptr;
    if (qi >= si.Qb) return;  // padded rows are written by the forward kernel
    int lo, hi;
    legal_range(qi, si.Qb, si.Kb, p.window, p.mask, lo, hi);
    const SplitSpan span = split_span(lo, hi, p.split_len);
    if (span.direct) return;  // written by the forward kernel
    const long long stride = (long long)p.B * p.Q * p.Hq;
    const long long first = (long long)span.first * stride + row;
    combine_one_row<T>(p.part_o + first * p.Dv, p.part_lse + first, stride, 0,
                       span.last - span.first + 1, p.Dv, orow, lse_out, lane);
}

template <typename T>
__global__ void __launch_bounds__(128) combine_flat_kernel(const float *o_parts,
                                                           const float *lse_parts, T *o,
                                                           float *lse, int nsplit,
                                                           long long rows, int Dv) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    combine_one_row<T>(o_parts, lse_parts, rows, row, nsplit, Dv, o + row * Dv,
                       lse ? lse + row : nullptr, lane);
}

template <typename T, int DVL>
int launch_generic_t(const AttnParams &p, cudaStream_t stream) {
    const int Dp = p.D | 1;
    const size_t smem = sizeof(float) * ((size_t)kRows * p.D + (size_t)kTK * Dp +
                                         (size_t)kTK * p.Dv);
    auto kern = generic_fwd_kernel<T, DVL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) {
        set_error("generic kernel: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return 3;
    }
    const long long rows = (long long)p.Q * p.G;
    dim3 grid((unsigned)((rows + kRows - 1) / kRows), (unsigned)(p.B * p.Hkv),
              (unsigned)p.nsplit);
    kern<<<grid, kWarps * 32, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("generic kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

template <typename T>
int launch_generic_dtype(const AttnParams &p, cudaStream_t stream) {
    if (p.Dv <= 32) return launch_generic_t<T, 1>(p, stream);
    if (p.Dv <= 64) return launch_generic_t<T, 2>(p, stream);
    if (p.Dv <= 128) return launch_generic_t<T, 4>(p, stream);
    if (p.Dv <= 256) return launch_generic_t<T, 8>(p, stream);
    return launch_generic_t<T, 16>(p, stream);
}

}  // namespace

int launch_generic(const AttnParams &p, int dtype, cudaStream_t stream) {
    if (p.Q * (long long)p.G / kRows + 1 > 0x7fffffffLL || p.B * (long long)p.Hkv > 65535 ||
        p.nsplit > 65535) {
        set_error("generic kernel: grid too large");
        return 2;
    }
    switch (dtype) {
        case 0: return launch_generic_dtype<float>(p, stream);
        case 1: return launch_generic_dtype<__half>(p, stream);
        case 2: return launch_generic_dtype<__nv_bfloat16>(p, stream);
    }
    set_error("generic kernel: bad dtype %d", dtype);
    return 1;
}

int launch_combine_rows(const AttnParams &p, int dtype, cudaStream_t stream) {
    const long long rows = (long long)p.B * p.Q * p.Hq;
    if (rows == 0) return 0;
    // programmatic dependent launch: the combine grid is scheduled while the
    // forward grid drains and waits in griddepcontrol.wait for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le = cudaSuccess;
    switch (dtype) {
        case 0: le = cudaLaunchKernelEx(&cfg, combine_rows_kernel<float>, p); break;
        case 1: le = cudaLaunchKernelEx(&cfg, combine_rows_kernel<__half>, p); break;
        case 2: le = cudaLaunchKernelEx(&cfg, combine_rows_kernel<__nv_bfloat16>, p); break;
        default: set_error("combine: bad dtype %d", dtype); return 1;
    }
    if (le != cudaSuccess) {
        set_error("combine kernel launch: %s", cudaGetErrorString(le));
        return 3;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("combine kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

// One warp per row, partials in a 16-bit storage type P (the merge of the
// key shards of several ranks, exchanged as they were written).
template <typename P, typename T>
__global__ void __launch_bounds__(128) combine_parts_kernel(const P *o_parts,
                                                            const float *lse_parts, T *o,
                                                            float *lse, int nsplit,
                                                            long long rows, int Dv) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    float mx = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) mx = fmaxf(mx, lse_parts[s * rows + row]);
    mx = warp_max(mx);
    T *orow = o + row * Dv;
    if (mx == -INFINITY) {
        for (int c = lane; c < Dv; c += 32) orow[c] = from_f32<T>(0.f);
        if (lane == 0 && lse) lse[row] = -INFINITY;
        return;
    }
    float wsum = 0.f;
    for (int s = lane; s < nsplit; s += 32) wsum += exp2f((lse_parts[s * rows + row] - mx) * kLog2e);
    wsum = warp_sum(wsum);
    const float inv = 1.f / wsum;
    for (int c = lane; c < Dv; c += 32) {
        float a = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float w = exp2f((lse_parts[s * rows + row] - mx) * kLog2e);
            a = fmaf(w, to_f32(o_parts[(s * rows + row) * Dv + c]), a);
        }
        orow[c] = from_f32<T>(a * inv);
    }
    if (lane == 0 && lse) lse[row] = mx + __logf(wsum);
}

int launch_combine_parts(const void *o_parts, int parts_dtype, const float *lse_parts, void *o,
                         float *lse, int nsplit, long long rows, int Dv, int dtype,
                         cudaStream_t stream) {
    if (rows == 0) return 0;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    if (parts_dtype == 1 && dtype == 1)
        combine_parts_kernel<__half, __half><<<blocks, 128, 0, stream>>>(
            static_cast<const __half *>(o_parts), lse_parts, static_cast<__half *>(o), lse,
            nsplit, rows, Dv);
    else if (parts_dtype == 2 && dtype == 2)
        combine_parts_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, 128, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(o_parts), lse_parts,
            static_cast<__nv_bfloat16 *>(o), lse, nsplit, rows, Dv);
    else {
        set_error("combine: 16-bit partials combine into the same dtype (parts %d, out %d)",
                  parts_dtype, dtype);
        return 2;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("combine kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

int launch_combine_flat(const float *o_parts, const float *lse_parts, void *o, float *lse,
                        int nsplit, long long rows, int Dv, int dtype, cudaStream_t stream) {
    if (rows == 0) return 0;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    switch (dtype) {
        case 0:
            combine_flat_kernel<float><<<blocks, 128, 0, stream>>>(
                o_parts, lse_parts, static_cast<float *>(o), lse, nsplit, rows, Dv);
            break;
        case 1:
            combine_flat_kernel<__half><<<blocks, 128, 0, stream>>>(
                o_parts, lse_parts, static_cast<__half *>(o), lse, nsplit, rows, Dv);
            break;
        case 2:
            combine_flat_kernel<__nv_bfloat16><<<blocks, 128, 0, stream>>>(
                o_parts, lse_parts, static_cast<__nv_bfloat16 *>(o), lse, nsplit, rows, Dv);
            break;
        default: set_error("combine: bad dtype %d", dtype); return 1;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("combine kernel launch: %s", cudaGetErrorString(e));
        return 3;
    }
    count_launch();
    return 0;
}

}  // namespace attn
