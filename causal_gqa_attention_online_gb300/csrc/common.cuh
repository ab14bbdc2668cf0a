// common.cuh -- problem descriptor and small device helpers shared by the
// kernels of libattn_gqa (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Device status detail codes (written once per launch by the first failing
// thread; read by attn_device_status()).
enum : int {
    kStatusOk = 0,
    kStatusTimeoutTmaFull = 0x101,
    kStatusTimeoutKvEmpty = 0x102,
    kStatusTimeoutMma = 0x103,
    kStatusTimeoutSoftmax = 0x104,
    kStatusTimeoutEpilogue = 0x105,
    kStatusTimeoutQ = 0x106,
    kStatusTimeoutDecode = 0x201,
};

// One attention problem.  Element strides are in elements of the storage type.
// The padded layout has cu_q == cu_k == nullptr; the packed layout has both.
struct AttnParams {
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;              // may be null
    int B, Hq, Hkv, G;       // G = Hq / Hkv
    int Q, K;                // padded capacities, or max lengths (packed)
    long long Tq, Tk;        // rows of the q/o and k/v buffers (B*Q, B*K when padded)
    int D, Dv;
    const int32_t *seqlens_q;  // padded layout, may be null
    const int32_t *seqlens_k;  // padded layout, may be null
    const int32_t *cu_q;       // packed layout
    const int32_t *cu_k;       // packed layout
    // paged K/V (block_table != null): k and v are pools of pages of
    // page_size (a power of two) rows, [num_pages * page_size][Hkv][D or Dv];
    // sequence b's key j lives in page block_table[b * max_pages + j / page_size]
    const int32_t *block_table;
    int page_size, page_shift, max_pages, num_pages;
    int window;              // <= 0: off
    int mask;                // attn_mask: 0 bottom-right causal, 1 top-left causal, 2 none
    float scale;             // multiplies Q.K
    float scale_log2;        // scale * log2(e)
    // split-KV
    int nsplit;              // 1: write final outputs directly
    int split_len;           // keys per split (multiple of the key tile)
    float *part_o;           // [nsplit][B][Q][Hq][Dv] fp32
    float *part_lse;         // [nsplit][B][Q][Hq] fp32, natural log
    int *status;             // device status word
    unsigned long long wait_ns;  // limit of the tcgen05 kernels' mbarrier waits (ns)
    // arbitrary mask (padded layout; null: none): key k of query row q of
    // sequence b and query head h is legal only if bit k % 32 of word k / 32 of
    // mask row ((b * mask_heads + hm) * Q + q) is set, hm = h when
    // mask_heads == Hq and 0 when mask_heads == 1; rows are mask_words apart
    const uint32_t *mask_bits;
    int mask_words, mask_heads;
};

// One backward problem: the forward problem (its o and lse hold the forward's
// outputs, read here) plus dO and the gradients.
struct BwdParams {
    AttnParams f;
    const void *dout;  // [rows of q][Hq][Dv], like o
    void *dq;          // like q
    void *dk;          // like k
    void *dv;          // like v
    float *delta;      // [Tq * Hq] workspace: rowsum(dO * O)
};

struct SeqInfo {
    long long q_off;  // first query row of the sequence in q / o (row = one token)
    long long k_off;  // first key row of the sequence in k / v
    int Qb, Kb;
};

__host__ __device__ __forceinline__ int clamp_len(int n, int cap) {
    return n < 0 ? 0 : (n > cap ? cap : n);
}

__device__ __forceinline__ SeqInfo seq_info(const AttnParams &p, int b) {
    SeqInfo s;
    if (p.cu_q != nullptr) {
        const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
        const int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
        s.q_off = q0;
        s.k_off = k0;
        // a sequence never reaches past the buffers, whatever cu_seqlens holds
        s.Qb = clamp_len(min((long long)(q1 - q0), p.Tq - q0), p.Q);
        s.Kb = clamp_len(min((long long)(k1 - k0), p.Tk - k0), p.K);
    } else {
        s.q_off = (long long)b * p.Q;
        s.k_off = (long long)b * p.K;
        s.Qb = p.seqlens_q ? clamp_len(__ldg(p.seqlens_q + b), p.Q) : p.Q;
        s.Kb = p.seqlens_k ? clamp_len(__ldg(p.seqlens_k + b), p.K) : p.K;
    }
    return s;
}

// Row of key `key` of sequence b in the k / v buffers.  Page numbers outside
// [0, num_pages) are clamped, so a bad table gives wrong keys, never a bad address.
__device__ __forceinline__ long long kv_row(const AttnParams &p, const SeqInfo &si, int b,
                                            int key) {
    if (p.block_table == nullptr) return si.k_off + key;
    int pg = __ldg(p.block_table + (long long)b * p.max_pages + (key >> p.page_shift));
    pg = min(max(pg, 0), p.num_pages - 1);
    return ((long long)pg << p.page_shift) + (key & (p.page_size - 1));
}

// Row of the arbitrary mask for query row qi of sequence b and query head h.
__device__ __forceinline__ const uint32_t *mask_row(const AttnParams &p, int b, int h, int qi) {
    const int hm = p.mask_heads == 1 ? 0 : h;
    return p.mask_bits + (((long long)b * p.mask_heads + hm) * p.Q + qi) * (long long)p.mask_words;
}

// Legal keys of query row qi: [lo, hi) (empty when hi <= lo).  Causal masks
// keep the keys up to the row's diagonal -- aligned to the end of the keys
// (bottom-right, the default) or to their start (top-left) -- and a window
// keeps the last `window` of those; no mask keeps every key of the sequence.
__host__ __device__ __forceinline__ void legal_range(int qi, int Qb, int Kb, int window,
                                                     int mask, int &lo, int &hi) {
    if (mask == 2) {
        lo = 0;
        hi = Kb;
        return;
    }
    const int diag = mask == 1 ? qi : qi + Kb - Qb;  // last legal key
    hi = min(diag + 1, Kb);
    lo = 0;
    if (window > 0) lo = max(0, diag - window + 1);
}

// Query positions [qf, qe) of a sequence that have a legal key in [k0, k1)
// (k0 < k1 <= Kb); empty when qe <= qf.  The causal masks' ranges
// [lo(qi), hi(qi)) both grow with qi, so the set is an interval.
__host__ __device__ __forceinline__ void rows_for_keys(int k0, int k1, int Qb, int Kb,
                                                       int window, int mask, int &qf, int &qe) {
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

// Split-KV ownership of one row with legal keys [lo, hi).  The key axis is cut
// into splits of `len` keys.  A row whose legal keys lie in one split (or that
// has none) is "direct": the block of split `first` writes its final O / LSE.
// Otherwise every split in [first, last] writes a partial and the combine
// kernel merges exactly those.
struct SplitSpan {
    int first, last;
    bool direct;
};

__host__ __device__ __forceinline__ SplitSpan split_span(int lo, int hi, int len) {
    SplitSpan s;
    if (hi <= lo) {
        s.first = s.last = 0;
        s.direct = true;
    } else {
        s.first = lo / len;
        s.last = (hi - 1) / len;
        s.direct = s.first == s.last;
    }
    return s;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) {
    return __float2half_rn(x);
}
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Records the first failure of a launch; later failures keep the first code.
__device__ __forceinline__ void report_status(int *status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace attn
