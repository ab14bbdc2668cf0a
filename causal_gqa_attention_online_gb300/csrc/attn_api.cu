// attn_api.cu -- the C ABI of libattn_gqa: argument validation, kernel choice,
// split-KV workspace from a library-owned stream-ordered pool, error strings
// and the device status word.  Declarations and contracts: include/attn_gqa.h.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "attn_gqa.h"
#include "common.cuh"
#include "launch.h"

namespace attn {

namespace {
thread_local char g_last_error[512] = "";
constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
cudaMemPool_t g_pools[kMaxDevices] = {};
int *g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
}  // namespace

std::atomic<unsigned long long> g_launches{0};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// The device status word (one per device, in this module's device image).
__device__ int g_device_status;

void clear_error() { g_last_error[0] = '\0'; }

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

int sm_count(int device) {
    if (device < 0 || device >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (g_sm_count[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
            return 0;
        g_sm_count[device] = n;
    }
    return g_sm_count[device];
}

namespace {

int current_device(int *dev) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
        set_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

// Address of the status word on `dev` (the current device).
int status_ptr(int dev, int **out) {
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_device_status);
        if (e != cudaSuccess) {
            set_error("cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        g_status_ptr[dev] = static_cast<int *>(ptr);
    }
    *out = g_status_ptr[dev];
    return ATTN_OK;
}

// Library-owned pool: freed blocks stay cached, so steady-state split-KV
// calls do not reach the driver allocator.
int pool_for(int dev, cudaMemPool_t *out) {
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (g_pools[dev] == nullptr) {
        cudaMemPoolProps props;
        memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) {
            set_error("cudaMemPoolCreate: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        uint64_t threshold = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &threshold);
        if (e != cudaSuccess) {
            set_error("cudaMemPoolSetAttribute: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return ATTN_OK;
}

bool ptr_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Host-side validation shared by both layouts.
int validate(const void *q, const void *k, const void *v, const void *o, const float *lse,
             int B, int Hq, int Hkv, int Q, int K, int D, int Dv, int dtype, int algo) {
    if (B < 0 || Hq < 0 || Hkv < 0 || Q < 0 || K < 0) {
        set_error("negative size (B=%d Hq=%d Hkv=%d Q=%d K=%d)", B, Hq, Hkv, Q, K);
        return ATTN_ERR_INVALID;
    }
    if (Hq > 0 && (Hkv == 0 || Hq % Hkv != 0)) {
        set_error("Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
        return ATTN_ERR_INVALID;
    }
    if (D < 1 || D > 512 || Dv < 1 || Dv > 512) {
        set_error("head widths must be in [1, 512] (D=%d Dv=%d)", D, Dv);
        return ATTN_ERR_INVALID;
    }
    if (dtype < ATTN_F32 || dtype > ATTN_BF16) {
        set_error("unknown dtype %d", dtype);
        return ATTN_ERR_INVALID;
    }
    if (algo < ATTN_ALGO_AUTO || algo > ATTN_ALGO_MMA) {
        set_error("unknown algo %d", algo);
        return ATTN_ERR_INVALID;
    }
    const bool any_q = (long long)B * Q * Hq > 0;
    if (any_q && (q == nullptr || o == nullptr)) {
        set_error("q and o must be non-null");
        return ATTN_ERR_INVALID;
    }
    if (any_q && K > 0 && (k == nullptr || v == nullptr)) {
        set_error("k and v must be non-null");
        return ATTN_ERR_INVALID;
    }
    if (!ptr_aligned16(q) || !ptr_aligned16(k) || !ptr_aligned16(v) || !ptr_aligned16(o) ||
        !ptr_aligned16(lse)) {
        set_error("tensor pointers must be 16-byte aligned");
        return ATTN_ERR_INVALID;
    }
    return ATTN_OK;
}

int plan_splits(AttnParams &p, int chosen, int nsm) {
    if (nsm < 1) {
        set_error("the device reports no multiprocessors");
        return ATTN_ERR_CUDA;
    }
    if (chosen == ATTN_ALGO_DECODE) {
        p.split_len = decode_split_len(p, nsm);
    } else {
        p.split_len = p.K > 0 ? p.K : 1;
        const long long units = (long long)p.B * p.Hkv * (((long long)p.Q * p.G + 31) / 32);
        const int min_split = 128;
        if (p.K > 2 * min_split && units < 2LL * nsm) {
            const long long want = (2LL * nsm + units - 1) / units;
            const long long most = (p.K + min_split - 1) / min_split;
            const long long ns = want < most ? want : most;
            if (ns > 1) {
                long long len = (p.K + ns - 1) / ns;
                p.split_len = (int)((len + 63) / 64 * 64);
            }
        }
    }
    if (p.split_len < 1) p.split_len = 1;
    p.nsplit = p.K > 0 ? (int)(((long long)p.K + p.split_len - 1) / p.split_len) : 1;
    return ATTN_OK;
}

unsigned long long split_workspace_bytes(const AttnParams &p) {
    if (p.nsplit <= 1) return 0;
    const unsigned long long rows = (unsigned long long)p.nsplit * p.B * p.Q * p.Hq;
    return sizeof(float) * rows * (unsigned long long)(p.Dv + 1);
}

void set_split_workspace(AttnParams &p, void *ws) {
    const long long rows = (long long)p.nsplit * p.B * p.Q * p.Hq;
    p.part_o = static_cast<float *>(ws);
    p.part_lse = p.part_o + rows * p.Dv;
}

int launch_split_kv(const AttnParams &p, int chosen, int dtype, cudaStream_t stream) {
    int rc = chosen == ATTN_ALGO_DECODE ? launch_decode(p, dtype, stream)
                                        : launch_generic(p, dtype, stream);
    if (rc == 0 && p.nsplit > 1) rc = launch_combine_rows(p, dtype, stream);
    return rc;
}

namespace {

int run(AttnParams &p, int dtype, int algo, cudaStream_t stream) {
    int dev = 0;
    int rc = current_device(&dev);
    if (rc) return rc;
    rc = status_ptr(dev, &p.status);
    if (rc) return rc;
    const int nsm = sm_count(dev);

    // Kernel choice.  An arbitrary mask runs on the tcgen05 prefill or the
    // CUDA-core kernel only.
    const bool masked = p.mask_bits != nullptr;
    if (masked && (algo == ATTN_ALGO_DECODE || algo == ATTN_ALGO_MMA)) {
        set_error("an arbitrary mask runs on the tcgen05 or the generic kernel only");
        return ATTN_ERR_UNSUPPORTED;
    }
    int chosen = algo;
    if (algo == ATTN_ALGO_AUTO) {
        chosen = ATTN_ALGO_GENERIC;
        if (dtype != ATTN_F32) {
            if (!masked && decode_supported(p, dtype))
                chosen = ATTN_ALGO_DECODE;
            else if (prefill_tc_supported(p, dtype) || prefill_wide_tc_supported(p, dtype))
                chosen = ATTN_ALGO_TCGEN05;
            else if (!masked && fwd_mma_supported(p, dtype))
                chosen = ATTN_ALGO_MMA;
        }
    } else if (algo == ATTN_ALGO_DECODE && !decode_supported(p, dtype)) {
        set_error("decode kernel does not take this shape/dtype");
        return ATTN_ERR_UNSUPPORTED;
    } else if (algo == ATTN_ALGO_TCGEN05 && !prefill_tc_supported(p, dtype) &&
               !prefill_wide_tc_supported(p, dtype)) {
        set_error("tcgen05 prefill kernel does not take this shape/dtype");
        return ATTN_ERR_UNSUPPORTED;
    } else if (algo == ATTN_ALGO_MMA && !fwd_mma_supported(p, dtype)) {
        set_error("mma forward kernel takes bf16/fp16 with D, Dv multiples of 8 up to 512");
        return ATTN_ERR_UNSUPPORTED;
    }

    if (chosen == ATTN_ALGO_TCGEN05 && !prefill_tc_supported(p, dtype))
        return launch_prefill_wide_tc(p, dtype, stream);
    if (chosen == ATTN_ALGO_TCGEN05) {
        // workspace: the unit order (ints), then the live-tile flags of a mask
        const long long n = prefill_tc_order_len(p), nlive = prefill_tc_live_len(p);
        if (n == 0 && nlive == 0) return launch_prefill_tc(p, dtype, stream, nullptr, nullptr);
        void *ws = nullptr;
        cudaMemPool_t pool = nullptr;
        rc = pool_for(dev, &pool);
        if (rc) return rc;
        const size_t order_bytes = (sizeof(int) * (size_t)n + 255) / 256 * 256;
        const size_t bytes = order_bytes + (size_t)nlive;
        cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, stream);
        if (e != cudaSuccess) {
            set_error("workspace cudaMallocFromPoolAsync(%zu): %s", bytes, cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        rc = launch_prefill_tc(p, dtype, stream, n > 0 ? static_cast<int *>(ws) : nullptr,
                               nlive > 0 ? static_cast<uint8_t *>(ws) + order_bytes : nullptr);
        e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == 0) {
            set_error("workspace cudaFreeAsync: %s", cudaGetErrorString(e));
            rc = ATTN_ERR_CUDA;
        }
        return rc;
    }
    if (chosen == ATTN_ALGO_MMA) return launch_fwd_mma(p, dtype, stream);

    // Split the key axis when the (sequence, KV head, row-block) units alone
    // would leave SMs idle.  A row whose legal keys fall in one split is
    // written directly; the others are merged by the combine kernel.
    rc = plan_splits(p, chosen, nsm);
    if (rc) return rc;

    void *ws = nullptr;
    if (p.nsplit > 1) {
        const size_t bytes = (size_t)split_workspace_bytes(p);
        cudaMemPool_t pool = nullptr;
        rc = pool_for(dev, &pool);
        if (rc) return rc;
        const cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, stream);
        if (e != cudaSuccess) {
            set_error("workspace cudaMallocFromPoolAsync(%zu): %s", bytes, cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        set_split_workspace(p, ws);
    }
    rc = launch_split_kv(p, chosen, dtype, stream);
    if (ws != nullptr) {
        const cudaError_t e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == 0) {
            set_error("workspace cudaFreeAsync: %s", cudaGetErrorString(e));
            rc = ATTN_ERR_CUDA;
        }
    }
    return rc;
}

int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
               int Hkv, long long Tq, long long Tk, int Q, int K, int D, int Dv,
               const int32_t *seqlens_q,
               const int32_t *seqlens_k, const int32_t *cu_q, const int32_t *cu_k, int window,
               float scale, int mask, int dtype, int algo, cudaStream_t stream,
               const int32_t *block_table = nullptr, int page_size = 0, int num_pages = 0,
               int max_pages = 0, const uint32_t *mask_bits = nullptr, int mask_words = 0,
               int mask_heads = 0) {
    clear_error();
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Q, K, D, Dv, dtype, algo);
    if (rc) return rc;
    if (mask < ATTN_MASK_CAUSAL || mask > ATTN_MASK_NONE) {
        set_error("unknown mask %d", mask);
        return ATTN_ERR_INVALID;
    }
    if (mask == ATTN_MASK_NONE && window > 0) {
        set_error("a window needs a causal mask (window=%d with ATTN_MASK_NONE)", window);
        return ATTN_ERR_INVALID;
    }
    if ((long long)B * Q * Hq == 0) return ATTN_OK;
    AttnParams p;
    memset(&p, 0, sizeof(p));
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Q = Q;
    p.K = K;
    p.Tq = Tq;
    p.Tk = Tk;
    p.D = D;
    p.Dv = Dv;
    p.seqlens_q = seqlens_q;
    p.seqlens_k = seqlens_k;
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    // A window of at least K keys keeps every causal key: same as no window
    // (this also keeps the kernels' window arithmetic far from overflow).
    p.window = (window <= 0 || window >= K) ? 0 : window;
    p.mask = mask;
    p.block_table = block_table;
    p.page_size = page_size;
    p.page_shift = 0;
    while (page_size > 0 && (1 << p.page_shift) < page_size) ++p.page_shift;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.mask_bits = K > 0 ? mask_bits : nullptr;  // no key: nothing to mask
    p.mask_words = mask_words;
    p.mask_heads = mask_heads;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.nsplit = 1;
    p.split_len = K > 0 ? K : 1;
    p.wait_ns = wait_limit_ns();
    return run(p, dtype, algo, stream);
}

int bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
               long long Tq, long long Tk, int Q, int K, int D, int Dv,
               const int32_t *seqlens_q, const int32_t *seqlens_k, const int32_t *cu_q,
               const int32_t *cu_k, int window, float scale, int mask, int dtype, int algo,
               cudaStream_t stream) {
    clear_error();
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Q, K, D, Dv, dtype, ATTN_ALGO_AUTO);
    if (rc) return rc;
    if (D > 256 || Dv > 256) {
        set_error("the backward takes head widths up to 256 (D=%d Dv=%d)", D, Dv);
        return ATTN_ERR_UNSUPPORTED;
    }
    if (algo != ATTN_ALGO_AUTO && algo != ATTN_ALGO_GENERIC && algo != ATTN_ALGO_MMA &&
        algo != ATTN_ALGO_TCGEN05) {
        set_error("backward algo must be ATTN_ALGO_AUTO, ATTN_ALGO_GENERIC, ATTN_ALGO_MMA or "
                  "ATTN_ALGO_TCGEN05 (got %d)", algo);
        return ATTN_ERR_INVALID;
    }
    if (mask < ATTN_MASK_CAUSAL || mask > ATTN_MASK_NONE) {
        set_error("unknown mask %d", mask);
        return ATTN_ERR_INVALID;
    }
    if (mask == ATTN_MASK_NONE && window > 0) {
        set_error("a window needs a causal mask (window=%d with ATTN_MASK_NONE)", window);
        return ATTN_ERR_INVALID;
    }
    const bool any_q = (long long)B * Q * Hq > 0;
    const bool any_k = (long long)B * K * Hkv > 0;
    if ((any_q && (lse == nullptr || dout == nullptr || dq == nullptr)) ||
        (any_k && (dk == nullptr || dv == nullptr))) {
        set_error("lse, dout, dq, dk and dv must be non-null");
        return ATTN_ERR_INVALID;
    }
    if (!ptr_aligned16(dout) || !ptr_aligned16(dq) || !ptr_aligned16(dk) || !ptr_aligned16(dv)) {
        set_error("tensor pointers must be 16-byte aligned");
        return ATTN_ERR_INVALID;
    }
    if (!any_q && !any_k) return ATTN_OK;
    BwdParams bp;
    memset(&bp, 0, sizeof(bp));
    AttnParams &p = bp.f;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = const_cast<void *>(o);
    p.lse = const_cast<float *>(lse);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hkv > 0 ? Hq / Hkv : 1;
    p.Q = Q;
    p.K = K;
    p.Tq = Tq;
    p.Tk = Tk;
    p.D = D;
    p.Dv = Dv;
    p.seqlens_q = seqlens_q;
    p.seqlens_k = seqlens_k;
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.window = (window <= 0 || window >= K) ? 0 : window;
    p.mask = mask;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.nsplit = 1;
    p.wait_ns = wait_limit_ns();
    bp.dout = dout;
    bp.dq = dq;
    bp.dk = dk;
    bp.dv = dv;
    const bool mma_ok = bwd_mma_supported(p, dtype);
    const bool tc_ok = mma_ok && bwd_dq_tc_supported(p, dtype);
    if (algo == ATTN_ALGO_MMA && !mma_ok) {
        set_error("mma backward kernels take bf16/fp16 with D, Dv multiples of 8 up to 128");
        return ATTN_ERR_UNSUPPORTED;
    }
    if (algo == ATTN_ALGO_TCGEN05 && !tc_ok) {
        set_error("the tcgen05 backward takes bf16/fp16 with D, Dv multiples of 16 in [64, 128]");
        return ATTN_ERR_UNSUPPORTED;
    }
    int mode = 0;  // CUDA cores
    if (algo == ATTN_ALGO_MMA) mode = 1;
    else if (algo == ATTN_ALGO_TCGEN05) mode = 2;
    else if (algo == ATTN_ALGO_AUTO) mode = tc_ok ? 2 : (mma_ok ? 1 : 0);
    int dev = 0;
    rc = current_device(&dev);
    if (rc) return rc;
    rc = status_ptr(dev, &p.status);
    if (rc) return rc;
    if (!any_q) {
        // no query rows: every key gets zero gradients
        const size_t es = dtype == ATTN_F32 ? 4 : 2;
        cudaError_t e = cudaMemsetAsync(dk, 0, (size_t)Tk * Hkv * D * es, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, (size_t)Tk * Hkv * Dv * es, stream);
        if (e != cudaSuccess) {
            set_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        return ATTN_OK;
    }
    cudaMemPool_t pool = nullptr;
    rc = pool_for(dev, &pool);
    if (rc) return rc;
    void *ws = nullptr;
    const size_t bytes = sizeof(float) * (size_t)(Tq * Hq);
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, stream);
    if (e != cudaSuccess) {
        set_error("workspace cudaMallocFromPoolAsync(%zu): %s", bytes, cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    bp.delta = static_cast<float *>(ws);
    rc = launch_bwd(bp, dtype, mode, stream);
    e = cudaFreeAsync(ws, stream);
    if (e != cudaSuccess && rc == 0) {
        set_error("workspace cudaFreeAsync: %s", cudaGetErrorString(e));
        rc = ATTN_ERR_CUDA;
    }
    return rc;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                const int32_t *seqlens_k, int window, float scale, int mask, int dtype, int algo,
                attn_stream_t stream) {
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, (long long)B * Q, (long long)B * K, Q, K, D, Dv,
                      seqlens_q, seqlens_k, nullptr, nullptr, window, scale, mask, dtype, algo,
                      reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages, void *o, float *lse,
                   int B, int Hq, int Hkv, int Q, int D, int Dv, const int32_t *block_table,
                   int max_pages, int page_size, int num_pages, const int32_t *seqlens_q,
                   const int32_t *seqlens_k, int window, float scale, int mask, int dtype,
                   int algo, attn_stream_t stream) {
    attn::clear_error();
    if (page_size < 1 || page_size > (1 << 20) || (page_size & (page_size - 1)) != 0) {
        set_error("page_size must be a power of two in [1, 2^20] (got %d)", page_size);
        return ATTN_ERR_INVALID;
    }
    if (num_pages < 1 || max_pages < 0 ||
        (long long)num_pages * page_size >= (1LL << 31) ||
        (long long)max_pages * page_size >= (1LL << 31)) {
        set_error("bad page counts (num_pages=%d max_pages=%d page_size=%d)", num_pages,
                  max_pages, page_size);
        return ATTN_ERR_INVALID;
    }
    if (B > 0 && (block_table == nullptr || seqlens_k == nullptr)) {
        set_error("paged K/V needs block_table and seqlens_k");
        return ATTN_ERR_INVALID;
    }
    const int K = max_pages * page_size;  // key capacity of a sequence
    return fwd_common(q, k_pages, v_pages, o, lse, B, Hq, Hkv, (long long)B * Q,
                      (long long)num_pages * page_size, Q, K, D, Dv, seqlens_q, seqlens_k, nullptr,
                      nullptr, window, scale, mask, dtype, algo,
                      reinterpret_cast<cudaStream_t>(stream), block_table, page_size, num_pages,
                      max_pages);
}

int attn_fwd_masked(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int Hq, int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                    const int32_t *seqlens_k, const uint32_t *mask_bits, int mask_words,
                    int mask_heads, int window, float scale, int mask, int dtype, int algo,
                    attn_stream_t stream) {
    attn::clear_error();
    if ((long long)B * Q * Hq > 0 && K > 0) {
        if (mask_bits == nullptr) {
            set_error("attn_fwd_masked: mask_bits must be non-null");
            return ATTN_ERR_INVALID;
        }
        if ((reinterpret_cast<uintptr_t>(mask_bits) & 15u) != 0) {
            set_error("attn_fwd_masked: mask_bits must be 16-byte aligned");
            return ATTN_ERR_INVALID;
        }
        const long long need = 4LL * (((long long)K + 127) / 128);
        if (mask_words < need || mask_words % 4 != 0) {
            set_error("attn_fwd_masked: mask_words (%d) must be a multiple of 4 and at least "
                      "4 * ceil(K / 128) = %lld",
                      mask_words, need);
            return ATTN_ERR_INVALID;
        }
        if (mask_heads != 1 && mask_heads != Hq) {
            set_error("attn_fwd_masked: mask_heads (%d) must be 1 or Hq (%d)", mask_heads, Hq);
            return ATTN_ERR_INVALID;
        }
    }
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, (long long)B * Q, (long long)B * K, Q, K, D, Dv,
                      seqlens_q, seqlens_k, nullptr, nullptr, window, scale, mask, dtype, algo,
                      reinterpret_cast<cudaStream_t>(stream), nullptr, 0, 0, 0, mask_bits,
                      mask_words, mask_heads);
}

int attn_fwd_algo(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                  int Hq, int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                  const int32_t *seqlens_k, int window, float scale, int dtype, int algo,
                  attn_stream_t stream) {
    return attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Q, K, D, Dv, seqlens_q, seqlens_k, window,
                       scale, ATTN_MASK_CAUSAL, dtype, algo, stream);
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
             const int32_t *seqlens_k, int window, float scale, int dtype,
             attn_stream_t stream) {
    return attn_fwd_algo(q, k, v, o, lse, B, Hq, Hkv, Q, K, D, Dv, seqlens_q, seqlens_k, window,
                         scale, dtype, ATTN_ALGO_AUTO, stream);
}

int attn_fwd_varlen_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int Hq, int Hkv, int total_q, int total_k, int max_Q, int max_K, int D,
                       int Dv, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                       int window, float scale, int mask, int dtype, int algo,
                       attn_stream_t stream) {
    if (B > 0 && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) {
        attn::set_error("cu_seqlens_q and cu_seqlens_k must be non-null");
        return ATTN_ERR_INVALID;
    }
    if (total_q < 0 || total_k < 0) {
        attn::set_error("negative size (total_q=%d total_k=%d)", total_q, total_k);
        return ATTN_ERR_INVALID;
    }
    if (total_q == 0) return ATTN_OK;
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, total_q, total_k, max_Q, max_K, D, Dv,
                      nullptr, nullptr, cu_seqlens_q, cu_seqlens_k, window, scale, mask, dtype,
                      algo, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_varlen_algo(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int Hq, int Hkv, int total_q, int total_k, int max_Q, int max_K,
                         int D, int Dv, const int32_t *cu_seqlens_q,
                         const int32_t *cu_seqlens_k, int window, float scale, int dtype,
                         int algo, attn_stream_t stream) {
    return attn_fwd_varlen_ex(q, k, v, o, lse, B, Hq, Hkv, total_q, total_k, max_Q, max_K, D, Dv,
                              cu_seqlens_q, cu_seqlens_k, window, scale, ATTN_MASK_CAUSAL, dtype,
                              algo, stream);
}

int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int Hq, int Hkv, int total_q, int total_k, int max_Q, int max_K, int D,
                    int Dv, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                    int window, float scale, int dtype, attn_stream_t stream) {
    return attn_fwd_varlen_algo(q, k, v, o, lse, B, Hq, Hkv, total_q, total_k, max_Q, max_K, D,
                                Dv, cu_seqlens_q,
                                cu_seqlens_k, window, scale, dtype, ATTN_ALGO_AUTO, stream);
}

int attn_lse_combine(const float *o_parts, const float *lse_parts, void *o, float *lse,
                     int nsplit, long long rows, int Dv, int dtype, attn_stream_t stream) {
    clear_error();
    if (nsplit < 1 || rows < 0 || Dv < 1 || Dv > 4096 || dtype < ATTN_F32 || dtype > ATTN_BF16) {
        attn::set_error("attn_lse_combine: bad size or dtype (nsplit=%d rows=%lld Dv=%d)",
                        nsplit, rows, Dv);
        return ATTN_ERR_INVALID;
    }
    if (rows > 0 && (o_parts == nullptr || lse_parts == nullptr || o == nullptr)) {
        attn::set_error("attn_lse_combine: null pointer");
        return ATTN_ERR_INVALID;
    }
    if (rows > (1LL << 40)) {
        attn::set_error("attn_lse_combine: too many rows");
        return ATTN_ERR_UNSUPPORTED;
    }
    return launch_combine_flat(o_parts, lse_parts, o, lse, nsplit, rows, Dv, dtype,
                               reinterpret_cast<cudaStream_t>(stream));
}

int attn_lse_combine_ex(const void *o_parts, const float *lse_parts, void *o, float *lse,
                        int nsplit, long long rows, int Dv, int parts_dtype, int dtype,
                        attn_stream_t stream) {
    clear_error();
    if (parts_dtype == ATTN_F32)
        return attn_lse_combine(static_cast<const float *>(o_parts), lse_parts, o, lse, nsplit,
                                rows, Dv, dtype, stream);
    if (nsplit < 1 || rows < 0 || Dv < 1 || Dv > 4096 || parts_dtype < ATTN_F32 ||
        parts_dtype > ATTN_BF16 || dtype < ATTN_F32 || dtype > ATTN_BF16) {
        attn::set_error("attn_lse_combine_ex: bad size or dtype (nsplit=%d rows=%lld Dv=%d)",
                        nsplit, rows, Dv);
        return ATTN_ERR_INVALID;
    }
    if (rows > 0 && (o_parts == nullptr || lse_parts == nullptr || o == nullptr)) {
        attn::set_error("attn_lse_combine_ex: null pointer");
        return ATTN_ERR_INVALID;
    }
    if (rows > (1LL << 40)) {
        attn::set_error("attn_lse_combine_ex: too many rows");
        return ATTN_ERR_UNSUPPORTED;
    }
    return launch_combine_parts(o_parts, parts_dtype, lse_parts, o, lse, nsplit, rows, Dv, dtype,
                                reinterpret_cast<cudaStream_t>(stream));
}

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Q, int K,
             int D, int Dv, const int32_t *seqlens_q, const int32_t *seqlens_k, int window,
             float scale, int mask, int dtype, int algo, attn_stream_t stream) {
    return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, (long long)B * Q,
                      (long long)B * K, Q, K, D, Dv, seqlens_q, seqlens_k, nullptr, nullptr,
                      window, scale, mask, dtype, algo, reinterpret_cast<cudaStream_t>(stream));
}

int attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                    const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                    int total_q, int total_k, int max_Q, int max_K, int D, int Dv,
                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int window,
                    float scale, int mask, int dtype, int algo, attn_stream_t stream) {
    if (B > 0 && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) {
        attn::set_error("cu_seqlens_q and cu_seqlens_k must be non-null");
        return ATTN_ERR_INVALID;
    }
    if (total_q < 0 || total_k < 0) {
        attn::set_error("negative size (total_q=%d total_k=%d)", total_q, total_k);
        return ATTN_ERR_INVALID;
    }
    return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, total_q, total_k, max_Q,
                      max_K, D, Dv, nullptr, nullptr, cu_seqlens_q, cu_seqlens_k, window, scale,
                      mask, dtype, algo, reinterpret_cast<cudaStream_t>(stream));
}

const char *attn_last_error(void) { return g_last_error; }

int attn_device_status(int *detail) {
    if (detail) *detail = 0;
    int dev = 0;
    int rc = current_device(&dev);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        attn::set_error("cudaDeviceSynchronize: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    int value = 0;
    e = cudaMemcpyFromSymbol(&value, g_device_status, sizeof(int));
    if (e != cudaSuccess) {
        attn::set_error("reading the status word: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) {
        attn::set_error("clearing the status word: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    if (detail) *detail = value;
    return value == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

unsigned long long attn_kernel_launches(void) {
    return g_launches.load(std::memory_order_relaxed);
}

unsigned long long attn_set_wait_limit(unsigned long long ns) {
    return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

const char *attn_version(void) { return "0.2.0"; }

}  // extern "C"
