// attn_noalloc.cu -- attn_fwd_decode_noalloc: the split-KV decode of attn_fwd
// with its scratch taken from a fixed device array instead of the allocator.
//
// Who needs it: a caller that must not allocate device memory while it runs
// attention -- for example a serving process that embeds this library under
// another runtime which owns every byte of device memory (its own caching
// allocator or a hard memory cap), or a latency-critical decode loop where an
// allocation, or the synchronisation an allocator may perform, is not
// allowed.  attn_fwd takes its split-KV partials from a stream-ordered pool;
// this entry point takes them from `g_noalloc_scratch` below and never calls
// cudaMalloc, cudaMallocAsync, cudaFree or any other allocating routine.
//
// The array is a file-scope __device__ object: every GPU on which this
// library's code is loaded holds kNoAllocScratchBytes of it until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it is only a stand-in object), so the device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first
// call made on it; that first call should therefore come before any stream
// capture.  All calls share the one array, which keeps whatever the previous
// call left in it: two calls that overlap on the GPU (different streams, or
// different host threads on one device) race on it and must be serialised by
// the caller.  Nothing in it has to start at zero: every partial result the
// combine step reads is written by the same call first.
#include <cstring>
#include <mutex>

#include "attn_gqa.h"
#include "common.cuh"
#include "launch.h"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        set_error("attn_fwd_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            set_error("attn_fwd_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return ATTN_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o,
                                       float *lse, int B, int Hq, int Hkv, int Q, int K, int D,
                                       int Dv, const int32_t *seqlens_q,
                                       const int32_t *seqlens_k, int window, float scale,
                                       int dtype, attn_stream_t stream) {
    using namespace attn;
    if (B < 0 || Hq < 0 || Hkv < 0 || Q < 0 || K < 0) {
        set_error("attn_fwd_decode_noalloc: negative size");
        return ATTN_ERR_INVALID;
    }
    if (Hq > 0 && (Hkv == 0 || Hq % Hkv != 0)) {
        set_error("attn_fwd_decode_noalloc: Hq (%d) must be a positive multiple of Hkv (%d)", Hq,
                  Hkv);
        return ATTN_ERR_INVALID;
    }
    if ((long long)B * Q * Hq == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr || (K > 0 && (k == nullptr || v == nullptr))) {
        set_error("attn_fwd_decode_noalloc: null tensor pointer");
        return ATTN_ERR_INVALID;
    }
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                          reinterpret_cast<uintptr_t>(lse);
    if (mis & 15u) {
        set_error("attn_fwd_decode_noalloc: tensor pointers must be 16-byte aligned");
        return ATTN_ERR_INVALID;
    }
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
    p.Tq = (long long)B * Q;
    p.Tk = (long long)B * K;
    p.D = D;
    p.Dv = Dv;
    p.seqlens_q = seqlens_q;
    p.seqlens_k = seqlens_k;
    p.window = (window <= 0 || window >= K) ? 0 : window;
    p.mask = 0;  // bottom-right causal, as attn_fwd
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    if (!decode_supported(p, dtype)) {
        set_error("attn_fwd_decode_noalloc: the decode kernel takes bf16/fp16, D and Dv in "
                  "{64, 128} or both 256, and Q * Hq / Hkv <= 16");
        return ATTN_ERR_UNSUPPORTED;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        set_error("attn_fwd_decode_noalloc: cudaGetDevice failed");
        return ATTN_ERR_CUDA;
    }
    // the same split of the key axis as attn_fwd, so both give the same result
    p.split_len = decode_split_len(p, sm_count(dev));
    if (p.split_len < 1) p.split_len = 1;
    p.nsplit = K > 0 ? (int)(((long long)K + p.split_len - 1) / p.split_len) : 1;
    if (p.nsplit > 1) {
        const long long rows = (long long)p.nsplit * B * Q * Hq;
        const unsigned long long need = 4ull * (unsigned long long)rows * (unsigned long long)(Dv + 1);
        if (need > kNoAllocScratchBytes) {
            set_error("attn_fwd_decode_noalloc: this problem needs %llu bytes of split-KV "
                      "scratch; the fixed scratch array holds %llu bytes (use attn_fwd)",
                      need, (unsigned long long)kNoAllocScratchBytes);
            return ATTN_ERR_UNSUPPORTED;
        }
        void *scratch = nullptr;
        const int rc = noalloc_scratch(&scratch);
        if (rc) return rc;
        p.part_o = static_cast<float *>(scratch);
        p.part_lse = p.part_o + rows * Dv;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = launch_decode(p, dtype, s);
    if (rc == 0 && p.nsplit > 1) rc = launch_combine_rows(p, dtype, s);
    return rc;
}
