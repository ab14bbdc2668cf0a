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

// Device address of the scratch array on `dev`, the current device (looked
// up once per device).
int noalloc_scratch(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch);
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
    clear_error();
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Q, K, D, Dv, dtype, ATTN_ALGO_DECODE);
    if (rc) return rc;
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
    p.wait_ns = wait_limit_ns();
    if (!decode_supported(p, dtype)) {
        set_error("attn_fwd_decode_noalloc: the decode kernel takes bf16/fp16, D and Dv in "
                  "{64, 128} or both 256, and Q * Hq / Hkv <= 16");
        return ATTN_ERR_UNSUPPORTED;
    }
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        set_error("attn_fwd_decode_noalloc: cudaGetDevice: %s (device %d)", cudaGetErrorString(e),
                  dev);
        return ATTN_ERR_CUDA;
    }
    // the split of the key axis that attn_fwd plans (the same helper), so both
    // entry points run the same launches
    rc = plan_splits(p, ATTN_ALGO_DECODE, sm_count(dev));
    if (rc) return rc;
    const unsigned long long need = split_workspace_bytes(p);
    if (need > kNoAllocScratchBytes) {
        set_error("attn_fwd_decode_noalloc: this problem needs %llu bytes of split-KV "
                  "scratch; the fixed scratch array holds %llu bytes (use attn_fwd)",
                  need, (unsigned long long)kNoAllocScratchBytes);
        return ATTN_ERR_UNSUPPORTED;
    }
    if (need > 0) {
        void *scratch = nullptr;
        rc = noalloc_scratch(dev, &scratch);
        if (rc) return rc;
        set_split_workspace(p, scratch);
    }
    return launch_split_kv(p, ATTN_ALGO_DECODE, dtype, reinterpret_cast<cudaStream_t>(stream));
}
