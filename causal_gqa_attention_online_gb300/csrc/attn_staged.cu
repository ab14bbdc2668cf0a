// attn_staged.cu -- attn_fwd on host-resident tensors: the batch is cut into
// chunks of sequences, and each chunk's host->device copy, attention launch and
// device->host copy run on three streams, so the copies of one chunk overlap
// the attention of another.  Only the valid rows of each sequence are copied
// in (padding is never read by the kernels).  Declared in include/attn_gqa.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "attn_gqa.h"
#include "common.cuh"
#include "launch.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 32;

// Per device: the copy-in and copy-out streams and the events that order them.
struct Staging {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kMaxChunks] = {};
    cudaEvent_t run_done[kMaxChunks] = {};
};
std::mutex g_staging_mutex[kMaxDevices];
Staging g_staging[kMaxDevices];

int staging_init(Staging &s) {
    if (s.ready) return 0;
    cudaError_t e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.end, cudaEventDisableTiming);
    for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
        e = cudaEventCreateWithFlags(&s.in_done[c], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.run_done[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        set_error("attn_fwd_staged: stream/event setup: %s", cudaGetErrorString(e));
        return ATTN_ERR_CUDA;
    }
    s.ready = true;
    return 0;
}

// Copies rows [0, n_b) of every sequence b in [b0, b1) of a padded tensor
// (`cap` rows of `row` bytes per sequence); runs of whole sequences go as one copy.
cudaError_t copy_rows(char *dst, const char *src, int b0, int b1, long long cap, size_t row,
                      const int32_t *n, cudaMemcpyKind kind, cudaStream_t st,
                      unsigned long long *bytes) {
    int b = b0;
    while (b < b1) {
        const long long nb = n ? std::min<long long>(std::max(n[b], 0), cap) : cap;
        if (nb == cap) {  // extend a run of whole sequences
            int e = b + 1;
            while (e < b1 && (n == nullptr || std::min<long long>(std::max(n[e], 0), cap) == cap))
                ++e;
            const size_t off = (size_t)b * cap * row, len = (size_t)(e - b) * cap * row;
            if (len) {
                const cudaError_t err = cudaMemcpyAsync(dst + off, src + off, len, kind, st);
                if (err != cudaSuccess) return err;
                *bytes += len;
            }
            b = e;
        } else {
            const size_t off = (size_t)b * cap * row, len = (size_t)nb * row;
            if (len) {
                const cudaError_t err = cudaMemcpyAsync(dst + off, src + off, len, kind, st);
                if (err != cudaSuccess) return err;
                *bytes += len;
            }
            ++b;
        }
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace attn

using namespace attn;

int attn_fwd_staged(const void *hq, const void *hk, const void *hv, void *ho, float *hlse,
                    void *q, void *k, void *v, void *o, float *lse, int B, int Hq, int Hkv, int Q,
                    int K, int D, int Dv, const int32_t *seqlens_q, const int32_t *seqlens_k,
                    const int32_t *seqlens_q_host, const int32_t *seqlens_k_host, int window,
                    float scale, int dtype, int chunks, unsigned long long *bytes_in,
                    unsigned long long *bytes_out, attn_stream_t stream) {
    if (bytes_in) *bytes_in = 0;
    if (bytes_out) *bytes_out = 0;
    if (B < 0 || Q < 0 || K < 0 || Hq < 0 || Hkv <= 0 || D <= 0 || Dv <= 0 ||
        dtype < ATTN_F32 || dtype > ATTN_BF16) {
        set_error("attn_fwd_staged: bad size or dtype");
        return ATTN_ERR_INVALID;
    }
    if ((seqlens_q == nullptr) != (seqlens_q_host == nullptr) ||
        (seqlens_k == nullptr) != (seqlens_k_host == nullptr)) {
        set_error("attn_fwd_staged: give each seqlens array both on the device and on the host, "
                  "or neither");
        return ATTN_ERR_INVALID;
    }
    if ((long long)B * Q * Hq == 0) return ATTN_OK;
    if (!hq || !hk || !hv || !ho || !q || !k || !v || !o || (hlse != nullptr && lse == nullptr)) {
        set_error("attn_fwd_staged: null buffer");
        return ATTN_ERR_INVALID;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_error("attn_fwd_staged: cudaGetDevice failed");
        return ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_staging_mutex[dev]);
    Staging &S = g_staging[dev];
    int rc = staging_init(S);
    if (rc) return rc;

    const int nch = std::max(1, std::min({chunks > 0 ? chunks : 4, B, kMaxChunks}));
    const size_t es = dtype == ATTN_F32 ? 4 : 2;
    const size_t qrow = (size_t)Hq * D * es, krow = (size_t)Hkv * D * es,
                 vrow = (size_t)Hkv * Dv * es, orow = (size_t)Hq * Dv * es, lrow = (size_t)Hq * 4;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long bin = 0, bout = 0;

    // the device buffers and the host outputs are free once the caller's
    // earlier work on `stream` is done
    cudaError_t e = cudaEventRecord(S.start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(S.in, S.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(S.out, S.start, 0);
    for (int c = 0; c < nch && e == cudaSuccess && rc == 0; ++c) {
        const int b0 = (int)((long long)B * c / nch), b1 = (int)((long long)B * (c + 1) / nch);
        // in: valid query rows, valid key / value rows
        e = copy_rows(static_cast<char *>(q), static_cast<const char *>(hq), b0, b1, Q, qrow,
                      seqlens_q_host, cudaMemcpyHostToDevice, S.in, &bin);
        if (e == cudaSuccess)
            e = copy_rows(static_cast<char *>(k), static_cast<const char *>(hk), b0, b1, K, krow,
                          seqlens_k_host, cudaMemcpyHostToDevice, S.in, &bin);
        if (e == cudaSuccess)
            e = copy_rows(static_cast<char *>(v), static_cast<const char *>(hv), b0, b1, K, vrow,
                          seqlens_k_host, cudaMemcpyHostToDevice, S.in, &bin);
        if (e == cudaSuccess) e = cudaEventRecord(S.in_done[c], S.in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, S.in_done[c], 0);
        if (e != cudaSuccess) break;
        // attention on the chunk
        rc = attn_fwd(static_cast<const char *>(q) + (size_t)b0 * Q * qrow,
                      static_cast<const char *>(k) + (size_t)b0 * K * krow,
                      static_cast<const char *>(v) + (size_t)b0 * K * vrow,
                      static_cast<char *>(o) + (size_t)b0 * Q * orow,
                      lse ? lse + (size_t)b0 * Q * Hq : nullptr, b1 - b0, Hq, Hkv, Q, K, D, Dv,
                      seqlens_q ? seqlens_q + b0 : nullptr, seqlens_k ? seqlens_k + b0 : nullptr,
                      window, scale, dtype, stream);
        if (rc) break;
        e = cudaEventRecord(S.run_done[c], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(S.out, S.run_done[c], 0);
        // out: every query row (padded rows hold +0 / -inf)
        if (e == cudaSuccess) {
            const size_t off = (size_t)b0 * Q * orow, len = (size_t)(b1 - b0) * Q * orow;
            e = cudaMemcpyAsync(static_cast<char *>(ho) + off, static_cast<const char *>(o) + off,
                                len, cudaMemcpyDeviceToHost, S.out);
            bout += len;
        }
        if (e == cudaSuccess && hlse) {
            const size_t off = (size_t)b0 * Q * lrow, len = (size_t)(b1 - b0) * Q * lrow;
            e = cudaMemcpyAsync(reinterpret_cast<char *>(hlse) + off,
                                reinterpret_cast<const char *>(lse) + off, len,
                                cudaMemcpyDeviceToHost, S.out);
            bout += len;
        }
    }
    // the caller's stream continues after the last copy out (and any copy in)
    cudaError_t e2 = cudaEventRecord(S.end, S.out);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, S.end, 0);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(S.end, S.in);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, S.end, 0);
    if (bytes_in) *bytes_in = bin;
    if (bytes_out) *bytes_out = bout;
    if (rc) return rc;
    if (e != cudaSuccess || e2 != cudaSuccess) {
        set_error("attn_fwd_staged: %s", cudaGetErrorString(e != cudaSuccess ? e : e2));
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}
