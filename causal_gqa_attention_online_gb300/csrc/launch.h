// launch.h -- host-side launchers of the kernels (internal to libattn_gqa).
// Each returns 0 on success, otherwise an attn_status code, and writes a
// message through set_error().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace attn {

void set_error(const char *fmt, ...);
void clear_error();   // the calling thread's message becomes ""
void count_launch();  // one successful kernel launch
int sm_count(int device);  // 0 if the device index or the query is bad
unsigned long long wait_limit_ns();  // limit of the tcgen05 kernels' mbarrier waits

// Host-side argument checks shared by the entry points (dtype, algo, sizes,
// pointers, 16-byte alignment); 0 or an attn_status code with a message.
int validate(const void *q, const void *k, const void *v, const void *o, const float *lse,
             int B, int Hq, int Hkv, int Q, int K, int D, int Dv, int dtype, int algo);

// Split-KV plan of a decode (chosen = ATTN_ALGO_DECODE) or CUDA-core problem:
// sets p.split_len and p.nsplit.  The partials need split_workspace_bytes(p)
// bytes (0 when nsplit == 1) at a 16-byte aligned address handed over with
// set_split_workspace; launch_split_kv then runs the kernel and, for
// nsplit > 1, the combine.
int plan_splits(AttnParams &p, int chosen, int nsm);
unsigned long long split_workspace_bytes(const AttnParams &p);
void set_split_workspace(AttnParams &p, void *ws);
int launch_split_kv(const AttnParams &p, int chosen, int dtype, cudaStream_t stream);

// CUDA-core online softmax (any dtype; D, Dv <= 512).  Honours p.nsplit.
int launch_generic(const AttnParams &p, int dtype, cudaStream_t stream);
// Split-KV partial merge, driven by the problem's layout.
int launch_combine_rows(const AttnParams &p, int dtype, cudaStream_t stream);
// Plain [nsplit, rows, Dv] merge for attn_lse_combine.
int launch_combine_flat(const float *o_parts, const float *lse_parts, void *o, float *lse,
                        int nsplit, long long rows, int Dv, int dtype, cudaStream_t stream);
// The same merge with fp16 / bf16 partials (parts_dtype == dtype).
int launch_combine_parts(const void *o_parts, int parts_dtype, const float *lse_parts, void *o,
                         float *lse, int nsplit, long long rows, int Dv, int dtype,
                         cudaStream_t stream);
// Tensor-core split-KV decode (bf16/fp16, Q*G <= 16).  Honours p.nsplit.
bool decode_supported(const AttnParams &p, int dtype);
int decode_split_len(const AttnParams &p, int nsm);
int launch_decode(const AttnParams &p, int dtype, cudaStream_t stream);
// tcgen05/TMEM prefill (bf16/fp16, D and Dv multiples of 16 in [64, 128]).
bool prefill_tc_supported(const AttnParams &p, int dtype);
// Ints of workspace the launch wants for its longest-first unit order (0: the
// natural order is used), and bytes for the live-tile flags of an arbitrary
// mask (0: no mask); order_ws / live_ws hold that many, or are null.
long long prefill_tc_order_len(const AttnParams &p);
long long prefill_tc_live_len(const AttnParams &p);
int launch_prefill_tc(const AttnParams &p, int dtype, cudaStream_t stream, int *order_ws,
                      uint8_t *live_ws);

// tcgen05/TMEM prefill for head widths above 128 (bf16/fp16, D and Dv multiples
// of 16 in [64, 512], at least one above 128; not paged, no arbitrary mask).
// Widths above 256 go to the 512-wide kernel (output columns in halves).
bool prefill_wide_tc_supported(const AttnParams &p, int dtype);
int launch_prefill_wide_tc(const AttnParams &p, int dtype, cudaStream_t stream);
bool prefill_wide512_tc_supported(const AttnParams &p, int dtype);
int launch_prefill_wide512_tc(const AttnParams &p, int dtype, cudaStream_t stream);

// mma.sync forward (bf16/fp16, D and Dv multiples of 8 up to 512): the
// tensor-core path for head widths the tcgen05 prefill kernel does not take.
bool fwd_mma_supported(const AttnParams &p, int dtype);
int launch_fwd_mma(const AttnParams &p, int dtype, cudaStream_t stream);

// 4-D TMA map over 16-bit elements [d3][d2][d1][d0] (d0 innermost), box
// {64, b1, b2, 1}, 128-byte swizzle; returns 0 or an attn_status code.
int make_tma_map_4d(CUtensorMap *map, const void *ptr, bool bf16, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t d3, uint32_t b1, uint32_t b2);

// tcgen05 dQ kernel of the backward (bf16/fp16, D and Dv multiples of 16 in
// [64, 128], not paged).  self_delta 0: bp.delta must already hold
// rowsum(dO * O); 1: the kernel computes it for its rows; 2: and writes it to
// bp.delta.
bool bwd_dq_tc_supported(const AttnParams &p, int dtype);
int launch_bwd_dq_tc(const BwdParams &bp, int dtype, cudaStream_t stream, int self_delta);
// tcgen05 dK/dV kernel: as bwd_dq_tc_supported, and Hq / Hkv divides 128.
// after_dq: launched as a programmatic dependent of the dQ launch just before
// it on the same stream (which writes bp.delta).
bool bwd_dkdv_tc_supported(const AttnParams &p, int dtype);
int launch_bwd_dkdv_tc(const BwdParams &bp, int dtype, cudaStream_t stream, bool after_dq);

// Backward: rowsum(dO * O), then dK/dV and dQ.  mode 0: the CUDA-core
// kernels; 1: the mma.sync kernels (bf16/fp16, bwd_mma_supported); 2: the
// tcgen05 dQ kernel (bwd_dq_tc_supported) and the tcgen05 dK/dV kernel where
// it applies (bwd_dkdv_tc_supported; then the dQ kernel computes rowsum(dO * O)
// and runs first), the mma.sync one otherwise.
bool bwd_mma_supported(const AttnParams &p, int dtype);
int launch_bwd(const BwdParams &bp, int dtype, int mode, cudaStream_t stream);

}  // namespace attn
