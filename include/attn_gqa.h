/*
 * attn_gqa.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention
 * forward library (libattn_gqa.so).
 *
 * Operation.  Every entry point computes, for each sequence b, query head h and
 * valid query row q, the softmax attention
 *
 *     O[q,h,:] = sum_k p_k V[k,kh,:],   p_k = exp(s_k - LSE[q,h]),
 *     s_k      = scale * <Q[q,h,:], K[k,kh,:]>,
 *     LSE[q,h] = log sum_{k legal} exp(s_k)            (natural log)
 *
 * over the legal keys of the row, with kh = h / (Hq / Hkv):
 *
 *     0 <= k < Kb,   k <= q + Kb - Qb,
 *     and, when window > 0,   k >= q + Kb - Qb - window + 1.
 *
 * Sources: "Attention execution mapping: 现状、缺口与有界实验"
 * (LuisaCompute), section 1 (bottom-right causal GQA, kh = h / (Hq/Hkv),
 * legal keys k <= q + K - Q, one online-softmax program for prefill and
 * decode with row max / row sum / accumulator carried across KV blocks) and
 * section 5 (split-KV needs a legal merge of the (max, sum, acc) state);
 * "快速後端" (Laya fast backends), numerical verification (sliding window,
 * int32 per-sequence lengths, empty sequences, finite padded output).
 * The window reading (the w most recent keys including the diagonal one),
 * the empty-row convention and the natural-log LSE are this library's
 * readings where the pages are silent.
 *
 * Rows with no legal key (Kb = 0, leading rows when Qb > Kb, or a window
 * that excludes every key) return O = +0.0 and LSE = -inf.  Padded query rows
 * q >= Qb of the padded layout are written as O = +0.0 and LSE = -inf.
 *
 * Memory and ownership.  All tensor and length pointers are DEVICE pointers
 * owned by the caller; the library never frees or retains them.  Tensors are
 * dense and contiguous (row-major in the order given), 16-byte aligned.
 * Key / value rows past a sequence's length are never used as values: they
 * may hold anything, NaN included.
 *
 * Asynchrony.  Every call validates its host-side arguments, enqueues its
 * kernels on `stream` and returns; nothing synchronises.  Split-KV calls take
 * their temporary workspace from a library-owned stream-ordered pool
 * (cudaMallocAsync / cudaFreeAsync on `stream`).
 *
 * Errors.  Calls return ATTN_OK or a status below; no exception crosses the
 * ABI.  attn_last_error() gives a message for the calling thread's last
 * failure.  Device-side contract violations found by the kernels (a bounded
 * wait that ran out) are recorded in a device status word read by
 * attn_device_status().
 */
#ifndef ATTN_GQA_H
#define ATTN_GQA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

/* Element types of q, k, v and o.  lse is always float32. */
enum attn_dtype { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 };

/* Status codes. */
enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,     /* null pointer, negative size, Hq % Hkv != 0 ... */
    ATTN_ERR_UNSUPPORTED = 2, /* dtype / head-width / algorithm combination */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    ATTN_ERR_TIMEOUT = 4      /* a kernel's bounded wait ran out (device status) */
};

/* Kernel selection for the *_algo entry points. */
enum attn_algo {
    ATTN_ALGO_AUTO = 0,     /* choose by dtype, head widths and query length */
    ATTN_ALGO_GENERIC = 1,  /* CUDA-core online softmax: any dtype, D, Dv <= 512 */
    ATTN_ALGO_TCGEN05 = 2,  /* tcgen05/TMEM prefill: bf16/fp16, D, Dv multiples of 16 in
                               [64, 512], not paged above 128; in the backward, the
                               tcgen05 dQ and dK/dV kernels (D, Dv in [64, 128]) */
    ATTN_ALGO_DECODE = 3,   /* split-KV tensor-core decode: bf16/fp16, Q*G <= 16 */
    ATTN_ALGO_MMA = 4       /* warp-level mma.sync tensor cores, bf16/fp16: the forward for
                               D, Dv multiples of 8 up to 512 (chosen by AUTO where the
                               tcgen05 and decode kernels do not apply), the backward for
                               D, Dv multiples of 8 up to 128 */
};

/* Which keys a query row may attend to (attn_fwd_ex, attn_fwd_varlen_ex). */
enum attn_mask {
    ATTN_MASK_CAUSAL = 0,          /* bottom-right causal: key k <= q + Kb - Qb (attn_fwd's) */
    ATTN_MASK_CAUSAL_TOP_LEFT = 1, /* top-left causal: key k <= q */
    ATTN_MASK_NONE = 2             /* every key k < Kb (no window allowed) */
};

/*
 * attn_fwd -- padded layout.
 *   q   [B, Q, Hq, D]    o   [B, Q, Hq, Dv]    lse [B, Q, Hq] (float32, may be NULL)
 *   k   [B, K, Hkv, D]   v   [B, K, Hkv, Dv]
 *   Q, K        padded capacities (query rows / key rows per sequence).
 *   seqlens_q   int32 [B] valid query rows per sequence, or NULL for all Q.
 *   seqlens_k   int32 [B] valid key rows per sequence, or NULL for all K.
 *               Values outside [0, Q] / [0, K] are clamped into range.
 *   window      > 0: keep the `window` most recent keys (diagonal included);
 *               <= 0: no window.
 *   scale       multiplies Q.K (pass 1/sqrt(D) for the usual scaling).
 *   dtype       attn_dtype of q, k, v and o.
 * Returns ATTN_OK, ATTN_ERR_INVALID (bad pointer or size, Hq % Hkv != 0,
 * D or Dv outside [1, 512]), ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 * B = 0, Q = 0 or Hq = 0 work is a successful no-op.
 */
ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
             const int32_t *seqlens_k, int window, float scale, int dtype,
             attn_stream_t stream);

/*
 * attn_fwd_varlen -- packed layout.
 *   q [Tq, Hq, D]  k [Tk, Hkv, D]  v [Tk, Hkv, Dv]  o [Tq, Hq, Dv]  lse [Tq, Hq] (may be NULL)
 *   total_q, total_k   rows of the packed buffers (Tq, Tk): bounds every read
 *               and write; cu_seqlens_q[B] <= total_q, cu_seqlens_k[B] <= total_k.
 *   cu_seqlens_q, cu_seqlens_k   int32 [B+1], cu[0] = 0, non-decreasing:
 *               sequence b owns query rows [cu_q[b], cu_q[b+1]) and key rows
 *               [cu_k[b], cu_k[b+1]); an empty sequence owns none.
 *   max_Q, max_K   upper bounds of the per-sequence lengths (sizes the grid;
 *               a sequence longer than them is cut to its first max_Q query
 *               rows / max_K key rows).
 * Other arguments and return codes as attn_fwd.  Rows outside every
 * sequence are not written.
 */
ATTN_API int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int Hq, int Hkv, int total_q, int total_k, int max_Q, int max_K, int D, int Dv,
                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int window,
                    float scale, int dtype, attn_stream_t stream);

/* The same two operations with an explicit kernel choice (attn_algo).  A
 * choice that cannot run the given shape returns ATTN_ERR_UNSUPPORTED. */
ATTN_API int attn_fwd_algo(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                  int Hq, int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                  const int32_t *seqlens_k, int window, float scale, int dtype, int algo,
                  attn_stream_t stream);
ATTN_API int attn_fwd_varlen_algo(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int Hq, int Hkv, int total_q, int total_k, int max_Q, int max_K,
                         int D, int Dv,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int window,
                         float scale, int dtype, int algo, attn_stream_t stream);

/*
 * attn_fwd_ex / attn_fwd_varlen_ex -- the two operations with an explicit
 * mask (attn_mask) and kernel choice (attn_algo).  The pages define the
 * bottom-right causal mask only; the top-left causal mask and no mask are
 * extensions of this library: the same online-softmax recurrence over a
 * different set of legal keys (a window applies to the causal masks only:
 * ATTN_MASK_NONE with window > 0 is ATTN_ERR_INVALID).
 */
ATTN_API int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int Hq, int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                         const int32_t *seqlens_k, int window, float scale, int mask, int dtype,
                         int algo, attn_stream_t stream);
ATTN_API int attn_fwd_varlen_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int total_q, int total_k, int max_Q,
                                int max_K, int D, int Dv, const int32_t *cu_seqlens_q,
                                const int32_t *cu_seqlens_k, int window, float scale, int mask,
                                int dtype, int algo, attn_stream_t stream);

/*
 * attn_lse_combine -- the legal merge of split-KV partial states (the
 * "(max, sum, acc)" merge of the LuisaCompute page, section 5), written as a
 * merge of normalised partials:
 *   o_parts   float32 [nsplit, rows, Dv]   each partial normalised by its own sum
 *   lse_parts float32 [nsplit, rows]       natural-log LSE of each partial;
 *                                          -inf marks a partial with no key
 *   o         [rows, Dv] in `dtype`;  lse [rows] float32 (may be NULL)
 *   L = log sum_s exp(lse_s);   o = sum_s exp(lse_s - L) o_s.
 * A row whose partials are all -inf gives o = +0 and lse = -inf.
 */
ATTN_API int attn_lse_combine(const float *o_parts, const float *lse_parts, void *o, float *lse,
                     int nsplit, long long rows, int Dv, int dtype, attn_stream_t stream);

/*
 * attn_lse_combine_ex -- attn_lse_combine with the partials in any storage
 * dtype: parts_dtype ATTN_F32 is attn_lse_combine; ATTN_F16 / ATTN_BF16 take
 * o_parts [nsplit, rows, Dv] in that dtype (as attn_fwd wrote them, each
 * normalised by its own sum) and need dtype == parts_dtype.  This merges the
 * outputs of one sequence's key shards computed on several GPUs and exchanged
 * as they are (the sharded decode of the Python package).  Accumulation is in
 * fp32; return codes as attn_lse_combine.
 */
ATTN_API int attn_lse_combine_ex(const void *o_parts, const float *lse_parts, void *o, float *lse,
                                 int nsplit, long long rows, int Dv, int parts_dtype, int dtype,
                                 attn_stream_t stream);

/*
 * attn_fwd_paged -- attn_fwd with the keys and values in pages: a serving
 * layout (the pages have no counterpart; the attention itself is unchanged).
 *   q [B, Q, Hq, D], o [B, Q, Hq, Dv], lse [B, Q, Hq] as in attn_fwd.
 *   k_pages [num_pages, page_size, Hkv, D], v_pages [num_pages, page_size, Hkv, Dv]:
 *               pools of pages of page_size key rows (a power of two).
 *   block_table int32 [B, max_pages] on the device: key j of sequence b is row
 *               j % page_size of page block_table[b][j / page_size].  Entries
 *               outside [0, num_pages) are clamped into it.
 *   seqlens_k   int32 [B] on the device (required), at most max_pages * page_size.
 *   mask, algo  as in attn_fwd_ex.  The tcgen05 prefill takes page sizes that
 *               are multiples of 128; the decode and fp32 kernels take any.
 * Return codes as attn_fwd.
 */
ATTN_API int attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages, void *o,
                            float *lse, int B, int Hq, int Hkv, int Q, int D, int Dv,
                            const int32_t *block_table, int max_pages, int page_size,
                            int num_pages, const int32_t *seqlens_q, const int32_t *seqlens_k,
                            int window, float scale, int mask, int dtype, int algo,
                            attn_stream_t stream);

/*
 * attn_fwd_masked -- attn_fwd_ex with an arbitrary boolean mask on top of the
 * mask mode and the window: key k is legal for query row q of sequence b and
 * query head h only if it is legal under `mask` / `window` and bit k % 32 of
 * word k / 32 of mask row ((b * mask_heads + hm) * Q + q) is set, where hm = h
 * when mask_heads == Hq and hm = 0 when mask_heads == 1 (one mask shared by
 * every head).  ATTN_MASK_NONE with this mask gives a purely arbitrary mask.
 * "Attention execution mapping" (LuisaCompute), section 7, names arbitrary
 * masks as a semantic extension beyond the pages' bottom-right rule; the rest
 * of the definition (the online softmax over the legal keys, +0 / -inf for a
 * row without one) is unchanged.
 *   mask_bits   uint32 [B, mask_heads, Q, mask_words] on the device, 16-byte
 *               aligned; bits of keys at or past a sequence's length are ignored
 *   mask_words  words per row: a multiple of 4, at least 4 * ceil(K / 128)
 *   mask_heads  1 or Hq
 * Padded layout only; other arguments as attn_fwd_ex.  The tcgen05 prefill
 * (ATTN_ALGO_AUTO's choice for bf16/fp16 widths 64..128) skips 128-key tiles in
 * which no row of a work unit has an allowed key, without loading them; the
 * CUDA-core kernel (ATTN_ALGO_GENERIC, and AUTO otherwise) tests every key.
 * ATTN_ALGO_DECODE and ATTN_ALGO_MMA return ATTN_ERR_UNSUPPORTED.  Extra
 * workspace from the library's pool: ceil(K / 128) bytes per query block and
 * head group.  Return codes as attn_fwd.
 */
ATTN_API int attn_fwd_masked(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int Hq, int Hkv, int Q, int K, int D, int Dv,
                             const int32_t *seqlens_q, const int32_t *seqlens_k,
                             const uint32_t *mask_bits, int mask_words, int mask_heads, int window,
                             float scale, int mask, int dtype, int algo, attn_stream_t stream);

/*
 * attn_fwd_decode_noalloc -- attn_fwd's split-KV decode for callers that may
 * not allocate device memory while attention runs: for example a serving
 * process whose device memory is owned by another runtime's allocator or held
 * under a hard cap, or a latency-critical decode loop where an allocation (or
 * a synchronisation it may bring) is not allowed.  The pages have no
 * counterpart to this entry point; it is a deployment aid of this library.
 *
 * Same arguments, layout and result as attn_fwd, restricted to the shapes the
 * decode kernel takes (bf16/fp16, D and Dv in {64, 128} or both 256, Q * Hq / Hkv <= 16).
 * The split-KV partials live in a fixed 32 MiB __device__ array that every
 * GPU using the library keeps until the process exits; the call makes no
 * allocation of any kind.  A problem whose partials would not fit returns
 * ATTN_ERR_UNSUPPORTED with a message giving the bytes needed.  The first
 * call on a device looks up the array's device address (make that call before
 * any stream capture).  All calls share the array: calls that overlap on the
 * GPU (other streams or host threads on the same device) race on it and must
 * be serialised by the caller.  Nothing in the array needs to start at zero.
 */
ATTN_API int attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o,
                                     float *lse, int B, int Hq, int Hkv, int Q, int K, int D,
                                     int Dv, const int32_t *seqlens_q, const int32_t *seqlens_k,
                                     int window, float scale, int dtype, attn_stream_t stream);

/*
 * attn_fwd_staged -- attn_fwd on tensors that live in host memory.  A
 * serving aid of this library (the pages have no counterpart): the batch is
 * cut into `chunks` groups of sequences (<= 0: 4; at most B and 32), and for
 * each group the host->device copy of its inputs, its attention launch (on
 * `stream`, exactly as attn_fwd) and the device->host copy of its outputs are
 * ordered by events across three streams, so the copies of one group overlap
 * the attention of another.
 *   hq, hk, hv, ho, hlse   host tensors, padded layout as in attn_fwd (hlse
 *                          may be NULL); page-locked memory is needed for the
 *                          copies to overlap anything
 *   q, k, v, o, lse        caller-owned device buffers of the same shapes,
 *                          used as staging (lse may be NULL only with hlse)
 *   seqlens_q, seqlens_k   as in attn_fwd (device int32 [B] or NULL), and
 *   seqlens_q_host, seqlens_k_host  the same values in host memory (NULL
 *                          exactly when the device array is NULL): only rows
 *                          [0, Qb) of q and [0, Kb) of k and v are copied in;
 *                          every row of o and lse is copied out
 *   bytes_in, bytes_out    (may be NULL) receive the bytes copied each way
 * Asynchronous like attn_fwd: `stream` is ordered after the last copy out.
 * Calls on one device are serialised inside the library (they share its two
 * copy streams).  Return codes as attn_fwd.
 */
ATTN_API int attn_fwd_staged(const void *hq, const void *hk, const void *hv, void *ho, float *hlse,
                             void *q, void *k, void *v, void *o, float *lse, int B, int Hq,
                             int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                             const int32_t *seqlens_k, const int32_t *seqlens_q_host,
                             const int32_t *seqlens_k_host, int window, float scale, int dtype,
                             int chunks, unsigned long long *bytes_in,
                             unsigned long long *bytes_out, attn_stream_t stream);

/*
 * attn_bwd -- gradients of attn_fwd_ex (padded layout) for a loss whose
 * gradient with respect to o is dout.  "Accelerating PyTorch on AMD GPUs
 * with FlyDSL", section on FMHA through AOTriton, describes such a backward
 * as separate dQ and dK/dV kernels reusing the forward's building blocks,
 * without its arithmetic; the arithmetic here is the derivative of the
 * forward definition (O = softmax(scale Q K^T + mask) V per row, with the
 * row's log-sum-exp kept).  With P = exp(scale q.k - LSE) over the row's legal
 * keys and Dq = sum(dO * O) over the row:
 *     dS = P (dO . v - Dq)
 *     dq = scale sum_k dS k
 *     dk = scale sum over rows of dS q
 *     dv = sum over rows of P dO
 * where a KV head's dk and dv sum over every query head of its group.
 *   q, k, v       the forward's inputs, shapes as in attn_fwd
 *   o, lse        the forward's outputs for those inputs (lse required);
 *                 P is recomputed from lse, nothing else is stored
 *   dout          [B, Q, Hq, Dv], same dtype as q
 *   dq, dk, dv    outputs shaped like q, k, v (same dtype), written in full:
 *                 rows past seqlens_q, keys past seqlens_k, rows without a
 *                 legal key and keys no row attends to get zeros
 *   seqlens_q, seqlens_k, window, scale, mask   as in attn_fwd_ex
 *   algo          ATTN_ALGO_AUTO (ATTN_ALGO_TCGEN05 where it applies, else
 *                 ATTN_ALGO_MMA, else the CUDA-core kernels), ATTN_ALGO_GENERIC,
 *                 ATTN_ALGO_MMA (mma.sync dK/dV and dQ; bf16/fp16, widths
 *                 multiples of 8 up to 128) or ATTN_ALGO_TCGEN05 (tcgen05
 *                 dQ and dK/dV kernels -- the dK/dV one when Hq / Hkv
 *                 divides 128, else mma.sync; bf16/fp16, widths multiples of
 *                 16 in [64, 128], padded or packed layout)
 * Head widths up to 256 (wider ones return ATTN_ERR_UNSUPPORTED).
 * All pointers are device memory, 16-byte aligned.  A workspace of
 * 4 * B * Q * Hq bytes comes from the library's stream-ordered pool.  The
 * result is deterministic (no atomics: dk/dv and dq are written by separate
 * kernels, each element by one thread).  Returns ATTN_OK, ATTN_ERR_INVALID,
 * ATTN_ERR_UNSUPPORTED (ATTN_ALGO_MMA on a shape it does not take) or
 * ATTN_ERR_CUDA; asynchronous on `stream`.
 */
ATTN_API int attn_bwd(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                      int Hq, int Hkv, int Q, int K, int D, int Dv, const int32_t *seqlens_q,
                      const int32_t *seqlens_k, int window, float scale, int mask, int dtype,
                      int algo, attn_stream_t stream);

/* attn_bwd on the packed layout of attn_fwd_varlen_ex: q, o, dout, dq
 * [total_q, Hq, *], k, v, dk, dv [total_k, Hkv, *], sequences given by
 * cu_seqlens_q / cu_seqlens_k (int32 [B + 1]).  Rows of dq, dk and dv
 * outside every sequence are not written. */
ATTN_API int attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int B, int Hq, int Hkv, int total_q, int total_k, int max_Q,
                             int max_K, int D, int Dv, const int32_t *cu_seqlens_q,
                             const int32_t *cu_seqlens_k, int window, float scale, int mask,
                             int dtype, int algo, attn_stream_t stream);

/* Message for the calling thread's most recent failed call ("" if none). */
ATTN_API const char *attn_last_error(void);

/* Reads and clears the device status word of the current device
 * (synchronises the device).  Returns ATTN_OK, ATTN_ERR_TIMEOUT, or
 * ATTN_ERR_CUDA if the read itself failed; *detail (may be NULL) receives the
 * kernel-specific detail code. */
ATTN_API int attn_device_status(int *detail);

/*
 * Sets the time limit of the mbarrier waits inside the tcgen05 kernels
 * (prefill, backward) for launches made after the call, in nanoseconds, for
 * every thread and device of the process; 0 restores the default of 2 s.
 * Returns the previous limit.  A wait that runs out records ATTN_ERR_TIMEOUT
 * and a detail code in the device status word (attn_device_status), and the
 * launch unwinds: its blocks wait (up to 2 s, whatever this limit) for their
 * own copies and tensor-core operations in flight, free their tensor memory
 * and return, leaving the outputs incomplete and the context usable.  A
 * diagnostic aid: a limit shorter than the kernel's run makes a correct launch
 * time out on purpose, which is how the timeout path is tested.  The pages
 * have no counterpart ("Attention execution mapping" records a submission
 * stall, section 21.9, which is why the waits are bounded at all).
 */
ATTN_API unsigned long long attn_set_wait_limit(unsigned long long ns);

/* Number of kernels this library has launched in the process so far (all
 * devices, all threads).  A measurement aid: the difference around a region
 * counts the library's launches inside it. */
ATTN_API unsigned long long attn_kernel_launches(void);

/* Library version, e.g. "0.1.0". */
ATTN_API const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GQA_H */
