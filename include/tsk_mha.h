/*
 * tsk_mha.h -- C ABI of the GB300 (sm_103a) mha_prefill library.
 *
 * Operation (TokenSpeed-kernel README, section "Public API": `mha_prefill`;
 * the workload is GPT-OSS attention -- grouped-query heads, attention sinks,
 * sliding-window and full-attention layers -- page "TokenSpeed-kernel:
 * multi-silicon ...", section "Числа: Gluon на AMD MI355X", and the ai-radar.it
 * article, section "AMD MI355X: la prova sul campo").  The pages do not spell
 * the formula out; this library computes, for every packed sequence s with
 * tokens [start, start+L), token t, query head h and KV head g = h / (Hq/Hkv):
 *
 *     J   = { j : max(start, t - W + 1) <= j <= t }      (W <= 0: no lower window bound)
 *     x_j = scale * <q[t,h,:], k[j,g,:]>
 *     out[t,h,:] = sum_{j in J} e^{x_j} v[j,g,:] / (sum_{j in J} e^{x_j} + e^{sink_h})
 *     lse[t,h]   = log(sum_{j in J} e^{x_j} + e^{sink_h})          (natural log)
 *
 * The sink is a raw logit (not multiplied by `scale`) that joins the softmax
 * normaliser with a zero value vector; without sinks its term is absent.
 *
 * All entry points are host functions; pointers marked "device" must be
 * device-accessible memory of the current CUDA device.  The caller owns every
 * buffer; nothing is retained after a call returns.
 */
#ifndef TSK_MHA_H_
#define TSK_MHA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define TSK_API __attribute__((visibility("default")))
#else
#define TSK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tsk_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  TSK_OK = 0,
  TSK_ERR_INVALID_ARG = -1,    /* NULL where a buffer is required, negative sizes, bad scale */
  TSK_ERR_UNSUPPORTED = -2,    /* D not 64 or 128, Hq % Hkv != 0, sizes beyond the limits below */
  TSK_ERR_ALIGNMENT = -3,      /* q/k/v/out not 16-byte aligned, sinks/lse/cu not 4-byte */
  TSK_ERR_DEVICE = -4,         /* no device, not compute capability 10.3, CUDA error */
  TSK_ERR_OOM = -5,            /* workspace allocation failed */
  TSK_ERR_LAUNCH = -6,         /* kernel launch failed */
  TSK_ERR_DEVICE_TIMEOUT = -7, /* a kernel gave up on a bounded wait (device status word) */
  TSK_ERR_BAD_SEQLENS = -8,    /* device check: cu_seqlens not 0..total_tokens non-decreasing */
  TSK_ERR_BOUNDS = -9          /* libraries built with -DTSK_DEBUG only: a computed global index or
                                  TMA coordinate fell outside its buffer; the access was skipped */
} tsk_status;

/*
 * tsk_mha_prefill -- causal grouped-query attention with sink and window
 * over packed variable-length sequences (the formula above).
 *
 *   q           device, bf16 [total_tokens, Hq, D], contiguous (row stride Hq*D)
 *   k, v        device, bf16 [total_tokens, Hkv, D], contiguous
 *   sinks       device, fp32 [Hq] sink logits, or NULL for no sink
 *   cu_seqlens  device, int32 [num_seqs + 1]; cu[0] = 0, non-decreasing,
 *               cu[num_seqs] = total_tokens.  Zero-length sequences are allowed.
 *   num_seqs    number of packed sequences (>= 0)
 *   total_tokens host copy of cu_seqlens[num_seqs] (the tensor-map extent; the
 *               kernels check it against the device array and report
 *               TSK_ERR_BAD_SEQLENS through tsk_get_device_status on mismatch,
 *               computing nothing in that case)
 *   Hq, Hkv     query / KV heads; Hq % Hkv == 0 (Hq == Hkv is plain MHA)
 *   D           head dimension: 64 (GPT-OSS shapes) or 128 (its own kernel)
 *   window      <= 0: full causal; W >= 1: token t sees keys t-W+1 .. t
 *   scale       multiplier of q.k (finite, > 0); not applied to sinks
 *   out         device, bf16 [total_tokens, Hq, D]; must not overlap q, k, v
 *   lse         device, fp32 [total_tokens, Hq] natural-log normaliser, or NULL
 *   stream      stream to enqueue on
 *
 * Limits: total_tokens * Hq < 2^31, num_seqs < 2^24.
 * Asynchronous: enqueues work on `stream` and returns; no host synchronisation.
 * Results are bitwise deterministic run to run (no split-K, no atomics in the
 * arithmetic).  Host-detectable errors return before anything is enqueued and
 * leave all memory untouched.  The library keeps a small device workspace per
 * (device, stream), created on first use; calls on one stream are ordered,
 * calls on different streams do not share it.  Not safe to call concurrently
 * from several host threads on the same stream.
 * CUDA graphs: once a stream's workspace is warm (an earlier eager call on
 * that stream with at least as many query tiles and sequences), a call
 * enqueues kernel launches only and may be captured on that stream.  The
 * graph keeps using that stream's workspace, so its replays must not overlap
 * other calls on the same stream; a replay reads the inputs the buffers hold
 * when it runs.  The same holds for every entry point below.
 */
TSK_API tsk_status tsk_mha_prefill(const void *q, const void *k, const void *v, const float *sinks,
                           const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                           int32_t Hq, int32_t Hkv, int32_t D, int32_t window, float scale,
                           void *out, float *lse, tsk_stream_t stream);

/*
 * tsk_mha_prefill_kvcache -- prefill over a key/value cache (README, section
 * "Public API": `mha_prefill_with_kvcache`; the pages give no formula).
 * Sequence s has Lq = cu_seqlens_q[s+1] - cu_seqlens_q[s] new query tokens
 * and Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s] >= Lq keys/values: the cached
 * prefix followed by the new tokens' own keys/values.  New token i sits at
 * key position P = Lk - Lq + i and attends to key positions
 * max(0, P - W + 1) .. P of its own sequence (causal aligned to the end of
 * the keys); otherwise as tsk_mha_prefill (sinks, scale, lse, GQA mapping).
 * With Lk == Lq for every sequence this is tsk_mha_prefill.
 *
 *   q             device, bf16 [total_q, Hq, D]
 *   k, v          device, bf16 [total_k, Hkv, D] (contiguous per sequence)
 *   cu_seqlens_q  device, int32 [num_seqs + 1], 0 .. total_q, non-decreasing
 *   cu_seqlens_k  device, int32 [num_seqs + 1], 0 .. total_k, non-decreasing
 *   total_q, total_k  host copies of the last offsets (total_k >= total_q)
 *   out           device, bf16 [total_q, Hq, D]; lse fp32 [total_q, Hq] or NULL
 *
 * Inconsistent offsets (including Lk < Lq for some sequence) are reported as
 * TSK_ERR_BAD_SEQLENS through tsk_get_device_status and nothing is computed.
 * Limits: total_q * Hq < 2^31 and total_k * Hkv < 2^31.
 */
TSK_API tsk_status tsk_mha_prefill_kvcache(const void *q, const void *k, const void *v,
                                           const float *sinks, const int32_t *cu_seqlens_q,
                                           const int32_t *cu_seqlens_k, int32_t num_seqs,
                                           int64_t total_q, int64_t total_k, int32_t Hq,
                                           int32_t Hkv, int32_t D, int32_t window, float scale,
                                           void *out, float *lse, tsk_stream_t stream);

/*
 * tsk_mha_decode_kvcache -- one decoding step over a key/value cache (README,
 * section "Public API": the decode call of the same runtime path; the pages
 * give no formula).  Sequence s has one new query token q[s] and
 * Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s] >= 1 keys/values whose last one is
 * the token's own; the token sits at key position Lk - 1 and attends to key
 * positions max(0, Lk - W) .. Lk - 1 (all of them for W <= 0), with the sink
 * of its head counted once.  Identical to tsk_mha_prefill_kvcache with one
 * query per sequence.  The keys of a sequence are split over several CTAs
 * when the batch alone would not fill the GPU; the last CTA of each
 * (sequence, KV head, block of query heads) to finish merges the splits'
 * partial softmax states.  Two launches: an offset check, then the split
 * kernel.
 *
 *   q             device, bf16 [num_seqs, Hq, D]
 *   k, v          device, bf16 [total_k, Hkv, D] (contiguous per sequence)
 *   sinks         device, fp32 [Hq] or NULL
 *   cu_seqlens_k  device, int32 [num_seqs + 1]: 0 = cu[0] < cu[1] < ... = total_k
 *   max_seqlen_k  host: an upper bound of every Lk (sizes the key splits);
 *                 1 <= max_seqlen_k <= total_k
 *   D             64 or 128; Hq % Hkv == 0 (any group size)
 *   out           device, bf16 [num_seqs, Hq, D]; lse fp32 [num_seqs, Hq] or NULL
 *
 * Offsets that are not strictly increasing, do not end at total_k or have a
 * length above max_seqlen_k are reported as TSK_ERR_BAD_SEQLENS through
 * tsk_get_device_status and nothing is written.  Limits: num_seqs <= 65535,
 * total_k * Hkv < 2^31.  The library keeps a per-(device, stream) buffer of
 * splits x num_seqs x Hq x (D + 2) floats for the partial states and one int
 * counter per (sequence, KV head, block of 16 query heads).
 */
TSK_API tsk_status tsk_mha_decode_kvcache(const void *q, const void *k, const void *v,
                                         const float *sinks, const int32_t *cu_seqlens_k,
                                         int32_t num_seqs, int64_t total_k, int32_t max_seqlen_k,
                                         int32_t Hq, int32_t Hkv, int32_t D, int32_t window,
                                         float scale, void *out, float *lse, tsk_stream_t stream);

/*
 * Paged key/value cache.  The cache is a pool of fixed-size pages: k_pages and
 * v_pages are bf16 [num_pages, page_size, Hkv, D]; block_table is an int32
 * [num_seqs, max_blocks_per_seq] device array whose row s lists the pages of
 * sequence s in order (key position x of the sequence is slot x % page_size
 * of page block_table[s][x / page_size]).  page_size is 8, 16, 32, 64 or a
 * multiple of 128 (a 128-key tile is then loaded as whole pages or one page
 * part).  cu_seqlens_k holds the prefix sums of the key counts (not pool
 * offsets); every page a sequence needs must be in [0, num_pages) and
 * ceil(Lk / page_size) <= max_blocks_per_seq, else TSK_ERR_BAD_SEQLENS (via
 * tsk_get_device_status) and nothing is computed.  Slots past Lk in a
 * sequence's last page are read (with zero weight) and must hold finite
 * values, e.g. a zero-initialised pool.  Other arguments and results as in
 * tsk_mha_prefill_kvcache / tsk_mha_decode_kvcache.
 */
TSK_API tsk_status tsk_mha_prefill_paged(const void *q, const void *k_pages, const void *v_pages,
                                        const float *sinks, const int32_t *cu_seqlens_q,
                                        const int32_t *cu_seqlens_k, const int32_t *block_table,
                                        int32_t max_blocks_per_seq, int32_t page_size,
                                        int32_t num_pages, int32_t num_seqs, int64_t total_q,
                                        int64_t total_k, int32_t Hq, int32_t Hkv, int32_t D,
                                        int32_t window, float scale, void *out, float *lse,
                                        tsk_stream_t stream);
TSK_API tsk_status tsk_mha_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                       const float *sinks, const int32_t *cu_seqlens_k,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       int32_t page_size, int32_t num_pages, int32_t num_seqs,
                                       int64_t total_k, int32_t max_seqlen_k, int32_t Hq,
                                       int32_t Hkv, int32_t D, int32_t window, float scale,
                                       void *out, float *lse, tsk_stream_t stream);

/*
 * tsk_mha_prefill_fp8 -- tsk_mha_prefill with FP8 inputs (the pages' model
 * serves FP8 weights; no formula is given for attention inputs): q8, k8, v8
 * are OCP E4M3 codes ([total_tokens, Hq, 64] and [total_tokens, Hkv, 64]
 * bytes) whose values are code * q_scale, code * k_scale, code * v_scale
 * (per-tensor fp32 scales, finite and > 0).  The result is the attention of
 * those values (scale, sinks, window, lse and out as in tsk_mha_prefill; out
 * stays bf16).  Head dimension 64 or 128.  Q K^T runs on E4M3 operands with
 * fp32 accumulation; P is rounded to bf16 for the PV product, whose V
 * operand is V's values in bf16 (exact), so outputs differ from the exact
 * attention of the dequantised inputs by up to sum_j (p_j / 256) |v_j| / l
 * per element plus bf16 rounding, as in tsk_mha_prefill.  Three launches:
 * the scheduler, a pre-pass (V as bf16; for D = 64 also the key-row norms),
 * the attention.  Extra device memory per (device, stream):
 * total_tokens * Hkv * D * 2 bytes for V in bf16.
 */
TSK_API tsk_status tsk_mha_prefill_fp8(const void *q8, const void *k8, const void *v8,
                                      float q_scale, float k_scale, float v_scale,
                                      const float *sinks, const int32_t *cu_seqlens,
                                      int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                      int32_t Hkv, int32_t D, int32_t window, float scale,
                                      void *out, float *lse, tsk_stream_t stream);

/*
 * tsk_mha_prefill_fp8_kvcache -- tsk_mha_prefill_fp8 over a contiguous key/value
 * cache: the arguments of tsk_mha_prefill_kvcache (per-sequence query and key
 * offsets cu_seqlens_q / cu_seqlens_k, Lk >= Lq, query i of a sequence at key
 * position Lk - Lq + i) with E4M3 q8 [total_q, Hq, D], k8 and v8
 * [total_k, Hkv, D] and the per-tensor scales of tsk_mha_prefill_fp8.
 * Head dimension 64 or 128; the same accuracy bound as tsk_mha_prefill_fp8;
 * total_k >= total_q (else TSK_ERR_INVALID_ARG); offsets are checked on the
 * device (TSK_ERR_BAD_SEQLENS through tsk_get_device_status).  Extra device
 * memory per (device, stream): total_k * Hkv * D * 2 bytes for V in bf16.
 */
TSK_API tsk_status tsk_mha_prefill_fp8_kvcache(const void *q8, const void *k8, const void *v8,
                                              float q_scale, float k_scale, float v_scale,
                                              const float *sinks, const int32_t *cu_seqlens_q,
                                              const int32_t *cu_seqlens_k, int32_t num_seqs,
                                              int64_t total_q, int64_t total_k, int32_t Hq,
                                              int32_t Hkv, int32_t D, int32_t window,
                                              float scale, void *out, float *lse,
                                              tsk_stream_t stream);

/* Human-readable name of a status code (static string). */
TSK_API const char *tsk_status_string(tsk_status s);

/* Text of the last CUDA error this library saw on the calling host thread
 * ("" if none): which step failed and CUDA's error name and message.  The
 * string stays valid until the next call on this thread. */
TSK_API const char *tsk_last_error(void);

/*
 * Synchronises `stream`, reads and clears the device status word of that
 * stream's workspace: TSK_OK, TSK_ERR_DEVICE_TIMEOUT (a bounded wait expired;
 * that call's outputs are incomplete) or TSK_ERR_BAD_SEQLENS.  Returns TSK_OK
 * if the stream has no workspace yet.
 */
TSK_API tsk_status tsk_get_device_status(tsk_stream_t stream);

/*
 * Timing hook.  While enabled, each tsk_mha_prefill call records CUDA events
 * on its stream around the scheduler pre-pass and around the attention
 * kernel.  tsk_profile_read synchronises on the last call's events and returns
 * the two durations in milliseconds.
 */
TSK_API tsk_status tsk_profile_enable(int enable);
TSK_API tsk_status tsk_profile_read(float *prepass_ms, float *attention_ms);

/* Number of kernels one tsk_mha_prefill call launches (0 for empty problems). */
TSK_API int32_t tsk_kernels_per_call(void);

/*
 * Benchmark helper (not part of the attention path): measures the current
 * device's throughput of the exponential instruction the softmax uses
 * (ex2.approx.f32), with 16 warps per SM running independent chains, and
 * stores it in *ex2_per_second (exponentials per second over the whole GPU).
 * Synchronises `stream`.  The benchmark states the softmax's exponentials
 * per second against this roof.
 */
TSK_API tsk_status tsk_bench_ex2_rate(double *ex2_per_second, tsk_stream_t stream);

/* Frees every cached workspace (synchronises the device first). */
TSK_API tsk_status tsk_release(void);

/*
 * Test hook for the device-side bounded waits.  `timeout_ns` is the limit of
 * every wait of later calls (0 restores the default of 2 s).  With `stall`
 * non-zero, the TMA producer of every CTA first waits on a barrier that
 * nothing signals, so each CTA runs into the limit: it records
 * TSK_ERR_DEVICE_TIMEOUT in the stream's status word, stops its other roles,
 * drains in-flight copies and MMAs (those keep a 2 s limit), frees TMEM and
 * returns without writing the outputs.  The CUDA context stays usable.
 */
TSK_API tsk_status tsk_debug_set_wait(unsigned long long timeout_ns, int stall);

/*
 * Profiling hook of builds compiled with -DTSK_TRACE (returns
 * TSK_ERR_UNSUPPORTED otherwise).  Synchronises the device and copies up to
 * n counters into `out`: out[i] = clock cycles spent at code site i, summed
 * over lane 0 of every warp that passed it, and out[64 + i] = the number of
 * passes; then clears them.  Sites 1..15 are the bounded waits (numbered as
 * the status word reports them), 20..28 softmax phases, 30 softmax total.
 * out[128 + b] (b < 1024) is the run time in ns of block b in the last
 * launch.
 */
TSK_API tsk_status tsk_debug_trace(unsigned long long *out, int32_t n);

/*
 * tsk_debug_shrink_extent -- test hook of libraries built with -DTSK_DEBUG
 * (otherwise TSK_ERR_UNSUPPORTED): later prefill calls check their q/out
 * accesses against an extent `rows` smaller than the real one (the tensor
 * maps keep the real extent, so every access it makes the checks skip is a
 * legal one).  The checks then report TSK_ERR_BOUNDS and leave the last
 * rows unwritten; 0 restores the real extent.
 */
TSK_API tsk_status tsk_debug_shrink_extent(int32_t rows);

/*
 * tsk_debug_timeline -- libraries built with -DTSK_TIMELINE only (otherwise
 * TSK_ERR_UNSUPPORTED): copies up to n entries of block 0's event record of
 * the last launch into host memory `out` and clears it.  Entry
 * [warp * 16384 + i] is event i of that warp: id in bits 56..63, SM clock in
 * bits 0..55; unused entries are 0.  Synchronises the device.
 */
TSK_API tsk_status tsk_debug_timeline(unsigned long long *out, int32_t n);

/*
 * tsk_mha_prefill_noalloc -- the same operation and arguments as
 * tsk_mha_prefill, for callers that must not allocate device memory during a
 * call: code running under a memory pool it does not own (a serving engine
 * that has reserved the whole device), latency-critical paths where an
 * allocation's implicit synchronisation is not acceptable, or processes that
 * forbid allocation after start-up.  (The pages have no counterpart of this
 * entry point; it is an addition of this library.)
 *
 * It calls no cudaMalloc/cudaFree or other allocating routine.  Its scratch
 * (status words, tile offsets, the sorted query-tile list, the key-norm
 * pre-pass's per-block maxima) is a fixed
 * ~1.8 MB array in the library's device memory, which every GPU that loads
 * the library holds until the process exits.  Limits: num_seqs <= 16384 and
 * total_tokens/128 + num_seqs + 1 <= 49152; larger problems are rejected with
 * TSK_ERR_UNSUPPORTED (tsk_last_error says which limit) before anything is
 * enqueued.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array: calls whose
 * work overlaps on the GPU (different streams, or host threads issuing
 * concurrently) race and must be serialised by the caller.  Each call clears
 * the status words it needs; device-side errors it detects (inconsistent
 * cu_seqlens, an expired bounded wait) leave the outputs unwritten and are
 * reported by tsk_noalloc_status (below), not by tsk_get_device_status.
 */
TSK_API tsk_status tsk_mha_prefill_noalloc(const void *q, const void *k, const void *v,
                                           const float *sinks, const int32_t *cu_seqlens,
                                           int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                           int32_t Hkv, int32_t D, int32_t window, float scale,
                                           void *out, float *lse, tsk_stream_t stream);

/*
 * tsk_noalloc_status -- the device-side status of the most recent
 * tsk_mha_prefill_noalloc call on the current device: TSK_OK, or
 * TSK_ERR_BAD_SEQLENS (-8, cu_seqlens inconsistent with num_seqs or
 * total_tokens; nothing was written) or TSK_ERR_DEVICE_TIMEOUT (-7, a bounded
 * wait expired).  Like tsk_get_device_status it synchronises `stream` (the
 * stream that call was made on) and clears a non-zero status after reading
 * it; it allocates nothing (two small synchronous copies of the fixed
 * array's status words).  Returns TSK_OK if no allocation-free call has been
 * made on this device.  (No counterpart in the pages: a companion of the
 * allocation-free entry point.)
 */
TSK_API tsk_status tsk_noalloc_status(tsk_stream_t stream);

/*
 * tsk_mha_prefill_host -- tsk_mha_prefill with every buffer in host memory:
 * q, k, v, sinks, cu_seqlens, out and lse are host pointers (same shapes,
 * types and meaning as for tsk_mha_prefill; cu_seqlens is read on the host,
 * so all of its checks happen before anything is enqueued and an invalid
 * array returns TSK_ERR_INVALID_ARG; so does `out` overlapping q, k or v).
 * The pages define the operation on
 * device tensors only; this entry point is an addition of this library for
 * callers whose inputs live in host memory.
 *
 * The packed token stream is cut into about eight chunks of consecutive
 * tokens (at least 2048 each; a chunk ends at a sequence end or at a
 * multiple of 128 rows from the start of the sequence it cuts, so every
 * query tile is the one tsk_mha_prefill forms).  Chunk c's attention is a prefill over a
 * key/value cache: its queries are the chunk's rows, its keys each touched
 * sequence's rows from the sequence start to the chunk end, all already on
 * the device.  Copies in (one stream), attention (two streams) and copies
 * out (one stream) then overlap across chunks; these streams belong to the
 * library, one set per (device, caller stream).  Results are bit for bit
 * those of tsk_mha_prefill (the same query tiles visit the same key tiles).
 *
 * Asynchronous: the call enqueues work and returns; `stream` continues once
 * every output byte has reached host memory, so the host buffers must stay
 * valid (and out/lse unread) until `stream` has passed that point (for
 * example cudaStreamSynchronize(stream)).  The work starts after everything
 * enqueued earlier on `stream`.  Copies overlap only with page-locked host
 * buffers (cudaHostAlloc / cudaHostRegister); with pageable memory the call
 * still works but the copies serialise the host.  Device memory: a
 * grow-only buffer of about (2*Hq + 2*Hkv)*D*2 + 4*Hq bytes per token plus the
 * workspaces of the library's streams, held per (device, caller stream)
 * until tsk_release.  Device-side errors of the chunks' kernels are reported
 * by tsk_get_device_status(stream).  Not capturable in a CUDA graph (it
 * waits on events recorded on its own streams).  Calls on one caller stream
 * are serialised by a library lock while they enqueue.
 */
TSK_API tsk_status tsk_mha_prefill_host(const void *q, const void *k, const void *v,
                                        const float *sinks, const int32_t *cu_seqlens,
                                        int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                        int32_t Hkv, int32_t D, int32_t window, float scale,
                                        void *out, float *lse, tsk_stream_t stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
TSK_API int32_t tsk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TSK_MHA_H_ */
