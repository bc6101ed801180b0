/*
 * kvq.h -- C ABI of libkvq: a paged KV cache held in dynamic low-bit form on
 * one GB300 (sm_103a), with the write path that fills it and the decode and
 * chunked-prefill attention that read it.
 *
 * Sources the operations follow (web pages, cited by title and section):
 *   [vLLM-INT4]  vLLM PR #40835 review summary, "INT4 per-token-head KV cache
 *                for the Triton backend": sections 功能与动机 (motivation: RHT
 *                plus asymmetric scale/zero point), 实现拆解 (implementation
 *                breakdown, items 2-4), 关键源码片段 (key source snippets:
 *                INT4_CONFIG range [-8, 7]; get_kv_cache_shape row size
 *                head_size//2 + scale_pad, scale_pad = 4), 风险与影响 (causal only).
 *   [FD-INT2]    FastDeploy PR #5173 "[Feature] support dynamic int2
 *                quantization cache kv": Motivation, Modifications, Usage.
 *   [FD-HEADWISE] FastDeploy PR #7718 "Optimize AppendAttention for discrete
 *                head-wise block_idx": Motivation (block_tables_headwise
 *                layout), Modifications "PR2-only delta" table (-1 sentinel,
 *                sink_size), Correctness gates.
 *   [ASCEND-INT8] vllm-ascend-quantized-kv-cache 0.2.0rc2 METADATA, "Ascend
 *                INT8 KV Cache Plugin", section 运行机制 (dynamic symmetric
 *                per-channel INT8, scales taken along tokens on the first K/V
 *                a layer receives; prefill gathers and dequantises pages).
 *   [FD-UINT8]   FastDeploy PR #7757 "fix cache_manager_v1 allocating kv cache
 *                with wrong dtype when kv_cache_quant_type is set", section 修复
 *                (every quantised cache is stored as 1-byte uint8).
 *
 * Conventions shared by every call
 *   - Every pointer is a DEVICE pointer on the current CUDA device unless the
 *     comment says "host".  The library allocates nothing at call time; its
 *     only state is a per-device record of kernel attributes it has set and,
 *     for kvq_decode_attn_noalloc, one static scratch array per device.
 *   - Calls enqueue work on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and never synchronise.  Outputs are valid
 *     once the stream reaches the work.
 *   - Host-detectable errors (NULL pointers, unsupported shapes, misaligned
 *     pointers, a too-small workspace, Hq % Hkv != 0) return a status before
 *     any launch and leave all device memory untouched.  A failed launch
 *     returns KVQ_ERR_CUDA; kvq_last_error() then holds the CUDA message.
 *   - Device-detectable contract violations (a block id >= num_blocks, a
 *     position beyond the table row, more new tokens than seq_len) OR a bit
 *     into *dev_error (KVQ_DEVERR_* below, nullable), and the offending row
 *     is skipped: it is never read nor written.  Read *dev_error after the
 *     stream synchronises.
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_ABI_VERSION 1

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, both/neither table, Hq % Hkv != 0 */
  KVQ_ERR_UNSUPPORTED = 2, /* head_dim, block_size, mode, dtype or GQA group not built */
  KVQ_ERR_CUDA = 3,        /* a kernel launch failed; see kvq_last_error() */
  KVQ_ERR_WORKSPACE = 4    /* decode workspace NULL or smaller than required */
} kvq_status;

/* Quantisation modes.
 * INT4 / INT2: per (token, kv_head) row: optional RHT, then asymmetric codes
 *   u in [0, 2^b - 1] with an fp16 scale s and fp16 zero point m (the value of
 *   code 0); the signed view q = u - 2^(b-1) covers [-8, 7] for INT4
 *   ([vLLM-INT4] 关键源码片段, INT4_CONFIG) and [-2, 1] for INT2 ([FD-INT2]).
 * INT8: dynamic symmetric per-channel codes in [-127, 127] with one fp32
 *   scale per (K|V, kv_head, channel) ([ASCEND-INT8] 运行机制); no RHT.
 * INT4_STEGO: the INT4 row layout, with the 4-byte pad an fp32 scale whose
 *   low 4 mantissa bits carry an integer zero point ([vLLM-INT4] 评论区精华,
 *   zero-point steganography).  Per row (after the optional RHT): the grid
 *   (u - zp) * s holds 0, so it spans lo = min(min, 0) .. hi = max(max, 0);
 *   s = (hi - lo) / 15 with its low 4 mantissa bits cleared, zp =
 *   clamp(rne(-lo / s), 0, 15), u = clamp(rne(x / s) + zp, 0, 15), pad =
 *   bits(s) | zp, value (u - zp) * s.
 * INT8_TOKEN_HEAD / FP8_TOKEN_HEAD: the per-token-head INT8 / FP8 modes the
 *   INT4 mode was built on ([vLLM-INT4] 功能与动机, 关联脉络): per row (after
 *   the optional RHT) one symmetric fp32 scale s = amax / 127 (INT8 codes
 *   clamp(rne(x / s), -127, 127)) or s = amax / 448 (FP8 E4M3 codes: x / s
 *   rounded to nearest even, saturating at 448); s = 0 gives zero codes;
 *   value code * s. */
typedef enum {
  KVQ_INT4_TOKEN_HEAD = 0,
  KVQ_INT2_TOKEN_HEAD = 1,
  KVQ_INT8_CHANNEL = 2,
  KVQ_INT4_STEGO = 3,
  KVQ_INT8_TOKEN_HEAD = 4,
  KVQ_FP8_TOKEN_HEAD = 5
} kvq_mode;

/* Element type of q / k / v inputs. */
typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1 } kvq_dtype;

/* Bits OR-ed into *dev_error by the kernels. */
#define KVQ_DEVERR_BLOCK_RANGE 1 /* table entry >= num_blocks: row skipped */
#define KVQ_DEVERR_TABLE_RANGE 2 /* position / block_size >= max_blocks: row skipped */
#define KVQ_DEVERR_SEQ_LEN 4     /* negative seq_len, or more new tokens than seq_len */
#define KVQ_DEVERR_TIMEOUT 8     /* a bounded wait for an asynchronous copy gave up (never expected) */
#define KVQ_DEVERR_BOUNDS 16     /* debug library only (libkvq_debug.so, built with -DKVQ_BOUNDS_CHECK):
                                     an index computed on the device fell outside its buffer; the access
                                     was skipped (never expected) */

/* One layer's paged cache (caller-allocated; store it as torch.uint8, cf.
 * [FD-UINT8] 修复).
 *
 * Page layout ([vLLM-INT4] 关键源码片段 get_kv_cache_shape gives the row;
 * K and V are kept in separate pools so that one (block, kv_head) page is
 * contiguous):
 *     k_pages, v_pages : uint8 [num_blocks][num_kv_heads][block_size][row_bytes]
 *     row_bytes        : kvq_row_bytes(mode, head_dim)
 *       INT4: head_dim/2 data bytes (element 2i in the low nibble of byte i),
 *             then 4 pad bytes = fp16 scale s, fp16 zero point m (little endian)
 *       INT2: head_dim/4 data bytes (element 4i+j in bits 2j..2j+1 of byte i),
 *             then the same 4 pad bytes
 *       INT8: head_dim bytes of two's-complement codes (no pad)
 *       INT8_TOKEN_HEAD / FP8_TOKEN_HEAD: head_dim code bytes (two's
 *             complement / E4M3), then the fp32 scale (little endian)
 *   Both pools must be 16-byte aligned.
 *
 * rht_signs: int8 [head_dim] of +1/-1 (device).  Non-NULL turns the random
 *   Hadamard transform on for INT4/INT2: y = H (signs * x), H the unnormalised
 *   Sylvester Walsh-Hadamard matrix ([vLLM-INT4] 功能与动机, 实现拆解 2); the
 *   same for INT4_STEGO and the INT8 / FP8 token-head modes.  One vector per
 *   layer, shared by K, V and every head.  Must be NULL for INT8_CHANNEL.
 *
 * ch_amax / ch_amax_ready (INT8 only, else NULL):
 *   ch_amax: fp32 [2][num_kv_heads][head_dim] (index 0 = K, 1 = V).  The scale
 *   of a channel is ch_amax / 127 (IEEE fp32 division).  While
 *   *ch_amax_ready == 0 the buffer must hold zeros: the next kvq_write takes
 *   the per-channel max |x| over ALL tokens it is given (also tokens whose page
 *   is -1), stores it here and sets *ch_amax_ready = 1 ([ASCEND-INT8] 运行机制:
 *   scales come from the first K/V a layer receives).  Later writes reuse it
 *   and saturate at +-127. */
typedef struct {
  uint8_t* k_pages;
  uint8_t* v_pages;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size; /* 16, 32 or 64 */
  int32_t head_dim;   /* 64 or 128 */
  int32_t mode;       /* kvq_mode */
  const int8_t* rht_signs;
  float* ch_amax;
  int32_t* ch_amax_ready;
} kvq_cache;

/* Paging state of one step.
 * Exactly one of the two tables is non-NULL ([FD-HEADWISE] Motivation):
 *   block_tables          int32 [batch][max_blocks]: row b serves every head
 *   block_tables_headwise int32 [batch * num_kv_heads][max_blocks]: row
 *                         b * num_kv_heads + h serves kv head h
 *   Token position p of a row lives in page table[row][p / block_size], slot
 *   p % block_size.  An entry < 0 (-1 sentinel) marks an evicted block: it is
 *   never dereferenced, writes to it are dropped and its keys contribute
 *   nothing ([FD-HEADWISE] PR2-only delta, Correctness gates).
 * seq_lens int32 [batch]: tokens in the cache for each sequence AFTER this
 *   step's write.  Decode queries sit at position seq_lens[b] - 1.
 * window_per_kv_head int32 [num_kv_heads] or NULL (= all heads full):
 *   0 = full attention; W > 0 = sliding window: a query at p sees key j iff
 *   j <= p and (j < sink_size or j > p - W) ([FD-HEADWISE] sink_size).
 */
typedef struct {
  const int32_t* block_tables;
  const int32_t* block_tables_headwise;
  int32_t max_blocks;
  int32_t batch;
  const int32_t* seq_lens;
  const int32_t* window_per_kv_head;
  int32_t sink_size;
} kvq_paging;

/* Bytes of one cache row for (mode, head_dim); 0 if unsupported. */
int32_t kvq_row_bytes(int32_t mode, int32_t head_dim);

/* kvq_write -- quantise new K/V tokens and scatter them into the pages.
 * ([vLLM-INT4] 实现拆解 2 and 4: rotate, per-token-head scale and zero point,
 * pack, scatter through the block table; [FD-INT2] Modifications: cache-write
 * kernels for the 2-bit cache; [ASCEND-INT8] 运行机制 for INT8.)
 *
 * k, v          : [num_tokens][num_kv_heads][head_dim] of `dtype` (row-major,
 *                 16-byte aligned).
 * cu_new_tokens : int32 [batch + 1], cu[0] = 0, non-decreasing, cu[batch] =
 *                 num_tokens.  Sequence b owns tokens cu[b] .. cu[b+1]-1, at
 *                 positions seq_lens[b] - n_b .. seq_lens[b] - 1 (n_b = its count).
 * Per row the codes are bit-exactly defined: fp32 sign flip and butterfly in
 * stage order 1, 2, 4, ..., head_dim/2; min/max canonicalised with +0.0f;
 * s = (max - min) / (2^b - 1) (IEEE); s, m rounded to fp16 (round to nearest
 * even, saturating at +-65504); u = clamp(rne((y - m) / s), 0, 2^b - 1), u = 0
 * when the fp16 scale is 0.  INT8: q = clamp(rne(x / (amax / 127)), -127, 127),
 * 0 when the scale is 0.  INT8 / FP8 token-head: amax = max |y| of the row,
 * s = amax / 127 or amax / 448 (IEEE), each code from y / s (IEEE division;
 * E4M3 by round to nearest even with saturation), all 0 when s is 0.
 * num_tokens == 0 is a no-op returning KVQ_OK. */
kvq_status kvq_write(const kvq_cache* cache, const kvq_paging* paging,
                     const void* k, const void* v, int32_t dtype,
                     const int32_t* cu_new_tokens, int32_t num_tokens,
                     int32_t* dev_error, void* stream);

/* kvq_gather -- read rows of given positions back from the pages as dense,
 * dequantised values in the input domain (inverse RHT applied): the gather
 * and dequantise step a prefill can run before dense attention ([FD-INT2]
 * review: the custom op dynamic_quant_get_kv_from_cache; [ASCEND-INT8]
 * 运行机制: chunked prefill gathers and dequantises the paged cache).
 *
 * cu_tokens    : int32 [batch + 1], the position map of kvq_write: sequence b's
 *                tokens cu[b] .. cu[b+1]-1 are its positions seq_lens[b] - n_b
 *                .. seq_lens[b] - 1 (n_b = seq_lens[b] gathers the whole sequence).
 * k_out, v_out : [num_tokens][num_kv_heads][head_dim] of out_dtype (KVQ_F32 or
 *                KVQ_BF16, round to nearest even), caller-allocated, 16-byte aligned.
 * Per row (fp32): INT4 / INT2 y = u * s + m; zero-point-in-scale INT4 (u -
 * zp) * s; INT8 channel q * (amax / 127); INT8 / FP8 token-head code * s;
 * then, with RHT signs, x = signs * (H y) / D by the same butterfly.  A row
 * whose table entry is -1 is written as zeros; rows that cannot be located
 * are written as zeros and set *dev_error bits as in kvq_write.  Window
 * fields of `paging` are ignored.  num_tokens == 0 is a no-op. */
kvq_status kvq_gather(const kvq_cache* cache, const kvq_paging* paging, const int32_t* cu_tokens,
                      int32_t num_tokens, void* k_out, void* v_out, int32_t out_dtype, int32_t* dev_error,
                      void* stream);

/* kvq_gather_chunk -- kvq_gather where the current chunk comes in full
 * precision: the gather for a prefill that attends to the chunk's own K / V
 * as given rather than as stored.
 * k_chunk, v_chunk : [rows][num_kv_heads][head_dim] of chunk_dtype (KVQ_F32 or
 *                    KVQ_BF16), 16-byte aligned: the rows kvq_write was given.
 * cu_chunk         : int32 [batch + 1]: sequence b's chunk is rows cu_chunk[b] ..
 *                    cu_chunk[b+1]-1, its positions the last m_b = cu_chunk[b+1] -
 *                    cu_chunk[b] of the sequence (kvq_write's cu_new_tokens map).
 * Positions before the chunk are gathered from the cache as kvq_gather does;
 * chunk positions are copied (fp32 or bf16 out) without the RHT or any
 * quantisation.  m_b < 0 or m_b > seq_lens[b] sets KVQ_DEVERR_SEQ_LEN and gives
 * zero rows.  NULL k_chunk (with v_chunk and cu_chunk NULL) is kvq_gather. */
kvq_status kvq_gather_chunk(const kvq_cache* cache, const kvq_paging* paging, const int32_t* cu_tokens,
                            int32_t num_tokens, const void* k_chunk, const void* v_chunk, int32_t chunk_dtype,
                            const int32_t* cu_chunk, void* k_out, void* v_out, int32_t out_dtype,
                            int32_t* dev_error, void* stream);

/* Workspace needed by kvq_decode_attn for `num_splits` (0 = the library's
 * choice).  Writes the byte count to *bytes (host) and the split count that
 * kvq_decode_attn will use to *splits_used (host, nullable). */
kvq_status kvq_decode_workspace_size(const kvq_cache* cache, const kvq_paging* paging,
                                     int32_t num_q_heads, int32_t num_splits,
                                     size_t* bytes, int32_t* splits_used);

/* kvq_decode_attn -- one decode query per sequence over the paged cache.
 * ([vLLM-INT4] 实现拆解 2: unpack, dequantise, attention; [FD-HEADWISE]
 * per-head row walk with -1 sentinel; [ASCEND-INT8] 运行机制: decode
 * dequantises inside the attention kernel.)
 *
 * q   : [batch][num_q_heads][head_dim] of `dtype`; q head hq reads kv head
 *       hq / (num_q_heads / num_kv_heads).  GQA group size 1..8.
 * out : fp32 [batch][num_q_heads][head_dim] = sum_j P_j v_j with
 *       P = softmax_j(softmax_scale * q . k_j) over the visible keys, where k_j
 *       and v_j are the dequantised rows mapped back through the inverse RHT.
 *       A query with no visible key gets zeros.
 * workspace : device scratch of >= kvq_decode_workspace_size() bytes, 256-byte
 *       aligned, owned by the caller; its contents on entry do not matter.
 * The work is split along the keys (split-KV); a second kernel merges the
 * splits and applies the inverse RHT. */
kvq_status kvq_decode_attn(const kvq_cache* cache, const kvq_paging* paging,
                           const void* q, int32_t dtype, int32_t num_q_heads,
                           float softmax_scale, float* out,
                           void* workspace, size_t workspace_bytes, int32_t num_splits,
                           int32_t* dev_error, void* stream);

/* kvq_write_decode_attn -- one decode step in one call: kvq_write of the
 * step's new tokens, then kvq_decode_attn, with the write done by the
 * decode's query-preparation kernel instead of a launch of its own.
 * ([vLLM-INT4] 关键源码片段 get_kv_cache_shape: the row the write produces
 * and the decode reads; 实现拆解 2: the write and read kernels.)
 *
 * k, v, kv_dtype, cu_new_tokens, num_tokens : as kvq_write (new rows
 *       [num_tokens][num_kv_heads][head_dim]; sequence b's new tokens are at
 *       positions seq_lens[b] - n_b .. seq_lens[b] - 1).
 * q, q_dtype, num_q_heads, softmax_scale, out, workspace, workspace_bytes,
 * num_splits : as kvq_decode_attn.
 * The pages and error bits are exactly those of kvq_write followed by
 * kvq_decode_attn: the rows come from the same row arithmetic.  Meant for
 * decode steps (a few new tokens per sequence: each (sequence, kv head)
 * writes its rows with one CTA).  KVQ_INT8_CHANNEL is not supported (its
 * first write takes the channel maxima over every token first):
 * KVQ_ERR_UNSUPPORTED. */
kvq_status kvq_write_decode_attn(const kvq_cache* cache, const kvq_paging* paging,
                                 const void* k, const void* v, int32_t kv_dtype,
                                 const int32_t* cu_new_tokens, int32_t num_tokens,
                                 const void* q, int32_t q_dtype, int32_t num_q_heads,
                                 float softmax_scale, float* out,
                                 void* workspace, size_t workspace_bytes, int32_t num_splits,
                                 int32_t* dev_error, void* stream);

/* kvq_prefill_attn -- causal chunked-prefill attention of a chunk of queries
 * against everything in the cache, the chunk itself included (write the chunk
 * with kvq_write first).  ([FD-INT2] Usage: chunked prefill; [vLLM-INT4]
 * 风险与影响: causal attention only; [ASCEND-INT8] 运行机制: chunked prefill
 * reads the paged cache.)
 *
 * q    : [total_q][num_q_heads][head_dim] of `dtype`.
 * cu_q : int32 [batch + 1]; sequence b's queries are rows cu_q[b] .. cu_q[b+1]-1
 *        at positions seq_lens[b] - n_b + i.
 * max_q_per_seq : host upper bound on n_b (sizes the grid).
 * out  : fp32 [total_q][num_q_heads][head_dim]. */
kvq_status kvq_prefill_attn(const kvq_cache* cache, const kvq_paging* paging,
                            const void* q, int32_t dtype, int32_t num_q_heads,
                            const int32_t* cu_q, int32_t total_q, int32_t max_q_per_seq,
                            float softmax_scale, float* out,
                            int32_t* dev_error, void* stream);

/* kvq_decode_attn_noalloc -- kvq_decode_attn for callers that cannot
 * allocate device memory (no counterpart on the pages; an addition of this
 * library).  Some callers must not or cannot call cudaMalloc at call time:
 * a plugin inside a host framework that owns all device memory and hands out
 * no scratch, or a latency-critical path where an allocation's implicit
 * synchronisation is unacceptable.  This entry point takes the same arguments
 * as kvq_decode_attn minus the workspace and allocates nothing: the split-KV
 * partials live in one static device array of KVQ_NOALLOC_SCRATCH_BYTES that
 * the library reserves on every GPU it is loaded on, until the process exits.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents.  Nothing in it needs to start at zero (the kernels
 *     write every partial before reading it), but calls whose work overlaps
 *     on the GPU (different streams, or different host threads) race on it:
 *     serialise them.
 *   - Returns KVQ_ERR_WORKSPACE, with a message, when the call would need more
 *     scratch than KVQ_NOALLOC_SCRATCH_BYTES (see kvq_decode_workspace_size). */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const kvq_paging* paging,
                                   const void* q, int32_t dtype, int32_t num_q_heads,
                                   float softmax_scale, float* out, int32_t num_splits,
                                   int32_t* dev_error, void* stream);

/* Human-readable name of a status. */
const char* kvq_status_string(int32_t status);

/* Message of the last KVQ_ERR_* returned on this host thread ("" if none). */
const char* kvq_last_error(void);

/* KVQ_ABI_VERSION of the loaded library. */
int32_t kvq_abi_version(void);

/* kvq_prefill_dense_attn -- causal chunked-prefill attention over DENSE bf16
 * K / V rows, the prefill that follows a gather ([FD-INT2] review: the
 * custom op dynamic_quant_get_kv_from_cache; [ASCEND-INT8] 运行机制: chunked
 * prefill gathers and dequantises the paged cache, then attends).  The same
 * tcgen05 kernel as kvq_prefill_attn with bf16 rows in place of codes: no
 * scale, no zero point, no RHT (the rows are in the input domain, as
 * kvq_gather writes them).
 *
 * k, v          : bf16 [rows][num_kv_heads][head_dim], 16-byte aligned; sequence
 *                 b's key j is row cu_kv[b] + j (kvq_gather with n_b = seq_lens[b]
 *                 writes exactly this layout).  The kernel converts the rows to
 *                 fp16 (round to nearest): exact for 0 and 2^-17 <= |x| <= 65504;
 *                 smaller magnitudes round to a multiple of 2^-24, larger ones
 *                 become 65504 or infinity, so keep the rows inside that range.
 * cu_kv         : int32 [batch + 1] (device); cu_kv[b + 1] - cu_kv[b] >= seq_lens[b],
 *                 else the sequence is skipped and KVQ_DEVERR_SEQ_LEN set.
 * num_kv_rows   : rows of k and v (host); cu_kv[batch] <= num_kv_rows.  The rows
 *                 move by tensor copies (one 64-row box of a head per tile).
 * paging        : seq_lens, batch, window_per_kv_head and sink_size as for the
 *                 paged calls; both block tables must be NULL.
 * q, dtype, num_q_heads, cu_q, total_q, max_q_per_seq, softmax_scale, out,
 * dev_error     : as in kvq_prefill_attn (queries at positions seq_lens[b] - n_b
 *                 + i, causal, window + sink per kv head). */
kvq_status kvq_prefill_dense_attn(const void* k, const void* v, const int32_t* cu_kv, int32_t num_kv_rows,
                                  int32_t num_kv_heads, int32_t head_dim, const kvq_paging* paging, const void* q,
                                  int32_t dtype, int32_t num_q_heads, const int32_t* cu_q, int32_t total_q,
                                  int32_t max_q_per_seq, float softmax_scale, float* out, int32_t* dev_error,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
