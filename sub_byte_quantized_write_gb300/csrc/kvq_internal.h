// kvq_internal.h -- kernel parameter blocks and launchers behind the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_common.cuh"

namespace kvq {

struct WriteParams {
  uint8_t* k_pages;
  uint8_t* v_pages;
  int num_blocks, num_kv_heads, block_size, head_dim, mode;
  int stego;                  // INT4 rows whose pad is an fp32 scale carrying the zero point
  const int8_t* signs;
  float* ch_amax;
  int32_t* ch_ready;
  const int32_t* table;
  int headwise, max_blocks, batch;
  const int32_t* seq_lens;
  const int32_t* cu_new;
  const void* k;
  const void* v;
  int dtype, num_tokens;
  int32_t* dev_error;
  // gather: dense outputs [num_tokens][Hkv][D] of out_dtype (DT_F32 / DT_BF16)
  void* out_k;
  void* out_v;
  int out_dtype;
  // gather with the current chunk in full precision (NULL chunk_k: plain
  // gather): sequence b's last cu_chunk[b+1] - cu_chunk[b] positions come
  // from rows cu_chunk[b] .. of chunk_k / chunk_v [rows][Hkv][D] of chunk_dtype
  const void* chunk_k;
  const void* chunk_v;
  const int32_t* cu_chunk;
  int chunk_dtype;
};

// Shared by the decode and prefill kernels.
struct AttnParams {
  const uint8_t* k_pages;
  const uint8_t* v_pages;
  int num_blocks, num_kv_heads, block_size, head_dim, mode;
  int stego;                  // INT4 rows whose pad is an fp32 scale carrying the zero point
  const int8_t* signs;        // NULL = RHT off
  const float* ch_amax;       // INT8: [2][Hkv][D]
  const int32_t* table;
  int headwise, max_blocks, batch;
  const int32_t* seq_lens;
  const int32_t* window;      // [Hkv] or NULL
  int sink;
  const void* q;
  int dtype, num_q_heads, group;
  float softmax_scale;
  float* out;
  int32_t* dev_error;
  // prefill
  const int32_t* cu_q;
  int total_q, max_q_per_seq;
  // dense prefill: sequence b's key j is row cu_kv[b] + j of k_pages / v_pages;
  // kv_map[0 | 1] view K / V as [rows][Hkv][D] bf16 in boxes of one 64-dim half
  // of 64 rows of one head, 128-byte swizzled.
  // decode (token-head modes): kv_map[0 | 1] view the K / V pool as 2-D tensors
  // of page chunks (decode_chunk_rows), one chunk per box row.
  const int32_t* cu_kv;
  int chunk_rows_total;   // decode: rows of the kv_map tensors (the kernel copies no row at or past it)
  // decode with the step's write (kvq_write_decode_attn): the preparation
  // kernel quantises and stores the new K / V rows [num_new][Hkv][D] of
  // new_dtype; sequence b's are rows cu_new[b] .. cu_new[b+1] - 1 (NULL new_k:
  // no write)
  const void* new_k;
  const void* new_v;
  int new_dtype, num_new;
  const int32_t* cu_new;
  CUtensorMap kv_map[2];  // 128-byte aligned by its own declaration
};

// Decode workspace (caller-owned scratch), carved by decode_ws_layout.
struct DecodeWs {
  int* tile_start;     // [B*Hkv + 1] first stream tile of each pair (written by the stream kernel's CTA 0)
  uint32_t* qfrag;     // [B*Hkv][32 lanes][NT * D/16 * 2] query B-operand images
  float4* qbg;         // [B*Hkv][4*NT] per-head logit constants (beta, gamma, key fold, 0)
  float2* part_ml;     // [n_partials][G] (running max in log2 units, sum of weights)
  float* part_o;       // [n_partials][G][D] unnormalised partial outputs
  int n_partials;      // stream workers + B*Hkv
  int nwall;           // stream warps launched
  int fixed_workers;   // > 0: use exactly this many workers
};

// Split-KV geometry shared by the host API and the kernels.
constexpr int DECODE_KEYS_PER_TILE = 32;
constexpr int DECODE_WARPS = 4;
constexpr int DECODE_MIN_TILES_PER_WARP = 8;

// How the stream kernel of one configuration is launched: CTAs per SM and
// warps per CTA.
struct DecodeShape {
  int ctas_per_sm, warps_per_cta;
};

struct DecodeLayout {
  size_t off_tile_start, off_qfrag, off_qbg, off_part_ml, off_part_o, total;
  int grid, nwall, n_partials;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout for one decode call; sm_count * ctas_per_sm CTAs of
// warps_per_cta warps.
inline DecodeLayout decode_ws_layout(int batch, int num_kv_heads, int group, int head_dim, int sm_count,
                                     DecodeShape shape) {
  DecodeLayout L;
  const int BH = batch * num_kv_heads;
  const int NT = group <= 4 ? 1 : 2;
  L.grid = sm_count * shape.ctas_per_sm;
  L.nwall = L.grid * shape.warps_per_cta;
  L.n_partials = L.nwall + BH;
  size_t o = 0;
  L.off_tile_start = o; o = align256(o + (size_t)(BH + 1) * 4);
  L.off_qfrag = o;      o = align256(o + (size_t)BH * 32 * NT * (head_dim / 16) * 2 * 4);
  L.off_qbg = o;        o = align256(o + (size_t)BH * 4 * NT * 16);
  L.off_part_ml = o;    o = align256(o + (size_t)L.n_partials * group * 8);
  L.off_part_o = o;     o = align256(o + (size_t)L.n_partials * group * head_dim * 4);
  L.total = o;
  return L;
}

DecodeShape decode_shape(int mode, int head_dim, int group);
// Key rows per page chunk that the decode's tensor copies move (16 or 8), or 0
// when the configuration copies its pages with cp.async (INT8 per channel).
// The caller's tensor maps kv_map[0 | 1] view the K / V pool as 2-D tensors
// of such chunks: row (block * Hkv + head) * (block_size / rows) + chunk.
int decode_chunk_rows(int mode, int head_dim, int group);

cudaError_t launch_write(const WriteParams& P, cudaStream_t stream);
cudaError_t launch_gather(const WriteParams& P, cudaStream_t stream);
cudaError_t launch_decode(const AttnParams& P, const DecodeWs& ws, int grid, cudaStream_t stream);
cudaError_t launch_prefill(const AttnParams& P, cudaStream_t stream);

// The prefill grid: x = query tiles of the longest chunk (PREFILL_ROWS_PER_CTA
// (query, q head) rows per CTA), y = kv heads, z = sequences.  Computed in 64
// bits so that no max_q_per_seq can wrap it; the host checks it against the
// launch limits before any launch.
constexpr int PREFILL_ROWS_PER_CTA = 128;
inline long long prefill_grid_x(int max_q_per_seq, int group) {
  const long long qb = PREFILL_ROWS_PER_CTA / group;
  return ((long long)max_q_per_seq + qb - 1) / qb;
}

}  // namespace kvq
