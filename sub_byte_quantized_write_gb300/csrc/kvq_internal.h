// kvq_internal.h -- kernel parameter blocks and launchers behind the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_common.cuh"

namespace kvq {

struct WriteParams {
  uint8_t* k_pages;
  uint8_t* v_pages;
  int num_blocks, num_kv_heads, block_size, head_dim, mode;
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
};

// Shared by the decode and prefill kernels.
struct AttnParams {
  const uint8_t* k_pages;
  const uint8_t* v_pages;
  int num_blocks, num_kv_heads, block_size, head_dim, mode;
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
  // decode
  int num_splits, tiles_per_split;  // tiles of 32 keys
  float* part_o;                    // [B][Hq][S][D]
  float2* part_ml;                  // [B][Hq][S]  (max in log2 units, sum)
  // prefill
  const int32_t* cu_q;
  int total_q, max_q_per_seq;
};

cudaError_t launch_write(const WriteParams& P, cudaStream_t stream);
cudaError_t launch_decode(const AttnParams& P, cudaStream_t stream);
cudaError_t launch_prefill(const AttnParams& P, cudaStream_t stream);

// Split-KV geometry shared by the host API and the kernels.
constexpr int DECODE_KEYS_PER_TILE = 32;
constexpr int DECODE_WARPS = 4;

}  // namespace kvq
