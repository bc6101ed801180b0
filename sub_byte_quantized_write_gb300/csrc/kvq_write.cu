// kvq_write.cu -- write path: rotate, quantise, pack and scatter new K/V rows;
// and its inverse, gathering rows back from the pages as dense values.
//
// INT4 / INT2 per (token, kv_head): vLLM PR #40835 review summary ("INT4
// per-token-head KV cache for the Triton backend"), 实现拆解 item 2 (the write
// kernel rotates each row with a random Hadamard transform, takes a per-token-
// head scale and zero point, rounds and packs nibbles) and 关键源码片段
// (row = head_size/2 data bytes + a 4-byte scale pad); FastDeploy PR #5173
// "support dynamic int2 quantization cache kv", Modifications (cache-write
// kernels of the dynamic 2-bit cache).
// INT8 per channel: vllm-ascend-quantized-kv-cache METADATA ("Ascend INT8 KV
// Cache Plugin"), 运行机制 (symmetric per-channel scales along tokens, from the
// first K/V a layer receives, separately for K and V).
// INT8 / FP8 per (token, kv_head): the same vLLM page, 功能与动机 and 关联脉络
// (the per-token-head INT8 / FP8 modes the INT4 mode builds on): one
// symmetric fp32 scale per row, stored after the D code bytes.
// Scatter through a uniform or head-wise block table with -1 sentinels:
// FastDeploy PR #7718 "Optimize AppendAttention for discrete head-wise
// block_idx", Motivation and PR2-only delta table.
//
// One warp per (token, kv_head, K|V) row; each lane holds D/32 consecutive
// elements.  The row's arithmetic is a fixed sequence of IEEE fp32 operations
// (sign flip, butterfly in stage order, exact min/max, one division, fp16 RNE,
// one subtract and one divide per element, round-half-even), so the packed
// bytes are identical to any other evaluation in the same order.

#include <algorithm>

#include "kvq_internal.h"
#include "kvq_row.cuh"

namespace kvq {

// Destination row of (token t, kv head h) for every lane of the warp;
// nullptr when the row is dropped (-1 sentinel) or invalid (error bit set).
// The owning sequence is found with one round of parallel loads: lane j
// holds cu[j + 32 i] and ballots whether it is <= t (cu is non-decreasing,
// so the ballot's population count locates the sequence).
__device__ __forceinline__ uint8_t* dest_row(const WriteParams& P, uint8_t* pages, int t, int h, int lane) {
  int b = -1, cu_b = 0, cu_b1 = 0, L = 0;
  int prev_c = 0, prev_l = 0;  // cu and seq_lens at the previous chunk's last lane
  for (int base = 0; base <= P.batch; base += 32) {
    const int j = base + lane;
    const int cj = j <= P.batch ? __ldg(P.cu_new + j) : 0x7FFFFFFF;
    const int lj = j < P.batch ? __ldg(P.seq_lens + j) : 0;
    const int cnt = __popc(__ballot_sync(0xffffffffu, cj <= t));
    if (cnt < 32) {  // the last entry <= t is in this chunk, or ended the previous one
      if (cnt == 0) {
        b = base - 1;
        cu_b = prev_c;
        L = prev_l;
        cu_b1 = __shfl_sync(0xffffffffu, cj, 0);
      } else {
        b = base + cnt - 1;
        cu_b = __shfl_sync(0xffffffffu, cj, cnt - 1);
        L = __shfl_sync(0xffffffffu, lj, cnt - 1);
        cu_b1 = __shfl_sync(0xffffffffu, cj, cnt);
      }
      break;
    }
    prev_c = __shfl_sync(0xffffffffu, cj, 31);
    prev_l = __shfl_sync(0xffffffffu, lj, 31);
  }
  if (b < 0 || b >= P.batch || t >= cu_b1) return nullptr;  // token outside every sequence
  const int n = cu_b1 - cu_b;
  if (L < 0 || n > L) {
    if (lane == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    return nullptr;
  }
  const int p = L - n + (t - cu_b);
  const int row = P.headwise ? b * P.num_kv_heads + h : b;
  const int lb = p / P.block_size;
  if (lb >= P.max_blocks) {
    if (lane == 0) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    return nullptr;
  }
  const int blk = __ldg(P.table + (size_t)row * P.max_blocks + lb);
  if (blk < 0) return nullptr;  // evicted slot: nothing is written
  if (blk >= P.num_blocks) {
    if (lane == 0) flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
    return nullptr;
  }
  const int R = row_bytes_of(P.mode, P.head_dim);
  const size_t slot = ((size_t)blk * P.num_kv_heads + h) * P.block_size + (p % P.block_size);
  if (!KVQ_IN_BOUNDS(slot < (size_t)P.num_blocks * P.num_kv_heads * P.block_size, P.dev_error)) return nullptr;
  return pages + slot * R;
}

// OR-combine `bits` (nbits per lane) of groups of 32/nbits lanes into one
// 32-bit word held by the first lane of each group.
template <int NBITS>
__device__ __forceinline__ uint32_t gather_word(uint32_t bits, int lane) {
  constexpr int LPW = 32 / NBITS;  // lanes per word
  uint32_t v = bits << ((lane % LPW) * NBITS);
#pragma unroll
  for (int o = 1; o < LPW; o <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int MODE, int D, bool STEGO>
__global__ void __launch_bounds__(256) write_token_head_kernel(WriteParams P) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  // a decode call after this write may start its query preparation now; it
  // waits for this grid before anything reads the pages written here
  allow_dependent_launch();
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int kv = (int)(wid & 1);
  const long long th = wid >> 1;
  const int h = (int)(th % P.num_kv_heads);
  const long long t = th / P.num_kv_heads;
  if (t >= P.num_tokens) return;
  float x[EPL];  // issued before the (dependent) table lookups
  load_row_elems<EPL>(kv ? P.v : P.k, P.dtype, ((size_t)t * P.num_kv_heads + h) * D + lane * EPL, x);
  const RowSigns<EPL> sg = load_row_signs<EPL>(P.signs, lane);
  uint8_t* dst = dest_row(P, kv ? P.v_pages : P.k_pages, (int)t, h, lane);
  if (dst == nullptr) return;  // warp-uniform
  quantise_store_row<MODE, D, STEGO, 32>(sg, x, dst, lane, true);
}

// INT8, pass 1 (only while *ready == 0): per-channel max |x| over all tokens.
// Column c = (kv * Hkv + h) * D + d; amax must start at zero; non-negative
// floats order like their bit patterns, so an integer atomicMax is exact.
__global__ void __launch_bounds__(256) int8_amax_kernel(WriteParams P, int tokens_per_block) {
  if (__ldg(P.ch_ready) != 0) return;
  const int cols = 2 * P.num_kv_heads * P.head_dim;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int per_kv = P.num_kv_heads * P.head_dim;
  const int kv = c / per_kv, hd = c % per_kv;
  const void* src = kv ? P.v : P.k;
  const int t0 = blockIdx.y * tokens_per_block;
  const int t1 = min(P.num_tokens, t0 + tokens_per_block);
  float a = 0.0f;
  for (int t = t0; t < t1; ++t) {
    float x[1];
    const size_t off = (size_t)t * per_kv + hd;
    x[0] = P.dtype == DT_F32 ? __ldg(reinterpret_cast<const float*>(src) + off)
                             : __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(src) + off) << 16);
    a = fmaxf(a, fabsf(x[0]));
  }
  atomicMax(reinterpret_cast<int*>(P.ch_amax) + c, __float_as_int(a));
}

// INT8, pass 2: q = clamp(rne(x / (amax / 127)), -127, 127).
template <int D>
__global__ void __launch_bounds__(256) int8_quant_kernel(WriteParams P) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  allow_dependent_launch();  // as in write_token_head_kernel
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blockIdx.x == 0 && threadIdx.x == 0) *P.ch_ready = 1;  // later calls reuse the scales
  const int kv = (int)(wid & 1);
  const long long th = wid >> 1;
  const int h = (int)(th % P.num_kv_heads);
  const long long t = th / P.num_kv_heads;
  if (t >= P.num_tokens) return;
  float x[EPL];
  load_row_elems<EPL>(kv ? P.v : P.k, P.dtype, ((size_t)t * P.num_kv_heads + h) * D + lane * EPL, x);
  uint8_t* dst = dest_row(P, kv ? P.v_pages : P.k_pages, (int)t, h, lane);
  if (dst == nullptr) return;
  const float* am = P.ch_amax + ((size_t)kv * P.num_kv_heads + h) * D + lane * EPL;
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const float s = __fdiv_rn(am[i], 127.0f);
    int q = 0;
    if (s != 0.0f) {
      float r = rintf(__fdiv_rn(x[i], s));
      r = fminf(fmaxf(r, -127.0f), 127.0f);
      q = (int)r;
    }
    bits |= ((uint32_t)q & 0xFFu) << (8 * i);
  }
  const uint32_t word = gather_word<EPL * 8>(bits, lane);
  constexpr int LPW = 32 / (EPL * 8);
  if (lane % LPW == 0) *reinterpret_cast<uint32_t*>(dst + 4 * (lane / LPW)) = word;
}

// ---------------------------------------------------------------------------
// Gather and dequantise: FastDeploy PR #5173 "support dynamic int2
// quantization cache kv" (its review lists the new custom op
// dynamic_quant_get_kv_from_cache) and the Ascend INT8 plugin, 运行机制
// (chunked prefill gathers and dequantises the paged cache).  The write's
// position map; each row's codes become fp32 values, the warp maps the row
// back through the inverse RHT d * (H y) / D, and the row is stored densely
// (fp32 or bf16).  A row the table marks -1, or that cannot be located, is
// stored as zeros.
//
// One warp per (GATHER_TOKENS consecutive tokens, kv head): lanes 0..7 locate
// one token each (binary search of cu, then the table), the warp then issues
// the loads of all 2 x GATHER_TOKENS rows (K and V share the lookup) before
// it converts and stores them, so each warp keeps 16 row loads in flight
// instead of one dependent chain per row.
constexpr int GATHER_TOKENS = 8;

// Byte offset of (token t, kv head h)'s row in a pool, -1 (evicted or
// invalid; invalid rows set their error bit), or -2 - r for row r of the
// full-precision chunk.
template <bool CHUNK>
__device__ __forceinline__ long long gather_row_offset(const WriteParams& P, int t, int h) {
  if (t >= P.num_tokens) return -1;
  int lo = 0, hi = P.batch - 1;  // the last sequence whose first token is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P.cu_new + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  const int cu_b = __ldg(P.cu_new + b), cu_b1 = __ldg(P.cu_new + b + 1);
  if (t < cu_b || t >= cu_b1) return -1;  // outside every sequence
  const int n = cu_b1 - cu_b, L = __ldg(P.seq_lens + b);
  if (L < 0 || n > L) {
    flag_error(P.dev_error, DEVERR_SEQ_LEN);
    return -1;
  }
  const int p = L - n + (t - cu_b);
  if constexpr (CHUNK) {
    const int c0 = __ldg(P.cu_chunk + b), m = __ldg(P.cu_chunk + b + 1) - c0;
    if (m < 0 || m > L) {
      flag_error(P.dev_error, DEVERR_SEQ_LEN);
      return -1;
    }
    if (p >= L - m) return -2 - (long long)(c0 + p - (L - m));
  }
  const int lb = p / P.block_size;
  if (lb >= P.max_blocks) {
    flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    return -1;
  }
  const int row = P.headwise ? b * P.num_kv_heads + h : b;
  const int blk = __ldg(P.table + (size_t)row * P.max_blocks + lb);
  if (blk < 0) return -1;
  if (blk >= P.num_blocks) {
    flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
    return -1;
  }
  const int R = row_bytes_of(P.mode, P.head_dim);
  const size_t slot = ((size_t)blk * P.num_kv_heads + h) * P.block_size + (p % P.block_size);
  if (!KVQ_IN_BOUNDS(slot < (size_t)P.num_blocks * P.num_kv_heads * P.block_size, P.dev_error)) return -1;
  return (long long)slot * R;
}

// tsign: the lane's d_i / D factors of the inverse RHT (0 = RHT off)
template <int MODE, int D, bool STEGO>
__device__ __forceinline__ void gather_dequant(const WriteParams& P, uint32_t w, uint32_t pad, int kv, int h,
                                               int lane, const float (&tsign)[D / 32], float (&y)[D / 32]) {
  constexpr int EPL = D / 32;
  constexpr int BITS = mode_bits(MODE);
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const uint32_t u = (w >> (e * BITS)) & ((1u << BITS) - 1u);
    if constexpr (MODE == MODE_INT8) {
      const int c = lane * EPL + e;
      const float s = __fdiv_rn(__ldg(P.ch_amax + ((size_t)kv * P.num_kv_heads + h) * D + c), 127.0f);
      y[e] = __fmul_rn((float)(int8_t)u, s);
    } else if constexpr (MODE == MODE_I8T) {
      y[e] = __fmul_rn((float)(int8_t)u, __uint_as_float(pad));
    } else if constexpr (MODE == MODE_F8T) {
      const float c = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)u, __NV_E4M3)));
      y[e] = __fmul_rn(c, __uint_as_float(pad));
    } else if constexpr (STEGO) {
      y[e] = __fmul_rn((float)((int)u - (int)(pad & 15u)), __uint_as_float(pad & ~15u));
    } else {
      const float S = __half2float(__ushort_as_half((unsigned short)(pad & 0xFFFFu)));
      const float M = __half2float(__ushort_as_half((unsigned short)(pad >> 16)));
      y[e] = __fadd_rn(__fmul_rn((float)u, S), M);
    }
  }
  if (MODE != MODE_INT8 && P.signs) {
    wht_warp<EPL>(y, lane);
#pragma unroll
    for (int e = 0; e < EPL; ++e) y[e] = __fmul_rn(y[e], tsign[e]);  // exact: +-1 / D
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void gather_store(void* out, size_t o, const float (&y)[D / 32]) {
  constexpr int EPL = D / 32;
  if constexpr (!BF16) {
    float* p = reinterpret_cast<float*>(out) + o;
    if constexpr (EPL == 4) *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
    else *reinterpret_cast<float2*>(p) = make_float2(y[0], y[1]);
  } else {
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(out) + o;
    const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]);
    if constexpr (EPL == 4) {
      const __nv_bfloat162 c = __floats2bfloat162_rn(y[2], y[3]);
      *reinterpret_cast<uint2*>(p) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c));
    } else {
      *reinterpret_cast<__nv_bfloat162*>(p) = a;
    }
  }
}

// Dequantise, map back and store the warp's 2 x GATHER_TOKENS rows.  Rows
// without data arrive as code word 0 and pad 0, which every mode turns into
// zeros (scale 0, or code 0 for INT8 per channel), so no branch is needed;
// full-precision chunk rows (off <= -2, warp-uniform) are copied as given.
template <int MODE, int D, bool STEGO, bool BF16, bool CHUNK>
__device__ __forceinline__ void gather_rows(const WriteParams& P, const uint32_t (&w)[2][GATHER_TOKENS],
                                            const uint32_t (&pad)[2][GATHER_TOKENS],
                                            const long long (&off)[GATHER_TOKENS], long long t0, int h, int lane,
                                            const float (&tsign)[D / 32]) {
  constexpr int EPL = D / 32;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv)
#pragma unroll
    for (int r = 0; r < GATHER_TOKENS; ++r) {
      float y[EPL];
      if (CHUNK && off[r] <= -2) {
        long long src = -2 - off[r];
        if (!KVQ_IN_BOUNDS(src < (long long)__ldg(P.cu_chunk + P.batch), P.dev_error)) src = 0;
        load_row_elems<EPL>(kv ? P.chunk_v : P.chunk_k, P.chunk_dtype,
                            ((size_t)src * P.num_kv_heads + h) * D + lane * EPL, y);
      } else {
        gather_dequant<MODE, D, STEGO>(P, w[kv][r], pad[kv][r], kv, h, lane, tsign, y);
      }
      const long long t = t0 + r;
      if (t < P.num_tokens) gather_store<D, BF16>(kv ? P.out_v : P.out_k, ((size_t)t * P.num_kv_heads + h) * D + lane * EPL, y);
    }
}

template <int MODE, int D, bool STEGO, bool CHUNK>
__global__ void __launch_bounds__(256) gather_kernel(WriteParams P) {
  constexpr int EPL = D / 32;
  constexpr int BITS = mode_bits(MODE);
  constexpr int DATA = data_bytes(MODE, D);
  constexpr int LB = EPL * BITS;  // bits per lane, a divisor of 32
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int h = (int)(wid % P.num_kv_heads);
  const long long t0 = (wid / P.num_kv_heads) * GATHER_TOKENS;
  if (t0 >= P.num_tokens) return;
  // 1. lanes 0..7 locate one token each
  long long my_off = -1;
  if (lane < GATHER_TOKENS) my_off = gather_row_offset<CHUNK>(P, (int)(t0 + lane), h);
  long long off[GATHER_TOKENS];
#pragma unroll
  for (int r = 0; r < GATHER_TOKENS; ++r) off[r] = __shfl_sync(0xffffffffu, my_off, r);
  float tsign[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e)
    tsign[e] = (P.signs && __ldg(P.signs + lane * EPL + e) < 0 ? -1.0f : 1.0f) / (float)D;
  // 2. every row's loads in flight together: the lane's code word and the pad
  const int word = (lane * LB) >> 5, shift = (lane * LB) & 31;
  uint32_t w[2][GATHER_TOKENS], pad[2][GATHER_TOKENS];
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const uint8_t* pool = kv ? P.v_pages : P.k_pages;
#pragma unroll
    for (int r = 0; r < GATHER_TOKENS; ++r) {
      w[kv][r] = 0;
      pad[kv][r] = 0;
      if (off[r] >= 0) {
        const uint8_t* src = pool + off[r];
        w[kv][r] = __ldg(reinterpret_cast<const uint32_t*>(src) + word) >> shift;
        if constexpr (MODE != MODE_INT8) pad[kv][r] = __ldg(reinterpret_cast<const uint32_t*>(src + DATA));
      }
    }
  }
  // 3. dequantise, inverse RHT, store
  if (P.out_dtype == DT_BF16) gather_rows<MODE, D, STEGO, true, CHUNK>(P, w, pad, off, t0, h, lane, tsign);
  else gather_rows<MODE, D, STEGO, false, CHUNK>(P, w, pad, off, t0, h, lane, tsign);
}

template <int MODE, bool STEGO>
void launch_gather_m(const WriteParams& P, int blocks, cudaStream_t stream) {
  // the full-precision chunk is a separate instantiation, so the plain
  // gather pays nothing for it
  if (P.chunk_k) {
    if (P.head_dim == 128) gather_kernel<MODE, 128, STEGO, true><<<blocks, 256, 0, stream>>>(P);
    else gather_kernel<MODE, 64, STEGO, true><<<blocks, 256, 0, stream>>>(P);
  } else {
    if (P.head_dim == 128) gather_kernel<MODE, 128, STEGO, false><<<blocks, 256, 0, stream>>>(P);
    else gather_kernel<MODE, 64, STEGO, false><<<blocks, 256, 0, stream>>>(P);
  }
}

cudaError_t launch_gather(const WriteParams& P, cudaStream_t stream) {
  const long long warps = (long long)((P.num_tokens + GATHER_TOKENS - 1) / GATHER_TOKENS) * P.num_kv_heads;
  const int blocks = (int)((warps + 7) / 8);
  switch (P.mode) {
    case MODE_INT4:
      if (P.stego) launch_gather_m<MODE_INT4, true>(P, blocks, stream);
      else launch_gather_m<MODE_INT4, false>(P, blocks, stream);
      break;
    case MODE_INT2: launch_gather_m<MODE_INT2, false>(P, blocks, stream); break;
    case MODE_INT8: launch_gather_m<MODE_INT8, false>(P, blocks, stream); break;
    case MODE_I8T: launch_gather_m<MODE_I8T, false>(P, blocks, stream); break;
    case MODE_F8T: launch_gather_m<MODE_F8T, false>(P, blocks, stream); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// The write of a long chunk: persistent warps, each taking units of four
// tokens of one kv head in turn (unit u: tokens 4 (u / Hkv) .. + 3, head
// u % Hkv).  Eight lanes per row: lane group g (lanes 8g .. 8g+7) takes token
// 4 (u / Hkv) + g, first its K row, then its V row.  With D/8 elements per
// lane the butterfly's first log2(D/8) stages and most of the min / max run
// in registers and the packed bytes form in lane (no word gather).  While a
// unit is quantised, the warp's next unit's input rows are already on their
// way into its shared-memory stage (cp.async) and lanes 0..3 have looked up
// its destinations (the gather's lookup, which flags the same errors as
// dest_row).  The row arithmetic is quantise_store_row's, so the bytes are
// those of write_token_head_kernel.
constexpr int WRITE_TOKENS = 4;
constexpr int WRITE_LPR = 32 / WRITE_TOKENS;  // lanes per row
constexpr int WRITE_BATCH_MIN_TOKENS = 512;
constexpr int WRITE_WARPS = 8;   // per CTA
constexpr int WRITE_STAGES = 2;  // input stages per warp
constexpr int WRITE_CTAS_PER_SM = 3;

// Shared memory of write_batch_kernel: per warp and stage, the unit's K rows
// then V rows as they are in the input ([4][D] of the input dtype each).
inline size_t write_batch_smem(int head_dim, int dtype) {
  return (size_t)WRITE_WARPS * WRITE_STAGES * 2 * WRITE_TOKENS * head_dim * (dtype == DT_F32 ? 4 : 2);
}

template <int MODE, int D, bool STEGO, bool F32>
__global__ void __launch_bounds__(WRITE_WARPS * 32, WRITE_CTAS_PER_SM) write_batch_kernel(WriteParams P) {
  constexpr int EPL = D / WRITE_LPR;
  constexpr int ESZ = F32 ? 4 : 2;
  constexpr int IN_ROW = D * ESZ;                        // bytes of one input row
  constexpr int UNIT = 2 * WRITE_TOKENS * IN_ROW;        // K rows, then V rows
  constexpr int CPR = IN_ROW / 16;                       // 16-byte pieces per row
  static_assert((UNIT / 16) % 32 == 0, "whole pieces per lane");
  extern __shared__ __align__(16) uint8_t wsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / WRITE_LPR, sub = lane % WRITE_LPR;
  allow_dependent_launch();  // as in write_token_head_kernel
  const int Hkv = P.num_kv_heads;
  const int groups = (P.num_tokens + WRITE_TOKENS - 1) / WRITE_TOKENS;
  uint8_t* buf = wsm + (size_t)warp * WRITE_STAGES * UNIT;
  const RowSigns<EPL> sg = load_row_signs<EPL>(P.signs, sub);  // shared by every row of this lane
  // unit u = grp * Hkv + h, taken by warps u, u + nw, u + 2 nw, ...
  const int nw = gridDim.x * WRITE_WARPS;
  const int step_g = nw / Hkv, step_h = nw % Hkv;
  const int w0 = blockIdx.x * WRITE_WARPS + warp;
  int grp = w0 / Hkv, h = w0 % Hkv;

  // input rows of unit (gg, hh) into stage st (rows past the input are not read)
  auto issue = [&](int gg, int hh, int st) {
    if (gg < groups) {
      uint8_t* dst = buf + st * UNIT;
#pragma unroll
      for (int k = 0; k < UNIT / 16 / 32; ++k) {
        const int c = lane + 32 * k;
        const int row = c / CPR, part = c % CPR;
        const int t = gg * WRITE_TOKENS + row % WRITE_TOKENS;
        if (t < P.num_tokens)
          cp_async16(dst + 16 * c,
                     static_cast<const uint8_t*>(row < WRITE_TOKENS ? P.k : P.v) + ((size_t)t * Hkv + hh) * IN_ROW +
                         16 * part,
                     16);
      }
    }
    cp_async_commit();
  };
  // destination byte offset of token WRITE_TOKENS gg + lane (lanes 0..3), -1: none
  auto lookup = [&](int gg, int hh) -> long long {
    if (gg >= groups || lane >= WRITE_TOKENS) return -1;
    return gather_row_offset<false>(P, gg * WRITE_TOKENS + lane, hh);
  };

  issue(grp, h, 0);
  long long my_off = lookup(grp, h);
  int st = 0;
  while (grp < groups) {
    int ng = grp + step_g, nh = h + step_h;
    if (nh >= Hkv) {
      nh -= Hkv;
      ++ng;
    }
    issue(ng, nh, st ^ 1);
    const long long next_off = lookup(ng, nh);
    cp_async_wait<1>();  // this unit's rows have landed
    __syncwarp();
    float x[2][EPL];
    const uint8_t* src = buf + st * UNIT + g * IN_ROW + sub * EPL * ESZ;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint8_t* r = src + kv * WRITE_TOKENS * IN_ROW;
#pragma unroll
      for (int c = 0; c < EPL * ESZ / 16; ++c) {
        const uint4 v = lds128(r + 16 * c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (F32) {
            x[kv][4 * c + k] = __uint_as_float(w[k]);
          } else {
            x[kv][8 * c + 2 * k] = __uint_as_float(w[k] << 16);
            x[kv][8 * c + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
          }
        }
      }
    }
    __syncwarp();  // every lane has read this stage before it is filled again
    const long long off = __shfl_sync(0xffffffffu, my_off, g);  // -1: an evicted, invalid or absent row
#pragma unroll
    for (int kv = 0; kv < 2; ++kv)
      quantise_store_row<MODE, D, STEGO, WRITE_LPR>(sg, x[kv], (kv ? P.v_pages : P.k_pages) + (off >= 0 ? off : 0),
                                                    lane, off >= 0);
    my_off = next_off;
    grp = ng;
    h = nh;
    st ^= 1;
  }
  cp_async_wait<0>();
}

template <int MODE, bool STEGO>
cudaError_t launch_write_m(const WriteParams& P, cudaStream_t stream) {
  if (P.num_tokens >= WRITE_BATCH_MIN_TOKENS) {
    // one CTA of eight persistent warps per unit group, at most
    // WRITE_CTAS_PER_SM per SM; the opt-in shared-memory size is set once per
    // device (not inside later calls, which may be captured into a graph)
    static bool attr_set[64] = {false};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = write_batch_smem(P.head_dim, P.dtype);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
      const int mx = (int)write_batch_smem(128, DT_F32);
      const void* fns[4] = {(const void*)write_batch_kernel<MODE, 128, STEGO, false>,
                            (const void*)write_batch_kernel<MODE, 128, STEGO, true>,
                            (const void*)write_batch_kernel<MODE, 64, STEGO, false>,
                            (const void*)write_batch_kernel<MODE, 64, STEGO, true>};
      for (const void* f : fns)
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    // units of four tokens of one kv head; the kernel counts them in 32 bits
    const long long units = (long long)((P.num_tokens + WRITE_TOKENS - 1) / WRITE_TOKENS) * P.num_kv_heads;
    const int blocks = (int)std::min<long long>((units + WRITE_WARPS - 1) / WRITE_WARPS, (long long)sms * WRITE_CTAS_PER_SM);
    const dim3 grid(blocks), block(WRITE_WARPS * 32);
    const bool f32 = P.dtype == DT_F32;
    if (P.head_dim == 128) {
      if (f32) write_batch_kernel<MODE, 128, STEGO, true><<<grid, block, smem, stream>>>(P);
      else write_batch_kernel<MODE, 128, STEGO, false><<<grid, block, smem, stream>>>(P);
    } else {
      if (f32) write_batch_kernel<MODE, 64, STEGO, true><<<grid, block, smem, stream>>>(P);
      else write_batch_kernel<MODE, 64, STEGO, false><<<grid, block, smem, stream>>>(P);
    }
  } else {
    const long long warps = (long long)P.num_tokens * P.num_kv_heads * 2;
    const int blocks = (int)((warps + 7) / 8);
    if (P.head_dim == 128) write_token_head_kernel<MODE, 128, STEGO><<<blocks, 256, 0, stream>>>(P);
    else write_token_head_kernel<MODE, 64, STEGO><<<blocks, 256, 0, stream>>>(P);
  }
  return cudaGetLastError();
}

cudaError_t launch_write(const WriteParams& P, cudaStream_t stream) {
  const long long warps = (long long)P.num_tokens * P.num_kv_heads * 2;
  const int blocks = (int)((warps + 7) / 8);
  if (P.mode == MODE_INT8) {
    const int tpb = 1024;
    dim3 g1((2 * P.num_kv_heads * P.head_dim + 255) / 256, (P.num_tokens + tpb - 1) / tpb);
    int8_amax_kernel<<<g1, 256, 0, stream>>>(P, tpb);
    if (P.head_dim == 128) int8_quant_kernel<128><<<blocks, 256, 0, stream>>>(P);
    else int8_quant_kernel<64><<<blocks, 256, 0, stream>>>(P);
    return cudaGetLastError();
  }
  if (P.mode == MODE_I8T) return launch_write_m<MODE_I8T, false>(P, stream);
  if (P.mode == MODE_F8T) return launch_write_m<MODE_F8T, false>(P, stream);
  if (P.mode == MODE_INT4 && P.stego) return launch_write_m<MODE_INT4, true>(P, stream);
  if (P.mode == MODE_INT4) return launch_write_m<MODE_INT4, false>(P, stream);
  return launch_write_m<MODE_INT2, false>(P, stream);
}

}  // namespace kvq
