// kvq_prefill_tc.cu -- causal chunked-prefill attention over the paged
// low-bit cache on the 5th-generation tensor cores (tcgen05, TMEM).
//
// What it computes: every query of the chunk (sequence b, position
// seq_lens[b] - n_b + i) attends causally to all keys visible at its
// position, the chunk's own keys included, all read back from the INT4 /
// INT2 / INT8 / FP8 pages (the chunk is written with kvq_write first).  Sources
// (page title, section): FastDeploy PR #5173 "support dynamic int2
// quantization cache kv", Usage (chunked prefill with 8192 batched tokens);
// vLLM PR #40835 review summary ("INT4 per-token-head KV cache for the Triton
// backend"), 实现拆解 item 2 and 风险与影响 (causal attention only);
// vllm-ascend-quantized-kv-cache METADATA ("Ascend INT8 KV Cache Plugin"),
// 运行机制 (chunked prefill reads and dequantises the paged cache); FastDeploy
// PR #7718 "Optimize AppendAttention for discrete head-wise block_idx"
// (head-wise rows, -1 sentinel, sink tokens).
//
// Design: one CTA of 14 warps per (128 rows, kv head, sequence); the 128
// rows are (query, q head of the GQA group) pairs, so every key tile is
// expanded once for the whole group.  Roles:
//   warps 0-7  softmax: row r belongs to warps r / 32 (keys 0-31 of each
//              tile) and r / 32 + 4 (keys 32-63).  Each half keeps its own
//              running maximum, sum and O accumulator (O0, O1 in TMEM), so
//              the two never wait for each other inside the key loop; it
//              reads its logits from TMEM, masks them, writes (P s) hi / lo
//              over them and rescales its O when its maximum grows.  In the
//              end the halves merge (log-sum-exp weights) and the row gets
//              the zero-point term, the inverse RHT and 1 / l.
//   warp 8     TMEM allocation; lane 0 issues every tcgen05.mma:
//              S_b = Q_hi K^T + Q_lo K^T (M=128, N=64, K=D) into one of two
//              TMEM buffers, then O0 += P_hi V + P_lo V over keys 0-31 and
//              O1 over keys 32-63 (M=128, N=D).
//   warps 9-12 producers: expansion of the codes into fp16 K (K-major) and
//              V^T (K-major, transposed with stmatrix) tiles in the 128-byte
//              swizzle layout.
//   warp 13    copy issuer: bulk copies of the raw page chunks.
// Codes enter the tensor cores as signed integers (exact in fp16); the
// query and (P s) are split into fp16 hi + lo terms so fp16 does not limit
// accuracy.  Every wait on an mbarrier is bounded; on a timeout the CTA
// reports KVQ_DEVERR_TIMEOUT, drains, frees its TMEM and returns.

#include <math_constants.h>

#include "kvq_internal.h"
#include "kvq_tc.cuh"

namespace kvq {

namespace {

constexpr int TP_ROWS = PREFILL_ROWS_PER_CTA;
constexpr int TP_KT = 64;
constexpr int TP_THREADS = 448;
constexpr int TP_SOFTMAX = 256;    // warps 0-7: warp w owns rows 32 (w % 4) .. + 31, keys 32 (w / 4) .. + 31 of a tile
constexpr int TP_MMA_WARP = 8;
constexpr int TP_PROD_WARP0 = 9;   // warps 9-12 expand codes
constexpr int TP_PRODUCERS = 128;
constexpr int TP_ISSUE_WARP = 13;
// O is rescaled only when a row's maximum grows by more than 2^TP_SLACK, so
// weights p reach at most 2^TP_SLACK and p * s stays inside fp16 for any
// scale s below 65504 / 2^TP_SLACK (4094).
constexpr float TP_SLACK = 4.0f;
// sleep between polls of a barrier wait, by role (ns): the softmax and the
// MMA issuer are the critical path, the copy issuer and the producers run ahead
constexpr uint32_t TP_NAP_SOFTMAX = 20, TP_NAP_MMA = 20, TP_NAP_PRODUCER = 100, TP_NAP_ISSUER = 200;

template <int MODE, int D>
struct TpCfg {
  static constexpr int DATA = data_bytes(MODE, D);  // code bytes before the pad (dense rows: D * 2, no pad)
  static_assert(DATA <= row_bytes_of(MODE, D), "the pad follows the codes");
  static constexpr int R = row_bytes_of(MODE, D);
  static constexpr int CHUNK = 16 * R;          // one 16-row chunk of a page (contiguous)
  static constexpr int RAW = TP_KT * R;         // raw bytes of one tensor per tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int KATOM = TP_KT * 128;     // one 64-wide atom of the K tile (8 KB)
  static constexpr int KTILE = (D / 64) * KATOM;
  static constexpr int VTILE = D * 128;         // V^T: D rows x 64 keys
  // expanded K / V^T stages and raw stages
  static constexpr int NKV = 3;
  static constexpr int NRAW = 3;
  // shared-memory layout (swizzled tiles at 1024-byte boundaries)
  static constexpr int OFF_K = 0;                                       // [NKV] K tiles
  static constexpr int OFF_VT = OFF_K + NKV * KTILE;                   // [NKV] V^T tiles
  static constexpr int OFF_RAW = OFF_VT + NKV * VTILE;                 // [NRAW][K,V][RAW]
  static constexpr int OFF_SC = OFF_RAW + NRAW * 2 * RAW;              // [NKV][ks, kz, vs, vz][64] f32
  static constexpr int OFF_KVAL = OFF_SC + NKV * 4 * TP_KT * 4;        // [NKV][4] chunk validity of the expanded tiles
  static constexpr int OFF_RAWVAL = OFF_KVAL + 64;                     // [NRAW][4] chunk validity of the raw tiles
  static constexpr int OFF_XMAX = OFF_RAWVAL + 64;                     // [2 key halves][128] f32 (epilogue)
  static constexpr int OFF_ROW = OFF_XMAX + 2 * 2 * TP_ROWS * 4;       // beta, gamma [128] f32, pos [128] int
  static constexpr int OFF_BAR = OFF_ROW + 3 * TP_ROWS * 4;            // mbarriers
  static constexpr int NBAR = 32;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;                  // tmem slot, abort flag, sequence
  static constexpr int SMEM = OFF_MISC + 16 + 1024;                    // + alignment slack
  // TMEM columns: S[2] (64 fp32 each; P hi / lo overwrite them), O0 (D fp32),
  // Q hi and Q lo (D / 2 columns each: two fp16 per column), O1 (D fp32)
  static constexpr int TM_O = 2 * TP_KT;
  static constexpr int TM_QHI = TM_O + D;
  static constexpr int TM_QLO = TM_QHI + D / 2;
  static constexpr int TM_O1 = TM_QLO + D / 2;  // O of the second key half
  static constexpr int TMEM_COLS = TM_O1 + D <= 256 ? 256 : 512;
  // the query rows are staged (fp16 hi / lo, rows padded by 16 bytes) in the
  // K / V^T stages before they are moved to TMEM
  static constexpr int QROW = 2 * D + 16;
  // the epilogue stages O rows (fp32, 16-byte pieces XOR-swizzled by row)
  // in the K / V^T stages, free once the last P.V is done
  static_assert(TP_ROWS * D * 4 <= NKV * (KTILE + VTILE), "epilogue staging does not fit");
  static_assert(2 * TP_ROWS * QROW <= NKV * (KTILE + VTILE), "query staging does not fit");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(CHUNK % 16 == 0 && R % 4 == 0, "bulk copies need 16-byte multiples");
};

// barriers: raw stage full [3] / empty [3], K/V stage full [3] / empty [3],
// S full [2] / empty [2], P full, O done, drain, and per row quad the
// epilogue's meeting of its two softmax warps [4]
enum {
  B_RAWFULL = 0, B_RAWEMPTY = 3, B_KVFULL = 6, B_KVEMPTY = 9, B_SFULL = 12, B_SEMPTY = 14, B_PFULL = 16, B_ODONE = 17,
  B_DRAIN = 18, B_EPI = 28
};

// Two bf16 values (low half first) as an fp16 pair, rounded to nearest.  A
// bf16 value carries 8 significant bits, so the conversion is exact for 0 and
// for 2^-17 <= |x| <= 65504 (fp16 normals, and the subnormals that are
// multiples of 2^-24).  Smaller magnitudes round to a multiple of 2^-24
// (error at most 2^-25); magnitudes above 65504 become 65504 or infinity.
__device__ __forceinline__ uint32_t bf16x2_to_half2_bits(uint32_t w) {
  const __half2 hv = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&hv);
}

// Eight consecutive codes (head dims 8c .. 8c+7) of a raw row as four exact
// fp16 pairs of signed codes u - 2^(b-1) (INT8: as stored; FP8: the E4M3
// value; dense rows: the bf16 values), in dim order.
template <int MODE>
__device__ __forceinline__ uint4 codes8(const uint8_t* raw_row, int c) {
  uint32_t o[4];
  if constexpr (MODE == MODE_DBF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(raw_row + 16 * c);
    o[0] = bf16x2_to_half2_bits(w.x);
    o[1] = bf16x2_to_half2_bits(w.y);
    o[2] = bf16x2_to_half2_bits(w.z);
    o[3] = bf16x2_to_half2_bits(w.w);
  } else if constexpr (MODE == MODE_INT4) {
    const uint32_t w = lds32(raw_row + 4 * c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = prmt(w, 0u, j | (4 << 4) | (j << 8) | (4 << 12));  // byte j in both halves
      o[j] = hsub2_bits(lop3_and_or(x, 0x00F0000Fu, 0x54006400u), 0x54806408u);
    }
  } else if constexpr (MODE == MODE_INT2) {
    const uint32_t w = *reinterpret_cast<const uint16_t*>(raw_row + 2 * c);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t x = prmt(w, 0u, j | (4 << 4) | (j << 8) | (4 << 12));
      o[2 * j] = hsub2_bits(lop3_and_or(x, 0x000C0003u, 0x5C006400u), 0x5C086402u);
      o[2 * j + 1] = hsub2_bits(lop3_and_or(x, 0x00C00030u, 0x4C005400u), 0x4C805420u);
    }
  } else if constexpr (MODE == MODE_F8T) {
    const uint2 w = make_uint2(lds32(raw_row + 8 * c), lds32(raw_row + 8 * c + 4));  // rows are D + 4 bytes
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = e4m3x2_to_half2_bits((j < 2 ? w.x : w.y) >> (16 * (j & 1)));
  } else {
    // INT8 channel rows (D bytes) are 8-byte aligned, token-head rows (D + 4) are not
    const uint2 w = MODE == MODE_INT8 ? lds64(raw_row + 8 * c)
                                      : make_uint2(lds32(raw_row + 8 * c), lds32(raw_row + 8 * c + 4));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t src = j < 2 ? w.x : w.y;
      const int bb = 2 * (j & 1);
      const uint32_t x = prmt(src, 0u, bb | (4 << 4) | ((bb + 1) << 8) | (4 << 12));
      o[j] = hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Dense raw tiles: D / 64 halves of DENSE_HALF bytes, each 64 rows of 128
// bytes (64 bf16 dims) with the 128-byte swizzle of the tensor copy.
constexpr int DENSE_HALF = 64 * 128;
// Dims 8c .. 8c+7 of row `row` as four fp16 pairs.
__device__ __forceinline__ uint4 dense_codes8(const uint8_t* raw, int row, int c) {
  const uint4 w = *reinterpret_cast<const uint4*>(raw + (c >> 3) * DENSE_HALF + tc::sw128_off(row, c & 7));
  return make_uint4(bf16x2_to_half2_bits(w.x), bf16x2_to_half2_bits(w.y), bf16x2_to_half2_bits(w.z),
                    bf16x2_to_half2_bits(w.w));
}
// Dims d, d+1 (d even) of row `row` as an fp16 pair (low half = dim d).
__device__ __forceinline__ uint32_t dense_codes2(const uint8_t* raw, int row, int d) {
  const int c = (d & 63) >> 3;
  return bf16x2_to_half2_bits(*reinterpret_cast<const uint32_t*>(raw + (d >> 6) * DENSE_HALF +
                                                                 tc::sw128_off(row, c) + 2 * (d & 7)));
}

// The two codes of head dims (d, d+1), d even, of a raw row as an exact fp16
// pair of signed codes (low half = dim d).
template <int MODE>
__device__ __forceinline__ uint32_t codes2(const uint8_t* raw_row, int d) {
  if constexpr (MODE == MODE_DBF16) {
    return bf16x2_to_half2_bits(*reinterpret_cast<const uint32_t*>(raw_row + 2 * d));
  } else if constexpr (MODE == MODE_INT4) {
    const uint32_t b = raw_row[d >> 1];
    const uint32_t x = b | (b << 16);
    return hsub2_bits(lop3_and_or(x, 0x00F0000Fu, 0x54006400u), 0x54806408u);
  } else if constexpr (MODE == MODE_INT2) {
    const uint32_t b = (uint32_t)raw_row[d >> 2] >> (2 * (d & 3));  // crumbs d, d+1 at bits 0-3
    const uint32_t x = b | (b << 16);
    return hsub2_bits(lop3_and_or(x, 0x000C0003u, 0x5C006400u), 0x5C086402u);
  } else if constexpr (MODE == MODE_F8T) {
    // V rows of masked keys may hold stale NaN codes (weight 0 times NaN is NaN)
    return e4m3x2_to_half2_bits(e4m3x4_no_nan(*reinterpret_cast<const uint16_t*>(raw_row + d)));
  } else {
    const uint32_t w = *reinterpret_cast<const uint16_t*>(raw_row + d);
    const uint32_t x = prmt(w, 0u, 0 | (4 << 4) | (1 << 8) | (4 << 12));
    return hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);
  }
}

}  // namespace

// Heaviest sequences first: CTA row z of the grid takes the sequence of
// rank z by 2 L - n (a proxy for its keys per query), so the long prefixes
// start in the first wave and the short ones fill the tail.  Batches above
// 64 sequences keep their order.
__device__ __forceinline__ int heavy_first_sequence(const AttnParams& P, int z) {
  if (P.batch > 64) return z;
  const int lane = threadIdx.x & 31;
  int key[2], me = -1;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int b = lane + 32 * k;
    key[k] = b < P.batch ? 2 * __ldg(P.seq_lens + b) - (__ldg(P.cu_q + b + 1) - __ldg(P.cu_q + b)) : INT_MIN;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int b = lane + 32 * k;
    int rank = 0;
    for (int j = 0; j < P.batch; ++j) {
      const int kj = __shfl_sync(0xffffffffu, key[j >> 5], j & 31);
      rank += (kj > key[k] || (kj == key[k] && j < b)) ? 1 : 0;
    }
    if (b < P.batch && rank == z) me = b;
  }
  const unsigned m = __ballot_sync(0xffffffffu, me >= 0);
  const int src = m ? __ffs(m) - 1 : 0;
  const int b = __shfl_sync(0xffffffffu, me, src);
  return m ? b : z;
}

template <int MODE, int D>
__global__ void __launch_bounds__(TP_THREADS, 1) prefill_tc_kernel(const __grid_constant__ AttnParams P) {
  using C = TpCfg<MODE, D>;
  constexpr int NKV = C::NKV;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* seq_slot = reinterpret_cast<int*>(sm + C::OFF_MISC + 8);
  if (warp == 0) {
    const int b0 = heavy_first_sequence(P, blockIdx.z);
    if (lane == 0) *seq_slot = b0;
  }
  __syncthreads();
  const int b = *seq_slot, h = blockIdx.y;
  const int qtile = gridDim.x - 1 - blockIdx.x;  // later queries (more keys) first
  const int G = P.group, Hq = P.num_q_heads, Hkv = P.num_kv_heads, bs = P.block_size;
  const int QB = TP_ROWS / G;

  const int cq0 = __ldg(P.cu_q + b);
  const int n = __ldg(P.cu_q + b + 1) - cq0;
  const int q0 = qtile * QB;
  if (q0 >= n) return;
  const int L = __ldg(P.seq_lens + b);
  if (n > L || L < 0) {
    if (tid == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    return;
  }
  int Leff = L;
  if (Leff > P.max_blocks * bs) {
    if (tid == 0) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    Leff = P.max_blocks * bs;
  }
  if constexpr (MODE == MODE_DBF16) {  // the sequence's dense rows must hold its L keys
    if (__ldg(P.cu_kv + b + 1) - __ldg(P.cu_kv + b) < L) {
      if (tid == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
      return;
    }
  }
  const int nq = min(QB, n - q0);
  const int p_min = L - n + q0, p_max = L - n + q0 + nq - 1;

  float* sc = reinterpret_cast<float*>(sm + C::OFF_SC);
  int* kval = reinterpret_cast<int*>(sm + C::OFF_KVAL);
  int* rawval = reinterpret_cast<int*>(sm + C::OFF_RAWVAL);
  float* rbeta = reinterpret_cast<float*>(sm + C::OFF_ROW);
  float* rgamma = rbeta + TP_ROWS;
  int* rpos = reinterpret_cast<int*>(rgamma + TP_ROWS);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);

  // ---- key tiles: [0, p_max] or, for a sliding-window head, the sink tiles
  // plus the tiles from the earliest window start of the CTA's rows
  const int W = P.window ? __ldg(P.window + h) : 0;
  const int n_total = min(p_max / TP_KT + 1, (Leff + TP_KT - 1) / TP_KT);
  int ns = 0, tw = 0;
  bool gap = false;
  if (W > 0) {
    const int kw = p_min - W + 1;
    if (kw > 0) {
      ns = (min(P.sink, Leff) + TP_KT - 1) / TP_KT;
      tw = kw / TP_KT;
      gap = tw > ns;
    }
  }
  const int n_virt = gap ? ns + (n_total - tw) : n_total;
  auto tile_of = [&](int v) { return (gap && v >= ns) ? tw + (v - ns) : v; };

  // ---- set-up: barriers, TMEM, query rows
  if (tid == 0) {
    for (int i = 0; i < C::NRAW; ++i) {
      mbar_init(bar + B_RAWFULL + i, 1);
      mbar_init(bar + B_RAWEMPTY + i, TP_PRODUCERS);
    }
    for (int i = 0; i < NKV; ++i) {
      mbar_init(bar + B_KVFULL + i, TP_PRODUCERS);
      mbar_init(bar + B_KVEMPTY + i, 1);
    }
    mbar_init(bar + B_SFULL + 0, 1);
    mbar_init(bar + B_SFULL + 1, 1);
    mbar_init(bar + B_PFULL, TP_SOFTMAX);
    mbar_init(bar + B_ODONE, 1);
    mbar_init(bar + B_DRAIN, 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar + B_EPI + i, 64);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == TP_MMA_WARP) tc::alloc(tmem_slot, C::TMEM_COLS);

  const float log2e = 1.4426950408889634f;
  const float dnorm = (MODE != MODE_INT8 && P.signs) ? (float)D : 1.0f;
  {
    constexpr int EPL = D / 32;
    uint8_t* qhi = sm + C::OFF_K;                      // [128 rows][QROW] fp16 hi
    uint8_t* qlo = sm + C::OFF_K + TP_ROWS * C::QROW;  // [128 rows][QROW] fp16 lo
    for (int r = warp; r < TP_ROWS; r += TP_THREADS / 32) {
      const int ql = r / G, i = r % G;
      const bool rv = ql < nq && KVQ_IN_BOUNDS(cq0 + q0 + ql < P.total_q, P.dev_error);  // warp-uniform
      float x[EPL];
      if (rv) {
        load_row_elems<EPL>(P.q, P.dtype, ((size_t)(cq0 + q0 + ql) * Hq + h * G + i) * D + lane * EPL, x);
        if constexpr (MODE == MODE_INT8) {
          const float* am = P.ch_amax + (size_t)h * D + lane * EPL;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x[e] *= __fdiv_rn(am[e], 127.0f);
        } else if (P.signs) {
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            if (__ldg(P.signs + lane * EPL + e) < 0) x[e] = -x[e];
          wht_warp<EPL>(x, lane);
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = 0.0f;
      }
      if (P.softmax_scale < 0.0f) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = -x[e];
      }
      float sum = 0.0f, amx = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        sum += x[e];
        amx = fmaxf(amx, fabsf(x[e]));
      }
      sum = warp_sum(sum);
      amx = warp_max(amx);
      const int ex = amx > 0.0f ? ilogbf(amx) : 0;
      const float scl = ldexpf(1.0f, 10 - ex);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int d = lane * EPL + e;
        const float v = x[e] * scl;
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        *reinterpret_cast<__half*>(qhi + r * C::QROW + 2 * d) = hi;
        *reinterpret_cast<__half*>(qlo + r * C::QROW + 2 * d) = lo;
      }
      if (lane == 0) {
        // logit = beta * (s c.q'') + gamma * z, beta > 0: a negative scale is
        // carried by q'' (negated above), a zero scale by a tiny beta
        const float sabs = fabsf(P.softmax_scale);
        rbeta[r] = fmaxf(sabs * log2e / (dnorm * scl), 1e-30f);
        rgamma[r] = sabs * log2e * sum / dnorm;
        rpos[r] = rv ? (L - n + q0 + ql) : -1;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  {
    const uint32_t tmem0 = *tmem_slot;
    // the softmax warps move the query rows into TMEM: warp w writes lanes
    // 32 (w % 4) .. + 31, half w / 4 of the columns of Q hi and of Q lo
    if (warp < TP_SOFTMAX / 32) {
      const int quad = warp & 3, hf = warp >> 2;
      const int r = quad * 32 + lane;
      const uint32_t lb = (uint32_t)(quad * 32) << 16;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const uint8_t* src = sm + C::OFF_K + part * TP_ROWS * C::QROW + r * C::QROW;
        const uint32_t col0 = (part == 0 ? C::TM_QHI : C::TM_QLO) + hf * (D / 4);
#pragma unroll 1
        for (int c = 0; c < D / 4; c += 16) {  // 16 columns = 32 dims
          uint32_t rr[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + 4 * (hf * (D / 4) + c) + 16 * j);
            rr[4 * j] = w.x;
            rr[4 * j + 1] = w.y;
            rr[4 * j + 2] = w.z;
            rr[4 * j + 3] = w.w;
          }
          tc::st16(tmem0 + lb + col0 + c, rr);
        }
      }
      tc::wait_st();
    }
  }
  tc::fence_before();
  __syncthreads();  // the query rows are in TMEM; the staging area is free again
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + C::TM_O;    // O of keys 0-31 of every tile
  const uint32_t tmem_o1 = tmem + C::TM_O1;  // O of keys 32-63

  if (warp == TP_ISSUE_WARP) {
    // ======================= raw page copies (one lane) =======================
    // Bulk copies of each tile's valid 16-row chunks into a ring of NRAW raw
    // stages, up to NRAW tiles ahead of the expansion; the page-table
    // entries are read two tiles ahead of the copies that use them.
    if (MODE == MODE_DBF16 && lane == 0) {
      // dense rows: the 64-row tile of this head per tensor, as D / 64
      // 128-byte-swizzled boxes of one 64-dim half each (tensor copies; rows
      // past the array arrive as zeros, rows of the next sequence are zeroed
      // by the producers)
      const int row0 = __ldg(P.cu_kv + b);
      int rs = 0, rphase = 0;
#pragma unroll 1
      for (int v = 0; v < n_virt; ++v) {
        if (!mbar_wait_bounded(bar + B_RAWEMPTY + rs, rphase ^ 1, TP_NAP_ISSUER) || *abort_flag) {
          *abort_flag = 1;
          flag_error(P.dev_error, DEVERR_TIMEOUT);
          break;
        }
        const int key0 = TP_KT * tile_of(v);
        const int nrows = max(0, min(TP_KT, Leff - key0));
        uint8_t* rk = sm + C::OFF_RAW + rs * 2 * C::RAW;
#pragma unroll
        for (int c = 0; c < 4; ++c) rawval[rs * 4 + c] = 16 * c < nrows ? 1 : 0;
        mbar_arrive_expect_tx(bar + B_RAWFULL + rs, (uint32_t)(2 * C::RAW));
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {  // one 64-dim half (64 swizzled lines of 128 B) per copy
          tc::tma_load_4d(rk + hh * DENSE_HALF, &P.kv_map[0], 0, hh, h, row0 + key0, bar + B_RAWFULL + rs);
          tc::tma_load_4d(rk + C::RAW + hh * DENSE_HALF, &P.kv_map[1], 0, hh, h, row0 + key0, bar + B_RAWFULL + rs);
        }
        if (++rs == C::NRAW) {
          rs = 0;
          rphase ^= 1;
        }
      }
    } else if (MODE != MODE_DBF16 && lane == 0) {
      const int trow = P.headwise ? b * Hkv + h : b;
      const int32_t* tbl = P.table + (size_t)trow * P.max_blocks;
      const size_t blk_stride = (size_t)Hkv * bs * C::R;
      const int bs_log2 = __ffs(bs) - 1;
      const uint8_t* kbase = P.k_pages + (size_t)h * bs * C::R;
      const uint8_t* vbase = P.v_pages + (size_t)h * bs * C::R;
      auto lookup = [&](int v, int (&out)[4]) {
#pragma unroll
        for (int c = 0; c < 4; ++c) out[c] = -1;
        if (v < n_virt) {
          const int key0 = TP_KT * tile_of(v);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int key = key0 + 16 * c;
            if (key < Leff) out[c] = __ldg(tbl + (key >> bs_log2));
          }
        }
      };
      int rs = 0, rphase = 0;
      // block ids of tiles v, v + 1, v + 2: each table load is issued three
      // tiles before its copies and moved between registers a tile after it
      // was issued, so no step waits on a load in flight
      int ids0[4], ids1[4], ids2[4];
      lookup(0, ids0);
      lookup(1, ids1);
      lookup(2, ids2);
#pragma unroll 1
      for (int v = 0; v < n_virt; ++v) {
        // the producers are done with this raw stage (tile v - NRAW)
        if (!mbar_wait_bounded(bar + B_RAWEMPTY + rs, rphase ^ 1, TP_NAP_ISSUER) || *abort_flag) {
          *abort_flag = 1;
          flag_error(P.dev_error, DEVERR_TIMEOUT);
          break;
        }
        const int key0 = TP_KT * tile_of(v);
        uint8_t* rk = sm + C::OFF_RAW + rs * 2 * C::RAW;
        uint8_t* rvp = rk + C::RAW;
        int valid = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (ids0[c] >= P.num_blocks) {
            flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
            ids0[c] = -1;
          }
          // the chunk's 16 rows lie inside the pool (kbase is head h's first page)
          if (ids0[c] >= 0 &&
              !KVQ_IN_BOUNDS((size_t)h * bs * C::R + (size_t)ids0[c] * blk_stride +
                                     (size_t)((key0 + 16 * c) & (bs - 1)) * C::R + C::CHUNK <=
                                 (size_t)P.num_blocks * P.num_kv_heads * bs * C::R,
                             P.dev_error))
            ids0[c] = -1;
          if (ids0[c] >= 0) valid |= 1 << c;
          rawval[rs * 4 + c] = ids0[c] >= 0 ? 1 : 0;
        }
        mbar_arrive_expect_tx(bar + B_RAWFULL + rs, (uint32_t)(__popc(valid) * 2 * C::CHUNK));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if ((valid >> c) & 1) {
            const int key = key0 + 16 * c;
            const size_t off = (size_t)ids0[c] * blk_stride + (size_t)(key & (bs - 1)) * C::R;
            bulk_g2s(rk + c * C::CHUNK, kbase + off, C::CHUNK, bar + B_RAWFULL + rs);
            bulk_g2s(rvp + c * C::CHUNK, vbase + off, C::CHUNK, bar + B_RAWFULL + rs);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ids0[c] = ids1[c];
          ids1[c] = ids2[c];
        }
        lookup(v + 3, ids2);
        if (++rs == C::NRAW) {
          rs = 0;
          rphase ^= 1;
        }
      }
    }
    __syncwarp();
  } else if (warp >= TP_PROD_WARP0) {
    // ======================= producers: code expansion =======================
    const int pt = tid - TP_PROD_WARP0 * 32;  // 0..127
    const int pwarp = warp - TP_PROD_WARP0;
    int kvs = 0, kv_phase = 0;  // K/V stage of tile v and its wrap count parity
    int rs = 0, rphase = 0;     // raw stage of tile v
#pragma unroll 1
    for (int v = 0; v < n_virt; ++v) {
      // raw tile v has landed; the tensor cores are done with this K/V stage
      const bool late = !mbar_wait_bounded(bar + B_RAWFULL + rs, rphase, TP_NAP_PRODUCER) ||
                        !mbar_wait_bounded(bar + B_KVEMPTY + kvs, kv_phase ^ 1, TP_NAP_PRODUCER);
      if (late || *abort_flag) {
        *abort_flag = 1;
        flag_error(P.dev_error, DEVERR_TIMEOUT);
        break;
      }
      const int key0 = TP_KT * tile_of(v);
      const int vmask = rawval[rs * 4 + 0] | (rawval[rs * 4 + 1] << 1) | (rawval[rs * 4 + 2] << 2) |
                        (rawval[rs * 4 + 3] << 3);
      if (pt < 4) kval[kvs * 4 + pt] = (vmask >> pt) & 1;
      const uint8_t* rk = sm + C::OFF_RAW + rs * 2 * C::RAW;
      const uint8_t* rvp = rk + C::RAW;
      uint8_t* kt = sm + C::OFF_K + kvs * C::KTILE;
      uint8_t* vt = sm + C::OFF_VT + kvs * C::VTILE;
      // K: key rows, 8 dims per 16-byte chunk (rows of skipped chunks hold
      // stale bytes: finite codes, masked in the softmax)
      {
        // thread pt always expands the same 8 dims (c8) of keys pt / (D/8) + step * j
        constexpr int ITEMS = TP_KT * (D / 8) / TP_PRODUCERS;
        constexpr int KSTEP = TP_PRODUCERS / (D / 8);
        static_assert(TP_KT * (D / 8) % TP_PRODUCERS == 0 && TP_PRODUCERS % (D / 8) == 0, "K expansion split");
        const int c8 = pt % (D / 8), key_0 = pt / (D / 8);
        const uint8_t* src = rk + key_0 * C::R;
        uint8_t* dst = kt + (c8 >> 3) * C::KATOM;
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
          const int key = key_0 + KSTEP * j;
          uint4 hv;
          if constexpr (MODE == MODE_DBF16) hv = dense_codes8(rk, key, c8);
          else hv = codes8<MODE>(src + KSTEP * j * C::R, c8);
          if (MODE == MODE_DBF16 && key0 + key >= Leff) hv = make_uint4(0u, 0u, 0u, 0u);  // not copied
          *reinterpret_cast<uint4*>(dst + tc::sw128_off(key, c8 & 7)) = hv;
        }
      }
      // V^T: 8 keys x 32 dims per stmatrix (four 8x8 blocks, stored transposed)
      {
        const int g8 = lane >> 2, t4 = lane & 3;
        constexpr int JOBS = (TP_KT / 8) * (D / 32);
        constexpr int PW = TP_PRODUCERS / 32;
        static_assert(JOBS % PW == 0, "V expansion split");
#pragma unroll
        for (int jj = 0; jj < JOBS / PW; ++jj) {
          const int job = pwarp + PW * jj;
          const int kb = job % (TP_KT / 8), db = job / (TP_KT / 8);  // key block, 32-dim block
          const uint8_t* row = rvp + (8 * kb + g8) * C::R;
          uint32_t r4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (MODE == MODE_DBF16) r4[i] = dense_codes2(rvp, 8 * kb + g8, 32 * db + 8 * i + 2 * t4);
            else r4[i] = codes2<MODE>(row, 32 * db + 8 * i + 2 * t4);
          }
          if (MODE == MODE_DBF16 && key0 + 8 * kb + g8 >= Leff) {  // not copied: stale bytes could be NaN
#pragma unroll
            for (int i = 0; i < 4; ++i) r4[i] = 0u;
          }
          const int mi = lane >> 3, rr = lane & 7;
          const int d = 32 * db + 8 * mi + rr;  // stored row of matrix mi
          tc::stsm_x4_t(smem_addr(vt + tc::sw128_off(d, kb)), r4[0], r4[1], r4[2], r4[3]);
        }
      }
      if constexpr (MODE != MODE_INT8) {
        // per-key scale and zero point; 0 for keys without data (skipped
        // chunks, rows past the sequence) so that masked keys add exact zeros
        for (int idx = pt; idx < 2 * TP_KT; idx += TP_PRODUCERS) {
          const int key = idx & (TP_KT - 1);
          const bool isv = idx >= TP_KT;
          const bool has = ((vmask >> (key >> 4)) & 1) && key0 + key < Leff;
          float s = 0.0f, z = 0.0f;
          if (has) {
            if constexpr (MODE == MODE_DBF16) {
              s = 1.0f;  // dense values: no scale, no zero point
            } else {
              const uint32_t pad = lds32((isv ? rvp : rk) + key * C::R + C::DATA);
              pad_scale_zero<MODE>(pad, P.stego != 0, s, z);  // z: the value of the signed code 0
            }
          }
          float* scs = sc + kvs * 4 * TP_KT;
          scs[(isv ? 2 : 0) * TP_KT + key] = s;
          scs[(isv ? 3 : 1) * TP_KT + key] = z;
        }
      }
      tc::mbar_arrive(bar + B_RAWEMPTY + rs);  // this thread is done reading the raw stage
      tc::fence_proxy_async();
      tc::mbar_arrive(bar + B_KVFULL + kvs);
      if (++kvs == NKV) {
        kvs = 0;
        kv_phase ^= 1;
      }
      if (++rs == C::NRAW) {
        rs = 0;
        rphase ^= 1;
      }
    }
  } else if (warp == TP_MMA_WARP) {
    // ======================= MMA issue =======================
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_f16(TP_ROWS, TP_KT);
      const uint32_t idesc_pv = tc::idesc_f16(TP_ROWS, D);
      // O0 += P V over the tile's keys 0-31 and O1 over keys 32-63, with P
      // (hi / lo interleaved per 16 keys, where the tile's S was) from TMEM
      // and V^T from shared memory
      auto pv = [&](int i, int kvs_i) -> bool {
        if (!mbar_wait_bounded(bar + B_PFULL, i & 1, TP_NAP_MMA)) return false;
        tc::fence_after();
        const uint32_t a_vt = smem_addr(sm + C::OFF_VT + kvs_i * C::VTILE);
        const uint32_t p_tm = tmem + (i & 1) * TP_KT;
#pragma unroll
        for (int kk = 0; kk < TP_KT / 16; ++kk) {
          const uint64_t bdesc = tc::sw128_desc(a_vt + 32 * kk);
          const uint32_t o_tm = kk < TP_KT / 32 ? tmem_o : tmem_o1;
          tc::mma_f16_ts(o_tm, p_tm + 16 * kk, bdesc, idesc_pv, (i > 0 || (kk % (TP_KT / 32)) > 0) ? 1u : 0u);
          tc::mma_f16_ts(o_tm, p_tm + 16 * kk + 8, bdesc, idesc_pv, 1u);
        }
        tc::commit(bar + B_ODONE);
        tc::commit(bar + B_KVEMPTY + kvs_i);
        return true;
      };
      bool ok = true;
      int kvs = 0, kv_phase = 0, kvs_prev = 0;
#pragma unroll 1
      for (int v = 0; v < n_virt && ok; ++v) {
        const int st = v & 1;
        // S(v) goes where P(v - 2) was: P.V(v - 2) was issued before it and
        // the tensor cores run this thread's MMAs in order
        if (!mbar_wait_bounded(bar + B_KVFULL + kvs, kv_phase, TP_NAP_MMA)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t a_k = smem_addr(sm + C::OFF_K + kvs * C::KTILE);
        const uint32_t s_tm = tmem + st * TP_KT;
#pragma unroll
        for (int s = 0; s < C::KSTEPS; ++s) {
          const uint64_t bdesc = tc::sw128_desc(a_k + (s >> 2) * C::KATOM + (s & 3) * 32);
          tc::mma_f16_ts(s_tm, tmem + C::TM_QHI + 8 * s, bdesc, idesc_qk, s > 0 ? 1u : 0u);
          tc::mma_f16_ts(s_tm, tmem + C::TM_QLO + 8 * s, bdesc, idesc_qk, 1u);
        }
        tc::commit(bar + B_SFULL + st);
        if (v >= 1) ok = pv(v - 1, kvs_prev);
        if (*abort_flag) ok = false;
        kvs_prev = kvs;
        if (++kvs == NKV) {
          kvs = 0;
          kv_phase ^= 1;
        }
      }
      if (ok && n_virt >= 1) ok = pv(n_virt - 1, kvs_prev);
      if (!ok) {
        *abort_flag = 1;
        flag_error(P.dev_error, DEVERR_TIMEOUT);
      }
      // drain: every MMA issued by this thread has completed
      tc::commit(bar + B_DRAIN);
      (void)mbar_wait_bounded(bar + B_DRAIN, 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax =======================
    // Row r is shared by warps r / 32 (keys 0-31 of each tile) and r / 32 + 4
    // (keys 32-63), which may both read TMEM lanes 32 (w % 4) ...  Each half
    // is an online softmax of its own over its keys, with its own maximum,
    // sums and O accumulator.  Per tile it makes two passes over its 32
    // logits (two 16-key chunks, kept in registers between the passes):
    // pass 1 forms y = s c.q'' + rho z (rho = gamma / beta), masks it and
    // takes the maximum; pass 2 forms p = 2^(beta y - m) and writes (p s)
    // hi / lo of its 32 keys to P, over the tile's S columns.
    const int quad = warp & 3, hf = warp >> 2;
    const int r = quad * 32 + lane;
    const float rb = rbeta[r];
    const float rho = rgamma[r] / rb;
    const int rp = rpos[r];
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tmem_oh = hf ? tmem_o1 : tmem_o;  // this half's O
    float* xmax = reinterpret_cast<float*>(sm + C::OFF_XMAX);
    float mrow = -CUDART_INF_F, lrow = 0.0f, pzrow = 0.0f;  // lrow, pzrow: this half's keys
    bool ok = true;
    int kvs = 0;
#pragma unroll 1
    for (int v = 0; v < n_virt; ++v) {
      const int st = v & 1;
      const int T = tile_of(v);
      // every decision around a .sync.aligned TMEM access is warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_SFULL + st, (v >> 1) & 1, TP_NAP_SOFTMAX))) {
        ok = false;
        break;
      }
      tc::fence_after();
      const float4* s4 = reinterpret_cast<const float4*>(sc + kvs * 4 * TP_KT);  // ks, kz, vs, vz: 16 float4 each
      const int kv4 = kval[kvs * 4 + 0] | (kval[kvs * 4 + 1] << 1) | (kval[kvs * 4 + 2] << 2) | (kval[kvs * 4 + 3] << 3);
      const int key0 = TP_KT * T;
      const bool full = kv4 == 15 && key0 + TP_KT - 1 <= rp && key0 + TP_KT <= Leff &&
                        (W <= 0 || key0 > rp - W || key0 + TP_KT <= P.sink);
      const bool all_full = __all_sync(0xffffffffu, full);
      const uint32_t s_col = tmem + lane_base + st * TP_KT;
      float ymax = -CUDART_INF_F;
      uint32_t yy[2][16];  // this half's 32 logits y, kept for pass 2
      tc::ld16(s_col + 16 * (2 * hf), yy[0]);
      tc::ld16(s_col + 16 * (2 * hf + 1), yy[1]);
      tc::wait_ld();
      tc::regs_after_wait(yy[0]);
      tc::regs_after_wait(yy[1]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hf + cc;
        uint32_t (&rr)[16] = yy[cc];
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          float4 ks = make_float4(0.f, 0.f, 0.f, 0.f), kz = ks;
          if constexpr (MODE != MODE_INT8) {
            ks = s4[4 * c + j4];
            kz = s4[16 + 4 * c + j4];
          }
          const float ksv[4] = {ks.x, ks.y, ks.z, ks.w}, kzv[4] = {kz.x, kz.y, kz.z, kz.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jj = 4 * j4 + e;
            const float dot = __uint_as_float(rr[jj]);
            rr[jj] = __float_as_uint(MODE == MODE_INT8 ? dot : fmaf(ksv[e], dot, rho * kzv[e]));
          }
        }
        if (!all_full) {  // warp-uniform: masks only where some row of the warp needs them
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = key0 + 16 * c + jj;
            bool vis = ((kv4 >> c) & 1) && j <= rp && j < Leff;
            if (W > 0) vis = vis && (j < P.sink || j > rp - W);
            if (!vis) rr[jj] = __float_as_uint(-CUDART_INF_F);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) ymax = fmaxf(ymax, __uint_as_float(rr[jj]));
      }
      // lazy rescale: keep the reference maximum until the row's maximum
      // over this half's keys passes it by more than 2^TP_SLACK
      const float tmax = rb * ymax;
      const bool grow = tmax > mrow + TP_SLACK;
      const float mref = grow ? tmax : mrow;
      const float muse = mref == -CUDART_INF_F ? 0.0f : mref;
      // the previous P.V must be done before O is rescaled (this wait also
      // keeps the softmax within one tile of the MMA warp's P barrier)
      if (v >= 1 && !__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_ODONE, (v - 1) & 1, TP_NAP_SOFTMAX))) {
        ok = false;
        break;
      }
      const bool resc = v >= 1 && grow && mrow != -CUDART_INF_F;
      if (__any_sync(0xffffffffu, resc)) {  // this half's O; rows keeping their reference scale by 1
        tc::fence_after();
        const float f = resc ? ex2(mrow - muse) : 1.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ra[16], rb2[16];
          tc::ld16(tmem_oh + lane_base + c0, ra);
          tc::ld16(tmem_oh + lane_base + c0 + 16, rb2);
          tc::wait_ld();
          tc::regs_after_wait(ra);
          tc::regs_after_wait(rb2);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            ra[j] = __float_as_uint(__uint_as_float(ra[j]) * f);
            rb2[j] = __float_as_uint(__uint_as_float(rb2[j]) * f);
          }
          tc::st16(tmem_oh + lane_base + c0, ra);
          tc::st16(tmem_oh + lane_base + c0 + 16, rb2);
        }
        tc::wait_st();
        lrow *= f;
        pzrow *= f;
      }
      mrow = mref;
      float tl = 0.0f, tpz = 0.0f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hf + cc;
        const uint32_t (&rr)[16] = yy[cc];
        uint32_t pw[16];  // P hi (8 columns) then P lo (8 columns) of these 16 keys
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          float4 vs = make_float4(1.f, 1.f, 1.f, 1.f), vz = make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (MODE != MODE_INT8) {
            vs = s4[32 + 4 * c + j4];
            vz = s4[48 + 4 * c + j4];
          }
          const float vsv[4] = {vs.x, vs.y, vs.z, vs.w}, vzv[4] = {vz.x, vz.y, vz.z, vz.w};
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            float w2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = 4 * j4 + 2 * e2 + e;
              const float p = ex2(fmaf(rb, __uint_as_float(rr[jj]), -muse));
              tl += p;
              if constexpr (MODE != MODE_INT8) tpz = fmaf(p, vzv[2 * e2 + e], tpz);
              w2[e] = MODE != MODE_INT8 ? p * vsv[2 * e2 + e] : p;
            }
            const __half2 hp = __floats2half2_rn(w2[0], w2[1]);
            const float2 hf2 = __half22float2(hp);
            const __half2 lp = __floats2half2_rn(w2[0] - hf2.x, w2[1] - hf2.y);
            pw[2 * j4 + e2] = *reinterpret_cast<const uint32_t*>(&hp);
            pw[8 + 2 * j4 + e2] = *reinterpret_cast<const uint32_t*>(&lp);
          }
        }
        tc::st16(s_col + 16 * c, pw);  // over the 16 y values just read
      }
      tc::wait_st();
      lrow += tl;
      pzrow += tpz;
      tc::fence_before();
      tc::mbar_arrive(bar + B_PFULL);
      if (++kvs == NKV) kvs = 0;
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        ok = false;
        break;
      }
    }
    // ---- epilogue: the pair's two halves merge (each weighted by 2^(its
    // maximum - the row's), half 0 staging its O in shared memory and half 1
    // adding its own), then per row a warp applies the zero-point term, the
    // inverse RHT (or the INT8 V channel scales) and 1 / l and stores the row
    // with coalesced writes.  Both warps of a pair pass the same three phases
    // of B_EPI + quad, whatever their status, so neither waits on a partner
    // that left; every wait is bounded.
    if (ok && n_virt >= 1 && !__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_ODONE, (n_virt - 1) & 1)))
      ok = false;
    float4* stage = reinterpret_cast<float4*>(sm + C::OFF_K);  // [128 rows][D / 4], piece j at j ^ (row & 7)
    float* xsum = reinterpret_cast<float*>(sm + C::OFF_RAW);    // [l, pz, ok half 0, ok half 1][128]
    constexpr int P4 = D / 4;
    xmax[hf * TP_ROWS + r] = mrow;
    xsum[(2 + hf) * TP_ROWS + r] = ok ? 1.0f : 0.0f;
    tc::mbar_arrive(bar + B_EPI + quad);
    bool good = mbar_wait_bounded(bar + B_EPI + quad, 0);
    good = __all_sync(0xffffffffu, ok && good && xsum[(2 + (hf ^ 1)) * TP_ROWS + r] != 0.0f);
    const float mrr = fmaxf(mrow, xmax[(hf ^ 1) * TP_ROWS + r]);
    const float fw = mrow == -CUDART_INF_F ? 0.0f : ex2(mrow - mrr);  // 0 for a half without visible keys
#pragma unroll 1
    for (int ph = 0; ph < 2; ++ph) {
      if (good && hf == ph) {  // every P.V is done: the K / V^T stages are free for staging
        xsum[0 * TP_ROWS + r] = (ph ? xsum[0 * TP_ROWS + r] : 0.0f) + fw * lrow;
        xsum[1 * TP_ROWS + r] = (ph ? xsum[1 * TP_ROWS + r] : 0.0f) + (MODE != MODE_INT8 ? fw * pzrow : 0.0f);
        if (n_virt >= 1) {  // whole warp reads its 32 TMEM rows, valid or not
          tc::fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ra[16], rb2[16];
            tc::ld16(tmem_oh + lane_base + c0, ra);
            tc::ld16(tmem_oh + lane_base + c0 + 16, rb2);
            tc::wait_ld();
            tc::regs_after_wait(ra);
            tc::regs_after_wait(rb2);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t* w = j < 4 ? ra + 4 * j : rb2 + 4 * (j - 4);
              float4& dst = stage[r * P4 + ((c0 / 4 + j) ^ (r & 7))];
              const float4 prev = ph ? dst : make_float4(0.f, 0.f, 0.f, 0.f);
              dst = make_float4(fmaf(fw, __uint_as_float(w[0]), prev.x), fmaf(fw, __uint_as_float(w[1]), prev.y),
                                fmaf(fw, __uint_as_float(w[2]), prev.z), fmaf(fw, __uint_as_float(w[3]), prev.w));
            }
          }
        } else if (ph == 0) {
          for (int j = 0; j < P4; ++j) stage[r * P4 + j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      tc::mbar_arrive(bar + B_EPI + quad);  // half ph has staged (or failed)
      good = __all_sync(0xffffffffu, mbar_wait_bounded(bar + B_EPI + quad, (ph + 1) & 1) && good);
    }
    if (!good) {
      *abort_flag = 1;
      if (lane == 0) flag_error(P.dev_error, DEVERR_TIMEOUT);
    } else {
      constexpr int EPL = D / 32;  // lane holds dims lane * EPL .. + EPL - 1
      for (int k = 16 * hf; k < 16 * hf + 16; ++k) {
        const int row = quad * 32 + k;
        const int ql = row / G, i = row % G;
        if (ql >= nq) continue;  // warp-uniform
        const float lr = xsum[0 * TP_ROWS + row];
        const float pz = xsum[1 * TP_ROWS + row];
        float o[EPL];
        const float* src = reinterpret_cast<const float*>(stage + row * P4 + ((lane * EPL / 4) ^ (row & 7))) +
                           (lane * EPL) % 4;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = src[e] + pz;
        if (lr == 0.0f) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
        } else if constexpr (MODE != MODE_INT8) {
          if (P.signs) {
            wht_warp<EPL>(o, lane);
            const float inv = 1.0f / ((float)D * lr);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = (__ldg(P.signs + lane * EPL + e) < 0 ? -o[e] : o[e]) * inv;
          } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] /= lr;
          }
        } else {
          const float* am = P.ch_amax + ((size_t)Hkv + h) * D + lane * EPL;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] = o[e] * __fdiv_rn(am[e], 127.0f) / lr;
        }
        float* orow = P.out + ((size_t)(cq0 + q0 + ql) * Hq + h * G + i) * D + lane * EPL;
        if (KVQ_IN_BOUNDS(cq0 + q0 + ql < P.total_q, P.dev_error)) {
          if constexpr (EPL == 4) {
            *reinterpret_cast<float4*>(orow) = make_float4(o[0], o[1], o[2], o[3]);
          } else {
            *reinterpret_cast<float2*>(orow) = make_float2(o[0], o[1]);
          }
        }
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == TP_MMA_WARP) {
    tc::fence_after();
    tc::dealloc(tmem, C::TMEM_COLS);
  }
}

template <int MODE, int D>
cudaError_t launch_prefill_tc_t(const AttnParams& P, cudaStream_t stream) {
  using C = TpCfg<MODE, D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<MODE, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid((unsigned)prefill_grid_x(P.max_q_per_seq, P.group), P.num_kv_heads, P.batch);  // TP_THREADS threads each
  prefill_tc_kernel<MODE, D><<<grid, TP_THREADS, C::SMEM, stream>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnParams& P, cudaStream_t stream) {
  switch (P.mode * 1000 + P.head_dim) {
    case MODE_INT4 * 1000 + 128: return launch_prefill_tc_t<MODE_INT4, 128>(P, stream);
    case MODE_INT4 * 1000 + 64: return launch_prefill_tc_t<MODE_INT4, 64>(P, stream);
    case MODE_INT2 * 1000 + 128: return launch_prefill_tc_t<MODE_INT2, 128>(P, stream);
    case MODE_INT2 * 1000 + 64: return launch_prefill_tc_t<MODE_INT2, 64>(P, stream);
    case MODE_INT8 * 1000 + 128: return launch_prefill_tc_t<MODE_INT8, 128>(P, stream);
    case MODE_INT8 * 1000 + 64: return launch_prefill_tc_t<MODE_INT8, 64>(P, stream);
    case MODE_I8T * 1000 + 128: return launch_prefill_tc_t<MODE_I8T, 128>(P, stream);
    case MODE_I8T * 1000 + 64: return launch_prefill_tc_t<MODE_I8T, 64>(P, stream);
    case MODE_F8T * 1000 + 128: return launch_prefill_tc_t<MODE_F8T, 128>(P, stream);
    case MODE_F8T * 1000 + 64: return launch_prefill_tc_t<MODE_F8T, 64>(P, stream);
    case MODE_DBF16 * 1000 + 128: return launch_prefill_tc_t<MODE_DBF16, 128>(P, stream);
    case MODE_DBF16 * 1000 + 64: return launch_prefill_tc_t<MODE_DBF16, 64>(P, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
