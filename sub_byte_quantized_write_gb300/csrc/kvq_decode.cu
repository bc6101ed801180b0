// kvq_decode.cu -- split-KV decode attention over the paged low-bit cache.
//
// What it computes: for every sequence b and q head hq, softmax attention of
// the decode query (position seq_lens[b]-1) over the visible cached keys,
// with keys and values read from INT4 / INT2 / INT8 / FP8 pages, dequantised
// and mapped back through the inverse RHT.  Sources (page title, section):
// vLLM PR #40835 review summary ("INT4 per-token-head KV cache for the Triton
// backend"), 实现拆解 item 2 (read kernel: unpack, dequantise, attention);
// FastDeploy PR #7718 "Optimize AppendAttention for discrete head-wise
// block_idx", Motivation and PR2-only delta table (per-head table rows, the
// -1 sentinel is skipped before any page address is formed, sink tokens);
// vllm-ascend-quantized-kv-cache METADATA ("Ascend INT8 KV Cache Plugin"),
// 运行机制 (decode dequantises inside the attention kernel).
//
// Design (GB300), three kernels per call, chained by programmatic dependent
// launch:
//  1. decode_prep_kernel: one CTA per (sequence, kv head) pair: the query
//     operand images (q' = H (d * q) split fp16 hi / lo, in the lane order of
//     the MMA operand) and the per-head logit constants, including the
//     constant the folded key unpack adds (INT4: 72 per dim; INT2: 66, 18 or
//     6 by the dim's crumb position).  With kvq_write_decode_attn it also
//     quantises and stores the step's new K / V rows of its pair, after the
//     kernels before it are done with the pools.
//  2. decode_tma_kernel (INT4 / INT2 / 8-bit token-head rows): persistent
//     warps, one CTA of 12 warps per SM for GQA groups up to 4 (two CTAs of 4
//     for groups up to 8).  The concatenated tile lists of all pairs (64-key tiles for the
//     4-bit and 2-bit rows at groups up to 4, else 32) are cut into one
//     contiguous, equal slice per warp ("stream-K"), balanced to within a tile
//     whatever the context lengths.  Each tile's K and V rows arrive by one
//     cp.async.bulk.tensor ... tile::gather4 copy each: the pool is viewed as
//     a 2-D tensor whose rows are page chunks of KT/4 key rows, so the tile's
//     four chunks (from four pages anywhere in the pool) are four row
//     coordinates of one copy, into the warp's ring of mbarrier-tracked
//     stages.  Lanes 0-3 look up the next tile's table entries one tile ahead;
//     a -1 entry or a chunk past the sequence points the copy at row 0 and is
//     masked, never turned into the page's own address.  Full tiles run a
//     body without masks.  CTA 0 publishes each pair's first tile for the
//     merge.  decode_stream_kernel (INT8 per channel) is the same algorithm
//     over 16-byte cp.async pieces with XOR-swizzled rows and its own scan.
//  3. decode_reduce_kernel: per (sequence, q head) the log-sum-exp merge of
//     the partials of the warps whose slices cover the pair, the inverse RHT
//     and 1 / l.
// The RHT and the dequantisation are folded into the query and the weights:
//   q . k_j = (s_j (q' . c_j) + z_j sum(q')) / D,   q' = H (d * q)
//   sum_j P_j v_j = d * H( sum_j (P_j s_j) c_j + sum_j P_j z_j ) / D
// with the signed code c = u - 2^(b-1) and z = m + 2^(b-1) s (the value of
// code 2^(b-1)); INT8 / FP8 token-head rows have c the stored code (an E4M3
// value for FP8) and z = 0.  So the hot loop multiplies codes (exact small integers in fp16) on
// the tensor cores: QK^T as m16n8k16 with M = 16 keys and N = 8 slots (4 q
// heads of the GQA group x {hi, lo} halves of q'), and P.V as m16n8k16 with
// M = 16 head dims, K = 16 keys, N = the same 8 slots of (P s) hi / lo.
// Splitting q' and (P s) into two fp16 terms keeps ~22 significant bits, so
// the fp16 operands do not limit accuracy.  Signed (centred) codes keep the
// fp32 accumulators small: with unsigned codes the P.V accumulator and the
// zero-point sum grow large with opposite signs and their rounding errors no
// longer cancel over tens of thousands of keys.

#include <math_constants.h>

#include <type_traits>

#include "kvq_internal.h"
#include "kvq_row.cuh"

namespace kvq {

template <int MODE, int D>
struct DecCfg {
  static constexpr int BITS = mode_bits(MODE);
  static constexpr int DATA = data_bytes(MODE, D);
  static constexpr int R = row_bytes_of(MODE, D);
  static constexpr int CHUNK = 16 * R;     // one 16-row chunk of a page
  static constexpr int TILE = 2 * CHUNK;   // 32 key rows of K (or V)
  static constexpr int STAGE = 2 * TILE;   // K tile then V tile
  static constexpr int NSTAGE = MODE == MODE_INT4 ? 4 : (MODE == MODE_INT2 ? 6 : 3);
  static constexpr int KSTEPS = D / 16;    // k16 steps of QK^T
  static constexpr int MT = D / 16;        // m16 tiles of P.V (rows = head dims)
  static constexpr int CPW = 32 / BITS;    // codes per 32-bit word
  static constexpr int KPW = CPW / 4;      // k-steps fed by one word of a key row
  static constexpr int WPL = KSTEPS / KPW; // words each lane reads per key row
  static constexpr int BPL = D * BITS / 128;  // bytes of a lane's V range (D/16 codes)
  static constexpr int PPR = D / 16;       // 16-byte pieces per INT8 row
};

// Byte offset of (row kappa, byte) inside a 32-row INT8 tile whose 16-byte
// pieces are XOR-swizzled by row so that lanes reading different rows hit
// different banks.
template <int D>
__device__ __forceinline__ int swz(int kappa, int byte) {
  constexpr int PPR = D / 16;
  return kappa * D + 16 * ((byte >> 4) ^ ((kappa >> 2) & (PPR - 1))) + (byte & 15);
}

template <int MODE, int D>
__device__ __forceinline__ uint32_t load_kword(const uint8_t* tile, int kappa, int w) {
  using C = DecCfg<MODE, D>;
  if constexpr (MODE == MODE_INT8) return lds32(tile + swz<D>(kappa, 4 * w));
  else return lds32(tile + kappa * C::R + 4 * w);
}

// The lane's range of D/16 consecutive codes (bytes gidx*BPL ...) of row kappa,
// shifted so that the first code sits at bit 0.
template <int MODE, int D>
__device__ __forceinline__ uint2 load_range(const uint8_t* tile, int kappa, int gidx) {
  using C = DecCfg<MODE, D>;
  const int off = gidx * C::BPL;
  if constexpr (MODE == MODE_INT8) {
    const uint8_t* p = tile + swz<D>(kappa, off);
    if constexpr (C::BPL == 8) return lds64(p);
    else return make_uint2(lds32(p), 0u);
  } else {
    const uint8_t* row = tile + kappa * C::R;
    if constexpr (C::BPL == 8) {  // 8-bit token-head rows: D + 4 bytes, 4-byte aligned
      return make_uint2(lds32(row + off), lds32(row + off + 4));
    } else if constexpr (C::BPL >= 4) {
      return make_uint2(lds32(row + off), 0u);
    } else {
      const uint32_t w = lds32(row + (off & ~3));
      return make_uint2(w >> (8 * (off & 3)), 0u);
    }
  }
}

// fp16 bit pattern of (magic + bias) in both halves, where `magic` places a
// code's lowest bit at bit `pos` of a half with weight 1 (1024, 256, 64, 16
// for pos 0, 2, 4, 6): OR-ing the code in gives magic + u exactly, and one
// sub.f16x2 with this value leaves the SIGNED code u - bias exactly.
__host__ __device__ constexpr uint32_t magic_minus(uint32_t magic_half, int pos, int bias) {
  return (magic_half | ((uint32_t)bias << pos)) * 0x00010001u;
}

// Two codes of one key row as an exact fp16 pair of signed codes
// q = u - 2^(b-1) (INT4 [-8, 7], INT2 [-2, 1], INT8 as stored, FP8 the E4M3
// value).  Pair P of
// word w holds head dims (d0, d1) = INT4 (8w+P, 8w+P+4), INT2 (16w+P,
// 16w+P+8), INT8 (4w+2P, 4w+2P+1); kpair_dims gives the same map for the
// query side.
template <int MODE, int P>
__device__ __forceinline__ uint32_t kpair(uint32_t w) {
  if constexpr (MODE == MODE_INT4) {
    constexpr int pos = (P & 1) ? 4 : 0;
    constexpr uint32_t mask = 0x000F000Fu << pos;
    constexpr uint32_t magic = (P & 1) ? 0x54005400u : 0x64006400u;  // 64 + u, 1024 + u
    const uint32_t src = (P >= 2) ? (w >> 8) : w;
    return hsub2_bits(lop3_and_or(src, mask, magic), magic_minus(magic & 0xFFFF, pos, 8));
  } else if constexpr (MODE == MODE_INT2) {
    constexpr int q = P & 3;
    constexpr uint32_t mask = 0x00030003u << (2 * q);
    constexpr uint32_t magic = q == 0 ? 0x64006400u : q == 1 ? 0x5C005C00u : q == 2 ? 0x54005400u : 0x4C004C00u;
    const uint32_t src = (P >= 4) ? (w >> 8) : w;
    return hsub2_bits(lop3_and_or(src, mask, magic), magic_minus(magic & 0xFFFF, 2 * q, 2));
  } else if constexpr (MODE == MODE_F8T) {
    return e4m3x2_to_half2_bits(w >> (16 * P));
  } else {
    constexpr uint32_t sel = (2 * P) | (4 << 4) | ((2 * P + 1) << 8) | (4 << 12);
    const uint32_t x = prmt(w, 0u, sel);
    return hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);  // 1152 + q - 1152
  }
}

// INT4 key pairs without the subtraction: every nibble is moved to bits 4-7
// of its half and OR-ed into 64.0, giving 64 + u = 72 + (u - 8) exactly; the
// constant 72 * sum(q'') per head is removed after the dot product (the
// query side supplies it).  Same pair-to-dims map as kpair.
template <int P>
__device__ __forceinline__ uint32_t kpair_int4_fold(uint32_t w) {
  const uint32_t src = P == 0 ? (w << 4) : P == 1 ? w : P == 2 ? (w >> 4) : (w >> 8);
  return lop3_and_or(src, 0x00F000F0u, 0x54005400u);
}
constexpr float KFOLD_INT4 = 72.0f;

// INT2 key pairs without the subtraction: crumb P of each half goes to bit 4,
// 6 or 8 of the half (from w << 4, w or w >> 6) and is OR-ed into 64, 16 or 4,
// the value whose unit in the last place puts weight 1 on that bit: M_P + u
// exactly, with M_P at most 64 so that the folded constant stays small next
// to the products.  Pair P holds head dims 16w+P and 16w+P+8 (as kpair).
template <int P>
__device__ __forceinline__ uint32_t kpair_int2_fold(uint32_t w) {
  constexpr int pos = (P == 0 || P == 2 || P == 5) ? 4 : (P == 1 || P == 3 || P == 6) ? 6 : 8;
  constexpr uint32_t magic = pos == 4 ? 0x54005400u : pos == 6 ? 0x4C004C00u : 0x44004400u;  // 64, 16, 4
  const uint32_t src = P <= 1 ? (w << 4) : P <= 4 ? w : (w >> 6);
  return lop3_and_or(src, 0x00030003u << pos, magic);
}
// M_P + 2 for the head dim d (P = d mod 8): what the folded INT2 key value
// adds to the signed code u - 2.
__host__ __device__ constexpr float kfold_int2(int d) {
  return (d & 7) == 4 || (d & 7) == 7 ? 6.0f : ((d & 7) == 1 || (d & 7) == 3 || (d & 7) == 6) ? 18.0f : 66.0f;
}

template <int MODE>
__device__ __forceinline__ void kpair_dims(int w, int P, int& d0, int& d1) {
  if (MODE == MODE_INT4) { d0 = 8 * w + P; d1 = d0 + 4; }
  else if (MODE == MODE_INT2) { d0 = 16 * w + P; d1 = d0 + 8; }
  else { d0 = 4 * w + 2 * P; d1 = d0 + 1; }
}

// Code C of the lane ranges of two keys (A: key e=0, B: key e=1) as an exact
// fp16 pair of signed codes (A's code in the low half).
template <int MODE, int C>
__device__ __forceinline__ uint32_t vpair(uint2 A, uint2 B) {
  if constexpr (MODE == MODE_INT4) {
    constexpr int byte = C / 2;
    constexpr uint32_t sel = byte | (byte << 4) | ((4 + byte) << 8) | ((4 + byte) << 12);
    const uint32_t x = prmt(A.x, B.x, sel);
    constexpr int pos = (C & 1) ? 4 : 0;
    constexpr uint32_t mask = 0x000F000Fu << pos;
    constexpr uint32_t magic = (C & 1) ? 0x54005400u : 0x64006400u;
    return hsub2_bits(lop3_and_or(x, mask, magic), magic_minus(magic & 0xFFFF, pos, 8));
  } else if constexpr (MODE == MODE_INT2) {
    constexpr int byte = C / 4, q = C % 4;
    constexpr uint32_t sel = byte | (byte << 4) | ((4 + byte) << 8) | ((4 + byte) << 12);
    const uint32_t x = prmt(A.x, B.x, sel);
    constexpr uint32_t mask = 0x00030003u << (2 * q);
    constexpr uint32_t magic = q == 0 ? 0x64006400u : q == 1 ? 0x5C005C00u : q == 2 ? 0x54005400u : 0x4C004C00u;
    return hsub2_bits(lop3_and_or(x, mask, magic), magic_minus(magic & 0xFFFF, 2 * q, 2));
  } else if constexpr (MODE == MODE_F8T) {
    constexpr int b = C & 3;
    return e4m3x2_to_half2_bits((C < 4) ? prmt(A.x, B.x, b | ((4 + b) << 4)) : prmt(A.y, B.y, b | ((4 + b) << 4)));
  } else {
    constexpr int b = C & 3;
    constexpr uint32_t sel = b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12);
    const uint32_t x = (C < 4) ? prmt(A.x, B.x, sel) : prmt(A.y, B.y, sel);
    return hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);
  }
}

template <int K, int MODE>
struct Unroll {
  template <typename F>
  __device__ __forceinline__ static void run(F&& f) {
    Unroll<K - 1, MODE>::run(f);
    f(std::integral_constant<int, K - 1>{});
  }
};
template <int MODE>
struct Unroll<0, MODE> {
  template <typename F>
  __device__ __forceinline__ static void run(F&&) {}
};

// ---------------------------------------------------------------------------
// Visible tile list of one (sequence, kv head): tiles [0, ns) and [tw, n_total)
// when a sliding window leaves a gap after the sink tiles, else [0, n_total).

struct TileList {
  int L, Leff, W, ns, tw, n_total, n_virt;
  bool gap;
};

__device__ __forceinline__ TileList tile_list(const AttnParams& P, int b, int h, bool flag_errors, int KT) {
  TileList t;
  int L = __ldg(P.seq_lens + b);
  if (L < 0) {
    if (flag_errors) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    L = 0;
  }
  t.L = L;
  t.Leff = L;
  if (t.Leff > P.max_blocks * P.block_size) {
    if (flag_errors) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    t.Leff = P.max_blocks * P.block_size;
  }
  t.W = P.window ? __ldg(P.window + h) : 0;
  t.n_total = (t.Leff + KT - 1) / KT;
  t.ns = 0;
  t.tw = 0;
  t.gap = false;
  if (t.W > 0) {
    const int kw = (L - 1) - t.W + 1;  // first key inside the window of the query at L - 1
    if (kw > 0) {
      t.ns = (min(P.sink, t.Leff) + KT - 1) / KT;
      t.tw = kw / KT;
      t.gap = t.tw > t.ns;
    }
  }
  t.n_virt = t.gap ? t.ns + (t.n_total - t.tw) : t.n_total;
  return t;
}

__device__ __forceinline__ int tile_of(const TileList& t, int v) {
  return (t.gap && v >= t.ns) ? t.tw + (v - t.ns) : v;
}

// Number of stream warps actually used for T tiles: at least MIN tiles each.
__device__ __forceinline__ int stream_workers(int T, int nwall, int fixed) {
  if (fixed > 0) return max(1, min(fixed, nwall));
  return max(1, min(nwall, T / DECODE_MIN_TILES_PER_WARP));
}
__device__ __forceinline__ int slice_lo(int w, int T, int nw) { return (int)((long long)w * T / nw); }
// The worker whose slice holds global tile x.
__device__ __forceinline__ int worker_of(int x, int T, int nw) {
  return min(nw - 1, (int)(((long long)(x + 1) * nw - 1) / T));
}

// ---------------------------------------------------------------------------
// Stream-kernel shape per configuration (from sweeps on the decode
// workloads): keys per tile, ring depth and CTAs per SM.  INT4 with GQA
// groups up to 4 takes 64-key tiles (two independent 32-key halves per step
// of a warp) at 3 CTAs per SM; the others 32-key tiles, NT == 1 kernels at 4
// CTAs per SM (3 for the larger 8-bit rows), NT == 2 kernels at 3 (2 for
// 8-bit rows).
template <int MODE, int D, int NT>
struct StreamCfg {
  static constexpr int KT = (MODE == MODE_INT4 && NT == 1) ? 64 : 32;
  static constexpr int NCH = KT / 16;  // 16-row page chunks per tile
  static constexpr int NH2 = KT / 32;  // 32-key halves per tile
  static constexpr int NSTAGE = NT == 1 ? (MODE == MODE_INT4 ? 2 : (MODE == MODE_INT2 ? 5 : 2))
                                        : (MODE == MODE_INT4 ? 4 : (MODE == MODE_INT2 ? 3 : 3));
  static constexpr bool BYTES = MODE == MODE_INT8 || byte_token_head(MODE);
  static constexpr int CTAS = NT == 1 ? (MODE == MODE_INT4 || BYTES ? 3 : 4) : (BYTES ? 2 : 3);
  static constexpr int TILE = KT * row_bytes_of(MODE, D);  // key rows of K (or V)
  static constexpr int STAGE = 2 * TILE;                   // K tile then V tile
};

template <int MODE, int D, int NT>
struct TmaCfg {
  static constexpr int R = row_bytes_of(MODE, D);
  static constexpr bool BYTES = byte_token_head(MODE);
  static constexpr int KT = (NT == 1 && !BYTES) ? 64 : 32;   // keys per tile
  static constexpr int NH2 = KT / 32;                         // 32-key halves per tile
  static constexpr int RPC = KT / 4;                          // key rows per gathered chunk
  static constexpr int RPC_LOG2 = RPC == 16 ? 4 : 3;
  static constexpr int TILE = KT * R;
  static constexpr int TILE_AL = (TILE + 127) / 128 * 128;
  static constexpr int STAGE = 2 * TILE_AL;                   // K tile then V tile
  static constexpr int NSTAGE = STAGE >= 8000 ? 2 : (STAGE >= 4000 ? 3 : 4);
  // one n-tile: one CTA of 12 warps per SM, so that the SM's warps are not
  // ranked by the age of the CTA they belong to (three CTAs of 4 warps finish
  // in the order they started); two n-tiles: two CTAs of 4 warps, which
  // measured faster there than one CTA of 8
  static constexpr int WARPS = NT == 1 ? 3 * DECODE_WARPS : DECODE_WARPS;
  static constexpr int CTAS = NT == 1 ? 1 : 2;
  static constexpr int XREG = 576;                            // exchange bytes per (half, n-tile)
  static constexpr bool XSMEM = NH2 * NT * XREG <= TILE;
  static_assert(RPC * R <= 2048 && (RPC * R) % 16 == 0, "a chunk must be one tensor-map box row");
  static_assert(MODE == MODE_INT8 || WARPS * NSTAGE * (STAGE + 8) + 1024 <= 227 * 1024,
                "the warps' rings must fit one SM");  // (INT8 per channel streams with cp.async instead)
};

// Rows per gathered chunk for the host's tensor maps (0: cp.async path),
// taken from the very configuration the launched kernel uses.
template <int MODE, int D>
int chunk_rows_md(int group) {
  return group <= 4 ? TmaCfg<MODE, D, 1>::RPC : TmaCfg<MODE, D, 2>::RPC;
}
int decode_chunk_rows(int mode, int head_dim, int group) {
  const bool d128 = head_dim == 128;
  switch (mode) {
    case MODE_INT4: return d128 ? chunk_rows_md<MODE_INT4, 128>(group) : chunk_rows_md<MODE_INT4, 64>(group);
    case MODE_INT2: return d128 ? chunk_rows_md<MODE_INT2, 128>(group) : chunk_rows_md<MODE_INT2, 64>(group);
    case MODE_I8T: return d128 ? chunk_rows_md<MODE_I8T, 128>(group) : chunk_rows_md<MODE_I8T, 64>(group);
    case MODE_F8T: return d128 ? chunk_rows_md<MODE_F8T, 128>(group) : chunk_rows_md<MODE_F8T, 64>(group);
    default: return 0;
  }
}

// Keys per tile of the stream kernel that runs a configuration (the prefix
// sum of tile counts and the slices must use the same tiles).
template <int MODE, int D, int NT>
__host__ __device__ constexpr int decode_tile_keys() {
  return MODE == MODE_INT8 ? StreamCfg<MODE, D, NT>::KT : TmaCfg<MODE, D, NT>::KT;
}

// ---------------------------------------------------------------------------
// 1. preparation

// The new tokens' K and V rows of pair (b, h), written as kvq_write writes
// them (the same row function, so the same bytes; a -1 destination is
// skipped, errors set the same bits): the step's write fused into the
// decode.  One warp per row, the CTA's four warps in turn.
template <int MODE, int D, bool STEGO>
__device__ __forceinline__ void fused_write_pair(const AttnParams& P, int b, int h) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = P.num_kv_heads, bs = P.block_size;
  const int t0 = __ldg(P.cu_new + b), n = __ldg(P.cu_new + b + 1) - t0;
  if (n <= 0) return;
  const int L = __ldg(P.seq_lens + b);
  if (L < 0 || n > L) {
    if (threadIdx.x == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    return;
  }
  const int R = row_bytes_of(MODE, D);
  const int32_t* tbl = P.table + (size_t)(P.headwise ? b * Hkv + h : b) * P.max_blocks;
  const RowSigns<EPL> sg = load_row_signs<EPL>(P.signs, lane);
  for (int r = warp; r < 2 * n; r += 4) {
    const int i = r >> 1, kv = r & 1;
    if (t0 + i < 0 || t0 + i >= P.num_new) continue;  // as the write: rows 0 .. num_tokens - 1 only
    const int p = L - n + i;
    const int lb = p / bs;
    if (lb >= P.max_blocks) {
      if (lane == 0) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
      continue;
    }
    const int blk = __ldg(tbl + lb);
    if (blk < 0) continue;  // evicted slot: nothing is written
    if (blk >= P.num_blocks) {
      if (lane == 0) flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
      continue;
    }
    if (!KVQ_IN_BOUNDS(((size_t)blk * Hkv + h) * bs + p % bs < (size_t)P.num_blocks * Hkv * bs, P.dev_error)) continue;
    float x[EPL];
    load_row_elems<EPL>(kv ? P.new_v : P.new_k, P.new_dtype, ((size_t)(t0 + i) * Hkv + h) * D + lane * EPL, x);
    uint8_t* pages = const_cast<uint8_t*>(kv ? P.v_pages : P.k_pages);
    quantise_store_row<MODE, D, STEGO, 32>(sg, x, pages + (((size_t)blk * Hkv + h) * bs + p % bs) * R, lane,
                                           true);
  }
}

template <int MODE, int D, int NT, bool STEGO>
__global__ void __launch_bounds__(128) decode_prep_kernel(AttnParams P, DecodeWs ws) {
  using C = DecCfg<MODE, D>;
  constexpr int EPL = D / 32;
  constexpr int NH = 4 * NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = P.num_kv_heads, G = P.group, Hq = P.num_q_heads;
  __shared__ __half qh[2][NH][D];
  allow_dependent_launch();  // the stream kernel may launch; it waits for this grid to finish
  // This kernel may start while the write kernel before it still runs
  // (programmatic launch): nothing here reads what the write produces except
  // the INT8 channel scales, so INT8 waits for the write first and the other
  // modes only before exiting -- the stream kernel, which waits for this
  // grid, then also sees the new tokens.
  if (MODE == MODE_INT8) grid_dependency_wait();
  // query fragments of one (sequence, kv head)
  const int bh = blockIdx.x;
  const int b = bh / Hkv, h = bh % Hkv;
  const float log2e = 1.4426950408889634f;
  const float dnorm = (MODE != MODE_INT8 && P.signs) ? (float)D : 1.0f;
  for (int i = warp; i < NH; i += 4) {
    float x[EPL];
    if (i < G) {
      const int hq = h * G + i;
      load_row_elems<EPL>(P.q, P.dtype, ((size_t)b * Hq + hq) * D + lane * EPL, x);
      if constexpr (MODE == MODE_INT8) {
        const float* am = P.ch_amax + (size_t)h * D + lane * EPL;  // K channel scales
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] *= __fdiv_rn(am[e], 127.0f);
      } else {
        if (P.signs) {
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            if (__ldg(P.signs + lane * EPL + e) < 0) x[e] = -x[e];
          wht_warp<EPL>(x, lane);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) x[e] = 0.0f;
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
    const float sc = ldexpf(1.0f, 10 - ex);  // max |q''| in [1024, 2048)
    // the folded key offset: sum over dims of the exact operand value (hi +
    // lo) times the constant the folded key unpack adds to the signed code
    float opsum = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float v = x[e] * sc;
      const __half hi = __float2half_rn(v);
      const __half lo = __float2half_rn(v - __half2float(hi));
      qh[0][i][lane * EPL + e] = hi;
      qh[1][i][lane * EPL + e] = lo;
      const float kc = MODE == MODE_INT4 ? KFOLD_INT4 : MODE == MODE_INT2 ? kfold_int2(lane * EPL + e) : 0.0f;
      opsum = fmaf(kc, __half2float(hi) + __half2float(lo), opsum);
    }
    opsum = warp_sum(opsum);
    if (lane == 0) {
      const float beta = i < G ? P.softmax_scale * log2e / (dnorm * sc) : 0.0f;
      const float gamma = i < G ? P.softmax_scale * log2e * sum / dnorm : 0.0f;
      const float corr = opsum;
      ws.qbg[(size_t)bh * NH + i] = make_float4(beta, gamma, corr, 0.0f);
    }
  }
  __syncthreads();
  // B-operand image: [lane][nt][kstep][reg]; slot gq of n-tile nt = head
  // 4 nt + gq/2, half gq & 1; the register pairs head dims in the order the
  // key-side unpack produces them (kpair_dims).
  constexpr int PER_LANE = NT * C::KSTEPS * 2;
  uint4* dst = reinterpret_cast<uint4*>(ws.qfrag + (size_t)bh * 32 * PER_LANE);
  // four consecutive image words per thread and 16-byte store
  for (int q4 = threadIdx.x; q4 < 32 * PER_LANE / 4; q4 += blockDim.x) {
    uint32_t wv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = 4 * q4 + k;
      const int ln = idx / PER_LANE, rest = idx % PER_LANE;
      const int nt = rest / (C::KSTEPS * 2), s = (rest / 2) % C::KSTEPS, r = rest & 1;
      const int g_ = ln >> 2, t_ = ln & 3;
      const int head = 4 * nt + (g_ >> 1), hl = g_ & 1;
      const int w = 4 * (s / C::KPW) + t_, sig = s % C::KPW;
      int d0, d1;
      kpair_dims<MODE>(w, 2 * sig + r, d0, d1);
      const __half2 pr = __halves2half2(qh[hl][head][d0], qh[hl][head][d1]);
      wv[k] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    dst[q4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
  if (MODE != MODE_INT8) grid_dependency_wait();
  if constexpr (MODE != MODE_INT8) {
    // the step's write, after the kernels before it are done with the pools
    if (P.new_k) fused_write_pair<MODE, D, STEGO>(P, b, h);
  }
}

// ---------------------------------------------------------------------------
// 2. stream kernel

// One (sequence, kv head) as seen by a cursor walking the global tile order.
struct Seg {
  int bh, h, start, end;
  TileList t;
  const int32_t* tbl;
};

// Pair bh whose tiles start at global tile `start`.
__device__ __forceinline__ void load_seg(const AttnParams& P, int bh, int start, Seg& s, int KT) {
  const int Hkv = P.num_kv_heads;
  s.bh = bh;
  const int b = bh / Hkv, h = bh % Hkv;
  s.h = h;
  s.t = tile_list(P, b, h, false, KT);
  s.start = start;
  s.end = start + s.t.n_virt;
  s.tbl = P.table + (size_t)(P.headwise ? bh : b) * P.max_blocks;
}

template <int MODE, int D, int NT>
__global__ void __launch_bounds__(128, (StreamCfg<MODE, D, NT>::CTAS)) decode_stream_kernel(AttnParams P, DecodeWs ws) {
  using C = DecCfg<MODE, D>;
  using SC = StreamCfg<MODE, D, NT>;
  constexpr int NSTAGE = SC::NSTAGE;
  constexpr int KT = SC::KT, NCH = SC::NCH, NH2 = SC::NH2;
  constexpr int NH = 4 * NT;
  constexpr int PER_LANE = NT * C::KSTEPS * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = P.group, Hkv = P.num_kv_heads, bs = P.block_size;
  const int BH = P.batch * Hkv;

  allow_dependent_launch();  // the merge kernel may launch; it waits for this grid to finish
  // Slices come from the tile counts themselves (a prefix scan per CTA over
  // all (sequence, kv head) pairs, thread t owning a contiguous run of
  // pairs), worked out while the kernels before still run.
  __shared__ int run_start[129];
  const int items = (BH + 127) / 128;
  {
    const int first = threadIdx.x * items;
    int tsum = 0;
    for (int k = 0; k < items && first + k < BH; ++k) {
      const int bh = first + k;
      tsum += tile_list(P, bh / Hkv, bh % Hkv, false, KT).n_virt;
    }
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ int wtot[DECODE_WARPS];
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wtot[w];
    run_start[threadIdx.x + 1] = before + incl;
    if (threadIdx.x == 0) run_start[0] = 0;
    if (blockIdx.x == 0) {
      // CTA 0 publishes every pair's first tile for the merge kernel, and
      // reports a negative seq_len or one past the table, once per sequence
      int x = before + incl - tsum;
      for (int k = 0; k < items && first + k < BH; ++k) {
        const int bh = first + k;
        ws.tile_start[bh] = x;
        x += tile_list(P, bh / Hkv, bh % Hkv, bh % Hkv == 0, KT).n_virt;
      }
      if (threadIdx.x == 127) ws.tile_start[BH] = before + incl;
    }
    __syncthreads();
  }
  const int T = run_start[128];
  const int nw = stream_workers(T, gridDim.x * DECODE_WARPS, ws.fixed_workers);
  const int gw = blockIdx.x * DECODE_WARPS + warp;
  if (gw >= nw) return;  // whole warp; no CTA-wide barrier follows
  const int lo = slice_lo(gw, T, nw), hi = slice_lo(gw + 1, T, nw);
  if (lo >= hi) return;

  // INT4 / INT2 pages move by 1-D bulk copies (one per 16-row chunk, tracked
  // by a per-stage mbarrier); INT8 rows are XOR-swizzled by 16-byte piece on
  // the way in, so they use per-lane cp.async.
  constexpr bool BULK = MODE != MODE_INT8;
  uint8_t* ring = smem + warp * NSTAGE * SC::STAGE;
  int* wvld = reinterpret_cast<int*>(smem + DECODE_WARPS * NSTAGE * SC::STAGE) + warp * NSTAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DECODE_WARPS * NSTAGE * SC::STAGE + DECODE_WARPS * NSTAGE * 4) +
                   warp * NSTAGE;
  if constexpr (BULK) {
    if (lane == 0) {
      for (int i = 0; i < NSTAGE; ++i) mbar_init(bars + i, 1);
      mbar_init_fence();
    }
    __syncwarp();
  }
  uint32_t phase_bits = 0;  // parity of the next completion to wait for, per stage

  // first (sequence, kv head) of the slice: the run holding tile lo, then
  // the pair inside it
  int a = 0, z = 128;
  while (z - a > 1) {
    const int mid = (a + z) >> 1;
    if (run_start[mid] <= lo) a = mid;
    else z = mid;
  }
  int bh0 = a * items, st0 = run_start[a];
  for (;;) {
    const int n0 = tile_list(P, bh0 / Hkv, bh0 % Hkv, false, KT).n_virt;
    if (st0 + n0 > lo) break;
    st0 += n0;
    ++bh0;
  }
  Seg is;  // lookup / issue cursor
  load_seg(P, bh0, st0, is, KT);
  Seg cs = is;  // compute cursor

  const size_t blk_stride = (size_t)Hkv * bs * C::R;
  const int bs_log2 = __ffs(bs) - 1;

  // Table lookups run one tile ahead of the copies that use them, so the
  // latency of the block-id load overlaps a whole tile of compute.
  int x_lookup = lo;                 // next tile to look up
  int nx_h = 0, nx_key = 0, nx_leff = 0;
  int nx_blk[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) nx_blk[c] = 0;
  bool nx_have = false;
  auto lookup = [&]() {
    nx_have = x_lookup < hi;
    if (nx_have) {
      while (x_lookup >= is.end) load_seg(P, is.bh + 1, is.end, is, KT);
      nx_h = is.h;
      nx_key = KT * tile_of(is.t, x_lookup - is.start);
      nx_leff = is.t.Leff;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int key = nx_key + 16 * c;
        nx_blk[c] = (key < nx_leff && KVQ_IN_BOUNDS((key >> bs_log2) < P.max_blocks, P.dev_error))
                        ? __ldg(is.tbl + (key >> bs_log2))
                        : -1;
      }
      ++x_lookup;
    }
  };

  int st_issue = 0;
  auto issue = [&]() {
    if (nx_have) {
      uint8_t* kt = ring + st_issue * SC::STAGE;
      uint8_t* vt = kt + SC::TILE;
      const uint8_t* kbase = P.k_pages + (size_t)nx_h * bs * C::R;
      const uint8_t* vbase = P.v_pages + (size_t)nx_h * bs * C::R;
      int valid = 0;
      size_t off[NCH];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int key = nx_key + 16 * c;
        const int blk = nx_blk[c];
        bool ok = blk >= 0;  // -1: evicted (never addressed) or beyond the sequence
        if (blk >= P.num_blocks) {
          ok = false;
          if (lane == 0) flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
        }
        off[c] = ok ? (size_t)blk * blk_stride + (size_t)(key & (bs - 1)) * C::R : 0;
        // the chunk's 16 rows lie inside the pool (kbase is head h's first page)
        if (ok && !KVQ_IN_BOUNDS((size_t)nx_h * bs * C::R + off[c] + (size_t)C::CHUNK <=
                                     (size_t)P.num_blocks * Hkv * bs * C::R,
                                 P.dev_error)) {
          ok = false;
          off[c] = 0;
        }
        valid |= (ok ? 1 : 0) << c;
      }
      if constexpr (BULK) {
        // lane 0 acts through predicates, so the warp forms no divergent region
        const bool l0 = lane == 0;
        if (l0) wvld[st_issue] = valid;
        mbar_arrive_expect_tx_if(l0, bars + st_issue, (uint32_t)(__popc(valid) * 2 * C::CHUNK));
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const bool go = l0 && ((valid >> c) & 1);
          bulk_g2s_if(go, kt + c * C::CHUNK, kbase + off[c], C::CHUNK, bars + st_issue);
          bulk_g2s_if(go, vt + c * C::CHUNK, vbase + off[c], C::CHUNK, bars + st_issue);
        }
      } else {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint8_t* ks = kbase + off[c];
          const uint8_t* vs = vbase + off[c];
          const int nbytes = ((valid >> c) & 1) ? 16 : 0;
#pragma unroll
          for (int i = 0; i < (C::R + 31) / 32; ++i) {
            const int q = lane + 32 * i;  // 16-byte piece of the 16-row chunk
            if (q < C::R) {
              const int kappa = 16 * c + q / C::PPR;
              const int dst = kappa * D + 16 * ((q % C::PPR) ^ ((kappa >> 2) & (C::PPR - 1)));
              cp_async16(kt + dst, ks + 16 * q, nbytes);
              cp_async16(vt + dst, vs + 16 * q, nbytes);
            }
          }
        }
        if (lane == 0) wvld[st_issue] = valid;
      }
      st_issue = st_issue + 1 == NSTAGE ? 0 : st_issue + 1;
    }
    if constexpr (!BULK) cp_async_commit();
    lookup();
  };

  // per-segment state
  uint32_t bq[NT][C::KSTEPS][2];
  float bet[NT], gam[NT], kcorr[NT];
  float oacc[NT][C::MT][4];
  float mrun[NT], lrun[NT], pmrun[NT];
  int part_id = 0;

  auto begin_seg = [&](int x) {
    // partial record id: slice index + pair index (unique, see reduce)
    part_id = gw + cs.bh;
    const int qbh = KVQ_IN_BOUNDS(cs.bh >= 0 && cs.bh < BH, P.dev_error) ? cs.bh : 0;
    const uint4* src = reinterpret_cast<const uint4*>(ws.qfrag + ((size_t)qbh * 32 + lane) * PER_LANE);
    uint32_t tmp[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE / 4; ++i) {
      const uint4 v = __ldg(src + i);
      tmp[4 * i] = v.x; tmp[4 * i + 1] = v.y; tmp[4 * i + 2] = v.z; tmp[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int s = 0; s < C::KSTEPS; ++s) {
        bq[nt][s][0] = tmp[(nt * C::KSTEPS + s) * 2];
        bq[nt][s][1] = tmp[(nt * C::KSTEPS + s) * 2 + 1];
      }
      const float4 bg = __ldg(ws.qbg + (size_t)qbh * NH + 4 * nt + tq);
      bet[nt] = bg.x;
      gam[nt] = bg.y;
      kcorr[nt] = bg.z;
      mrun[nt] = -CUDART_INF_F;
      lrun[nt] = 0.0f;
      pmrun[nt] = 0.0f;
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) oacc[nt][mt][r] = 0.0f;
    }
  };

  auto flush_seg = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = lrun[nt], pm = pmrun[nt];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l += __shfl_xor_sync(0xffffffffu, l, o);
        pm += __shfl_xor_sync(0xffffffffu, pm, o);
      }
      const int head = 4 * nt + tq;
      if (head < G && KVQ_IN_BOUNDS(part_id >= 0 && part_id < ws.n_partials, P.dev_error)) {
        float* po = ws.part_o + ((size_t)part_id * G + head) * D;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          po[gq * (D / 16) + mt] = oacc[nt][mt][0] + oacc[nt][mt][1] + pm;
          po[(8 + gq) * (D / 16) + mt] = oacc[nt][mt][2] + oacc[nt][mt][3] + pm;
        }
        if (gq == 0) ws.part_ml[(size_t)part_id * G + head] = make_float2(mrun[nt], l);
      }
    }
  };

  lookup();
  // Copies wait for the kernels before: the write of this step's tokens may
  // still run (the preparation kernel starts alongside it), and the query
  // images and per-head constants must be ready.
  grid_dependency_wait();
#pragma unroll 1
  for (int k = 0; k < NSTAGE - 1; ++k) issue();

  begin_seg(lo);
  int st = 0;
  // per-lane shared-memory offsets (loop invariant): key rows 4gq + 2m + hh,
  // value rows 8tq + 4m' + 2h' + e
  const int koff = 4 * gq * C::R + 4 * tq;
  const bool stego = P.stego != 0;
  const int poff = 4 * gq * C::R + C::DATA;
  const int vrow = 8 * tq * C::R;
  bool timed_out = false;
#pragma unroll 1
  for (int x = lo; x < hi; ++x) {
    if constexpr (BULK) {
      if (!mbar_wait_bounded(bars + st, (phase_bits >> st) & 1)) {
        timed_out = true;
        break;
      }
      phase_bits ^= 1u << st;
    } else {
      cp_async_wait<NSTAGE - 2>();
    }
    __syncwarp();
    issue();
    if (x >= cs.end) {
      flush_seg();
      do load_seg(P, cs.bh + 1, cs.end, cs, KT);
      while (x >= cs.end);
      begin_seg(x);
    }
    const uint8_t* kt = ring + st * SC::STAGE;
    const uint8_t* vt = kt + SC::TILE;
    const int valid = wvld[st];
    st = st + 1 == NSTAGE ? 0 : st + 1;
    const int key0 = KT * tile_of(cs.t, x - cs.start);
    const int Leff = cs.t.Leff, W = cs.t.W, p_q = cs.t.L - 1;
    // every key of the tile visible (the common case): no per-key masks
    const bool full = valid == (1 << NCH) - 1 && key0 + KT <= Leff &&
                      (W <= 0 || key0 > p_q - W || key0 + KT <= P.sink);

    // ---- S^T = U_K (keys x D) . Q (D x slots), per 32-key half h2; lane
    // rows: keys 32 h2 + 4gq + 2m + hh
    float sacc[NH2][2][NT][4];
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) sacc[h2][m][nt][r] = 0.0f;
#pragma unroll
    for (int wi = 0; wi < C::WPL; ++wi) {
      uint32_t kw[NH2][2][2];
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if constexpr (MODE == MODE_INT8)
              kw[h2][m][hh] = load_kword<MODE, D>(kt, 32 * h2 + 4 * gq + 2 * m + hh, 4 * wi + tq);
            else kw[h2][m][hh] = lds32(kt + koff + (32 * h2 + 2 * m + hh) * C::R + 16 * wi);
          }
      Unroll<C::KPW, MODE>::run([&](auto sig_c) {
        constexpr int sig = decltype(sig_c)::value;
        const int s = C::KPW * wi + sig;
#pragma unroll
        for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            uint32_t a[4];
            if constexpr (MODE == MODE_INT4) {
              a[0] = kpair_int4_fold<2 * sig>(kw[h2][m][0]);
              a[1] = kpair_int4_fold<2 * sig>(kw[h2][m][1]);
              a[2] = kpair_int4_fold<2 * sig + 1>(kw[h2][m][0]);
              a[3] = kpair_int4_fold<2 * sig + 1>(kw[h2][m][1]);
            } else {
              a[0] = kpair<MODE, 2 * sig>(kw[h2][m][0]);
              a[1] = kpair<MODE, 2 * sig>(kw[h2][m][1]);
              a[2] = kpair<MODE, 2 * sig + 1>(kw[h2][m][0]);
              a[3] = kpair<MODE, 2 * sig + 1>(kw[h2][m][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[h2][m][nt], a, bq[nt][s][0], bq[nt][s][1]);
          }
      });
    }

    // ---- logits (log2 units), masks, online softmax
    float lg[NH2][2][2][NT];
    float sv_[NH2][2][2], mv_[NH2][2][2];
    bool vk[NH2][2][2];
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kappa = 32 * h2 + 4 * gq + 2 * m + hh;
          bool ok = true;
          if (!full) {
            const int j = key0 + kappa;
            ok = ((valid >> (kappa >> 4)) & 1) && j < Leff;
            if (W > 0) ok = ok && (j < P.sink || j > p_q - W);
          }
          vk[h2][m][hh] = ok;
          float sk = 0.0f, mk = 0.0f;
          if constexpr (MODE != MODE_INT8) {
            const uint32_t pk = lds32(kt + poff + (32 * h2 + 2 * m + hh) * C::R);
            const uint32_t pv = lds32(vt + poff + (32 * h2 + 2 * m + hh) * C::R);
            pad_scale_zero<MODE>(pk, stego, sk, mk);
            pad_scale_zero<MODE>(pv, stego, sv_[h2][m][hh], mv_[h2][m][hh]);
          } else {
            sv_[h2][m][hh] = 1.0f;
            mv_[h2][m][hh] = 0.0f;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float cdot = sacc[h2][m][nt][2 * hh] + sacc[h2][m][nt][2 * hh + 1];  // hi + lo slots
            if constexpr (MODE == MODE_INT4) cdot -= kcorr[nt];
            float zz;
            if constexpr (MODE == MODE_INT8) zz = bet[nt] * cdot;
            else if constexpr (byte_token_head(MODE)) zz = (bet[nt] * sk) * cdot;
            else zz = fmaf(bet[nt] * sk, cdot, gam[nt] * mk);
            lg[h2][m][hh][nt] = ok ? zz : -CUDART_INF_F;
          }
        }

    uint32_t xh[NH2][NT][2], xl[NH2][NT][2];  // packed (P s) hi / lo per (h2, m): (key hh=0, key hh=1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
        tmax = fmaxf(tmax, fmaxf(fmaxf(lg[h2][0][0][nt], lg[h2][0][1][nt]), fmaxf(lg[h2][1][0][nt], lg[h2][1][1][nt])));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mnew = fmaxf(mrun[nt], tmax);
      const float muse = mnew == -CUDART_INF_F ? 0.0f : mnew;
      const float f = ex2(mrun[nt] - muse);
      mrun[nt] = mnew;
      if (__any_sync(0xffffffffu, f != 1.0f)) {
        lrun[nt] *= f;
        pmrun[nt] *= f;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) oacc[nt][mt][r] *= f;
      }
      float tl = 0.0f, tpm = 0.0f;  // tile-local sums, added once per tile
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float wv[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float p = ex2(lg[h2][m][hh][nt] - muse);
            const bool ok = vk[h2][m][hh];
            tl += ok ? p : 0.0f;
            if constexpr (MODE != MODE_INT8 && !byte_token_head(MODE)) tpm += ok ? p * mv_[h2][m][hh] : 0.0f;
            wv[hh] = ok ? p * sv_[h2][m][hh] : 0.0f;
          }
          const __half2 hp = __floats2half2_rn(wv[0], wv[1]);
          const float2 hf = __half22float2(hp);
          const __half2 lp = __floats2half2_rn(wv[0] - hf.x, wv[1] - hf.y);
          xh[h2][nt][m] = *reinterpret_cast<const uint32_t*>(&hp);
          xl[h2][nt][m] = *reinterpret_cast<const uint32_t*>(&lp);
        }
      lrun[nt] += tl;
      pmrun[nt] += tpm;
    }

    // ---- P.V: O^T (D x slots) += U_V^T (D x 16 keys) . Wslots (16 keys x slots)
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int mp = 0; mp < 2; ++mp) {
        uint32_t bw[NT][2];
        const int src = ((2 * tq + mp) << 2) | (gq >> 1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t a0 = __shfl_sync(0xffffffffu, xh[h2][nt][0], src);
          const uint32_t b0 = __shfl_sync(0xffffffffu, xl[h2][nt][0], src);
          const uint32_t a1 = __shfl_sync(0xffffffffu, xh[h2][nt][1], src);
          const uint32_t b1 = __shfl_sync(0xffffffffu, xl[h2][nt][1], src);
          bw[nt][0] = (gq & 1) ? b0 : a0;
          bw[nt][1] = (gq & 1) ? b1 : a1;
        }
        uint2 vl[2][2], vh[2][2];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if constexpr (MODE == MODE_INT8) {
              const int kappa = 32 * h2 + 8 * tq + 4 * mp + 2 * hp + e;
              vl[hp][e] = load_range<MODE, D>(vt, kappa, gq);
              vh[hp][e] = load_range<MODE, D>(vt, kappa, 8 + gq);
            } else {
              const uint8_t* vr = vt + vrow + (32 * h2 + 4 * mp + 2 * hp + e) * C::R;
              vl[hp][e] = load_range<MODE, D>(vr, 0, gq);
              vh[hp][e] = load_range<MODE, D>(vr, 0, 8 + gq);
            }
          }
        if constexpr (MODE == MODE_F8T) {
          if (!full) {  // warp-uniform; masked rows may hold stale NaN codes
#pragma unroll
            for (int hp = 0; hp < 2; ++hp)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                vl[hp][e] = make_uint2(e4m3x4_no_nan(vl[hp][e].x), e4m3x4_no_nan(vl[hp][e].y));
                vh[hp][e] = make_uint2(e4m3x4_no_nan(vh[hp][e].x), e4m3x4_no_nan(vh[hp][e].y));
              }
          }
        }
        Unroll<C::MT, MODE>::run([&](auto mt_c) {
          constexpr int mt = decltype(mt_c)::value;
          const uint32_t a[4] = {vpair<MODE, mt>(vl[0][0], vl[0][1]), vpair<MODE, mt>(vh[0][0], vh[0][1]),
                                 vpair<MODE, mt>(vl[1][0], vl[1][1]), vpair<MODE, mt>(vh[1][0], vh[1][1])};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[nt][mt], a, bw[nt][0], bw[nt][1]);
        });
      }
  }
  if (timed_out) {
    // a copy never arrived: report it, give the copies in flight one more
    // bounded chance to land, and leave without writing this slice's partial
    if (lane == 0) flag_error(P.dev_error, DEVERR_TIMEOUT);
    if constexpr (BULK)
      for (int i = 0; i < NSTAGE; ++i) (void)mbar_wait_bounded(bars + i, (phase_bits >> i) & 1);
    return;
  }
  flush_seg();
  if constexpr (!BULK) cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// merge helpers (used by the merge kernel)

// Merge records w0 + bh .. w0 + nrec - 1 + bh of q head i of pair bh
// (log-sum-exp weights), apply the output transform (inverse RHT with the
// signs tsign, or the INT8 V channel scales) and 1 / l, and store the D
// outputs at `out`; one warp, element d = lane + 32 e in lane `lane`.
// Records are read through L2 (they may come from other SMs of this grid).
template <int D>
__device__ __forceinline__ void merge_records(const AttnParams& P, const DecodeWs& ws, int bh, int i, int w0,
                                              int nrec, const float (&tsign)[D / 32], float* out, int lane) {
  constexpr int EPL = D / 32;
  const int G = P.group;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
  // one round trip for the first 32 records' sums and the first four
  // records' outputs; lane j holds record w0 + j
  // every record index w0 + r + bh must lie in the workspace
  if (!KVQ_IN_BOUNDS(w0 >= 0 && nrec >= 1 && w0 + nrec - 1 + bh < ws.n_partials, P.dev_error)) nrec = 0;
  float2 ml0 = make_float2(-CUDART_INF_F, 0.0f);
  if (lane < nrec) ml0 = __ldcg(ws.part_ml + (size_t)(w0 + lane + bh) * G + i);
  constexpr int V0 = 8;  // records whose outputs load in the first round trip
  float v0[V0][EPL];
#pragma unroll
  for (int u = 0; u < V0; ++u) {
    const float* po = ws.part_o + ((size_t)(u < nrec ? w0 + u + bh : 0) * G + i) * D;
#pragma unroll
    for (int e = 0; e < EPL; ++e) v0[u][e] = u < nrec ? __ldcg(po + lane + 32 * e) : 0.0f;
  }
  float M = ml0.y > 0.0f ? ml0.x : -CUDART_INF_F;
  for (int j = 32 + lane; j < nrec; j += 32) {
    const float2 ml = __ldcg(ws.part_ml + (size_t)(w0 + j + bh) * G + i);
    if (ml.y > 0.0f) M = fmaxf(M, ml.x);
  }
  M = warp_max(M);
  if (M == -CUDART_INF_F) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = 0.0f;
    return;
  }
  float l = 0.0f;
  for (int c0 = 0; c0 < nrec; c0 += 32) {
    float2 ml = ml0;
    if (c0 > 0) {
      ml = make_float2(-CUDART_INF_F, 0.0f);
      if (c0 + lane < nrec) ml = __ldcg(ws.part_ml + (size_t)(w0 + c0 + lane + bh) * G + i);
    }
    const float f = (c0 + lane < nrec && ml.y > 0.0f) ? ex2(ml.x - M) : 0.0f;
    l += f * ml.y;
    const int n = min(32, nrec - c0);
    int kfirst = 0;
    if (c0 == 0) {  // the first V0 records: outputs loaded with the sums above
#pragma unroll
      for (int u = 0; u < V0; ++u) {
        const float fk = __shfl_sync(0xffffffffu, f, u);
        const bool use = u < n && fk != 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = fmaf(use ? fk : 0.0f, use ? v0[u][e] : 0.0f, o[e]);
      }
      kfirst = V0;
    }
    // then four records per round, their loads issued together
    for (int k0 = kfirst; k0 < n; k0 += 4) {
      float fk[4];
      float v[4][EPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        fk[u] = __shfl_sync(0xffffffffu, f, (k0 + u) & 31);
        const bool use = k0 + u < n && fk[u] != 0.0f;
        const float* po = ws.part_o + ((size_t)(w0 + c0 + k0 + u + bh) * G + i) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[u][e] = use ? __ldcg(po + lane + 32 * e) : 0.0f;
        if (!use) fk[u] = 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = fmaf(fk[u], v[u][e], o[e]);
    }
  }
  l = warp_sum(l);
  // element d = lane + 32 e: lane bits are d bits 0-4, e bits are d bits 5-6
  if (P.mode != MODE_INT8 && P.signs) {
#pragma unroll
    for (int lm = 1; lm < 32; lm <<= 1) {
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float x = __shfl_xor_sync(0xffffffffu, o[e], lm);
        o[e] = upper ? x - o[e] : o[e] + x;
      }
    }
#pragma unroll
    for (int hstep = 1; hstep < EPL; hstep <<= 1)
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        if (e & hstep) continue;
        const float a = o[e], c = o[e + hstep];
        o[e] = a + c;
        o[e + hstep] = a - c;
      }
    const float inv = 1.0f / ((float)D * l);
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = tsign[e] * o[e] * inv;
  } else if (P.mode == MODE_INT8) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = o[e] * tsign[e] / l;
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = o[e] / l;
  }
}

// Output transform constants of kv head h for element d = lane + 32 e: the
// RHT signs (+-1), or the INT8 V channel scales.
template <int D>
__device__ __forceinline__ void output_signs(const AttnParams& P, int h, int lane, float (&tsign)[D / 32]) {
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    const int d = lane + 32 * e;
    if (P.mode == MODE_INT8) tsign[e] = __fdiv_rn(__ldg(P.ch_amax + ((size_t)P.num_kv_heads + h) * D + d), 127.0f);
    else tsign[e] = (P.signs && __ldg(P.signs + d) < 0) ? -1.0f : 1.0f;
  }
}

// ---------------------------------------------------------------------------
// 2b. stream kernel over tensor-copied tiles (INT4 / INT2 rows, also with the
// zero point in the scale, and INT8 / FP8 token-head rows)
//
// Same work split, records and arithmetic as decode_stream_kernel, with the
// per-tile overheads taken out of the steady-state loop:
//  * a tile's K (or V) rows arrive by ONE `tile::gather4` tensor copy: the
//    pool is viewed as a 2-D tensor whose rows are page chunks of KT/4 key
//    rows, so the four chunks of a tile (from up to four pages) are four row
//    coordinates of one copy.  The four table lookups run on lanes 0-3.  A
//    chunk with no data (a -1 entry, past the sequence) is pointed at a
//    chunk that exists and is masked: no coordinate outside the pool is ever
//    formed, and no -1 entry becomes an address.
//  * tiles whose keys are all visible take a body without any mask.
//  * the logit of key j is s_j (beta q''.c_j + kappa) + gamma m_j, with
//    kappa = 2^(b-1) gamma - beta (key fold) per head (z = m + 2^(b-1) s).
//  * the (P s) hi / lo weights move from the score layout to the P.V operand
//    layout through shared memory (the consumed K tile), two 16-byte stores
//    and four 8-byte loads per lane, bank-conflict free.

template <int MODE, int D, int NT, bool STEGO>
__global__ void __launch_bounds__(TmaCfg<MODE, D, NT>::WARPS * 32, (TmaCfg<MODE, D, NT>::CTAS))
    decode_tma_kernel(const __grid_constant__ AttnParams P, DecodeWs ws) {
  using C = DecCfg<MODE, D>;
  using TC = TmaCfg<MODE, D, NT>;
  constexpr int NSTAGE = TC::NSTAGE, KT = TC::KT, NH2 = TC::NH2, R = TC::R;
  constexpr int NH = 4 * NT;
  constexpr int PER_LANE = NT * C::KSTEPS * 2;
  constexpr uint32_t VMASK = 0xFu;  // four chunks per tile
  constexpr float HR = (float)(1 << (mode_bits(MODE) - 1));
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = P.group, Hkv = P.num_kv_heads, bs = P.block_size;
  const int BH = P.batch * Hkv;

  allow_dependent_launch();  // the merge kernel may launch; it waits for this grid to finish
  __shared__ int run_start[129];
  const int items = (BH + 127) / 128;
  {
    // the first 128 threads scan: thread t owns pairs t * items ..
    const bool scanner = threadIdx.x < 128;
    const int first = threadIdx.x * items;
    int tsum = 0, incl = 0;
    __shared__ int wtot[4];
    if (scanner) {
      for (int k = 0; k < items && first + k < BH; ++k) {
        const int bh = first + k;
        tsum += tile_list(P, bh / Hkv, bh % Hkv, false, KT).n_virt;
      }
      incl = tsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wtot[warp] = incl;
    }
    __syncthreads();
    if (scanner) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += wtot[w];
      run_start[threadIdx.x + 1] = before + incl;
      if (threadIdx.x == 0) run_start[0] = 0;
      if (blockIdx.x == 0) {
        // CTA 0 publishes every pair's first tile for the merge kernel, and
        // reports a negative seq_len or one past the table, once per sequence
        int x = before + incl - tsum;
        for (int k = 0; k < items && first + k < BH; ++k) {
          const int bh = first + k;
          ws.tile_start[bh] = x;
          x += tile_list(P, bh / Hkv, bh % Hkv, bh % Hkv == 0, KT).n_virt;
        }
        if (threadIdx.x == 127) ws.tile_start[BH] = before + incl;
      }
    }
    __syncthreads();
  }
  const int T = run_start[128];
  const int nw = stream_workers(T, gridDim.x * TC::WARPS, ws.fixed_workers);
  const int gw = blockIdx.x * TC::WARPS + warp;
  if (gw >= nw) return;  // whole warp; no CTA-wide barrier follows
  const int lo = slice_lo(gw, T, nw), hi = slice_lo(gw + 1, T, nw);
  if (lo >= hi) return;

  // first (sequence, kv head) of the slice: the run holding tile lo, then
  // the pair inside it
  int a = 0, z = 128;
  while (z - a > 1) {
    const int mid = (a + z) >> 1;
    if (run_start[mid] <= lo) a = mid;
    else z = mid;
  }
  int bh0 = a * items, st0 = run_start[a];
  for (;;) {
    const int n0 = tile_list(P, bh0 / Hkv, bh0 % Hkv, false, KT).n_virt;
    if (st0 + n0 > lo) break;
    st0 += n0;
    ++bh0;
  }
  uint8_t* ring = smem + warp * NSTAGE * TC::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TC::WARPS * NSTAGE * TC::STAGE) + warp * NSTAGE;
  if (lane == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(bars + i, 1);
    mbar_init_fence();
  }
  __syncwarp();
  uint32_t phase_bits = 0;  // parity of the next completion to wait for, per stage

  Seg is;  // lookup / issue cursor
  load_seg(P, bh0, st0, is, KT);
  Seg cs = is;  // compute cursor

  const int bs_log2 = __ffs(bs) - 1;
  const int cpb_log2 = bs_log2 - TC::RPC_LOG2;  // chunks per page (bs >= RPC)

  // The next tile to copy: lane c < 4 loads the table entry of its chunk c
  // (-1: no data) one tile before the copy, so that the load's latency
  // overlaps a tile of work; the copy turns it into a tensor row.
  int x_lookup = lo;
  int nx_e = -1, nx_sub = 0, nx_h = 0;
  bool nx_have = false;
  auto lookup = [&]() {
    nx_have = x_lookup < hi;
    if (nx_have) {
      while (x_lookup >= is.end) load_seg(P, is.bh + 1, is.end, is, KT);
      const int key = KT * tile_of(is.t, x_lookup - is.start) + TC::RPC * (lane & 3);
      nx_e = (lane < 4 && key < is.t.Leff && KVQ_IN_BOUNDS((key >> bs_log2) < P.max_blocks, P.dev_error))
                 ? __ldg(is.tbl + (key >> bs_log2))
                 : -1;
      nx_sub = (key & (bs - 1)) >> TC::RPC_LOG2;
      nx_h = is.h;
      ++x_lookup;
    }
  };

  int st_issue = 0;
  // the K / V rows are read once per call: with one n-tile they are copied
  // evict-first, so that the partial records written mid-call stay in L2 for
  // the merge kernel (1.1 us less per INT4 call; with two n-tiles, where the
  // stream runs longer per byte, the plain copy measured faster)
  const uint64_t kv_policy = l2_evict_first_policy();
  uint32_t vq = 0;  // chunk masks of the tiles in flight, oldest in the low bits
  int vpos = 0;
  int err_bits = 0;  // error bits of this lane, published once after the loop
  auto issue = [&]() {
    if (nx_have) {
      const bool out_of_pool = nx_e >= P.num_blocks;
      int nx_row = (nx_e >= 0 && !out_of_pool) ? ((nx_e * Hkv + nx_h) << cpb_log2) + nx_sub : -1;
      // a row at or past the tensor map's end (a map that does not match this kernel) is never copied
      const bool past_map = nx_row >= P.chunk_rows_total;
      nx_row = past_map ? -1 : nx_row;
      err_bits |= (out_of_pool || past_map) ? DEVERR_BLOCK_RANGE : 0;
      const uint32_t nx_valid = __ballot_sync(0xffffffffu, nx_row >= 0) & VMASK;
      // chunks without data copy chunk row 0 of the pool instead (masked later)
      const int rr = nx_row >= 0 ? nx_row : 0;
      const int r0 = __shfl_sync(0xffffffffu, rr, 0);
      const int r1 = __shfl_sync(0xffffffffu, rr, 1);
      const int r2 = __shfl_sync(0xffffffffu, rr, 2);
      const int r3 = __shfl_sync(0xffffffffu, rr, 3);
      uint8_t* kt = ring + st_issue * TC::STAGE;
      const bool l0 = lane == 0;
      mbar_arrive_expect_tx_if(l0, bars + st_issue, (uint32_t)(2 * TC::TILE));
      if constexpr (NT == 1) {
        tma_gather4_hint_if(l0, kt, &P.kv_map[0], r0, r1, r2, r3, bars + st_issue, kv_policy);
        tma_gather4_hint_if(l0, kt + TC::TILE_AL, &P.kv_map[1], r0, r1, r2, r3, bars + st_issue, kv_policy);
      } else {
        tma_gather4_if(l0, kt, &P.kv_map[0], r0, r1, r2, r3, bars + st_issue);
        tma_gather4_if(l0, kt + TC::TILE_AL, &P.kv_map[1], r0, r1, r2, r3, bars + st_issue);
      }
      vq |= nx_valid << vpos;
      vpos += 4;
      st_issue = st_issue + 1 == NSTAGE ? 0 : st_issue + 1;
    }
    lookup();
  };

  // per-segment state
  uint32_t bq[NT][C::KSTEPS][2];
  float bet[NT], gam[NT], kap[NT];
  float oacc[NT][C::MT][4];
  float mrun[NT], lrun[NT], pmrun[NT];
  int part_id = 0;

  auto begin_seg = [&]() {
    part_id = gw + cs.bh;  // partial record id: slice index + pair index (unique, see reduce)
    const int qbh = KVQ_IN_BOUNDS(cs.bh >= 0 && cs.bh < BH, P.dev_error) ? cs.bh : 0;
    const uint4* src = reinterpret_cast<const uint4*>(ws.qfrag + ((size_t)qbh * 32 + lane) * PER_LANE);
    uint32_t tmp[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE / 4; ++i) {
      const uint4 v = __ldg(src + i);
      tmp[4 * i] = v.x; tmp[4 * i + 1] = v.y; tmp[4 * i + 2] = v.z; tmp[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int s = 0; s < C::KSTEPS; ++s) {
        bq[nt][s][0] = tmp[(nt * C::KSTEPS + s) * 2];
        bq[nt][s][1] = tmp[(nt * C::KSTEPS + s) * 2 + 1];
      }
      const float4 bg = __ldg(ws.qbg + (size_t)qbh * NH + 4 * nt + tq);
      bet[nt] = bg.x;
      gam[nt] = TC::BYTES ? 0.0f : bg.y;
      kap[nt] = TC::BYTES ? 0.0f : fmaf(-bg.x, bg.z, HR * bg.y);  // 2^(b-1) gamma - beta fold
      mrun[nt] = -CUDART_INF_F;
      lrun[nt] = 0.0f;
      pmrun[nt] = 0.0f;
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) oacc[nt][mt][r] = 0.0f;
    }
  };

  auto flush_seg = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float l = lrun[nt], pm = pmrun[nt];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l += __shfl_xor_sync(0xffffffffu, l, o);
        pm += __shfl_xor_sync(0xffffffffu, pm, o);
      }
      const int head = 4 * nt + tq;
      if (head < G && KVQ_IN_BOUNDS(part_id >= 0 && part_id < ws.n_partials, P.dev_error)) {
        float* po = ws.part_o + ((size_t)part_id * G + head) * D;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          po[gq * (D / 16) + mt] = oacc[nt][mt][0] + oacc[nt][mt][1] + pm;
          po[(8 + gq) * (D / 16) + mt] = oacc[nt][mt][2] + oacc[nt][mt][3] + pm;
        }
        if (gq == 0) ws.part_ml[(size_t)part_id * G + head] = make_float2(mrun[nt], l);
      }
    }
  };

  // per-lane shared-memory offsets (loop invariant): key rows 4gq + 2m + hh,
  // value rows 8tq + 4m' + 2h' + e; the weight exchange writes this lane's
  // 16 bytes at xw and reads its operand pair at xr (+ 320 for m' = 1)
  const int koff = 4 * gq * R + 4 * tq;
  const int poff = 4 * gq * R + C::DATA;
  const int vrow = 8 * tq * R;
  const int xw = 64 * (gq >> 1) + 16 * tq + 320 * (gq & 1);
  const int xr = 64 * tq + 8 * gq;

  // One tile: S = codes . q'', online softmax, O += codes^T . (P s).
  auto tile = [&](auto full_c, const uint8_t* kt, const uint8_t* vt, uint32_t cur, int key0, int Leff, int W,
                  int p_q) {
    constexpr bool FULL = decltype(full_c)::value;
    float sacc[NH2][2][NT][4];
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) sacc[h2][m][nt][r] = 0.0f;
#pragma unroll
    for (int wi = 0; wi < C::WPL; ++wi) {
      uint32_t kw[NH2][2][2];
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) kw[h2][m][hh] = lds32(kt + koff + (32 * h2 + 2 * m + hh) * R + 16 * wi);
      Unroll<C::KPW, MODE>::run([&](auto sig_c) {
        constexpr int sig = decltype(sig_c)::value;
        const int s = C::KPW * wi + sig;
#pragma unroll
        for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            uint32_t av[4];
            if constexpr (MODE == MODE_INT4) {
              av[0] = kpair_int4_fold<2 * sig>(kw[h2][m][0]);
              av[1] = kpair_int4_fold<2 * sig>(kw[h2][m][1]);
              av[2] = kpair_int4_fold<2 * sig + 1>(kw[h2][m][0]);
              av[3] = kpair_int4_fold<2 * sig + 1>(kw[h2][m][1]);
            } else if constexpr (MODE == MODE_INT2) {
              av[0] = kpair_int2_fold<2 * sig>(kw[h2][m][0]);
              av[1] = kpair_int2_fold<2 * sig>(kw[h2][m][1]);
              av[2] = kpair_int2_fold<2 * sig + 1>(kw[h2][m][0]);
              av[3] = kpair_int2_fold<2 * sig + 1>(kw[h2][m][1]);
            } else {
              av[0] = kpair<MODE, 2 * sig>(kw[h2][m][0]);
              av[1] = kpair<MODE, 2 * sig>(kw[h2][m][1]);
              av[2] = kpair<MODE, 2 * sig + 1>(kw[h2][m][0]);
              av[3] = kpair<MODE, 2 * sig + 1>(kw[h2][m][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[h2][m][nt], av, bq[nt][s][0], bq[nt][s][1]);
          }
      });
    }

    // logits (log2 units) and the per-key value scale / zero-point value
    float lg[NH2][2][2][NT];
    float sv_[NH2][2][2], zv_[NH2][2][2];
    bool vk[NH2][2][2];
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          bool ok = true;
          if constexpr (!FULL) {
            const int kappa = 32 * h2 + 4 * gq + 2 * m + hh;
            const int j = key0 + kappa;
            ok = ((cur >> (kappa / TC::RPC)) & 1) && j < Leff;
            if (W > 0) ok = ok && (j < P.sink || j > p_q - W);
          }
          vk[h2][m][hh] = ok;
          const uint32_t pk = lds32(kt + poff + (32 * h2 + 2 * m + hh) * R);
          const uint32_t pv = lds32(vt + poff + (32 * h2 + 2 * m + hh) * R);
          float sk, mk;
          [[maybe_unused]] float zst = 0.0f;  // STEGO: the key's zero point
          if constexpr (TC::BYTES) {
            sk = __uint_as_float(pk);
            mk = 0.0f;
            sv_[h2][m][hh] = __uint_as_float(pv);
            zv_[h2][m][hh] = 0.0f;
          } else if constexpr (STEGO) {
            sk = __uint_as_float(pk & ~15u);
            mk = 0.0f;
            zst = (float)(int)(pk & 15u);
            const float s_v = __uint_as_float(pv & ~15u);
            sv_[h2][m][hh] = s_v;
            zv_[h2][m][hh] = s_v * (float)(8 - (int)(pv & 15u));
          } else {
            const float2 fk = __half22float2(*reinterpret_cast<const __half2*>(&pk));
            const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&pv));
            sk = fk.x;
            mk = fk.y;
            sv_[h2][m][hh] = fv.x;
            zv_[h2][m][hh] = fmaf(HR, fv.x, fv.y);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float cdot = sacc[h2][m][nt][2 * hh] + sacc[h2][m][nt][2 * hh + 1];  // hi + lo slots
            float zz;
            if constexpr (TC::BYTES) {
              zz = sk * (bet[nt] * cdot);
            } else if constexpr (STEGO) {
              zz = sk * fmaf(-gam[nt], zst, fmaf(bet[nt], cdot, kap[nt]));
            } else {
              zz = fmaf(sk, fmaf(bet[nt], cdot, kap[nt]), gam[nt] * mk);
            }
            lg[h2][m][hh][nt] = FULL ? zz : (ok ? zz : -CUDART_INF_F);
          }
        }

    uint32_t xh[NH2][NT][2], xl[NH2][NT][2];  // packed (P s) hi / lo per (h2, m): (key hh=0, key hh=1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
        tmax = fmaxf(tmax, fmaxf(fmaxf(lg[h2][0][0][nt], lg[h2][0][1][nt]), fmaxf(lg[h2][1][0][nt], lg[h2][1][1][nt])));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mnew = fmaxf(mrun[nt], tmax);
      const float muse = mnew == -CUDART_INF_F ? 0.0f : mnew;
      const float f = ex2(mrun[nt] - muse);
      mrun[nt] = mnew;
      if (__any_sync(0xffffffffu, f != 1.0f)) {
        lrun[nt] *= f;
        pmrun[nt] *= f;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) oacc[nt][mt][r] *= f;
      }
      float tl = 0.0f, tpm = 0.0f;  // tile-local sums, added once per tile
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float wv[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float p = ex2(lg[h2][m][hh][nt] - muse);
            if constexpr (FULL) {
              tl += p;
              if constexpr (!TC::BYTES) tpm = fmaf(p, zv_[h2][m][hh], tpm);
              wv[hh] = p * sv_[h2][m][hh];
            } else {
              // select after the product: a masked row's scale may be any bits
              const bool ok = vk[h2][m][hh];
              tl += ok ? p : 0.0f;
              if constexpr (!TC::BYTES) tpm += ok ? p * zv_[h2][m][hh] : 0.0f;
              wv[hh] = ok ? p * sv_[h2][m][hh] : 0.0f;
            }
          }
          const __half2 hp = __floats2half2_rn(wv[0], wv[1]);
          const float2 hf = __half22float2(hp);
          const __half2 lp = __floats2half2_rn(wv[0] - hf.x, wv[1] - hf.y);
          xh[h2][nt][m] = *reinterpret_cast<const uint32_t*>(&hp);
          xl[h2][nt][m] = *reinterpret_cast<const uint32_t*>(&lp);
        }
      lrun[nt] += tl;
      pmrun[nt] += tpm;
    }

    // the weights in the P.V operand layout: lane (gq, tq) takes, for keys
    // 8tq + 4m' + {0..3}, slot gq = (head gq/2, hi or lo) from lane (2tq + m', gq/2)
    uint32_t bw[NH2][2][NT][2];
    if constexpr (TC::XSMEM) {
      uint8_t* xb = const_cast<uint8_t*>(kt);  // this stage's K rows are consumed
      __syncwarp();
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          sts128(xb + (h2 * NT + nt) * TC::XREG + xw,
                 make_uint4(xh[h2][nt][0], xh[h2][nt][1], xl[h2][nt][0], xl[h2][nt][1]));
      __syncwarp();
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int mp = 0; mp < 2; ++mp)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = lds64(xb + (h2 * NT + nt) * TC::XREG + xr + 320 * mp);
            bw[h2][mp][nt][0] = b.x;
            bw[h2][mp][nt][1] = b.y;
          }
    } else {
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          const int src = ((2 * tq + mp) << 2) | (gq >> 1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint32_t a0 = __shfl_sync(0xffffffffu, xh[h2][nt][0], src);
            const uint32_t b0 = __shfl_sync(0xffffffffu, xl[h2][nt][0], src);
            const uint32_t a1 = __shfl_sync(0xffffffffu, xh[h2][nt][1], src);
            const uint32_t b1 = __shfl_sync(0xffffffffu, xl[h2][nt][1], src);
            bw[h2][mp][nt][0] = (gq & 1) ? b0 : a0;
            bw[h2][mp][nt][1] = (gq & 1) ? b1 : a1;
          }
        }
    }

    // P.V: O^T (D x slots) += U_V^T (D x 16 keys) . Wslots (16 keys x slots)
#pragma unroll
    for (int h2 = 0; h2 < NH2; ++h2)
#pragma unroll
      for (int mp = 0; mp < 2; ++mp) {
        uint2 vl[2][2], vh[2][2];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint8_t* vr = vt + vrow + (32 * h2 + 4 * mp + 2 * hp + e) * R;
            vl[hp][e] = load_range<MODE, D>(vr, 0, gq);
            vh[hp][e] = load_range<MODE, D>(vr, 0, 8 + gq);
          }
        if constexpr (MODE == MODE_F8T && !FULL) {  // masked rows may hold stale NaN codes
#pragma unroll
          for (int hp = 0; hp < 2; ++hp)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              vl[hp][e] = make_uint2(e4m3x4_no_nan(vl[hp][e].x), e4m3x4_no_nan(vl[hp][e].y));
              vh[hp][e] = make_uint2(e4m3x4_no_nan(vh[hp][e].x), e4m3x4_no_nan(vh[hp][e].y));
            }
        }
        Unroll<C::MT, MODE>::run([&](auto mt_c) {
          constexpr int mt = decltype(mt_c)::value;
          const uint32_t av[4] = {vpair<MODE, mt>(vl[0][0], vl[0][1]), vpair<MODE, mt>(vh[0][0], vh[0][1]),
                                  vpair<MODE, mt>(vl[1][0], vl[1][1]), vpair<MODE, mt>(vh[1][0], vh[1][1])};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[nt][mt], av, bw[h2][mp][nt][0], bw[h2][mp][nt][1]);
        });
      }
  };

  lookup();
  // Copies wait for the kernel before: the write of this step's tokens may
  // still run (this grid starts alongside it).
  grid_dependency_wait();
#pragma unroll 1
  for (int k = 0; k < NSTAGE - 1; ++k) issue();

  int st = 0;
  bool timed_out = false;
#pragma unroll 1
  for (int x = lo; x < hi; ++x) {
    if (x == lo || x >= cs.end) {  // a new (sequence, kv head): its query fragments (one code path)
      if (x > lo) {
        flush_seg();
        do load_seg(P, cs.bh + 1, cs.end, cs, KT);
        while (x >= cs.end);
      }
      begin_seg();
    }
    if (!mbar_wait_bounded(bars + st, (phase_bits >> st) & 1)) {
      timed_out = true;
      break;
    }
    phase_bits ^= 1u << st;
    __syncwarp();
    issue();
    const uint32_t cur = vq & VMASK;
    vq >>= 4;
    vpos -= 4;
    const uint8_t* kt = ring + st * TC::STAGE;
    st = st + 1 == NSTAGE ? 0 : st + 1;
    const int key0 = KT * tile_of(cs.t, x - cs.start);
    const int Leff = cs.t.Leff, W = cs.t.W, p_q = cs.t.L - 1;
    const bool full = cur == VMASK && key0 + KT <= Leff && (W <= 0 || key0 > p_q - W || key0 + KT <= P.sink);
    if (full) tile(std::true_type{}, kt, kt + TC::TILE_AL, cur, key0, Leff, W, p_q);
    else tile(std::false_type{}, kt, kt + TC::TILE_AL, cur, key0, Leff, W, p_q);
  }
  err_bits = __reduce_or_sync(0xffffffffu, err_bits);
  if (err_bits && lane == 0) flag_error(P.dev_error, err_bits);
  if (timed_out) {
    // a copy never arrived: report it, give the copies in flight one more
    // bounded chance to land, and leave without writing this slice's partial
    if (lane == 0) flag_error(P.dev_error, DEVERR_TIMEOUT);
    for (int i = 0; i < NSTAGE; ++i) (void)mbar_wait_bounded(bars + i, (phase_bits >> i) & 1);
    return;
  }
  flush_seg();
}

// ---------------------------------------------------------------------------
// 3. merge of the partials of one (sequence, q head) + inverse RHT

template <int D>
__global__ void __launch_bounds__(256) decode_reduce_kernel(AttnParams P, DecodeWs ws) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int Hq = P.num_q_heads, G = P.group, Hkv = P.num_kv_heads;
  if (wid >= (long long)P.batch * Hq) return;
  const int b = (int)(wid / Hq), hq = (int)(wid % Hq);
  const int h = hq / G, i = hq % G;
  const int bh = b * Hkv + h;
  const int BH = P.batch * Hkv;
  float* out = P.out + (size_t)wid * D;
  // the output transform's constants do not depend on the kernels before
  float tsign[EPL];
  output_signs<D>(P, h, lane, tsign);
  grid_dependency_wait();  // every partial of the stream kernel is written
  const int T = ws.tile_start[BH];
  const int start = ws.tile_start[bh], end = ws.tile_start[bh + 1];
  if (start >= end || !KVQ_IN_BOUNDS(start >= 0 && end <= T, P.dev_error)) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = 0.0f;
    return;
  }
  // the slices holding this pair's tiles are workers w_first .. w_last; the
  // record of (worker w, pair bh) is w + bh, written by this call
  const int nw = stream_workers(T, ws.nwall, ws.fixed_workers);
  const int w0 = worker_of(start, T, nw), w1 = worker_of(end - 1, T, nw);
  merge_records<D>(P, ws, bh, i, w0, w1 - w0 + 1, tsign, out, lane);
}

// ---------------------------------------------------------------------------
// launch

template <int MODE, int D, int NT>
size_t stream_smem_bytes() {
  using SC = StreamCfg<MODE, D, NT>;
  constexpr int NSTAGE = SC::NSTAGE;
  return (size_t)DECODE_WARPS * NSTAGE * SC::STAGE + DECODE_WARPS * NSTAGE * 4 + DECODE_WARPS * NSTAGE * 8;
}

// CTAs per SM and warps per CTA of the stream kernel one configuration launches
template <int D, int NT>
DecodeShape decode_shape_dnt(int mode) {
  switch (mode) {
    case MODE_INT4: return {TmaCfg<MODE_INT4, D, NT>::CTAS, TmaCfg<MODE_INT4, D, NT>::WARPS};
    case MODE_INT2: return {TmaCfg<MODE_INT2, D, NT>::CTAS, TmaCfg<MODE_INT2, D, NT>::WARPS};
    case MODE_INT8: return {StreamCfg<MODE_INT8, D, NT>::CTAS, DECODE_WARPS};
    case MODE_I8T: return {TmaCfg<MODE_I8T, D, NT>::CTAS, TmaCfg<MODE_I8T, D, NT>::WARPS};
    default: return {TmaCfg<MODE_F8T, D, NT>::CTAS, TmaCfg<MODE_F8T, D, NT>::WARPS};
  }
}

DecodeShape decode_shape(int mode, int head_dim, int group) {
  if (head_dim == 64) return group > 4 ? decode_shape_dnt<64, 2>(mode) : decode_shape_dnt<64, 1>(mode);
  return group > 4 ? decode_shape_dnt<128, 2>(mode) : decode_shape_dnt<128, 1>(mode);
}

template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int MODE, int D, int NT, bool STEGO>
cudaError_t launch_decode_t(const AttnParams& P, const DecodeWs& ws, int grid, cudaStream_t stream) {
  constexpr bool TMA = MODE != MODE_INT8;
  using TC = TmaCfg<MODE, D, NT>;
  const size_t smem = TMA ? (size_t)TC::WARPS * TC::NSTAGE * TC::STAGE + TC::WARPS * TC::NSTAGE * 8
                          : stream_smem_bytes<MODE, D, NT>();
  // the opt-in shared-memory size is set once per device (not inside later
  // calls, which may be captured into a CUDA graph)
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    if constexpr (TMA)
      e = cudaFuncSetAttribute(decode_tma_kernel<MODE, D, NT, STEGO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    else
      e = cudaFuncSetAttribute(decode_stream_kernel<MODE, D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int BH = P.batch * P.num_kv_heads;
  e = launch_dependent(decode_prep_kernel<MODE, D, NT, STEGO>, dim3(BH), dim3(128), 0, stream, P, ws);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the stream and merge kernels launch programmatically: their CTAs become
  // resident while the previous kernel drains and wait on its completion
  if constexpr (TMA)
    e = launch_dependent(decode_tma_kernel<MODE, D, NT, STEGO>, dim3(grid), dim3(TC::WARPS * 32), smem, stream, P,
                         ws);
  else
    e = launch_dependent(decode_stream_kernel<MODE, D, NT>, dim3(grid), dim3(128), smem, stream, P, ws);
  if (e != cudaSuccess) return e;
  const long long warps = (long long)P.batch * P.num_q_heads;
  return launch_dependent(decode_reduce_kernel<D>, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, stream, P, ws);
}

template <int MODE, int D>
cudaError_t launch_decode_md(const AttnParams& P, const DecodeWs& ws, int grid, cudaStream_t stream) {
  if constexpr (MODE == MODE_INT4) {
    if (P.stego) {
      if (P.group <= 4) return launch_decode_t<MODE, D, 1, true>(P, ws, grid, stream);
      return launch_decode_t<MODE, D, 2, true>(P, ws, grid, stream);
    }
  }
  if (P.group <= 4) return launch_decode_t<MODE, D, 1, false>(P, ws, grid, stream);
  return launch_decode_t<MODE, D, 2, false>(P, ws, grid, stream);
}

cudaError_t launch_decode(const AttnParams& P, const DecodeWs& ws, int grid, cudaStream_t stream) {
  switch (P.mode * 1000 + P.head_dim) {
    case MODE_INT4 * 1000 + 128: return launch_decode_md<MODE_INT4, 128>(P, ws, grid, stream);
    case MODE_INT4 * 1000 + 64: return launch_decode_md<MODE_INT4, 64>(P, ws, grid, stream);
    case MODE_INT2 * 1000 + 128: return launch_decode_md<MODE_INT2, 128>(P, ws, grid, stream);
    case MODE_INT2 * 1000 + 64: return launch_decode_md<MODE_INT2, 64>(P, ws, grid, stream);
    case MODE_INT8 * 1000 + 128: return launch_decode_md<MODE_INT8, 128>(P, ws, grid, stream);
    case MODE_INT8 * 1000 + 64: return launch_decode_md<MODE_INT8, 64>(P, ws, grid, stream);
    case MODE_I8T * 1000 + 128: return launch_decode_md<MODE_I8T, 128>(P, ws, grid, stream);
    case MODE_I8T * 1000 + 64: return launch_decode_md<MODE_I8T, 64>(P, ws, grid, stream);
    case MODE_F8T * 1000 + 128: return launch_decode_md<MODE_F8T, 128>(P, ws, grid, stream);
    case MODE_F8T * 1000 + 64: return launch_decode_md<MODE_F8T, 64>(P, ws, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
