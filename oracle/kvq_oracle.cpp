// kvq_oracle.cpp -- plain, slow CPU oracle of the paged low-bit KV cache.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library (sub_byte_quantized_write_gb300/)
// includes, links or calls this file; only tests/, the smoke check and the
// bench's CPU-baseline leg load it.  It shares no header, helper, table or
// constant with the CUDA path: every step is written out here from the pages.
//
// What it computes (sources by page title and section):
//   * Write, INT4 / INT2 per (token, kv_head) row -- vLLM PR #40835 review
//     summary ("INT4 per-token-head KV cache for the Triton backend"),
//     功能与动机 and 实现拆解 item 2: rotate with a random Hadamard transform,
//     then an asymmetric scale and zero point per token-head, round, pack two
//     4-bit codes per byte; 关键源码片段 INT4_CONFIG: signed range [-8, 7];
//     get_kv_cache_shape: row = head_size/2 data bytes + 4 pad bytes.
//     FastDeploy PR #5173 "support dynamic int2 quantization cache kv",
//     Motivation / Modifications: the same dynamic scheme at 2 bits.
//   * Write, INT8 per channel -- vllm-ascend-quantized-kv-cache METADATA
//     ("Ascend INT8 KV Cache Plugin"), 运行机制: symmetric per-channel scales
//     taken along the token axis on the first K/V a layer receives, separately
//     for K and V.
//   * Write, INT4 with the zero point hidden in the scale -- same vLLM page,
//     评论区精华 (zero-point steganography): the 4-bit zero point is stored in
//     the low 4 bits of the fp32 scale, so the row needs no extra bytes.
//   * Write, INT8 / FP8 per (token, kv_head) row -- same vLLM page, 功能与动机
//     and 关联脉络: the INT4 mode is added on top of the INT8 / FP8
//     per-token-head modes of the base PR #40633, one scale per token-head.
//   * Paging -- FastDeploy PR #7718 "Optimize AppendAttention for discrete
//     head-wise block_idx", Motivation: uniform [batch, block] table or
//     head-wise [batch * kv_heads, block] table; PR2-only delta table and
//     Correctness gates: a -1 entry is an evicted sliding-window block whose
//     keys contribute nothing and whose page is never addressed; sink_size.
//   * Gather and dequantise -- FastDeploy PR #5173 (the review notes a new
//     custom op dynamic_quant_get_kv_from_cache) and the Ascend INT8 plugin,
//     运行机制 (prefill gathers and dequantises the paged cache when needed):
//     rows of given positions read back through the table, dequantised and
//     mapped through the inverse RHT to dense K / V.
//   * Attention -- the textbook definition: softmax(scale * q . k_j) weights
//     over the visible dequantised keys, output sum_j P_j v_j, in double.
//
// Readings taken where the pages are silent:
//   RHT unnormalised forward y = H (d * x), inverse x = d * (H y) / D; butterfly
//   stage order h = 1, 2, ..., D/2 in fp32; the zero point m is the value of
//   code 0 (the row minimum); fp16 round-to-nearest-even saturating at 65504;
//   codes by round-half-to-even; element 2i in the low nibble; element 4i+j in
//   bits 2j; pad = fp16 s then fp16 m; INT8 range [-127, 127] with scale
//   amax / 127; a query at p sees key j iff j <= p and (no window, or j < sink,
//   or j > p - W) and its block entry is a valid id.  Zero-point-in-scale
//   INT4: the grid (u - zp) * s always holds 0, so it spans [min(min, 0),
//   max(max, 0)]: s = (max(max, 0) - min(min, 0)) / 15 with its low 4
//   mantissa bits cleared; zero point zp = clamp(rne(-min(min, 0) / s), 0, 15);
//   codes clamp(rne(x / s) + zp, 0, 15); pad = bits(s) | zp; value (u - zp) * s.
//   INT8 / FP8 per token-head: symmetric, RHT optional as for INT4; amax =
//   max |x| of the (rotated) row; s = amax / 127 with codes clamp(rne(x / s),
//   -127, 127), or s = amax / 448 with codes the nearest E4M3 value of x / s
//   (ties to even, saturating at 448); row = D code bytes + fp32 s; s = 0
//   gives all-zero codes.
//
// Built with -O2 -ffp-contract=off -fno-fast-math so that the fp32 write path
// is evaluated exactly in the order written.

#include <algorithm>
#include <atomic>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

enum { MODE_INT4 = 0, MODE_INT2 = 1, MODE_INT8 = 2, MODE_INT4_STEGO = 3, MODE_INT8_TOKEN_HEAD = 4,
       MODE_FP8_TOKEN_HEAD = 5 };
enum { DT_F32 = 0, DT_BF16 = 1 };
enum { ERR_BLOCK_RANGE = 1, ERR_TABLE_RANGE = 2, ERR_SEQ_LEN = 4 };

// ---------------------------------------------------------------------------
// IEEE-754 binary16 conversions, from the format's definition:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 encodes
// subnormals (fraction * 2^-24), exponent 31 encodes Inf/NaN.

uint16_t f16_encode_exact(double v /* >= 0, exactly representable in binary16 */) {
  if (v == 0.0) return 0;
  if (v < std::ldexp(1.0, -14)) {  // subnormal: v = frac * 2^-24
    return (uint16_t)(v / std::ldexp(1.0, -24));
  }
  int e2;
  double fr = std::frexp(v, &e2);  // v = fr * 2^e2, fr in [0.5, 1)
  int e = e2 - 1;                  // v = (2 fr) * 2^e, 2 fr in [1, 2)
  if (e > 15) return 0x7C00;       // infinity
  double frac = (2.0 * fr - 1.0) * 1024.0;  // exact integer 0..1023
  return (uint16_t)(((e + 15) << 10) | (int)frac);
}

// Round a float to binary16, nearest representable value, ties to even;
// magnitudes at or beyond 65520 (half an ulp above the largest finite 65504)
// become infinity, as IEEE rounding prescribes.
uint16_t f16_round_nearest_even(float x) {
  uint32_t bits;
  std::memcpy(&bits, &x, 4);
  uint16_t sign = (uint16_t)((bits >> 31) << 15);
  if (std::isnan(x)) return (uint16_t)(sign | 0x7E00);
  double a = std::fabs((double)x);
  if (std::isinf(x)) return (uint16_t)(sign | 0x7C00);
  // spacing of binary16 values around a: 2^(e-10) in binade [2^e, 2^(e+1)),
  // e >= -14; subnormal spacing 2^-24 below 2^-14.
  double ulp;
  if (a < std::ldexp(1.0, -14)) {
    ulp = std::ldexp(1.0, -24);
  } else {
    int e2;
    std::frexp(a, &e2);
    ulp = std::ldexp(1.0, (e2 - 1) - 10);
  }
  double q = a / ulp;                 // exact: ulp is a power of two
  double r = std::nearbyint(q);       // ties to even (default rounding mode)
  double v = r * ulp;
  if (v >= 65520.0) return (uint16_t)(sign | 0x7C00);
  return (uint16_t)(sign | f16_encode_exact(v));
}

float f16_decode(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0) v = std::ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = std::ldexp(1.0 + f / 1024.0, e - 15);
  return (float)(s ? -v : v);
}

// Saturating variant used for the stored scale and zero point: values beyond
// the largest finite binary16 are clamped to +-65504 before rounding.
uint16_t f16_saturate(float x) {
  if (x > 65504.0f) x = 65504.0f;
  if (x < -65504.0f) x = -65504.0f;
  return f16_round_nearest_even(x);
}

// ---------------------------------------------------------------------------
// FP8 E4M3, the variant without infinities, from the format's definition:
// 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; exponent field 0
// encodes subnormals (fraction * 2^-9); only S.1111.111 is NaN, so the
// largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448.

double e4m3_decode(uint8_t c) {
  const int e = (c >> 3) & 15, f = c & 7;
  double v;
  if (e == 15 && f == 7) v = NAN;
  else if (e == 0) v = std::ldexp((double)f, -9);
  else v = std::ldexp(1.0 + f / 8.0, e - 7);
  return (c & 0x80) ? -v : v;
}

// Nearest E4M3 value of a finite float, ties to even; magnitudes that round
// above 448 saturate to 448.  The input's sign is kept (-0 gives 0x80).
uint8_t e4m3_round_saturate(float x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs((double)x);
  // spacing of E4M3 values around a: 2^(e-3) in binade [2^e, 2^(e+1)),
  // e >= -6; subnormal spacing 2^-9 below 2^-6
  double ulp;
  if (a < std::ldexp(1.0, -6)) {
    ulp = std::ldexp(1.0, -9);
  } else {
    int e2;
    std::frexp(a, &e2);
    ulp = std::ldexp(1.0, (e2 - 1) - 3);
  }
  double v = std::nearbyint(a / ulp) * ulp;  // exact: ulp is a power of two
  if (v > 448.0) v = 448.0;
  uint8_t mag;
  if (v < std::ldexp(1.0, -6)) {
    mag = (uint8_t)(v / std::ldexp(1.0, -9));
  } else {
    int e2;
    const double fr = std::frexp(v, &e2);  // v = (2 fr) * 2^(e2 - 1)
    mag = (uint8_t)(((e2 - 1 + 7) << 3) | (int)((2.0 * fr - 1.0) * 8.0));
  }
  return (uint8_t)(sign | mag);
}

float widen(const void* base, int dtype, size_t idx) {
  if (dtype == DT_F32) return ((const float*)base)[idx];
  uint16_t b = ((const uint16_t*)base)[idx];
  uint32_t u = (uint32_t)b << 16;  // bf16 -> fp32 is exact: append 16 zero bits
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

int code_bits(int mode) { return (mode == MODE_INT4 || mode == MODE_INT4_STEGO) ? 4 : (mode == MODE_INT2 ? 2 : 8); }
bool byte_token_head(int mode) { return mode == MODE_INT8_TOKEN_HEAD || mode == MODE_FP8_TOKEN_HEAD; }

int row_bytes(int mode, int D) {
  if (D != 64 && D != 128) return 0;
  if (mode == MODE_INT4) return D / 2 + 4;  // nibbles + fp16 s + fp16 m
  if (mode == MODE_INT4_STEGO) return D / 2 + 4;  // nibbles + fp32 s carrying the zero point
  if (mode == MODE_INT2) return D / 4 + 4;  // crumbs + fp16 s + fp16 m
  if (mode == MODE_INT8) return D;
  if (byte_token_head(mode)) return D + 4;  // code bytes + fp32 s
  return 0;
}

// ---------------------------------------------------------------------------
// Random Hadamard transform (forward), fp32, fixed order: sign flip, then the
// Walsh-Hadamard butterfly with stride h = 1, 2, 4, ..., D/2; each pair
// (j, j+h) with (j & h) == 0 becomes (x_j + x_{j+h}, x_j - x_{j+h}).
void rht_forward_f32(float* x, int D, const int8_t* signs) {
  if (signs) {
    for (int i = 0; i < D; ++i)
      if (signs[i] < 0) x[i] = -x[i];
  }
  for (int h = 1; h < D; h <<= 1) {
    for (int j = 0; j < D; ++j) {
      if (j & h) continue;
      float a = x[j], b = x[j + h];
      x[j] = a + b;
      x[j + h] = a - b;
    }
  }
}

// Unnormalised Walsh-Hadamard product in double (used for the inverse).
void wht_double(double* x, int D) {
  for (int h = 1; h < D; h <<= 1)
    for (int j = 0; j < D; ++j) {
      if (j & h) continue;
      double a = x[j], b = x[j + h];
      x[j] = a + b;
      x[j + h] = a - b;
    }
}

// ---------------------------------------------------------------------------
// Code packing.  INT4: byte i = u[2i] | u[2i+1] << 4.  INT2: byte i =
// sum_j u[4i+j] << 2j.  INT8: byte i = two's complement of the signed code.
void pack_codes(int mode, const uint8_t* u, int D, uint8_t* out) {
  if (mode == MODE_INT4 || mode == MODE_INT4_STEGO) {
    for (int i = 0; i < D / 2; ++i) out[i] = (uint8_t)((u[2 * i] & 15) | ((u[2 * i + 1] & 15) << 4));
  } else if (mode == MODE_INT2) {
    for (int i = 0; i < D / 4; ++i) {
      int b = 0;
      for (int j = 0; j < 4; ++j) b |= (u[4 * i + j] & 3) << (2 * j);
      out[i] = (uint8_t)b;
    }
  } else {
    for (int i = 0; i < D; ++i) out[i] = u[i];
  }
}

void unpack_codes(int mode, const uint8_t* bytes, int D, uint8_t* u) {
  if (mode == MODE_INT4 || mode == MODE_INT4_STEGO) {
    for (int i = 0; i < D / 2; ++i) {
      u[2 * i] = bytes[i] & 15;
      u[2 * i + 1] = bytes[i] >> 4;
    }
  } else if (mode == MODE_INT2) {
    for (int i = 0; i < D / 4; ++i)
      for (int j = 0; j < 4; ++j) u[4 * i + j] = (bytes[i] >> (2 * j)) & 3;
  } else {
    for (int i = 0; i < D; ++i) u[i] = bytes[i];
  }
}

// ---------------------------------------------------------------------------
// One INT4 / INT2 row: RHT (optional), per-row asymmetric scale and zero point,
// codes, packing, pad = [fp16 s | fp16 m].
void quant_row_token_head(int mode, const float* xin, int D, const int8_t* signs, uint8_t* row) {
  std::vector<float> x(xin, xin + D);
  if (signs) rht_forward_f32(x.data(), D, signs);  // NULL signs: RHT off
  float mn = x[0], mx = x[0];
  for (int i = 1; i < D; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  mn = mn + 0.0f;  // -0 -> +0, so the result does not depend on min order
  mx = mx + 0.0f;
  const int levels = (1 << code_bits(mode)) - 1;
  float s = (mx - mn) / (float)levels;
  uint16_t s_h = f16_saturate(s);
  uint16_t m_h = f16_saturate(mn);
  float S = f16_decode(s_h), M = f16_decode(m_h);
  std::vector<uint8_t> u(D);
  for (int i = 0; i < D; ++i) {
    if (S == 0.0f) {
      u[i] = 0;
      continue;
    }
    float t = (x[i] - M) / S;
    float r = std::nearbyint(t);  // round half to even
    if (r < 0.0f) r = 0.0f;
    if (r > (float)levels) r = (float)levels;
    u[i] = (uint8_t)r;
  }
  const int data = D * code_bits(mode) / 8;
  pack_codes(mode, u.data(), D, row);
  row[data + 0] = (uint8_t)(s_h & 0xFF);
  row[data + 1] = (uint8_t)(s_h >> 8);
  row[data + 2] = (uint8_t)(m_h & 0xFF);
  row[data + 3] = (uint8_t)(m_h >> 8);
}

// One INT4 row whose 4-byte pad is an fp32 scale with the integer zero point
// in its low 4 mantissa bits.
float bits_to_float(uint32_t b) {
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}
uint32_t float_to_bits(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return b;
}
void quant_row_stego(const float* xin, int D, const int8_t* signs, uint8_t* row) {
  std::vector<float> x(xin, xin + D);
  if (signs) rht_forward_f32(x.data(), D, signs);
  float mn = x[0], mx = x[0];
  for (int i = 1; i < D; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  const float lo = mn < 0.0f ? mn : 0.0f;  // the grid holds 0 (code zp)
  const float hi = mx > 0.0f ? mx : 0.0f;
  float s = (hi - lo) / 15.0f;
  const uint32_t sb = float_to_bits(s) & ~15u;  // the low 4 bits carry the zero point
  const float st = bits_to_float(sb);
  int zp = 0;
  if (st != 0.0f) {
    float r = std::nearbyint(-lo / st);
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    zp = (int)r;
  }
  std::vector<uint8_t> u(D);
  for (int i = 0; i < D; ++i) {
    if (st == 0.0f) {
      u[i] = 0;
      continue;
    }
    float r = std::nearbyint(x[i] / st) + (float)zp;
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    u[i] = (uint8_t)r;
  }
  pack_codes(MODE_INT4_STEGO, u.data(), D, row);
  const uint32_t pad = sb | (uint32_t)zp;
  for (int b = 0; b < 4; ++b) row[D / 2 + b] = (uint8_t)(pad >> (8 * b));
}

// One INT8 / FP8 row with a symmetric scale per (token, kv_head): RHT
// (optional), amax = max |x|, s = amax / 127 (INT8) or amax / 448 (FP8, the
// largest E4M3 value), code of x / s per element, pad = fp32 s.
void quant_row_byte_token_head(int mode, const float* xin, int D, const int8_t* signs, uint8_t* row) {
  std::vector<float> x(xin, xin + D);
  if (signs) rht_forward_f32(x.data(), D, signs);
  float amax = 0.0f;
  for (int i = 0; i < D; ++i) {
    const float a = std::fabs(x[i]);
    if (a > amax) amax = a;
  }
  const float s = amax / (mode == MODE_INT8_TOKEN_HEAD ? 127.0f : 448.0f);
  for (int i = 0; i < D; ++i) {
    uint8_t c = 0;
    if (s != 0.0f) {
      const float t = x[i] / s;
      if (mode == MODE_INT8_TOKEN_HEAD) {
        float r = std::nearbyint(t);
        if (r < -127.0f) r = -127.0f;
        if (r > 127.0f) r = 127.0f;
        c = (uint8_t)(int8_t)(int)r;
      } else {
        c = e4m3_round_saturate(t);
      }
    }
    row[i] = c;
  }
  const uint32_t pad = float_to_bits(s);
  for (int b = 0; b < 4; ++b) row[D + b] = (uint8_t)(pad >> (8 * b));
}

void quant_row_int8(const float* x, int D, const float* amax, uint8_t* row) {
  for (int c = 0; c < D; ++c) {
    float s = amax[c] / 127.0f;
    int q = 0;
    if (s != 0.0f) {
      float r = std::nearbyint(x[c] / s);
      if (r < -127.0f) r = -127.0f;
      if (r > 127.0f) r = 127.0f;
      q = (int)r;
    }
    row[c] = (uint8_t)(int8_t)q;
  }
}

// Dequantised row mapped back to the input domain, in double.
void dequant_row(int mode, const uint8_t* row, int D, const int8_t* signs, const float* amax,
                 double* out) {
  std::vector<uint8_t> u(D);
  unpack_codes(mode, row, D, u.data());
  if (mode == MODE_INT8) {
    for (int c = 0; c < D; ++c) {
      float s = amax[c] / 127.0f;
      out[c] = (double)(int8_t)u[c] * (double)s;
    }
    return;
  }
  const int data = D * code_bits(mode) / 8;
  if (byte_token_head(mode)) {
    const uint32_t pad = (uint32_t)row[D] | ((uint32_t)row[D + 1] << 8) | ((uint32_t)row[D + 2] << 16) |
                         ((uint32_t)row[D + 3] << 24);
    const double S = bits_to_float(pad);
    for (int i = 0; i < D; ++i)
      out[i] = (mode == MODE_INT8_TOKEN_HEAD ? (double)(int8_t)u[i] : e4m3_decode(u[i])) * S;
  } else if (mode == MODE_INT4_STEGO) {
    const uint32_t pad = (uint32_t)row[data] | ((uint32_t)row[data + 1] << 8) | ((uint32_t)row[data + 2] << 16) |
                         ((uint32_t)row[data + 3] << 24);
    const int zp = (int)(pad & 15u);
    const double S = bits_to_float(pad & ~15u);
    for (int i = 0; i < D; ++i) out[i] = (double)((int)u[i] - zp) * S;
  } else {
    uint16_t s_h = (uint16_t)(row[data] | (row[data + 1] << 8));
    uint16_t m_h = (uint16_t)(row[data + 2] | (row[data + 3] << 8));
    double S = f16_decode(s_h), M = f16_decode(m_h);
    for (int i = 0; i < D; ++i) out[i] = (double)u[i] * S + M;
  }
  if (signs) {  // inverse RHT: d * (H y) / D
    wht_double(out, D);
    for (int i = 0; i < D; ++i) out[i] = out[i] * (double)signs[i] / (double)D;
  }
}

}  // namespace

// ===========================================================================
// exported C entry points (ctypes)

extern "C" {

struct OrcCache {
  uint8_t* k_pages;
  uint8_t* v_pages;
  int32_t num_blocks, num_kv_heads, block_size, head_dim, mode;
  const int8_t* signs;
  float* ch_amax;   // [2][Hkv][D]
  int32_t* ch_ready;
};

struct OrcPaging {
  const int32_t* table;  // [rows][max_blocks]
  int32_t headwise;
  int32_t max_blocks;
  int32_t batch;
  const int32_t* seq_lens;
  const int32_t* window;  // [Hkv] or NULL
  int32_t sink;
};

int32_t orc_row_bytes(int32_t mode, int32_t D) { return row_bytes(mode, D); }
uint16_t orc_f16_round(float x) { return f16_round_nearest_even(x); }
uint16_t orc_f16_saturate(float x) { return f16_saturate(x); }
float orc_f16_decode(uint16_t h) { return f16_decode(h); }
void orc_rht_forward(float* x, int32_t D, const int8_t* signs) { rht_forward_f32(x, D, signs); }
void orc_pack_codes(int32_t mode, const uint8_t* u, int32_t D, uint8_t* out) { pack_codes(mode, u, D, out); }
void orc_unpack_codes(int32_t mode, const uint8_t* b, int32_t D, uint8_t* u) { unpack_codes(mode, b, D, u); }
int32_t orc_signed_code(int32_t mode, int32_t u) {
  // INT4 / INT2 offset encoding: stored u in [0, 2^b - 1] is q = u - 2^(b-1).
  return u - (1 << (code_bits(mode) - 1));
}
double orc_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
uint8_t orc_e4m3_round(float x) { return e4m3_round_saturate(x); }
void orc_quant_row(int32_t mode, const float* x, int32_t D, const int8_t* signs, uint8_t* row) {
  if (mode == MODE_INT4_STEGO) quant_row_stego(x, D, signs, row);
  else if (byte_token_head(mode)) quant_row_byte_token_head(mode, x, D, signs, row);
  else quant_row_token_head(mode, x, D, signs, row);
}
void orc_dequant_row(int32_t mode, const uint8_t* row, int32_t D, const int8_t* signs,
                     const float* amax, double* out) {
  dequant_row(mode, row, D, signs, amax, out);
}

static int32_t table_row(const OrcPaging* pg, int b, int h, int Hkv) {
  return pg->headwise ? b * Hkv + h : b;
}

// Quantise `num_tokens` new tokens of K and V and scatter them.  Returns the
// OR of ERR_* bits for rows it had to skip.
int32_t orc_write(const OrcCache* c, const OrcPaging* pg, const void* k, const void* v, int32_t dtype,
                  const int32_t* cu_new, int32_t num_tokens) {
  const int D = c->head_dim, Hkv = c->num_kv_heads, bs = c->block_size, mode = c->mode;
  const int R = row_bytes(mode, D);
  int32_t err = 0;
  if (num_tokens <= 0) return 0;
  if (mode == MODE_INT8 && *c->ch_ready == 0) {
    // First K/V of the layer: channel amax over every token given.
    for (int kv = 0; kv < 2; ++kv) {
      const void* src = kv ? v : k;
      for (int h = 0; h < Hkv; ++h)
        for (int ch = 0; ch < D; ++ch) {
          float a = 0.0f;
          for (int t = 0; t < num_tokens; ++t) {
            float x = std::fabs(widen(src, dtype, ((size_t)t * Hkv + h) * D + ch));
            if (x > a) a = x;
          }
          c->ch_amax[((size_t)kv * Hkv + h) * D + ch] = a;
        }
    }
    *c->ch_ready = 1;
  }
  std::vector<float> x(D);
  for (int b = 0; b < pg->batch; ++b) {
    const int n = cu_new[b + 1] - cu_new[b];
    const int L = pg->seq_lens[b];
    if (n == 0) continue;
    if (L < 0 || n > L) {
      err |= ERR_SEQ_LEN;
      continue;
    }
    for (int i = 0; i < n; ++i) {
      const int t = cu_new[b] + i;
      const int p = L - n + i;
      for (int h = 0; h < Hkv; ++h) {
        const int row = table_row(pg, b, h, Hkv);
        const int lb = p / bs;
        if (lb >= pg->max_blocks) {
          err |= ERR_TABLE_RANGE;
          continue;
        }
        const int blk = pg->table[(size_t)row * pg->max_blocks + lb];
        if (blk < 0) continue;  // evicted: nothing is written
        if (blk >= c->num_blocks) {
          err |= ERR_BLOCK_RANGE;
          continue;
        }
        for (int kv = 0; kv < 2; ++kv) {
          const void* src = kv ? v : k;
          for (int d = 0; d < D; ++d) x[d] = widen(src, dtype, ((size_t)t * Hkv + h) * D + d);
          uint8_t* pages = kv ? c->v_pages : c->k_pages;
          uint8_t* dst = pages + (((size_t)blk * Hkv + h) * bs + (p % bs)) * R;
          if (mode == MODE_INT8)
            quant_row_int8(x.data(), D, c->ch_amax + ((size_t)kv * Hkv + h) * D, dst);
          else if (mode == MODE_INT4_STEGO)
            quant_row_stego(x.data(), D, c->signs, dst);
          else if (byte_token_head(mode))
            quant_row_byte_token_head(mode, x.data(), D, c->signs, dst);
          else
            quant_row_token_head(mode, x.data(), D, c->signs, dst);
        }
      }
    }
  }
  return err;
}

// Gather and dequantise the K and V rows of `num_tokens` positions.  Sequence
// b's tokens cu[b] .. cu[b+1]-1 are its positions seq_lens[b] - n_b ..
// seq_lens[b] - 1 (the map of orc_write).  out: double [num_tokens][Hkv][D]
// each; a -1 table entry gives a zero row; a row that cannot be located
// (too many tokens for the sequence, a position past the table row, a block
// id past the pool) gives a zero row and an ERR_* bit.
int32_t orc_gather_chunk(const OrcCache* c, const OrcPaging* pg, const int32_t* cu, int32_t num_tokens,
                         const void* k_chunk, const void* v_chunk, int32_t chunk_dtype, const int32_t* cu_chunk,
                         double* k_out, double* v_out);

int32_t orc_gather(const OrcCache* c, const OrcPaging* pg, const int32_t* cu, int32_t num_tokens, double* k_out,
                   double* v_out) {
  return orc_gather_chunk(c, pg, cu, num_tokens, nullptr, nullptr, DT_F32, nullptr, k_out, v_out);
}

// The same gather where the current chunk comes in full precision (the Ascend
// INT8 plugin's 运行机制 and FastDeploy PR #5173 attend to the chunk being
// written; this variant takes its K / V as given, not as stored): positions
// seq_lens[b] - m_b .. seq_lens[b] - 1, m_b = cu_chunk[b+1] - cu_chunk[b], are
// read from rows cu_chunk[b] .. of k_chunk / v_chunk [rows][Hkv][D] (fp32 or
// bf16 bits, the layout kvq_write reads), the earlier ones from the cache.
// NULL k_chunk gives the plain gather.
int32_t orc_gather_chunk(const OrcCache* c, const OrcPaging* pg, const int32_t* cu, int32_t num_tokens,
                         const void* k_chunk, const void* v_chunk, int32_t chunk_dtype, const int32_t* cu_chunk,
                         double* k_out, double* v_out) {
  const int D = c->head_dim, Hkv = c->num_kv_heads, bs = c->block_size, mode = c->mode;
  const int R = row_bytes(mode, D);
  int32_t err = 0;
  for (size_t i = 0; i < (size_t)num_tokens * Hkv * D; ++i) k_out[i] = v_out[i] = 0.0;
  for (int b = 0; b < pg->batch; ++b) {
    const int n = cu[b + 1] - cu[b];
    const int L = pg->seq_lens[b];
    if (n == 0) continue;
    if (L < 0 || n > L) {
      err |= ERR_SEQ_LEN;
      continue;
    }
    const int m = k_chunk ? cu_chunk[b + 1] - cu_chunk[b] : 0;
    if (m < 0 || m > L) {
      err |= ERR_SEQ_LEN;
      continue;
    }
    for (int i = 0; i < n; ++i) {
      const int t = cu[b] + i;
      const int p = L - n + i;
      for (int h = 0; h < Hkv; ++h) {
        if (p >= L - m) {  // the current chunk, as given
          const size_t src = ((size_t)(cu_chunk[b] + p - (L - m)) * Hkv + h) * D;
          const size_t o = ((size_t)t * Hkv + h) * D;
          for (int d = 0; d < D; ++d) {
            k_out[o + d] = widen(k_chunk, chunk_dtype, src + d);
            v_out[o + d] = widen(v_chunk, chunk_dtype, src + d);
          }
          continue;
        }
        const int lb = p / bs;
        if (lb >= pg->max_blocks) {
          err |= ERR_TABLE_RANGE;
          continue;
        }
        const int blk = pg->table[(size_t)table_row(pg, b, h, Hkv) * pg->max_blocks + lb];
        if (blk < 0) continue;  // evicted: a zero row
        if (blk >= c->num_blocks) {
          err |= ERR_BLOCK_RANGE;
          continue;
        }
        const size_t off = (((size_t)blk * Hkv + h) * bs + (p % bs)) * R;
        const size_t o = ((size_t)t * Hkv + h) * D;
        dequant_row(mode, c->k_pages + off, D, c->signs, c->ch_amax ? c->ch_amax + (size_t)h * D : nullptr,
                    k_out + o);
        dequant_row(mode, c->v_pages + off, D, c->signs,
                    c->ch_amax ? c->ch_amax + ((size_t)Hkv + h) * D : nullptr, v_out + o);
      }
    }
  }
  return err;
}

// Keys and values one (sequence, kv head) can see, in the input domain.
struct Deq {
  int b = -1, h = -1, n = 0;
  std::vector<double> K, V;
  std::vector<char> ok;
};

// Sequence and position of every selected query row.  Decode (cu_q == NULL):
// row i is sequence i's query at seq_lens[i] - 1.  Prefill: row i in
// [cu_q[b], cu_q[b+1]) is at seq_lens[b] - n_b + (i - cu_q[b]).
static void query_rows(const OrcPaging* pg, const int32_t* cu_q, int32_t total_q, const int32_t* rows,
                       int32_t& n_rows, std::vector<int32_t>& sel, std::vector<int32_t>& seq,
                       std::vector<int32_t>& pos) {
  if (rows) sel.assign(rows, rows + n_rows);
  else {
    for (int i = 0; i < total_q; ++i) sel.push_back(i);
    n_rows = total_q;
  }
  seq.assign(n_rows, 0);
  pos.assign(n_rows, 0);
  for (int r = 0; r < n_rows; ++r) {
    const int i = sel[r];
    int b = 0, p = 0;
    if (!cu_q) {
      b = i;
      p = pg->seq_lens[b] - 1;
    } else {
      while (b + 1 <= pg->batch && cu_q[b + 1] <= i) ++b;
      const int n = cu_q[b + 1] - cu_q[b];
      p = pg->seq_lens[b] - n + (i - cu_q[b]);
    }
    seq[r] = b;
    pos[r] = p;
  }
}

// Softmax attention per (selected row, q head), in double, over the keys of
// `deq` that the row's position sees (causal, window + sink).
static void attention_rows(const OrcPaging* pg, const std::vector<Deq>& deq, const std::vector<int32_t>& sel,
                           const std::vector<int32_t>& seq, const std::vector<int32_t>& pos, int32_t n_rows,
                           const void* q, int32_t dtype, int32_t Hq, int Hkv, int D, float scale, double* out,
                           int32_t threads) {
  const int g = Hq / Hkv;
  std::atomic<int> next(0);
  const int n_items = n_rows * Hq;
  auto attn_worker = [&]() {
    std::vector<double> z, qd(D);
    for (;;) {
      int w = next.fetch_add(1);
      if (w >= n_items) break;
      const int r = w / Hq, hq = w % Hq, h = hq / g;
      const int b = seq[r], p = pos[r];
      const Deq& dq = deq[(size_t)b * Hkv + h];
      double* o = out + ((size_t)r * Hq + hq) * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int d = 0; d < D; ++d) qd[d] = (double)widen(q, dtype, ((size_t)sel[r] * Hq + hq) * D + d);
      const int W = pg->window ? pg->window[h] : 0;
      z.assign(dq.n, -INFINITY);
      double zmax = -INFINITY;
      for (int j = 0; j < dq.n && j <= p; ++j) {
        if (!dq.ok[j]) continue;
        if (W > 0 && !(j < pg->sink || j > p - W)) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * dq.K[(size_t)j * D + d];
        z[j] = (double)scale * dot;
        if (z[j] > zmax) zmax = z[j];
      }
      if (zmax == -INFINITY) continue;  // no visible key: output 0
      double l = 0.0;
      for (int j = 0; j < dq.n && j <= p; ++j) {
        if (z[j] == -INFINITY) continue;
        const double e = std::exp(z[j] - zmax);
        l += e;
        for (int d = 0; d < D; ++d) o[d] += e * dq.V[(size_t)j * D + d];
      }
      for (int d = 0; d < D; ++d) o[d] /= l;
    }
  };
  if (threads < 1) threads = 1;
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) pool.emplace_back(attn_worker);
  for (auto& th : pool) th.join();
}

// Largest position each (sequence, kv head) must provide keys up to.
static std::vector<int> needed_keys(const OrcPaging* pg, int Hkv, const std::vector<int32_t>& seq,
                                    const std::vector<int32_t>& pos, int32_t n_rows) {
  std::vector<int> need((size_t)pg->batch * Hkv, -1);
  for (int r = 0; r < n_rows; ++r)
    for (int h = 0; h < Hkv; ++h) {
      int& m = need[(size_t)seq[r] * Hkv + h];
      if (pos[r] > m) m = pos[r];
    }
  return need;
}

// Attention for selected query rows over the paged cache.  `rows` lists the
// query rows to compute (NULL = all total_q); out is double [n_rows][Hq][D].
int32_t orc_attention(const OrcCache* c, const OrcPaging* pg, const void* q, int32_t dtype, int32_t Hq,
                      const int32_t* cu_q, int32_t total_q, float scale, const int32_t* rows,
                      int32_t n_rows, double* out, int32_t threads) {
  const int D = c->head_dim, Hkv = c->num_kv_heads, bs = c->block_size, mode = c->mode;
  const int R = row_bytes(mode, D);
  if (Hq % Hkv) return -1;
  std::vector<int32_t> sel, seq, pos;
  query_rows(pg, cu_q, total_q, rows, n_rows, sel, seq, pos);
  int32_t err = 0;
  // Phase 1: dequantise the keys each needed (sequence, kv head) can see.
  std::vector<Deq> deq((size_t)pg->batch * Hkv);
  const std::vector<int> need = needed_keys(pg, Hkv, seq, pos, n_rows);
  std::vector<int> items;
  for (size_t it = 0; it < need.size(); ++it)
    if (need[it] >= 0) items.push_back((int)it);
  if (threads < 1) threads = 1;
  std::atomic<int> next(0);
  std::atomic<int32_t> aerr(0);
  auto deq_worker = [&]() {
    for (;;) {
      int w = next.fetch_add(1);
      if (w >= (int)items.size()) break;
      const int it = items[w];
      const int b = it / Hkv, h = it % Hkv;
      Deq& dq = deq[it];
      dq.b = b;
      dq.h = h;
      dq.n = std::min(need[it] + 1, pg->seq_lens[b]);
      if (dq.n < 0) dq.n = 0;
      dq.K.assign((size_t)dq.n * D, 0.0);
      dq.V.assign((size_t)dq.n * D, 0.0);
      dq.ok.assign(dq.n, 0);
      const int row = table_row(pg, b, h, Hkv);
      for (int j = 0; j < dq.n; ++j) {
        const int lb = j / bs;
        if (lb >= pg->max_blocks) {
          aerr |= ERR_TABLE_RANGE;
          continue;
        }
        const int blk = pg->table[(size_t)row * pg->max_blocks + lb];
        if (blk < 0) continue;  // evicted: never addressed
        if (blk >= c->num_blocks) {
          aerr |= ERR_BLOCK_RANGE;
          continue;
        }
        const size_t off = (((size_t)blk * Hkv + h) * bs + (j % bs)) * R;
        dequant_row(mode, c->k_pages + off, D, c->signs,
                    c->ch_amax ? c->ch_amax + ((size_t)0 * Hkv + h) * D : nullptr,
                    &dq.K[(size_t)j * D]);
        dequant_row(mode, c->v_pages + off, D, c->signs,
                    c->ch_amax ? c->ch_amax + ((size_t)1 * Hkv + h) * D : nullptr,
                    &dq.V[(size_t)j * D]);
        dq.ok[j] = 1;
      }
    }
  };
  {
    std::vector<std::thread> pool;
    for (int t = 0; t < threads; ++t) pool.emplace_back(deq_worker);
    for (auto& th : pool) th.join();
  }
  // Phase 2: softmax attention per (row, q head), in double.
  attention_rows(pg, deq, sel, seq, pos, n_rows, q, dtype, Hq, Hkv, D, scale, out, threads);
  return err | aerr.load();
}

// Attention over dense K / V rows: the dense prefill that follows a gather
// (FastDeploy PR #5173, the dynamic_quant_get_kv_from_cache op; Ascend INT8
// plugin, 运行机制: prefill gathers and dequantises, then attends).  Sequence
// b's key j is row cu_kv[b] + j of k, v [rows][Hkv][D] (fp32 values or bf16
// bits, `kv_dtype`); the table fields of `pg` are not used; queries and
// visibility as in orc_attention.
int32_t orc_dense_attention(const void* k, const void* v, int32_t kv_dtype, const int32_t* cu_kv,
                            const OrcPaging* pg, int32_t Hkv, int32_t D, const void* q, int32_t dtype, int32_t Hq,
                            const int32_t* cu_q, int32_t total_q, float scale, const int32_t* rows, int32_t n_rows,
                            double* out, int32_t threads) {
  if (Hq % Hkv) return -1;
  std::vector<int32_t> sel, seq, pos;
  query_rows(pg, cu_q, total_q, rows, n_rows, sel, seq, pos);
  std::vector<Deq> deq((size_t)pg->batch * Hkv);
  const std::vector<int> need = needed_keys(pg, Hkv, seq, pos, n_rows);
  int32_t err = 0;
  for (int b = 0; b < pg->batch; ++b)
    if (cu_kv[b + 1] - cu_kv[b] != pg->seq_lens[b]) err |= ERR_SEQ_LEN;
  if (err) return err;
  for (size_t it = 0; it < need.size(); ++it) {
    if (need[it] < 0) continue;
    const int b = (int)it / Hkv, h = (int)it % Hkv;
    Deq& dq = deq[it];
    dq.b = b;
    dq.h = h;
    dq.n = std::max(0, std::min(need[it] + 1, pg->seq_lens[b]));
    dq.K.assign((size_t)dq.n * D, 0.0);
    dq.V.assign((size_t)dq.n * D, 0.0);
    dq.ok.assign(dq.n, 1);
    for (int j = 0; j < dq.n; ++j)
      for (int d = 0; d < D; ++d) {
        const size_t idx = ((size_t)(cu_kv[b] + j) * Hkv + h) * D + d;
        dq.K[(size_t)j * D + d] = widen(k, kv_dtype, idx);
        dq.V[(size_t)j * D + d] = widen(v, kv_dtype, idx);
      }
  }
  attention_rows(pg, deq, sel, seq, pos, n_rows, q, dtype, Hq, Hkv, D, scale, out, threads);
  return 0;
}

int32_t orc_rounding_mode_is_nearest(void) { return std::fegetround() == FE_TONEAREST; }

}  // extern "C"
