// kvq_row.cuh -- the write path's row arithmetic, shared by every kernel that
// writes cache rows (the write kernels and the decode's fused write).
//
// vLLM PR #40835 review summary ("INT4 per-token-head KV cache for the Triton
// backend"), 实现拆解 item 2: rotate each row with a random Hadamard transform,
// take a per-token-head scale and zero point, round and pack; 关键源码片段:
// row = head_size/2 data bytes + a 4-byte scale pad.  The INT8 / FP8
// token-head rows (same page, 功能与动机 / 关联脉络): one symmetric fp32 scale
// per row after the D code bytes.
#pragma once

#include "kvq_common.cuh"

namespace kvq {

// The quantiser's code before clamping is rint(RN(d / s)).  It is first
// taken as the nearest integer k of t = RN(d r), r = RN(1 / s):
// t = (d / s)(1 + e1)(1 + e2) with |e1|, |e2| <= 2^-24, so |t - d/s| <=
// |d/s| 2^-22.99, below 2^-14.9 while |t| < 256.  Where t is farther than
// 2^-14 from every half-integer, the exact quotient and its correctly rounded
// value lie on the same side of the same half-integer as t and round to k;
// where |t| >= 256 every code in use (at most 127 in size) clamps to the same
// end either way.  near_half marks the elements within 2^-14 of a
// half-integer (ties among them; for |t| >= 2^22 possibly more, which only
// costs time); a lane with one of them, or whose 1 / s is not a finite
// float, recomputes its codes with the correctly rounded division.  k comes from adding and
// removing 1.5 * 2^23 (round-half-even for |t| < 2^22; a larger |t| keeps its
// sign and size, which is all the clamp needs).
__device__ __forceinline__ float quotient_rint_fast(float d, float r, bool& near_half) {
  const float t = __fmul_rn(d, r);
  const float k = __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);
  near_half |= fabsf(__fsub_rn(t, k)) >= 0.49993896484375f;  // 0.5 - 2^-14
  return k;
}

// The RHT signs of a lane's EPL elements as float sign-bit masks (0 or
// 0x80000000): x XOR mask is the exact product with the +-1 sign.  Loaded
// once and reused for every row the lane rotates.
template <int EPL>
struct RowSigns {
  uint32_t m[EPL];
  bool on;
};
template <int EPL>
__device__ __forceinline__ RowSigns<EPL> load_row_signs(const int8_t* signs, int sub) {
  RowSigns<EPL> r;
  r.on = signs != nullptr;
#pragma unroll
  for (int i = 0; i < EPL; ++i) r.m[i] = 0;
  if (!r.on) return r;
  const int8_t* p = signs + sub * EPL;
  if constexpr (EPL % 4 == 0) {
    if ((reinterpret_cast<uintptr_t>(signs) & (EPL >= 16 ? 15 : EPL - 1)) == 0) {  // whole words
      uint32_t w[EPL / 4];
      if constexpr (EPL >= 16) {
#pragma unroll
        for (int v = 0; v < EPL / 16; ++v) {
          const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + v);
          w[4 * v] = q.x; w[4 * v + 1] = q.y; w[4 * v + 2] = q.z; w[4 * v + 3] = q.w;
        }
      } else if constexpr (EPL == 8) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = q.x; w[1] = q.y;
      } else {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i) r.m[i] = (w[i / 4] << (24 - 8 * (i % 4))) & 0x80000000u;
      return r;
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) r.m[i] = (uint32_t)(__ldg(p + i) & 0x80) << 24;
  return r;
}

// Rotate, quantise, pack and store one row at dst.  The row is held by LPR
// consecutive lanes (32: a warp per row; 8: four rows per warp), lane `sub`
// of the group holding elements sub * EPL .. + EPL - 1 (EPL = D / LPR).
// Every step is one IEEE operation in a fixed order (butterfly stages
// h = 1, 2, ..., D/2, exact min / max, one division for the scale, fp16 RNE,
// one subtract and one correctly rounded divide per element (reached through
// a multiply wherever that provably gives the same integer),
// round-half-even), so the bytes
// match any other evaluation in that order, whatever LPR.  Every lane of
// the warp must call this (the shuffles span the warp); `store` is false
// for a group whose row is not written.
template <int MODE, int D, bool STEGO, int LPR>
__device__ __forceinline__ void quantise_store_row(const RowSigns<D / LPR>& sg, float (&x)[D / LPR], uint8_t* dst,
                                                   int lane, bool store) {
  constexpr int EPL = D / LPR;
  constexpr int BITS = mode_bits(MODE);
  constexpr int LEVELS = (1 << BITS) - 1;
  constexpr int DATA = data_bytes(MODE, D);
  const int sub = lane & (LPR - 1);
  if (sg.on) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) x[i] = __uint_as_float(__float_as_uint(x[i]) ^ sg.m[i]);
    // stages h = 1 .. EPL/2 in lane, then h = EPL .. D/2 over the group's lanes
#pragma unroll
    for (int h = 1; h < EPL; h <<= 1) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (i & h) continue;
        const float a = x[i], c = x[i + h];
        x[i] = __fadd_rn(a, c);
        x[i + h] = __fsub_rn(a, c);
      }
    }
#pragma unroll
    for (int lm = 1; lm < LPR; lm <<= 1) {
      // lower lane holds x_j: x_j + x_{j+h}; upper lane holds x_{j+h}: x_j - x_{j+h},
      // both as one exact fma(+-1, x, o)
      const float sg = (sub & lm) ? -1.0f : 1.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, x[i], lm);
        x[i] = __fmaf_rn(sg, x[i], o);
      }
    }
  }
  // codes: NBITS = EPL * BITS bits per lane, in NW words (at least one)
  constexpr int NBITS = EPL * BITS;
  constexpr int NW = NBITS >= 32 ? NBITS / 32 : 1;
  constexpr int CPW = 32 / BITS;  // codes per word
  uint32_t bits[NW];
#pragma unroll
  for (int k = 0; k < NW; ++k) bits[k] = 0;
  uint32_t pad;
  if constexpr (byte_token_head(MODE)) {
    // symmetric: s = amax / 127 (INT8) or amax / 448 (largest E4M3 value)
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int lm = 1; lm < LPR; lm <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, lm));
    const float s = __fdiv_rn(amax, MODE == MODE_I8T ? 127.0f : 448.0f);
    if (s != 0.0f) {
      if constexpr (MODE == MODE_I8T) {
        const float rs = __frcp_rn(s);
        bool exact = !(rs <= 3.402823466e38f);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const float k = quotient_rint_fast(x[i], rs, exact);
          bits[i / CPW] |= ((uint32_t)(int)fminf(fmaxf(k, -127.0f), 127.0f) & 0xFFu) << ((i % CPW) * BITS);
        }
        if (exact) {  // rare: recompute this lane's codes with the division
#pragma unroll
          for (int k = 0; k < NW; ++k) bits[k] = 0;
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const float k = rintf(__fdiv_rn(x[i], s));
            bits[i / CPW] |= ((uint32_t)(int)fminf(fmaxf(k, -127.0f), 127.0f) & 0xFFu) << ((i % CPW) * BITS);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const uint32_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[i], s), __NV_SATFINITE, __NV_E4M3);  // nearest even
          bits[i / CPW] |= c << ((i % CPW) * BITS);
        }
      }
    }
    pad = __float_as_uint(s);
  } else {
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < EPL; ++i) {
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
#pragma unroll
    for (int lm = 1; lm < LPR; lm <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, lm));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, lm));
    }
    mn = __fadd_rn(mn, 0.0f);  // canonical +0
    mx = __fadd_rn(mx, 0.0f);
    if constexpr (STEGO) {
      // the grid (u - zp) * s holds 0: it spans min(mn, 0) .. max(mx, 0); the
      // scale's low 4 mantissa bits are cleared and carry the zero point
      const float lo = mn < 0.0f ? mn : 0.0f, hi = mx > 0.0f ? mx : 0.0f;
      const uint32_t sb = __float_as_uint(__fdiv_rn(__fsub_rn(hi, lo), (float)LEVELS)) & ~15u;
      const float st = __uint_as_float(sb);
      float zp = 0.0f;
      if (st != 0.0f) zp = fminf(fmaxf(rintf(__fdiv_rn(-lo, st)), 0.0f), (float)LEVELS);
      if (st != 0.0f) {
        const float rst = __frcp_rn(st);
        bool exact = !(rst <= 3.402823466e38f);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const float r = __fadd_rn(quotient_rint_fast(x[i], rst, exact), zp);
          bits[i / CPW] |= (uint32_t)fminf(fmaxf(r, 0.0f), (float)LEVELS) << ((i % CPW) * BITS);
        }
        if (exact) {  // rare: recompute this lane's codes with the division
#pragma unroll
          for (int k = 0; k < NW; ++k) bits[k] = 0;
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const float r = __fadd_rn(rintf(__fdiv_rn(x[i], st)), zp);
            bits[i / CPW] |= (uint32_t)fminf(fmaxf(r, 0.0f), (float)LEVELS) << ((i % CPW) * BITS);
          }
        }
      }
      pad = sb | (uint32_t)zp;
    } else {
      const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)LEVELS);
      const uint16_t s_h = f16_sat_bits(s);
      const uint16_t m_h = f16_sat_bits(mn);
      const float S = __half2float(__ushort_as_half(s_h));
      const float M = __half2float(__ushort_as_half(m_h));
      if (S != 0.0f) {
        const float rS = __frcp_rn(S);
        bool exact = !(rS <= 3.402823466e38f);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const float k = quotient_rint_fast(__fsub_rn(x[i], M), rS, exact);
          bits[i / CPW] |= (uint32_t)fminf(fmaxf(k, 0.0f), (float)LEVELS) << ((i % CPW) * BITS);
        }
        if (exact) {  // rare: recompute this lane's codes with the division
#pragma unroll
          for (int k = 0; k < NW; ++k) bits[k] = 0;
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const float k = rintf(__fdiv_rn(__fsub_rn(x[i], M), S));
            bits[i / CPW] |= (uint32_t)fminf(fmaxf(k, 0.0f), (float)LEVELS) << ((i % CPW) * BITS);
          }
        }
      }
      pad = (uint32_t)s_h | ((uint32_t)m_h << 16);
    }
  }
  if constexpr (NBITS >= 32) {
    // this lane's bytes sub * NBITS/8 ..: whole words (rows are 4-byte aligned)
    if (store) {
#pragma unroll
      for (int k = 0; k < NW; ++k) *reinterpret_cast<uint32_t*>(dst + sub * (NBITS / 8) + 4 * k) = bits[k];
    }
  } else {
    // 32 / NBITS lanes share a word: OR their bits into the group's first lane
    constexpr int LPW = 32 / NBITS;
    uint32_t v = bits[0] << ((sub % LPW) * NBITS);
#pragma unroll
    for (int o = 1; o < LPW; o <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    if (store && sub % LPW == 0) *reinterpret_cast<uint32_t*>(dst + 4 * (sub / LPW)) = v;
  }
  if (store && sub == 0) *reinterpret_cast<uint32_t*>(dst + DATA) = pad;
}

}  // namespace kvq
