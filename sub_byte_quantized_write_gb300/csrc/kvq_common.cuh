// kvq_common.cuh -- device helpers shared by the libkvq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace kvq {

// Kernel code families.  The API's zero-point-in-scale INT4 mode (3) runs as
// MODE_INT4 with the `stego` flag of the parameters; 4 and 5 are the INT8 /
// FP8 rows with one fp32 scale per (token, kv head); 6 is the dense prefill's
// bf16 rows (no codes, no scale).
enum { MODE_INT4 = 0, MODE_INT2 = 1, MODE_INT8 = 2, MODE_I8T = 4, MODE_F8T = 5, MODE_DBF16 = 6 };
enum { DT_F32 = 0, DT_BF16 = 1 };
enum { DEVERR_BLOCK_RANGE = 1, DEVERR_TABLE_RANGE = 2, DEVERR_SEQ_LEN = 4, DEVERR_TIMEOUT = 8, DEVERR_BOUNDS = 16 };

__host__ __device__ constexpr int mode_bits(int mode) {
  return mode == MODE_INT4 ? 4 : (mode == MODE_INT2 ? 2 : (mode == MODE_DBF16 ? 16 : 8));
}
__host__ __device__ constexpr int data_bytes(int mode, int D) { return D * mode_bits(mode) / 8; }
__host__ __device__ constexpr int row_bytes_of(int mode, int D) {
  return (mode == MODE_INT8 || mode == MODE_DBF16) ? data_bytes(mode, D) : data_bytes(mode, D) + 4;
}
// INT8 / FP8 codes with a symmetric fp32 scale per row (no zero point)
__host__ __device__ constexpr bool byte_token_head(int mode) { return mode == MODE_I8T || mode == MODE_F8T; }

// Two E4M3 codes (bits 0-7 and 8-15 of `pair`) as an fp16 pair, the first in
// the low half; exact, since every E4M3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_half2_bits(uint32_t pair) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(pair & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Four E4M3 bytes with the NaN pattern S.1111.111 replaced by S.1111.110.
// The write path never stores it, but stale bytes of masked rows may, and a
// NaN times a zero weight still poisons a tensor-core sum.  Per byte, the low
// 7 bits plus one carry into bit 7 only when they are all ones.
__device__ __forceinline__ uint32_t e4m3x4_no_nan(uint32_t w) {
  return w ^ ((((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u) >> 7);
}

__device__ __forceinline__ void flag_error(int32_t* dev_error, int bit) {
  if (dev_error) atomicOr(dev_error, bit);
}

// Debug builds (-DKVQ_BOUNDS_CHECK, libkvq_debug.so): indices that a kernel
// computes are checked against their buffers before the access; a failed
// check sets DEVERR_BOUNDS and the access is skipped.  Release builds compile
// the checks away: there the conditions hold by construction.
#ifdef KVQ_BOUNDS_CHECK
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* dev_error) {
  if (!ok) flag_error(dev_error, DEVERR_BOUNDS);
  return ok;
}
#define KVQ_IN_BOUNDS(ok, err) ::kvq::in_bounds((ok), (err))
#else
#define KVQ_IN_BOUNDS(ok, err) true
#endif

// Load EPL consecutive input elements (fp32 or bf16) as fp32 (EPL = 2, 4, 8
// or 16; elem_off a multiple of EPL, so the vector loads are aligned).
template <int EPL>
__device__ __forceinline__ void load_row_elems(const void* base, int dtype, size_t elem_off, float (&x)[EPL]) {
  if (dtype == DT_F32) {
    const float* p = reinterpret_cast<const float*>(base) + elem_off;
    if constexpr (EPL >= 4) {
#pragma unroll
      for (int c = 0; c < EPL / 4; ++c) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p) + c);
        x[4 * c] = v.x; x[4 * c + 1] = v.y; x[4 * c + 2] = v.z; x[4 * c + 3] = v.w;
      }
    } else {
      float2 v = __ldg(reinterpret_cast<const float2*>(p));
      x[0] = v.x; x[1] = v.y;
    }
  } else {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base) + elem_off;
    if constexpr (EPL >= 8) {
#pragma unroll
      for (int c = 0; c < EPL / 8; ++c) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[8 * c + 2 * k] = __uint_as_float(w[k] << 16);
          x[8 * c + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
      }
    } else if constexpr (EPL == 4) {
      uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xFFFF0000u);
      x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    } else {
      uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p));
      x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xFFFF0000u);
    }
  }
}

// Warp-wide Walsh-Hadamard butterfly over D = 32 * EPL elements, lane l
// holding elements l*EPL .. l*EPL+EPL-1.  Stage order h = 1, 2, ..., D/2, each
// pair (j, j+h) -> (x_j + x_{j+h}, x_j - x_{j+h}) in fp32: every stage is a
// single IEEE add or subtract per element, so the result is bit-identical to
// a sequential evaluation in the same stage order.
template <int EPL>
__device__ __forceinline__ void wht_warp(float (&x)[EPL], int lane) {
#pragma unroll
  for (int h = 1; h < EPL; h <<= 1) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (i & h) continue;
      const float a = x[i], b = x[i + h];
      x[i] = __fadd_rn(a, b);
      x[i + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int lm = 1; lm < 32; lm <<= 1) {
    // lower lane holds x_j: x_j + x_{j+h}; upper lane holds x_{j+h}: x_j - x_{j+h}.
    // Both as one fma(+-1, x, o): the product is exact, so the result is the
    // correctly rounded sum or difference, bit for bit.
    const float sg = (lane & lm) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], lm);
      x[i] = __fmaf_rn(sg, x[i], o);
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// fp32 -> fp16 bits, round to nearest even, saturating at +-65504.
__device__ __forceinline__ uint16_t f16_sat_bits(float x) {
  x = fminf(fmaxf(x, -65504.0f), 65504.0f);
  return __half_as_ushort(__float2half_rn(x));
}

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;  // (a & b) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// cp.async 16 bytes global -> shared; src_bytes = 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk (TMA) copies.  Every wait is bounded: after
// WAIT_LIMIT_CYCLES of polling the caller gets `false` and must report an
// error instead of spinning on.

constexpr long long WAIT_LIMIT_CYCLES = 1000000000LL;  // about 0.5 s at 2 GHz

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread until the phase completes (or
// `hint_ns` nanoseconds pass), so waiting warps do not keep polling shared
// memory and taking issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// The polling loop is one out-of-line function shared by every call site,
// so the kernels' hot loops stay small in the instruction cache.  Between
// polls the thread sleeps `sleep_ns`, so that warps waiting off the critical
// path leave the issue slots to the warps that work.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint32_t sleep_ns) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 1000000u)) {
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) return false;
    if (sleep_ns) __nanosleep(sleep_ns);
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, sleep_ns);
}
// Predicated forms for code run by a whole warp where one lane acts: no
// divergent branch around them.
__device__ __forceinline__ void mbar_arrive_expect_tx_if(bool pred, uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}\n" ::"r"(
          smem_addr(bar)),
      "r"(bytes), "r"((int)pred)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_if(bool pred, void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}\n" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "r"((int)pred)
      : "memory");
}
// global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte
// aligned), completion counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Gather of four rows of a 2-D tensor map (`tile::gather4`): rows r0..r3
// (each one box row of the map's width) land back to back at `dst`;
// completion counted on `bar`.  Only lanes with `pred` set issue it.  Every
// row coordinate passed here must lie inside the tensor.
__device__ __forceinline__ void tma_gather4_if(bool pred, void* dst, const void* map, int r0, int r1, int r2, int r3,
                                               uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %7, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {0, %2, %3, %4, %5}], [%6];\n\t}\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_addr(bar)), "r"((int)pred)
      : "memory");
}

// Same copy with an L2 cache policy (`policy` from l2_evict_first_policy()).
__device__ __forceinline__ void tma_gather4_hint_if(bool pred, void* dst, const void* map, int r0, int r1, int r2,
                                                    int r3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %7, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {0, %2, %3, %4, %5}], [%6], %8;\n\t}\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_addr(bar)), "r"((int)pred),
      "l"(policy)
      : "memory");
}

// An L2 policy under which the lines a load brings in are the first to be
// evicted: for data read once, so that it does not push out data written
// for a later kernel.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor runs; it must call
// grid_dependency_wait() before touching anything the predecessor writes.
// The predecessor lets it launch early with allow_dependent_launch().
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Scale s and the value z of the signed code 0 (stored code 2^(b-1)) from an
// INT4 / INT2 row's 4-byte pad: fp16 s then fp16 m (z = m + 2^(b-1) s), or,
// for zero-point-in-scale INT4 rows, an fp32 s whose low 4 bits hold the zero
// point zp (z = (8 - zp) s, exact).  INT8 / FP8 token-head rows: the pad is
// the fp32 scale and z = 0.
template <int MODE>
__device__ __forceinline__ void pad_scale_zero(uint32_t pad, bool stego, float& s, float& z) {
  constexpr float half_range = (float)(1 << (mode_bits(MODE) - 1));
  if constexpr (byte_token_head(MODE)) {
    s = __uint_as_float(pad);
    z = 0.0f;
  } else if (MODE == MODE_INT4 && stego) {
    s = __uint_as_float(pad & ~15u);
    z = s * (float)(8 - (int)(pad & 15u));
  } else {
    s = __half2float(__ushort_as_half((unsigned short)(pad & 0xFFFF)));
    z = fmaf(half_range, s, __half2float(__ushort_as_half((unsigned short)(pad >> 16))));
  }
}
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void sts128(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

}  // namespace kvq
