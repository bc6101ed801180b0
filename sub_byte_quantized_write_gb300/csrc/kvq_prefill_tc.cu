// kvq_prefill_tc.cu -- causal chunked-prefill attention over the paged
// low-bit cache on the 5th-generation tensor cores (tcgen05, TMEM).
//
// What it computes: every query of the chunk (sequence b, position
// seq_lens[b] - n_b + i) attends causally to all keys visible at its
// position, the chunk's own keys included, all read back from the INT4 /
// INT2 / INT8 pages (the chunk is written with kvq_write first).  Sources
// (page title, section): FastDeploy PR #5173 "support dynamic int2
// quantization cache kv", Usage (chunked prefill with 8192 batched tokens);
// vLLM PR #40835 review summary ("INT4 per-token-head KV cache for the Triton
// backend"), 实现拆解 item 2 and 风险与影响 (causal attention only);
// vllm-ascend-quantized-kv-cache METADATA ("Ascend INT8 KV Cache Plugin"),
// 运行机制 (chunked prefill reads and dequantises the paged cache); FastDeploy
// PR #7718 "Optimize AppendAttention for discrete head-wise block_idx"
// (head-wise rows, -1 sentinel, sink tokens).
//
// Design: one CTA of 8 warps per (128 rows, kv head, sequence); the 128
// rows are (query, q head of the GQA group) pairs, so every key tile is
// expanded once for the whole group.  Roles:
//   warps 0-3  softmax: thread r owns row r; reads its row of S from TMEM,
//              applies masks, online softmax, writes (P s) hi / lo rows to
//              shared memory, rescales its O row in TMEM when the max grows,
//              and in the end applies the zero-point term, the inverse RHT and
//              1 / l to its O row.
//   warp 4     TMEM allocation; lane 0 issues every tcgen05.mma:
//              S_b = Q_hi K^T + Q_lo K^T (M=128, N=64, K=D) into one of two
//              TMEM buffers, then O += P_hi V + P_lo V (M=128, N=D, K=64).
//   warps 5-7  producers: cp.async of the raw page chunks (double-buffered),
//              expansion of the codes into fp16 K (K-major) and V^T (K-major,
//              transposed with stmatrix) tiles in the 128-byte swizzle layout.
// Codes enter the tensor cores as signed integers (exact in fp16); the
// query and (P s) are split into fp16 hi + lo terms so fp16 does not limit
// accuracy.  Every wait on an mbarrier is bounded; on a timeout the CTA
// reports KVQ_DEVERR_TIMEOUT, drains, frees its TMEM and returns.

#include <math_constants.h>

#include "kvq_internal.h"
#include "kvq_tc.cuh"

namespace kvq {

namespace {

constexpr int TP_ROWS = 128;
constexpr int TP_KT = 64;
constexpr int TP_THREADS = 256;
constexpr int TP_PRODUCERS = 96;  // warps 5-7
constexpr int TP_MMA_WARP = 4;

template <int MODE, int D>
struct TpCfg {
  static constexpr int BITS = mode_bits(MODE);
  static constexpr int DATA = data_bytes(MODE, D);
  static constexpr int R = row_bytes_of(MODE, D);
  static constexpr int CHUNK = 16 * R;
  static constexpr int RAW = TP_KT * R;         // raw bytes of one tensor per tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int QATOM = TP_ROWS * 128;   // one 64-wide K atom of Q (16 KB)
  static constexpr int KATOM = TP_KT * 128;     // one 64-wide atom of the K tile (8 KB)
  // shared-memory layout (swizzled tiles at 1024-byte boundaries)
  static constexpr int OFF_QHI = 0;
  static constexpr int OFF_QLO = OFF_QHI + (D / 64) * QATOM;
  static constexpr int OFF_K = OFF_QLO + (D / 64) * QATOM;            // [2] K tiles
  static constexpr int OFF_VT = OFF_K + 2 * (D / 64) * KATOM;          // [2] V^T tiles (D rows x 128 B)
  static constexpr int OFF_PHI = OFF_VT + 2 * D * 128;
  static constexpr int OFF_PLO = OFF_PHI + TP_ROWS * 128;
  static constexpr int OFF_RAW = OFF_PLO + TP_ROWS * 128;              // [2][K,V][RAW]
  static constexpr int OFF_SC = OFF_RAW + ((4 * RAW + 15) / 16) * 16;  // [2][ks, kz, vs, vz][64] f32
  static constexpr int OFF_KVAL = OFF_SC + 2 * 4 * TP_KT * 4;          // [2][4] chunk validity of the expanded tiles
  static constexpr int OFF_RAWVAL = OFF_KVAL + 32;                     // [2][4] chunk validity of the raw tiles
  static constexpr int OFF_ROW = OFF_RAWVAL + 32;                      // beta, gamma [128] f32, pos [128] int
  static constexpr int OFF_BAR = OFF_ROW + 3 * TP_ROWS * 4;            // mbarriers
  static constexpr int NBAR = 12;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;                  // tmem slot, abort flag
  static constexpr int SMEM = OFF_MISC + 16 + 1024;                    // + alignment slack
  static constexpr int TMEM_COLS = 256;                                // S[2] (64 each) + O (D)
};

enum { B_KVFULL = 0, B_KVEMPTY = 2, B_SFULL = 4, B_SEMPTY = 6, B_PFULL = 8, B_ODONE = 9, B_DRAIN = 10 };

// Eight consecutive codes (head dims 8c .. 8c+7) of a raw row as four exact
// fp16 pairs of signed codes u - 2^(b-1) (INT8: as stored), in dim order.
template <int MODE>
__device__ __forceinline__ uint4 codes8(const uint8_t* raw_row, int c) {
  uint32_t o[4];
  if constexpr (MODE == MODE_INT4) {
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
  } else {
    const uint2 w = lds64(raw_row + 8 * c);
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

// The two codes of head dims (d, d+1), d even, of a raw row as an exact fp16
// pair of signed codes (low half = dim d).
template <int MODE>
__device__ __forceinline__ uint32_t codes2(const uint8_t* raw_row, int d) {
  if constexpr (MODE == MODE_INT4) {
    const uint32_t b = raw_row[d >> 1];
    const uint32_t x = b | (b << 16);
    return hsub2_bits(lop3_and_or(x, 0x00F0000Fu, 0x54006400u), 0x54806408u);
  } else if constexpr (MODE == MODE_INT2) {
    const uint32_t b = (uint32_t)raw_row[d >> 2] >> (2 * (d & 3));  // crumbs d, d+1 at bits 0-3
    const uint32_t x = b | (b << 16);
    return hsub2_bits(lop3_and_or(x, 0x000C0003u, 0x5C006400u), 0x5C086402u);
  } else {
    const uint32_t w = *reinterpret_cast<const uint16_t*>(raw_row + d);
    const uint32_t x = prmt(w, 0u, 0 | (4 << 4) | (1 << 8) | (4 << 12));
    return hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);
  }
}

}  // namespace

template <int MODE, int D>
__global__ void __launch_bounds__(TP_THREADS, 1) prefill_tc_kernel(AttnParams P) {
  using C = TpCfg<MODE, D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    mbar_init(bar + B_KVFULL + 0, TP_PRODUCERS);
    mbar_init(bar + B_KVFULL + 1, TP_PRODUCERS);
    mbar_init(bar + B_KVEMPTY + 0, 1);
    mbar_init(bar + B_KVEMPTY + 1, 1);
    mbar_init(bar + B_SFULL + 0, 1);
    mbar_init(bar + B_SFULL + 1, 1);
    mbar_init(bar + B_SEMPTY + 0, TP_ROWS);
    mbar_init(bar + B_SEMPTY + 1, TP_ROWS);
    mbar_init(bar + B_PFULL, TP_ROWS);
    mbar_init(bar + B_ODONE, 1);
    mbar_init(bar + B_DRAIN, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == TP_MMA_WARP) tc::alloc(tmem_slot, C::TMEM_COLS);

  const float log2e = 1.4426950408889634f;
  const float dnorm = (MODE != MODE_INT8 && P.signs) ? (float)D : 1.0f;
  {
    constexpr int EPL = D / 32;
    uint8_t* qhi = sm + C::OFF_QHI;
    uint8_t* qlo = sm + C::OFF_QLO;
    for (int r = warp; r < TP_ROWS; r += TP_THREADS / 32) {
      const int ql = r / G, i = r % G;
      const bool rv = ql < nq;
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
        const int off = (d >> 6) * C::QATOM + tc::sw128_off(r, (d & 63) >> 3) + 2 * (d & 7);
        *reinterpret_cast<__half*>(qhi + off) = hi;
        *reinterpret_cast<__half*>(qlo + off) = lo;
      }
      if (lane == 0) {
        rbeta[r] = P.softmax_scale * log2e / (dnorm * scl);
        rgamma[r] = P.softmax_scale * log2e * sum / dnorm;
        rpos[r] = rv ? (L - n + q0 + ql) : -1;
      }
    }
  }
  tc::fence_proxy_async();  // query tiles are read by the tensor cores
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 128;  // O after the two 64-column S buffers

  if (warp >= 5) {
    // ======================= producers =======================
    const int pt = tid - 5 * 32;  // 0..95
    const int pwarp = warp - 5;
    const int trow = P.headwise ? b * Hkv + h : b;
    const int32_t* tbl = P.table + (size_t)trow * P.max_blocks;
    const size_t blk_stride = (size_t)Hkv * bs * C::R;
    const uint8_t* kbase = P.k_pages + (size_t)h * bs * C::R;
    const uint8_t* vbase = P.v_pages + (size_t)h * bs * C::R;
    auto issue_raw = [&](int v) {
      if (v < n_virt) {
        const int T = tile_of(v);
        uint8_t* rk = sm + C::OFF_RAW + (v & 1) * 2 * C::RAW;
        uint8_t* rvp = rk + C::RAW;
        for (int idx = pt; idx < 4 * C::R; idx += TP_PRODUCERS) {
          const int c = idx / C::R, q = idx % C::R;
          const int key = TP_KT * T + 16 * c;
          bool ok = key < Leff;
          int blk = 0;
          if (ok) {
            blk = __ldg(tbl + key / bs);
            if (blk < 0) ok = false;
            else if (blk >= P.num_blocks) {
              ok = false;
              if (q == 0) flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
            }
          }
          const size_t off = ok ? (size_t)blk * blk_stride + (size_t)(key % bs) * C::R : 0;
          cp_async16(rk + c * C::CHUNK + 16 * q, kbase + off + 16 * q, ok ? 16 : 0);
          cp_async16(rvp + c * C::CHUNK + 16 * q, vbase + off + 16 * q, ok ? 16 : 0);
          if (q == 0) rawval[(v & 1) * 4 + c] = ok ? 1 : 0;
        }
      }
      cp_async_commit();
    };
    // producer-only named barrier with an OR reduction: every producer leaves
    // the loop at the same iteration
    auto producers_any = [&](bool pred) -> bool {
      uint32_t out;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
          : "=r"(out)
          : "r"((uint32_t)pred), "n"(TP_PRODUCERS)
          : "memory");
      return out != 0;
    };
    issue_raw(0);
#pragma unroll 1
    for (int v = 0; v < n_virt; ++v) {
      // all producers are done expanding tile v - 1 (its raw stage is refilled next)
      if (producers_any(*abort_flag != 0)) break;
      const int st = v & 1;
      issue_raw(v + 1);
      cp_async_wait<1>();
      // the tensor cores are done with this stage's K / V^T tiles (tile v - 2)
      const bool late = !mbar_wait_bounded(bar + B_KVEMPTY + st, ((v >> 1) & 1) ^ 1);
      if (producers_any(late)) {  // also: raw tile v visible to every producer
        *abort_flag = 1;
        flag_error(P.dev_error, DEVERR_TIMEOUT);
        break;
      }
      if (pt < 4) kval[st * 4 + pt] = rawval[st * 4 + pt];
      const uint8_t* rk = sm + C::OFF_RAW + st * 2 * C::RAW;
      const uint8_t* rvp = rk + C::RAW;
      uint8_t* kt = sm + C::OFF_K + st * (D / 64) * C::KATOM;
      uint8_t* vt = sm + C::OFF_VT + st * D * 128;
      // K: key rows, 8 dims per 16-byte chunk
      for (int it = pt; it < TP_KT * (D / 8); it += TP_PRODUCERS) {
        const int key = it / (D / 8), c8 = it % (D / 8);
        const uint4 hv = codes8<MODE>(rk + key * C::R, c8);
        *reinterpret_cast<uint4*>(kt + (c8 >> 3) * C::KATOM + tc::sw128_off(key, c8 & 7)) = hv;
      }
      // V^T: 8 keys x 32 dims per stmatrix (four 8x8 blocks, stored transposed)
      {
        const int g8 = lane >> 2, t4 = lane & 3;
        constexpr int JOBS = (TP_KT / 8) * (D / 32);
        for (int job = pwarp; job < JOBS; job += TP_PRODUCERS / 32) {
          const int kb = job % (TP_KT / 8), db = job / (TP_KT / 8);  // key block, 32-dim block
          const uint8_t* row = rvp + (8 * kb + g8) * C::R;
          uint32_t r4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) r4[i] = codes2<MODE>(row, 32 * db + 8 * i + 2 * t4);
          const int mi = lane >> 3, rr = lane & 7;
          const int d = 32 * db + 8 * mi + rr;  // stored row of matrix mi
          tc::stsm_x4_t(smem_addr(vt + tc::sw128_off(d, kb)), r4[0], r4[1], r4[2], r4[3]);
        }
      }
      if constexpr (MODE != MODE_INT8) {
        for (int idx = pt; idx < 2 * TP_KT; idx += TP_PRODUCERS) {
          const int key = idx & (TP_KT - 1);
          const bool isv = idx >= TP_KT;
          const uint32_t pad = lds32((isv ? rvp : rk) + key * C::R + C::DATA);
          constexpr float half_range = (float)(1 << (C::BITS - 1));
          const float s = __half2float(__ushort_as_half((unsigned short)(pad & 0xFFFF)));
          const float m = __half2float(__ushort_as_half((unsigned short)(pad >> 16)));
          float* scs = sc + st * 4 * TP_KT;
          scs[(isv ? 2 : 0) * TP_KT + key] = s;
          scs[(isv ? 3 : 1) * TP_KT + key] = fmaf(half_range, s, m);  // value of the signed code 0
        }
      }
      tc::fence_proxy_async();
      tc::mbar_arrive(bar + B_KVFULL + st);
    }
    cp_async_wait<0>();
  } else if (warp == TP_MMA_WARP) {
    // ======================= MMA issue =======================
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_f16(TP_ROWS, TP_KT);
      const uint32_t idesc_pv = tc::idesc_f16(TP_ROWS, D);
      const uint32_t a_qhi = smem_addr(sm + C::OFF_QHI), a_qlo = smem_addr(sm + C::OFF_QLO);
      const uint32_t a_phi = smem_addr(sm + C::OFF_PHI), a_plo = smem_addr(sm + C::OFF_PLO);
      auto pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait_bounded(bar + B_PFULL, i & 1)) return false;
        tc::fence_after();
        const uint32_t a_vt = smem_addr(sm + C::OFF_VT + st * D * 128);
#pragma unroll
        for (int kk = 0; kk < TP_KT / 16; ++kk)
          tc::mma_f16(tmem_o, tc::sw128_desc(a_phi + 32 * kk), tc::sw128_desc(a_vt + 32 * kk), idesc_pv,
                      (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < TP_KT / 16; ++kk)
          tc::mma_f16(tmem_o, tc::sw128_desc(a_plo + 32 * kk), tc::sw128_desc(a_vt + 32 * kk), idesc_pv, 1u);
        tc::commit(bar + B_ODONE);
        tc::commit(bar + B_KVEMPTY + st);
        return true;
      };
      bool ok = true;
#pragma unroll 1
      for (int v = 0; v < n_virt && ok; ++v) {
        const int st = v & 1;
        if (!mbar_wait_bounded(bar + B_KVFULL + st, (v >> 1) & 1) ||
            !mbar_wait_bounded(bar + B_SEMPTY + st, ((v >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t a_k = smem_addr(sm + C::OFF_K + st * (D / 64) * C::KATOM);
        const uint32_t s_tm = tmem + st * TP_KT;
#pragma unroll
        for (int s = 0; s < C::KSTEPS; ++s) {
          const uint32_t ao = (s >> 2) * C::QATOM + (s & 3) * 32, bo = (s >> 2) * C::KATOM + (s & 3) * 32;
          tc::mma_f16(s_tm, tc::sw128_desc(a_qhi + ao), tc::sw128_desc(a_k + bo), idesc_qk, s > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int s = 0; s < C::KSTEPS; ++s) {
          const uint32_t ao = (s >> 2) * C::QATOM + (s & 3) * 32, bo = (s >> 2) * C::KATOM + (s & 3) * 32;
          tc::mma_f16(s_tm, tc::sw128_desc(a_qlo + ao), tc::sw128_desc(a_k + bo), idesc_qk, 1u);
        }
        tc::commit(bar + B_SFULL + st);
        if (v >= 1) ok = pv(v - 1);
        if (*abort_flag) ok = false;
      }
      if (ok && n_virt >= 1) ok = pv(n_virt - 1);
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
    // ======================= softmax (thread r = row r) =======================
    const int r = tid;
    const float rb = rbeta[r], rg = rgamma[r];
    const int rp = rpos[r];
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float mrow = -CUDART_INF_F, lrow = 0.0f, pzrow = 0.0f;
    uint8_t* phi = sm + C::OFF_PHI;
    uint8_t* plo = sm + C::OFF_PLO;
    bool ok = true;
#pragma unroll 1
    for (int v = 0; v < n_virt; ++v) {
      const int st = v & 1;
      const int T = tile_of(v);
      // every decision around a .sync.aligned TMEM access is warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_SFULL + st, (v >> 1) & 1))) {
        ok = false;
        break;
      }
      tc::fence_after();
      float z[TP_KT];
      {
        uint32_t rr[TP_KT / 16][16];
#pragma unroll
        for (int c = 0; c < TP_KT / 16; ++c) tc::ld16(tmem + lane_base + st * TP_KT + 16 * c, rr[c]);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < TP_KT / 16; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j) z[16 * c + j] = __uint_as_float(rr[c][j]);
      }
      tc::fence_before();
      tc::mbar_arrive(bar + B_SEMPTY + st);
      // logits (log2 units) and masks
      const float* scs = sc + st * 4 * TP_KT;
      const int kv4 = kval[st * 4 + 0] | (kval[st * 4 + 1] << 1) | (kval[st * 4 + 2] << 2) | (kval[st * 4 + 3] << 3);
      const int key0 = TP_KT * T;
      const bool full = kv4 == 15 && key0 + TP_KT - 1 <= rp && key0 + TP_KT <= Leff &&
                        (W <= 0 || key0 > rp - W || key0 + TP_KT <= P.sink);
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < TP_KT; ++k) {
        float zz;
        if constexpr (MODE == MODE_INT8) zz = rb * z[k];
        else zz = fmaf(rb * scs[k], z[k], rg * scs[TP_KT + k]);
        if (!full) {
          const int j = key0 + k;
          bool vis = ((kv4 >> (k >> 4)) & 1) && j <= rp && j < Leff;
          if (W > 0) vis = vis && (j < P.sink || j > rp - W);
          zz = vis ? zz : -CUDART_INF_F;
        }
        z[k] = zz;
        tmax = fmaxf(tmax, zz);
      }
      const float mnew = fmaxf(mrow, tmax);
      const float muse = mnew == -CUDART_INF_F ? 0.0f : mnew;
      // the previous P.V must be done before P is overwritten or O rescaled
      if (v >= 1 && !__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_ODONE, (v - 1) & 1))) {
        ok = false;
        break;
      }
      const bool grow = v >= 1 && mnew > mrow && mrow != -CUDART_INF_F;
      if (__any_sync(0xffffffffu, grow)) {  // whole warp: rows that did not grow scale by 1
        tc::fence_after();
        const float f = grow ? ex2(mrow - muse) : 1.0f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t rr[16];
          tc::ld16(tmem_o + lane_base + c0, rr);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
          tc::st16(tmem_o + lane_base + c0, rr);
        }
        tc::wait_st();
        lrow *= f;
        pzrow *= f;
      }
      mrow = mnew;
      float tl = 0.0f, tpz = 0.0f;
#pragma unroll
      for (int c = 0; c < TP_KT / 8; ++c) {
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float w2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 8 * c + 2 * j + e;
            const float p = ex2(z[k] - muse);
            tl += p;
            if constexpr (MODE != MODE_INT8) {
              tpz += p * scs[3 * TP_KT + k];
              w2[e] = p * scs[2 * TP_KT + k];
            } else {
              w2[e] = p;
            }
          }
          const __half2 hp = __floats2half2_rn(w2[0], w2[1]);
          const float2 hf = __half22float2(hp);
          const __half2 lp = __floats2half2_rn(w2[0] - hf.x, w2[1] - hf.y);
          hv[j] = *reinterpret_cast<const uint32_t*>(&hp);
          lv[j] = *reinterpret_cast<const uint32_t*>(&lp);
        }
        *reinterpret_cast<uint4*>(phi + tc::sw128_off(r, c)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(plo + tc::sw128_off(r, c)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
      lrow += tl;
      pzrow += tpz;
      tc::fence_proxy_async();
      tc::fence_before();
      tc::mbar_arrive(bar + B_PFULL);
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        ok = false;
        break;
      }
    }
    // ---- epilogue: O row, zero-point term, inverse RHT, 1 / l
    if (ok && n_virt >= 1 && !__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_ODONE, (n_virt - 1) & 1)))
      ok = false;
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) flag_error(P.dev_error, DEVERR_TIMEOUT);
    } else {
      const int ql = r / G, i = r % G;
      float o[D];
      if (n_virt >= 1) {  // whole warp reads its 32 TMEM rows, valid or not
        tc::fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t rr[16];
          tc::ld16(tmem_o + lane_base + c0, rr);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) o[c0 + j] = __uint_as_float(rr[j]);
        }
      } else {
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] = 0.0f;
      }
      if (ql < nq) {
        float* orow = P.out + ((size_t)(cq0 + q0 + ql) * Hq + h * G + i) * D;
        if (lrow == 0.0f) {
#pragma unroll
          for (int d = 0; d < D; d += 4) *reinterpret_cast<float4*>(orow + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          if constexpr (MODE != MODE_INT8) {
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] += pzrow;
            if (P.signs) {
#pragma unroll
              for (int hs = 1; hs < D; hs <<= 1)
#pragma unroll
                for (int d = 0; d < D; ++d) {
                  if (d & hs) continue;
                  const float a = o[d], c = o[d + hs];
                  o[d] = a + c;
                  o[d + hs] = a - c;
                }
              const float inv = 1.0f / ((float)D * lrow);
#pragma unroll
              for (int d = 0; d < D; ++d) o[d] = (__ldg(P.signs + d) < 0 ? -o[d] : o[d]) * inv;
            } else {
#pragma unroll
              for (int d = 0; d < D; ++d) o[d] /= lrow;
            }
          } else {
            const float* am = P.ch_amax + ((size_t)Hkv + h) * D;
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] = o[d] * __fdiv_rn(am[d], 127.0f) / lrow;
          }
#pragma unroll
          for (int d = 0; d < D; d += 4) *reinterpret_cast<float4*>(orow + d) = make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]);
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
  const int QB = TP_ROWS / P.group;
  dim3 grid((P.max_q_per_seq + QB - 1) / QB, P.num_kv_heads, P.batch);
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
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
