// kvq_prefill.cu -- causal chunked-prefill attention over the paged low-bit cache.
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
// Design: one CTA of 4 warps per (query tile, kv head, sequence).  The 64
// rows of the CTA are (query, q head of the GQA group) pairs, so every key
// tile is dequantised once for the whole group.  Per 64-key tile, raw page
// chunks arrive by cp.async (double-buffered); the CTA expands the codes into
// fp16 tiles in shared memory (exact small integers; per-key scale and zero
// point kept aside), and each warp runs QK^T and P.V on the tensor cores
// (m16n8k16) with the query and (P s) each split into fp16 hi + lo terms.
// Codes enter the tensor cores signed (u - 2^(b-1)) with the zero point
// moved to the value of code 2^(b-1), which keeps the fp32 accumulators
// small over long prefixes.
// The RHT is folded in: q' = H(d * q) once per row, and the epilogue applies
// d * H(.) / D to the output rows.

#include <math_constants.h>

#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int PF_ROWS = 64;   // (query, head) rows per CTA
constexpr int PF_KT = 64;     // keys per tile
constexpr int PF_THREADS = 128;

template <int MODE, int D>
struct PfCfg {
  static constexpr int DATA = data_bytes(MODE, D);
  static constexpr int R = row_bytes_of(MODE, D);
  static constexpr int CHUNK = 16 * R;
  static constexpr int RAW = PF_KT * R;          // raw bytes of one tensor per tile
  static constexpr int KSTEPS = D / 16;
  static constexpr int NDT = D / 8;              // n8 tiles of the output row
  static constexpr int HT = PF_KT * D * 2;       // bytes of one fp16 tile
  // smem offsets
  static constexpr int OFF_RAW = 0;                          // [2 buf][K,V][RAW]
  static constexpr int OFF_KH = OFF_RAW + 4 * RAW;           // fp16 K tile (also q staging)
  static constexpr int OFF_VH = OFF_KH + HT;                 // fp16 V tile
  static constexpr int OFF_SC = OFF_VH + HT;                 // ks, km, vs, vm [4][KT] f32
  static constexpr int OFF_KV = OFF_SC + 4 * PF_KT * 4;      // chunk validity [2][4] int
  static constexpr int OFF_ROW = OFF_KV + 8 * 4;             // beta, gamma [ROWS] f32, pos [ROWS] int
  static constexpr int SMEM = OFF_ROW + 3 * PF_ROWS * 4;
};

// 16-byte chunk swizzle of an fp16 tile with rows of D halves.
template <int D>
__device__ __forceinline__ int hsw(int row, int chunk) {
  return row * (2 * D) + 16 * (chunk ^ (row & 7));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

// Eight consecutive codes (head dims 8c .. 8c+7) of a raw row as four exact
// fp16 pairs in dim order, as signed codes u - 2^(b-1) (INT8: as stored).
// The magic constants put a code's low bit at weight 1 (1024 + u for bits
// 0-3, 64 + u for bits 4-7, 256 / 16 for the 2-bit positions 2 and 6); the
// subtrahend is magic + 2^(b-1).
template <int MODE>
__device__ __forceinline__ uint4 codes8(const uint8_t* raw_row, int c) {
  uint32_t o[4];
  if constexpr (MODE == MODE_INT4) {
    const uint32_t w = lds32(raw_row + 4 * c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = prmt(w, 0u, j | (4 << 4) | (j << 8) | (4 << 12));  // byte j in both halves
      // low half: low nibble -> 1024 + u; high half: high nibble -> 64 + u
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

}  // namespace

template <int MODE, int D>
__global__ void __launch_bounds__(PF_THREADS, 2) prefill_kernel(AttnParams P) {
  using C = PfCfg<MODE, D>;
  constexpr int EPL = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = P.group, Hq = P.num_q_heads, Hkv = P.num_kv_heads, bs = P.block_size;
  const int QB = PF_ROWS / G;  // queries per CTA

  const int cq0 = __ldg(P.cu_q + b);
  const int n = __ldg(P.cu_q + b + 1) - cq0;
  const int q0 = qtile * QB;
  if (q0 >= n) return;
  const int L = __ldg(P.seq_lens + b);
  if (n > L || L < 0) {
    if (threadIdx.x == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    return;
  }
  int Leff = L;
  if (Leff > P.max_blocks * bs) {
    if (threadIdx.x == 0) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    Leff = P.max_blocks * bs;
  }
  const int nq = min(QB, n - q0);
  const int p_min = L - n + q0, p_max = L - n + q0 + nq - 1;

  uint8_t* raw = smem + C::OFF_RAW;
  uint8_t* kh = smem + C::OFF_KH;
  uint8_t* vh = smem + C::OFF_VH;
  float* ks = reinterpret_cast<float*>(smem + C::OFF_SC);
  float* km = ks + PF_KT;
  float* vs = km + PF_KT;
  float* vm = vs + PF_KT;
  int* kval = reinterpret_cast<int*>(smem + C::OFF_KV);
  float* rbeta = reinterpret_cast<float*>(smem + C::OFF_ROW);
  float* rgamma = rbeta + PF_ROWS;
  int* rpos = reinterpret_cast<int*>(rgamma + PF_ROWS);

  // ---- query rows: q' (RHT or INT8 channel scale), power-of-two scale, fp16 hi / lo
  const float log2e = 1.4426950408889634f;
  const float dnorm = (MODE != MODE_INT8 && P.signs) ? (float)D : 1.0f;
  uint8_t* qst_hi = kh;  // staging, [ROWS][D] fp16, swizzled (reuses the K/V tiles)
  uint8_t* qst_lo = vh;
  for (int rr = 0; rr < 16; ++rr) {
    const int r = warp * 16 + rr;
    const int ql = r / G, i = r % G;
    const bool rv = ql < nq;
    float x[EPL];
    if (rv) {
      const int hq = h * G + i;
      load_row_elems<EPL>(P.q, P.dtype, ((size_t)(cq0 + q0 + ql) * Hq + hq) * D + lane * EPL, x);
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
    const float sc = ldexpf(1.0f, 10 - ex);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int d = lane * EPL + e;
      const float v = x[e] * sc;
      const __half hi = __float2half_rn(v);
      const __half lo = __float2half_rn(v - __half2float(hi));
      const int off = hsw<D>(r, d >> 3) + 2 * (d & 7);
      *reinterpret_cast<__half*>(qst_hi + off) = hi;
      *reinterpret_cast<__half*>(qst_lo + off) = lo;
    }
    if (lane == 0) {
      rbeta[r] = P.softmax_scale * log2e / (dnorm * sc);
      rgamma[r] = P.softmax_scale * log2e * sum / dnorm;
      rpos[r] = rv ? (L - n + q0 + ql) : -1;
    }
  }
  __syncthreads();
  uint32_t ahi[C::KSTEPS][4], alo[C::KSTEPS][4];
  {
    const int r0 = warp * 16 + gq, r1 = r0 + 8;
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) {
      const int oa = hsw<D>(r0, 2 * s) + 4 * tq, ob = hsw<D>(r1, 2 * s) + 4 * tq;
      const int oc = hsw<D>(r0, 2 * s + 1) + 4 * tq, od = hsw<D>(r1, 2 * s + 1) + 4 * tq;
      ahi[s][0] = lds32(qst_hi + oa); ahi[s][1] = lds32(qst_hi + ob);
      ahi[s][2] = lds32(qst_hi + oc); ahi[s][3] = lds32(qst_hi + od);
      alo[s][0] = lds32(qst_lo + oa); alo[s][1] = lds32(qst_lo + ob);
      alo[s][2] = lds32(qst_lo + oc); alo[s][3] = lds32(qst_lo + od);
    }
  }
  float rb[2], rg[2];
  int rp[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int r = warp * 16 + gq + 8 * x;
    rb[x] = rbeta[r];
    rg[x] = rgamma[r];
    rp[x] = rpos[r];
  }

  // ---- key tiles: [0, p_max] or, for a sliding-window head, the sink tiles
  // plus the tiles from the earliest window start of the CTA's rows.
  const int W = P.window ? __ldg(P.window + h) : 0;
  const int n_total = min(p_max / PF_KT + 1, (Leff + PF_KT - 1) / PF_KT);
  int ns = 0, tw = 0;
  bool gap = false;
  if (W > 0) {
    const int kw = p_min - W + 1;
    if (kw > 0) {
      ns = (min(P.sink, Leff) + PF_KT - 1) / PF_KT;
      tw = kw / PF_KT;
      gap = tw > ns;
    }
  }
  const int n_virt = gap ? ns + (n_total - tw) : n_total;
  const int trow = P.headwise ? b * Hkv + h : b;
  const int32_t* tbl = P.table + (size_t)trow * P.max_blocks;
  const size_t blk_stride = (size_t)Hkv * bs * C::R;
  const uint8_t* kbase = P.k_pages + (size_t)h * bs * C::R;
  const uint8_t* vbase = P.v_pages + (size_t)h * bs * C::R;
  auto tile_of = [&](int v) { return (gap && v >= ns) ? tw + (v - ns) : v; };

  __syncthreads();  // q staging consumed before the tiles overwrite it

  auto issue = [&](int v) {
    if (v < n_virt) {
      const int T = tile_of(v);
      uint8_t* rk = raw + (v & 1) * 2 * C::RAW;
      uint8_t* rv = rk + C::RAW;
      for (int idx = threadIdx.x; idx < 4 * C::R; idx += PF_THREADS) {
        const int c = idx / C::R, q = idx % C::R;
        const int key = PF_KT * T + 16 * c;
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
        cp_async16(rv + c * C::CHUNK + 16 * q, vbase + off + 16 * q, ok ? 16 : 0);
        if (q == 0) kval[(v & 1) * 4 + c] = ok ? 1 : 0;
      }
    }
    cp_async_commit();
  };

  float oacc[C::NDT][4];
#pragma unroll
  for (int nd = 0; nd < C::NDT; ++nd)
#pragma unroll
    for (int r = 0; r < 4; ++r) oacc[nd][r] = 0.0f;
  float mrow[2] = {-CUDART_INF_F, -CUDART_INF_F}, lrow[2] = {0.0f, 0.0f}, pmrow[2] = {0.0f, 0.0f};

  issue(0);
#pragma unroll 1
  for (int v = 0; v < n_virt; ++v) {
    issue(v + 1);
    cp_async_wait<1>();
    __syncthreads();
    const int T = tile_of(v);
    // ---- expand codes of this tile into fp16 tiles
    {
      const uint8_t* rk = raw + (v & 1) * 2 * C::RAW;
      const uint8_t* rv = rk + C::RAW;
      constexpr int ITEMS = PF_KT * (D / 8);
      for (int idx = threadIdx.x; idx < 2 * ITEMS; idx += PF_THREADS) {
        const int tsel = idx / ITEMS, it = idx % ITEMS;
        const int key = it / (D / 8), c8 = it % (D / 8);
        const uint8_t* src = (tsel ? rv : rk) + key * C::R;
        const uint4 hv = codes8<MODE>(src, c8);
        *reinterpret_cast<uint4*>((tsel ? vh : kh) + hsw<D>(key, c8)) = hv;
      }
      if constexpr (MODE != MODE_INT8) {
        const int key = threadIdx.x & (PF_KT - 1);
        const bool isv = threadIdx.x >= PF_KT;
        const uint32_t pad = lds32((isv ? rv : rk) + key * C::R + C::DATA);
        constexpr float half_range = (float)(MODE == MODE_INT4 ? 8 : 2);
        const float s = __half2float(__ushort_as_half((unsigned short)(pad & 0xFFFF)));
        const float m = __half2float(__ushort_as_half((unsigned short)(pad >> 16)));
        (isv ? vs : ks)[key] = s;
        (isv ? vm : km)[key] = fmaf(half_range, s, m);  // value of the signed code 0
      }
    }
    __syncthreads();
    const int kv_valid = (kval[(v & 1) * 4 + 0]) | (kval[(v & 1) * 4 + 1] << 1) |
                         (kval[(v & 1) * 4 + 2] << 2) | (kval[(v & 1) * 4 + 3] << 3);

    // ---- S = Q K^T over 64 keys (8 n-tiles)
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) sacc[nt][r] = 0.0f;
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bm[4];
        const int mi = lane >> 3;
        const int key = 8 * (2 * np + (mi >> 1)) + (lane & 7);
        ldsm_x4(bm, kh + hsw<D>(key, 2 * s + (mi & 1)));
        mma_16816(sacc[2 * np], ahi[s], bm[0], bm[1]);
        mma_16816(sacc[2 * np], alo[s], bm[0], bm[1]);
        mma_16816(sacc[2 * np + 1], ahi[s], bm[2], bm[3]);
        mma_16816(sacc[2 * np + 1], alo[s], bm[2], bm[3]);
      }
    }
    // ---- logits, masks, online softmax (rows gq and gq + 8 of the warp)
    float tmax[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = r >> 1;
        const int kk = 8 * nt + 2 * tq + (r & 1);
        const int j = PF_KT * T + kk;
        bool ok = ((kv_valid >> (kk >> 4)) & 1) && j <= rp[x] && j < Leff;
        if (W > 0) ok = ok && (j < P.sink || j > rp[x] - W);
        float z;
        if constexpr (MODE == MODE_INT8) z = rb[x] * sacc[nt][r];
        else z = fmaf(rb[x] * ks[kk], sacc[nt][r], rg[x] * km[kk]);
        sacc[nt][r] = ok ? z : -CUDART_INF_F;
        tmax[x] = fmaxf(tmax[x], sacc[nt][r]);
      }
    float muse[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      tmax[x] = fmaxf(tmax[x], __shfl_xor_sync(0xffffffffu, tmax[x], 1));
      tmax[x] = fmaxf(tmax[x], __shfl_xor_sync(0xffffffffu, tmax[x], 2));
      const float mnew = fmaxf(mrow[x], tmax[x]);
      muse[x] = mnew == -CUDART_INF_F ? 0.0f : mnew;
      const float f = ex2(mrow[x] - muse[x]);
      mrow[x] = mnew;
      lrow[x] *= f;
      pmrow[x] *= f;
#pragma unroll
      for (int nd = 0; nd < C::NDT; ++nd) {
        oacc[nd][2 * x] *= f;
        oacc[nd][2 * x + 1] *= f;
      }
    }
    uint32_t whi[4][4], wlo[4][4];  // A fragments of (P s) per 16-key step
    float tl[2] = {0.0f, 0.0f}, tpm[2] = {0.0f, 0.0f};  // tile-local sums
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float w[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int x = r >> 1;
        const int kk = 8 * nt + 2 * tq + (r & 1);
        const float p = ex2(sacc[nt][r] - muse[x]);  // masked logits give 0
        tl[x] += p;
        if constexpr (MODE != MODE_INT8) {
          tpm[x] += p * vm[kk];
          w[r] = p * vs[kk];
        } else {
          w[r] = p;
        }
      }
      const int kk16 = nt >> 1, half = nt & 1;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const __half h0 = __float2half_rn(w[2 * x]), h1 = __float2half_rn(w[2 * x + 1]);
        const __half2 hp = __halves2half2(h0, h1);
        const __half2 lp = __floats2half2_rn(w[2 * x] - __half2float(h0), w[2 * x + 1] - __half2float(h1));
        whi[kk16][2 * half + x] = *reinterpret_cast<const uint32_t*>(&hp);
        wlo[kk16][2 * half + x] = *reinterpret_cast<const uint32_t*>(&lp);
      }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      lrow[x] += tl[x];
      pmrow[x] += tpm[x];
    }
    // ---- O += (P s) V
#pragma unroll
    for (int kk16 = 0; kk16 < 4; ++kk16) {
#pragma unroll
      for (int np = 0; np < C::NDT / 2; ++np) {
        uint32_t bm[4];
        const int mi = lane >> 3;
        const int key = 16 * kk16 + 8 * (mi & 1) + (lane & 7);
        ldsm_x4_t(bm, vh + hsw<D>(key, 2 * np + (mi >> 1)));
        mma_16816(oacc[2 * np], whi[kk16], bm[0], bm[1]);
        mma_16816(oacc[2 * np], wlo[kk16], bm[0], bm[1]);
        mma_16816(oacc[2 * np + 1], whi[kk16], bm[2], bm[3]);
        mma_16816(oacc[2 * np + 1], wlo[kk16], bm[2], bm[3]);
      }
    }
    __syncthreads();  // tiles fully consumed before the next expansion
  }
  cp_async_wait<0>();

  // ---- epilogue: row totals, zero-point term, inverse RHT, 1 / l
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    lrow[x] += __shfl_xor_sync(0xffffffffu, lrow[x], 1);
    lrow[x] += __shfl_xor_sync(0xffffffffu, lrow[x], 2);
    pmrow[x] += __shfl_xor_sync(0xffffffffu, pmrow[x], 1);
    pmrow[x] += __shfl_xor_sync(0xffffffffu, pmrow[x], 2);
  }
  // element (nd, r): row x = r >> 1, head dim d = 8 nd + 2 tq + (r & 1)
  if constexpr (MODE != MODE_INT8) {
#pragma unroll
    for (int nd = 0; nd < C::NDT; ++nd)
#pragma unroll
      for (int r = 0; r < 4; ++r) oacc[nd][r] += pmrow[r >> 1];
    if (P.signs) {
      // stride 1: in register; strides 2, 4: lanes tq ^ 1, tq ^ 2; strides >= 8: across nd
#pragma unroll
      for (int nd = 0; nd < C::NDT; ++nd)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const float a = oacc[nd][2 * x], c = oacc[nd][2 * x + 1];
          oacc[nd][2 * x] = a + c;
          oacc[nd][2 * x + 1] = a - c;
        }
#pragma unroll
      for (int lm = 1; lm <= 2; lm <<= 1) {
        const bool upper = (tq & lm) != 0;
#pragma unroll
        for (int nd = 0; nd < C::NDT; ++nd)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float o = __shfl_xor_sync(0xffffffffu, oacc[nd][r], lm);
            oacc[nd][r] = upper ? o - oacc[nd][r] : oacc[nd][r] + o;
          }
      }
#pragma unroll
      for (int hs = 1; hs < C::NDT; hs <<= 1)
#pragma unroll
        for (int nd = 0; nd < C::NDT; ++nd) {
          if (nd & hs) continue;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = oacc[nd][r], c = oacc[nd + hs][r];
            oacc[nd][r] = a + c;
            oacc[nd + hs][r] = a - c;
          }
        }
    }
  }
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int r = warp * 16 + gq + 8 * x;
    const int ql = r / G, i = r % G;
    if (ql >= nq) continue;
    const int hq = h * G + i;
    float* orow = P.out + ((size_t)(cq0 + q0 + ql) * Hq + hq) * D;
    const float l = lrow[x];
#pragma unroll
    for (int nd = 0; nd < C::NDT; ++nd) {
      const int d = 8 * nd + 2 * tq;
      float o0 = oacc[nd][2 * x], o1 = oacc[nd][2 * x + 1];
      if (l == 0.0f) {
        o0 = 0.0f;
        o1 = 0.0f;
      } else if constexpr (MODE == MODE_INT8) {
        const float* am = P.ch_amax + ((size_t)Hkv + h) * D;
        o0 = o0 * __fdiv_rn(am[d], 127.0f) / l;
        o1 = o1 * __fdiv_rn(am[d + 1], 127.0f) / l;
      } else if (P.signs) {
        const float inv = 1.0f / ((float)D * l);
        o0 = (__ldg(P.signs + d) < 0 ? -o0 : o0) * inv;
        o1 = (__ldg(P.signs + d + 1) < 0 ? -o1 : o1) * inv;
      } else {
        o0 /= l;
        o1 /= l;
      }
      *reinterpret_cast<float2*>(orow + d) = make_float2(o0, o1);
    }
  }
}

template <int MODE, int D>
cudaError_t launch_prefill_t(const AttnParams& P, cudaStream_t stream) {
  using C = PfCfg<MODE, D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<MODE, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int QB = PF_ROWS / P.group;
  dim3 grid((P.max_q_per_seq + QB - 1) / QB, P.num_kv_heads, P.batch);
  prefill_kernel<MODE, D><<<grid, PF_THREADS, C::SMEM, stream>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnParams& P, cudaStream_t stream) {
  switch (P.mode * 1000 + P.head_dim) {
    case MODE_INT4 * 1000 + 128: return launch_prefill_t<MODE_INT4, 128>(P, stream);
    case MODE_INT4 * 1000 + 64: return launch_prefill_t<MODE_INT4, 64>(P, stream);
    case MODE_INT2 * 1000 + 128: return launch_prefill_t<MODE_INT2, 128>(P, stream);
    case MODE_INT2 * 1000 + 64: return launch_prefill_t<MODE_INT2, 64>(P, stream);
    case MODE_INT8 * 1000 + 128: return launch_prefill_t<MODE_INT8, 128>(P, stream);
    case MODE_INT8 * 1000 + 64: return launch_prefill_t<MODE_INT8, 64>(P, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
