// kvq_decode.cu -- split-KV decode attention over the paged low-bit cache.
//
// What it computes: for every sequence b and q head hq, softmax attention of
// the decode query (position seq_lens[b]-1) over the visible cached keys,
// with keys and values read from INT4 / INT2 / INT8 pages, dequantised and
// mapped back through the inverse RHT.  Sources (page title, section):
// vLLM PR #40835 review summary ("INT4 per-token-head KV cache for the Triton
// backend"), 实现拆解 item 2 (read kernel: unpack, dequantise, attention);
// FastDeploy PR #7718 "Optimize AppendAttention for discrete head-wise
// block_idx", Motivation and PR2-only delta table (per-head table rows, the
// -1 sentinel is skipped before any page address is formed, sink tokens);
// vllm-ascend-quantized-kv-cache METADATA ("Ascend INT8 KV Cache Plugin"),
// 运行机制 (decode dequantises inside the attention kernel).
//
// Design (GB300): one CTA of 4 warps per (sequence, kv head, split).  Each
// warp streams 32-key tiles (two 16-row page chunks each of K and V) through
// its own cp.async ring in shared memory and keeps its own online softmax.
// The RHT and the dequantisation are folded into the query and the weights:
//   q . k_j = (s_j (q' . c_j) + z_j sum(q')) / D,   q' = H (d * q)
//   sum_j P_j v_j = d * H( sum_j (P_j s_j) c_j + sum_j P_j z_j ) / D
// with the signed code c = u - 2^(b-1) and z = m + 2^(b-1) s (the value of
// code 2^(b-1)), so the hot loop multiplies codes (exact small integers in fp16) on
// the tensor cores: QK^T as m16n8k16 with M = 16 keys and N = 8 slots (4 q
// heads of the GQA group x {hi, lo} halves of q'), and P.V as m16n8k16 with
// M = 16 head dims, K = 16 keys, N = the same 8 slots of (P s) hi / lo.
// Splitting q' and (P s) into two fp16 terms keeps ~22 significant bits, so
// the fp16 operands do not limit accuracy.  Signed (centred) codes keep the
// fp32 accumulators small: with unsigned codes the P.V accumulator and the
// zero-point sum grow large with opposite signs and their rounding errors no
// longer cancel over tens of thousands of keys.  A second kernel merges the
// splits (log-sum-exp) and applies the inverse RHT.

#include <math_constants.h>

#include <type_traits>

#include "kvq_internal.h"

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
    if constexpr (C::BPL >= 4) {
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
// q = u - 2^(b-1) (INT4 [-8, 7], INT2 [-2, 1], INT8 as stored).  Pair P of
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
  } else {
    constexpr uint32_t sel = (2 * P) | (4 << 4) | ((2 * P + 1) << 8) | (4 << 12);
    const uint32_t x = prmt(w, 0u, sel);
    return hsub2_bits(lop3_and_xor(x, 0x00FF00FFu, 0x64806480u), 0x64806480u);  // 1152 + q - 1152
  }
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

template <int MODE, int D, int NT>
__global__ void __launch_bounds__(128, (NT == 1 ? 3 : 2)) decode_split_kernel(AttnParams P) {
  using C = DecCfg<MODE, D>;
  constexpr int EPL = D / 32;
  constexpr int NH = 4 * NT;  // head slots of the CTA (g <= NH)
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;  // mma groupID / thread-in-group
  const int G = P.group, Hq = P.num_q_heads, S = P.num_splits, Hkv = P.num_kv_heads;
  const int bs = P.block_size;

  // smem carve-up: stage rings | q hi/lo (fp16) | per-head constants | chunk validity
  uint8_t* rings = smem;
  __half* qh = reinterpret_cast<__half*>(smem + DECODE_WARPS * C::NSTAGE * C::STAGE);  // [2][NH][D]
  float* qbeta = reinterpret_cast<float*>(qh + 2 * NH * D);                            // [NH]
  float* qgamma = qbeta + NH;                                                           // [NH]
  int* vld = reinterpret_cast<int*>(qgamma + NH);                                       // [4][NSTAGE]

  // ---- visible tile list of this (sequence, kv head)
  int L = __ldg(P.seq_lens + b);
  if (L < 0) {
    if (threadIdx.x == 0) flag_error(P.dev_error, DEVERR_SEQ_LEN);
    L = 0;
  }
  const int p_q = L - 1;  // query position
  int Leff = L;
  if (Leff > P.max_blocks * bs) {
    if (threadIdx.x == 0 && split == 0) flag_error(P.dev_error, DEVERR_TABLE_RANGE);
    Leff = P.max_blocks * bs;
  }
  const int W = P.window ? __ldg(P.window + h) : 0;
  const int n_total = (Leff + 31) >> 5;
  int ns = 0, tw = 0;
  bool gap = false;
  if (W > 0) {
    const int kw = p_q - W + 1;  // first key of the window
    if (kw > 0) {
      const int sk = min(P.sink, Leff);
      ns = (sk + 31) >> 5;
      tw = kw >> 5;
      gap = tw > ns;
    }
  }
  const int n_virt = gap ? ns + (n_total - tw) : n_total;
  const int v0 = split * P.tiles_per_split;
  const int v1 = min(n_virt, v0 + P.tiles_per_split);
  const size_t part_base = ((size_t)b * Hq + (size_t)h * G) * S + split;  // + i * S for head i
  if (v0 >= v1) {
    if (threadIdx.x < G) P.part_ml[part_base + (size_t)threadIdx.x * S] = make_float2(-CUDART_INF_F, 0.0f);
    return;
  }
  const int trow = P.headwise ? b * Hkv + h : b;
  const int32_t* tbl = P.table + (size_t)trow * P.max_blocks;
  const uint8_t* kbase = P.k_pages + (size_t)h * bs * C::R;
  const uint8_t* vbase = P.v_pages + (size_t)h * bs * C::R;
  const size_t blk_stride = (size_t)Hkv * bs * C::R;

  // ---- query preparation (once per CTA): q' = H(d * q) (or q * channel
  // scale for INT8), scaled by a power of two, split into fp16 hi + lo.
  const float log2e = 1.4426950408889634f;
  const float dnorm = (MODE != MODE_INT8 && P.signs) ? (float)D : 1.0f;
  for (int i = warp; i < NH; i += DECODE_WARPS) {
    float x[EPL];
    if (i < G) {
      const int hq = h * G + i;
      load_row_elems<EPL>(P.q, P.dtype, ((size_t)b * Hq + hq) * D + lane * EPL, x);
      if constexpr (MODE == MODE_INT8) {
        const float* am = P.ch_amax + (size_t)h * D + lane * EPL;  // K scales
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
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float v = x[e] * sc;
      const __half hi = __float2half_rn(v);
      const __half lo = __float2half_rn(v - __half2float(hi));
      qh[(0 * NH + i) * D + lane * EPL + e] = hi;
      qh[(1 * NH + i) * D + lane * EPL + e] = lo;
    }
    if (lane == 0) {
      qbeta[i] = i < G ? P.softmax_scale * log2e / (dnorm * sc) : 0.0f;
      qgamma[i] = i < G ? P.softmax_scale * log2e * sum / dnorm : 0.0f;
    }
  }
  __syncthreads();

  // B fragments of QK^T: slot gq of n-tile nt = head 4*nt + gq/2, half gq&1.
  uint32_t bq[NT][C::KSTEPS][2];
  float bet[NT], gam[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + (gq >> 1);
    const __half* src = qh + ((gq & 1) * NH + head) * D;
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) {
      const int w = 4 * (s / C::KPW) + tq, sig = s % C::KPW;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        int d0, d1;
        kpair_dims<MODE>(w, 2 * sig + r, d0, d1);
        const __half2 pr = __halves2half2(src[d0], src[d1]);
        bq[nt][s][r] = *reinterpret_cast<const uint32_t*>(&pr);
      }
    }
    bet[nt] = qbeta[4 * nt + tq];
    gam[nt] = qgamma[4 * nt + tq];
  }

  // ---- this warp's tiles: virtual indices v0 + warp, v0 + warp + 4, ...
  const int first = v0 + warp;
  const int n_my = first < v1 ? (v1 - first + DECODE_WARPS - 1) / DECODE_WARPS : 0;
  uint8_t* ring = rings + warp * C::NSTAGE * C::STAGE;
  int* wvld = vld + warp * C::NSTAGE;

  auto tile_of = [&](int k) {
    const int v = first + DECODE_WARPS * k;
    return (gap && v >= ns) ? tw + (v - ns) : v;
  };

  auto issue = [&](int k) {
    if (k < n_my) {
      const int T = tile_of(k);
      uint8_t* kt = ring + (k % C::NSTAGE) * C::STAGE;
      uint8_t* vt = kt + C::TILE;
      int valid = 0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int key = 32 * T + 16 * c;
        bool ok = key < Leff;
        int blk = 0;
        if (ok) {
          blk = __ldg(tbl + key / bs);
          if (blk < 0) ok = false;  // evicted: never addressed
          else if (blk >= P.num_blocks) {
            ok = false;
            flag_error(P.dev_error, DEVERR_BLOCK_RANGE);
          }
        }
        const size_t off = ok ? (size_t)blk * blk_stride + (size_t)(key % bs) * C::R : 0;
        const uint8_t* ks = kbase + off;
        const uint8_t* vs = vbase + off;
        const int nbytes = ok ? 16 : 0;
        for (int q = lane; q < C::R; q += 32) {
          int dst;
          if constexpr (MODE == MODE_INT8) {
            const int kappa = 16 * c + q / C::PPR;
            dst = kappa * D + 16 * ((q % C::PPR) ^ ((kappa >> 2) & (C::PPR - 1)));
          } else {
            dst = c * C::CHUNK + 16 * q;
          }
          cp_async16(kt + dst, ks + 16 * q, nbytes);
          cp_async16(vt + dst, vs + 16 * q, nbytes);
        }
        valid |= (ok ? 1 : 0) << c;
      }
      if (lane == 0) wvld[k % C::NSTAGE] = valid;
    }
    cp_async_commit();
  };

  float oacc[NT][C::MT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) oacc[nt][mt][r] = 0.0f;
  float mrun[NT], lrun[NT], pmrun[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mrun[nt] = -CUDART_INF_F;
    lrun[nt] = 0.0f;
    pmrun[nt] = 0.0f;
  }

#pragma unroll 1
  for (int k = 0; k < C::NSTAGE - 1; ++k) issue(k);

#pragma unroll 1
  for (int k = 0; k < n_my; ++k) {
    cp_async_wait<C::NSTAGE - 2>();
    __syncwarp();
    issue(k + C::NSTAGE - 1);
    const uint8_t* kt = ring + (k % C::NSTAGE) * C::STAGE;
    const uint8_t* vt = kt + C::TILE;
    const int valid = wvld[k % C::NSTAGE];
    const int key0 = 32 * tile_of(k);

    // ---- S^T = U_K (keys x D) . Q (D x slots); lane rows: keys 4gq + 2m + hh
    float sacc[2][NT][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) sacc[m][nt][r] = 0.0f;
#pragma unroll
    for (int wi = 0; wi < C::WPL; ++wi) {
      uint32_t kw[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) kw[m][hh] = load_kword<MODE, D>(kt, 4 * gq + 2 * m + hh, 4 * wi + tq);
      Unroll<C::KPW, MODE>::run([&](auto sig_c) {
        constexpr int sig = decltype(sig_c)::value;
        const int s = C::KPW * wi + sig;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t a[4] = {kpair<MODE, 2 * sig>(kw[m][0]), kpair<MODE, 2 * sig>(kw[m][1]),
                                 kpair<MODE, 2 * sig + 1>(kw[m][0]), kpair<MODE, 2 * sig + 1>(kw[m][1])};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[m][nt], a, bq[nt][s][0], bq[nt][s][1]);
        }
      });
    }

    // ---- logits (log2 units), masks, online softmax
    float lg[2][2][NT];
    float sv_[2][2], mv_[2][2];
    bool vk[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int kappa = 4 * gq + 2 * m + hh;
        const int j = key0 + kappa;
        bool ok = ((valid >> (kappa >> 4)) & 1) && j < Leff;
        if (W > 0) ok = ok && (j < P.sink || j > p_q - W);
        vk[m][hh] = ok;
        float sk = 0.0f, mk = 0.0f;
        if constexpr (MODE != MODE_INT8) {
          const uint32_t pk = lds32(kt + kappa * C::R + C::DATA);
          const uint32_t pv = lds32(vt + kappa * C::R + C::DATA);
          constexpr float half_range = (float)(1 << (C::BITS - 1));
          sk = __half2float(__ushort_as_half((unsigned short)(pk & 0xFFFF)));
          mk = fmaf(half_range, sk, __half2float(__ushort_as_half((unsigned short)(pk >> 16))));
          sv_[m][hh] = __half2float(__ushort_as_half((unsigned short)(pv & 0xFFFF)));
          mv_[m][hh] = fmaf(half_range, sv_[m][hh], __half2float(__ushort_as_half((unsigned short)(pv >> 16))));
        } else {
          sv_[m][hh] = 1.0f;
          mv_[m][hh] = 0.0f;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float cdot = sacc[m][nt][2 * hh] + sacc[m][nt][2 * hh + 1];  // hi + lo slots
          float z;
          if constexpr (MODE == MODE_INT8) z = bet[nt] * cdot;
          else z = fmaf(bet[nt] * sk, cdot, gam[nt] * mk);
          lg[m][hh][nt] = ok ? z : -CUDART_INF_F;
        }
      }

    uint32_t xh[NT][2], xl[NT][2];  // packed (P s) hi / lo per m: (key hh=0, key hh=1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float tmax = fmaxf(fmaxf(lg[0][0][nt], lg[0][1][nt]), fmaxf(lg[1][0][nt], lg[1][1][nt]));
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
      for (int m = 0; m < 2; ++m) {
        float wv[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float p = ex2(lg[m][hh][nt] - muse);
          const bool ok = vk[m][hh];
          tl += ok ? p : 0.0f;
          if constexpr (MODE != MODE_INT8) tpm += ok ? p * mv_[m][hh] : 0.0f;
          wv[hh] = ok ? p * sv_[m][hh] : 0.0f;
        }
        const __half h0 = __float2half_rn(wv[0]), h1 = __float2half_rn(wv[1]);
        const __half2 hp = __halves2half2(h0, h1);
        const __half2 lp = __floats2half2_rn(wv[0] - __half2float(h0), wv[1] - __half2float(h1));
        xh[nt][m] = *reinterpret_cast<const uint32_t*>(&hp);
        xl[nt][m] = *reinterpret_cast<const uint32_t*>(&lp);
      }
      lrun[nt] += tl;
      pmrun[nt] += tpm;
    }

    // ---- P.V: O^T (D x slots) += U_V^T (D x 16 keys) . Wslots (16 keys x slots)
#pragma unroll
    for (int mp = 0; mp < 2; ++mp) {
      uint32_t bw[NT][2];
      const int src = ((2 * tq + mp) << 2) | (gq >> 1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t a0 = __shfl_sync(0xffffffffu, xh[nt][0], src);
        const uint32_t b0 = __shfl_sync(0xffffffffu, xl[nt][0], src);
        const uint32_t a1 = __shfl_sync(0xffffffffu, xh[nt][1], src);
        const uint32_t b1 = __shfl_sync(0xffffffffu, xl[nt][1], src);
        bw[nt][0] = (gq & 1) ? b0 : a0;
        bw[nt][1] = (gq & 1) ? b1 : a1;
      }
      uint2 vl[2][2], vh[2][2];
#pragma unroll
      for (int hp = 0; hp < 2; ++hp)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kappa = 8 * tq + 4 * mp + 2 * hp + e;
          vl[hp][e] = load_range<MODE, D>(vt, kappa, gq);
          vh[hp][e] = load_range<MODE, D>(vt, kappa, 8 + gq);
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

  // ---- per-warp totals, then merge the 4 warps of the CTA
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lrun[nt] += __shfl_xor_sync(0xffffffffu, lrun[nt], o);
      pmrun[nt] += __shfl_xor_sync(0xffffffffu, pmrun[nt], o);
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  float* osm = reinterpret_cast<float*>(rings);               // [4][NH][2][D]
  float* stat = osm + DECODE_WARPS * NH * 2 * D;               // [4][NH][3]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + tq;
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int rg = (r < 2) ? gq : 8 + gq;
        const int d = rg * (D / 16) + mt;
        osm[((warp * NH + head) * 2 + (r & 1)) * D + d] = oacc[nt][mt][r];
      }
    if (gq == 0) {
      float* st = stat + (warp * NH + head) * 3;
      st[0] = mrun[nt];
      st[1] = lrun[nt];
      st[2] = pmrun[nt];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < DECODE_WARPS; ++w) M = fmaxf(M, stat[(w * NH + i) * 3]);
    const size_t pidx = part_base + (size_t)i * S;
    if (M == -CUDART_INF_F) {
      if (d == 0) P.part_ml[pidx] = make_float2(-CUDART_INF_F, 0.0f);
      continue;
    }
    float o = 0.0f, l = 0.0f, pm = 0.0f;
#pragma unroll
    for (int w = 0; w < DECODE_WARPS; ++w) {
      const float* st = stat + (w * NH + i) * 3;
      const float f = ex2(st[0] - M);
      o += f * (osm[((w * NH + i) * 2 + 0) * D + d] + osm[((w * NH + i) * 2 + 1) * D + d]);
      l += f * st[1];
      pm += f * st[2];
    }
    P.part_o[pidx * D + d] = o + pm;
    if (d == 0) P.part_ml[pidx] = make_float2(M, l);
  }
}

// Merge the splits of one (sequence, q head): log-sum-exp weights, then the
// inverse RHT (d * H o / D) or the INT8 value-channel scales, then 1 / l.
template <int D>
__global__ void __launch_bounds__(256) decode_reduce_kernel(AttnParams P) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int Hq = P.num_q_heads, S = P.num_splits;
  if (wid >= (long long)P.batch * Hq) return;
  const int hq = (int)(wid % Hq);
  const int h = hq / P.group;
  const size_t base = (size_t)wid * S;
  float* out = P.out + (size_t)wid * D;
  float M = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, P.part_ml[base + s].x);
  M = warp_max(M);
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
  if (M == -CUDART_INF_F) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = 0.0f;
    return;
  }
  float l = 0.0f;
  for (int s = 0; s < S; ++s) {
    const float2 ml = P.part_ml[base + s];
    if (ml.y == 0.0f) continue;
    const float f = ex2(ml.x - M);
    l += f * ml.y;
    const float* po = P.part_o + (base + s) * D;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] += f * po[lane + 32 * e];
  }
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
    for (int e = 0; e < EPL; ++e) {
      const int d = lane + 32 * e;
      out[d] = (__ldg(P.signs + d) < 0 ? -o[e] : o[e]) * inv;
    }
  } else if (P.mode == MODE_INT8) {
    const float* am = P.ch_amax + ((size_t)1 * P.num_kv_heads + h) * D;  // V scales
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int d = lane + 32 * e;
      out[d] = o[e] * __fdiv_rn(am[d], 127.0f) / l;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = o[e] / l;
  }
}

template <int MODE, int D, int NT>
size_t decode_smem_bytes() {
  using C = DecCfg<MODE, D>;
  constexpr int NH = 4 * NT;
  const size_t rings = (size_t)DECODE_WARPS * C::NSTAGE * C::STAGE;
  const size_t merge = (size_t)DECODE_WARPS * NH * 2 * D * 4 + DECODE_WARPS * NH * 3 * 4;
  const size_t first = rings > merge ? rings : merge;
  return first + 2 * NH * D * 2 + 2 * NH * 4 + DECODE_WARPS * C::NSTAGE * 4;
}

template <int MODE, int D, int NT>
cudaError_t launch_decode_t(const AttnParams& P, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes<MODE, D, NT>();
  // the opt-in shared-memory size is set once per device (not inside later
  // calls, which may be captured into a CUDA graph)
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_split_kernel<MODE, D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(P.num_splits, P.num_kv_heads, P.batch);
  decode_split_kernel<MODE, D, NT><<<grid, 128, smem, stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = (long long)P.batch * P.num_q_heads;
  decode_reduce_kernel<D><<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(P);
  return cudaGetLastError();
}

template <int MODE, int D>
cudaError_t launch_decode_md(const AttnParams& P, cudaStream_t stream) {
  if (P.group <= 4) return launch_decode_t<MODE, D, 1>(P, stream);
  return launch_decode_t<MODE, D, 2>(P, stream);
}

cudaError_t launch_decode(const AttnParams& P, cudaStream_t stream) {
  switch (P.mode * 1000 + P.head_dim) {
    case MODE_INT4 * 1000 + 128: return launch_decode_md<MODE_INT4, 128>(P, stream);
    case MODE_INT4 * 1000 + 64: return launch_decode_md<MODE_INT4, 64>(P, stream);
    case MODE_INT2 * 1000 + 128: return launch_decode_md<MODE_INT2, 128>(P, stream);
    case MODE_INT2 * 1000 + 64: return launch_decode_md<MODE_INT2, 64>(P, stream);
    case MODE_INT8 * 1000 + 128: return launch_decode_md<MODE_INT8, 128>(P, stream);
    case MODE_INT8 * 1000 + 64: return launch_decode_md<MODE_INT8, 64>(P, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
