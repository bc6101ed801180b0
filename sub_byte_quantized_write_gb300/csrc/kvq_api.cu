// kvq_api.cu -- the C ABI of libkvq: argument validation, launch geometry,
// status codes.  Every call validates everything it can on the host before
// any launch (a bad call leaves device memory untouched) and then enqueues
// its kernels on the caller's stream without synchronising.

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status st, const char* msg) {
  g_last_error = msg;
  return st;
}

kvq_status cuda_fail(cudaError_t e) {
  g_last_error = std::string("CUDA: ") + cudaGetErrorString(e);
  return KVQ_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Kernel code family of an API mode: the zero-point-in-scale INT4 rows are
// INT4 rows with another pad (the `stego` flag of the kernel parameters).
int kernel_mode(int32_t mode) { return mode == KVQ_INT4_STEGO ? kvq::MODE_INT4 : mode; }

kvq_status check_cache(const kvq_cache* c) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (!c->k_pages || !c->v_pages) return fail(KVQ_ERR_INVALID_ARG, "k_pages / v_pages is NULL");
  if (!aligned(c->k_pages, 16) || !aligned(c->v_pages, 16))
    return fail(KVQ_ERR_INVALID_ARG, "k_pages / v_pages must be 16-byte aligned");
  if (c->mode != KVQ_INT4_TOKEN_HEAD && c->mode != KVQ_INT2_TOKEN_HEAD && c->mode != KVQ_INT8_CHANNEL &&
      c->mode != KVQ_INT4_STEGO && c->mode != KVQ_INT8_TOKEN_HEAD && c->mode != KVQ_FP8_TOKEN_HEAD)
    return fail(KVQ_ERR_UNSUPPORTED, "unknown mode");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(KVQ_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->block_size != 16 && c->block_size != 32 && c->block_size != 64)
    return fail(KVQ_ERR_UNSUPPORTED, "block_size must be 16, 32 or 64");
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return fail(KVQ_ERR_INVALID_ARG, "num_blocks / num_kv_heads must be > 0");
  if (c->mode == KVQ_INT8_CHANNEL) {
    if (c->rht_signs) return fail(KVQ_ERR_INVALID_ARG, "INT8 per-channel mode takes no RHT signs");
    if (!c->ch_amax || !c->ch_amax_ready) return fail(KVQ_ERR_INVALID_ARG, "INT8 mode needs ch_amax and ch_amax_ready");
    if (!aligned(c->ch_amax, 16)) return fail(KVQ_ERR_INVALID_ARG, "ch_amax must be 16-byte aligned");
  }
  return KVQ_OK;
}

kvq_status check_paging(const kvq_paging* p, int num_kv_heads) {
  (void)num_kv_heads;
  if (!p) return fail(KVQ_ERR_INVALID_ARG, "paging is NULL");
  if ((p->block_tables == nullptr) == (p->block_tables_headwise == nullptr))
    return fail(KVQ_ERR_INVALID_ARG, "exactly one of block_tables / block_tables_headwise must be set");
  if (p->batch < 0) return fail(KVQ_ERR_INVALID_ARG, "batch < 0");
  if (p->batch > 0 && (!p->seq_lens || p->max_blocks <= 0))
    return fail(KVQ_ERR_INVALID_ARG, "seq_lens is NULL or max_blocks <= 0");
  if (p->sink_size < 0) return fail(KVQ_ERR_INVALID_ARG, "sink_size < 0");
  if (p->batch > 65535) return fail(KVQ_ERR_UNSUPPORTED, "batch > 65535");
  return KVQ_OK;
}

kvq::AttnParams attn_params(const kvq_cache* c, const kvq_paging* p, const void* q, int32_t dtype,
                            int32_t hq, float scale, float* out, int32_t* dev_error) {
  kvq::AttnParams a;
  std::memset(&a, 0, sizeof(a));
  a.k_pages = c->k_pages;
  a.v_pages = c->v_pages;
  a.num_blocks = c->num_blocks;
  a.num_kv_heads = c->num_kv_heads;
  a.block_size = c->block_size;
  a.head_dim = c->head_dim;
  a.mode = kernel_mode(c->mode);
  a.stego = c->mode == KVQ_INT4_STEGO;
  a.signs = c->mode == KVQ_INT8_CHANNEL ? nullptr : c->rht_signs;
  a.ch_amax = c->ch_amax;
  a.headwise = p->block_tables_headwise != nullptr;
  a.table = a.headwise ? p->block_tables_headwise : p->block_tables;
  a.max_blocks = p->max_blocks;
  a.batch = p->batch;
  a.seq_lens = p->seq_lens;
  a.window = p->window_per_kv_head;
  a.sink = p->sink_size;
  a.q = q;
  a.dtype = dtype;
  a.num_q_heads = hq;
  a.group = hq / c->num_kv_heads;
  a.softmax_scale = scale;
  a.out = out;
  a.dev_error = dev_error;
  return a;
}

kvq_status check_q(const kvq_cache* c, const void* q, int32_t dtype, int32_t hq, const float* out) {
  if (!q || !out) return fail(KVQ_ERR_INVALID_ARG, "q / out is NULL");
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return fail(KVQ_ERR_UNSUPPORTED, "dtype must be KVQ_F32 or KVQ_BF16");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(KVQ_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  if (hq <= 0 || hq % c->num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (hq / c->num_kv_heads > 8) return fail(KVQ_ERR_UNSUPPORTED, "GQA group size above 8");
  return KVQ_OK;
}

// The prefill launch's grid (query tiles, kv heads, sequences) must fit the
// launch limits: x < 2^31, y and z <= 65535.
kvq_status check_prefill_grid(const kvq::AttnParams& P) {
  if (kvq::prefill_grid_x(P.max_q_per_seq, P.group) > 0x7FFFFFFFLL)
    return fail(KVQ_ERR_UNSUPPORTED, "max_q_per_seq gives more query tiles than one launch can hold");
  if (P.num_kv_heads > 65535) return fail(KVQ_ERR_UNSUPPORTED, "num_kv_heads > 65535 for the prefill launch");
  if (P.batch > 65535) return fail(KVQ_ERR_UNSUPPORTED, "batch > 65535");
  return KVQ_OK;
}

kvq::DecodeLayout decode_layout(const kvq_cache* c, const kvq_paging* p, int32_t num_q_heads) {
  const int group = num_q_heads / c->num_kv_heads;
  return kvq::decode_ws_layout(p->batch, c->num_kv_heads, group, c->head_dim, sm_count(),
                               kvq::decode_shape(kernel_mode(c->mode), c->head_dim, group));
}

// Scratch of kvq_decode_attn_noalloc: one static device array per GPU that
// loads the library.  Host code must not use the symbol's host-side name as a
// pointer; the device address is looked up once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

kvq_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return fail(KVQ_ERR_UNSUPPORTED, "device index >= 64");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

int32_t kvq_row_bytes(int32_t mode, int32_t head_dim) {
  if (head_dim != 64 && head_dim != 128) return 0;
  if (mode == KVQ_INT4_TOKEN_HEAD || mode == KVQ_INT4_STEGO) return head_dim / 2 + 4;
  if (mode == KVQ_INT2_TOKEN_HEAD) return head_dim / 4 + 4;
  if (mode == KVQ_INT8_CHANNEL) return head_dim;
  if (mode == KVQ_INT8_TOKEN_HEAD || mode == KVQ_FP8_TOKEN_HEAD) return head_dim + 4;
  return 0;
}

int32_t kvq_abi_version(void) { return KVQ_ABI_VERSION; }

const char* kvq_status_string(int32_t s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    default: return "KVQ_UNKNOWN_STATUS";
  }
}

const char* kvq_last_error(void) { return g_last_error.c_str(); }

kvq_status kvq_write(const kvq_cache* cache, const kvq_paging* paging, const void* k, const void* v,
                     int32_t dtype, const int32_t* cu_new_tokens, int32_t num_tokens, int32_t* dev_error,
                     void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0 || paging->batch == 0) return KVQ_OK;
  if (!k || !v || !cu_new_tokens) return fail(KVQ_ERR_INVALID_ARG, "k / v / cu_new_tokens is NULL");
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return fail(KVQ_ERR_UNSUPPORTED, "dtype must be KVQ_F32 or KVQ_BF16");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(KVQ_ERR_INVALID_ARG, "k / v must be 16-byte aligned");
  if ((long long)num_tokens * cache->num_kv_heads * 2 / 8 + 1 > 0x7FFFFFFFLL)
    return fail(KVQ_ERR_UNSUPPORTED, "too many tokens for one call");
  kvq::WriteParams P;
  std::memset(&P, 0, sizeof(P));
  P.k_pages = cache->k_pages;
  P.v_pages = cache->v_pages;
  P.num_blocks = cache->num_blocks;
  P.num_kv_heads = cache->num_kv_heads;
  P.block_size = cache->block_size;
  P.head_dim = cache->head_dim;
  P.mode = kernel_mode(cache->mode);
  P.stego = cache->mode == KVQ_INT4_STEGO;
  P.signs = cache->mode == KVQ_INT8_CHANNEL ? nullptr : cache->rht_signs;
  P.ch_amax = cache->ch_amax;
  P.ch_ready = cache->ch_amax_ready;
  P.headwise = paging->block_tables_headwise != nullptr;
  P.table = P.headwise ? paging->block_tables_headwise : paging->block_tables;
  P.max_blocks = paging->max_blocks;
  P.batch = paging->batch;
  P.seq_lens = paging->seq_lens;
  P.cu_new = cu_new_tokens;
  P.k = k;
  P.v = v;
  P.dtype = dtype;
  P.num_tokens = num_tokens;
  P.dev_error = dev_error;
  cudaError_t e = kvq::launch_write(P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KVQ_OK;
}

kvq_status kvq_gather(const kvq_cache* cache, const kvq_paging* paging, const int32_t* cu_tokens,
                      int32_t num_tokens, void* k_out, void* v_out, int32_t out_dtype, int32_t* dev_error,
                      void* stream) {
  return kvq_gather_chunk(cache, paging, cu_tokens, num_tokens, nullptr, nullptr, KVQ_F32, nullptr, k_out, v_out,
                          out_dtype, dev_error, stream);
}

kvq_status kvq_gather_chunk(const kvq_cache* cache, const kvq_paging* paging, const int32_t* cu_tokens,
                            int32_t num_tokens, const void* k_chunk, const void* v_chunk, int32_t chunk_dtype,
                            const int32_t* cu_chunk, void* k_out, void* v_out, int32_t out_dtype,
                            int32_t* dev_error, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0 || paging->batch == 0) return KVQ_OK;
  if (!k_out || !v_out || !cu_tokens) return fail(KVQ_ERR_INVALID_ARG, "k_out / v_out / cu_tokens is NULL");
  if (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16)
    return fail(KVQ_ERR_UNSUPPORTED, "out_dtype must be KVQ_F32 or KVQ_BF16");
  if (!aligned(k_out, 16) || !aligned(v_out, 16)) return fail(KVQ_ERR_INVALID_ARG, "k_out / v_out must be 16-byte aligned");
  if ((k_chunk == nullptr) != (v_chunk == nullptr) || (k_chunk && !cu_chunk))
    return fail(KVQ_ERR_INVALID_ARG, "k_chunk, v_chunk and cu_chunk go together");
  if (k_chunk && chunk_dtype != KVQ_F32 && chunk_dtype != KVQ_BF16)
    return fail(KVQ_ERR_UNSUPPORTED, "chunk_dtype must be KVQ_F32 or KVQ_BF16");
  if (k_chunk && (!aligned(k_chunk, 16) || !aligned(v_chunk, 16)))
    return fail(KVQ_ERR_INVALID_ARG, "k_chunk / v_chunk must be 16-byte aligned");
  if ((long long)num_tokens * cache->num_kv_heads * 2 / 8 + 1 > 0x7FFFFFFFLL)
    return fail(KVQ_ERR_UNSUPPORTED, "too many tokens for one call");
  kvq::WriteParams P;
  std::memset(&P, 0, sizeof(P));
  P.k_pages = cache->k_pages;
  P.v_pages = cache->v_pages;
  P.num_blocks = cache->num_blocks;
  P.num_kv_heads = cache->num_kv_heads;
  P.block_size = cache->block_size;
  P.head_dim = cache->head_dim;
  P.mode = kernel_mode(cache->mode);
  P.stego = cache->mode == KVQ_INT4_STEGO;
  P.signs = cache->mode == KVQ_INT8_CHANNEL ? nullptr : cache->rht_signs;
  P.ch_amax = cache->ch_amax;
  P.headwise = paging->block_tables_headwise != nullptr;
  P.table = P.headwise ? paging->block_tables_headwise : paging->block_tables;
  P.max_blocks = paging->max_blocks;
  P.batch = paging->batch;
  P.seq_lens = paging->seq_lens;
  P.cu_new = cu_tokens;
  P.num_tokens = num_tokens;
  P.dev_error = dev_error;
  P.out_k = k_out;
  P.out_v = v_out;
  P.out_dtype = out_dtype;
  P.chunk_k = k_chunk;
  P.chunk_v = v_chunk;
  P.cu_chunk = cu_chunk;
  P.chunk_dtype = chunk_dtype;
  cudaError_t e = kvq::launch_gather(P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_cache* cache, const kvq_paging* paging, int32_t num_q_heads,
                                     int32_t num_splits, size_t* bytes, int32_t* splits_used) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return fail(KVQ_ERR_INVALID_ARG, "bad num_q_heads");
  if (num_q_heads / cache->num_kv_heads > 8) return fail(KVQ_ERR_UNSUPPORTED, "GQA group size above 8");
  const kvq::DecodeLayout L = decode_layout(cache, paging, num_q_heads);
  *bytes = L.total;
  if (splits_used) *splits_used = num_splits > 0 ? (num_splits < L.nwall ? num_splits : L.nwall) : L.nwall;
  return KVQ_OK;
}

}  // extern "C"

namespace {
bool page_chunk_map(CUtensorMap* map, const void* pages, int num_blocks, int Hkv, int block_size, int row_bytes,
                    int chunk_rows);
}

extern "C" {

}  // extern "C"

namespace {

// Fields of the step's write for the fused call (new_k == nullptr: none).
struct FusedWrite {
  const void* k = nullptr;
  const void* v = nullptr;
  int32_t dtype = 0;
  const int32_t* cu_new = nullptr;
  int32_t num_tokens = 0;
};

kvq_status decode_call(const kvq_cache* cache, const kvq_paging* paging, const void* q, int32_t dtype,
                       int32_t num_q_heads, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                       int32_t num_splits, int32_t* dev_error, void* stream, const FusedWrite& fw) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (paging->batch == 0) return KVQ_OK;
  if ((st = check_q(cache, q, dtype, num_q_heads, out)) != KVQ_OK) return st;
  if ((long long)paging->batch * cache->num_kv_heads + 1 > 0x7FFFFFFFLL)
    return fail(KVQ_ERR_UNSUPPORTED, "batch * num_kv_heads too large");
  const kvq::DecodeLayout L = decode_layout(cache, paging, num_q_heads);
  if (!workspace || workspace_bytes < L.total) return fail(KVQ_ERR_WORKSPACE, "workspace missing or too small");
  if (!aligned(workspace, 256)) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  kvq::AttnParams P = attn_params(cache, paging, q, dtype, num_q_heads, softmax_scale, out, dev_error);
  const int rpc = kvq::decode_chunk_rows(P.mode, P.head_dim, P.group);
  if (rpc > 0) {  // the stream kernel's tensor copies: one map per pool
    const int R = kvq_row_bytes(cache->mode, cache->head_dim);
    if ((long long)cache->num_blocks * cache->num_kv_heads * (cache->block_size / rpc) > 0x7FFFFFFFLL)
      return fail(KVQ_ERR_UNSUPPORTED, "pool too large for 32-bit chunk coordinates");
    P.chunk_rows_total = cache->num_blocks * cache->num_kv_heads * (cache->block_size / rpc);
    if (!page_chunk_map(&P.kv_map[0], cache->k_pages, cache->num_blocks, cache->num_kv_heads, cache->block_size, R, rpc) ||
        !page_chunk_map(&P.kv_map[1], cache->v_pages, cache->num_blocks, cache->num_kv_heads, cache->block_size, R, rpc))
      return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K / V pools");
  }
  uint8_t* w = static_cast<uint8_t*>(workspace);
  kvq::DecodeWs ws;
  ws.tile_start = reinterpret_cast<int*>(w + L.off_tile_start);
  ws.qfrag = reinterpret_cast<uint32_t*>(w + L.off_qfrag);
  ws.qbg = reinterpret_cast<float4*>(w + L.off_qbg);
  ws.part_ml = reinterpret_cast<float2*>(w + L.off_part_ml);
  ws.part_o = reinterpret_cast<float*>(w + L.off_part_o);
  ws.n_partials = L.n_partials;
  ws.nwall = L.nwall;
  ws.fixed_workers = num_splits > 0 ? num_splits : 0;
  P.new_k = fw.k;
  P.new_v = fw.v;
  P.new_dtype = fw.dtype;
  P.cu_new = fw.cu_new;
  P.num_new = fw.num_tokens;
  cudaError_t e = kvq::launch_decode(P, ws, L.grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attn(const kvq_cache* cache, const kvq_paging* paging, const void* q, int32_t dtype,
                           int32_t num_q_heads, float softmax_scale, float* out, void* workspace,
                           size_t workspace_bytes, int32_t num_splits, int32_t* dev_error, void* stream) {
  return decode_call(cache, paging, q, dtype, num_q_heads, softmax_scale, out, workspace, workspace_bytes, num_splits,
                     dev_error, stream, FusedWrite());
}

kvq_status kvq_write_decode_attn(const kvq_cache* cache, const kvq_paging* paging, const void* k, const void* v,
                                 int32_t kv_dtype, const int32_t* cu_new_tokens, int32_t num_tokens, const void* q,
                                 int32_t q_dtype, int32_t num_q_heads, float softmax_scale, float* out,
                                 void* workspace, size_t workspace_bytes, int32_t num_splits, int32_t* dev_error,
                                 void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (cache->mode == KVQ_INT8_CHANNEL)
    return fail(KVQ_ERR_UNSUPPORTED, "the fused write + decode does not take INT8 per-channel caches");
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "num_tokens < 0");
  FusedWrite fw;
  if (num_tokens > 0 && paging->batch > 0) {
    if (!k || !v || !cu_new_tokens) return fail(KVQ_ERR_INVALID_ARG, "k / v / cu_new_tokens is NULL");
    if (kv_dtype != KVQ_F32 && kv_dtype != KVQ_BF16)
      return fail(KVQ_ERR_UNSUPPORTED, "kv_dtype must be KVQ_F32 or KVQ_BF16");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(KVQ_ERR_INVALID_ARG, "k / v must be 16-byte aligned");
    fw.k = k;
    fw.v = v;
    fw.dtype = kv_dtype;
    fw.cu_new = cu_new_tokens;
    fw.num_tokens = num_tokens;
  }
  return decode_call(cache, paging, q, q_dtype, num_q_heads, softmax_scale, out, workspace, workspace_bytes,
                     num_splits, dev_error, stream, fw);
}

kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const kvq_paging* paging, const void* q,
                                   int32_t dtype, int32_t num_q_heads, float softmax_scale, float* out,
                                   int32_t num_splits, int32_t* dev_error, void* stream) {
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_size(cache, paging, num_q_heads, num_splits, &need, nullptr);
  if (st != KVQ_OK) return st;
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "decode needs %zu bytes of scratch; the static scratch holds %u",
                  need, (unsigned)KVQ_NOALLOC_SCRATCH_BYTES);
    return fail(KVQ_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != KVQ_OK) return st;
  return kvq_decode_attn(cache, paging, q, dtype, num_q_heads, softmax_scale, out, ws,
                         (size_t)KVQ_NOALLOC_SCRATCH_BYTES, num_splits, dev_error, stream);
}

kvq_status kvq_prefill_attn(const kvq_cache* cache, const kvq_paging* paging, const void* q, int32_t dtype,
                            int32_t num_q_heads, const int32_t* cu_q, int32_t total_q, int32_t max_q_per_seq,
                            float softmax_scale, float* out, int32_t* dev_error, void* stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if ((st = check_paging(paging, cache->num_kv_heads)) != KVQ_OK) return st;
  if (total_q < 0 || max_q_per_seq < 0) return fail(KVQ_ERR_INVALID_ARG, "total_q / max_q_per_seq < 0");
  if (paging->batch == 0 || total_q == 0 || max_q_per_seq == 0) return KVQ_OK;
  if ((st = check_q(cache, q, dtype, num_q_heads, out)) != KVQ_OK) return st;
  if (!cu_q) return fail(KVQ_ERR_INVALID_ARG, "cu_q is NULL");
  kvq::AttnParams P = attn_params(cache, paging, q, dtype, num_q_heads, softmax_scale, out, dev_error);
  P.cu_q = cu_q;
  P.total_q = total_q;
  P.max_q_per_seq = max_q_per_seq;
  if ((st = check_prefill_grid(P)) != KVQ_OK) return st;
  cudaError_t e = kvq::launch_prefill(P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KVQ_OK;
}

}  // extern "C"

namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows][Hkv][D] bf16 seen as a 4-D tensor (64, D / 64, Hkv, rows): a box of
// 64 elements x 1 half x 1 head x 64 rows is one 64-dim half of the tile of
// one head, 64 lines of 128 bytes whose 16-byte pieces land XOR-swizzled by
// the line index (128-byte swizzle), so that the expansion's reads of one
// column across eight rows fall in eight different banks.
bool dense_rows_map(CUtensorMap* map, const void* base, int64_t rows, int Hkv, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || D % 64 != 0) return false;
  const cuuint64_t dims[4] = {64, (cuuint64_t)D / 64, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[3] = {128, (cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, 1, 64};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The K or V pool as a 2-D tensor of page chunks for the decode's gathers:
// row (block * Hkv + head) * (block_size / chunk_rows) + chunk holds key rows
// chunk * chunk_rows .. of that page, chunk_rows * row_bytes bytes (a
// multiple of 16, at most 2048) read as 8-byte elements, one row per box.
// No L2 promotion: a chunk (1088 bytes for the INT4 rows) starts at any
// 64-byte offset, and promoting its lines to 256-byte sectors fetched bytes of
// the neighbouring heads' chunks (the INT4 decode call ran 1.5 us longer).
bool page_chunk_map(CUtensorMap* map, const void* pages, int num_blocks, int Hkv, int block_size, int row_bytes,
                    int chunk_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t chunk = (cuuint64_t)chunk_rows * row_bytes;
  if (chunk % 16 != 0 || chunk > 2048) return false;
  const cuuint64_t dims[2] = {chunk / 8, (cuuint64_t)num_blocks * Hkv * (block_size / chunk_rows)};
  const cuuint64_t strides[1] = {chunk};
  const cuuint32_t box[2] = {(cuuint32_t)(chunk / 8), 1};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(pages), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

kvq_status kvq_prefill_dense_attn(const void* k, const void* v, const int32_t* cu_kv, int32_t num_kv_rows,
                                  int32_t num_kv_heads, int32_t head_dim, const kvq_paging* paging, const void* q,
                                  int32_t dtype, int32_t num_q_heads, const int32_t* cu_q, int32_t total_q,
                                  int32_t max_q_per_seq, float softmax_scale, float* out, int32_t* dev_error,
                                  void* stream) {
  if (!paging) return fail(KVQ_ERR_INVALID_ARG, "paging is NULL");
  if (paging->block_tables || paging->block_tables_headwise)
    return fail(KVQ_ERR_INVALID_ARG, "dense attention takes no block table");
  if (paging->batch < 0 || total_q < 0 || max_q_per_seq < 0)
    return fail(KVQ_ERR_INVALID_ARG, "batch / total_q / max_q_per_seq < 0");
  if (head_dim != 64 && head_dim != 128) return fail(KVQ_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (num_kv_heads <= 0 || num_kv_rows < 0) return fail(KVQ_ERR_INVALID_ARG, "num_kv_heads <= 0 or num_kv_rows < 0");
  if (paging->batch == 0 || total_q == 0 || max_q_per_seq == 0) return KVQ_OK;
  if (num_kv_rows == 0) return fail(KVQ_ERR_INVALID_ARG, "no K / V rows");
  if (!k || !v || !cu_kv || !cu_q || !paging->seq_lens) return fail(KVQ_ERR_INVALID_ARG, "k / v / cu_kv / cu_q / seq_lens is NULL");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(KVQ_ERR_INVALID_ARG, "k / v must be 16-byte aligned");
  if (!q || !out) return fail(KVQ_ERR_INVALID_ARG, "q / out is NULL");
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return fail(KVQ_ERR_UNSUPPORTED, "dtype must be KVQ_F32 or KVQ_BF16");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(KVQ_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (num_q_heads / num_kv_heads > 8) return fail(KVQ_ERR_UNSUPPORTED, "GQA group size above 8");
  kvq::AttnParams P;
  std::memset(&P, 0, sizeof(P));
  P.k_pages = static_cast<const uint8_t*>(k);
  P.v_pages = static_cast<const uint8_t*>(v);
  P.num_kv_heads = num_kv_heads;
  P.block_size = 16;          // no pages: positions are bounded by cu_kv instead
  P.max_blocks = 1 << 26;
  P.head_dim = head_dim;
  P.mode = kvq::MODE_DBF16;
  P.batch = paging->batch;
  P.seq_lens = paging->seq_lens;
  P.window = paging->window_per_kv_head;
  P.sink = paging->sink_size;
  P.q = q;
  P.dtype = dtype;
  P.num_q_heads = num_q_heads;
  P.group = num_q_heads / num_kv_heads;
  P.softmax_scale = softmax_scale;
  P.out = out;
  P.dev_error = dev_error;
  P.cu_q = cu_q;
  P.total_q = total_q;
  P.max_q_per_seq = max_q_per_seq;
  P.cu_kv = cu_kv;
  if (const kvq_status gs = check_prefill_grid(P); gs != KVQ_OK) return gs;
  if (!dense_rows_map(&P.kv_map[0], k, num_kv_rows, num_kv_heads, head_dim) ||
      !dense_rows_map(&P.kv_map[1], v, num_kv_rows, num_kv_heads, head_dim))
    return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for the dense K / V rows");
  cudaError_t e = kvq::launch_prefill(P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return KVQ_OK;
}

}  // extern "C"
