// C ABI entry points: host-side validation, then one or a few kernel launches
// on the caller's stream.  Nothing here allocates device memory or
// synchronises the device.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kvint4.h"
#include "internal.h"

namespace kvint4 {

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int sm_count(int dev) {
  static std::atomic<int> cache[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// The two driver calls are reached through the runtime's entry-point query,
// so the library links the static runtime only.
uint64_t current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool workspace_layout(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                      int head_size, WorkspaceLayout* L) {
  if (num_seqs < 0 || num_q_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0) return false;
  if (num_q_heads % num_kv_heads) return false;
  const int64_t group = num_q_heads / num_kv_heads;
  int64_t tile_tokens = kPrefillRows / group;
  if (tile_tokens < 1) tile_tokens = 1;
  const int64_t S = num_seqs, T = num_q_tokens, Hq = num_q_heads, Hkv = num_kv_heads, D = head_size;
  size_t off = 0;
  L->plan = off;
  off = align256(off + 64 * sizeof(int32_t));
  L->dseq = off;
  off = align256(off + (size_t)S * 4 * sizeof(int32_t));
  L->dprefix = off;
  off = align256(off + (size_t)(S + 1) * sizeof(int64_t));
  L->max_prefill_items = (T / tile_tokens + S) * Hkv;
  L->pitems = off;
  off = align256(off + (size_t)L->max_prefill_items * 4 * sizeof(int32_t));
  L->plist = off;
  off = align256(off + (size_t)L->max_prefill_items * 2 * sizeof(int32_t));
  L->qrot = off;
  off = align256(off + (size_t)T * Hq * D * 2);
  L->direct_o = off;
  off = align256(off + (size_t)S * Hkv * kDecodeCols * D * sizeof(float));
  L->direct_ml = off;
  off = align256(off + (size_t)S * Hkv * kDecodeCols * 2 * sizeof(float));
  L->warp_o = off;
  off = align256(off + (size_t)kMaxDecodeWarps * kDecodeCols * D * sizeof(float));
  L->warp_ml = off;
  off = align256(off + (size_t)kMaxDecodeWarps * kDecodeCols * 2 * sizeof(float));
  L->total = off;
  return true;
}

static bool head_size_ok(int d) { return d == 64 || d == 96 || d == 128 || d == 192 || d == 256; }
static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static bool aligned(const void* p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }

}  // namespace kvint4

using namespace kvint4;

extern "C" {

int kv_int4_version(void) { return 4; }

const char* kv_int4_status_string(int status) {
  switch (status) {
    case KV_INT4_OK: return "ok";
    case KV_INT4_ERR_NULL: return "a required pointer is NULL";
    case KV_INT4_ERR_HEAD_SIZE: return "unsupported head_size (expected 64, 96, 128, 192 or 256)";
    case KV_INT4_ERR_HEADS: return "invalid head counts (num_q_heads must be a positive multiple of num_kv_heads, at most 64 times it)";
    case KV_INT4_ERR_BLOCK_SIZE: return "unsupported block_size (expected 16)";
    case KV_INT4_ERR_ALIGN:
      return "a pointer breaks its alignment rule (16 bytes for K/V/Q/out and code caches, 8 for slot_mapping, "
             "4 for scale caches and int32 metadata) or a token stride is not a multiple of 8 elements";
    case KV_INT4_ERR_WORKSPACE: return "workspace is NULL or smaller than kv_int4_attention_workspace_size()";
    case KV_INT4_ERR_SIZE: return "a count is negative or a size overflows the index types";
    case KV_INT4_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case KV_INT4_ERR_SCRATCH_LIMIT:
      return "the call needs more workspace than the static no-allocation scratch holds "
             "(KV_INT4_NOALLOC_SCRATCH_BYTES); use kv_int4_attention with a caller workspace";
    default: return "unknown status";
  }
}

static int validate_write(const void* k, int64_t ks, const void* v, int64_t vs, const int64_t* slots,
                          int num_tokens, const uint8_t* kc, const uint8_t* vc, const float* ksc,
                          const float* vsc, int num_blocks, int block_size, int hkv, int d,
                          const int8_t* signs, bool need_signs) {
  if (num_tokens < 0 || num_blocks < 0 || hkv <= 0) return num_tokens < 0 || num_blocks < 0 ? KV_INT4_ERR_SIZE : KV_INT4_ERR_HEADS;
  if (!head_size_ok(d)) return KV_INT4_ERR_HEAD_SIZE;
  if (block_size != 16) return KV_INT4_ERR_BLOCK_SIZE;
  if (num_tokens == 0) return KV_INT4_OK;  // a no-op; empty tensors may carry NULL pointers
  if (!k || !v || !slots || !kc || !vc || !ksc || !vsc || (need_signs && !signs)) return KV_INT4_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc) || (ks % 8) || (vs % 8) || ks < 0 || vs < 0)
    return KV_INT4_ERR_ALIGN;
  if (!aligned(slots, 8) || !aligned(ksc, 4) || !aligned(vsc, 4)) return KV_INT4_ERR_ALIGN;
  if ((int64_t)num_tokens * 2 * hkv >= (1ll << 31)) return KV_INT4_ERR_SIZE;
  return KV_INT4_OK;
}

// One write path for every format and layout.  in-slot: kc is the combined
// [blocks][2][16][Hkv][P] cache (vc, ksc, vsc unused by the caller).
static int do_write(const void* k, int64_t ks, const void* v, int64_t vs, const int64_t* slots, int num_tokens,
                    uint8_t* kc, uint8_t* vc, float* ksc, float* vsc, int num_blocks, int block_size, int hkv,
                    int d, const int8_t* signs, int32_t* status, void* stream, bool prerot, bool int8,
                    bool inslot) {
  const int cb = int8 ? d : d / 2;  // code bytes per head vector (valid d only; checked below)
  if (inslot) {
    if (!kc && num_tokens > 0) return KV_INT4_ERR_NULL;
    const int P = inslot_bytes(cb);
    vc = kc ? kc + 16ll * hkv * P : nullptr;
    ksc = kc ? reinterpret_cast<float*>(kc + cb) : nullptr;
    vsc = kc ? reinterpret_cast<float*>(kc + 16ll * hkv * P + cb) : nullptr;
  }
  int e = validate_write(k, ks, v, vs, slots, num_tokens, kc, vc, ksc, vsc, num_blocks, block_size, hkv, d, signs,
                         !prerot && !int8);
  if (e != KV_INT4_OK) return e;
  if (num_tokens == 0) return KV_INT4_OK;
  const CacheGeo geo = inslot ? inslot_geo(hkv, cb) : separate_geo(hkv, cb);
  if ((int64_t)num_blocks * geo.cblk >= (1ll << 62)) return KV_INT4_ERR_SIZE;
  if (current_device() < 0) return KV_INT4_ERR_CUDA;
  WriteArgs a{k, ks, v, vs, slots, num_tokens, kc, vc, ksc, vsc, num_blocks, block_size, hkv, d, signs, status, geo};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return int8 ? launch_write_int8(a, st) : launch_write(a, prerot, st);
}

int kv_int4_write(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                  const int64_t* slot_mapping, int num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                  float* k_scale_cache, float* v_scale_cache, int num_blocks, int block_size, int num_kv_heads,
                  int head_size, const int8_t* signs, int32_t* dev_status, void* stream) {
  return do_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, k_cache, v_cache, k_scale_cache,
                  v_scale_cache, num_blocks, block_size, num_kv_heads, head_size, signs, dev_status, stream, false,
                  false, false);
}

int kv_int8_write(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                  const int64_t* slot_mapping, int num_tokens, int8_t* k_cache, int8_t* v_cache, float* k_scale_cache,
                  float* v_scale_cache, int num_blocks, int block_size, int num_kv_heads, int head_size,
                  int32_t* dev_status, void* stream) {
  return do_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, reinterpret_cast<uint8_t*>(k_cache),
                  reinterpret_cast<uint8_t*>(v_cache), k_scale_cache, v_scale_cache, num_blocks, block_size,
                  num_kv_heads, head_size, nullptr, dev_status, stream, false, true, false);
}

int kv_int4_write_prerotated(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                             const int64_t* slot_mapping, int num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                             float* k_scale_cache, float* v_scale_cache, int num_blocks, int block_size,
                             int num_kv_heads, int head_size, int32_t* dev_status, void* stream) {
  return do_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, k_cache, v_cache, k_scale_cache,
                  v_scale_cache, num_blocks, block_size, num_kv_heads, head_size, nullptr, dev_status, stream, true,
                  false, false);
}

int kv_int4_inslot_slot_bytes(int head_size, int int8) {
  if (!head_size_ok(head_size)) return 0;
  return inslot_bytes(int8 ? head_size : head_size / 2);
}

int kv_int4_write_inslot(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                         const int64_t* slot_mapping, int num_tokens, uint8_t* kv_cache, int num_blocks,
                         int block_size, int num_kv_heads, int head_size, const int8_t* signs, int32_t* dev_status,
                         void* stream) {
  return do_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, kv_cache, nullptr, nullptr,
                  nullptr, num_blocks, block_size, num_kv_heads, head_size, signs, dev_status, stream, false, false,
                  true);
}

int kv_int8_write_inslot(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                         const int64_t* slot_mapping, int num_tokens, uint8_t* kv_cache, int num_blocks,
                         int block_size, int num_kv_heads, int head_size, int32_t* dev_status, void* stream) {
  return do_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, kv_cache, nullptr, nullptr,
                  nullptr, num_blocks, block_size, num_kv_heads, head_size, nullptr, dev_status, stream, false, true,
                  true);
}

size_t kv_int4_attention_workspace_size(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                                        int head_size) {
  if (!head_size_ok(head_size)) return 0;
  WorkspaceLayout L;
  if (!workspace_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_size, &L)) return 0;
  return L.total;
}

static int do_attention(const void* q, int64_t q_token_stride, const uint8_t* k_cache, const uint8_t* v_cache,
                        const float* k_scale_cache, const float* v_scale_cache, const int32_t* block_table,
                        int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc,
                        int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len, int num_q_heads,
                        int num_kv_heads, int head_size, int block_size, int num_blocks, float softmax_scale,
                        int causal, int sliding_window, const int8_t* signs, void* out, int64_t out_token_stride,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream, bool int8,
                        bool inslot) {
  if (inslot && head_size_ok(head_size) && num_kv_heads > 0 && k_cache) {
    // k_cache is the combined [blocks][2][16][Hkv][P] cache
    const int cb = int8 ? head_size : head_size / 2, P = inslot_bytes(cb);
    v_cache = k_cache + 16ll * num_kv_heads * P;
    k_scale_cache = reinterpret_cast<const float*>(k_cache + cb);
    v_scale_cache = reinterpret_cast<const float*>(v_cache + cb);
  }
  if (num_seqs < 0 || num_q_tokens < 0 || max_query_len < 0 || max_seq_len < 0 || num_blocks < 0 ||
      max_blocks_per_seq < 0 || sliding_window < 0)
    return KV_INT4_ERR_SIZE;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > kPrefillRows)
    return KV_INT4_ERR_HEADS;
  if (!head_size_ok(head_size)) return KV_INT4_ERR_HEAD_SIZE;
  if (block_size != 16) return KV_INT4_ERR_BLOCK_SIZE;
  if (num_seqs == 0 || num_q_tokens == 0) return KV_INT4_OK;
  if (!q || !k_cache || !v_cache || !k_scale_cache || !v_scale_cache || !block_table || !seq_lens ||
      !query_start_loc || (!int8 && !signs) || !out || !workspace)
    return !workspace ? KV_INT4_ERR_WORKSPACE : KV_INT4_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) || (q_token_stride % 8) ||
      (out_token_stride % 8) || q_token_stride < 0 || out_token_stride < 0 || ((uintptr_t)workspace & 255u))
    return KV_INT4_ERR_ALIGN;
  if (!aligned(k_scale_cache, 4) || !aligned(v_scale_cache, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(query_start_loc, 4) || !aligned(dev_status, 4))
    return KV_INT4_ERR_ALIGN;
  if ((int64_t)max_blocks_per_seq * block_size >= (1ll << 31) || (int64_t)num_q_tokens * num_q_heads >= (1ll << 31))
    return KV_INT4_ERR_SIZE;
  WorkspaceLayout L;
  if (!workspace_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_size, &L)) return KV_INT4_ERR_SIZE;
  if (workspace_bytes < L.total) return KV_INT4_ERR_WORKSPACE;
  if (current_device() < 0) return KV_INT4_ERR_CUDA;
  AttnArgs a{q, q_token_stride, k_cache, v_cache, k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
             seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len, max_seq_len, num_q_heads,
             num_kv_heads, head_size, block_size, num_blocks, softmax_scale, causal, sliding_window, signs, out,
             out_token_stride, workspace, workspace_bytes, dev_status, int8,
             inslot ? inslot_geo(num_kv_heads, int8 ? head_size : head_size / 2)
                    : separate_geo(num_kv_heads, int8 ? head_size : head_size / 2)};
  if ((int64_t)num_blocks * a.geo.cblk >= (1ll << 62)) return KV_INT4_ERR_SIZE;
  return launch_attention(a, static_cast<cudaStream_t>(stream));
}

int kv_int4_attention(const void* q, int64_t q_token_stride, const uint8_t* k_cache, const uint8_t* v_cache,
                      const float* k_scale_cache, const float* v_scale_cache, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc,
                      int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len, int num_q_heads,
                      int num_kv_heads, int head_size, int block_size, int num_blocks, float softmax_scale,
                      int causal, int sliding_window, const int8_t* signs, void* out, int64_t out_token_stride,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return do_attention(q, q_token_stride, k_cache, v_cache, k_scale_cache, v_scale_cache, block_table,
                      max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len,
                      max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
                      causal, sliding_window, signs, out, out_token_stride, workspace, workspace_bytes, dev_status,
                      stream, false, false);
}

int kv_int8_attention(const void* q, int64_t q_token_stride, const int8_t* k_cache, const int8_t* v_cache,
                      const float* k_scale_cache, const float* v_scale_cache, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc,
                      int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len, int num_q_heads,
                      int num_kv_heads, int head_size, int block_size, int num_blocks, float softmax_scale,
                      int causal, int sliding_window, void* out, int64_t out_token_stride, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return do_attention(q, q_token_stride, reinterpret_cast<const uint8_t*>(k_cache),
                      reinterpret_cast<const uint8_t*>(v_cache), k_scale_cache, v_scale_cache, block_table,
                      max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len,
                      max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
                      causal, sliding_window, nullptr, out, out_token_stride, workspace, workspace_bytes, dev_status,
                      stream, true, false);
}

int kv_int4_attention_inslot(const void* q, int64_t q_token_stride, const uint8_t* kv_cache,
                             const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                             const int32_t* query_start_loc, int num_seqs, int num_q_tokens, int max_query_len,
                             int max_seq_len, int num_q_heads, int num_kv_heads, int head_size, int block_size,
                             int num_blocks, float softmax_scale, int causal, int sliding_window, const int8_t* signs,
                             void* out, int64_t out_token_stride, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream) {
  return do_attention(q, q_token_stride, kv_cache, kv_cache, nullptr, nullptr, block_table, max_blocks_per_seq,
                      seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len, max_seq_len, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, softmax_scale, causal, sliding_window, signs,
                      out, out_token_stride, workspace, workspace_bytes, dev_status, stream, false, true);
}

int kv_int8_attention_inslot(const void* q, int64_t q_token_stride, const uint8_t* kv_cache,
                             const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                             const int32_t* query_start_loc, int num_seqs, int num_q_tokens, int max_query_len,
                             int max_seq_len, int num_q_heads, int num_kv_heads, int head_size, int block_size,
                             int num_blocks, float softmax_scale, int causal, int sliding_window, void* out,
                             int64_t out_token_stride, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             void* stream) {
  return do_attention(q, q_token_stride, kv_cache, kv_cache, nullptr, nullptr, block_table, max_blocks_per_seq,
                      seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len, max_seq_len, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, softmax_scale, causal, sliding_window, nullptr,
                      out, out_token_stride, workspace, workspace_bytes, dev_status, stream, true, true);
}

}  // extern "C"
