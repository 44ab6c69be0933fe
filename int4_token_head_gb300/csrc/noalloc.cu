// kv_int4_attention_noalloc: attention for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a workspace: code running inside a
// framework or plugin host that owns every device allocation and hands out
// none, or a pipeline whose buffers were all sized up front and that may not
// call cudaMalloc in its steady state (an allocation there can synchronise
// the device or fail under memory pressure).  For them this entry point uses a
// workspace that already exists: a fixed-size array in this file that the
// CUDA driver places on every GPU when it loads the library, and frees only
// when the process exits.  The caller still provides every input and output.
//
// Set-up: the first call on a device, with that device current, asks the
// runtime for the array's device address (cudaGetSymbolAddress) and keeps it
// for later calls on that device (and looks it up again after a
// cudaDeviceReset, which gives the device a new context).  That first call
// may load the library's device code on the device, so make it before any
// stream capture begins.
//
// Sharing: every call on a device uses the same array, and the array keeps
// whatever the previous call left there.  The attention kernels never read a
// workspace byte they have not written earlier in the same call (the schedule
// counters are reset by the first kernel of each call), so nothing needs to be
// cleared between calls.  Two calls whose work overlaps on the GPU (different
// streams, or different host threads without ordering) race on the array and
// produce wrong results: order them, for example by issuing them on one stream.

#include <cuda_runtime.h>

#include "../../include/kvint4.h"
#include "internal.h"

namespace kvint4 {
namespace {

// The whole workspace of kv_int4_attention_noalloc, per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KV_INT4_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on device `dev` (which must be
// current), looked up once per device and CUDA context: after a
// cudaDeviceReset the array lives in a new context, possibly elsewhere.
int scratch_address(int dev, void** out) {
  static PerContext<void*> address;
  const bool ok = address.get(dev, [](void** p) {
    return cudaGetSymbolAddress(p, g_noalloc_scratch) == cudaSuccess && *p != nullptr;
  }, out);
  return ok ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}

}  // namespace
}  // namespace kvint4

extern "C" int kv_int4_attention_noalloc(
    const void* q, int64_t q_token_stride, const uint8_t* k_cache, const uint8_t* v_cache,
    const float* k_scale_cache, const float* v_scale_cache, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs, int num_q_tokens, int max_query_len,
    int max_seq_len, int num_q_heads, int num_kv_heads, int head_size, int block_size, int num_blocks,
    float softmax_scale, int causal, int sliding_window, const int8_t* signs, void* out, int64_t out_token_stride,
    int32_t* dev_status, void* stream) {
  const size_t need =
      kv_int4_attention_workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_size);
  if (need > KV_INT4_NOALLOC_SCRATCH_BYTES) return KV_INT4_ERR_SCRATCH_LIMIT;
  if (need == 0 || num_seqs == 0 || num_q_tokens == 0) {
    // invalid sizes or an empty batch: the regular entry point reports it
    // without touching any workspace
    return kv_int4_attention(q, q_token_stride, k_cache, v_cache, k_scale_cache, v_scale_cache, block_table,
                             max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len,
                             max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                             softmax_scale, causal, sliding_window, signs, out, out_token_stride, nullptr, 0,
                             dev_status, stream);
  }
  const int dev = kvint4::current_device();
  if (dev < 0) return KV_INT4_ERR_CUDA;
  void* scratch = nullptr;
  const int rc = kvint4::scratch_address(dev, &scratch);
  if (rc != KV_INT4_OK) return rc;
  return kv_int4_attention(q, q_token_stride, k_cache, v_cache, k_scale_cache, v_scale_cache, block_table,
                           max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_q_tokens, max_query_len,
                           max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, num_blocks, softmax_scale,
                           causal, sliding_window, signs, out, out_token_stride, scratch,
                           KV_INT4_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
