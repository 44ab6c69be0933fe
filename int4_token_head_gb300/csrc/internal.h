// Host-side internal interface between the C ABI (api.cu) and the kernel
// launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace kvint4 {

constexpr int kMaxDevices = 64;

// current device index (clamped to [0, kMaxDevices)); -1 on failure
int current_device();
// cached multiprocessor count of device `dev`
int sm_count(int dev);
// A unique id of the calling thread's current CUDA context (0 when there is
// none yet or the driver cannot say).  cudaDeviceReset replaces a device's
// primary context, and with it every function attribute set and every
// address taken in the old one.
uint64_t current_context_id();

// A launch setting (a function attribute set, an occupancy, a symbol
// address) computed once per device and CUDA context and shared by all host
// threads.  The first caller in a new context computes it under the lock;
// a failed computation caches nothing.
template <typename T>
class PerContext {
 public:
  template <typename Make>
  bool get(int dev, Make&& make, T* out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    const uint64_t ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mutex_);
    Slot& s = slot_[dev];
    if (!s.valid || s.ctx != ctx) {
      T v{};
      if (!make(&v)) return false;
      s.value = v;
      s.ctx = ctx;
      s.valid = true;
    }
    *out = s.value;
    return true;
  }

 private:
  struct Slot {
    bool valid = false;
    uint64_t ctx = 0;
    T value{};
  };
  std::mutex mutex_;
  Slot slot_[kMaxDevices];
};

// Where the codes and the scale of (slot, kv head) live.  A slot is
// (block, row) = (slot / 16, slot % 16); codes start at
//   code base + block * cblk + row * crow + head * chead        (bytes)
// and the f32 scale at
//   scale base + block * sblk + row * srow + head * shead       (floats).
// Separate caches ([blocks][16][Hkv][code bytes] + [blocks][16][Hkv] f32):
// crow = Hkv * code bytes, chead = code bytes, srow = Hkv, shead = 1.
// In-slot caches ([blocks][2 (K, V)][16][Hkv][P] bytes, the scale at byte
// code bytes of each P-byte slot): crow = Hkv * P, chead = P, and the same
// strides in floats for the scales.
struct CacheGeo {
  int64_t cblk, crow;
  int32_t chead;
  int64_t sblk, srow;
  int32_t shead;
};
inline CacheGeo separate_geo(int hkv, int code_bytes) {
  return CacheGeo{16ll * hkv * code_bytes, (int64_t)hkv * code_bytes, code_bytes, 16ll * hkv, hkv, 1};
}
// bytes of one in-slot (token, head) slot: codes + f32 scale, rounded up to 16
inline int inslot_bytes(int code_bytes) { return (code_bytes + 4 + 15) / 16 * 16; }
inline CacheGeo inslot_geo(int hkv, int code_bytes) {
  const int P = inslot_bytes(code_bytes);
  return CacheGeo{32ll * hkv * P, (int64_t)hkv * P, P, 8ll * hkv * P, (int64_t)hkv * P / 4, P / 4};
}
#ifdef __CUDACC__
// Store a head vector's scale at p (the scale's place for its slot and head).
// In the in-slot layout (a scale stride of more than one float) the scale and
// the padding after it are the slot's last 16 bytes (the code bytes are a
// multiple of 16): they are stored whole, the scale then zeros, so that the
// DRAM sectors a write touches are written in full (a lone 4-byte store
// leaves the padding's sector to be merged with DRAM contents: measured on
// GB300, the long-context bulk write into the in-slot layout 0.63 -> 0.70 of
// the HBM copy bandwidth).
__device__ __forceinline__ void store_scale(float* p, const CacheGeo& g, float sc) {
  if (g.shead != 1)
    *reinterpret_cast<uint4*>(p) = make_uint4(__float_as_uint(sc), 0u, 0u, 0u);
  else
    *p = sc;
}
#endif

struct WriteArgs {
  const void* k;
  int64_t k_stride;
  const void* v;
  int64_t v_stride;
  const int64_t* slot_mapping;
  int num_tokens;
  uint8_t* k_cache;
  uint8_t* v_cache;
  float* k_scale;
  float* v_scale;
  int num_blocks;
  int block_size;
  int num_kv_heads;
  int head_size;
  const int8_t* signs;
  int32_t* dev_status;
  CacheGeo geo;
};

int launch_write(const WriteArgs& a, bool prerotated, cudaStream_t stream);
// int8_per_token_head write (write_int8.cu): caches of d bytes per head vector
int launch_write_int8(const WriteArgs& a, cudaStream_t stream);

struct AttnArgs {
  const void* q;
  int64_t q_stride;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int num_seqs;
  int num_q_tokens;
  int max_query_len;
  int max_seq_len;
  int num_q_heads;
  int num_kv_heads;
  int head_size;
  int block_size;
  int num_blocks;
  float softmax_scale;
  int causal;
  int sliding_window;  // 0: none
  const int8_t* signs;
  void* out;
  int64_t out_stride;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  bool int8;  // int8_per_token_head cache (int8 codes, no rotation, no signs)
  CacheGeo geo;
};

// Workspace layout, shared by the size query and the launcher.
struct WorkspaceLayout {
  size_t plan;          // int32 counters + per-seq schedule
  size_t dseq;          // int4 [num_seqs] decode sequences: (sequence id, seq_len, first query token, q_len)
  size_t dprefix;       // int64 [num_seqs + 1] block prefix over decode sequences
  size_t pitems;        // int2 [num_seqs + 1] prefill sequence table (region sized for max_prefill_items int4)
  size_t plist;         // int2 [max_prefill_items] prefill (sequence-table index, tile) pairs, longest first
  size_t qrot;          // f16 [num_q_tokens][Hq][d] rotated, pre-scaled queries
  size_t direct_o;      // f32 [num_seqs][Hkv][8][d]
  size_t direct_ml;     // f32 [num_seqs][Hkv][8][2]
  size_t warp_o;        // f32 [kMaxDecodeWarps][8][d] (one slot per (decode CTA, head of its group))
  size_t warp_ml;       // f32 [kMaxDecodeWarps][8][2]
  size_t total;
  int64_t max_prefill_items;
};

constexpr int kMaxDecodeWarps = 4096;
constexpr int kDecodeCols = 8;      // query columns (q token x q head) per decode work unit
constexpr int kPrefillRows = 64;    // query rows (q token x q head) per prefill tile

bool workspace_layout(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                      int head_size, WorkspaceLayout* out);

int launch_attention(const AttnArgs& a, cudaStream_t stream);

// opt-in kernel timing (timing.cu); kinds match the order documented in kvint4.h
enum TimedKind { kTimedWrite = 0, kTimedPrep = 1, kTimedPrefill = 2, kTimedDecode = 3, kTimedReduce = 4 };
constexpr int kTimedKinds = 5;
void timing_begin(TimedKind kind, cudaStream_t stream);
void timing_end(TimedKind kind, cudaStream_t stream);

}  // namespace kvint4
