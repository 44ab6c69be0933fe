// kv_int8_write: the int8_per_token_head sibling mode's write path ("[Feature]
// Triton INT4 per-token-head KV cache quantization", PR #40835, review thread:
// int8 cache dtype, raw-cache round reference; "vLLM -- Attention Kernels &
// KV Cache Quantization", Merged contribution: this mode never rotates).
// Per (token, kv head) vector x of K and of V (bf16, no rotation):
//   a = max |x_i|,  s = fp32(a / 127),  c_i = rne(x_i * fp32(1 / s))
// (s = 0 and c = 0 when a < 2^-119), c stored as int8 at cache[slot][h][:]
// and s at scale[slot][h].
//
// HBM-bound: 2d bytes read, d + 4 written per vector.  Lane l of a warp step
// owns elements [16c, 16c + 16) (c = l mod (d/16)) of vector l / (d/16): a
// step covers 32 / (d/16) vectors with two 16-byte loads and one 16-byte
// store per lane, U steps loaded before any is processed.  The absmax is reduced over the vector's lanes with
// redux.sync; s and 1/s come from two exact 128-entry tables (a is a bf16
// value (1 + m/128) 2^e, so fp32(a/127) = fp32((1 + m/128)/127) 2^e and
// fp32(1/s) = fp32(1/fp32((1 + m/128)/127)) 2^-e, all normal above the flush
// bound); fma(x, r, 1.5 * 2^23) rounds half to even and leaves the code's
// two's-complement byte in the low bits.

#include <cuda_runtime.h>

#include "../../include/kvint4.h"
#include "common.cuh"
#include "internal.h"

namespace kvint4 {
namespace {

constexpr int kI8Warps = 8;
constexpr float kI8Flush = 1.50463276905252801e-36f;  // 2^-119
constexpr float kI8Magic = 12582912.0f;                // 1.5 * 2^23

struct I8Args {
  const uint16_t* k;
  int64_t k_stride;
  const uint16_t* v;
  int64_t v_stride;
  const int64_t* slots;
  int64_t num_vectors;  // num_tokens * 2 * hkv, (token, K heads then V heads)
  uint8_t* k_cache;
  uint8_t* v_cache;
  float* k_scale;
  float* v_scale;
  int64_t num_slots;
  int hkv;
  int32_t* status;
  FastDiv upt;  // vectors per token (2 hkv)
  CacheGeo geo;
};

template <int D>
__global__ void __launch_bounds__(kI8Warps * 32) write_int8_kernel(I8Args a) {
  constexpr int CH = D / 16;    // lanes per vector, 16 elements (two 16-byte chunks) each
  constexpr int VPS = 32 / CH;  // vectors per warp step
  constexpr int U = 2;          // warp steps in flight
  __shared__ uint32_t stab[256];
  if (threadIdx.x < 128) {
    const float t = __fdiv_rn(1.0f + (float)threadIdx.x * 0.0078125f, 127.0f);
    stab[threadIdx.x] = __float_as_uint(t);
    stab[128 + threadIdx.x] = __float_as_uint(__frcp_rn(t));
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int vsub = lane / CH, c = lane - vsub * CH;
  const bool active = vsub < VPS;
  unsigned gmask;  // the lanes of this lane's vector (lanes past the last vector form their own group)
  if constexpr (CH == 32) gmask = 0xffffffffu;
  else gmask = ((1u << CH) - 1u) << (vsub * CH);
  const int upt = 2 * a.hkv;
  const int nv = (int)a.num_vectors;  // < 2^31 (host-checked)
  const int gw = blockIdx.x * kI8Warps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kI8Warps;
  for (int base = gw * VPS * U; base < nv; base += nw * VPS * U) {
    uint4 x[U][2];
    int64_t sl[U];  // slots, loaded with the data so their latency overlaps
    int unit[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int vec = base + u * VPS + vsub;
      x[u][0] = x[u][1] = make_uint4(0, 0, 0, 0);
      sl[u] = -1;
      const int tok = (int)a.upt.div((uint32_t)vec);
      unit[u] = vec - tok * upt;
      if (active && vec < nv) {
        sl[u] = a.slots[tok];
        const bool kv = unit[u] >= a.hkv;
        const uint16_t* src = (kv ? a.v + (int64_t)tok * a.v_stride + (unit[u] - a.hkv) * D
                                  : a.k + (int64_t)tok * a.k_stride + unit[u] * D) + 16 * c;
        x[u][0] = reinterpret_cast<const uint4*>(src)[0];
        x[u][1] = reinterpret_cast<const uint4*>(src)[1];
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      const uint32_t w8[8] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w,
                              x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
      uint32_t am = 0;
#pragma unroll
      for (int j = 0; j < 8; j++) am = absmax_bf16x2(am, w8[j]);
      uint32_t a16 = max(am & 0x7fffu, (am >> 16) & 0x7fffu);
      a16 = __reduce_max_sync(gmask, a16);
      // table scale (exact above the flush bound), selected without branches
      const uint32_t m = a16 & 0x7fu;
      const uint32_t esh = (uint32_t)((int)(a16 >> 7) - 127) << 23;
      const bool keep = __uint_as_float(a16 << 16) >= kI8Flush;
      float sc = keep ? __uint_as_float(stab[m] + esh) : 0.f;
      float r = keep ? __uint_as_float(stab[128 + m] - esh) : 0.f;
      if (a16 >= 0x7f80u) {  // inf / NaN input
        sc = __fdiv_rn(__uint_as_float(a16 << 16), 127.0f);
        r = __frcp_rn(sc);
      }
      const float2 r2 = make_float2(r, r), magic2 = make_float2(kI8Magic, kI8Magic);
      uint32_t b[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float2 tq = f2fma(make_float2(__uint_as_float(w8[j] << 16), __uint_as_float(w8[j] & 0xffff0000u)), r2,
                                magic2);
        b[j] = __byte_perm(__float_as_uint(tq.x), __float_as_uint(tq.y), 0x0040);  // two code bytes
      }
      const uint4 codes = make_uint4(__byte_perm(b[0], b[1], 0x5410), __byte_perm(b[2], b[3], 0x5410),
                                     __byte_perm(b[4], b[5], 0x5410), __byte_perm(b[6], b[7], 0x5410));
      const int64_t slot = sl[u];
      if (slot < 0) continue;  // padding token, lane past the end, or inactive lane
      if (slot >= a.num_slots) {
        if (c == 0 && unit[u] == 0) flag(a.status, KV_INT4_DEV_BAD_SLOT);
        continue;
      }
      const bool kv = unit[u] >= a.hkv;
      const int h = kv ? unit[u] - a.hkv : unit[u];
      *reinterpret_cast<uint4*>((kv ? a.v_cache : a.k_cache) + code_off(a.geo, slot, h) + 16 * c) = codes;
      if (c == 0) store_scale((kv ? a.v_scale : a.k_scale) + scale_off(a.geo, slot, h), a.geo, sc);
    }
  }
}

template <int D>
int launch_t(const I8Args& a, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return KV_INT4_ERR_CUDA;
  constexpr int per_warp = (32 / (D / 16)) * 2;
  const int64_t warps = (a.num_vectors + per_warp - 1) / per_warp;
  int64_t grid = (warps + kI8Warps - 1) / kI8Warps;
  const int64_t cap = (int64_t)sm_count(dev) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  timing_begin(kTimedWrite, stream);
  write_int8_kernel<D><<<(unsigned)grid, kI8Warps * 32, 0, stream>>>(a);
  timing_end(kTimedWrite, stream);
  return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}

}  // namespace

int launch_write_int8(const WriteArgs& w, cudaStream_t stream) {
  I8Args a{static_cast<const uint16_t*>(w.k), w.k_stride, static_cast<const uint16_t*>(w.v), w.v_stride,
           w.slot_mapping, (int64_t)w.num_tokens * 2 * w.num_kv_heads, w.k_cache, w.v_cache, w.k_scale,
           w.v_scale, (int64_t)w.num_blocks * w.block_size, w.num_kv_heads, w.dev_status,
           FastDiv((uint32_t)(2 * w.num_kv_heads)), w.geo};
  switch (w.head_size) {
    case 64: return launch_t<64>(a, stream);
    case 96: return launch_t<96>(a, stream);
    case 128: return launch_t<128>(a, stream);
    case 192: return launch_t<192>(a, stream);
    case 256: return launch_t<256>(a, stream);
    default: return KV_INT4_ERR_HEAD_SIZE;
  }
}

}  // namespace kvint4
