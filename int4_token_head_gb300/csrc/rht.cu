// kv_int4_rht: the block-diagonal randomized Hadamard rotation on its own
// ("vLLM -- Attention Kernels & KV Cache Quantization", PR #56198, Merged
// contribution; D before H per "Rotate KV into RHT domain in the INT4
// unified attn test", PR #62881, Details / Root cause).
//
//   forward: y = (I_n (x) H_b) . D . x        inverse: y = D . (I_n (x) H_b) . x / b
//
// Kernels, all HBM-bound (2 bytes read and 2 or 4 written per element):
//  - cache head sizes (64, 96, 128, 192, 256), rows 16-byte aligned: 16-byte
//    chunks per lane, several rows per warp step, butterflies in registers
//    and across lanes (rht_vec_kernel);
//  - the same head sizes otherwise: one warp per row in registers, lane l
//    holding elements l + 32k; stages h < 32 pair lanes (shfl.xor), stages
//    h >= 32 pair a lane's own registers;
//  - any other head size up to 4096: the row is staged in shared memory and
//    every stage h < b pairs elements i and i + h with (i mod 2h) < h, which
//    never crosses a b-block because 2h divides b.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/kvint4.h"
#include "common.cuh"
#include "internal.h"

namespace kvint4 {
namespace {

constexpr int kRhtWarps = 8;           // rows in flight per CTA
constexpr int kRhtMaxSmemHead = 4096;  // largest head size of the shared-memory kernel

struct RhtArgs {
  const uint16_t* x;
  int64_t xs;
  void* y;
  int64_t ys;
  int64_t rows;
  const int8_t* signs;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

template <bool F32>
__device__ __forceinline__ void store_elem(void* y, int64_t idx, float v) {
  if constexpr (F32) static_cast<float*>(y)[idx] = v;
  else static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
}

template <int D, bool INV, bool F32>
__global__ void __launch_bounds__(kRhtWarps * 32) rht_reg_kernel(RhtArgs a) {
  constexpr int B = Head<D>::b;
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  float sg[PER];
#pragma unroll
  for (int k = 0; k < PER; k++) sg[k] = a.signs[lane + 32 * k] < 0 ? -1.f : 1.f;
  const float post = INV ? 1.f / (float)B : 1.f;  // exact: B is a power of two
  const int64_t nwarps = (int64_t)gridDim.x * kRhtWarps;
  for (int64_t row = (int64_t)blockIdx.x * kRhtWarps + (threadIdx.x >> 5); row < a.rows; row += nwarps) {
    const uint16_t* src = a.x + row * a.xs;
    float x[PER];
#pragma unroll
    for (int k = 0; k < PER; k++) {
      const float v = bf16_to_f32(src[lane + 32 * k]);
      x[k] = INV ? v : v * sg[k];
    }
#pragma unroll
    for (int hh = 1; hh < B && hh < 32; hh <<= 1) {
      const float f = (lane & hh) ? -1.f : 1.f;  // upper element: partner - self
#pragma unroll
      for (int k = 0; k < PER; k++) x[k] = fmaf(f, x[k], __shfl_xor_sync(0xffffffffu, x[k], hh));
    }
#pragma unroll
    for (int m = 1; 32 * m < B; m <<= 1) {
#pragma unroll
      for (int k = 0; k < PER; k++) {
        if ((k & m) == 0) {
          const float p = x[k], q = x[k + m];
          x[k] = p + q;
          x[k + m] = p - q;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < PER; k++) store_elem<F32>(a.y, row * a.ys + lane + 32 * k, INV ? x[k] * sg[k] * post : x[k]);
  }
}

// 16-byte variant of the register kernel (rows 16-byte aligned): lane l of a
// warp step owns chunk c = l mod CH (elements 8c .. 8c+7) of row l / CH, so a
// step covers 32 / CH rows with one 16-byte load per lane.  Stages h < 8 pair
// a lane's own elements; stages h >= 8 pair chunks c and c ^ (h / 8), i.e.
// lanes l and l ^ (h / 8) (each row's chunks start at a multiple of b / 8
// lanes).  U steps are loaded before any is computed.
template <int D, bool INV, bool F32>
__global__ void __launch_bounds__(kRhtWarps * 32) rht_vec_kernel(RhtArgs a) {
  constexpr int B = Head<D>::b;
  constexpr int CH = D / 8;       // 16-byte chunks per row
  constexpr int RPW = 32 / CH;    // rows per warp step
  constexpr int U = 4;            // warp steps in flight
  static_assert(RPW >= 1 && (RPW * CH) % (B / 8 > 0 ? B / 8 : 1) == 0, "row layout");
  const int lane = threadIdx.x & 31;
  const int rsub = lane / CH, c = lane - rsub * CH;
  const bool active = rsub < RPW;
  float sg[8];
#pragma unroll
  for (int j = 0; j < 8; j++) sg[j] = (active && a.signs[8 * c + j] < 0) ? -1.f : 1.f;
  const float post = INV ? 1.f / (float)B : 1.f;
  const int64_t gw = (int64_t)blockIdx.x * kRhtWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kRhtWarps;
  for (int64_t base = gw * RPW * U; base < a.rows; base += nwarps * RPW * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t row = base + u * RPW + rsub;
      v[u] = make_uint4(0, 0, 0, 0);
      if (active && row < a.rows) v[u] = *reinterpret_cast<const uint4*>(a.x + row * a.xs + 8 * c);
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float e[8];
#pragma unroll
      for (int j = 0; j < 4; j++) {
        e[2 * j] = __uint_as_float(w[j] << 16);
        e[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
      if constexpr (!INV) {
#pragma unroll
        for (int j = 0; j < 8; j++) e[j] *= sg[j];
      }
#pragma unroll
      for (int hh = 1; hh < 8 && hh < B; hh <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; j++) {
          if ((j & hh) == 0) {
            const float p = e[j], q = e[j + hh];
            e[j] = p + q;
            e[j + hh] = p - q;
          }
        }
      }
#pragma unroll
      for (int m = 1; 8 * m < B; m <<= 1) {
        const float f = (c & m) ? -1.f : 1.f;  // upper chunk: partner - self
#pragma unroll
        for (int j = 0; j < 8; j++) e[j] = fmaf(f, e[j], __shfl_xor_sync(0xffffffffu, e[j], m));
      }
      if constexpr (INV) {
#pragma unroll
        for (int j = 0; j < 8; j++) e[j] = e[j] * sg[j] * post;
      }
      const int64_t row = base + u * RPW + rsub;
      if (!active || row >= a.rows) continue;
      if constexpr (F32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.y) + row * a.ys + 8 * c);
        dst[0] = make_float4(e[0], e[1], e[2], e[3]);
        dst[1] = make_float4(e[4], e[5], e[6], e[7]);
      } else {
        uint4 o;
        o.x = pack_bf16x2_rn(e[0], e[1]);
        o.y = pack_bf16x2_rn(e[2], e[3]);
        o.z = pack_bf16x2_rn(e[4], e[5]);
        o.w = pack_bf16x2_rn(e[6], e[7]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.y) + row * a.ys + 8 * c) = o;
      }
    }
  }
}

template <bool INV, bool F32>
__global__ void __launch_bounds__(kRhtWarps * 32) rht_smem_kernel(RhtArgs a, int d) {
  extern __shared__ float srow[];  // [kRhtWarps][d]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* r = srow + (size_t)warp * d;
  const int b = d & -d;
  const float post = INV ? 1.f / (float)b : 1.f;
  const int64_t nwarps = (int64_t)gridDim.x * kRhtWarps;
  for (int64_t row = (int64_t)blockIdx.x * kRhtWarps + warp; row < a.rows; row += nwarps) {
    const uint16_t* src = a.x + row * a.xs;
    for (int i = lane; i < d; i += 32) {
      const float v = bf16_to_f32(src[i]);
      r[i] = (!INV && a.signs[i] < 0) ? -v : v;
    }
    __syncwarp();
    int lh = 0;
    for (int hh = 1; hh < b; hh <<= 1, lh++) {
      for (int p = lane; p < d / 2; p += 32) {
        const int i = ((p >> lh) << (lh + 1)) + (p & (hh - 1));
        const float u = r[i], w = r[i + hh];
        r[i] = u + w;
        r[i + hh] = u - w;
      }
      __syncwarp();
    }
    for (int i = lane; i < d; i += 32) {
      const float v = INV ? (a.signs[i] < 0 ? -r[i] : r[i]) * post : r[i];
      store_elem<F32>(a.y, row * a.ys + i, v);
    }
    __syncwarp();  // the row buffer is reused by the next row
  }
}

int64_t grid_for(int64_t rows, int dev) {
  int64_t grid = (rows + kRhtWarps - 1) / kRhtWarps;
  const int64_t cap = (int64_t)sm_count(dev) * 8;  // persistent rows loop beyond 8 CTAs per SM
  return grid < cap ? grid : cap;
}

template <int D, bool INV, bool F32>
int launch_reg(const RhtArgs& a, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return KV_INT4_ERR_CUDA;
  const bool vec = ((uintptr_t)a.x & 15u) == 0 && ((uintptr_t)a.y & 15u) == 0 && a.xs % 8 == 0 &&
                   a.ys % (F32 ? 4 : 8) == 0;
  if (vec) {
    constexpr int rows_per_warp = (32 / (D / 8)) * 4;
    const int64_t warps = (a.rows + rows_per_warp - 1) / rows_per_warp;
    int64_t grid = (warps + kRhtWarps - 1) / kRhtWarps;
    const int64_t cap = (int64_t)sm_count(dev) * 8;
    if (grid > cap) grid = cap;
    rht_vec_kernel<D, INV, F32><<<(unsigned)grid, kRhtWarps * 32, 0, stream>>>(a);
  } else {
    rht_reg_kernel<D, INV, F32><<<(unsigned)grid_for(a.rows, dev), kRhtWarps * 32, 0, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}

template <bool INV, bool F32>
int launch_smem(const RhtArgs& a, int d, cudaStream_t stream) {
  const int smem = kRhtWarps * d * (int)sizeof(float);
  static PerContext<int> attr;
  const int dev = current_device();
  if (dev < 0) return KV_INT4_ERR_CUDA;
  int set = 0;
  if (!attr.get(dev, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(rht_smem_kernel<INV, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kRhtWarps * kRhtMaxSmemHead * (int)sizeof(float)) == cudaSuccess;
      }, &set))
    return KV_INT4_ERR_CUDA;
  rht_smem_kernel<INV, F32><<<(unsigned)grid_for(a.rows, dev), kRhtWarps * 32, smem, stream>>>(a, d);
  return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}

template <bool INV, bool F32>
int dispatch(const RhtArgs& a, int d, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_reg<64, INV, F32>(a, stream);
    case 96: return launch_reg<96, INV, F32>(a, stream);
    case 128: return launch_reg<128, INV, F32>(a, stream);
    case 192: return launch_reg<192, INV, F32>(a, stream);
    case 256: return launch_reg<256, INV, F32>(a, stream);
    default: return launch_smem<INV, F32>(a, d, stream);
  }
}

}  // namespace
}  // namespace kvint4

extern "C" int kv_int4_rht(const void* x, int64_t x_row_stride, void* y, int64_t y_row_stride, int y_f32,
                           int64_t num_rows, int head_size, const int8_t* signs, int inverse, void* stream) {
  using namespace kvint4;
  if (num_rows < 0) return KV_INT4_ERR_SIZE;
  if (head_size < 1 || head_size > kRhtMaxSmemHead) return KV_INT4_ERR_HEAD_SIZE;
  if (num_rows == 0) return KV_INT4_OK;
  if (!x || !y || !signs) return KV_INT4_ERR_NULL;
  const uintptr_t ya = y_f32 ? 3u : 1u;
  if (((uintptr_t)x & 1u) || ((uintptr_t)y & ya) || x_row_stride < head_size || y_row_stride < head_size)
    return KV_INT4_ERR_ALIGN;
  RhtArgs a{static_cast<const uint16_t*>(x), x_row_stride, y, y_row_stride, num_rows, signs};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (inverse) return y_f32 ? dispatch<true, true>(a, head_size, s) : dispatch<true, false>(a, head_size, s);
  return y_f32 ? dispatch<false, true>(a, head_size, s) : dispatch<false, false>(a, head_size, s);
}
