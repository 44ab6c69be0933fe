// reshape_and_cache_int4 for sm_103a: rotate (block-diagonal randomized
// Hadamard), round through bf16, per-(token, kv head) absmax scale, signed
// INT4 codes packed two per byte, scatter through slot_mapping.
//
// Method: "Rotate KV into RHT domain in the INT4 unified attn test" (vLLM PR
// #62881), Details / Root cause and Fix; block-diagonal H_b from "vLLM --
// Attention Kernels & KV Cache Quantization" (PR #56198); cache layout from
// "[Feature] Triton INT4 per-token-head KV cache quantization" (PR #40835).
//
// Design (HBM-bound; ~10-15 ALU ops per element must stay under the copy
// time):
//  * A persistent grid walks tiles of UT head vectors ("units"; unit =
//    (token, K-or-V, kv head), token-major so that a tile's stores are
//    contiguous per token).  Tiles are staged global->shared with 16-byte
//    cp.async in a STAGES-deep pipeline; each vector sits at a padded stride
//    (2d+16 bytes, an odd number of 16-byte bank groups) so that threads
//    reading their own vectors are bank-conflict free.
//  * A vector is split across TPV threads, each owning SEG = min(b, 64)
//    consecutive outputs.  H_b = H_F (x) H_SEG (Sylvester, F = b/SEG), so a
//    thread first combines F input segments with the signs of row jj of H_F
//    (reading its F segments from shared memory) and then runs an in-register
//    SEG-point butterfly.  No warp shuffles are needed for the transform.
//  * Rounding to bf16 is one cvt per pair; the absmax is a packed
//    max.xorsign.abs on bf16x2; the per-vector absmax across the TPV threads
//    goes through shared memory.
//  * code = rint(y * r): fma(y, r, 1.5*2^23 + 8) rounds the exact product to
//    an integer (ties to even, since 1.5*2^23 + 8 is even) and leaves c + 8 in
//    the low 4 bits of the result; pairs are merged with one integer
//    multiply-add and four bytes gathered with byte permutes.

#include "common.cuh"
#include "internal.h"

namespace kvint4 {

// n / d for 0 <= n < 2^31 by a precomputed multiplier (round-up method of
// Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with s = ceil(log2 d) and m' = 2^32 + m =
// ceil(2^(32+s) / d), floor(n / d) = floor(n * m' / 2^(32+s)).
struct FastDiv {
  uint32_t d, m, s;
  __host__ FastDiv(uint32_t d_) : d(d_) {
    s = 0;
    while ((1ull << s) < d) s++;
    m = (uint32_t)((((1ull << 32) * ((1ull << s) - d)) / d) + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return (uint32_t)(((uint64_t)__umulhi(n, m) + n) >> s);
  }
};

template <int D>
struct WriteGeom {
  static constexpr int B = Head<D>::b;
  static constexpr int SEG = B < 64 ? B : 64;  // outputs per thread
  static constexpr int F = B / SEG;            // input segments combined first (1, 2 or 4)
  static constexpr int TPV = D / SEG;          // threads per head vector
  static constexpr int UT = TPV == 1 ? 256 : TPV == 2 ? 128 : 64;  // vectors per tile
  static constexpr int NT = UT * TPV;          // threads per CTA
  static constexpr int VSTRIDE = 2 * D + 16;   // padded smem bytes per staged vector
  static constexpr int STAGE_BYTES = UT * VSTRIDE;
  static constexpr int STAGES = 3;
  static constexpr int CHUNKS = D / 8;         // 16-byte chunks per bf16 vector
  static constexpr int SMEM = STAGES * STAGE_BYTES + D * 4 /*sign masks*/ + TPV * UT * 4 /*absmax*/;
  static_assert(SEG % 16 == 0, "segments must cover whole 16-byte chunks");
  static_assert(VSTRIDE % 32 == 16, "padded stride must be an odd number of 16-byte units");
};

template <int SEG>
__device__ __forceinline__ void wht_inplace(float (&w)[SEG]) {
#pragma unroll
  for (int h = 1; h < SEG; h <<= 1) {
#pragma unroll
    for (int i = 0; i < SEG; i++) {
      if ((i & h) == 0) {
        float a = w[i], c = w[i + h];
        w[i] = a + c;
        w[i + h] = a - c;
      }
    }
  }
}

// 2.0^-120: absmax below this is stored as scale 0 and all-zero codes.
__device__ constexpr float kFlushAbsmax = 7.52316384526264005e-37f;
// 1.5 * 2^23 + 8
__device__ constexpr float kCodeMagic = 12582920.0f;

template <int D, bool PREROT>
__global__ void __launch_bounds__(WriteGeom<D>::NT)
write_kernel(const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v,
             int64_t v_stride, const int64_t* __restrict__ slot_mapping, int num_tokens,
             uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
             float* __restrict__ v_scale, int64_t num_slots, int hkv, FastDiv div2h,
             const int8_t* __restrict__ signs, int32_t* status) {
  using G = WriteGeom<D>;
  constexpr int B = G::B, SEG = G::SEG, F = G::F, TPV = G::TPV, UT = G::UT, NT = G::NT;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* stages = smem;
  uint32_t* smask = reinterpret_cast<uint32_t*>(smem + G::STAGES * G::STAGE_BYTES);  // [D/2][2]
  uint32_t* samax = smask + D;                                                        // [TPV][UT]

  const int tid = threadIdx.x;
  const int64_t units = (int64_t)num_tokens * 2 * hkv;
  const int64_t num_tiles = (units + UT - 1) / UT;

  if (!PREROT) {
    for (int p = tid; p < D / 2; p += NT) {
      int s0 = signs[2 * p], s1 = signs[2 * p + 1];
      if (blockIdx.x == 0 && ((s0 != 1 && s0 != -1) || (s1 != 1 && s1 != -1))) flag(status, KV_INT4_DEV_BAD_SIGNS);
      smask[2 * p + 0] = s0 < 0 ? 0x80000000u : 0u;  // low element, applied after <<16
      smask[2 * p + 1] = s1 < 0 ? 0x80000000u : 0u;  // high element
    }
  }

  // issue the copies of one tile into one stage
  auto issue = [&](int64_t tile, int stage) {
    uint8_t* dst = stages + stage * G::STAGE_BYTES;
    const int64_t u0 = tile * UT;
    for (int idx = tid; idx < UT * G::CHUNKS; idx += NT) {
      const int uu = idx / G::CHUNKS;
      const int c = idx - uu * G::CHUNKS;
      const int64_t ug = u0 + uu;
      if (ug < units) {
        const uint32_t t = div2h.div((uint32_t)ug);  // units < 2^31 (checked on the host)
        const int rem = (int)(ug - (int64_t)t * 2 * hkv);
        const int kv = rem >= hkv;
        const int h = rem - kv * hkv;
        const uint16_t* src = (kv ? v + (int64_t)t * v_stride : k + (int64_t)t * k_stride) + h * D + c * 8;
        cp_async16(dst + uu * G::VSTRIDE + c * 16, src);
      }
    }
  };

  const int j = tid / UT;       // segment index within the vector
  const int u = tid - j * UT;   // vector index within the tile
  const int blk = j / F;        // Hadamard block
  const int jj = j - blk * F;   // row of H_F

  int64_t tile = blockIdx.x;
  const int64_t tstep = gridDim.x;
#pragma unroll 1
  for (int s = 0; s < G::STAGES - 1; s++) {
    int64_t tt = tile + s * tstep;
    if (tt < num_tiles) issue(tt, s);
    cp_async_commit();
  }
  __syncthreads();  // sign masks visible

  int stage = 0;
#pragma unroll 1
  for (int64_t it = 0; tile < num_tiles; tile += tstep, it++) {
    {
      int64_t tn = tile + (G::STAGES - 1) * tstep;
      if (tn < num_tiles) issue(tn, (stage + G::STAGES - 1) % G::STAGES);
      cp_async_commit();
    }
    cp_async_wait<G::STAGES - 1>();
    __syncthreads();

    const uint8_t* sv = stages + stage * G::STAGE_BYTES + u * G::VSTRIDE;
    const int64_t ug = tile * UT + u;
    const bool active = ug < units;

    uint32_t packed[SEG / 2];
    uint32_t amax = 0;
    if (active) {
      if (PREROT) {
        const uint4* src = reinterpret_cast<const uint4*>(sv + (blk * B + jj * SEG) * 2);
#pragma unroll
        for (int c = 0; c < SEG / 8; c++) {
          uint4 q = src[c];
          packed[4 * c + 0] = q.x;
          packed[4 * c + 1] = q.y;
          packed[4 * c + 2] = q.z;
          packed[4 * c + 3] = q.w;
        }
      } else {
        float w[SEG];
#pragma unroll
        for (int m = 0; m < F; m++) {
          const int e0 = blk * B + m * SEG;
          const uint4* src = reinterpret_cast<const uint4*>(sv + e0 * 2);
          const bool neg = (__popc(jj & m) & 1) != 0;  // H_F[jj][m] = -1
#pragma unroll
          for (int c = 0; c < SEG / 8; c++) {
            uint4 q = src[c];
            uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int p = 0; p < 4; p++) {
              const int e = e0 + 8 * c + 2 * p;  // element index of the low half
              float lo = __uint_as_float((words[p] << 16) ^ smask[e]);
              float hi = __uint_as_float((words[p] & 0xffff0000u) ^ smask[e + 1]);
              const int i = 8 * c + 2 * p;
              if (m == 0) {
                w[i] = lo;
                w[i + 1] = hi;
              } else if (neg) {
                w[i] -= lo;
                w[i + 1] -= hi;
              } else {
                w[i] += lo;
                w[i + 1] += hi;
              }
            }
          }
        }
        wht_inplace<SEG>(w);
#pragma unroll
        for (int p = 0; p < SEG / 2; p++) packed[p] = pack_bf16x2_rn(w[2 * p], w[2 * p + 1]);
      }
#pragma unroll
      for (int p = 0; p < SEG / 2; p++) amax = absmax_bf16x2(amax, packed[p]);
      uint32_t alo = amax & 0x7fffu, ahi = (amax >> 16) & 0x7fffu;
      amax = alo > ahi ? alo : ahi;
    }
    if (TPV > 1) {
      samax[j * UT + u] = amax;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < TPV; q++) {
        uint32_t o = samax[q * UT + u];
        amax = o > amax ? o : amax;
      }
    }

    if (active) {
      const uint32_t t = div2h.div((uint32_t)ug);
      const int rem = (int)(ug - (int64_t)t * 2 * hkv);
      const int kv = rem >= hkv;
      const int h = rem - kv * hkv;
      const int64_t slot = slot_mapping[t];
      if (slot >= num_slots) {
        if (j == 0) flag(status, KV_INT4_DEV_BAD_SLOT);
      } else if (slot >= 0) {
        const float a = __uint_as_float(amax << 16);
        float sc = 0.f, r = 0.f;
        if (a >= kFlushAbsmax) {
          sc = __fdiv_rn(a, 7.0f);
          r = __frcp_rn(sc);
        }
        uint32_t out[SEG / 8];
#pragma unroll
        for (int wq = 0; wq < SEG / 8; wq++) {
          uint32_t bytes[4];
#pragma unroll
          for (int p = 0; p < 4; p++) {
            const uint32_t pw = packed[4 * wq + p];
            const uint32_t tl = __float_as_uint(fmaf(bf16lo_to_f32(pw), r, kCodeMagic));
            const uint32_t th = __float_as_uint(fmaf(bf16hi_to_f32(pw), r, kCodeMagic));
            bytes[p] = tl + (th << 4);  // low byte: (c_lo + 8) + 16 (c_hi + 8)
          }
          const uint32_t x01 = __byte_perm(bytes[0], bytes[1], 0x0040);
          const uint32_t x23 = __byte_perm(bytes[2], bytes[3], 0x0040);
          out[wq] = __byte_perm(x01, x23, 0x5410) ^ 0x88888888u;  // offset binary -> two's complement
        }
        uint8_t* cache = kv ? v_cache : k_cache;
        uint4* dst = reinterpret_cast<uint4*>(cache + (slot * hkv + h) * (int64_t)(D / 2) + (blk * B + jj * SEG) / 2);
#pragma unroll
        for (int q = 0; q < SEG / 32; q++) dst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
        if (j == 0) (kv ? v_scale : k_scale)[slot * hkv + h] = sc;
      }
    }
    __syncthreads();  // the stage (and the absmax buffer) may now be overwritten
    stage = (stage + 1) % G::STAGES;
  }
  cp_async_wait<0>();
}

template <int D, bool PREROT>
static int launch_write_t(const WriteArgs& a, cudaStream_t stream) {
  using G = WriteGeom<D>;
  auto kern = write_kernel<D, PREROT>;
  const int dev = current_device();
  static bool configured[kMaxDevices] = {};
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM) != cudaSuccess)
      return KV_INT4_ERR_CUDA;
    configured[dev] = true;
  }
  static int occ[kMaxDevices] = {};
  if (!occ[dev]) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, G::NT, G::SMEM) != cudaSuccess || o < 1) return KV_INT4_ERR_CUDA;
    occ[dev] = o;
  }
  const int64_t units = (int64_t)a.num_tokens * 2 * a.num_kv_heads;
  const int64_t tiles = (units + G::UT - 1) / G::UT;
  const int64_t cap = (int64_t)sm_count(dev) * occ[dev];
  const int grid = (int)(tiles < cap ? tiles : cap);
  timing_begin(kTimedWrite, stream);
  write_kernel<D, PREROT><<<grid, G::NT, G::SMEM, stream>>>(
      static_cast<const uint16_t*>(a.k), a.k_stride, static_cast<const uint16_t*>(a.v), a.v_stride,
      a.slot_mapping, a.num_tokens, a.k_cache, a.v_cache, a.k_scale, a.v_scale,
      (int64_t)a.num_blocks * a.block_size, a.num_kv_heads, FastDiv(2u * a.num_kv_heads), a.signs,
      a.dev_status);
  timing_end(kTimedWrite, stream);
  return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
}

int launch_write(const WriteArgs& a, bool prerotated, cudaStream_t stream) {
  switch (a.head_size) {
#define KVINT4_CASE(DD) \
  case DD:              \
    return prerotated ? launch_write_t<DD, true>(a, stream) : launch_write_t<DD, false>(a, stream);
    KVINT4_CASE(64)
    KVINT4_CASE(96)
    KVINT4_CASE(128)
    KVINT4_CASE(192)
    KVINT4_CASE(256)
#undef KVINT4_CASE
    default:
      return KV_INT4_ERR_HEAD_SIZE;
  }
}

}  // namespace kvint4
