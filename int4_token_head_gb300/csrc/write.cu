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
             float* __restrict__ v_scale, CacheGeo geo, int64_t num_slots, int hkv, FastDiv div2h,
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
        uint4* dst = reinterpret_cast<uint4*>(cache + code_off(geo, slot, h) + (blk * B + jj * SEG) / 2);
#pragma unroll
        for (int q = 0; q < SEG / 32; q++) dst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
        if (j == 0) store_scale((kv ? v_scale : k_scale) + scale_off(geo, slot, h), geo, sc);
      }
    }
    __syncthreads();  // the stage (and the absmax buffer) may now be overwritten
    stage = (stage + 1) % G::STAGES;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Token-aligned variant (used whenever a token's 2*Hkv head vectors fit in one
// tile): a tile is TT whole tokens, so every thread's copy sources and its
// compute unit's (token offset, K/V, head) are fixed per thread and only the
// tile's first token changes.  Sign masks are packed per element pair and the
// butterflies run on packed fp32 pairs (two IEEE adds per instruction, the
// same roundings as the scalar form).
// ---------------------------------------------------------------------------
template <int D, bool PREROT>
__global__ void __launch_bounds__(WriteGeom<D>::NT)
write_kernel_tok(const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v,
                 int64_t v_stride, const int64_t* __restrict__ slot_mapping, int num_tokens,
                 uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
                 float* __restrict__ v_scale, CacheGeo geo, int64_t num_slots, int hkv, int tt_per_tile,
                 const int8_t* __restrict__ signs, int32_t* status) {
  using G = WriteGeom<D>;
  constexpr int B = G::B, SEG = G::SEG, F = G::F, TPV = G::TPV, UT = G::UT, NT = G::NT;
  constexpr int CPT = (UT * G::CHUNKS) / NT;  // copy chunks per thread per tile
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* stages = smem;
  uint2* smask = reinterpret_cast<uint2*>(smem + G::STAGES * G::STAGE_BYTES);  // [D/2] (lo, hi) sign bits
  uint32_t* samax = reinterpret_cast<uint32_t*>(smask + D / 2);                 // [TPV][UT]

  const int tid = threadIdx.x;
  const int units_per_token = 2 * hkv;
  const int units = tt_per_tile * units_per_token;  // <= UT
  const int num_tiles = (num_tokens + tt_per_tile - 1) / tt_per_tile;

  if (!PREROT) {
    for (int p = tid; p < D / 2; p += NT) {
      const int s0 = signs[2 * p], s1 = signs[2 * p + 1];
      if (blockIdx.x == 0 && ((s0 != 1 && s0 != -1) || (s1 != 1 && s1 != -1))) flag(status, KV_INT4_DEV_BAD_SIGNS);
      smask[p] = make_uint2(s0 < 0 ? 0x80000000u : 0u, s1 < 0 ? 0x80000000u : 0u);
    }
  }

  // copy slots of this thread (tile-invariant): chunk idx = tid + NT * q
  const uint16_t* c_src[CPT];
  int c_tok[CPT];    // token offset within the tile, or -1 if unused
  int64_t c_strd[CPT];
#pragma unroll
  for (int q = 0; q < CPT; q++) {
    const int idx = tid + NT * q;
    const int uu = idx / G::CHUNKS, c = idx % G::CHUNKS;
    const int tt = uu / units_per_token, w = uu % units_per_token;
    const int kv = w >= hkv, h = kv ? w - hkv : w;
    c_tok[q] = uu < units ? tt : -1;
    c_src[q] = (kv ? v : k) + (int64_t)tt * (kv ? v_stride : k_stride) + h * D + c * 8;
    c_strd[q] = (int64_t)tt_per_tile * (kv ? v_stride : k_stride);
  }
  auto issue = [&](int tile, int stage) {
    const uint32_t dst0 = smem_addr(stages + stage * G::STAGE_BYTES);
    const int t0 = tile * tt_per_tile;
#pragma unroll
    for (int q = 0; q < CPT; q++) {
      const int idx = tid + NT * q;
      const int uu = idx / G::CHUNKS, c = idx % G::CHUNKS;
      if (c_tok[q] >= 0 && t0 + c_tok[q] < num_tokens) {
        const uint16_t* src = c_src[q] + (int64_t)tile * c_strd[q];
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst0 + uu * G::VSTRIDE + c * 16), "l"(src));
      }
    }
  };

  const int j = tid / UT;       // segment index within the vector
  const int u = tid - j * UT;   // vector index within the tile
  const int blk = j / F;        // Hadamard block
  const int jj = j - blk * F;   // row of H_F
  const int u_tt = u / units_per_token, u_w = u % units_per_token;
  const int u_kv = u_w >= hkv, u_h = u_kv ? u_w - hkv : u_w;
  uint8_t* const u_cache = u_kv ? v_cache : k_cache;
  float* const u_scale = u_kv ? v_scale : k_scale;

  int tile = blockIdx.x;
  const int tstep = gridDim.x;
#pragma unroll 1
  for (int s = 0; s < G::STAGES - 1; s++) {
    const int tt = tile + s * tstep;
    if (tt < num_tiles) issue(tt, s);
    cp_async_commit();
  }
  __syncthreads();  // sign masks visible

  int stage = 0;
#pragma unroll 1
  for (; tile < num_tiles; tile += tstep) {
    {
      const int tn = tile + (G::STAGES - 1) * tstep;
      if (tn < num_tiles) issue(tn, (stage + G::STAGES - 1) % G::STAGES);
      cp_async_commit();
    }
    cp_async_wait<G::STAGES - 1>();
    __syncthreads();

    const uint8_t* sv = stages + stage * G::STAGE_BYTES + u * G::VSTRIDE;
    const int t = tile * tt_per_tile + u_tt;
    const bool active = u < units && t < num_tokens;

    uint32_t packed[SEG / 2];
    uint32_t amax = 0;
    if (active) {
      if (PREROT) {
        const uint4* src = reinterpret_cast<const uint4*>(sv + (blk * B + jj * SEG) * 2);
#pragma unroll
        for (int c = 0; c < SEG / 8; c++) {
          const uint4 qv = src[c];
          packed[4 * c + 0] = qv.x;
          packed[4 * c + 1] = qv.y;
          packed[4 * c + 2] = qv.z;
          packed[4 * c + 3] = qv.w;
        }
      } else {
        float2 W[SEG / 2];  // element pairs (2i, 2i+1)
#pragma unroll
        for (int m = 0; m < F; m++) {
          const int e0 = blk * B + m * SEG;
          const uint4* src = reinterpret_cast<const uint4*>(sv + e0 * 2);
          const uint4* msk = reinterpret_cast<const uint4*>(smask + e0 / 2);
          const bool neg = (__popc(jj & m) & 1) != 0;  // H_F[jj][m] = -1
#pragma unroll
          for (int c = 0; c < SEG / 8; c++) {
            const uint4 qv = src[c];
            const uint4 m01 = msk[2 * c], m23 = msk[2 * c + 1];
            const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
            const uint32_t mlo[4] = {m01.x, m01.z, m23.x, m23.z};
            const uint32_t mhi[4] = {m01.y, m01.w, m23.y, m23.w};
#pragma unroll
            for (int p = 0; p < 4; p++) {
              const float lo = __uint_as_float(words[p] * 65536u + mlo[p]);    // adding 2^31 flips the sign bit
              const float hi = __uint_as_float((words[p] & 0xffff0000u) ^ mhi[p]);
              const float2 z = make_float2(lo, hi);
              const int i = 4 * c + p;
              if (m == 0) W[i] = z;
              else W[i] = neg ? f2sub(W[i], z) : f2add(W[i], z);
            }
          }
        }
        // H_SEG: the stage pairing adjacent elements inside a pair, then packed stages
#pragma unroll
        for (int i = 0; i < SEG / 2; i++) W[i] = make_float2(W[i].x + W[i].y, W[i].x - W[i].y);
#pragma unroll
        for (int hp = 1; hp < SEG / 2; hp <<= 1) {
#pragma unroll
          for (int i = 0; i < SEG / 2; i++) {
            if ((i & hp) == 0) {
              const float2 a = W[i], b = W[i + hp];
              W[i] = f2add(a, b);
              W[i + hp] = f2sub(a, b);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < SEG / 2; i++) packed[i] = pack_bf16x2_rn(W[i].x, W[i].y);
      }
#pragma unroll
      for (int p = 0; p < SEG / 2; p++) amax = absmax_bf16x2(amax, packed[p]);
      const uint32_t alo = amax & 0x7fffu, ahi = (amax >> 16) & 0x7fffu;
      amax = alo > ahi ? alo : ahi;
    }
    if (TPV > 1) {
      samax[j * UT + u] = amax;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < TPV; q++) {
        const uint32_t o = samax[q * UT + u];
        amax = o > amax ? o : amax;
      }
    }

    if (active) {
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
        const float2 r2 = make_float2(r, r), magic2 = make_float2(kCodeMagic, kCodeMagic);
        uint32_t out[SEG / 8];
#pragma unroll
        for (int wq = 0; wq < SEG / 8; wq++) {
          uint32_t bytes[4];
#pragma unroll
          for (int p = 0; p < 4; p++) {
            const uint32_t pw = packed[4 * wq + p];
            const float2 tq = f2fma(make_float2(__uint_as_float(pw * 65536u), __uint_as_float(pw & 0xffff0000u)), r2, magic2);
            bytes[p] = __float_as_uint(tq.y) * 16u + __float_as_uint(tq.x);  // low byte: (c_lo + 8) + 16 (c_hi + 8)
          }
          const uint32_t x01 = __byte_perm(bytes[0], bytes[1], 0x0040);
          const uint32_t x23 = __byte_perm(bytes[2], bytes[3], 0x0040);
          out[wq] = __byte_perm(x01, x23, 0x5410) ^ 0x88888888u;  // offset binary -> two's complement
        }
        uint4* dst = reinterpret_cast<uint4*>(u_cache + code_off(geo, slot, u_h) + (blk * B + jj * SEG) / 2);
#pragma unroll
        for (int q = 0; q < SEG / 32; q++) dst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
        if (j == 0) store_scale(u_scale + scale_off(geo, slot, u_h), geo, sc);
      }
    }
    __syncthreads();  // the stage (and the absmax buffer) may now be overwritten
    stage = (stage + 1) % G::STAGES;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Tensor-core variant of the rotation (the default for head sizes up to 192).
//
// H_b = H_{b/16} (x) H_16 (Sylvester; the group index is the high part of
// the element index), so for each 16-element group q the 16-point transform
// of the sign-flipped inputs, z_q = H_16 . D_q . x_q, is a 16 x 16 matrix
// product with exact +-1 entries: one bf16 mma.sync (inputs exact, fp32
// accumulation) handles 16 head vectors x one group x 8 outputs.  The
// remaining log2(b/16) stages across groups of a Hadamard block are fp32
// butterflies on values that the same thread already holds for every group.
// The output columns of the MMA are permuted (B_q's columns) so that each lane
// ends up with four consecutive outputs, i.e. two whole code bytes, per group.
// ---------------------------------------------------------------------------
template <int D>
struct TcGeom {
  static constexpr int B = D & -D;
  static constexpr int NG = D / 16;        // 16-element groups per head vector
  static constexpr int GB = B / 16;        // groups per Hadamard block
  static constexpr int WARPS = 4;
  static constexpr int NT = WARPS * 32;
  static constexpr int UT = WARPS * 16;    // head vectors per tile (16 rows per warp)
  static constexpr int ROWB = 2 * D;       // bytes of one bf16 head vector
  // Staging: a warp's 16 head vectors sit in 8 pairs, each pair contiguous
  // (one bulk copy fills it when the two vectors are neighbours in memory)
  // and padded by 16 bytes.  MMA rows g and g + 8 are vectors 2g and 2g + 1,
  // so the eight rows an ldmatrix reads are first (or second) vectors of
  // eight pairs, 16 bytes apart modulo 128: no bank conflicts.  Each warp
  // owns its rows of every stage and waits on its own barrier, so warps never
  // wait for one another.  Stages and CTAs per SM per head size (measured on
  // GB300: warps per SM matter more than depth).
  static constexpr int PSTRIDE = 2 * ROWB + 16;  // bytes per staged pair
  static constexpr int WSTAGE = 8 * PSTRIDE;     // one warp's rows of one stage
  static constexpr int STAGES = D == 96 ? 4 : 2;
  static constexpr int MIN_CTAS = D == 192 ? 3 : 4;
  static constexpr int STAGE_BYTES = WARPS * WSTAGE;
  static constexpr int BFRAG_BYTES = NG * 2 * 32 * 8;
  static constexpr int SCALE_TABLE_BYTES = 2 * 128 * 4;
  static constexpr int SMEM = STAGES * STAGE_BYTES + BFRAG_BYTES + SCALE_TABLE_BYTES + WARPS * STAGES * 8;
};

// byte offset of head vector v (0..15) within a warp's stage rows
template <int D>
__device__ __forceinline__ int tc_vec_off(int v) { return (v >> 1) * TcGeom<D>::PSTRIDE + (v & 1) * TcGeom<D>::ROWB; }

// output o (0..15) of MMA column n of n-tile t: lane c holds columns 2c, 2c+1,
// i.e. outputs 4c + 2t and 4c + 2t + 1
__device__ __forceinline__ int tc_out_index(int t, int n) { return 4 * (n >> 1) + 2 * t + (n & 1); }

template <int D>
__global__ void __launch_bounds__(TcGeom<D>::NT, TcGeom<D>::MIN_CTAS)
write_kernel_tc(const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v, int64_t v_stride,
                const int64_t* __restrict__ slot_mapping, int num_tokens, uint8_t* __restrict__ k_cache,
                uint8_t* __restrict__ v_cache, float* __restrict__ k_scale, float* __restrict__ v_scale,
                CacheGeo geo, int64_t num_slots, int hkv, int tt_per_tile, const int8_t* __restrict__ signs,
                int32_t* status) {
  using G = TcGeom<D>;
  constexpr int NG = G::NG, GB = G::GB, NT = G::NT;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* stages = smem;
  uint2* sbfrag = reinterpret_cast<uint2*>(smem + G::STAGES * G::STAGE_BYTES);  // [NG][2][32]
  uint32_t* stab = reinterpret_cast<uint32_t*>(smem + G::STAGES * G::STAGE_BYTES + G::BFRAG_BYTES);  // [2][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int units_per_token = 2 * hkv;
  const int units = tt_per_tile * units_per_token;  // <= UT
  const int num_tiles = (num_tokens + tt_per_tile - 1) / tt_per_tile;
  // this warp's stage barriers [STAGES]
  const uint32_t bars =
      smem_addr(smem + G::STAGES * G::STAGE_BYTES + G::BFRAG_BYTES + G::SCALE_TABLE_BYTES) + warp * G::STAGES * 8;

  // B_q fragments of D_q . H_16 (columns permuted), bf16 +-1
  for (int e = tid; e < NG * 2 * 32; e += NT) {
    const int q = e / 64, t = (e / 32) & 1, l = e & 31;
    const int lg = l >> 2, lc = l & 3;
    const int o = tc_out_index(t, lg);
    uint32_t w[2];
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t pair = 0;
#pragma unroll
      for (int e2 = 0; e2 < 2; e2++) {
        const int i = 2 * lc + 8 * half + e2;  // k index (input element within the group)
        const int sgn = signs[16 * q + i];
        const bool neg = ((__popc(i & o) & 1) != 0) != (sgn < 0);
        pair |= (neg ? 0xbf80u : 0x3f80u) << (16 * e2);
        if (blockIdx.x == 0 && t == 0 && lg == 0 && sgn != 1 && sgn != -1) flag(status, KV_INT4_DEV_BAD_SIGNS);
      }
      w[half] = pair;
    }
    sbfrag[e] = make_uint2(w[0], w[1]);
  }
  // Scale tables.  absmax is a bf16 value (1 + m/128) 2^e, so
  // s = fp32(absmax / 7) = fp32((1 + m/128) / 7) 2^e and fp32(1 / s) =
  // fp32(1 / fp32((1 + m/128) / 7)) 2^-e exactly (all normal numbers above
  // the flush bound): one correctly rounded division and reciprocal per m.
  if (tid < 128) {
    const float t7 = __fdiv_rn(1.0f + (float)tid * 0.0078125f, 7.0f);
    stab[tid] = __float_as_uint(t7);
    stab[128 + tid] = __float_as_uint(__frcp_rn(t7));
  }
  if (lane == 0) {
    for (int s = 0; s < G::STAGES; s++) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
  }

  // copies: lane cv < 16 owns head vector warp * 16 + cv of every tile.  With
  // an even head count the two vectors of a pair are neighbouring heads of
  // one token, so the even lane copies both with one bulk copy.
  const bool paired = (hkv & 1) == 0;
  const int cv = lane & 15;
  const int cu = warp * 16 + cv;
  const bool c_used = lane < 16 && cu < units && (!paired || (cv & 1) == 0);
  const int c_tt = cu / units_per_token, c_w = cu % units_per_token;
  const int c_kv = c_w >= hkv, c_h = c_kv ? c_w - hkv : c_w;
  const uint16_t* const c_src = (c_kv ? v : k) + (int64_t)c_tt * (c_kv ? v_stride : k_stride) + c_h * D;
  const int64_t c_tstride = (int64_t)tt_per_tile * (c_kv ? v_stride : k_stride);
  const uint32_t c_dst = smem_addr(stages + warp * G::WSTAGE + tc_vec_off<D>(cv));
  const uint32_t c_bytes = paired ? 2 * G::ROWB : G::ROWB;
  auto issue = [&](int tl, int stage) {
    const bool go = c_used && tl * tt_per_tile + c_tt < num_tokens;
    const unsigned m = __ballot_sync(0xffffffffu, go);
    const uint32_t bar = bars + 8 * stage;
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(m) * c_bytes);
    __syncwarp();
    if (go) bulk_g2s(c_dst + stage * G::STAGE_BYTES, c_src + (int64_t)tl * c_tstride, c_bytes, bar);
  };

  // this thread's two MMA rows g and g + 8 are head vectors 2g and 2g + 1
  int r_tt[2], r_kv[2], r_h[2];
#pragma unroll
  for (int rr = 0; rr < 2; rr++) {
    const int uu = warp * 16 + 2 * g + rr;
    r_tt[rr] = uu < units ? uu / units_per_token : -1;
    const int w = uu % units_per_token;
    r_kv[rr] = w >= hkv;
    r_h[rr] = r_kv[rr] ? w - hkv : w;
  }
  // ldmatrix row for this lane: matrices (rows 0-7|8-15) x (k 0-7|8-15);
  // MMA row m is vector 2 (m & 7) + (m >> 3)
  const int a_m = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int a_off = warp * G::WSTAGE + tc_vec_off<D>(2 * (a_m & 7) + (a_m >> 3));
  const int a_half = lane >> 4;  // which 16-byte half of a 16-element group

  __syncthreads();  // B fragments, scale tables and barrier initialisation visible

  int tile = blockIdx.x;
  const int tstep = gridDim.x;
#pragma unroll 1
  for (int s = 0; s < G::STAGES - 1; s++) {
    const int tt = tile + s * tstep;
    if (tt < num_tiles) issue(tt, s);
  }
  // slots of this thread's rows, loaded one tile ahead
  auto load_slots = [&](int tl, int64_t (&sl)[2]) {
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      const int tok = tl * tt_per_tile + r_tt[rr];
      sl[rr] = (tl < num_tiles && r_tt[rr] >= 0 && tok < num_tokens) ? slot_mapping[tok] : -1;
    }
  };
  int64_t next_slot[2];
  load_slots(tile, next_slot);

  int stage = 0;
  uint32_t phase = 0;  // bit s: parity of stage s's next completion
  bool stalled = false;
#pragma unroll 1
  for (; tile < num_tiles; tile += tstep) {
    int64_t r_slot[2] = {next_slot[0], next_slot[1]};
    load_slots(tile + tstep, next_slot);
    {
      // refill the stage this warp finished with at its previous tile
      const int tn = tile + (G::STAGES - 1) * tstep;
      if (tn < num_tiles) issue(tn, stage == 0 ? G::STAGES - 1 : stage - 1);
    }
    if (!mbar_wait_bounded(bars + 8 * stage, (phase >> stage) & 1)) {
      stalled = true;
      break;
    }
    phase ^= 1u << stage;

    uint8_t* const wbase = stages + stage * G::STAGE_BYTES + warp * G::WSTAGE;
    const uint8_t* sa = stages + stage * G::STAGE_BYTES + a_off;
    uint32_t pk[2][NG][2];  // [n-tile][group][row g / row g+8]: bf16x2 of outputs (4c+2t, 4c+2t+1)
#pragma unroll
    for (int t = 0; t < 2; t++) {
      float cacc[NG][4];
#pragma unroll
      for (int q = 0; q < NG; q++) {
        uint32_t a[4];
        ldmatrix_x4(a, sa + (2 * q + a_half) * 16);
        const uint2 bf = sbfrag[(q * 2 + t) * 32 + lane];
        mma_16816_bf16_z(cacc[q], a, bf.x, bf.y);
      }
      // cross-group stages of each Hadamard block
#pragma unroll
      for (int h = 1; h < GB; h <<= 1) {
#pragma unroll
        for (int q = 0; q < NG; q++) {
          if ((q & h) == 0) {
            const float2 a0 = make_float2(cacc[q][0], cacc[q][1]), a1 = make_float2(cacc[q][2], cacc[q][3]);
            const float2 b0 = make_float2(cacc[q + h][0], cacc[q + h][1]), b1 = make_float2(cacc[q + h][2], cacc[q + h][3]);
            const float2 s0 = f2add(a0, b0), s1 = f2add(a1, b1), d0 = f2sub(a0, b0), d1 = f2sub(a1, b1);
            cacc[q][0] = s0.x; cacc[q][1] = s0.y; cacc[q][2] = s1.x; cacc[q][3] = s1.y;
            cacc[q + h][0] = d0.x; cacc[q + h][1] = d0.y; cacc[q + h][2] = d1.x; cacc[q + h][3] = d1.y;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NG; q++) {
        pk[t][q][0] = pack_bf16x2_rn(cacc[q][0], cacc[q][1]);
        pk[t][q][1] = pack_bf16x2_rn(cacc[q][2], cacc[q][3]);
      }
    }

    // this thread's rows: slot (or -1: nothing to store)
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      if (r_slot[rr] >= num_slots) {
        if (cq == 0 && r_kv[rr] == 0 && r_h[rr] == 0) flag(status, KV_INT4_DEV_BAD_SLOT);
        r_slot[rr] = -1;
      }
    }
    // per row: absmax over the 4 lanes of the quad, scale, codes.  The codes
    // are staged in the row's own (already consumed) input bytes.
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      uint32_t am = 0;
#pragma unroll
      for (int t = 0; t < 2; t++)
#pragma unroll
        for (int q = 0; q < NG; q++) am = absmax_bf16x2(am, pk[t][q][rr]);
      uint32_t a16 = max(am & 0x7fffu, (am >> 16) & 0x7fffu);
      a16 = max(a16, __shfl_xor_sync(0xffffffffu, a16, 1));
      a16 = max(a16, __shfl_xor_sync(0xffffffffu, a16, 2));
      const float amax = __uint_as_float(a16 << 16);
      float sc = 0.f, r = 0.f;
      if (amax >= kFlushAbsmax) {
        if (a16 < 0x7f80u) {
          const uint32_t m = a16 & 0x7fu;
          const int e = (int)(a16 >> 7) - 127;
          sc = __uint_as_float(stab[m] + (uint32_t)(e << 23));
          r = __uint_as_float(stab[128 + m] - (uint32_t)(e << 23));
        } else {  // inf / NaN input
          sc = __fdiv_rn(amax, 7.0f);
          r = __frcp_rn(sc);
        }
      }
      const float2 r2 = make_float2(r, r), magic2 = make_float2(kCodeMagic, kCodeMagic);
      uint8_t* orow = wbase + tc_vec_off<D>(2 * g + rr);
#pragma unroll
      for (int q = 0; q < NG; q++) {
        uint32_t bytes[2];
#pragma unroll
        for (int t = 0; t < 2; t++) {
          const uint32_t pw = pk[t][q][rr];
          const float2 tq = f2fma(make_float2(__uint_as_float(pw * 65536u), __uint_as_float(pw & 0xffff0000u)), r2, magic2);
          bytes[t] = __float_as_uint(tq.y) * 16u + __float_as_uint(tq.x);  // (c_lo + 8) | (c_hi + 8) << 4 (mod 16)
        }
        // outputs 4cq..4cq+3 of group q = bytes 8q + 2cq, 8q + 2cq + 1; the xor
        // turns the four offset-binary nibbles into two's complement at once
        *reinterpret_cast<uint16_t*>(orow + 8 * q + 2 * cq) = (uint16_t)(__byte_perm(bytes[0], bytes[1], 0x0040) ^ 0x8888u);
      }
      if (cq == 0 && r_slot[rr] >= 0) store_scale((r_kv[rr] ? v_scale : k_scale) + scale_off(geo, r_slot[rr], r_h[rr]), geo, sc);
    }
    __syncwarp();
    // 16-byte stores: the quad of rows g, g + 8 stores those rows' chunks
    constexpr int CPR = D / 32;  // 16-byte chunks per code row
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      if (r_slot[rr] < 0) continue;
      uint8_t* dst = (r_kv[rr] ? v_cache : k_cache) + code_off(geo, r_slot[rr], r_h[rr]);
#pragma unroll
      for (int ch = cq; ch < CPR; ch += 4)
        *reinterpret_cast<uint4*>(dst + ch * 16) = *reinterpret_cast<const uint4*>(wbase + tc_vec_off<D>(2 * g + rr) + ch * 16);
    }
    // this tile's shared-memory reads and writes come before the bulk copy
    // that refills the stage at the next tile
    fence_proxy_async_smem();
    __syncwarp();
    stage = stage + 1 == G::STAGES ? 0 : stage + 1;
  }
  if (stalled) {
    // report, then let the copies this warp still has in flight land (each
    // wait again bounded) before the CTA's shared memory is released
    if (lane == 0) flag(status, KV_INT4_DEV_TIMEOUT);
    for (int j = 0; j < G::STAGES; j++) {  // tiles tile .. tile + (STAGES - 1) * tstep
      const int sj = (stage + j) % G::STAGES;
      if (tile + j * tstep < num_tiles && !mbar_wait_bounded(bars + 8 * sj, (phase >> sj) & 1)) break;
    }
  }
}

template <int D, bool PREROT>
static int launch_write_t(const WriteArgs& a, cudaStream_t stream) {
  using G = WriteGeom<D>;
  auto kern = write_kernel<D, PREROT>;
  const int dev = current_device();
  // each kernel's shared-memory limit and CTAs per SM, set once per device context
  auto setup = [](auto k, int threads, int smem, int* o) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(o, k, threads, smem) == cudaSuccess && *o >= 1;
  };
  static PerContext<int> occ_cache;
  int occ = 0;
  if (!occ_cache.get(dev, [&](int* o) { return setup(kern, G::NT, G::SMEM, o); }, &occ)) return KV_INT4_ERR_CUDA;
  if constexpr (!PREROT && D <= 192) {
    using T = TcGeom<D>;
    if (2 * a.num_kv_heads <= T::UT) {
      auto tckern = write_kernel_tc<D>;
      static PerContext<int> tc_occ_cache;
      int tc_occ = 0;
      if (!tc_occ_cache.get(dev, [&](int* o) { return setup(tckern, T::NT, T::SMEM, o); }, &tc_occ))
        return KV_INT4_ERR_CUDA;
      const int tt = T::UT / (2 * a.num_kv_heads);
      const int64_t tiles = ((int64_t)a.num_tokens + tt - 1) / tt;
      const int64_t tcap = (int64_t)sm_count(dev) * tc_occ;
      const int grid = (int)(tiles < tcap ? tiles : tcap);
      timing_begin(kTimedWrite, stream);
      tckern<<<grid, T::NT, T::SMEM, stream>>>(
          static_cast<const uint16_t*>(a.k), a.k_stride, static_cast<const uint16_t*>(a.v), a.v_stride,
          a.slot_mapping, a.num_tokens, a.k_cache, a.v_cache, a.k_scale, a.v_scale, a.geo,
          (int64_t)a.num_blocks * a.block_size, a.num_kv_heads, tt, a.signs, a.dev_status);
      timing_end(kTimedWrite, stream);
      return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
    }
  }
  const int64_t cap = (int64_t)sm_count(dev) * occ;
  if (2 * a.num_kv_heads <= G::UT) {
    auto tkern = write_kernel_tok<D, PREROT>;
    static PerContext<int> tok_attr;
    int set = 0;
    if (!tok_attr.get(dev, [&](int* v) {
          *v = 1;
          return cudaFuncSetAttribute(tkern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM) == cudaSuccess;
        }, &set))
      return KV_INT4_ERR_CUDA;
    const int tt = G::UT / (2 * a.num_kv_heads);
    const int64_t tiles = ((int64_t)a.num_tokens + tt - 1) / tt;
    const int grid = (int)(tiles < cap ? tiles : cap);
    timing_begin(kTimedWrite, stream);
    tkern<<<grid, G::NT, G::SMEM, stream>>>(
        static_cast<const uint16_t*>(a.k), a.k_stride, static_cast<const uint16_t*>(a.v), a.v_stride,
        a.slot_mapping, a.num_tokens, a.k_cache, a.v_cache, a.k_scale, a.v_scale, a.geo,
        (int64_t)a.num_blocks * a.block_size, a.num_kv_heads, tt, a.signs, a.dev_status);
    timing_end(kTimedWrite, stream);
    return cudaGetLastError() == cudaSuccess ? KV_INT4_OK : KV_INT4_ERR_CUDA;
  }
  const int64_t units = (int64_t)a.num_tokens * 2 * a.num_kv_heads;
  const int64_t tiles = (units + G::UT - 1) / G::UT;
  const int grid = (int)(tiles < cap ? tiles : cap);
  timing_begin(kTimedWrite, stream);
  write_kernel<D, PREROT><<<grid, G::NT, G::SMEM, stream>>>(
      static_cast<const uint16_t*>(a.k), a.k_stride, static_cast<const uint16_t*>(a.v), a.v_stride,
      a.slot_mapping, a.num_tokens, a.k_cache, a.v_cache, a.k_scale, a.v_scale, a.geo,
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
