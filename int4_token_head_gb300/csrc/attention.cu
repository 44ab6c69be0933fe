// unified_attention_int4 for sm_103a: varlen prefill + decode with GQA over
// the paged INT4 per-token-head cache, computed in the rotated domain.
//
// Method ("Rotate KV into RHT domain in the INT4 unified attn test", vLLM PR
// #62881, Details / Root cause; b in place of d per "vLLM -- Attention
// Kernels & KV Cache Quantization", PR #56198):
//   q' = (I_n (x) H_b) D q,  score_t = softmax_scale/b * q' . (c_t s_t),
//   o' = sum_t softmax_t * (c_t^v s_t^v),  out = D (I_n (x) H_b) o' / b.
//
// Launch sequence (all on the caller's stream):
//  1. prep: CTA 0 builds the schedule from seq_lens / query_start_loc (decode
//     sequence list with block prefix sums, prefill tile list); the other
//     CTAs rotate every query once and pre-scale it by
//     softmax_scale * log2(e) / b, stored as f16 (scores are then base-2).
//  2. prefill (only for sequences whose q_len * G exceeds the decode column
//     budget, or G > 8): one CTA per 64-row tile of (query token x q head of
//     one kv group), FA2-style mma.sync with K/V dequantised once per block
//     into f16 shared tiles.
//  3. decode: stream-K over the flattened (decode sequence, head group,
//     position) space, a position being one or two consecutive 16-key
//     blocks; every CTA takes an equal contiguous range, so the split-KV
//     load balance is exact.  The CTA stages each block of its head group
//     into shared memory; per block a warp computes S^T = K Q'^T for its
//     head with the 16 keys as the MMA M dimension (q_len*G <= 8 query
//     columns as N; two blocks of a position share the 8 columns),
//     converting INT4 nibbles straight into f16 A fragments in registers
//     (the in-register order of head dimensions is a permutation applied
//     consistently to q', which leaves q'.K unchanged); P is transposed with
//     movmatrix into the B operand of O'^T += V^T P^T.  Each segment piece
//     writes (o', m, l) to the workspace.
//  4. reduce: merges the pieces of every decode segment with the log-sum-exp
//     rule, normalises, applies the inverse rotation and writes bf16.
//
// Device-side checks never trap: bad blocks are masked, bad sequences
// skipped, and a KV_INT4_DEV_* bit is ORed into the caller's status word.

#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace kvint4 {

constexpr float kLog2e = 1.4426950408889634f;

struct PlanView {
  int32_t* plan;      // [0] n_dseq, [1] n_prefill_items, [2] prefill work counter, [3] n_pseq
  int32_t* dseq;
  int64_t* dprefix;
  int2* ptab;         // prefill sequences in order: (seq id, index of its first item); [n_pseq].y = items
  __half* qrot;
  float* direct_o;
  float* direct_ml;
  float* warp_o;
  float* warp_ml;
};

static PlanView plan_view(void* ws, const WorkspaceLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  PlanView v;
  v.plan = reinterpret_cast<int32_t*>(b + L.plan);
  v.dseq = reinterpret_cast<int32_t*>(b + L.dseq);
  v.dprefix = reinterpret_cast<int64_t*>(b + L.dprefix);
  v.ptab = reinterpret_cast<int2*>(b + L.pitems);
  v.qrot = reinterpret_cast<__half*>(b + L.qrot);
  v.direct_o = reinterpret_cast<float*>(b + L.direct_o);
  v.direct_ml = reinterpret_cast<float*>(b + L.direct_ml);
  v.warp_o = reinterpret_cast<float*>(b + L.warp_o);
  v.warp_ml = reinterpret_cast<float*>(b + L.warp_ml);
  return v;
}

// KV cache formats: INT4 codes of the rotated vectors, two per byte (the
// method), or int8 codes of the unrotated vectors (the int8_per_token_head
// sibling mode).
enum KvFmt { kFmtInt4 = 0, kFmtInt8 = 1 };

struct Common {
  const uint16_t* q;
  int64_t q_stride;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  CacheGeo geo;  // cache strides (separate or in-slot scales)
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int num_seqs;
  int num_q_tokens;
  int hq;
  int hkv;
  int group;
  FastDiv gdiv{1};  // division by group
  int num_blocks;
  int causal;
  int window;    // sliding window (0: none): the query at position p sees no key at p - window or before
  float qscale;  // softmax_scale * log2(e) / b
  const int8_t* signs;
  uint16_t* out;
  int64_t out_stride;
  int32_t* status;
  int tile_tokens;  // prefill: query tokens per 64-row tile
  int hg;           // decode: kv heads per CTA (largest divisor of hkv <= 8)
  int ng;           // decode: head groups per sequence (hkv / hg)
  int np;           // decode: 16-key blocks per schedule position (1 or 2)
  int dcols;        // decode: query columns per block (8 / np); longer queries go to prefill
  long long max_items;  // capacity of the prefill item list
};

// first key position visible to the query at position qpos
__device__ __forceinline__ int window_lo(const Common& c, int qpos) {
  return c.window > 0 ? max(0, qpos - c.window + 1) : 0;
}
// first 16-key block a sequence's attention reads: blocks wholly before the
// window of its earliest query (position L - q_len) are never visible
__device__ __forceinline__ int first_block(const Common& c, int L, int ql) { return window_lo(c, L - ql) >> 4; }

__device__ __forceinline__ bool is_decode_kind(int qlen, const Common& c) {
  return c.group <= c.dcols && qlen * c.group <= c.dcols;
}

// ---------------------------------------------------------------------------
// 1. prep: schedule (CTA 0) + query rotation (CTAs 1..)
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
// query rotation: one thread per piece of kPrepPiece(D) consecutive elements
// of a row (a whole 16-element Hadamard block, or 16 elements of a longer
// one, its later stages by shuffles: more threads in flight per SM than
// longer pieces, measured faster)
__host__ __device__ constexpr int kPrepPiece(int d) { return (d & -d) < 16 ? (d & -d) : 16; }

template <typename T>
__device__ T block_exclusive_scan(T v, T* total, T* sbuf /*[kPrepThreads/32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sbuf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = lane < kPrepThreads / 32 ? sbuf[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kPrepThreads / 32) sbuf[lane] = w;
  }
  __syncthreads();
  T before = warp > 0 ? sbuf[warp - 1] : T(0);
  *total = sbuf[kPrepThreads / 32 - 1];
  __syncthreads();
  return before + x - v;
}

template <int D, bool ROT>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(Common c, PlanView pv) {
  if (blockIdx.x == 0) {
    __shared__ int32_t s_i32[kPrepThreads / 32];
    __shared__ long long s_i64[kPrepThreads / 32];
    int n_dseq = 0, n_pseq = 0;
    long long dpre = 0, n_items = 0;
    for (int base = 0; base < c.num_seqs; base += kPrepThreads) {
      const int s = base + threadIdx.x;
      int kind = 0, nblk = 0, ntiles = 0, ql = 0, L = 0;
      if (s < c.num_seqs) {
        const int q0 = c.qsl[s], q1 = c.qsl[s + 1];
        L = c.seq_lens[s];
        ql = q1 - q0;
        const bool bad = q0 < 0 || q1 > c.num_q_tokens || ql < 0 || L < ql ||
                         (long long)L > (long long)c.max_blocks * 16;
        if (bad) {
          flag(c.status, KV_INT4_DEV_BAD_SEQ);
        } else if (ql > 0) {
          kind = is_decode_kind(ql, c) ? 1 : 2;
          nblk = (L + 15) / 16;
          if (kind == 2) ntiles = (ql + c.tile_tokens - 1) / c.tile_tokens;
        }
      }
      int tot_a, tot_p;
      long long tot_b, tot_c;
      const int ex_a = block_exclusive_scan<int>(kind == 1, &tot_a, s_i32);
      const int npos = kind == 1 ? (nblk - first_block(c, L, ql) + c.np - 1) / c.np : 0;
      const long long ex_b = block_exclusive_scan<long long>(npos, &tot_b, s_i64);
      const int ex_p = block_exclusive_scan<int>(kind == 2, &tot_p, s_i32);
      const long long ex_c = block_exclusive_scan<long long>((long long)ntiles * c.hkv, &tot_c, s_i64);
      if (kind == 1) {
        pv.dseq[n_dseq + ex_a] = s;
        pv.dprefix[n_dseq + ex_a] = dpre + ex_b;
      } else if (kind == 2) {
        // the prefill kernel expands (tile, kv head) items from this table
        pv.ptab[n_pseq + ex_p] = make_int2(s, (int)min(n_items + ex_c, (long long)INT_MAX));
      }
      n_dseq += tot_a;
      dpre += tot_b;
      n_pseq += tot_p;
      n_items += tot_c;
    }
    if (threadIdx.x == 0) {
      pv.dprefix[n_dseq] = dpre;
      pv.plan[0] = n_dseq;
      // more items than the workspace was sized for only happens with
      // inconsistent query_start_loc: the prefill part is dropped and flagged
      const bool over = n_items > c.max_items || n_items > INT_MAX;
      if (over) flag(c.status, KV_INT4_DEV_BAD_SEQ);
      pv.ptab[n_pseq] = make_int2(-1, over ? 0 : (int)n_items);
      pv.plan[1] = over ? 0 : (int)n_items;
      pv.plan[2] = 0;
      pv.plan[3] = n_pseq;
    }
    return;
  }

  // query rotation: q' = (I_n (x) H_b) D q * qscale as f16.  A thread holds
  // E = min(b, 16) consecutive elements of one row (16-byte loads and
  // stores): D is applied as sign-bit XOR masks on the bf16 pairs, the
  // Hadamard stages below E run in registers (packed f32x2), the stages from
  // E to b across the b / E threads of the block (adjacent lanes).
  constexpr int B = Head<D>::b;
  constexpr int E = kPrepPiece(D);
  constexpr int TPB = B / E;  // threads per Hadamard block: 1 .. 16
  constexpr int PPR = D / E;  // pieces per row
  __shared__ __align__(16) uint32_t smask[D / 2];
  if constexpr (ROT) {
    for (int i = threadIdx.x; i < D / 2; i += kPrepThreads)
      smask[i] = (c.signs[2 * i] < 0 ? 0x8000u : 0u) | (c.signs[2 * i + 1] < 0 ? 0x80000000u : 0u);
    __syncthreads();
  }
  const long long piece = (long long)(blockIdx.x - 1) * kPrepThreads + threadIdx.x;
  // the pieces of one Hadamard block are adjacent lanes and all valid or all
  // not (PPR is a multiple of TPB): every lane stays for the shuffles
  const bool live = piece < (long long)c.num_q_tokens * c.hq * PPR;
  const long long row = live ? piece / PPR : 0;
  const int e0 = (int)(piece - (piece / PPR) * PPR) * E;
  const long long t = row / c.hq;
  const int h = (int)(row - t * c.hq);
  const uint16_t* src = c.q + t * c.q_stride + (long long)h * D + e0;
  float x[E];
#pragma unroll
  for (int v = 0; v < E / 8; v++) {
    uint4 w = live ? reinterpret_cast<const uint4*>(src)[v] : make_uint4(0, 0, 0, 0);
    if constexpr (ROT) {
      const uint4 m = *reinterpret_cast<const uint4*>(smask + (e0 >> 1) + 4 * v);
      w.x ^= m.x; w.y ^= m.y; w.z ^= m.z; w.w ^= m.w;
    }
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      x[8 * v + 2 * k] = bf16lo_to_f32(ww[k]);
      x[8 * v + 2 * k + 1] = bf16hi_to_f32(ww[k]);
    }
  }
  if constexpr (ROT) {
    // stage 1: pairs (i, i + 1); packed as (x_i, x_{i+2}) +- (x_{i+1}, x_{i+3})
#pragma unroll
    for (int i = 0; i < E; i += 4) {
      const float2 a = make_float2(x[i], x[i + 2]), b = make_float2(x[i + 1], x[i + 3]);
      const float2 u = f2add(a, b), w = f2sub(a, b);
      x[i] = u.x; x[i + 2] = u.y; x[i + 1] = w.x; x[i + 3] = w.y;
    }
    // stages 2 .. E/2: pairs (i, i + hh) and (i + 1, i + 1 + hh) together
#pragma unroll
    for (int hh = 2; hh < E; hh <<= 1) {
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        if ((i & hh) == 0) {
          const float2 a = make_float2(x[i], x[i + 1]), b = make_float2(x[i + hh], x[i + hh + 1]);
          const float2 u = f2add(a, b), w = f2sub(a, b);
          x[i] = u.x; x[i + 1] = u.y; x[i + hh] = w.x; x[i + hh + 1] = w.y;
        }
      }
    }
    // stages E .. b/2: the partner piece is lane ^ m (upper element = partner - self)
#pragma unroll
    for (int m = 1; m < TPB; m <<= 1) {
      const float f = (threadIdx.x & m) ? -1.f : 1.f;
#pragma unroll
      for (int k = 0; k < E; k++) x[k] = fmaf(f, x[k], __shfl_xor_sync(0xffffffffu, x[k], m));
    }
  }
  if (live) {
    __half* dst = pv.qrot + row * D + e0;
    const float2 qs = make_float2(c.qscale, c.qscale);
#pragma unroll
    for (int v = 0; v < E / 8; v++) {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const float2 y = __fmul2_rn(make_float2(x[8 * v + 2 * k], x[8 * v + 2 * k + 1]), qs);
        o[k] = pack_f16x2(y.x, y.y);
      }
      reinterpret_cast<uint4*>(dst)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// 3. decode: stream-K over (segment, position) units, one CTA per head group
// ---------------------------------------------------------------------------
// A position is NP consecutive 16-key blocks of one segment.  With NP > 1 the
// blocks share one score accumulator: block j owns query columns
// [j * COLS, (j + 1) * COLS) (COLS = 8 / NP >= the sequence's q_len * G), so
// one softmax pass, one barrier and one V offset correction serve NP blocks.
// Each column keeps its own running (m, l, o'); the reduce kernel merges the
// NP columns of a query with the log-sum-exp rule like any other split.
template <int D, int NP, int FMT>
struct DecGeom {
  static constexpr int COLS = kDecodeCols / NP;  // query columns per block
  // ring of single-block slots: NP consumed per iteration, the rest in flight
  static constexpr int NS = NP == 1 ? 4 : 2 * NP + 1;
  static constexpr int WAIT = NS - 2 * NP;  // copy groups that may stay pending at a wait
  static constexpr int CB = FMT == kFmtInt8 ? D : D / 2;  // code bytes per head vector
  static constexpr int KROW = CB;           // K tile row stride (bytes)
  // V tile row stride: an odd multiple of 16 bytes, so that the 8 rows of
  // an ldmatrix piece fall in distinct bank groups
  static constexpr int VROW = (CB / 16) % 2 ? CB : CB + 16;
  static constexpr int KTILE = 16 * KROW;
  static constexpr int VTILE = 16 * VROW;
  // one head's K and V codes of one block, padded to 64 mod 128 bytes so that
  // the copies of neighbouring heads' rows fall in different bank halves
  static constexpr int HTILE = ((KTILE + VTILE + 63) / 128) * 128 + 64;
  static constexpr int KW = CB / 16;    // K words per row per thread (quarter row)
  static constexpr int KSTEPS = D / 16; // MMA k-steps of a block's K (and m-tiles of its V)
  static constexpr int CHR = CB / 16;   // 16-byte chunks per code row
  // per slot: hg head tiles, then scales [K/V][hg][16]
  __host__ __device__ static constexpr int slot_bytes(int hg) { return hg * (HTILE + 128); }
  __host__ __device__ static constexpr int smem_bytes(int hg) { return NS * slot_bytes(hg) + 32; }
  static_assert(HTILE % 16 == 0, "tile alignment");
  static_assert(WAIT >= 0 && NS <= 8, "slot ring");
};

// Walk over the decode units (sequence i, head group grp, position kp).
struct DecWalk {
  int i;      // index into the decode-sequence list
  int grp;    // head group
  int kp;     // position within the sequence
  int npos;   // positions of the sequence
  int nblk;   // 16-key blocks of the sequence
  int fb;     // first block read (the sliding window's)
  int seq;    // sequence id
};

template <int NP>
__device__ __forceinline__ void walk_load(DecWalk& w, const Common& c, const PlanView& pv) {
  w.seq = pv.dseq[w.i];
  const int L = c.seq_lens[w.seq];
  w.nblk = (L + 15) / 16;
  w.fb = first_block(c, L, c.qsl[w.seq + 1] - c.qsl[w.seq]);
  w.npos = (w.nblk - w.fb + NP - 1) / NP;
}
template <int NP>
__device__ __forceinline__ void walk_next(DecWalk& w, const Common& c, const PlanView& pv) {
  if (++w.kp == w.npos) {
    w.kp = 0;
    if (++w.grp == c.ng) {
      w.grp = 0;
      ++w.i;
      walk_load<NP>(w, c, pv);
    }
  }
}

template <int N, int BYTES>
__device__ __forceinline__ void lds_words(uint32_t (&w)[N], const uint8_t* p) {
  static_assert(N * 4 == BYTES, "word count");
  if constexpr (BYTES % 16 == 0) {
#pragma unroll
    for (int k = 0; k < N / 4; k++) {
      uint4 v = reinterpret_cast<const uint4*>(p)[k];
      w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
    }
  } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
    for (int k = 0; k < N / 2; k++) {
      uint2 v = reinterpret_cast<const uint2*>(p)[k];
      w[2 * k] = v.x; w[2 * k + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < N; k++) w[k] = reinterpret_cast<const uint32_t*>(p)[k];
  }
}

// O'^T += V^T P'^T.  ldmatrix.trans of an 8-key x 16-byte piece of the V
// tile gives each lane one word holding bytes (2g, 2g+1) of keys 2cq and
// 2cq+1.
// INT4: one lop3 yields an A-fragment register (two keys, one head
// dimension) and a shift by 8 exposes the second byte.  Chunk ch (bytes
// [16 ch, 16 ch + 16) of each V row) feeds m-tiles 2 ch and 2 ch + 1, whose
// rows g and g + 8 are head dimensions 32 ch + 4g + 2e and 32 ch + 4g + 2e + 1
// (e = 0, 1; the odd ones carry the factor 16 of the high nibble).
// int8: the word, made offset-binary by an xor, gives its two head
// dimensions' registers by one byte permute each (0x64nn is 1024 + nn):
// chunk ch feeds m-tile ch, rows g and g + 8 being dimensions 16 ch + 2g and
// 16 ch + 2g + 1.  With CORR the block's offset correction follows every
// m-tile's MMA.
template <int D, bool CORR, int FMT>
__device__ __forceinline__ void pv_mma_chunk(float (&oacc)[D / 16][4], int ch, uint32_t r_lo, uint32_t r_hi,
                                             uint32_t b0, uint32_t b1, const uint32_t (&vcorr)[4]) {
  if constexpr (FMT == kFmtInt4) {
    const uint32_t s_lo = r_lo >> 8, s_hi = r_hi >> 8;
    const uint32_t a0[4] = {nib_lo(r_lo), nib_hi(r_lo), nib_lo(r_hi), nib_hi(r_hi)};
    mma_16816(oacc[2 * ch], a0, b0, b1);
    if constexpr (CORR) mma_16816(oacc[2 * ch], vcorr, b0, b1);
    const uint32_t a1[4] = {nib_lo(s_lo), nib_hi(s_lo), nib_lo(s_hi), nib_hi(s_hi)};
    mma_16816(oacc[2 * ch + 1], a1, b0, b1);
    if constexpr (CORR) mma_16816(oacc[2 * ch + 1], vcorr, b0, b1);
  } else {
    const uint32_t lo = r_lo ^ 0x80808080u, hi = r_hi ^ 0x80808080u;
    const uint32_t a[4] = {__byte_perm(lo, kBytes64, 0x4240), __byte_perm(lo, kBytes64, 0x4341),
                           __byte_perm(hi, kBytes64, 0x4240), __byte_perm(hi, kBytes64, 0x4341)};
    mma_16816(oacc[ch], a, b0, b1);
    if constexpr (CORR) mma_16816(oacc[ch], vcorr, b0, b1);
  }
}

// vaddr: shared address of this lane's ldmatrix row in chunk pair 0 (lane l
// addresses key 8 ((l >> 3) & 1) + (l & 7) of chunk (l >> 4))
template <int D, bool CORR, int FMT>
__device__ __forceinline__ void pv_mmas(float (&oacc)[D / 16][4], uint32_t vaddr, uint32_t b0, uint32_t b1,
                                        const uint32_t (&vcorr)[4]) {
  constexpr int CH = (FMT == kFmtInt8 ? D : D / 2) / 16;  // 16-byte chunks per V row
#pragma unroll
  for (int p = 0; p < CH / 2; p++) {
    uint32_t r[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(vaddr + p * 32));
    pv_mma_chunk<D, CORR, FMT>(oacc, 2 * p, r[0], r[1], b0, b1, vcorr);
    pv_mma_chunk<D, CORR, FMT>(oacc, 2 * p + 1, r[2], r[3], b0, b1, vcorr);
  }
  if constexpr (CH % 2) {
    uint32_t r[2];
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(vaddr + (CH / 2) * 32));
    pv_mma_chunk<D, CORR, FMT>(oacc, CH - 1, r[0], r[1], b0, b1, vcorr);
  }
}

struct DecParams {
  Common c;
  PlanView pv;
  int num_ctas;
};

// Work decomposition: stream-K over the flattened (decode sequence, head
// group, position) units; CTA r takes units [T*r/R, T*(r+1)/R).  A CTA has
// one warp per kv head of the group; for every block all its threads copy
// the block's codes and scales of the group's heads -- contiguous runs of the
// cache -- into per-head padded tiles, and each warp then computes its own
// head.  Every (segment, head) piece of a CTA's range writes (o', m, l) for
// all 8 columns: to the sequence's direct slot if the piece starts the
// segment, else to the CTA's slot.
//
// Score arithmetic.  A K fragment holds 1032 + c at the low-nibble positions
// and 1152 + 16c at the high-nibble ones; the q' fragment carries 16 q' at the
// low positions and q' at the high ones, so the MMA yields
//   acc = 16 (q' . c) + bias,  bias = sum_low 16 q' * 1032 + sum_high q' * 1152,
// and bias is itself one MMA of a constant A fragment against q' per segment.
// The V side works the same way: even head dimensions accumulate
// p'(1032 + c), odd ones p'(1152 + 16c); right after each position's MMAs a
// further MMA of a constant (-1032 / -1152) A fragment against the same P'^T
// removes that position's offset, so the running accumulator only ever holds
// one block's worth of offset per column (accumulating the offset over
// thousands of keys would cost the fp32 accumulator the signal's low bits).
template <int D, int NP, int FMT>
__global__ void __launch_bounds__(256) decode_kernel(DecParams prm) {
  using G = DecGeom<D, NP, FMT>;
  constexpr bool I8 = FMT == kFmtInt8;
  const Common& c = prm.c;
  const PlanView& pv = prm.pv;
  extern __shared__ __align__(16) uint8_t smem[];
  const int HG = c.hg;
  const int tid = threadIdx.x, nthr = HG * 32;
  const int hl = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int SB = G::slot_bytes(HG);
  int* sflag = reinterpret_cast<int*>(smem + G::NS * SB);

  const int n_dseq = pv.plan[0];
  if (n_dseq == 0) return;
  const long long Tu = pv.dprefix[n_dseq] * c.ng;
  const int R = prm.num_ctas;
  const long long P0 = Tu * blockIdx.x / R, P1 = Tu * (blockIdx.x + 1) / R;
  if (P0 >= P1) return;

  // locate P0: largest i with dprefix[i] * ng <= P0 (32-ary search, per warp)
  int lo = 0, hi = n_dseq;  // invariant: key(lo) <= P0 < key(hi)
  while (hi - lo > 1) {
    const long long span = hi - lo;
    const int probe = lo + (int)((span * lane) / 32);
    const bool le = lane == 0 || pv.dprefix[probe] * c.ng <= P0;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz(m);
    const int nlo = lo + (int)((span * last) / 32);
    const int nhi = last == 31 ? hi : lo + (int)((span * (last + 1)) / 32);
    lo = nlo;
    hi = nhi > nlo ? nhi : nlo + 1;
  }
  DecWalk cw;
  cw.i = lo;
  walk_load<NP>(cw, c, pv);
  {
    const long long off = P0 - pv.dprefix[cw.i] * c.ng;
    cw.grp = (int)(off / cw.npos);
    cw.kp = (int)(off - (long long)cw.grp * cw.npos);
  }
  DecWalk pw = cw;

  // thread-constant parts of the staging addresses: CHR chunks per thread
  // (chunk index ((kv * 16 + r) * HG + h) * CHR + col: consecutive threads read
  // consecutive bytes of the cache)
  uint32_t c_saddr[G::CHR];      // shared address within slot 0
  const uint8_t* c_src[G::CHR];  // cache address within block 0, head group 0
#pragma unroll
  for (int j = 0; j < G::CHR; j++) {
    const int idx = tid + nthr * j;
    const int col = idx % G::CHR;
    const int rest = idx / G::CHR;
    const int h = rest % HG;
    const int kvr = rest / HG;
    const int kv = kvr / 16, r = kvr % 16;
    c_saddr[j] = smem_addr(smem) + h * G::HTILE + (kv ? G::KTILE + r * G::VROW : r * G::KROW) + col * 16;
    c_src[j] = (kv ? c.v_cache : c.k_cache) + r * c.geo.crow + (long long)h * c.geo.chead + col * 16;
  }
  // one 4-byte scale per thread: [K/V][row][h]
  const int s_kv = tid / (16 * HG), s_rem = tid % (16 * HG);
  const int s_r = s_rem / HG, s_h = s_rem % HG;
  const uint32_t s_saddr = smem_addr(smem) + HG * G::HTILE + (s_kv * HG + s_h) * 64 + s_r * 4;
  const float* s_src = (s_kv ? c.v_scale : c.k_scale) + s_r * c.geo.srow + (long long)s_h * c.geo.shead;
  const uint64_t blk_bytes = (uint64_t)c.geo.cblk, blk_scales = (uint64_t)c.geo.sblk;

  // block j of a position, or kAbsent past the end of the sequence (NP > 1)
  constexpr int kAbsent = -0x7fffffff - 1;
  auto block_at = [&](const DecWalk& w, int j) {
    const int kb = w.fb + w.kp * NP + j;
    return kb < w.nblk ? c.block_table[(long long)w.seq * c.max_blocks + kb] : kAbsent;
  };
  auto issue = [&](int blk, int grp, int slot) {
    const bool ok = blk >= 0 && blk < c.num_blocks;
    if (ok) {
      const uint32_t soff = (uint32_t)(slot * SB);
      const uint64_t goff = (uint64_t)(grp * HG) * c.geo.chead;
#pragma unroll
      for (int j = 0; j < G::CHR; j++) {
        const uint8_t* src = c_src[j] + (uint64_t)(uint32_t)blk * blk_bytes + goff;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(c_saddr[j] + soff), "l"(src));
      }
      const float* ssrc = s_src + (uint64_t)(uint32_t)blk * blk_scales + (uint64_t)(grp * HG) * c.geo.shead;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s_saddr + soff), "l"(ssrc));
    }
    if (tid == 0) {
      sflag[slot] = ok;
      if (!ok && blk != kAbsent) flag(c.status, KV_INT4_DEV_BAD_BLOCK);
    }
  };

  // producer: one block per call into the next ring slot, the next block id
  // loaded one call ahead; one commit group per call (empty past the range)
  long long ppos = P0;
  int pj = 0, ps = 0;
  int pblk = block_at(pw, 0);
  auto produce = [&]() {
    if (ppos < P1) {
      issue(pblk, pw.grp, ps);
      ps = ps + 1 == G::NS ? 0 : ps + 1;
      if (++pj == NP) {
        pj = 0;
        if (++ppos < P1) walk_next<NP>(pw, c, pv);
      }
      if (ppos < P1) pblk = block_at(pw, pj);
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int s = 0; s < G::NS - NP; s++) produce();

  // per-segment state of this warp's head
  uint32_t qb[G::KSTEPS][2];
  float oacc[G::KSTEPS][4];
  float m0, m1, l0, l1, bias0, bias1;
  int lim0, lim1;  // keys visible to columns 2cq, 2cq+1: positions [lo, lim)
  int lo0, lo1;
  int lim_warp;    // smallest of all columns' limits
  int lo_warp;     // largest of all columns' first visible positions
  bool first_piece = cw.kp == 0;

  auto begin_segment = [&]() {
    const int seq = cw.seq;
    const int head = cw.grp * HG + hl;
    const int q0 = c.qsl[seq];
    const int ql = c.qsl[seq + 1] - q0;
    const int L = c.seq_lens[seq];
    const int ctx = L - ql;
    // B fragments of this lane's column g, which holds query column g % COLS
    const int n = g & (G::COLS - 1);
    const bool colok = n < ql * c.group;
    const int j = n / c.group, jj = n - j * c.group;
    const __half* qrow = pv.qrot + ((long long)(q0 + (colok ? j : 0)) * c.hq + head * c.group + (colok ? jj : 0)) * D;
    if constexpr (!I8) {
      const __half2 x16 = __float2half2_rn(16.f);
#pragma unroll
      for (int w = 0; w < G::KW; w++) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (colok) v = *reinterpret_cast<const uint4*>(qrow + 8 * (cq * G::KW + w));
        uint32_t lo0 = __byte_perm(v.x, v.z, 0x5410), lo1 = __byte_perm(v.y, v.w, 0x5410);
        __half2 h0 = __hmul2(*reinterpret_cast<__half2*>(&lo0), x16);
        __half2 h1 = __hmul2(*reinterpret_cast<__half2*>(&lo1), x16);
        qb[2 * w][0] = *reinterpret_cast<uint32_t*>(&h0);
        qb[2 * w][1] = __byte_perm(v.x, v.z, 0x7632);
        qb[2 * w + 1][0] = *reinterpret_cast<uint32_t*>(&h1);
        qb[2 * w + 1][1] = __byte_perm(v.y, v.w, 0x7632);
      }
    } else {
      // k-step s of this lane's quarter: dimensions cq D/4 + 4s + {0, 1} and + {2, 3}
#pragma unroll
      for (int w = 0; w < G::KW; w++) {
        uint2 v = make_uint2(0, 0);
        if (colok) v = *reinterpret_cast<const uint2*>(qrow + cq * (D / 4) + 4 * w);
        qb[w][0] = v.x;
        qb[w][1] = v.y;
      }
    }
    float bacc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t abias[4] = {I8 ? kF16x2_1152 : kF16x2_1032, I8 ? kF16x2_1152 : kF16x2_1032, kF16x2_1152,
                               kF16x2_1152};
#pragma unroll
    for (int s = 0; s < G::KSTEPS; s++) mma_16816(bacc, abias, qb[s][0], qb[s][1]);
    bias0 = bacc[0];
    bias1 = bacc[1];
    const int col0 = (2 * cq) & (G::COLS - 1), col1 = (2 * cq + 1) & (G::COLS - 1);
    const int j0 = min(col0 / c.group, max(ql - 1, 0)), j1 = min(col1 / c.group, max(ql - 1, 0));
    lim0 = c.causal ? min(L, ctx + j0 + 1) : L;
    lim1 = c.causal ? min(L, ctx + j1 + 1) : L;
    lo0 = window_lo(c, ctx + j0);
    lo1 = window_lo(c, ctx + j1);
    lim_warp = min(lim0, lim1);
    lo_warp = max(lo0, lo1);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      lim_warp = min(lim_warp, __shfl_xor_sync(0xffffffffu, lim_warp, o));
      lo_warp = max(lo_warp, __shfl_xor_sync(0xffffffffu, lo_warp, o));
    }
#pragma unroll
    for (int i = 0; i < G::KSTEPS; i++) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  };

  auto flush = [&]() {
    float a0 = l0, a1 = l1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      a0 += __shfl_xor_sync(0xffffffffu, a0, o);
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    }
    float* dst_o;
    float* dst_ml;
    if (first_piece) {
      const long long slot = (long long)cw.i * c.hkv + cw.grp * HG + hl;
      dst_o = pv.direct_o + slot * kDecodeCols * D;
      dst_ml = pv.direct_ml + slot * kDecodeCols * 2;
    } else {
      const long long slot = (long long)blockIdx.x * HG + hl;
      dst_o = pv.warp_o + slot * kDecodeCols * D;
      dst_ml = pv.warp_ml + slot * kDecodeCols * 2;
    }
    if constexpr (!I8) {
      // m-tiles 2ch, 2ch+1 hold d = 32 ch + 4g + {0, 1, 2, 3} (odd d scaled by 16)
      float* o0 = dst_o + (2 * cq) * D + 4 * g;
      float* o1 = dst_o + (2 * cq + 1) * D + 4 * g;
#pragma unroll
      for (int i = 0; i < G::KSTEPS; i += 2) {
        *reinterpret_cast<float4*>(o0 + 16 * i) =
            make_float4(oacc[i][0], oacc[i][2] * 0.0625f, oacc[i + 1][0], oacc[i + 1][2] * 0.0625f);
        *reinterpret_cast<float4*>(o1 + 16 * i) =
            make_float4(oacc[i][1], oacc[i][3] * 0.0625f, oacc[i + 1][1], oacc[i + 1][3] * 0.0625f);
      }
    } else {
      // m-tile t holds d = 16 t + 2g (row g) and 16 t + 2g + 1 (row g + 8)
      float* o0 = dst_o + (2 * cq) * D + 2 * g;
      float* o1 = dst_o + (2 * cq + 1) * D + 2 * g;
#pragma unroll
      for (int i = 0; i < G::KSTEPS; i++) {
        *reinterpret_cast<float2*>(o0 + 16 * i) = make_float2(oacc[i][0], oacc[i][2]);
        *reinterpret_cast<float2*>(o1 + 16 * i) = make_float2(oacc[i][1], oacc[i][3]);
      }
    }
    if (g == 0) {
      dst_ml[(2 * cq) * 2 + 0] = m0;
      dst_ml[(2 * cq) * 2 + 1] = a0;
      dst_ml[(2 * cq + 1) * 2 + 0] = m1;
      dst_ml[(2 * cq + 1) * 2 + 1] = a1;
    }
  };

  begin_segment();
  const int jb = (cq * NP) >> 2;  // block of this thread's score columns 2cq, 2cq+1
  const int jv = (g * NP) >> 3;   // block of this lane's P'^T column g
  // this lane's ldmatrix row of the V tile in slot 0
  const uint32_t v_lane = smem_addr(smem) + hl * G::HTILE + G::KTILE +
                          (((lane >> 3) & 1) * 8 + (lane & 7)) * G::VROW + (lane >> 4) * 16;
  int cs = 0;                     // slot of the iteration's first block
  const int nunits = (int)(P1 - P0);
  // INT4: rows g (even d: offset 1032) and g + 8 (odd d: offset 1152); int8: 1152
  const uint32_t vcorr[4] = {I8 ? kF16x2_M1152 : kF16x2_M1032, kF16x2_M1152, I8 ? kF16x2_M1152 : kF16x2_M1032,
                             kF16x2_M1152};
#pragma unroll 1
  for (int it = 0; it < nunits; it++) {
    cp_async_wait<G::WAIT>();
    __syncthreads();  // this position's copies visible; every warp done with the previous slots
#pragma unroll
    for (int j = 0; j < NP; j++) produce();

    int slot[NP];
    slot[0] = cs;
#pragma unroll
    for (int j = 1; j < NP; j++) slot[j] = slot[j - 1] + 1 == G::NS ? 0 : slot[j - 1] + 1;
    bool allok = true;
    int my = slot[0];
#pragma unroll
    for (int j = 0; j < NP; j++) {
      allok = allok && sflag[slot[j]] != 0;
      if (j > 0 && jb == j) my = slot[j];
    }
    const uint8_t* mstg = smem + my * SB;
    const bool bok = sflag[my] != 0;
    const float* sks = reinterpret_cast<const float*>(mstg + HG * G::HTILE + hl * 64);
    const float* svs = reinterpret_cast<const float*>(mstg + HG * G::HTILE + (HG + hl) * 64);

    // ---- S^T = K Q'^T (biased, x16), one accumulator per block ----
    float sacc[NP][4];
#pragma unroll
    for (int j = 0; j < NP; j++) {
      sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
      const uint8_t* st = smem + slot[j] * SB + hl * G::HTILE;
      uint32_t xk[G::KW], yk[G::KW];
      lds_words<G::KW, G::CB / 4>(xk, st + g * G::KROW + cq * (G::CB / 4));
      lds_words<G::KW, G::CB / 4>(yk, st + (g + 8) * G::KROW + cq * (G::CB / 4));
#pragma unroll
      for (int w = 0; w < G::KW; w++) {
        if constexpr (!I8) {
          const uint32_t x = xk[w], y = yk[w], x8 = x >> 8, y8 = y >> 8;
          const uint32_t a0[4] = {nib_lo(x), nib_lo(y), nib_hi(x), nib_hi(y)};
          mma_16816(sacc[j], a0, qb[2 * w][0], qb[2 * w][1]);
          const uint32_t a1[4] = {nib_lo(x8), nib_lo(y8), nib_hi(x8), nib_hi(y8)};
          mma_16816(sacc[j], a1, qb[2 * w + 1][0], qb[2 * w + 1][1]);
        } else {
          // four int8 codes of key g (x) and key g + 8 (y): 1152 + c per f16
          const uint32_t x = xk[w] ^ 0x80808080u, y = yk[w] ^ 0x80808080u;
          const uint32_t a[4] = {__byte_perm(x, kBytes64, 0x4140), __byte_perm(y, kBytes64, 0x4140),
                                 __byte_perm(x, kBytes64, 0x4342), __byte_perm(y, kBytes64, 0x4342)};
          mma_16816(sacc[j], a, qb[w][0], qb[w][1]);
        }
      }
    }
    float sa[4] = {sacc[0][0], sacc[0][1], sacc[0][2], sacc[0][3]};
#pragma unroll
    for (int j = 1; j < NP; j++)
#pragma unroll
      for (int e = 0; e < 4; e++) sa[e] = jb == j ? sacc[j][e] : sa[e];

    const int kb0 = cw.fb + cw.kp * NP;
    const int pos0 = (kb0 + jb) * 16 + g, pos1 = pos0 + 8;
    // INT4 scores carry the factor 16 of q' at the low-nibble positions
    const float ks0 = sks[g] * (I8 ? 1.f : 0.0625f), ks1 = sks[g + 8] * (I8 ? 1.f : 0.0625f);
    float s00 = (sa[0] - bias0) * ks0, s01 = (sa[1] - bias1) * ks0;
    float s10 = (sa[2] - bias0) * ks1, s11 = (sa[3] - bias1) * ks1;
    // keys outside a column's visible range [lo, lim) (or in an invalid or
    // absent block) only occur in positions that reach past the warp's
    // smallest limit or start before its largest window start
    const bool full = allok && (kb0 + NP) * 16 <= lim_warp && kb0 * 16 >= lo_warp;
    if (!full) {
      s00 = (bok && pos0 < lim0 && pos0 >= lo0) ? s00 : -INFINITY;
      s01 = (bok && pos0 < lim1 && pos0 >= lo1) ? s01 : -INFINITY;
      s10 = (bok && pos1 < lim0 && pos1 >= lo0) ? s10 : -INFINITY;
      s11 = (bok && pos1 < lim1 && pos1 >= lo1) ? s11 : -INFINITY;
    }
    float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
    // exact running max: reduce across the key lanes only when some lane
    // holds a score above its column's current max
    if (__any_sync(0xffffffffu, mx0 > m0 || mx1 > m1)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // a column with no visible key yet keeps m = -inf (and alpha = 1)
      const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int i = 0; i < G::KSTEPS; i++) {
        oacc[i][0] *= al0;
        oacc[i][1] *= al1;
        oacc[i][2] *= al0;
        oacc[i][3] *= al1;
      }
    }
    const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
    const float p00 = fast_exp2(s00 - mu0), p01 = fast_exp2(s01 - mu1);
    const float p10 = fast_exp2(s10 - mu0), p11 = fast_exp2(s11 - mu1);
    l0 += p00 + p10;
    l1 += p01 + p11;
    const float vs0 = svs[g], vs1 = svs[g + 8];
    float q00 = p00 * vs0, q01 = p01 * vs0, q10 = p10 * vs1, q11 = p11 * vs1;
    if (!full) {  // masked keys may carry unwritten (NaN) scales: select, do not multiply
      q00 = s00 == -INFINITY ? 0.f : q00;
      q01 = s01 == -INFINITY ? 0.f : q01;
      q10 = s10 == -INFINITY ? 0.f : q10;
      q11 = s11 == -INFINITY ? 0.f : q11;
    }
    const uint32_t M0 = pack_f16x2(q00, q01);
    const uint32_t M1 = pack_f16x2(q10, q11);
    const uint32_t b0 = movmatrix_trans(M0), b1 = movmatrix_trans(M1);

    // ---- O'^T += V^T P'^T (offset removed per position) ----
    if constexpr (NP == 1) {
      pv_mmas<D, true, FMT>(oacc, v_lane + slot[0] * SB, b0, b1, vcorr);
    } else {
#pragma unroll
      for (int j = 0; j < NP; j++) {
        // block j's probabilities only: the other blocks' columns are zero
        const uint32_t bj0 = jv == j ? b0 : 0u, bj1 = jv == j ? b1 : 0u;
        pv_mmas<D, false, FMT>(oacc, v_lane + slot[j] * SB, bj0, bj1, vcorr);
      }
#pragma unroll
      for (int i = 0; i < G::KSTEPS; i++) mma_16816(oacc[i], vcorr, b0, b1);
    }

    const bool last_in_seg = cw.kp == cw.npos - 1;
    const bool last_in_range = it + 1 == nunits;
    if (last_in_seg || last_in_range) flush();
    if (!last_in_range) {
      walk_next<NP>(cw, c, pv);
      if (last_in_seg) {
        first_piece = true;
        begin_segment();
      }
    }
    cs += NP;
    if (cs >= G::NS) cs -= G::NS;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// 4. reduce: merge decode pieces, normalise, inverse-rotate, write bf16
// ---------------------------------------------------------------------------
struct RedParams {
  Common c;
  PlanView pv;
  int num_ctas;
  int cps;  // warps (query columns) per segment: min(dcols, max_query_len * group)
};

template <int D, bool ROT>
__global__ void __launch_bounds__(kDecodeCols * 32) reduce_kernel(RedParams prm) {
  const Common& c = prm.c;
  const PlanView& pv = prm.pv;
  constexpr int B = Head<D>::b;
  __shared__ float srow[kDecodeCols][D];
  // a warp per (segment, query column): the CTA's dcols warps cover
  // dcols / cps segments of cps columns each
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * (c.dcols / prm.cps) + warp / prm.cps;
  const int col = warp % prm.cps;
  const int n_dseq = pv.plan[0];
  if (seg >= n_dseq * c.hkv) return;
  const int i = seg / c.hkv, h = seg - i * c.hkv;
  const int seq = pv.dseq[i];
  const int q0 = c.qsl[seq], ql = c.qsl[seq + 1] - q0;
  if (col >= ql * c.group) return;  // ql * group <= cps
  const int nblk = (c.seq_lens[seq] + 15) / 16;
  const int npos = (nblk - first_block(c, c.seq_lens[seq], ql) + c.np - 1) / c.np;
  const int grp = h / c.hg, hl = h - grp * c.hg;
  const long long Tu = pv.dprefix[n_dseq] * c.ng;
  const long long sbeg = pv.dprefix[i] * c.ng + (long long)grp * npos, send = sbeg + npos;
  const int W = prm.num_ctas;
  auto wstart = [&](long long w) { return Tu * w / W; };

  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; k++) acc[k] = 0.f;
  float M = -INFINITY, Lsum = 0.f;
  // a piece's columns col, col + dcols, ... hold the same query over
  // disjoint key blocks
  auto merge_slot = [&](const float* o_base, const float* ml_base) {
    for (int sub = 0; sub < c.np; sub++) {
      const int cc = col + sub * c.dcols;
      const float* ow = o_base + cc * D;
      const float mw = ml_base[cc * 2], lw = ml_base[cc * 2 + 1];
      const float Mn = fmaxf(M, mw);
      const float Mu = Mn == -INFINITY ? 0.f : Mn;
      const float a = fast_exp2(M - Mu), b = fast_exp2(mw - Mu);
#pragma unroll
      for (int k = 0; k < PER; k++) acc[k] = acc[k] * a + ow[lane + 32 * k] * b;
      Lsum = Lsum * a + lw * b;
      M = Mn;
    }
  };
  merge_slot(pv.direct_o + (long long)seg * kDecodeCols * D, pv.direct_ml + (long long)seg * kDecodeCols * 2);
  // the other pieces: CTAs whose non-empty range starts strictly inside the
  // segment.  Walk the CTAs or the positions, whichever are fewer.
  auto merge_cta = [&](long long w) {
    const long long slot = w * c.hg + hl;
    merge_slot(pv.warp_o + slot * kDecodeCols * D, pv.warp_ml + slot * kDecodeCols * 2);
  };
  const long long w_first = ((sbeg + 1) * W + Tu - 1) / Tu;  // first CTA starting after sbeg
  const long long w_end = (send * W + Tu - 1) / Tu;          // first CTA starting at or after send
  if (w_end - w_first <= send - sbeg - 1) {
    for (long long w = w_first; w < w_end; w++)
      if (wstart(w + 1) > wstart(w)) merge_cta(w);
  } else {
    for (long long p = sbeg + 1; p < send; p++) {
      const long long w = ((p + 1) * W + Tu - 1) / Tu - 1;  // last CTA starting at or before p
      if (wstart(w) == p) merge_cta(w);
    }
  }
  float* r = srow[warp];
  const float inv = 1.f / (Lsum * (ROT ? (float)B : 1.f));
#pragma unroll
  for (int k = 0; k < PER; k++) r[lane + 32 * k] = acc[k] * inv;
  __syncwarp();
  if constexpr (ROT) {
#pragma unroll 1
    for (int hh = 1; hh < B; hh <<= 1) {
      for (int p = lane; p < D / 2; p += 32) {
        const int ii = (p / hh) * 2 * hh + (p % hh);
        const float a = r[ii], b = r[ii + hh];
        r[ii] = a + b;
        r[ii + hh] = a - b;
      }
      __syncwarp();
    }
  }
  const int j = col / c.group, jj = col - j * c.group;
  uint16_t* dst = c.out + (long long)(q0 + j) * c.out_stride + (long long)(h * c.group + jj) * D;
  for (int p = lane; p < D / 2; p += 32) {
    const float x0 = (ROT && c.signs[2 * p] < 0) ? -r[2 * p] : r[2 * p];
    const float x1 = (ROT && c.signs[2 * p + 1] < 0) ? -r[2 * p + 1] : r[2 * p + 1];
    reinterpret_cast<uint32_t*>(dst)[p] = pack_bf16x2_rn(x0, x1);
  }
}

// ---------------------------------------------------------------------------
// 2. prefill: FA2-style, 64 query rows x 16 keys per step, mma.sync
// ---------------------------------------------------------------------------
template <int D, int FMT>
struct PreGeom {
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int ROWS = kPrefillRows;  // 16 per warp
  static constexpr int STAGES = 3;
  static constexpr int CB = FMT == kFmtInt8 ? D : D / 2;  // code bytes per head vector
  static constexpr int TILE = 16 * CB;
  static constexpr int STAGE = 2 * TILE + 2 * 16 * 4;
  static constexpr int HSTRIDE = D + 8;  // halves per row of the f16 tiles (odd multiple of 16 B)
  static constexpr int SMEM = STAGES * STAGE + ROWS * HSTRIDE * 2 + 2 * 16 * HSTRIDE * 2 + D * 4 + 64;
};

struct PreParams {
  Common c;
  PlanView pv;
};

template <int D, int FMT>
__global__ void __launch_bounds__(PreGeom<D, FMT>::THREADS) prefill_kernel(PreParams prm) {
  using G = PreGeom<D, FMT>;
  constexpr bool ROT = FMT == kFmtInt4;
  constexpr int B = Head<D>::b;
  constexpr int NT = D / 8;  // n-tiles of the output
  const Common& c = prm.c;
  const PlanView& pv = prm.pv;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* stages = smem;
  __half* sQ = reinterpret_cast<__half*>(smem + G::STAGES * G::STAGE);
  __half* sK = sQ + G::ROWS * G::HSTRIDE;
  __half* sV = sK + 16 * G::HSTRIDE;
  float* ssign = reinterpret_cast<float*>(sV + 16 * G::HSTRIDE);
  int* sitem = reinterpret_cast<int*>(ssign + D);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  for (int i = tid; i < D; i += G::THREADS) ssign[i] = (ROT && c.signs[i] < 0) ? -1.f : 1.f;
  const int n_items = pv.plan[1], n_pseq = pv.plan[3];

#pragma unroll 1
  while (true) {
    if (tid == 0) {
      // next item: (prefill sequence, tile in descending order of work, kv head)
      const int itn = atomicAdd(&pv.plan[2], 1);
      int4 it = make_int4(-1, 0, 0, 0);
      if (itn < n_items) {
        int lo = 0, hi = n_pseq;  // ptab[lo].y <= itn < ptab[hi].y
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (pv.ptab[mid].y <= itn) lo = mid;
          else hi = mid;
        }
        const int s = pv.ptab[lo].x, r = itn - pv.ptab[lo].y;
        const int qa = c.qsl[s], qn = c.qsl[s + 1] - qa, Ls = c.seq_lens[s];
        const int ntiles = (qn + c.tile_tokens - 1) / c.tile_tokens;
        const int t = ntiles - 1 - r / c.hkv;
        const int keys = c.causal ? Ls - qn + min(qn, (t + 1) * c.tile_tokens) : Ls;
        it = make_int4(s, r % c.hkv, t, (keys + 15) / 16);
      }
      sitem[0] = it.x; sitem[1] = it.y; sitem[2] = it.z; sitem[3] = it.w;
    }
    __syncthreads();
    const int4 item = make_int4(sitem[0], sitem[1], sitem[2], sitem[3]);
    __syncthreads();
    if (item.x < 0) break;
    const int seq = item.x, h = item.y, tile = item.z, nkb = item.w;
    const int q0 = c.qsl[seq], ql = c.qsl[seq + 1] - q0;
    const int L = c.seq_lens[seq], ctx = L - ql;
    const int tok0 = tile * c.tile_tokens;
    const int ntok = min(c.tile_tokens, ql - tok0);
    const int nrows = ntok * c.group;

    // Q tile -> shared (rows beyond the tile are zero)
    for (int idx = tid; idx < G::ROWS * (D / 8); idx += G::THREADS) {
      const int r = idx / (D / 8), ch = idx - r * (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < nrows) {
        const int j = r / c.group, jj = r - j * c.group;
        v = *reinterpret_cast<const uint4*>(pv.qrot + ((long long)(q0 + tok0 + j) * c.hq + h * c.group + jj) * D + ch * 8);
      }
      *reinterpret_cast<uint4*>(sQ + r * G::HSTRIDE + ch * 8) = v;
    }

    auto issue = [&](int kb, int stage) {
      uint8_t* st = stages + stage * G::STAGE;
      const int blk = c.block_table[(long long)seq * c.max_blocks + kb];
      if (blk < 0 || blk >= c.num_blocks) return;  // reported and masked by the consumer
      const long long cb0 = (long long)blk * c.geo.cblk, sb0 = (long long)blk * c.geo.sblk;
      for (int q = tid; q < G::CB; q += G::THREADS) {  // 16 rows x CB/16 chunks
        const int r = q / (G::CB / 16), col = q - r * (G::CB / 16);
        const long long goff = cb0 + r * c.geo.crow + (long long)h * c.geo.chead + col * 16;
        cp_async16(st + r * G::CB + col * 16, c.k_cache + goff);
        cp_async16(st + G::TILE + r * G::CB + col * 16, c.v_cache + goff);
      }
      if (tid < 32) {
        const int r = tid & 15;
        const long long soff = sb0 + r * c.geo.srow + (long long)h * c.geo.shead;
        if (tid < 16) cp_async4(st + 2 * G::TILE + r * 4, c.k_scale + soff);
        else cp_async4(st + 2 * G::TILE + 64 + r * 4, c.v_scale + soff);
      }
    };

    // blocks wholly before the window of the tile's earliest query are skipped
    const int kb0 = window_lo(c, ctx + tok0) >> 4;
    for (int s = 0; s < G::STAGES - 1; s++) {
      if (kb0 + s < nkb) issue(kb0 + s, s);
      cp_async_commit();
    }

    float oacc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; t++) oacc[t][0] = oacc[t][1] = oacc[t][2] = oacc[t][3] = 0.f;
    float mr0 = -INFINITY, mr1 = -INFINITY, lr0 = 0.f, lr1 = 0.f;
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    const int qp0 = ctx + tok0 + (r0 < nrows ? r0 / c.group : 0);
    const int qp1 = ctx + tok0 + (r1 < nrows ? r1 / c.group : 0);
    const int lim0 = c.causal ? min(L, qp0 + 1) : L;
    const int lim1 = c.causal ? min(L, qp1 + 1) : L;
    const int lo0 = window_lo(c, qp0), lo1 = window_lo(c, qp1);

#pragma unroll 1
    for (int kb = kb0; kb < nkb; kb++) {
      const int stage = (kb - kb0) % G::STAGES;
      if (kb + G::STAGES - 1 < nkb) issue(kb + G::STAGES - 1, (kb - kb0 + G::STAGES - 1) % G::STAGES);
      cp_async_commit();
      cp_async_wait<G::STAGES - 1>();
      __syncthreads();
      const int blk = c.block_table[(long long)seq * c.max_blocks + kb];
      const bool bok = blk >= 0 && blk < c.num_blocks;
      if (!bok && tid == 0) flag(c.status, KV_INT4_DEV_BAD_BLOCK);
      const uint8_t* st = stages + stage * G::STAGE;
      // dequantise K and V codes of this block into f16 rows (natural order)
      constexpr int WPR = G::CB / 4;  // code words per row
      for (int q = tid; q < 2 * 16 * WPR; q += G::THREADS) {
        const int which = q / (16 * WPR);
        const int rem = q - which * 16 * WPR;
        const int r = rem / WPR, w = rem - r * WPR;
        const uint32_t x0 = bok ? reinterpret_cast<const uint32_t*>(st + which * G::TILE + r * G::CB)[w] : 0u;
        __half* dst = (which ? sV : sK) + r * G::HSTRIDE;
        if constexpr (ROT) {
          const uint32_t x = bok ? x0 : 0x88888888u;
          const uint32_t p0 = nib_to_f16x2(x), p1 = nib_to_f16x2(x >> 4), p2 = nib_to_f16x2(x >> 8),
                         p3 = nib_to_f16x2(x >> 12);
          // p_k = (element k, element k+4) -> natural order 0..7
          uint4 o;
          o.x = __byte_perm(p0, p1, 0x5410);
          o.y = __byte_perm(p2, p3, 0x5410);
          o.z = __byte_perm(p0, p1, 0x7632);
          o.w = __byte_perm(p2, p3, 0x7632);
          *reinterpret_cast<uint4*>(dst + w * 8) = o;
        } else {
          // four int8 codes: 0x64uu (u = c + 128) is 1024 + u, minus 1152 is c, exactly
          const uint32_t x = x0 ^ 0x80808080u;
          const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0x6480),
                                             __ushort_as_half((unsigned short)0x6480));  // 1152
          uint32_t h01 = __byte_perm(x, kBytes64, 0x4140), h23 = __byte_perm(x, kBytes64, 0x4342);
          __half2 a = __hsub2(*reinterpret_cast<__half2*>(&h01), off), b = __hsub2(*reinterpret_cast<__half2*>(&h23), off);
          *reinterpret_cast<uint2*>(dst + w * 4) =
              make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
        }
      }
      __syncthreads();
      const float* sks = reinterpret_cast<const float*>(st + 2 * G::TILE);
      const float* svs = sks + 16;

      // S = Q' K^T : 16 rows x 16 keys per warp
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int s = 0; s < D / 16; s++) {
        uint32_t a[4], bk[4];
        {
          const int mi = lane >> 3, rr = lane & 7;
          ldmatrix_x4(a, sQ + (warp * 16 + (mi & 1) * 8 + rr) * G::HSTRIDE + 16 * s + (mi >> 1) * 8);
          ldmatrix_x4(bk, sK + ((mi >> 1) * 8 + rr) * G::HSTRIDE + 16 * s + (mi & 1) * 8);
        }
        mma_16816(sacc[0], a, bk[0], bk[1]);
        mma_16816(sacc[1], a, bk[2], bk[3]);
      }
      // scale, mask, online softmax (rows r0, r1; keys 2cq, 2cq+1, 8+2cq, 9+2cq)
      float sv[2][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; nt++) {
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const int key = nt * 8 + 2 * cq + e;
          const int pos = kb * 16 + key;
          const float ks = sks[key];
          sv[nt][e] = (bok && pos < lim0 && pos >= lo0) ? sacc[nt][e] * ks : -INFINITY;
          sv[nt][2 + e] = (bok && pos < lim1 && pos >= lo1) ? sacc[nt][2 + e] * ks : -INFINITY;
          mx0 = fmaxf(mx0, sv[nt][e]);
          mx1 = fmaxf(mx1, sv[nt][2 + e]);
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(mr0 - mu0), al1 = fast_exp2(mr1 - mu1);
      mr0 = mn0;
      mr1 = mn1;
      uint32_t pa[4];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; nt++) {
        float pw[4];
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const int key = nt * 8 + 2 * cq + e;
          const float vs = svs[key];
          const float p0 = fast_exp2(sv[nt][e] - mu0);
          const float p1 = fast_exp2(sv[nt][2 + e] - mu1);
          ps0 += p0;
          ps1 += p1;
          pw[e] = sv[nt][e] == -INFINITY ? 0.f : p0 * vs;
          pw[2 + e] = sv[nt][2 + e] == -INFINITY ? 0.f : p1 * vs;
        }
        pa[2 * nt + 0] = pack_f16x2(pw[0], pw[1]);  // row r0, keys nt*8 + 2cq..
        pa[2 * nt + 1] = pack_f16x2(pw[2], pw[3]);  // row r1
      }
      lr0 = lr0 * al0 + ps0;
      lr1 = lr1 * al1 + ps1;
      // A fragment order: (r0, k 0-7), (r1, k 0-7), (r0, k 8-15), (r1, k 8-15)
      const uint32_t afr[4] = {pa[0], pa[1], pa[2], pa[3]};
#pragma unroll
      for (int t = 0; t < NT; t += 2) {
        uint32_t bv[4];
        const int mi = lane >> 3, rr = lane & 7;
        ldmatrix_x4_trans(bv, sV + ((mi & 1) * 8 + rr) * G::HSTRIDE + 8 * (t + (mi >> 1)));
        oacc[t][0] *= al0; oacc[t][1] *= al0; oacc[t][2] *= al1; oacc[t][3] *= al1;
        oacc[t + 1][0] *= al0; oacc[t + 1][1] *= al0; oacc[t + 1][2] *= al1; oacc[t + 1][3] *= al1;
        mma_16816(oacc[t], afr, bv[0], bv[1]);
        mma_16816(oacc[t + 1], afr, bv[2], bv[3]);
      }
    }
    cp_async_wait<0>();

    // epilogue: normalise, inverse rotation over d, signs, /b, bf16 store
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      lr0 += __shfl_xor_sync(0xffffffffu, lr0, o);
      lr1 += __shfl_xor_sync(0xffffffffu, lr1, o);
    }
    const float bn = ROT ? (float)B : 1.f;
    const float inv0 = 1.f / (lr0 * bn), inv1 = 1.f / (lr1 * bn);
    // thread values: row r0 -> oacc[t][0..1] (d = 8t + 2cq + e), row r1 -> oacc[t][2..3]
    if constexpr (ROT) {
#pragma unroll
    for (int t = 0; t < NT; t++) {  // stage h = 1
      float a = oacc[t][0], b = oacc[t][1];
      oacc[t][0] = a + b; oacc[t][1] = a - b;
      a = oacc[t][2]; b = oacc[t][3];
      oacc[t][2] = a + b; oacc[t][3] = a - b;
    }
#pragma unroll
    for (int lb = 0; lb < 2; lb++) {  // stages h = 2, 4 across the quad
      if ((2 << lb) >= B) break;
      const bool upper = (cq >> lb) & 1;
#pragma unroll
      for (int t = 0; t < NT; t++) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const float mine = oacc[t][e];
          const float other = __shfl_xor_sync(0xffffffffu, mine, 1 << lb);
          oacc[t][e] = upper ? other - mine : mine + other;
        }
      }
    }
#pragma unroll
    for (int ht = 1; ht < NT; ht <<= 1) {  // stages h = 8, 16, ... over t
      if (8 * ht >= B) break;
#pragma unroll
      for (int t = 0; t < NT; t++) {
        if ((t & ht) == 0) {
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const float a = oacc[t][e], b = oacc[t + ht][e];
            oacc[t][e] = a + b;
            oacc[t + ht][e] = a - b;
          }
        }
      }
    }
    }  // ROT
    if (r0 < nrows) {
      const int j = r0 / c.group, jj = r0 - j * c.group;
      uint16_t* dst = c.out + (long long)(q0 + tok0 + j) * c.out_stride + (long long)(h * c.group + jj) * D;
#pragma unroll
      for (int t = 0; t < NT; t++) {
        const int d = 8 * t + 2 * cq;
        reinterpret_cast<uint32_t*>(dst + d)[0] =
            pack_bf16x2_rn(oacc[t][0] * inv0 * ssign[d], oacc[t][1] * inv0 * ssign[d + 1]);
      }
    }
    if (r1 < nrows) {
      const int j = r1 / c.group, jj = r1 - j * c.group;
      uint16_t* dst = c.out + (long long)(q0 + tok0 + j) * c.out_stride + (long long)(h * c.group + jj) * D;
#pragma unroll
      for (int t = 0; t < NT; t++) {
        const int d = 8 * t + 2 * cq;
        reinterpret_cast<uint32_t*>(dst + d)[0] =
            pack_bf16x2_rn(oacc[t][2] * inv1 * ssign[d], oacc[t][3] * inv1 * ssign[d + 1]);
      }
    }
    __syncthreads();
  }
}

#include "prefill_ws.cuh"

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
template <typename K>
static bool configure(K kern, int smem, int threads, int* occ_out, bool* done, int* occ_cache) {
  if (!*done) {
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess || o < 1) return false;
    *occ_cache = o;
    *done = true;
  }
  *occ_out = *occ_cache;
  return true;
}

// CTAs per SM for a kernel that allocates tensor memory: the occupancy API
// answers 1 for any such kernel, so the count is taken from the kernel's
// registers and shared memory and the TMEM columns each CTA holds
template <typename K>
static bool configure_tmem(K kern, int smem, int threads, int tmem_cols, int* occ_out, bool* done, int* occ_cache) {
  if (!*done) {
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return false;
    cudaFuncAttributes fa;
    int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
      return false;
    const int warps = (threads + 31) / 32;
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;  // allocated per warp in 256-register units
    const int by_regs = regs_sm / (regs_warp * ((warps + 3) / 4 * 4));  // and per group of four warps
    const int by_smem = smem_sm / (smem + fa.sharedSizeBytes + reserved);
    const int by_tmem = 512 / tmem_cols;
    const int o = min(by_regs, min(by_smem, by_tmem));
    if (o < 1) return false;
    *occ_cache = o;
    *done = true;
  }
  *occ_out = *occ_cache;
  return true;
}

template <int D, int FMT>
static int launch_attention_t(const AttnArgs& a, cudaStream_t stream) {
  WorkspaceLayout L;
  workspace_layout(a.num_seqs, a.num_q_tokens, a.num_q_heads, a.num_kv_heads, a.head_size, &L);
  PlanView pv = plan_view(a.workspace, L);
  const int dev = current_device();
  const int sms = sm_count(dev);
  Common c;
  c.q = static_cast<const uint16_t*>(a.q);
  c.q_stride = a.q_stride;
  c.k_cache = a.k_cache;
  c.v_cache = a.v_cache;
  c.k_scale = a.k_scale;
  c.v_scale = a.v_scale;
  c.geo = a.geo;
  c.block_table = a.block_table;
  c.max_blocks = a.max_blocks_per_seq;
  c.seq_lens = a.seq_lens;
  c.qsl = a.query_start_loc;
  c.num_seqs = a.num_seqs;
  c.num_q_tokens = a.num_q_tokens;
  c.hq = a.num_q_heads;
  c.hkv = a.num_kv_heads;
  c.group = a.num_q_heads / a.num_kv_heads;
  c.gdiv = FastDiv((uint32_t)c.group);
  c.num_blocks = a.num_blocks;
  c.causal = a.causal;
  c.window = a.sliding_window;
  constexpr bool ROT = FMT == kFmtInt4;
  c.qscale = a.softmax_scale * kLog2e / (ROT ? (float)Head<D>::b : 1.f);
  c.signs = a.signs;
  c.out = static_cast<uint16_t*>(a.out);
  c.out_stride = a.out_stride;
  c.status = a.dev_status;
  // prefill items: 256 rows on the warp-specialised tensor-core kernel
  // (head sizes up to 192), 64 on the warp-MMA one
  constexpr bool kTcPrefill = D <= 192;
  constexpr int kTileRows = kTcPrefill ? kWsRows : kPrefillRows;
  c.tile_tokens = kTileRows / c.group > 0 ? kTileRows / c.group : 1;
  c.max_items = L.max_prefill_items;
  // kv heads per decode CTA: the largest divisor of Hkv up to 4 whose
  // staging ring fits in shared memory (int8 tiles are twice as large).
  // Four 4-warp CTAs per SM beat two 8-warp ones (independent barrier
  // domains; measured on GB300: long-context decode 0.76 vs 0.73 of the HBM
  // peak); the in-slot layout keeps up to 8, its unaligned slots read
  // better in longer contiguous runs
  constexpr int kMaxSmem = 227 * 1024;
  const bool inslot = a.geo.chead != (FMT == kFmtInt8 ? D : D / 2);
  int hg_cap = inslot ? 8 : 4;
  while (hg_cap > 1 && DecGeom<D, 1, FMT>::smem_bytes(hg_cap) > kMaxSmem) hg_cap--;
  c.hg = 1;
  for (int h = hg_cap; h >= 1; h--)
    if (a.num_kv_heads % h == 0) {
      c.hg = h;
      break;
    }
  c.ng = a.num_kv_heads / c.hg;
  if (c.group > kPrefillRows) return KV_INT4_ERR_HEADS;

  // decode configuration: blocks per schedule position and the kernel's
  // occupancy.  Pairing blocks needs q_len * G <= 4 for every decode
  // sequence; when the batch also holds prefills (q_len * G > 8 somewhere),
  // decode is sized for single-token queries and longer ones go to prefill.
  const bool any_decode = c.group <= kDecodeCols;
  int dec_occ = 0;
  if (any_decode) {
    static bool attr_done[kMaxDevices][2] = {};
    static int occ_cache[kMaxDevices][2][9] = {};
    auto occupancy = [&](auto kern, int np, int smem_max, int smem) -> int {
      if (smem > kMaxSmem) return 0;  // this ring does not fit
      if (!attr_done[dev][np - 1]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, min(smem_max, kMaxSmem)) !=
            cudaSuccess)
          return 0;
        attr_done[dev][np - 1] = true;
      }
      if (!occ_cache[dev][np - 1][c.hg]) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, c.hg * 32, smem) != cudaSuccess || o < 1) return 0;
        occ_cache[dev][np - 1][c.hg] = o;
      }
      return occ_cache[dev][np - 1][c.hg];
    };
    const int occ1 = occupancy(decode_kernel<D, 1, FMT>, 1, DecGeom<D, 1, FMT>::smem_bytes(8), DecGeom<D, 1, FMT>::smem_bytes(c.hg));
    if (occ1 < 1) return KV_INT4_ERR_CUDA;
    const long long mq = (long long)(a.max_query_len > 0 ? a.max_query_len : 1) * c.group;
    const long long cols = mq <= kDecodeCols ? mq : c.group;
    c.np = 1;
    dec_occ = occ1;
    if (cols <= kDecodeCols / 2) {
      const int occ2 =
          occupancy(decode_kernel<D, 2, FMT>, 2, DecGeom<D, 2, FMT>::smem_bytes(8), DecGeom<D, 2, FMT>::smem_bytes(c.hg));
      if (occ2 >= 1 && occ2 >= occ1) {  // 0: the paired ring does not fit
        c.np = 2;
        dec_occ = occ2;
      }
    }
  } else {
    c.np = 1;
  }
  c.dcols = kDecodeCols / c.np;

  // 1. prep
  {
    const long long rows = (long long)a.num_q_tokens * a.num_q_heads;
    const long long pieces = rows * (D / kPrepPiece(D));
    const long long grid = 1 + (pieces + kPrepThreads - 1) / kPrepThreads;
    if (grid > 0x7fffffff) return KV_INT4_ERR_SIZE;
    timing_begin(kTimedPrep, stream);
    prep_kernel<D, ROT><<<(unsigned)grid, kPrepThreads, 0, stream>>>(c, pv);
    timing_end(kTimedPrep, stream);
    if (cudaGetLastError() != cudaSuccess) return KV_INT4_ERR_CUDA;
  }
  // 2. prefill
  const bool may_prefill = c.group > c.dcols || (long long)a.max_query_len * c.group > c.dcols;
  if (may_prefill) {
    static bool done[kMaxDevices] = {};
    static int occ_c[kMaxDevices] = {};
    int occ = 0;
    if constexpr (kTcPrefill) {
      using G = WsGeom<D, FMT>;
      if (!configure_tmem(prefill_ws_kernel<D, FMT>, G::SMEM, G::THREADS, G::TMEM_COLS, &occ, &done[dev], &occ_c[dev]))
        return KV_INT4_ERR_CUDA;
      long long grid = (long long)sms * occ;
      if (grid > L.max_prefill_items) grid = L.max_prefill_items;
      if (grid < 1) grid = 1;
      timing_begin(kTimedPrefill, stream);
      prefill_ws_kernel<D, FMT><<<(unsigned)grid, G::THREADS, G::SMEM, stream>>>(PreParams{c, pv});
      timing_end(kTimedPrefill, stream);
    } else {
      using G = PreGeom<D, FMT>;
      if (!configure(prefill_kernel<D, FMT>, G::SMEM, G::THREADS, &occ, &done[dev], &occ_c[dev]))
        return KV_INT4_ERR_CUDA;
      long long grid = (long long)sms * occ;
      if (grid > L.max_prefill_items) grid = L.max_prefill_items;
      if (grid < 1) grid = 1;
      timing_begin(kTimedPrefill, stream);
      prefill_kernel<D, FMT><<<(unsigned)grid, G::THREADS, G::SMEM, stream>>>(PreParams{c, pv});
      timing_end(kTimedPrefill, stream);
    }
    if (cudaGetLastError() != cudaSuccess) return KV_INT4_ERR_CUDA;
  }
  // 3. decode + 4. reduce
  if (any_decode) {
    long long grid = (long long)sms * dec_occ;
    if (grid * c.hg > kMaxDecodeWarps) grid = kMaxDecodeWarps / c.hg;
    const int num_ctas = (int)grid;
    const int threads = c.hg * 32;
    timing_begin(kTimedDecode, stream);
    if (c.np == 2)
      decode_kernel<D, 2, FMT><<<(unsigned)grid, threads, DecGeom<D, 2, FMT>::smem_bytes(c.hg), stream>>>(
          DecParams{c, pv, num_ctas});
    else
      decode_kernel<D, 1, FMT><<<(unsigned)grid, threads, DecGeom<D, 1, FMT>::smem_bytes(c.hg), stream>>>(
          DecParams{c, pv, num_ctas});
    timing_end(kTimedDecode, stream);
    if (cudaGetLastError() != cudaSuccess) return KV_INT4_ERR_CUDA;
    // query columns a decode segment can need: q_len * G, at most dcols
    const long long mcols = (long long)(a.max_query_len > 0 ? a.max_query_len : 1) * c.group;
    int cps = c.dcols;
    while (cps > 1 && cps / 2 >= mcols) cps /= 2;  // a divisor of dcols (a power of two)
    const long long spc = c.dcols / cps;  // segments per CTA
    const long long rgrid = ((long long)a.num_seqs * a.num_kv_heads + spc - 1) / spc;
    if (rgrid > 0x7fffffff) return KV_INT4_ERR_SIZE;
    timing_begin(kTimedReduce, stream);
    reduce_kernel<D, ROT><<<(unsigned)rgrid, c.dcols * 32, 0, stream>>>(RedParams{c, pv, num_ctas, cps});
    timing_end(kTimedReduce, stream);
    if (cudaGetLastError() != cudaSuccess) return KV_INT4_ERR_CUDA;
  }
  return KV_INT4_OK;
}

template <int FMT>
static int launch_fmt(const AttnArgs& a, cudaStream_t stream) {
  switch (a.head_size) {
    case 64: return launch_attention_t<64, FMT>(a, stream);
    case 96: return launch_attention_t<96, FMT>(a, stream);
    case 128: return launch_attention_t<128, FMT>(a, stream);
    case 192: return launch_attention_t<192, FMT>(a, stream);
    case 256: return launch_attention_t<256, FMT>(a, stream);
    default: return KV_INT4_ERR_HEAD_SIZE;
  }
}

int launch_attention(const AttnArgs& a, cudaStream_t stream) {
  return a.int8 ? launch_fmt<kFmtInt8>(a, stream) : launch_fmt<kFmtInt4>(a, stream);
}

}  // namespace kvint4
