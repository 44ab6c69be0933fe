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
  int4* dseq;         // decode sequences in order: (sequence id, seq_len, first query token, q_len)
  int64_t* dprefix;
  int2* ptab;         // prefill sequences in order: (seq id, index of its first item); [n_pseq].y = items
  int2* plist;        // prefill (sequence, tile) pairs, longest first; pair i gives items i Hkv .. i Hkv + Hkv - 1
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
  v.dseq = reinterpret_cast<int4*>(b + L.dseq);
  v.dprefix = reinterpret_cast<int64_t*>(b + L.dprefix);
  v.ptab = reinterpret_cast<int2*>(b + L.pitems);
  v.plist = reinterpret_cast<int2*>(b + L.plist);
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
  int max_qlen;  // the caller's max_query_len: launch sizes assume no q_len above it
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
  int hg;           // decode: kv heads per CTA (largest divisor of hkv <= 4)
  int ng;           // decode: head groups per sequence (hkv / hg)
  int nl;           // decode: lanes (a divisor of ng): CTA r serves the head groups g with g mod nl = r mod nl
  int np;           // decode: 16-key blocks per schedule position (1, 2 or 4)
  int dcols;        // decode: query columns per block (8 / np); longer queries go to prefill
  long long max_items;  // capacity of the prefill item list
};

// floor(n / d) for 0 <= n, 0 < d: one 32-bit division when both fit (the
// usual case for schedule arithmetic), the 64-bit routine otherwise
__device__ __forceinline__ long long div_nn(long long n, long long d) {
  return ((n | d) >> 31) == 0 ? (long long)((uint32_t)n / (uint32_t)d) : n / d;
}

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

// keys that prefill tile t of a sequence (kv length L, q_len qn) attends:
// up to its last query's causal horizon, or all
__device__ __forceinline__ int prefill_tile_keys(const Common& c, int L, int qn, int t) {
  return c.causal ? L - qn + min(qn, (t + 1) * c.tile_tokens) : L;
}
// prefill item itn in the prep kernel's longest-first order: (sequence, kv
// head, tile, 16-key blocks), or sequence -1 past the last item
__device__ __forceinline__ int4 prefill_item(const Common& c, const PlanView& pv, int itn, int n_items) {
  if (itn >= n_items) return make_int4(-1, 0, 0, 0);
  const int pi = itn / c.hkv;
  const int2 st = pv.plist[pi];
  const int qa = c.qsl[st.x], qn = c.qsl[st.x + 1] - qa;
  const int keys = prefill_tile_keys(c, c.seq_lens[st.x], qn, st.y);
  return make_int4(st.x, itn - pi * c.hkv, st.y, (keys + 15) / 16);
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
      int kind = 0, nblk = 0, ntiles = 0, ql = 0, L = 0, q0 = 0;
      if (s < c.num_seqs) {
        q0 = c.qsl[s];
        const int q1 = c.qsl[s + 1];
        L = c.seq_lens[s];
        ql = q1 - q0;
        // a q_len above max_query_len would fall outside the launches sized
        // from it (decode columns, the prefill launch, the reduce segments)
        const bool bad = q0 < 0 || q1 > c.num_q_tokens || ql < 0 || L < ql || ql > c.max_qlen ||
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
        pv.dseq[n_dseq + ex_a] = make_int4(s, L, q0, ql);
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
    // the prefill (sequence, tile) pairs, longest first: a counting sort over
    // buckets of 16-key blocks (descending), so that the longest items start
    // first and the shortest fill the end of the launch (within a bucket the
    // order is arbitrary; every item computes the same rows either way)
    constexpr int kBuckets = 2048;
    __shared__ int hist[kBuckets];
    if (n_pseq > 0 && n_items <= c.max_items && n_items <= INT_MAX) {
      int sh = 0;
      while ((((long long)c.max_blocks + 1) >> sh) >= kBuckets) sh++;
      auto bucket = [&](int nkb) { return kBuckets - 1 - min(kBuckets - 1, nkb >> sh); };
      for (int i = threadIdx.x; i < kBuckets; i += kPrepThreads) hist[i] = 0;
      __syncthreads();  // the sequence table and the histogram
      for (int p = threadIdx.x; p < n_pseq; p += kPrepThreads) {
        const int sq = pv.ptab[p].x, qn = c.qsl[sq + 1] - c.qsl[sq], Ls = c.seq_lens[sq];
        const int nt = (qn + c.tile_tokens - 1) / c.tile_tokens;
        for (int t = 0; t < nt; t++) atomicAdd(&hist[bucket((prefill_tile_keys(c, Ls, qn, t) + 15) / 16)], 1);
      }
      __syncthreads();
      // exclusive prefix over the buckets: thread j owns buckets [8j, 8j + 8)
      constexpr int PER = kBuckets / kPrepThreads;
      int mine = 0;
#pragma unroll
      for (int i = 0; i < PER; i++) mine += hist[threadIdx.x * PER + i];
      int total;
      int run = block_exclusive_scan<int>(mine, &total, s_i32);
#pragma unroll
      for (int i = 0; i < PER; i++) {
        const int hb = hist[threadIdx.x * PER + i];
        hist[threadIdx.x * PER + i] = run;
        run += hb;
      }
      __syncthreads();
      for (int p = threadIdx.x; p < n_pseq; p += kPrepThreads) {
        const int sq = pv.ptab[p].x, qn = c.qsl[sq + 1] - c.qsl[sq], Ls = c.seq_lens[sq];
        const int nt = (qn + c.tile_tokens - 1) / c.tile_tokens;
        for (int t = 0; t < nt; t++)
          pv.plist[atomicAdd(&hist[bucket((prefill_tile_keys(c, Ls, qn, t) + 15) / 16)], 1)] = make_int2(sq, t);
      }
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
        // INT4: each 8-element group in the nibble order of the code words,
        // (0, 4), (1, 5), (2, 6), (3, 7): the order the attention kernels'
        // K tiles and fragments use, so that they read q' as stored
        const float2 y = ROT ? __fmul2_rn(make_float2(x[8 * v + k], x[8 * v + k + 4]), qs)
                             : __fmul2_rn(make_float2(x[8 * v + 2 * k], x[8 * v + 2 * k + 1]), qs);
        o[k] = pack_f16x2(y.x, y.y);
      }
      reinterpret_cast<uint4*>(dst)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

#include "decode.cuh"

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
  // a warp per (segment, query column): the CTA's dcols warps cover
  // dcols / cps segments of cps columns each
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * (c.dcols / prm.cps) + warp / prm.cps;
  const int col = warp % prm.cps;
  const int n_dseq = pv.plan[0];
  if (seg >= n_dseq * c.hkv) return;
  const int i = seg / c.hkv, h = seg - i * c.hkv;
  const int4 di = pv.dseq[i];  // (sequence, seq_len, first query token, q_len)
  const int q0 = di.z, ql = di.w;
  if (col >= ql * c.group) return;  // ql * group <= cps
  const int nblk = (di.y + 15) / 16;
  const int npos = (nblk - first_block(c, di.y, ql) + c.np - 1) / c.np;
  const int grp = h / c.hg, hl = h - grp * c.hg;
  // the lane of the segment's head group, and the group's place in its lane
  const int gpl = c.ng / c.nl, lane_g = grp % c.nl, gs = grp / c.nl;
  const long long Tu = pv.dprefix[n_dseq] * gpl;
  const long long sbeg = pv.dprefix[i] * gpl + (long long)gs * npos, send = sbeg + npos;
  const int W = prm.num_ctas / c.nl;  // the lane's CTAs
  auto wstart = [&](long long w) { return div_nn(Tu * w, W); };

  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; k++) acc[k] = 0.f;
  float M = -INFINITY, Lsum = 0.f;
  // The pieces (the direct slot of the piece that starts the segment, then
  // every CTA whose non-empty range starts strictly inside it) are merged a
  // chunk at a time: all of a chunk's loads are issued before any of its
  // arithmetic (the chunk's largest maximum first, then every piece weighted
  // by 2^(m - that maximum)), so a segment's pieces cost one or two memory
  // round trips instead of one each.  With two blocks per position a
  // piece's columns col and col + dcols hold the same query over disjoint key
  // blocks; with four the decode merged them into column col.
  const int nsub = c.np == 2 ? 2 : 1;
  constexpr int CH = 4;  // pieces per chunk
  int64_t chunk[CH];     // piece slots: -1 the direct slot, else the CTA slot index
  int nch = 0;
  auto o_of = [&](int64_t sl) {
    return sl < 0 ? pv.direct_o + (long long)seg * kDecodeCols * D : pv.warp_o + sl * kDecodeCols * D;
  };
  auto ml_of = [&](int64_t sl) {
    return sl < 0 ? pv.direct_ml + (long long)seg * kDecodeCols * 2 : pv.warp_ml + sl * kDecodeCols * 2;
  };
  auto merge_chunk = [&]() {
    float mw[CH][2], lw[CH][2], ov[CH][2][PER];
#pragma unroll
    for (int j = 0; j < CH; j++) {
#pragma unroll
      for (int sub = 0; sub < 2; sub++) {
        const bool use = j < nch && sub < nsub;
        const int cc = col + sub * c.dcols;
        const float* ml = ml_of(use ? chunk[j] : -1);
        const float* o = o_of(use ? chunk[j] : -1);
        mw[j][sub] = use ? ml[cc * 2] : -INFINITY;
        lw[j][sub] = use ? ml[cc * 2 + 1] : 0.f;
#pragma unroll
        for (int k = 0; k < PER; k++) ov[j][sub][k] = use ? o[cc * D + lane + 32 * k] : 0.f;
      }
    }
    float Mc = -INFINITY;
#pragma unroll
    for (int j = 0; j < CH; j++) Mc = fmaxf(Mc, fmaxf(mw[j][0], mw[j][1]));
    const float Mn = fmaxf(M, Mc);
    const float Mu = Mn == -INFINITY ? 0.f : Mn;
    const float a = fast_exp2(M - Mu);
#pragma unroll
    for (int k = 0; k < PER; k++) acc[k] *= a;
    Lsum *= a;
#pragma unroll
    for (int j = 0; j < CH; j++) {
#pragma unroll
      for (int sub = 0; sub < 2; sub++) {
        const float wgt = fast_exp2(mw[j][sub] - Mu);  // 0 for an unused entry
#pragma unroll
        for (int k = 0; k < PER; k++) acc[k] += ov[j][sub][k] * wgt;
        Lsum += lw[j][sub] * wgt;
      }
    }
    M = Mn;
    nch = 0;
  };
  auto add_piece = [&](int64_t sl) {
#pragma unroll
    for (int j = 0; j < CH; j++)
      if (j == nch) chunk[j] = sl;  // a register, not local memory
    if (++nch == CH) merge_chunk();
  };
  add_piece(-1);
  // the other pieces: CTAs whose non-empty range starts strictly inside the
  // segment.  Walk the CTAs or the positions, whichever are fewer.
  auto add_cta = [&](long long w) { add_piece((w * c.nl + lane_g) * c.hg + hl); };
  const long long w_first = div_nn((sbeg + 1) * W + Tu - 1, Tu);  // first CTA starting after sbeg
  const long long w_end = div_nn(send * W + Tu - 1, Tu);          // first CTA starting at or after send
  if (w_end - w_first <= send - sbeg - 1) {
    for (long long w = w_first; w < w_end; w++)
      if (wstart(w + 1) > wstart(w)) add_cta(w);
  } else {
    for (long long p = sbeg + 1; p < send; p++) {
      const long long w = div_nn((p + 1) * W + Tu - 1, Tu) - 1;  // last CTA starting at or before p
      if (wstart(w) == p) add_cta(w);
    }
  }
  if (nch > 0) merge_chunk();
  // normalise, then D (I_n (x) H_b) (.) / b in registers: element e = lane +
  // 32 k of the head vector is acc[k] of lane e % 32, and a butterfly stage of
  // span hs pairs e with e ^ hs (Sylvester order) -- across lanes by warp
  // shuffles for spans below 32, across this lane's registers above
  const float inv = 1.f / (Lsum * (ROT ? (float)B : 1.f));
#pragma unroll
  for (int k = 0; k < PER; k++) acc[k] *= inv;
  if constexpr (ROT) {
#pragma unroll
    for (int hs = 1; hs < (B < 32 ? B : 32); hs <<= 1) {
      const bool upper = (lane & hs) != 0;
#pragma unroll
      for (int k = 0; k < PER; k++) {
        const float o = __shfl_xor_sync(0xffffffffu, acc[k], hs);
        acc[k] = upper ? o - acc[k] : acc[k] + o;
      }
    }
#pragma unroll
    for (int hs = 32; hs < B; hs <<= 1) {
      const int hk = hs / 32;
#pragma unroll
      for (int k = 0; k < PER; k++)
        if (!(k & hk)) {
          const float a = acc[k], b = acc[k + hk];
          acc[k] = a + b;
          acc[k + hk] = a - b;
        }
    }
  }
  const int j = col / c.group, jj = col - j * c.group;
  uint16_t* dst = c.out + (long long)(q0 + j) * c.out_stride + (long long)(h * c.group + jj) * D;
#pragma unroll
  for (int k = 0; k < PER; k++) {
    const int e = lane + 32 * k;
    const float x = (ROT && c.signs[e] < 0) ? -acc[k] : acc[k];
    dst[e] = (uint16_t)(pack_bf16x2_rn(x, 0.f) & 0xffffu);  // coalesced: a warp writes 64 contiguous bytes per k
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
  const int n_items = pv.plan[1];

#pragma unroll 1
  while (true) {
    if (tid == 0) {
      // next item, longest first: (prefill sequence, kv head, tile, blocks)
      const int4 it = prefill_item(c, pv, atomicAdd(&pv.plan[2], 1), n_items);
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
          // p_k = (element k, element k+4): K rows stay in this nibble order
          // (q' is stored in it), V rows, whose dims are the output's, go to
          // natural order 0..7
          uint4 o = make_uint4(p0, p1, p2, p3);
          if (which) {
            o.x = __byte_perm(p0, p1, 0x5410);
            o.y = __byte_perm(p2, p3, 0x5410);
            o.z = __byte_perm(p0, p1, 0x7632);
            o.w = __byte_perm(p2, p3, 0x7632);
          }
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
// sets the kernel's shared-memory limit and gives its CTAs per SM
template <typename K>
static bool configure(K kern, int smem, int threads, int* occ_out) {
  if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return false;
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess || o < 1) return false;
  *occ_out = o;
  return true;
}

// CTAs per SM for a kernel that allocates tensor memory: the occupancy API
// answers 1 for any such kernel, so the count is taken from the kernel's
// registers and shared memory and the TMEM columns each CTA holds
template <typename K>
static bool configure_tmem(K kern, int smem, int threads, int tmem_cols, int* occ_out) {
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
  *occ_out = o;
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
  c.max_qlen = a.max_query_len;
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
  // peak), for the in-slot layout too since the head-group lanes put the
  // CTAs reading one row's slots side by side (long-context in-slot decode
  // 2.226 -> 2.200 ms, Phi-3 46.6 -> 43.3 us against eight-head CTAs)
  constexpr int kMaxSmem = 227 * 1024;
  const bool inslot = a.geo.chead != (FMT == kFmtInt8 ? D : D / 2);
  int hg_cap = 4;
  while (hg_cap > 1 && DecGeom<D, 1, FMT>::smem_bytes(hg_cap) > kMaxSmem) hg_cap--;
  c.hg = 1;
  for (int h = hg_cap; h >= 1; h--)
    if (a.num_kv_heads % h == 0) {
      c.hg = h;
      break;
    }
  c.ng = a.num_kv_heads / c.hg;
  c.nl = 1;
  if (c.group > kPrefillRows) return KV_INT4_ERR_HEADS;

  // decode configuration: blocks per schedule position and the kernel's
  // occupancy.  Pairing blocks needs q_len * G <= 4 for every decode
  // sequence; when the batch also holds prefills (q_len * G > 8 somewhere),
  // decode is sized for single-token queries and longer ones go to prefill.
  const bool any_decode = c.group <= kDecodeCols;
  int dec_occ = 0;
  // the 16-byte scale rows (and at INT4 d = 128 the deeper decode ring)
  // serve the separate-scale layout with four heads per CTA and 16-byte
  // aligned scale rows; the in-slot layout's eight-head CTAs read better with
  // the shallower ring (measured on GB300: in-slot decode 2.20 vs 2.63 ms)
  const bool dec_deep = !inslot && c.hg == 4 && (reinterpret_cast<uintptr_t>(a.k_scale) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(a.v_scale) & 15) == 0 && (a.geo.srow * 4) % 16 == 0 &&
                        (a.geo.sblk * 4) % 16 == 0 && a.geo.shead == 1;
  if (any_decode) {
    // one cache per kernel and head group: (blocks per position, ring depth, hg)
    static PerContext<int> occ_cache[4][2][9];
    auto occupancy = [&](auto kern, int np, int smem_max, int smem) -> int {
      if (smem > kMaxSmem) return 0;  // this ring does not fit
      int o = 0;
      const bool ok = occ_cache[np - 1][dec_deep][c.hg].get(dev, [&](int* v) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, min(smem_max, kMaxSmem)) !=
            cudaSuccess)
          return false;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, c.hg * 32, smem) == cudaSuccess && *v >= 1;
      }, &o);
      return ok ? o : 0;
    };
    using E1 = DecodeEntry<D, 1, FMT>;
    using E2 = DecodeEntry<D, 2, FMT>;
    const int occ1 = occupancy(E1::kernel(dec_deep), 1, E1::smem(dec_deep, 8), E1::smem(dec_deep, c.hg));
    if (occ1 < 1) return KV_INT4_ERR_CUDA;
    const long long mq = (long long)(a.max_query_len > 0 ? a.max_query_len : 1) * c.group;
    const long long cols = mq <= kDecodeCols ? mq : c.group;
    c.np = 1;
    dec_occ = occ1;
    if (cols <= kDecodeCols / 2) {
      const int occ2 = occupancy(E2::kernel(dec_deep), 2, E2::smem(dec_deep, 8), E2::smem(dec_deep, c.hg));
      if (occ2 >= 1 && occ2 >= occ1) {  // 0: the paired ring does not fit
        c.np = 2;
        dec_occ = occ2;
        // four blocks per position when every block needs at most 2 columns
        // (one query per kv head: Phi-3's shape): the position's fixed work
        // serves twice the keys.  INT4 with four-head CTAs and 16-byte scale
        // rows only (the other instances of the four-block kernel spill),
        // while at least three CTAs fit per SM (measured on GB300 at d = 128,
        // G = 1 and 2, three CTAs of the eight-slot ring against four of the
        // six-slot one: 1-3 % faster; d = 192 and 256 would drop to two)
        if constexpr (FMT == kFmtInt4) {
          if (cols <= kDecodeCols / 4 && dec_deep) {
            using E4 = DecodeEntry<D, 4, FMT>;
            const int occ4 = occupancy(E4::kernel(true), 4, E4::smem(true, 8), E4::smem(true, c.hg));
            if (occ4 >= 1 && (occ4 >= occ2 || occ4 >= 3)) {
              c.np = 4;
              dec_occ = occ4;
            }
          }
        }
      }
    }
  } else {
    c.np = 1;
  }
  c.dcols = kDecodeCols / c.np;
  // the decode launch's CTAs
  int dec_grid = 0;
  if (any_decode) {
    long long grid = (long long)sms * dec_occ;
    if (grid * c.hg > kMaxDecodeWarps) grid = kMaxDecodeWarps / c.hg;
    // lanes: the CTAs of all (or as many as divide evenly) head groups walk
    // the same positions side by side, so the groups' slices of a block's
    // code and scale rows are read together and each cache line leaves DRAM
    // once (measured on GB300, Phi-3 shape, 32 kv heads in 8 groups: DRAM
    // reads 1.79x the cache bytes when a CTA walks its groups one after the
    // other)
    for (int l = (int)(grid < c.ng ? grid : c.ng); l >= 1; l--)
      if (c.ng % l == 0) {
        c.nl = l;
        break;
      }
    grid = grid / c.nl * c.nl;
    dec_grid = (int)grid;
  }

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
    static PerContext<int> occ_c;
    int occ = 0;
    if constexpr (kTcPrefill) {
      using G = WsGeom<D, FMT>;
      if (!occ_c.get(dev, [](int* o) {
            return configure_tmem(prefill_ws_kernel<D, FMT>, G::SMEM, G::THREADS, G::TMEM_COLS, o);
          }, &occ))
        return KV_INT4_ERR_CUDA;
      long long grid = (long long)sms * occ;
      if (grid > L.max_prefill_items) grid = L.max_prefill_items;
      if (grid < 1) grid = 1;
      timing_begin(kTimedPrefill, stream);
      prefill_ws_kernel<D, FMT><<<(unsigned)grid, G::THREADS, G::SMEM, stream>>>(PreParams{c, pv});
      timing_end(kTimedPrefill, stream);
    } else {
      using G = PreGeom<D, FMT>;
      if (!occ_c.get(dev, [](int* o) { return configure(prefill_kernel<D, FMT>, G::SMEM, G::THREADS, o); }, &occ))
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
    const long long grid = dec_grid;
    const int num_ctas = dec_grid;
    const int threads = c.hg * 32;
    timing_begin(kTimedDecode, stream);
    if (c.np == 4) {
      if constexpr (FMT == kFmtInt4)
        DecodeEntry<D, 4, FMT>::kernel(true)<<<(unsigned)grid, threads, DecodeEntry<D, 4, FMT>::smem(true, c.hg), stream>>>(
            DecParams{c, pv, num_ctas});
    } else if (c.np == 2)
      DecodeEntry<D, 2, FMT>::kernel(dec_deep)<<<(unsigned)grid, threads, DecodeEntry<D, 2, FMT>::smem(dec_deep, c.hg), stream>>>(
          DecParams{c, pv, num_ctas});
    else
      DecodeEntry<D, 1, FMT>::kernel(dec_deep)<<<(unsigned)grid, threads, DecodeEntry<D, 1, FMT>::smem(dec_deep, c.hg), stream>>>(
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
