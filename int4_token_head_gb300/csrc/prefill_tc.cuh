// Prefill on the 5th-generation tensor cores (tcgen05), included by
// attention.cu after the schedule and parameter types it shares.
//
// One CTA of 4 warps per tile of 128 query rows (query token x q head of one
// kv group: the MMA's M), 64 keys (four cache blocks) per step:
//   1. the codes of the step's four blocks were staged by cp.async during
//      the previous step; all threads dequantise them (exactly, as f16) into
//      a K tile and a V tile in shared memory, 128-byte swizzled;
//   2. one thread issues S = Q' K^T (D/16 MMAs of 128 x 64 x 16) into TMEM;
//   3. each thread owns one query row: it reads its 64 scores with
//      tcgen05.ld, scales them by the keys' K scales, masks them (causal,
//      window, length, bad blocks), runs the base-2 online softmax and
//      writes its row of P' = p * v_scale into a swizzled P tile.  The
//      exponent reference m_ref of a row moves (and its O row in TMEM is
//      rescaled) only when the row max passes m_ref + tau: tau = 8 while
//      every V scale of the step is below 128, so p <= 2^8 keeps P' below
//      2^15 in f16; otherwise tau = 0 (the exact running max);
//   4. one thread issues O' += P' V (4 MMAs of 128 x D x 16, V read as an
//      MN-major operand) into TMEM;
//   5. the epilogue reads each row's O', normalises it and (INT4) applies
//      D (I_n (x) H_b) (.) / b in registers, one thread per row.
// INT4 tiles keep each 8-element group in nibble order (elements 0,4,1,5,
// 2,6,3,7: two nibble lanes of a 32-bit word per f16x2, no byte shuffles);
// Q' is stored with the same permutation, which leaves Q' K^T unchanged,
// and the epilogue undoes it on O' (its columns are V's dims) by register
// renaming.
// Shared-memory operands: K-major tiles are [D/64 blocks][rows][128 bytes]
// with the 16-byte chunk index XORed by row % 8 (1024-byte atoms; leading
// byte offset unused, stride byte offset 1024); the V tile uses the same
// bytes as an MN-major operand (dims are the MMA's N: leading byte offset =
// one 64-dim block = 64 keys x 128 bytes, stride byte offset = 8 keys).

template <int D, int FMT>
struct TcPreGeom {
  static constexpr int ROWS = 128;                   // query rows per tile (MMA M)
  static constexpr int NK = 64;                      // keys per step
  static constexpr int KB = (D + 63) / 64;           // 128-byte blocks of an f16 head vector
  static constexpr int QBYTES = ROWS * 128 * KB;
  static constexpr int KVBYTES = NK * 128 * KB;      // K tile; the V tile has the same size
  static constexpr int PBYTES = ROWS * 128;          // P' tile: 128 rows x 64 keys
  static constexpr int CB = FMT == kFmtInt8 ? D : D / 2;  // code bytes per head vector
  static constexpr int SC_OFF = 4 * 2 * 16 * CB;     // staging: codes [block][K/V][16][CB], then scales
  static constexpr int FL_OFF = SC_OFF + 4 * 2 * 16 * 4;  // then four block flags
  static constexpr int STG = FL_OFF + 16;
  // P' reuses the K tile's bytes (K is dead once S is complete)
  static constexpr int KPBYTES = KVBYTES > PBYTES ? KVBYTES : PBYTES;
  static constexpr int TMEM_COLS = NK + D <= 256 ? 256 : 512;  // S at [0, 64), O' at [64, 64 + D)
  static constexpr int USED = 1024 + QBYTES + KPBYTES + KVBYTES + STG + 2 * NK * 4 + 32 + D * 4 + 64;
  // two CTAs per SM: their tensor-core and CUDA-core phases overlap; the
  // floor keeps a third (which would wait for TMEM) off the SM
  static constexpr int SMEM = USED > 80 * 1024 ? USED : 80 * 1024;
  static_assert(D % 32 == 0 && D <= 192, "head sizes served by the tensor-core prefill");
};

// byte offset of 16-byte chunk c (elements 8c .. 8c+7) of row r in a
// 128-byte-swizzled K-major tile of `rows` rows
__device__ __forceinline__ uint32_t sw128(int rows, int r, int c) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// position i of an INT4 8-element group holds element nib_order(i)
__host__ __device__ constexpr int nib_order(int i) { return (i >> 1) + ((i & 1) << 2); }

// 8 exact f16 values of the codes at src (INT4: one word, 8 codes, nibble
// order; int8: two words, natural order); `ok` false gives zeros
template <int FMT>
__device__ __forceinline__ uint4 dequant8(const uint8_t* src, bool ok) {
  uint4 o;
  if constexpr (FMT == kFmtInt4) {
    const uint32_t x = ok ? *reinterpret_cast<const uint32_t*>(src) : 0u;  // code 0
    const uint32_t y = x >> 8;
    // low nibbles of bytes (0, 2) -> 1032 + c, exact; minus 1032
    // high nibbles of bytes (0, 2) -> 1152 + 16c, exact; / 16 - 72 in one rounding of an exact value
    const uint32_t n1032 = kF16x2_M1032, h16 = 0x2c002c00u, m72 = 0xd480d480u;  // (-1032, -1032), (1/16, 1/16), (-72, -72)
    const __half2 m1032 = *reinterpret_cast<const __half2*>(&n1032);
    const __half2 inv16 = *reinterpret_cast<const __half2*>(&h16), n72 = *reinterpret_cast<const __half2*>(&m72);
    uint32_t a = nib_lo(x), b = nib_hi(x), e = nib_lo(y), f = nib_hi(y);
    __half2 ha = __hadd2(*reinterpret_cast<__half2*>(&a), m1032);
    __half2 hb = __hfma2(*reinterpret_cast<__half2*>(&b), inv16, n72);
    __half2 he = __hadd2(*reinterpret_cast<__half2*>(&e), m1032);
    __half2 hf = __hfma2(*reinterpret_cast<__half2*>(&f), inv16, n72);
    // (e0, e4), (e1, e5), (e2, e6), (e3, e7)
    o.x = *reinterpret_cast<uint32_t*>(&ha);
    o.y = *reinterpret_cast<uint32_t*>(&hb);
    o.z = *reinterpret_cast<uint32_t*>(&he);
    o.w = *reinterpret_cast<uint32_t*>(&hf);
  } else {
    const uint2 w = ok ? *reinterpret_cast<const uint2*>(src) : make_uint2(0, 0);
    const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
    const uint32_t a = w.x ^ 0x80808080u, b = w.y ^ 0x80808080u;
    uint32_t h[4] = {__byte_perm(a, kBytes64, 0x4140), __byte_perm(a, kBytes64, 0x4342), __byte_perm(b, kBytes64, 0x4140),
                     __byte_perm(b, kBytes64, 0x4342)};
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      __half2 v = __hsub2(*reinterpret_cast<__half2*>(&h[i]), off);  // 1024 + (c + 128) - 1152 = c, exactly
      r[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    o = make_uint4(r[0], r[1], r[2], r[3]);
  }
  return o;
}

__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_bounded(bar, parity)) return true;
  flag(status, KV_INT4_DEV_TIMEOUT);
  return false;
}

template <int D, int FMT>
__global__ void __launch_bounds__(128, 1) prefill_tc_kernel(PreParams prm) {
  using G = TcPreGeom<D, FMT>;
  constexpr bool ROT = FMT == kFmtInt4;
  constexpr int B = Head<D>::b;
  constexpr int KSTEPS = D / 16;
  constexpr int NK = G::NK, ROWS = G::ROWS;
  constexpr uint32_t IDESC_S = umma_idesc_f16(ROWS, NK, false);
  constexpr uint32_t IDESC_O = umma_idesc_f16(ROWS, D, true);
  const Common& c = prm.c;
  const PlanView& pv = prm.pv;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* const sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const sQ = sm;
  uint8_t* const sK = sQ + G::QBYTES;
  uint8_t* const sP = sK;  // after S
  uint8_t* const sV = sK + G::KPBYTES;
  uint8_t* const stg = sV + G::KVBYTES;
  float* const sks = reinterpret_cast<float*>(stg + G::STG);  // the step's K scales [64], then V scales [64]
  float* const svs = sks + NK;
  // [4] block usable (copy of the staged flags), then [2] per-warp vote "every V scale of the step is below 128"
  int* const sflag = reinterpret_cast<int*>(svs + NK);
  float* const ssign = reinterpret_cast<float*>(sflag + 8);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(ssign + D);  // S done, O' done
  uint32_t* const tslot = reinterpret_cast<uint32_t*>(bars + 2);
  int* const sitem = reinterpret_cast<int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < D; i += 128) ssign[i] = (ROT && c.signs[i] < 0) ? -1.f : 1.f;
  const uint32_t bar_s = smem_addr(&bars[0]), bar_o = smem_addr(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tslot), G::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem, tO = tmem + NK;
  uint32_t ph_s = 0, ph_o = 0;
  bool o_pending = false;  // an O' MMA group was committed and not yet waited for
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
    if (item.x < 0) break;
    const int seq = item.x, h = item.y, tile = item.z, nkb = item.w;
    const int q0 = c.qsl[seq], ql = c.qsl[seq + 1] - q0;
    const int L = c.seq_lens[seq], ctx = L - ql;
    const int tok0 = tile * c.tile_tokens;
    const int ntok = min(c.tile_tokens, ql - tok0);
    const int nrows = ntok * c.group;
    const int kb0 = window_lo(c, ctx + tok0) >> 4;  // blocks before the earliest row's window are skipped
    const int nsteps = (nkb - kb0 + 3) / 4;

    // this thread's query row: Q' tile row, key range [lo, lim)
    const int r = tid;
    const int j = r / c.group, jj = r - j * c.group;
    const bool rok = r < nrows;
    {
      const __half* src = pv.qrot + ((long long)(q0 + tok0 + (rok ? j : 0)) * c.hq + h * c.group + (rok ? jj : 0)) * D;
#pragma unroll 4
      for (int ch = 0; ch < D / 8; ch++) {
        uint4 v = rok ? reinterpret_cast<const uint4*>(src)[ch] : make_uint4(0, 0, 0, 0);
        if constexpr (FMT == kFmtInt4) {
          // the tiles' nibble order: (q0, q4), (q1, q5), (q2, q6), (q3, q7)
          v = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                         __byte_perm(v.y, v.w, 0x7632));
        }
        *reinterpret_cast<uint4*>(sQ + sw128(ROWS, r, ch)) = v;
      }
    }
    const int qp = ctx + tok0 + (rok ? j : 0);
    const int lim = c.causal ? min(L, qp + 1) : L;
    const int lo = window_lo(c, qp);
    float m_ref = -INFINITY, l_run = 0.f;  // exponent reference of the row, sum of its weights

    // stage the codes, scales and block flags of step `st` (four 16-key
    // blocks): thread (block b4, K/V, row) copies one code row and its scale
    auto issue = [&](int st) {
      const int b4 = tid >> 5, kv = (tid >> 4) & 1, row = tid & 15;
      const int kb = kb0 + st * 4 + b4;
      const int blk = kb < nkb ? c.block_table[(long long)seq * c.max_blocks + kb] : -1;
      const bool ok = kb < nkb && blk >= 0 && blk < c.num_blocks;
      if (ok) {
        const uint8_t* src = (kv ? c.v_cache : c.k_cache) + (long long)blk * c.geo.cblk + row * c.geo.crow +
                             (long long)h * c.geo.chead;
        uint8_t* dst = stg + ((b4 * 2 + kv) * 16 + row) * G::CB;
#pragma unroll
        for (int col = 0; col < G::CB / 16; col++) cp_async16(dst + col * 16, src + col * 16);
        cp_async4(stg + G::SC_OFF + ((b4 * 2 + kv) * 16 + row) * 4,
                  (kv ? c.v_scale : c.k_scale) + (long long)blk * c.geo.sblk + row * c.geo.srow +
                      (long long)h * c.geo.shead);
      }
      if (kv == 0 && row == 0) {
        reinterpret_cast<int*>(stg + G::FL_OFF)[b4] = ok;
        if (kb < nkb && !ok) flag(c.status, KV_INT4_DEV_BAD_BLOCK);
      }
    };

    issue(0);
    cp_async_commit();
#pragma unroll 1
    for (int st = 0; st < nsteps; st++) {
      cp_async_wait<0>();
      // the previous O' MMAs read sV and sP (the K tile): done before they are rewritten
      if (o_pending) {
        mbar_wait_spin(bar_o, ph_o, c.status);
        ph_o ^= 1;
        o_pending = false;
      }
      __syncthreads();
      const uint8_t* sb = stg;
      const int* sfl = reinterpret_cast<const int*>(sb + G::FL_OFF);
      // the step's scales and flags outlive the staging (refilled below)
      if (tid < NK) {
        const float vsc = reinterpret_cast<const float*>(sb + G::SC_OFF)[(tid >> 4) * 32 + 16 + (tid & 15)];
        sks[tid] = reinterpret_cast<const float*>(sb + G::SC_OFF)[(tid >> 4) * 32 + (tid & 15)];
        svs[tid] = vsc;
        // unusable blocks' stale scales count too: the vote only ever errs towards tau = 0
        const bool small = __all_sync(0xffffffffu, fabsf(vsc) < 128.f);
        if ((tid & 31) == 0) sflag[4 + warp] = small;
      } else if (tid < NK + 4) {
        sflag[tid - NK] = sfl[tid - NK];
      }
      const int fmask = (sfl[0] != 0) | (sfl[1] != 0) << 1 | (sfl[2] != 0) << 2 | (sfl[3] != 0) << 3;
      // dequantise the step's K and V codes into the swizzled f16 tiles
      constexpr int CPK = D / 8;                               // 16-byte f16 chunks per key
      constexpr int CBYTES = FMT == kFmtInt8 ? 8 : 4;          // code bytes of 8 elements
#pragma unroll 4
      for (int q = tid; q < NK * CPK; q += 128) {
        const int k = q / CPK, ch = q - k * CPK;
        const int b4 = k >> 4;
        const bool ok = (fmask >> b4) & 1;
        const uint8_t* ksrc = sb + (b4 * 16 + k) * G::CB + ch * CBYTES;  // row (b4, K, k & 15)
        const uint32_t off = sw128(NK, k, ch);
        *reinterpret_cast<uint4*>(sK + off) = dequant8<FMT>(ksrc, ok);
        *reinterpret_cast<uint4*>(sV + off) = dequant8<FMT>(ksrc + 16 * G::CB, ok);
      }
      fence_proxy_async_smem();  // the tiles are read by the tensor cores
      tc_fence_before();
      __syncthreads();
      // the staging is free: fetch the next step's codes while this one computes
      if (st + 1 < nsteps) issue(st + 1);
      cp_async_commit();
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ks++)
          umma_f16(tS, umma_desc(smem_addr(sQ) + (ks >> 2) * ROWS * 128 + (ks & 3) * 32, 16, 1024),
                   umma_desc(smem_addr(sK) + (ks >> 2) * NK * 128 + (ks & 3) * 32, 16, 1024), IDESC_S, ks > 0);
        umma_commit(bar_s);
      }
      mbar_wait_spin(bar_s, ph_s, c.status);
      ph_s ^= 1;
      tc_fence_after();

      // ---- online softmax of this thread's row over the step's 64 keys ----
      float sv[NK];
      {
        float t0[32], t1[32];
        tmem_ld32(tS + lane_off, t0);
        tmem_ld32(tS + lane_off + 32, t1);
#pragma unroll
        for (int k = 0; k < 32; k++) {
          sv[k] = t0[k];
          sv[32 + k] = t1[k];
        }
      }
      const int pos0 = (kb0 + st * 4) * 16;
      const float tau = (sflag[4] && sflag[5]) ? 8.f : 0.f;
      // a step wholly inside the row's visible range over usable blocks needs no mask
      const bool full = pos0 >= lo && pos0 + NK <= lim && sflag[0] && sflag[1] && sflag[2] && sflag[3];
      const float4* ks4 = reinterpret_cast<const float4*>(sks);
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int k = 0; k < NK; k += 4) {
          const float4 f = ks4[k / 4];
          const float2 a = __fmul2_rn(make_float2(sv[k], sv[k + 1]), make_float2(f.x, f.y));
          const float2 b = __fmul2_rn(make_float2(sv[k + 2], sv[k + 3]), make_float2(f.z, f.w));
          sv[k] = a.x; sv[k + 1] = a.y; sv[k + 2] = b.x; sv[k + 3] = b.y;
          mx4[0] = fmaxf(mx4[0], a.x); mx4[1] = fmaxf(mx4[1], a.y);
          mx4[2] = fmaxf(mx4[2], b.x); mx4[3] = fmaxf(mx4[3], b.y);
        }
      } else {
#pragma unroll
        for (int k = 0; k < NK; k++) {
          const int pos = pos0 + k;
          const bool vis = sflag[k >> 4] != 0 && pos >= lo && pos < lim;
          sv[k] = vis ? sv[k] * sks[k] : -INFINITY;
          mx4[k & 3] = fmaxf(mx4[k & 3], sv[k]);
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // the reference moves when the row max passes it by more than tau; a
      // row with no visible key so far (O' = 0, l = 0) takes the max as is
      const bool grow = m_ref != -INFINITY && mx > m_ref + tau;
      const float alpha = grow ? fast_exp2(m_ref - mx) : 1.f;
      if (grow || m_ref == -INFINITY) m_ref = mx;
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; cc++) {
          float o[32];
          tmem_ld32(tO + lane_off + cc * 32, o);
#pragma unroll
          for (int i = 0; i < 32; i++) o[i] *= alpha;
          tmem_st32(tO + lane_off + cc * 32, o);
        }
      }
      l_run *= alpha;
      uint32_t pk[NK / 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      const float4* vs4 = reinterpret_cast<const float4*>(svs);
      if (full) {
        // every key visible: no selects
        const float2 nm = make_float2(-m_ref, -m_ref);
#pragma unroll
        for (int k = 0; k < NK; k += 4) {
          const float4 f = vs4[k / 4];
          const float2 da = __fadd2_rn(make_float2(sv[k], sv[k + 1]), nm);
          const float2 db = __fadd2_rn(make_float2(sv[k + 2], sv[k + 3]), nm);
          const float2 pa = make_float2(fast_exp2(da.x), fast_exp2(da.y));
          const float2 pb = make_float2(fast_exp2(db.x), fast_exp2(db.y));
          ps[0] += pa.x; ps[1] += pa.y; ps[2] += pb.x; ps[3] += pb.y;
          const float2 wa = __fmul2_rn(pa, make_float2(f.x, f.y));
          const float2 wb = __fmul2_rn(pb, make_float2(f.z, f.w));
          pk[k / 2] = pack_f16x2(wa.x, wa.y);
          pk[k / 2 + 1] = pack_f16x2(wb.x, wb.y);
        }
      } else {
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
        for (int k = 0; k < NK; k += 2) {
          const float p0 = sv[k] == -INFINITY ? 0.f : fast_exp2(sv[k] - mu);
          const float p1 = sv[k + 1] == -INFINITY ? 0.f : fast_exp2(sv[k + 1] - mu);
          ps[k & 3] += p0;
          ps[(k & 3) + 1] += p1;
          // masked keys may carry unwritten (NaN) scales: select, do not multiply
          const float w0 = p0 == 0.f ? 0.f : p0 * svs[k];
          const float w1 = p1 == 0.f ? 0.f : p1 * svs[k + 1];
          pk[k / 2] = pack_f16x2(w0, w1);
        }
      }
      l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
#pragma unroll
      for (int cc = 0; cc < 8; cc++)
        *reinterpret_cast<uint4*>(sP + r * 128 + ((cc ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; kk++)
          umma_f16(tO, umma_desc(smem_addr(sP) + kk * 32, 16, 1024),
                   umma_desc(smem_addr(sV) + kk * 2048, NK * 128, 1024), IDESC_O, st > 0 || kk > 0);
        umma_commit(bar_o);
      }
      o_pending = true;
    }
    cp_async_wait<0>();

    // ---- epilogue: normalise, inverse rotation (INT4), bf16 store ----
    if (o_pending) {
      mbar_wait_spin(bar_o, ph_o, c.status);
      ph_o ^= 1;
      o_pending = false;
    }
    tc_fence_after();
    const float inv = l_run > 0.f ? 1.f / (l_run * (ROT ? (float)B : 1.f)) : 0.f;
    uint16_t* dst = c.out + (long long)(q0 + tok0 + (rok ? j : 0)) * c.out_stride + (long long)(h * c.group + jj) * D;
    constexpr int CHUNK = (ROT && B > 32) ? B : 32;  // columns handled together (one Hadamard block)
#pragma unroll 1
    for (int base = 0; base < D; base += CHUNK) {
      float o[CHUNK];
#pragma unroll
      for (int cc = 0; cc < CHUNK / 32; cc++) {
        float t[32];
        tmem_ld32(tO + lane_off + base + cc * 32, t);
#pragma unroll
        for (int i = 0; i < 32; i++) o[cc * 32 + (FMT == kFmtInt4 ? (i & ~7) + nib_order(i & 7) : i)] = t[i];
      }
      if constexpr (ROT) {
        // H_b over each b-block of this chunk (CHUNK is a multiple of b)
#pragma unroll
        for (int hh = 1; hh < B; hh <<= 1) {
#pragma unroll
          for (int i = 0; i < CHUNK; i++) {
            if ((i & hh) == 0) {
              const float a0 = o[i], b0 = o[i + hh];
              o[i] = a0 + b0;
              o[i + hh] = a0 - b0;
            }
          }
        }
      }
      if (rok) {
#pragma unroll
        for (int i = 0; i < CHUNK; i += 8) {
          uint4 w;
          w.x = pack_bf16x2_rn(o[i] * inv * ssign[base + i], o[i + 1] * inv * ssign[base + i + 1]);
          w.y = pack_bf16x2_rn(o[i + 2] * inv * ssign[base + i + 2], o[i + 3] * inv * ssign[base + i + 3]);
          w.z = pack_bf16x2_rn(o[i + 4] * inv * ssign[base + i + 4], o[i + 5] * inv * ssign[base + i + 5]);
          w.w = pack_bf16x2_rn(o[i + 6] * inv * ssign[base + i + 6], o[i + 7] * inv * ssign[base + i + 7]);
          *reinterpret_cast<uint4*>(dst + base + i) = w;
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM, sQ and the staging may be reused by the next tile
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, G::TMEM_COLS);
}
