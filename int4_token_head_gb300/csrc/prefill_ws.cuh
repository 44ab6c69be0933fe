// Warp-specialised prefill on the 5th-generation tensor cores (tcgen05),
// included by attention.cu after the schedule and parameter types it uses.
//
// One CTA per SM (all 512 TMEM columns), one item = 256 query rows
// (query token x q head of one kv group) in two halves of 128, the MMA's M;
// 64 keys (four cache blocks) per step.  Sixteen warps in three roles, each
// role running its own item loop so that a register budget can be set per
// warpgroup (softmax 160 a thread, the others 96); the roles meet only at
// mbarriers, so that the next item starts while the current one's epilogue
// runs:
//   * dequant warps (8-14): claim the next item (longest first) and pass it
//     to the other roles through a two-entry ring; stage the step's code rows
//     and scales with cp.async into one of two staging buffers (block ids
//     loaded a step ahead), load the item's Q' rows once every score MMA of
//     the previous item is complete, dequantise K into one of two f16 tiles
//     (one where shared memory is short) and V into one of two, exactly (an
//     INT4 nibble u becomes the f16 pattern 0x6400 | u = 1024 + u, an int8
//     byte u the pattern 0x64uu), and copy the step's K/V scales, block flags
//     and the V-scale vote into a three-entry ring;
//   * MMA warp (15, lane 0 issues): S_h = Q_h K^T into TMEM columns
//     [64h, 64h + 64); O_h += P_h V with P_h read from TMEM (the A operand
//     of the MMA may live in tensor memory) into columns
//     [128 + hD, 128 + (h+1)D).  Issue order S0 S1 | PV0 S0' | PV1 S1' | ...
//     lets each half's softmax run while the other half's MMAs do;
//   * softmax warps (0-3 for half 0, 4-7 for half 1): one query row per
//     thread, a masked base-2 online softmax whose exponent reference m_ref
//     moves (and the row's O in TMEM is rescaled) only when the row max
//     passes m_ref + tau: tau = 8 while every V scale of the step's
//     existing keys is below 128, so p <= 2^8 keeps P' below 2^15 in f16,
//     else tau = 0 (the exact running max); P' = p * v_scale is written back
//     as f16 pairs over the row's S columns.  The epilogue normalises O,
//     applies D (I_n (x) H_b) (.) / b in registers (packed f32x2 butterflies)
//     and writes the bf16 rows straight from registers (where the transform
//     comes in 64-column groups, each lane quad first transposes its 32-byte
//     units so that one store writes a 128-byte run per quad), leaving
//     shared memory to the next item.
// INT4 tiles keep each 8-element group in nibble order (elements 0,4,1,5,
// 2,6,3,7: the two nibble lanes of a 32-bit word per f16x2, no byte
// shuffles); the prep kernel stores Q' with the same permutation, which
// leaves Q' K^T unchanged, and the epilogue undoes it on O (its columns are
// V's dims) by register renaming.
// Shared-memory operands: K-major tiles are [D/64 blocks][rows][128 bytes]
// with the 16-byte chunk index XORed by row % 8 (1024-byte atoms; leading
// byte offset unused, stride byte offset 1024); the V tiles use the same
// layout as MN-major operands (dims are the MMA's N: leading byte offset =
// one 64-dim block = 64 keys x 128 bytes, stride byte offset = 8 keys).
// Hand-offs are mbarriers (every wait bounded; a wait that runs out sets
// KV_INT4_DEV_TIMEOUT and a CTA-wide abort flag that ends every later
// wait at once, so a fault in the pipeline costs one time-out, not one
// per step).  Each comes in a pair, per K/V tile, per half or per item ring
// entry, so that no barrier can complete twice before its waiter has seen
// the first:
//   ifull[e] (dequant -> MMA, softmax)  item ring entry e written
//   ifree[e] (MMA, softmax -> dequant)  item ring entry e read
//   kfull[b] (dequant -> MMA)  K tile b and the step's ring entry written
//                              (for an item's first step also its Q' rows)
//   vfull[b] (dequant -> MMA)  V tile b written
//   kfree[b] (MMA commit -> dequant) S0 and S1 that read K tile b complete
//   vfree[b] (MMA commit -> dequant) PV0 and PV1 that read V tile b complete
//   sfull[h] (MMA commit -> softmax h) S_h complete (and every earlier MMA)
//   pfull[h] (softmax h -> MMA) P_h in TMEM, O_h rescaled if it had to be
//   odone    (MMA commit -> softmax) the item's last PV complete
// The ring entry of step j is rewritten at step j + 3, after S of step
// j + 1 completed, which follows both halves' P of step j.  Across items:
// the next item's Q' rows and K tiles are written once the previous item's
// last S is complete (kfree), its V tiles and first ring entries once the
// previous item's last PV is (vfree: every P, so every softmax read of the
// ring, came before it); its first PV overwrites O only after its first P,
// which the softmax warps write after their epilogue's last TMEM load.

constexpr int kWsRows = 256;  // query rows per item

// byte offset of 16-byte chunk c (elements 8c .. 8c+7) of row r in a
// 128-byte-swizzled K-major tile of `rows` rows: [c / 8][rows][128 bytes],
// the chunk index within a 128-byte row XORed by r % 8
__device__ __forceinline__ uint32_t sw128(int rows, int r, int c) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, int FMT>
struct WsGeom {
  static constexpr int ROWS = kWsRows;
  static constexpr int NK = 64;                       // keys per step
  static constexpr int KB = (D + 63) / 64;            // 128-byte blocks of an f16 head vector
  static constexpr int QBYTES = ROWS * 128 * KB;
  static constexpr int KVBYTES = NK * 128 * KB;       // one K or V tile
  static constexpr int CB = FMT == kFmtInt8 ? D : D / 2;
  // staging: code rows [block][K/V][16] at a stride of an odd number of
  // 16-byte units (eight consecutive rows hit eight bank groups), then
  // scales, then flags
  static constexpr int SROW = CB + ((CB / 16) % 2 == 0 ? 16 : 0);
  static constexpr int SC_OFF = 4 * 2 * 16 * SROW;
  static constexpr int FL_OFF = SC_OFF + 4 * 2 * 16 * 4;
  static constexpr int STG = (FL_OFF + 16 + 127) / 128 * 128;
  static constexpr int RING = 2 * NK * 4 + 32;        // K scales, V scales, 4 block flags, 2 votes
  static constexpr int NRING = 3;                     // ring entries: step j's is rewritten at step j + 3
  static constexpr int TMEM_COLS = 128 + 2 * D <= 256 ? 256 : 512;
  static constexpr int NBARS = 18;
  // item ring [2][4], abort flag, TMEM base
  static constexpr int fixed_bytes(int kbuf) {
    return 1024 + QBYTES + (kbuf + 2) * KVBYTES + 2 * STG + NRING * RING + D * 4 + NBARS * 8 + 48;
  }
  // two K tiles (dequantise K(j + 1) while S(j) runs) where shared memory allows
  static constexpr int KBUF = fixed_bytes(2) <= 227 * 1024 ? 2 : 1;
  static constexpr int USED = fixed_bytes(KBUF);
  static constexpr int SMEM = USED;
  static constexpr int THREADS = 16 * 32;
  static constexpr int DQ_WARPS = 7;  // warps 8 .. 14
  static_assert(D % 32 == 0 && D <= 192, "head sizes served by the warp-specialised prefill");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// a bounded mbarrier wait that gives up at once after any wait of the CTA
// has run out (abort flag set)
__device__ __forceinline__ bool ws_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status) {
  for (int n = 0; n < kMaxWaitIters; n++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255) == 255 && *abort) return false;
  }
  *abort = 1;
  flag(status, KV_INT4_DEV_TIMEOUT);
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// 8 exact f16 values of one 32-bit word of INT4 codes, in nibble order
// (elements 0,4,1,5,2,6,3,7): the low nibbles of bytes (0, 2) become
// 1032 + c exactly (minus 1032), the high ones 1152 + 16c (/ 16 - 72 in one
// rounding of an exact value)
__device__ __forceinline__ uint4 dq_word_int4(uint32_t x) {
  const uint32_t y = x >> 8;
  const uint32_t n1032 = kF16x2_M1032, h16 = 0x2c002c00u, m72 = 0xd480d480u;  // (-1032), (1/16), (-72)
  const __half2 m1032 = *reinterpret_cast<const __half2*>(&n1032);
  const __half2 inv16 = *reinterpret_cast<const __half2*>(&h16), n72 = *reinterpret_cast<const __half2*>(&m72);
  uint32_t a = nib_lo(x), b = nib_hi(x), e = nib_lo(y), f = nib_hi(y);
  __half2 ha = __hadd2(*reinterpret_cast<__half2*>(&a), m1032);
  __half2 hb = __hfma2(*reinterpret_cast<__half2*>(&b), inv16, n72);
  __half2 he = __hadd2(*reinterpret_cast<__half2*>(&e), m1032);
  __half2 hf = __hfma2(*reinterpret_cast<__half2*>(&f), inv16, n72);
  return make_uint4(*reinterpret_cast<uint32_t*>(&ha), *reinterpret_cast<uint32_t*>(&hb),
                    *reinterpret_cast<uint32_t*>(&he), *reinterpret_cast<uint32_t*>(&hf));
}
// 8 exact f16 values of two words of int8 codes, natural order: the byte
// c + 128 paired with 0x64 is 1024 + (c + 128); minus 1152
__device__ __forceinline__ uint4 dq_pair_int8(uint32_t wx, uint32_t wy) {
  const uint32_t a = wx ^ 0x80808080u, b = wy ^ 0x80808080u, m1152 = kF16x2_M1152;
  const __half2 off = *reinterpret_cast<const __half2*>(&m1152);
  uint32_t h[4] = {__byte_perm(a, kBytes64, 0x4140), __byte_perm(a, kBytes64, 0x4342), __byte_perm(b, kBytes64, 0x4140),
                   __byte_perm(b, kBytes64, 0x4342)};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    __half2 v = __hadd2(*reinterpret_cast<__half2*>(&h[i]), off);
    r[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// per-thread register budget of the calling warpgroup (all four warps execute it)
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }

// named barrier over the dequant warps only
__device__ __forceinline__ void dq_sync() { asm volatile("bar.sync 1, 224;\n" ::: "memory"); }

template <int D, int FMT>
__global__ void __launch_bounds__(16 * 32, 1) prefill_ws_kernel(PreParams prm) {
  using G = WsGeom<D, FMT>;
  constexpr bool ROT = FMT == kFmtInt4;
  constexpr int B = Head<D>::b;
  constexpr int KSTEPS = D / 16;
  constexpr int NK = G::NK, ROWS = G::ROWS;
  constexpr uint32_t IDESC_S = umma_idesc_f16(128, NK, false);
  constexpr uint32_t IDESC_O = umma_idesc_f16(128, D, true);
  const Common& c = prm.c;
  const PlanView& pv = prm.pv;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* const sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const sQ = sm;                     // [KB][256 rows][128 B], swizzled
  uint8_t* const sK = sQ + G::QBYTES;         // KBUF K tiles [KB][64 keys][128 B]
  uint8_t* const sV = sK + G::KBUF * G::KVBYTES;  // two V tiles
  uint8_t* const stg = sV + 2 * G::KVBYTES;   // two staging buffers
  uint8_t* const ring = stg + 2 * G::STG;     // two entries: K scales [64], V scales [64], flags [4], votes [2]
  float* const ssign = reinterpret_cast<float*>(ring + G::NRING * G::RING);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(ssign + D);
  int* const sitem = reinterpret_cast<int*>(bars + G::NBARS);  // item ring [2][4], abort flag
  uint32_t* const tslot = reinterpret_cast<uint32_t*>(sitem + 10);
  volatile int* const abort_flag = sitem + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // barrier indices
  // two of each pair: per K/V tile (full, free) or per half (S, P); every
  // barrier is waited once per completion, in order
  enum { KFULL = 0, VFULL = 2, KFREE = 4, VFREE = 6, SFULL = 8, PFULL = 10, ODONE = 12, DRAIN = 13, IFULL = 14, IFREE = 16 };
  auto bar = [&](int i) { return smem_addr(&bars[i]); };
  for (int i = tid; i < D; i += G::THREADS) ssign[i] = (ROT && c.signs[i] < 0) ? -1.f : 1.f;
  if (tid == 0) {
    mbar_init(bar(KFULL), G::DQ_WARPS);
    mbar_init(bar(KFULL + 1), G::DQ_WARPS);
    mbar_init(bar(VFULL), G::DQ_WARPS);
    mbar_init(bar(VFULL + 1), G::DQ_WARPS);
    mbar_init(bar(KFREE), 1);
    mbar_init(bar(KFREE + 1), 1);
    mbar_init(bar(VFREE), 1);
    mbar_init(bar(VFREE + 1), 1);
    mbar_init(bar(SFULL), 1);
    mbar_init(bar(SFULL + 1), 1);
    mbar_init(bar(PFULL), 4);
    mbar_init(bar(PFULL + 1), 4);
    mbar_init(bar(ODONE), 1);
    mbar_init(bar(DRAIN), 1);
    mbar_init(bar(IFULL), 1);
    mbar_init(bar(IFULL + 1), 1);
    mbar_init(bar(IFREE), 9);  // the eight softmax warps and the MMA warp
    mbar_init(bar(IFREE + 1), 9);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tslot), G::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // registers: the launch gives 128 a thread to all four warpgroups (65,536);
  // the softmax warpgroups take 160, the dequant/MMA ones keep 96
  // (2 x 128 x 160 + 2 x 128 x 96 = 65,536: the increase can always be met)
  const int n_items = pv.plan[1];
  // each role runs its own item loop (the same items, handed over through
  // the item ring), so that the register budget set for its warpgroups
  // covers only its own code
  static_assert(G::THREADS == 512, "four warpgroups");
  auto item_at = [&](int e) { return make_int4(sitem[4 * e], sitem[4 * e + 1], sitem[4 * e + 2], sitem[4 * e + 3]); };
  // a consumer's wait for ring entry e, warp-uniform (a wait that gives up
  // on the abort flag may do so in some lanes only)
  auto take_item = [&](int e, uint32_t& ph, int4& item) {
    const bool ok = __all_sync(0xffffffffu, ws_wait(bar(IFULL + e), (ph >> e) & 1, abort_flag, c.status));
    ph ^= 1u << e;
    if (!ok) return false;
    item = item_at(e);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(IFREE + e));
    return item.x >= 0;
  };
  if (warp < 8) {
    // ======================= softmax warpgroups =======================
    regs_inc<160>();
    // phase bits of the barriers the role waits on (one completion per wait)
    uint32_t ph_sfull = 0, ph_odone = 0, ph_ifull = 0;
#pragma unroll 1
    for (int itc = 0;; itc++) {
      int4 item;
      if (!take_item(itc & 1, ph_ifull, item)) break;
      const int seq = item.x, h = item.y, tile = item.z, nkb = item.w;
      const int q0 = c.qsl[seq], ql = c.qsl[seq + 1] - q0;
      const int L = c.seq_lens[seq], ctx = L - ql;
      const int tok0 = tile * c.tile_tokens;
      const int ntok = min(c.tile_tokens, ql - tok0);
      const int nrows = ntok * c.group;
      const int kb0 = window_lo(c, ctx + tok0) >> 4;  // blocks before the earliest row's window are skipped
      const int nsteps = (nkb - kb0 + 3) / 4;
      // ================= softmax warps: half hf, one query row per thread =================
      const int hf = warp >> 2;
      const int r = tid;  // row of the item (half hf holds rows [128 hf, 128 hf + 128))
      const int j = (int)c.gdiv.div((uint32_t)r);  // token of the row within the item
      const bool rok = r < nrows;
      const int qp = ctx + tok0 + (rok ? j : 0);
      const int lim = c.causal ? min(L, qp + 1) : L;
      const int lo = window_lo(c, qp);
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + 64 * hf + lane_off, tO = tmem + 128 + hf * D + lane_off;
      float m_ref = -INFINITY, l_run = 0.f;  // exponent reference of the row, sum of its weights
#pragma unroll 1
      for (int st = 0; st < nsteps; st++) {
        const uint8_t* re = ring + (st % G::NRING) * G::RING;
        const float* sks = reinterpret_cast<const float*>(re);
        const float* svs = sks + NK;
        const int* sfl = reinterpret_cast<const int*>(re + 2 * NK * 4);
        ws_wait(bar(SFULL + hf), ph_sfull, abort_flag, c.status);
        ph_sfull ^= 1;
        tc_fence_after();
        float sv[NK];
        {
          float t0[32], t1[32];
          tmem_ld32(tS, t0);
          tmem_ld32(tS + 32, t1);
#pragma unroll
          for (int k = 0; k < 32; k++) {
            sv[k] = t0[k];
            sv[32 + k] = t1[k];
          }
        }
        const int pos0 = (kb0 + st * 4) * 16;
        const float tau = (sfl[4] && sfl[5]) ? 8.f : 0.f;
        // a step wholly inside the row's visible range over usable blocks needs no mask
        const bool full = pos0 >= lo && pos0 + NK <= lim && sfl[0] && sfl[1] && sfl[2] && sfl[3];
        const float4* ks4 = reinterpret_cast<const float4*>(sks);
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (full) {
#pragma unroll
          for (int k = 0; k < NK; k += 4) {
            const float4 f = ks4[k / 4];
            const float2 a = __fmul2_rn(make_float2(sv[k], sv[k + 1]), make_float2(f.x, f.y));
            const float2 bb = __fmul2_rn(make_float2(sv[k + 2], sv[k + 3]), make_float2(f.z, f.w));
            sv[k] = a.x; sv[k + 1] = a.y; sv[k + 2] = bb.x; sv[k + 3] = bb.y;
            mx4[(k >> 2) & 1] = fmax3(mx4[(k >> 2) & 1], a.x, a.y);
            mx4[2 + ((k >> 2) & 1)] = fmax3(mx4[2 + ((k >> 2) & 1)], bb.x, bb.y);
          }
        } else {
#pragma unroll
          for (int k = 0; k < NK; k++) {
            const int pos = pos0 + k;
            const bool vis = sfl[k >> 4] != 0 && pos >= lo && pos < lim;
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
          // O' of this half is complete up to the previous step (S_h of this step was issued after it)
#pragma unroll 1
          for (int cc = 0; cc < D / 32; cc++) {
            float o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; i++) o[i] *= alpha;
            tmem_st32(tO + cc * 32, o);
          }
        }
        l_run *= alpha;
        float pf[NK / 2];  // P' as f16 pairs (bit patterns)
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float4* vs4 = reinterpret_cast<const float4*>(svs);
        if (full) {
          const float2 nm = make_float2(-m_ref, -m_ref);
#pragma unroll
          for (int k = 0; k < NK; k += 4) {
            const float4 f = vs4[k / 4];
            const float2 da = __fadd2_rn(make_float2(sv[k], sv[k + 1]), nm);
            const float2 db = __fadd2_rn(make_float2(sv[k + 2], sv[k + 3]), nm);
            const float2 pa = make_float2(fast_exp2(da.x), fast_exp2(da.y));
            const float2 pb = make_float2(fast_exp2(db.x), fast_exp2(db.y));
            ps2[0] = f2add(ps2[0], pa);
            ps2[1] = f2add(ps2[1], pb);
            const float2 wa = __fmul2_rn(pa, make_float2(f.x, f.y));
            const float2 wb = __fmul2_rn(pb, make_float2(f.z, f.w));
            pf[k / 2] = __uint_as_float(pack_f16x2(wa.x, wa.y));
            pf[k / 2 + 1] = __uint_as_float(pack_f16x2(wb.x, wb.y));
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
            pf[k / 2] = __uint_as_float(pack_f16x2(w0, w1));
          }
        }
        l_run += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps2[0].x + ps2[0].y) + (ps2[1].x + ps2[1].y));
        tmem_st32(tS, pf);  // P' over the row's first 32 S columns (S is consumed)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(PFULL + hf));
      }

      // ---- epilogue: normalise, inverse rotation (INT4), bf16 store ----
      ws_wait(bar(ODONE), ph_odone, abort_flag, c.status);
      ph_odone ^= 1;
      tc_fence_after();
      const bool live = l_run > 0.f;  // a row that saw no usable key is written as zeros
      const float inv = live ? 1.f / (l_run * (ROT ? (float)B : 1.f)) : 0.f;
      // The output leaves straight from registers (shared memory is left to
      // the next item, whose Q' and first tiles load meanwhile).  A thread
      // holds its row, and the rows of a lane quad are the group's q heads of
      // one token (contiguous when the group has four heads): where a whole
      // 64-column group is transformed at once, the quad transposes its
      // 32-byte units so that each store instruction writes a full 128-byte
      // run per quad; elsewhere a thread stores its own row 32 bytes at a time.
      uint16_t* const orow =
          c.out + (long long)(q0 + tok0 + (rok ? j : 0)) * c.out_stride + (long long)(h * c.group + (rok ? r - j * c.group : 0)) * D;
      const int qi = lane & 3;  // position in the lane quad
      // the output rows start on 32-byte boundaries (else two 16-byte stores)
      const bool al32 = ((reinterpret_cast<uintptr_t>(c.out) | (uintptr_t)(c.out_stride * 2) | (uintptr_t)(D * 2)) & 31) == 0;
      auto st32 = [&](uint16_t* dst, const uint4& a, const uint4& b) {
        if (al32) {
          asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(dst), "r"(a.x), "r"(a.y), "r"(a.z),
                       "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                       : "memory");
        } else {
          reinterpret_cast<uint4*>(dst)[0] = a;
          reinterpret_cast<uint4*>(dst)[1] = b;
        }
      };
      // bf16 words of the 8 outputs from column col: normalised, signs
      // applied, zeros for a row that saw no usable key
      auto cvt8 = [&](int col, const float* y) {
        const float4 s0 = *reinterpret_cast<const float4*>(ssign + col);
        const float4 s1 = *reinterpret_cast<const float4*>(ssign + col + 4);
        const float2 iv = make_float2(inv, inv);
        const float2 z0 = __fmul2_rn(__fmul2_rn(make_float2(y[0], y[1]), iv), make_float2(s0.x, s0.y));
        const float2 z1 = __fmul2_rn(__fmul2_rn(make_float2(y[2], y[3]), iv), make_float2(s0.z, s0.w));
        const float2 z2 = __fmul2_rn(__fmul2_rn(make_float2(y[4], y[5]), iv), make_float2(s1.x, s1.y));
        const float2 z3 = __fmul2_rn(__fmul2_rn(make_float2(y[6], y[7]), iv), make_float2(s1.z, s1.w));
        const uint4 w = make_uint4(pack_bf16x2_rn(z0.x, z0.y), pack_bf16x2_rn(z1.x, z1.y), pack_bf16x2_rn(z2.x, z2.y),
                                   pack_bf16x2_rn(z3.x, z3.y));
        return live ? w : make_uint4(0, 0, 0, 0);
      };
      // 16 outputs from column col (a multiple of 16) of this thread's row
      auto put16 = [&](int col, const float (&y)[16]) {
        const uint4 a = cvt8(col, y), b = cvt8(col + 8, y + 8);
        if (rok) st32(orow + col, a, b);
      };
      // TMEM column slot of natural element i within a chunk: INT4 columns are
      // in nibble order, so elements i and i + 4 (i % 8 < 4) sit in slots s, s + 1
      auto slot = [](int i) { return FMT == kFmtInt4 ? (i & ~7) + (i & 3) * 2 + ((i >> 2) & 1) : i; };
      constexpr int CHUNK = (ROT && B > 32) ? (B > 64 ? 64 : B) : 32;  // columns transformed in registers
      constexpr bool QUAD = CHUNK == 64 && !(ROT && B > 64);              // whole 64-column groups stored here
      // the quad's rows (lane quad position t): output row, or null past the item's rows
      uint16_t* qrow[4];
#pragma unroll
      for (int t = 0; t < 4; t++) {
        const unsigned long long pr = rok ? reinterpret_cast<unsigned long long>(orow) : 0ull;
        qrow[t] = reinterpret_cast<uint16_t*>(__shfl_sync(0xffffffffu, pr, (lane & ~3) | t));
      }
#pragma unroll 1
      for (int base = 0; base < D; base += CHUNK) {
        float o[CHUNK];  // TMEM column order
#pragma unroll
        for (int cc = 0; cc < CHUNK / 32; cc++) tmem_ld32(tO + base + cc * 32, *reinterpret_cast<float(*)[32]>(o + cc * 32));
        if constexpr (ROT) {
          // H over each CHUNK-block (H_b itself when b <= 64): the stride-4
          // level pairs the two halves of a slot pair, every other level
          // pairs slot pairs with packed f32x2 arithmetic
#pragma unroll
          for (int hh = 1; hh < (B < CHUNK ? B : CHUNK); hh <<= 1) {
            if (hh == 4) {
#pragma unroll
              for (int i = 0; i < CHUNK; i++) {
                if ((i & 4) == 0) {
                  const float a0 = o[slot(i)], b0 = o[slot(i + 4)];
                  o[slot(i)] = a0 + b0;
                  o[slot(i + 4)] = a0 - b0;
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < CHUNK; i++) {
                if ((i & hh) == 0 && (i & 4) == 0) {
                  const int sa = slot(i), sb = slot(i + hh);
                  const float2 x = make_float2(o[sa], o[sa + 1]), y = make_float2(o[sb], o[sb + 1]);
                  const float2 u = f2add(x, y), v = f2sub(x, y);
                  o[sa] = u.x; o[sa + 1] = u.y;
                  o[sb] = v.x; o[sb + 1] = v.y;
                }
              }
            }
          }
        }
        if constexpr (ROT && B > 64) {
          // b = 128: park the H_64 halves in TMEM in natural order for the last stage
          float nat[CHUNK];
#pragma unroll
          for (int i = 0; i < CHUNK; i++) nat[i] = o[slot(i)];
#pragma unroll
          for (int cc = 0; cc < CHUNK / 32; cc++) tmem_st32(tO + base + cc * 32, *reinterpret_cast<float(*)[32]>(nat + cc * 32));
        } else if constexpr (QUAD) {
          // u[t]: 32-byte unit t (columns base + 16 t ..) of this thread's row
          uint4 u[4][2];
#pragma unroll
          for (int t = 0; t < 4; t++) {
            float y[16];
#pragma unroll
            for (int e = 0; e < 16; e++) y[e] = o[slot(16 * t + e)];
            u[t][0] = cvt8(base + 16 * t, y);
            u[t][1] = cvt8(base + 16 * t + 8, y + 8);
          }
          // 4 x 4 transpose over the quad (row = quad position, column =
          // unit), by two exchanges with the partners at xor 1 and xor 2:
          // afterwards u[t] is unit qi of the quad's row t
#pragma unroll
          for (int x = 1; x <= 2; x <<= 1) {
            const bool hi = (qi & x) != 0;
#pragma unroll
            for (int a = 0; a < 4; a++) {
              if (a & x) continue;  // pairs (a, a + x)
#pragma unroll
              for (int k = 0; k < 2; k++) {
                const uint4 snd = hi ? u[a][k] : u[a + x][k];
                uint4 rcv;
                rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, x);
                rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, x);
                rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, x);
                rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, x);
                if (hi) u[a][k] = rcv;
                else u[a + x][k] = rcv;
              }
            }
          }
#pragma unroll
          for (int t = 0; t < 4; t++)
            if (qrow[t] != nullptr) st32(qrow[t] + base + 16 * qi, u[t][0], u[t][1]);
        } else {
#pragma unroll
          for (int i = 0; i < CHUNK; i += 16) {
            float y[16];
#pragma unroll
            for (int e = 0; e < 16; e++) y[e] = o[slot(i + e)];
            put16(base + i, y);
          }
        }
      }
      if constexpr (ROT && B > 64) {
        static_assert(B == 128, "the two-pass epilogue takes b = 128");
        // H_128 = (H_2 (x) I_64)(I_2 (x) H_64): pair natural columns i and i + 64 of each 128-block
#pragma unroll 1
        for (int base = 0; base < D; base += 128) {
#pragma unroll 1
          for (int q = 0; q < 64; q += 32) {
            float a[32], b2[32];
            tmem_ld32(tO + base + q, a);
            tmem_ld32(tO + base + 64 + q, b2);
#pragma unroll
            for (int i = 0; i < 32; i += 16) {
              float y0[16], y1[16];
#pragma unroll
              for (int e = 0; e < 16; e++) {
                y0[e] = a[i + e] + b2[i + e];
                y1[e] = a[i + e] - b2[i + e];
              }
              put16(base + q + i, y0);
              put16(base + 64 + q + i, y1);
            }
          }
        }
      }
    }
  } else {
    // ==================== dequant and MMA warpgroups ====================
    regs_dec<96>();
    uint32_t ph_kfull = 0, ph_vfull = 0, ph_kfree = 0, ph_vfree = 0, ph_pfull = 0;
    if (warp < 15) {
      // ================= dequant warps =================
      const int dt = tid - 256;
      uint32_t ph_ifree = 0;
      int prev_steps = 0;  // steps of the previous item
      // the previous item's MMA completions that its step loop did not wait
      // for: the S of its last KBUF steps (and with them every S, so every
      // read of its Q' and K tiles), the last PV of each V tile (and with it
      // every P, so every softmax read of its ring entries)
      auto wait_kfree_tail = [&](int ns) {
        for (int st = ns - G::KBUF < 0 ? 0 : ns - G::KBUF; st < ns; st++) {
          ws_wait(bar(KFREE + (st & 1)), (ph_kfree >> (st & 1)) & 1, abort_flag, c.status);
          ph_kfree ^= 1u << (st & 1);
        }
      };
      auto wait_vfree_tail = [&](int ns) {
        for (int b = 0; b < 2 && b < ns; b++) {
          ws_wait(bar(VFREE + b), (ph_vfree >> b) & 1, abort_flag, c.status);
          ph_vfree ^= 1u << b;
        }
      };
#pragma unroll 1
      for (int itc = 0;; itc++) {
        const int e = itc & 1;
        if (dt == 0) {
          // claim the next item and publish it in ring entry e, whose
          // previous item (itc - 2) every consumer has read
          if (itc >= 2) {
            ws_wait(bar(IFREE + e), (ph_ifree >> e) & 1, abort_flag, c.status);
            ph_ifree ^= 1u << e;
          }
          const int4 it = prefill_item(c, pv, *abort_flag ? n_items : atomicAdd(&pv.plan[2], 1), n_items);
          sitem[4 * e] = it.x;
          sitem[4 * e + 1] = it.y;
          sitem[4 * e + 2] = it.z;
          sitem[4 * e + 3] = it.w;
          mbar_arrive(bar(IFULL + e));
        }
        dq_sync();
        const int4 item = item_at(e);
        if (item.x < 0) {
          wait_kfree_tail(prev_steps);
          wait_vfree_tail(prev_steps);
          break;
        }
        const int seq = item.x, h = item.y, tile = item.z, nkb = item.w;
        const int q0 = c.qsl[seq], ql = c.qsl[seq + 1] - q0;
        const int L = c.seq_lens[seq], ctx = L - ql;
        const int tok0 = tile * c.tile_tokens;
        const int ntok = min(c.tile_tokens, ql - tok0);
        const int nrows = ntok * c.group;
        const int kb0 = window_lo(c, ctx + tok0) >> 4;  // blocks before the earliest row's window are skipped
        const int nsteps = (nkb - kb0 + 3) / 4;
        // staging is done by the first 128 dequant threads: thread (block b4,
        // K/V, row) copies one code row and its scale; the block id of a step
        // is loaded a step before its copies are issued
        auto block_of = [&](int st) -> int {
          const int kb = kb0 + st * 4 + (dt >> 5);
          return (dt < 128 && kb < nkb) ? c.block_table[(long long)seq * c.max_blocks + kb] : -1;
        };
        auto issue = [&](int st, uint8_t* sb, int blk) {
          if (dt >= 128) return;
          const int b4 = dt >> 5, kv = (dt >> 4) & 1, row = dt & 15;
          const int kb = kb0 + st * 4 + b4;
          const bool ok = kb < nkb && blk >= 0 && blk < c.num_blocks;
          if (ok) {
            const uint8_t* src = (kv ? c.v_cache : c.k_cache) + (long long)blk * c.geo.cblk + row * c.geo.crow +
                                 (long long)h * c.geo.chead;
            uint8_t* dst = sb + ((b4 * 2 + kv) * 16 + row) * G::SROW;
#pragma unroll
            for (int col = 0; col < G::CB / 16; col++) cp_async16(dst + col * 16, src + col * 16);
            cp_async4(sb + G::SC_OFF + ((b4 * 2 + kv) * 16 + row) * 4,
                      (kv ? c.v_scale : c.k_scale) + (long long)blk * c.geo.sblk + row * c.geo.srow +
                          (long long)h * c.geo.shead);
          }
          if (kv == 0 && row == 0) {
            reinterpret_cast<int*>(sb + G::FL_OFF)[b4] = ok;
            if (kb < nkb && !ok) flag(c.status, KV_INT4_DEV_BAD_BLOCK);
          }
        };
        // dequantise the K (kv = 0) or V (kv = 1) codes of staging sb into a
        // tile: a thread takes 16 code bytes (one shared load) of one key;
        // consecutive threads take consecutive keys, so that the eight keys
        // of a store phase cover the eight swizzled 16-byte positions
        auto dequant = [&](const uint8_t* sb, uint8_t* tile_dst, int kv, int fmask) {
          constexpr int UC = FMT == kFmtInt8 ? 2 : 4;  // 8-element chunks per 16 code bytes
          constexpr int UPK = D / 8 / UC;              // 16-byte code units per key
#pragma unroll 2
          for (int q = dt; q < NK * UPK; q += 32 * G::DQ_WARPS) {
            const int k = q & (NK - 1), g = q >> 6;
            const int b4 = k >> 4, x7 = k & 7;
            uint4 w = *reinterpret_cast<const uint4*>(sb + (k + (b4 + kv) * 16) * G::SROW + g * 16);
            if (!((fmask >> b4) & 1)) w = make_uint4(0, 0, 0, 0);  // code 0 in both formats
            uint8_t* const dst = tile_dst + (((g * UC) >> 3) * NK + k) * 128;
            if constexpr (FMT == kFmtInt4) {
              const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int i = 0; i < 4; i++)
                *reinterpret_cast<uint4*>(dst + ((((g * 4 + i) & 7) ^ x7) << 4)) = dq_word_int4(wv[i]);
            } else {
              *reinterpret_cast<uint4*>(dst + ((((g * 2) & 7) ^ x7) << 4)) = dq_pair_int8(w.x, w.y);
              *reinterpret_cast<uint4*>(dst + ((((g * 2 + 1) & 7) ^ x7) << 4)) = dq_pair_int8(w.z, w.w);
            }
          }
        };
        // the first two steps' copies go out at once (the staging buffers are
        // free: the previous item's last dequantisation is done)
        issue(0, stg, block_of(0));
        cp_async_commit();
        if (nsteps > 1) issue(1, stg + G::STG, block_of(1));
        cp_async_commit();
        int blk_next = block_of(2);
        // Q' rows of the item, once every S of the previous item is complete;
        // consecutive threads on consecutive 16-byte chunks (the rows of one
        // token's group are contiguous; INT4 q' is stored in the tiles'
        // nibble order).  They land with step 0's copies, before kfull.
        wait_kfree_tail(prev_steps);
        {
          constexpr int CPR = D / 8;  // 16-byte chunks of a row
#pragma unroll 4
          for (int u = dt; u < ROWS * CPR; u += 32 * G::DQ_WARPS) {
            const int rr = u / CPR, ch = u - rr * CPR;
            uint8_t* d = sQ + sw128(ROWS, rr, ch);
            if (rr < nrows) {
              const int tj = (int)c.gdiv.div((uint32_t)rr), tjj = rr - tj * c.group;
              cp_async16(d, reinterpret_cast<const uint8_t*>(
                                pv.qrot + ((long long)(q0 + tok0 + tj) * c.hq + h * c.group + tjj) * D) + ch * 16);
            } else {
              *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
            }
          }
          cp_async_commit();
        }
        // V tiles and the first ring entries: every PV of the previous item
        // is complete
        wait_vfree_tail(prev_steps);
#pragma unroll 1
        for (int j = 0; j < nsteps; j++) {
          const int b = j & 1;
          uint8_t* const sb = stg + b * G::STG;
          if (j == 0)
            cp_async_wait<0>();  // with the item's Q' rows
          else
            cp_async_wait<1>();
          dq_sync();  // every thread's copies of step j have landed
          // the K tile of step j is free once S of step j - KBUF is complete;
          // the ring entry of step j once the softmax of step j - 3 is (S of
          // step j - 2 follows both halves' P of step j - 3)
          if (j >= G::KBUF) {
            const int fb = (j - G::KBUF) & 1;
            ws_wait(bar(KFREE + fb), (ph_kfree >> fb) & 1, abort_flag, c.status);
            ph_kfree ^= 1u << fb;
          }
          const int* sfl = reinterpret_cast<const int*>(sb + G::FL_OFF);
          uint8_t* const re = ring + (j % G::NRING) * G::RING;
          const int fmask = (sfl[0] != 0) | (sfl[1] != 0) << 1 | (sfl[2] != 0) << 2 | (sfl[3] != 0) << 3;
          if (dt < NK) {
            const float* scs = reinterpret_cast<const float*>(sb + G::SC_OFF);
            const float vsc = scs[(dt >> 4) * 32 + 16 + (dt & 15)];
            reinterpret_cast<float*>(re)[dt] = scs[(dt >> 4) * 32 + (dt & 15)];
            reinterpret_cast<float*>(re)[NK + dt] = vsc;
            // the vote reads only keys that exist (usable block, position below the
            // sequence length): the threshold, and so the rounding, depend on the
            // cache's contents alone
            const bool exists = ((fmask >> (dt >> 4)) & 1) && (kb0 + j * 4) * 16 + dt < L;
            const bool small = __all_sync(0xffffffffu, !exists || fabsf(vsc) < 128.f);
            if (lane == 0) reinterpret_cast<int*>(re + 2 * NK * 4)[4 + (dt >> 5)] = small;
          } else if (dt < NK + 4) {
            reinterpret_cast<int*>(re + 2 * NK * 4)[dt - NK] = sfl[dt - NK];
          }
          dequant(sb, sK + (G::KBUF == 2 ? b : 0) * G::KVBYTES, 0, fmask);
          fence_proxy_async_smem();  // the tile is read by the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(KFULL + b));
          if (j >= 2) {
            ws_wait(bar(VFREE + b), (ph_vfree >> b) & 1, abort_flag, c.status);  // PVs of step j - 2 done
            ph_vfree ^= 1u << b;
          }
          dequant(sb, sV + b * G::KVBYTES, 1, fmask);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(VFULL + b));
          dq_sync();  // every thread is done with staging b
          if (j + 2 < nsteps) issue(j + 2, sb, blk_next);
          cp_async_commit();
          blk_next = block_of(j + 3);
        }
        if (nsteps == 0) cp_async_wait<0>();  // no step waited for this item's Q' copies
        prev_steps = nsteps;
      }
      cp_async_wait<0>();
    } else {
      // ================= MMA warp (lane 0 issues, the warp waits together) =================
      const bool leader = lane == 0;
      uint32_t ph_ifull = 0;
      // operand descriptors: the start address is the low 14-bit field of
      // (address >> 4), so an offset below 256 KB adds to the descriptor
      const uint64_t dq = umma_desc(smem_addr(sQ), 16, 1024);
      const uint64_t dk = umma_desc(smem_addr(sK), 16, 1024);
      const uint64_t dv = umma_desc(smem_addr(sV), NK * 128, 1024);
#pragma unroll 1
      for (int itc = 0;; itc++) {
        int4 item;
        if (!take_item(itc & 1, ph_ifull, item)) break;
        const int seq = item.x, tile = item.z, nkb = item.w;
        const int ql = c.qsl[seq + 1] - c.qsl[seq];
        const int ctx = c.seq_lens[seq] - ql;
        const int kb0 = window_lo(c, ctx + tile * c.tile_tokens) >> 4;  // blocks before the earliest row's window are skipped
        const int nsteps = (nkb - kb0 + 3) / 4;
        // S_h = Q_h K^T over the head dimension into TMEM columns [64h, 64h + 64)
        auto issue_s = [&](int hh, int st) {
          if (leader) {
            const uint64_t kt = dk + (uint64_t)((G::KBUF == 2 ? (st & 1) : 0) * (G::KVBYTES >> 4));
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ks++)
              umma_f16(tmem + 64 * hh, dq + (uint64_t)(((ks >> 2) * ROWS * 128 + hh * 128 * 128 + (ks & 3) * 32) >> 4),
                       kt + (uint64_t)(((ks >> 2) * NK * 128 + (ks & 3) * 32) >> 4), IDESC_S, ks > 0);
          }
        };
        // O_h += P_h V_b, P_h the f16 pairs over S_h's first 32 columns
        auto issue_pv = [&](int hh, int b, bool first) {
          if (leader) {
            const uint64_t vt = dv + (uint64_t)(b * (G::KVBYTES >> 4));
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
              umma_f16_ts(tmem + 128 + hh * D, tmem + 64 * hh + kk * 8, vt + (uint64_t)(kk * (2048 >> 4)), IDESC_O,
                          !first || kk > 0);
          }
        };
        auto commit = [&](int i) {
          if (leader) umma_commit(bar(i));
          __syncwarp();
        };
        // kfull of step 0 also covers the item's Q' rows
        if (nsteps > 0) {
          ws_wait(bar(KFULL), ph_kfull & 1, abort_flag, c.status);
          ph_kfull ^= 1;
          tc_fence_after();
          issue_s(0, 0);
          commit(SFULL);
          issue_s(1, 0);
          commit(SFULL + 1);
          commit(KFREE);
        }
#pragma unroll 1
        for (int j = 0; j < nsteps; j++) {
          const int b = j & 1, nb = (j + 1) & 1;
          // V of this step and K of the next are normally ready long before
          // P: wait for them first, so that PV and the next S issue as soon
          // as the half's P lands (neither waits on anything this warp issues
          // later: V(j) follows PV(j - 2), K(j + 1) follows S(j + 1 - KBUF))
          ws_wait(bar(VFULL + b), (ph_vfull >> b) & 1, abort_flag, c.status);
          ph_vfull ^= 1u << b;
          if (j + 1 < nsteps) {
            ws_wait(bar(KFULL + nb), (ph_kfull >> nb) & 1, abort_flag, c.status);
            ph_kfull ^= 1u << nb;
          }
          ws_wait(bar(PFULL), ph_pfull & 1, abort_flag, c.status);
          ph_pfull ^= 1;
          tc_fence_after();
          issue_pv(0, b, j == 0);
          if (j + 1 < nsteps) {
            issue_s(0, j + 1);
            commit(SFULL);
          }
          ws_wait(bar(PFULL + 1), (ph_pfull >> 1) & 1, abort_flag, c.status);
          ph_pfull ^= 2;
          tc_fence_after();
          issue_pv(1, b, j == 0);
          commit(VFREE + b);
          if (j + 1 < nsteps) {
            issue_s(1, j + 1);
            commit(SFULL + 1);
            commit(KFREE + nb);
          }
        }
        commit(ODONE);
      }
    }
  }
  if (warp == 15) {
    // after a time-out MMAs may still be in flight: they end by themselves
    // (they wait on nothing) and must end before the columns are freed
    if (lane == 0) umma_commit(bar(DRAIN));
    __syncwarp();
    if (!mbar_wait_bounded(bar(DRAIN), 0)) flag(c.status, KV_INT4_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, G::TMEM_COLS);
}
