// Paged decode attention on INT4 / int8 per-token-head codes, included by
// attention.cu after the schedule and parameter types it uses (Common,
// PlanView).  Kept in its own file so that a change elsewhere in the
// attention path leaves this kernel's source, and the DRAM traffic recorded
// against it, untouched.

// ---------------------------------------------------------------------------
// 3. decode: stream-K over (segment, position) units, one CTA per head group
// ---------------------------------------------------------------------------
// A position is NP consecutive 16-key blocks of one segment.  With NP > 1 the
// blocks share one score accumulator: block j owns query columns
// [j * COLS, (j + 1) * COLS) (COLS = 8 / NP >= the sequence's q_len * G), so
// one softmax pass, one barrier and one V offset correction serve NP blocks.
// Each column keeps its own running (m, l, o'); the reduce kernel merges the
// NP columns of a query with the log-sum-exp rule like any other split
// (with NP = 4 the piece's flush merges them first).
template <int D, int NP, int FMT, bool DEEP = false>
struct DecGeom {
  static constexpr int COLS = kDecodeCols / NP;  // query columns per block
  static constexpr int CB = FMT == kFmtInt8 ? D : D / 2;  // code bytes per head vector
  // 64-byte code rows: V rows unpadded, 16-byte chunk c of row r stored at
  // chunk c ^ ((r >> 1) & 3), which spreads an ldmatrix piece's 8 rows over
  // all bank groups; other sizes pad the V row instead
  static constexpr bool VSWZ = CB == 64;
  // ring of single-block slots: NP consumed per iteration, the rest in
  // flight.  The copies in flight per SM set the decode's pace; DEEP (four
  // heads per CTA, four CTAs per SM, separate 16-byte aligned scales) takes
  // one more slot where the slots are small enough to keep four CTAs per SM
  // (swizzled 64-byte rows, or rows of at most 48 bytes), and stages a
  // block's scales as 16-byte rows of the group's four heads
  static constexpr int NS = NP == 1 ? 4 : NP == 4 ? 8 : 2 * NP + (DEEP && (VSWZ || CB <= 48) ? 2 : 1);
  static constexpr int WAIT = NS - 2 * NP;  // copy groups that may stay pending at a wait
  static constexpr int KROW = CB;           // K tile row stride (bytes)
  // V tile row stride: an odd multiple of 16 bytes, so that the 8 rows of
  // an ldmatrix piece fall in distinct bank groups (or swizzled, above)
  static constexpr int VROW = VSWZ || (CB / 16) % 2 ? CB : CB + 16;
  static constexpr int KTILE = 16 * KROW;
  static constexpr int VTILE = 16 * VROW;
  // one head's K and V codes of one block, padded to 64 mod 128 bytes so that
  // the copies of neighbouring heads' rows fall in different bank halves
  static constexpr int HTILE = ((KTILE + VTILE + 63) / 128) * 128 + 64;
  static constexpr int KW = CB / 16;    // K words per row per thread (quarter row)
  static constexpr int KSTEPS = D / 16; // MMA k-steps of a block's K (and m-tiles of its V)
  static constexpr int CHR = CB / 16;   // 16-byte chunks per code row
  // per slot: hg head tiles, then scales [K/V][hg][16] ([K/V][16][hg] with DEEP)
  __host__ __device__ static constexpr int slot_bytes(int hg) { return hg * (HTILE + 128); }
  __host__ __device__ static constexpr int smem_bytes(int hg) { return NS * slot_bytes(hg) + 32; }
  static_assert(HTILE % 16 == 0, "tile alignment");
  static_assert(WAIT >= 0 && NS <= 8, "slot ring");
};

// Walk over a lane's decode units (sequence i, head group grp, position kp).
struct DecWalk {
  int i;      // index into the decode-sequence list
  int grp;    // head group (grp mod nl = lane)
  int lane;   // the CTA's lane
  int kp;     // position within the sequence
  int npos;   // positions of the sequence
  int nblk;   // 16-key blocks of the sequence
  int fb;     // first block read (the sliding window's)
  int seq;    // sequence id
};

// one 16-byte record per decode sequence, written by the prep kernel
template <int NP>
__device__ __forceinline__ void walk_load(DecWalk& w, const Common& c, const PlanView& pv) {
  const int4 di = pv.dseq[w.i];  // (sequence, seq_len, first query token, q_len)
  w.seq = di.x;
  w.nblk = (di.y + 15) / 16;
  w.fb = first_block(c, di.y, di.w);
  w.npos = (w.nblk - w.fb + NP - 1) / NP;
}
template <int NP>
__device__ __forceinline__ void walk_next(DecWalk& w, const Common& c, const PlanView& pv) {
  if (++w.kp == w.npos) {
    w.kp = 0;
    if ((w.grp += c.nl) >= c.ng) {
      w.grp = w.lane;
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
// addresses key 8 ((l >> 3) & 1) + (l & 7) of chunk (l >> 4)); chunk pair p
// is at vaddr + p * vstep (32 in a padded tile, +-32 by row in a swizzled one)
template <int D, bool CORR, int FMT>
__device__ __forceinline__ void pv_mmas(float (&oacc)[D / 16][4], uint32_t vaddr, int vstep, uint32_t b0, uint32_t b1,
                                        const uint32_t (&vcorr)[4]) {
  constexpr int CH = (FMT == kFmtInt8 ? D : D / 2) / 16;  // 16-byte chunks per V row
#pragma unroll
  for (int p = 0; p < CH / 2; p++) {
    uint32_t r[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(vaddr + p * vstep));
    pv_mma_chunk<D, CORR, FMT>(oacc, 2 * p, r[0], r[1], b0, b1, vcorr);
    pv_mma_chunk<D, CORR, FMT>(oacc, 2 * p + 1, r[2], r[3], b0, b1, vcorr);
  }
  if constexpr (CH % 2) {
    uint32_t r[2];
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(vaddr + (CH / 2) * vstep));
    pv_mma_chunk<D, CORR, FMT>(oacc, CH - 1, r[0], r[1], b0, b1, vcorr);
  }
}

struct DecParams {
  Common c;
  PlanView pv;
  int num_ctas;
};

// Work decomposition: nl lanes (nl divides the head-group count; as a rule
// every group has its own lane), CTA r in lane r mod nl.  Each lane runs
// stream-K over its flattened (decode sequence, head group, position) units:
// the lane's k-th CTA takes units [T*k/R, T*(k+1)/R) of its T, with R the
// lane's CTAs.  The lanes' ranges line up, so the CTAs that read the
// different head groups' slices of one block do so at about the same time
// and the cache lines they share are read from DRAM once.  A CTA has
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
template <int D, int NP, int FMT, bool DEEP>
__device__ __forceinline__ void decode_body(const DecParams& prm) {
  using G = DecGeom<D, NP, FMT, DEEP>;
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
  // lane blockIdx.x mod nl: its head groups, the lane's (blockIdx.x / nl)-th
  // share of their units
  const int gpl = c.ng / c.nl;  // head groups per lane
  const int my_lane = blockIdx.x % c.nl, rr = blockIdx.x / c.nl;
  const long long Tu = pv.dprefix[n_dseq] * gpl;
  const int R = prm.num_ctas / c.nl;
  const long long P0 = Tu * rr / R, P1 = Tu * (rr + 1) / R;
  if (P0 >= P1) return;
  const int nunits = (int)(P1 - P0);

  // locate P0: largest i with dprefix[i] * gpl <= P0 (32-ary search, per warp)
  int lo = 0, hi = n_dseq;  // invariant: key(lo) <= P0 < key(hi)
  while (hi - lo > 1) {
    const long long span = hi - lo;
    const int probe = lo + (int)((span * lane) / 32);
    const bool le = lane == 0 || pv.dprefix[probe] * gpl <= P0;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz(m);
    const int nlo = lo + (int)((span * last) / 32);
    const int nhi = last == 31 ? hi : lo + (int)((span * (last + 1)) / 32);
    lo = nlo;
    hi = nhi > nlo ? nhi : nlo + 1;
  }
  DecWalk cw;
  cw.i = lo;
  cw.lane = my_lane;
  walk_load<NP>(cw, c, pv);
  {
    const long long off = P0 - pv.dprefix[cw.i] * gpl;
    const int gs = (int)(off / cw.npos);
    cw.grp = gs * c.nl + my_lane;
    cw.kp = (int)(off - (long long)gs * cw.npos);
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
    const int vcol = G::VSWZ ? col ^ ((r >> 1) & 3) : col;
    c_saddr[j] = smem_addr(smem) + h * G::HTILE + (kv ? G::KTILE + r * G::VROW + vcol * 16 : r * G::KROW + col * 16);
    c_src[j] = (kv ? c.v_cache : c.k_cache) + r * c.geo.crow + (long long)h * c.geo.chead + col * 16;
  }
  // scales: DEEP (four heads) one 16-byte row [K/V][row][h] for each of
  // threads 0..31, else one 4-byte scale [K/V][h][row] per thread
  const int s_kv = DEEP ? tid >> 4 : tid / (16 * HG), s_rem = DEEP ? tid & 15 : tid % (16 * HG);
  const int s_r = DEEP ? s_rem : s_rem / HG, s_h = DEEP ? 0 : s_rem % HG;
  const uint32_t s_saddr = smem_addr(smem) + HG * G::HTILE +
                           (DEEP ? (s_kv * 16 + s_r) * 16 : (s_kv * HG + s_h) * 64 + s_r * 4);
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
      if constexpr (DEEP) {
        if (tid < 32) asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s_saddr + soff), "l"(ssrc));
      } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s_saddr + soff), "l"(ssrc));
      }
    }
    if (tid == 0) {
      sflag[slot] = ok;
      if (!ok && blk != kAbsent) flag(c.status, KV_INT4_DEV_BAD_BLOCK);
    }
  };

  // producer: one block per call into the next ring slot, the next block id
  // loaded one call ahead; one commit group per call (empty past the range)
  int ppos = 0;
  int pj = 0, ps = 0;
  // the prologue's block ids, loaded together when its NS - NP blocks lie in
  // the first segment (one latency instead of one per block): this serves
  // short ranges; the DEEP ring's CTAs run long ranges and keep the registers
  constexpr int PRO = DEEP ? 1 : G::NS - NP;
  static_assert(PRO <= 4, "prologue depth");
  int pro[4];
  const int pro_n = PRO > 1 && pw.kp + (PRO + NP - 1) / NP <= pw.npos && (PRO + NP - 1) / NP <= nunits ? PRO : 1;
#pragma unroll
  for (int j = 0; j < 4; j++)
    if (j < pro_n) {
      const int kb = pw.fb + pw.kp * NP + j;
      pro[j] = kb < pw.nblk ? c.block_table[(long long)pw.seq * c.max_blocks + kb] : kAbsent;
    }
  if (pro_n == 1) pro[0] = block_at(pw, 0);
  int pro_left = pro_n - 1;  // prefetched ids after the current one, shifted down pro[1..3]
  int pblk = pro[0];
  auto produce = [&]() {
    if (ppos < nunits) {
      issue(pblk, pw.grp, ps);
      ps = ps + 1 == G::NS ? 0 : ps + 1;
      if (++pj == NP) {
        pj = 0;
        if (++ppos < nunits) walk_next<NP>(pw, c, pv);
      }
      if (ppos < nunits) {
        if (pro_left > 0) {
          pblk = pro[1];
          pro[1] = pro[2];
          pro[2] = pro[3];
          --pro_left;
        } else {
          pblk = block_at(pw, pj);
        }
      }
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
    const int head = cw.grp * HG + hl;
    const int4 di = pv.dseq[cw.i];  // (sequence, seq_len, first query token, q_len)
    const int q0 = di.z, ql = di.w, L = di.y;
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
        // q' is stored in nibble order: v = (e0, e4), (e1, e5), (e2, e6), (e3, e7)
        uint4 v = make_uint4(0, 0, 0, 0);
        if (colok) v = *reinterpret_cast<const uint4*>(qrow + 8 * (cq * G::KW + w));
        __half2 h0 = __hmul2(*reinterpret_cast<__half2*>(&v.x), x16);
        __half2 h1 = __hmul2(*reinterpret_cast<__half2*>(&v.z), x16);
        qb[2 * w][0] = *reinterpret_cast<uint32_t*>(&h0);
        qb[2 * w][1] = v.y;
        qb[2 * w + 1][0] = *reinterpret_cast<uint32_t*>(&h1);
        qb[2 * w + 1][1] = v.w;
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
    // with four blocks per position the piece's blocks hold the same queries
    // in columns c, c + 2, c + 4, c + 6 (lanes whose cq differs): merge them
    // here with the log-sum-exp rule, so that only columns 0 and 1 leave the
    // CTA and the reduce reads one partial per piece instead of four (with
    // two blocks the reduce merges the pair: the extra code here measured
    // 1631 -> 1641 us on the long-context decode)
    float mm0 = m0, mm1 = m1;
    if constexpr (NP == 4) {
#pragma unroll
      for (int x = G::COLS / 2; x < 4; x <<= 1) {
        const float p0 = __shfl_xor_sync(0xffffffffu, mm0, x), p1 = __shfl_xor_sync(0xffffffffu, mm1, x);
        const float n0 = fmaxf(mm0, p0), n1 = fmaxf(mm1, p1);
        const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
        const float sa0 = fast_exp2(mm0 - u0), sb0 = fast_exp2(p0 - u0);
        const float sa1 = fast_exp2(mm1 - u1), sb1 = fast_exp2(p1 - u1);
        a0 = a0 * sa0 + __shfl_xor_sync(0xffffffffu, a0, x) * sb0;
        a1 = a1 * sa1 + __shfl_xor_sync(0xffffffffu, a1, x) * sb1;
#pragma unroll
        for (int i = 0; i < G::KSTEPS; i++) {
          oacc[i][0] = oacc[i][0] * sa0 + __shfl_xor_sync(0xffffffffu, oacc[i][0], x) * sb0;
          oacc[i][2] = oacc[i][2] * sa0 + __shfl_xor_sync(0xffffffffu, oacc[i][2], x) * sb0;
          oacc[i][1] = oacc[i][1] * sa1 + __shfl_xor_sync(0xffffffffu, oacc[i][1], x) * sb1;
          oacc[i][3] = oacc[i][3] * sa1 + __shfl_xor_sync(0xffffffffu, oacc[i][3], x) * sb1;
        }
        mm0 = n0;
        mm1 = n1;
      }
    }
    if (NP == 4 && cq > 0) return;  // columns 2 .. 7 are merged into columns 0 and 1
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
      dst_ml[(2 * cq) * 2 + 0] = mm0;
      dst_ml[(2 * cq) * 2 + 1] = a0;
      dst_ml[(2 * cq + 1) * 2 + 0] = mm1;
      dst_ml[(2 * cq + 1) * 2 + 1] = a1;
    }
  };

  begin_segment();
  const int jb = (cq * NP) >> 2;  // block of this thread's score columns 2cq, 2cq+1
  const int jv = (g * NP) >> 3;   // block of this lane's P'^T column g
  // this lane's ldmatrix row of the V tile in slot 0
  const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7), vx = G::VSWZ ? (vrow >> 1) & 3 : 0;
  const uint32_t v_lane =
      smem_addr(smem) + hl * G::HTILE + G::KTILE + vrow * G::VROW + (((lane >> 4) ^ (vx & 1)) + 2 * (vx >> 1)) * 16;
  const int vstep = vx >> 1 ? -32 : 32;
  int cs = 0;                     // slot of the iteration's first block
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
    const float* sks = reinterpret_cast<const float*>(mstg + HG * G::HTILE + (DEEP ? hl * 4 : hl * 64));
    const float* svs = reinterpret_cast<const float*>(mstg + HG * G::HTILE + (DEEP ? 256 + hl * 4 : (HG + hl) * 64));
    constexpr int SR = DEEP ? 4 : 1;  // scale stride between rows (floats)

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
    const float ks0 = sks[g * SR] * (I8 ? 1.f : 0.0625f), ks1 = sks[(g + 8) * SR] * (I8 ? 1.f : 0.0625f);
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
    const float vs0 = svs[g * SR], vs1 = svs[(g + 8) * SR];
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
      pv_mmas<D, true, FMT>(oacc, v_lane + slot[0] * SB, vstep, b0, b1, vcorr);
    } else {
#pragma unroll
      for (int j = 0; j < NP; j++) {
        // block j's probabilities only: the other blocks' columns are zero
        const uint32_t bj0 = jv == j ? b0 : 0u, bj1 = jv == j ? b1 : 0u;
        pv_mmas<D, false, FMT>(oacc, v_lane + slot[j] * SB, vstep, bj0, bj1, vcorr);
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

// Register ceilings (allocated in steps of 8 a thread) for four 4-warp CTAs
// per SM up to head size 96, three at 128 (int8) and 192 (INT4); int8 at 192
// and both formats at 256 keep the compiler's choice (two CTAs, no spills).
__host__ __device__ constexpr int decode_max_regs(int d, int fmt) {
  return d <= 96 ? 128 : (d <= 128 || (d <= 192 && fmt == kFmtInt4)) ? 168 : 255;
}
template <int D, int NP, int FMT, bool DEEP = false>
__global__ void __maxnreg__(decode_max_regs(D, FMT)) decode_kernel(DecParams prm) {
  decode_body<D, NP, FMT, DEEP>(prm);
}
// INT4 head size 128 (the long-context shape): at most 128 registers a
// thread, so that four 4-warp CTAs (or two 8-warp ones) share an SM
template <int NP, bool DEEP>
__global__ void __launch_bounds__(256, 2) decode_kernel_i4d128(DecParams prm) {
  decode_body<128, NP, kFmtInt4, DEEP>(prm);
}
// The decode kernel for a format and head size, with the 16-byte scale rows
// (and, for 64-byte code rows, the deeper ring) where it has them (`deep`),
// and its dynamic shared memory for hg heads per CTA.  INT4 head size 128
// takes them with paired blocks, where the deeper ring changes the slot
// count; the other INT4 head sizes take the scale rows alone.
template <int D, int NP, int FMT>
struct DecodeEntry {
  static constexpr bool HAS_DEEP =
      FMT == kFmtInt4 && (D != 128 || NP == 4 || DecGeom<D, NP, FMT, true>::NS != DecGeom<D, NP, FMT>::NS);
  static void (*kernel(bool deep))(DecParams) {
    if constexpr (NP == 4) {  // launched with four-head CTAs and 16-byte scale rows only
      static_assert(HAS_DEEP, "four blocks per position: INT4");
      (void)deep;
      if constexpr (D == 128) return decode_kernel_i4d128<NP, true>;
      else return decode_kernel<D, NP, FMT, true>;
    } else if constexpr (FMT == kFmtInt4 && D == 128) {
      if constexpr (HAS_DEEP) {
        if (deep) return decode_kernel_i4d128<NP, true>;
      }
      return decode_kernel_i4d128<NP, false>;
    } else {
      if constexpr (HAS_DEEP) {
        if (deep) return decode_kernel<D, NP, FMT, true>;
      }
      return decode_kernel<D, NP, FMT, false>;
    }
  }
  static int smem(bool deep, int hg) {
    return deep && HAS_DEEP ? DecGeom<D, NP, FMT, true>::smem_bytes(hg) : DecGeom<D, NP, FMT>::smem_bytes(hg);
  }
};
