// bsfa_xs.cuh -- the single-head gated prefill kernel: one query head per
// CTA, one 128-row query tile per unit, key tiles of BK = 128 or 224 keys,
// each key tile one semantic block (Bq = 128, Bk = BK).
//
// BK = 128, the pipelined schedule (the default for gated 128 x 128 calls):
// the scores of key tiles t, t+1 and t+2 live in three TMEM buffers, and a
// warp of its own issues Q.K^T of tile t+3 as soon as tile t is done with its
// buffer -- skipped (the softmax frees it right after the vote) or its P.V
// complete ("Skipping attention blocks was the easy part", section
// "Cross-stage P": the next tile's Q.K^T does not wait for the current
// tile's P.V).  Two tiles' Q.K^T then run while a third is being decided,
// which is what a run of skipped tiles needs.
//
// BK = 224, the H100 deployment tile of "Block Sparse Flash Attention"
// ("Loss & Training": a 128-row query tile and a 224-key tile): one 224-column
// score buffer (two would not fit next to O in the 512 TMEM columns), so the
// next Q.K^T follows the current decision or P.V.  Key Designs 2 notes that
// a single j = i index does not map the diagonal for unequal tiles: a key
// tile is a candidate when all its keys precede the query tile's first row,
// and every other visible key tile is in the diagonal region (kept, masked).
//
// What it computes is the same gated, renormalised attention as
// bsfa_fwd_kernel (Key Designs 2 and 3; the lambda gate of "Vote, then
// skip"): every visible tile's scores are computed, the tile maximum (or
// each row's maximum against its running max) decides the tile, and a
// skipped tile gets no V load, no exp and no P.V.  With CALIB the kernel
// only computes Q.K^T and records sigma * (tile maximum) of every candidate
// tile (the calibration pass of Key Designs 1).  With CORR (mean correction,
// "FlashPrefill V2") a unit's key tiles are followed by ceil(I / 128)
// correction tiles through the same roles: the producer loads key means,
// the V loader value means, and the softmax runs them in a loop of its own
// after the key tiles (see the CORR note at the kernel).
//
// Roles (384 threads, one CTA per SM, persistent over a heaviest-first list
// of (KV head, query tile, query head) units):
//   warp 0      TMA producer: Q per unit, K for every visible tile.
//   warp 1      P.V issuer (calibration: Q.K^T issuer), TMEM owner.
//   warp 2      Q.K^T issuer (not calibration).
//   warp 3      V loader: V of the tiles the gate keeps (of every tile when
//               the gate is compiled out or with VALL).
//   warps 4-11  softmax: warp 4 + 4 ch + wq holds, for rows 32 wq .. 32 wq
//               + 31, the tile's keys [BK/2 ch, BK/2 ch + BK/2).
//
// TMEM: score buffer b at columns [128 b, 128 b + BK) (P overwrites its first
// BK/2 columns as 16-bit pairs), O after them (XsLayout::O_COL).
#pragma once
#include "bsfa_fwd.cuh"

namespace bsfa {

struct XsCtrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4];  // K ring (XsLayout::KST <= 4 stages)
  uint64_t v_full[2], v_empty[2];  // V ring (XsLayout::VST <= 2 stages)
  uint64_t s_full[3];    // per S buffer: scores of its current tile ready
  uint64_t ph_full[3];   // per S buffer: P of the first half of the keys written (or skipped)
  uint64_t p_full[3];    // per S buffer: P of the second half written (or skipped)
  uint64_t dec_full[3];  // per S buffer: decision word published (32 arrivals, one warp)
  uint64_t pv_done[2];   // per kept-tile parity: that kept tile's P.V and all before it done
  uint64_t buf_free[3];  // per S buffer: its tile is done with it (skipped, or P.V complete)
  uint64_t o_full, o_empty;
  uint64_t drain, drain_qk;
  uint32_t tmem_base;
  uint32_t dec[3];       // per S buffer: tile stamp << DEC_BITS | keep bit
  float xmax[2][2][128]; // per (tile parity, column half, row): half-row maximum
  float xl[2][128];      // per (column half, row): share of the normaliser
  float xw[2][8];        // calibration: per (tile parity, softmax warp) maximum
  // Mean correction: kept bits of the unit's candidate key blocks (bit j of
  // word j / 32 = block j kept), written by the bookkeeping warp.
  uint32_t kbits[CORR_WORDS];
  int abort;
};

template <int D, int BK, bool CALIB>
struct XsLayout {
  static constexpr int NB = BK == 128 ? 3 : 1;                        // score buffers
  static constexpr int KST = BK == 128 ? 3 : (D == 128 ? 1 : 2);      // K ring stages
  static constexpr int VST = CALIB ? 0 : 2;                           // V ring stages
  static constexpr int TQ = TILE * D * 2;  // bytes of the 128-row Q tile
  static constexpr int TKV = BK * D * 2;   // bytes of one K or V tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TQ;
  static constexpr int V_OFF = K_OFF + KST * TKV;
  static constexpr int C_OFF = V_OFF + VST * TKV;
  static constexpr int RAW = C_OFF + (((int)sizeof(XsCtrl) + 15) & ~15) + 1024;
  // At least 120 KB, so that one CTA is resident per SM (the persistent grid
  // and the whole-TMEM allocation assume it).
  static constexpr int BYTES = RAW > 120 * 1024 ? RAW : 120 * 1024;
  static constexpr int NCOLS = 512;
  static constexpr int NTHREADS = 384;
  // O after the score buffers: [384, 384 + D) with three 128-column buffers,
  // [256, 256 + D) after the single 224-column one.
  static constexpr uint32_t O_COL = BK == 128 ? NB * 128 : 256;
  static_assert(O_COL + D <= NCOLS, "TMEM columns");
  static_assert(BYTES <= 227 * 1024, "shared memory");
  static_assert(BK == 128 || BK == 224, "key tile");
  static_assert(KST <= 4 && VST <= 2 && NB <= 3, "ring sizes of XsCtrl");
};

// The CTA's units, in order.  Each KV head's units (heaviest first) are dealt
// in waves of gridDim.x, and the waves alternate direction over the CTAs
// (boustrophedon): the CTA that takes a wave's heaviest unit takes the next
// wave's lightest, so the CTAs' cumulative work stays level and the units of
// a wave stream the KV head's K/V prefix together, close enough in time for
// each tile to be fetched into L2 once.  The first wave's direction flips
// from one KV head to the next, which also levels the partial last waves.
// (Dealt round-robin, the first CTAs took the heaviest unit of every wave
// and drifted a whole unit ahead of the last ones within a KV head.)  Every
// role of the CTA walks the same sequence.
struct XsUnits {
  int per_kv, hkv, h, w, u;  // u: the current unit, -1 past the end
  __device__ __forceinline__ XsUnits(int per_kv_, int hkv_)
      : per_kv(per_kv_), hkv(hkv_), h(0), w(-1), u(-1) {
    next();
  }
  __device__ __forceinline__ bool valid() const { return u >= 0; }
  __device__ __forceinline__ void next() {
    const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    for (;;) {
      if (++w * g >= per_kv) {  // past this KV head's last wave
        w = 0;
        if (++h >= hkv) {
          u = -1;
          return;
        }
      }
      const int ul = w * g + (((w + h) & 1) ? g - 1 - b : b);
      if (ul < per_kv) {
        u = h * per_kv + ul;
        return;
      }
    }
  }
};

// Key tiles visible to query tile I of a length-len sequence: those starting
// at or before the tile's last row.
template <int BK>
__device__ __forceinline__ int xs_ntiles(int I, int len) {
  return min(I * TILE + TILE - 1, len - 1) / BK + 1;
}

// S = Q K^T for one tile: D/16 K-steps of M = 128, N = BK, K = 16.  Q's and
// K's 64-column swizzled halves sit TILE*128 and BK*128 bytes apart.
template <int D, int BK>
__device__ __forceinline__ void xs_issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk,
                                            uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t oq = (((kk >> 2) * (TILE * 128)) + (kk & 3) * 32) >> 4;
    const uint64_t ok = (((kk >> 2) * (BK * 128)) + (kk & 3) * 32) >> 4;
    umma_ss(d_tmem, dq + oq, dk + ok, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V over K-steps [k0, k1) of 16 keys: P (16-bit pairs) in TMEM
// columns [8 kk, 8 kk + 8) of the score buffer, V MN-major (16 keys = 2048 B
// per 64-column half).
__device__ __forceinline__ void xs_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                            uint32_t idesc, uint32_t acc, int k0, int k1) {
#pragma unroll
  for (int kk = k0; kk < k1; ++kk)
    umma_ts(d_tmem, p_tmem + kk * 8, dv + ((kk * 2048) >> 4), idesc, (kk > 0 || acc) ? 1u : 0u);
}

// CORR (gated, BK = 128, contiguous K/V): mean correction.  After a unit's key
// tiles come ceil(I / 128) correction tiles through the same pipeline: their
// "keys" and "values" are the block means of 128 consecutive key blocks
// (tmKb, tmVb), and only the candidate blocks this head skipped enter them,
// with the logit shifted by ln(Bk) so that one mean stands for the block's Bk
// keys ("FlashPrefill V2", mean correction).
template <int D, int BK, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED,
          bool CORR = false>
__global__ void __launch_bounds__(384, 1)
    bsfa_xs_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmKb,
                   const __grid_constant__ CUtensorMap tmVb, const DevParams p) {
  static_assert(!CORR || (GATING && !CALIB && !VALL && !PAGED && BK == 128), "mean correction");
  using LY = XsLayout<D, BK, CALIB>;
  constexpr int NB = LY::NB, KST = LY::KST, VST = LY::VST;
  // Q.K^T from a warp of its own (warp 2) when there are several score
  // buffers; with one, each Q.K^T waits for the previous tile anyway and is
  // issued in order after its P.V by warp 1.
  constexpr bool SPLIT = !CALIB && NB > 1;
  constexpr int VSTN = VST > 0 ? VST : 1;  // divisor for V ring indices (no V ring: unused)
  constexpr int TQ = LY::TQ, TKV = LY::TKV;
  constexpr int QHALF = TILE * 128;  // bytes of one 64-column swizzled half of Q
  constexpr int KHALF = BK * 128;    // the same for a K or V tile
  constexpr int NHALF = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base + LY::Q_OFF;
  uint8_t* sK = base + LY::K_OFF;
  uint8_t* sV = base + LY::V_OFF;
  XsCtrl* c = reinterpret_cast<XsCtrl*>(base + LY::C_OFF);
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_empty, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(&c->s_full[b], 1);
      mbar_init(&c->ph_full[b], 128);
      mbar_init(&c->p_full[b], 128);
      mbar_init(&c->dec_full[b], 32);
      c->dec[b] = 0xFFFFFFFFu;  // no stamp matches
    }
    for (int b = 0; b < 2; ++b) mbar_init(&c->pv_done[b], 1);
    for (int b = 0; b < 3; ++b) mbar_init(&c->buf_free[b], 1);
    mbar_init(&c->o_full, 1);
    mbar_init(&c->o_empty, 256);
    mbar_init(&c->drain, 1);
    mbar_init(&c->drain_qk, 1);
    c->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    if (!CALIB) prefetch_tensormap(&tmV);
    if (CORR) {
      prefetch_tensormap(&tmKb);
      prefetch_tensormap(&tmVb);
    }
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, LY::NCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;

  // Unit order: KV head slowest, then query tiles heaviest first, then the
  // query heads of the group (the group's CTAs stream the same K/V tiles
  // together, out of L2).
  const int ntot = *p.ntiles_total;
  const int per_kv = ntot * p.group;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t kc = 0, uc = 0;
    int last_q = -1;  // index of the last unit whose Q load was issued
    bool ok = true;
    for (XsUnits it(per_kv, p.Hkv); ok && it.valid(); it.next(), ++uc) {
      const int u = it.u;
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int h = kvh * p.group + rem % p.group;
      const int4 si = p.seqinfo[t.x];
      const int n = xs_ntiles<BK>(t.y, si.y);
      const int ntt = n + (CORR ? (t.y + TILE - 1) / TILE : 0);  // + correction tiles
      if (!(ok = wait_all(&c->q_empty, (uc & 1) ^ 1, abort, p.err, ERR_WAIT_Q_EMPTY))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&c->q_full, TQ);
        for (int hf = 0; hf < NHALF; ++hf)
          tma_load_4d(sQ + hf * QHALF, &tmQ, &c->q_full, hf * 64, si.x + t.y * TILE, h, si.w);
      }
      __syncwarp();
      last_q = static_cast<int>(uc);
      for (int J = 0; J < ntt; ++J) {
        // A K tile's coordinates: the sequence's token base, or (paged, BK =
        // 128 only) its page from the block table.  A correction tile reads
        // the key means of blocks [128 (J - n), +128) of the sequence.
        const int2 cc = PAGED ? kv_tile_coord<PAGED>(p, si, t.x, J)
                              : make_int2(si.x + J * BK, si.w);
        const bool mean_tile = CORR && J >= n;
        {
          const uint32_t st = kc % KST;
          // With as many K stages as score buffers, Q.K^T number kc reads K
          // stage kc % KST and writes score buffer kc % NB, the same index:
          // the stage is free once that buffer's scores are complete.
          uint64_t* kfree = (KST == NB) ? &c->s_full[st] : &c->k_empty[st];
          if (!(ok = wait_all(kfree, ((kc / KST) & 1) ^ 1, abort, p.err, ERR_WAIT_K_EMPTY)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&c->k_full[st], TKV);
            for (int hf = 0; hf < NHALF; ++hf) {
              if (mean_tile)
                tma_load_4d(sK + st * TKV + hf * KHALF, &tmKb, &c->k_full[st], hf * 64,
                            si.z + (J - n) * TILE, kvh, 0);
              else
                tma_load_4d(sK + st * TKV + hf * KHALF, &tmK, &c->k_full[st], hf * 64, cc.x, kvh,
                            cc.y);
            }
          }
          __syncwarp();
          ++kc;
        }
      }
    }
    if (!ok) {
      // Let every copy already issued land before the CTA can exit.
      if (last_q >= 0) drain_wait(&c->q_full, last_q & 1);
      for (uint32_t i = 0; i < KST && i < kc; ++i) {
        const uint32_t f = kc - 1 - i;
        drain_wait(&c->k_full[f % KST], (f / KST) & 1);
      }
    }
  } else if (!CALIB && warp == 3) {
    // ------------------------------------------------------------ V loader
    // V of a tile is requested as soon as the softmax publishes a keep (with
    // VALL, or with the gate compiled out: for every tile, as soon as a stage
    // is free).  A warp of its own, so that K loads never queue behind V.
    uint32_t vc = 0, tc = 0;
    bool ok = true;
    for (XsUnits it(per_kv, p.Hkv); ok && it.valid(); it.next()) {
      const int u = it.u;
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int4 si = p.seqinfo[t.x];
      const int n = xs_ntiles<BK>(t.y, si.y);
      const int ntt = n + (CORR ? (t.y + TILE - 1) / TILE : 0);
      for (int J = 0; J < ntt; ++J, ++tc) {
        const int2 cc = PAGED ? kv_tile_coord<PAGED>(p, si, t.x, J)
                              : make_int2(si.x + J * BK, si.w);  // before the waits
        // Also in a unit whose gate keeps everything, V waits for each
        // published decision: issued as early as a stage is free (as with
        // VALL), the V copies delay the K copies the Q.K^T issuer waits on.
        bool need = VALL || !GATING;
        if constexpr (GATING && !VALL) {
          // The decision word of the tile's S buffer carries the tile stamp.  A
          // word stamped with a later tile also means a skip: a kept tile's
          // P.V waits for its V, and the next Q.K^T into that buffer (whose
          // decision overwrites the word) is issued only after that P.V.
          const uint32_t b = tc % NB;
          const uint32_t w = wait_decision<NB>(&c->dec[b], &c->dec_full[b], tc, abort, p.err, &ok);
          if (!ok) break;
          need = stamp_dist(w, tc) == 0 && (w & DEC_MASK) != 0u;
        }
        if (!need) continue;
        const uint32_t st = vc % VSTN;
        if (!(ok = wait_all(&c->v_empty[st], ((vc / VSTN) & 1) ^ 1, abort, p.err,
                            ERR_WAIT_V_EMPTY)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&c->v_full[st], TKV);
          for (int hf = 0; hf < NHALF; ++hf) {
            if (CORR && J >= n)  // value means of key blocks [128 (J - n), +128)
              tma_load_4d(sV + st * TKV + hf * KHALF, &tmVb, &c->v_full[st], hf * 64,
                          si.z + (J - n) * TILE, kvh, 0);
            else
              tma_load_4d(sV + st * TKV + hf * KHALF, &tmV, &c->v_full[st], hf * 64, cc.x, kvh,
                          cc.y);
          }
        }
        __syncwarp();
        ++vc;
      }
    }
    if (!ok) {
      if constexpr (VST > 0) {
        for (uint32_t i = 0; i < static_cast<uint32_t>(VST) && i < vc; ++i) {
          const uint32_t f = vc - 1 - i;
          drain_wait(&c->v_full[f % VSTN], (f / VSTN) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- P.V issuer
    // The whole warp runs the loop and the waits; one elected lane issues
    // every MMA and commit.  For each tile t: its decision; if kept, P.V (P
    // in two halves) and the commit of pv_done.  A skipped tile needs nothing
    // here (every access and commit of this warp queues behind the MMAs in
    // flight).  With SPLIT, a kept tile also commits buf_free (its score
    // buffer may take the Q.K^T of tile t + NB once that P.V is complete) and
    // warp 2 issues every Q.K^T, as soon as a buffer is free and its K tile
    // has landed, so a run of skipped tiles never waits for this warp.
    // Without SPLIT (one 224-column buffer) this warp issues the Q.K^T of
    // tile t + NB itself, in issue order after t's P.V.  Calibration: this
    // warp issues the Q.K^T, each after the softmax's release of the buffer.
    constexpr uint32_t IDESC_QK = idesc_f32acc<F16>(128, BK, false, false);
    constexpr uint32_t IDESC_PV = idesc_f32acc<F16>(128, D, false, true);
    constexpr int KSTEPS = BK / 16, KHALFSTEPS = BK / 32;
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sV), KHALF, 1024);
    const uint32_t d_o = tmem + LY::O_COL;
    uint32_t kc = 0, vc = 0, tc = 0, uc = 0;
    uint32_t kp = 0;  // kept tiles so far (pv_done phases)
    bool ok = true;
    // Q.K^T of the unit's tile j into score buffer b.
    auto issue_s = [&](int j, int n, uint32_t b) -> bool {
      const uint32_t kst = kc % KST;
      if (!__all_sync(0xffffffffu, mbar_test_wait(&c->k_full[kst], (kc / KST) & 1)) &&
          !wait_all(&c->k_full[kst], (kc / KST) & 1, abort, p.err, ERR_WAIT_K_FULL))
        return false;
      if (elect_one()) {
        xs_issue_qk<D, BK>(tmem + b * 128, dQ, dK + ((kst * TKV) >> 4), IDESC_QK);
        umma_commit(&c->s_full[b]);
        if constexpr (KST != NB) umma_commit(&c->k_empty[kst]);
        if (j == n - 1) umma_commit(&c->q_empty);
      }
      __syncwarp();
      ++kc;
      return true;
    };
    for (XsUnits it(per_kv, p.Hkv); ok && it.valid(); it.next(), ++uc) {
      const int u = it.u;
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int nk = xs_ntiles<BK>(t.y, p.seqinfo[t.x].y);
      const int n = nk + (CORR ? (t.y + TILE - 1) / TILE : 0);  // + correction tiles
      // A unit whose gate keeps everything: no decision to read for its key
      // tiles (the softmax still publishes them, so the phases stay one per
      // tile).  Correction tiles are read even then.
      const bool triv = GATING && !CALIB && unit_gate_trivial(p, kvh * p.group + rem % p.group, t.y);
      if constexpr (!SPLIT) {
        if (!(ok = wait_all(&c->q_full, uc & 1, abort, p.err, ERR_WAIT_Q_FULL))) break;
        for (int j = 0; j < NB && j < n; ++j)
          if (!(ok = issue_s(j, n, (tc + j) % NB))) break;
        if (!ok) break;
      }
      bool first = true;  // no P.V of this unit issued yet
      for (int J = 0; J < n && ok; ++J, ++tc) {
        const uint32_t b = tc % NB, ppar = (tc / NB) & 1;
        if constexpr (CALIB) {
          // The softmax has read the scores (both halves arrive per tile).
          if (!(ok = wait_all(&c->ph_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL))) break;
          if (!(ok = wait_all(&c->p_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL))) break;
          tc_fence_after();
          if (J + NB < n && !(ok = issue_s(J + NB, n, b))) break;
          continue;
        }
        // The decision first: a skipped tile needs nothing else, and each
        // shared-memory access of this warp (probes included) queues behind
        // the operand reads of the MMAs in flight.  A kept tile then probes
        // V and both halves of P back to back and blocks only on what is
        // missing.  Warp-uniform: a phase counts as complete when every lane
        // saw it so.
        const uint32_t vst = vc % VSTN;
        bool keep = true;
        if (triv && (!CORR || J < nk)) {
          // keep
        } else if constexpr (GATING && SPLIT) {
          // Q.K^T run ahead of this warp through skipped tiles, so the word
          // may already carry a later tile's decision: that means tile tc was
          // skipped (a kept tile's buffer takes no later Q.K^T before this
          // warp's P.V of it), and a reader that is behind never waits on a
          // phase by parity alone.
          const uint32_t w = wait_decision<NB>(&c->dec[b], &c->dec_full[b], tc, abort, p.err, &ok);
          if (!ok) break;
          keep = stamp_dist(w, tc) == 0 && (w & DEC_MASK) != 0u;
        } else if constexpr (GATING) {
          // Lane 0's reading of the word, for the whole warp.
          uint32_t w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          if ((w >> DEC_BITS) != (tc & DEC_STAMP_MASK)) {  // not published yet
            if (!(ok = wait_all(&c->dec_full[b], ppar, abort, p.err, ERR_WAIT_DEC))) break;
            w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          }
          keep = (w & DEC_MASK) != 0u;
        }
        bool v_ok = false, ph_ok = false, p_ok = false;
        if (keep || (GATING && VALL))
          v_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->v_full[vst], (vc / VSTN) & 1));
        if (keep) {
          ph_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->ph_full[b], ppar));
          p_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->p_full[b], ppar));
        }
        const bool vload = keep || (GATING && VALL);  // this tile's V stage was filled
        if (vload && !v_ok &&
            !(ok = wait_all(&c->v_full[vst], (vc / VSTN) & 1, abort, p.err, ERR_WAIT_V_FULL)))
          break;
        if (keep) {
          if (PAGED && J == n - 1) {
            // Keys of the last tile past the sequence end: a paged pool may
            // hold anything there (NaN included), and P = 0 does not cancel
            // NaN in P.V.
            const int valid = p.seqinfo[t.x].y - J * TILE;
            if (valid < TILE) zero_tile_rows<D>(sV + vst * TKV, valid, lane);
          }
          uint32_t acc = 1u;
          if (first) {
            if (!(ok = wait_all(&c->o_empty, (uc & 1) ^ 1, abort, p.err, ERR_WAIT_O_EMPTY)))
              break;
            acc = 0u;
            first = false;
          }
          const uint32_t d_p = tmem + b * 128;
          const uint64_t dv_st = dV + ((vst * TKV) >> 4);
          if (ph_ok && p_ok) {
            tc_fence_after();
            if (elect_one()) xs_issue_pv(d_o, d_p, dv_st, IDESC_PV, acc, 0, KSTEPS);
            __syncwarp();
          } else {
            if (!ph_ok && !(ok = wait_all(&c->ph_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL)))
              break;
            tc_fence_after();
            if (elect_one()) xs_issue_pv(d_o, d_p, dv_st, IDESC_PV, acc, 0, KHALFSTEPS);
            __syncwarp();
            if (!p_ok && !(ok = wait_all(&c->p_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL)))
              break;
            tc_fence_after();
            if (elect_one()) xs_issue_pv(d_o, d_p, dv_st, IDESC_PV, 1u, KHALFSTEPS, KSTEPS);
            __syncwarp();
          }
        } else {
          // A skipped tile has no P: its scores were read before the vote
          // barrier that preceded the decision, so the buffer may be refilled.
          tc_fence_after();
        }
        if (elect_one()) {
          if (keep) {
            umma_commit(&c->pv_done[kp & 1]);
            if (SPLIT) umma_commit(&c->buf_free[b]);
          }
          if (vload) umma_commit(&c->v_empty[vst]);
        }
        __syncwarp();
        if (keep) ++kp;
        if (vload) ++vc;
        if constexpr (!SPLIT) {
          if (J + NB < n && !(ok = issue_s(J + NB, n, b))) break;
        }
      }
      if (!ok) break;
      if constexpr (!CALIB) {
        if (elect_one()) umma_commit(&c->o_full);
        __syncwarp();
      }
    }
    // Drain: every issued MMA completes before TMEM can be released.
    if (elect_one()) umma_commit(&c->drain);
    __syncwarp();
    drain_wait(&c->drain, 0);
  } else if (SPLIT && warp == 2) {
    // ------------------------------------------------------ Q.K^T issuer
    // Q.K^T number g (the CTA's g-th tile, in unit order) goes into score
    // buffer g % NB once tile g - NB is done with it (buf_free: the softmax
    // arrives for a skip, the P.V issuer commits after a kept tile's P.V)
    // and K tile g has landed.  Its commit on s_full also frees K stage g %
    // KST when KST == NB.  Probes first, waits only on what is missing.
    constexpr uint32_t IDESC_QK = idesc_f32acc<F16>(128, BK, false, false);
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    uint32_t g = 0, uc = 0;
    bool ok = true;
    for (XsUnits it(per_kv, p.Hkv); ok && it.valid(); it.next(), ++uc) {
      const int u = it.u;
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int n = xs_ntiles<BK>(t.y, p.seqinfo[t.x].y) + (CORR ? (t.y + TILE - 1) / TILE : 0);
      if (!(ok = wait_all(&c->q_full, uc & 1, abort, p.err, ERR_WAIT_Q_FULL))) break;
      for (int j = 0; j < n; ++j, ++g) {
        const uint32_t b = g % NB, kst = g % KST;
        const uint32_t fpar = ((g / NB) & 1) ^ 1, kpar = (g / KST) & 1;
        const bool f_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->buf_free[b], fpar));
        const bool k_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->k_full[kst], kpar));
        if (!f_ok && !(ok = wait_all(&c->buf_free[b], fpar, abort, p.err, ERR_WAIT_P_FULL)))
          break;
        if (!k_ok && !(ok = wait_all(&c->k_full[kst], kpar, abort, p.err, ERR_WAIT_K_FULL)))
          break;
        tc_fence_after();
        if (elect_one()) {
          xs_issue_qk<D, BK>(tmem + b * 128, dQ, dK + ((kst * TKV) >> 4), IDESC_QK);
          umma_commit(&c->s_full[b]);
          if constexpr (KST != NB) umma_commit(&c->k_empty[kst]);
          if (j == n - 1) umma_commit(&c->q_empty);
        }
        __syncwarp();
      }
    }
    if (elect_one()) umma_commit(&c->drain_qk);
    __syncwarp();
    drain_wait(&c->drain_qk, 0);
  } else if (warp < 4) {
    // idle
  } else {
    // -------------------------------------------------------------- softmax
    // Warp 4 + 4 ch + wq: rows 32 wq .. 32 wq + 31, keys [HK ch, HK ch + HK)
    // of each tile.  A thread loads its HK scores once (the reducing TMEM
    // load also gives their maximum), votes, and takes its exp pass from
    // registers.  One barrier per tile joins the 256 softmax threads: its
    // count carries the gate's vote, the failure consensus and whether some
    // row needs the exact maximum of its two halves (a rise of the lazily
    // rescaled reference, or of the lambda running max); only then are the
    // half maxima exchanged through shared memory.
    constexpr int HK = BK / 2, NCH = HK / 32, TAIL = HK % 32;  // TAIL is 0 or 16
    static_assert(TAIL == 0 || TAIL == 16, "key split");
    const int ch = (warp - 4) >> 2;  // column half
    const int wq = warp & 3;         // TMEM lane quarter
    const int row = wq * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(wq * 32) << 16;
    constexpr int DH = D / 2;        // my output columns
    const uint32_t tO = tmem + tlane + LY::O_COL + ch * DH;
    // Counts and bitmap words: every lane of warp 4 keeps them (lane 0 stores).
    const bool lead_warp = warp == 4;
    constexpr uint32_t bar_id = 1;
    constexpr uint32_t NBAR = 256;
    const float sc = p.sigma_log2;
    const bool lambda_mode = GATING && !CALIB && p.mode == 1;
    // ln(lambda) = -inf keeps every block: no running max to keep exact, so
    // no exchange of half-row maxima for it.
    const bool lambda_vote = lambda_mode && p.log_lambda != -CUDART_INF_F;
    uint32_t tc = 0, uc = 0;
    uint32_t kn = 0;  // kept tiles so far (pv_done phases)
    bool ok = true;
    uint32_t cnt_kept = 0, cnt_cand = 0, cnt_diag = 0;

    for (XsUnits it(per_kv, p.Hkv); ok && it.valid(); it.next(), ++uc) {
      const int u = it.u;
      int I, len, h;
      {
        const int kvh = u / per_kv, rem = u - kvh * per_kv;
        const int2 t = p.tiles[rem / p.group];
        I = t.y;
        len = p.seqinfo[t.x].y;
        h = kvh * p.group + rem % p.group;
      }
      const int n = xs_ntiles<BK>(I, len);
      const int rabs = I * TILE + row;  // my row's position in the sequence
      const bool rvalid = rabs < len;
      float tq = 0.f;
      if (GATING && !CALIB && p.mode == 0) tq = p.thr[(long long)h * p.nT + min(I, p.nT - 1)];
      // m_used: reference of P (trails the running max by at most 2^8 in P
      // units); m_true: exact running max over kept blocks (lambda gate); l:
      // this half's share of the normaliser.
      float m_used = -CUDART_INF_F, m_true = -CUDART_INF_F, l = 0.f;
      bool o_init = false;
      bool prev_kept = false;  // lambda vote: the unit's previous tile was kept
      uint32_t bm_word = 0;

      for (int J = 0; J < n; ++J, ++tc) {
        const uint32_t b = tc % NB;
        // Every thread reaches the tile barrier below, also after its own
        // bounded wait gave up, so the 256 threads leave together.
        const bool okl = wait_bar(&c->s_full[b], (tc / NB) & 1, abort, p.err, ERR_WAIT_S_FULL);
        __syncwarp();  // the TMEM loads below are warp-wide
        tc_fence_after();
        // A candidate: every key precedes the query tile's first row; any
        // other visible tile is in the diagonal region (kept, masked).
        const bool cand = (J + 1) * BK <= I * TILE;
        const int kbase = J * BK + ch * HK;  // position of my first key
        const uint32_t tS = tmem + tlane + b * 128 + ch * HK;  // my score columns

        // ---- my HK scores and their maximum (masked outside the candidates)
        uint32_t sr[NCH][32];
        uint32_t stl[16];
        float lm = -CUDART_INF_F;
        {
          float qm[NCH];
#pragma unroll
          for (int q = 0; q < NCH; ++q) tmem_ld32_max(tS + q * 32, sr[q], qm[q]);
          if constexpr (TAIL > 0) tmem_ld16(tS + NCH * 32, stl);
          // Lambda vote: the other half's maximum of the previous (kept) tile,
          // stored before that tile's barrier, joins the running max here,
          // while the TMEM loads are in flight.
          if (lambda_vote && prev_kept)
            m_true = fmaxf(m_true, c->xmax[(tc - 1) & 1][ch ^ 1][row]);
          tmem_wait_ld();
          if (cand) {
#pragma unroll
            for (int q = 0; q < NCH; ++q) lm = fmaxf(lm, qm[q]);
#pragma unroll
            for (int e = 0; e < TAIL; ++e) lm = fmaxf(lm, __uint_as_float(stl[e]));
          } else {
#pragma unroll
            for (int e = 0; e < HK; ++e) {
              const float x = __uint_as_float(e < NCH * 32 ? sr[e >> 5][e & 31] : stl[e & 15]);
              if (kbase + e <= rabs) lm = fmaxf(lm, x);
            }
          }
        }

        if constexpr (CALIB) {
          // sigma * (tile maximum) of a candidate: the maximum over the valid
          // rows of both halves, combined through shared memory.
          const float wm = warp_max_f32(rvalid ? lm : -CUDART_INF_F);
          if (lane == 0) c->xw[tc & 1][warp - 4] = wm;
          tc_fence_before();
          ok = bar_red_and(bar_id, NBAR, okl);
          if (!ok) break;
          if (cand && threadIdx.x == 128) {
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < 8; ++w) mx = fmaxf(mx, c->xw[tc & 1][w]);
            p.blockmax[((long long)h * p.cal_nq + I) * p.cal_nk + J] = mx * p.sigma;
          }
          mbar_arrive(ch == 0 ? &c->ph_full[b] : &c->p_full[b]);
          continue;
        }

        // ---- votes.  Threshold: my half of the row wants the tile when
        // sigma * (half max) >= T; the tile maximum clears T exactly when some
        // half row does.  Lambda: a row wants the tile when
        // sigma * (rowmax - m_true) >= ln(lambda); m_true is the same in both
        // halves of a row, so this is the OR of the halves' tests.
        bool want = false;
        if constexpr (GATING) {
          if (!lambda_mode) want = rvalid && lm * p.sigma >= tq;
          else want = rvalid && (lm - m_true) * p.sigma >= p.log_lambda;
        }
        // With a lambda vote each half stores its maximum before the tile
        // barrier, every tile; the other half folds it into its running max
        // at the next tile (above), which is the first vote that needs it.
        // The exchange after the barrier happens only when some row needs the
        // exact maximum now (a rise of the lazily rescaled reference).
        if (lambda_vote) c->xmax[tc & 1][ch][row] = lm;
        const bool need_x = rvalid && (lm - m_used) * sc > RESCALE_LOG2;
        // Every read of S is complete (tcgen05.wait::ld above); the fence
        // orders it before the barrier, after which the MMA warp may refill a
        // skipped tile's buffer and the other half's P may overwrite my
        // score columns.
        tc_fence_before();
        // The barrier's count is X + 16 V: lane 0 of each warp counts 1 when
        // a lane stopped or needs the exchange, lanes 1..16 count 1 each when
        // a row of the warp wants the tile (X, V <= 8).
        const bool wx = __any_sync(0xffffffffu, !okl || need_x);
        const bool wv = __any_sync(0xffffffffu, want);
        const uint32_t nv = bar_red_popc(bar_id, NBAR, lane == 0 ? wx : (lane <= 16 && wv));
        const bool kept = !GATING || !cand || nv >= 16u;
        float rowmax = lm;  // the row's maximum over both halves (exact when exchanged)
        const bool exact = (nv & 15u) != 0u;
        if ((nv & 15u) != 0u) {  // an exchange, or a thread that stopped
          if (!lambda_vote) c->xmax[tc & 1][ch][row] = lm;
          ok = bar_red_and(bar_id, NBAR, okl);
          if (!ok) break;
        }
        if (exact) rowmax = fmaxf(lm, c->xmax[tc & 1][ch ^ 1][row]);
        if (lambda_mode && kept) m_true = fmaxf(m_true, rowmax);
        prev_kept = kept;
        if (GATING && lead_warp) {  // all 32 lanes: same value, 32 arrivals
          st_release_u32(&c->dec[b], ((tc & DEC_STAMP_MASK) << DEC_BITS) | (kept ? 1u : 0u));
          mbar_arrive(&c->dec_full[b]);
          // A skipped tile's buffer is free: every read of its scores was
          // fenced before the barrier above.
          if (SPLIT && !kept && elect_one()) mbar_arrive(&c->buf_free[b]);
          __syncwarp();
        }

        // ---- online softmax over my half of a kept tile
        if (kept) {
          if (exact) {  // rowmax is exact: rescale when the reference must rise
            const float m_new = fmaxf(m_used, rowmax);
            const bool resc = (m_new - m_used) * sc > RESCALE_LOG2;
            float alpha = 1.f;
            if (resc) {
              alpha = ex2_approx((m_used - m_new) * sc);
              m_used = m_new;
              l *= alpha;
            }
            // O may still be accumulating an earlier tile's P.V (with several
            // score buffers this tile's Q.K^T was issued before it): wait
            // until every P.V so far is done.  The TMEM loads and stores are
            // warp-wide, so the warp rescales together, with alpha = 1 in rows
            // that keep their reference.  A wait that gives up raises the
            // abort flag, which the next tile barrier turns into a common exit.
            if (o_init && __any_sync(0xffffffffu, resc)) {
              wait_bar(&c->pv_done[(kn - 1) & 1], ((kn - 1) >> 1) & 1, abort, p.err,
                       ERR_WAIT_O_FULL);
              __syncwarp();
              tc_fence_after();
#pragma unroll 1
              for (int q = 0; q < DH / 16; ++q) {
                uint32_t orr[16];
                tmem_ld16(tO + q * 16, orr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_st16(tO + q * 16, orr);
              }
            }
          }
          // P = exp2(sigma*log2e*(S - m_used)) over my visible keys, packed as
          // 16-bit pairs into my HK/2 P columns of the tile's score buffer.
          const uint32_t tP = tmem + tlane + b * 128 + ch * (HK / 2);
          const float mb = (m_used == -CUDART_INF_F) ? 0.f : m_used * sc;
          const uint64_t sc2 = f2_pack(sc, sc), nmb2 = f2_pack(-mb, -mb);
          uint64_t lsum2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < NCH; ++q) {  // 32 of my keys per step, 16 P columns
            uint32_t pk[16];
            if (cand) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const uint64_t x2 = f2_pack(__uint_as_float(sr[q][2 * e]),
                                            __uint_as_float(sr[q][2 * e + 1]));
                float y0, y1;
                f2_unpack(f2_fma(x2, sc2, nmb2), y0, y1);
                const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                lsum2 = f2_add(lsum2, f2_pack(p0, p1));
                pk[e] = pack_x2<F16>(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int key = kbase + q * 32 + 2 * e;
                const float x0 = __uint_as_float(sr[q][2 * e]);
                const float x1 = __uint_as_float(sr[q][2 * e + 1]);
                const float p0 = key <= rabs ? ex2_approx(fmaf(x0, sc, -mb)) : 0.f;
                const float p1 = key + 1 <= rabs ? ex2_approx(fmaf(x1, sc, -mb)) : 0.f;
                lsum2 = f2_add(lsum2, f2_pack(p0, p1));
                pk[e] = pack_x2<F16>(p0, p1);
              }
            }
            tmem_st16(tP + q * 16, pk);
          }
          if constexpr (TAIL > 0) {  // the last 16 of my keys, 8 P columns
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int key = kbase + NCH * 32 + 2 * e;
              const float x0 = __uint_as_float(stl[2 * e]);
              const float x1 = __uint_as_float(stl[2 * e + 1]);
              const float p0 = (cand || key <= rabs) ? ex2_approx(fmaf(x0, sc, -mb)) : 0.f;
              const float p1 = (cand || key + 1 <= rabs) ? ex2_approx(fmaf(x1, sc, -mb)) : 0.f;
              lsum2 = f2_add(lsum2, f2_pack(p0, p1));
              pk[e] = pack_x2<F16>(p0, p1);
            }
            tmem_st8(tP + NCH * 16, pk);
          }
          float ls0, ls1;
          f2_unpack(lsum2, ls0, ls1);
          l += ls0 + ls1;
          tmem_wait_st();
          o_init = true;
          ++kn;
        }
        // My half of P is written (or the tile skipped): one arrival per
        // thread and tile on this half's barrier (first half: ph_full).
        tc_fence_before();
        mbar_arrive(ch == 0 ? &c->ph_full[b] : &c->p_full[b]);

        // ---- bookkeeping: bitmap words and block counts (lead warp)
        if (lead_warp) {
          if (cand) {
            ++cnt_cand;
            cnt_kept += kept ? 1u : 0u;
          } else {
            ++cnt_diag;
          }
          if (kept) bm_word |= 1u << (J & 31);
          // Mean correction: the kept bits of the candidates, complete before
          // the diagonal tile's barrier, which every correction tile follows.
          if (CORR && cand && lane == 0 && ((J & 31) == 31 || J == I - 1))
            c->kbits[J >> 5] = bm_word;
          if ((p.bitmap != nullptr || CORR) && ((J & 31) == 31 || J == n - 1)) {
            if (p.bitmap != nullptr) {
              const int4 si = p.seqinfo[p.tiles[(u % per_kv) / p.group].x];
              if (lane == 0)
                p.bitmap[((long long)(si.z + I) * p.Hq + h) * (long long)p.words + (J >> 5)] =
                    bm_word;
            }
            bm_word = 0;
          }
        }
      }
      if (!ok) break;
      if constexpr (CALIB) continue;

      if constexpr (CORR) {
        // ---- correction tiles, a loop of their own so that the key tiles'
        // loop stays as without the option.  Tile ci holds the means of key
        // blocks [128 ci, 128 ci + 128); my 64 entries are blocks kb0 ..
        // kb0 + 63.  An entry enters when its block is a candidate (block <
        // I) that this head skipped (the kept bits are complete: the diagonal
        // tile's barrier came after the last of them), with ln(Bk) added to
        // its logit (corr_shift, raw score units).  The tile is kept when
        // some entry enters; then the same vote barrier, exchange, rescale and
        // P hand-off as a key tile.
        const int nct = (I + TILE - 1) / TILE;
        for (int ci = 0; ci < nct; ++ci, ++tc) {
          const uint32_t b = tc % NB;
          const bool okl = wait_bar(&c->s_full[b], (tc / NB) & 1, abort, p.err, ERR_WAIT_S_FULL);
          __syncwarp();
          tc_fence_after();
          const int kb0 = ci * TILE + ch * HK;
          const uint32_t tS = tmem + tlane + b * 128 + ch * HK;
          uint32_t sr[2][32], inc[2];
          tmem_ld32(tS, sr[0]);
          tmem_ld32(tS + 32, sr[1]);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int lim = I - kb0 - 32 * q;
            const uint32_t cm = lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : (1u << lim) - 1u);
            inc[q] = lim > 0 ? cm & ~c->kbits[(kb0 >> 5) + q] : 0u;
          }
          tmem_wait_ld();
          float lm = -CUDART_INF_F;
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if ((inc[q] >> e) & 1u) lm = fmaxf(lm, __uint_as_float(sr[q][e]));
          if (lm != -CUDART_INF_F) lm += p.corr_shift;
          const bool need_x = rvalid && (lm - m_used) * sc > RESCALE_LOG2;
          tc_fence_before();
          const bool wx = __any_sync(0xffffffffu, !okl || need_x);
          const bool wv = (inc[0] | inc[1]) != 0u;  // the same in every row of my half
          const uint32_t nv = bar_red_popc(bar_id, NBAR, lane == 0 ? wx : (lane <= 16 && wv));
          const bool kept = nv >= 16u;
          float rowmax = lm;
          const bool exact = (nv & 15u) != 0u;
          if (exact) {
            c->xmax[tc & 1][ch][row] = lm;
            ok = bar_red_and(bar_id, NBAR, okl);
            if (!ok) break;
            rowmax = fmaxf(lm, c->xmax[tc & 1][ch ^ 1][row]);
          }
          if (lead_warp) {
            st_release_u32(&c->dec[b], ((tc & DEC_STAMP_MASK) << DEC_BITS) | (kept ? 1u : 0u));
            mbar_arrive(&c->dec_full[b]);
            if (!kept && elect_one()) mbar_arrive(&c->buf_free[b]);
            __syncwarp();
          }
          if (kept) {
            if (exact) {
              const float m_new = fmaxf(m_used, rowmax);
              const bool resc = (m_new - m_used) * sc > RESCALE_LOG2;
              float alpha = 1.f;
              if (resc) {
                alpha = ex2_approx((m_used - m_new) * sc);
                m_used = m_new;
                l *= alpha;
              }
              if (o_init && __any_sync(0xffffffffu, resc)) {
                wait_bar(&c->pv_done[(kn - 1) & 1], ((kn - 1) >> 1) & 1, abort, p.err,
                         ERR_WAIT_O_FULL);
                __syncwarp();
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < DH / 16; ++q) {
                  uint32_t orr[16];
                  tmem_ld16(tO + q * 16, orr);
                  tmem_wait_ld();
#pragma unroll
                  for (int e = 0; e < 16; ++e)
                    orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                  tmem_st16(tO + q * 16, orr);
                }
              }
            }
            const uint32_t tP = tmem + tlane + b * 128 + ch * (HK / 2);
            const float bias =
                p.corr_shift * sc - ((m_used == -CUDART_INF_F) ? 0.f : m_used * sc);
            float lsum = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float x0 = __uint_as_float(sr[q][2 * e]);
                const float x1 = __uint_as_float(sr[q][2 * e + 1]);
                const float p0 =
                    ((inc[q] >> (2 * e)) & 1u) ? ex2_approx(fmaf(x0, sc, bias)) : 0.f;
                const float p1 =
                    ((inc[q] >> (2 * e + 1)) & 1u) ? ex2_approx(fmaf(x1, sc, bias)) : 0.f;
                lsum += p0 + p1;
                pk[e] = pack_x2<F16>(p0, p1);
              }
              tmem_st16(tP + q * 16, pk);
            }
            l += lsum;
            tmem_wait_st();
            o_init = true;
            ++kn;
          }
          tc_fence_before();
          mbar_arrive(ch == 0 ? &c->ph_full[b] : &c->p_full[b]);
        }
        if (!ok) break;
      }

      // ---- epilogue: O / l -> 16-bit, log-sum-exp, bitmap tail
      const int4 si = p.seqinfo[p.tiles[(u % per_kv) / p.group].x];
      if (lead_warp && p.bitmap != nullptr) {
        const long long bm_row = ((long long)(si.z + I) * p.Hq + h) * (long long)p.words;
        for (int w = ((n - 1) >> 5) + 1 + lane; w < p.words; w += 32) p.bitmap[bm_row + w] = 0u;
      }
      c->xl[ch][row] = l;
      {
        const bool okl = wait_bar(&c->o_full, uc & 1, abort, p.err, ERR_WAIT_O_FULL);
        if (!(ok = bar_red_and(bar_id, NBAR, okl))) break;
      }
      tc_fence_after();
      const float lt = l + c->xl[ch ^ 1][row];
      const float inv_l = (lt > 0.f) ? 1.f / lt : 0.f;
      uint16_t* orow = p.o + (long long)si.w * p.o_sb + (long long)h * p.o_sh +
                       (long long)(si.x + rabs) * p.o_st + ch * DH;
#pragma unroll
      for (int q = 0; q < DH / 16; ++q) {
        uint32_t orr[16];
        tmem_ld16(tO + q * 16, orr);
        tmem_wait_ld();
        if (rvalid) {
          uint4 pk4[2];
          uint32_t* pw = reinterpret_cast<uint32_t*>(pk4);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pw[e] = pack_x2<F16>(__uint_as_float(orr[2 * e]) * inv_l,
                                 __uint_as_float(orr[2 * e + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 16);
          dst[0] = pk4[0];
          dst[1] = pk4[1];
        }
      }
      if (ch == 0 && p.lse != nullptr && rvalid)
        p.lse[(long long)h * p.lse_rows +
              (p.varlen ? (long long)si.x : (long long)si.w * p.batch_len) + rabs] =
            m_used * p.sigma + logf(lt);
      // The next unit's first P.V overwrites O once all 256 threads are here.
      tc_fence_before();
      mbar_arrive(&c->o_empty);
    }
    if (!CALIB && p.counts != nullptr && lead_warp && lane == 0 && (cnt_cand | cnt_diag) != 0u) {
      atomicAdd(&p.counts[0], (unsigned long long)cnt_kept);
      atomicAdd(&p.counts[1], (unsigned long long)cnt_cand);
      atomicAdd(&p.counts[2], (unsigned long long)cnt_diag);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, LY::NCOLS);
  }
}

}  // namespace bsfa
