// bsfa_xs.cuh -- the pipelined gated prefill kernel for 128 x 128 semantic
// blocks: one query head per CTA, the scores of key tiles t and t+1 in two
// TMEM buffers, so that Q.K^T of tile t+2 is issued as soon as tile t's gate
// decision (a skip) or its P (a keep) is in.  The gate then sits on the
// softmax warps' path only, not on the tensor pipe's: a run of skipped
// tiles streams Q.K^T back to back.
//
// What it computes is the same gated, renormalised attention as
// bsfa_fwd_kernel ("Block Sparse Flash Attention", Key Designs 2 and 3;
// the lambda gate of "Skipping attention blocks was the easy part", section
// "Vote, then skip"): every visible 128 x 128 tile's scores are computed,
// the tile maximum (or each row's maximum against its running max) decides
// the tile, and a skipped tile gets no V load, no exp and no P.V.  The
// schedule follows that page's "Cross-stage P" section in spirit: the next
// tile's Q.K^T does not wait for the current tile's P.V.
//
// Roles (384 threads, one CTA per SM, persistent over a heaviest-first
// list of (KV head, query tile, query head) units):
//   warp 0      TMA producer: Q per unit, K for every visible tile (3-stage
//               ring), V for every tile when the gate is compiled out.
//   warp 1      MMA issuer, TMEM owner.
//   warp 3      (gate on) V loader: V of the tiles the gate keeps.
//   warps 4-11  softmax: warp 4 + 4 ch + wq holds, for rows 32 wq .. 32 wq
//               + 31, the tile's keys [64 ch, 64 ch + 64).
//
// TMEM: S buffers at columns [0, 128) and [128, 256) (tile t uses buffer
// t % 2; P overwrites its first 64 columns as 16-bit pairs), O at [256,
// 256 + D).
#pragma once
#include "bsfa_fwd.cuh"

namespace bsfa {

constexpr int XS_KST = 3;  // K ring stages (Q.K^T runs up to two tiles ahead)
constexpr int XS_VST = 2;  // V ring stages

struct XsCtrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[XS_KST], k_empty[XS_KST];
  uint64_t v_full[XS_VST], v_empty[XS_VST];
  uint64_t s_full[2];    // per S buffer: scores of its current tile ready
  uint64_t ph_full[2];   // per S buffer: P of keys 0-63 written (or tile skipped), 128 arrivals
  uint64_t p_full[2];    // per S buffer: P of keys 64-127 written (or tile skipped), 128 arrivals
  uint64_t dec_full[2];  // per S buffer: decision word published, 32 arrivals
  uint64_t pv_done[2];   // per tile parity: that tile's P.V (if any) and all before it complete
  uint64_t o_full, o_empty;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t dec[2];       // per S buffer: tile stamp << DEC_BITS | keep bit
  float xmax[2][2][128]; // per (tile parity, column half, row): half-row maximum
  float xl[2][128];      // per (column half, row): share of the normaliser
  int abort;
};

template <int D>
struct XsLayout {
  static constexpr int TB = TILE * D * 2;  // bytes of one 128-row 16-bit tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TB;
  static constexpr int V_OFF = K_OFF + XS_KST * TB;
  static constexpr int C_OFF = V_OFF + XS_VST * TB;
  static constexpr int RAW = C_OFF + (((int)sizeof(XsCtrl) + 15) & ~15) + 1024;
  // At least 120 KB, so that one CTA is resident per SM (the persistent grid
  // and the whole-TMEM allocation assume it).
  static constexpr int BYTES = RAW > 120 * 1024 ? RAW : 120 * 1024;
  static constexpr int NCOLS = 512;
  static constexpr int NTHREADS = 384;
  static constexpr uint32_t O_COL = 256;
};

// Signed distance, modulo the 28-bit decision stamp, of a decision word's
// stamp from tile counter tc (the initial word 0xFFFFFFFF reads as -1 at 0).
__device__ __forceinline__ int32_t xs_stamp_dist(uint32_t w, uint32_t tc) {
  return static_cast<int32_t>(((w >> DEC_BITS) - tc) << (32 - 28)) >> (32 - 28);
}

template <int D, bool GATING, bool F16, bool VALL, bool PAGED>
__global__ void __launch_bounds__(384, 1)
    bsfa_xs_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const DevParams p) {
  using LY = XsLayout<D>;
  constexpr int TB = LY::TB;
  constexpr int HALF = TILE * 128;  // bytes of one 64-column swizzled half
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
    for (int i = 0; i < XS_KST; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < XS_VST; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c->s_full[b], 1);
      mbar_init(&c->ph_full[b], 128);
      mbar_init(&c->p_full[b], 128);
      mbar_init(&c->dec_full[b], 32);
      mbar_init(&c->pv_done[b], 1);
      c->dec[b] = 0xFFFFFFFFu;  // no stamp matches
    }
    mbar_init(&c->o_full, 1);
    mbar_init(&c->o_empty, 256);
    mbar_init(&c->drain, 1);
    c->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
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
  const int total_units = per_kv * p.Hkv;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t kc = 0, vc = 0, uc = 0;
    int last_q = -1;  // index of the last unit whose Q load was issued
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int h = kvh * p.group + rem % p.group;
      const int4 si = p.seqinfo[t.x];
      const int n = t.y + 1;
      if (!(ok = wait_all(&c->q_empty, (uc & 1) ^ 1, abort, p.err, ERR_WAIT_Q_EMPTY))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&c->q_full, TB);
        for (int hf = 0; hf < NHALF; ++hf)
          tma_load_4d(sQ + hf * HALF, &tmQ, &c->q_full, hf * 64, si.x + t.y * TILE, h, si.w);
      }
      __syncwarp();
      last_q = static_cast<int>(uc);
      for (int J = 0; J < n; ++J) {
        {
          const uint32_t st = kc % XS_KST;
          const int2 cc = kv_tile_coord<PAGED>(p, si, t.x, J);  // before the wait
          if (!(ok = wait_all(&c->k_empty[st], ((kc / XS_KST) & 1) ^ 1, abort, p.err,
                              ERR_WAIT_K_EMPTY)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&c->k_full[st], TB);
            for (int hf = 0; hf < NHALF; ++hf)
              tma_load_4d(sK + st * TB + hf * HALF, &tmK, &c->k_full[st], hf * 64, cc.x, kvh, cc.y);
          }
          __syncwarp();
          ++kc;
        }
        if constexpr (!GATING) {
          const uint32_t st = vc % XS_VST;
          const int2 cc = kv_tile_coord<PAGED>(p, si, t.x, J);
          if (!(ok = wait_all(&c->v_empty[st], ((vc / XS_VST) & 1) ^ 1, abort, p.err,
                              ERR_WAIT_V_EMPTY)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&c->v_full[st], TB);
            for (int hf = 0; hf < NHALF; ++hf)
              tma_load_4d(sV + st * TB + hf * HALF, &tmV, &c->v_full[st], hf * 64, cc.x, kvh, cc.y);
          }
          __syncwarp();
          ++vc;
        }
      }
    }
    if (!ok) {
      // Let every copy already issued land before the CTA can exit.
      if (last_q >= 0) drain_wait(&c->q_full, last_q & 1);
      for (uint32_t i = 0; i < XS_KST && i < kc; ++i) {
        const uint32_t f = kc - 1 - i;
        drain_wait(&c->k_full[f % XS_KST], (f / XS_KST) & 1);
      }
      for (uint32_t i = 0; i < XS_VST && i < vc; ++i) {
        const uint32_t f = vc - 1 - i;
        drain_wait(&c->v_full[f % XS_VST], (f / XS_VST) & 1);
      }
    }
  } else if (GATING && warp == 3) {
    // ----------------------------------------------------- V loader (gated)
    // V of a tile is requested as soon as the softmax publishes a keep (with
    // VALL: for every tile, as soon as a stage is free).
    uint32_t vc = 0, tc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int4 si = p.seqinfo[t.x];
      const int n = t.y + 1;
      for (int J = 0; J < n; ++J, ++tc) {
        const int2 cc = kv_tile_coord<PAGED>(p, si, t.x, J);  // before the waits
        bool need = VALL;
        if constexpr (!VALL) {
          // The decision word of the tile's S buffer carries the tile stamp.  A
          // word stamped with a later tile also means a skip: a kept tile's
          // P.V waits for its V, and the next Q.K^T into that buffer (whose
          // decision overwrites the word) is issued only after that P.V.  Only
          // a word from an earlier tile needs the wait; then the barrier's
          // phase for this tile has not completed, so its parity is safe.
          const uint32_t b = tc & 1;
          uint32_t w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          if (xs_stamp_dist(w, tc) < 0) {
            if (!(ok = wait_all(&c->dec_full[b], (tc >> 1) & 1, abort, p.err, ERR_WAIT_DEC)))
              break;
            w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          }
          need = xs_stamp_dist(w, tc) == 0 && (w & DEC_MASK) != 0u;
        }
        if (!need) continue;
        const uint32_t st = vc % XS_VST;
        if (!(ok = wait_all(&c->v_empty[st], ((vc / XS_VST) & 1) ^ 1, abort, p.err,
                            ERR_WAIT_V_EMPTY)))
          break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&c->v_full[st], TB);
          for (int hf = 0; hf < NHALF; ++hf)
            tma_load_4d(sV + st * TB + hf * HALF, &tmV, &c->v_full[st], hf * 64, cc.x, kvh, cc.y);
        }
        __syncwarp();
        ++vc;
      }
    }
    if (!ok) {
      for (uint32_t i = 0; i < XS_VST && i < vc; ++i) {
        const uint32_t f = vc - 1 - i;
        drain_wait(&c->v_full[f % XS_VST], (f / XS_VST) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and the waits; one elected lane issues
    // every MMA and commit.  Per unit: Q.K^T of tiles 0 and 1, then for each
    // tile t: its decision; if kept, P.V (P in two halves); the commit of
    // pv_done; then Q.K^T of tile t + 2 into t's S buffer (in issue order
    // after t's P.V, which reads P from that buffer).
    constexpr uint32_t IDESC_QK = idesc_f32acc<F16>(128, 128, false, false);
    constexpr uint32_t IDESC_PV = idesc_f32acc<F16>(128, D, false, true);
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sV), HALF, 1024);
    const uint32_t d_o = tmem + LY::O_COL;
    uint32_t kc = 0, vc = 0, tc = 0, uc = 0;
    bool ok = true;
    // Q.K^T of the unit's tile j (j = tile index) into S buffer b.
    auto issue_s = [&](int j, int n, uint32_t b) -> bool {
      const uint32_t kst = kc % XS_KST;
      if (!__all_sync(0xffffffffu, mbar_test_wait(&c->k_full[kst], (kc / XS_KST) & 1)) &&
          !wait_all(&c->k_full[kst], (kc / XS_KST) & 1, abort, p.err, ERR_WAIT_K_FULL))
        return false;
      if (elect_one()) {
        issue_qk<D, 1>(tmem + b * 128, dQ, dK + ((kst * TB) >> 4), IDESC_QK);
        umma_commit(&c->s_full[b]);
        umma_commit(&c->k_empty[kst]);
        if (j == n - 1) umma_commit(&c->q_empty);
      }
      __syncwarp();
      ++kc;
      return true;
    };
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.group];
      const int n = t.y + 1;
      if (!(ok = wait_all(&c->q_full, uc & 1, abort, p.err, ERR_WAIT_Q_FULL))) break;
      tc_fence_after();
      for (int j = 0; j < 2 && j < n; ++j)
        if (!(ok = issue_s(j, n, (tc + j) & 1))) break;
      if (!ok) break;
      bool first = true;  // no P.V of this unit issued yet
      for (int J = 0; J < n && ok; ++J, ++tc) {
        const uint32_t b = tc & 1, ppar = (tc >> 1) & 1;
        // Probe everything this step may need back to back (one shared-memory
        // round trip), then block only on what is missing.
        const uint32_t vst = vc % XS_VST;
        // (warp-uniform: a phase counts as complete when every lane saw it so)
        const bool v_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->v_full[vst], (vc / XS_VST) & 1));
        const bool ph_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->ph_full[b], ppar));
        const bool p_ok = __all_sync(0xffffffffu, mbar_test_wait(&c->p_full[b], ppar));
        bool keep = true;
        if constexpr (GATING) {
          // Lane 0's reading of the word, for the whole warp.
          uint32_t w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          if ((w >> DEC_BITS) != (tc & DEC_STAMP_MASK)) {  // not published yet
            if (!(ok = wait_all(&c->dec_full[b], ppar, abort, p.err, ERR_WAIT_DEC))) break;
            w = __shfl_sync(0xffffffffu, ld_acquire_u32(&c->dec[b]), 0);
          }
          keep = (w & DEC_MASK) != 0u;
        }
        const bool vload = keep || (GATING && VALL);  // this tile's V stage was filled
        if (vload && !v_ok &&
            !(ok = wait_all(&c->v_full[vst], (vc / XS_VST) & 1, abort, p.err, ERR_WAIT_V_FULL)))
          break;
        if (keep) {
          if (PAGED && J == n - 1) {
            // Keys of the last tile past the sequence end: a paged pool may
            // hold anything there (NaN included), and P = 0 does not cancel
            // NaN in P.V.
            const int valid = p.seqinfo[t.x].y - J * TILE;
            if (valid < TILE) zero_tile_rows<D>(sV + vst * TB, valid, lane);
          }
          uint32_t acc = 1u;
          if (first) {
            if (!(ok = wait_all(&c->o_empty, (uc & 1) ^ 1, abort, p.err, ERR_WAIT_O_EMPTY)))
              break;
            acc = 0u;
            first = false;
          }
          const uint32_t d_p = tmem + b * 128;
          const uint64_t dv_st = dV + ((vst * TB) >> 4);
          if (ph_ok && p_ok) {
            tc_fence_after();
            if (elect_one()) issue_pv<D, 1>(d_o, d_p, dv_st, IDESC_PV, acc);
            __syncwarp();
          } else {
            if (!ph_ok && !(ok = wait_all(&c->ph_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL)))
              break;
            tc_fence_after();
            if (elect_one()) issue_pv_half<D, 1>(d_o, d_p, dv_st, IDESC_PV, acc, 0);
            __syncwarp();
            if (!p_ok && !(ok = wait_all(&c->p_full[b], ppar, abort, p.err, ERR_WAIT_P_FULL)))
              break;
            tc_fence_after();
            if (elect_one()) issue_pv_half<D, 1>(d_o, d_p, dv_st, IDESC_PV, 1u, 1);
            __syncwarp();
          }
        } else {
          // A skipped tile has no P: its scores were read before the vote
          // barrier that preceded the decision, so the buffer may be refilled.
          tc_fence_after();
        }
        if (elect_one()) {
          umma_commit(&c->pv_done[tc & 1]);
          if (vload) umma_commit(&c->v_empty[vst]);
        }
        __syncwarp();
        if (vload) ++vc;
        if (J + 2 < n && !(ok = issue_s(J + 2, n, b))) break;
      }
      if (!ok) break;
      if (elect_one()) umma_commit(&c->o_full);
      __syncwarp();
    }
    // Drain: every issued MMA completes before TMEM can be released.
    if (elect_one()) umma_commit(&c->drain);
    __syncwarp();
    drain_wait(&c->drain, 0);
  } else if (warp < 4) {
    // idle
  } else {
    // -------------------------------------------------------------- softmax
    // Warp 4 + 4 ch + wq: rows 32 wq .. 32 wq + 31, keys [64 ch, 64 ch + 64)
    // of each tile.  A thread loads its 64 scores once (the reducing TMEM
    // load also gives their maximum), votes, and takes its exp pass from
    // registers.  One barrier per tile joins the 256 softmax threads: its
    // count carries the gate's vote, the failure consensus and whether some
    // row needs the exact maximum of its two halves (a rise of the lazily
    // rescaled reference, or of the lambda running max); only then are the
    // half maxima exchanged through shared memory.
    const int ch = (warp - 4) >> 2;  // column half
    const int wq = warp & 3;         // TMEM lane quarter
    const int row = wq * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(wq * 32) << 16;
    constexpr int DH = D / 2;        // my output columns
    const uint32_t tO = tmem + tlane + LY::O_COL + ch * DH;
    // Counts and bitmap words: every lane of warp 4 keeps them (lane 0 stores).
    const bool lead_warp = warp == 4;
    constexpr uint32_t bar_id = 1;
    constexpr uint32_t NB = 256;
    const float sc = p.sigma_log2;
    const bool lambda_mode = GATING && p.mode == 1;
    uint32_t tc = 0, uc = 0;
    bool ok = true;
    uint32_t cnt_kept = 0, cnt_cand = 0;

    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      int I, len, h;
      {
        const int kvh = u / per_kv, rem = u - kvh * per_kv;
        const int2 t = p.tiles[rem / p.group];
        I = t.y;
        len = p.seqinfo[t.x].y;
        h = kvh * p.group + rem % p.group;
      }
      const bool rvalid = I * TILE + row < len;
      float tq = 0.f;
      if (GATING && p.mode == 0) tq = p.thr[(long long)h * p.nT + min(I, p.nT - 1)];
      // m_used: reference of P (trails the running max by at most 2^8 in P
      // units); m_true: exact running max over kept blocks (lambda gate); l:
      // this half's share of the normaliser.
      float m_used = -CUDART_INF_F, m_true = -CUDART_INF_F, l = 0.f;
      bool o_init = false;
      uint32_t bm_word = 0;

      for (int J = 0; J <= I; ++J, ++tc) {
        const uint32_t b = tc & 1;
        // Every thread reaches the tile barrier below, also after its own
        // bounded wait gave up, so the 256 threads leave together.
        const bool okl = wait_bar(&c->s_full[b], (tc >> 1) & 1, abort, p.err, ERR_WAIT_S_FULL);
        __syncwarp();  // the TMEM loads below are warp-wide
        tc_fence_after();
        const bool diag_tile = (J == I);
        const uint32_t tS = tmem + tlane + b * 128 + ch * 64;  // my 64 score columns

        // ---- my 64 scores and their maximum (masked on the diagonal tile)
        uint32_t sr[2][32];
        float lm;
        {
          float qm0, qm1;
          tmem_ld32_max(tS, sr[0], qm0);
          tmem_ld32_max(tS + 32, sr[1], qm1);
          tmem_wait_ld();
          if (!diag_tile) {
            lm = fmaxf(qm0, qm1);
          } else {
            lm = -CUDART_INF_F;
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (ch * 64 + e <= row) lm = fmaxf(lm, __uint_as_float(sr[e >> 5][e & 31]));
          }
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
        const bool need_x =
            rvalid && (((lm - m_used) * sc > RESCALE_LOG2) || (lambda_mode && lm > m_true));
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
        const uint32_t n = bar_red_popc(bar_id, NB, lane == 0 ? wx : (lane <= 16 && wv));
        const bool kept = !GATING || diag_tile || n >= 16u;
        float rowmax = lm;  // the row's maximum over both halves (exact when exchanged)
        if ((n & 15u) != 0u) {
          c->xmax[tc & 1][ch][row] = lm;
          ok = bar_red_and(bar_id, NB, okl);
          if (!ok) break;
          rowmax = fmaxf(lm, c->xmax[tc & 1][ch ^ 1][row]);
        }
        if (lambda_mode && kept) m_true = fmaxf(m_true, rowmax);
        if (GATING && lead_warp) {  // all 32 lanes: same value, 32 arrivals
          st_release_u32(&c->dec[b], ((tc & DEC_STAMP_MASK) << DEC_BITS) | (kept ? 1u : 0u));
          mbar_arrive(&c->dec_full[b]);
        }

        // ---- online softmax over my half of a kept tile
        if (kept) {
          if ((n & 15u) != 0u) {  // rowmax is exact: rescale when the reference must rise
            const float m_new = fmaxf(m_used, rowmax);
            const bool resc = (m_new - m_used) * sc > RESCALE_LOG2;
            float alpha = 1.f;
            if (resc) {
              alpha = ex2_approx((m_used - m_new) * sc);
              m_used = m_new;
              l *= alpha;
            }
            // O may still be accumulating the previous tile's P.V (Q.K^T of
            // this tile was issued before it): wait until every P.V so far
            // is done.  The TMEM loads and stores are warp-wide, so the warp
            // rescales together, with alpha = 1 in rows that keep their
            // reference.  A wait that gives up raises the abort flag, which
            // the next tile barrier turns into a common exit.
            if (o_init && __any_sync(0xffffffffu, resc)) {
              wait_bar(&c->pv_done[(tc - 1) & 1], ((tc - 1) >> 1) & 1, abort, p.err,
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
          // 16-bit pairs into my 32 P columns of the tile's S buffer.
          const uint32_t tP = tmem + tlane + b * 128 + ch * 32;
          const float mb = (m_used == -CUDART_INF_F) ? 0.f : m_used * sc;
          const uint64_t sc2 = f2_pack(sc, sc), nmb2 = f2_pack(-mb, -mb);
          uint64_t lsum2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {  // 32 of my keys per step, 16 P columns
            uint32_t pk[16];
            if (!diag_tile) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const uint64_t x2 = f2_pack(__uint_as_float(sr[hq][2 * e]),
                                            __uint_as_float(sr[hq][2 * e + 1]));
                float y0, y1;
                f2_unpack(f2_fma(x2, sc2, nmb2), y0, y1);
                const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                lsum2 = f2_add(lsum2, f2_pack(p0, p1));
                pk[e] = pack_x2<F16>(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int key = ch * 64 + hq * 32 + 2 * e;
                const float x0 = __uint_as_float(sr[hq][2 * e]);
                const float x1 = __uint_as_float(sr[hq][2 * e + 1]);
                const float p0 = key <= row ? ex2_approx(fmaf(x0, sc, -mb)) : 0.f;
                const float p1 = key + 1 <= row ? ex2_approx(fmaf(x1, sc, -mb)) : 0.f;
                lsum2 = f2_add(lsum2, f2_pack(p0, p1));
                pk[e] = pack_x2<F16>(p0, p1);
              }
            }
            tmem_st16(tP + hq * 16, pk);
          }
          float ls0, ls1;
          f2_unpack(lsum2, ls0, ls1);
          l += ls0 + ls1;
          tmem_wait_st();
          o_init = true;
        }
        // My half of P is written (or the tile skipped): one arrival per
        // thread and tile on this half's barrier (keys 0-63: ph_full).
        tc_fence_before();
        mbar_arrive(ch == 0 ? &c->ph_full[b] : &c->p_full[b]);

        // ---- bookkeeping: bitmap words and block counts (lead warp)
        if (lead_warp) {
          if (!diag_tile) {
            ++cnt_cand;
            cnt_kept += kept ? 1u : 0u;
          }
          if (kept) bm_word |= 1u << (J & 31);
          if (p.bitmap != nullptr && ((J & 31) == 31 || diag_tile)) {
            const int4 si = p.seqinfo[p.tiles[(u % per_kv) / p.group].x];
            if (lane == 0)
              p.bitmap[((long long)(si.z + I) * p.Hq + h) * (long long)p.words + (J >> 5)] = bm_word;
            bm_word = 0;
          }
        }
      }
      if (!ok) break;

      // ---- epilogue: O / l -> 16-bit, log-sum-exp, bitmap tail
      const int4 si = p.seqinfo[p.tiles[(u % per_kv) / p.group].x];
      if (lead_warp && p.bitmap != nullptr) {
        const long long bm_row = ((long long)(si.z + I) * p.Hq + h) * (long long)p.words;
        for (int w = (I >> 5) + 1 + lane; w < p.words; w += 32) p.bitmap[bm_row + w] = 0u;
      }
      c->xl[ch][row] = l;
      {
        const bool okl = wait_bar(&c->o_full, uc & 1, abort, p.err, ERR_WAIT_O_FULL);
        if (!(ok = bar_red_and(bar_id, NB, okl))) break;
      }
      tc_fence_after();
      const float lt = l + c->xl[ch ^ 1][row];
      const float inv_l = (lt > 0.f) ? 1.f / lt : 0.f;
      const int qpos = I * TILE + row;
      uint16_t* orow = p.o + (long long)si.w * p.o_sb + (long long)h * p.o_sh +
                       (long long)(si.x + qpos) * p.o_st + ch * DH;
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
              (p.varlen ? (long long)si.x : (long long)si.w * p.batch_len) + qpos] =
            m_used * p.sigma + logf(lt);
      // The next unit's first P.V overwrites O once all 256 threads are here.
      tc_fence_before();
      mbar_arrive(&c->o_empty);
    }
    if (p.counts != nullptr && lead_warp && lane == 0 && uc != 0u) {
      atomicAdd(&p.counts[0], (unsigned long long)cnt_kept);
      atomicAdd(&p.counts[1], (unsigned long long)cnt_cand);
      atomicAdd(&p.counts[2], (unsigned long long)uc);  // one diagonal block per unit
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
