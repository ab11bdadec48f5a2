// bsfa_fwd.cuh -- the persistent, warp-specialised gated prefill kernel for
// sm_103a, and its calibration variant.
//
// What it computes ("Block Sparse Flash Attention", Key Designs 2 and 3; the
// lambda gate from "Skipping attention blocks was the easy part", section
// "Vote, then skip"): for every causally visible 128x128 score tile
// S = Q K^T (tcgen05 MMA, bf16 in, fp32 in TMEM) the semantic Bq x Bk blocks
// inside it are gated; a kept block goes through online softmax and O += P V
// (P in TMEM, V by TMA only after the decision); a skipped block leaves the
// running max, the normaliser and O untouched and its V is never fetched.
//
// Roles (one CTA per SM, persistent over a heaviest-first unit list):
//   warp 0          TMA producer: Q per unit, K for every visible tile (and V
//                   for every tile when the gate is compiled out).
//   warp 3          (gate on) V loader: V for the tiles that some slot keeps,
//                   issued as soon as the decision is published.
//   warp 1          MMA issuer (one thread): S_s = Q_s K^T, O_s += P_s V.
//                   Also owns the TMEM allocation.
//   warps 4..       one softmax warpgroup per query slot s (NQ slots = NQ
//                   query heads of one GQA group sharing the K/V stream);
//                   thread t owns query row t of the slot's 128-row tile.
//
// TMEM columns: S_s at [128 s, 128 s + 128) (P_s overwrites its first 64
// columns as packed bf16 pairs), O_s at [128 NQ + D s, 128 NQ + D (s+1)).
//
// Compiled-in options (template parameters, so that no option costs the
// others a branch): the gate or none, the calibration variant (Q.K^T and
// block maxima only), fp16 or bf16 elements, V for every tile (an A/B of the
// gated V load), K/V read from page pools through a block table, and
// mean-correction tiles after a unit's key tiles.
#pragma once
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace bsfa {

constexpr int TILE = 128;
constexpr int KST = 2;  // K ring stages
// Mean correction: words of kept-candidate bits kept per softmax warp (one
// bit per candidate key block), so sequences of up to 32 * CORR_WORDS * 128
// = 512K tokens.
constexpr int CORR_WORDS = 128;
constexpr int VST = 2;  // V ring stages
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
// Lazy rescale: P is taken against a maximum that may trail the true running
// maximum by up to 8 in log2 units (P entries up to 2^8); only a larger rise
// rescales O and l.
constexpr float RESCALE_LOG2 = 8.0f;
// Decision words carry the tile counter (its low 28 bits) above the four
// decision bits, so a reader can tell a published decision from the word of
// two tiles earlier.
constexpr uint32_t DEC_BITS = 4;
constexpr uint32_t DEC_MASK = (1u << DEC_BITS) - 1u;
constexpr uint32_t DEC_STAMP_MASK = 0x0FFFFFFFu;
// Register split for two slots (384 threads): warpgroup 0 (copies, MMA issue)
// drops to COPY_REGS, the two softmax warpgroups rise to SOFTMAX_REGS.  The
// host checks 128*COPY_REGS + 256*SOFTMAX_REGS against the registers the
// kernel is launched with before the first launch.
constexpr int COPY_REGS = 104;
constexpr int SOFTMAX_REGS = 200;

// Device error word codes (site of the wait that ran out).
enum : unsigned {
  ERR_WAIT_Q_EMPTY = 0x101, ERR_WAIT_K_EMPTY, ERR_WAIT_V_EMPTY, ERR_WAIT_DEC,
  ERR_WAIT_Q_FULL, ERR_WAIT_K_FULL, ERR_WAIT_V_FULL, ERR_WAIT_P_FULL, ERR_WAIT_O_EMPTY,
  ERR_WAIT_S_FULL, ERR_WAIT_WG, ERR_WAIT_O_FULL, ERR_WAIT_DRAIN, ERR_WAIT_RED,
  ERR_WAIT_SELFTEST = 0x1FF
};

struct DevParams {
  uint16_t* o;                // bf16 or f16 elements (the kernel's element type)
  long long o_sb, o_sh, o_st;
  int Hq, Hkv, group, pairs;  // pairs = group / NQ
  int varlen;
  int batch_len;              // batched layout: tokens per sequence (lse row = b*batch_len + pos)
  int Bq, Bk;
  float sigma, sigma_log2;
  int mode;                   // 0 threshold, 1 lambda, 2 dense
  const float* thr;
  int nT;
  float log_lambda;
  uint32_t* bitmap;
  int words;                  // bitmap words per row; layout [query-block rows][Hq][words]
  float* lse;
  long long lse_rows;
  unsigned long long* counts; // [3]
  const int4* seqinfo;        // {tok0, len, rowbase, bcoord}
  const int2* tiles;          // {b, I} sorted by I descending
  const int* ntiles_total;
  float* blockmax;            // calibration: [Hq][cal_nq][cal_nk]
  int cal_nq, cal_nk;
  // Paged K/V: null for contiguous K/V.  Key tile J of sequence b lives in
  // page btab[b * bt_stride + J / tiles_per_page], 128-token slot
  // J % tiles_per_page (a 128-key tile never straddles two pages).
  const int* btab;
  int bt_stride, tiles_per_page;
  // Mean correction: ln(Bk) / sigma, the stand-in logit's shift in the raw
  // score units the kernel keeps its maxima in.
  float corr_shift;
  unsigned* err;
};

// TMA coordinates (token, outermost) of key tile J of sequence b: contiguous
// K/V address it by the sequence's first token and batch index; paged K/V by
// the token slot inside its page and the page index from the block table.
template <bool PAGED>
__device__ __forceinline__ int2 kv_tile_coord(const DevParams& p, const int4& si, int b, int J) {
  if constexpr (!PAGED) return make_int2(si.x + J * TILE, si.w);
  const int pg = __ldg(p.btab + (long long)b * p.bt_stride + J / p.tiles_per_page);
  return make_int2((J % p.tiles_per_page) * TILE, pg);
}

template <int D, int NQ>
struct Ctrl {
  uint64_t q_full[NQ];
  uint64_t q_empty;
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[NQ], o_full[NQ], o_empty[NQ];
  // Per tile parity: P written (or the tile skipped) by all 128 threads of a
  // slot; calibration maxima of a slot's four warps in (128 arrivals); the
  // decision word published by the slot's first warp (32 arrivals).
  uint64_t p_full[NQ][2];
  uint64_t ph_full[NQ][2];  // first half of P (keys 0-63) written
  uint64_t red_full[NQ][2];
  uint64_t dec_full[NQ][2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t dec[NQ][2];
  float red[NQ][2][4][2];
  alignas(16) uint32_t vote[NQ][2][4];   // per warp: bit k = some row wants key half k
  alignas(16) uint32_t vote2[NQ][2][4];  // lambda, second key half
  int abort;
};

template <int D, int NQ, bool CALIB, bool CORR = false>
struct Layout {
  static constexpr int TB = TILE * D * 2;  // bytes of one 128-row bf16 tile
  static constexpr int NV = CALIB ? 0 : VST;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQ * TB;
  static constexpr int V_OFF = K_OFF + KST * TB;
  static constexpr int C_OFF = V_OFF + NV * TB;
  // + alignment slack; at least 120 KB so that a single CTA is resident per SM
  // (the persistent grid assumes it and the TMEM allocation is not shared).
  // Mean correction: kept-candidate bit words, [slot][warp][CORR_WORDS].
  static constexpr int KB_OFF = C_OFF + (((int)sizeof(Ctrl<D, NQ>) + 15) & ~15);
  static constexpr int KB_BYTES = CORR ? NQ * 4 * CORR_WORDS * 4 : 0;
  static constexpr int RAW = KB_OFF + KB_BYTES + 1024;
  static constexpr int BYTES = RAW > 120 * 1024 ? RAW : 120 * 1024;
  static constexpr int NCOLS = (NQ * 128 + NQ * D) <= 256 ? 256 : 512;
  static constexpr int NTHREADS = 128 + 128 * NQ;
};

// Bounded wait: true when the phase of `parity` completed; false after the
// time bound (error word set, abort raised) or when another role aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         unsigned* err, unsigned site,
                                         uint64_t timeout_ns = WAIT_TIMEOUT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        atomicCAS(err, 0u, site);
        return false;
      }
    }
  }
}

// wait_bar executed by every lane of a warp, with the lanes agreeing on the
// outcome (a phase seen complete by one lane is complete for all of them;
// only a lane that timed out can disagree, and then the whole warp stops).
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         unsigned* err, unsigned site) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, err, site));
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Bounded wait used only on the abort path: ignores the abort flag so that
// copies / MMAs already in flight can land before the CTA releases resources.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > WAIT_TIMEOUT_NS / 20) return;
}

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Barrier over the `n` threads of a warpgroup that also ANDs a predicate:
// every thread learns whether all of them are still running.
__device__ __forceinline__ bool bar_red_and(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Barrier over the `n` threads of a warpgroup that counts the threads whose
// predicate is true.
__device__ __forceinline__ uint32_t bar_red_popc(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r;
}

// A compile-time bool as a value (to instantiate a generic lambda twice).
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

// Semantic block class of key block j for query block i (length-L sequence):
// 1 = candidate (every key precedes every row), 2 = diagonal region, 0 = none.
__device__ __forceinline__ int block_class(int i, int j, int Bq, int Bk, int L) {
  const int first_row = i * Bq;
  const int last_row = min((i + 1) * Bq, L) - 1;
  const int first_key = j * Bk;
  if (first_row > last_row || first_key >= L) return 0;
  if ((j + 1) * Bk <= first_row) return 1;
  if (first_key <= last_row) return 2;
  return 0;
}

// Signed distance, modulo the 28-bit decision stamp, of a decision word's
// stamp from tile counter tc (the initial word 0xFFFFFFFF reads as -1 at 0).
__device__ __forceinline__ int32_t stamp_dist(uint32_t w, uint32_t tc) {
  return static_cast<int32_t>(((w >> DEC_BITS) - tc) << (32 - 28)) >> (32 - 28);
}

// The decision word of tile tc (or a later one) of one slot and tile parity,
// read by a whole warp.  The barrier completes once per publication of that
// word, in tile order, so each try targets the phase right after the stamp the
// word carries, whose predecessor has completed; the word is re-read after
// every try, so a parity try that aliases a later phase (the publisher having
// moved on meanwhile) only costs a retry, and a reader that ran ahead (through
// units without votes) finds an older stamp and waits for it.  Bounded like
// every other wait: on timeout it sets the error word and the abort flag and
// *ok = false.
template <int NW = 2>  // words in the ring: tile tc publishes into word tc % NW
__device__ __forceinline__ uint32_t wait_decision(const uint32_t* word, uint64_t* bar,
                                                  uint32_t tc, volatile int* abort,
                                                  unsigned* err, bool* ok) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    const uint32_t w = __shfl_sync(0xffffffffu, ld_acquire_u32(word), 0);
    if (stamp_dist(w, tc) >= 0) return w;
    // The word's tiles are published in order tc % NW, tc % NW + NW, ...;
    // the initial word has no stamp, and its first publication is phase 0.
    const uint32_t next = (w == 0xFFFFFFFFu) ? (tc % NW) : ((w >> DEC_BITS) + NW);
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, (next / NW) & 1u))) continue;
    if ((n & 15u) == 15u) {
      const bool give_up = *abort || globaltimer_ns() - t0 > WAIT_TIMEOUT_NS;
      if (__any_sync(0xffffffffu, give_up)) {
        if (!*abort) {
          *abort = 1;
          atomicCAS(err, 0u, static_cast<unsigned>(ERR_WAIT_DEC));
        }
        *ok = false;
        return w;
      }
    }
  }
}

// True when the gate keeps every block of query tile I of head h: its
// threshold entries are all -inf (calibration gives -inf to query blocks with
// fewer than k candidates), or ln(lambda) = -inf.  Such a unit needs no vote:
// the softmax, the MMA warp and the V loader all take every decision as a
// keep without exchanging it.
__device__ __forceinline__ bool unit_gate_trivial(const DevParams& p, int h, int I) {
  if (p.mode == 1) return p.log_lambda == -CUDART_INF_F;
  if (p.mode != 0) return false;
  const int QS = TILE / p.Bq;
  const int iq = (I * TILE) / p.Bq;
  for (int q = 0; q < QS; ++q)
    if (p.thr[(long long)h * p.nT + min(iq + q, p.nT - 1)] != -CUDART_INF_F) return false;
  return true;
}

// Zero rows [first_row, 128) of a 128-row tile in shared memory as TMA wrote
// it (D/64 swizzled halves of 128 rows x 128 bytes; the 128-byte swizzle only
// permutes 16-byte chunks inside a row, so whole rows are zeroed in place).
// All 32 lanes of the calling warp take part; the proxy fence and the warp
// barrier order the writes before an MMA that the warp then issues.
template <int D>
__device__ __forceinline__ void zero_tile_rows(uint8_t* tile, int first_row, int lane) {
  constexpr int NHALF = D / 64;
  const int chunks = (TILE - first_row) * NHALF * 8;
  for (int c = lane; c < chunks; c += 32) {
    const int r = first_row + c / (NHALF * 8);
    const int hf = (c / 8) % NHALF, ch = c % 8;
    *reinterpret_cast<uint4*>(tile + hf * (TILE * 128) + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_shared();
  __syncwarp();
}

// S = Q K^T for one slot: D/16 K-steps of M=128, N=128, K=16.  Operand
// halves (64 columns, 16 KB each) sit TILE*128 bytes apart.
template <int D, int NQ>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (((kk >> 2) * (TILE * 128)) + (kk & 3) * 32) >> 4;
    umma_ss(d_tmem, dq + off, dk + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V for one slot: 8 K-steps of 16 keys; P (bf16 pairs) in TMEM
// columns [8 kk, 8 kk + 8) of the S region, V MN-major (16 keys = 2048 B).
template <int D, int NQ>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                         uint32_t idesc, uint32_t acc) {
#pragma unroll
  for (int kk = 0; kk < TILE / 16; ++kk)
    umma_ts(d_tmem, p_tmem + kk * 8, dv + ((kk * 2048) >> 4), idesc, (kk > 0 || acc) ? 1u : 0u);
}

// One half of O (+)= P V: K-steps [4 half, 4 half + 4), i.e. keys
// [64 half, 64 half + 64), whose P lives in TMEM columns [32 half, 32 half + 32).
template <int D, int NQ>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                              uint32_t idesc, uint32_t acc, int half) {
#pragma unroll
  for (int k = 0; k < TILE / 32; ++k) {
    const int kk = half * (TILE / 32) + k;
    umma_ts(d_tmem, p_tmem + kk * 8, dv + ((kk * 2048) >> 4), idesc, (kk > 0 || acc) ? 1u : 0u);
  }
}

// VALL (gated only): load V for every visible tile, kept or not.
// PAGED: K and V come from page pools through the block table.
// CORR (gated, Bq = Bk = 128): mean correction.  After a unit's key tiles,
// ceil(I / 128) correction tiles run through the same pipeline: their "keys"
// and "values" are the block means of 128 consecutive key blocks (tmKb,
// tmVb), and only the blocks this slot skipped enter them, with the logit
// shifted by ln(Bk) so that one mean stands for the block's Bk keys.
template <int D, int NQ, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED, bool CORR>
__global__ void __launch_bounds__(Layout<D, NQ, CALIB, CORR>::NTHREADS, 1)
    bsfa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmKb,
                    const __grid_constant__ CUtensorMap tmVb, const DevParams p) {
  using LY = Layout<D, NQ, CALIB, CORR>;
  constexpr int TB = LY::TB;
  constexpr int HALF = TILE * 128;  // bytes of one 64-column swizzled half
  constexpr int NHALF = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base + LY::Q_OFF;
  uint8_t* sK = base + LY::K_OFF;
  uint8_t* sV = base + LY::V_OFF;
  Ctrl<D, NQ>* c = reinterpret_cast<Ctrl<D, NQ>*>(base + LY::C_OFF);
  uint32_t* kbits = reinterpret_cast<uint32_t*>(base + LY::KB_OFF);  // CORR only
  volatile int* abort = &c->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&c->q_full[s], 1);
      mbar_init(&c->s_full[s], 1);
      mbar_init(&c->o_full[s], 1);
      mbar_init(&c->o_empty[s], 128);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&c->p_full[s][b], 128);
        mbar_init(&c->red_full[s][b], 128);
        mbar_init(&c->ph_full[s][b], 128);
        mbar_init(&c->dec_full[s][b], 32);
      }
    }
    mbar_init(&c->q_empty, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    mbar_init(&c->drain, 1);
    for (int s = 0; s < NQ; ++s) c->dec[s][0] = c->dec[s][1] = 0xFFFFFFFFu;  // no stamp matches
    c->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    if (!CALIB) prefetch_tensormap(&tmV);
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
  // q-head pairs of the group.  Each wave of resident CTAs then streams one
  // KV head's K/V prefix, which stays resident in L2 while every CTA of the
  // wave walks it (with the KV head fastest the wave streamed all heads and
  // re-read K/V from DRAM many times over).
  const int ntot = *p.ntiles_total;
  const int per_kv = ntot * p.pairs;
  const int total_units = per_kv * p.Hkv;

  // Register split (two slots): each role sets its own limit at the top of
  // its branch, so the compiler allocates each branch against its limit.

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (NQ == 2) setmaxnreg_dec<COPY_REGS>();
    // The whole warp runs the loop and the waits (so every value it uses is
    // warp-uniform); one elected lane issues each copy.
    uint32_t kc = 0, vc = 0, tc = 0, uc = 0;
    int last_q = -1;  // index of the last unit whose Q load was issued
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.pairs];
      const int pr = rem % p.pairs;
      const int4 si = p.seqinfo[t.x];
      const int I = t.y, nkt = I + 1;
      const int ntt = nkt + (CORR ? (I + TILE - 1) / TILE : 0);  // + correction tiles
      const int row0 = si.x + I * TILE;
      if (!(ok = wait_all(&c->q_empty, (uc & 1) ^ 1, abort, p.err, ERR_WAIT_Q_EMPTY))) break;
      if (elect_one()) {
        for (int s = 0; s < NQ; ++s) {
          const int h = kvh * p.group + pr * NQ + s;
          mbar_arrive_expect_tx(&c->q_full[s], TB);
          for (int hf = 0; hf < NHALF; ++hf)
            tma_load_4d(sQ + s * TB + hf * HALF, &tmQ, &c->q_full[s], hf * 64, row0, h, si.w);
        }
      }
      __syncwarp();
      last_q = static_cast<int>(uc);
      for (int J = -1; J < ntt; ++J) {
        // K for tile J + 1 (tile 0 before the loop proper), then V for tile J.
        if (J + 1 < ntt) {
          const uint32_t st = kc % KST;
          // A paged tile's page comes from the block table: issue that load
          // before the stage wait so that its latency hides behind it.
          const int2 kc2 = (!CORR || J + 1 < nkt) ? kv_tile_coord<PAGED>(p, si, t.x, J + 1)
                                                 : make_int2(0, 0);
          if (!(ok = wait_all(&c->k_empty[st], ((kc / KST) & 1) ^ 1, abort, p.err,
                              ERR_WAIT_K_EMPTY)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&c->k_full[st], TB);
            if (!CORR || J + 1 < nkt) {
              for (int hf = 0; hf < NHALF; ++hf)
                tma_load_4d(sK + st * TB + hf * HALF, &tmK, &c->k_full[st], hf * 64, kc2.x, kvh,
                            kc2.y);
            } else {  // block means of key blocks [128 (J + 1 - nkt), +128)
              for (int hf = 0; hf < NHALF; ++hf)
                tma_load_4d(sK + st * TB + hf * HALF, &tmKb, &c->k_full[st], hf * 64,
                            si.z + (J + 1 - nkt) * TILE, kvh, 0);
            }
          }
          __syncwarp();
          ++kc;
        }
        if (J < 0) continue;
        if constexpr (!CALIB && !GATING) {
          {
            const uint32_t st = vc % VST;
            const int2 vc2 = kv_tile_coord<PAGED>(p, si, t.x, J);  // before the wait
            if (!(ok = wait_all(&c->v_empty[st], ((vc / VST) & 1) ^ 1, abort, p.err,
                                ERR_WAIT_V_EMPTY)))
              break;
            if (elect_one()) {
              mbar_arrive_expect_tx(&c->v_full[st], TB);
              for (int hf = 0; hf < NHALF; ++hf)
                tma_load_4d(sV + st * TB + hf * HALF, &tmV, &c->v_full[st], hf * 64, vc2.x, kvh,
                            vc2.y);
            }
            __syncwarp();
            ++vc;
          }
        }
        ++tc;
      }
    }
    if (!ok) {
      // Let every copy already issued land before the CTA can exit.
      for (int s = 0; s < NQ && last_q >= 0; ++s) drain_wait(&c->q_full[s], last_q & 1);
      for (uint32_t i = 0; i < KST && i < kc; ++i) {
        const uint32_t f = kc - 1 - i;
        drain_wait(&c->k_full[f % KST], (f / KST) & 1);
      }
      for (uint32_t i = 0; i < VST && i < vc; ++i) {
        const uint32_t f = vc - 1 - i;
        drain_wait(&c->v_full[f % VST], (f / VST) & 1);
      }
    }
  } else if (GATING && !CALIB && warp == 3) {
    // ----------------------------------------------------- V loader (gated)
    // A warp of its own, so that a kept tile's V is requested as soon as a
    // slot publishes its decision (the producer is busy with K then).
    if constexpr (NQ == 2) setmaxnreg_dec<COPY_REGS>();
    uint32_t vc = 0, tc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.pairs];
      const int4 si = p.seqinfo[t.x];
      const int nkt = t.y + 1;
      const int ntt = nkt + (CORR ? (t.y + TILE - 1) / TILE : 0);
      for (int J = 0; J < ntt; ++J, ++tc) {
        // Every slot's decision is read on every tile (V is issued on the
        // first one that keeps the tile), so this warp consumes each
        // decision phase in order instead of skipping some.  With VALL no
        // decision is read: V of every tile is issued as early as a stage
        // is free, like the gate-compiled-out producer does.
        bool need = VALL, issued = false;
        // The tile's V coordinates (a block-table load when paged) are read
        // before the decision waits, off the path from a keep to its copy.
        const int2 vc2 = (!CORR || J < nkt) ? kv_tile_coord<PAGED>(p, si, t.x, J) : make_int2(0, 0);
        for (int s = 0; s < NQ && ok; ++s) {
          if constexpr (!VALL) {
            // Every decision phase is consumed in order, also in units whose
            // gate keeps everything (their decisions are published as
            // keeps): so this warp never runs ahead of the decisions, and
            // it trails them by at most one tile -- it only blocks, besides
            // here, on the V stage of a kept tile, whose P.V (and so every
            // later decision of that slot) waits for that V.  The parity wait
            // therefore never falls two phases behind.
            if (!(ok = wait_all(&c->dec_full[s][tc & 1], (tc >> 1) & 1, abort, p.err,
                                ERR_WAIT_DEC)))
              break;
            need = need || (c->dec[s][tc & 1] & DEC_MASK) != 0u;
          }
          if (!need || issued) continue;
          issued = true;
          const uint32_t st = vc % VST;
          if (!(ok = wait_all(&c->v_empty[st], ((vc / VST) & 1) ^ 1, abort, p.err,
                              ERR_WAIT_V_EMPTY)))
            break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&c->v_full[st], TB);
            if (!CORR || J < nkt) {
              for (int hf = 0; hf < NHALF; ++hf)
                tma_load_4d(sV + st * TB + hf * HALF, &tmV, &c->v_full[st], hf * 64, vc2.x, kvh,
                            vc2.y);
            } else {  // value means of key blocks [128 (J - nkt), +128)
              for (int hf = 0; hf < NHALF; ++hf)
                tma_load_4d(sV + st * TB + hf * HALF, &tmVb, &c->v_full[st], hf * 64,
                            si.z + (J - nkt) * TILE, kvh, 0);
            }
          }
          __syncwarp();
          ++vc;
        }
        if (!ok) break;
      }
    }
    if (!ok) {
      for (uint32_t i = 0; i < VST && i < vc; ++i) {
        const uint32_t f = vc - 1 - i;
        drain_wait(&c->v_full[f % VST], (f / VST) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if constexpr (NQ == 2) setmaxnreg_dec<COPY_REGS>();
    // The whole warp runs the loop and the waits; one elected lane (always
    // the same lane: all 32 are active) issues every MMA and commit, so each
    // commit tracks that lane's earlier MMAs.
    constexpr uint32_t IDESC_QK = idesc_f32acc<F16>(128, 128, false, false);
    constexpr uint32_t IDESC_PV = idesc_f32acc<F16>(128, D, false, true);
    uint32_t kc = 0, vc = 0, tc = 0, uc = 0;
    bool ok = true;
    // Descriptors: one 64-bit base per operand buffer; a K-step adds its
    // byte offset >> 4 to the start-address field (bits 0-13; every
    // shared-memory address here is < 2^18, so the field never carries).
    const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sV), HALF, 1024);
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      const int2 t = p.tiles[(u % per_kv) / p.pairs];
      const int nkt = t.y + 1;
      const int ntt = nkt + (CORR ? (t.y + TILE - 1) / TILE : 0);
      // Slots whose gate keeps every block of this unit: no decision to read.
      uint32_t triv = 0;
      if constexpr (GATING && !CALIB && !CORR) {
        const int h0 = (u / per_kv) * p.group + ((u % per_kv) % p.pairs) * NQ;
        for (int s = 0; s < NQ; ++s)
          if (unit_gate_trivial(p, h0 + s, t.y)) triv |= 1u << s;
      }
      for (int s = 0; s < NQ && ok; ++s)
        ok = wait_all(&c->q_full[s], uc & 1, abort, p.err, ERR_WAIT_Q_FULL);
      if (!ok) break;
      {
        const uint32_t st = kc % KST;
        if (!(ok = wait_all(&c->k_full[st], (kc / KST) & 1, abort, p.err, ERR_WAIT_K_FULL))) break;
        if (elect_one()) {
          for (int s = 0; s < NQ; ++s) {
            issue_qk<D, NQ>(tmem + s * 128, dQ + ((s * TB) >> 4), dK + ((st * TB) >> 4), IDESC_QK);
            umma_commit(&c->s_full[s]);
          }
          umma_commit(&c->k_empty[st]);
          if (ntt == 1) umma_commit(&c->q_empty);
        }
        __syncwarp();
        ++kc;
      }
      uint32_t first_mask = (1u << NQ) - 1u;  // slots whose O has not been written yet
      for (int J = 0; J < ntt && ok; ++J, ++tc) {
        const int tb = tc & 1;
        const uint32_t vst = vc % VST;
        const uint32_t kst = kc % KST;
        bool vready = false, any = false;
        for (int s = 0; s < NQ; ++s) {
          bool do_pv = false;
          uint32_t acc = 1u;
          const bool do_qk = J + 1 < ntt;
          const uint32_t ppar = (tc >> 1) & 1u;
          // Every shared-memory access of this warp queues behind the
          // operand reads of the MMAs it has just issued (Q.K^T reads both
          // operands from shared memory at the full shared-memory rate), so
          // one access costs hundreds of cycles.  Probe everything this step
          // may need -- the decision word, V, P and the next K tile -- back
          // to back without blocking (one round trip for all of them), and
          // block only on what was not ready.
          const bool v_ok = CALIB || vready || mbar_test_wait(&c->v_full[vst], (vc / VST) & 1);
          const bool p_ok = mbar_test_wait(&c->p_full[s][tb], ppar);
          const bool k_ok = !(do_qk && s == 0) || mbar_test_wait(&c->k_full[kst], (kc / KST) & 1);
          const uint32_t dw = (GATING && !CALIB) ? ld_acquire_u32(&c->dec[s][tb]) : 0u;
          if constexpr (!CALIB) {
            uint32_t dec = 1u;
            if (GATING && !((triv >> s) & 1u)) {
              uint32_t w = dw;
              if ((w >> DEC_BITS) != (tc & DEC_STAMP_MASK)) {  // not published yet
                if (!(ok = wait_all(&c->dec_full[s][tb], ppar, abort, p.err, ERR_WAIT_DEC))) break;
                w = ld_acquire_u32(&c->dec[s][tb]);
              }
              dec = w & DEC_MASK;
            }
            if (dec != 0u) {
              any = true;
              do_pv = true;
              if (!vready) {
                // V arrives by TMA into shared memory: the mbarrier completion
                // orders it before the MMA (no TMEM hand-off, no tcgen05 fence).
                if (!v_ok && !(ok = wait_all(&c->v_full[vst], (vc / VST) & 1, abort, p.err,
                                             ERR_WAIT_V_FULL)))
                  break;
                vready = true;
                if (PAGED && J == nkt - 1) {
                  // Keys of the last tile past the sequence end: a paged pool
                  // may hold anything there (NaN included), and P = 0 does
                  // not cancel NaN in P.V.
                  const int valid = p.seqinfo[t.x].y - J * TILE;
                  if (valid < TILE) zero_tile_rows<D>(sV + vst * TB, valid, lane);
                }
              }
              if (first_mask & (1u << s)) {
                if (!(ok = wait_all(&c->o_empty[s], (uc & 1) ^ 1, abort, p.err,
                                    ERR_WAIT_O_EMPTY)))
                  break;
                acc = 0u;
                first_mask &= ~(1u << s);
              }
            }
          }
          // A skipped tile has no P: its S was read before the decision was
          // published, so the next S may be issued now.  The P barrier of
          // this tile parity is then not waited on: its previous phase (tile
          // tc - 2) completed before this tile's S was issued (that issue
          // followed either the P of tile tc - 1, or a skip decision, which
          // is published only after the vote barrier of tile tc - 1, which
          // each thread reaches after its arrival for tile tc - 2), so a
          // later wait on it never falls two phases behind.  The barrier of
          // P's first half (ph_full) gets one arrival per thread per tile as
          // well, before that thread's P arrival, so the same holds for it.
          if (CALIB) {
            if (!p_ok && !(ok = wait_all(&c->p_full[s][tb], ppar, abort, p.err, ERR_WAIT_P_FULL)))
              break;
            tc_fence_after();
          } else if (do_pv) {
            // P.V for this tile first: it does not need the next K tile.
            const uint32_t d_o = tmem + NQ * 128 + s * D, d_p = tmem + s * 128;
            const uint64_t dv_st = dV + ((vst * TB) >> 4);
            if (GATING && !p_ok) {
              // The softmax hands P off in two halves: start on keys 0-63
              // while it still computes keys 64-127.
              if (!(ok = wait_all(&c->ph_full[s][tb], ppar, abort, p.err, ERR_WAIT_P_FULL)))
                break;
              tc_fence_after();
              if (elect_one()) issue_pv_half<D, NQ>(d_o, d_p, dv_st, IDESC_PV, acc, 0);
              __syncwarp();
              if (!(ok = wait_all(&c->p_full[s][tb], ppar, abort, p.err, ERR_WAIT_P_FULL))) break;
              tc_fence_after();
              if (elect_one()) issue_pv_half<D, NQ>(d_o, d_p, dv_st, IDESC_PV, 1u, 1);
              __syncwarp();
            } else {
              if (!GATING && !p_ok &&
                  !(ok = wait_all(&c->p_full[s][tb], ppar, abort, p.err, ERR_WAIT_P_FULL)))
                break;
              tc_fence_after();
              if (elect_one()) issue_pv<D, NQ>(d_o, d_p, dv_st, IDESC_PV, acc);
              __syncwarp();
            }
          } else {
            tc_fence_after();
          }
          if (do_qk && s == 0 && !k_ok) {
            if (!(ok = wait_all(&c->k_full[kst], (kc / KST) & 1, abort, p.err, ERR_WAIT_K_FULL)))
              break;
          }
          if (elect_one()) {
            if (do_qk) {
              issue_qk<D, NQ>(tmem + s * 128, dQ + ((s * TB) >> 4), dK + ((kst * TB) >> 4),
                              IDESC_QK);
              umma_commit(&c->s_full[s]);
              if (s == NQ - 1) {
                umma_commit(&c->k_empty[kst]);
                if (J + 1 == ntt - 1) umma_commit(&c->q_empty);
              }
            }
          }
          __syncwarp();
          if (do_qk && s == NQ - 1) ++kc;
        }
        if (!ok) break;
        if constexpr (GATING && !CALIB && VALL) {
          // This tile's V was loaded whether or not a slot kept it.
          if (!vready) {
            if (!(ok = wait_all(&c->v_full[vst], (vc / VST) & 1, abort, p.err, ERR_WAIT_V_FULL)))
              break;
            any = true;
          }
        }
        if (!CALIB && any) {
          if (elect_one()) umma_commit(&c->v_empty[vst]);
          __syncwarp();
          ++vc;
        }
      }
      if (!ok) break;
      if constexpr (!CALIB) {
        if (elect_one())
          for (int s = 0; s < NQ; ++s) umma_commit(&c->o_full[s]);
        __syncwarp();
      }
    }
    // Drain: every issued MMA completes before TMEM can be released.
    if (elect_one()) umma_commit(&c->drain);
    __syncwarp();
    drain_wait(&c->drain, 0);
  } else if (warp < 4) {
    if constexpr (NQ == 2) setmaxnreg_dec<COPY_REGS>();
  } else {
    // -------------------------------------------------------------- softmax
    if constexpr (NQ == 2) setmaxnreg_inc<SOFTMAX_REGS>();
    const int s = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + tlane + s * 128;
    const uint32_t tO = tmem + tlane + NQ * 128 + s * D;
    const int QS = TILE / p.Bq, KS = TILE / p.Bk;
    const bool simple = (QS == 1 && KS == 1);  // one semantic block per 128x128 tile
    const int myqs = (p.Bq == 64) ? (row >> 6) : 0;
    // The warp holding the first row of a semantic query block keeps that
    // block's counts and bitmap words.  Every lane of it keeps the same
    // values (gate decisions are warp-uniform), so the bookkeeping never
    // splits the warp (a one-lane branch here slowed the whole warp's
    // exp pass); lane 0 alone stores.
    const bool lead_warp = ((wq * 32) % p.Bq) == 0;
    const uint32_t bar_id = 1 + s;  // named barrier of this warpgroup (gated kernel)
    const float sc = p.sigma_log2;
    uint32_t tc = 0, uc = 0;
    bool ok = true;
    unsigned long long cnt_kept = 0, cnt_cand = 0, cnt_diag = 0;

    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++uc) {
      const int kvh = u / per_kv, rem = u - kvh * per_kv;
      const int2 t = p.tiles[rem / p.pairs];
      const int pr = rem % p.pairs;
      const int4 si = p.seqinfo[t.x];
      const int I = t.y, nkt = I + 1, len = si.y;
      const int h = kvh * p.group + pr * NQ + s;
      const int qpos = I * TILE + row;
      const bool rvalid = qpos < len;
      const int iq_base = (I * TILE) / p.Bq;  // semantic query block of row 0
      const int my_i = iq_base + myqs;
      float thr[2] = {0.f, 0.f};
      if (GATING && !CALIB && p.mode == 0) {
        thr[0] = p.thr[(long long)h * p.nT + min(iq_base, p.nT - 1)];
        if (QS == 2) thr[1] = p.thr[(long long)h * p.nT + min(iq_base + 1, p.nT - 1)];
      }
      // A unit whose gate keeps everything takes no vote and no per-tile
      // barrier; a bounded wait that gives up inside it is carried to the
      // unit's epilogue barrier (`failed`), where the warpgroup leaves together.
      const bool trivial = GATING && !CALIB && !CORR && unit_gate_trivial(p, h, I);
      bool failed = false;
      float m_used = -CUDART_INF_F, m_true = -CUDART_INF_F, l = 0.f;
      bool o_init = false;
      uint32_t bm_word = 0;
      int bm_idx = 0;
      const bool bm_on = (p.bitmap != nullptr) && lead_warp && (my_i * p.Bq < len);
      const long long bm_row = ((long long)(si.z + my_i) * p.Hq + h) * (long long)p.words;
      // Mean correction (Bq = Bk = 128: the candidates of query block I are
      // key blocks 0 .. I-1): kept bits of the candidates, one word per 32
      // blocks, in this warp's own shared-memory row.
      const int nct = CORR ? (I + TILE - 1) / TILE : 0;  // correction tiles after the keys
      uint32_t* my_kbits = kbits + (s * 4 + wq) * CORR_WORDS;
      uint32_t kbit_acc = 0;

      // The tile loop, compiled twice: once for units whose gate keeps
      // everything (no vote, no per-tile barrier) and once for the rest,
      // so that neither pays for the other's branches.
      auto tile_loop = [&](auto triv_c) {
        constexpr bool TRIV = decltype(triv_c)::value;
        for (int J = 0; J < nkt; ++J, ++tc) {
          const int tb = tc & 1;
          const uint32_t ph = (tc >> 1) & 1u;  // phase parity of the per-tile-parity barriers
          // Waits here are bounded.  In the gated kernel every thread joins the
          // per-tile vote barrier even after its own wait gave up, and the
          // barrier's count tells all of them, so the warpgroup leaves together
          // (its named barriers can never strand a warp).  The other kernels use
          // no named barrier in this loop: a warp that gives up leaves alone and
          // the others' bounded waits see the abort flag.
          bool okl;
          if constexpr (GATING && !CALIB) {
            okl = wait_bar(&c->s_full[s], tc & 1, abort, p.err, ERR_WAIT_S_FULL);
          } else {
            if (!(ok = wait_all(&c->s_full[s], tc & 1, abort, p.err, ERR_WAIT_S_FULL))) break;
            okl = true;
          }
          tc_fence_after();
          const bool diag_tile = (J == I);  // keys beyond a row exist only in the last tile

          // ---- pass 1: row maxima of the two 64-key halves of S
          float rm0 = -CUDART_INF_F, rm1 = -CUDART_INF_F;
          uint32_t sr[4][32];
          // Unconditional, even for a thread whose wait gave up (it then reads
          // stale S from its own TMEM columns and the vote barrier stops the
          // warpgroup): a per-thread guard around the .sync.aligned loads cost
          // the gated kernel about 2% of its tile period.
          {
            // The reducing TMEM load returns each 32-column quarter's maximum
            // along with the values, so a tile below the diagonal needs no
            // max instructions at all; the diagonal tile masks and reduces the
            // values itself.
            float qm[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32_max(tS + q * 32, sr[q], qm[q]);
            tmem_wait_ld();
            if (!diag_tile) {
              rm0 = fmaxf(qm[0], qm[1]);
              rm1 = fmaxf(qm[2], qm[3]);
            } else {
  #pragma unroll
              for (int e = 0; e < 128; ++e) {
                const float x = (e > row) ? -CUDART_INF_F : __uint_as_float(sr[e >> 5][e & 31]);
                if (e < 64) rm0 = fmaxf(rm0, x); else rm1 = fmaxf(rm1, x);
              }
            }
            if (KS == 1) {
              rm0 = fmaxf(rm0, rm1);
              rm1 = rm0;
            }
          }

          // Block classes of the (query, key) sub-blocks of this tile.
          int cls[2][2] = {{0, 0}, {0, 0}};
          if (simple) {
            cls[0][0] = diag_tile ? 2 : 1;
          } else {
  #pragma unroll
            for (int q = 0; q < 2; ++q)
  #pragma unroll
              for (int k = 0; k < 2; ++k)
                if (q < QS && k < KS)
                  cls[q][k] = block_class(iq_base + q, (J * TILE) / p.Bk + k, p.Bq, p.Bk, len);
          }

          // ---- gate votes.  Threshold: row r wants key half k when
          // sigma * rowmax_r(k) >= T.  The tile maximum clears T exactly when
          // some row's maximum does (scaling by sigma > 0 is monotone in fp32),
          // so the OR of the row votes equals comparing s_max(i,j) with T.
          // Lambda: row r wants the first sub-block when
          // sigma * (rowmax_r - m_r) >= ln(lambda).
          const bool lambda_mode = GATING && !CALIB && p.mode == 1;
          if constexpr (CALIB) {
            const float w0 = warp_max_f32(rvalid ? rm0 : -CUDART_INF_F);
            const float w1 = (KS == 1) ? w0 : warp_max_f32(rvalid ? rm1 : -CUDART_INF_F);
            c->red[s][tb][wq][0] = w0;  // every lane: same value
            c->red[s][tb][wq][1] = w1;
            tc_fence_before();
            mbar_arrive(&c->red_full[s][tb]);
            // Calibration: the slot's first warp records sigma * s_max of each
            // candidate block once every warp's maxima are in.
            if (wq == 0) {
              if (!(ok = wait_all(&c->red_full[s][tb], ph, abort, p.err, ERR_WAIT_RED))) break;
              if (lane == 0) {
                for (int q = 0; q < QS; ++q)
                  for (int k = 0; k < KS; ++k) {
                    if (cls[q][k] != 1) continue;
                    float mx = -CUDART_INF_F;
                    for (int w = 0; w < 4; ++w)
                      if (QS == 1 || (w >> 1) == q) mx = fmaxf(mx, c->red[s][tb][w][k]);
                    const long long idx =
                        ((long long)h * p.cal_nq + iq_base + q) * p.cal_nk + (J * TILE) / p.Bk + k;
                    p.blockmax[idx] = mx * p.sigma;
                  }
              }
              __syncwarp();
            }
            mbar_arrive(&c->p_full[s][tb]);
            continue;
          } else {
            // ---- gate: decide every sub-block of this tile
            bool keep[2][2];
  #pragma unroll
            for (int q = 0; q < 2; ++q)
  #pragma unroll
              for (int k = 0; k < 2; ++k) keep[q][k] = cls[q][k] != 0;
            if constexpr (GATING && TRIV) {
              failed = failed || !okl;
            } else if constexpr (GATING) {
              bool w0, w1 = false;
              if (!lambda_mode) {
                const float tq = (myqs ? thr[1] : thr[0]);
                w0 = rvalid && rm0 * p.sigma >= tq;
                w1 = rvalid && rm1 * p.sigma >= tq;
              } else {
                w0 = rvalid && (myqs ? cls[1][0] : cls[0][0]) == 1 &&
                     ((rm0 - m_true) * p.sigma >= p.log_lambda);
              }
              // Every read of S is complete here (tcgen05.wait::ld above); the
              // fence orders it before the barrier, so that the MMA warp may
              // overwrite S as soon as it reads a skip decision.
              tc_fence_before();
              if (simple) {
                // One 128x128 semantic block per tile: the hardware barrier
                // itself carries the vote (no shared-memory traffic, which
                // queues behind the MMAs' operand reads).  Lane 0 of each warp
                // counts 1 when some lane of the warp has stopped, lanes 1..8
                // count 1 each when some row of the warp wants the block, so the
                // count is F + 8 V with F, V <= 4.
                const bool wf = __any_sync(0xffffffffu, !okl);
                const bool wv = __any_sync(0xffffffffu, w0);
                const uint32_t n = bar_red_popc(bar_id, 128, lane == 0 ? wf : (lane <= 8 && wv));
                ok = (n & 7u) == 0u;
                if (!ok) break;
                if (!diag_tile) keep[0][0] = n >= 8u;
              } else {
                c->vote[s][tb][wq] = (__any_sync(0xffffffffu, w0) ? 1u : 0u) |
                                     ((KS == 2 && __any_sync(0xffffffffu, w1)) ? 2u : 0u);
                ok = bar_red_and(bar_id, 128, okl);
                if (!ok) break;
                // OR the warp votes of each query half (warps 0-1 hold rows 0-63).
                const uint4 vv = *reinterpret_cast<const uint4*>(&c->vote[s][tb][0]);
                uint32_t vq0 = vv.x | vv.y, vq1 = vv.z | vv.w;
                if (QS == 1) vq0 = vq1 = vq0 | vq1;
  #pragma unroll
                for (int k = 0; k < 2; ++k) {
                  if (cls[0][k] == 1) keep[0][k] = (vq0 >> k) & 1u;
                  if (cls[1][k] == 1) keep[1][k] = (vq1 >> k) & 1u;
                }
              }
              if (lambda_mode) {
                // Sub-blocks in ascending key order; a row's running max moves
                // only with the blocks it keeps, so the second key half is voted
                // on after the first half's decision.
                if ((myqs ? keep[1][0] : keep[0][0])) m_true = fmaxf(m_true, rm0);
                if (KS == 2) {
                  if (cls[0][1] == 1 || cls[1][1] == 1) {
                    const bool v1 = rvalid && (myqs ? cls[1][1] : cls[0][1]) == 1 &&
                                    ((rm1 - m_true) * p.sigma >= p.log_lambda);
                    c->vote2[s][tb][wq] = __any_sync(0xffffffffu, v1) ? 1u : 0u;
                    // Every thread passed the vote barrier above, so all of them
                    // reach this one.
                    named_bar_sync(bar_id, 128);
                    const uint4 v2 = *reinterpret_cast<const uint4*>(&c->vote2[s][tb][0]);
                    uint32_t u0 = v2.x | v2.y, u1 = v2.z | v2.w;
                    if (QS == 1) u0 = u1 = u0 | u1;
                    if (cls[0][1] == 1) keep[0][1] = u0 & 1u;
                    if (cls[1][1] == 1) keep[1][1] = u1 & 1u;
                  }
                  if ((myqs ? keep[1][1] : keep[0][1])) m_true = fmaxf(m_true, rm1);
                }
              }
            }
            uint32_t decbits = 0;
  #pragma unroll
            for (int q = 0; q < 2; ++q)
  #pragma unroll
              for (int k = 0; k < 2; ++k)
                if (keep[q][k]) decbits |= 1u << (q * 2 + k);
            if (GATING && wq == 0) {  // all 32 lanes: same value, 32 arrivals
              // Release: a reader that sees this tile's stamp also sees every
              // S read the decision depended on (the votes it waited for).
              st_release_u32(&c->dec[s][tb], ((tc & DEC_STAMP_MASK) << DEC_BITS) | decbits);
              mbar_arrive(&c->dec_full[s][tb]);
            }

            // ---- online softmax over the kept sub-blocks of this slot
            if (decbits != 0u) {
              const bool k0 = (myqs ? keep[1][0] : keep[0][0]);
              const bool k1 = (KS == 1) ? k0 : (myqs ? keep[1][1] : keep[0][1]);
              float rmk = -CUDART_INF_F;
              if (k0) rmk = fmaxf(rmk, rm0);
              if (k1) rmk = fmaxf(rmk, rm1);
              const float m_new = fmaxf(m_used, rmk);
              const bool resc = (m_new - m_used) * sc > RESCALE_LOG2;
              float alpha = 1.f;
              if (resc) {
                alpha = ex2_approx((m_used - m_new) * sc);
                m_used = m_new;
                l *= alpha;
              }
              if (o_init && __any_sync(0xffffffffu, resc)) {
  #pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                  uint32_t orr[32];
                  tmem_ld32(tO + q * 32, orr);
                  tmem_wait_ld();
  #pragma unroll
                  for (int e = 0; e < 32; ++e)
                    orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                  tmem_st32(tO + q * 32, orr);
                }
              }
              // Pass 2: P = exp2(sigma*log2e*(S - m)) for the kept, visible
              // entries, packed as bf16 pairs into the first 64 columns of the
              // S region (half hf -> P columns [32 hf, 32 hf + 32); those S
              // columns have been read by then).
              const float mb = (m_used == -CUDART_INF_F) ? 0.f : m_used * sc;
              const uint64_t sc2 = f2_pack(sc, sc), nmb2 = f2_pack(-mb, -mb);
              uint64_t lsum2 = f2_pack(0.f, 0.f);
              const bool fast = !diag_tile && k0 && k1;
  #pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const bool kk = (hf == 0) ? k0 : k1;
                // Re-read this half of S from TMEM (cheaper than holding the
                // whole row in registers across the gate).
                tmem_ld32(tS + hf * 64, sr[2 * hf]);
                tmem_ld32(tS + hf * 64 + 32, sr[2 * hf + 1]);
                tmem_wait_ld();
                uint32_t pk[32];
                if (fast) {
  #pragma unroll
                  for (int e = 0; e < 32; ++e) {
                    const uint64_t x2 = f2_pack(__uint_as_float(sr[2 * hf + (e >> 4)][(2 * e) & 31]),
                                                __uint_as_float(sr[2 * hf + (e >> 4)][(2 * e + 1) & 31]));
                    float y0, y1;
                    f2_unpack(f2_fma(x2, sc2, nmb2), y0, y1);
                    const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                    const uint64_t pp = f2_pack(p0, p1);
                    lsum2 = f2_add(lsum2, pp);
                    pk[e] = pack_x2<F16>(p0, p1);
                  }
                } else {
  #pragma unroll
                  for (int e = 0; e < 32; ++e) {
                    const int cc = hf * 64 + 2 * e;
                    const bool vis0 = kk && !(diag_tile && cc > row);
                    const bool vis1 = kk && !(diag_tile && cc + 1 > row);
                    const float x0 = __uint_as_float(sr[2 * hf + (e >> 4)][(2 * e) & 31]);
                    const float x1 = __uint_as_float(sr[2 * hf + (e >> 4)][(2 * e + 1) & 31]);
                    const float p0 = vis0 ? ex2_approx(fmaf(x0, sc, -mb)) : 0.f;
                    const float p1 = vis1 ? ex2_approx(fmaf(x1, sc, -mb)) : 0.f;
                    lsum2 = f2_add(lsum2, f2_pack(p0, p1));
                    pk[e] = pack_x2<F16>(p0, p1);
                  }
                }
                tmem_st32(tS + hf * 32, pk);
                if (GATING && hf == 0) {  // hand off the first half of P
                  tmem_wait_st();
                  tc_fence_before();
                  mbar_arrive(&c->ph_full[s][tb]);
                }
              }
              float ls0, ls1;
              f2_unpack(lsum2, ls0, ls1);
              l += ls0 + ls1;
              tmem_wait_st();
              o_init = true;
            }
            if (GATING && decbits == 0u) mbar_arrive(&c->ph_full[s][tb]);  // one phase per tile
            tc_fence_before();
            mbar_arrive(&c->p_full[s][tb]);

            // ---- bookkeeping: bitmap words and block counts (after the
            // hand-off of P, off the path to the next MMA)
            if constexpr (CORR) {
              if (J < I) {  // a candidate: record whether this slot kept it
                kbit_acc |= (keep[0][0] ? 1u : 0u) << (J & 31);
                if ((J & 31) == 31 || J == I - 1) {
                  my_kbits[J >> 5] = kbit_acc;  // every lane: same value
                  kbit_acc = 0u;
                }
              }
            }
            if (lead_warp && my_i * p.Bq < len) {
  #pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int cl = (myqs ? cls[1][k] : cls[0][k]);
                if (cl == 0) continue;
                const int j = (J * TILE) / p.Bk + k;
                if (cl == 1) {
                  ++cnt_cand;
                  cnt_kept += (myqs ? keep[1][k] : keep[0][k]) ? 1 : 0;
                } else {
                  ++cnt_diag;
                }
                if (bm_on) {
                  if ((j >> 5) != bm_idx) {
                    if (lane == 0) p.bitmap[bm_row + bm_idx] = bm_word;
                    bm_idx = j >> 5;
                    bm_word = 0;
                  }
                  if ((myqs ? keep[1][k] : keep[0][k])) bm_word |= 1u << (j & 31);
                }
              }
            }
          }
        }
      };
      if (trivial)
        tile_loop(BoolC<true>{});
      else
        tile_loop(BoolC<false>{});
      if (!ok) break;

      if constexpr (CORR && GATING && !CALIB) {
        // ---- mean-correction tiles: S = Q Kbar^T over the means of key
        // blocks [jb, jb + 128).  Entry e enters iff key block jb + e is a
        // candidate (jb + e < I) that this slot skipped; its logit carries
        // ln(Bk) (corr_shift in raw score units), so one mean stands for the
        // block's Bk keys.  The same hand-offs as a key tile: the vote
        // barrier keeps the warpgroup together, the first warp publishes the
        // decision (any entry), P goes over S and the MMA warp adds P Vbar.
        for (int ci = 0; ci < nct; ++ci, ++tc) {
          const int tb = tc & 1;
          const int jb = ci * TILE;
          uint32_t inc[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int lim = I - jb - 32 * q;
            const uint32_t cand = lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : (1u << lim) - 1u);
            inc[q] = cand & ~my_kbits[(jb >> 5) + q];
          }
          const bool any_in = (inc[0] | inc[1] | inc[2] | inc[3]) != 0u;
          const bool okl = wait_bar(&c->s_full[s], tc & 1, abort, p.err, ERR_WAIT_S_FULL);
          tc_fence_after();
          float mx = -CUDART_INF_F;
          if (okl && any_in) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t sq[32];
              tmem_ld32(tS + q * 32, sq);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if ((inc[q] >> e) & 1u) mx = fmaxf(mx, __uint_as_float(sq[e]));
            }
          }
          tc_fence_before();
          if (!(ok = bar_red_and(bar_id, 128, okl))) break;
          if (wq == 0) {  // all 32 lanes: same value, 32 arrivals
            st_release_u32(&c->dec[s][tb],
                           ((tc & DEC_STAMP_MASK) << DEC_BITS) | (any_in ? 1u : 0u));
            mbar_arrive(&c->dec_full[s][tb]);
          }
          if (any_in) {
            const float m_new = fmaxf(m_used, mx + p.corr_shift);
            const bool resc = (m_new - m_used) * sc > RESCALE_LOG2;
            float alpha = 1.f;
            if (resc) {
              alpha = ex2_approx((m_used - m_new) * sc);
              m_used = m_new;
              l *= alpha;
            }
            if (o_init && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
              for (int q = 0; q < D / 32; ++q) {
                uint32_t orr[32];
                tmem_ld32(tO + q * 32, orr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_st32(tO + q * 32, orr);
              }
            }
            const float bias = p.corr_shift * sc - ((m_used == -CUDART_INF_F) ? 0.f : m_used * sc);
            float lsum = 0.f;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
              // Re-read this half of S (64 columns) before P overwrites the
              // first 32 columns of the S region with it.
              uint32_t sh[2][32];
              tmem_ld32(tS + hf * 64, sh[0]);
              tmem_ld32(tS + hf * 64 + 32, sh[1]);
              tmem_wait_ld();
              const uint32_t m0 = inc[2 * hf], m1 = inc[2 * hf + 1];
              uint32_t pk[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int c0 = 2 * e, c1 = 2 * e + 1;  // columns within this half
                const uint32_t w0 = c0 < 32 ? m0 : m1, w1 = c1 < 32 ? m0 : m1;
                const float x0 = __uint_as_float(sh[c0 >> 5][c0 & 31]);
                const float x1 = __uint_as_float(sh[c1 >> 5][c1 & 31]);
                const float p0 = ((w0 >> (c0 & 31)) & 1u) ? ex2_approx(fmaf(x0, sc, bias)) : 0.f;
                const float p1 = ((w1 >> (c1 & 31)) & 1u) ? ex2_approx(fmaf(x1, sc, bias)) : 0.f;
                lsum += p0 + p1;
                pk[e] = pack_x2<F16>(p0, p1);
              }
              tmem_st32(tS + hf * 32, pk);
              if (hf == 0) {
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&c->ph_full[s][tb]);
              }
            }
            l += lsum;
            tmem_wait_st();
            o_init = true;
          }
          if (!any_in) mbar_arrive(&c->ph_full[s][tb]);
          tc_fence_before();
          mbar_arrive(&c->p_full[s][tb]);
        }
        if (!ok) break;
      }

      if constexpr (!CALIB) {
        // ---- epilogue: O / l -> bf16, log-sum-exp, bitmap tail
        if (bm_on)
          for (int w = bm_idx + lane; w < p.words; w += 32)
            p.bitmap[bm_row + w] = (w == bm_idx) ? bm_word : 0u;
        if constexpr (GATING) {
          const bool okl = wait_bar(&c->o_full[s], uc & 1, abort, p.err, ERR_WAIT_O_FULL);
          if (!(ok = bar_red_and(bar_id, 128, okl && !failed))) break;
        } else {
          if (!(ok = wait_all(&c->o_full[s], uc & 1, abort, p.err, ERR_WAIT_O_FULL))) break;
        }
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        uint16_t* orow = p.o + (long long)si.w * p.o_sb + (long long)h * p.o_sh +
                              (long long)(si.x + qpos) * p.o_st;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t orr[32];
          tmem_ld32(tO + q * 32, orr);
          tmem_wait_ld();
          if (rvalid) {
            uint4 pk[4];
            uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pw[e] = pack_x2<F16>(__uint_as_float(orr[2 * e]) * inv_l,
                                   __uint_as_float(orr[2 * e + 1]) * inv_l);
            uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = pk[e];
          }
        }
        if (p.lse != nullptr && rvalid)
          p.lse[(long long)h * p.lse_rows +
                (p.varlen ? (long long)si.x : (long long)si.w * p.batch_len) + qpos] =
              m_used * p.sigma + logf(l);
        tc_fence_before();
        mbar_arrive(&c->o_empty[s]);
      }
    }
    if (p.counts != nullptr && lane == 0 && (cnt_cand | cnt_diag) != 0ull) {
      atomicAdd(&p.counts[0], cnt_kept);
      atomicAdd(&p.counts[1], cnt_cand);
      atomicAdd(&p.counts[2], cnt_diag);
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
