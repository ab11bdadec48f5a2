/*
 * bsfa.h -- C ABI of libbsfa.so: block-sparse gated causal prefill attention
 * (Block Sparse Flash Attention form) for NVIDIA GB300 (sm_103a).
 *
 * Operations and where they are defined:
 *
 *   bsfa_prefill_fwd   "Block Sparse Flash Attention" (papernotes.org note on
 *                      arXiv 2512.07011), Key Designs 2 "Exact-Score Gating"
 *                      (displayed equation: s_max(i,j) over the whole
 *                      Bq x Bk tile of QK^T/sqrt(d); keep iff s_max >= T) and
 *                      Key Designs 3 "Selective Streaming Aggregation"
 *                      (a rejected tile gets no V load, no exp, no P.V and no
 *                      update of the running max, the normaliser or the output
 *                      accumulator; the output is renormalised over the
 *                      retained blocks).  The lambda-relative mode follows
 *                      "Skipping attention blocks was the easy part"
 *                      (yash-agarwal.org, BLASST), section "Vote, then skip".
 *   bsfa_calibrate     same BSFA note, Key Designs 1 "Offline Threshold
 *                      Calibration": per head and query block, the k-th
 *                      largest maximum over the visible off-diagonal key
 *                      blocks, averaged over calibration samples; -inf when
 *                      fewer than k candidates exist.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers unless a parameter says "host".
 *     The caller owns every buffer; the library never allocates device memory
 *     at run time (scratch comes from the caller's workspace).  Its only
 *     device memory of its own is static: the device error word and the
 *     fixed scratch array of bsfa_prefill_fwd_noalloc.
 *   - Calls are asynchronous on `stream` and never synchronise the host,
 *     except bsfa_device_error which synchronises `stream` by design.
 *   - Errors that the host can detect are returned before anything is
 *     launched: a rejected call writes no memory the caller can see.  A
 *     device-side wait that ran out of time (a hang guard, never expected in
 *     a correct run) sets a device error word; it is reported by
 *     bsfa_device_error.
 *   - No C++ exception crosses this boundary.
 *   - Size limits (BSFA_ERR_UNSUPPORTED beyond them): at most 4096 sequences
 *     per call; at most 16384 query tiles of 128 rows per sequence (2M tokens);
 *     for calibration, at most 16 budgets per call and 8192 key blocks per
 *     sample.
 *
 * Block geometry (all positions local to a sequence):
 *   query block i covers rows [i*Bq, min((i+1)*Bq, L)); key block j covers
 *   keys [j*Bk, min((j+1)*Bk, L)).  Key block j is a CANDIDATE for query
 *   block i when (j+1)*Bk <= i*Bq (every key precedes every row: the tile lies
 *   strictly below the causal diagonal).  A visible block that is not a
 *   candidate belongs to the diagonal region: it is always kept and the
 *   causal mask is applied to it.
 */
#ifndef BSFA_H
#define BSFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bsfa_stream_t; /* same handle as cudaStream_t */

typedef enum {
  BSFA_OK = 0,
  BSFA_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, GQA mismatch, bad stride */
  BSFA_ERR_UNSUPPORTED = 2,   /* head_dim / block sizes / alignment not supported */
  BSFA_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  BSFA_ERR_DEVICE_TIMEOUT = 4,/* a device-side wait exceeded its bound */
  BSFA_ERR_WORKSPACE = 5      /* workspace pointer null/misaligned or too small */
} bsfa_status;

typedef enum {
  BSFA_GATE_THRESHOLD = 0, /* keep candidate (i,j) iff sigma*max(QK^T tile) >= T[h][min(i,nT-1)] */
  BSFA_GATE_LAMBDA = 1,    /* skip candidate iff for every row r: sigma*(rowmax_r - m_r) < log_lambda,
                              m_r = exact running max over kept blocks, blocks in ascending key
                              order with the diagonal region last */
  BSFA_GATE_NONE = 2       /* dense causal attention: a kernel built with the gate compiled out
                              (the zero-skip overhead reference) */
} bsfa_gate_mode;

/* Element type of Q, K, V and O (one type for all four).  The tensor-core
 * products accumulate in fp32 for either; P is rounded to this type before
 * the PV product and O is rounded to it once, at the end. */
typedef enum {
  BSFA_DTYPE_BF16 = 0,
  BSFA_DTYPE_F16 = 1
} bsfa_dtype;

/* Bits of bsfa_fwd_params.flags. */
typedef enum {
  /* THRESHOLD and LAMBDA modes: load the V tile of every visible key tile,
   * kept or not, ahead of the gate (as the BLASST SM100 kernel does, "V is
   * still loaded" in its discussion of skipped blocks); skipped tiles still
   * get no exp, no P.V and no m/l/O update, so results are bit-identical to
   * flags = 0.  Exists to measure what skipping the V load saves. */
  BSFA_FLAG_V_ALWAYS = 1,
  /* THRESHOLD and LAMBDA modes: mean correction for skipped blocks ("FlashPrefill
   * V2" summary, agihunt.info, mean correction).  Every skipped candidate block J
   * of a query block enters that block's softmax through a zero-order stand-in:
   * with the block's mean key kbar_J and mean value vbar_J, each row adds the
   * weight Bk * exp(sigma * q . kbar_J) to the denominator and that weight times
   * vbar_J to the numerator.  The gate's decisions, the bitmap and the counts are
   * unchanged.  The block means are computed in fp32 from K and V and stored in
   * the element type in the workspace (bsfa_prefill_workspace_size includes
   * them).  Requires block_q == block_k == 128, contiguous K/V (block_table
   * NULL), no BSFA_FLAG_V_ALWAYS, sequences of at most 524288 tokens and
   * head_dim * num_heads_kv <= 1024 (one thread per element in the block-mean
   * pass: Hkv <= 8 at d = 128, <= 16 at d = 64); else BSFA_ERR_UNSUPPORTED,
   * returned before anything is launched. */
  BSFA_FLAG_MEAN_CORRECTION = 2,
  /* THRESHOLD, LAMBDA and NONE modes: the pipelined schedule instead of the
   * paired one.  Same results up to rounding order (the gate's decisions and
   * the bitmap are the same; outputs differ only in the fp32 summation order
   * of the normaliser).  Paired (flags = 0): a CTA holds two query heads of
   * one GQA group that share every K/V tile, with one score buffer each; a
   * head's next Q.K^T waits for its current P.V.  Pipelined: a CTA holds one
   * query head with three score buffers, and a warp of its own issues the
   * Q.K^T of tile t + 3 as soon as tile t is done with its buffer (skipped,
   * or its P.V complete), ahead of the P.V in flight ("Skipping attention
   * blocks was the easy part", section "Cross-stage P").  Requires
   * block_q == 128 and block_k == 128 or 224, else BSFA_ERR_UNSUPPORTED;
   * mean correction runs in both schedules (block_k == 128).  It is the
   * faster schedule for gated calls (threshold or lambda) with 128 x 128
   * blocks once tiles are skipped (the Python binding's default picks it
   * there); with the gate compiled out the two are within a few percent of
   * each other.  The 128 x 224 tile always runs one query head per CTA (its
   * 224-column score buffer fits TMEM once, not twice), with or without this
   * flag. */
  BSFA_FLAG_PIPELINED = 4
} bsfa_flag;

/*
 * Parameters of one prefill call.  Q, K, V, O share one 16-bit element type
 * (`dtype`: bf16 or fp16) with the head dimension contiguous; every other dimension is addressed through strides
 * given in ELEMENTS as {batch, head, token}.  Two layouts are accepted:
 *   - batched  (cu_seqlens == NULL): `batch` sequences of `seqlen` tokens,
 *     e.g. [B, H, L, d] or [B, L, H, d];
 *   - varlen   (cu_seqlens != NULL): `batch` sequences packed along tokens,
 *     `seqlen` = total packed tokens, sequence b owns tokens
 *     [cu_seqlens[b], cu_seqlens[b+1]); the batch stride is ignored.
 *     cu_seqlens lives in device memory and is read by the kernels only, so
 *     the library cannot check it without a synchronisation: the caller
 *     guarantees 0 <= cu_seqlens[0] <= cu_seqlens[1] <= ... <=
 *     cu_seqlens[batch] <= seqlen and every length <= max_seqlen.  Offsets
 *     that break this make the kernels read and write out of bounds.
 * Strides must be multiples of 8 elements (16 bytes) and the base pointers
 * 16-byte aligned (TMA requirement).  q-head h reads KV head h / (Hq/Hkv).
 */
typedef struct {
  const void* q;              /* [.., Hq, .., d]  */
  const void* k;              /* [.., Hkv, .., d] */
  const void* v;              /* [.., Hkv, .., d] */
  void* o;                    /* same shape as q; rows past a sequence end untouched */
  int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3]; /* {batch, head, token} */
  int batch;                  /* number of sequences (>= 0; 0 is a no-op) */
  int num_heads_q;            /* Hq */
  int num_heads_kv;           /* Hkv, Hq % Hkv == 0 */
  int seqlen;                 /* tokens per sequence (batched) or total tokens (varlen) */
  int head_dim;               /* d: 64 or 128 */
  const int32_t* cu_seqlens;  /* device int32 [batch+1], nullable (batched layout) */
  int max_seqlen;             /* varlen: an upper bound on every sequence length */
  int block_q, block_k;       /* semantic gate blocks Bq, Bk: each 64 or 128, or Bq = 128
                                 with Bk = 224 (the H100 tile of the BSFA note, "Loss &
                                 Training"; contiguous K/V and no mean correction, else
                                 BSFA_ERR_UNSUPPORTED).  Any other pair:
                                 BSFA_ERR_UNSUPPORTED */
  float softmax_scale;        /* sigma; <= 0 selects 1/sqrt(d) */
  int mode;                   /* bsfa_gate_mode */
  const float* thresholds;    /* device fp32 [Hq][thresholds_nq] (THRESHOLD mode): the
                                 slice for one (budget, layer); natural-log units of the
                                 scaled scores; -inf keeps everything */
  int thresholds_nq;          /* nT >= 1; query blocks i >= nT use T[h][nT-1] */
  float log_lambda;           /* natural log of lambda (LAMBDA mode) */
  uint32_t* kept_bitmap;      /* nullable device output [rows][Hq][words_per_row] (see
                                 bsfa_bitmap_words_per_row): bit j of
                                 row (h, row_base(b) + i) = keep(i,j); diagonal-region bits
                                 are 1; invisible blocks 0; every word of every row written */
  float* lse;                 /* nullable device fp32 output [Hq][rows]: natural-log
                                 log-sum-exp of the kept scaled scores, row = b*seqlen+pos
                                 (batched) or cu_seqlens[b]+pos (varlen) */
  unsigned long long* block_counts; /* nullable device u64[3], overwritten: kept candidate
                                 blocks, visible candidate blocks, diagonal-region blocks
                                 (semantic Bq x Bk blocks, all heads and sequences) */
  void* workspace;            /* device scratch, >= bsfa_prefill_workspace_size bytes,
                                 256-byte aligned; its contents are not preserved */
  size_t workspace_bytes;
  int dtype;                  /* bsfa_dtype of q, k, v and o; 0 (a zeroed struct) is bf16;
                                 any other value is BSFA_ERR_UNSUPPORTED */
  unsigned int flags;         /* bsfa_flag bits (0 = default); unknown bits are
                                 BSFA_ERR_UNSUPPORTED */
  /* Paged K/V, the layout a serving KV cache uses ("FlashPrefill V2" summary,
   * agihunt.info: the sparse kernel reads K/V through the page table, so it
   * plugs into a paged cache with continuous batching).  block_table == NULL
   * (a zeroed struct) keeps the contiguous K/V layouts above.  When set:
   *   - k and v point to page pools: page p holds page_size consecutive tokens
   *     of every KV head; element (p, h, t, :) sits at
   *     base + p*stride[0] + h*stride[1] + t*stride[2] (the "batch" stride
   *     addresses pages), e.g. [num_pages, page_size, Hkv, d];
   *   - key position pos of sequence b is token pos % page_size of page
   *     block_table[b*block_table_stride + pos/page_size];
   *   - q, o, lse and the bitmap keep their batched or varlen layout.
   * Pool rows past a sequence's last key may hold anything, NaN included:
   * the kernel zeroes them in shared memory before they reach P.V.  A table
   * entry outside [0, num_pages) reads as zero keys and values (the TMA
   * bounds check) and never addresses memory outside the pools. */
  const int32_t* block_table; /* device int32 [batch][block_table_stride] */
  int block_table_stride;     /* entries per sequence, >= ceil(max_len / page_size) */
  int page_size;              /* tokens per page: a positive multiple of 128, else
                                 BSFA_ERR_UNSUPPORTED */
  int num_pages;              /* pages in each pool (>= 1) */
} bsfa_fwd_params;

/* Bytes of workspace bsfa_prefill_fwd needs for these parameters (reads the
 * shape fields only).  Returns 0 for invalid parameters. */
size_t bsfa_prefill_workspace_size(const bsfa_fwd_params* p);

/* Shape of the optional kept-block bitmap: *rows = Hq * sum_b ceil(L_b/Bq) is
 * not knowable on the host in varlen mode without the lengths, so the host
 * passes an upper bound through the call below:
 *   words_per_row = ceil(ceil(max_len / Bk) / 32), max_len = seqlen (batched)
 *   or max_seqlen (varlen);
 *   rows_per_head = batch * ceil(seqlen / Bq) (batched) or
 *   sum_b ceil(L_b / Bq) (varlen, computed by the caller from its lengths);
 *   row_base(b) = sum_{b' < b} ceil(L_b' / Bq).
 * Returns BSFA_OK or BSFA_ERR_INVALID_ARG. */
bsfa_status bsfa_bitmap_words_per_row(const bsfa_fwd_params* p, int* words_per_row);

/* Gated causal prefill.  Validates `p`, then enqueues on `stream` a small
 * scheduling kernel, the block-mean kernel when BSFA_FLAG_MEAN_CORRECTION is
 * set, and the persistent attention kernel.  Asynchronous.
 * Errors: BSFA_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE before any launch;
 * BSFA_ERR_CUDA if a launch or descriptor encode fails. */
bsfa_status bsfa_prefill_fwd(const bsfa_fwd_params* p, bsfa_stream_t stream);

/*
 * bsfa_prefill_fwd_noalloc -- the same gated prefill for callers that cannot
 * allocate device memory at call time.  The paper has no counterpart to this
 * entry point; it exists for the calling environment, not for the method.
 *
 * Who needs it: callers whose device memory is planned once, up front, and
 * who may not call cudaMalloc (or any allocator) while attention runs --
 * real-time serving loops with a fixed memory plan, plugins hosted by a
 * framework that owns the allocator, embedded runtimes with a static memory
 * map.  bsfa_prefill_fwd asks for a caller-provided workspace; this entry
 * point takes none.
 *
 * Behaviour: identical to bsfa_prefill_fwd, except that p->workspace and
 * p->workspace_bytes are ignored.  The scratch (sequence table and tile
 * schedule) lives in a fixed 256 KiB array of device memory that the library
 * sets aside on every GPU that loads it, for the life of the process.
 *   - Limit: the call's bsfa_prefill_workspace_size(p) must not exceed
 *     262144 bytes (for example 32 sequences of 32K tokens need about 66 KiB;
 *     one sequence may have up to 16384 query tiles of 128 rows).  A larger
 *     request returns BSFA_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address and
 *     caches it; make that first call before any stream capture begins.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents.  Each call rewrites every scratch byte it later reads,
 *     so nothing has to start at zero.  Calls that may overlap on the GPU
 *     (different streams with no ordering between them) race on the array:
 *     order them on one stream, or use bsfa_prefill_fwd with separate
 *     workspaces.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
bsfa_status bsfa_prefill_fwd_noalloc(const bsfa_fwd_params* p, bsfa_stream_t stream);

/*
 * Offline threshold calibration for one layer and a set of budgets.
 *   q_samples / k_samples: HOST arrays of n_samples DEVICE pointers to
 *     tensors (element type `dtype`, a bsfa_dtype) of one sample each, layout [H, L, d] addressed by the strides
 *     {head, token} in elements (d contiguous), equal L for every sample.
 *   ks: HOST array of n_k budgets (each >= 1).
 *   block_q, block_k: 64 or 128 each, or 128 with 224.
 *   thresholds_out: device fp32 [n_k][Hq][ceil(L/Bq)], overwritten with the
 *     mean over samples of the k-th largest candidate block maximum (scaled
 *     by sigma), -inf where a sample has fewer than k candidates.
 *   workspace: >= bsfa_calibrate_workspace_size(...) bytes, 256-byte aligned.
 * Asynchronous on `stream`.
 */
size_t bsfa_calibrate_workspace_size(int num_heads_q, int seqlen, int block_q, int block_k);

bsfa_status bsfa_calibrate(const void* const* q_samples, const void* const* k_samples,
                           int n_samples, int num_heads_q, int num_heads_kv, int seqlen,
                           int head_dim, int dtype,
                           const int64_t q_stride[2], const int64_t k_stride[2],
                           int block_q, int block_k, float softmax_scale,
                           const int* ks, int n_k, float* thresholds_out,
                           void* workspace, size_t workspace_bytes, bsfa_stream_t stream);

/* Synchronises `stream`, then reports (and clears) the device error word set
 * by a kernel whose bounded wait ran out.  *code receives the raw word (0 if
 * none).  Returns BSFA_ERR_DEVICE_TIMEOUT if it was set, BSFA_ERR_CUDA if the
 * synchronisation failed, else BSFA_OK. */
bsfa_status bsfa_device_error(bsfa_stream_t stream, unsigned int* code);

/* Hang-guard self test.  Launches one warp on `stream` that waits, through
 * the same bounded-wait routine the attention kernels use, on a barrier that
 * nothing ever completes.  After timeout_us microseconds (1 .. 10^7) the wait
 * gives up, records code 0x1FF in the device error word and the kernel exits
 * normally.  bsfa_device_error then returns BSFA_ERR_DEVICE_TIMEOUT with that
 * code, and the context stays usable.  No fault, trap or hang is involved. */
bsfa_status bsfa_selftest_wait_guard(unsigned int timeout_us, bsfa_stream_t stream);

/* Static description of a status code. */
const char* bsfa_status_string(bsfa_status s);

/* Library version, e.g. 0x000100 for 0.1.0. */
int bsfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSFA_H */
