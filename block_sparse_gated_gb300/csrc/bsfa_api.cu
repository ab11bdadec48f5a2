// bsfa_api.cu -- host side of libbsfa.so: argument validation, TMA
// descriptors, the scheduling pre-pass and the calibration selection kernel.
// The C ABI is declared in include/bsfa.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "bsfa.h"
#include "bsfa_launch.h"

namespace bsfa {

// Device error word: set by a kernel whose bounded wait ran out.
static __device__ unsigned g_device_error = 0u;

constexpr int MAX_BATCH = 4096;          // sequences per call
constexpr int MAX_TILES_PER_SEQ = 16384; // 128-row tiles per sequence (2M tokens)
constexpr int MAX_BUDGETS = 16;          // budgets per calibration call
constexpr int MAX_CAL_BLOCKS = 8192;     // key blocks per calibration row
constexpr int PREP_THREADS = 1024;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ scheduling pre-pass
// One CTA.  From the sequence lengths it writes
//   seqinfo[b] = {first token, length, first semantic query-block row, batch coordinate}
//   tiles[]    = every (b, I) 128-row query tile, sorted by I descending (the
//                number of key tiles a unit streams is I + 1: heaviest first)
//   *ntot      = number of tiles;  counts[0..2] = 0 when non-null.
__global__ void __launch_bounds__(PREP_THREADS)
    prep_kernel(const int32_t* cu, int batch, int seqlen, int varlen, int Bq, int max_tiles,
                int4* seqinfo, int2* tiles, int* ntot, unsigned long long* counts) {
  extern __shared__ int sh[];
  int* nt = sh;                       // [batch] tiles per sequence
  int* cnt = sh + batch;              // [max_tiles] sequences with more than I tiles
  __shared__ int part[PREP_THREADS];  // per-thread partial sums for the scan
  const int tid = threadIdx.x;
  for (int b = tid; b < batch; b += blockDim.x) {
    const int len = varlen ? (cu[b + 1] - cu[b]) : seqlen;
    nt[b] = (len + TILE - 1) / TILE;
  }
  if (counts != nullptr && tid < 3) counts[tid] = 0ull;
  __syncthreads();
  if (tid == 0) {  // semantic query-block row base: prefix over sequences
    int rb = 0;
    for (int b = 0; b < batch; ++b) {
      const int len = varlen ? (cu[b + 1] - cu[b]) : seqlen;
      seqinfo[b] = make_int4(varlen ? cu[b] : 0, len, rb, varlen ? 0 : b);
      rb += (len + Bq - 1) / Bq;
    }
  }
  for (int I = tid; I < max_tiles; I += blockDim.x) {
    int n = 0;
    for (int b = 0; b < batch; ++b) n += (nt[b] > I) ? 1 : 0;
    cnt[I] = n;
  }
  __syncthreads();
  // Exclusive scan of cnt in descending I: off(I) = sum_{I' > I} cnt[I'].
  // Thread t owns the contiguous descending chunk [t*per, (t+1)*per).
  const int per = (max_tiles + PREP_THREADS - 1) / PREP_THREADS;
  int local = 0;
  for (int r = tid * per; r < min((tid + 1) * per, max_tiles); ++r) local += cnt[max_tiles - 1 - r];
  part[tid] = local;
  __syncthreads();
  for (int off = 1; off < PREP_THREADS; off <<= 1) {
    const int v = (tid >= off) ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - local;  // exclusive prefix of this chunk
  for (int r = tid * per; r < min((tid + 1) * per, max_tiles); ++r) {
    const int I = max_tiles - 1 - r;
    int pos = run;
    for (int b = 0; b < batch; ++b)
      if (nt[b] > I) tiles[pos++] = make_int2(b, I);
    run += cnt[I];
  }
  if (tid == PREP_THREADS - 1) *ntot = part[tid];
}

// ------------------------------------------------------------ calibration selection
struct SelectArgs {
  const float* blockmax;  // [Hq][nq][nk], sigma * s_max for candidate blocks
  float* out;             // [n_k][Hq][nq]
  int Hq, nq, nk, Bq, Bk, L;
  int n_k;
  int ks[MAX_BUDGETS];
  int sample, n_samples;
};

// One CTA per (query block i, head h): sort the candidate maxima descending
// (bitonic network, -inf padding) and accumulate the k-th largest of each
// budget; the last sample divides the sum by the sample count.
__global__ void __launch_bounds__(1024) select_kernel(const SelectArgs a) {
  extern __shared__ float v[];
  const int i = blockIdx.x, h = blockIdx.y;
  // Candidates of query block i: key blocks j with (j+1)*Bk <= i*Bq.
  const int ncand = min((i * a.Bq) / a.Bk, a.nk);
  int n = 1;
  while (n < ncand) n <<= 1;
  const float* row = a.blockmax + ((long long)h * a.nq + i) * a.nk;
  for (int t = threadIdx.x; t < n; t += blockDim.x) v[t] = (t < ncand) ? row[t] : -CUDART_INF_F;
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const int u = t ^ j;
        if (u > t) {
          const float x = v[t], y = v[u];
          const bool descending_run = (t & k) == 0;
          if (descending_run ? (x < y) : (x > y)) {
            v[t] = y;
            v[u] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  if (threadIdx.x < a.n_k) {
    const int kk = a.ks[threadIdx.x];
    const float t = (ncand >= kk) ? v[kk - 1] : -CUDART_INF_F;
    float* o = a.out + ((long long)threadIdx.x * a.Hq + h) * a.nq + i;
    float acc = (a.sample == 0) ? t : (*o + t);
    if (a.sample == a.n_samples - 1) acc = acc / static_cast<float>(a.n_samples);
    *o = acc;
  }
}

// ------------------------------------------------------------ block means (mean correction)
// One CTA per 128-row query tile of the schedule (with Bq = Bk = 128 that is
// one key block), blockDim = {d, KV heads}: thread (e, h) averages element e
// of the block's keys and values of KV head h in fp32 and stores the means in
// the element type at row seqinfo.z + I of the tables [Hkv][rows][d] (the
// same row numbering as the kept-block bitmap).
template <bool F16>
__global__ void __launch_bounds__(1024)
    block_mean_kernel(const uint16_t* k, const uint16_t* v, long long k_sb, long long k_sh,
                      long long k_st, long long v_sb, long long v_sh, long long v_st,
                      const int4* seqinfo, const int2* tiles, const int* ntot, uint16_t* kbar,
                      uint16_t* vbar, int rows) {
  if (static_cast<int>(blockIdx.x) >= *ntot) return;
  const int2 t = tiles[blockIdx.x];
  const int4 si = seqinfo[t.x];
  const int e = threadIdx.x, h = threadIdx.y, d = blockDim.x;
  const int r0 = t.y * TILE, r1 = min(r0 + TILE, si.y);
  const uint16_t* kp = k + (long long)si.w * k_sb + (long long)h * k_sh + e;
  const uint16_t* vp = v + (long long)si.w * v_sb + (long long)h * v_sh + e;
  float sk = 0.f, sv = 0.f;
#pragma unroll 8
  for (int r = r0; r < r1; ++r) {
    const long long tok = si.x + r;
    const uint16_t a = kp[tok * k_st], b = vp[tok * v_st];
    if (F16) {
      sk += __half2float(__ushort_as_half(a));
      sv += __half2float(__ushort_as_half(b));
    } else {
      sk += __bfloat162float(__ushort_as_bfloat16(a));
      sv += __bfloat162float(__ushort_as_bfloat16(b));
    }
  }
  const float inv = 1.f / static_cast<float>(r1 - r0);
  const long long o = ((long long)h * rows + si.z + t.y) * d + e;
  if (F16) {
    kbar[o] = __half_as_ushort(__float2half_rn(sk * inv));
    vbar[o] = __half_as_ushort(__float2half_rn(sv * inv));
  } else {
    kbar[o] = __bfloat16_as_ushort(__float2bfloat16_rn(sk * inv));
    vbar[o] = __bfloat16_as_ushort(__float2bfloat16_rn(sv * inv));
  }
}

// ------------------------------------------------------------ hang-guard self test
// One warp waits, through the attention kernel's own bounded-wait helper, on
// an mbarrier that nothing ever arrives on.  The wait gives up after
// timeout_ns, records ERR_WAIT_SELFTEST in the device error word and the
// kernel returns normally, leaving the context usable.
__global__ void __launch_bounds__(32) wait_guard_selftest_kernel(unsigned long long timeout_ns,
                                                                 unsigned* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0)
    wait_bar(&bar, 0, &abort_flag, err, ERR_WAIT_SELFTEST, timeout_ns);
}

// ------------------------------------------------------------ TMA descriptors
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled get_encoder() {
  static EncodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

// 4-D map of 16-bit elements (bf16 or fp16) {d, tokens, heads, batch}, box {64, box_rows,
// 1, 1} (128 rows, or 224 for the keys and values of the 128 x 224 tile), 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* ptr, bool f16, int d, long long tokens, int heads,
                     int batch, long long st_tok, long long st_head, long long st_batch,
                     int box_rows = TILE) {
  EncodeTiled enc = get_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)tokens, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)st_tok * 2, (cuuint64_t)st_head * 2,
                           (cuuint64_t)st_batch * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static unsigned* error_word() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(ptr);
}

template <bool CALIB, bool F16, bool G, bool VA, bool PG, bool CR>
static cudaError_t dispatch_dn(int d, int nq, const Maps& m, const DevParams& p, int grid,
                               cudaStream_t st) {
  if (d == 128) return nq == 2 ? launch_fwd<128, 2, G, CALIB, F16, VA, PG, CR>(m, p, grid, st)
                               : launch_fwd<128, 1, G, CALIB, F16, VA, PG, CR>(m, p, grid, st);
  return nq == 2 ? launch_fwd<64, 2, G, CALIB, F16, VA, PG, CR>(m, p, grid, st)
                 : launch_fwd<64, 1, G, CALIB, F16, VA, PG, CR>(m, p, grid, st);
}

struct Variant {
  bool gating, vall, paged, corr;
};

template <bool CALIB, bool F16>
static cudaError_t dispatch_t(int d, int nq, Variant v, const Maps& m, const DevParams& p,
                              int grid, cudaStream_t st) {
  if constexpr (CALIB) {
    return dispatch_dn<true, F16, true, false, false, false>(d, nq, m, p, grid, st);
  } else {
    if (v.corr) return dispatch_dn<false, F16, true, false, false, true>(d, nq, m, p, grid, st);
    if (v.paged)
      return v.gating ? dispatch_dn<false, F16, true, false, true, false>(d, nq, m, p, grid, st)
                      : dispatch_dn<false, F16, false, false, true, false>(d, nq, m, p, grid, st);
    if (v.gating && v.vall)
      return dispatch_dn<false, F16, true, true, false, false>(d, nq, m, p, grid, st);
    return v.gating ? dispatch_dn<false, F16, true, false, false, false>(d, nq, m, p, grid, st)
                    : dispatch_dn<false, F16, false, false, false, false>(d, nq, m, p, grid, st);
  }
}

// The pipelined schedule (bsfa_xs_kernel, BSFA_FLAG_PIPELINED): 128 x 128
// semantic blocks (with or without mean correction), or the 128 x 224 tile.
template <int D, int BK, bool F16>
static cudaError_t dispatch_xs_d(Variant v, const Maps& m, const DevParams& p, int grid,
                                 cudaStream_t st) {
  if constexpr (BK == 128) {
    if (v.corr) return launch_xs<D, BK, true, false, F16, false, false, true>(m, p, grid, st);
    if (v.paged) return v.gating ? launch_xs<D, BK, true, false, F16, false, true>(m, p, grid, st)
                                 : launch_xs<D, BK, false, false, F16, false, true>(m, p, grid, st);
  }
  if (v.gating && v.vall) return launch_xs<D, BK, true, false, F16, true, false>(m, p, grid, st);
  return v.gating ? launch_xs<D, BK, true, false, F16, false, false>(m, p, grid, st)
                  : launch_xs<D, BK, false, false, F16, false, false>(m, p, grid, st);
}

// The single-head kernels: key tiles of 128 (BSFA_FLAG_PIPELINED) or 224.
template <bool F16>
static cudaError_t dispatch_xs_t(int d, int bk, Variant v, const Maps& m, const DevParams& p,
                                 int grid, cudaStream_t st) {
  if (bk == 224)
    return d == 128 ? dispatch_xs_d<128, 224, F16>(v, m, p, grid, st)
                    : dispatch_xs_d<64, 224, F16>(v, m, p, grid, st);
  return d == 128 ? dispatch_xs_d<128, 128, F16>(v, m, p, grid, st)
                  : dispatch_xs_d<64, 128, F16>(v, m, p, grid, st);
}

template <bool CALIB>
static cudaError_t dispatch(bool f16, int d, int nq, Variant v, const Maps& m,
                            const DevParams& p, int grid, cudaStream_t st) {
  return f16 ? dispatch_t<CALIB, true>(d, nq, v, m, p, grid, st)
             : dispatch_t<CALIB, false>(d, nq, v, m, p, grid, st);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool stride_ok(long long s) { return s > 0 && (s % 8) == 0; }

struct Carve {
  int4* seqinfo;
  int2* tiles;
  int* ntot;
  float* blockmax;
  uint16_t* kbar;
  uint16_t* vbar;
  size_t bytes;
};

// Workspace layout: seqinfo | tiles | ntot | (calibration) blockmax |
// (mean correction) key means | value means, each [Hkv][rows][d] 16-bit.
static Carve carve(void* base, int batch, int max_tiles_total, size_t blockmax_elems,
                   size_t mean_elems = 0) {
  Carve c{};
  size_t off = 0;
  uint8_t* b = static_cast<uint8_t*>(base);
  c.seqinfo = reinterpret_cast<int4*>(b + off);
  off = align_up(off + sizeof(int4) * (size_t)batch, 256);
  c.tiles = reinterpret_cast<int2*>(b + off);
  off = align_up(off + sizeof(int2) * (size_t)max_tiles_total, 256);
  c.ntot = reinterpret_cast<int*>(b + off);
  off = align_up(off + sizeof(int), 256);
  c.blockmax = reinterpret_cast<float*>(b + off);
  off = align_up(off + sizeof(float) * blockmax_elems, 256);
  c.kbar = reinterpret_cast<uint16_t*>(b + off);
  off = align_up(off + sizeof(uint16_t) * mean_elems, 256);
  c.vbar = reinterpret_cast<uint16_t*>(b + off);
  off = align_up(off + sizeof(uint16_t) * mean_elems, 256);
  c.bytes = off;
  return c;
}

static long long max_len_of(const bsfa_fwd_params* p) {
  return p->cu_seqlens ? p->max_seqlen : p->seqlen;
}

static long long tiles_bound(const bsfa_fwd_params* p) {
  if (p->cu_seqlens) return (p->seqlen + TILE - 1) / TILE + p->batch;
  return (long long)p->batch * ((p->seqlen + TILE - 1) / TILE);
}

static bool corr_on(const bsfa_fwd_params* p) {
  return (p->flags & BSFA_FLAG_MEAN_CORRECTION) != 0;
}

// Elements of one block-mean table (mean correction), 0 when it is off.
static size_t mean_elems(const bsfa_fwd_params* p) {
  if (!corr_on(p) || p->num_heads_kv <= 0 || p->head_dim <= 0) return 0;
  return (size_t)p->num_heads_kv * (size_t)tiles_bound(p) * (size_t)p->head_dim;
}

static bsfa_status validate(const bsfa_fwd_params* p) {
  if (p == nullptr) return BSFA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->seqlen < 0) return BSFA_ERR_INVALID_ARG;
  if (p->num_heads_q <= 0 || p->num_heads_kv <= 0 || p->num_heads_q % p->num_heads_kv)
    return BSFA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return BSFA_ERR_UNSUPPORTED;
  if (p->dtype != BSFA_DTYPE_BF16 && p->dtype != BSFA_DTYPE_F16) return BSFA_ERR_UNSUPPORTED;
  if (p->flags & ~static_cast<unsigned>(BSFA_FLAG_V_ALWAYS | BSFA_FLAG_MEAN_CORRECTION |
                                        BSFA_FLAG_PIPELINED))
    return BSFA_ERR_UNSUPPORTED;
  // The pipelined schedule: Bq = 128, Bk = 128 or 224 (mean correction with
  // Bk = 128 only, as in every schedule).
  if ((p->flags & BSFA_FLAG_PIPELINED) &&
      (p->block_q != TILE || (p->block_k != TILE && p->block_k != 224)))
    return BSFA_ERR_UNSUPPORTED;
  // Semantic blocks: Bq, Bk in {64, 128}, or the 128 x 224 tile.
  const bool tile224 = p->block_q == TILE && p->block_k == 224;
  if (!tile224 &&
      ((p->block_q != 64 && p->block_q != 128) || (p->block_k != 64 && p->block_k != 128)))
    return BSFA_ERR_UNSUPPORTED;
  // The 128 x 224 tile: contiguous K/V (a 224-key tile would straddle pages)
  // and no mean correction.
  if (tile224 && (p->block_table != nullptr || (p->flags & BSFA_FLAG_MEAN_CORRECTION)))
    return BSFA_ERR_UNSUPPORTED;
  if (p->mode < BSFA_GATE_THRESHOLD || p->mode > BSFA_GATE_NONE) return BSFA_ERR_INVALID_ARG;
  if (p->batch > MAX_BATCH) return BSFA_ERR_UNSUPPORTED;
  if (p->cu_seqlens && p->seqlen > 0 && p->max_seqlen <= 0) return BSFA_ERR_INVALID_ARG;
  if ((max_len_of(p) + TILE - 1) / TILE > MAX_TILES_PER_SEQ) return BSFA_ERR_UNSUPPORTED;
  if (corr_on(p)) {
    // Stand-ins need gating, 128 x 128 blocks (one key block per tile),
    // contiguous K/V and at most 32 * CORR_WORDS candidate blocks per row.
    if (p->mode == BSFA_GATE_NONE || p->block_q != TILE || p->block_k != TILE ||
        p->block_table != nullptr || (p->flags & BSFA_FLAG_V_ALWAYS) ||
        (max_len_of(p) + TILE - 1) / TILE > 32 * CORR_WORDS)
      return BSFA_ERR_UNSUPPORTED;
    // The block-mean pass runs one thread per (element, KV head) in one CTA.
    if (p->head_dim * p->num_heads_kv > 1024) return BSFA_ERR_UNSUPPORTED;
  }
  if (p->batch == 0 || p->seqlen == 0) return BSFA_OK;
  if (!p->q || !p->k || !p->v || !p->o) return BSFA_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->o))
    return BSFA_ERR_UNSUPPORTED;
  const int first = p->cu_seqlens ? 1 : 0;
  const bool paged = p->block_table != nullptr;
  for (int i = first; i < 3; ++i)
    if (!stride_ok(p->q_stride[i]) || !stride_ok(p->k_stride[i]) || !stride_ok(p->v_stride[i]) ||
        !stride_ok(p->o_stride[i]))
      return BSFA_ERR_UNSUPPORTED;
  if (paged) {
    // Pages are addressed through the "batch" stride of K and V, in either layout.
    if (!stride_ok(p->k_stride[0]) || !stride_ok(p->v_stride[0])) return BSFA_ERR_UNSUPPORTED;
    if (p->page_size <= 0 || p->page_size % TILE != 0) return BSFA_ERR_UNSUPPORTED;
    if (p->flags & BSFA_FLAG_V_ALWAYS) return BSFA_ERR_UNSUPPORTED;  // no paged V-always kernels
    if (p->num_pages < 1) return BSFA_ERR_INVALID_ARG;
    if ((long long)p->block_table_stride * p->page_size < max_len_of(p))
      return BSFA_ERR_INVALID_ARG;
  }
  if (p->mode == BSFA_GATE_THRESHOLD && (p->thresholds == nullptr || p->thresholds_nq < 1))
    return BSFA_ERR_INVALID_ARG;
  if (p->mode == BSFA_GATE_LAMBDA && std::isnan(p->log_lambda)) return BSFA_ERR_INVALID_ARG;
  if (p->workspace == nullptr || (reinterpret_cast<uintptr_t>(p->workspace) & 255u))
    return BSFA_ERR_WORKSPACE;
  return BSFA_OK;
}

}  // namespace bsfa

using namespace bsfa;

extern "C" {

int bsfa_version(void) { return 0x000100; }

const char* bsfa_status_string(bsfa_status s) {
  switch (s) {
    case BSFA_OK: return "ok";
    case BSFA_ERR_INVALID_ARG: return "invalid argument";
    case BSFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case BSFA_ERR_CUDA: return "CUDA call failed";
    case BSFA_ERR_DEVICE_TIMEOUT: return "device-side wait exceeded its bound";
    case BSFA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

size_t bsfa_prefill_workspace_size(const bsfa_fwd_params* p) {
  if (p == nullptr || p->batch < 0 || p->seqlen < 0 || p->batch > MAX_BATCH) return 0;
  if (p->cu_seqlens != nullptr && p->max_seqlen < 0) return 0;
  return carve(nullptr, p->batch, (int)tiles_bound(p), 0, mean_elems(p)).bytes;
}

bsfa_status bsfa_bitmap_words_per_row(const bsfa_fwd_params* p, int* words_per_row) {
  if (p == nullptr || words_per_row == nullptr || p->block_k <= 0) return BSFA_ERR_INVALID_ARG;
  const long long nk = (max_len_of(p) + p->block_k - 1) / p->block_k;
  *words_per_row = (int)((nk + 31) / 32);
  return BSFA_OK;
}

bsfa_status bsfa_prefill_fwd(const bsfa_fwd_params* p, bsfa_stream_t stream_) {
  const bsfa_status v = validate(p);
  if (v != BSFA_OK) return v;
  if (p->batch == 0 || p->seqlen == 0) return BSFA_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const long long tb = tiles_bound(p);
  const Carve cv = carve(p->workspace, p->batch, (int)tb, 0, mean_elems(p));
  if (p->workspace_bytes < cv.bytes) return BSFA_ERR_WORKSPACE;
  const bool corr = corr_on(p);

  const int d = p->head_dim;
  const int g = p->num_heads_q / p->num_heads_kv;
  const int nq = (g % 2 == 0) ? 2 : 1;
  const bool varlen = p->cu_seqlens != nullptr;
  const int bdim = varlen ? 1 : p->batch;
  const long long max_len = max_len_of(p);
  const int max_tiles = (int)((max_len + TILE - 1) / TILE);

  Maps m;
  // The batch stride is unused in varlen mode; give the map a valid one.
  auto bstride = [&](const int64_t* st, int heads) {
    return varlen ? (long long)st[1] * heads : (long long)st[0];
  };
  const bool f16 = p->dtype == BSFA_DTYPE_F16;
  const bool paged = p->block_table != nullptr;
  const int kv_rows = p->block_k == 224 ? 224 : TILE;  // rows of one K or V tile
  if (!make_map(&m.q, p->q, f16, d, p->seqlen, p->num_heads_q, bdim, p->q_stride[2], p->q_stride[1],
                bstride(p->q_stride, p->num_heads_q)))
    return BSFA_ERR_CUDA;
  if (paged) {
    // Page pools: {d, tokens of a page, KV heads, pages}.
    if (!make_map(&m.k, p->k, f16, d, p->page_size, p->num_heads_kv, p->num_pages, p->k_stride[2],
                  p->k_stride[1], p->k_stride[0]) ||
        !make_map(&m.v, p->v, f16, d, p->page_size, p->num_heads_kv, p->num_pages, p->v_stride[2],
                  p->v_stride[1], p->v_stride[0]))
      return BSFA_ERR_CUDA;
  } else if (!make_map(&m.k, p->k, f16, d, p->seqlen, p->num_heads_kv, bdim, p->k_stride[2],
                       p->k_stride[1], bstride(p->k_stride, p->num_heads_kv), kv_rows) ||
             !make_map(&m.v, p->v, f16, d, p->seqlen, p->num_heads_kv, bdim, p->v_stride[2],
                       p->v_stride[1], bstride(p->v_stride, p->num_heads_kv), kv_rows)) {
    return BSFA_ERR_CUDA;
  }
  m.kb = m.k;
  m.vb = m.v;
  if (corr) {
    // Block-mean tables [Hkv][tb][d]: row r is key block r of the bitmap's
    // row numbering.
    if (!make_map(&m.kb, cv.kbar, f16, d, tb, p->num_heads_kv, 1, d, tb * d,
                  tb * d * p->num_heads_kv) ||
        !make_map(&m.vb, cv.vbar, f16, d, tb, p->num_heads_kv, 1, d, tb * d,
                  tb * d * p->num_heads_kv))
      return BSFA_ERR_CUDA;
  }

  DevParams dp{};
  dp.o = static_cast<uint16_t*>(p->o);
  dp.o_sb = varlen ? 0 : p->o_stride[0];
  dp.o_sh = p->o_stride[1];
  dp.o_st = p->o_stride[2];
  dp.Hq = p->num_heads_q;
  dp.Hkv = p->num_heads_kv;
  dp.group = g;
  dp.pairs = g / nq;
  dp.varlen = varlen ? 1 : 0;
  dp.batch_len = varlen ? 0 : p->seqlen;
  dp.Bq = p->block_q;
  dp.Bk = p->block_k;
  dp.sigma = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt((float)d);
  dp.sigma_log2 = dp.sigma * 1.4426950408889634f;
  dp.mode = p->mode;
  dp.thr = p->thresholds;
  dp.nT = p->thresholds_nq > 0 ? p->thresholds_nq : 1;
  dp.log_lambda = p->log_lambda;
  dp.bitmap = p->kept_bitmap;
  int words = 0;
  bsfa_bitmap_words_per_row(p, &words);
  dp.words = words;
  dp.lse = p->lse;
  dp.lse_rows = varlen ? p->seqlen : (long long)p->batch * p->seqlen;
  dp.counts = p->block_counts;
  dp.seqinfo = cv.seqinfo;
  dp.tiles = cv.tiles;
  dp.ntiles_total = cv.ntot;
  dp.btab = paged ? p->block_table : nullptr;
  dp.bt_stride = paged ? p->block_table_stride : 0;
  dp.tiles_per_page = paged ? p->page_size / TILE : 1;
  dp.corr_shift = std::log(static_cast<float>(p->block_k)) / dp.sigma;
  dp.err = error_word();
  if (dp.err == nullptr) return BSFA_ERR_CUDA;

  const size_t prep_smem = sizeof(int) * ((size_t)p->batch + (size_t)max_tiles);
  if (prep_smem > 48 * 1024 &&
      cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)prep_smem) != cudaSuccess)
    return BSFA_ERR_CUDA;
  prep_kernel<<<1, PREP_THREADS, prep_smem, stream>>>(p->cu_seqlens, p->batch, p->seqlen,
                                                       varlen ? 1 : 0, p->block_q, max_tiles,
                                                       cv.seqinfo, cv.tiles, cv.ntot,
                                                       p->block_counts);
  if (cudaGetLastError() != cudaSuccess) return BSFA_ERR_CUDA;
  if (corr) {
    const dim3 mb_block(d, p->num_heads_kv);  // d * Hkv <= 1024, checked by validate()
    const auto* kk = static_cast<const uint16_t*>(p->k);
    const auto* vv = static_cast<const uint16_t*>(p->v);
    const long long ksb = varlen ? 0 : p->k_stride[0], vsb = varlen ? 0 : p->v_stride[0];
    if (f16)
      block_mean_kernel<true><<<(unsigned)tb, mb_block, 0, stream>>>(
          kk, vv, ksb, p->k_stride[1], p->k_stride[2], vsb, p->v_stride[1], p->v_stride[2],
          cv.seqinfo, cv.tiles, cv.ntot, cv.kbar, cv.vbar, (int)tb);
    else
      block_mean_kernel<false><<<(unsigned)tb, mb_block, 0, stream>>>(
          kk, vv, ksb, p->k_stride[1], p->k_stride[2], vsb, p->v_stride[1], p->v_stride[2],
          cv.seqinfo, cv.tiles, cv.ntot, cv.kbar, cv.vbar, (int)tb);
    if (cudaGetLastError() != cudaSuccess) return BSFA_ERR_CUDA;
  }
  const int sms = num_sms();
  if (sms <= 0) return BSFA_ERR_CUDA;
  const bool vall = (p->flags & BSFA_FLAG_V_ALWAYS) != 0;
  const Variant var{p->mode != BSFA_GATE_NONE, vall, paged, corr};
  if ((p->flags & BSFA_FLAG_PIPELINED) || p->block_k == 224) {
    // One query head per CTA: units are (KV head, query tile, query head).
    const long long units_xs = tb * p->num_heads_q;
    const int grid_xs = (int)(units_xs < sms ? units_xs : sms);
    const cudaError_t e = f16 ? dispatch_xs_t<true>(d, p->block_k, var, m, dp, grid_xs, stream)
                              : dispatch_xs_t<false>(d, p->block_k, var, m, dp, grid_xs, stream);
    return e == cudaSuccess ? BSFA_OK : BSFA_ERR_CUDA;
  }
  const long long units = tb * p->num_heads_kv * (g / nq);
  const int grid = (int)(units < sms ? units : sms);
  if (dispatch<false>(f16, d, nq, var, m, dp, grid, stream) != cudaSuccess)
    return BSFA_ERR_CUDA;
  return BSFA_OK;
}

size_t bsfa_calibrate_workspace_size(int Hq, int L, int Bq, int Bk) {
  if (Hq <= 0 || L <= 0 || Bq <= 0 || Bk <= 0) return 0;
  const size_t nq = (L + Bq - 1) / Bq, nk = (L + Bk - 1) / Bk;
  return carve(nullptr, 1, (L + TILE - 1) / TILE, (size_t)Hq * nq * nk).bytes;
}

bsfa_status bsfa_calibrate(const void* const* q_samples, const void* const* k_samples,
                           int n_samples, int Hq, int Hkv, int L, int d, int dtype,
                           const int64_t q_stride[2], const int64_t k_stride[2], int Bq, int Bk,
                           float softmax_scale, const int* ks, int n_k, float* out,
                           void* workspace, size_t workspace_bytes, bsfa_stream_t stream_) {
  if (!q_samples || !k_samples || n_samples <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || L <= 0 ||
      !q_stride || !k_stride || !ks || n_k <= 0 || !out)
    return BSFA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return BSFA_ERR_UNSUPPORTED;
  if (dtype != BSFA_DTYPE_BF16 && dtype != BSFA_DTYPE_F16) return BSFA_ERR_UNSUPPORTED;
  const bool f16 = dtype == BSFA_DTYPE_F16;
  const bool tile224 = Bq == TILE && Bk == 224;  // the 128 x 224 tile
  if (!tile224 && ((Bq != 64 && Bq != 128) || (Bk != 64 && Bk != 128)))
    return BSFA_ERR_UNSUPPORTED;
  if (n_k > MAX_BUDGETS) return BSFA_ERR_UNSUPPORTED;
  for (int i = 0; i < n_k; ++i)
    if (ks[i] < 1) return BSFA_ERR_INVALID_ARG;
  const int nqb = (L + Bq - 1) / Bq, nkb = (L + Bk - 1) / Bk;
  if (nkb > MAX_CAL_BLOCKS || (L + TILE - 1) / TILE > MAX_TILES_PER_SEQ) return BSFA_ERR_UNSUPPORTED;
  for (int i = 0; i < 2; ++i)
    if (!stride_ok(q_stride[i]) || !stride_ok(k_stride[i])) return BSFA_ERR_UNSUPPORTED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return BSFA_ERR_WORKSPACE;
  const int max_tiles = (L + TILE - 1) / TILE;
  const Carve cv = carve(workspace, 1, max_tiles, (size_t)Hq * nqb * nkb);
  if (workspace_bytes < cv.bytes) return BSFA_ERR_WORKSPACE;
  for (int n = 0; n < n_samples; ++n)
    if (!q_samples[n] || !k_samples[n] || !aligned16(q_samples[n]) || !aligned16(k_samples[n]))
      return BSFA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  const int g = Hq / Hkv;
  const int nq = (g % 2 == 0) ? 2 : 1;
  DevParams dp{};
  dp.Hq = Hq;
  dp.Hkv = Hkv;
  dp.group = g;
  dp.pairs = g / nq;
  dp.Bq = Bq;
  dp.Bk = Bk;
  dp.sigma = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)d);
  dp.sigma_log2 = dp.sigma * 1.4426950408889634f;
  dp.mode = BSFA_GATE_THRESHOLD;
  dp.seqinfo = cv.seqinfo;
  dp.tiles = cv.tiles;
  dp.ntiles_total = cv.ntot;
  dp.blockmax = cv.blockmax;
  dp.cal_nq = nqb;
  dp.cal_nk = nkb;
  dp.err = error_word();
  if (dp.err == nullptr) return BSFA_ERR_CUDA;

  const int sms = num_sms();
  if (sms <= 0) return BSFA_ERR_CUDA;
  const long long units = (long long)max_tiles * Hkv * (g / nq);
  const int grid = (int)(units < sms ? units : sms);

  SelectArgs sa{};
  sa.blockmax = cv.blockmax;
  sa.out = out;
  sa.Hq = Hq;
  sa.nq = nqb;
  sa.nk = nkb;
  sa.Bq = Bq;
  sa.Bk = Bk;
  sa.L = L;
  sa.n_k = n_k;
  for (int i = 0; i < n_k; ++i) sa.ks[i] = ks[i];
  sa.n_samples = n_samples;
  int sort_n = 1;
  while (sort_n < nkb) sort_n <<= 1;
  const size_t sel_smem = sizeof(float) * (size_t)sort_n;
  if (sel_smem > 48 * 1024 &&
      cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sel_smem) != cudaSuccess)
    return BSFA_ERR_CUDA;
  const int sel_threads = sort_n < 1024 ? (sort_n < 32 ? 32 : sort_n) : 1024;
  if (sel_threads < n_k) return BSFA_ERR_UNSUPPORTED;  // never: n_k <= 16 < 32

  prep_kernel<<<1, PREP_THREADS, sizeof(int) * (1 + (size_t)max_tiles), stream>>>(
      nullptr, 1, L, 0, Bq, max_tiles, cv.seqinfo, cv.tiles, cv.ntot, nullptr);
  if (cudaGetLastError() != cudaSuccess) return BSFA_ERR_CUDA;

  for (int n = 0; n < n_samples; ++n) {
    Maps m;
    if (!make_map(&m.q, q_samples[n], f16, d, L, Hq, 1, q_stride[1], q_stride[0],
                  (long long)q_stride[0] * Hq) ||
        !make_map(&m.k, k_samples[n], f16, d, L, Hkv, 1, k_stride[1], k_stride[0],
                  (long long)k_stride[0] * Hkv, tile224 ? 224 : TILE))
      return BSFA_ERR_CUDA;
    m.v = m.kb = m.vb = m.k;
    cudaError_t e;
    if (tile224) {
      // The single-head calibration kernel: one 224-key tile per semantic block.
      const long long units_xs = (long long)max_tiles * Hq;
      const int grid_xs = (int)(units_xs < sms ? units_xs : sms);
      if (d == 128)
        e = f16 ? launch_xs<128, 224, true, true, true, false, false>(m, dp, grid_xs, stream)
                : launch_xs<128, 224, true, true, false, false, false>(m, dp, grid_xs, stream);
      else
        e = f16 ? launch_xs<64, 224, true, true, true, false, false>(m, dp, grid_xs, stream)
                : launch_xs<64, 224, true, true, false, false, false>(m, dp, grid_xs, stream);
    } else {
      e = dispatch<true>(f16, d, nq, Variant{true, false, false, false}, m, dp, grid, stream);
    }
    if (e != cudaSuccess) return BSFA_ERR_CUDA;
    sa.sample = n;
    select_kernel<<<dim3(nqb, Hq), sel_threads, sel_smem, stream>>>(sa);
    if (cudaGetLastError() != cudaSuccess) return BSFA_ERR_CUDA;
  }
  return BSFA_OK;
}

bsfa_status bsfa_selftest_wait_guard(unsigned int timeout_us, bsfa_stream_t stream_) {
  if (timeout_us == 0 || timeout_us > 10000000u) return BSFA_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (err == nullptr) return BSFA_ERR_CUDA;
  wait_guard_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(
      1000ull * timeout_us, err);
  return cudaGetLastError() == cudaSuccess ? BSFA_OK : BSFA_ERR_CUDA;
}

bsfa_status bsfa_device_error(bsfa_stream_t stream_, unsigned int* code) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BSFA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return BSFA_ERR_CUDA;
  if (code) *code = v;
  if (v != 0u) {
    const unsigned zero = 0u;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return BSFA_ERR_CUDA;
    return BSFA_ERR_DEVICE_TIMEOUT;
  }
  return BSFA_OK;
}

}  // extern "C"
