// Pipelined attention kernels (one query head per CTA, two S buffers) for
// 128 x 128 semantic blocks.
#include "bsfa_launch.h"
#include "bsfa_xs.cuh"

namespace bsfa {

template <int D, bool GATING, bool F16, bool VALL, bool PAGED>
cudaError_t launch_xs(const Maps& m, const DevParams& p, int grid, cudaStream_t stream) {
  using LY = XsLayout<D>;
  auto* fn = &bsfa_xs_kernel<D, GATING, F16, VALL, PAGED>;
  static bool configured[64] = {};  // the attribute is per device; set once on each
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  fn<<<grid, LY::NTHREADS, LY::BYTES, stream>>>(m.q, m.k, m.v, p);
  return cudaGetLastError();
}

#define BSFA_XS(D, G, F, VA, PG) \
  template cudaError_t launch_xs<D, G, F, VA, PG>(const Maps&, const DevParams&, int, cudaStream_t);
BSFA_XS(128, true, false, false, false)
BSFA_XS(128, true, true, false, false)
BSFA_XS(128, false, false, false, false)
BSFA_XS(128, false, true, false, false)
BSFA_XS(128, true, false, true, false)
BSFA_XS(128, true, true, true, false)
BSFA_XS(128, true, false, false, true)
BSFA_XS(128, true, true, false, true)
BSFA_XS(128, false, false, false, true)
BSFA_XS(128, false, true, false, true)
BSFA_XS(64, true, false, false, false)
BSFA_XS(64, true, true, false, false)
BSFA_XS(64, false, false, false, false)
BSFA_XS(64, false, true, false, false)
BSFA_XS(64, true, false, true, false)
BSFA_XS(64, true, true, true, false)
BSFA_XS(64, true, false, false, true)
BSFA_XS(64, true, true, false, true)
BSFA_XS(64, false, false, false, true)
BSFA_XS(64, false, true, false, true)
#undef BSFA_XS

}  // namespace bsfa
