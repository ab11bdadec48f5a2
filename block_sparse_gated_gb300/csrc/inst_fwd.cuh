// inst_fwd.cuh -- explicit instantiation helper for the attention kernel.
#pragma once
#include "bsfa_launch.h"

namespace bsfa {

template <int D, int NQ, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED, bool CORR>
cudaError_t launch_fwd(const Maps& m, const DevParams& p, int grid, cudaStream_t stream) {
  using LY = Layout<D, NQ, CALIB, CORR>;
  auto* fn = &bsfa_fwd_kernel<D, NQ, GATING, CALIB, F16, VALL, PAGED, CORR>;
  static bool configured[64] = {};  // the attribute is per device; set once on each
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (NQ == 2) {
      // setmaxnreg moves registers between warpgroups inside the block's own
      // allocation; an increase the allocation cannot cover would never
      // complete, so refuse to launch rather than risk it.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      if (128 * COPY_REGS + 256 * SOFTMAX_REGS > LY::NTHREADS * fa.numRegs)
        return cudaErrorInvalidConfiguration;
    }
    if (dev < 64) configured[dev] = true;
  }
  fn<<<grid, LY::NTHREADS, LY::BYTES, stream>>>(m.q, m.k, m.v, m.kb, m.vb, p);
  return cudaGetLastError();
}

}  // namespace bsfa

#define BSFA_INSTANTIATE(D, NQ, G, C, F) BSFA_INSTANTIATE_X(D, NQ, G, C, F, false, false, false)
#define BSFA_INSTANTIATE_V(D, NQ, G, C, F, VA) BSFA_INSTANTIATE_X(D, NQ, G, C, F, VA, false, false)
#define BSFA_INSTANTIATE_VP(D, NQ, G, C, F, VA, PG) BSFA_INSTANTIATE_X(D, NQ, G, C, F, VA, PG, false)
#define BSFA_INSTANTIATE_X(D, NQ, G, C, F, VA, PG, CR)                                  \
  template cudaError_t bsfa::launch_fwd<D, NQ, G, C, F, VA, PG, CR>(const Maps&,        \
                                                                    const DevParams&, int, \
                                                                    cudaStream_t);
