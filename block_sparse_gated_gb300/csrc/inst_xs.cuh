// inst_xs.cuh -- explicit instantiation helper for the single-head kernel.
#pragma once
#include "bsfa_launch.h"
#include "bsfa_xs.cuh"

namespace bsfa {

template <int D, int BK, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED, bool CORR>
cudaError_t launch_xs(const Maps& m, const DevParams& p, int grid, cudaStream_t stream) {
  using LY = XsLayout<D, BK, CALIB>;
  auto* fn = &bsfa_xs_kernel<D, BK, GATING, CALIB, F16, VALL, PAGED, CORR>;
  static bool configured[64] = {};  // the attribute is per device; set once on each
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  fn<<<grid, LY::NTHREADS, LY::BYTES, stream>>>(m.q, m.k, m.v, m.kb, m.vb, p);
  return cudaGetLastError();
}

}  // namespace bsfa
