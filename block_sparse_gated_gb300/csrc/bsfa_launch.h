// bsfa_launch.h -- internal declarations shared by the host API and the
// translation units that instantiate the attention kernel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsfa_fwd.cuh"

namespace bsfa {

struct Maps {
  CUtensorMap q, k, v;
  CUtensorMap kb, vb;  // block-mean tables (mean correction); copies of k, v otherwise
};

// Launches bsfa_fwd_kernel<D, NQ, GATING, CALIB, F16, VALL, PAGED, CORR> with its shared-memory size.
template <int D, int NQ, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED, bool CORR>
cudaError_t launch_fwd(const Maps& m, const DevParams& p, int grid, cudaStream_t stream);

// Launches bsfa_xs_kernel<D, BK, GATING, CALIB, F16, VALL, PAGED, CORR> (one
// query head per CTA, 128-row query tiles, key tiles of BK = 128 or 224; CORR:
// mean correction, BK = 128).
template <int D, int BK, bool GATING, bool CALIB, bool F16, bool VALL, bool PAGED,
          bool CORR = false>
cudaError_t launch_xs(const Maps& m, const DevParams& p, int grid, cudaStream_t stream);

}  // namespace bsfa
