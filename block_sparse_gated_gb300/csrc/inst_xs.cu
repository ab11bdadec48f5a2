// Pipelined attention kernels (one query head per CTA, two S buffers) for
// 128 x 128 semantic blocks.
#include "inst_xs.cuh"

namespace bsfa {

#define BSFA_XS(D, G, F, VA, PG) \
  template cudaError_t launch_xs<D, 128, G, false, F, VA, PG>(const Maps&, const DevParams&, int, \
                                                              cudaStream_t);
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
// Mean correction (gated, contiguous K/V).
template cudaError_t launch_xs<128, 128, true, false, false, false, false, true>(
    const Maps&, const DevParams&, int, cudaStream_t);
template cudaError_t launch_xs<128, 128, true, false, true, false, false, true>(
    const Maps&, const DevParams&, int, cudaStream_t);
template cudaError_t launch_xs<64, 128, true, false, false, false, false, true>(
    const Maps&, const DevParams&, int, cudaStream_t);
template cudaError_t launch_xs<64, 128, true, false, true, false, false, true>(
    const Maps&, const DevParams&, int, cudaStream_t);

}  // namespace bsfa
