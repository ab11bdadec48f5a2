// Single-head attention kernels for the 128 x 224 tile (Bq = 128, Bk = 224),
// and the calibration kernels for that tile.
#include "inst_xs.cuh"

namespace bsfa {

#define BSFA_XS224(D, G, C, F, VA) \
  template cudaError_t launch_xs<D, 224, G, C, F, VA, false>(const Maps&, const DevParams&, int, \
                                                             cudaStream_t);
BSFA_XS224(128, true, false, false, false)
BSFA_XS224(128, true, false, true, false)
BSFA_XS224(128, false, false, false, false)
BSFA_XS224(128, false, false, true, false)
BSFA_XS224(128, true, false, false, true)
BSFA_XS224(128, true, false, true, true)
BSFA_XS224(64, true, false, false, false)
BSFA_XS224(64, true, false, true, false)
BSFA_XS224(64, false, false, false, false)
BSFA_XS224(64, false, false, true, false)
BSFA_XS224(64, true, false, false, true)
BSFA_XS224(64, true, false, true, true)
BSFA_XS224(128, true, true, false, false)
BSFA_XS224(128, true, true, true, false)
BSFA_XS224(64, true, true, false, false)
BSFA_XS224(64, true, true, true, false)
#undef BSFA_XS224

}  // namespace bsfa
