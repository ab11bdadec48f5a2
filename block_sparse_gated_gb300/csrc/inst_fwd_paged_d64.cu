// Attention kernels reading K/V from page pools, head_dim 64 (gated and
// gate-compiled-out).
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE_VP(64, 2, true, false, false, false, true)
BSFA_INSTANTIATE_VP(64, 2, true, false, true, false, true)
BSFA_INSTANTIATE_VP(64, 1, true, false, false, false, true)
BSFA_INSTANTIATE_VP(64, 1, true, false, true, false, true)
BSFA_INSTANTIATE_VP(64, 2, false, false, false, false, true)
BSFA_INSTANTIATE_VP(64, 2, false, false, true, false, true)
BSFA_INSTANTIATE_VP(64, 1, false, false, false, false, true)
BSFA_INSTANTIATE_VP(64, 1, false, false, true, false, true)
}  // namespace bsfa
