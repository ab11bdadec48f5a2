// Gated attention kernels that load V for every visible tile (kept or not),
// for measuring what skipping the load of a skipped tile's V saves.
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE_V(128, 2, true, false, false, true)
BSFA_INSTANTIATE_V(128, 2, true, false, true, true)
BSFA_INSTANTIATE_V(128, 1, true, false, false, true)
BSFA_INSTANTIATE_V(128, 1, true, false, true, true)
BSFA_INSTANTIATE_V(64, 2, true, false, false, true)
BSFA_INSTANTIATE_V(64, 2, true, false, true, true)
BSFA_INSTANTIATE_V(64, 1, true, false, false, true)
BSFA_INSTANTIATE_V(64, 1, true, false, true, true)
}  // namespace bsfa
