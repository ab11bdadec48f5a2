// Attention kernels for head_dim 128 (gated and gate-compiled-out).
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE(128, 2, true, false, false)
BSFA_INSTANTIATE(128, 2, true, false, true)
BSFA_INSTANTIATE(128, 1, true, false, false)
BSFA_INSTANTIATE(128, 1, true, false, true)
BSFA_INSTANTIATE(128, 2, false, false, false)
BSFA_INSTANTIATE(128, 2, false, false, true)
BSFA_INSTANTIATE(128, 1, false, false, false)
BSFA_INSTANTIATE(128, 1, false, false, true)
}  // namespace bsfa
