// Attention kernels for head_dim 64 (gated and gate-compiled-out).
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE(64, 2, true, false)
BSFA_INSTANTIATE(64, 1, true, false)
BSFA_INSTANTIATE(64, 2, false, false)
BSFA_INSTANTIATE(64, 1, false, false)
}  // namespace bsfa
