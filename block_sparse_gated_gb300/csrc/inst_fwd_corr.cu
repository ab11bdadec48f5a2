// Gated attention kernels with mean correction for skipped blocks (head_dim
// 128 and 64, bf16 and fp16, one or two q-head slots).
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE_X(128, 2, true, false, false, false, false, true)
BSFA_INSTANTIATE_X(128, 2, true, false, true, false, false, true)
BSFA_INSTANTIATE_X(128, 1, true, false, false, false, false, true)
BSFA_INSTANTIATE_X(128, 1, true, false, true, false, false, true)
BSFA_INSTANTIATE_X(64, 2, true, false, false, false, false, true)
BSFA_INSTANTIATE_X(64, 2, true, false, true, false, false, true)
BSFA_INSTANTIATE_X(64, 1, true, false, false, false, false, true)
BSFA_INSTANTIATE_X(64, 1, true, false, true, false, false, true)
}  // namespace bsfa
