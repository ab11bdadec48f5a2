// Calibration variants of the attention kernel (Q.K^T tiles and block maxima only).
#include "inst_fwd.cuh"
namespace bsfa {
BSFA_INSTANTIATE(128, 2, true, true, false)
BSFA_INSTANTIATE(128, 2, true, true, true)
BSFA_INSTANTIATE(128, 1, true, true, false)
BSFA_INSTANTIATE(128, 1, true, true, true)
BSFA_INSTANTIATE(64, 2, true, true, false)
BSFA_INSTANTIATE(64, 2, true, true, true)
BSFA_INSTANTIATE(64, 1, true, true, false)
BSFA_INSTANTIATE(64, 1, true, true, true)
}  // namespace bsfa
