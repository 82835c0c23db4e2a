// tcgen05 split kernel, d_head = 64: f16 and bf16, with and without the causal tail.
#include "gqa_tc.cuh"

namespace gqa {
GQA_DEFINE_TC_UNIT(tc_d64, 64)
}  // namespace gqa
