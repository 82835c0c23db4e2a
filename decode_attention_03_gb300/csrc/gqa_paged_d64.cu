// Instances of the split-KV decode kernels: paged, d_head = 64, f16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_PAGED_UNIT(paged_d64, 64, false, false)
}  // namespace gqa
