// Instances of the split-KV decode kernels: paged, d_head = 128, f16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_PAGED_UNIT(paged_d128, 128, false, false)
}  // namespace gqa
