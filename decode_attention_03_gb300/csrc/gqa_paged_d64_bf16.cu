// Instances of the split-KV decode kernels: paged, d_head = 64, bf16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_PAGED_UNIT(paged_d64_bf16, 64, true, false)
}  // namespace gqa
