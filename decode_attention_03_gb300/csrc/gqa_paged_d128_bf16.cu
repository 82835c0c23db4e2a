// Instances of the split-KV decode kernels: paged, d_head = 128, bf16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_PAGED_UNIT(paged_d128_bf16, 128, true, false)
}  // namespace gqa
