// Instances of the split-KV decode kernel: d_head = 128, paged = true.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_UNIT(paged_d128, 128, true)
}  // namespace gqa
