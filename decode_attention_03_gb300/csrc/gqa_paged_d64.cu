// Instances of the split-KV decode kernel: d_head = 64, paged = true.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_UNIT(paged_d64, 64, true)
}  // namespace gqa
