// Instances of the split-KV decode kernel: d_head = 128, paged = false.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_UNIT(contig_d128, 128, false)
}  // namespace gqa
