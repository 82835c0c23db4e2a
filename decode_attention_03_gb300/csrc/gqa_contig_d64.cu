// Instances of the split-KV decode kernel: d_head = 64, paged = false.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_UNIT(contig_d64, 64, false)
}  // namespace gqa
