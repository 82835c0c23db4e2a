// Instances of the split-KV decode kernels: contiguous K/V, d_head = 64, f16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_CONTIG_UNIT(contig_d64, 64, false, false)
}  // namespace gqa
