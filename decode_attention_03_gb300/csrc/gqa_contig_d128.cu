// Instances of the split-KV decode kernels: contiguous K/V, d_head = 128, f16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_CONTIG_UNIT(contig_d128, 128, false, false)
}  // namespace gqa
