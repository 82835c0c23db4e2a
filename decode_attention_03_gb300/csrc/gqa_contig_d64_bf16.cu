// Instances of the split-KV decode kernels: contiguous K/V, d_head = 64, bf16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_CONTIG_UNIT(contig_d64_bf16, 64, true, false)
}  // namespace gqa
