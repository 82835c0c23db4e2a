// Instances of the split-KV decode kernels, cluster variant (the splits of a unit merged through
// distributed shared memory): contiguous K/V, d_head = 64, bf16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_CONTIG_UNIT(cluster_d64_bf16, 64, true, true)
}  // namespace gqa
