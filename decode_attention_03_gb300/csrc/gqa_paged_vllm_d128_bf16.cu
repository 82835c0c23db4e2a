// Instances of the persistent paged kernel over the vLLM cache layout (key cache
// [blocks, KV heads, d/8, block, 8], value cache [blocks, KV heads, d, block]), d_head = 128,
// bfloat16 elements.
#include "gqa_instances.cuh"

namespace gqa {
GQA_DEFINE_PAGED_UNIT(paged_vllm_d128_bf16, 128, true, true)
}  // namespace gqa
