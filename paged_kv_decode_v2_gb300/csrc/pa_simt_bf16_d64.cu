// CUDA-core attention kernels (V2 phase 1 and V1, up to 8 query rows per
// KV head) for bf16 storage, head_dim 64.
#include "pa_simt.cuh"

namespace pa {
PA_DEFINE_SIMT_OPS(__nv_bfloat16, simt_ops_bf16_d64, 64)
} // namespace pa
