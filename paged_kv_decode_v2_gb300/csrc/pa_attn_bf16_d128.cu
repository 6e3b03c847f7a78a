// Attention kernels (V2 phase 1 and V1) for bf16 storage, head_dim 128.
#include "pa_attn.cuh"

namespace pa {
PA_DEFINE_ATTN_OPS(__nv_bfloat16, attn_ops_bf16_d128, 128)
} // namespace pa
