// Attention kernels (V2 phase 1 and V1) for f16 storage, head_dim 128.
#include "pa_attn.cuh"

namespace pa {
PA_DEFINE_ATTN_OPS(__half, attn_ops_f16_d128, 128)
} // namespace pa
