// Attention kernels (V2 phase 1 and V1) for f16 storage, head_dim 64.
#include "pa_attn.cuh"

namespace pa {
PA_DEFINE_ATTN_OPS(__half, attn_ops_f16_d64, 64)
} // namespace pa
