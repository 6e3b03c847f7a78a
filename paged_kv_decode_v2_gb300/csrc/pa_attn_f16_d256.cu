// Attention kernels (V2 phase 1 and V1) for f16 storage, head_dim 256.
#include "pa_attn.cuh"

namespace pa {
PA_DEFINE_ATTN_OPS(__half, attn_ops_f16_d256, 256)
} // namespace pa
