// CUDA-core attention kernels (V2 phase 1 and V1, up to 8 query rows per
// KV head) for f16 storage, head_dim 64.
#include "pa_simt.cuh"

namespace pa {
PA_DEFINE_SIMT_OPS(__half, simt_ops_f16_d64, 64)
} // namespace pa
