// tcgen05 attention kernels (V2 phase 1 and V1, many query rows per KV head)
// for bf16 storage, head_dim 128.
#include "pa_tc.cuh"

namespace pa {
PA_DEFINE_TC_OPS(__nv_bfloat16, tc_ops_bf16_d128, 128)
} // namespace pa
