// tcgen05 attention kernels (V2 phase 1 and V1, many query rows per KV head)
// for f16 storage, head_dim 256.
#include "pa_tc.cuh"

namespace pa {
PA_DEFINE_TC_OPS(__half, tc_ops_f16_d256, 256)
} // namespace pa
