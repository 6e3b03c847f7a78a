// Attention kernels (V2 phase 1 and V1) instantiated for bfloat16 storage.
#include "pa_attn.cuh"

namespace pa {

cudaError_t attn_prepare_bf16(int block_size, int group, bool v1, int optin_bytes, size_t *limit)
{
    return attn_prepare<__nv_bfloat16>(block_size, group, v1, optin_bytes, limit);
}

cudaError_t launch_attn_bf16(const AttnLaunch &L, cudaStream_t stream)
{
    return attn_launch<__nv_bfloat16>(L, stream);
}

int attn_occupancy_bf16(int block_size, int group, bool v1, int warps, size_t smem_bytes)
{
    return attn_occupancy_t<__nv_bfloat16>(block_size, group, v1, warps, smem_bytes);
}

} // namespace pa
