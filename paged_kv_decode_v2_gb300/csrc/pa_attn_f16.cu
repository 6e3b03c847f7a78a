// Attention kernels (V2 phase 1 and V1) instantiated for binary16 storage.
#include "pa_attn.cuh"

namespace pa {

cudaError_t attn_prepare_f16(int block_size, int group, bool v1, int optin_bytes, size_t *limit)
{
    return attn_prepare<__half>(block_size, group, v1, optin_bytes, limit);
}

cudaError_t launch_attn_f16(const AttnLaunch &L, cudaStream_t stream)
{
    return attn_launch<__half>(L, stream);
}

int attn_occupancy_f16(int block_size, int group, bool v1, int warps, size_t smem_bytes)
{
    return attn_occupancy_t<__half>(block_size, group, v1, warps, smem_bytes);
}

} // namespace pa
