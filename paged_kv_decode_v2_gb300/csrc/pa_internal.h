// pa_internal.h -- host-side interface between the C ABI (pa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 16;        // query heads per KV head
constexpr int kMaxWarps = 8;         // warps per attention CTA
constexpr int kMaxStages = 8;        // TMA ring stages per warp
constexpr int kMergeThreads = 128;   // phase-2 CTA size

// Arguments of the attention kernel (phase 1 of V2, or V1).
struct AttnParams {
    const void *query;           // [S, H, 128]
    const int32_t *block_tables; // [S, max_blocks]
    const int32_t *seq_lens;     // [S]
    int num_heads;
    int num_kv_heads;
    int group;                   // G = H / KV
    int num_blocks;
    int max_blocks;
    int seq_len_cap;             // lengths are clamped to [0, cap]
    float scale;
    int part_blocks;             // V2: blocks per partition
    int stages;                  // TMA ring stages per warp
    int max_num_partitions;      // V2: partition capacity of the intermediates
    float *tmp_output;           // V2: [S, H, NPcap, 128]
    float *exp_sums;             // V2: [S, H, NPcap]
    float *max_logits;           // V2: [S, H, NPcap]
    void *out;                   // V1: [S, H, 128]
    int32_t *status;
};

struct AttnLaunch {
    AttnParams p;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    int block_size;              // 16 or 32
    int dtype;                   // PA_F16 / PA_BF16
    bool v1;
    dim3 grid;
    int warps;
    size_t smem_bytes;
};

struct MergeParams {
    const int32_t *seq_lens;
    int num_heads;
    int seq_len_cap;
    int partition_size;
    int max_num_partitions;
    const float *tmp_output;
    const float *exp_sums;
    const float *max_logits;
    void *out;
    int32_t *status;
};

// Per-warp shared-memory ring bytes for one stage: K and V tiles, 2 halves of 128-byte lines.
inline size_t stage_bytes(int block_size) { return static_cast<size_t>(block_size) * 512; }

// Scratch one warp needs to hand its partial {m, l, o} to the CTA merge.
inline size_t warp_scratch_bytes(int group)
{
    int heads = group <= 8 ? 8 : 16;
    return static_cast<size_t>(heads) * (2 + 132) * 4;
}

cudaError_t launch_attn_f16(const AttnLaunch &L, cudaStream_t stream);
cudaError_t launch_attn_bf16(const AttnLaunch &L, cudaStream_t stream);
cudaError_t attn_prepare_f16(int block_size, int group, bool v1, int optin_bytes, size_t *limit);
cudaError_t attn_prepare_bf16(int block_size, int group, bool v1, int optin_bytes, size_t *limit);
cudaError_t launch_merge(int dtype, const MergeParams &p, int num_seqs, int num_sms,
                         cudaStream_t stream);
int attn_occupancy(int dtype, int block_size, int group, bool v1, int warps, size_t smem_bytes);
int attn_occupancy_f16(int block_size, int group, bool v1, int warps, size_t smem_bytes);
int attn_occupancy_bf16(int block_size, int group, bool v1, int warps, size_t smem_bytes);
cudaError_t launch_wait_selftest(int32_t *status, unsigned long long limit_ns, cudaStream_t stream);

} // namespace pa
