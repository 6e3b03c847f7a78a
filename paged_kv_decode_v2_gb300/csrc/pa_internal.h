// pa_internal.h -- host-side interface between the C ABI (pa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_decode.h"

namespace pa {

constexpr int kMaxGroup = 16;        // query rows (columns) one attention CTA serves
constexpr int kMaxQLen = 4096;       // new tokens per sequence
constexpr int kMaxGQA = 64;          // query heads per KV head
constexpr int kMaxWarps = 8;         // warps per attention CTA
constexpr int kMaxStages = 8;        // TMA ring stages per warp
constexpr int kMergeThreads = 128;   // phase-2 CTA size
constexpr int kTcRows = 128;         // tcgen05 kernel: query rows per CTA (the MMA's M)
constexpr int kTcTok = 64;           // tcgen05 kernel: tokens per K/V tile
constexpr float kTcRescaleLog2 = 8.f; // tcgen05 kernel: max P = 2^8 before m moves
constexpr int kTcThreads = 192;      // tcgen05 kernel: 4 row warps, MMA warp, TMA warp
constexpr int kTc2Tok = 128;         // two-tile tcgen05 kernel: tokens per K/V tile
constexpr int kTc2Threads = 320;     // two-tile tcgen05 kernel: 8 row warps, MMA warp, TMA warp

// Arguments of the attention kernel (phase 1 of V2, or V1).
struct AttnParams {
    const void *query;           // [S, q_len, H, D]
    const int32_t *block_tables; // [S, max_blocks]
    const int32_t *seq_lens;     // [S]
    int num_heads;
    int num_kv_heads;
    int group;                   // G = H / KV
    int q_len;                   // new tokens per sequence (query rows per (seq, head))
    int cols;                    // G * q_len query rows per KV head
    int col_groups;              // CTAs that split those rows (16 rows each when > 1)
    int num_blocks;
    int max_blocks;
    int seq_len_cap;             // lengths are clamped to [0, cap]
    float scale;
    int partition_size;          // V2: tokens per partition (any positive value)
    int stages;                  // TMA ring stages per warp (tcgen05 kernel: K ring stages)
    int v_stages;                // tcgen05 kernel: V ring stages
    int q_half;                  // tcgen05 one-tile kernel: only Q rows 64-127 stored (<= 64 rows)
    int max_num_partitions;      // V2: partition capacity of the intermediates
    float *tmp_output;           // V2: [S, q_len, H, NPcap, D]
    float *exp_sums;             // V2: [S, q_len, H, NPcap]
    float *max_logits;           // V2: [S, q_len, H, NPcap]
    void *out;                   // V1 and fused V2: [S, q_len, H, D]
    int32_t *counters;           // fused V2: [S, KV] tickets, zero between calls
    const int32_t *vh_flag;      // binary16 copy of V: its flag, 0 when the copy holds V
    const int32_t *vh_offs;      // binary16 copy of V: each sequence's first block in it
    int vh_blocks;               // and the blocks one KV head's part of it holds
    int32_t *status;
};

struct AttnLaunch {
    AttnParams p;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    CUtensorMap tmap_vh;         // the binary16 copy of V (two-tile bf16 kernel reading it)
    int head_dim;                // 64, 128 or 256
    int block_size;              // 8, 16, 32 or 64
    int dtype;                   // PA_F16 / PA_BF16
    bool v1;
    bool fused;                  // V2 with the merge in the last CTA of each (seq, KV head)
    bool simt;                   // the CUDA-core kernel (up to 8 rows) instead of mma.sync
    bool tc;                     // a tcgen05 kernel
    int tc_tiles;                // its 128-row query tiles per CTA (1 or 2)
    bool vh;                     // two tiles, bf16: V from the binary16 copy, binary16 P.V
    int cta_cols;                // query rows one CTA serves (<= 16): picks the n-tile count
    dim3 grid;
    int warps;
    size_t smem_bytes;
};

struct MergeParams {
    const int32_t *seq_lens;
    int q_len;                   // rows of the grid's y dimension are (sequence, new token)
    int num_heads;
    int head_dim;
    int seq_len_cap;
    int partition_size;
    int max_num_partitions;
    const float *tmp_output;
    const float *exp_sums;
    const float *max_logits;
    void *out;
    int32_t *status;
};

// The binary16 copy of the V blocks a multi-query call reads (bf16 caches):
// the blocks the sequences use, packed -- sequence s's logical block j at
// index offs[s] + j of a [blocks][KV][block_size][head_dim] array (offs the
// exclusive prefix sum of ceil(L_s / block_size)), rows past a sequence's
// end zero -- and a flag word, 1 when the copy is not to be used: a finite
// value of 2^16 or more in magnitude, or more blocks than `copy_blocks`.
struct VhParams {
    const void *value_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int num_seqs;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int num_blocks;
    int max_blocks;
    int seq_len_cap;
    long long copy_blocks;       // blocks the copy's space holds
    int32_t *offs;               // [num_seqs], written by the offsets pass
    void *copy;
    int32_t *flag;
};
cudaError_t launch_v_half(const VhParams &p, int num_sms, cudaStream_t stream);
// Query rows per KV head below which the copy is not made (unless
// pa_set_rows_kernel(4) forces the two-tile kernel): the copy costs one read
// and one write of the V blocks whatever the rows, while the binary16 P.V it
// enables saves MMA work in proportion to them.  On uniform batches of 1 to
// 8192 tokens it paid from 1024 rows per KV head and lost at 256.
constexpr int kVhMinRows = 1024;

// Per-warp shared-memory ring bytes for one stage: a K tile and a V tile of
// block_size rows (at least 16: an 8-token block size stages two blocks) x
// head_dim 16-bit values.
inline size_t stage_bytes(int block_size, int head_dim)
{
    return static_cast<size_t>(block_size < 16 ? 16 : block_size) * head_dim * 4;
}

// Scratch one warp needs to hand its partial {m, l, o} to the CTA merge.
inline size_t warp_scratch_bytes(int cta_cols, int head_dim)
{
    int heads = cta_cols <= 8 ? 8 : 16;
    return static_cast<size_t>(heads) * (2 + head_dim + 4) * 4;
}

// Entry points of the attention kernels for one (storage type, head_dim).
// `variant`: 0 = V2 phase 1, 1 = V1, 2 = fused V2 (mma.sync kernels only).
struct AttnOps {
    cudaError_t (*prepare)(int block_size, int cta_cols, int variant, int optin_bytes,
                           size_t *limit);
    int (*occupancy)(int block_size, int cta_cols, int variant, int warps, size_t smem_bytes);
    cudaError_t (*launch)(const AttnLaunch &L, cudaStream_t stream);
};
const AttnOps *attn_ops_f16_d64();
const AttnOps *attn_ops_f16_d128();
const AttnOps *attn_ops_f16_d256();
const AttnOps *attn_ops_bf16_d64();
const AttnOps *attn_ops_bf16_d128();
const AttnOps *attn_ops_bf16_d256();

inline int attn_variant(const AttnLaunch &L) { return L.v1 ? 1 : L.fused ? 2 : 0; }

inline const AttnOps *attn_ops(int dtype, int head_dim)
{
    if (dtype == PA_BF16)
        return head_dim == 64 ? attn_ops_bf16_d64() : head_dim == 128 ? attn_ops_bf16_d128()
                                                                       : attn_ops_bf16_d256();
    return head_dim == 64 ? attn_ops_f16_d64() : head_dim == 128 ? attn_ops_f16_d128()
                                                                  : attn_ops_f16_d256();
}

// The CUDA-core (SIMT) attention kernels for up to 8 query rows per KV head:
// same launch shape, ring and outputs as the mma.sync kernels above.
const AttnOps *simt_ops_f16_d64();
const AttnOps *simt_ops_f16_d128();
const AttnOps *simt_ops_f16_d256();
const AttnOps *simt_ops_bf16_d64();
const AttnOps *simt_ops_bf16_d128();
const AttnOps *simt_ops_bf16_d256();

inline const AttnOps *simt_ops(int dtype, int head_dim)
{
    if (dtype == PA_BF16)
        return head_dim == 64 ? simt_ops_bf16_d64() : head_dim == 128 ? simt_ops_bf16_d128()
                                                                       : simt_ops_bf16_d256();
    return head_dim == 64 ? simt_ops_f16_d64() : head_dim == 128 ? simt_ops_f16_d128()
                                                                  : simt_ops_f16_d256();
}

// Dynamic shared memory of the tcgen05 kernel: the Q tile, k_stages K tiles
// and v_stages V tiles, and 1 KB to align the base to the 1024-byte swizzle
// atom.
inline size_t tc_smem_bytes(int head_dim, int k_stages, int v_stages, bool q_half = false)
{
    return 1024 + (size_t)(q_half ? kTcRows / 2 : kTcRows) * head_dim * 2 +
           (size_t)(k_stages + v_stages) * kTcTok * head_dim * 2;
}

// Dynamic shared memory of the two-tile tcgen05 kernel: two Q tiles, k_stages
// K tiles and v_stages V tiles of 128 tokens, and the 1 KB alignment slack.
inline size_t tc2_smem_bytes(int head_dim, int k_stages, int v_stages)
{
    return 1024 + (size_t)2 * kTcRows * head_dim * 2 +
           (size_t)(k_stages + v_stages) * kTc2Tok * head_dim * 2;
}

// Entry points of the tcgen05 attention kernels for one (storage type, head_dim).
struct TcOps {
    cudaError_t (*prepare)(int block_size, bool v1, int tiles, bool vh, int optin_bytes,
                           size_t *limit);
    cudaError_t (*launch)(const AttnLaunch &L, cudaStream_t stream);
};
const TcOps *tc_ops_f16_d64();
const TcOps *tc_ops_f16_d128();
const TcOps *tc_ops_f16_d256();
const TcOps *tc_ops_bf16_d64();
const TcOps *tc_ops_bf16_d128();
const TcOps *tc_ops_bf16_d256();

inline const TcOps *tc_ops(int dtype, int head_dim)
{
    if (dtype == PA_BF16)
        return head_dim == 64 ? tc_ops_bf16_d64() : head_dim == 128 ? tc_ops_bf16_d128()
                                                                     : tc_ops_bf16_d256();
    return head_dim == 64 ? tc_ops_f16_d64() : head_dim == 128 ? tc_ops_f16_d128()
                                                                : tc_ops_f16_d256();
}

// Merge form: 1 one CTA per (head, row, slice of head_dim), 2 one warp per
// (row, head); `forced` 1 or 2 picks it, 0 lets the rule choose.
int merge_form(const MergeParams &p, int num_seqs, int num_sms, int forced);
cudaError_t launch_merge(int dtype, const MergeParams &p, int num_seqs, int num_sms, int form,
                         cudaStream_t stream);

cudaError_t launch_wait_selftest(int32_t *status, unsigned long long limit_ns, cudaStream_t stream);

} // namespace pa
