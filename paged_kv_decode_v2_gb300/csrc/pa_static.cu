// pa_static.cu -- pa_decode_v2_static: the two-pass decode for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain the three phase-1 intermediates
// (tmp_output, exp_sums, max_logits): code that runs inside a host
// framework owning every device allocation, embedded or plug-in runtimes
// that are given a fixed memory budget up front, or hot paths where a
// cudaMalloc (an implicit device synchronisation) is not allowed.  This
// entry point keeps those intermediates in one array that lives in the
// library itself, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable of PA_STATIC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  In
// host code its name is only a stand-in, so its device address is looked
// up with cudaGetSymbolAddress once per device, with that device current,
// on the first call made on that device, and kept for the life of the
// process.  A cudaDeviceReset unloads the library's device code, so the
// kept address would then be stale: this entry point must not be called on
// a device after that device has been reset.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "pa_decode.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_static_scratch[PA_STATIC_SCRATCH_BYTES / sizeof(float)];

// Device address of g_static_scratch, per device (null until looked up).
std::atomic<float *> g_scratch_addr[kMaxDevices];

float *scratch_address(int dev)
{
    float *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p)
        return p;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scratch) != cudaSuccess ||
        p == nullptr)
        return nullptr;
    g_scratch_addr[dev].store(p, std::memory_order_release);
    return p;
}

} // namespace

extern "C" PA_API int pa_decode_v2_static(const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          const int32_t *seq_lens, int num_seqs, int num_heads,
                                          int num_kv_heads, int head_dim, int num_blocks,
                                          int block_size, int max_blocks_per_seq,
                                          int max_seq_len_hint, float scale, int partition_size,
                                          int dtype, void *out, int32_t *status,
                                          pa_stream_t stream)
{
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq <= 0 || partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    // Partitions the call needs: the same count pa_decode_v2 launches.
    const long long full = (long long)max_blocks_per_seq * block_size;
    const long long cap = (max_seq_len_hint > 0 && max_seq_len_hint < full) ? max_seq_len_hint : full;
    const long long np = (cap + partition_size - 1) / partition_size;
    // rows * (head_dim + 2) * 4 bytes must fit the array, rows = num_seqs *
    // num_heads * np.  Compared by successive division, which cannot overflow:
    // for positive integers, np <= floor(floor(R / H) / S) exactly when
    // np * H * S <= R.
    const long long max_rows = (long long)PA_STATIC_SCRATCH_BYTES /
                               (((long long)head_dim + 2) * (long long)sizeof(float));
    if (np < 1 || np > INT32_MAX || np > max_rows / num_heads / num_seqs)
        return PA_ERR_WORKSPACE;
    const long long rows = (long long)num_seqs * num_heads * np;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    float *base = scratch_address(dev);
    if (!base)
        return PA_ERR_CUDA;

    // [tmp_output: rows x head_dim][exp_sums: rows][max_logits: rows].  Every
    // slot that phase 2 reads is written by phase 1 of the same call, so the
    // previous call's contents never need clearing.
    float *tmp_output = base;
    float *exp_sums = tmp_output + rows * head_dim;
    float *max_logits = exp_sums + rows;
    return pa_decode_v2(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, num_heads,
                        num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                        max_seq_len_hint, scale, partition_size, dtype, out, tmp_output, exp_sums,
                        max_logits, (int)np, status, stream);
}
