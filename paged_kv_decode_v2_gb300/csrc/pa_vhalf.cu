// pa_vhalf.cu -- a binary16 copy of the V blocks one multi-query call reads,
// for bf16 caches.
//
// Every bf16 value below 2^16 in magnitude has an exact binary16 form (its 8
// significant bits fit in 11 and its exponent in binary16's range; below
// 2^-14 binary16's subnormal spacing of 2^-24 loses at most 2^-25), and inf
// and NaN map to inf and NaN.  With V in binary16, P.V of the two-tile
// tcgen05 kernel runs on binary16 P and V, one MMA per K-step, where bf16's P
// needs a hi + lo pair.  A finite value of 2^16 or more sets *flag, and the
// attention kernel then reads the bf16 cache with the hi + lo pair instead.
//
// Layout of the copy: [S][KV][max_blocks][block_size][head_dim], the
// sequence's logical block j at index j; rows past the sequence's end are
// zero.  A block id outside [0, num_blocks) reads block 0, as the attention
// kernels do.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kVhBlocks = 16;   // blocks of one (sequence, KV head) per CTA
constexpr int kVhRound = 8;     // chunks per thread in flight
constexpr int kVhThreads = 256;

__global__ void __launch_bounds__(kVhThreads) v_half_kernel(const VhParams p)
{
    __shared__ int s_id[kVhBlocks]; // physical block of each of the CTA's blocks, -1 past the end
    const int s = blockIdx.z;
    const int kv = blockIdx.y;
    const int j0 = blockIdx.x * kVhBlocks;
    int L = __ldg(&p.seq_lens[s]);
    L = L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
    const int nb = (L + p.block_size - 1) / p.block_size;
    if (threadIdx.x < kVhBlocks) {
        const int j = j0 + threadIdx.x;
        int id = -1;
        if (j < nb) {
            id = __ldg(p.block_tables + (size_t)s * p.max_blocks + j);
            if (id < 0 || id >= p.num_blocks)
                id = 0;
        }
        s_id[threadIdx.x] = id;
    }
    __syncthreads();
    const int per_row = p.head_dim / 8;            // 16-byte chunks of a row
    const int chunks = p.block_size * per_row;     // of one block's slice
    const int total = kVhBlocks * chunks;
    const uint4 *__restrict__ src = static_cast<const uint4 *>(p.value_cache);
    uint4 *__restrict__ dst = static_cast<uint4 *>(p.copy) +
                              (((size_t)s * p.num_kv_heads + kv) * p.max_blocks + j0) * chunks;
    uint32_t big = 0u;
    // kVhRound chunks per thread in flight: all loads of a round before any use.
    for (int base = threadIdx.x; base < total; base += kVhRound * kVhThreads) {
        uint4 x[kVhRound];
        int ok[kVhRound];
#pragma unroll
        for (int u = 0; u < kVhRound; ++u) {
            const int i = base + u * kVhThreads;
            const int jj = i / chunks;
            const int c = i - jj * chunks;
            const int id = i < total ? s_id[jj] : -1;
            // 1: a token row, 0: a row past the sequence's end, -1: a block past it.
            ok[u] = id < 0 ? -1 : ((j0 + jj) * p.block_size + c / per_row < L ? 1 : 0);
            x[u] = ok[u] == 1 ? __ldg(src + ((size_t)id * p.num_kv_heads + kv) * chunks + c)
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kVhRound; ++u) {
            if (ok[u] < 0)
                continue;
            uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // Per half: 0x4780 (2^16) <= |bits| < 0x7f80 (inf): finite and too large.
                const uint32_t m = w[k] & 0x7fff7fffu;
                big |= __vcmpgeu2(m, 0x47804780u) & __vcmpltu2(m, 0x7f807f80u);
                const __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16),
                                                    __uint_as_float(w[k] & 0xffff0000u));
                w[k] = *reinterpret_cast<const uint32_t *>(&h);
            }
            dst[base + u * kVhThreads] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    if (__any_sync(0xffffffffu, big != 0u) && (threadIdx.x & 31) == 0)
        atomicOr(p.flag, 1);
}

cudaError_t launch_v_half(const VhParams &p, int num_seqs, cudaStream_t stream)
{
    const int nb_max = (p.seq_len_cap + p.block_size - 1) / p.block_size;
    if (nb_max == 0)
        return cudaSuccess;
    const dim3 grid((unsigned)((nb_max + kVhBlocks - 1) / kVhBlocks), (unsigned)p.num_kv_heads,
                    (unsigned)num_seqs);
    v_half_kernel<<<grid, kVhThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace pa
