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
// Layout of the copy: [KV][copy_blocks][block_size][head_dim], the blocks the
// sequences use packed within each KV head's part: sequence s's logical block
// j at index offs[s] + j, offs the exclusive prefix sum of ceil(L_s /
// block_size) that the offsets pass writes, so that the blocks one
// (sequence, KV head) pair reads lie back to back; rows past a sequence's end
// are zero.  The offsets pass also sets the flag when the packed copy would not
// fit its space, and the copy pass then writes nothing.  A block id outside
// [0, num_blocks) reads block 0, as the attention kernels do.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kVhScanThreads = 1024;

// One CTA: offs[s] = sum of ceil(L_t / block_size) over t < s, and the flag:
// 1 if the total exceeds copy_blocks, else 0 (the copy pass may raise it).
__global__ void __launch_bounds__(kVhScanThreads) v_half_offsets_kernel(const VhParams p)
{
    __shared__ long long part[kVhScanThreads];
    const int per = (p.num_seqs + kVhScanThreads - 1) / kVhScanThreads;
    const int s0 = threadIdx.x * per;
    const int s1 = min(s0 + per, p.num_seqs);
    auto nblocks = [&](int s) {
        int L = __ldg(&p.seq_lens[s]);
        L = L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
        return (long long)((L + p.block_size - 1) / p.block_size);
    };
    long long sum = 0;
    for (int s = s0; s < s1; ++s)
        sum += nblocks(s);
    part[threadIdx.x] = sum;
    __syncthreads();
    // Inclusive scan of the per-thread sums (Hillis-Steele, in place).
    for (int d = 1; d < kVhScanThreads; d <<= 1) {
        const long long v = threadIdx.x >= d ? part[threadIdx.x - d] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    long long run = part[threadIdx.x] - sum; // exclusive start of this thread's range
    for (int s = s0; s < s1; ++s) {
        p.offs[s] = (int32_t)min(run, (long long)INT32_MAX);
        run += nblocks(s);
    }
    if (threadIdx.x == kVhScanThreads - 1)
        *p.flag = part[kVhScanThreads - 1] > p.copy_blocks ? 1 : 0;
}

constexpr int kVhBlocks = 16;   // packed blocks of one KV head per work item
constexpr int kVhRound = 8;     // chunks per thread in flight
constexpr int kVhThreads = 256;
constexpr int kVhCtasPerSm = 4;

// Persistent: CTAs stride over work items, item = (KV head kv, kVhBlocks
// consecutive packed blocks of it), kv-major, so that neighbouring CTAs write
// neighbouring parts of the copy and no CTA is launched for blocks past the
// sequences' ends.  Packed block q belongs to the last sequence s with
// offs[s] <= q (empty sequences share their offset with the next one).
__global__ void __launch_bounds__(kVhThreads, kVhCtasPerSm) v_half_kernel(const VhParams p)
{
    __shared__ int s_id[kVhBlocks];   // physical block of each of the item's blocks, -1 past the total
    __shared__ int s_rows[kVhBlocks]; // its rows inside the sequence
    __shared__ int s_skip;
    // The flag already set (the packed copy does not fit): nothing to write.
    // Read once, so that the whole CTA takes the same branch.
    if (threadIdx.x == 0)
        s_skip = __ldcg(p.flag);
    __syncthreads();
    if (s_skip != 0)
        return;
    auto length = [&](int t) {
        const int L = __ldg(&p.seq_lens[t]);
        return L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
    };
    const int last = p.num_seqs - 1;
    const long long total =
        (long long)__ldg(&p.offs[last]) + (length(last) + p.block_size - 1) / p.block_size;
    const long long per_kv = (total + kVhBlocks - 1) / kVhBlocks;
    const long long items = per_kv * p.num_kv_heads;
    const int per_row = p.head_dim / 8;                  // 16-byte chunks of a row (a power of two)
    const int chunks = p.block_size * per_row;           // of one block's slice (a power of two)
    const int lg_row = __ffs(per_row) - 1;
    const int lg_chunks = __ffs(chunks) - 1;
    const int span = kVhBlocks * chunks;
    const uint4 *__restrict__ src = static_cast<const uint4 *>(p.value_cache);
    uint4 *__restrict__ dst = static_cast<uint4 *>(p.copy);
    uint32_t big = 0u;
    for (long long item = blockIdx.x; item < items; item += gridDim.x) {
        const int kv = (int)(item / per_kv);
        const long long q0 = (item - (long long)kv * per_kv) * kVhBlocks;
        if (threadIdx.x < kVhBlocks) {
            const long long q = q0 + threadIdx.x;
            int id = -1, rows = 0;
            if (q < total) {
                int lo = 0, hi = last; // the last s with offs[s] <= q
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if ((long long)__ldg(&p.offs[mid]) <= q)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int j = (int)(q - __ldg(&p.offs[lo]));
                id = __ldg(p.block_tables + (size_t)lo * p.max_blocks + j);
                if (id < 0 || id >= p.num_blocks)
                    id = 0;
                rows = min(p.block_size, length(lo) - j * p.block_size);
            }
            s_id[threadIdx.x] = id;
            s_rows[threadIdx.x] = rows;
        }
        __syncthreads();
        uint4 *__restrict__ out = dst + ((size_t)kv * p.copy_blocks + q0) * chunks;
        // kVhRound chunks per thread in flight: all loads of a round before any use.
        for (int base = threadIdx.x; base < span; base += kVhRound * kVhThreads) {
            uint4 x[kVhRound];
            int ok[kVhRound];
#pragma unroll
            for (int u = 0; u < kVhRound; ++u) {
                const int i = base + u * kVhThreads;
                const int jj = i >> lg_chunks;
                const int c = i & (chunks - 1);
                const int id = i < span ? s_id[jj] : -1;
                // 1: a token row, 0: a row past the sequence's end, -1: past the total.
                ok[u] = id < 0 ? -1 : ((c >> lg_row) < s_rows[jj] ? 1 : 0);
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
                out[base + u * kVhThreads] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        __syncthreads(); // s_id / s_rows are rewritten for the next item
    }
    if (__any_sync(0xffffffffu, big != 0u) && (threadIdx.x & 31) == 0)
        atomicOr(p.flag, 1);
}

cudaError_t launch_v_half(const VhParams &p, int num_sms, cudaStream_t stream)
{
    v_half_offsets_kernel<<<1, kVhScanThreads, 0, stream>>>(p);
    // Work items at most: every sequence at the capacity, within the copy's space.
    const long long nb_max = (p.seq_len_cap + p.block_size - 1) / p.block_size;
    long long blocks = nb_max * p.num_seqs;
    if (blocks > p.copy_blocks)
        blocks = p.copy_blocks;
    const long long items = (blocks + kVhBlocks - 1) / kVhBlocks * p.num_kv_heads;
    if (items == 0)
        return cudaGetLastError();
    const long long slots = (long long)num_sms * kVhCtasPerSm;
    v_half_kernel<<<(unsigned)(items < slots ? items : slots), kVhThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

} // namespace pa
