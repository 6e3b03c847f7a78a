// pa_merge.cu -- phase 2 of split-K decode: the cross-partition
// log-sum-exp merge ("paged_attention_v2_pytorch.py" commit 9cb7f9d,
// "Implementation", Phase 2):
//     global_max = max_p max_logits[p]
//     rescale_p  = exp(max_logits[p] - global_max) * exp_sums[p]
//     out        = sum_p (rescale_p / sum_q rescale_q) * tmp_output[p]
// and the self-test kernel of the bounded wait.
//
// One CTA per (query head, sequence).  Warp w takes partitions w, w + 8, ...
// and each lane 4 consecutive dims (one float4 per partition), so a warp
// reads one 512-byte partition row per step; the eight warps' partial sums
// meet in shared memory.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p)
{
    using E = Elem<T>;
    constexpr int kWarps = kMergeThreads / 32;
    __shared__ float4 s_acc[kWarps][32];
    __shared__ float s_w[kWarps];
    __shared__ float s_max[kWarps];

    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    int L = __ldg(&p.seq_lens[b]);
    L = L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
    const int np = (L + p.partition_size - 1) / p.partition_size;
    const size_t bh = (size_t)b * p.num_heads + h;
    T *out = static_cast<T *>(p.out) + bh * kHeadDim;
    if (np == 0) {
        if (threadIdx.x < kHeadDim)
            out[threadIdx.x] = E::from_float(0.f);
        return;
    }
    const float *ml = p.max_logits + bh * p.max_num_partitions;
    const float *es = p.exp_sums + bh * p.max_num_partitions;
    const float4 *tmp = reinterpret_cast<const float4 *>(p.tmp_output + bh * p.max_num_partitions * kHeadDim);

    // global_max
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < np; i += kMergeThreads)
        mx = fmaxf(mx, __ldg(ml + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0)
        s_max[warp] = mx;
    __syncthreads();
    float gmax = s_max[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
        gmax = fmaxf(gmax, s_max[w]);
    const float gmax2 = gmax * kLog2e;

    // sum_p rescale_p * o_p and sum_p rescale_p
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
#pragma unroll 4
    for (int i = warp; i < np; i += kWarps) {
        const float w = fast_exp2(fmaf(__ldg(ml + i), kLog2e, -gmax2)) * __ldg(es + i);
        const float4 v = __ldg(tmp + (size_t)i * (kHeadDim / 4) + lane);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
        wsum += w;
    }
    s_acc[warp][lane] = acc;
    if (lane == 0)
        s_w[warp] = wsum;
    __syncthreads();

    if (threadIdx.x < kHeadDim) {
        const int d = threadIdx.x;
        float total = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            total += s_w[w];
            const float *a = reinterpret_cast<const float *>(&s_acc[w][d >> 2]);
            o += a[d & 3];
        }
        out[d] = E::from_float(o / total);
    }
}

cudaError_t launch_merge(int dtype, const MergeParams &p, int num_seqs, cudaStream_t stream)
{
    dim3 grid(p.num_heads, num_seqs);
    if (dtype == PA_BF16)
        merge_kernel<__nv_bfloat16><<<grid, kMergeThreads, 0, stream>>>(p);
    else
        merge_kernel<__half><<<grid, kMergeThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// One warp waits on a barrier that nothing completes; the bounded wait must
// give up after limit_ns and report PA_STATUS_TIMEOUT.
__global__ void wait_selftest_kernel(int32_t *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    const uint32_t a = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(a, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(a, 0, limit_ns);
    if (!ok && threadIdx.x == 0)
        set_status(status, PA_STATUS_TIMEOUT);
}

cudaError_t launch_wait_selftest(int32_t *status, unsigned long long limit_ns, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

} // namespace pa
