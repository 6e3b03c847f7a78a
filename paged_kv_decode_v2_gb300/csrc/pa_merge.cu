// pa_merge.cu -- phase 2 of split-K decode: the cross-partition
// log-sum-exp merge ("paged_attention_v2_pytorch.py" commit 9cb7f9d,
// "Implementation", Phase 2):
//     global_max = max_p max_logits[p]
//     rescale_p  = exp(max_logits[p] - global_max) * exp_sums[p]
//     out        = sum_p (rescale_p / sum_q rescale_q) * tmp_output[p]
// and the self-test kernel of the bounded wait.
//
// One CTA per (query head, sequence, slice of head_dim); the slice is at
// most 128 dims, and smaller (down to 16) when there are few (seq, head)
// pairs.  A group of lanes owns one partition at a time and reads the
// slice as float4s (contiguous bytes); the groups of a CTA take partitions
// round robin and their running states meet in shared memory.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int DD>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p)
{
    using E = Elem<T>;
    constexpr int kGroup = DD / 4;                 // lanes per partition (one float4 each)
    constexpr int kSlots = kMergeThreads / kGroup; // partitions in flight per CTA
    __shared__ float s_m[kSlots];
    __shared__ float s_l[kSlots];
    __shared__ float4 s_acc[kSlots][kGroup];

    const int h = blockIdx.x;
    const int row = blockIdx.y;       // (sequence, new token) = b * q_len + i
    const int b = row / p.q_len;
    const int D = p.head_dim;
    const int d0 = blockIdx.z * DD;
    const int slot = threadIdx.x / kGroup; // partitions slot, slot + kSlots, ...
    const int c = threadIdx.x % kGroup;    // float4 column within the CTA's dims

    // The next call's attention grid may be scheduled while this one runs; it
    // waits for this grid's completion before it touches global memory.
    asm volatile("griddepcontrol.launch_dependents;");
    // Inputs not written by phase 1 may be read before the dependency wait.
    int L = __ldg(&p.seq_lens[b]);
    L = L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
    const int np = (L + p.partition_size - 1) / p.partition_size;
    const size_t bh = (size_t)row * p.num_heads + h;
    T *out = static_cast<T *>(p.out) + bh * D + d0;
    if (np == 0) {
        if (threadIdx.x < DD)
            out[threadIdx.x] = E::from_float(0.f);
        return;
    }
    const float *ml = p.max_logits + bh * p.max_num_partitions;
    const float *es = p.exp_sums + bh * p.max_num_partitions;
    const float4 *tmp = reinterpret_cast<const float4 *>(p.tmp_output + bh * p.max_num_partitions * D + d0);
    const int row4 = D / 4; // float4s between partitions

    // Phase 1's results are visible only after this point.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // One pass over the partitions with a running maximum: the pages' rule
    // rescale_p = exp(m_p - M) * l_p, with M raised as larger maxima appear
    // and the partial sums multiplied by exp(M_old - M_new).
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int i = slot; i < np; i += kSlots) {
        const float mp = __ldg(ml + i);
        const float lp = __ldg(es + i);
        const float4 v = __ldg(tmp + (size_t)i * row4 + c);
        if (lp == 0.f) // a partition none of whose tokens this query sees
            continue;
        const float mn = fmaxf(m, mp);
        const float a = fast_exp2((m - mn) * kLog2e); // 0 while m is -inf
        const float w = fast_exp2((mp - mn) * kLog2e) * lp;
        acc.x = fmaf(acc.x, a, w * v.x);
        acc.y = fmaf(acc.y, a, w * v.y);
        acc.z = fmaf(acc.z, a, w * v.z);
        acc.w = fmaf(acc.w, a, w * v.w);
        l = fmaf(l, a, w);
        m = mn;
    }
    s_acc[slot][c] = acc;
    if (c == 0) {
        s_m[slot] = m;
        s_l[slot] = l;
    }
    __syncthreads();

    if (threadIdx.x < DD) {
        const int d = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
            M = fmaxf(M, s_m[s]);
        float total = 0.f, o = 0.f;
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const float f = s_m[s] == -INFINITY ? 0.f : fast_exp2((s_m[s] - M) * kLog2e);
            total = fmaf(f, s_l[s], total);
            const float *a = reinterpret_cast<const float *>(&s_acc[s][d >> 2]);
            o = fmaf(f, a[d & 3], o);
        }
        out[d] = E::from_float(total > 0.f ? o / total : 0.f); // 0: the query sees no token
    }
}

template <typename T>
static cudaError_t launch_merge_t(cudaLaunchConfig_t &cfg, int dd, const MergeParams &p)
{
    switch (dd) {
    case 16: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 16>, p);
    case 32: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 32>, p);
    case 64: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 64>, p);
    default: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 128>, p);
    }
}

cudaError_t launch_merge(int dtype, const MergeParams &p, int num_seqs, int num_sms,
                         cudaStream_t stream)
{
    // A CTA owns at most 128 dims of head_dim; split further (down to 16
    // dims) while the grid has fewer than about two CTAs per SM -- a finer
    // split only adds CTAs of very little work.
    const long long pairs = (long long)p.num_heads * num_seqs * p.q_len;
    int dd = p.head_dim < 128 ? p.head_dim : 128;
    while (dd > 16 && pairs * (p.head_dim / dd) < 2LL * num_sms)
        dd /= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_heads, num_seqs * p.q_len, p.head_dim / dd);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // Programmatic dependent launch: this grid may be scheduled while the
    // attention grid before it drains; griddepcontrol.wait orders the reads.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == PA_BF16)
        return launch_merge_t<__nv_bfloat16>(cfg, dd, p);
    return launch_merge_t<__half>(cfg, dd, p);
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
