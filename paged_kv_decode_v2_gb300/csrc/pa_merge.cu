// pa_merge.cu -- phase 2 of split-K decode: the cross-partition
// log-sum-exp merge ("paged_attention_v2_pytorch.py" commit 9cb7f9d,
// "Implementation", Phase 2):
//     global_max = max_p max_logits[p]
//     rescale_p  = exp(max_logits[p] - global_max) * exp_sums[p]
//     out        = sum_p (rescale_p / sum_q rescale_q) * tmp_output[p]
// and the self-test kernel of the bounded wait.
//
// Two forms.  The slice form: one CTA per (query head, sequence, slice of
// head_dim); the slice is at most 128 dims, and smaller (down to 16) when
// there are few (seq, head) pairs.  A group of lanes owns one partition at a
// time and reads the slice as float4s (contiguous bytes); the groups of a
// CTA take partitions round robin, and their running states meet by warp
// shuffles and then in shared memory.  The row form: one warp per (row,
// head), its lanes spanning head_dim, walking the partitions in order --
// for calls with few partitions and many (row, head) pairs, where a CTA per
// pair would leave most of its threads idle and the grid's size, not the
// bytes, would set the time.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Folds the running state (mo, lo, ao) into (m, l, a): the same
// exp(m_old - M) rule as the partitions' own merge; a state with m = -inf
// (no partition seen) adds nothing.
__device__ __forceinline__ void merge_state(float &m, float &l, float4 &a, float mo, float lo,
                                            float4 ao)
{
    const float M = fmaxf(m, mo);
    const float f = m == -INFINITY ? 0.f : fast_exp2((m - M) * kLog2e);
    const float g = mo == -INFINITY ? 0.f : fast_exp2((mo - M) * kLog2e);
    l = fmaf(l, f, lo * g);
    a.x = fmaf(a.x, f, ao.x * g);
    a.y = fmaf(a.y, f, ao.y * g);
    a.z = fmaf(a.z, f, ao.z * g);
    a.w = fmaf(a.w, f, ao.w * g);
    m = M;
}

template <typename T, int DD, int NTH>
__global__ void __launch_bounds__(NTH) merge_kernel(const MergeParams p)
{
    using E = Elem<T>;
    constexpr int kGroup = DD / 4;         // lanes per partition (one float4 each)
    constexpr int kSlots = NTH / kGroup;   // partitions in flight per CTA
    constexpr int kWarps = NTH / 32;
    __shared__ float s_m[kWarps][kGroup];
    __shared__ float s_l[kWarps][kGroup];
    __shared__ float4 s_acc[kWarps][kGroup];

    const int h = blockIdx.x;
    const int row = blockIdx.y;       // (sequence, new token) = b * q_len + i
    const int b = row / p.q_len;
    const int D = p.head_dim;
    const int d0 = blockIdx.z * DD;
    const int slot = threadIdx.x / kGroup; // partitions slot, slot + kSlots, ...
    const int c = threadIdx.x % kGroup;    // float4 column within the CTA's dims
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

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
    // The slots of one warp (lanes with the same column c) meet by shuffles,
    // then the warps meet in shared memory.
#pragma unroll
    for (int off = kGroup; off < 32; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float lo = __shfl_xor_sync(0xffffffffu, l, off);
        float4 ao;
        ao.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
        ao.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
        ao.z = __shfl_xor_sync(0xffffffffu, acc.z, off);
        ao.w = __shfl_xor_sync(0xffffffffu, acc.w, off);
        merge_state(m, l, acc, mo, lo, ao);
    }
    if (lane < kGroup) {
        s_m[warp][c] = m;
        s_l[warp][c] = l;
        s_acc[warp][c] = acc;
    }
    __syncthreads();

    if (threadIdx.x < kGroup) {
        float M = s_m[0][c], tot = s_l[0][c];
        float4 o = s_acc[0][c];
#pragma unroll
        for (int w = 1; w < kWarps; ++w)
            merge_state(M, tot, o, s_m[w][c], s_l[w][c], s_acc[w][c]);
        const float inv = tot > 0.f ? 1.f / tot : 0.f; // 0: the query sees no token
        T *o4 = out + 4 * c;
        o4[0] = E::from_float(o.x * inv);
        o4[1] = E::from_float(o.y * inv);
        o4[2] = E::from_float(o.z * inv);
        o4[3] = E::from_float(o.w * inv);
    }
}

// The row form: warp w of CTA x merges pair x * kRowWarps + w, i.e. (row,
// head) with row = pair / num_heads; lane l owns dims [l * DL, l * DL + DL).
// The partitions are folded in index order with the same running-maximum
// rule as the slice form.
template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) merge_rows_kernel(const MergeParams p, int pairs)
{
    using E = Elem<T>;
    constexpr int DL = D / 32;            // 2, 4 or 8 floats per lane
    constexpr int kRowWarps = kMergeThreads / 32;
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x * kRowWarps + (threadIdx.x >> 5);

    asm volatile("griddepcontrol.launch_dependents;");
    if (pair >= pairs)
        return;
    const int row = pair / p.num_heads;   // (sequence, new token) = b * q_len + i
    const int b = row / p.q_len;
    int L = __ldg(&p.seq_lens[b]);
    L = L < 0 ? 0 : (L > p.seq_len_cap ? p.seq_len_cap : L);
    const int np = (L + p.partition_size - 1) / p.partition_size;
    T *out = static_cast<T *>(p.out) + (size_t)pair * D + lane * DL;
    if (np == 0) {
#pragma unroll
        for (int j = 0; j < DL; ++j)
            out[j] = E::from_float(0.f);
        return;
    }
    const float *ml = p.max_logits + (size_t)pair * p.max_num_partitions;
    const float *es = p.exp_sums + (size_t)pair * p.max_num_partitions;
    const float *tmp = p.tmp_output + (size_t)pair * p.max_num_partitions * D + lane * DL;

    asm volatile("griddepcontrol.wait;" ::: "memory");

    float m = -INFINITY, l = 0.f;
    float acc[DL];
#pragma unroll
    for (int j = 0; j < DL; ++j)
        acc[j] = 0.f;
#pragma unroll 4
    for (int i = 0; i < np; ++i) {
        const float mp = __ldg(ml + i);
        const float lp = __ldg(es + i);
        float v[DL];
        if constexpr (DL == 2) {
            const float2 t = __ldg(reinterpret_cast<const float2 *>(tmp + (size_t)i * D));
            v[0] = t.x;
            v[1] = t.y;
        } else {
#pragma unroll
            for (int q = 0; q < DL / 4; ++q) {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(tmp + (size_t)i * D) + q);
                v[4 * q] = t.x;
                v[4 * q + 1] = t.y;
                v[4 * q + 2] = t.z;
                v[4 * q + 3] = t.w;
            }
        }
        if (lp == 0.f) // a partition none of whose tokens this query sees
            continue;
        const float mn = fmaxf(m, mp);
        const float a = fast_exp2((m - mn) * kLog2e); // 0 while m is -inf
        const float w = fast_exp2((mp - mn) * kLog2e) * lp;
#pragma unroll
        for (int j = 0; j < DL; ++j)
            acc[j] = fmaf(acc[j], a, w * v[j]);
        l = fmaf(l, a, w);
        m = mn;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f; // 0: the query sees no token
#pragma unroll
    for (int j = 0; j < DL; ++j)
        out[j] = E::from_float(acc[j] * inv);
}

template <typename T>
static cudaError_t launch_rows_t(cudaLaunchConfig_t &cfg, int head_dim, const MergeParams &p,
                                 int pairs)
{
    switch (head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, merge_rows_kernel<T, 64>, p, pairs);
    case 256: return cudaLaunchKernelEx(&cfg, merge_rows_kernel<T, 256>, p, pairs);
    default: return cudaLaunchKernelEx(&cfg, merge_rows_kernel<T, 128>, p, pairs);
    }
}

template <typename T>
static cudaError_t launch_merge_t(cudaLaunchConfig_t &cfg, int dd, const MergeParams &p)
{
    switch (dd) {
    case 16: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 16, kMergeThreads>, p);
    case 32: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 32, kMergeThreads>, p);
    case 64: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 64, kMergeThreads>, p);
    default: return cudaLaunchKernelEx(&cfg, merge_kernel<T, 128, kMergeThreads>, p);
    }
}

int merge_form(const MergeParams &p, int num_seqs, int num_sms, int forced)
{
    // The row form's grid counts pairs / 4 CTAs in one dimension: up to 2^30
    // pairs.
    const long long pairs = (long long)p.num_heads * num_seqs * p.q_len;
    if (forced == 1 || (forced == 2 && pairs <= (1LL << 30)))
        return forced;
    // Row form when the slice form would launch more than 16 CTAs per SM and
    // every sequence has at most 8 partitions, or, from 32 pairs per SM, at
    // most 32: the slice form's CTA per pair leaves most of its lanes idle
    // when a batch's pairs have few partitions each, and the row form's warps
    // take a long pair's partitions one after another.  Measured on GB300 (us
    // per call, slice / row form): ragged batch (64 sequences, lognormal
    // lengths to 32K) with 2, 4, 8, 16 new tokens 144.8 / 140.4, 197.7 /
    // 187.3, 220.3 / 196.4, 285.3 / 237.4 (16 to 32 partitions, 8K to 64K
    // pairs); the same batch with one new token 142.5 / 143.6 (64 partitions,
    // 4K pairs); one 100K-token sequence 37.1 / 69.7; stress at 2 sequences
    // 159.5 / 179.0.
    const int np_max = (p.seq_len_cap + p.partition_size - 1) / p.partition_size;
    const bool many = pairs > 16LL * num_sms && pairs <= (1LL << 30);
    return many && (np_max <= 8 || (np_max <= 32 && pairs >= 32LL * num_sms)) ? 2 : 1;
}

cudaError_t launch_merge(int dtype, const MergeParams &p, int num_seqs, int num_sms, int form,
                         cudaStream_t stream)
{
    // A CTA owns at most 128 dims of head_dim (dd); split further, down to 16
    // dims, (a) while the grid has fewer than about two CTAs per SM, or (b)
    // while the longest sequence has more partitions than one unrolled round
    // of 4 per slot covers (slots = 128 threads / (dd / 4) lanes) and the
    // grid stays within 16 CTAs per SM.  The CTA stays at 128 threads, so
    // that these CTAs fit beside the attention kernel's (their registers come
    // from what that kernel leaves free) and wait, already resident, for it
    // to finish.  Measured on GB300 (us the merge adds to a call, same box):
    // 8 x 131072 tokens at 1024 per partition (128 partitions): 7.3-8.5 at
    // 128 dims per CTA; 256- and 512-thread CTAs cost the 100K-token and
    // ragged batches 1.3 and 2.5 us instead, from not fitting beside the
    // attention kernel.
    const long long pairs = (long long)p.num_heads * num_seqs * p.q_len;
    const int np_max = (p.seq_len_cap + p.partition_size - 1) / p.partition_size;
    int dd = p.head_dim < 128 ? p.head_dim : 128;
    while (dd > 16) {
        const long long ctas = pairs * (p.head_dim / dd);
        const int slots = kMergeThreads / (dd / 4);
        if (ctas < 2LL * num_sms || (np_max > 4 * slots && 2 * ctas <= 16LL * num_sms))
            dd /= 2;
        else
            break;
    }
    const long long pairs_all = (long long)p.num_heads * num_seqs * p.q_len;
    const bool rows = merge_form(p, num_seqs, num_sms, form) == 2;
    cudaLaunchConfig_t cfg = {};
    if (rows)
        cfg.gridDim = dim3((unsigned)((pairs_all + kMergeThreads / 32 - 1) / (kMergeThreads / 32)));
    else
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
    if (rows) {
        if (dtype == PA_BF16)
            return launch_rows_t<__nv_bfloat16>(cfg, p.head_dim, p, (int)pairs_all);
        return launch_rows_t<__half>(cfg, p.head_dim, p, (int)pairs_all);
    }
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
