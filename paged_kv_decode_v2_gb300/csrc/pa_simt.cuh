// pa_simt.cuh -- the attention kernel of phase 1 (and of V1) on the CUDA
// cores alone: Q.K dot products and the softmax max / sum reduced with warp
// shuffles, P.V as scalar FMAs, no tensor-core instruction.
//
// It is the design the method's GQA decode suggests when the query group is
// small ("paged_attention_v2_pytorch.py" commit 15ef28e, "Key changes": one
// KV head broadcast over its G query heads): a G x 16 score tile is far from
// a dense MMA tile at G = 1..4.  It serves up to 8 query rows per KV head
// (NH = 1, 2, 4 or 8 after padding) and exists beside the mma.sync kernel
// (pa_attn.cuh) so the two can be timed and profiled on the same launch
// shapes; the library picks the mma.sync kernel unless told otherwise
// (pa_set_rows_kernel), because it measured faster at every G.
//
// Data movement is the mma.sync kernel's: each warp owns a ring of TMA
// stages, takes units j = warp, warp + W, ... of its CTA's range, and reads
// block ids one 32-unit chunk ahead.  Per 16-token tile of a unit:
//   Q.K   kTG lanes serve one token (kTP = 32 / kTG tokens per pass); a lane
//         holds kDQ dims of Q for the NH heads in registers (fp32) and reads
//         the same dims of K as 16-byte shared-memory loads; the NH partial
//         sums are reduce-scattered over the first log2(NH) lane bits of the
//         group and summed over the rest, so each lane ends with one
//         head's score for its token.
//   max   per head over the tile: local max over the lane's tokens, then a
//         shuffle max across the token groups; running {m, l} rescaled by
//         exp(m_old - m_new) ("paged_attn.py" commit 490ff98, the
//         summary_statistics paragraph).
//   P.V   p = exp(s - m) goes through a 16 x NH shared tile; each lane owns
//         D / 32 dims of O for the NH heads and adds p * V over the 16 tokens.
// At the end the warps' {m, l, o} are merged with the same rule and written
// as the partition's max_logits, exp_sums and normalised tmp_output
// ("paged_attention_v2_pytorch.py" commit 9cb7f9d, "Implementation",
// Phase 1), or as out for V1.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int NH>
struct SimtShape {
    static constexpr int kRaw = D * NH / 64;
    static constexpr int kTG = kRaw < 8 ? 8 : (kRaw > 32 ? 32 : kRaw); // lanes per token in Q.K
    static constexpr int kTP = 32 / kTG;                                 // tokens per pass
    static constexpr int kDQ = D / kTG;                                  // Q.K dims per lane
    static constexpr int kCQ = kDQ / 8;                                  // 16-byte chunks per lane
    static constexpr int kDL = D / 32;                                   // P.V dims per lane
    static constexpr int kPasses = 16 / kTP;                             // passes per 16-token tile
    static_assert(kCQ >= 1 && kCQ <= 4 && kDQ * NH <= 64, "Q registers per lane");
};

// Eight 16-bit values (one 16-byte chunk) to fp32.
template <typename T>
__device__ __forceinline__ void chunk_to_float(const uint4 &c, float (&f)[8])
{
    using E = Elem<T>;
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = E::lo(w[i]);
        f[2 * i + 1] = E::hi(w[i]);
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Bits [0, n) of x reversed (n <= 3).
__device__ __forceinline__ int bitrev(int x, int n)
{
    int r = 0;
    for (int i = 0; i < n; ++i)
        r |= ((x >> i) & 1) << (n - 1 - i);
    return r;
}

template <typename T, int D, int BS, int NH, bool V1>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    simt_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const AttnParams p)
{
    using E = Elem<T>;
    using SS = SimtShape<D, NH>;
    constexpr int kTG = SS::kTG, kTP = SS::kTP, kCQ = SS::kCQ, kDL = SS::kDL;
    constexpr int kPasses = SS::kPasses;
    constexpr int kLogNH = NH == 1 ? 0 : NH == 2 ? 1 : NH == 4 ? 2 : 3;
    constexpr int kSlices = D / 64;
    constexpr int kUB = BS < 16 ? 16 / BS : 1;        // blocks per unit
    constexpr int kUT = BS * kUB;                     // tokens per unit
    constexpr uint32_t kHalfBytes = kUT * 128;        // one 64-dim slice of a K or V unit
    constexpr uint32_t kStageBytes = 2 * kSlices * kHalfBytes;
    constexpr int kTiles = kUT / 16;
    constexpr int kHeads = 8;                         // scratch rows, as the mma.sync kernel's
    constexpr int kScr = D + 4;

    __shared__ uint64_t bars[kMaxWarps * kMaxStages];
    __shared__ __align__(16) float s_p[kMaxWarps][16 * NH + NH]; // p [token][head], alpha[head]
    __shared__ float s_factor[kMaxWarps][kMaxGroup];
    __shared__ float s_stat[3][kMaxGroup];
    extern __shared__ uint8_t dyn_smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int grp = lane / kTG;       // token group of Q.K
    const int j = lane % kTG;         // lane within the group
    // Head this lane's Q.K sum ends with (the reduce-scatter keeps the low
    // log2(NH) lane bits in reversed order).
    const int hmine = bitrev(j & (NH - 1), kLogNH);

    const int part = V1 ? 0 : (int)blockIdx.x;
    const int kv = blockIdx.y;
    const int b = blockIdx.z;

    if (threadIdx.x == 0)
        prefetch_tensormap(&tmap_k);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    const int head0 = kv * p.group;
    const int ncols = p.cols; // <= NH: one CTA serves every row of the KV head
    auto col_row = [&](int n) -> size_t {
        return ((size_t)b * p.q_len + n / p.group) * p.num_heads + head0 + n % p.group;
    };
    const int tokA = V1 ? 0 : part * p.partition_size;
    const int blk0 = tokA / BS;
    const int range_max =
        V1 ? p.max_blocks
           : (int)min(((long long)tokA + p.partition_size + BS - 1) / BS, (long long)p.max_blocks) -
                 blk0;
    const int32_t *bt_row = p.block_tables + (size_t)b * p.max_blocks + blk0;
    const int Lraw = __ldg(&p.seq_lens[b]);
    auto load_ids = [&](int chunk, int bound, int32_t(&dst)[kUB]) {
        const int u = warp + nwarps * (chunk * 32 + lane);
#pragma unroll
        for (int k = 0; k < kUB; ++k) {
            const int bi = u * kUB + k;
            dst[k] = bi < bound ? __ldg(bt_row + bi) : 0;
        }
    };
    int32_t ids_cur[kUB], ids_next[kUB];
    load_ids(0, range_max, ids_cur);
    load_ids(1, range_max, ids_next);

    // Q for this lane's Q.K dims, fp32: chunk step s of lane j covers chunk
    // cg(s) = j * kCQ + (s + j / (8 / kCQ)) % kCQ.  The rotation puts the 8
    // lanes of each quarter-warp on 8 different 16-byte bank groups.
    auto chunk_of = [&](int s) { return j * kCQ + (s + j / (8 / kCQ)) % kCQ; };
    float qreg[NH][kCQ][8];
    {
        // 4-byte loads: the query is only required to be 4-byte aligned.
        const uint32_t *q32 = static_cast<const uint32_t *>(p.query);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const bool has = h < ncols;
            const size_t row = col_row(has ? h : 0);
#pragma unroll
            for (int s = 0; s < kCQ; ++s) {
                const uint32_t *src = q32 + row * (D / 2) + chunk_of(s) * 4;
                uint4 c = make_uint4(0, 0, 0, 0);
                if (has)
                    c = make_uint4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
                chunk_to_float<T>(c, qreg[h][s]);
                // The scale and log2(e) are folded into Q: scores come out in exp2 units.
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    qreg[h][s][e] *= p.scale * kLog2e;
            }
        }
    }

    int L = Lraw;
    if (L < 0 || L > p.seq_len_cap) {
        if (threadIdx.x == 0 && part == 0 && kv == 0)
            set_status(p.status, PA_STATUS_BAD_SEQ_LEN);
        L = L < 0 ? 0 : p.seq_len_cap;
    }
    if (!V1 && tokA >= L)
        return;
    const int tok0 = blk0 * BS;
    const int lo = tokA - tok0;
    const int ntok = V1 ? L : (int)(min((long long)tokA + p.partition_size, (long long)L) - tok0);
    const int nblk = (ntok + BS - 1) / BS;
    const int nunit = (ntok + kUT - 1) / kUT;

    if (V1 && nblk == 0) {
        T *out = static_cast<T *>(p.out);
        for (int idx = threadIdx.x; idx < ncols * D; idx += blockDim.x)
            out[col_row(idx / D) * D + idx % D] = E::from_float(0.f);
        return;
    }

    // Visible positions of this lane's head column: rows r - lo < vis.
    unsigned vis;
    {
        const int last = (hmine < ncols ? L - p.q_len + hmine / p.group : L - 1) - tok0;
        vis = (unsigned)max(min(last + 1, ntok) - lo, 0);
    }

    const uint32_t smem0 = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    const uint32_t ring = smem0 + (uint32_t)warp * (uint32_t)p.stages * kStageBytes;
    const uint32_t bar0 = smem_addr(&bars[warp * kMaxStages]);
    const int stages = p.stages;
    const int cnt = warp < nunit ? (nunit - warp + nwarps - 1) / nwarps : 0;

    if (lane == 0) {
        for (int s = 0; s < stages; ++s)
            mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
        if (warp == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
    }
    __syncwarp();

    const uint64_t policy = l2_evict_first_policy();
    int32_t status_bits = 0;
    int chunk_cur = 0;

    auto issue = [&](int i, int s) {
        const int c = i >> 5;
        if (c != chunk_cur) {
#pragma unroll
            for (int k = 0; k < kUB; ++k)
                ids_cur[k] = ids_next[k];
            load_ids(c + 1, nblk, ids_next);
            chunk_cur = c;
        }
        const int u = warp + nwarps * i;
        const int nb = kUB == 1 ? 1 : min(kUB, nblk - u * kUB);
        const uint32_t bar = bar0 + 8 * s;
        const uint32_t dst = ring + (uint32_t)s * kStageBytes;
        if (lane == 0)
            mbar_arrive_expect_tx(bar, kUB == 1 ? kStageBytes : (uint32_t)nb * BS * 256u * kSlices);
#pragma unroll
        for (int k = 0; k < kUB; ++k) {
            int32_t phys = __shfl_sync(0xffffffffu, ids_cur[k], i & 31);
            if (k < nb) {
                if (phys < 0 || phys >= p.num_blocks) {
                    status_bits |= PA_STATUS_BAD_BLOCK_ID;
                    phys = 0;
                }
                if (lane == 0) {
                    const int row = (int)(((long long)phys * p.num_kv_heads + kv) * BS);
#pragma unroll
                    for (int sl = 0; sl < kSlices; ++sl)
                        tma_load_3d(dst + sl * kHalfBytes + k * BS * 128, &tmap_k, 0, sl, row, bar,
                                    policy);
#pragma unroll
                    for (int sl = 0; sl < kSlices; ++sl)
                        tma_load_3d(dst + (kSlices + sl) * kHalfBytes + k * BS * 128, &tmap_v, 0, sl,
                                    row, bar, policy);
                }
            }
        }
    };

    int issued = 0;
    for (; issued < cnt && issued < stages; ++issued)
        issue(issued, issued);

    // Running state: m (exp2 units) and this lane's share of l for head
    // hmine; O for the lane's P.V dims and every head.
    float m_run = -INFINITY, l_run = 0.f;
    float o[NH][kDL];
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int e = 0; e < kDL; ++e)
            o[h][e] = 0.f;

    float *pw = s_p[warp];
    // P.V dims of this lane: [lane * kDL, lane * kDL + kDL), in slice dsl,
    // 16-byte chunk dch of that slice, byte offset doff within the chunk.
    const int dsl = (lane * kDL) / 64;
    const int dch = ((lane * kDL) % 64) / 8;
    const int doff = ((lane * kDL) % 8) * 2;

    int i = 0;
    for (; i < cnt; ++i) {
        const int s = i % stages;
        const uint32_t parity = (uint32_t)(i / stages) & 1u;
        if (!mbar_wait_bounded(bar0 + 8 * s, parity, kWaitLimitNs)) {
            status_bits |= PA_STATUS_TIMEOUT;
            break;
        }
        const int jblk = warp + nwarps * i;
        const int valid = min(kUT, ntok - jblk * kUT);
        const uint32_t kbase = ring + (uint32_t)s * kStageBytes;
        const uint32_t vbase = kbase + kSlices * kHalfBytes;

        if (valid < kUT) {
            const int nchunks = (kUT - valid) * kSlices * 8;
            for (int c = lane; c < nchunks; c += 32) {
                const int r = valid + c / (kSlices * 8);
                const int sl = (c >> 3) % kSlices;
                st_shared_zero16(vbase + sl * kHalfBytes + r * 128 + (c & 7) * 16);
            }
            __syncwarp();
        }

#pragma unroll
        for (int tile = 0; tile < kTiles; ++tile) {
            if (tile * 16 >= valid)
                break;
            // ---- scores of the lane's tokens t = tile * 16 + pass * kTP + grp, head hmine
            float sc[kPasses];
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                const int t = tile * 16 + ps * kTP + grp;
                const uint32_t rbase = kbase + (uint32_t)t * 128;
                float acc[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    acc[h] = 0.f;
#pragma unroll
                for (int st = 0; st < kCQ; ++st) {
                    const int cg = chunk_of(st);
                    float kf[8];
                    chunk_to_float<T>(lds128(rbase + (cg >> 3) * kHalfBytes + (((cg & 7) ^ (t & 7)) << 4)),
                                      kf);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[h] = fmaf(qreg[h][st][e], kf[e], acc[h]);
                }
                // Reduce-scatter over lane bits 0 .. log2(NH) - 1 of the group:
                // lanes whose bit is 1 keep the upper half of the heads.
#pragma unroll
                for (int lv = 0; lv < kLogNH; ++lv) {
                    const int half = NH >> (lv + 1);
                    const bool up = (j >> lv) & 1;
#pragma unroll
                    for (int h = 0; h < half; ++h) {
                        const float keep = up ? acc[h + half] : acc[h];
                        const float send = up ? acc[h] : acc[h + half];
                        acc[h] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << lv);
                    }
                }
                // Then sum over the remaining lanes of the group.
#pragma unroll
                for (int off = NH; off < kTG; off <<= 1)
                    acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
                const unsigned r = (unsigned)(jblk * kUT + t - lo);
                sc[ps] = r < vis ? acc[0] : -INFINITY;
            }

            // ---- streaming softmax for head hmine over the tile's 16 tokens
            float mx = sc[0];
#pragma unroll
            for (int ps = 1; ps < kPasses; ++ps)
                mx = fmaxf(mx, sc[ps]);
#pragma unroll
            for (int off = kTG; off < 32; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float mn = fmaxf(m_run, mx);
            const bool live = mn != -INFINITY;
            const float alpha = live ? fast_exp2(m_run - mn) : 1.f;
            const float mb = live ? mn : 0.f;
            m_run = mn;
            float lsum = 0.f;
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                const float pv = fast_exp2(sc[ps] - mb);
                lsum += pv;
                if (j < NH)
                    pw[(ps * kTP + grp) * NH + hmine] = pv;
            }
            l_run = fmaf(l_run, alpha, lsum);
            if (lane < NH)
                pw[16 * NH + hmine] = alpha;
            __syncwarp();

            // ---- O += P V over the tile
            {
                float al[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    al[h] = pw[16 * NH + h];
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                    for (int e = 0; e < kDL; ++e)
                        o[h][e] *= al[h];
            }
#pragma unroll 4
            for (int t = 0; t < 16; ++t) {
                const int row = tile * 16 + t;
                const uint32_t va = vbase + dsl * kHalfBytes + (uint32_t)row * 128 +
                                    ((dch ^ (row & 7)) << 4) + doff;
                float vf[kDL];
                if constexpr (kDL == 2) {
                    const uint32_t w = lds32(va);
                    vf[0] = E::lo(w);
                    vf[1] = E::hi(w);
                } else if constexpr (kDL == 4) {
                    const uint2 w = lds64(va);
                    vf[0] = E::lo(w.x);
                    vf[1] = E::hi(w.x);
                    vf[2] = E::lo(w.y);
                    vf[3] = E::hi(w.y);
                } else {
                    float f8[8];
                    chunk_to_float<T>(lds128(va), f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        vf[e] = f8[e];
                }
                float pt[NH];
                if constexpr (NH >= 4) {
#pragma unroll
                    for (int h = 0; h < NH; h += 4) {
                        const float4 q4 = *reinterpret_cast<const float4 *>(pw + t * NH + h);
                        pt[h] = q4.x;
                        pt[h + 1] = q4.y;
                        pt[h + 2] = q4.z;
                        pt[h + 3] = q4.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        pt[h] = pw[t * NH + h];
                }
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                    for (int e = 0; e < kDL; ++e)
                        o[h][e] = fmaf(pt[h], vf[e], o[h][e]);
            }
            __syncwarp();
        }
        if (issued < cnt) {
            if (valid < kUT)
                fence_proxy_async();
            issue(issued, s);
            ++issued;
        }
    }

    if (status_bits & PA_STATUS_TIMEOUT) {
        for (int k = i; k < issued; ++k)
            mbar_wait_bounded(bar0 + 8 * (k % stages), (uint32_t)(k / stages) & 1u, kWaitLimitNs);
    }
    if (status_bits && lane == 0)
        set_status(p.status, status_bits);

    // ---- hand the warp's {m, l, o} to the CTA merge (scratch = this warp's ring).
    // m is in exp2 units here; the merge and the outputs use natural-log units.
#pragma unroll
    for (int off = kTG; off < 32; off <<= 1)
        l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
    float *scr = reinterpret_cast<float *>(dyn_smem + (ring - smem_addr(dyn_smem)));
    float *scr_m = scr;
    float *scr_l = scr + kHeads;
    float *scr_o = scr + 2 * kHeads;
    __syncwarp();
    if (lane < NH) {
        scr_m[hmine] = m_run == -INFINITY ? -INFINITY : m_run * (1.f / kLog2e);
        scr_l[hmine] = l_run;
    }
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int e = 0; e < kDL; ++e)
            scr_o[h * kScr + lane * kDL + e] = o[h][e];
    __syncthreads();

    const uint32_t warp_stride = (uint32_t)stages * kStageBytes / 4;
    const float *scr0 = reinterpret_cast<const float *>(dyn_smem + (smem0 - smem_addr(dyn_smem)));
    if (threadIdx.x < ncols) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < nwarps; ++w)
            M = fmaxf(M, scr0[w * warp_stride + h]);
        float lsum = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            const float mw = scr0[w * warp_stride + h];
            const float f = mw == -INFINITY ? 0.f : fast_exp2((mw - M) * kLog2e);
            s_factor[w][h] = f;
            lsum = fmaf(f, scr0[w * warp_stride + kHeads + h], lsum);
        }
        s_stat[0][h] = M;
        s_stat[1][h] = lsum;
        s_stat[2][h] = lsum > 0.f ? 1.f / lsum : 0.f;
    }
    __syncthreads();

    constexpr int kQuads = D / 4;
    for (int idx = threadIdx.x; idx < ncols * kQuads; idx += blockDim.x) {
        const int h = idx / kQuads;
        const int d = (idx % kQuads) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < nwarps; ++w) {
            const float f = s_factor[w][h];
            const float4 v =
                *reinterpret_cast<const float4 *>(scr0 + w * warp_stride + 2 * kHeads + h * kScr + d);
            acc.x = fmaf(f, v.x, acc.x);
            acc.y = fmaf(f, v.y, acc.y);
            acc.z = fmaf(f, v.z, acc.z);
            acc.w = fmaf(f, v.w, acc.w);
        }
        const float inv = s_stat[2][h];
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const size_t bh = col_row(h);
        if (V1) {
            T *o4 = static_cast<T *>(p.out) + bh * D + d;
            o4[0] = E::from_float(acc.x);
            o4[1] = E::from_float(acc.y);
            o4[2] = E::from_float(acc.z);
            o4[3] = E::from_float(acc.w);
        } else {
            const size_t slot = bh * p.max_num_partitions + part;
            *reinterpret_cast<float4 *>(p.tmp_output + slot * D + d) = acc;
            if (d == 0) {
                p.exp_sums[slot] = s_stat[1][h];
                p.max_logits[slot] = s_stat[0][h];
            }
        }
    }
}

// Kernel dispatch on block size, padded rows NH and V1/V2, for one head_dim.
template <typename T, int D>
static const void *simt_kernel_ptr(int block_size, int cols, int v1)
{
    if (v1 == 2) // no fused variant of this kernel
        return nullptr;
    const int nh = cols <= 1 ? 1 : cols <= 2 ? 2 : cols <= 4 ? 4 : 8;
#define PA_SIMT_NH(BS, NH)                                                                        \
    if (nh == NH)                                                                                 \
        return v1 == 1 ? reinterpret_cast<const void *>(&simt_attn_kernel<T, D, BS, NH, true>)         \
                       : reinterpret_cast<const void *>(&simt_attn_kernel<T, D, BS, NH, false>);
#define PA_SIMT_BS(BS)                                                                            \
    if (block_size == BS) {                                                                       \
        PA_SIMT_NH(BS, 1)                                                                         \
        PA_SIMT_NH(BS, 2)                                                                         \
        PA_SIMT_NH(BS, 4)                                                                         \
        PA_SIMT_NH(BS, 8)                                                                         \
    }
    PA_SIMT_BS(8)
    PA_SIMT_BS(16)
    PA_SIMT_BS(32)
    PA_SIMT_BS(64)
#undef PA_SIMT_BS
#undef PA_SIMT_NH
    return nullptr;
}

template <typename T, int D>
static cudaError_t simt_prepare(int block_size, int cols, int v1, int optin_bytes, size_t *limit)
{
    const void *fn = simt_kernel_ptr<T, D>(block_size, cols, v1);
    if (!fn)
        return cudaErrorInvalidValue;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess)
        return e;
    if ((size_t)optin_bytes <= fa.sharedSizeBytes)
        return cudaErrorInvalidValue;
    *limit = (size_t)optin_bytes - fa.sharedSizeBytes;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)*limit);
}

template <typename T, int D>
static int simt_occupancy(int block_size, int cols, int v1, int warps, size_t smem_bytes)
{
    const void *fn = simt_kernel_ptr<T, D>(block_size, cols, v1);
    int n = 0;
    if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, warps * 32, smem_bytes) !=
                   cudaSuccess)
        return 0;
    return n;
}

template <typename T, int D>
static cudaError_t simt_launch(const AttnLaunch &L, cudaStream_t stream)
{
    const void *fn = simt_kernel_ptr<T, D>(L.block_size, L.cta_cols, attn_variant(L));
    if (!fn)
        return cudaErrorInvalidValue;
    void *args[] = {const_cast<CUtensorMap *>(&L.tmap_k), const_cast<CUtensorMap *>(&L.tmap_v),
                    const_cast<AttnParams *>(&L.p)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = dim3(L.warps * 32);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

#define PA_DEFINE_SIMT_OPS(T, NAME, D)                                                            \
    const AttnOps *NAME()                                                                         \
    {                                                                                             \
        static const AttnOps ops = {&simt_prepare<T, D>, &simt_occupancy<T, D>,                   \
                                    &simt_launch<T, D>};                                          \
        return &ops;                                                                              \
    }

} // namespace pa
