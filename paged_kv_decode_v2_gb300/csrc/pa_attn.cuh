// pa_attn.cuh -- the attention kernel: phase 1 of split-K decode ("V2") and
// the single-pass form ("V1").
//
// One CTA owns one (partition p, KV head k, sequence b) -- for V1 the
// "partition" is the whole sequence.  It serves the whole GQA group of G
// query heads that share KV head k, so every K/V byte is read from HBM once
// per call ("paged_attention_v2_pytorch.py" commit 15ef28e, "Key changes":
// GQA by broadcasting the KV head instead of replicating it).
//
// Data movement.  Each warp of the CTA owns a private ring of `stages`
// shared-memory stages and walks the units j = warp, warp + W, ... of the
// CTA's range; a unit is one paged block, or two for 8-token blocks so that
// a unit fills a 16-row MMA tile.  A stage holds a unit's K tile and V tile
// (tokens x head_dim each), brought in by TMA tensor loads (one per block
// and 64-dim slice of K and of V) that complete on the stage's mbarrier.
// Block ids are read from the block table a full chunk of 32 units ahead of
// use.  Loads use 128-byte swizzling, so the ldmatrix reads below touch 32
// distinct banks.
//
// Math (fp32 accumulation on the tensor cores, mma.sync m16n8k16).  Tokens
// are the M dimension and query heads the N dimension (8 per n-tile), so a
// GQA group of 8 fills an n-tile exactly:
//     S^T[16 tokens x 8 heads]  = K_tile[16 x D] . Q^T[D x 8]   (D/16 MMAs)
//     O^T[D x 8 heads]         += V_tile^T[D x 16] . P^T[16 x 8] (D/16 MMAs)
// Q^T lives in registers for the whole CTA.  The S^T accumulator fragment is
// turned into the P^T operand fragment with two movmatrix transposes.  The
// softmax is the streaming {m, l, o} accumulator with the merge factor
// exp(m_old - m_new) ("paged_attn.py" commit 490ff98, the
// summary_statistics paragraph), kept per warp and merged across warps at
// the end with the same rule.
//
// Output.  V2 writes, per query head of the group, the partition's
//     max_logits = m_p,  exp_sums = l_p = sum exp(s - m_p),
//     tmp_output = sum exp(s - m_p) V / l_p
// ("paged_attention_v2_pytorch.py" commit 9cb7f9d, "Implementation",
// Phase 1).  V1 writes out = o / l rounded to the storage type.
//
// FUSED (V2 only) adds phase 2 to the same grid: after writing its
// partials, each CTA takes a ticket from a per-(sequence, KV head) counter,
// and the CTA that takes the last one merges that group's partitions into
// out -- the single-kernel alternative to the separate reduction pass that
// "paged_attn.py" commit 490ff98 sets against CCCL's two-pass dispatch.
// The merging CTA reads the partitions in index order, so the result does
// not depend on which CTA finishes last.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Phase-1 CTAs that serve 16 query rows (NT = 2) of up to 128 dims run at
// most 4 warps, so that three CTAs fit an SM (<= 170 registers, no spills);
// every other kernel runs up to 8 warps.
template <int D, int NT, bool V1>
struct AttnBounds {
    static constexpr bool kNarrow = NT == 2 && !V1 && D <= 128;
    static constexpr int kThreads = kNarrow ? 128 : kMaxWarps * 32;
    static constexpr int kMinBlocks = kNarrow ? 3 : 1;
};

template <typename T, int D, int BS, int NT, bool V1, bool FUSED = false>
__global__ void __launch_bounds__(AttnBounds<D, NT, V1>::kThreads,
                                  AttnBounds<D, NT, V1>::kMinBlocks)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p)
{
    using E = Elem<T>;
    constexpr int kKS = D / 16;                       // 16-dim steps of Q.K, 16-dim tiles of O
    constexpr int kSlices = D / 64;                   // 64-dim slices: one TMA load each
    // A ring stage holds one "unit" of kUB blocks, at least the 16 tokens of an MMA tile.
    constexpr int kUB = BS < 16 ? 16 / BS : 1;        // blocks per unit
    constexpr int kUT = BS * kUB;                     // tokens per unit
    constexpr uint32_t kHalfBytes = kUT * 128;        // one 64-dim slice of a K or V unit
    constexpr uint32_t kStageBytes = 2 * kSlices * kHalfBytes; // K slices, then V slices
    constexpr int kTiles = kUT / 16;                  // 16-row MMA tiles per unit
    constexpr int kHeads = NT * 8;
    constexpr int kScr = D + 4;                       // scratch row stride (floats)

    __shared__ uint64_t bars[kMaxWarps * kMaxStages];
    __shared__ float s_factor[kMaxWarps][kMaxGroup];
    __shared__ float s_stat[3][kMaxGroup]; // merged max, merged sum, 1 / sum (0 when empty)
    extern __shared__ uint8_t dyn_smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int g4 = lane >> 2; // row group of the mma fragments
    const int t4 = lane & 3;  // thread within the group

    // blockIdx.x = partition * col_groups + column group (V1: the column group).
    const int cgi = V1 ? (int)blockIdx.x : (int)blockIdx.x % p.col_groups;
    const int part = V1 ? 0 : (int)blockIdx.x / p.col_groups;
    const int kv = blockIdx.y;
    const int b = blockIdx.z;

    // This grid is launched with programmatic stream serialisation, so its
    // CTAs may become resident while the kernel before it in the stream is
    // still running.  Nothing global is read or written before this wait,
    // which returns once that kernel has completed and its writes are
    // visible.  Then the grid after this one (the merge) may be scheduled
    // early; it waits the same way before reading what this grid writes.
    if (threadIdx.x == 0)
        prefetch_tensormap(&tmap_k);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    // ---- loads that do not depend on the sequence length, issued together:
    // the length, the first two chunks of block ids and the Q fragments.
    const int head0 = kv * p.group;
    // Columns of this CTA: query rows (new token i, head head0 + g) for the
    // global column c = col0 + n = i * group + g, n < ncols.
    const int col0 = cgi * kHeads;
    const int ncols = min(kHeads, p.cols - col0);
    auto col_row = [&](int n) -> size_t { // row of [S * q_len * H] for local column n
        const int c = col0 + n;
        return ((size_t)b * p.q_len + c / p.group) * p.num_heads + head0 + c % p.group;
    };
    // V2: partition `part` holds tokens [tokA, tokA + partition_size), which
    // may begin and end inside a block; blocks from blk0 cover it.
    const int tokA = V1 ? 0 : part * p.partition_size;
    const int blk0 = tokA / BS;
    const int range_max =
        V1 ? p.max_blocks
           : (int)min(((long long)tokA + p.partition_size + BS - 1) / BS, (long long)p.max_blocks) -
                 blk0;
    const int32_t *bt_row = p.block_tables + (size_t)b * p.max_blocks + blk0;
    const int Lraw = __ldg(&p.seq_lens[b]);
    // Block ids of the warp's units (unit u = warp + nwarps * i) for i in a
    // 32-unit chunk, one unit per lane; blocks at or past `bound` read as 0.
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

    // Q^T fragments (B operand of S^T = K Q^T): head 8j + g4, dims 16ks + 2t4 (+1, +8, +9)
    uint32_t qf[NT][kKS][2];
    {
        const uint32_t *q32 = static_cast<const uint32_t *>(p.query);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int n = j * 8 + g4;
            const bool has = n < ncols;
            const size_t rowbase = col_row(has ? n : 0) * (D / 2);
#pragma unroll
            for (int ks = 0; ks < kKS; ++ks) {
                qf[j][ks][0] = has ? __ldg(q32 + rowbase + ks * 8 + t4) : 0u;
                qf[j][ks][1] = has ? __ldg(q32 + rowbase + ks * 8 + 4 + t4) : 0u;
            }
        }
    }

    // ---- sequence range owned by this CTA
    int L = Lraw;
    if (L < 0 || L > p.seq_len_cap) {
        if (threadIdx.x == 0 && part == 0 && kv == 0)
            set_status(p.status, PA_STATUS_BAD_SEQ_LEN);
        L = L < 0 ? 0 : p.seq_len_cap;
    }
    if (!V1 && tokA >= L) {
        // Partition past the end of this sequence: nothing to write -- except
        // in the fused form for an empty sequence, whose zero output row no
        // merge would write: partition 0's CTAs write it.
        if (FUSED && part == 0 && L == 0) {
            T *out = static_cast<T *>(p.out);
            for (int idx = threadIdx.x; idx < ncols * D; idx += blockDim.x)
                out[col_row(idx / D) * D + idx % D] = E::from_float(0.f);
        }
        return;
    }
    // Token positions below are counted from tok0, the first token of block blk0;
    // the range is [lo, ntok) of them.
    const int tok0 = blk0 * BS;
    const int lo = tokA - tok0;
    const int ntok = V1 ? L : (int)(min((long long)tokA + p.partition_size, (long long)L) - tok0);
    const int nblk = (ntok + BS - 1) / BS;   // blocks of the range
    const int nunit = (ntok + kUT - 1) / kUT; // ring stages' worth

    if (V1 && nblk == 0) { // empty sequence: zero output
        T *out = static_cast<T *>(p.out);
        for (int idx = threadIdx.x; idx < ncols * D; idx += blockDim.x)
            out[col_row(idx / D) * D + idx % D] = E::from_float(0.f);
        return;
    }

    // Visible tokens of this lane's columns 8j + 2t4 (+1): position t - tok0 = lo + r
    // with r < vis: new token i sees positions <= L - q_len + i, and none
    // outside the range [tokA, tok0 + ntok) (a straddling block also holds
    // tokens of the neighbouring partitions).  Padding columns (past ncols)
    // keep the whole range and are never stored.
    unsigned vis[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int n = j * 8 + 2 * t4 + k;
            const int last = (n < ncols ? L - p.q_len + (col0 + n) / p.group : L - 1) - tok0;
            vis[j][k] = (unsigned)max(min(last + 1, ntok) - lo, 0);
        }

    const uint32_t smem0 = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    const uint32_t ring = smem0 + (uint32_t)warp * (uint32_t)p.stages * kStageBytes;
    const uint32_t bar0 = smem_addr(&bars[warp * kMaxStages]);
    const int stages = p.stages;

    // Units of this warp: u = warp + nwarps * i, i < cnt.
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

    // Issue the TMA loads of the warp's i-th unit into stage s (warp-uniform call).
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
        const int nb = kUB == 1 ? 1 : min(kUB, nblk - u * kUB); // blocks in the unit
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
                    phys = 0; // read a valid block instead of memory outside the cache
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

    // Running softmax state of this lane's heads 8j + 2t4 (+1): natural-log units.
    float m_run[NT][2], l_run[NT][2];
    float o[NT][kKS][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        m_run[j][0] = m_run[j][1] = -INFINITY;
        l_run[j][0] = l_run[j][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt)
            o[j][mt][0] = o[j][mt][1] = o[j][mt][2] = o[j][mt][3] = 0.f;
    }

    // Per-lane ldmatrix row offsets.  ldmatrix lane L addresses row (L & 7) of 8x8 matrix L >> 3.
    const int mrow = lane & 7;
    const int mq = lane >> 3;
    // K (non-transposed A operand): matrix q covers rows (q & 1) * 8 .., dims (q >> 1) * 8 ..
    const int k_row = (mq & 1) * 8 + mrow;
    const int k_chunk_hi = mq >> 1;
    // V (transposed A operand): matrix q covers dims (q & 1) * 8 .., tokens (q >> 1) * 8 ..
    const int v_row = (mq >> 1) * 8 + mrow;
    const int v_chunk_lo = mq & 1;

    const float scale = p.scale;
    int i = 0;
    for (; i < cnt; ++i) {
        const int s = i % stages;
        const uint32_t parity = (uint32_t)(i / stages) & 1u;
        if (!mbar_wait_bounded(bar0 + 8 * s, parity, kWaitLimitNs)) {
            status_bits |= PA_STATUS_TIMEOUT;
            break;
        }
        const int jblk = warp + nwarps * i; // unit
        const int valid = min(kUT, ntok - jblk * kUT);
        const uint32_t kbase = ring + (uint32_t)s * kStageBytes;
        const uint32_t vbase = kbase + kSlices * kHalfBytes;

        if (valid < kUT) {
            // Rows past the end of the range (or of the unit's loaded blocks):
            // zero V so no stale value reaches P.V.  A row is kSlices lines of
            // eight 16-byte chunks.
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
            // ---- S^T = K_tile Q^T
            uint32_t ka[kKS][4];
            {
                const int r = tile * 16 + k_row;
                const uint32_t rbase = kbase + r * 128;
#pragma unroll
                for (int ks = 0; ks < kKS; ++ks) {
                    const int chunk = ((ks & 3) << 1) | k_chunk_hi;
                    ldsm_x4(rbase + (ks >> 2) * kHalfBytes + ((chunk ^ mrow) << 4), ka[ks]);
                }
            }
            float sacc[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float e[4] = {0.f, 0.f, 0.f, 0.f};
                float f[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < kKS; ks += 2) {
                    E::mma(e, ka[ks], qf[j][ks][0], qf[j][ks][1]);
                    E::mma(f, ka[ks + 1], qf[j][ks + 1][0], qf[j][ks + 1][1]);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sacc[j][c] = e[c] + f[c];
            }

            // ---- scale, mask, streaming softmax update
            // token rows of c0/c1 and (r0 + 8) of c2/c3, from tok0 + lo (an
            // unsigned compare with vis also masks the rows before lo)
            const unsigned r0 = (unsigned)(jblk * kUT + tile * 16 + g4 - lo);
            uint32_t pb[NT][2][2]; // [n-tile][hi/lo][b0/b1]
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float sv[4];
                sv[0] = r0 < vis[j][0] ? sacc[j][0] * scale : -INFINITY;
                sv[1] = r0 < vis[j][1] ? sacc[j][1] * scale : -INFINITY;
                sv[2] = r0 + 8u < vis[j][0] ? sacc[j][2] * scale : -INFINITY;
                sv[3] = r0 + 8u < vis[j][1] ? sacc[j][3] * scale : -INFINITY;
                float mx0 = fmaxf(sv[0], sv[2]);
                float mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[j][0], mx0);
                const float mn1 = fmaxf(m_run[j][1], mx1);
                // A column with no visible token yet (max still -inf) keeps l = o = 0.
                const bool live0 = mn0 != -INFINITY, live1 = mn1 != -INFINITY;
                const float a0 = live0 ? fast_exp2((m_run[j][0] - mn0) * kLog2e) : 1.f;
                const float a1 = live1 ? fast_exp2((m_run[j][1] - mn1) * kLog2e) : 1.f;
                m_run[j][0] = mn0;
                m_run[j][1] = mn1;
                const float mb0 = live0 ? mn0 * kLog2e : 0.f, mb1 = live1 ? mn1 * kLog2e : 0.f;
                float pv[4];
                pv[0] = fast_exp2(fmaf(sv[0], kLog2e, -mb0));
                pv[1] = fast_exp2(fmaf(sv[1], kLog2e, -mb1));
                pv[2] = fast_exp2(fmaf(sv[2], kLog2e, -mb0));
                pv[3] = fast_exp2(fmaf(sv[3], kLog2e, -mb1));
                l_run[j][0] = fmaf(l_run[j][0], a0, pv[0] + pv[2]);
                l_run[j][1] = fmaf(l_run[j][1], a1, pv[1] + pv[3]);
#pragma unroll
                for (int mt = 0; mt < kKS; ++mt) {
                    o[j][mt][0] *= a0;
                    o[j][mt][1] *= a1;
                    o[j][mt][2] *= a0;
                    o[j][mt][3] *= a1;
                }
                // P^T fragments: pack (token row, head pair) and transpose to (token pair, head).
                const uint32_t h01 = E::pack(pv[0], pv[1]);
                const uint32_t h23 = E::pack(pv[2], pv[3]);
                pb[j][0][0] = movmatrix_trans(h01);
                pb[j][0][1] = movmatrix_trans(h23);
                if (E::kSplitP) {
                    const uint32_t l01 = E::pack(pv[0] - E::lo(h01), pv[1] - E::hi(h01));
                    const uint32_t l23 = E::pack(pv[2] - E::lo(h23), pv[3] - E::hi(h23));
                    pb[j][1][0] = movmatrix_trans(l01);
                    pb[j][1][1] = movmatrix_trans(l23);
                }
            }

            // ---- O^T += V_tile^T P^T
            {
                const int r = tile * 16 + v_row;
                const uint32_t rbase = vbase + r * 128;
#pragma unroll
                for (int mt = 0; mt < kKS; ++mt) {
                    uint32_t va[4];
                    const int chunk = ((mt & 3) << 1) | v_chunk_lo;
                    ldsm_x4_trans(rbase + (mt >> 2) * kHalfBytes + ((chunk ^ mrow) << 4), va);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        E::mma(o[j][mt], va, pb[j][0][0], pb[j][0][1]);
                        if (E::kSplitP)
                            E::mma(o[j][mt], va, pb[j][1][0], pb[j][1][1]);
                    }
                }
            }
        }
        __syncwarp();
        if (issued < cnt) {
            if (valid < kUT)
                fence_proxy_async();
            issue(issued, s);
            ++issued;
        }
    }

    if (status_bits & PA_STATUS_TIMEOUT) {
        // Let copies still in flight into this warp's ring land before the
        // shared memory is reused or released (bounded again).
        for (int k = i; k < issued; ++k)
            mbar_wait_bounded(bar0 + 8 * (k % stages), (uint32_t)(k / stages) & 1u, kWaitLimitNs);
    }
    if (status_bits && lane == 0)
        set_status(p.status, status_bits);

    // ---- hand the warp's {m, l, o} to the CTA merge (scratch = this warp's own ring)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_run[j][0] += __shfl_xor_sync(0xffffffffu, l_run[j][0], off);
            l_run[j][1] += __shfl_xor_sync(0xffffffffu, l_run[j][1], off);
        }
    }
    float *scr = reinterpret_cast<float *>(dyn_smem + (ring - smem_addr(dyn_smem)));
    float *scr_m = scr;
    float *scr_l = scr + kHeads;
    float *scr_o = scr + 2 * kHeads; // [kHeads][kScr]
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int hA = j * 8 + 2 * t4;
        if (g4 == 0) {
            scr_m[hA] = m_run[j][0];
            scr_m[hA + 1] = m_run[j][1];
            scr_l[hA] = l_run[j][0];
            scr_l[hA + 1] = l_run[j][1];
        }
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) {
            const int d = mt * 16 + g4;
            scr_o[hA * kScr + d] = o[j][mt][0];
            scr_o[(hA + 1) * kScr + d] = o[j][mt][1];
            scr_o[hA * kScr + d + 8] = o[j][mt][2];
            scr_o[(hA + 1) * kScr + d + 8] = o[j][mt][3];
        }
    }
    __syncthreads();

    // ---- merge the warps: M = max m_w, f_w = exp(m_w - M), l = sum f_w l_w, o = sum f_w o_w / l
    const uint32_t warp_stride = (uint32_t)stages * kStageBytes / 4; // floats between warp scratches
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
        // lsum == 0: no token of this range is visible to the column (only with
        // several new tokens): an empty partition, or a zero output in V1.
        s_stat[2][h] = lsum > 0.f ? 1.f / lsum : 0.f;
    }
    __syncthreads();

    // Four consecutive dims per thread and pass (16-byte shared loads and a
    // 16-byte partials store), the reciprocal of the sum taken once per head.
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

    if constexpr (!V1 && FUSED) {
        // ---- phase 2 in the last CTA of this (sequence, KV head).  Each
        // thread's partial writes are made visible device-wide before the
        // ticket is taken; the ticket counter wraps to 0 on the last ticket,
        // which leaves it ready for the next call.
        __shared__ int s_last;
        __threadfence();
        __syncthreads();
        const int np_b = (L + p.partition_size - 1) / p.partition_size;
        if (threadIdx.x == 0) {
            const unsigned total = (unsigned)np_b * (unsigned)p.col_groups;
            unsigned *ctr = reinterpret_cast<unsigned *>(p.counters) +
                            (size_t)b * p.num_kv_heads + kv;
            s_last = atomicInc(ctr, total - 1u) == total - 1u;
        }
        __syncthreads();
        if (!s_last)
            return;
        __threadfence();
        // One (query row, 4 dims) per thread and pass, over every row of the
        // KV head (all column groups): M = max m_p, w_p = exp(m_p - M) l_p,
        // out = sum w_p o_p / sum w_p, with M raised as larger maxima appear
        // ("paged_attention_v2_pytorch.py" commit 9cb7f9d, "Implementation",
        // Phase 2).  Loads bypass L1 (other CTAs wrote them in this grid).
        for (int idx = threadIdx.x; idx < p.cols * kQuads; idx += blockDim.x) {
            const int n = idx / kQuads;
            const int d = (idx % kQuads) * 4;
            const size_t bh =
                ((size_t)b * p.q_len + n / p.group) * p.num_heads + head0 + n % p.group;
            const float *ml = p.max_logits + bh * p.max_num_partitions;
            const float *es = p.exp_sums + bh * p.max_num_partitions;
            const float *tp = p.tmp_output + bh * p.max_num_partitions * D + d;
            float m = -INFINITY, l = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int q = 0; q < np_b; ++q) {
                const float mp = __ldcg(ml + q);
                const float lp = __ldcg(es + q);
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(tp + (size_t)q * D));
                if (lp == 0.f)
                    continue;
                const float mn = fmaxf(m, mp);
                const float a = fast_exp2((m - mn) * kLog2e);
                const float w = fast_exp2((mp - mn) * kLog2e) * lp;
                acc.x = fmaf(acc.x, a, w * v.x);
                acc.y = fmaf(acc.y, a, w * v.y);
                acc.z = fmaf(acc.z, a, w * v.z);
                acc.w = fmaf(acc.w, a, w * v.w);
                l = fmaf(l, a, w);
                m = mn;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T *o4 = static_cast<T *>(p.out) + bh * D + d;
            o4[0] = E::from_float(acc.x * inv);
            o4[1] = E::from_float(acc.y * inv);
            o4[2] = E::from_float(acc.z * inv);
            o4[3] = E::from_float(acc.w * inv);
        }
    }
}

// Kernel dispatch on block size, n-tiles (<= 8 or <= 16 columns) and V1 /
// V2 / fused V2, for one head_dim.  `v1` is 1 for V1, 0 for V2 and 2 for
// the fused V2.
template <typename T, int D>
static const void *attn_kernel_ptr(int block_size, int cols, int v1)
{
    const bool nt2 = cols > 8;
#define PA_PICK_NT(BS, NT)                                                                        \
    return v1 == 1   ? reinterpret_cast<const void *>(&attn_kernel<T, D, BS, NT, true>)           \
           : v1 == 2 ? reinterpret_cast<const void *>(&attn_kernel<T, D, BS, NT, false, true>)    \
                     : reinterpret_cast<const void *>(&attn_kernel<T, D, BS, NT, false>);
#define PA_PICK(BS)                                                                               \
    if (block_size == BS) {                                                                       \
        if (nt2) {                                                                                \
            PA_PICK_NT(BS, 2)                                                                     \
        }                                                                                         \
        PA_PICK_NT(BS, 1)                                                                         \
    }
    PA_PICK(8)
    PA_PICK(16)
    PA_PICK(32)
    PA_PICK(64)
#undef PA_PICK
#undef PA_PICK_NT
    return nullptr;
}

// Opts the kernel in to the largest dynamic shared memory the device allows
// next to its static shared memory; returns that limit in *limit.
template <typename T, int D>
static cudaError_t attn_prepare(int block_size, int cols, int v1, int optin_bytes, size_t *limit)
{
    const void *fn = attn_kernel_ptr<T, D>(block_size, cols, v1);
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

// Resident CTAs per SM for a launch shape (0 on error).
template <typename T, int D>
static int attn_occupancy(int block_size, int cols, int v1, int warps, size_t smem_bytes)
{
    const void *fn = attn_kernel_ptr<T, D>(block_size, cols, v1);
    int n = 0;
    if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, warps * 32, smem_bytes) !=
                   cudaSuccess)
        return 0;
    return n;
}

template <typename T, int D>
static cudaError_t attn_launch(const AttnLaunch &L, cudaStream_t stream)
{
    const void *fn = attn_kernel_ptr<T, D>(L.block_size, L.cta_cols, attn_variant(L));
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

// The table one translation unit exports for its (storage type, head_dim).
#define PA_DEFINE_ATTN_OPS(T, NAME, D)                                                            \
    const AttnOps *NAME()                                                                         \
    {                                                                                             \
        static const AttnOps ops = {&attn_prepare<T, D>, &attn_occupancy<T, D>,                   \
                                    &attn_launch<T, D>};                                          \
        return &ops;                                                                              \
    }

} // namespace pa
