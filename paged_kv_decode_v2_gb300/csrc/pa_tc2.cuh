// pa_tc2.cuh -- the tcgen05 attention kernel for many query rows per KV head
// (long multi-token steps, chunked prefill), two query tiles per CTA.
//
// It computes what pa_tc.cuh's kernel computes (paged-attention pages,
// "PagedAttention V2": per (sequence, KV head, partition) the partition's
// softmax statistics and partition-normalised softmax.V of every query row,
// or V1's final output), arranged for throughput when a KV head has more
// than 128 query rows:
//
//   * one CTA per SM holds two 128-row query tiles that share every K/V tile,
//     so each K/V byte brought to the SM serves 256 rows;
//   * K/V tiles are 128 tokens, so S = Q K^T is N = 128 per tcgen05.mma;
//   * per tile q, TMEM holds O (head_dim columns) and S (128 columns); P
//     (16-bit, hi + lo halves for bf16) is written over the S columns it was
//     computed from, so the next S of that tile is issued right after its
//     P.V, in order on the tensor pipe;
//   * the MMA thread alternates the tiles: while one tile's rows run their
//     softmax, the tensor cores run the other tile's P.V and next S;
//   * as in pa_tc.cuh, the running max m moves only when a row would
//     otherwise see P > 2^8, so O is rarely rescaled; a V2 partial reports
//     the true max with l rescaled to it.
//
// Warp roles: warps 0-3 own the rows of tile 0 and warps 4-7 those of tile
// 1 (one row per thread), warp 8 issues the MMAs and owns the TMEM
// allocation, two lanes of warp 9 load the K and V tiles with TMA.
//
// bf16 caches: the VH form reads V from the packed binary16 copy of the
// call's V blocks (pa_vhalf.cu) and runs P.V on binary16 P and V, one MMA per K-step,
// as for fp16 caches; the other form splits P into bf16 hi + lo halves.
// S = Q K^T stays in bf16.  The VH kernel holds both forms and takes the bf16
// one when the copy's flag is set.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

template <int D>
struct Tc2Cfg {
    static constexpr int kSlices = D / 64;
    static constexpr uint32_t kQSlice = kTcRows * 128;                // bytes of one Q slice
    static constexpr uint32_t kKVSlice = kTc2Tok * 128;               // bytes of one K or V slice
    static constexpr uint32_t kQBytes = kQSlice * kSlices;            // one query tile
    static constexpr uint32_t kKVBytes = kKVSlice * kSlices;          // one K (or V) tile
    // TMEM of tile q: O at q * 256 + [0, D), S / P at q * 256 + [128, 256).
    static constexpr uint32_t kTileCols = 256;
    static constexpr uint32_t kSCol = 128;
};

// The kernel's body for one P format: H, V from the binary16 copy and P in
// binary16 (bf16 caches only); otherwise the cache's own form.
template <typename T, int D, int BS, bool V1, bool H>
__device__ __forceinline__ void tc2_body(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                         const CUtensorMap &tmap_vh, const AttnParams &p)
{
    static_assert(D <= 128, "two query tiles need O + S of each in 256 TMEM columns");
    using C = Tc2Cfg<D>;
    using E = Elem<T>;
    constexpr bool kBf16 = E::kSplitP;
    constexpr int kBPT = kTc2Tok / BS; // blocks per tile

    __shared__ uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages],
        v_empty[kMaxStages];
    __shared__ uint64_t q_full, s_full[2], p_full[2], drained;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    extern __shared__ uint8_t dyn_smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cgi = V1 ? (int)blockIdx.x : (int)blockIdx.x % p.col_groups; // pair of row tiles
    const int part = V1 ? 0 : (int)blockIdx.x / p.col_groups;
    const int kv = blockIdx.y;
    const int b = blockIdx.z;

    static_assert(!H || kBf16, "the binary16 copy is for bf16 caches");
    constexpr bool use_h = H;

    int L = __ldg(&p.seq_lens[b]);
    if (L < 0 || L > p.seq_len_cap) {
        if (threadIdx.x == 0 && part == 0 && kv == 0 && cgi == 0)
            set_status(p.status, PA_STATUS_BAD_SEQ_LEN);
        L = L < 0 ? 0 : p.seq_len_cap;
    }
    const int tokA = V1 ? 0 : part * p.partition_size;
    if (!V1 && tokA >= L)
        return; // partition past the end of the sequence: nothing to write

    // Rows of the CTA: [c0, c0 + nrows) of the KV head's cols = q_len * G;
    // tile q holds [c0 + 128 q, ...).  Tile 1 may be empty.
    const int c0 = cgi * 2 * kTcRows;
    const int nrows = min(2 * kTcRows, p.cols - c0);
    const int ntq = nrows > kTcRows ? 2 : 1; // query tiles with rows
    const int i_last = (c0 + nrows - 1) / p.group;
    long long e = V1 ? (long long)L : min((long long)L, (long long)tokA + p.partition_size);
    e = min(e, (long long)L - p.q_len + i_last + 1);
    const int tokE = (int)e;
    const int blk0 = tokA / BS;
    const int tok0 = blk0 * BS;
    const int ntiles = tokE > tokA ? (tokE - tok0 + kTc2Tok - 1) / kTc2Tok : 0;
    const int nblk = tokE > tokA ? (tokE - tok0 + BS - 1) / BS : 0;

    // This thread's row (warps 0-7): tile q, row r of the tile.
    const int q = threadIdx.x >> 7;
    const int r = threadIdx.x & 127;
    const bool row_ok = threadIdx.x < 2 * kTcRows && 128 * q + r < nrows;
    const int ci = c0 + (row_ok ? 128 * q + r : 0);
    const int qi = ci / p.group;
    const int head = kv * p.group + ci % p.group;
    const size_t qrow = ((size_t)b * p.q_len + qi) * p.num_heads + head;

    // The row's first 256 bytes of Q are fetched now, so their latency
    // overlaps the TMEM allocation and barrier set-up below.
    constexpr int kQChunks = D / 8;                       // 16-byte chunks of a row
    constexpr int kEarly = kQChunks < 16 ? kQChunks : 16; // chunks held in registers
    const uint32_t *q32 = static_cast<const uint32_t *>(p.query) + qrow * (D / 2);
    // Rows are D * 2 bytes apart, so one base check covers every row.
    const bool q_vec = (reinterpret_cast<uintptr_t>(p.query) & 15u) == 0;
    auto q_chunk = [&](int ch) -> uint4 {
        if (!row_ok)
            return make_uint4(0u, 0u, 0u, 0u);
        if (q_vec)
            return __ldg(reinterpret_cast<const uint4 *>(q32) + ch);
        return make_uint4(__ldg(q32 + ch * 4), __ldg(q32 + ch * 4 + 1), __ldg(q32 + ch * 4 + 2),
                          __ldg(q32 + ch * 4 + 3));
    };
    uint4 q_early[kEarly];
#pragma unroll
    for (int ch = 0; ch < kEarly; ++ch)
        q_early[ch] = q_chunk(ch);

    if (ntiles == 0) {
        if (row_ok) {
            if (V1) {
                T *out = static_cast<T *>(p.out) + qrow * D;
                for (int d = 0; d < D; ++d)
                    out[d] = E::from_float(0.f);
            } else {
                const size_t slot = qrow * p.max_num_partitions + part;
                float4 *tmp = reinterpret_cast<float4 *>(p.tmp_output + slot * D);
                for (int d = 0; d < D / 4; ++d)
                    tmp[d] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.exp_sums[slot] = 0.f;
                p.max_logits[slot] = -INFINITY;
            }
        }
        return;
    }

    const int kst = p.stages;
    const int vst = p.v_stages;
    const uint32_t smem0 = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    const uint32_t q_sm = smem0; // two query tiles
    const uint32_t k_sm = smem0 + 2 * C::kQBytes;
    const uint32_t v_sm = k_sm + (uint32_t)kst * C::kKVBytes;
    const uint32_t b_k_full = smem_addr(k_full), b_v_full = smem_addr(v_full);
    const uint32_t b_k_empty = smem_addr(k_empty), b_v_empty = smem_addr(v_empty);
    const uint32_t b_q_full = smem_addr(&q_full), b_drained = smem_addr(&drained);
    const uint32_t b_s_full = smem_addr(s_full), b_p_full = smem_addr(p_full);
    volatile int *abort_flag = &abort_sh;

    if (warp == 8) {
        tmem_alloc(smem_addr(&tmem_base_sh), 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 288) {
        for (int s = 0; s < kst; ++s) {
            mbar_init(b_k_full + 8 * s, 1);
            mbar_init(b_k_empty + 8 * s, 1);
        }
        for (int s = 0; s < vst; ++s) {
            mbar_init(b_v_full + 8 * s, 1);
            mbar_init(b_v_empty + 8 * s, 1);
        }
        mbar_init(b_q_full, kTcRows * ntq);
        for (int t = 0; t < 2; ++t) {
            mbar_init(b_s_full + 8 * t, 1);
            mbar_init(b_p_full + 8 * t, kTcRows);
        }
        mbar_init(b_drained, 1);
        abort_sh = 0;
        mbar_init_fence();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    int32_t status_bits = 0;

    if (warp == 9) {
        // ---------------------------------------------------------- producers
        // Lane 0 loads the K tiles, lane 1 the V tiles, each into its own ring:
        // a K stage is free once S of both query tiles is computed, a V stage
        // once P.V of both is.  Block ids are fetched a tile ahead.
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap *map = is_k ? &tmap_k : use_h ? &tmap_vh : &tmap_v;
            // The binary16 copy, [KV][vh_blocks][block_size] rows, holds the
            // sequence's logical block j of KV head kv at kv * vh_blocks + vh_offs[b] + j.
            const long long vh_blk0 =
                use_h ? (long long)kv * p.vh_blocks + __ldg(&p.vh_offs[b]) + blk0 : 0;
            const uint32_t ring = is_k ? k_sm : v_sm;
            const uint32_t full = is_k ? b_k_full : b_v_full;
            const uint32_t empty = is_k ? b_k_empty : b_v_empty;
            const int stages = is_k ? kst : vst;
            const uint64_t policy = l2_evict_normal_policy();
            const int32_t *bt = p.block_tables + (size_t)b * p.max_blocks + blk0;
            int32_t ids[kBPT], nxt[kBPT];
            auto fetch = [&](int t, int32_t(&dst)[kBPT]) {
#pragma unroll
                for (int k = 0; k < kBPT; ++k) {
                    const int bi = t * kBPT + k;
                    int32_t id = 0;
                    if (t < ntiles && bi < nblk) {
                        id = __ldg(bt + bi);
                        if (id < 0 || id >= p.num_blocks) {
                            status_bits |= PA_STATUS_BAD_BLOCK_ID;
                            id = 0; // read a valid block instead of memory outside the cache
                        }
                    }
                    dst[k] = id;
                }
            };
            fetch(0, nxt);
            int issued = 0;
            int s = 0;         // ring stage of tile t
            uint32_t ph = 0u;  // its fill round & 1
            for (int t = 0; t < ntiles; ++t) {
#pragma unroll
                for (int k = 0; k < kBPT; ++k)
                    ids[k] = nxt[k];
                fetch(t + 1, nxt);
                if (t >= stages && !mbar_wait_abortable(empty + 8 * s, ph ^ 1u, abort_flag)) {
                    status_bits |= PA_STATUS_TIMEOUT;
                    *abort_flag = 1;
                    break;
                }
                const int nb = min(kBPT, nblk - t * kBPT);
                mbar_arrive_expect_tx(full + 8 * s, (uint32_t)nb * BS * 128u * C::kSlices);
#pragma unroll
                for (int k = 0; k < kBPT; ++k) {
                    if (k < nb) {
                        const int row =
                            !is_k && use_h
                                ? (int)((vh_blk0 + t * kBPT + k) * BS)
                                : (int)(((long long)ids[k] * p.num_kv_heads + kv) * BS);
#pragma unroll
                        for (int sl = 0; sl < C::kSlices; ++sl)
                            tma_load_3d(ring + s * C::kKVBytes + sl * C::kKVSlice + k * BS * 128, map,
                                        0, sl, row, full + 8 * s, policy);
                    }
                }
                issued = t + 1;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            for (int t = max(0, issued - stages); t < issued; ++t)
                mbar_wait_bounded(full + 8 * (t % stages), (uint32_t)(t / stages) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 8) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16<kBf16>(kTcRows, kTc2Tok, false);
            constexpr uint32_t idesc_o = idesc_f16<kBf16>(kTcRows, D, true);
            constexpr uint32_t idesc_o16 = idesc_f16<false>(kTcRows, D, true);
            const bool split = kBf16 && !use_h; // P in hi + lo halves
            // Descriptors are linear in the address (start / 16 in the low
            // bits, shared memory < 256 KB): offsets are added to a base.
            const uint64_t qd = smem_desc_sw128(q_sm, 16, 1024);
            const uint64_t kd = smem_desc_sw128(k_sm, 16, 1024);
            const uint64_t vd = smem_desc_sw128(v_sm, C::kKVSlice, 1024);
            // S_q = Q_q K^T of the K tile in ring stage ks into tile q's S columns.
            auto issue_s = [&](int qq, int ks_stage) {
                const uint64_t kb = kd + (((uint32_t)ks_stage * C::kKVBytes) >> 4);
                const uint64_t qb = qd + (((uint32_t)qq * C::kQBytes) >> 4);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off_q = (ks >> 2) * C::kQSlice + (ks & 3) * 32;
                    const uint32_t off_k = (ks >> 2) * C::kKVSlice + (ks & 3) * 32;
                    tc_mma_ss(tmem + qq * C::kTileCols + C::kSCol, qb + (off_q >> 4), kb + (off_k >> 4),
                              idesc_s, ks > 0);
                }
            };
            // O_q += P_q V of tile t in ring stage vs_stage: P's 16 tokens of
            // K-step kt sit at S column 32 (kt / 2) + 8 (kt % 2), the lo
            // halves 16 columns further.
            auto issue_pv = [&](int qq, int vs_stage, int t) {
                const uint64_t vb = vd + (((uint32_t)vs_stage * C::kKVBytes) >> 4);
                const uint32_t pc = tmem + qq * C::kTileCols + C::kSCol;
#pragma unroll
                for (int kt = 0; kt < kTc2Tok / 16; ++kt) {
                    const uint32_t a = pc + 32 * (kt >> 1) + 8 * (kt & 1);
                    const uint64_t bd = vb + ((kt * 2048) >> 4);
                    tc_mma_ts(tmem + qq * C::kTileCols, a, bd, split ? idesc_o : idesc_o16,
                              (t > 0 || kt > 0) ? 1u : 0u);
                    if (split)
                        tc_mma_ts(tmem + qq * C::kTileCols, a + 16, bd, idesc_o, 1u);
                }
            };
            bool ok = mbar_wait_abortable(b_q_full, 0, abort_flag) &&
                      mbar_wait_abortable(b_k_full, 0, abort_flag);
            if (ok) {
                tc_fence_after();
                for (int qq = 0; qq < ntq; ++qq) {
                    issue_s(qq, 0);
                    tc_commit(b_s_full + 8 * qq);
                }
                tc_commit(b_k_empty);
            }
            int vs = 0;                          // V ring stage of tile t
            uint32_t vph = 0u;                   // and its fill round & 1
            int ks1 = kst > 1 ? 1 : 0;           // K ring stage of tile t + 1
            uint32_t kph1 = kst > 1 ? 0u : 1u;
            for (int t = 0; ok && t < ntiles; ++t) {
                ok = mbar_wait_abortable(b_v_full + 8 * vs, vph, abort_flag);
                for (int qq = 0; ok && qq < ntq; ++qq) {
                    ok = mbar_wait_abortable(b_p_full + 8 * qq, (uint32_t)t & 1u, abort_flag);
                    if (ok && qq == 0 && t + 1 < ntiles)
                        ok = mbar_wait_abortable(b_k_full + 8 * ks1, kph1, abort_flag);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_pv(qq, vs, t);
                    if (t + 1 < ntiles)
                        issue_s(qq, ks1);
                    // Arrives once P.V(t) and S(t + 1) of tile qq are done (the
                    // last tile: once its final P.V is).
                    tc_commit(b_s_full + 8 * qq);
                }
                if (!ok)
                    break;
                tc_commit(b_v_empty + 8 * vs);
                if (t + 1 < ntiles)
                    tc_commit(b_k_empty + 8 * ks1);
                if (++vs == vst) {
                    vs = 0;
                    vph ^= 1u;
                }
                if (++ks1 == kst) {
                    ks1 = 0;
                    kph1 ^= 1u;
                }
            }
            if (!ok) {
                status_bits |= PA_STATUS_TIMEOUT;
                *abort_flag = 1;
            }
            tc_commit(b_drained);
            mbar_wait_bounded(b_drained, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (q < ntq) {
        // ---------------------------------------------------------- rows of tile q
        {
            const uint32_t qb = q_sm + (uint32_t)q * C::kQBytes;
#pragma unroll
            for (int ch = 0; ch < kQChunks; ++ch) {
                const uint4 v = ch < kEarly ? q_early[ch] : q_chunk(ch);
                const uint32_t addr =
                    qb + (ch >> 3) * C::kQSlice + r * 128 + ((((ch & 7) ^ (r & 7))) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            fence_proxy_async();
            mbar_arrive(b_q_full);
        }
        const int hi = row_ok ? min(tokE, L - p.q_len + qi + 1) : tokA;
        const unsigned span = (unsigned)max(hi - tokA, 0);
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t o_col = lane_base + q * C::kTileCols;
        const uint32_t s_col = o_col + C::kSCol;
        const uint32_t b_sf = b_s_full + 8 * q, b_pf = b_p_full + 8 * q;
        const float scale = p.scale;
        // m_run: the max P and O are relative to; m_true: the row's max.
        float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            // S_q(t) is ready, and P.V of the previous tile is done (O is stable).
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(b_sf, (uint32_t)t & 1u, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int off = tok0 + t * kTc2Tok - tokA;
            const bool whole =
                __all_sync(0xffffffffu, scale > 0.f && off >= 0 && off + kTc2Tok <= (int)span);
            // Pass 1: the row max over the tile's 128 scores, loaded with one
            // wait.  x: the raw score on whole tiles with scale > 0 (scale
            // folded into cf: max(s) * scale = max(s * scale)), else masked
            // s * scale.
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            {
                uint32_t sr[4][32];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tmem_ld32_async(s_col + 32 * k, sr[k]);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tmem_ld_wait(sr[k]);
                if (whole) {
#pragma unroll
                    for (int c = 0; c < kTc2Tok; c += 2)
                        mq[(c >> 1) & 3] = fmax3(mq[(c >> 1) & 3], __uint_as_float(sr[c >> 5][c & 31]),
                                                 __uint_as_float(sr[c >> 5][(c & 31) + 1]));
                } else {
#pragma unroll
                    for (int c = 0; c < kTc2Tok; ++c) {
                        const float s = __uint_as_float(sr[c >> 5][c & 31]);
                        mq[c & 3] = fmaxf(mq[c & 3],
                                          (unsigned)(off + c) < span ? s * scale : -INFINITY);
                    }
                }
            }
            float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            float cf = kLog2e;
            if (whole) {
                mx *= scale;
                cf = scale * kLog2e;
            }
            m_true = fmaxf(m_true, mx);
            // m moves only when a row of the warp would otherwise see P > 2^8
            // (always on its first visible tile, where m_run = -inf).
            float a = 1.f;
            if (__any_sync(0xffffffffu, (mx - m_run) * kLog2e > kTcRescaleLog2)) {
                const float mn = fmaxf(m_run, mx);
                a = mn != -INFINITY ? fast_exp2((m_run - mn) * kLog2e) : 1.f;
                m_run = mn;
            }
            const float mb = m_run != -INFINITY ? m_run * kLog2e : 0.f;
            // Pass 2, 64 tokens at a time: P = exp(x * cf - mb), written over
            // the S columns just read: per 32 tokens, hi halves at [32k, 32k +
            // 16), lo at [32k + 16, 32k + 32).
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            uint64_t ls2[2] = {0ull, 0ull}; // packed row sums of the binary16 form
            const uint64_t cf2 = f2_pack(cf, cf), nmb2 = f2_pack(-mb, -mb);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t sr[2][32];
                tmem_ld32_async(s_col + 64 * h, sr[0]);
                tmem_ld32_async(s_col + 64 * h + 32, sr[1]);
                tmem_ld_wait(sr[0]);
                tmem_ld_wait(sr[1]);
                if (!whole) {
#pragma unroll
                    for (int k = 0; k < 2; ++k)
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const float s = __uint_as_float(sr[k][c]);
                            sr[k][c] = __float_as_uint(
                                (unsigned)(off + 64 * h + 32 * k + c) < span ? s * scale : -INFINITY);
                        }
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t ph[16], pl[16];
                    const uint32_t col = s_col + 64 * h + 32 * k;
                    if (kBf16 && !use_h) {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float x0 = __uint_as_float(sr[k][c]), x1 = __uint_as_float(sr[k][c + 1]);
                            const float p0 = fast_exp2(fmaf(x0, cf, -mb));
                            const float p1 = fast_exp2(fmaf(x1, cf, -mb));
                            ls[(c >> 1) & 3] += p0 + p1;
                            const uint32_t hh = E::pack(p0, p1);
                            ph[c >> 1] = hh;
                            pl[c >> 1] = E::pack(p0 - E::lo(hh), p1 - E::hi(hh));
                        }
                        tmem_st16x2(col, ph, col + 16, pl);
                    } else {
                        // binary16 P: fp16 caches, or bf16 with V from the copy
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            float y0, y1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k][c]), __uint_as_float(sr[k][c + 1])),
                                             cf2, nmb2),
                                      y0, y1);
                            const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                            ls2[(c >> 1) & 1] = f2_add(ls2[(c >> 1) & 1], f2_pack(p0, p1));
                            ph[c >> 1] = Elem<__half>::pack(p0, p1);
                        }
                        tmem_st16_async(col, ph);
                    }
                }
            }
            // One wait for the tile's P stores (tcgen05.st takes its registers
            // when issued), before the arrival below lets P.V read them.
            if (!(kBf16 && !use_h))
                tmem_st_wait();
            if (!(kBf16 && !use_h)) {
                f2_unpack(f2_add(ls2[0], ls2[1]), ls[0], ls[1]);
            }
            l_run = fmaf(l_run, a, (ls[0] + ls[1]) + (ls[2] + ls[3]));
            // Rescale O when m moved (O holds P.V of earlier tiles only from t = 1).
            if (t > 0 && __any_sync(0xffffffffu, a != 1.f)) {
#pragma unroll 1
                for (int cc = 0; cc < D; cc += 64) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32_async(o_col + cc, o0);
                    tmem_ld32_async(o_col + cc + 32, o1);
                    tmem_ld_wait(o0);
                    tmem_ld_wait(o1);
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        o0[k] = __float_as_uint(__uint_as_float(o0[k]) * a);
                        o1[k] = __float_as_uint(__uint_as_float(o1[k]) * a);
                    }
                    tmem_st32x2(o_col + cc, o0, o_col + cc + 32, o1);
                }
            }

            if (t == ntiles - 1 && q == 0) {
                // Tile rows past the range may hold anything: zero them in V so
                // that 0 * garbage cannot reach O (tile 0's P.V runs first).
                const int vt = tokE - (tok0 + t * kTc2Tok);
                if (vt < kTc2Tok) {
                    const int s = t % vst;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_abortable(b_v_full + 8 * s, (uint32_t)(t / vst) & 1u,
                                                        abort_flag))) {
                        ok = false;
                        break;
                    }
                    const uint32_t vb = v_sm + (uint32_t)s * C::kKVBytes;
                    const int nchunks = (kTc2Tok - vt) * 8 * C::kSlices;
                    for (int idx = r; idx < nchunks; idx += kTcRows) {
                        const int sl = idx % C::kSlices;
                        const int rest = idx / C::kSlices;
                        st_shared_zero16(vb + sl * C::kKVSlice + (vt + rest / 8) * 128 + (rest & 7) * 16);
                    }
                    fence_proxy_async();
                }
            }
            tc_fence_before();
            mbar_arrive(b_pf);
        }
        // The last P.V of the tile has completed once s_full completes once more.
        if (ok && !__all_sync(0xffffffffu,
                              mbar_wait_abortable(b_sf, (uint32_t)ntiles & 1u, abort_flag)))
            ok = false;
        if (!ok) {
            status_bits |= PA_STATUS_TIMEOUT;
            *abort_flag = 1;
        } else {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            if (V1) {
                uint32_t *out = reinterpret_cast<uint32_t *>(static_cast<T *>(p.out) + qrow * D);
#pragma unroll 1
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t o[32];
                    tmem_ld32(o_col + cc, o);
                    if (row_ok) {
#pragma unroll
                        for (int k = 0; k < 32; k += 2)
                            out[(cc + k) / 2] = E::pack(__uint_as_float(o[k]) * inv,
                                                        __uint_as_float(o[k + 1]) * inv);
                    }
                }
            } else {
                const size_t slot = qrow * p.max_num_partitions + part;
                float4 *tmp = reinterpret_cast<float4 *>(p.tmp_output + slot * D);
#pragma unroll 1
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t o[32];
                    tmem_ld32(o_col + cc, o);
                    if (row_ok) {
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            tmp[(cc + k) / 4] = make_float4(
                                __uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                                __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
                    }
                }
                if (row_ok) {
                    // The partition's statistics relative to its true max.
                    p.exp_sums[slot] =
                        m_true != -INFINITY ? l_run * fast_exp2((m_run - m_true) * kLog2e) : 0.f;
                    p.max_logits[slot] = m_true;
                }
            }
        }
    }

    if (status_bits)
        set_status(p.status, status_bits);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// VH = false: the form of the cache's type.  VH = true (bf16): V from the
// binary16 copy with binary16 P, unless the copy's flag is set (a value
// binary16 cannot hold, or a copy too large for its space), in which case the
// bf16 form with hi + lo P on the cache; the flag is final once the previous
// grid (the copy pass) has completed, so every thread reads the same value.
template <typename T, int D, int BS, bool V1, bool VH = false>
__global__ void __launch_bounds__(kTc2Threads)
    tc2_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_vh,
                    const __grid_constant__ AttnParams p)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if constexpr (VH) {
        if (__ldcg(p.vh_flag) == 0)
            tc2_body<T, D, BS, V1, true>(tmap_k, tmap_v, tmap_vh, p);
        else
            tc2_body<T, D, BS, V1, false>(tmap_k, tmap_v, tmap_vh, p);
    } else {
        tc2_body<T, D, BS, V1, false>(tmap_k, tmap_v, tmap_vh, p);
    }
}

} // namespace pa
