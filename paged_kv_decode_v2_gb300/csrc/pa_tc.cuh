// pa_tc.cuh -- paged attention for many query rows per KV head on the
// tcgen05 tensor cores: several new tokens per sequence (checking speculated
// tokens) up to chunked prefill, where a chunk of new tokens attends to the
// cached prefix and, causally, to itself.
//
// Paged-attention pages, "PagedAttention V2" and its split-K description:
// phase 1 computes, per (sequence, KV head, partition), the softmax
// statistics and the partition-normalised softmax.V of every query row of
// the GQA group; phase 2 (pa_merge.cu) merges partitions by log-sum-exp.
// The same kernel also runs as V1 (one range covering the whole sequence,
// final output written directly).  The pages' kernels tile
// [kv_head, gqa, q_len, tile]; this one takes 128 query rows (new token i,
// head g of the group, row = i * group + g) per CTA as the M of the MMA:
//
//   S   = Q K_t^T         tcgen05.mma, M = 128 rows, N = 64 tokens, K = D;
//                         A = Q and B = K tile in shared memory, S in TMEM
//   P   = exp(S - m)      one thread per row reads its S row from TMEM,
//                         masks, keeps the running max m and sum l, and
//                         writes P (16-bit, split into hi + lo for bf16)
//                         back to TMEM over its S
//   O  += P V_t           tcgen05.mma, M = 128, N = D, K = 64 tokens; A = P
//                         in TMEM, B = V tile (MN-major) in shared memory,
//                         O in TMEM
//
// S/P has two TMEM buffers, tile t in buffer t & 1, so the MMA thread runs
// S of tile t + 2 right behind P.V of tile t and the rows never wait for a
// P.V before writing their next P.  The running max m used for P and for O
// moves only when a row's max grows by more than 2^8 in exp2 terms (P then
// stays <= 2^8, which fp32 and the 16-bit hi + lo pair hold with the same
// relative precision as values <= 1); O is rescaled, after waiting for the
// last P.V, only then.  O / l does not depend
// on which m was used.  The true max is tracked beside it, and a V2 partial
// reports that max with l rescaled to it, as the merge expects.
//
// Half Q tile (p.q_half, a KV head of at most 64 rows): the rows sit at M
// indices 64-127, so only those 64 rows of Q are stored, 8 KB per 64-dim
// slice instead of 16.  The S MMA still reads 128 rows: its descriptor
// starts 8 KB before each stored slice, so the padding rows 0-63 read
// whatever lies there (the end of the K ring, or the previous slice).  MMA
// rows are independent and those rows' S, P and O are never stored, so the
// saved 16 KB (head_dim 128) buy a third ring stage at two CTAs per SM.
//
// Warp roles: warps 0-3 own the 128 rows (softmax, epilogue), warp 4 issues
// the MMAs (one thread) and owns the TMEM allocation, two lanes of warp 5
// gather the K and the V blocks of each 64-token tile with TMA, each into its
// own ring (p.stages K stages, p.v_stages V stages).
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tc2.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

template <int D>
struct TcCfg {
    static constexpr int kSlices = D / 64;                          // 128-byte swizzled column slices
    static constexpr uint32_t kQSlice = kTcRows * 128;              // bytes of one Q slice
    static constexpr uint32_t kKVSlice = kTcTok * 128;              // bytes of one K or V slice
    static constexpr uint32_t kQBytes = kQSlice * kSlices;
    static constexpr uint32_t kKVBytes = kKVSlice * kSlices;        // one K (or V) tile
    // TMEM columns: O at [0, D), S/P buffer j at [D + 64 j, D + 64 j + 64).
    // P is written over its S: hi at the buffer's first 32 columns, lo at
    // the next 32 (two 16-bit values per column).
    static constexpr uint32_t kSCol = D;
    static constexpr uint32_t kCols = D + 2 * kTcTok <= 256 ? 256 : 512;
};

template <typename T, int D, int BS, bool V1>
__global__ void __launch_bounds__(kTcThreads, D <= 128 ? 2 : 1)
    tc_attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const AttnParams p)
{
    using C = TcCfg<D>;
    using E = Elem<T>;
    constexpr bool kBf16 = E::kSplitP;
    constexpr int kBPT = kTcTok / BS; // blocks per tile

    __shared__ uint64_t k_full[kMaxStages], v_full[kMaxStages], k_empty[kMaxStages],
        v_empty[kMaxStages];
    __shared__ uint64_t q_full, s_full[2], p_full[2], o_done[2], drained;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    extern __shared__ uint8_t dyn_smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rt = V1 ? (int)blockIdx.x : (int)blockIdx.x % p.col_groups; // row tile
    const int part = V1 ? 0 : (int)blockIdx.x / p.col_groups;
    const int kv = blockIdx.y;
    const int b = blockIdx.z;

    // Programmatic stream serialisation: nothing global is touched before
    // the previous grid in the stream has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    int L = __ldg(&p.seq_lens[b]);
    if (L < 0 || L > p.seq_len_cap) {
        if (threadIdx.x == 0 && part == 0 && kv == 0 && rt == 0)
            set_status(p.status, PA_STATUS_BAD_SEQ_LEN);
        L = L < 0 ? 0 : p.seq_len_cap;
    }
    const int tokA = V1 ? 0 : part * p.partition_size;
    if (!V1 && tokA >= L)
        return; // partition past the end of the sequence: nothing to write

    // Rows [c0, c0 + nrows) of the KV head's cols = q_len * group rows.
    const int c0 = rt * kTcRows;
    const int nrows = min(kTcRows, p.cols - c0);
    const int i_last = (c0 + nrows - 1) / p.group;
    // Tokens the CTA needs: [tokA, tokE), the range cut by the causal limit
    // of its last new token (new token i sees positions <= L - q_len + i).
    long long e = V1 ? (long long)L : min((long long)L, (long long)tokA + p.partition_size);
    e = min(e, (long long)L - p.q_len + i_last + 1);
    const int tokE = (int)e;
    const int blk0 = tokA / BS;
    const int tok0 = blk0 * BS;
    const int ntiles = tokE > tokA ? (tokE - tok0 + kTcTok - 1) / kTcTok : 0;
    const int nblk = tokE > tokA ? (tokE - tok0 + BS - 1) / BS : 0;

    // This thread's row (warps 0-3).  A tile of fewer than 128 rows puts them
    // in the highest warps (M index = roff + row): whole warps of padding rows
    // then sit on the schedulers of the MMA and TMA warps and skip the
    // softmax, while the rows run on schedulers of their own.
    const int roff = kTcRows - (nrows + 31) / 32 * 32;
    const int r = threadIdx.x;
    const bool row_ok = r < kTcRows && r >= roff && r - roff < nrows;
    const int ci = c0 + (row_ok ? r - roff : 0);
    const int qi = ci / p.group;                 // new token
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
        // No row sees a token of the range: an empty partition (m = -inf,
        // l = 0, o = 0), or a zero output in V1.
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

    const int kst = p.stages;   // K ring stages
    const int vst = p.v_stages; // V ring stages
    const uint32_t smem0 = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    // Layout: [Q | K ring | V ring], or with a half Q tile [K ring | Q | V
    // ring], the K ring then holding the 8 KB the first slice's padding rows
    // alias (kst >= 1 K stages of >= 8 KB each).
    const bool q_half = p.q_half != 0;
    const uint32_t q_slice = q_half ? C::kQSlice / 2 : C::kQSlice; // bytes between Q slices
    const uint32_t k_sm = q_half ? smem0 : smem0 + C::kQBytes;
    const uint32_t q_sm = q_half ? k_sm + (uint32_t)kst * C::kKVBytes : smem0;
    const uint32_t v_sm = q_half ? q_sm + C::kQBytes / 2 : k_sm + (uint32_t)kst * C::kKVBytes;
    const uint32_t b_k_full = smem_addr(k_full), b_v_full = smem_addr(v_full);
    const uint32_t b_k_empty = smem_addr(k_empty), b_v_empty = smem_addr(v_empty);
    const uint32_t b_q_full = smem_addr(&q_full), b_s_full = smem_addr(s_full);
    const uint32_t b_p_full = smem_addr(p_full), b_o_done = smem_addr(o_done);
    const uint32_t b_drained = smem_addr(&drained);
    volatile int *abort_flag = &abort_sh;

    if (warp == 4) {
        tmem_alloc(smem_addr(&tmem_base_sh), C::kCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 160) {
        for (int s = 0; s < kst; ++s) {
            mbar_init(b_k_full + 8 * s, 1);
            mbar_init(b_k_empty + 8 * s, 1);
        }
        for (int s = 0; s < vst; ++s) {
            mbar_init(b_v_full + 8 * s, 1);
            mbar_init(b_v_empty + 8 * s, 1);
        }
        mbar_init(b_q_full, kTcRows);
        for (int j = 0; j < 2; ++j) {
            mbar_init(b_s_full + 8 * j, 1);
            mbar_init(b_p_full + 8 * j, kTcRows);
            mbar_init(b_o_done + 8 * j, 1);
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

    if (warp == 5) {
        // ---------------------------------------------------------- producers
        // Lane 0 loads the K tiles, lane 1 the V tiles, each into its own
        // ring and at its own pace: a K stage is free again once S of its
        // tile is computed, a V stage once P.V is.  Block ids are fetched a
        // tile ahead of their use.
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
            const uint32_t ring = is_k ? k_sm : v_sm;
            const uint32_t full = is_k ? b_k_full : b_v_full;
            const uint32_t empty = is_k ? b_k_empty : b_v_empty;
            const int stages = is_k ? kst : vst;
            const uint64_t policy =
                p.col_groups == 1 ? l2_evict_first_policy() : l2_evict_normal_policy();
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
                        const int row = (int)(((long long)ids[k] * p.num_kv_heads + kv) * BS);
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
            // Let copies still in flight land before the CTA's shared memory
            // is released (they have normally been consumed long ago).
            for (int t = max(0, issued - stages); t < issued; ++t)
                mbar_wait_bounded(full + 8 * (t % stages), (uint32_t)(t / stages) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 4) {
        // ---------------------------------------------------------- MMA issuer
        // Order: S(0), S(1), then per tile P.V(t) followed by S(t + 2) into
        // the buffer P(t) occupied.  tcgen05 MMAs of one thread run in issue
        // order, so S(t + 2) overwrites P(t) only after P.V(t) has read it,
        // and a commit that S(t) signals also covers every earlier P.V.
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16<kBf16>(kTcRows, kTcTok, false);
            constexpr uint32_t idesc_o = idesc_f16<kBf16>(kTcRows, D, true);
            // Descriptors are linear in the address (start / 16 in the low
            // bits, shared memory < 256 KB): offsets are added to a base.
            // With a half Q tile, each slice's descriptor starts 64 rows (8 KB)
            // before its stored rows 64-127.
            const uint64_t qd = smem_desc_sw128(q_half ? q_sm - C::kQSlice / 2 : q_sm, 16, 1024);
            const uint64_t kd = smem_desc_sw128(k_sm, 16, 1024);
            const uint64_t vd = smem_desc_sw128(v_sm, C::kKVSlice, 1024);
            int ks_next = 0;       // K ring stage of the next S
            uint32_t kph = 0u;     // and its fill round & 1
            // S(t) into buffer t & 1 once K tile t has landed.
            auto issue_s = [&](int t) -> bool {
                if (!mbar_wait_abortable(b_k_full + 8 * ks_next, kph, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t sc = tmem + C::kSCol + (uint32_t)(t & 1) * kTcTok;
                const uint64_t kb = kd + (((uint32_t)ks_next * C::kKVBytes) >> 4);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off_q = (ks >> 2) * q_slice + (ks & 3) * 32;
                    const uint32_t off_k = (ks >> 2) * C::kKVSlice + (ks & 3) * 32;
                    tc_mma_ss(sc, qd + (off_q >> 4), kb + (off_k >> 4), idesc_s, ks > 0);
                }
                tc_commit(b_s_full + 8 * (t & 1));
                tc_commit(b_k_empty + 8 * ks_next);
                if (++ks_next == kst) {
                    ks_next = 0;
                    kph ^= 1u;
                }
                return true;
            };
            bool ok = mbar_wait_abortable(b_q_full, 0, abort_flag) && issue_s(0) &&
                      (ntiles == 1 || issue_s(1));
            int vs = 0;            // V ring stage of tile t
            uint32_t vph = 0u;
            for (int t = 0; ok && t < ntiles; ++t) {
                const uint32_t pc = tmem + C::kSCol + (uint32_t)(t & 1) * kTcTok;
                ok = mbar_wait_abortable(b_p_full + 8 * (t & 1), (uint32_t)(t >> 1) & 1u, abort_flag) &&
                     mbar_wait_abortable(b_v_full + 8 * vs, vph, abort_flag);
                if (!ok)
                    break;
                tc_fence_after();
                const uint64_t vb = vd + (((uint32_t)vs * C::kKVBytes) >> 4);
#pragma unroll
                for (int kt = 0; kt < kTcTok / 16; ++kt)
                    tc_mma_ts(tmem, pc + kt * 8, vb + ((kt * 2048) >> 4), idesc_o,
                              (t > 0 || kt > 0) ? 1u : 0u);
                if (kBf16) {
#pragma unroll
                    for (int kt = 0; kt < kTcTok / 16; ++kt)
                        tc_mma_ts(tmem, pc + 32 + kt * 8, vb + ((kt * 2048) >> 4), idesc_o, 1u);
                }
                tc_commit(b_o_done + 8 * (t & 1));
                tc_commit(b_v_empty + 8 * vs);
                if (++vs == vst) {
                    vs = 0;
                    vph ^= 1u;
                }
                if (t + 2 < ntiles)
                    ok = issue_s(t + 2);
            }
            if (!ok) {
                status_bits |= PA_STATUS_TIMEOUT;
                *abort_flag = 1;
            }
            // Every MMA issued has completed once this commit arrives.
            tc_commit(b_drained);
            mbar_wait_bounded(b_drained, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- rows
        // Q row -> shared memory, 128-byte swizzled (16-byte chunk c of a row
        // of 64 dims at (c ^ (row & 7)) * 16), zero for padding rows; with a
        // half Q tile only rows 64-127 are stored, at row - 64.
        if (!q_half || r >= kTcRows / 2) {
            const int qr = q_half ? r - kTcRows / 2 : r;
#pragma unroll
            for (int ch = 0; ch < kQChunks; ++ch) {
                const uint4 v = ch < kEarly ? q_early[ch] : q_chunk(ch);
                const uint32_t addr =
                    q_sm + (ch >> 3) * q_slice + qr * 128 + ((((ch & 7) ^ (r & 7))) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
        }
        fence_proxy_async();
        mbar_arrive(b_q_full);
        if (warp * 32 + 32 <= roff) {
            // A warp of padding rows only: one arrival on "P ready" per tile,
            // after that tile's S, keeps the barrier's count (never a phase
            // early); its P lanes are never read into a row that is stored.
            for (int t = 0; t < ntiles; ++t) {
                if (!__all_sync(0xffffffffu, mbar_wait_abortable(b_s_full + 8 * (t & 1),
                                                                 (uint32_t)(t >> 1) & 1u, abort_flag))) {
                    status_bits |= PA_STATUS_TIMEOUT;
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive(b_p_full + 8 * (t & 1));
            }
        } else {
            // Visible tokens of this row: tokA <= t < hi (unsigned span from tokA).
            const int hi = row_ok ? min(tokE, L - p.q_len + qi + 1) : tokA;
            const unsigned span = (unsigned)max(hi - tokA, 0);
            const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
            const float scale = p.scale;
            // m_run: the max P and O are relative to; m_true: the row's max.
            float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const uint32_t sc = lane_base + C::kSCol + (uint32_t)(t & 1) * kTcTok;
                // Waits end in a warp-uniform decision: tcgen05.ld / st are warp-collective.
                if (!__all_sync(0xffffffffu, mbar_wait_abortable(b_s_full + 8 * (t & 1),
                                                                 (uint32_t)(t >> 1) & 1u, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32_async(sc, sr[0]);
                tmem_ld32_async(sc + 32, sr[1]);
                tmem_ld_wait(sr[0]);
                tmem_ld_wait(sr[1]);

                const int off = tok0 + t * kTcTok - tokA; // token (t's first) - tokA
                // x: the exp2 argument is x * cf - mb.  On a tile every row of the
                // warp sees whole (the common case) with scale > 0, x is the raw
                // score and the scale folds into cf (max(s) * scale = max(s * scale)
                // for scale > 0); otherwise x = s * scale, or -inf where masked.
                float x[kTcTok];
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}; // independent chains
                float mx, cf;
                // Padding rows of a partly filled warp vote yes: their P reaches only
                // O rows that are never stored.
                if (__all_sync(0xffffffffu,
                               !row_ok || (scale > 0.f && off >= 0 && off + kTcTok <= (int)span))) {
#pragma unroll
                    for (int c = 0; c < kTcTok; ++c) {
                        x[c] = __uint_as_float(sr[c >> 5][c & 31]);
                        mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    }
                    mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * scale;
                    cf = scale * kLog2e;
                } else {
#pragma unroll
                    for (int c = 0; c < kTcTok; ++c) {
                        const float s = __uint_as_float(sr[c >> 5][c & 31]);
                        x[c] = (unsigned)(off + c) < span ? s * scale : -INFINITY;
                        mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    }
                    mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                    cf = kLog2e;
                }
                m_true = fmaxf(m_true, mx);
                // Move m when a row of the warp would otherwise see P > 2^8 (the
                // first visible tile always: m_run = -inf).  NaN (both -inf) is no.
                float a = 1.f;
                if (__any_sync(0xffffffffu, row_ok && (mx - m_run) * kLog2e > kTcRescaleLog2)) {
                    const float mn = fmaxf(m_run, mx);
                    // A row with no visible token yet (max still -inf) keeps l = o = 0.
                    a = mn != -INFINITY ? fast_exp2((m_run - mn) * kLog2e) : 1.f;
                    m_run = mn;
                    // O is rescaled once the last P.V has landed (tile 0 has no O yet).
                    if (t > 0 && __any_sync(0xffffffffu, row_ok && a != 1.f)) {
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait_abortable(b_o_done + 8 * ((t - 1) & 1),
                                                            (uint32_t)((t - 1) >> 1) & 1u, abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < D; cc += 64) {
                            uint32_t o0[32], o1[32];
                            tmem_ld32_async(lane_base + cc, o0);
                            tmem_ld32_async(lane_base + cc + 32, o1);
                            tmem_ld_wait(o0);
                            tmem_ld_wait(o1);
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                o0[k] = __float_as_uint(__uint_as_float(o0[k]) * a);
                                o1[k] = __float_as_uint(__uint_as_float(o1[k]) * a);
                            }
                            tmem_st32x2(lane_base + cc, o0, lane_base + cc + 32, o1);
                        }
                    }
                }
                const float mb = m_run != -INFINITY ? m_run * kLog2e : 0.f;
                uint32_t ph[32], pl[32];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < kTcTok; c += 2) {
                    const float p0 = fast_exp2(fmaf(x[c], cf, -mb));
                    const float p1 = fast_exp2(fmaf(x[c + 1], cf, -mb));
                    ls[(c >> 1) & 3] += p0 + p1;
                    const uint32_t h = E::pack(p0, p1);
                    ph[c >> 1] = h;
                    pl[c >> 1] = kBf16 ? E::pack(p0 - E::lo(h), p1 - E::hi(h)) : 0u;
                }
                const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
                l_run = fmaf(l_run, a, lsum);

                // P over S in the same buffer: its S was read above, and P.V(t - 2),
                // the last reader of the buffer, completed before S(t) did.
                if (kBf16)
                    tmem_st32x2(sc, ph, sc + 32, pl);
                else
                    tmem_st32(sc, ph);

                if (t == ntiles - 1) {
                    // Tile rows past the range (unloaded blocks, slots past the
                    // sequence end) may hold anything: zero them in V so that
                    // 0 * garbage cannot reach O.
                    const int vt = tokE - (tok0 + t * kTcTok);
                    if (vt < kTcTok) {
                        const int s = t % vst;
                        // The parity wait for V(t) is unambiguous once the stage's
                        // previous fill, V(t - vst), has landed.  S(t) followed
                        // P.V(t - 2), so that holds for vst >= 2; a one-stage ring
                        // waits for P.V(t - 1) first.
                        if (vst == 1 && t > 0 &&
                            !__all_sync(0xffffffffu,
                                        mbar_wait_abortable(b_o_done + 8 * ((t - 1) & 1),
                                                            (uint32_t)((t - 1) >> 1) & 1u, abort_flag))) {
                            ok = false;
                            break;
                        }
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait_abortable(b_v_full + 8 * s, (uint32_t)(t / vst) & 1u,
                                                            abort_flag))) {
                            ok = false;
                            break;
                        }
                        const uint32_t vb = v_sm + (uint32_t)s * C::kKVBytes;
                        const int nchunks = (kTcTok - vt) * 8 * C::kSlices;
                        for (int idx = r - roff; idx < nchunks; idx += kTcRows - roff) {
                            const int sl = idx % C::kSlices;
                            const int rest = idx / C::kSlices;
                            st_shared_zero16(vb + sl * C::kKVSlice + (vt + rest / 8) * 128 + (rest & 7) * 16);
                        }
                        fence_proxy_async();
                    }
                }
                tc_fence_before();
                mbar_arrive(b_p_full + 8 * (t & 1));
            }
            // P.V(ntiles - 1), the last MMA; P.V(ntiles - 3) completed before
            // S(ntiles - 1), so the parity wait cannot be a phase early.
            if (ok && !__all_sync(0xffffffffu,
                                  mbar_wait_abortable(b_o_done + 8 * ((ntiles - 1) & 1),
                                                      (uint32_t)((ntiles - 1) >> 1) & 1u, abort_flag)))
                ok = false;
            if (!ok) {
                status_bits |= PA_STATUS_TIMEOUT;
                *abort_flag = 1;
            } else {
                tc_fence_after();
                // ---- epilogue: O / l for the row
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                if (V1) {
                    uint32_t *out = reinterpret_cast<uint32_t *>(static_cast<T *>(p.out) + qrow * D);
#pragma unroll 1
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_base + cc, o);
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
                        tmem_ld32(lane_base + cc, o);
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
    }

    if (status_bits)
        set_status(p.status, status_bits);
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kCols);
    }
}

// Kernel dispatch on block size, V1/V2, query tiles per CTA (two only for
// head_dim <= 128) and, for two tiles and bf16, whether V comes from the
// binary16 copy.
template <typename T, int D>
static const void *tc_kernel_ptr(int block_size, bool v1, int tiles, bool vh)
{
#define PA_PICK(K, BS)                                                                            \
    if (block_size == BS)                                                                         \
        return v1 ? reinterpret_cast<const void *>(&K<T, D, BS, true>)                            \
                  : reinterpret_cast<const void *>(&K<T, D, BS, false>);
#define PA_PICK_VH(BS)                                                                            \
    if (block_size == BS)                                                                         \
        return v1 ? reinterpret_cast<const void *>(&tc2_attn_kernel<T, D, BS, true, true>)        \
                  : reinterpret_cast<const void *>(&tc2_attn_kernel<T, D, BS, false, true>);
    if (tiles == 2) {
        if constexpr (D <= 128) {
            if (vh) {
                if constexpr (Elem<T>::kSplitP) {
                    PA_PICK_VH(8)
                    PA_PICK_VH(16)
                    PA_PICK_VH(32)
                    PA_PICK_VH(64)
                }
                return nullptr;
            }
            PA_PICK(tc2_attn_kernel, 8)
            PA_PICK(tc2_attn_kernel, 16)
            PA_PICK(tc2_attn_kernel, 32)
            PA_PICK(tc2_attn_kernel, 64)
        }
        return nullptr;
    }
#undef PA_PICK_VH
    PA_PICK(tc_attn_kernel, 8)
    PA_PICK(tc_attn_kernel, 16)
    PA_PICK(tc_attn_kernel, 32)
    PA_PICK(tc_attn_kernel, 64)
#undef PA_PICK
    return nullptr;
}

template <typename T, int D>
static cudaError_t tc_prepare(int block_size, bool v1, int tiles, bool vh, int optin_bytes,
                              size_t *limit)
{
    const void *fn = tc_kernel_ptr<T, D>(block_size, v1, tiles, vh);
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
static cudaError_t tc_launch(const AttnLaunch &L, cudaStream_t stream)
{
    const void *fn = tc_kernel_ptr<T, D>(L.block_size, L.v1, L.tc_tiles, L.vh);
    if (!fn)
        return cudaErrorInvalidValue;
    // The two-tile kernel also takes the binary16 copy's map (the V map when
    // there is no copy; it is then not read).
    const CUtensorMap *vh = L.vh ? &L.tmap_vh : &L.tmap_v;
    void *args1[] = {const_cast<CUtensorMap *>(&L.tmap_k), const_cast<CUtensorMap *>(&L.tmap_v),
                     const_cast<AttnParams *>(&L.p)};
    void *args2[] = {const_cast<CUtensorMap *>(&L.tmap_k), const_cast<CUtensorMap *>(&L.tmap_v),
                     const_cast<CUtensorMap *>(vh), const_cast<AttnParams *>(&L.p)};
    void **args = L.tc_tiles == 2 ? args2 : args1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = dim3(L.tc_tiles == 2 ? kTc2Threads : kTcThreads);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

#define PA_DEFINE_TC_OPS(T, NAME, D)                                                              \
    const TcOps *NAME()                                                                           \
    {                                                                                             \
        static const TcOps ops = {&tc_prepare<T, D>, &tc_launch<T, D>};                           \
        return &ops;                                                                              \
    }

} // namespace pa
