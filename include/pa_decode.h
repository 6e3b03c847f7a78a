/*
 * pa_decode.h -- C ABI of the split-K paged-attention decode library
 * (libpa_decode.so, CUDA for sm_103a).
 *
 * Operation (what every entry point computes)
 * -------------------------------------------
 * For each sequence b < num_seqs and query head h < num_heads, with
 * G = num_heads / num_kv_heads and KV head k = h / G (one KV head serves a
 * contiguous group of G query heads -- the GQA broadcast of the
 * "paged_attention_v2_pytorch.py" commit 15ef28e, "Key changes"):
 *
 *     K_t = key_cache  [block_tables[b][t / block_size], k, t % block_size, :]
 *     V_t = value_cache[block_tables[b][t / block_size], k, t % block_size, :]
 *     s_t = scale * <query[b, h, :], K_t>                  for t < seq_lens[b]
 *     out[b, h, :] = sum_t softmax(s)_t * V_t
 *
 * pa_decode_v2 computes it in the two passes of the pages' "V2"
 * ("paged_attention_v2_pytorch.py" commit 9cb7f9d, "Implementation"):
 *   phase 1, per (sequence, head, partition p of partition_size tokens):
 *       max_logits[b,h,p] = m_p = max_{t in p} s_t
 *       exp_sums  [b,h,p] = l_p = sum_{t in p} exp(s_t - m_p)
 *       tmp_output[b,h,p,:] = o_p = sum_{t in p} exp(s_t - m_p) V_t / l_p
 *   phase 2, per (sequence, head), the log-sum-exp merge:
 *       M = max_p m_p,  w_p = exp(m_p - M) * l_p,
 *       out[b,h,:] = sum_p (w_p / sum_q w_q) * o_p
 * over the ceil(seq_lens[b] / partition_size) partitions of sequence b.
 * pa_decode_v1 is the single-pass form (one CTA per (sequence, KV head)
 * walks every block with a running {m, l, o}; "vllm/_custom_ops.py" commit
 * 900ae0b, "V1: 1 CTA iterates ... partitions sequentially").  pa_decode
 * chooses between them ("paged_attn.py" commit 490ff98, change 1: restore
 * the V1/V2 adaptive dispatch), with a rule re-measured on this GPU (see
 * pa_decode_choose).
 *
 * Layouts (all row-major, contiguous, device memory)
 * --------------------------------------------------
 *   query        [num_seqs, num_heads, head_dim]                 dtype
 *   key_cache    [num_blocks, num_kv_heads, block_size, head_dim] dtype
 *   value_cache  [num_blocks, num_kv_heads, block_size, head_dim] dtype
 *   block_tables [num_seqs, max_blocks_per_seq]                  int32
 *                entries past ceil(seq_len / block_size) are never read
 *   seq_lens     [num_seqs]                                      int32
 *   out          [num_seqs, num_heads, head_dim]                 dtype
 *   tmp_output   [num_seqs, num_heads, max_num_partitions, head_dim] float32
 *   exp_sums     [num_seqs, num_heads, max_num_partitions]       float32
 *   max_logits   [num_seqs, num_heads, max_num_partitions]       float32
 *   dtype is PA_F16 (IEEE binary16) or PA_BF16 (bfloat16); arithmetic is
 *   fp32 throughout; out is rounded to dtype to nearest-even.
 *   Partition slots p >= ceil(seq_lens[b]/partition_size) are left untouched.
 *   A sequence with seq_len 0 gets a zero output row.
 *
 * Supported shapes: head_dim 64, 128 or 256; block_size 8, 16, 32 or 64;
 * partition_size any positive value (a partition may begin or end inside a
 * block; a block that straddles two partitions is read by both); G = num_heads /
 * num_kv_heads an integer in [1, 64]; q_len in [1, 4096] with num_seqs *
 * q_len <= 65535 (the _mq entry points).  Other shapes return
 * PA_ERR_UNSUPPORTED.  key_cache and value_cache must be 16-byte aligned
 * (they are read with the Tensor Memory Accelerator), tmp_output 16-byte
 * aligned, and query, out, block_tables, seq_lens, exp_sums, max_logits and
 * status 4-byte aligned; a misaligned pointer is PA_ERR_INVALID_ARG.
 *
 * Ownership, synchronisation, errors
 * ----------------------------------
 * Every pointer is owned and allocated by the caller; the library never
 * allocates, frees or synchronises.  Work is enqueued on `stream` (NULL is
 * the legacy default stream) and is asynchronous.  Arguments are validated
 * on the host before anything is enqueued: an invalid call returns a
 * non-zero PA_ERR_* code and launches nothing.  A launch failure returns
 * PA_ERR_CUDA.  Problems only the device can see are OR-ed as PA_STATUS_*
 * bits into *status (a device int32 the caller zeroes; may be NULL):
 *   PA_STATUS_BAD_BLOCK_ID  a needed block_tables entry is outside
 *                           [0, num_blocks); that block is read from
 *                           physical block 0 instead (the output is then
 *                           meaningless but no memory outside the caches
 *                           is touched);
 *   PA_STATUS_BAD_SEQ_LEN   seq_lens[b] < 0 or > max_blocks_per_seq *
 *                           block_size; the length is clamped into range;
 *   PA_STATUS_TIMEOUT       a bounded wait for a shared-memory copy gave up
 *                           (after about a second) instead of hanging.
 * The caller reads *status after synchronising the stream.
 * Entry points are thread-safe; the only global state is a per-device
 * cache of the multiprocessor count and of the kernels' shared-memory
 * opt-in, plus a small per-thread cache of encoded TMA descriptors keyed
 * by cache address and shape.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_API __attribute__((visibility("default")))

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *pa_stream_t;

enum { PA_F16 = 0, PA_BF16 = 1 };

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, inconsistent sizes */
    PA_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim, block_size, G) */
    PA_ERR_WORKSPACE = 3,   /* max_num_partitions too small for the sequences */
    PA_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
};

enum {
    PA_STATUS_BAD_BLOCK_ID = 1,
    PA_STATUS_BAD_SEQ_LEN = 2,
    PA_STATUS_TIMEOUT = 4
};

/*
 * Number of partitions ceil(max_seq_len / partition_size) that phase 1 uses
 * for the longest sequence ("vllm/_custom_ops.py" commit 900ae0b, change 1:
 * 100K tokens / 1024 = 98 partitions).  Returns -1 for invalid arguments.
 */
PA_API int pa_v2_num_partitions(int max_seq_len, int partition_size);

/*
 * Bytes of the three phase-1 intermediates (tmp_output, exp_sums,
 * max_logits) for the given capacity: num_seqs * num_heads *
 * max_num_partitions * (head_dim + 2) * 4.  The caller allocates them once
 * and reuses them ("paged_attn.py" commit 490ff98, change 2: pre-allocate
 * the V2 intermediates).  Returns 0 for invalid arguments.
 */
PA_API size_t pa_v2_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                    int max_num_partitions);

/*
 * Two-pass split-K decode (phase 1 then phase 2 on `stream`), see above.
 * max_seq_len_hint: if > 0, an upper bound of every seq_lens[b] known on the
 *   host; phase 1 then launches ceil(hint / partition_size) partitions per
 *   sequence.  If <= 0, ceil(max_blocks_per_seq * block_size /
 *   partition_size) are launched and the unused ones exit at once.  A
 *   sequence longer than the hint sets PA_STATUS_BAD_SEQ_LEN.
 * max_num_partitions: the partition capacity (third dimension) of
 *   tmp_output / exp_sums / max_logits; it must be >= the launched count,
 *   else PA_ERR_WORKSPACE.
 */
PA_API int pa_decode_v2(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                        int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                        int partition_size, int dtype, void *out, float *tmp_output,
                        float *exp_sums, float *max_logits, int max_num_partitions,
                        int32_t *status, pa_stream_t stream);

/*
 * Single-kernel V2: the same result as pa_decode_v2 (within the stated
 * tolerances; the merge sums in another order), with phase 2 done inside
 * the phase-1 grid.  Each CTA writes its partition's partials, then takes a
 * ticket from counters[b * num_kv_heads + k]; the CTA that takes the last
 * ticket of its (sequence b, KV head k) merges that group's partitions into
 * out -- the single-kernel alternative to the separate reduction pass that
 * "paged_attn.py" commit 490ff98 sets against CCCL's two-pass dispatch
 * ("Architecture follows CCCL's two-pass dispatch", "vllm/_custom_ops.py"
 * commit 900ae0b).  The merging CTA reads partitions in index order, so the
 * output does not depend on which CTA finishes last.
 *   counters  [num_seqs, num_kv_heads] int32, device memory owned by the
 *             caller, all zero before the first call; every call that
 *             completes leaves them zero again (each counter wraps to 0 on
 *             its last ticket), so one zeroing at allocation suffices.  Calls
 *             that overlap on the GPU must not share a counters array.
 * The other arguments are pa_decode_v2's; tmp_output, exp_sums and
 * max_logits hold the partials afterwards exactly as after pa_decode_v2.
 * Runs on the mma.sync kernel whatever the group size (no tcgen05 or SIMT
 * variant).  Measured against pa_decode_v2 on GB300 it is faster only when
 * the merge is trivial and the call latency-bound (one 1000-token sequence:
 * 10.4 vs 11.3 us) and slower otherwise, most of all with many partitions,
 * whose merge then runs on one CTA (one 100K-token sequence at 512 tokens
 * per partition: 97.5 vs 38.0 us); pa_decode never picks it.
 */
PA_API int pa_decode_v2_fused(const void *query, const void *key_cache, const void *value_cache,
                              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, int max_blocks_per_seq, int max_seq_len_hint,
                              float scale, int partition_size, int dtype, void *out,
                              float *tmp_output, float *exp_sums, float *max_logits,
                              int max_num_partitions, int32_t *counters, int32_t *status,
                              pa_stream_t stream);

/*
 * Phase 1 alone: writes tmp_output, exp_sums and max_logits for every
 * partition (same arguments as pa_decode_v2 without `out`).
 */
PA_API int pa_decode_v2_phase1(const void *query, const void *key_cache, const void *value_cache,
                               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                               int block_size, int max_blocks_per_seq, int max_seq_len_hint,
                               float scale, int partition_size, int dtype, float *tmp_output,
                               float *exp_sums, float *max_logits, int max_num_partitions,
                               int32_t *status, pa_stream_t stream);

/*
 * Phase 2 alone: the log-sum-exp merge of the partitions phase 1 wrote
 * (reads ceil(seq_lens[b] / partition_size) partitions of each (b, h)).
 */
PA_API int pa_decode_v2_phase2(const int32_t *seq_lens, int num_seqs, int num_heads,
                               int head_dim, int max_seq_len, int partition_size, int dtype,
                               const float *tmp_output, const float *exp_sums,
                               const float *max_logits, int max_num_partitions, void *out,
                               int32_t *status, pa_stream_t stream);

/*
 * Several new tokens per sequence (multi-query decode, e.g. checking q_len
 * speculated tokens at once).  The pages batch [kv_h, gqa, q_len, tile] in
 * the "paged_attn.py" commit 490ff98 online-softmax paragraph; the causal
 * mask they leave implicit is read as: new token i of sequence b sits at
 * position L - q_len + i, where L = seq_lens[b] already counts the q_len new
 * tokens, and attends to keys t <= L - q_len + i.  A new token that sees no
 * key (L - q_len + i < 0) gets a zero output row.
 *   query       [num_seqs, q_len, num_heads, head_dim]   dtype
 *   out         [num_seqs, q_len, num_heads, head_dim]   dtype
 *   tmp_output  [num_seqs, q_len, num_heads, max_num_partitions, head_dim]
 *   exp_sums, max_logits  [num_seqs, q_len, num_heads, max_num_partitions]
 * A partition holding none of the tokens a query sees is written as
 * max_logits = -inf, exp_sums = 0, tmp_output = 0 and adds nothing to the
 * merge.  The K/V cache is read once per call for all q_len * G query rows
 * of a KV head: up to 31 rows an mma.sync kernel serves 16 rows per CTA,
 * from 32 rows a tcgen05 kernel serves 128 rows per CTA (see
 * pa_set_rows_kernel); CTAs that split the rows of one range run side by
 * side, so their reads meet in L2.  Chunked prefill is this call with q_len
 * the chunk length, the chunk's own K/V already written to the cache (it
 * attends to the prefix and causally to itself).  q_len = 1 is
 * pa_decode_v2 / _v1.
 */
PA_API int pa_decode_v2_mq(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int num_blocks, int block_size, int max_blocks_per_seq,
                           int max_seq_len_hint, float scale, int partition_size, int dtype,
                           void *out, float *tmp_output, float *exp_sums, float *max_logits,
                           int max_num_partitions, int32_t *status, pa_stream_t stream);

PA_API int pa_decode_v1_mq(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int num_blocks, int block_size, int max_blocks_per_seq,
                           int max_seq_len_hint, float scale, int dtype, void *out,
                           int32_t *status, pa_stream_t stream);

/*
 * Which variant pa_decode_mq runs for q_len new tokens per sequence on the
 * current device: returns 1 (V1) or 2 (V2), or a negative PA_ERR_* code.
 * Host only.  With R = q_len * G query rows per KV head:
 *   - one partition covers max_seq_len: V1;
 *   - R < 32 (the mma.sync kernel): V2, for q_len >= 2 at the partition
 *     size pa_decode_mq_partition returns (1024 tokens unless
 *     partition_size is larger or the grid would leave SMs idle; V1 when
 *     that partition covers max_seq_len), for q_len = 1 at partition_size;
 *   - R >= 32 (the tcgen05 kernels) and few (sequence, KV head, row tile)
 *     groups, at most half the CTAs resident at once: V2 on partitions
 *     sized so that the longest sequence's CTAs make one wave (a multiple
 *     of 64 tokens, at least partition_size), V1 if one partition covers it;
 *   - otherwise 32 <= R <= 128 (one query tile): V2 at the partition size
 *     pa_decode_mq_partition returns (2048 tokens unless partition_size is
 *     larger, or the grid would leave SMs idle), or V1 when that partition
 *     covers max_seq_len;
 *   - otherwise R > 128 (chunked prefill): V1 when the V1 grid (num_seqs *
 *     num_kv_heads CTAs per 128-row tile) gives every SM a CTA -- or, for
 *     sequences of 8192 tokens and more, V2 on two partitions when V1's
 *     waves of CTAs would leave more than a tenth of the resident slots
 *     idle and two partitions pack them better -- else V2.
 * There is no counterpart in the method's description, which dispatches
 * single-token decode only; the rule is measured on GB300.
 */
PA_API int pa_decode_mq_choose(int num_seqs, int q_len, int num_heads, int num_kv_heads,
                               int head_dim, int max_seq_len, int partition_size);

/*
 * The partition size pa_decode_mq runs V2 with for these sizes: at least
 * partition_size (the intermediates sized for partition_size therefore
 * always suffice), or 0 when it runs V1.  Negative PA_ERR_* code for invalid arguments.  Host
 * only.  No counterpart in the method's description.
 */
PA_API int pa_decode_mq_partition(int num_seqs, int q_len, int num_heads, int num_kv_heads,
                                  int head_dim, int max_seq_len, int partition_size);

/*
 * pa_decode_v2_mq or pa_decode_v1_mq, as pa_decode_mq_choose picks (the
 * capacity max_seq_len_hint if > 0, else max_blocks_per_seq * block_size, is
 * its max_seq_len), V2 at the partition size pa_decode_mq_partition returns.
 * The V2 intermediates, sized for partition_size, must be valid whenever V2
 * can be chosen; after a V2 call they hold the partials of that (possibly
 * coarser) partitioning -- at a stride of max_num_partitions, except in the
 * case below.
 *
 * bf16 caches whose rows would take the two-tile tcgen05 kernel under
 * fp16's rule (R > 128, head_dim <= 128, max_seq_len >= 1024), with R >=
 * 1024 (any R and length with pa_set_rows_kernel(4); never with modes 1, 3
 * and 6): tmp_output, when large enough, also holds a binary16 copy of the
 * V blocks the call reads, and P.V runs on binary16 P and V (one MMA per
 * K-step where bf16 needs a hi + lo pair of P halves).  Below 1024 rows per
 * KV head the copy's extra read and write of V outweighs what it saves.
 * Layout, in bytes from tmp_output (num_seqs * q_len * num_heads *
 * max_num_partitions * head_dim * 4 bytes in all): the partials at a stride
 * of the partitions used (np, 0 for V1), num_seqs * q_len * num_heads * np *
 * head_dim * 4 bytes; at the next multiple of 256, num_seqs 32-bit block
 * offsets, offs[s] = the sum of ceil(L_t / block_size) over t < s with L_t
 * clamped to the capacity, and a 32-bit flag after them; at the next
 * multiple of 256 after the flag the copy, [num_kv_heads][copy_blocks]
 * [block_size][head_dim] binary16, copy_blocks as many as the rest of
 * tmp_output holds (at most 2^31 rows in all): a sequence's logical block j
 * at index offs[s] + j of each KV head's part, rows past its end zero, an
 * out-of-range block id read as block 0.  The flag is set to 1 when the
 * sequences' blocks do not fit copy_blocks (the lengths are device data) or
 * a finite value of magnitude 2^16 or more was met (binary16 cannot hold
 * it): the call then reads the bf16 cache with P in hi + lo halves instead
 * (the attention kernel reads the flag once the copy pass has completed and
 * takes its bf16 form, still on two tiles).  Every bf16 value
 * below 2^16 has an exact binary16 form, so the copy loses nothing.  When
 * tmp_output cannot hold the offsets, the flag and one block, there is no
 * copy and the call runs the one-tile kernel with hi + lo P.  The copy adds
 * one read and one write of the V blocks' bytes to the call.
 */
PA_API int pa_decode_mq(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int q_len, int num_heads, int num_kv_heads, int head_dim,
                        int num_blocks, int block_size, int max_blocks_per_seq,
                        int max_seq_len_hint, float scale, int partition_size, int dtype,
                        void *out, float *tmp_output, float *exp_sums, float *max_logits,
                        int max_num_partitions, int32_t *status, pa_stream_t stream);

/*
 * Single-pass decode: one CTA per (sequence, KV head) walks all blocks with
 * a running {m, l, o} and writes `out` directly.  No intermediates.
 */
PA_API int pa_decode_v1(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                        int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                        int dtype, void *out, int32_t *status, pa_stream_t stream);

/*
 * Which variant pa_decode runs for these sizes on the current device:
 * returns 1 (V1) or 2 (V2), or a negative PA_ERR_* code.  Host only.
 * The rule, measured on GB300 ("paged_attn.py" commit 490ff98, change 1,
 * restores a V1/V2 dispatch; its 8192-token switch point was set on other
 * hardware): with NP = ceil(max_seq_len / partition_size),
 *   V1 if NP <= 1 (a merge of one partition would only copy), or if NP == 2
 *      and num_seqs * num_kv_heads (V1's CTAs) is at most the number of SMs
 *      (a latency-bound call, where the merge's second launch costs more
 *      than splitting each sequence in two);
 *   V2 otherwise.
 */
PA_API int pa_decode_choose(int num_seqs, int num_kv_heads, int max_seq_len, int partition_size);

/*
 * V1/V2 dispatch: runs pa_decode_v1 or pa_decode_v2 as pa_decode_choose
 * says for (num_seqs, num_kv_heads, L, partition_size), where L is
 * max_seq_len_hint if > 0, else max_blocks_per_seq * block_size.  The V2
 * intermediates must be valid whenever V2 can be chosen.
 */
PA_API int pa_decode(const void *query, const void *key_cache, const void *value_cache,
                     const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                     int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                     int partition_size, int dtype, void *out, float *tmp_output,
                     float *exp_sums, float *max_logits, int max_num_partitions,
                     int32_t *status, pa_stream_t stream);

/*
 * Launch-shape override for the attention kernels, process-wide: warps per
 * CTA (1..8) and TMA ring stages per warp (1..8); 0 keeps the built-in
 * choice for that field.  The override never changes results, only speed.
 * Returns PA_ERR_INVALID_ARG for out-of-range values.
 */
PA_API int pa_set_launch_config(int warps_per_cta, int stages_per_warp);

/*
 * Kernel choice for the query rows of a KV head (rows = q_len * G),
 * process-wide: 0 (default) picks by row count -- up to 31 rows the
 * mma.sync kernel (16 rows per CTA), from 32 rows a tcgen05 kernel (128-row
 * query tiles, S and O accumulated in tensor memory; two tiles sharing each
 * K/V tile per CTA for fp16 when a KV head has more than 128 rows, head_dim
 * <= 128 and sequences reach 1024 tokens, else one tile and two CTAs per
 * SM); 1 always the mma.sync kernel; 2 always a tcgen05 kernel; 3 always
 * the one-tile tcgen05 kernel; 4 always the two-tile one (one tile for
 * head_dim 256); 5 the CUDA-core kernel (Q.K and the softmax reduced with
 * warp shuffles, P.V as scalar FMAs, no tensor-core instruction) up to 8
 * rows, else as 0; 6 always the one-tile tcgen05 kernel with its whole
 * 128-row Q tile stored (by default a KV head of at most 64 rows stores only
 * the 64 rows it uses and spends the space on a deeper ring).  Either kernel
 * computes the same
 * result within the stated tolerances; the choice changes only speed.  The
 * tcgen05 kernel takes its K ring stages from pa_set_launch_config's
 * stages_per_warp and its V ring stages from warps_per_cta when those are
 * set.  Returns PA_ERR_INVALID_ARG for other
 * values.  There is no counterpart in the method's description: this is a
 * tuning and test hook.
 */
PA_API int pa_set_rows_kernel(int mode);

/*
 * Form of phase 2 (the merge), process-wide: 0 (default) by rule -- one warp
 * per (row, head) when there are more than 16 (row, head) pairs per SM and
 * the longest sequence has at most 8 partitions, or at most 32 with 32 pairs
 * per SM or more; else one CTA per (head, row, slice of head_dim); 1 always
 * the CTA-per-slice form; 2 always the
 * warp-per-pair form (up to 2^30 pairs, else the CTA form).  Both fold the
 * partitions with the same rule; the choice changes only speed.  Returns
 * PA_ERR_INVALID_ARG for other values.  A tuning and test hook, with no
 * counterpart in the method's description.
 */
PA_API int pa_set_merge_form(int form);

/*
 * Size of the intermediates array that pa_decode_v2_static keeps inside the
 * library: 16 MiB of device memory on every GPU that loads the library,
 * held until the process exits.
 */
#define PA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * pa_decode_v2 for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for callers that must
 * not or cannot call cudaMalloc -- code inside a host framework that owns
 * every device allocation, runtimes handed a fixed memory budget up front,
 * or hot paths where an allocation (and the implicit device synchronisation
 * it brings) is not allowed.  The caller passes only inputs and outputs,
 * with the same meaning as in pa_decode_v2; tmp_output, exp_sums and
 * max_logits live in a PA_STATIC_SCRATCH_BYTES array owned by the library.
 * Nothing is allocated or freed by this call.
 *   - Limit: num_seqs * num_heads * ceil(L / partition_size) *
 *     (head_dim + 2) * 4 bytes must fit in PA_STATIC_SCRATCH_BYTES, where L
 *     is max_seq_len_hint if > 0, else max_blocks_per_seq * block_size.
 *     Larger calls return PA_ERR_WORKSPACE and launch nothing.
 *   - Set-up: the first call on a device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture.  The address is kept for the
 *     life of the process, so do not call this entry point on a device
 *     after cudaDeviceReset on it (the reset unloads the array and the kept
 *     address goes stale).
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents.  No slot needs clearing (each slot the merge
 *     reads is written earlier in the same call), but two calls that
 *     overlap on the GPU (different streams, or different host threads)
 *     race on the array and corrupt each other's results: keep such calls
 *     ordered on one stream.
 */
PA_API int pa_decode_v2_static(const void *query, const void *key_cache, const void *value_cache,
                               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                               int block_size, int max_blocks_per_seq, int max_seq_len_hint,
                               float scale, int partition_size, int dtype, void *out,
                               int32_t *status, pa_stream_t stream);

/* Human-readable name of a PA_* return code (static string). */
PA_API const char *pa_status_string(int code);

/*
 * Self-test of the bounded-wait path used by every kernel above: launches
 * one warp that waits on a shared-memory barrier nothing ever completes,
 * for at most limit_ns nanoseconds, then ORs PA_STATUS_TIMEOUT into
 * *status and returns.  Shows that a stuck copy turns into an error status
 * instead of a hung GPU.  limit_ns must be in (0, 2e9].
 */
PA_API int pa_selftest_wait_timeout(int32_t *status, long long limit_ns, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
