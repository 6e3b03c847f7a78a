// pa_api.cu -- the C ABI declared in include/pa_decode.h: host-side
// validation, TMA descriptor encoding, launch sizing, V1/V2 dispatch.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_decode.h"
#include "pa_internal.h"

using namespace pa;

namespace {

constexpr int kMaxDevices = 64;

// A binary16 copy of the V blocks of one multi-query call (bf16 caches) and
// the flag word that says whether it holds every value exactly.
struct VhCopy {
    void *copy;
    int32_t *flag;
    const int32_t *offs;         // each sequence's first block in the packed copy
    int copy_blocks;             // blocks the copy's space holds
};

std::atomic<int> g_tune_warps{0};
std::atomic<int> g_tune_stages{0};
// Kernel for the query rows of a KV head: 0 = by row count, 1 = always the
// mma.sync kernel, 2 = always a tcgen05 kernel (query tiles by row count),
// 3 = the one-tile tcgen05 kernel, 4 = the two-tile one (head_dim <= 128),
// 5 = the CUDA-core (SIMT) kernel up to 8 rows, else as 0, 6 = the one-tile
// tcgen05 kernel with the whole 128-row Q tile stored at every row count.
std::atomic<int> g_rows_kernel{0};
// Phase-2 form: 0 = by rule, 1 = a CTA per (head, row, slice of head_dim),
// 2 = a warp per (row, head).
std::atomic<int> g_merge_form{0};
// From this many query rows per KV head (q_len * G) up, the tcgen05 kernel
// (128 rows per CTA) runs instead of the mma.sync one (up to 16 per CTA).
// Measured on GB300 (best of V1 / V2 per kernel, mma.sync vs tcgen05):
// 16 rows 99 vs 155 us; 32 rows: batch decode 152 vs 151, fp16 138 vs 140,
// a 100K-token sequence 64.5 vs 54.8; 48 rows 211 vs 161; 64 rows 291 vs 157.
constexpr int kTcMinRows = 32;

// Per-device cached multiprocessor count (0 = not queried yet).
std::atomic<int> g_sm_count[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

int current_device(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices)
        return PA_ERR_CUDA;
    return PA_OK;
}

int sm_count(int dev)
{
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return -1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by every attention entry point.  No CUDA call.
int check_shape(const void *query, const void *key_cache, const void *value_cache,
                const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_heads,
                int num_kv_heads, int head_dim, int num_blocks, int block_size,
                int max_blocks_per_seq, float scale, int dtype)
{
    if (!query || !key_cache || !value_cache || !block_tables || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64)
        return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > kMaxGQA)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    // TMA row coordinates and token indices are 32-bit.
    if ((int64_t)num_blocks * num_kv_heads * block_size > INT32_MAX ||
        (int64_t)max_blocks_per_seq * block_size > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(query, 4) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int seq_cap(int max_blocks_per_seq, int block_size, int hint)
{
    const int full = max_blocks_per_seq * block_size;
    return (hint > 0 && hint < full) ? hint : full;
}

// 3-D view of a cache for the TMA: dims {64 (a slice of head_dim), head_dim / 64
// (slices), rows = num_blocks * KV * block_size}, 128-byte swizzle, box
// {64, 1, block_size}: one load brings one 64-dim slice of a block's tile.
int encode_cache_map_uncached(CUtensorMap *map, const void *base, int dtype, int num_blocks,
                              int num_kv_heads, int block_size, int head_dim)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn)
        return PA_ERR_CUDA;
    const cuuint64_t rows = (cuuint64_t)num_blocks * num_kv_heads * block_size;
    const cuuint64_t dims[3] = {64, (cuuint64_t)head_dim / 64, rows};
    const cuuint64_t strides[2] = {128, (cuuint64_t)head_dim * 2}; // bytes of dim 1 and dim 2
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)block_size};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Small per-thread cache of encoded descriptors: a decode loop calls with the
// same caches every step, so encoding happens once per (cache, shape).
struct MapCacheEntry {
    CUtensorMap map;
    const void *base;
    int dtype, num_blocks, num_kv_heads, block_size, head_dim;
    bool valid;
};
constexpr int kMapCacheSize = 8;
thread_local MapCacheEntry t_map_cache[kMapCacheSize];
thread_local int t_map_next = 0;

int encode_cache_map(CUtensorMap *map, const void *base, int dtype, int num_blocks,
                     int num_kv_heads, int block_size, int head_dim)
{
    for (int i = 0; i < kMapCacheSize; ++i) {
        const MapCacheEntry &e = t_map_cache[i];
        if (e.valid && e.base == base && e.dtype == dtype && e.num_blocks == num_blocks &&
            e.num_kv_heads == num_kv_heads && e.block_size == block_size &&
            e.head_dim == head_dim) {
            *map = e.map;
            return PA_OK;
        }
    }
    int rc = encode_cache_map_uncached(map, base, dtype, num_blocks, num_kv_heads, block_size,
                                       head_dim);
    if (rc)
        return rc;
    MapCacheEntry &e = t_map_cache[t_map_next];
    t_map_next = (t_map_next + 1) % kMapCacheSize;
    e.map = *map;
    e.base = base;
    e.dtype = dtype;
    e.num_blocks = num_blocks;
    e.num_kv_heads = num_kv_heads;
    e.block_size = block_size;
    e.head_dim = head_dim;
    e.valid = true;
    return PA_OK;
}

// Index of a kernel instantiation: storage type x head_dim x block size x
// row variant (mma.sync with one or two n-tiles, or the SIMT kernel padded
// to 1, 2, 4 or 8 rows) x V2 / V1 / fused V2.
constexpr int kKernelSlots = 2 * 3 * 4 * 6 * 3;

int kernel_slot(const AttnLaunch &L)
{
    const int di = L.head_dim == 64 ? 0 : L.head_dim == 128 ? 1 : 2;
    const int bi = L.block_size == 8 ? 3 : L.block_size == 16 ? 0 : L.block_size == 32 ? 1 : 2;
    const int c = L.cta_cols;
    const int vi = L.simt ? (c <= 1 ? 2 : c <= 2 ? 3 : c <= 4 ? 4 : 5) : (c > 8 ? 1 : 0);
    return ((((L.dtype == PA_BF16 ? 1 : 0) * 3 + di) * 4 + bi) * 6 + vi) * 3 + attn_variant(L);
}

// The kernel table of a launch: the SIMT or the mma.sync kernels.
const AttnOps *ops_of(const AttnLaunch &L)
{
    return L.simt ? simt_ops(L.dtype, L.head_dim) : attn_ops(L.dtype, L.head_dim);
}

// Per-device, per-kernel dynamic shared memory limit after the opt-in (0 = not yet).
std::atomic<int> g_smem_limit[kMaxDevices][kKernelSlots];
// Per-device resident CTAs per SM by [kernel][warps][stages], stored + 1 (0 = not queried).
std::atomic<int> g_occ[kMaxDevices][kKernelSlots][kMaxWarps + 1][kMaxStages + 1];

// Opts the kernel in to the device's largest dynamic shared memory (once per
// device) and returns that limit, or 0 on error.
size_t smem_limit(int dev, const AttnLaunch &L)
{
    const int slot = kernel_slot(L);
    const int have = g_smem_limit[dev][slot].load(std::memory_order_acquire);
    if (have > 0)
        return (size_t)have;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    size_t limit = 0;
    cudaError_t e = ops_of(L)->prepare(L.block_size, L.cta_cols, attn_variant(L), optin, &limit);
    if (e != cudaSuccess)
        return 0;
    g_smem_limit[dev][slot].store((int)limit, std::memory_order_release);
    return limit;
}

size_t attn_smem(const AttnLaunch &L, int warps, int stages)
{
    return 1024 + (size_t)warps * stages * stage_bytes(L.block_size, L.head_dim);
}

int occupancy(int dev, const AttnLaunch &L, int warps, int stages, size_t limit)
{
    const size_t smem = attn_smem(L, warps, stages);
    if (smem > limit || warps < 1 || warps > kMaxWarps || stages < 1 || stages > kMaxStages)
        return 0;
    const int slot = kernel_slot(L);
    const int c = g_occ[dev][slot][warps][stages].load(std::memory_order_relaxed);
    if (c)
        return c - 1;
    const int n = ops_of(L)->occupancy(L.block_size, L.cta_cols, attn_variant(L), warps, smem);
    g_occ[dev][slot][warps][stages].store(n + 1, std::memory_order_relaxed);
    return n;
}

// Launch shape of the attention kernel, from a warps x stages sweep on
// GB300.  Phase 1 aims at about 64 KB of ring per CTA (three CTAs per SM)
// with 4 warps when a stage is small enough: two stages per warp (one block
// computing, one landing) for stages up to 8 KB (16-token blocks of 128
// dims), one stage beyond (a larger stage would otherwise cut the CTAs per
// SM), and fewer warps for 32 KB and 64 KB stages.  When the grid would take
// a few waves at that size but fits one wave with narrower CTAs, the
// narrower CTAs win (no wave tail).  V1 has only num_seqs * num_kv_heads
// CTAs, so it takes the widest CTA that fits about 200 KB with two stages.
void size_attn(AttnLaunch &L, int dev, int sms, size_t limit)
{
    const int tune_w = g_tune_warps.load(std::memory_order_relaxed);
    const int tune_s = g_tune_stages.load(std::memory_order_relaxed);
    const size_t sb = stage_bytes(L.block_size, L.head_dim);
    const size_t scratch = warp_scratch_bytes(L.cta_cols, L.head_dim);
    auto clampi = [](long long v, int lo, int hi) { return (int)(v < lo ? lo : v > hi ? hi : v); };
    const int w_fit = clampi((long long)(65536 / sb), 1, 4);
    int stages = tune_s > 0 ? tune_s : (L.v1 ? 2 : clampi((long long)(65536 / (w_fit * sb)), 1, 2));
    while ((size_t)stages * sb < scratch)
        ++stages;
    int warps;
    if (tune_w > 0) {
        warps = tune_w;
    } else if (L.v1) {
        warps = clampi((long long)(200 * 1024 / (2 * sb)), 1, kMaxWarps);
    } else {
        const int w0 = w_fit;
        warps = w0;
        const long long ctas = (long long)L.grid.x * L.grid.y * L.grid.z;
        const long long occ0 = occupancy(dev, L, w0, stages, limit);
        if (occ0 > 0 && ctas > occ0 * sms && ctas <= 3 * occ0 * sms) {
            for (int w1 = w0 / 2; w1 >= 1; w1 /= 2) {
                if (ctas <= (long long)occupancy(dev, L, w1, stages, limit) * sms) {
                    warps = w1;
                    break;
                }
            }
        }
    }
    // Phase-1 kernels for 16 query rows of up to 128 dims are compiled for at
    // most 4 warps (three CTAs per SM).
    if (!L.v1 && L.cta_cols > 8 && L.head_dim <= 128 && warps > 4)
        warps = 4;
    while (attn_smem(L, warps, stages) > limit && stages > 1 && (size_t)(stages - 1) * sb >= scratch)
        --stages;
    while (attn_smem(L, warps, stages) > limit && warps > 1)
        --warps;
    L.warps = warps;
    L.p.stages = stages;
    L.smem_bytes = attn_smem(L, warps, stages);
}

// Per-device dynamic shared memory limit of each tcgen05 kernel after the opt-in.
constexpr int kTcSlots = 2 * 3 * 4 * 2 * 2 * 2;
std::atomic<int> g_tc_smem_limit[kMaxDevices][kTcSlots];

int tc_slot(int dtype, int head_dim, int block_size, bool v1, int tiles, bool vh)
{
    const int di = head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2;
    const int bi = block_size == 8 ? 3 : block_size == 16 ? 0 : block_size == 32 ? 1 : 2;
    return (((((dtype == PA_BF16 ? 1 : 0) * 3 + di) * 4 + bi) * 2 + (v1 ? 1 : 0)) * 2 +
            (tiles - 1)) * 2 + (vh ? 1 : 0);
}

// The tcgen05 kernels.  One query tile: as many K and V ring stages as keep
// two CTAs per SM for head_dim <= 128 (one for 256 dims, whose TMEM takes
// the whole SM): 2 + 2 stages of 64 tokens at head_dim 128, 4 + 4 at 64.  A
// KV head of at most 64 rows stores only the 64 Q rows it uses (half Q
// tile), and at head_dim 128 the 16 KB saved hold a third V stage.  Two
// query tiles (one CTA per SM, all 512 TMEM columns): 2 + 2 stages of 128
// tokens at head_dim 128, 4 + 4 at 64.  pa_set_launch_config's
// stages_per_warp overrides the K stages and its warps_per_cta the V
// stages.
int prepare_and_launch_tc(AttnLaunch &L, int dev, cudaStream_t stream)
{
    const int tiles = L.tc_tiles;
    const int slot = tc_slot(L.dtype, L.head_dim, L.block_size, L.v1, tiles, L.vh);
    size_t limit = (size_t)g_tc_smem_limit[dev][slot].load(std::memory_order_acquire);
    if (limit == 0) {
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        if (tc_ops(L.dtype, L.head_dim)->prepare(L.block_size, L.v1, tiles, L.vh, optin, &limit) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        g_tc_smem_limit[dev][slot].store((int)limit, std::memory_order_release);
    }
    const bool q_half = L.p.q_half != 0;
    auto bytes = [&](int ks, int vs) {
        return tiles == 2 ? tc2_smem_bytes(L.head_dim, ks, vs)
                          : tc_smem_bytes(L.head_dim, ks, vs, q_half);
    };
    const int tune_s = g_tune_stages.load(std::memory_order_relaxed);
    const int tune_w = g_tune_warps.load(std::memory_order_relaxed);
    int ks = L.head_dim == 64 ? 4 : 2, vs = ks;
    if (q_half && L.head_dim == 128)
        vs = 3;
    if (tune_s > 0)
        ks = tune_s;
    if (tune_w > 0)
        vs = tune_w;
    while (bytes(ks, vs) > limit && (ks > 1 || vs > 1)) {
        if (ks >= vs)
            --ks;
        else
            --vs;
    }
    if (bytes(ks, vs) > limit)
        return PA_ERR_UNSUPPORTED;
    L.p.stages = ks;
    L.p.v_stages = vs;
    L.warps = (tiles == 2 ? kTc2Threads : kTcThreads) / 32;
    L.smem_bytes = bytes(ks, vs);
    return tc_ops(L.dtype, L.head_dim)->launch(L, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int prepare_and_launch_attn(AttnLaunch &L, cudaStream_t stream)
{
    int dev;
    if (current_device(&dev))
        return PA_ERR_CUDA;
    if (L.tc)
        return prepare_and_launch_tc(L, dev, stream);
    const int sms = sm_count(dev);
    if (sms <= 0)
        return PA_ERR_CUDA;
    const size_t limit = smem_limit(dev, L);
    if (limit == 0)
        return PA_ERR_CUDA;
    size_attn(L, dev, sms, limit);
    if (L.smem_bytes > limit)
        return PA_ERR_UNSUPPORTED;
    cudaError_t e = ops_of(L)->launch(L, stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Whether the query rows of a KV head (q_len * G of them) go to a tcgen05 kernel.
bool use_tc(int cols)
{
    const int mode = g_rows_kernel.load(std::memory_order_relaxed);
    if ((mode >= 2 && mode <= 4) || mode == 6)
        return true;
    return (mode == 0 || mode == 5) && cols >= kTcMinRows;
}

// 128-row query tiles per CTA of the tcgen05 kernel.  Two tiles (one CTA per
// SM, two tiles' O and S in the SM's 512 TMEM columns, each K/V tile shared)
// need head_dim <= 128.  By default they are taken for fp16 when a KV head
// has more than 128 rows and sequences reach 1024 tokens; bf16, whose split
// P doubles the P.V work, and short sequences run faster with one tile and
// two CTAs per SM.  (The multi-query dispatch gives bf16 the fp16 rule when it
// can make a binary16 copy of V: pa_decode_mq.)  Measured on GB300 (V1, one vs two tiles): chunked prefill
// (2 x 2048 new tokens after 30K) bf16 2384 vs 2495 us, fp16 2137 vs 1903;
// 4 x 1024 new after 3072 bf16 323 vs 351, fp16 296 vs 282; 8 x 512 new
// tokens, no prefix, fp16 75 vs 87.
int tc_tiles(int cols, int head_dim, int dtype, int max_seq_len)
{
    const int mode = g_rows_kernel.load(std::memory_order_relaxed);
    if (head_dim > 128 || mode == 3 || mode == 6)
        return 1;
    if (mode == 4)
        return 2;
    return (dtype == PA_F16 && cols > kTcRows && max_seq_len >= 1024) ? 2 : 1;
}

// CTAs that split the query rows of one KV head and range.
int row_ctas(int cols, int head_dim, int dtype, int max_seq_len)
{
    if (use_tc(cols)) {
        const int rows = kTcRows * tc_tiles(cols, head_dim, dtype, max_seq_len);
        return (cols + rows - 1) / rows;
    }
    return cols <= 8 ? 1 : (cols + kMaxGroup - 1) / kMaxGroup;
}

// Builds the attention launch (V2 phase 1 or V1) after validation.
int build_attn(AttnLaunch &L, const void *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int q_len,
               int num_heads,
               int num_kv_heads, int head_dim, int num_blocks, int block_size,
               int max_blocks_per_seq, int cap, float scale, int dtype, bool v1,
               int num_partitions, int partition_size,
               float *tmp_output, float *exp_sums, float *max_logits, int max_num_partitions,
               void *out, int32_t *status, int32_t *counters = nullptr,
               const VhCopy *vh = nullptr)
{
    L = AttnLaunch{};
    // The fused V2 (counters given) runs on the mma.sync kernel at any row count.
    const bool fused = counters != nullptr;
    int rc = encode_cache_map(&L.tmap_k, key_cache, dtype, num_blocks, num_kv_heads, block_size,
                              head_dim);
    if (rc)
        return rc;
    rc = encode_cache_map(&L.tmap_v, value_cache, dtype, num_blocks, num_kv_heads, block_size,
                          head_dim);
    if (rc)
        return rc;
    if (vh) {
        // The copy is [KV][copy_blocks][block_size][head_dim] binary16: as rows,
        // the cache map's shape with copy_blocks blocks.
        rc = encode_cache_map(&L.tmap_vh, vh->copy, PA_F16, vh->copy_blocks, num_kv_heads,
                              block_size, head_dim);
        if (rc)
            return rc;
        L.p.vh_offs = vh->offs;
        L.p.vh_blocks = vh->copy_blocks;
        L.p.vh_flag = vh->flag;
    }
    // With the binary16 copy, bf16 rows take the kernel fp16's would.
    const int tile_dtype = vh ? PA_F16 : dtype;
    AttnParams &p = L.p;
    p.query = query;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_heads / num_kv_heads;
    p.q_len = q_len;
    p.cols = p.group * q_len;
    L.tc = !fused && use_tc(p.cols);
    if (L.tc) {
        // 128 rows per query tile; the CTAs of one range split the rows.
        L.cta_cols = kMaxGroup;
        L.tc_tiles = tc_tiles(p.cols, head_dim, tile_dtype, cap);
        // At most 64 rows on one tile: only Q rows 64-127 are stored.
        p.q_half = (L.tc_tiles == 1 && p.cols <= kTcRows / 2 &&
                    g_rows_kernel.load(std::memory_order_relaxed) != 6)
                       ? 1
                       : 0;
        p.col_groups = row_ctas(p.cols, head_dim, tile_dtype, cap);
    } else {
        // Up to 8 query rows: one n-tile (or the SIMT kernel when asked for);
        // more: 16 per CTA, split over CTAs.
        L.cta_cols = p.cols <= 8 ? p.cols : kMaxGroup;
        p.col_groups = (p.cols + L.cta_cols - 1) / L.cta_cols;
        L.simt = !fused && p.cols <= 8 && g_rows_kernel.load(std::memory_order_relaxed) == 5;
    }
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.seq_len_cap = cap;
    p.scale = scale;
    p.partition_size = v1 ? 0 : partition_size;
    p.max_num_partitions = max_num_partitions;
    p.tmp_output = tmp_output;
    p.exp_sums = exp_sums;
    p.max_logits = max_logits;
    p.out = out;
    p.counters = counters;
    p.status = status;
    L.fused = fused;
    L.vh = vh && L.tc && L.tc_tiles == 2 && dtype == PA_BF16;
    L.head_dim = head_dim;
    L.block_size = block_size;
    L.dtype = dtype;
    L.v1 = v1;
    // Column groups of one partition are adjacent in x, so they are scheduled
    // together and their K/V reads meet in L2.
    L.grid = dim3((unsigned)(v1 ? 1 : num_partitions) * p.col_groups, num_kv_heads, num_seqs);
    return PA_OK;
}

int check_q_len(int num_seqs, int q_len)
{
    if (q_len < 1)
        return PA_ERR_INVALID_ARG;
    if (q_len > kMaxQLen || (long long)num_seqs * q_len > 65535)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

int v2_phase1_impl(const void *query, const void *key_cache, const void *value_cache,
                   const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int q_len,
                   int num_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
                   int max_blocks_per_seq, int max_seq_len_hint, float scale, int partition_size,
                   int dtype, float *tmp_output, float *exp_sums, float *max_logits,
                   int max_num_partitions, int32_t *status, cudaStream_t stream, int *cap_out,
                   void *fused_out = nullptr, int32_t *counters = nullptr,
                   const VhCopy *vh = nullptr)
{
    int rc = check_shape(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, scale, dtype);
    if (rc)
        return rc;
    rc = check_q_len(num_seqs, q_len);
    if (rc)
        return rc;
    if (partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (!tmp_output || !exp_sums || !max_logits || max_num_partitions <= 0)
        return PA_ERR_INVALID_ARG;
    if (!aligned(tmp_output, 16) || !aligned(exp_sums, 4) || !aligned(max_logits, 4) ||
        (status && !aligned(status, 4)))
        return PA_ERR_INVALID_ARG;
    const int cap = seq_cap(max_blocks_per_seq, block_size, max_seq_len_hint);
    const int np = pa_v2_num_partitions(cap, partition_size);
    if (np > max_num_partitions)
        return PA_ERR_WORKSPACE;
    if (cap_out)
        *cap_out = cap;
    if (np == 0)
        return PA_OK;
    AttnLaunch L;
    rc = build_attn(L, query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                    num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                    cap, scale, dtype, false, np, partition_size, tmp_output, exp_sums, max_logits,
                    max_num_partitions, fused_out, status, counters, vh);
    if (rc)
        return rc;
    return prepare_and_launch_attn(L, stream);
}

int v2_phase2_impl(const int32_t *seq_lens, int num_seqs, int q_len, int num_heads, int head_dim,
                   int max_seq_len, int partition_size, int dtype, const float *tmp_output,
                   const float *exp_sums, const float *max_logits, int max_num_partitions,
                   void *out, int32_t *status, cudaStream_t stream)
{
    if (!seq_lens || !tmp_output || !exp_sums || !max_logits || !out)
        return PA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
        partition_size <= 0 || max_num_partitions <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return PA_ERR_UNSUPPORTED;
    if (num_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    const int qrc = check_q_len(num_seqs, q_len);
    if (qrc)
        return qrc;
    if (!aligned(tmp_output, 16) || !aligned(out, 4) || !aligned(seq_lens, 4) ||
        !aligned(exp_sums, 4) || !aligned(max_logits, 4) || (status && !aligned(status, 4)))
        return PA_ERR_INVALID_ARG;
    if (pa_v2_num_partitions(max_seq_len, partition_size) > max_num_partitions)
        return PA_ERR_WORKSPACE;
    MergeParams p;
    p.seq_lens = seq_lens;
    p.q_len = q_len;
    p.num_heads = num_heads;
    p.head_dim = head_dim;
    p.seq_len_cap = max_seq_len;
    p.partition_size = partition_size;
    p.max_num_partitions = max_num_partitions;
    p.tmp_output = tmp_output;
    p.exp_sums = exp_sums;
    p.max_logits = max_logits;
    p.out = out;
    p.status = status;
    int dev;
    if (current_device(&dev))
        return PA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0)
        return PA_ERR_CUDA;
    return launch_merge(dtype, p, num_seqs, sms, g_merge_form.load(std::memory_order_relaxed),
                        stream) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int choose_variant(int num_seqs, int num_kv_heads, int max_seq_len, int partition_size, int sms)
{
    // One partition: V2's merge would only copy, so V1.  Two partitions and a
    // V1 grid of at most one CTA per SM: the call is latency-bound and the
    // merge's fixed cost (a second launch behind the first) outweighs
    // splitting each sequence in two, so V1.  Otherwise V2.  Measured on
    // GB300 (us, V1 vs V2, 32 / 8 or 8 / 2 heads, P = 512): 1 seq x 1000
    // tokens 9.6 vs 10.6, 8 x 600 7.9 vs 10.9, 8 x 1000 10.4 vs 11.8; from
    // three partitions V2 wins (1 x 1500: 12.7 vs 10.6; 4 x 2000: 16.2 vs
    // 11.9), and with two partitions on a large grid too (512 x <= 1024:
    // 195.8 vs 177.4; 32 seqs of U{1..8192}: 97.2 vs 85.2).
    const int np = pa_v2_num_partitions(max_seq_len, partition_size);
    if (np <= 1)
        return 1;
    if (np == 2 && (long long)num_seqs * num_kv_heads <= sms)
        return 1;
    return 2;
}

// Several new tokens per sequence: which variant pa_decode_mq runs, and with
// which partition size (*part_out) if V2.
//
// The tcgen05 kernel with few (sequence, KV head, row tile) groups -- at
// most half the CTAs that are resident at once -- runs V2 on partitions
// sized so that the longest sequence's CTAs make exactly one wave (rounded
// up to the 64-token tile, never finer than partition_size).  Measured on
// GB300, one 100K-token sequence, 32 / 4 heads (us; 2048-token partitions
// vs one wave): 4 new tokens 48.0 vs 41.8, 8 tokens 51.5 vs 44.0, 16 tokens
// 62.0 vs 49.8, 32 tokens (two row tiles) 109.9 vs 76.3; one CTA per SM
// with rings of 4 + 4 to 6 + 6 stages instead: 47.0, 49.6, 56.3, 97.0.
//
// Otherwise, 32 to 128 query rows per KV head (one 128-row tile):
// V2 at a coarse partition of kTcV2Partition tokens (never finer than the
// caller's partition_size, and halved down to it while the grid would give
// fewer CTAs than SMs), or V1 when that partition covers max_seq_len.  The
// tcgen05 V2 pays a fixed set-up per CTA (TMEM allocation, barriers, the Q
// tile, filling and draining its rings); 2048-token partitions amortise it
// while still splitting the longest sequences, which bound V1.  Measured on
// GB300 (us per call; V1 / V2 at 512 / 1024 / 2048 / 4096 tokens):
//   32 seqs <= 8192 tokens (batch decode), 8 new tokens (32 rows):
//     152.2 / 151.9 / 129.5 / 129.4 / 146.8
//   the same, 16 new tokens (64 rows): 156.8 / 174.0 / 145.6 / 141.6 / 159.0
//   the same, 32 new tokens (128 rows): 175.7 / 235.6 / 187.0 / 177.1 / 193.6
//   one 100K-token sequence, 4 new tokens (32 rows): V2 55.2 / 54.3 / 49.5 / 69.9
//   the same, 16 new tokens (128 rows): V2 88.6 / 74.2 / 61.1 / 81.4
//   64 seqs, lognormal lengths <= 32768, 16 new tokens (128 rows):
//     253.7 / 354.3 / 279.4 / 250.6 / 254.1
// More rows (chunked prefill): V1 when the V1 grid (num_seqs * num_kv_heads
// CTAs per row split) gives every SM a CTA, else V2 at the caller's
// partition size; its partials grow with the rows (chunked prefill, 2 x
// 2048 new tokens after 30K: V1 2384 vs V2 4867 us at 512 tokens).  When
// V1's long CTAs would end on a mostly empty wave, V2 on two partitions:
// the same step, 1024 CTAs in waves of 304, bf16 V1 2456-2526 vs two
// partitions 2299-2327 us (three: 2357-2375; four: 2355-2388), fp16 1908 vs
// 1849-1852; 4 x 1024 new tokens after 3072 (short CTAs) V1 332 vs 452.
// Fewer rows (the mma.sync kernel, 2 or more new tokens): V2 on partitions
// of max(partition_size, 1024) tokens, halved the same way (us; V1 / V2 at
// 512 / 1024 / 2048): batch decode, 2 new tokens (8 rows) 96.5 / 86.1 /
// 86.6 / 122.8; 4 tokens (16 rows) 107.8 / 97.9 / 96.3 / 149.8; ragged, 2
// tokens (16 rows) 157.1 / 139.4 / 119.3 / 118.8; the 100K-token sequence,
// 2 tokens (16 rows) V2 44.2 / 41.1 / 42.9.  A single new token takes the
// caller's partition size, as pa_decode does.
constexpr int kTcV2Partition = 2048;
constexpr int kTcV2MaxRows = kTcRows;
constexpr int kMmaV2Partition = 1024;

int choose_variant_mq(int num_seqs, int q_len, int group, int num_kv_heads, int head_dim,
                      int max_seq_len, int partition_size, int sms, int *part_out)
{
    *part_out = partition_size;
    if (pa_v2_num_partitions(max_seq_len, partition_size) <= 1)
        return 1;
    const int cols = q_len * group;
    if (!use_tc(cols)) {
        if (q_len == 1)
            return 2;
        const long long per_part_mma = (long long)num_seqs * num_kv_heads *
                                       row_ctas(cols, head_dim, PA_BF16, max_seq_len);
        int pc = partition_size > kMmaV2Partition ? partition_size : kMmaV2Partition;
        while (pc / 2 >= partition_size &&
               per_part_mma * pa_v2_num_partitions(max_seq_len, pc) < sms)
            pc /= 2;
        if (pa_v2_num_partitions(max_seq_len, pc) <= 1)
            return 1;
        *part_out = pc;
        return 2;
    }
    // CTAs per partition index, and how many CTAs are resident at once (two
    // per SM for the one-tile kernel up to head_dim 128, one otherwise).
    const int tiles = tc_tiles(cols, head_dim, PA_BF16, max_seq_len);
    const long long per_part =
        (long long)num_seqs * num_kv_heads * row_ctas(cols, head_dim, PA_BF16, max_seq_len);
    const long long slots = (long long)sms * (tiles == 1 && head_dim <= 128 ? 2 : 1);
    if (2 * per_part <= slots) {
        // Few (sequence, KV head, row tile) groups: partitions sized so that
        // the longest sequence's CTAs fill exactly one wave (a multiple of
        // the 64-token tile), each group split over several SMs.
        const long long parts = slots / per_part;
        long long pc = ((long long)max_seq_len + parts - 1) / parts;
        pc = (pc + kTcTok - 1) / kTcTok * kTcTok;
        if (pc < partition_size)
            pc = partition_size;
        if (pa_v2_num_partitions(max_seq_len, (int)pc) <= 1)
            return 1;
        *part_out = (int)pc;
        return 2;
    }
    if (cols <= kTcV2MaxRows) {
        int pc = partition_size > kTcV2Partition ? partition_size : kTcV2Partition;
        while (pc / 2 >= partition_size &&
               per_part * pa_v2_num_partitions(max_seq_len, pc) < sms)
            pc /= 2;
        if (pa_v2_num_partitions(max_seq_len, pc) <= 1)
            return 1;
        *part_out = pc;
        return 2;
    }
    if (per_part < sms)
        return 2;
    // Many rows (chunked prefill), V1's grid fills the SMs: its CTAs run in
    // waves of `slots`.  When they are long (sequences of 8192 tokens and
    // more, so that a partial's fixed cost is small beside a CTA's work), the
    // waves would leave more than a tenth of the slots idle, and two
    // partitions per sequence pack them better: V2 on two partitions (a
    // multiple of 64 tokens).  Otherwise V1.
    const long long waves1 = (per_part + slots - 1) / slots;
    const long long waves2 = (2 * per_part + slots - 1) / slots;
    if (max_seq_len >= 4 * kTcV2Partition && 10 * per_part < 9 * slots * waves1 &&
        waves2 < 2 * waves1 && max_seq_len >= 2 * partition_size) {
        long long pc = ((long long)max_seq_len + 1) / 2;
        pc = (pc + kTcTok - 1) / kTcTok * kTcTok;
        if (pc >= partition_size && pa_v2_num_partitions(max_seq_len, (int)pc) == 2) {
            *part_out = (int)pc;
            return 2;
        }
    }
    return 1;
}


// bf16 rows that would take the two-tile kernel under fp16's rule, kVhMinRows
// or more of them per KV head (any number when pa_set_rows_kernel(4) forces
// two tiles): a binary16 copy of the V blocks the call reads, packed per KV
// head, in tmp_output past the
// partials of np_used partitions (0 for V1): the per-sequence block offsets
// and the flag word at the next multiple of 256 bytes, the copy at the next
// multiple of 256 after them, filling the rest of tmp_output.  The offsets
// pass sets the flag when the packed copy does not fit (lengths are device
// data); the attention kernels then read the bf16 cache.  vh->copy stays null
// when the rule does not apply or not even the offsets fit.
int make_v_half_copy(VhCopy *vh, const void *value_cache, const int32_t *block_tables,
                     const int32_t *seq_lens, int num_seqs, int q_len, int num_heads,
                     int num_kv_heads, int head_dim, int num_blocks, int block_size,
                     int max_blocks_per_seq, int cap, float *tmp_output, int max_num_partitions,
                     int np_used, cudaStream_t stream)
{
    const int cols = q_len * (num_heads / num_kv_heads);
    const bool forced = g_rows_kernel.load(std::memory_order_relaxed) == 4;
    if (!use_tc(cols) || tc_tiles(cols, head_dim, PA_F16, cap) != 2 ||
        (cols < kVhMinRows && !forced) || !tmp_output ||
        !aligned(tmp_output, 16) || max_num_partitions <= 0 || np_used > max_num_partitions)
        return PA_OK;
    auto round256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t off = round256((size_t)num_seqs * q_len * num_heads * np_used * head_dim * 4);
    const size_t copy_off = off + round256((size_t)(num_seqs + 1) * 4);
    const size_t have =
        (size_t)num_seqs * q_len * num_heads * (size_t)max_num_partitions * head_dim * 4;
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * 2;
    if (copy_off + block_bytes > have)
        return PA_OK;
    // Blocks the space holds, kept within 32-bit TMA row coordinates.
    long long copy_blocks = (long long)((have - copy_off) / block_bytes);
    const long long max_rows_blocks = (long long)INT32_MAX / ((long long)num_kv_heads * block_size);
    if (copy_blocks > max_rows_blocks)
        copy_blocks = max_rows_blocks;
    char *base = reinterpret_cast<char *>(tmp_output);
    VhParams vp;
    vp.value_cache = value_cache;
    vp.block_tables = block_tables;
    vp.seq_lens = seq_lens;
    vp.num_seqs = num_seqs;
    vp.num_kv_heads = num_kv_heads;
    vp.head_dim = head_dim;
    vp.block_size = block_size;
    vp.num_blocks = num_blocks;
    vp.max_blocks = max_blocks_per_seq;
    vp.seq_len_cap = cap;
    vp.copy_blocks = copy_blocks;
    vp.offs = reinterpret_cast<int32_t *>(base + off);
    vp.flag = vp.offs + num_seqs;
    vp.copy = base + copy_off;
    int dev;
    if (current_device(&dev))
        return PA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0)
        return PA_ERR_CUDA;
    if (launch_v_half(vp, sms, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    vh->copy = vp.copy;
    vh->flag = vp.flag;
    vh->offs = vp.offs;
    vh->copy_blocks = (int)copy_blocks;
    return PA_OK;
}

// V2 for several new tokens (phase 1 and the merge); vh: a binary16 copy of
// V for the two-tile kernel, or null.
int v2_mq_impl(const void *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int q_len,
               int num_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
               int max_blocks_per_seq, int max_seq_len_hint, float scale, int partition_size,
               int dtype, void *out, float *tmp_output, float *exp_sums, float *max_logits,
               int max_num_partitions, int32_t *status, cudaStream_t stream, const VhCopy *vh)
{
    if (!out || !aligned(out, 4))
        return PA_ERR_INVALID_ARG;
    int cap = 0;
    int rc = v2_phase1_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                            num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                            max_blocks_per_seq, max_seq_len_hint, scale, partition_size, dtype,
                            tmp_output, exp_sums, max_logits, max_num_partitions, status, stream,
                            &cap, nullptr, nullptr, vh);
    if (rc)
        return rc;
    return v2_phase2_impl(seq_lens, num_seqs, q_len, num_heads, head_dim, cap, partition_size,
                          dtype, tmp_output, exp_sums, max_logits, max_num_partitions, out, status,
                          stream);
}

// V1 for several new tokens; vh as for v2_mq_impl.
int v1_mq_impl(const void *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int q_len,
               int num_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
               int max_blocks_per_seq, int max_seq_len_hint, float scale, int dtype, void *out,
               int32_t *status, cudaStream_t stream, const VhCopy *vh)
{
    int rc = check_shape(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, scale, dtype);
    if (rc)
        return rc;
    rc = check_q_len(num_seqs, q_len);
    if (rc)
        return rc;
    if (!out || !aligned(out, 4) || (status && !aligned(status, 4)))
        return PA_ERR_INVALID_ARG;
    const int cap = seq_cap(max_blocks_per_seq, block_size, max_seq_len_hint);
    AttnLaunch L;
    rc = build_attn(L, query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                    num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                    cap, scale, dtype, true, 1, 0, nullptr, nullptr, nullptr, 0, out, status,
                    nullptr, vh);
    if (rc)
        return rc;
    return prepare_and_launch_attn(L, stream);
}

} // namespace

extern "C" {

PA_API int pa_v2_num_partitions(int max_seq_len, int partition_size)
{
    if (max_seq_len < 0 || partition_size <= 0)
        return -1;
    return (int)(((long long)max_seq_len + partition_size - 1) / partition_size);
}

PA_API size_t pa_v2_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                    int max_num_partitions)
{
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_num_partitions <= 0)
        return 0;
    return (size_t)num_seqs * num_heads * max_num_partitions * (size_t)(head_dim + 2) * 4;
}

PA_API int pa_decode_v2_phase1(const void *query, const void *key_cache, const void *value_cache,
                               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                               int block_size, int max_blocks_per_seq, int max_seq_len_hint,
                               float scale, int partition_size, int dtype, float *tmp_output,
                               float *exp_sums, float *max_logits, int max_num_partitions,
                               int32_t *status, pa_stream_t stream)
{
    return v2_phase1_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, 1,
                          num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                          max_blocks_per_seq, max_seq_len_hint, scale, partition_size, dtype,
                          tmp_output, exp_sums, max_logits, max_num_partitions, status,
                          (cudaStream_t)stream, nullptr);
}

PA_API int pa_decode_v2_phase2(const int32_t *seq_lens, int num_seqs, int num_heads,
                               int head_dim, int max_seq_len, int partition_size, int dtype,
                               const float *tmp_output, const float *exp_sums,
                               const float *max_logits, int max_num_partitions, void *out,
                               int32_t *status, pa_stream_t stream)
{
    return v2_phase2_impl(seq_lens, num_seqs, 1, num_heads, head_dim, max_seq_len, partition_size,
                          dtype, tmp_output, exp_sums, max_logits, max_num_partitions, out,
                          status, (cudaStream_t)stream);
}

PA_API int pa_decode_v2_mq(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int num_blocks, int block_size, int max_blocks_per_seq,
                           int max_seq_len_hint, float scale, int partition_size, int dtype,
                           void *out, float *tmp_output, float *exp_sums, float *max_logits,
                           int max_num_partitions, int32_t *status, pa_stream_t stream)
{
    return v2_mq_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                      num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                      max_seq_len_hint, scale, partition_size, dtype, out, tmp_output, exp_sums,
                      max_logits, max_num_partitions, status, (cudaStream_t)stream, nullptr);
}

PA_API int pa_decode_v2(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                        int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                        int partition_size, int dtype, void *out, float *tmp_output,
                        float *exp_sums, float *max_logits, int max_num_partitions,
                        int32_t *status, pa_stream_t stream)
{
    return pa_decode_v2_mq(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                           max_blocks_per_seq, max_seq_len_hint, scale, partition_size, dtype, out,
                           tmp_output, exp_sums, max_logits, max_num_partitions, status, stream);
}

PA_API int pa_decode_v2_fused(const void *query, const void *key_cache, const void *value_cache,
                              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, int max_blocks_per_seq, int max_seq_len_hint,
                              float scale, int partition_size, int dtype, void *out,
                              float *tmp_output, float *exp_sums, float *max_logits,
                              int max_num_partitions, int32_t *counters, int32_t *status,
                              pa_stream_t stream)
{
    if (!out || !aligned(out, 4) || !counters || !aligned(counters, 4))
        return PA_ERR_INVALID_ARG;
    int cap = 0;
    int rc = v2_phase1_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, 1,
                            num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                            max_blocks_per_seq, max_seq_len_hint, scale, partition_size, dtype,
                            tmp_output, exp_sums, max_logits, max_num_partitions, status,
                            (cudaStream_t)stream, &cap, out, counters);
    return rc;
}

PA_API int pa_decode_v1_mq(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int num_blocks, int block_size, int max_blocks_per_seq,
                           int max_seq_len_hint, float scale, int dtype, void *out,
                           int32_t *status, pa_stream_t stream)
{
    return v1_mq_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                      num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                      max_seq_len_hint, scale, dtype, out, status, (cudaStream_t)stream, nullptr);
}

PA_API int pa_decode_v1(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                        int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                        int dtype, void *out, int32_t *status, pa_stream_t stream)
{
    return pa_decode_v1_mq(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                           max_blocks_per_seq, max_seq_len_hint, scale, dtype, out, status, stream);
}

PA_API int pa_decode_choose(int num_seqs, int num_kv_heads, int max_seq_len, int partition_size)
{
    if (num_seqs <= 0 || num_kv_heads <= 0 || max_seq_len < 0 || partition_size <= 0)
        return -PA_ERR_INVALID_ARG;
    int dev;
    if (current_device(&dev))
        return -PA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0)
        return -PA_ERR_CUDA;
    return choose_variant(num_seqs, num_kv_heads, max_seq_len, partition_size, sms);
}

PA_API int pa_decode_mq_choose(int num_seqs, int q_len, int num_heads, int num_kv_heads,
                               int head_dim, int max_seq_len, int partition_size)
{
    if (num_seqs <= 0 || q_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || max_seq_len < 0 || partition_size <= 0)
        return -PA_ERR_INVALID_ARG;
    int dev;
    if (current_device(&dev))
        return -PA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0)
        return -PA_ERR_CUDA;
    int part = 0;
    return choose_variant_mq(num_seqs, q_len, num_heads / num_kv_heads, num_kv_heads, head_dim,
                             max_seq_len, partition_size, sms, &part);
}

PA_API int pa_decode_mq_partition(int num_seqs, int q_len, int num_heads, int num_kv_heads,
                                  int head_dim, int max_seq_len, int partition_size)
{
    if (num_seqs <= 0 || q_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || max_seq_len < 0 || partition_size <= 0)
        return -PA_ERR_INVALID_ARG;
    int dev;
    if (current_device(&dev))
        return -PA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0)
        return -PA_ERR_CUDA;
    int part = 0;
    const int v = choose_variant_mq(num_seqs, q_len, num_heads / num_kv_heads, num_kv_heads,
                                    head_dim, max_seq_len, partition_size, sms, &part);
    return v == 2 ? part : 0;
}

PA_API int pa_decode_mq(const void *query, const void *key_cache, const void *value_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                        int q_len, int num_heads, int num_kv_heads, int head_dim,
                        int num_blocks, int block_size, int max_blocks_per_seq,
                        int max_seq_len_hint, float scale, int partition_size, int dtype,
                        void *out, float *tmp_output, float *exp_sums, float *max_logits,
                        int max_num_partitions, int32_t *status, pa_stream_t stream)
{
    int rc = check_shape(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, scale, dtype);
    if (rc)
        return rc;
    rc = check_q_len(num_seqs, q_len);
    if (rc)
        return rc;
    if (partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    const int cap = seq_cap(max_blocks_per_seq, block_size, max_seq_len_hint);
    const int which =
        pa_decode_mq_choose(num_seqs, q_len, num_heads, num_kv_heads, head_dim, cap, partition_size);
    if (which < 0)
        return -which;
    const int part = which == 2 ? pa_decode_mq_partition(num_seqs, q_len, num_heads, num_kv_heads,
                                                         head_dim, cap, partition_size)
                                : partition_size;
    if (part < 0)
        return -part;
    const cudaStream_t st = (cudaStream_t)stream;
    // The arguments the entry points below check, checked here too: nothing
    // may be launched for a call that is then refused.
    if (!out || !aligned(out, 4) || (status && !aligned(status, 4)))
        return PA_ERR_INVALID_ARG;
    if (which == 2 && (!tmp_output || !exp_sums || !max_logits || max_num_partitions <= 0 ||
                       !aligned(tmp_output, 16) || !aligned(exp_sums, 4) ||
                       !aligned(max_logits, 4)))
        return PA_ERR_INVALID_ARG;
    if (which == 2 && pa_v2_num_partitions(cap, part) > max_num_partitions)
        return PA_ERR_WORKSPACE;
    VhCopy vh{nullptr, nullptr, nullptr, 0};
    const int np_used = which == 2 ? pa_v2_num_partitions(cap, part) : 0;
    if (dtype == PA_BF16) {
        rc = make_v_half_copy(&vh, value_cache, block_tables, seq_lens, num_seqs, q_len, num_heads,
                              num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                              cap, tmp_output, max_num_partitions, np_used, st);
        if (rc)
            return rc;
    }
    const VhCopy *vhp = vh.copy ? &vh : nullptr;
    if (which == 1)
        return v1_mq_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                          num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                          max_blocks_per_seq, max_seq_len_hint, scale, dtype, out, status, st, vhp);
    return v2_mq_impl(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, q_len,
                      num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                      max_seq_len_hint, scale, part, dtype, out, tmp_output, exp_sums, max_logits,
                      vhp ? np_used : max_num_partitions, status, st, vhp);
}

PA_API int pa_decode(const void *query, const void *key_cache, const void *value_cache,
                     const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                     int block_size, int max_blocks_per_seq, int max_seq_len_hint, float scale,
                     int partition_size, int dtype, void *out, float *tmp_output,
                     float *exp_sums, float *max_logits, int max_num_partitions,
                     int32_t *status, pa_stream_t stream)
{
    int rc = check_shape(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, scale, dtype);
    if (rc)
        return rc;
    if (partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    const int cap = seq_cap(max_blocks_per_seq, block_size, max_seq_len_hint);
    const int which = pa_decode_choose(num_seqs, num_kv_heads, cap, partition_size);
    if (which < 0)
        return -which;
    if (which == 1)
        return pa_decode_v1(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                            num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                            max_blocks_per_seq, max_seq_len_hint, scale, dtype, out, status,
                            stream);
    return pa_decode_v2(query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                        num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                        max_blocks_per_seq, max_seq_len_hint, scale, partition_size, dtype, out,
                        tmp_output, exp_sums, max_logits, max_num_partitions, status, stream);
}

PA_API const char *pa_status_string(int code)
{
    switch (code) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    default: return "PA_UNKNOWN";
    }
}

PA_API int pa_set_launch_config(int warps_per_cta, int stages_per_warp)
{
    if (warps_per_cta < 0 || warps_per_cta > kMaxWarps || stages_per_warp < 0 ||
        stages_per_warp > kMaxStages)
        return PA_ERR_INVALID_ARG;
    g_tune_warps.store(warps_per_cta, std::memory_order_relaxed);
    g_tune_stages.store(stages_per_warp, std::memory_order_relaxed);
    return PA_OK;
}

PA_API int pa_set_rows_kernel(int mode)
{
    if (mode < 0 || mode > 6)
        return PA_ERR_INVALID_ARG;
    g_rows_kernel.store(mode, std::memory_order_relaxed);
    return PA_OK;
}

PA_API int pa_set_merge_form(int form)
{
    if (form < 0 || form > 2)
        return PA_ERR_INVALID_ARG;
    g_merge_form.store(form, std::memory_order_relaxed);
    return PA_OK;
}

PA_API int pa_selftest_wait_timeout(int32_t *status, long long limit_ns, pa_stream_t stream)
{
    if (!status || !aligned(status, 4) || limit_ns <= 0 || limit_ns > 2000000000LL)
        return PA_ERR_INVALID_ARG;
    return launch_wait_selftest(status, (unsigned long long)limit_ns, (cudaStream_t)stream) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

} // extern "C"
