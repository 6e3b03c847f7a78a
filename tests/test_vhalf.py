"""GPU parity of the multi-query dispatch's binary16 copy of V (bf16 caches).

For bf16 rows that take the two-tile tcgen05 kernel with 1024 or more query rows
per KV head (head_dim <= 128, sequences of 1024+ tokens; any rows and lengths
with pa_set_rows_kernel(4)), pa_decode_mq writes a binary16 copy of the V
blocks the call reads into tmp_output past the partials, packed per KV head,
and P.V runs on binary16 P and V.  Every bf16 value below 2^16 in magnitude
converts exactly; a finite value at or above it, or a packed copy too large
for its space, sets the copy's flag and the call falls back to bf16 V with P
in hi + lo halves.  The outputs are compared element by element with the fp64
oracle; the copy itself is compared bit for bit with torch's bf16 -> fp16
conversion of the blocks it mirrors, and its block offsets with the prefix
sum of the sequences' block counts.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import OUT_ABS, check_out, half_ulp, mq, oracle_problem, ramp_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(0)
    yield
    cuda_lib.pa_set_rows_kernel(0)


def run_dispatch(inp, P, status=None, npmax=None):
    import paged_kv_decode_v2_gb300 as pa
    w = inp.workload
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    # Room for the copy: a workspace for partitions 8 times finer than P.
    npmax = npmax or 8 * max(1, pa.num_partitions(cap, P))
    tmp, es, ml = pa.alloc_workspace(S, H, D, npmax, q_len=Q)
    for t in (tmp, es, ml):
        t.fill_(float("nan"))
    out = torch.full_like(inp.query, float("nan"))
    pa.pa_decode_mq(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                    w.scale, P, out, tmp, es, ml, status=status)
    torch.cuda.synchronize()
    return out, tmp


def copy_region(inp, P, tmp):
    """(copy [KV, blocks, bs, D] fp16, offs [S], flag) where the dispatch puts them
    (include/pa_decode.h): the offsets and the flag 256-byte aligned past the partials at the
    stride of the partitions used, the packed copy at the next 256 bytes, filling the rest."""
    import paged_kv_decode_v2_gb300 as pa
    w = inp.workload
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    which = pa.pa_decode_mq_choose(S, Q, H, w.num_kv_heads, D, cap, P)
    np_used = pa.num_partitions(cap, pa.pa_decode_mq_partition(S, Q, H, w.num_kv_heads, D, cap, P)) \
        if which == 2 else 0
    r256 = lambda x: -(-x // 256) * 256
    off = r256(S * Q * H * np_used * D * 4)
    raw = tmp.view(-1).view(torch.uint8)
    meta = raw[off:off + 4 * (S + 1)].view(torch.int32)
    offs, flag = meta[:S].clone(), int(meta[S].item())
    copy_off = off + r256(4 * (S + 1))
    block = w.num_kv_heads * w.block_size * D * 2
    nblk = (raw.numel() - copy_off) // block
    copy = raw[copy_off:copy_off + nblk * block].view(torch.float16).view(
        w.num_kv_heads, nblk, w.block_size, D)
    return copy, offs, flag


def check_offsets(inp, offs):
    """offs is the exclusive prefix sum of each sequence's block count."""
    bs = inp.workload.block_size
    nb = [-(-L // bs) for L in inp.seq_lens.tolist()]
    want = [sum(nb[:b]) for b in range(len(nb))]
    assert offs.tolist() == want


def check_copy(inp, copy, offs):
    """Blocks j < ceil(L / block_size) of each sequence, at index offs[s] + j of every KV
    head's part, equal torch's
    bf16 -> fp16 conversion of the cache blocks they mirror, bit for bit, with rows past the
    sequence's end zero."""
    w = inp.workload
    check_offsets(inp, offs)
    for b, L in enumerate(inp.seq_lens.tolist()):
        nb = -(-L // w.block_size)
        ids = inp.block_tables[b, :nb].long()
        blocks = inp.value_cache[ids].to(torch.float16)          # [nb, KV, bs, D]
        tok = torch.arange(nb * w.block_size, device=blocks.device).view(nb, 1, w.block_size, 1)
        blocks = torch.where(tok < L, blocks, torch.zeros_like(blocks)).permute(1, 0, 2, 3)
        o = int(offs[b])
        got = copy[:, o:o + nb]
        bad = (got.view(torch.int16) != blocks.contiguous().view(torch.int16)).sum().item()
        assert bad == 0, f"sequence {b}: {bad} values differ"


def prefill(name, q_len, G, lens, KV=2, D=128, bs=16, seed=0):
    return wl.make_inputs(mq(name, q_len, G, lens, bs=bs, P=512, D=D, KV=KV, seed=seed),
                          device="cuda")


# 1024 query rows per KV head (256 new tokens x 4 query heads): the copy under the default rule.
QL, GR = 256, 4


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32), (128, 64), (128, 8)])
def test_copy_used_and_parity(D, bs):
    """1024 rows per KV head, sequences up to 2000 tokens (one shorter than the chunk): the copy
    is made, holds every block it mirrors bit for bit (zero past each sequence's end), its flag
    is clear, and the output matches the oracle."""
    inp = prefill("vh_parity", QL, GR, (300, 1100, 2000, 41), D=D, bs=bs, seed=9400 + D + bs)
    out, tmp = run_dispatch(inp, 512)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy, offs)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_parity")


def test_copy_on_the_v1_path():
    """A shape the dispatch runs as V1 (sequences below 4096 tokens, more row tiles than a wave
    holds) takes the copy from the whole workspace."""
    import paged_kv_decode_v2_gb300 as pa
    lens = tuple(1100 + 37 * i for i in range(6))
    inp = prefill("vh_v1", 128, 8, lens, KV=8, seed=9450)
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    assert pa.pa_decode_mq_choose(S, Q, H, 8, D, cap, 512) == 1
    out, tmp = run_dispatch(inp, 512)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy, offs)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_v1")


def test_values_beyond_binary16_set_the_flag():
    """A finite value of 2^16 or more anywhere in the blocks read sets the flag; the call then
    reads the bf16 cache (P in hi + lo halves) and still matches the oracle, with the bound
    widened by 2^-11 * sum(p |v|) / l as in the tcgen05 suite's large-value test."""
    inp = prefill("vh_wide", QL, GR, (300, 1100, 2000), seed=9500)
    bs = 16
    tables = inp.block_tables.cpu()
    t = 1100 // 2
    inp.value_cache[int(tables[1, t // bs]), :, t % bs, 3] = 7.0e4
    out, tmp = run_dispatch(inp, 512)
    flag = copy_region(inp, 512, tmp)[2]
    assert flag == 1
    arrays = wl.to_oracle_arrays(inp)
    ref = oracle.decode(oracle.Problem.from_arrays(arrays))
    arrays["value_cache"] = arrays["value_cache"] & np.uint16(0x7FFF)
    ref_abs = oracle.decode(oracle.Problem.from_arrays(arrays))
    o = out.cpu().to(torch.float64).numpy()
    assert np.isfinite(o).all()
    assert (np.abs(o - ref) <= OUT_ABS + half_ulp(ref, wl.BF16) + 2.0 ** -11 * ref_abs).all()


def test_values_beyond_binary16_on_the_v1_path():
    """The V1 shape of test_copy_on_the_v1_path with one value of 2^16 or more: the flag is set
    and the two-tile kernel takes its bf16 form (hi + lo P on the cache) in the same launch."""
    import paged_kv_decode_v2_gb300 as pa
    lens = tuple(1100 + 37 * i for i in range(6))
    inp = prefill("vh_v1_wide", 128, 8, lens, KV=8, seed=9460)
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    assert pa.pa_decode_mq_choose(S, Q, H, 8, D, cap, 512) == 1
    t = 777
    inp.value_cache[int(inp.block_tables.cpu()[2, t // 16]), 5, t % 16, 9] = -9.0e4
    out, tmp = run_dispatch(inp, 512)
    assert copy_region(inp, 512, tmp)[2] == 1
    arrays = wl.to_oracle_arrays(inp)
    ref = oracle.decode(oracle.Problem.from_arrays(arrays))
    arrays["value_cache"] = arrays["value_cache"] & np.uint16(0x7FFF)
    ref_abs = oracle.decode(oracle.Problem.from_arrays(arrays))
    o = out.cpu().to(torch.float64).numpy()
    assert np.isfinite(o).all()
    assert (np.abs(o - ref) <= OUT_ABS + half_ulp(ref, wl.BF16) + 2.0 ** -11 * ref_abs).all()


def test_copy_path_is_reproducible():
    """Three calls on the same inputs through the copy (offsets pass, copy pass, two-tile kernel,
    merge) give bitwise the same output."""
    inp = prefill("vh_repro", QL, GR, (300, 1100, 2000), seed=9560)
    first, _ = run_dispatch(inp, 512)
    for _ in range(2):
        again, _ = run_dispatch(inp, 512)
        assert torch.equal(first, again)


def test_poison_does_not_set_the_flag():
    """NaN in every slot the call must not read (unreferenced blocks, rows past each sequence's
    end) changes nothing, bit for bit, and leaves the flag clear."""
    inp = prefill("vh_poison", QL, GR, (300, 1100, 2000), seed=9550)
    clean, tmp = run_dispatch(inp, 512)
    wl.poison_unreferenced(inp, float("nan"))
    dirty, tmp2 = run_dispatch(inp, 512)
    assert torch.equal(clean, dirty)
    assert copy_region(inp, 512, tmp2)[2] == 0


def test_small_workspace_skips_the_copy():
    """A workspace with room for the partials only: no copy, bf16 hi + lo P on one tile, same
    parity."""
    inp = prefill("vh_small", QL, GR, (300, 1100, 2000), seed=9600)
    out, tmp = run_dispatch(inp, 512, npmax=np_used(inp, 512))
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_small")


def test_below_the_rows_threshold_makes_no_copy():
    """160 rows per KV head under the default rule: the one-tile kernel with hi + lo P and
    nothing written past the partials."""
    inp = prefill("vh_rows", 40, 4, (300, 1100, 2000), seed=9610)
    out, tmp = run_dispatch(inp, 512)
    n = np_used(inp, 512)
    import paged_kv_decode_v2_gb300 as pa
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    if pa.pa_decode_mq_choose(S, Q, H, 2, D, cap, 512) == 1:
        n = 0
    assert torch.isnan(tmp[..., n:, :]).all()
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_rows")


def np_used(inp, P):
    import paged_kv_decode_v2_gb300 as pa
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * inp.workload.block_size
    part = pa.pa_decode_mq_partition(S, Q, H, inp.workload.num_kv_heads, D, cap, P)
    return pa.num_partitions(cap, part if part > 0 else P)


def test_packed_copy_fits_where_a_dense_one_would_not(cuda_lib):
    """pa_set_rows_kernel(4), 160 rows: four spare partitions of workspace hold the 213 blocks
    the sequences use (1.7 MB) but not a block-table-shaped copy (3 x 125 blocks, 3.1 MB): the
    copy is made and used."""
    cuda_lib.pa_set_rows_kernel(4)
    inp = prefill("vh_packed", 40, 4, (300, 1100, 2000), seed=9620)
    out, tmp = run_dispatch(inp, 512, npmax=np_used(inp, 512) + 4)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert copy.shape[1] >= 213 and copy.shape[1] < 3 * inp.block_tables.shape[1]
    assert flag == 0
    check_copy(inp, copy, offs)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_packed")


def test_copy_that_does_not_fit_sets_the_flag(cuda_lib):
    """pa_set_rows_kernel(4), 160 rows: one spare partition holds about 60 blocks, fewer than
    the 213 the sequences use: the offsets pass sets the flag, nothing is copied, and the bf16
    kernel gives the output."""
    cuda_lib.pa_set_rows_kernel(4)
    inp = prefill("vh_nofit", 40, 4, (300, 1100, 2000), seed=9640)
    out, tmp = run_dispatch(inp, 512, npmax=np_used(inp, 512) + 1)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert 0 < copy.shape[1] < 213
    assert flag == 1
    check_offsets(inp, offs)
    nan_bits = torch.tensor([float("nan")], dtype=torch.float32).view(torch.int32).item()
    assert (copy.view(torch.int32) == nan_bits).all()  # the workspace's NaN fill, untouched
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_nofit")


def test_bad_block_id_reads_block_zero_and_sets_status():
    inp = prefill("vh_status", QL, GR, (300, 1100), seed=9650)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp.block_tables[1, 5] = 10 ** 6
    out, tmp = run_dispatch(inp, 512, status=status)
    assert int(status.item()) & 1  # PA_STATUS_BAD_BLOCK_ID
    assert torch.isfinite(out).all()


def test_copy_with_empty_sequences_mixed_in():
    """Zero-length sequences between others: no block of theirs is copied or read, and their
    rows come out zero."""
    inp = prefill("vh_empty", QL, GR, (0, 1100, 0, 2000, 37), seed=9700)
    out, tmp = run_dispatch(inp, 512)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy, offs)
    ref = oracle.decode(oracle_problem(inp))
    check_out(out, ref, wl.BF16, what="vh_empty")
    assert (ref[0] == 0).all() and (ref[2] == 0).all()


def test_forced_two_tiles_on_short_sequences_use_the_copy(cuda_lib):
    """pa_set_rows_kernel(4) takes the two-tile kernel, and with it the copy, below 1024 tokens."""
    cuda_lib.pa_set_rows_kernel(4)
    inp = prefill("vh_short", 40, 4, (45, 300, 700), seed=9750)
    out, tmp = run_dispatch(inp, 512)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy, offs)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_short")


@pytest.mark.parametrize("c,period", [(1.5, None), (0.3, None), (4.0, 256)])
def test_copy_with_rising_and_falling_scores(cuda_lib, c, period):
    """pa_set_rows_kernel(4), 160 rows, scores rising on half the heads (the tcgen05 suite's ramps):
    through the copy, with binary16 P, the lazy rescale of O and l still matches the oracle."""
    cuda_lib.pa_set_rows_kernel(4)
    inp = ramp_scores(prefill("vh_ramp", 40, 4, (700, 300, 1000, 65), seed=9720 + int(10 * c)), c,
                      period)
    out, tmp = run_dispatch(inp, 512)
    copy, offs, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy, offs)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what=f"vh_ramp c={c}")


def test_one_tile_mode_makes_no_copy(cuda_lib):
    """pa_set_rows_kernel(3) keeps the one-tile kernel: nothing is written past the partials."""
    cuda_lib.pa_set_rows_kernel(3)
    inp = prefill("vh_none", 40, 4, (300, 1100, 2000), seed=9800)
    out, tmp = run_dispatch(inp, 512)
    import paged_kv_decode_v2_gb300 as pa
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    part = pa.pa_decode_mq_partition(S, Q, H, 2, D, cap, 512)
    np_used = pa.num_partitions(cap, part) if part > 0 else 0
    # Partials at the caller's stride (no copy, so no compaction): slots past np_used untouched.
    assert torch.isnan(tmp[..., np_used:, :]).all()
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_none")
