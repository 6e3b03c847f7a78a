"""GPU parity of the multi-query dispatch's binary16 copy of V (bf16 caches).

For bf16 rows that take the two-tile tcgen05 kernel (more than 128 query rows
per KV head, head_dim <= 128, sequences of 1024+ tokens), pa_decode_mq writes
a binary16 copy of the V blocks the call reads into tmp_output past the
partials, and P.V runs on binary16 P and V.  Every bf16 value below 2^16 in
magnitude converts exactly; a finite value at or above it sets the copy's flag
and the call falls back to bf16 V with P in hi + lo halves.  The outputs are
compared element by element with the fp64 oracle; the copy itself is compared
bit for bit with torch's bf16 -> fp16 conversion of the blocks it mirrors.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import OUT_ABS, check_out, half_ulp, mq, oracle_problem

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
    """(copy [S, KV, max_blocks, bs, D] fp16, flag) where the dispatch puts them: past the
    partials at the stride of the partitions it uses, 256-byte aligned (include/pa_decode.h)."""
    import paged_kv_decode_v2_gb300 as pa
    w = inp.workload
    S, Q, H, D = inp.query.shape
    maxb = inp.block_tables.shape[1]
    cap = maxb * w.block_size
    which = pa.pa_decode_mq_choose(S, Q, H, w.num_kv_heads, D, cap, P)
    np_used = pa.num_partitions(cap, pa.pa_decode_mq_partition(S, Q, H, w.num_kv_heads, D, cap, P)) \
        if which == 2 else 0
    off = -(-(S * Q * H * np_used * D * 4) // 256) * 256
    nbytes = S * w.num_kv_heads * maxb * w.block_size * D * 2
    raw = tmp.view(-1).view(torch.uint8)
    copy = raw[off:off + nbytes].view(torch.float16).view(S, w.num_kv_heads, maxb, w.block_size, D)
    fo = off + -(-nbytes // 256) * 256
    flag = int(raw[fo:fo + 4].view(torch.int32).item())
    return copy, flag


def check_copy(inp, copy):
    """Blocks j < ceil(L / block_size) of each sequence equal torch's bf16 -> fp16 conversion of
    the cache blocks they mirror, bit for bit, with rows past the sequence's end zero (blocks
    past it are never written or read)."""
    w = inp.workload
    for b, L in enumerate(inp.seq_lens.tolist()):
        nb = -(-L // w.block_size)
        ids = inp.block_tables[b, :nb].long()
        blocks = inp.value_cache[ids].to(torch.float16)          # [nb, KV, bs, D]
        tok = torch.arange(nb * w.block_size, device=blocks.device).view(nb, 1, w.block_size, 1)
        blocks = torch.where(tok < L, blocks, torch.zeros_like(blocks)).permute(1, 0, 2, 3)
        got = copy[b, :, :nb]
        bad = (got.view(torch.int16) != blocks.contiguous().view(torch.int16)).sum().item()
        assert bad == 0, f"sequence {b}: {bad} values differ"


def prefill(name, q_len, G, lens, KV=2, D=128, bs=16, seed=0):
    return wl.make_inputs(mq(name, q_len, G, lens, bs=bs, P=512, D=D, KV=KV, seed=seed),
                          device="cuda")


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32), (128, 64), (128, 8)])
def test_copy_used_and_parity(D, bs):
    """160 rows per KV head, sequences up to 2000 tokens: the copy is made, holds every block
    it mirrors bit for bit (zero past each sequence's end), its flag is clear, and the output
    matches the oracle."""
    inp = prefill("vh_parity", 40, 4, (300, 1100, 2000, 41), D=D, bs=bs, seed=9400 + D + bs)
    out, tmp = run_dispatch(inp, 512)
    copy, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_parity")


def test_copy_on_the_v1_path():
    """A shape the dispatch runs as V1 (every SM has a CTA, sequences below 8192 tokens) takes
    the copy from the whole workspace."""
    import paged_kv_decode_v2_gb300 as pa
    lens = tuple(1100 + 37 * i for i in range(10))
    inp = prefill("vh_v1", 20, 8, lens, KV=8, seed=9450)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    which = pa.pa_decode_mq_choose(S, Q, H, 8, D, cap, 512)
    per_part = S * 8 * 2  # (sequence, KV head, pair of 128-row tiles) CTAs
    assert which == (2 if per_part <= sms else 1)
    out, tmp = run_dispatch(inp, 512)
    copy, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_v1")


def test_values_beyond_binary16_set_the_flag():
    """A finite value of 2^16 or more anywhere in the blocks read sets the flag; the call then
    reads the bf16 cache (P in hi + lo halves) and still matches the oracle, with the bound
    widened by 2^-11 * sum(p |v|) / l as in the tcgen05 suite's large-value test."""
    inp = prefill("vh_wide", 40, 4, (300, 1100, 2000), seed=9500)
    bs = 16
    tables = inp.block_tables.cpu()
    t = 1100 // 2
    inp.value_cache[int(tables[1, t // bs]), :, t % bs, 3] = 7.0e4
    out, tmp = run_dispatch(inp, 512)
    _, flag = copy_region(inp, 512, tmp)
    assert flag == 1
    arrays = wl.to_oracle_arrays(inp)
    ref = oracle.decode(oracle.Problem.from_arrays(arrays))
    arrays["value_cache"] = arrays["value_cache"] & np.uint16(0x7FFF)
    ref_abs = oracle.decode(oracle.Problem.from_arrays(arrays))
    o = out.cpu().to(torch.float64).numpy()
    assert np.isfinite(o).all()
    assert (np.abs(o - ref) <= OUT_ABS + half_ulp(ref, wl.BF16) + 2.0 ** -11 * ref_abs).all()


def test_poison_does_not_set_the_flag():
    """NaN in every slot the call must not read (unreferenced blocks, rows past each sequence's
    end) changes nothing, bit for bit, and leaves the flag clear."""
    inp = prefill("vh_poison", 40, 4, (300, 1100, 2000), seed=9550)
    clean, tmp = run_dispatch(inp, 512)
    wl.poison_unreferenced(inp, float("nan"))
    dirty, tmp2 = run_dispatch(inp, 512)
    assert torch.equal(clean, dirty)
    assert copy_region(inp, 512, tmp2)[1] == 0


def test_small_workspace_skips_the_copy():
    """A workspace with room for the partials only: no copy, bf16 hi + lo P on one tile, same
    parity."""
    inp = prefill("vh_small", 40, 4, (300, 1100, 2000), seed=9600)
    import paged_kv_decode_v2_gb300 as pa
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    part = pa.pa_decode_mq_partition(S, Q, H, 2, D, cap, 512)
    np_used = pa.num_partitions(cap, part if part > 0 else 512)
    out, tmp = run_dispatch(inp, 512, npmax=np_used)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_small")


def test_bad_block_id_reads_block_zero_and_sets_status():
    inp = prefill("vh_status", 40, 4, (300, 1100), seed=9650)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp.block_tables[1, 5] = 10 ** 6
    out, tmp = run_dispatch(inp, 512, status=status)
    assert int(status.item()) & 1  # PA_STATUS_BAD_BLOCK_ID
    assert torch.isfinite(out).all()


def test_copy_with_empty_sequences_mixed_in():
    """Zero-length sequences between others: no block of theirs is copied or read, and their
    rows come out zero."""
    inp = prefill("vh_empty", 40, 4, (0, 1100, 0, 2000, 37), seed=9700)
    out, tmp = run_dispatch(inp, 512)
    copy, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy)
    ref = oracle.decode(oracle_problem(inp))
    check_out(out, ref, wl.BF16, what="vh_empty")
    assert (ref[0] == 0).all() and (ref[2] == 0).all()


def test_forced_two_tiles_on_short_sequences_use_the_copy(cuda_lib):
    """pa_set_rows_kernel(4) takes the two-tile kernel, and with it the copy, below 1024 tokens."""
    cuda_lib.pa_set_rows_kernel(4)
    inp = prefill("vh_short", 40, 4, (45, 300, 700), seed=9750)
    out, tmp = run_dispatch(inp, 512)
    copy, flag = copy_region(inp, 512, tmp)
    assert flag == 0
    check_copy(inp, copy)
    check_out(out, oracle.decode(oracle_problem(inp)), wl.BF16, what="vh_short")


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
