"""GPU parity of the single-kernel V2 (pa_decode_v2_fused) against the fp64 oracle.

The last CTA of each (sequence, KV head) to finish merges that group's
partitions, found with a ticket counter per group.  Checked: out against the
oracle and the partials against the oracle's per-partition statistics; the
counters are back at zero after every call, so repeated calls on one counter
array keep giving the same result.
"""
import pytest
import torch

import oracle
import workloads as wl
from parity_util import check_out, check_partitions, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(0)


def run_fused(pa, inp, P, hint=0, counters=None, status=None):
    w = inp.workload
    S, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    if hint > 0:
        cap = min(cap, hint)
    npmax = max(1, pa.num_partitions(cap, P))
    tmp, es, ml = pa.alloc_workspace(S, H, D, npmax)
    for t in (tmp, es, ml):
        t.fill_(float("nan"))
    if counters is None:
        counters = pa.alloc_counters(S, w.num_kv_heads)
    out = torch.full_like(inp.query, float("nan"))
    pa.pa_decode_v2_fused(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                          inp.seq_lens, w.scale, P, out, tmp, es, ml, counters,
                          max_seq_len_hint=hint, status=status)
    torch.cuda.synchronize()
    assert int(counters.abs().sum().item()) == 0, "ticket counters not back at zero"
    return out, tmp, es, ml


def fused_check(pa, inp, P, hint=0):
    prob = oracle_problem(inp)
    ref = oracle.decode(prob)
    out, tmp, es, ml = run_fused(pa, inp, P, hint=hint)
    check_out(out, ref, inp.workload.dtype, what=f"{inp.workload.name}/fused")
    check_partitions(inp, P, tmp, es, ml, prob=prob)
    return out


def test_tiny(cuda_lib):
    fused_check(cuda_lib, wl.make_inputs(wl.TINY, device="cuda"), 512)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 4, 8, 16, 64])
@pytest.mark.parametrize("P", [64, 512])
def test_fused_fuzz_grid(cuda_lib, dtype, bs, G, P):
    lens = (1, bs - 1, bs, bs + 1, P - 1, P, P + 1, 2 * P + bs + 3, 3 * P + 5)
    w = wl.Workload("fused_fuzz", len(lens), 2 * G, 2, 128, bs, P, dtype, "list", seq_lens=lens,
                    seed=11000 + 7 * G + bs + P + dtype)
    fused_check(cuda_lib, wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("G", [1, 8])
def test_fused_head_dims(cuda_lib, D, G):
    lens = (1, 15, 129, 700)
    w = wl.Workload("fused_d", len(lens), 2 * G, 2, D, 16, 128, wl.BF16, "list", seq_lens=lens,
                    seed=11500 + D + G)
    fused_check(cuda_lib, wl.make_inputs(w, device="cuda"), 128)


@pytest.mark.parametrize("bs,P", [(16, 300), (32, 200), (64, 100), (8, 12)])
def test_fused_partition_not_a_multiple_of_block_size(cuda_lib, bs, P):
    lens = sorted({1, bs + 1, P - 1, P, P + 1, 2 * P + 3, 700})
    w = wl.Workload("fused_pnb", len(lens), 8, 2, 128, bs, P, wl.BF16, "list",
                    seq_lens=tuple(lens), seed=11700 + bs + P)
    fused_check(cuda_lib, wl.make_inputs(w, device="cuda"), P)


def test_fused_empty_sequences(cuda_lib):
    w = wl.Workload("fused_empty", 5, 8, 2, 128, 16, 64, wl.BF16, "list",
                    seq_lens=(0, 1, 0, 65, 0), seed=77)
    inp = wl.make_inputs(w, device="cuda", max_blocks=8)
    out = fused_check(cuda_lib, inp, 64)
    assert (out[0] == 0).all() and (out[2] == 0).all() and (out[4] == 0).all()


def test_fused_all_empty(cuda_lib):
    w = wl.Workload("fused_allempty", 3, 8, 2, 128, 16, 64, wl.F16, "list", seq_lens=(0, 0, 0),
                    seed=3)
    inp = wl.make_inputs(w, device="cuda", max_blocks=4)
    assert (run_fused(cuda_lib, inp, 64)[0] == 0).all()


def test_fused_max_seq_len_hint(cuda_lib):
    w = wl.Workload("fused_hint", 3, 32, 4, 128, 16, 512, wl.BF16, "list",
                    seq_lens=(900, 1700, 33), seed=9)
    fused_check(cuda_lib, wl.make_inputs(w, device="cuda", max_blocks=400), 512, hint=1700)


def test_fused_repeated_calls_share_one_counter_array(cuda_lib):
    """Ten calls in a row on one counter array (left zero by each call), on two
    different shapes alternately, give the same outputs every time."""
    pa = cuda_lib
    a = wl.make_inputs(wl.TINY, device="cuda")
    w2 = wl.Workload("fused_rep", 1, 8, 2, 128, 16, 64, wl.BF16, "list", seq_lens=(5000,), seed=5)
    b = wl.make_inputs(w2, device="cuda")
    counters = pa.alloc_counters(1, 2)
    first = {}
    for k in range(10):
        inp, P = (a, 512) if k % 2 == 0 else (b, 64)
        out = run_fused(pa, inp, P, counters=counters)[0]
        if inp.workload.name in first:
            assert torch.equal(out, first[inp.workload.name])
        else:
            first[inp.workload.name] = out
    check_out(first["tiny"], oracle.decode(oracle_problem(a)), a.workload.dtype, what="tiny")
    check_out(first["fused_rep"], oracle.decode(oracle_problem(b)), b.workload.dtype,
              what="fused_rep")


def test_fused_bad_block_id_sets_status(cuda_lib):
    inp = wl.make_inputs(wl.TINY, device="cuda")
    inp.block_tables[0, 5] = inp.key_cache.shape[0] + 7
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_fused(cuda_lib, inp, 512, status=st)
    assert int(st.item()) & 1


def test_fused_relabelling_is_bitwise_invariant(cuda_lib):
    inp = wl.make_inputs(wl.TINY, device="cuda")
    r = wl.relabel_blocks(inp, seed=123)
    assert torch.equal(run_fused(cuda_lib, inp, 512)[0], run_fused(cuda_lib, r, 512)[0])


def test_fused_batch_decode_full_size_every_element(cuda_lib):
    fused_check(cuda_lib, wl.make_inputs(wl.BATCH, device="cuda"), wl.BATCH.partition_size)


@pytest.mark.parametrize("P", [512, 1024])
def test_fused_long_100k_full_size_every_element(cuda_lib, P):
    fused_check(cuda_lib, wl.make_inputs(wl.LONG, device="cuda"), P)
