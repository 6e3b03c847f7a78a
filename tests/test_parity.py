"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output element; the full-size workloads compare
every element where the oracle is fast enough and sampled sequences
(compacted into a small pool) where it is not.  Tolerances are those of
parity_util.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import (check_out, check_partitions, compact_subset, oracle_out, oracle_problem,
                         run_v2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    yield
    cuda_lib.pa_set_launch_config(0, 0)


def full_check(inp, P, entries=("v2", "v1", "dispatch"), hint=0):
    prob = oracle_problem(inp)
    ref = oracle.decode(prob)
    for e in entries:
        out, tmp, es, ml = run_v2(inp, P, hint=hint, entry=e)
        check_out(out, ref, inp.workload.dtype, what=f"{inp.workload.name}/{e}")
        if e == "v2":
            check_partitions(inp, P, tmp, es, ml, prob=prob)


# ---------------------------------------------------------------- small, every element

def test_tiny_workload_all_entries():
    full_check(wl.make_inputs(wl.TINY, device="cuda"), wl.TINY.partition_size)


def test_split_phases_equal_fused_call_bitwise():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    a = run_v2(inp, 512, entry="v2")
    b = run_v2(inp, 512, entry="split")
    assert torch.equal(a[0], b[0])


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("P", [64, 512])
def test_fuzz_grid(dtype, bs, G, P):
    lens = (1, bs - 1, bs, bs + 1, P - 1, P, P + 1, 2 * P + bs + 3, 3 * P + 5)
    w = wl.Workload("fuzz", len(lens), 2 * G, 2, 128, bs, P, dtype, "list", seq_lens=lens,
                    seed=1000 + 7 * G + bs + P + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 8, 16])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_fuzz_head_dims(D, bs, G, dtype):
    P = 128
    lens = (1, bs - 1, bs + 1, P - 1, P + 1, 3 * P + bs + 3)
    w = wl.Workload("fuzz_d", len(lens), 2 * G, 2, D, bs, P, dtype, "list", seq_lens=lens,
                    seed=2000 + D + 7 * G + bs + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("P", [128, 512])
def test_fuzz_block_size_64(dtype, G, P):
    lens = (1, 63, 64, 65, P - 1, P + 1, 2 * P + 67)
    w = wl.Workload("fuzz_bs64", len(lens), 2 * G, 2, 128, 64, P, dtype, "list", seq_lens=lens,
                    seed=3000 + 7 * G + P + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("bs,P", [(16, 300), (32, 200), (64, 100), (16, 8), (32, 48), (64, 1000),
                                  (16, 17), (32, 1), (8, 300), (8, 4), (8, 12)])
@pytest.mark.parametrize("G", [4, 16])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_partition_not_a_multiple_of_block_size(bs, P, G, dtype):
    """Partitions that begin and end inside a block: a straddling block is read
    by both partitions, each keeping only its own tokens."""
    lens = sorted({1, bs - 1, bs + 1, P - 1 or 1, P, P + 1, 2 * P + 3, 3 * P + bs + 5, 700})
    if P < 8:  # keep the partition count (and the oracle's work) small
        lens = [1, 2, 3, bs + 1, 40]
    w = wl.Workload("fuzz_pnb", len(lens), 2 * G, 2, 128, bs, P, dtype, "list", seq_lens=tuple(lens),
                    seed=7000 + bs + P + G + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("warps,stages", [(1, 1), (2, 2), (8, 1), (3, 3)])
def test_launch_shapes_other_head_dims(cuda_lib, D, warps, stages):
    w = wl.Workload("shapes_d", 3, 16, 2, D, 32, 256, wl.BF16, "list", seq_lens=(700, 2049, 5),
                    seed=56 + D)
    inp = wl.make_inputs(w, device="cuda")
    cuda_lib.pa_set_launch_config(warps, stages)
    try:
        full_check(inp, 256, entries=("v2", "v1"))
    finally:
        cuda_lib.pa_set_launch_config(0, 0)


@pytest.mark.parametrize("warps,stages", [(1, 1), (1, 2), (2, 1), (2, 4), (8, 2), (3, 3), (4, 8)])
@pytest.mark.parametrize("bs", [8, 16])
def test_launch_shapes_do_not_change_results(cuda_lib, warps, stages, bs):
    w = wl.Workload("shapes", 4, 16, 2, 128, bs, 256, wl.BF16, "list",
                    seq_lens=(1, 700, 2049, 4096), seed=55 + bs)
    inp = wl.make_inputs(w, device="cuda")
    cuda_lib.pa_set_launch_config(warps, stages)
    try:
        full_check(inp, 256, entries=("v2", "v1"))
    finally:
        cuda_lib.pa_set_launch_config(0, 0)


def test_empty_and_short_sequences():
    w = wl.Workload("empty", 5, 8, 2, 128, 16, 64, wl.BF16, "list", seq_lens=(0, 1, 0, 65, 0),
                    seed=77)
    inp = wl.make_inputs(w, device="cuda", max_blocks=8)
    full_check(inp, 64)
    for e in ("v2", "v1"):
        out = run_v2(inp, 64, entry=e)[0]
        assert (out[0] == 0).all() and (out[2] == 0).all() and (out[4] == 0).all()


def test_all_sequences_empty():
    w = wl.Workload("allempty", 3, 8, 2, 128, 16, 64, wl.F16, "list", seq_lens=(0, 0, 0), seed=3)
    inp = wl.make_inputs(w, device="cuda", max_blocks=4)
    for e in ("v2", "v1", "dispatch"):
        out = run_v2(inp, 64, entry=e)[0]
        assert (out == 0).all()


def test_max_seq_len_hint():
    w = wl.Workload("hint", 3, 32, 4, 128, 16, 512, wl.BF16, "list", seq_lens=(900, 1700, 33),
                    seed=9)
    inp = wl.make_inputs(w, device="cuda", max_blocks=400)
    full_check(inp, 512, hint=1700)


@pytest.mark.parametrize("bs", [8, 16])
def test_unreferenced_and_tail_slots_never_reach_the_output(bs):
    w = wl.Workload("poison", 4, 16, 2, 128, bs, 128, wl.BF16, "list", seq_lens=(37, 16, 300, 5),
                    seed=21 + bs)
    inp = wl.make_inputs(w, device="cuda", max_blocks=480 // bs)
    clean = [run_v2(inp, 128, entry=e)[0] for e in ("v2", "v1")]
    wl.poison_unreferenced(inp, float("nan"))
    dirty = [run_v2(inp, 128, entry=e)[0] for e in ("v2", "v1")]
    for a, b in zip(clean, dirty):
        assert torch.equal(a, b)
    wl.poison_unreferenced(inp, 1e30)
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_v2(inp, 128, entry=e)[0])


def test_physical_relabelling_is_bitwise_invariant():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    r = wl.relabel_blocks(inp, seed=123)
    for e in ("v2", "v1"):
        assert torch.equal(run_v2(inp, 512, entry=e)[0], run_v2(r, 512, entry=e)[0])


# ---------------------------------------------------------------- device-side status

def test_bad_block_id_sets_status_and_stays_in_bounds():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    inp.block_tables[0, 5] = inp.key_cache.shape[0] + 7
    for e in ("v2", "v1"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        run_v2(inp, 512, entry=e, status=st)
        assert int(st.item()) & 1


def test_seq_len_over_hint_sets_status():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_v2(inp, 512, hint=600, status=st)
    assert int(st.item()) & 2


def test_clean_call_leaves_status_zero():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_v2(inp, 512, status=st)
    run_v2(inp, 512, entry="v1", status=st)
    assert int(st.item()) == 0


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.pa_selftest_wait_timeout(st, 20_000_000)
    torch.cuda.synchronize()
    assert int(st.item()) == cuda_lib.PA_STATUS_TIMEOUT
    full_check(wl.make_inputs(wl.TINY, device="cuda"), 512, entries=("v2",))


# ---------------------------------------------------------------- full-size workloads

def test_batch_decode_full_size_every_element():
    inp = wl.make_inputs(wl.BATCH, device="cuda")
    full_check(inp, wl.BATCH.partition_size, entries=("v2", "v1", "dispatch"))


def test_dispatch_rule(cuda_lib):
    """V1 when the longest sequence fits one partition, or fits two and V1's grid (sequences x
    KV heads) has at most one CTA per SM; else V2."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert cuda_lib.pa_decode_choose(32, 8, 512, 512) == 1
    assert cuda_lib.pa_decode_choose(4096, 8, 300, 512) == 1
    assert cuda_lib.pa_decode_choose(1, 4, 513, 512) == 1          # two partitions, 4 CTAs
    assert cuda_lib.pa_decode_choose(1, 2, 1000, 512) == 1         # the tiny workload
    assert cuda_lib.pa_decode_choose(sms, 1, 1024, 512) == 1
    assert cuda_lib.pa_decode_choose(sms + 1, 1, 1024, 512) == 2
    assert cuda_lib.pa_decode_choose(1, 4, 1025, 512) == 2         # three partitions
    assert cuda_lib.pa_decode_choose(512, 8, 1024, 512) == 2
    assert cuda_lib.pa_decode_choose(1, 4, 100000, 1024) == 2


@pytest.mark.parametrize("P", [512, 1024])
def test_long_100k_full_size_every_element(P):
    inp = wl.make_inputs(wl.LONG, device="cuda")
    full_check(inp, P, entries=("v2",))


def _sampled(inp, P, seqs, heads):
    sub = compact_subset(inp, seqs)
    prob = oracle_problem(sub)
    pairs = [(i, h) for i in range(len(seqs)) for h in heads]
    ref = oracle.decode(prob, pairs=pairs)
    out, tmp, es, ml = run_v2(inp, P, entry="v2")
    g = torch.stack([out[b, h] for b in seqs for h in heads])
    check_out(g, ref, inp.workload.dtype, what=inp.workload.name)
    sel = torch.tensor(seqs, device=tmp.device)
    check_partitions(sub, P, tmp[sel], es[sel], ml[sel], pairs=pairs, prob=prob)


def test_ragged_serving_full_size_sampled():
    inp = wl.make_inputs(wl.RAGGED, device="cuda")
    lens = inp.seq_lens.tolist()
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    seqs = sorted({order[0], order[1], order[len(lens) // 2], order[-2], order[-1]})
    _sampled(inp, wl.RAGGED.partition_size, seqs, heads=range(0, 64, 5))


def test_stress_full_size_sampled():
    inp = wl.make_inputs(wl.STRESS, device="cuda")
    _sampled(inp, wl.STRESS.partition_size, [0, 7], heads=[0, 9, 31, 63])
