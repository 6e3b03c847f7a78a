"""GPU parity of the CUDA-core (SIMT) attention kernel against the fp64 oracle.

pa_set_rows_kernel(5) sends every call with up to 8 query rows per KV head to
the SIMT kernel (Q.K and the softmax reduced with warp shuffles, P.V as scalar
FMAs); the default mma.sync kernel is compared on the same inputs where the
two must agree only within the tolerances (different summation orders).
"""
import pytest
import torch

import workloads as wl
from parity_util import check_mq, mq, run_v2
from test_parity import full_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _simt(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(5)
    yield
    cuda_lib.pa_set_rows_kernel(0)
    cuda_lib.pa_set_launch_config(0, 0)


def _kernel_names(pa, mode, inp):
    from torch.profiler import ProfilerActivity, profile
    pa.pa_set_rows_kernel(mode)
    try:
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            run_v2(inp, 512, entry="v2")
            torch.cuda.synchronize()
    finally:
        pa.pa_set_rows_kernel(5)
    return [e.name for e in prof.events() if "attn_kernel" in e.name]


def test_mode_5_runs_the_simt_kernel(cuda_lib):
    """The kernel that runs under pa_set_rows_kernel(5) is the CUDA-core one (its name, as
    the CUDA profiler records it), and under mode 0 the mma.sync one."""
    inp = wl.make_inputs(wl.TINY, device="cuda")
    _kernel_names(cuda_lib, 0, inp)  # the profiler's first session may miss kernels
    simt = _kernel_names(cuda_lib, 5, inp)
    mma = _kernel_names(cuda_lib, 0, inp)
    if not simt and not mma:
        pytest.skip("the CUDA profiler recorded no kernel names here")
    assert simt and all("simt_attn_kernel" in n for n in simt), simt
    assert mma and not any("simt" in n or "tc_attn" in n for n in mma), mma


def test_tiny_workload_all_entries():
    full_check(wl.make_inputs(wl.TINY, device="cuda"), wl.TINY.partition_size)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("P", [64, 512])
def test_simt_fuzz_grid(dtype, bs, G, P):
    lens = (1, bs - 1, bs, bs + 1, P - 1, P, P + 1, 2 * P + bs + 3, 3 * P + 5)
    w = wl.Workload("simt_fuzz", len(lens), 2 * G, 2, 128, bs, P, dtype, "list", seq_lens=lens,
                    seed=9000 + 7 * G + bs + P + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_simt_head_dims(D, bs, G, dtype):
    P = 128
    lens = (1, bs - 1, bs + 1, P - 1, P + 1, 3 * P + bs + 3)
    w = wl.Workload("simt_d", len(lens), 2 * G, 2, D, bs, P, dtype, "list", seq_lens=lens,
                    seed=9500 + D + 7 * G + bs + dtype)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("bs,P", [(16, 300), (32, 200), (64, 100), (16, 17), (8, 12)])
@pytest.mark.parametrize("G", [1, 4])
def test_simt_partition_not_a_multiple_of_block_size(bs, P, G):
    lens = sorted({1, bs - 1, bs + 1, P - 1, P, P + 1, 2 * P + 3, 3 * P + bs + 5, 700})
    w = wl.Workload("simt_pnb", len(lens), 2 * G, 2, 128, bs, P, wl.BF16, "list",
                    seq_lens=tuple(lens), seed=9700 + bs + P + G)
    full_check(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("warps,stages", [(1, 1), (2, 2), (8, 1), (3, 3), (8, 4)])
def test_simt_launch_shapes(cuda_lib, warps, stages):
    w = wl.Workload("simt_shapes", 4, 8, 2, 128, 16, 256, wl.BF16, "list",
                    seq_lens=(1, 700, 2049, 4096), seed=9800)
    inp = wl.make_inputs(w, device="cuda")
    cuda_lib.pa_set_launch_config(warps, stages)
    try:
        full_check(inp, 256, entries=("v2", "v1"))
    finally:
        cuda_lib.pa_set_launch_config(0, 0)


@pytest.mark.parametrize("q_len,G", [(2, 4), (8, 1), (4, 2), (3, 2), (2, 1)])
def test_simt_several_new_tokens(q_len, G):
    """Up to 8 query rows per KV head from q_len new tokens x G heads, causal prefix."""
    P = 64
    lens = (1, q_len, P - 1, P + q_len, 3 * P + 5, 200)
    w = mq("simt_mq", q_len, G, lens, P=P, seed=9900 + 13 * q_len + G)
    check_mq(wl.make_inputs(w, device="cuda"), P)


def test_simt_empty_sequences():
    w = wl.Workload("simt_empty", 5, 8, 2, 128, 16, 64, wl.BF16, "list",
                    seq_lens=(0, 1, 0, 65, 0), seed=77)
    inp = wl.make_inputs(w, device="cuda", max_blocks=8)
    full_check(inp, 64)
    for e in ("v2", "v1"):
        out = run_v2(inp, 64, entry=e)[0]
        assert (out[0] == 0).all() and (out[2] == 0).all() and (out[4] == 0).all()


@pytest.mark.parametrize("bs", [8, 16])
def test_simt_unreferenced_and_tail_slots_never_reach_the_output(bs):
    w = wl.Workload("simt_poison", 4, 8, 2, 128, bs, 128, wl.BF16, "list",
                    seq_lens=(37, 16, 300, 5), seed=21 + bs)
    inp = wl.make_inputs(w, device="cuda", max_blocks=480 // bs)
    clean = [run_v2(inp, 128, entry=e)[0] for e in ("v2", "v1")]
    wl.poison_unreferenced(inp, float("nan"))
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_v2(inp, 128, entry=e)[0])


def test_simt_relabelling_is_bitwise_invariant():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    r = wl.relabel_blocks(inp, seed=123)
    for e in ("v2", "v1"):
        assert torch.equal(run_v2(inp, 512, entry=e)[0], run_v2(r, 512, entry=e)[0])


def test_simt_bad_block_id_sets_status():
    inp = wl.make_inputs(wl.TINY, device="cuda")
    inp.block_tables[0, 5] = inp.key_cache.shape[0] + 7
    for e in ("v2", "v1"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        run_v2(inp, 512, entry=e, status=st)
        assert int(st.item()) & 1


def test_simt_batch_decode_full_size_every_element():
    """The batch-decode workload (G = 4) on the SIMT kernel, every output element."""
    inp = wl.make_inputs(wl.BATCH, device="cuda")
    full_check(inp, wl.BATCH.partition_size, entries=("v2",))


def test_simt_long_100k_full_size_every_element():
    """The 100K-token workload (G = 8) on the SIMT kernel, every output element."""
    inp = wl.make_inputs(wl.LONG, device="cuda")
    full_check(inp, 512, entries=("v2",))

