"""pa_decode_v2_static: the decode entry point that allocates nothing.

It serves callers that cannot call cudaMalloc -- a framework that owns all
device memory, a runtime with a fixed budget, a hot path where allocating
would synchronise the device -- by keeping the phase-1 intermediates in an
array inside the library.  These tests call it through the C ABI several
times in a row on differently shaped problems, so each call finds the
previous call's leftovers in the shared array, and check every output
against the fp64 oracle at the parity tolerance and, bitwise, against
pa_decode_v2 (the same kernels) on the same inputs.  The file is named so
that pytest collects it last.
"""
import pytest
import torch

import workloads as wl
from parity_util import check_out, oracle_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _with_workspace(pa, inp, P):
    """pa_decode_v2 with caller-allocated intermediates."""
    w = inp.workload
    S, H, D = inp.query.shape
    npmax = pa.num_partitions(inp.block_tables.shape[1] * w.block_size, P)
    tmp, es, ml = pa.alloc_workspace(S, H, D, npmax)
    out = torch.empty_like(inp.query)
    pa.pa_decode_v2(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                    w.scale, P, out, tmp, es, ml)
    return out


def _static(pa, inp, P, status):
    w = inp.workload
    out = torch.full_like(inp.query, float("nan"))
    pa.pa_decode_v2_static(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                           inp.seq_lens, w.scale, P, out, status=status)
    return out


def _check_calls(pa, calls):
    """Runs the static entry point on each (inputs, P) in order, then checks each
    output against the oracle and bitwise against pa_decode_v2."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [_static(pa, inp, P, status) for inp, P in calls]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (inp, P), got in zip(calls, outs):
        what = f"static/{inp.workload.name}/P{P}"
        check_out(got, oracle_out(inp), inp.workload.dtype, what=what)
        ref = _with_workspace(pa, inp, P)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"{what}: differs from pa_decode_v2 on the same inputs"


def test_small_then_larger_call(cuda_lib):
    first = wl.make_inputs(wl.TINY, device="cuda")
    w2 = wl.Workload("no_alloc_second", 4, 32, 4, 128, 16, 512, wl.BF16, "list",
                     seq_lens=(3000, 17, 1024, 9000), seed=4242)
    second = wl.make_inputs(w2, device="cuda")
    _check_calls(cuda_lib, [(first, 512), (second, 512)])


def test_large_call_then_smaller_calls_over_its_leftovers(cuda_lib):
    """A call that fills most of the array (the full batch-decode workload: 32 x 32
    x 16 partitions of 130 floats, 8.5 MB), then smaller calls with other head counts
    and partition sizes: every slot they read holds the first call's finite values
    until they overwrite it."""
    big = wl.make_inputs(wl.BATCH, device="cuda")
    w2 = wl.Workload("no_alloc_after_big", 3, 16, 16, 128, 32, 256, wl.F16, "list",
                     seq_lens=(700, 1, 2049), seed=4343)
    w3 = wl.Workload("no_alloc_after_big_g8", 2, 16, 2, 128, 16, 100, wl.BF16, "list",
                     seq_lens=(1000, 333), seed=4444)
    _check_calls(cuda_lib, [(big, 512), (wl.make_inputs(w2, device="cuda"), 256),
                            (wl.make_inputs(w3, device="cuda"), 100)])


def test_rejects_sizes_beyond_the_array(cuda_lib):
    pa = cuda_lib
    inp = wl.make_inputs(wl.RAGGED.with_(seq_len_kind="list", num_seqs=64,
                                         seq_lens=tuple([32768] + [16] * 63)), device="cuda")
    out = torch.full_like(inp.query, 7.0)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_v2_static(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                               inp.seq_lens, inp.workload.scale, 512, out)
    assert e.value.code == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 7.0).all()
