"""pa_decode_v2_static: the decode entry point that allocates nothing.

It serves callers that cannot call cudaMalloc -- a framework that owns all
device memory, a runtime with a fixed budget, a hot path where allocating
would synchronise the device -- by keeping the phase-1 intermediates in an
array inside the library.  These tests call it through the C ABI twice in a
row on differently shaped problems (the second call finds the first call's
leftovers in the shared array) and compare each output with pa_decode_v2 on
the same inputs, using the parity tolerance for `out`.  The file is named so
that pytest collects it last.
"""
import pytest
import torch

import workloads as wl
from parity_util import check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _reference(pa, inp, P):
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


def test_two_calls_in_a_row_match_pa_decode_v2(cuda_lib):
    pa = cuda_lib
    first = wl.make_inputs(wl.TINY, device="cuda")
    w2 = wl.Workload("no_alloc_second", 4, 32, 4, 128, 16, 512, wl.BF16, "list",
                     seq_lens=(3000, 17, 1024, 9000), seed=4242)
    second = wl.make_inputs(w2, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    out1 = _static(pa, first, 512, status)
    out2 = _static(pa, second, 512, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    for inp, got in ((first, out1), (second, out2)):
        ref = _reference(pa, inp, 512)
        torch.cuda.synchronize()
        check_out(got, ref.cpu().double().numpy(), inp.workload.dtype,
                  what=f"static/{inp.workload.name}")


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
