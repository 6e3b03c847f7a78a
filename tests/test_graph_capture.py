"""The entry points inside a CUDA graph: captured once, replayed, bit for bit the eager call.

Serving loops capture each decode step into a graph; the library launches only
on the caller's stream, allocates nothing and never synchronises, so a capture
holds the whole call (tensor maps are encoded on the host at capture time).
Covered: the single-token dispatch (V2 with the merge), the multi-query
dispatch on the tcgen05 kernel, and the bf16 path through the binary16 copy of
V (the offsets pass, the copy pass, the attention kernel and the merge).
"""
import pytest
import torch

import workloads as wl
from parity_util import mq

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(0)


def captured_equals_eager(run):
    """run() launches one call on the current stream and returns its output tensor."""
    eager = run().clone()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()  # a warm call on the capture stream (descriptor caches, function attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = run()
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_single_token_dispatch_in_a_graph():
    import paged_kv_decode_v2_gb300 as pa
    w = wl.Workload("graph_v2", 6, 32, 8, 128, 16, 256, wl.BF16, "list",
                    seq_lens=(1, 300, 1500, 2048, 77, 999), seed=9900)
    inp = wl.make_inputs(w, device="cuda")
    S, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    assert pa.pa_decode_choose(S, w.num_kv_heads, cap, 256) == 2
    tmp, es, ml = pa.alloc_workspace(S, H, D, pa.num_partitions(cap, 256))
    out = torch.empty_like(inp.query)

    def run():
        pa.pa_decode(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                     w.scale, 256, out, tmp, es, ml)
        return out
    captured_equals_eager(run)


@pytest.mark.parametrize("q_len,G,dtype", [(16, 4, wl.BF16), (40, 4, wl.BF16), (40, 4, wl.F16),
                                           (256, 4, wl.BF16)])
def test_multi_query_dispatch_in_a_graph(q_len, G, dtype):
    """64 rows (one-tile V2); 160 rows: two tiles for fp16, one with hi + lo P for bf16; 1024
    bf16 rows: two tiles through the binary16 copy."""
    import paged_kv_decode_v2_gb300 as pa
    inp = wl.make_inputs(mq("graph_mq", q_len, G, (300, 1100, 2000), P=512, dtype=dtype,
                            seed=9950 + q_len + dtype), device="cuda")
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    tmp, es, ml = pa.alloc_workspace(S, H, D, 8 * pa.num_partitions(cap, 512), q_len=Q)
    out = torch.empty_like(inp.query)

    def run():
        pa.pa_decode_mq(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                        inp.seq_lens, inp.workload.scale, 512, out, tmp, es, ml)
        return out
    captured_equals_eager(run)
