"""GPU parity at softmax scales other than 1/sqrt(head_dim): zero, negative and large.

The kernels fold a positive scale into the exponent on tiles every row sees
whole (max(s) * scale = max(s * scale) only when scale > 0) and take the
masked path otherwise, so a zero or negative scale exercises the other branch
on every tile.  Each kernel form is compared element by element with the fp64
oracle at the same scale: the mma.sync kernel (V2, V1, fused), the CUDA-core
kernel, the multi-query mma.sync kernel, both tcgen05 kernels, and the bf16
path through the binary16 copy of V.
"""
import pytest
import torch

import oracle
import workloads as wl
from parity_util import check_out, mq

pytestmark = pytest.mark.gpu

SCALES = [0.0, -0.06, 0.5]


@pytest.fixture(autouse=True)
def _defaults(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(0)
    yield
    cuda_lib.pa_set_rows_kernel(0)


def reference(inp, scale):
    arrays = wl.to_oracle_arrays(inp)
    arrays["scale"] = scale
    return oracle.decode(oracle.Problem.from_arrays(arrays))


def single(G, seed, dtype=wl.BF16):
    lens = (1, 17, 300, 700, 1025)
    w = wl.Workload("scale_single", len(lens), 2 * G, 2, 128, 16, 256, dtype, "list",
                    seq_lens=lens, seed=seed)
    return wl.make_inputs(w, device="cuda")


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("entry", ["v2", "v1", "fused", "simt"])
def test_single_token(cuda_lib, scale, entry):
    import paged_kv_decode_v2_gb300 as pa
    inp = single(4, 9980 + SCALES.index(scale))
    S, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    tmp, es, ml = pa.alloc_workspace(S, H, D, pa.num_partitions(cap, 256))
    out = torch.full_like(inp.query, float("nan"))
    args = (inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens, scale)
    if entry == "v2":
        pa.pa_decode_v2(*args, 256, out, tmp, es, ml)
    elif entry == "v1":
        pa.pa_decode_v1(*args, out)
    elif entry == "fused":
        counters = pa.alloc_counters(S, 2)
        pa.pa_decode_v2_fused(*args, 256, out, tmp, es, ml, counters)
    else:
        cuda_lib.pa_set_rows_kernel(5)
        pa.pa_decode_v2(*args, 256, out, tmp, es, ml)
    torch.cuda.synchronize()
    check_out(out, reference(inp, scale), wl.BF16, what=f"scale {scale} {entry}")


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("q_len,G,mode,dtype", [(4, 4, 0, wl.BF16),     # 16 rows: mma.sync
                                               (16, 4, 3, wl.BF16),    # 64 rows: one tile, half Q
                                               (40, 4, 4, wl.F16),     # 160 rows: two tiles
                                               (40, 4, 4, wl.BF16)])   # bf16 via the binary16 copy
def test_multi_query(cuda_lib, scale, q_len, G, mode, dtype):
    import paged_kv_decode_v2_gb300 as pa
    cuda_lib.pa_set_rows_kernel(mode)
    inp = wl.make_inputs(mq("scale_mq", q_len, G, (q_len, 300, 1100, 2000), P=512, dtype=dtype,
                            seed=9990 + q_len + mode + SCALES.index(scale)), device="cuda")
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * 16
    tmp, es, ml = pa.alloc_workspace(S, H, D, 8 * pa.num_partitions(cap, 512), q_len=Q)
    out = torch.full_like(inp.query, float("nan"))
    pa.pa_decode_mq(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                    scale, 512, out, tmp, es, ml)
    torch.cuda.synchronize()
    check_out(out, reference(inp, scale), dtype, what=f"scale {scale} mq rows {q_len * G}")
