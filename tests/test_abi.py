"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pa_decode.h")

FAKE = 0x10000  # a 64 KiB-aligned address that is never dereferenced on these paths


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("pa_decode_v2", "pa_decode_v1", "pa_decode", "pa_decode_v2_phase1",
              "pa_decode_v2_phase2", "pa_v2_num_partitions", "pa_v2_workspace_bytes",
              "pa_status_string", "pa_decode_choose", "pa_selftest_wait_timeout",
              "pa_set_launch_config", "pa_set_rows_kernel", "pa_set_merge_form", "pa_decode_mq",
              "pa_decode_mq_choose"):
        assert n in names


def test_library_exports_every_declared_symbol(cuda_lib):
    lib = ctypes.CDLL(cuda_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_num_partitions(cuda_lib):
    assert cuda_lib.num_partitions(100000, 1024) == 98
    assert cuda_lib.num_partitions(100000, 512) == 196
    assert cuda_lib.num_partitions(1000, 512) == 2
    assert cuda_lib.num_partitions(0, 512) == 0
    assert cuda_lib.num_partitions(512, 512) == 1
    assert cuda_lib.num_partitions(513, 512) == 2
    assert cuda_lib.num_partitions(-1, 512) == -1
    assert cuda_lib.num_partitions(10, 0) == -1


def test_workspace_bytes(cuda_lib):
    assert cuda_lib.workspace_bytes(1, 32, 128, 196) == 32 * 196 * 130 * 4
    assert cuda_lib.workspace_bytes(0, 32, 128, 196) == 0


def test_status_strings(cuda_lib):
    assert cuda_lib.status_string(0) == "PA_OK"
    assert cuda_lib.status_string(3) == "PA_ERR_WORKSPACE"
    assert cuda_lib.status_string(99) == "PA_UNKNOWN"


def _v2(lib, **kw):
    a = dict(query=FAKE, key_cache=FAKE, value_cache=FAKE, block_tables=FAKE, seq_lens=FAKE,
             num_seqs=1, num_heads=8, num_kv_heads=2, head_dim=128, num_blocks=128, block_size=16,
             max_blocks=63, hint=0, scale=0.088, partition_size=512, dtype=0, out=FAKE, tmp=FAKE,
             es=FAKE, ml=FAKE, max_np=2, status=None, stream=None)
    a.update(kw)
    return lib.pa_decode_v2(a["query"], a["key_cache"], a["value_cache"], a["block_tables"],
                            a["seq_lens"], a["num_seqs"], a["num_heads"], a["num_kv_heads"],
                            a["head_dim"], a["num_blocks"], a["block_size"], a["max_blocks"],
                            a["hint"], a["scale"], a["partition_size"], a["dtype"], a["out"],
                            a["tmp"], a["es"], a["ml"], a["max_np"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(query=None), 1),
    (dict(out=None), 1),
    (dict(tmp=None), 1),
    (dict(num_seqs=0), 1),
    (dict(num_heads=6, num_kv_heads=4), 1),
    (dict(dtype=2), 1),
    (dict(scale=float("nan")), 1),
    (dict(head_dim=96), 2),
    (dict(head_dim=512), 2),
    (dict(block_size=48), 2),
    (dict(block_size=4), 2),
    (dict(num_heads=256, num_kv_heads=2), 2),
    (dict(partition_size=-16), 1),
    (dict(partition_size=0), 1),
    (dict(key_cache=FAKE + 8), 1),
    (dict(query=FAKE + 2), 1),
    (dict(out=FAKE + 2), 1),
    (dict(block_tables=FAKE + 2), 1),
    (dict(seq_lens=FAKE + 1), 1),
    (dict(status=FAKE + 2), 1),
    (dict(max_np=1), 3),
    (dict(hint=600, max_np=1), 3),
])
def test_invalid_arguments_fail_before_launch(cuda_lib, kw, code):
    assert _v2(cuda_lib.load(), **kw) == code


def test_invalid_arguments_v1_and_dispatch(cuda_lib):
    lib = cuda_lib.load()
    args = [FAKE] * 5 + [1, 8, 2, 80, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_v1(*args, 0, FAKE, None, None) == 2
    args = [FAKE] * 5 + [1, 8, 2, 128, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_v1(*args, 0, None, None, None) == 1
    assert lib.pa_decode_v1(*args, 0, FAKE + 2, None, None) == 1   # out must be 4-byte aligned
    assert lib.pa_decode(*args, -500, 0, FAKE, FAKE, FAKE, FAKE, 2, None, None) == 1
    assert lib.pa_decode_v2_phase2(FAKE, 1, 8, 128, 1000, 512, 0, FAKE, FAKE, FAKE, 1, FAKE,
                                   None, None) == 3
    assert lib.pa_decode_v2_phase2(None, 1, 8, 128, 1000, 512, 0, FAKE, FAKE, FAKE, 2, FAKE,
                                   None, None) == 1


def test_launch_config_override_validation(cuda_lib):
    assert cuda_lib.load().pa_set_launch_config(9, 2) == 1
    assert cuda_lib.load().pa_set_launch_config(4, 9) == 1
    assert cuda_lib.load().pa_set_launch_config(0, 0) == 0


def test_multi_query_dispatch_validation(cuda_lib):
    lib = cuda_lib.load()
    assert lib.pa_decode_mq_choose(0, 4, 32, 8, 128, 1000, 512) == -1
    assert lib.pa_decode_mq_choose(4, 0, 32, 8, 128, 1000, 512) == -1
    assert lib.pa_decode_mq_choose(4, 4, 30, 8, 128, 1000, 512) == -1
    assert lib.pa_decode_mq_choose(4, 4, 32, 8, 0, 1000, 512) == -1
    assert lib.pa_decode_mq_choose(4, 4, 32, 8, 128, 1000, 0) == -1
    args = [FAKE] * 5 + [1, 0, 8, 2, 128, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_mq(*args, 512, 0, FAKE, FAKE, FAKE, FAKE, 2, None, None) == 1
    args = [FAKE] * 5 + [1, 4, 8, 2, 128, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_mq(*args, 0, 0, FAKE, FAKE, FAKE, FAKE, 2, None, None) == 1


def test_merge_form_override_validation(cuda_lib):
    lib = cuda_lib.load()
    assert lib.pa_set_merge_form(-1) == 1
    assert lib.pa_set_merge_form(3) == 1
    for f in (2, 1, 0):
        assert lib.pa_set_merge_form(f) == 0


def test_rows_kernel_override_validation(cuda_lib):
    lib = cuda_lib.load()
    assert lib.pa_set_rows_kernel(-1) == 1
    assert lib.pa_set_rows_kernel(7) == 1
    assert lib.pa_set_rows_kernel(6) == 0
    assert lib.pa_set_rows_kernel(5) == 0
    assert lib.pa_set_rows_kernel(4) == 0
    assert lib.pa_set_rows_kernel(2) == 0
    assert lib.pa_set_rows_kernel(0) == 0


def test_selftest_rejects_bad_limits(cuda_lib):
    lib = cuda_lib.load()
    assert lib.pa_selftest_wait_timeout(None, 1000, None) == 1
    assert lib.pa_selftest_wait_timeout(FAKE + 2, 1000, None) == 1
    assert lib.pa_selftest_wait_timeout(FAKE, 0, None) == 1
    assert lib.pa_selftest_wait_timeout(FAKE, 3_000_000_000, None) == 1


def test_binding_refuses_cpu_tensors(cuda_lib):
    import torch
    import workloads as wl
    inp = wl.make_inputs(wl.TINY)
    out = torch.empty_like(inp.query)
    with pytest.raises(ValueError):
        cuda_lib.pa_decode_v1(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                              inp.seq_lens, 0.088, out)


def _static(lib, **kw):
    a = dict(num_seqs=1, num_heads=8, num_kv_heads=2, head_dim=128, num_blocks=128, block_size=16,
             max_blocks=63, hint=0, partition_size=512)
    a.update(kw)
    fn = lib.pa_decode_v2_static
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, P, P]
    fn.restype = I
    return fn(FAKE, FAKE, FAKE, FAKE, FAKE, a["num_seqs"], a["num_heads"], a["num_kv_heads"],
              a["head_dim"], a["num_blocks"], a["block_size"], a["max_blocks"], a["hint"], 0.088,
              a["partition_size"], 0, FAKE, None, None)


@pytest.mark.parametrize("kw", [
    # products far past 2^63 if multiplied out: must be rejected, not wrapped
    dict(num_seqs=2**31 - 1, num_heads=2**31 - 1, max_blocks=2**31 - 1, block_size=1,
         partition_size=1),
    dict(num_seqs=65535, num_heads=65535 * 64, num_kv_heads=65535, max_blocks=2**30, block_size=2),
    dict(head_dim=2**31 - 3),
    # just past the 16 MiB array: 32 x 32 x 32 partitions x 130 x 4 B = 17.0 MB
    dict(num_seqs=32, num_heads=32, num_kv_heads=8, max_blocks=1024, partition_size=512),
])
def test_static_entry_rejects_sizes_beyond_its_array_on_the_host(cuda_lib, kw):
    """The no-allocation entry point refuses, before any CUDA call, every size whose
    intermediates would not fit its array -- including sizes whose byte count would
    overflow a 64-bit product."""
    assert _static(cuda_lib.load(), **kw) == cuda_lib.PA_ERR_WORKSPACE


def test_fused_entry_rejects_missing_or_misaligned_counters(cuda_lib):
    lib = cuda_lib.load()
    args = [FAKE] * 5 + [1, 8, 2, 128, 128, 16, 63, 0, 0.088, 512, 0, FAKE, FAKE, FAKE, FAKE, 2]
    assert lib.pa_decode_v2_fused(*args, None, None, None) == 1
    assert lib.pa_decode_v2_fused(*args, FAKE + 2, None, None) == 1
    bad_out = list(args)
    bad_out[16] = None
    assert lib.pa_decode_v2_fused(*bad_out, FAKE, None, None) == 1
    small_ws = list(args)
    small_ws[-1] = 1
    assert lib.pa_decode_v2_fused(*small_ws, FAKE, None, None) == 3
