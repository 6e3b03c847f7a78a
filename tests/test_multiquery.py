"""GPU parity for several new tokens per sequence (q_len > 1, causal prefix).

New token i of a sequence with L tokens (the q_len new ones included) sees
keys t <= L - q_len + i.  The CUDA path (pa_decode_v2_mq / pa_decode_v1_mq
through the C ABI) is compared element by element with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import check_mq, check_out, mq, run_mq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)


@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_mq_fuzz(q_len, G, dtype):
    P = 64
    lens = (1, q_len - 1 or 1, q_len, P - 1, P, P + 1, P + q_len, 3 * P + 5, 200)
    w = mq("mq_fuzz", q_len, G, lens, P=P, dtype=dtype, seed=4000 + 13 * q_len + G + dtype)
    check_mq(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("G", [1, 8])
def test_mq_empty_sequences_mixed_in(G):
    """Zero-length sequences between others: V1 writes zero rows, V2 no partition and the merge
    zero rows (the mma.sync kernel: q_len * G < 64)."""
    w = mq("mq_empty", 4, G, (0, 70, 0, 2, 500, 0), P=64, seed=4500 + G)
    ref = check_mq(wl.make_inputs(w, device="cuda"), 64)
    assert (ref[0] == 0).all() and (ref[2] == 0).all() and (ref[5] == 0).all()


@pytest.mark.parametrize("q_len,G", [(4, 8), (8, 4), (3, 16), (64, 1), (16, 8)])
def test_mq_rows_split_over_ctas(q_len, G):
    """More than 16 query rows per KV head: rows split over side-by-side CTAs."""
    lens = (q_len, 2 * q_len + 3, 700)
    w = mq("mq_split", q_len, G, lens, P=256, seed=5000 + q_len + G)
    check_mq(wl.make_inputs(w, device="cuda"), 256)


@pytest.mark.parametrize("D,bs", [(64, 32), (256, 16), (128, 64), (128, 8), (64, 8)])
def test_mq_other_shapes(D, bs):
    w = mq("mq_shapes", 4, 4, (5, 130, 333), bs=bs, P=128, D=D, seed=6000 + D + bs)
    check_mq(wl.make_inputs(w, device="cuda"), 128)


@pytest.mark.parametrize("q_len,G,bs,P", [(3, 4, 16, 300), (4, 8, 32, 40), (8, 2, 64, 100)])
def test_mq_partition_not_a_multiple_of_block_size(q_len, G, bs, P):
    lens = (1, q_len, P - 1, P + 1, P + q_len, 2 * P + 7, 650)
    w = mq("mq_pnb", q_len, G, lens, bs=bs, P=P, seed=6500 + q_len + G + bs + P)
    check_mq(wl.make_inputs(w, device="cuda"), P)


def test_mq_dispatch_rule_and_entry(cuda_lib):
    """pa_decode_mq runs the variant pa_decode_mq_choose names, at the partition size
    pa_decode_mq_partition names (bitwise the same output as that entry point)."""
    import paged_kv_decode_v2_gb300 as pa
    # batch decode shapes (32 seqs, 32 / 8 heads, up to 8192 tokens, P = 512)
    assert pa.pa_decode_mq_choose(32, 2, 32, 8, 128, 8192, 512) == 2   # 8 rows per KV head
    assert pa.pa_decode_mq_choose(32, 4, 32, 8, 128, 8192, 512) == 2   # 16 rows (mma.sync)
    assert pa.pa_decode_mq_partition(32, 4, 32, 8, 128, 8192, 512) == 1024
    assert pa.pa_decode_mq_partition(32, 1, 32, 8, 128, 8192, 512) == 512   # one new token
    assert pa.pa_decode_mq_choose(32, 4, 32, 8, 128, 1024, 512) == 1   # one 1024 partition
    for q in (8, 16, 32):                                                # 32..128 rows (tcgen05)
        assert pa.pa_decode_mq_choose(32, q, 32, 8, 128, 8192, 512) == 2
        assert pa.pa_decode_mq_partition(32, q, 32, 8, 128, 8192, 512) == 2048
    assert pa.pa_decode_mq_partition(32, 16, 32, 8, 128, 8192, 4096) == 4096
    assert pa.pa_decode_mq_choose(32, 16, 32, 8, 128, 2048, 512) == 1   # one 2048 partition
    assert pa.pa_decode_mq_partition(32, 16, 32, 8, 128, 2048, 512) == 0
    assert pa.pa_decode_mq_choose(32, 64, 32, 8, 128, 8192, 512) == 1  # 256 rows: V1
    assert pa.pa_decode_mq_choose(1, 16, 32, 4, 128, 100000, 512) == 2  # one long sequence:
    sms = torch.cuda.get_device_properties(0).multi_processor_count   # one wave of 2 CTAs per SM
    parts = 2 * sms // 4
    assert pa.pa_decode_mq_partition(1, 16, 32, 4, 128, 100000, 512) == -(-(-(-100000 // parts)) // 64) * 64
    # chunked prefill (2 x 2048 new tokens after 30K, 32 / 8 heads): 1024 V1 CTAs in waves of
    # 2 per SM; two partitions when they pack the waves better
    n, slots = 2 * 8 * 64, 2 * sms
    w1, w2 = -(-n // slots), -(-2 * n // slots)
    two = 10 * n < 9 * slots * w1 and w2 < 2 * w1
    assert pa.pa_decode_mq_choose(2, 2048, 32, 8, 128, 32768, 512) == (2 if two else 1)
    assert pa.pa_decode_mq_partition(2, 2048, 32, 8, 128, 32768, 512) == (16384 if two else 0)
    assert pa.pa_decode_mq_choose(4, 1024, 32, 8, 128, 4096, 512) == 1     # short CTAs: V1
    parts = 2 * sms // 8                                                  # 256 rows: two row tiles
    assert pa.pa_decode_mq_partition(1, 32, 32, 4, 128, 100000, 512) == -(-(-(-100000 // parts)) // 64) * 64
    assert pa.pa_decode_mq_partition(1, 16, 32, 4, 128, 20000, 512) == 512  # 160 CTAs at 512
    assert pa.pa_decode_mq_choose(1, 16, 32, 4, 128, 512, 512) == 1     # one partition
    for (q_len, G, lens, P) in ((4, 4, (3, 100, 700, 1500), 256),
                                (16, 4, (3, 100, 2500, 6000, 777), 256)):
        w = mq("mq_dispatch", q_len, G, lens, P=P, seed=79 + q_len)
        inp = wl.make_inputs(w, device="cuda")
        S, Q, H, D = inp.query.shape
        cap = inp.block_tables.shape[1] * w.block_size
        want = pa.pa_decode_mq_choose(S, Q, H, w.num_kv_heads, D, cap, P)
        part = pa.pa_decode_mq_partition(S, Q, H, w.num_kv_heads, D, cap, P)
        assert (want == 1) == (part == 0)
        ref = run_mq(inp, part if want == 2 else P, entry="v1" if want == 1 else "v2")[0]
        tmp, es, ml = pa.alloc_workspace(S, H, D, pa.num_partitions(cap, P), q_len=Q)
        out = torch.full_like(inp.query, float("nan"))
        pa.pa_decode_mq(inp.query, inp.key_cache, inp.value_cache, inp.block_tables,
                        inp.seq_lens, w.scale, P, out, tmp, es, ml)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        check_out(out, oracle.decode(oracle.Problem.from_arrays(wl.to_oracle_arrays(inp))),
                  w.dtype, what=f"mq_dispatch q{q_len}")


def test_mq_single_token_matches_the_single_query_entry():
    import paged_kv_decode_v2_gb300 as pa
    inp = wl.make_inputs(wl.TINY, device="cuda")
    S, H, D = inp.query.shape
    tmp, es, ml = pa.alloc_workspace(S, H, D, 2)
    a = torch.empty_like(inp.query)
    pa.pa_decode_v2(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                    wl.TINY.scale, 512, a, tmp, es, ml)
    b = torch.empty_like(inp.query)[:, None]
    tmp2, es2, ml2 = pa.alloc_workspace(S, H, D, 2, q_len=1)
    pa.pa_decode_v2_mq(inp.query[:, None].contiguous(), inp.key_cache, inp.value_cache,
                       inp.block_tables, inp.seq_lens, wl.TINY.scale, 512, b, tmp2, es2, ml2)
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])


def test_mq_speculative_batch_full_size():
    """Batch decode (32 seqs up to 8192 tokens, 32/8 heads) checking 4 speculated tokens each."""
    w = wl.BATCH.with_(name="batch_spec4", q_len=4)
    inp = wl.make_inputs(w, device="cuda")
    check_mq(inp, w.partition_size)


def test_mq_rejects_bad_q_len(cuda_lib):
    lib = cuda_lib.load()
    FAKE = 0x10000
    args = [FAKE] * 5 + [1, 0, 8, 2, 128, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_v1_mq(*args, 0, FAKE, None, None) == cuda_lib.PA_ERR_INVALID_ARG
    args = [FAKE] * 5 + [1, 4097, 8, 2, 128, 128, 16, 63, 0, 0.088]
    assert lib.pa_decode_v1_mq(*args, 0, FAKE, None, None) == cuda_lib.PA_ERR_UNSUPPORTED


def test_mq_unreferenced_slots_and_relabelling():
    """Poison never reaches the output; relabelling physical blocks changes nothing (bitwise)."""
    w = mq("mq_poison", 4, 4, (3, 37, 200, 64), bs=16, P=64, seed=77)
    inp = wl.make_inputs(w, device="cuda", max_blocks=20)
    clean = [run_mq(inp, 64, entry=e)[0] for e in ("v2", "v1")]
    wl.poison_unreferenced(inp, float("nan"))
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_mq(inp, 64, entry=e)[0])
    r = wl.relabel_blocks(inp, seed=9)
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_mq(r, 64, entry=e)[0])


def test_mq_bad_block_id_sets_status():
    w = mq("mq_status", 2, 4, (100, 300), P=64, seed=78)
    inp = wl.make_inputs(w, device="cuda")
    inp.block_tables[1, 3] = inp.key_cache.shape[0] + 1
    for e in ("v2", "v1"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        run_mq(inp, 64, entry=e, status=st)
        assert int(st.item()) & 1


def _random_mq_cases(n, seed):
    """n seeded (q_len, G, D, bs, P, dtype, lens) draws over the shapes the entry points take."""
    import random
    rng = random.Random(seed)
    cases = []
    for k in range(n):
        q_len = rng.choice([2, 3, 5, 8, 13, 16, 33, 64, 100, 200])
        G = rng.choice([1, 2, 4, 8, 16])
        D = rng.choice([64, 128, 128, 256])
        bs = rng.choice([8, 16, 16, 32, 64])
        P = rng.choice([bs, 4 * bs, 512, rng.randint(1, 700)])
        dtype = rng.choice([wl.F16, wl.BF16])
        S = rng.randint(1, 4)
        lens = tuple(rng.choice([0, 1, rng.randint(1, q_len + 2), rng.randint(1, 1500)]) for _ in range(S))
        cases.append((q_len, G, D, bs, P, dtype, lens, 7000 + k))
    return cases


@pytest.mark.parametrize("case", _random_mq_cases(32, 20261203), ids=lambda c: f"q{c[0]}g{c[1]}d{c[2]}b{c[3]}p{c[4]}")
def test_mq_random_shapes_default_dispatch(case):
    """Seeded random shapes through the default kernel choice (mma.sync below 32 rows per KV head,
    a tcgen05 kernel from 32), V1 and V2, element by element against the oracle."""
    q_len, G, D, bs, P, dtype, lens, seed = case
    w = mq("mq_random", q_len, G, lens, bs=bs, P=P, D=D, dtype=dtype, seed=seed)
    check_mq(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("case", _random_mq_cases(12, 20261204), ids=lambda c: f"q{c[0]}g{c[1]}d{c[2]}b{c[3]}p{c[4]}")
def test_mq_random_shapes_through_the_dispatch(case):
    """Seeded random shapes through pa_decode_mq, whose V2 may run on partitions coarser than the
    caller's (pa_decode_mq_partition), element by element against the oracle."""
    import paged_kv_decode_v2_gb300 as pa
    q_len, G, D, bs, P, dtype, lens, seed = case
    w = mq("mq_dispatch_random", q_len, G, lens, bs=bs, P=P, D=D, dtype=dtype, seed=seed + 50)
    inp = wl.make_inputs(w, device="cuda")
    S, Q, H, Dh = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    tmp, es, ml = pa.alloc_workspace(S, H, Dh, max(1, pa.num_partitions(cap, P)), q_len=Q)
    out = torch.full_like(inp.query, float("nan"))
    pa.pa_decode_mq(inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens,
                    w.scale, P, out, tmp, es, ml)
    torch.cuda.synchronize()
    check_out(out, oracle.decode(oracle.Problem.from_arrays(wl.to_oracle_arrays(inp))), dtype,
              what="mq_dispatch_random")
