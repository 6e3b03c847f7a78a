"""GPU parity for the tcgen05 kernel: 128 query rows (new token i, head g of
the GQA group) per CTA, S = Q K^T and O += P V on the fifth-generation
tensor cores with S, P and O in tensor memory.

Every test forces each tcgen05 kernel form in turn (one 128-row query tile per
CTA, storing only 64 Q rows for KV heads of at most 64 rows; the same with the
whole Q tile stored; two tiles per CTA; pa_set_rows_kernel 3, 6 and 4) and
compares the CUDA path,
V2 (partials + merge) and V1, element by element with the fp64 oracle,
with the tolerances of parity_util: row counts below, at and above one CTA's
128 rows, every head_dim and block size, K/V tiles that end inside a block,
partitions that begin inside a block, K and V rings of one to five stages, chunked
prefill (a chunk of new tokens attending to a cached prefix and causally to
itself), poisoned caches and bad block ids.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import (OUT_ABS, check_mq, check_out, check_partitions, half_ulp, mq, ramp_scores,
                         oracle_problem, run_mq, run_v2)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[3, 6, 4], ids=["one_tile", "one_tile_full_q", "two_tiles"])
def _force_tc(request, cuda_lib):
    """Each test runs with the one-tile kernel (128 query rows per CTA; at most 64 rows store
    only their half of the Q tile), the one-tile kernel with the whole Q tile stored at every
    row count, and the two-tile kernel (two 128-row tiles sharing each 128-token K/V tile;
    head_dim 256 stays on one tile)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    cuda_lib.pa_set_rows_kernel(request.param)
    yield
    cuda_lib.pa_set_rows_kernel(0)
    cuda_lib.pa_set_launch_config(0, 0)


def check_single(inp, P):
    """q_len = 1 (query [S, H, D]) through pa_decode_v2 and pa_decode_v1."""
    prob = oracle_problem(inp)
    ref = oracle.decode(prob)
    for e in ("v2", "v1"):
        out, tmp, es, ml = run_v2(inp, P, entry=e)
        check_out(out, ref, inp.workload.dtype, what=f"{inp.workload.name}/{e}")
        if e == "v2":
            check_partitions(inp, P, tmp, es, ml, prob=prob)


@pytest.mark.parametrize("q_len,G", [(2, 16), (4, 8), (8, 4), (3, 16), (5, 4), (20, 4), (24, 4),
                                     (32, 4), (16, 8), (33, 4)])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_row_counts(q_len, G, dtype):
    """20 to 132 rows per KV head: a tile's rows in one, two, three or four warps (whole warps of
    padding rows idle), exactly one CTA, two CTAs."""
    P = 128
    lens = (1, q_len, 63, 64, 65, P - 1, P + 1, 2 * P + 70, 700)
    w = mq("tc_rows", q_len, G, lens, P=P, dtype=dtype, seed=8000 + 31 * q_len + G + dtype)
    check_mq(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("G", [1, 8, 64])
def test_tc_single_query(G):
    P = 256
    lens = (1, 64, 255, 257, 1000)
    w = wl.Workload("tc_q1", len(lens), 2 * G, 2, 128, 16, P, wl.BF16, "list", seq_lens=lens,
                    seed=8100 + G)
    check_single(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_head_dims_and_block_sizes(D, bs, dtype):
    P = 128
    lens = (5, bs - 1, bs + 1, 130, 333)
    w = mq("tc_shapes", 4, 8, lens, bs=bs, P=P, D=D, dtype=dtype, seed=8200 + D + bs + dtype)
    check_mq(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("k_stages,v_stages", [(1, 1), (3, 1), (1, 3), (2, 2), (5, 4)])
def test_tc_ring_stages(cuda_lib, k_stages, v_stages):
    """The K and V rings wrap many times (V1 walks 1000+ tokens)."""
    cuda_lib.pa_set_launch_config(v_stages, k_stages)
    w = mq("tc_stages", 8, 4, (700, 1100, 64), P=256, seed=8300 + 8 * k_stages + v_stages)
    check_mq(wl.make_inputs(w, device="cuda"), 256)


@pytest.mark.parametrize("bs,P", [(16, 100), (32, 300), (16, 8), (64, 1000), (8, 100), (8, 4)])
def test_tc_partition_not_a_multiple_of_block_size(bs, P):
    lens = (1, 8, P - 1, P + 1, 2 * P + 7, 650)
    w = mq("tc_pnb", 8, 4, lens, bs=bs, P=P, seed=8400 + bs + P)
    check_mq(wl.make_inputs(w, device="cuda"), P)


@pytest.mark.parametrize("q_len,prefix", [(128, 0), (128, 37), (300, 1000), (64, 4000)])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_chunked_prefill(q_len, prefix, dtype):
    """A chunk of q_len new tokens whose K/V are already in the cache after a
    prefix: new token i attends to the prefix and to chunk tokens <= i."""
    lens = (prefix + q_len, q_len + 5)
    w = mq("tc_prefill", q_len, 4, lens, P=512, dtype=dtype, seed=8500 + q_len + prefix + dtype)
    check_mq(wl.make_inputs(w, device="cuda"), 512)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_values_beyond_binary16(dtype):
    """V values of magnitude 2^16 and more in a few visible tokens (first, middle and last K/V
    tile of a sequence; fp16 storage gets values near its own limit instead), through every
    tcgen05 kernel form.

    Tolerance: the parity bound (2e-3 plus half an ulp of the output) assumes V of unit scale.
    P is rounded to the storage type before P.V (11 significant bits for fp16; hi + lo halves,
    about 16, for bf16), so each term p * v moves by at most 2^-12 of p * |v|; this test adds
    2^-11 * sum(p |v|) / l, the oracle's output on |V|, to that bound.  A large value lost or
    clamped anywhere on the way would miss it by far."""
    P = 512
    lens = (300, 1100, 2000)
    w = mq("tc_wide", 40, 4, lens, P=P, dtype=dtype, seed=8750 + dtype)  # 160 rows per KV head
    inp = wl.make_inputs(w, device="cuda")
    big = [7.0e4, -2.5e5, 65536.0, -1.0e6] if dtype == wl.BF16 else [6.0e4, -6.5e4, 3.0e4, -5.0e4]
    bs = w.block_size
    tables = inp.block_tables.cpu()
    for b, L in enumerate(lens):
        for k, t in enumerate((5, L // 2, L - 1)):
            blk = int(tables[b, t // bs])
            inp.value_cache[blk, :, t % bs, (7 * k + b) % w.head_dim] = big[(k + b) % len(big)]
    arrays = wl.to_oracle_arrays(inp)
    ref = oracle.decode(oracle.Problem.from_arrays(arrays))
    arrays["value_cache"] = arrays["value_cache"] & np.uint16(0x7FFF)  # |V|: sign bit cleared
    ref_abs = oracle.decode(oracle.Problem.from_arrays(arrays))
    tol = OUT_ABS + half_ulp(ref, dtype) + 2.0 ** -11 * ref_abs
    for e in ("v2", "v1"):
        out = run_mq(inp, P, entry=e)[0].cpu().to(torch.float64).numpy()
        assert np.isfinite(out).all(), e
        err = np.abs(out - ref)
        assert (err <= tol).all(), (e, int((err > tol).sum()), float((err - tol).max()))


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16])
@pytest.mark.parametrize("c,period", [(1.5, None), (0.3, None), (4.0, 256)])
def test_tc_rising_and_falling_scores(c, period, dtype):
    """On half the rows the running max grows past the rescale threshold every tile (c = 1.5), every
    few tiles (c = 0.3), or by ~22 per tile for four tiles and then repeats without growing (c = 4,
    period 256); on the others it never grows.  O is rescaled for some rows of a warp and not the
    rest; V2's partition statistics still report the true max.  Logits stay below ~130, where fp32
    scores keep the exp_sums tolerance.  fp16 as well as bf16, so that every P format runs the ramps
    (fp16 on two tiles: binary16 P, ~5, ~24 and ~65 in exp2 terms per 128-token tile)."""
    w = mq("tc_ramp", 8, 4, (700, 300, 1000, 65), P=256, dtype=dtype, seed=8900 + int(10 * c) + dtype)
    inp = ramp_scores(wl.make_inputs(w, device="cuda"), c, period)
    check_mq(inp, 256)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_empty_sequences_mixed_in(dtype):
    """Zero-length sequences between others (and a sequence shorter than q_len): V1 writes zero
    rows for them, V2 writes no partition and the merge zero rows."""
    lens = (0, 300, 0, 5, 1200, 0)
    w = mq("tc_empty", 16, 8, lens, P=256, dtype=dtype, seed=9000 + dtype)
    inp = wl.make_inputs(w, device="cuda")
    ref = check_mq(inp, 256)
    assert (ref[0] == 0).all() and (ref[2] == 0).all() and (ref[5] == 0).all()


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_tc_maximum_q_len(dtype):
    """q_len 4096, the largest the entry points take: 4096 new tokens after a 100-token prefix, one
    query head per KV head (4096 rows per KV head), sampled rows (first, last, tile and partition
    edges) of both heads, V1 and V2, against the oracle."""
    Q = 4096
    w = mq("tc_qmax", Q, 1, (Q + 100,), P=512, dtype=dtype, seed=9100 + dtype)
    inp = wl.make_inputs(w, device="cuda")
    prob = oracle_problem(inp)
    rows = [0, 1, 127, 128, 411, 412, 2047, 2048, Q - 129, Q - 1]
    pairs = [(r, h) for r in rows for h in range(w.num_heads)]
    ref = oracle.decode(prob, pairs=pairs)
    for e in ("v1", "v2"):
        out = run_mq(inp, 512, entry=e)[0]
        g = torch.stack([out[r // Q, r % Q, h] for r, h in pairs])
        check_out(g, ref, w.dtype, what=f"{w.name}/{e}")


def test_tc_agrees_with_the_mma_sync_kernel(cuda_lib):
    """Both kernels on the same inputs, each against the oracle and against the other."""
    w = mq("tc_vs_mma", 8, 4, (3, 100, 513, 900), P=256, seed=8600)
    inp = wl.make_inputs(w, device="cuda")
    ref = check_mq(inp, 256)
    tc_out = run_mq(inp, 256)[0]
    cuda_lib.pa_set_rows_kernel(1)
    mma_out = run_mq(inp, 256)[0]
    check_out(mma_out, ref, w.dtype, what="mma.sync")
    d = (tc_out.float() - mma_out.float()).abs().max().item()
    assert d <= 2 * 2e-3 + 2 ** -8, d


def test_tc_unreferenced_slots_and_relabelling():
    """Poison never reaches the output; relabelling physical blocks changes nothing (bitwise)."""
    w = mq("tc_poison", 8, 4, (3, 37, 200, 64), bs=16, P=64, seed=8700)
    inp = wl.make_inputs(w, device="cuda", max_blocks=20)
    clean = [run_mq(inp, 64, entry=e)[0] for e in ("v2", "v1")]
    wl.poison_unreferenced(inp, float("nan"))
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_mq(inp, 64, entry=e)[0])
    r = wl.relabel_blocks(inp, seed=11)
    for a, e in zip(clean, ("v2", "v1")):
        assert torch.equal(a, run_mq(r, 64, entry=e)[0])


def test_tc_bad_block_id_sets_status_and_clean_call_does_not():
    w = mq("tc_status", 8, 4, (100, 300), P=64, seed=8800)
    inp = wl.make_inputs(w, device="cuda")
    for e in ("v2", "v1"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        run_mq(inp, 64, entry=e, status=st)
        assert int(st.item()) == 0
    inp.block_tables[1, 3] = inp.key_cache.shape[0] + 1
    for e in ("v2", "v1"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        run_mq(inp, 64, entry=e, status=st)
        assert int(st.item()) & 1


def test_tc_speculative_batch_full_size():
    """Batch decode (32 seqs up to 8192 tokens, 32/8 heads) checking 8 speculated tokens each."""
    w = wl.BATCH.with_(name="batch_spec8", q_len=8)
    check_mq(wl.make_inputs(w, device="cuda"), w.partition_size)


def test_tc_spec_verify_16_full_size():
    """Batch decode checking 16 speculated tokens (64 query rows per KV head), every element."""
    w = wl.SPEC_VERIFY16
    check_mq(wl.make_inputs(w, device="cuda"), w.partition_size)


def test_tc_chunked_prefill_full_size_sampled():
    """2 x (30,720-token prefix + 2048-token chunk): sampled query rows (first, last, tile and
    chunk edges) of three heads, V1 and V2, against the oracle."""
    w = wl.CHUNKED_PREFILL
    inp = wl.make_inputs(w, device="cuda")
    prob = oracle_problem(inp)
    Q = w.q_len
    rows = [0, 1, 63, 64, 1000, Q - 1, Q, Q + 517, 2 * Q - 1]
    heads = [0, 7, 31]
    pairs = [(r, h) for r in rows for h in heads]
    ref = oracle.decode(prob, pairs=pairs)
    for e in ("v1", "v2"):
        out = run_mq(inp, w.partition_size, entry=e)[0]
        g = torch.stack([out[r // Q, r % Q, h] for r, h in pairs])
        check_out(g, ref, w.dtype, what=f"{w.name}/{e}")
