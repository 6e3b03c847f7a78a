"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test fixes the oracle to a fact the pages or mathematics determine:
printed counts, hand-worked closed forms, invariants, special cases that
reduce to a library routine, and a pure-Python brute force on tiny inputs.
The mutation tests at the end plant single mistakes into a copy of the
oracle's C source and check that at least one pin catches each of them.
"""
import json
import math
import os
import re
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads as wl
from conftest import golden_path, ROOT

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ---------------------------------------------------------------- helpers

def small(name="small", S=3, H=8, KV=2, D=32, bs=16, P=64, dtype=wl.BF16, seq_lens=(1, 70, 200),
          seed=7, **kw):
    return wl.Workload(name, S, H, KV, D, bs, P, dtype, "list", seq_lens=tuple(seq_lens),
                       seed=seed, **kw)


def problem_of(inp: wl.Inputs) -> oracle.Problem:
    return oracle.Problem.from_arrays(wl.to_oracle_arrays(inp))


def decoded(t: torch.Tensor) -> np.ndarray:
    """fp16/bf16 tensor -> float64 numpy via torch's own conversion (a library routine)."""
    return t.detach().cpu().to(torch.float64).numpy()


def dense_kv(inp: wl.Inputs, b: int):
    """Logical [L, KV, D] K and V of sequence b, gathered with plain indexing."""
    bs = inp.workload.block_size
    L = int(inp.seq_lens[b])
    n = wl.blocks_for(L, bs)
    ids = inp.block_tables[b, :n].long()
    k = inp.key_cache[ids].permute(0, 2, 1, 3).reshape(n * bs, inp.workload.num_kv_heads, -1)[:L]
    v = inp.value_cache[ids].permute(0, 2, 1, 3).reshape(n * bs, inp.workload.num_kv_heads, -1)[:L]
    return k, v


# ---------------------------------------------------------------- storage decoding

def test_binary16_decoding_all_patterns():
    """The oracle's own binary16 decoding equals numpy's float16 for all 65536 patterns."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode_scalar(int(b), oracle.F16) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), bits[~same][:10]


def test_bfloat16_decoding_all_patterns():
    """The oracle's own bfloat16 decoding equals torch.bfloat16 -> float64 for all patterns."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_scalar(int(b), oracle.BF16) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), bits[~same][:10]


# ---------------------------------------------------------------- printed values

def test_golden_partition_counts_from_pages():
    cases = json.load(open(golden_path("partition_counts.json")))["cases"]
    w = small(S=1, H=1, KV=1, D=8, bs=16, P=512, seq_lens=(100000,))
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    for c in cases:
        if "blocks" in c:
            # The table width the oracle needs is exactly the printed block count:
            # the last needed entry is read (an invalid id there is an error) ...
            assert inp.block_tables.shape[1] == c["blocks"]
            bad = wl.to_oracle_arrays(inp)
            bad["block_tables"] = bad["block_tables"].copy()
            bad["block_tables"][0, c["blocks"] - 1] = -1
            with pytest.raises(RuntimeError):
                oracle.decode(oracle.Problem.from_arrays(bad), pairs=[(0, 0)])
            # ... and one block fewer cannot hold the sequence.
            short = wl.to_oracle_arrays(inp)
            short["block_tables"] = short["block_tables"][:, : c["blocks"] - 1].copy()
            with pytest.raises(RuntimeError):
                oracle.decode(oracle.Problem.from_arrays(short), pairs=[(0, 0)])
        else:
            _, _, _, num = oracle.partition_stats(prob, c["partition_size"], pairs=[(0, 0)])
            assert int(num[0]) == c["partitions"], c["cite"]


def test_hand_worked_three_tokens():
    import sympy
    g = json.load(open(golden_path("hand3.json")))
    ev = lambda e: float(sympy.N(sympy.sympify(e), 30))
    q = torch.tensor(g["query"], dtype=torch.float16)
    kc = torch.tensor(g["key_cache"], dtype=torch.float16)
    vc = torch.tensor(g["value_cache"], dtype=torch.float16)
    bt = np.array(g["block_tables"], dtype=np.int32)
    sl = np.array(g["seq_lens"], dtype=np.int32)
    u16 = lambda t: t.numpy().view(np.uint16)
    prob = oracle.Problem(u16(q), u16(kc), u16(vc), bt, sl, g["scale"], oracle.F16)
    out = oracle.decode(prob)[0, 0]
    exp_out = np.array([ev(e) for e in g["out"]])
    np.testing.assert_allclose(out, exp_out, rtol=0, atol=1e-15)
    o, m, l, num = oracle.partition_stats(prob, g["partition_size"])
    assert int(num[0]) == 2
    np.testing.assert_allclose(m[0, :2], [ev(e) for e in g["partitions"]["max_logits"]], atol=1e-15)
    np.testing.assert_allclose(l[0, :2], [ev(e) for e in g["partitions"]["exp_sums"]], atol=1e-15)
    np.testing.assert_allclose(o[0, :2], [[ev(e) for e in r] for r in g["partitions"]["tmp_output"]],
                               atol=1e-15)
    np.testing.assert_allclose(oracle.merge(o[0, :2], m[0, :2], l[0, :2]), exp_out, atol=1e-15)


# ---------------------------------------------------------------- closed forms

def test_uniform_keys_give_mean_of_values():
    """All K rows equal -> every logit equal -> out = mean of V; l_p = tokens in p."""
    w = small(seq_lens=(1, 70, 200, 513), S=4, P=64)
    inp = wl.make_inputs(w)
    inp.key_cache[:] = inp.key_cache[0, 0, 0]  # one row everywhere
    prob = problem_of(inp)
    out = oracle.decode(prob)
    o, m, l, num = oracle.partition_stats(prob, w.partition_size)
    G = w.group_size
    k0 = decoded(inp.key_cache[0, 0, 0])
    for b in range(w.num_seqs):
        L = int(inp.seq_lens[b])
        _, v = dense_kv(inp, b)
        vv = decoded(v)
        for h in range(w.num_heads):
            np.testing.assert_allclose(out[b, h], vv[:, h // G].mean(axis=0), rtol=0, atol=1e-13)
            common = w.scale * float(decoded(inp.query[b, h]) @ k0)
            i = b * w.num_heads + h
            for p in range(int(num[i])):
                ntok = min(L, (p + 1) * w.partition_size) - p * w.partition_size
                assert l[i, p] == pytest.approx(ntok, rel=1e-14)
                assert m[i, p] == pytest.approx(common, rel=1e-13, abs=1e-13)


def test_one_dominant_logit_selects_its_value_row():
    """q = e_0, K_t*[0] = 64 and |K_t[0]| <= 4 elsewhere: margin >= 60, out = V_t* within L e^-60 max|V|."""
    w = small(S=1, H=2, KV=1, D=16, seq_lens=(300,), P=64, dtype=wl.F16)
    inp = wl.make_inputs(w)
    inp.query.zero_()
    inp.query[..., 0] = 1.0
    inp.key_cache.clamp_(-4, 4)
    tstar = 217
    blk = int(inp.block_tables[0, tstar // w.block_size])
    inp.key_cache[blk, 0, tstar % w.block_size, 0] = 64.0
    prob = oracle.Problem.from_arrays({**wl.to_oracle_arrays(inp), "scale": 1.0})
    out = oracle.decode(prob)
    _, v = dense_kv(inp, 0)
    vstar = decoded(v[tstar, 0])
    bound = 300 * math.exp(-60) * np.abs(decoded(v)).max()
    for h in range(2):
        assert np.abs(out[0, h] - vstar).max() <= bound + 1e-16


def test_single_token_returns_its_value_row_exactly():
    w = small(S=2, H=4, KV=2, D=32, seq_lens=(1, 1))
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    out = oracle.decode(prob)
    o, m, l, num = oracle.partition_stats(prob, w.partition_size)
    for b in range(2):
        k, v = dense_kv(inp, b)
        for h in range(4):
            assert np.array_equal(out[b, h], decoded(v[0, h // 2]))
            i = b * 4 + h
            assert num[i] == 1 and l[i, 0] == 1.0
            s0 = w.scale * float(decoded(inp.query[b, h]) @ decoded(k[0, h // 2]))
            assert m[i, 0] == pytest.approx(s0, rel=1e-14)


def test_two_tokens_closed_form_with_scale():
    """Two tokens with logit gap d: out = V0 + sigmoid(d) (V1 - V0); checks scale is applied once."""
    w = small(S=1, H=1, KV=1, D=8, seq_lens=(2,), dtype=wl.F16)
    inp = wl.make_inputs(w)
    inp.query.zero_()
    inp.query[0, 0, 0] = 2.0
    b0 = int(inp.block_tables[0, 0])
    inp.key_cache[b0, 0, 0].zero_()
    inp.key_cache[b0, 0, 1].zero_()
    inp.key_cache[b0, 0, 1, 0] = 1.5  # raw dot 3.0
    for scale in (1.0, 0.125, 0.7):
        prob = oracle.Problem.from_arrays({**wl.to_oracle_arrays(inp), "scale": scale})
        out = oracle.decode(prob)[0, 0]
        d = 3.0 * scale
        v0, v1 = decoded(inp.value_cache[b0, 0, 0]), decoded(inp.value_cache[b0, 0, 1])
        expect = v0 + (v1 - v0) / (1.0 + math.exp(-d))
        np.testing.assert_allclose(out, expect, rtol=0, atol=1e-14)


def test_gqa_contiguous_groups():
    """KV head k holds V == k+1 everywhere; query head h must read KV head h // G."""
    for H, KV in ((8, 2), (8, 8), (8, 1), (12, 3)):
        w = small(S=1, H=H, KV=KV, D=16, seq_lens=(40,))
        inp = wl.make_inputs(w)
        for k in range(KV):
            inp.value_cache[:, k] = float(k + 1)
        out = oracle.decode(problem_of(inp))
        G = H // KV
        for h in range(H):
            np.testing.assert_allclose(out[0, h], float(h // G + 1), rtol=1e-14, atol=0)


def test_empty_sequence_is_zero():
    w = small(S=2, seq_lens=(0, 5))
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    out = oracle.decode(prob)
    assert np.all(out[0] == 0.0)
    _, _, _, num = oracle.partition_stats(prob, 64)
    assert np.all(num[: w.num_heads] == 0)
    assert np.all(oracle.merge(np.zeros((0, 32)), np.zeros(0), np.zeros(0)) == 0.0)


# ---------------------------------------------------------------- library routine / brute force

@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_matches_dense_torch_softmax(dtype):
    """Reduces to a library routine: gather K/V densely, torch.softmax in float64, then @ V."""
    w = small(S=3, H=8, KV=2, D=128, bs=16, seq_lens=(1000, 17, 333), dtype=dtype)
    inp = wl.make_inputs(w)
    out = oracle.decode(problem_of(inp))
    for b in range(3):
        k, v = dense_kv(inp, b)
        for h in range(8):
            q = inp.query[b, h].to(torch.float64)
            s = (k[:, h // 4].to(torch.float64) @ q) * w.scale
            ref = torch.softmax(s, dim=0) @ v[:, h // 4].to(torch.float64)
            np.testing.assert_allclose(out[b, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_matches_pure_python_brute_force():
    w = small(S=2, H=4, KV=2, D=8, bs=4, seq_lens=(13, 1), dtype=wl.F16)
    inp = wl.make_inputs(w)
    out = oracle.decode(problem_of(inp))
    ref = brute.decode(decoded(inp.query), decoded(inp.key_cache), decoded(inp.value_cache),
                       inp.block_tables.numpy(), inp.seq_lens.numpy(), w.scale)
    np.testing.assert_allclose(out, np.array(ref), rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- the method's algebra

@pytest.mark.parametrize("P", [512, 1024, 300, 7, 1])
def test_partition_then_merge_equals_unpartitioned(P):
    """Phase 1 + phase 2 (pages' V2) == full softmax, for divisor and non-divisor P."""
    lens = (1000, 1, 5000, 512, 1024, 2049)
    w = small(S=len(lens), H=4, KV=2, D=32, bs=16, seq_lens=lens, P=P)
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    full = oracle.decode(prob)
    o, m, l, num = oracle.partition_stats(prob, P)
    for i in range(w.num_seqs * w.num_heads):
        b, h = divmod(i, w.num_heads)
        assert num[i] == -(-lens[b] // P)
        merged = oracle.merge(o[i, : num[i]], m[i, : num[i]], l[i, : num[i]])
        np.testing.assert_allclose(merged, full[b, h], rtol=1e-12, atol=1e-13)


def test_partition_then_merge_at_100k_tokens():
    w = small(S=1, H=2, KV=1, D=16, bs=16, seq_lens=(100000,), P=512)
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    full = oracle.decode(prob)
    for P in (512, 1024):
        o, m, l, num = oracle.partition_stats(prob, P)
        for h in range(2):
            merged = oracle.merge(o[h, : num[h]], m[h, : num[h]], l[h, : num[h]])
            np.testing.assert_allclose(merged, full[0, h], rtol=1e-11, atol=1e-13)


def test_physical_block_relabelling_is_bitwise_invariant():
    w = small(S=3, H=8, KV=2, D=32, bs=16, seq_lens=(300, 17, 64))
    inp = wl.make_inputs(w)
    a = oracle.decode(problem_of(inp))
    b = oracle.decode(problem_of(wl.relabel_blocks(inp, seed=99)))
    assert np.array_equal(a, b)
    pa = oracle.partition_stats(problem_of(inp), 64)
    pb = oracle.partition_stats(problem_of(wl.relabel_blocks(inp, seed=5)), 64)
    for x, y in zip(pa, pb):
        assert np.array_equal(np.nan_to_num(x, nan=-7.0), np.nan_to_num(y, nan=-7.0))


def test_unreferenced_slots_are_never_read():
    """Poison (inf/nan) in unused pool blocks, tail rows and -1 table padding changes nothing."""
    w = small(S=3, H=4, KV=2, D=32, bs=16, seq_lens=(37, 16, 5), dtype=wl.F16)
    inp = wl.make_inputs(w, max_blocks=9)
    clean = oracle.decode(problem_of(inp))
    wl.poison_unreferenced(inp, float("nan"))
    assert (inp.block_tables == -1).any()
    dirty = oracle.decode(problem_of(inp))
    assert np.array_equal(clean, dirty)


def test_pairs_subset_matches_full():
    w = small()
    inp = wl.make_inputs(w)
    prob = problem_of(inp)
    full = oracle.decode(prob)
    pairs = [(2, 7), (0, 0), (1, 3)]
    sub = oracle.decode(prob, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[b, h])


# ---------------------------------------------------------------- several new tokens (q_len > 1)

def mq_workload(q_len, lens, H=8, KV=2, D=32, bs=16, P=64, dtype=wl.BF16, seed=11):
    return wl.Workload("mq", len(lens), H, KV, D, bs, P, dtype, "list", seq_lens=tuple(lens),
                       q_len=q_len, seed=seed)


def mq_torch_reference(inp):
    """Dense gather + torch.softmax(float64) over each query's causal prefix t <= L - Q + i."""
    w = inp.workload
    Q, G = w.q_len, w.group_size
    S = w.num_seqs
    out = np.zeros(tuple(inp.query.shape), dtype=np.float64)
    for b in range(S):
        L = int(inp.seq_lens[b])
        if L == 0:
            continue
        k, v = dense_kv(inp, b)
        for i in range(Q):
            vis = min(L, max(0, L - Q + i + 1))
            if vis == 0:
                continue
            for h in range(w.num_heads):
                s = (k[:vis, h // G].to(torch.float64) @ inp.query[b, i, h].to(torch.float64)) * w.scale
                out[b, i, h] = (torch.softmax(s, 0) @ v[:vis, h // G].to(torch.float64)).numpy()
    return out


def test_mq_single_token_is_the_single_query_decode():
    w1 = small(seq_lens=(5, 300, 64))
    inp1 = wl.make_inputs(w1)
    arrs = wl.to_oracle_arrays(inp1)
    single = oracle.decode(oracle.Problem.from_arrays(arrs))
    arrs4 = dict(arrs, query=arrs["query"][:, None])  # [S, 1, H, D]
    multi = oracle.decode(oracle.Problem.from_arrays(arrs4))
    assert multi.shape == (3, 1, 8, 32)
    assert np.array_equal(multi[:, 0], single)


@pytest.mark.parametrize("q_len", [2, 3, 7])
def test_mq_matches_causal_prefix_softmax(q_len):
    inp = wl.make_inputs(mq_workload(q_len, (1, 2, q_len, 17, 200)))
    out = oracle.decode(problem_of(inp))
    np.testing.assert_allclose(out, mq_torch_reference(inp), rtol=1e-12, atol=1e-13)
    L0 = 1  # sequence 0 is shorter than q_len: its first queries see nothing
    assert np.all(out[0, : q_len - L0] == 0.0)


@pytest.mark.parametrize("P", [16, 64, 48])
def test_mq_partition_then_merge_equals_unpartitioned(P):
    inp = wl.make_inputs(mq_workload(4, (3, 63, 64, 65, 129, 200)))
    prob = problem_of(inp)
    full = oracle.decode(prob).reshape(-1, prob.D)
    o, m, l, num = oracle.partition_stats(prob, P)
    for idx in range(full.shape[0]):
        n = int(num[idx])
        merged = oracle.merge(o[idx, :n], m[idx, :n], l[idx, :n])
        np.testing.assert_allclose(merged, full[idx], rtol=1e-12, atol=1e-13)
    # a partition holding none of a query's visible tokens is empty, not NaN
    assert np.isfinite(o[~np.isnan(o)]).all()
    assert (l[~np.isnan(l)] >= 0).all()


def test_mq_matches_pure_python_brute_force():
    inp = wl.make_inputs(mq_workload(3, (7, 2), H=4, KV=2, D=8, bs=4))
    out = oracle.decode(problem_of(inp))
    ref = brute.decode(decoded(inp.query), decoded(inp.key_cache), decoded(inp.value_cache),
                       inp.block_tables.numpy(), inp.seq_lens.numpy(), inp.workload.scale, q_len=3)
    np.testing.assert_allclose(out, np.array(ref), rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    # phase 2 without the exp_sum factor in the rescale
    "merge_drops_exp_sum": ("total_sum += exp(m_p[i] - global_max) * l_p[i];",
                            "total_sum += exp(m_p[i] - global_max);"),
    # GQA mapping by modulo instead of contiguous groups
    "gqa_modulo": ("int k = h / (p->H / p->KV);\n    for (int t = t0",
                   "int k = h % p->KV;\n    for (int t = t0"),
    # scale dropped from the logits
    "no_scale": ("s[t - t0] = p->scale * dot;", "s[t - t0] = dot;"),
    # wrong row inside a block
    "row_index": ("+ t % p->bs) * p->D", "+ (t / p->bs) % p->bs) * p->D"),
    # flipped sign in the softmax exponent
    "exp_sign": ("double w = exp(s[t - t0] - m);", "double w = exp(m - s[t - t0]);"),
    # binary16 exponent bias off by one
    "f16_bias": ("expo - 25", "expo - 24"),
    # causal limit of a new token off by one
    "causal_off_by_one": ("int visible = L - p->Q + r % p->Q + 1;", "int visible = L - p->Q + r % p->Q;"),
    # query row of new token i taken from the wrong position
    "mq_row": ("int b = r / p->Q;\n", "int b = r % p->S;\n"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "pa_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / f"{name}.so")
    oracle.build(force=True, src=str(path), out=so)
    return oracle.OracleLib(so)


def _pins_pass(lib: "oracle.OracleLib") -> bool:
    """A compact run of the pins above against a given oracle build; False if any fails."""
    try:
        # storage decoding
        for bits in (0x3C00, 0x0001, 0x7BFF, 0xC500):
            ref = float(np.array([bits], dtype=np.uint16).view(np.float16)[0])
            if lib.decode_scalar(bits, oracle.F16) != ref:
                return False
        # library routine
        w = small(S=2, H=8, KV=2, D=32, seq_lens=(100, 7), dtype=wl.BF16)
        inp = wl.make_inputs(w)
        prob = problem_of(inp)
        out = lib.decode(prob)
        for b in range(2):
            k, v = dense_kv(inp, b)
            for h in range(8):
                s = (k[:, h // 4].to(torch.float64) @ inp.query[b, h].to(torch.float64)) * w.scale
                ref = (torch.softmax(s, 0) @ v[:, h // 4].to(torch.float64)).numpy()
                if not np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-13):
                    return False
        # partition + merge
        o, m, l, num = lib.partition_stats(prob, 16)
        for i in range(16):
            b, h = divmod(i, 8)
            merged = lib.merge(o[i, : num[i]], m[i, : num[i]], l[i, : num[i]])
            if not np.allclose(merged, out[b, h], rtol=1e-12, atol=1e-13):
                return False
        # several new tokens: causal prefix softmax
        inp = wl.make_inputs(mq_workload(3, (2, 40, 9)))
        mq = lib.decode(problem_of(inp))
        if not np.allclose(mq, mq_torch_reference(inp), rtol=1e-12, atol=1e-13):
            return False
        return True
    except RuntimeError:
        return False


def test_pins_pass_on_the_real_oracle(tmp_path):
    assert _pins_pass(oracle.lib())


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    assert not _pins_pass(_build_mutant(tmp_path, name)), f"pins missed mutant {name}"
