"""Helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, and compare with the stated tolerances.

Tolerances (fp32-accumulated fp16/bf16 decode against the fp64 oracle):
  out         |gpu - ref| <= 2e-3 + half an ulp of the storage type at |ref|
              (out is stored in fp16/bf16, so its own rounding is added to
              the 2e-3 bound of the fp32 result), and
              max|gpu - ref| / max|ref| <= 1e-2 (norm-relative);
  tmp_output  |gpu - ref| <= 2e-3 (fp32, no storage rounding);
  max_logits  |gpu - ref| <= 1e-4 * max(1, |ref|);
  exp_sums    |gpu - ref| <= 1e-4 * ref.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as wl

OUT_ABS = 2e-3
OUT_NORM_REL = 1e-2
TMP_ABS = 2e-3
MAXLOGIT_REL = 1e-4
EXPSUM_REL = 1e-4


def half_ulp(ref: np.ndarray, dtype: int) -> np.ndarray:
    """Half the spacing of the storage type at |ref| (binary16 or bfloat16)."""
    a = np.abs(ref)
    mant = 10 if dtype == wl.F16 else 7
    emin = -14 if dtype == wl.F16 else -126
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return 0.5 * np.exp2(np.maximum(e, emin) - mant)


def oracle_problem(inp: wl.Inputs) -> oracle.Problem:
    return oracle.Problem.from_arrays(wl.to_oracle_arrays(inp))


def compact_subset(inp: wl.Inputs, seqs) -> wl.Inputs:
    """The listed sequences only, with their blocks gathered into a compact pool (for large configs)."""
    w = inp.workload
    bs = w.block_size
    tabs, ids = [], []
    pos = 0
    lens = [int(inp.seq_lens[b]) for b in seqs]
    width = inp.block_tables.shape[1]
    for b, L in zip(seqs, lens):
        n = wl.blocks_for(L, bs)
        row = torch.full((width,), -1, dtype=torch.int32)
        row[:n] = torch.arange(pos, pos + n, dtype=torch.int32)
        ids.append(inp.block_tables[b, :n].long().cpu())
        tabs.append(row)
        pos += n
    idx = torch.cat(ids) if ids else torch.zeros(0, dtype=torch.long)
    if pos == 0:
        idx = torch.zeros(1, dtype=torch.long)
    dev = inp.key_cache.device
    return wl.Inputs(w, inp.query[list(seqs)].cpu(), inp.key_cache[idx.to(dev)].cpu(),
                     inp.value_cache[idx.to(dev)].cpu(), torch.stack(tabs),
                     torch.tensor(lens, dtype=torch.int32), inp.outlier_channels)


def run_v2(inp: wl.Inputs, P: int, hint: int = 0, entry: str = "v2", status=None):
    import paged_kv_decode_v2_gb300 as pa
    w = inp.workload
    S, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    if hint > 0:
        cap = min(cap, hint)
    npmax = max(1, pa.num_partitions(cap, P))
    tmp, es, ml = pa.alloc_workspace(S, H, D, npmax)
    tmp.fill_(float("nan"))
    es.fill_(float("nan"))
    ml.fill_(float("nan"))
    out = torch.full_like(inp.query, float("nan"))
    args = (inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens, w.scale)
    if entry == "v2":
        pa.pa_decode_v2(*args, P, out, tmp, es, ml, max_seq_len_hint=hint, status=status)
    elif entry == "split":
        pa.pa_decode_v2_phase1(*args, P, tmp, es, ml, max_seq_len_hint=hint, status=status)
        pa.pa_decode_v2_phase2(inp.seq_lens, cap, P, tmp, es, ml, out, status=status)
    elif entry == "v1":
        pa.pa_decode_v1(*args, out, max_seq_len_hint=hint, status=status)
    elif entry == "dispatch":
        pa.pa_decode(*args, P, out, tmp, es, ml, max_seq_len_hint=hint, status=status)
    else:
        raise ValueError(entry)
    torch.cuda.synchronize()
    return out, tmp, es, ml


def check_out(gpu_out: torch.Tensor, ref: np.ndarray, dtype: int, what: str = "out"):
    g = gpu_out.detach().cpu().to(torch.float64).numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    tol = OUT_ABS + half_ulp(ref, dtype)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements over tolerance; worst "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    denom = max(np.abs(ref).max(), 1e-30)
    assert err.max() / denom <= OUT_NORM_REL, f"{what}: norm-relative error {err.max() / denom:.3e}"
    return float(err.max())


def check_partitions(inp: wl.Inputs, P: int, tmp, es, ml, pairs=None, prob=None):
    """Compare phase-1 intermediates with the oracle's per-partition statistics."""
    prob = prob or oracle_problem(inp)
    S, H = inp.query.shape[:2]
    if pairs is None:
        pairs = [(b, h) for b in range(S) for h in range(H)]
    o, m, l, num = oracle.partition_stats(prob, P, pairs=pairs, max_partitions=tmp.shape[2])
    tmp_c, es_c, ml_c = tmp.cpu().double().numpy(), es.cpu().double().numpy(), ml.cpu().double().numpy()
    worst = [0.0, 0.0, 0.0]
    for i, (b, h) in enumerate(pairs):
        n = int(num[i])
        if n == 0:
            continue
        dt = np.abs(tmp_c[b, h, :n] - o[i, :n])
        assert np.isfinite(tmp_c[b, h, :n]).all()
        assert dt.max() <= TMP_ABS, f"tmp_output ({b},{h}) err {dt.max():.3e}"
        # Empty partitions (a query that sees none of their tokens): l = 0, m = -inf.
        empty = l[i, :n] == 0.0
        assert (es_c[b, h, :n][empty] == 0.0).all(), f"exp_sums ({b},{h}) of an empty partition"
        assert (ml_c[b, h, :n][empty] == -np.inf).all(), f"max_logits ({b},{h}) of an empty partition"
        full = ~empty
        if not full.any():
            continue
        dm = np.abs(ml_c[b, h, :n][full] - m[i, :n][full])
        assert (dm <= MAXLOGIT_REL * np.maximum(1.0, np.abs(m[i, :n][full]))).all(), \
            f"max_logits ({b},{h}) err {dm.max():.3e}"
        de = np.abs(es_c[b, h, :n][full] - l[i, :n][full]) / l[i, :n][full]
        assert (de <= EXPSUM_REL).all(), f"exp_sums ({b},{h}) rel err {de.max():.3e}"
        worst = [max(worst[0], dt.max()), max(worst[1], dm.max()), max(worst[2], de.max())]
    return worst


def oracle_out(inp: wl.Inputs, pairs=None, prob=None):
    prob = prob or oracle_problem(inp)
    return oracle.decode(prob, pairs=pairs)


# ---------------------------------------------------------------- several new tokens per sequence

def run_mq(inp, P, entry="v2", hint=0, status=None):
    import paged_kv_decode_v2_gb300 as pa
    w = inp.workload
    S, Q, H, D = inp.query.shape
    cap = inp.block_tables.shape[1] * w.block_size
    if hint > 0:
        cap = min(cap, hint)
    npmax = max(1, pa.num_partitions(cap, P))
    tmp, es, ml = pa.alloc_workspace(S, H, D, npmax, q_len=Q)
    for t in (tmp, es, ml):
        t.fill_(float("nan"))
    out = torch.full_like(inp.query, float("nan"))
    args = (inp.query, inp.key_cache, inp.value_cache, inp.block_tables, inp.seq_lens, w.scale)
    if entry == "v2":
        pa.pa_decode_v2_mq(*args, P, out, tmp, es, ml, max_seq_len_hint=hint, status=status)
    else:
        pa.pa_decode_v1_mq(*args, out, max_seq_len_hint=hint, status=status)
    torch.cuda.synchronize()
    return out, tmp, es, ml


def check_mq(inp, P, entries=("v2", "v1")):
    prob = oracle_problem(inp)
    ref = oracle.decode(prob)  # [S, Q, H, D]
    S, Q, H, D = inp.query.shape
    for e in entries:
        out, tmp, es, ml = run_mq(inp, P, entry=e)
        check_out(out, ref, inp.workload.dtype, what=f"{inp.workload.name}/{e}")
        if e == "v2":
            pairs = [(r, h) for r in range(S * Q) for h in range(H)]
            check_partitions(inp, P, tmp.view(S * Q, H, *tmp.shape[3:]), es.view(S * Q, H, -1),
                             ml.view(S * Q, H, -1), pairs=pairs, prob=prob)
    return ref


def mq(name, q_len, G, lens, bs=16, P=64, dtype=wl.BF16, D=128, KV=2, seed=0):
    return wl.Workload(name, len(lens), G * KV, KV, D, bs, P, dtype, "list", seq_lens=tuple(lens),
                       q_len=q_len, seed=seed)


def ramp_scores(inp, c, period=None):
    """Add c * position (modulo period) to dimension 0 of every key and set dimension 0 of the queries
    to +1 for even heads and -1 for odd ones: scores rise by ~c * scale per token on even heads and
    fall on odd heads, so rows of one warp disagree on whether their running max moves."""
    w = inp.workload
    bs = w.block_size
    q = inp.query
    sign = torch.ones(w.num_heads, device=q.device)
    sign[1::2] = -1.0
    q[..., 0] = sign.to(q.dtype)
    lens = inp.seq_lens.tolist()
    for b, L in enumerate(lens):
        nb = -(-L // bs)
        ids = inp.block_tables[b, :nb].long()
        pos = torch.arange(nb * bs, device=q.device, dtype=torch.float32).view(nb, 1, bs)
        if period:
            pos = pos % period
        inp.key_cache[ids, :, :, 0] = (c * pos).expand(nb, w.num_kv_heads, bs).to(inp.key_cache.dtype)
    return inp
