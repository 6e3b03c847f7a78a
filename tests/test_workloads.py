"""Seeded input generators: determinism, shapes and the structure each workload promises."""
import math

import pytest
import torch

import workloads as wl


def test_same_seed_same_inputs():
    a = wl.make_inputs(wl.TINY)
    b = wl.make_inputs(wl.TINY)
    for x, y in ((a.query, b.query), (a.key_cache, b.key_cache), (a.value_cache, b.value_cache),
                 (a.block_tables, b.block_tables), (a.seq_lens, b.seq_lens)):
        assert torch.equal(x, y)


def test_tiny_shape_and_table():
    inp = wl.make_inputs(wl.TINY)
    assert inp.query.shape == (1, 8, 128) and inp.query.dtype == torch.float16
    assert inp.key_cache.shape == (128, 2, 16, 128)
    assert inp.seq_lens.tolist() == [1000]
    assert inp.block_tables.shape == (1, 63)       # ceil(1000 / 16)
    ids = inp.block_tables[0].tolist()
    assert len(set(ids)) == 63 and min(ids) >= 0 and max(ids) < 128
    assert inp.kv_bytes == 1000 * 2 * 128 * 2 * 2


def test_batch_lengths_and_pool():
    lens = wl.draw_seq_lens(wl.BATCH)
    assert len(lens) == 32 and min(lens) >= 1 and max(lens) <= 8192
    used = sum(wl.blocks_for(L, 16) for L in lens)
    assert math.ceil(1.25 * used) >= used


def test_ragged_lengths_are_clipped_lognormal():
    lens = wl.draw_seq_lens(wl.RAGGED)
    assert len(lens) == 64 and min(lens) >= 16 and max(lens) <= 32768
    med = sorted(lens)[32]
    assert 500 < med < 8000


def test_ragged_outlier_channels():
    w = wl.RAGGED.with_(num_seqs=2, seq_len_kind="list", seq_lens=(40, 70))
    inp = wl.make_inputs(w)
    assert len(inp.outlier_channels) == round(0.05 * 128)
    k = inp.key_cache.float()
    ch = torch.tensor(inp.outlier_channels)
    mask = torch.zeros(128, dtype=torch.bool)
    mask[ch] = True
    ratio = k[..., mask].std() / k[..., ~mask].std()
    assert 6.0 < ratio < 10.0


def test_block_tables_distinct_and_padded():
    w = wl.Workload("t", 4, 4, 2, 128, 16, 64, wl.BF16, "list", seq_lens=(1, 16, 17, 100))
    inp = wl.make_inputs(w, max_blocks=10)
    tab = inp.block_tables
    used = [wl.blocks_for(L, 16) for L in (1, 16, 17, 100)]
    flat = []
    for b, n in enumerate(used):
        assert (tab[b, n:] == -1).all()
        flat += tab[b, :n].tolist()
    assert len(set(flat)) == len(flat)


def test_relabel_keeps_logical_rows():
    w = wl.Workload("t", 2, 4, 2, 128, 16, 64, wl.F16, "list", seq_lens=(33, 70))
    inp = wl.make_inputs(w)
    r = wl.relabel_blocks(inp, seed=3)
    for b in range(2):
        for j in range(wl.blocks_for(int(inp.seq_lens[b]), 16)):
            assert torch.equal(inp.key_cache[inp.block_tables[b, j]],
                               r.key_cache[r.block_tables[b, j]])


def test_poison_touches_only_unread_slots():
    w = wl.Workload("t", 2, 4, 2, 128, 16, 64, wl.F16, "list", seq_lens=(33, 16))
    inp = wl.make_inputs(w)
    before = inp.key_cache.clone()
    wl.poison_unreferenced(inp, 1000.0)
    b0_last = int(inp.block_tables[0, 2])
    assert (inp.key_cache[b0_last, :, 1:] == 1000.0).all()
    assert torch.equal(inp.key_cache[b0_last, :, :1], before[b0_last, :, :1])
    for b, n in ((0, 2), (1, 1)):
        for j in range(n):
            blk = int(inp.block_tables[b, j])
            assert torch.equal(inp.key_cache[blk], before[blk])
