"""GPU parity of phase 2's two forms, each forced through pa_set_merge_form.

Form 1 runs one CTA per (head, row, slice of head_dim) and folds the
partitions round robin over its lanes; form 2 runs one warp per (row, head)
and folds them in index order.  Both compute the log-sum-exp merge of
"paged_attention_v2_pytorch.py" commit 9cb7f9d, "Implementation", Phase 2,
and each is compared element by element with the fp64 oracle (they are not
bitwise equal to each other: the order of the fold differs).
"""
import pytest
import torch

import oracle
import workloads as wl
from parity_util import check_mq, check_out, check_partitions, mq, oracle_problem, run_v2

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cuda_lib.pa_set_launch_config(0, 0)
    yield
    cuda_lib.pa_set_merge_form(0)


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_merge_form_single_token(cuda_lib, form, D, dtype):
    """One new token: up to 16 partitions of 64 tokens, empty sequences, a partition of one token."""
    cuda_lib.pa_set_merge_form(form)
    lens = (0, 1, 63, 64, 65, 500, 0, 1000)
    w = wl.Workload("merge_single", len(lens), 8, 2, D, 16, 64, dtype, "list", seq_lens=lens,
                    seed=9100 + 7 * form + D + dtype)
    inp = wl.make_inputs(w, device="cuda")
    prob = oracle_problem(inp)
    out, tmp, es, ml = run_v2(inp, 64, entry="v2")
    check_out(out, oracle.decode(prob), dtype, what=f"merge_single/form{form}")
    check_partitions(inp, 64, tmp, es, ml, prob=prob)


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("q_len,G", [(4, 8), (16, 4), (2, 1)])
def test_merge_form_causal_rows(cuda_lib, form, q_len, G):
    """Several new tokens: the early rows of a sequence see none of its last partition (a zero
    exp_sum the merge skips)."""
    cuda_lib.pa_set_merge_form(form)
    lens = (q_len, 64 + q_len // 2, 0, 129, 300)
    w = mq("merge_causal", q_len, G, lens, P=64, seed=9200 + 11 * form + q_len + G)
    check_mq(wl.make_inputs(w, device="cuda"), 64, entries=("v2",))


def test_merge_form_rule(cuda_lib):
    """The default picks the warp-per-pair form for many pairs with few partitions; the
    results of the default equal those of the form it picks, bit for bit."""
    from parity_util import run_mq
    w = mq("merge_rule", 8, 8, tuple(range(100, 100 + 64 * 40, 64)), P=512, KV=8,
           seed=9300)
    inp = wl.make_inputs(w, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = 40 * 8 * 64
    assert pairs > 16 * sms  # 8 partitions at most (lengths below 4096): the row form
    cuda_lib.pa_set_merge_form(0)
    out0 = run_mq(inp, 512, entry="v2")[0].clone()
    cuda_lib.pa_set_merge_form(2)
    out2 = run_mq(inp, 512, entry="v2")[0].clone()
    assert torch.equal(out0, out2)


@pytest.mark.parametrize("longest,form", [(20 * 512, 2), (40 * 512, 1)])
def test_merge_form_rule_partition_bound(cuda_lib, longest, form):
    """From 32 pairs per SM the default takes the warp-per-pair form up to 32 partitions at the
    longest (20 here) and the CTA-per-slice form beyond (40); its output equals that form's bit for
    bit."""
    from parity_util import run_mq
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S, Q, G, KV = 20, 8, 4, 8
    assert S * Q * G * KV >= 32 * sms
    lens = tuple(max(Q, longest - 997 * i) for i in range(S))
    w = mq("merge_bound", Q, G, lens, P=512, KV=KV, seed=9350 + longest // 512)
    inp = wl.make_inputs(w, device="cuda")
    cuda_lib.pa_set_merge_form(0)
    out0 = run_mq(inp, 512, entry="v2")[0].clone()
    cuda_lib.pa_set_merge_form(form)
    outf = run_mq(inp, 512, entry="v2")[0].clone()
    assert torch.equal(out0, outf)
