"""Failure detection on the GPU, without a GPU fault.

Every wait in the library's kernels is bounded: a wait that runs out records
MLA_DEV_TIMEOUT in the caller's status word, raises the abort flag of its CTA
and of the other CTA of its pair, drains and returns.  Every kernel that
starts with MLA_DEV_TIMEOUT already in the status word does no work.  These
tests make a wait run out on purpose (a barrier that nothing arrives at, with
a limit of a few milliseconds), check the status and the timings, and check
that each stage then leaves its outputs untouched.  Nothing here faults,
traps or waits without a limit.
"""
import numpy as np
import pytest
import torch

import mla_prefill_attention_plan_gb300 as mla
from workloads import WORKLOADS, make_attention_operands, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_NS = 5_000_000   # 5 ms


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_prefill_attention_plan_gb300 import build
    build.build()
    mla.load()


def _selftest(cluster):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    el = torch.full((cluster,), -2, dtype=torch.int64, device=DEV)
    mla.check(mla.mla_selftest_bounded_wait(st, el, LIMIT_NS, cluster))
    torch.cuda.synchronize()
    return int(st.item()), el.cpu().tolist()


def test_one_cta_wait_runs_out_and_reports():
    status, (t,) = _selftest(1)
    assert status == mla.MLA_DEV_TIMEOUT
    assert LIMIT_NS <= t < 500_000_000


def test_pair_gives_up_together():
    """CTA 1 waits 5 ms, CTA 0 the full 2 s limit: CTA 0 must come back as soon
    as CTA 1's abort flag reaches it, not after its own limit."""
    status, (t0, t1) = _selftest(2)
    assert status == mla.MLA_DEV_TIMEOUT
    assert LIMIT_NS <= t1 < 500_000_000
    assert 0 <= t0 < 500_000_000      # far below the 2 s it would otherwise wait


def test_selftest_repeats_and_context_stays_usable():
    for _ in range(3):
        assert _selftest(2)[0] == mla.MLA_DEV_TIMEOUT
    x = torch.arange(1024, device=DEV, dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


def test_stages_do_nothing_after_a_timeout():
    """With MLA_DEV_TIMEOUT in the status word, the plan, gather, projection and
    attention kernels launch, return at once and leave their outputs as they
    were; the status word keeps the timeout."""
    w = WORKLOADS["tiny_ragged"]
    inp = make_inputs(w)
    B, H, T, S, mc = inp["B"], w.H, inp["T_q"], w.buffer_token_size, w.max_chunks
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    el = torch.zeros(2, dtype=torch.int64, device=DEV)
    mla.check(mla.mla_selftest_bounded_wait(st, el, LIMIT_NS, 2))
    d = {k: inp[k].to(DEV) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache",
                                     "page_table", "w_k", "w_uv")}
    bro = torch.full((mc, B + 1), -7, dtype=torch.int32, device=DEV)
    co = torch.full((mc, B), -7, dtype=torch.int32, device=DEV)
    bl = torch.full((mc,), -7, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill_plan(bro, co, bl, d["input_row_offsets"], d["cache_lengths"], B, mc, S,
                                   st))
    # Tables the later stages can run on (written by the host, as the plan
    # would): one chunk holding every context row.
    tot = int((inp["new_lens"] + inp["cache_lens"]).sum())
    S1 = 128
    bro1 = torch.tensor([[0, int(inp["new_lens"][0] + inp["cache_lens"][0]), tot]], dtype=torch.int32,
                        device=DEV)
    co1 = torch.zeros(1, B, dtype=torch.int32, device=DEV)
    bl1 = torch.tensor([tot], dtype=torch.int32, device=DEV)
    ckv = torch.full((S1, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    kr = torch.full((S1, 64), 7.0, dtype=torch.bfloat16, device=DEV)
    mla.check(mla.mla_gather_latent(ckv, kr, d["kv_cache"], d["page_table"], inp["num_pages"],
                                    inp["page_size"], inp["max_pages"], bro1, co1, bl1, 0, B, S1,
                                    mla.MLA_BF16, st))
    kn = torch.full((S1, H, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    vv = torch.full((S1, H, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    mla.check(mla.mla_upproject(kn, vv, ckv, d["w_k"], d["w_uv"], bl1, 0, S1, H, mla.MLA_BF16,
                                d_status=st))
    k2, v2, r2 = (t.to(DEV) for t in make_attention_operands(w, S1))
    out = torch.full((T, H, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device=DEV)
    mla.check(mla.mla_prefill_attention(out, lse, None, None, d["q"], k2, v2, r2,
                                        d["input_row_offsets"], d["cache_lengths"], bro1, co1, bl1,
                                        0, 1, B, H, inp["max_prompt_len"], T, S1, inp["scale"],
                                        d_status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == mla.MLA_DEV_TIMEOUT
    assert (bro == -7).all() and (co == -7).all() and (bl == -7).all()
    for t in (ckv, kr, kn, vv, out, lse):
        assert (t.float() == 7.0).all()
    # The same calls with a clear status word do their work.
    st.zero_()
    mla.check(mla.mla_prefill_attention(out, lse, None, None, d["q"], k2, v2, r2,
                                        d["input_row_offsets"], d["cache_lengths"], bro1, co1, bl1,
                                        0, 1, B, H, inp["max_prompt_len"], T, S1, inp["scale"],
                                        d_status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert not (out.float() == 7.0).all()
