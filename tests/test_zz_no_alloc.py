"""The allocation-free attention entry point, on the GPU.

Some callers of this library cannot allocate device memory: a custom operator
loaded into a host framework that owns the whole device memory pool and hands
it no allocator, or a loop that must not call cudaMalloc because cudaMalloc
synchronises the device.  mla_prefill_attention_noalloc serves them by keeping
the cross-chunk fp32 merge state in a fixed array inside the library.

These tests run multi-chunk plans through that entry point twice in a row and
compare each result with the regular entry point (which takes the scratch from
the caller), within the tolerance the parity tests use, and check that calls
larger than the fixed array are refused.  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import mla_prefill_attention_plan_gb300 as mla
from workloads import WORKLOADS, make_attention_operands, make_inputs, scaled

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_ABS, MEAN_REL, LSE_ABS = 2e-2, 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_prefill_attention_plan_gb300 import build
    build.build()
    mla.load()


def _case(w, **kw):
    inp = make_inputs(w, **kw)
    B, H, T = inp["B"], w.H, inp["T_q"]
    S = w.buffer_token_size
    mc = -(-int((inp["new_lens"] + inp["cache_lens"]).sum()) // S)
    bro = torch.empty(mc, B + 1, dtype=torch.int32, device=DEV)
    co = torch.empty(mc, B, dtype=torch.int32, device=DEV)
    bl = torch.empty(mc, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = {k: inp[k].to(DEV) for k in ("q", "input_row_offsets", "cache_lengths")}
    mla.check(mla.mla_prefill_plan(bro, co, bl, d["input_row_offsets"], d["cache_lengths"], B, mc,
                                   S, st))
    ops = [tuple(t.to(DEV) for t in make_attention_operands(w, S, seed_offset=21 + c))
           for c in range(mc)]
    return inp, d, (bro, co, bl), ops, st, mc


def _run(noalloc, inp, d, tabs, ops, st, mc):
    w = inp["workload"]
    B, H, T, S = inp["B"], w.H, inp["T_q"], w.buffer_token_size
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, H, dtype=torch.float32, device=DEV)
    if not noalloc:
        oacc = torch.empty(T, H, 128, dtype=torch.float32, device=DEV)
        lacc = torch.empty(T, H, dtype=torch.float32, device=DEV)
    for c in range(mc):
        kn, vv, kr = ops[c]
        common = (d["q"], kn, vv, kr, d["input_row_offsets"], d["cache_lengths"], *tabs, c, mc, B,
                  H, inp["max_prompt_len"], T, S, inp["scale"])
        if noalloc:
            code = mla.mla_prefill_attention_noalloc(out, lse, *common, d_status=st)
        else:
            code = mla.mla_prefill_attention(out, lse, oacc, lacc, *common, d_status=st)
        mla.check(code)
    torch.cuda.synchronize()
    assert st.item() == 0, mla.status_string(int(st.item()))
    return out.float(), lse


def _close(a, b):
    d = (a - b).abs()
    assert torch.isfinite(a).all()
    assert d.max().item() <= MAX_ABS
    assert (d.sum() / b.abs().sum()).item() <= MEAN_REL


@pytest.mark.parametrize("shape", ["tiny", "ragged"])
def test_noalloc_matches_caller_scratch_on_two_calls(shape):
    if shape == "tiny":
        w = WORKLOADS["tiny_ragged"]
        args = {}
    else:
        w = scaled(WORKLOADS["ragged_chunked_cache"], B=3, H=4, buffer_token_size=700,
                   new_range=(100, 900), cache_range=(0, 1200))
        args = {}
    inp, d, tabs, ops, st, mc = _case(w, **args)
    assert mc > 1 and inp["T_q"] * w.H <= mla.MLA_NOALLOC_MAX_ROWS
    ref_out, ref_lse = _run(False, inp, d, tabs, ops, st, mc)
    for _ in range(2):   # the fixed scratch keeps the previous call's contents
        out, lse = _run(True, inp, d, tabs, ops, st, mc)
        _close(out, ref_out)
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS


def test_noalloc_refuses_calls_larger_than_its_scratch():
    rows = mla.MLA_NOALLOC_MAX_ROWS
    code = mla.mla_prefill_attention_noalloc(16, None, 16, 16, 16, 16, 16, 16, 16, 16, 16, 0, 2,
                                             1, 1, rows + 1, rows + 1, 64, 0.1, stream=0)
    assert code == mla.MLA_ERR_WORKSPACE
