"""GPU parity of the absorbed decode branch ("mla_prefill_decode_graph_bf16",
Args w_uk, w_uv, num_partitions_in) against the oracle's mla_decode, through
the C ABI.  Tolerance as for bf16 prefill: max-abs 2e-2 and mean-rel 1e-2
(sum|gpu - ref| / sum|ref|); the natural-log LSE within 5e-3."""
import numpy as np
import pytest
import torch

import mla_prefill_attention_plan_gb300 as mla
import oracle as O
from workloads import (DECODE_WORKLOADS, WORKLOADS, make_attention_sinks, make_inputs,
                       make_sparse_indices, scaled)

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_ABS, MEAN_REL, LSE_ABS = 2e-2, 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_prefill_attention_plan_gb300 import build
    build.build()
    mla.load()


def _decode_workload(B, H, new, cache, page_size=128, shuffle=True, seed=0):
    return scaled(DECODE_WORKLOADS["v3_decode"], B=B, H=H, new_lens=tuple(new), cache_lens=tuple(cache),
                  page_size=page_size, shuffle_pages=shuffle, seed=seed)


def run_decode(inp, parts=0, lse=True, sink=None, indices=None, stride=0, topk=None, status=None):
    w = inp["workload"]
    B, H, T = inp["B"], w.H, inp["T_q"]
    max_new = int(inp["new_lens"].max())
    max_seq = int((inp["new_lens"] + inp["cache_lens"]).max())
    max_keys = min(stride, max_seq) if indices is not None else max_seq
    nparts = parts or mla.mla_decode_partitions(B, H, max_new, max_keys)
    nbytes = mla.mla_decode_workspace_bytes(H, T, nparts)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    l = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV) if lse else None
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=DEV)
    d = {k: inp[k].to(DEV) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache", "page_table",
                                     "w_uk", "w_uv")}
    mla.check(mla.mla_decode(out, l, d["q"], d["input_row_offsets"], d["cache_lengths"], d["kv_cache"],
                             d["page_table"], inp["num_pages"], inp["page_size"], inp["max_pages"],
                             d["w_uk"], d["w_uv"], B, H, T, max_new, max_seq, parts, inp["scale"],
                             d_indices=indices, indices_stride=stride, topk_lengths=topk, attn_sink=sink,
                             workspace=ws, workspace_bytes=nbytes, d_status=st))
    torch.cuda.synchronize()
    if status is None:
        assert int(st.item()) == 0, mla.status_string(int(st.item()))
    return out, l


def oracle_decode(inp, heads=None, seqs=None, parts=1):
    """The oracle on a sample: the given heads (heads are independent) and
    sequences (their query rows renumbered)."""
    w = inp["workload"]
    H = w.H
    hs = list(range(H)) if heads is None else list(heads)
    bs = list(range(inp["B"])) if seqs is None else list(seqs)
    iro = inp["input_row_offsets"].numpy().astype(np.int64)
    rows = np.concatenate([np.arange(iro[b], iro[b + 1]) for b in bs])
    new = np.array([iro[b + 1] - iro[b] for b in bs])
    iro_s = np.concatenate([[0], np.cumsum(new)])
    q = O.decode(O.codes(inp["q"]), "bf16")[rows][:, hs]
    w_uk = O.decode(O.codes(inp["w_uk"]), "bf16")[hs]
    w_uv = O.decode(O.codes(inp["w_uv"]), "bf16")[hs]
    pt = O.codes(inp["page_table"])[bs]
    cache = O.codes(inp["cache_lengths"])[bs]
    res = O.mla_decode(q, O.codes(inp["kv_cache"]), pt, inp["page_size"], w_uk, w_uv, iro_s, cache,
                       inp["scale"], num_partitions=parts)
    out = {}
    for (bi, hi), (tok, o, l) in res.items():
        out[(bs[bi], hs[hi])] = (rows[tok], o, l)
    return out


def _compare(out, lse, ref):
    g = out.float().cpu().double().numpy()
    gl = None if lse is None else lse.cpu().double().numpy()
    max_abs, num, den, lse_err = 0.0, 0.0, 0.0, 0.0
    for (b, h), (tok, o, l) in ref.items():
        diff = np.abs(g[tok, h] - o)
        assert np.isfinite(g[tok, h]).all()
        max_abs = max(max_abs, float(diff.max()))
        num += float(diff.sum())
        den += float(np.abs(o).sum())
        if gl is not None:
            lse_err = max(lse_err, float(np.abs(gl[tok, h] - l).max()))
    assert max_abs <= MAX_ABS, max_abs
    assert num / den <= MEAN_REL, num / den
    assert lse_err <= LSE_ABS, lse_err
    return max_abs, num / den


@pytest.mark.parametrize("parts", [1, 3])
def test_decode_small_pages_gathered_rows(parts):
    """Page size 16: the 64-key tiles cross pages, so the kernel gathers rows
    four at a time; several tokens per sequence (causal among them)."""
    w = _decode_workload(3, 4, (1, 2, 3), (5, 130, 300), page_size=16)
    inp = make_inputs(w, with_w_uk=True)
    out, lse = run_decode(inp, parts)
    _compare(out, lse, oracle_decode(inp))


@pytest.mark.parametrize("parts", [1, 2, 5])
def test_decode_page128_tiles(parts):
    """Page size 128: every 64-key tile is one rectangular load; 128 heads."""
    w = _decode_workload(4, 128, (1, 1, 2, 1), (200, 1000, 77, 3000))
    inp = make_inputs(w, with_w_uk=True)
    out, lse = run_decode(inp, parts)
    _compare(out, lse, oracle_decode(inp, heads=[0, 1, 63, 64, 127]))


def test_decode_replays_in_a_cuda_graph():
    """The four launches of a decode call (programmatic dependent launches)
    captured in a CUDA graph: two replays give the eager call's output and LSE
    bit for bit."""
    w = _decode_workload(3, 16, [1, 2, 1], [300, 1000, 77])
    inp = make_inputs(w, with_w_uk=True)
    ref_out, ref_lse = run_decode(inp)
    B, H, T = inp["B"], w.H, inp["T_q"]
    max_new = int(inp["new_lens"].max())
    max_seq = int((inp["new_lens"] + inp["cache_lens"]).max())
    nparts = mla.mla_decode_partitions(B, H, max_new, max_seq)
    nbytes = mla.mla_decode_workspace_bytes(H, T, nparts)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = {k: inp[k].to(DEV) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache", "page_table",
                                     "w_uk", "w_uv")}

    def call():
        mla.check(mla.mla_decode(out, lse, d["q"], d["input_row_offsets"], d["cache_lengths"], d["kv_cache"],
                                 d["page_table"], inp["num_pages"], inp["page_size"], inp["max_pages"],
                                 d["w_uk"], d["w_uv"], B, H, T, max_new, max_seq, 0, inp["scale"],
                                 workspace=ws, workspace_bytes=nbytes, d_status=st))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0, mla.status_string(int(st.item()))
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)


def test_decode_small_heads_many_tokens():
    """16 heads: one 128-row tile holds 8 tokens of a sequence; a sequence of
    20 new tokens spans three tiles, each with its own causal limit."""
    w = _decode_workload(2, 16, (20, 3), (500, 64))
    inp = make_inputs(w, with_w_uk=True)
    out, lse = run_decode(inp, 2)
    _compare(out, lse, oracle_decode(inp))


def test_decode_one_head():
    """One head: a 128-row tile holds 128 tokens of a sequence, so a sequence
    of 150 new tokens spans two tiles with different causal limits."""
    w = _decode_workload(2, 1, (150, 2), (300, 1000))
    inp = make_inputs(w, with_w_uk=True)
    out, lse = run_decode(inp, 3)
    _compare(out, lse, oracle_decode(inp))


def test_decode_partition_count_invariance():
    w = _decode_workload(3, 8, (2, 1, 1), (700, 2000, 1))
    inp = make_inputs(w, with_w_uk=True)
    ref = oracle_decode(inp)
    outs = [run_decode(inp, p) for p in (1, 4, 9, 40)]
    for o, l in outs:
        _compare(o, l, ref)
    # more partitions than tiles: empty partitions contribute nothing
    assert torch.isfinite(outs[-1][0].float()).all()


def test_decode_full_size_sampled():
    """The DeepSeek-V3 decode workload (64 sequences, 1-2 new tokens over 4k-16k
    cached, shuffled pages) in the launch configuration the benchmark times;
    the oracle checks 3 heads of 6 sequences."""
    w = DECODE_WORKLOADS["v3_decode"]
    inp = make_inputs(w, with_w_uk=True)
    out, lse = run_decode(inp)
    _compare(out, lse, oracle_decode(inp, heads=[0, 77, 127], seqs=[0, 9, 21, 40, 52, 63]))


def test_decode_bad_page_reports_status():
    w = _decode_workload(2, 4, (1, 1), (100, 150))
    inp = make_inputs(w, with_w_uk=True)
    inp["page_table"][1, 0] = inp["num_pages"] + 5
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_decode(inp, 1, status=st)
    assert int(st.item()) == mla.MLA_DEV_BAD_PAGE


def oracle_sparse(inp, idx, topk, sink=None, heads=None, seqs=None):
    """The oracle's sparse decode on a sample of heads and sequences."""
    w = inp["workload"]
    hs = list(range(w.H)) if heads is None else list(heads)
    bs = list(range(inp["B"])) if seqs is None else list(seqs)
    iro = inp["input_row_offsets"].numpy().astype(np.int64)
    rows = np.concatenate([np.arange(iro[b], iro[b + 1]) for b in bs])
    new = np.array([iro[b + 1] - iro[b] for b in bs])
    iro_s = np.concatenate([[0], np.cumsum(new)])
    q = O.decode(O.codes(inp["q"]), "bf16")[rows][:, hs]
    w_uk = O.decode(O.codes(inp["w_uk"]), "bf16")[hs]
    w_uv = O.decode(O.codes(inp["w_uv"]), "bf16")[hs]
    res = O.mla_sparse_decode(q, O.codes(inp["kv_cache"]), inp["page_size"], w_uk, w_uv, iro_s,
                              idx.numpy()[bs], None if topk is None else topk.numpy()[bs], inp["scale"],
                              attn_sink=None if sink is None else sink.numpy()[bs])
    return {(bs[bi], hs[hi]): (rows[tok], o, l) for (bi, hi), (tok, o, l) in res.items()}


@pytest.mark.parametrize("with_sink", [False, True])
def test_sparse_decode_listed_rows(with_sink):
    """Sparse decode over top-k lists of physical rows (4 rows a gather), with
    counts below the list stride (garbage past them is never read), several
    tokens per sequence sharing one list, and optional sinks."""
    w = _decode_workload(3, 8, (1, 3, 2), (300, 90, 1000), page_size=32)
    inp = make_inputs(w, with_w_uk=True)
    idx, topk = make_sparse_indices(inp, 150, stride=160, pad=2 ** 30)
    sink = make_attention_sinks(3) if with_sink else None
    out, lse = run_decode(inp, 2, indices=idx.to(DEV), stride=160, topk=topk.to(DEV),
                          sink=None if sink is None else sink.to(DEV))
    _compare(out, lse, oracle_sparse(inp, idx, topk, sink))


def test_sparse_decode_empty_and_single_lists():
    """A sequence with no listed row (LSE -inf, output 0; with a sink, LSE =
    sink) and one with a single row (output = w_uv[h] times that row)."""
    w = _decode_workload(3, 4, (1, 1, 2), (64, 200, 10), page_size=16)
    inp = make_inputs(w, with_w_uk=True)
    idx, cnt = make_sparse_indices(inp, 40, stride=40)
    topk = torch.tensor([0, 1, int(cnt[2])], dtype=torch.int32)
    for sink in (None, make_attention_sinks(3, seed=3)):
        out, lse = run_decode(inp, 3, indices=idx.to(DEV), stride=40, topk=topk.to(DEV),
                              sink=None if sink is None else sink.to(DEV))
        ref = oracle_sparse(inp, idx, topk, sink, seqs=[1, 2])
        _compare(out, lse, ref)
        assert (out[0].float() == 0).all()
        expect = float("-inf") if sink is None else float(sink[0])
        assert torch.all(lse[0].cpu() == expect)


def test_dense_decode_with_sink_equals_sparse_over_the_context():
    """Dense decode with sinks equals the oracle's sparse decode listing each
    sequence's whole context (one new token each, so the causal limit is the
    whole context)."""
    w = _decode_workload(3, 16, (1, 1, 1), (700, 64, 1500))
    inp = make_inputs(w, with_w_uk=True)
    L = inp["new_lens"] + inp["cache_lens"]
    idx, topk = make_sparse_indices(inp, int(L.max()))
    sink = make_attention_sinks(3, seed=5)
    out, lse = run_decode(inp, 3, sink=sink.to(DEV))
    _compare(out, lse, oracle_sparse(inp, idx, topk, sink))


def test_sparse_decode_full_size_sampled():
    """64 sequences over 4k-16k cached tokens, top-2048 lists, per-batch sinks:
    the launch configuration the benchmark times; 3 heads of 6 sequences."""
    w = DECODE_WORKLOADS["v3_sparse_decode"]
    inp = make_inputs(w, with_w_uk=True)
    idx, topk = make_sparse_indices(inp, 2048)
    sink = make_attention_sinks(w.B)
    out, lse = run_decode(inp, indices=idx.to(DEV), stride=2048, topk=topk.to(DEV), sink=sink.to(DEV))
    _compare(out, lse, oracle_sparse(inp, idx, topk, sink, heads=[0, 50, 127], seqs=[0, 7, 19, 33, 48, 63]))


def test_sparse_decode_bad_row_reports_status():
    w = _decode_workload(2, 4, (1, 1), (100, 150), page_size=16)
    inp = make_inputs(w, with_w_uk=True)
    idx, topk = make_sparse_indices(inp, 30)
    idx[1, 3] = inp["num_pages"] * inp["page_size"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_decode(inp, 1, indices=idx.to(DEV), stride=30, topk=topk.to(DEV), status=st)
    assert int(st.item()) == mla.MLA_DEV_BAD_PAGE
