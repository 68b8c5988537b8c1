"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Plan and gather must match bit for bit; the projection
within bf16 (or e4m3) rounding; attention within max-abs 2e-2 / mean-rel 1e-2
for bf16 (6e-2 / 3e-2 for e4m3), mean-rel = sum|gpu-ref| / sum|ref|."""
import math

import numpy as np
import pytest
import torch

import mla_prefill_attention_plan_gb300 as mla
import oracle as O
from oracle import mla_oracle as M
from workloads import (WORKLOADS, lengths, make_attention_operands, make_cache_write_operands,
                       make_inputs, scaled)

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {"bf16": (2e-2, 1e-2), "e4m3": (6e-2, 3e-2)}
LSE_TOL = {"bf16": 5e-3, "e4m3": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_prefill_attention_plan_gb300 import build
    build.build()
    mla.load()
    assert torch.cuda.is_available()


@pytest.fixture
def bf16_kernel():
    """The bf16 attention kernel: one kernel (two-SM pairs), no fallback."""
    assert mla.mla_attention_kernel(mla.MLA_BF16) == "pair"
    return "pair"


def _dt(w):
    return mla.MLA_BF16 if w.dtype == "bf16" else mla.MLA_E4M3


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int64).astype(np.int32)).to(DEV)


def gpu_plan(iro, cache, S, max_chunks):
    B = len(cache)
    bro = torch.full((max_chunks, B + 1), -7, dtype=torch.int32, device=DEV)
    co = torch.full((max_chunks, max(B, 1)), -7, dtype=torch.int32, device=DEV)
    bl = torch.full((max_chunks,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill_plan(bro, co, bl, _i32(iro), _i32(cache) if B else _i32([0]), B,
                                   max_chunks, S, st))
    torch.cuda.synchronize()
    return (bro.cpu().numpy().astype(np.int64), co.cpu().numpy()[:, :B].astype(np.int64),
            bl.cpu().numpy().astype(np.int64), int(st.item()))


def _assert_plan_equal(iro, cache, S, mc):
    g = gpu_plan(iro, cache, S, mc)
    o = O.prefill_plan(iro, cache, S, mc)
    assert g[3] == o[3]
    if o[3] in (0, M.STATUS_TOO_MANY_CHUNKS):
        np.testing.assert_array_equal(g[0], o[0])
        np.testing.assert_array_equal(g[1], o[1])
        np.testing.assert_array_equal(g[2], o[2])


# ----------------------------------------------------------------------------- plan

@pytest.mark.parametrize("name", list(WORKLOADS))
def test_plan_workloads_bit_exact(name):
    w = WORKLOADS[name]
    new, cache = lengths(w)
    iro = np.concatenate([[0], np.cumsum(new)])
    _assert_plan_equal(iro, cache, w.buffer_token_size, w.max_chunks)


def test_plan_random_fuzz():
    rng = np.random.default_rng(5)
    for _ in range(150):
        B = int(rng.integers(1, 60))
        new = rng.integers(0, 300, B)
        cache = rng.integers(0, 300, B)
        S = int(rng.integers(1, 700))
        need = -(-int((new + cache).sum()) // S)
        mc = max(1, need + int(rng.integers(-2, 3)))
        _assert_plan_equal(np.concatenate([[0], np.cumsum(new)]), cache, S, mc)


@pytest.mark.parametrize("B", [4096, 4097, 20000, 300000])
def test_plan_many_sequences(B):
    """Multi-tile plans (tiles of 2048 sequences); 300000 sequences make 147 tiles."""
    rng = np.random.default_rng(B)
    new = rng.integers(0, 64, B)
    cache = rng.integers(0, 64, B)
    S = max(20000, int((new + cache).sum()) // 3)
    need = -(-int((new + cache).sum()) // S)
    _assert_plan_equal(np.concatenate([[0], np.cumsum(new)]), cache, S, need + 1)


def test_plan_many_tiles_garbage_tables():
    """600000 sequences (293 tiles of 2048), with the tables full of garbage
    beforehand (row 0 of cache_offsets holds scratch during
    the call and must come out zero); called twice on the same buffers."""
    rng = np.random.default_rng(41)
    B = 600_000
    new, cache = rng.integers(0, 64, B), rng.integers(0, 64, B)
    iro = np.concatenate([[0], np.cumsum(new)])
    S = int((new + cache).sum()) // 2 + 1
    mc = 3
    o = O.prefill_plan(iro, cache, S, mc)
    bro = torch.full((mc, B + 1), -7, dtype=torch.int32, device=DEV)
    co = torch.full((mc, B), -7, dtype=torch.int32, device=DEV)
    bl = torch.full((mc,), -7, dtype=torch.int32, device=DEV)
    iro_d, cl_d = _i32(iro).to(DEV), _i32(cache).to(DEV)
    for _ in range(2):
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        mla.check(mla.mla_prefill_plan(bro, co, bl, iro_d, cl_d, B, mc, S, st))
        torch.cuda.synchronize()
        assert int(st.item()) == o[3] == 0
        np.testing.assert_array_equal(bro.cpu().numpy(), o[0])
        np.testing.assert_array_equal(co.cpu().numpy(), o[1])
        np.testing.assert_array_equal(bl.cpu().numpy(), o[2])


def test_plan_multi_tile_status_codes():
    """Status codes from the multi-tile path: a decreasing offset in a middle
    tile, a total of 2^31 tokens or more, and too few chunk rows."""
    B = 50000
    new = np.full(B, 3)
    cache = np.full(B, 5)
    iro = np.concatenate([[0], np.cumsum(new)])
    bad = iro.copy()
    bad[30001] = bad[30000] - 1
    assert gpu_plan(bad, cache, 1000, 500)[3] == mla.MLA_DEV_BAD_OFFSETS
    big = np.full(B, 50000)     # 2.5e9 context tokens
    assert gpu_plan(iro, big, 1 << 30, 4)[3] == mla.MLA_DEV_BAD_OFFSETS
    assert gpu_plan(iro, cache, 1000, 399)[3] == mla.MLA_DEV_TOO_MANY_CHUNKS
    _assert_plan_equal(iro, cache, 1000, 399)        # the rows that exist are still right


def test_plan_unaligned_tables():
    """Tables and inputs 4 bytes off a 16-byte boundary (the plan takes any
    4-byte aligned pointers): same tables."""
    rng = np.random.default_rng(5)
    B = 70000
    new, cache = rng.integers(0, 64, B), rng.integers(0, 64, B)
    iro = np.concatenate([[0], np.cumsum(new)])
    S = int((new + cache).sum()) // 3 + 1
    mc = 4
    def shifted(n, fill):
        t = torch.full((n + 1,), fill, dtype=torch.int32, device=DEV)
        return t, t.data_ptr() + 4
    bro_t, bro_p = shifted(mc * (B + 1), -7)
    co_t, co_p = shifted(mc * B, -7)
    bl = torch.full((mc,), -7, dtype=torch.int32, device=DEV)
    iro_t, iro_p = shifted(B + 1, 0)
    iro_t[1:] = _i32(iro)
    cl_t, cl_p = shifted(B, 0)
    cl_t[1:] = _i32(cache)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill_plan(bro_p, co_p, bl, iro_p, cl_p, B, mc, S, st))
    torch.cuda.synchronize()
    o = O.prefill_plan(iro, cache, S, mc)
    assert int(st.item()) == o[3] == 0
    np.testing.assert_array_equal(bro_t[1:].cpu().numpy().reshape(mc, B + 1), o[0])
    np.testing.assert_array_equal(co_t[1:].cpu().numpy().reshape(mc, B), o[1])
    np.testing.assert_array_equal(bl.cpu().numpy(), o[2])


def test_plan_empty_batch():
    """No sequences: every chunk is unused (length -1, row [0])."""
    bro, co, bl, st = gpu_plan([0], [], 8, 3)
    o = O.prefill_plan([0], [], 8, 3)
    assert st == o[3] == 0
    np.testing.assert_array_equal(bro, o[0])
    np.testing.assert_array_equal(bl, o[2])
    assert list(bl) == [-1, -1, -1]


def test_plan_status_codes():
    assert gpu_plan([0, 10], [0], 4, 2)[3] == mla.MLA_DEV_TOO_MANY_CHUNKS
    _assert_plan_equal([0, 10], [0], 4, 2)          # truncated rows still written
    assert gpu_plan([1, 3], [0], 4, 2)[3] == mla.MLA_DEV_BAD_OFFSETS
    assert gpu_plan([0, 5, 3], [0, 0], 4, 4)[3] == mla.MLA_DEV_BAD_OFFSETS
    bro, co, bl, st = gpu_plan([0, 0, 0], [0, 0], 8, 3)
    assert st == 0 and list(bl) == [-1, -1, -1]


# ----------------------------------------------------------------------------- latent-cache write

def _assert_rounded(gpu_codes, exact, dtype, what, allow):
    """Storage codes from the GPU against exact float64 values.  The oracle's
    rounding (nearest even) must match, except where the exact value lies
    within `allow` (the float32 error bound of the kernel's arithmetic for that
    element) of a rounding midpoint: the kernel rounds its float32 result, so
    there either neighbour is a correct rounding."""
    want = M.bf16_encode(exact) if dtype == "bf16" else M.e4m3_encode(exact)
    diff = np.asarray(gpu_codes) != want
    if diff.any():
        g = O.decode(np.asarray(gpu_codes)[diff], dtype)
        w = O.decode(want[diff], dtype)
        x = exact[diff]
        near_tie = np.abs(x - 0.5 * (g + w)) <= allow[diff]
        assert near_tie.all(), (f"{what}: {int((~near_tie).sum())} codes differ away from a tie, e.g. exact "
                                f"{x[~near_tie][:3]} gpu {g[~near_tie][:3]} oracle {w[~near_tie][:3]}")
    return int(diff.sum())


def _rope_allow(x):
    """Error bound of a float32 rotation of interleaved pairs (a, b): each
    output is a*c -/+ b*s with |c|, |s| <= 1, so it is off by at most a few
    units of 2**-24 times |a| + |b|."""
    x = np.asarray(x, dtype=np.float64)
    m = np.abs(x[..., 0::2]) + np.abs(x[..., 1::2])
    return 1e-6 * np.repeat(m, 2, axis=-1)


def _cache_write_case(w, cache_dtype="bf16", inv_scale=1.0, with_q=True, freqs_rows=None,
                      drop_page=None):
    inp = make_inputs(scaled(w, dtype="bf16"))
    T, B = inp["T_q"], inp["B"]
    L = inp["new_lens"] + inp["cache_lens"]
    lat, gamma, freqs = make_cache_write_operands(w, T, int(L.max()) + 1)
    if freqs_rows is not None:
        freqs = freqs[:freqs_rows].contiguous()
    cache = inp["kv_cache"] if cache_dtype == "bf16" else inp["kv_cache"].float().to(torch.float8_e4m3fn)
    pt = inp["page_table"].clone()
    if drop_page is not None:
        pt[drop_page] = -1
    eps = 1e-6
    kv_d = cache.to(DEV)
    q_d = inp["q"].to(DEV) if with_q else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_latent_cache_write(
        kv_d, q_d, lat.to(DEV), gamma.to(DEV), freqs.to(DEV), inp["input_row_offsets"].to(DEV),
        inp["cache_lengths"].to(DEV), pt.to(DEV), inp["num_pages"], inp["page_size"],
        inp["max_pages"], B, w.H, T, freqs.shape[0], eps, inv_scale,
        mla.MLA_BF16 if cache_dtype == "bf16" else mla.MLA_E4M3, st))
    torch.cuda.synchronize()
    lat64 = O.decode(O.codes(lat), "bf16")
    q64 = O.decode(O.codes(inp["q"]), "bf16") if with_q else None
    kv_o, q_o, st_o = O.latent_cache_write(lat64, q64, gamma.numpy(), freqs.numpy(),
                                           inp["input_row_offsets"].numpy(), inp["cache_lengths"].numpy(),
                                           pt.numpy(), inp["page_size"], O.codes(cache), eps,
                                           dtype=cache_dtype, inv_scale=inv_scale)
    return dict(inp=inp, lat64=lat64, gamma=gamma.numpy(), freqs=freqs.numpy(), pt=pt.numpy(),
                kv_gpu=O.codes(kv_d.cpu()), q_gpu=O.codes(q_d.cpu()) if with_q else None,
                st_gpu=int(st.item()), kv_o=kv_o, q_o=q_o, st_o=st_o, eps=eps)


def _check_cache_write(c, cache_dtype, inv_scale=1.0):
    """Rows the oracle did not write are bit-identical; written rows and q's
    rope parts agree with the oracle's exact values up to ties."""
    inp = c["inp"]
    assert c["st_gpu"] == c["st_o"]
    iro, cl, ps = inp["input_row_offsets"].numpy(), inp["cache_lengths"].numpy(), inp["page_size"]
    written = np.zeros(c["kv_o"].shape[:2], dtype=bool)
    exact_rows = {}
    for b in range(inp["B"]):
        for i in range(int(iro[b + 1] - iro[b])):
            p = int(cl[b]) + i
            if p >= c["freqs"].shape[0]:
                continue
            pg = c["pt"][b, p // ps] if p // ps < c["pt"].shape[1] else -1
            if pg < 0:
                continue
            t = int(iro[b]) + i
            row = np.concatenate([O.rms_norm(c["lat64"][t, :512], c["gamma"], c["eps"]),
                                  O.rope_rotate(c["lat64"][t, 512:], c["freqs"][p])])
            # float32 RMSNorm: a relative error well under 5e-5 (512-term sum of squares,
            # square root, two products); rotation: see _rope_allow.
            allow = np.concatenate([5e-5 * np.abs(row[:512]), _rope_allow(c["lat64"][t, 512:])])
            written[pg, p % ps] = True
            exact_rows[(pg, p % ps)] = (row * inv_scale, allow * inv_scale)
    np.testing.assert_array_equal(c["kv_gpu"][~written], c["kv_o"][~written])
    keys = sorted(exact_rows)
    ties = 0
    if keys:
        gpu = np.stack([c["kv_gpu"][k] for k in keys])
        ex = np.stack([exact_rows[k][0] for k in keys])
        allow = np.stack([exact_rows[k][1] for k in keys])
        ties += _assert_rounded(gpu, ex, cache_dtype, "cache rows", allow)
    if c["q_gpu"] is not None:
        q_in = O.decode(O.codes(inp["q"]), "bf16")
        np.testing.assert_array_equal(c["q_gpu"][:, :, :128], O.codes(inp["q"])[:, :, :128])
        ties += _assert_rounded(c["q_gpu"][:, :, 128:], c["q_o"][:, :, 128:], "bf16", "q rope",
                                _rope_allow(q_in[:, :, 128:]))
    return ties


def test_cache_write_tiny_ragged_bf16():
    w = scaled(WORKLOADS["tiny_ragged"], H=4, page_size=8, shuffle_pages=True)
    c = _cache_write_case(w)
    _check_cache_write(c, "bf16")


def test_cache_write_ragged_chunked_bf16():
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=3)
    c = _cache_write_case(w)
    ties = _check_cache_write(c, "bf16")
    n = c["inp"]["T_q"] * (576 + 3 * 64)
    assert ties < 1e-3 * n


def test_cache_write_e4m3_cache_scaled():
    w = scaled(WORKLOADS["tiny_ragged"], H=2, page_size=16)
    c = _cache_write_case(w, cache_dtype="e4m3", inv_scale=2.0, with_q=False)
    _check_cache_write(c, "e4m3", inv_scale=2.0)


def test_cache_write_v3_full_size():
    """The DeepSeek-V3 shape in full: 4096 new tokens, 128 heads, every cache
    row and every q rope value compared."""
    c = _cache_write_case(WORKLOADS["v3_prefill"])
    ties = _check_cache_write(c, "bf16")
    assert ties < 1e-3 * 4096 * (576 + 128 * 64)


def test_cache_write_status_codes():
    w = scaled(WORKLOADS["tiny_ragged"], H=2, page_size=8)
    # Positions past the frequency table: those tokens are skipped entirely.
    c = _cache_write_case(w, freqs_rows=50)
    assert c["st_gpu"] == c["st_o"] == mla.MLA_DEV_BAD_OFFSETS
    _check_cache_write(c, "bf16")
    # A missing page where sequence 1's new tokens go: its rows stay unwritten.
    c = _cache_write_case(w, drop_page=(1, 6))
    assert c["st_gpu"] == c["st_o"] == mla.MLA_DEV_BAD_PAGE
    _check_cache_write(c, "bf16")


def test_cache_write_then_prefill_matches_oracle():
    """The write feeds the prefill: the fused path over the written cache,
    with the rotated q, matches the oracle's prefill over the oracle's cache."""
    w = scaled(WORKLOADS["tiny_ragged"], H=3, page_size=8)
    c = _cache_write_case(w)
    bf16 = lambda codes: torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(torch.bfloat16)
    gpu_in = dict(c["inp"], kv_cache=bf16(c["kv_gpu"]), q=bf16(c["q_gpu"]))
    ora_in = dict(c["inp"], kv_cache=bf16(c["kv_o"]), q=bf16(M.bf16_encode(c["q_o"])))
    out, lse = run_fused(gpu_in)
    _compare(out, oracle_fused(ora_in), "bf16", lse)


# ----------------------------------------------------------------------------- gather

def _gather_case(w, **kw):
    inp = make_inputs(w, **kw)
    c = {k: O.codes(inp[k]) for k in ("kv_cache", "page_table", "input_row_offsets", "cache_lengths")}
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], w.buffer_token_size, w.max_chunks)
    S = w.buffer_token_size
    B = inp["B"]
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, w.max_chunks)
    tdt = inp["kv_cache"].dtype
    kv = inp["kv_cache"].to(DEV)
    pt = inp["page_table"].to(DEV)
    bro = torch.as_tensor(g[0].astype(np.int32)).to(DEV)
    co = torch.as_tensor(g[1].astype(np.int32)).to(DEV)
    bl = torch.as_tensor(g[2].astype(np.int32)).to(DEV)
    for ch in range(w.max_chunks):
        ckv = torch.full((S, 512), 0.5, dtype=torch.float32).to(tdt).to(DEV)
        kr = torch.full((S, 64), 0.5, dtype=torch.float32).to(tdt).to(DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        mla.check(mla.mla_gather_latent(ckv, kr, kv, pt, inp["num_pages"], inp["page_size"],
                                        inp["max_pages"], bro, co, bl, ch, B, S, _dt(w), st))
        torch.cuda.synchronize()
        assert st.item() == 0
        o_ckv, o_kr, ost = O.gather_latent(c["kv_cache"], c["page_table"], inp["page_size"], plan, ch)
        assert ost == 0
        n = max(int(plan[2][ch]), 0)
        g_ckv, g_kr = O.codes(ckv.cpu()), O.codes(kr.cpu())
        np.testing.assert_array_equal(g_ckv[:n], o_ckv)
        np.testing.assert_array_equal(g_kr[:n], o_kr)
        # rows past the chunk's length are left untouched
        sentinel = O.codes(torch.full((1,), 0.5).to(tdt))[0]
        assert np.all(g_ckv[n:] == sentinel) and np.all(g_kr[n:] == sentinel)


def test_gather_tiny_ragged():
    _gather_case(WORKLOADS["tiny_ragged"])


def test_gather_shuffled_pages_multi_chunk():
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=1, buffer_token_size=1000, max_chunks=16,
               new_range=(1, 500), cache_range=(0, 900), page_size=16)
    _gather_case(w)


def test_gather_e4m3():
    w = scaled(WORKLOADS["longctx_fp8"], H=1, new_lens=(300,), cache_lens=(200,),
               buffer_token_size=192, max_chunks=3, page_size=64)
    _gather_case(w)


@pytest.mark.parametrize("name", ["ragged_chunked_cache", "longctx_fp8"])
def test_gather_full_size_every_chunk_bit_exact(name):
    """The full-size gathers the benchmark runs (seeded shuffled pages and 8192-row
    chunks; 16k + 16k e4m3 tokens), every chunk compared bit for bit with the
    oracle, the rows past the chunk untouched."""
    _gather_case(WORKLOADS[name])


def test_gather_bad_page_reports_status():
    w = WORKLOADS["tiny_ragged"]
    inp = make_inputs(w)
    pt = inp["page_table"].clone()
    pt[1, 2] = inp["num_pages"] + 5
    g = gpu_plan(O.codes(inp["input_row_offsets"]), O.codes(inp["cache_lengths"]), 32, 4)
    ckv = torch.zeros(32, 512, dtype=torch.bfloat16, device=DEV)
    kr = torch.zeros(32, 64, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    for ch in range(4):
        mla.check(mla.mla_gather_latent(ckv, kr, inp["kv_cache"].to(DEV), pt.to(DEV),
                                        inp["num_pages"], 16, inp["max_pages"], *tabs, ch, 2, 32,
                                        mla.MLA_BF16, st))
    torch.cuda.synchronize()
    assert st.item() == mla.MLA_DEV_BAD_PAGE


# ----------------------------------------------------------------------------- up-projection

@pytest.mark.parametrize("dtype,H,rows,S", [("bf16", 4, 89, 96), ("bf16", 3, 300, 320),
                                            ("bf16", 16, 1000, 1024), ("e4m3", 4, 200, 256)])
def test_upproject(dtype, H, rows, S):
    w = scaled(WORKLOADS["tiny_ragged" if dtype == "bf16" else "longctx_fp8"], H=H)
    gen = torch.Generator().manual_seed(H * 1000 + rows)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
    ckv = torch.randn(S, 512, generator=gen).to(tdt)
    wstd, wsc = (1 / math.sqrt(512), 1.0) if dtype == "bf16" else (1.0, 1 / math.sqrt(512))
    wk = (torch.randn(H * 128, 512, generator=gen) * wstd).to(tdt)
    wuv = (torch.randn(H, 128, 512, generator=gen) * wstd).to(tdt)
    kn = torch.full((S, H, 128), 3.0).to(tdt).to(DEV)
    vv = torch.full((S, H, 128), 3.0).to(torch.bfloat16 if dtype == "bf16" else torch.float16).to(DEV)
    bl = torch.tensor([rows], dtype=torch.int32, device=DEV)
    mla.check(mla.mla_upproject(kn, vv, ckv.to(DEV), wk.to(DEV), wuv.to(DEV), bl, 0, S, H,
                                mla.MLA_BF16 if dtype == "bf16" else mla.MLA_E4M3, 1.0, wsc, 1.0))
    torch.cuda.synchronize()
    rk, rv = O.upproject(O.decode(O.codes(ckv), dtype)[:rows], O.decode(O.codes(wk), dtype) * wsc,
                         O.decode(O.codes(wuv), dtype) * wsc)
    gk = kn.float().cpu().double().numpy()
    gv = vv.float().cpu().double().numpy()
    if dtype == "bf16":
        bound = lambda ref: 2.0 ** -8 * np.abs(ref) + 1e-3
    else:
        bound = lambda ref: 2.0 ** -3 * np.abs(ref) + 2.0 ** -8
    assert np.all(np.abs(gk[:rows] - rk) <= bound(rk))
    assert np.all(np.abs(gv[:rows] - rv) <= bound(rv))
    if dtype == "e4m3":
        # V is stored as f16 but must hold exactly the e4m3-rounded values
        assert np.array_equal(gv[:rows], O.round_to_e4m3(gv[:rows]))
    pad = min(S, -(-rows // 128) * 128)
    assert np.all(gk[rows:pad] == 0) and np.all(gv[rows:pad] == 0)   # zero-filled tile tail
    assert np.all(gk[pad:] == 3.0) and np.all(gv[pad:] == 3.0)       # untouched beyond it


def gpu_cache_rows(inp, tabs, S, mc, st=None, pt=None):
    """mla_chunk_cache_rows for all chunks: [mc, S] int32 on the device."""
    rows = torch.full((mc, S), -7, dtype=torch.int32, device=DEV)
    pt = inp["page_table"].to(DEV) if pt is None else pt
    mla.check(mla.mla_chunk_cache_rows(rows, pt, inp["num_pages"], inp["page_size"], inp["max_pages"],
                                       *tabs, mc, inp["B"], S, st))
    return rows


@pytest.mark.parametrize("name,kw", [
    ("tiny_ragged", {}),
    ("tiny_ragged", {"page_size": 1, "shuffle_pages": True}),
    ("ragged_chunked_cache", {"H": 1, "B": 300, "buffer_token_size": 512, "max_chunks": 8,
                              "new_range": (1, 5), "cache_range": (0, 4), "page_size": 3}),
    ("ragged_chunked_cache", {}),
    ("longctx_fp8", {}),
])
def test_chunk_cache_rows_bit_exact(name, kw):
    """The table of every chunk equals the oracle's, entry for entry (entries
    past a chunk's rows are 0), on the full-size workloads too."""
    w = scaled(WORKLOADS[name], **kw) if kw else WORKLOADS[name]
    inp = make_inputs(w)
    c = {k: O.codes(inp[k]) for k in ("input_row_offsets", "cache_lengths", "page_table")}
    S, mc = w.buffer_token_size, w.max_chunks
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows = gpu_cache_rows(inp, tabs, S, mc, st).cpu().numpy()
    assert st.item() == 0
    for ch in range(mc):
        ref, ost = O.chunk_cache_rows(c["page_table"], inp["page_size"], inp["num_pages"], plan, ch, S)
        assert ost == 0
        np.testing.assert_array_equal(rows[ch], ref)


def test_chunk_cache_rows_bad_page_reports_status():
    w = scaled(WORKLOADS["tiny_ragged"], page_size=16)
    inp = make_inputs(w)
    c = {k: O.codes(inp[k]) for k in ("input_row_offsets", "cache_lengths", "page_table")}
    S, mc = w.buffer_token_size, w.max_chunks
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    pt = inp["page_table"].clone()
    pt[inp["B"] - 1, 0] = inp["num_pages"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows = gpu_cache_rows(inp, tabs, S, mc, st, pt=pt.to(DEV))
    torch.cuda.synchronize()
    assert st.item() == mla.MLA_DEV_BAD_PAGE
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    for ch in range(mc):
        ref, _ = O.chunk_cache_rows(O.codes(pt), inp["page_size"], inp["num_pages"], plan, ch, S)
        np.testing.assert_array_equal(rows[ch].cpu().numpy(), ref)


def _paged_upproject_case(w, oracle=True, bad_page=False):
    """mla_upproject_paged, c_kv rows read from the paged cache through the
    chunk's cache-row table, every chunk: (1) bit for bit equal to
    mla_gather_latent + mla_upproject over the whole K and V buffers (the
    zeroed tile tail and the untouched rows past it included), and (2) within
    rounding of the oracle's projection of the oracle's gathered rows.  With
    bad_page, one table entry points outside the cache: reported, no fault."""
    inp = make_inputs(w)
    dt = w.dtype
    c = {k: O.codes(inp[k]) for k in ("kv_cache", "page_table", "input_row_offsets", "cache_lengths",
                                      "w_k", "w_uv")}
    S, mc, B, H = w.buffer_token_size, w.max_chunks, inp["B"], w.H
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    bro, co, bl = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    kv, pt = inp["kv_cache"].to(DEV), inp["page_table"].to(DEV)
    wk, wuv = inp["w_k"].to(DEV), inp["w_uv"].to(DEV)
    wsc = inp["w_scale"]
    paging = (inp["num_pages"], inp["page_size"], inp["max_pages"])
    ncr = inp["num_pages"] * inp["page_size"]
    rows_t = gpu_cache_rows(inp, [bro, co, bl], S, mc)
    if bad_page:
        rows_t[:, 5] = ncr + 7        # a table entry outside the cache
    vdt = torch.bfloat16 if dt == "bf16" else torch.float16
    st_bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    for ch in range(mc):
        res = {}
        for mode in ("paged",) if bad_page else ("buffer", "paged"):
            kn = torch.full((S, H, 128), 3.0).to(kv.dtype).to(DEV)
            vv = torch.full((S, H, 128), 3.0, dtype=vdt, device=DEV)
            st = st_bad if bad_page else torch.zeros(1, dtype=torch.int32, device=DEV)
            if mode == "buffer":
                ckv = torch.zeros(S, 512, dtype=kv.dtype, device=DEV)
                kr = torch.zeros(S, 64, dtype=kv.dtype, device=DEV)
                mla.check(mla.mla_gather_latent(ckv, kr, kv, pt, *paging, bro, co, bl, ch, B, S, _dt(w), st))
                mla.check(mla.mla_upproject(kn, vv, ckv, wk, wuv, bl, ch, S, H, _dt(w), 1.0, wsc, 1.0, st))
            else:
                mla.check(mla.mla_upproject_paged(kn, vv, kv, rows_t[ch], ncr, bl, ch, S, wk, wuv, H, _dt(w),
                                                  1.0, wsc, 1.0, st))
            torch.cuda.synchronize()
            res[mode] = (kn, vv, int(st.item()))
        if bad_page:
            continue
        assert res["buffer"][2] == 0 and res["paged"][2] == 0
        for i in (0, 1):
            assert torch.equal(res["buffer"][i].view(torch.uint8), res["paged"][i].view(torch.uint8)), (ch, i)
        n = max(int(plan[2][ch]), 0)
        if not oracle or n == 0:
            continue
        o_ckv, _, ost = O.gather_latent(c["kv_cache"], c["page_table"], inp["page_size"], plan, ch)
        assert ost == 0
        rk, rv = O.upproject(O.decode(o_ckv, dt), O.decode(c["w_k"], dt) * wsc,
                             O.decode(c["w_uv"], dt) * wsc)
        gk = res["paged"][0].float().cpu().double().numpy()[:n]
        gv = res["paged"][1].float().cpu().double().numpy()[:n]
        if dt == "bf16":
            bound = lambda ref: 2.0 ** -8 * np.abs(ref) + 1e-3
        else:
            bound = lambda ref: 2.0 ** -3 * np.abs(ref) + 2.0 ** -8
        assert np.all(np.abs(gk - rk) <= bound(rk))
        assert np.all(np.abs(gv - rv) <= bound(rv))
    if bad_page:
        assert int(st_bad.item()) == mla.MLA_DEV_BAD_PAGE


def test_paged_upproject_shuffled_pages_multi_chunk():
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=2, B=3, buffer_token_size=700, max_chunks=4,
               new_range=(100, 600), cache_range=(0, 900), page_size=16)
    _paged_upproject_case(w)


def test_paged_upproject_many_short_sequences():
    """300 sequences of 1..8 tokens: every 128-row tile spans dozens of them
    (the row -> sequence search), one-row pages."""
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=2, B=300, buffer_token_size=512, max_chunks=8,
               new_range=(1, 5), cache_range=(0, 4), page_size=1)
    _paged_upproject_case(w)


def test_paged_upproject_e4m3():
    w = scaled(WORKLOADS["longctx_fp8"], H=2, B=2, new_lens=(300, 41), cache_lens=(200, 0),
               buffer_token_size=192, max_chunks=3, page_size=64, shuffle_pages=True)
    _paged_upproject_case(w)


@pytest.mark.parametrize("name", ["ragged_chunked_cache", "longctx_fp8"])
def test_paged_upproject_full_size_equals_buffered(name):
    """Full size, every chunk: bit for bit equal to gather + buffered
    projection (whose own parity is covered above and by the fused tests)."""
    _paged_upproject_case(WORKLOADS[name], oracle=False)


def test_paged_upproject_bad_page_reports_status():
    w = scaled(WORKLOADS["tiny_ragged"], page_size=16)
    _paged_upproject_case(w, bad_page=True)


# ----------------------------------------------------------------------------- attention

def _compare(out, ref, dtype, lse=None):
    tol_abs, tol_rel = TOL[dtype]
    max_abs, num, den, lse_err = 0.0, 0.0, 0.0, 0.0
    out = out.float().cpu().double().numpy()
    lse_np = None if lse is None else lse.cpu().double().numpy()
    for (b, h), (tok, o, l) in ref.items():
        if tok.size == 0:
            continue
        g = out[tok, h]
        assert np.all(np.isfinite(g))
        d = np.abs(g - o)
        max_abs = max(max_abs, float(d.max()))
        num += float(d.sum())
        den += float(np.abs(o).sum())
        if lse_np is not None:
            lse_err = max(lse_err, float(np.abs(lse_np[tok, h] - l).max()))
    mean_rel = num / max(den, 1e-30)
    assert max_abs <= tol_abs, (max_abs, mean_rel)
    assert mean_rel <= tol_rel, (max_abs, mean_rel)
    assert lse_err <= LSE_TOL[dtype], lse_err
    return max_abs, mean_rel


def _attention_stage(w, seed_base=11):
    """Attention alone over seeded K/V buffers, chunk by chunk, with the merge
    scratch carried between calls."""
    inp = make_inputs(w)
    dt = w.dtype
    c = {k: O.codes(inp[k]) for k in ("q", "input_row_offsets", "cache_lengths")}
    S, mc, B, H, T = w.buffer_token_size, w.max_chunks, inp["B"], w.H, inp["T_q"]
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    ops = [make_attention_operands(w, S, seed_offset=seed_base + ch) for ch in range(mc)]
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, H, dtype=torch.float32, device=DEV)
    oacc = torch.empty(T, H, 128, dtype=torch.float32, device=DEV)
    lacc = torch.empty(T, H, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = inp["q"].to(DEV)
    for ch in range(mc):
        kn, vv, kr = (t.to(DEV) for t in ops[ch])
        mla.check(mla.mla_prefill_attention(out, lse, oacc, lacc, q, kn, vv, kr,
                                            inp["input_row_offsets"].to(DEV),
                                            inp["cache_lengths"].to(DEV), *tabs, ch, mc, B, H,
                                            inp["max_prompt_len"], T, S, inp["scale"],
                                            dtype=_dt(w), d_status=st))
    torch.cuda.synchronize()
    assert st.item() == 0

    def operands(ch):
        kn, vv, kr = ops[ch]
        # V of the e4m3 path is float16 holding e4m3 values: read it exactly
        v64 = vv.double().numpy() if dt == "e4m3" else O.decode(O.codes(vv), dt)
        return (O.decode(O.codes(kn), dt), O.decode(O.codes(kr), dt), v64)
    ref = O.attention_over_chunks(O.decode(c["q"], dt), operands, plan,
                                  c["input_row_offsets"], c["cache_lengths"], inp["scale"])
    return _compare(out, ref, dt, lse)


def test_attention_stage_multi_chunk(bf16_kernel):
    _attention_stage(WORKLOADS["tiny_ragged"])


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_attention_strongly_negative_scores(dtype):
    """Every score of every row near -140 (about -200 in log2 units, far below
    the fp32 exponent range once shifted by anything but the row's own
    maximum): the output is right only if each tile's maximum is taken over
    exactly its own scores.  q_nope = 4, k_nope = -4 plus a seeded multiple of
    1/4 (exact in bf16 and e4m3), rope parts zero, two sequences with two and
    one key tiles."""
    rng = np.random.default_rng(5)
    new, cache = np.array([150, 60]), np.array([0, 40])
    B, H, S = 2, 2, 256
    iro = np.concatenate([[0], np.cumsum(new)]).astype(np.int64)
    T = int(iro[-1])
    plan = O.prefill_plan(iro, cache, S, 1)
    g = gpu_plan(iro, cache, S, 1)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    store = torch.bfloat16 if dtype == "bf16" else torch.float8_e4m3fn
    q = torch.zeros(T, H, 192, dtype=torch.float32)
    q[:, :, :128] = 4.0
    q = q.to(store)
    kn = torch.as_tensor((-4.0 + rng.integers(0, 3, size=(S, H, 128)) / 4.0).astype(np.float32)).to(store)
    kr = torch.zeros(S, 64, dtype=torch.float32).to(store)
    vv = torch.as_tensor(rng.standard_normal((S, H, 128)).astype(np.float32)).to(store)
    if dtype == "e4m3":
        vv = vv.to(torch.float16)   # V of the e4m3 path: float16 holding e4m3 values
    scale = 1.0 / math.sqrt(192.0)
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, H, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill_attention(out, lse, None, None, q.to(DEV), kn.to(DEV), vv.to(DEV), kr.to(DEV),
                                        _i32(iro), _i32(cache), *tabs, 0, 1, B, H, int(new.max()), T, S, scale,
                                        dtype=mla.MLA_BF16 if dtype == "bf16" else mla.MLA_E4M3, d_status=st))
    torch.cuda.synchronize()
    assert st.item() == 0
    dec = lambda t: O.decode(O.codes(t), dtype)
    v64 = vv.double().numpy() if dtype == "e4m3" else dec(vv)
    ref = O.attention_over_chunks(dec(q), lambda ch: (dec(kn), dec(kr), v64), plan, iro, cache, scale)
    _compare(out, ref, dtype, lse)


def test_attention_offsets_past_total_q_tokens():
    """input_row_offsets[B] beyond total_q_tokens: the device reports bad
    offsets, leaves that sequence out and writes no row at or past
    total_q_tokens (the guard row past the declared output stays as it was);
    the sequence inside the bound is still computed."""
    w = scaled(WORKLOADS["tiny_ragged"], buffer_token_size=128, max_chunks=1)
    inp = make_inputs(w)
    c = {k: O.codes(inp[k]) for k in ("input_row_offsets", "cache_lengths")}
    S, B, H, T = 128, inp["B"], w.H, inp["T_q"]
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, 1)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    kn, vv, kr = (t.to(DEV) for t in make_attention_operands(w, S))
    out = torch.full((T, H, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), 3.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill_attention(out, lse, None, None, inp["q"].to(DEV), kn, vv, kr,
                                        inp["input_row_offsets"].to(DEV),
                                        inp["cache_lengths"].to(DEV), *tabs, 0, 1, B, H,
                                        inp["max_prompt_len"], T - 1, S, inp["scale"], d_status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == mla.MLA_DEV_BAD_OFFSETS
    n0 = int(inp["new_lens"][0])
    assert (out[n0:].float() == 3.0).all() and (lse[n0:] == 3.0).all()
    assert not (out[:n0].float() == 3.0).any()


def test_head_split_equals_full_call_bit_for_bit():
    """The multi-GPU split of the path is by heads (w_k, w_uv, q, K/V and out
    sliced on H, no collective): two attention calls on heads [0, H/2) and
    [H/2, H), each given its own contiguous slices, reproduce the full-H
    call bit for bit, on a multi-chunk plan."""
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=8, B=3, buffer_token_size=700, max_chunks=5,
               new_range=(100, 600), cache_range=(0, 900))
    inp = make_inputs(w)
    c = {k: O.codes(inp[k]) for k in ("input_row_offsets", "cache_lengths")}
    S, B, H, T = w.buffer_token_size, inp["B"], w.H, inp["T_q"]
    mc = -(-int((inp["new_lens"] + inp["cache_lens"]).sum()) // S)
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    ops = [tuple(t.to(DEV) for t in make_attention_operands(w, S, seed_offset=31 + ch)) for ch in range(mc)]
    q = inp["q"].to(DEV)
    iro, cl = inp["input_row_offsets"].to(DEV), inp["cache_lengths"].to(DEV)

    def run(h0, h1):
        hs = h1 - h0
        out = torch.empty(T, hs, 128, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(T, hs, dtype=torch.float32, device=DEV)
        oacc = torch.empty(T, hs, 128, dtype=torch.float32, device=DEV)
        lacc = torch.empty(T, hs, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        qs = q[:, h0:h1].contiguous()
        for ch in range(mc):
            kn, vv, kr = ops[ch]
            mla.check(mla.mla_prefill_attention(out, lse, oacc, lacc, qs, kn[:, h0:h1].contiguous(),
                                                vv[:, h0:h1].contiguous(), kr, iro, cl, *tabs, ch, mc, B,
                                                hs, inp["max_prompt_len"], T, S, inp["scale"], d_status=st))
        torch.cuda.synchronize()
        assert st.item() == 0
        return out, lse
    full_o, full_l = run(0, H)
    lo_o, lo_l = run(0, H // 2)
    hi_o, hi_l = run(H // 2, H)
    assert torch.equal(torch.cat([lo_o, hi_o], 1).view(torch.int16), full_o.view(torch.int16))
    assert torch.equal(torch.cat([lo_l, hi_l], 1), full_l)


def _paged_attention_case(w, seed_base=41, oracle=True, bad_page=False):
    """mla_prefill_attention_paged, k_rope read from the paged cache through
    the chunk's cache-row table, chunk by chunk: (1) bit for bit equal to
    mla_prefill_attention given the gathered k_rope rows (the masked keys past
    a sequence read other rows in the two calls and must change nothing), and
    (2) against the oracle, whose k_rope for a key is the cache row of its
    context position.  With bad_page, one table entry points outside the
    cache: reported, no fault."""
    inp = make_inputs(w)
    dt = w.dtype
    c = {k: O.codes(inp[k]) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache",
                                      "page_table")}
    S, mc, B, H, T = w.buffer_token_size, w.max_chunks, inp["B"], w.H, inp["T_q"]
    plan = O.prefill_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    g = gpu_plan(c["input_row_offsets"], c["cache_lengths"], S, mc)
    tabs = [torch.as_tensor(x.astype(np.int32)).to(DEV) for x in g[:3]]
    kv, pt = inp["kv_cache"].to(DEV), inp["page_table"].to(DEV)
    q = inp["q"].to(DEV)
    iro, cl = inp["input_row_offsets"].to(DEV), inp["cache_lengths"].to(DEV)
    paging = (inp["num_pages"], inp["page_size"], inp["max_pages"])
    ncr = inp["num_pages"] * inp["page_size"]
    rows_t = gpu_cache_rows(inp, tabs, S, mc)
    if bad_page:
        rows_t[:, 3] = -2             # a table entry outside the cache
    res = {}
    for mode in ("paged",) if bad_page else ("buffer", "paged"):
        out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
        oacc = torch.empty(T, H, 128, dtype=torch.float32, device=DEV)
        lacc = torch.empty(T, H, dtype=torch.float32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        for ch in range(mc):
            kn, vv, _ = (t.to(DEV) for t in make_attention_operands(w, S, seed_offset=seed_base + ch))
            if mode == "buffer":
                ckv = torch.zeros(S, 512, dtype=kv.dtype, device=DEV)
                kr = torch.zeros(S, 64, dtype=kv.dtype, device=DEV)
                mla.check(mla.mla_gather_latent(ckv, kr, kv, pt, *paging, *tabs, ch, B, S, _dt(w), st))
                mla.check(mla.mla_prefill_attention(out, lse, oacc, lacc, q, kn, vv, kr, iro, cl, *tabs,
                                                    ch, mc, B, H, inp["max_prompt_len"], T, S,
                                                    inp["scale"], dtype=_dt(w), d_status=st))
            else:
                mla.check(mla.mla_prefill_attention_paged(out, lse, oacc, lacc, q, kn, vv, kv, rows_t[ch],
                                                          ncr, iro, cl, *tabs, ch, mc, B, H,
                                                          inp["max_prompt_len"], T, S, inp["scale"],
                                                          dtype=_dt(w), d_status=st))
        torch.cuda.synchronize()
        res[mode] = (out, lse, int(st.item()))
    if bad_page:
        assert res["paged"][2] == mla.MLA_DEV_BAD_PAGE
        return None
    assert res["buffer"][2] == 0 and res["paged"][2] == 0
    assert torch.equal(res["buffer"][0].view(torch.int16), res["paged"][0].view(torch.int16))
    assert torch.equal(res["buffer"][1], res["paged"][1])
    if not oracle:
        return None

    def operands(ch):
        kn, vv, _ = make_attention_operands(w, S, seed_offset=seed_base + ch)
        _, kr, ost = O.gather_latent(c["kv_cache"], c["page_table"], inp["page_size"], plan, ch)
        assert ost == 0
        v64 = vv.double().numpy() if dt == "e4m3" else O.decode(O.codes(vv), dt)
        return (O.decode(O.codes(kn), dt), O.decode(kr, dt), v64)
    ref = O.attention_over_chunks(O.decode(c["q"], dt), operands, plan, c["input_row_offsets"],
                                  c["cache_lengths"], inp["scale"])
    return _compare(res["paged"][0], ref, dt, res["paged"][1])


def test_paged_attention_shuffled_pages_multi_chunk(bf16_kernel):
    """Shuffled 16-row pages (a 64-key half tile spans four pages), ragged
    sequences, several chunks."""
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=2, B=3, buffer_token_size=700, max_chunks=4,
               new_range=(100, 600), cache_range=(0, 900), page_size=16)
    _paged_attention_case(w)


def test_paged_attention_one_row_pages(bf16_kernel):
    """page_size 1: every key on a page of its own."""
    w = scaled(WORKLOADS["tiny_ragged"], page_size=1, shuffle_pages=True)
    _paged_attention_case(w)


def test_paged_attention_e4m3():
    w = scaled(WORKLOADS["longctx_fp8"], H=2, B=2, new_lens=(300, 41), cache_lens=(200, 0),
               buffer_token_size=192, max_chunks=3, page_size=64, shuffle_pages=True)
    _paged_attention_case(w)


@pytest.mark.parametrize("name", ["ragged_chunked_cache", "longctx_fp8"])
def test_paged_attention_full_size_equals_buffered(name):
    """The full-size workloads (seeded shuffled pages, every chunk): the paged
    call equals the buffered call bit for bit; the buffered call's own
    parity with the oracle at these sizes is covered by the fused tests."""
    _paged_attention_case(WORKLOADS[name], oracle=False)


def test_paged_attention_bad_page_reports_status():
    w = scaled(WORKLOADS["tiny_ragged"], page_size=16)
    _paged_attention_case(w, bad_page=True)


def test_attention_stage_e4m3_multi_chunk():
    w = scaled(WORKLOADS["longctx_fp8"], H=2, B=2, new_lens=(300, 41), cache_lens=(200, 0),
               buffer_token_size=192, max_chunks=3, page_size=64)
    _attention_stage(w)


def test_attention_stage_e4m3_tiles():
    w = scaled(WORKLOADS["longctx_fp8"], H=3, new_lens=(700,), cache_lens=(333,),
               buffer_token_size=1033, max_chunks=1, page_size=64)
    _attention_stage(w)


def run_fused(inp, S=None, max_chunks=None, lse=True):
    w = inp["workload"]
    S = S or w.buffer_token_size
    mc = max_chunks or w.max_chunks
    B, H, T = inp["B"], w.H, inp["T_q"]
    dt = _dt(w)
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse_t = torch.empty(T, H, dtype=torch.float32, device=DEV) if lse else None
    nbytes = mla.mla_prefill_workspace_bytes(B, H, T, mc, S, dt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    st = torch.full((1,), 99, dtype=torch.int32, device=DEV)
    mla.check(mla.mla_prefill(out, lse_t, inp["q"].to(DEV), inp["input_row_offsets"].to(DEV),
                              inp["cache_lengths"].to(DEV), inp["kv_cache"].to(DEV),
                              inp["page_table"].to(DEV), inp["num_pages"], inp["page_size"],
                              inp["max_pages"], inp["w_k"].to(DEV), inp["w_uv"].to(DEV), B, H, T,
                              inp["max_prompt_len"], S, mc, inp["scale"], inp["q_scale"],
                              inp["ckv_scale"], inp["w_scale"], dt, ws, nbytes, st))
    torch.cuda.synchronize()
    assert st.item() == 0, mla.status_string(int(st.item()))
    return out, lse_t


@pytest.mark.parametrize("name,heads", [("tiny_ragged", 4), ("ragged_chunked_cache", 4)])
def test_fused_call_replays_in_a_cuda_graph(name, heads, bf16_kernel):
    """The fused call (the plan, then per chunk the gather, projection and
    attention, every kernel a programmatic dependent launch) captured in a CUDA
    graph: two replays give the eager call's output and LSE bit for bit."""
    w = scaled(WORKLOADS[name], H=heads)
    inp = make_inputs(w)
    ref_out, ref_lse = run_fused(inp)
    S, mc, B, H, T = w.buffer_token_size, w.max_chunks, inp["B"], w.H, inp["T_q"]
    dt = _dt(w)
    dev_in = {k: inp[k].to(DEV) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache",
                                           "page_table", "w_k", "w_uv")}
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, H, dtype=torch.float32, device=DEV)
    nbytes = mla.mla_prefill_workspace_bytes(B, H, T, mc, S, dt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)

    def call():
        mla.check(mla.mla_prefill(out, lse, dev_in["q"], dev_in["input_row_offsets"],
                                  dev_in["cache_lengths"], dev_in["kv_cache"], dev_in["page_table"],
                                  inp["num_pages"], inp["page_size"], inp["max_pages"], dev_in["w_k"],
                                  dev_in["w_uv"], B, H, T, inp["max_prompt_len"], S, mc, inp["scale"],
                                  inp["q_scale"], inp["ckv_scale"], inp["w_scale"], dt, ws, nbytes, st))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()   # warm-up outside the capture (first-use set-up of the kernels)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert st.item() == 0, mla.status_string(int(st.item()))
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)


def oracle_fused(inp, S=None, max_chunks=None, heads=None, rows=None):
    w = inp["workload"]
    c = {k: O.codes(inp[k]) for k in ("q", "kv_cache", "page_table", "w_k", "w_uv",
                                      "input_row_offsets", "cache_lengths")}
    ref, _ = O.mla_prefill(c["q"], c["kv_cache"], c["page_table"], inp["page_size"], c["w_k"],
                           c["w_uv"], c["input_row_offsets"], c["cache_lengths"],
                           S or w.buffer_token_size, max_chunks or w.max_chunks, inp["scale"],
                           dtype=w.dtype, q_scale=inp["q_scale"], ckv_scale=inp["ckv_scale"],
                           w_scale=inp["w_scale"], heads=heads, rows=rows)
    return ref


def _sample_rows(new_lens, cache_lens, S, k, seed):
    """First, last, tile-edge and chunk-edge rows plus random ones, per sequence."""
    rng = np.random.default_rng(seed)
    out = []
    start = 0
    for n, cb in zip(new_lens, cache_lens):
        n, cb = int(n), int(cb)
        cand = {0, n - 1, min(127, n - 1), min(128, n - 1), n // 2}
        # rows whose position sits on a chunk boundary of the packed order
        for edge in range((start // S + 1) * S, start + cb + n, S):
            i = edge - start - cb
            for d in (-1, 0, 1):
                if 0 <= i + d < n:
                    cand.add(i + d)
        cand |= set(rng.integers(0, n, size=k).tolist()) if n > 0 else set()
        out.append(np.array(sorted(x for x in cand if 0 <= x < n), dtype=np.int64))
        start += cb + n
    return out


def test_fused_tiny_ragged_all_rows(bf16_kernel):
    inp = make_inputs(WORKLOADS["tiny_ragged"])
    out, lse = run_fused(inp)
    _compare(out, oracle_fused(inp), "bf16", lse)


@pytest.mark.parametrize("H", [1, 2])
def test_fused_one_and_two_heads(H, bf16_kernel):
    """One or two heads: a projection tile of 256 columns holds a single
    head's K (and a V tile the same head's V), and a head group is the whole
    head count; every row of the multi-chunk tiny workload is checked."""
    inp = make_inputs(scaled(WORKLOADS["tiny_ragged"], H=H))
    out, lse = run_fused(inp)
    _compare(out, oracle_fused(inp), "bf16", lse)


@pytest.mark.parametrize("S", [7, 64, 200])
def test_fused_buffer_size_invariance(S, bf16_kernel):
    """Different buffer sizes cut the context differently; the result is the same."""
    w = WORKLOADS["tiny_ragged"]
    inp = make_inputs(w)
    mc = -(-89 // S)
    out, lse = run_fused(inp, S=S, max_chunks=mc)
    _compare(out, oracle_fused(inp, S=S, max_chunks=mc), "bf16", lse)
    out_ref, _ = run_fused(inp)
    assert (out.float() - out_ref.float()).abs().max().item() <= 2e-2


def test_fused_v2lite_shape_small_heads(bf16_kernel):
    inp = make_inputs(scaled(WORKLOADS["v2lite_prefill"], H=2))
    out, lse = run_fused(inp)
    rows = _sample_rows(inp["new_lens"], inp["cache_lens"], 4096, 40, 1)
    _compare(out, oracle_fused(inp, rows=rows), "bf16", lse)


def test_fused_v3_full_length_small_heads(bf16_kernel):
    inp = make_inputs(scaled(WORKLOADS["v3_prefill"], H=2))
    out, lse = run_fused(inp)
    rows = _sample_rows(inp["new_lens"], inp["cache_lens"], 4096, 60, 2)
    _compare(out, oracle_fused(inp, rows=rows), "bf16", lse)


def test_fused_ragged_chunked_small_heads(bf16_kernel):
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=2)
    inp = make_inputs(w)
    out, lse = run_fused(inp)
    rows = _sample_rows(inp["new_lens"], inp["cache_lens"], w.buffer_token_size, 24, 3)
    _compare(out, oracle_fused(inp, rows=rows), "bf16", lse)


def test_fused_edge_cases(bf16_kernel):
    # an empty sequence, a cache-only sequence, a single token, a tile-edge length,
    # a buffer smaller than one sequence
    w = scaled(WORKLOADS["tiny_ragged"], H=3, page_size=8, buffer_token_size=50, max_chunks=12)
    new, cache = (0, 1, 129, 0, 5), (0, 0, 17, 30, 70)
    inp = make_inputs(w, new_lens=new, cache_lens=cache)
    mc = -(-sum(a + b for a, b in zip(new, cache)) // 50)
    out, lse = run_fused(inp, max_chunks=mc)
    _compare(out, oracle_fused(inp, max_chunks=mc), "bf16", lse)


def test_fused_pair_boundaries(bf16_kernel):
    """Query-tile pairs with an odd tile count (the second tile of the last pair
    is empty), one-tile sequences, and chunk cuts that leave one tile of a
    pair with no visible keys of a chunk while its partner has some."""
    w = scaled(WORKLOADS["tiny_ragged"], H=3, page_size=16, buffer_token_size=384, max_chunks=8)
    new, cache = (300, 129, 1, 257, 640), (0, 500, 37, 130, 90)
    inp = make_inputs(w, new_lens=new, cache_lens=cache)
    mc = -(-sum(a + b for a, b in zip(new, cache)) // 384)
    out, lse = run_fused(inp, max_chunks=mc)
    _compare(out, oracle_fused(inp, max_chunks=mc), "bf16", lse)


def test_fused_sequence_alone_equals_in_batch(bf16_kernel):
    w = scaled(WORKLOADS["ragged_chunked_cache"], H=2, B=3, buffer_token_size=256,
               new_range=(100, 300), cache_range=(0, 400))
    inp = make_inputs(w)
    mc = -(-int((inp["new_lens"] + inp["cache_lens"]).sum()) // 256)
    out, _ = run_fused(inp, max_chunks=mc)
    b = 1
    alone = make_inputs(scaled(w, B=1), new_lens=[inp["new_lens"][b]], cache_lens=[inp["cache_lens"][b]])
    # same sequence content: copy its q rows, pages and weights
    iro = inp["input_row_offsets"].numpy()
    alone["q"] = inp["q"][iro[b]:iro[b + 1]].clone()
    pages = inp["page_table"][b]
    pages = pages[pages >= 0]
    alone["kv_cache"] = inp["kv_cache"][pages.long()].clone()
    alone["page_table"] = torch.arange(len(pages), dtype=torch.int32)[None, :]
    alone["num_pages"], alone["max_pages"] = len(pages), len(pages)
    alone["w_k"], alone["w_uv"] = inp["w_k"], inp["w_uv"]
    mc1 = -(-int(inp["new_lens"][b] + inp["cache_lens"][b]) // 256)
    out1, _ = run_fused(alone, max_chunks=mc1)
    d = (out[iro[b]:iro[b + 1]].float() - out1.float()).abs().max().item()
    assert d <= 2e-2


def test_fused_e4m3_full_length_small_heads():
    w = scaled(WORKLOADS["longctx_fp8"], H=2)
    inp = make_inputs(w)
    out, lse = run_fused(inp)
    rows = _sample_rows(inp["new_lens"], inp["cache_lens"], w.buffer_token_size, 40, 5)
    _compare(out, oracle_fused(inp, rows=rows), "e4m3", lse)


@pytest.mark.parametrize("name", ["v2lite_prefill", "v3_prefill", "ragged_chunked_cache",
                                  "longctx_fp8"])
def test_fused_full_size_sampled(name, bf16_kernel):
    """Full sizes, the launch configuration the benchmark times; the oracle
    checks a sample of heads and rows."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    out, lse = run_fused(inp)
    heads = [0, w.H // 2 + 1, w.H - 1]
    rows = _sample_rows(inp["new_lens"], inp["cache_lens"], w.buffer_token_size, 12, 4)
    _compare(out, oracle_fused(inp, heads=heads, rows=rows), w.dtype, lse)
    assert torch.isfinite(out.float()).all()


def test_fused_is_deterministic(bf16_kernel):
    """No atomics in the arithmetic: repeated calls agree bit for bit (a
    pipeline race shows up here first)."""
    inp = make_inputs(scaled(WORKLOADS["ragged_chunked_cache"], H=2, B=4, buffer_token_size=2048,
                             new_range=(100, 900), cache_range=(0, 1500)))
    mc = -(-int((inp["new_lens"] + inp["cache_lens"]).sum()) // 2048)
    outs = [run_fused(inp, max_chunks=mc) for _ in range(4)]
    for o, l in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(l, outs[0][1])
