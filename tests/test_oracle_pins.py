"""Pins for the CPU oracle: each oracle function is checked against something
other than itself -- hand-worked tables, brute force written independently,
closed forms, invariants and library routines.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from oracle import mla_oracle as M
from workloads import WORKLOADS, make_cache_write_operands, make_inputs, scaled


# ----------------------------------------------------------------------------
# Latent-cache write: RMSNorm, RoPE rotation, the paged store
# ----------------------------------------------------------------------------

def test_rms_norm_closed_forms_and_library():
    rng = np.random.default_rng(3)
    g = 1.0 + 0.1 * rng.standard_normal(512)
    # A constant row normalises to the weights times its sign (eps = 0).
    np.testing.assert_allclose(O.rms_norm(np.full(512, -2.5), g, 0.0), -g, rtol=1e-15)
    # A one-hot row a*e_j has mean square a**2/512.
    x = np.zeros(512)
    x[17] = 3.0
    out = O.rms_norm(x, g, 1e-3)
    assert out[17] == pytest.approx(g[17] * 3.0 / math.sqrt(9.0 / 512 + 1e-3), rel=1e-14)
    assert np.count_nonzero(out) == 1
    # Scale invariance and a unit mean square of out / g (eps = 0).
    x = rng.standard_normal((4, 512))
    np.testing.assert_allclose(O.rms_norm(7.0 * x, g, 0.0), O.rms_norm(x, g, 0.0), rtol=1e-13)
    np.testing.assert_allclose(np.mean((O.rms_norm(x, g, 0.0) / g) ** 2, axis=-1), 1.0, rtol=1e-13)
    # The library routine (torch, float64), with epsilon.
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (512,), torch.from_numpy(g), eps=1e-5)
    np.testing.assert_allclose(O.rms_norm(x, g, 1e-5), ref.numpy(), rtol=1e-13)


def _freqs_from_angles(ang):
    f = np.empty(ang.shape[:-1] + (2 * ang.shape[-1],))
    f[..., 0::2] = np.cos(ang)
    f[..., 1::2] = np.sin(ang)
    return f


def test_rope_rotation_special_cases():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64))
    # Angle 0 is the identity; a quarter turn maps each pair (a, b) to (-b, a).
    np.testing.assert_array_equal(O.rope_rotate(x, np.tile([1.0, 0.0], 32)), x)
    quarter = O.rope_rotate(x, np.tile([0.0, 1.0], 32))
    np.testing.assert_array_equal(quarter[:, 0::2], -x[:, 1::2])
    np.testing.assert_array_equal(quarter[:, 1::2], x[:, 0::2])
    # Unit-modulus factors keep every pair's length; theta then -theta, and
    # theta1 then theta2 against theta1 + theta2.
    a1, a2 = rng.uniform(-7, 7, 32), rng.uniform(-7, 7, 32)
    y = O.rope_rotate(x, _freqs_from_angles(a1))
    np.testing.assert_allclose(np.hypot(y[:, 0::2], y[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]), rtol=1e-13)
    np.testing.assert_allclose(O.rope_rotate(y, _freqs_from_angles(-a1)), x, atol=1e-13)
    np.testing.assert_allclose(O.rope_rotate(y, _freqs_from_angles(a2)),
                               O.rope_rotate(x, _freqs_from_angles(a1 + a2)), atol=1e-12)
    # The library's complex product over the same interleaved layout.
    f = rng.standard_normal(64)
    z = torch.view_as_complex(torch.from_numpy(x).reshape(3, 32, 2).contiguous())
    w = torch.view_as_complex(torch.from_numpy(f).reshape(32, 2).contiguous())
    ref = torch.view_as_real(z * w).reshape(3, 64).numpy()
    np.testing.assert_allclose(O.rope_rotate(x, f), ref, rtol=1e-14, atol=1e-15)


def _cache_write_case(w, dtype="bf16", inv_scale=1.0, shuffle=False):
    inp = make_inputs(scaled(w, dtype="bf16", shuffle_pages=shuffle))
    T = inp["T_q"]
    L = inp["new_lens"] + inp["cache_lens"]
    lat, gamma, freqs = make_cache_write_operands(w, T, int(L.max()) + 1)
    cache = O.codes(inp["kv_cache"])
    if dtype == "e4m3":
        cache = M.e4m3_encode(M.bf16_decode(cache))
    return inp, O.decode(O.codes(lat), "bf16"), gamma.numpy().astype(np.float64), freqs.numpy(), cache


def test_cache_write_round_trip_through_cache():
    """Each sequence's context read back from the paged cache (an oracle
    function of its own): cached tokens untouched, new tokens normalised and
    rotated at their positions; q's nope parts untouched."""
    w = scaled(WORKLOADS["tiny_ragged"], H=3, page_size=8)
    inp, lat, gamma, freqs, cache = _cache_write_case(w, shuffle=True)
    q = O.decode(O.codes(inp["q"]), "bf16")
    iro, cl = inp["input_row_offsets"].numpy(), inp["cache_lengths"].numpy()
    kv, q2, st = O.latent_cache_write(lat, q, gamma, freqs, iro, cl, inp["page_table"].numpy(),
                                      inp["page_size"], cache, 1e-6)
    assert st == 0
    L = inp["new_lens"] + inp["cache_lens"]
    before = O.context_latents(cache, inp["page_table"].numpy(), inp["page_size"], L)
    after = O.context_latents(kv, inp["page_table"].numpy(), inp["page_size"], L)
    for b in range(inp["B"]):
        c = int(cl[b])
        np.testing.assert_array_equal(after[b][:c], before[b][:c])
        rows = lat[iro[b]:iro[b + 1]]
        want = np.concatenate([O.rms_norm(rows[:, :512], gamma, 1e-6),
                               O.rope_rotate(rows[:, 512:], freqs[c:c + len(rows)])], axis=1)
        np.testing.assert_array_equal(after[b][c:], M.bf16_encode(want))
        np.testing.assert_array_equal(q2[iro[b]:iro[b + 1], :, :128], q[iro[b]:iro[b + 1], :, :128])
        for i in range(len(rows)):
            np.testing.assert_allclose(q2[iro[b] + i, :, 128:], O.rope_rotate(q[iro[b] + i, :, 128:], freqs[c + i]),
                                       rtol=0, atol=0)
    # Pages no sequence uses hold exactly what they held.
    used = set(inp["page_table"].numpy().ravel().tolist()) - {-1}
    for pg in range(cache.shape[0]):
        if pg not in used:
            np.testing.assert_array_equal(kv[pg], cache[pg])


def test_cache_write_page_permutation_and_e4m3():
    """Relabelling the physical pages relabels the written cache; the e4m3
    store is the e4m3 rounding of the row times the inverse scale."""
    w = scaled(WORKLOADS["tiny_ragged"], H=2, page_size=8)
    inp, lat, gamma, freqs, cache = _cache_write_case(w)
    iro, cl, pt = inp["input_row_offsets"].numpy(), inp["cache_lengths"].numpy(), inp["page_table"].numpy()
    kv, _, st = O.latent_cache_write(lat, None, gamma, freqs, iro, cl, pt, 8, cache, 1e-6)
    perm = np.random.default_rng(9).permutation(cache.shape[0])
    inv = np.argsort(perm)                 # new page id of old page j is inv[j]
    pt2 = np.where(pt >= 0, inv[np.maximum(pt, 0)], -1)
    kv2, _, st2 = O.latent_cache_write(lat, None, gamma, freqs, iro, cl, pt2, 8, cache[perm], 1e-6)
    assert st == st2 == 0
    np.testing.assert_array_equal(kv2, kv[perm])
    _, _, _, _, cache8 = _cache_write_case(w, dtype="e4m3")
    kv8, _, st8 = O.latent_cache_write(lat, None, gamma, freqs, iro, cl, pt, 8, cache8, 1e-6,
                                       dtype="e4m3", inv_scale=0.5)
    assert st8 == 0
    L = inp["new_lens"] + inp["cache_lens"]
    got = O.context_latents(kv8, pt, 8, L)
    for b in range(inp["B"]):
        c = int(cl[b])
        rows = lat[iro[b]:iro[b + 1]]
        want = np.concatenate([O.rms_norm(rows[:, :512], gamma, 1e-6),
                               O.rope_rotate(rows[:, 512:], freqs[c:c + len(rows)])], axis=1)
        np.testing.assert_array_equal(M.e4m3_decode(got[b][c:]), M.round_to_e4m3(0.5 * want))


def test_cache_write_status():
    w = scaled(WORKLOADS["tiny_ragged"], H=1, page_size=8)
    inp, lat, gamma, freqs, cache = _cache_write_case(w)
    iro, cl, pt = inp["input_row_offsets"].numpy(), inp["cache_lengths"].numpy(), inp["page_table"].numpy()
    # A position past the frequency table.
    _, _, st = O.latent_cache_write(lat, None, gamma, freqs[:10], iro, cl, pt, 8, cache, 1e-6)
    assert st == M.STATUS_BAD_OFFSETS
    # A missing page where new tokens go (sequence 1 writes positions 40..72).
    pt2 = pt.copy()
    pt2[1, 6] = -1
    _, _, st = O.latent_cache_write(lat, None, gamma, freqs, iro, cl, pt2, 8, cache, 1e-6)
    assert st == M.STATUS_BAD_PAGE


# ----------------------------------------------------------------------------
# Plan
# ----------------------------------------------------------------------------

def _read_plan_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.split() for p in line.split("|")]
            rows.append(([int(x) for x in parts[1]], [int(x) for x in parts[2]], int(parts[3][0])))
    return rows


def test_plan_hand_worked_tiny_ragged(golden_dir):
    rows = _read_plan_golden(os.path.join(golden_dir, "plan_tiny_ragged.txt"))
    bro, co, bl, st = O.prefill_plan([0, 16, 49], [0, 40], 32, 4)
    assert st == 0
    for c, (b, k, n) in enumerate(rows):
        assert list(bro[c]) == b
        assert list(co[c]) == k
        assert bl[c] == n


def _token_walk(new, cache, S, max_chunks):
    """Independent plan: walk every context token in packed order and drop it
    into the current chunk, opening a new chunk when S rows are used."""
    B = len(new)
    L = [int(a) + int(b) for a, b in zip(new, cache)]
    chunks = []           # per chunk: list over b of [first_pos or None, count]
    cur = None
    used = S
    for b in range(B):
        for pos in range(L[b]):
            if used == S:
                cur = [[None, 0] for _ in range(B)]
                chunks.append(cur)
                used = 0
            if cur[b][0] is None:
                cur[b][0] = pos
            cur[b][1] += 1
            used += 1
    bro = np.zeros((max_chunks, B + 1), np.int64)
    co = np.zeros((max_chunks, B), np.int64)
    bl = np.full(max_chunks, -1, np.int64)
    # position of each seq's progress at the start of each chunk
    done = [0] * B
    for c in range(max_chunks):
        row = 0
        for b in range(B):
            bro[c, b] = row
            if c < len(chunks) and chunks[c][b][1] > 0:
                co[c, b] = chunks[c][b][0]
                row += chunks[c][b][1]
            else:
                co[c, b] = done[b]
        bro[c, B] = row
        if c < len(chunks):
            bl[c] = row
            for b in range(B):
                done[b] += chunks[c][b][1]
    return bro, co, bl, len(chunks)


def test_plan_matches_token_walk_random():
    """10^4 random tiny cases (B <= 6, lengths <= 40, S in [1, 50])."""
    rng = np.random.default_rng(1234)
    for _ in range(10000):
        B = int(rng.integers(0, 7))
        new = rng.integers(0, 41, size=B)
        cache = rng.integers(0, 41, size=B)
        S = int(rng.integers(1, 51))
        iro = np.concatenate([[0], np.cumsum(new)])
        need = -(-int((new + cache).sum()) // S)
        max_chunks = need + int(rng.integers(0, 3))
        bro, co, bl, st = O.prefill_plan(iro, cache, S, max_chunks)
        wbro, wco, wbl, nc = _token_walk(new, cache, S, max_chunks)
        assert st == 0 and nc == need
        np.testing.assert_array_equal(bro, wbro)
        np.testing.assert_array_equal(co, wco)
        np.testing.assert_array_equal(bl, wbl)


def test_plan_invariants_ragged_chunked_cache():
    w = WORKLOADS["ragged_chunked_cache"]
    from workloads import lengths
    new, cache = lengths(w)
    iro = np.concatenate([[0], np.cumsum(new)])
    bro, co, bl, st = O.prefill_plan(iro, cache, w.buffer_token_size, w.max_chunks)
    assert st == 0
    L = new + cache
    n = bro[:, 1:] - bro[:, :-1]
    np.testing.assert_array_equal(n.sum(axis=0), L)           # every token exactly once
    used = bl >= 0
    assert used.sum() == -(-L.sum() // w.buffer_token_size)
    assert np.all(bl[used][:-1] == w.buffer_token_size)       # all chunks but the last are full
    assert np.all(bro[:, -1][used] == bl[used])
    for b in range(w.B):                                       # contiguous in position
        for c in range(w.max_chunks - 1):
            if n[c, b] > 0 and co[c, b] + n[c, b] < L[b]:
                assert co[c + 1, b] == co[c, b] + n[c, b]


def test_plan_edge_cases():
    # nothing to do: every chunk unused
    bro, co, bl, st = O.prefill_plan([0, 0, 0], [0, 0], 8, 3)
    assert st == 0 and list(bl) == [-1, -1, -1] and not bro.any() and not co.any()
    # empty batch
    bro, co, bl, st = O.prefill_plan([0], [], 8, 2)
    assert st == 0 and bro.shape == (2, 1) and list(bl) == [-1, -1]
    # one token per chunk
    bro, co, bl, st = O.prefill_plan([0, 2], [1], 1, 3)
    assert list(bl) == [1, 1, 1] and list(co[:, 0]) == [0, 1, 2]
    # too few chunk rows: status 1, the rows that exist still written
    bro, co, bl, st = O.prefill_plan([0, 10], [0], 4, 2)
    assert st == M.STATUS_TOO_MANY_CHUNKS and list(bl) == [4, 4]
    # malformed offsets: status 2
    assert O.prefill_plan([1, 3], [0], 4, 2)[3] == M.STATUS_BAD_OFFSETS
    assert O.prefill_plan([0, 5, 3], [0, 0], 4, 4)[3] == M.STATUS_BAD_OFFSETS
    with pytest.raises(ValueError):
        O.prefill_plan([0, 1], [0], 0, 1)


# ----------------------------------------------------------------------------
# Gather
# ----------------------------------------------------------------------------

def _coded_cache(new, cache, ps, shuffle_seed=None):
    """A cache whose every element encodes (sequence, position, column), so
    the expected gather output follows from the token walk alone."""
    L = [int(a) + int(b) for a, b in zip(new, cache)]
    pages = [(x + ps - 1) // ps for x in L]
    num_pages = max(1, sum(pages))
    perm = np.arange(num_pages)
    if shuffle_seed is not None:
        perm = np.random.default_rng(shuffle_seed).permutation(num_pages)
    pt = np.full((len(L), max(1, max(pages, default=1))), -1, np.int64)
    kv = np.zeros((num_pages, ps, M.DC), np.int64)
    k = 0
    for b, Lb in enumerate(L):
        for p in range(pages[b]):
            pt[b, p] = perm[k]
            for s in range(ps):
                pos = p * ps + s
                kv[perm[k], s] = (b * 1000 + pos) * 1000 + np.arange(M.DC)
            k += 1
    return kv, pt


def test_gather_by_construction():
    rng = np.random.default_rng(7)
    for trial in range(30):
        B = int(rng.integers(1, 5))
        new = rng.integers(0, 30, size=B)
        cache = rng.integers(0, 30, size=B)
        ps = int(rng.integers(1, 9))
        S = int(rng.integers(1, 40))
        iro = np.concatenate([[0], np.cumsum(new)])
        nc = max(1, -(-int((new + cache).sum()) // S))
        kv, pt = _coded_cache(new, cache, ps, shuffle_seed=trial)
        plan = O.prefill_plan(iro, cache, S, nc)
        wbro, wco, wbl, _ = _token_walk(new, cache, S, nc)
        for c in range(nc):
            ckv, kr, st = O.gather_latent(kv, pt, ps, plan, c)
            assert st == 0
            for b in range(B):
                for t in range(wbro[c, b + 1] - wbro[c, b]):
                    pos = wco[c, b] + t
                    expect = (b * 1000 + pos) * 1000 + np.arange(M.DC)
                    np.testing.assert_array_equal(ckv[wbro[c, b] + t], expect[:M.R])
                    np.testing.assert_array_equal(kr[wbro[c, b] + t], expect[M.R:])


def test_gather_page_permutation_invariant():
    new, cache, ps, S = [20, 7, 33], [5, 40, 0], 4, 24
    iro = np.concatenate([[0], np.cumsum(new)])
    plan = O.prefill_plan(iro, cache, S, 5)
    kv0, pt0 = _coded_cache(new, cache, ps, None)
    kv1, pt1 = _coded_cache(new, cache, ps, 99)
    assert not np.array_equal(pt0, pt1)
    for c in range(5):
        a = O.gather_latent(kv0, pt0, ps, plan, c)
        b = O.gather_latent(kv1, pt1, ps, plan, c)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_gather_bad_page_status():
    kv, pt = _coded_cache([4], [4], 4)
    plan = O.prefill_plan([0, 4], [4], 8, 1)
    pt = pt.copy()
    pt[0, 1] = kv.shape[0]          # out of range
    assert O.gather_latent(kv, pt, 4, plan, 0)[2] == M.STATUS_BAD_PAGE


def test_chunk_cache_rows_by_construction():
    """Every element of the coded cache names its (sequence, position), so the
    row a table entry points at must carry the code of the buffer row's own
    token, taken from the token walk; entries past the chunk are 0."""
    rng = np.random.default_rng(11)
    for trial in range(30):
        B = int(rng.integers(1, 5))
        new = rng.integers(0, 30, size=B)
        cache = rng.integers(0, 30, size=B)
        ps = int(rng.integers(1, 9))
        S = int(rng.integers(1, 40))
        iro = np.concatenate([[0], np.cumsum(new)])
        nc = max(1, -(-int((new + cache).sum()) // S))
        kv, pt = _coded_cache(new, cache, ps, shuffle_seed=100 + trial)
        flat = kv.reshape(-1, M.DC)
        plan = O.prefill_plan(iro, cache, S, nc)
        wbro, wco, wbl, _ = _token_walk(new, cache, S, nc)
        for c in range(nc):
            rows, st = O.chunk_cache_rows(pt, ps, kv.shape[0], plan, c, S)
            assert st == 0 and rows.shape == (S,)
            n = max(int(wbl[c]), 0)
            assert np.all(rows[n:] == 0)
            for b in range(B):
                for t in range(wbro[c, b + 1] - wbro[c, b]):
                    expect = (b * 1000 + wco[c, b] + t) * 1000
                    assert flat[rows[wbro[c, b] + t], 0] == expect


def test_chunk_cache_rows_identity_pages():
    """One sequence on pages 0, 1, 2, ... in order: buffer row r of chunk c is
    cache row c * S + r (the context positions themselves)."""
    new, cache, ps, S = [37], [20], 8, 16
    kv, pt = _coded_cache(new, cache, ps, None)
    plan = O.prefill_plan([0, 37], cache, S, 4)
    for c in range(4):
        rows, st = O.chunk_cache_rows(pt, ps, kv.shape[0], plan, c, S)
        n = min(S, 57 - c * S)
        np.testing.assert_array_equal(rows[:n], c * S + np.arange(n))


def test_chunk_cache_rows_bad_page_status():
    kv, pt = _coded_cache([4], [4], 4)
    plan = O.prefill_plan([0, 4], [4], 8, 1)
    pt = pt.copy()
    pt[0, 1] = kv.shape[0]          # out of range
    rows, st = O.chunk_cache_rows(pt, 4, kv.shape[0], plan, 0, 8)
    assert st == M.STATUS_BAD_PAGE
    assert np.all(rows[4:] == 0) and np.array_equal(rows[:4], pt[0, 0] * 4 + np.arange(4))


# ----------------------------------------------------------------------------
# Up-projection
# ----------------------------------------------------------------------------

def test_upproject_bruteforce():
    rng = np.random.default_rng(3)
    rows, H = 3, 2
    c = rng.standard_normal((rows, M.R))
    wk = rng.standard_normal((H * M.DN, M.R))
    wuv = rng.standard_normal((H, M.DV, M.R))
    k, v = O.upproject(c, wk, wuv)
    for r in range(rows):
        for h in range(H):
            for d in (0, 5, 127):
                ek = sum(c[r, i] * wk[h * M.DN + d, i] for i in range(M.R))
                ev = sum(c[r, i] * wuv[h, d, i] for i in range(M.R))
                assert abs(k[r, h, d] - ek) < 1e-9 and abs(v[r, h, d] - ev) < 1e-9


def test_upproject_identity_and_heads_subset():
    rng = np.random.default_rng(4)
    c = rng.standard_normal((17, M.R))
    wk = rng.standard_normal((4 * M.DN, M.R))
    wuv = rng.standard_normal((4, M.DV, M.R))
    k, v = O.upproject(c, wk, wuv)
    x = rng.standard_normal(M.DN)
    for h in range(4):
        lhs = k[:, h] @ x
        rhs = c @ (wk[h * M.DN:(h + 1) * M.DN].T @ x)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-9)
    k2, v2 = O.upproject(c, wk, wuv, heads=[3, 1])
    np.testing.assert_array_equal(k2[:, 0], k[:, 3])
    np.testing.assert_array_equal(v2[:, 1], v[:, 1])


def test_upproject_store_rounding():
    rng = np.random.default_rng(5)
    c = rng.standard_normal((8, M.R))
    wk = rng.standard_normal((M.DN, M.R)) / math.sqrt(M.R)
    wuv = rng.standard_normal((1, M.DV, M.R)) / math.sqrt(M.R)
    k, v = O.upproject(c, wk, wuv)
    kb, vb = O.upproject(c, wk, wuv, store="bf16")
    kt = torch.tensor(k.astype(np.float32)).to(torch.bfloat16).double().numpy()
    # float64 -> bf16 equals float32 -> bf16 except where the float32 rounding
    # lands exactly on a bf16 tie; allow at most a handful of those
    assert (kb != kt).sum() <= 2
    assert np.all(np.abs(vb - v) <= np.abs(v) * 2.0 ** -8 + 1e-30)


# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------

def test_bf16_codec_against_torch():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16)
    np.testing.assert_array_equal(M.bf16_encode(x.astype(np.float64)),
                                  ref.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(M.bf16_decode(M.bf16_encode(x.astype(np.float64))),
                                  ref.double().numpy())


def test_e4m3_spec_values():
    # OCP FP8 E4M3 table values
    assert M.e4m3_encode(np.array([1.0]))[0] == 0x38
    assert M.e4m3_encode(np.array([448.0]))[0] == 0x7E
    assert M.e4m3_encode(np.array([1e6]))[0] == 0x7E          # saturate
    assert M.e4m3_encode(np.array([-448.0]))[0] == 0xFE
    assert M.e4m3_encode(np.array([2.0 ** -9]))[0] == 0x01    # smallest subnormal
    assert M.e4m3_encode(np.array([2.0 ** -6]))[0] == 0x08    # smallest normal
    assert M.e4m3_encode(np.array([1.0625]))[0] == 0x38       # tie -> even mantissa
    assert M.e4m3_encode(np.array([1.1875]))[0] == 0x3A       # tie -> even mantissa (up)
    assert M.e4m3_decode(np.array([0x7F]))[0] != M.e4m3_decode(np.array([0x7F]))[0]  # NaN
    allc = np.arange(256, dtype=np.uint8)
    finite = ~np.isnan(M.e4m3_decode(allc))
    np.testing.assert_array_equal(M.e4m3_encode(M.e4m3_decode(allc[finite]))[allc[finite] != 0x80],
                                  allc[finite][allc[finite] != 0x80])


def test_e4m3_codec_against_torch():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-8, 6, 100000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(M.e4m3_encode(x.astype(np.float64)), ref.view(torch.uint8).numpy())
    np.testing.assert_array_equal(M.e4m3_decode(ref.view(torch.uint8).numpy()), ref.double().numpy())


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------

def _tiny_context(seed=0, H=4, new=(16, 33), cache=(0, 40)):
    rng = np.random.default_rng(seed)
    T = sum(new)
    q = rng.standard_normal((T, H, M.DQ))
    kn = [rng.standard_normal((n + c, H, M.DN)) for n, c in zip(new, cache)]
    kr = [rng.standard_normal((n + c, M.DR)) for n, c in zip(new, cache)]
    v = [rng.standard_normal((n + c, H, M.DV)) for n, c in zip(new, cache)]
    return q, kn, kr, v, np.array(new), np.array(cache)


def test_attention_bruteforce_tiny():
    q, kn, kr, v, new, cache = _tiny_context()
    scale = 1 / math.sqrt(192)
    res = O.attention_reference(q, kn, kr, v, new, cache, scale)
    iro = [0, 16, 49]
    for b in range(2):
        L = new[b] + cache[b]
        for h in (0, 3):
            tok, o, lse = res[(b, h)]
            for i in range(new[b]):
                t = iro[b] + i
                mask = [[j <= cache[b] + ii for j in range(L)] for ii in range(new[b])]
                s = []
                for j in range(L):
                    if not mask[i][j]:
                        continue
                    acc = 0.0
                    for d in range(M.DN):
                        acc += q[t, h, d] * kn[b][j, h, d]
                    for d in range(M.DR):
                        acc += q[t, h, M.DN + d] * kr[b][j, d]
                    s.append((j, acc * scale))
                mx = max(x for _, x in s)
                den = sum(math.exp(x - mx) for _, x in s)
                assert abs(lse[i] - (mx + math.log(den))) < 1e-10
                for d in (0, 77, 127):
                    num = sum(math.exp(x - mx) * v[b][j, h, d] for j, x in s)
                    assert abs(o[i, d] - num / den) < 1e-10


def test_softmax_rows_sum_to_one_and_mask():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((50, 70)) * 5
    vis = np.arange(70)[None, :] <= (np.arange(50)[:, None] + 3)
    w, lse = M.softmax_weights(np.where(vis, s, -np.inf))
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(w[~vis] == 0)
    w, lse = M.softmax_weights(np.full((2, 5), -np.inf))
    assert np.all(w == 0) and np.all(np.isneginf(lse))


def test_attention_closed_forms():
    q, kn, kr, v, new, cache = _tiny_context(seed=1)
    scale = 1 / math.sqrt(192)
    res = O.attention_reference(q, kn, kr, v, new, cache, scale)
    # first new token of a sequence without cache sees only key 0
    _, o, lse = res[(0, 2)]
    np.testing.assert_allclose(o[0], v[0][0, 2], atol=1e-13)
    s00 = scale * (q[0, 2, :M.DN] @ kn[0][0, 2] + q[0, 2, M.DN:] @ kr[0][0])
    assert abs(lse[0] - s00) < 1e-12
    # zero queries weight every visible key equally
    q0 = np.zeros_like(q)
    res0 = O.attention_reference(q0, kn, kr, v, new, cache, scale)
    _, o, lse = res0[(1, 1)]
    for i in (0, 10, 32):
        nvis = cache[1] + i + 1
        np.testing.assert_allclose(o[i], v[1][:nvis, 1].mean(axis=0), atol=1e-12)
        assert abs(lse[i] - math.log(nvis)) < 1e-12


def test_attention_batch_permutation():
    q, kn, kr, v, new, cache = _tiny_context(seed=3, new=(5, 9, 3), cache=(7, 0, 12))
    scale = 0.1
    res = O.attention_reference(q, kn, kr, v, new, cache, scale)
    perm = [2, 0, 1]
    iro = np.concatenate([[0], np.cumsum(new)])
    qp = np.concatenate([q[iro[b]:iro[b + 1]] for b in perm])
    resp = O.attention_reference(qp, [kn[b] for b in perm], [kr[b] for b in perm],
                                 [v[b] for b in perm], new[perm], cache[perm], scale)
    for nb, b in enumerate(perm):
        for h in range(4):
            np.testing.assert_allclose(resp[(nb, h)][1], res[(b, h)][1], atol=1e-13)


def test_merge_split_equals_one_shot():
    rng = np.random.default_rng(8)
    n, m = 20, 60
    qn, qr = rng.standard_normal((n, M.DN)), rng.standard_normal((n, M.DR))
    kn, kr, v = rng.standard_normal((m, M.DN)), rng.standard_normal((m, M.DR)), rng.standard_normal((m, M.DV))
    q_pos = rng.integers(0, m, n)
    k_pos = rng.permutation(m)
    o, lse = O.partial_attention(qn, qr, kn, kr, v, q_pos, k_pos, 0.2)
    part = rng.random(m) < 0.5
    oa, la = O.partial_attention(qn, qr, kn[part], kr[part], v[part], q_pos, k_pos[part], 0.2)
    ob, lb = O.partial_attention(qn, qr, kn[~part], kr[~part], v[~part], q_pos, k_pos[~part], 0.2)
    om, lm = O.merge_partials(oa, la, ob, lb)
    np.testing.assert_allclose(om, o, atol=1e-12)
    np.testing.assert_allclose(lm, lse, atol=1e-12)
    # merging with an empty part is the identity
    oe, le = O.merge_partials(oa, la, np.zeros_like(oa), np.full(n, -np.inf))
    np.testing.assert_array_equal(oe, oa)


def _oracle_inputs(w, **kw):
    inp = make_inputs(w, with_w_uk=True, **kw)
    return inp, {k: O.codes(inp[k]) for k in ("q", "kv_cache", "w_k", "w_uv", "w_uk",
                                              "input_row_offsets", "cache_lengths", "page_table")}


def _unchunked_pipeline(inp, c, dtype="bf16", store=True):
    """Definition path: context latents straight from the paged cache (no
    plan), projected per head, attended over in one shot."""
    new, cache = inp["new_lens"], inp["cache_lens"]
    ctx = O.context_latents(c["kv_cache"], c["page_table"], inp["page_size"], new + cache)
    wk = O.decode(c["w_k"], dtype) * inp["w_scale"]
    wuv = O.decode(c["w_uv"], dtype) * inp["w_scale"]
    kn, kr, vv = [], [], []
    for x in ctx:
        lat = O.decode(x, dtype) * inp["ckv_scale"]
        k, v = O.upproject(lat[:, :M.R], wk, wuv, store=dtype if store else None)
        kn.append(k)
        vv.append(v)
        kr.append(lat[:, M.R:])
    q = O.decode(c["q"], dtype) * inp["q_scale"]
    return O.attention_reference(q, kn, kr, vv, new, cache, inp["scale"])


@pytest.mark.parametrize("S", [32, 7, 1000])
def test_chunked_pipeline_equals_unchunked(S):
    w = WORKLOADS["tiny_ragged"]
    inp, c = _oracle_inputs(w)
    ref = _unchunked_pipeline(inp, c)
    nc = -(-int((inp["new_lens"] + inp["cache_lens"]).sum()) // S) + 1
    res, plan = O.mla_prefill(c["q"], c["kv_cache"], c["page_table"], inp["page_size"],
                              c["w_k"], c["w_uv"], c["input_row_offsets"], c["cache_lengths"],
                              S, nc, inp["scale"])
    assert plan[3] == 0
    for key, (tok, o, lse) in ref.items():
        np.testing.assert_array_equal(res[key][0], tok)
        np.testing.assert_allclose(res[key][1], o, atol=1e-10)
        np.testing.assert_allclose(res[key][2], lse, atol=1e-10)


def test_chunked_pipeline_shuffled_pages_random_lengths():
    w = scaled(WORKLOADS["ragged_chunked_cache"], B=3, H=2, page_size=8, buffer_token_size=40,
               max_chunks=8, new_range=(1, 30), cache_range=(0, 60))
    inp, c = _oracle_inputs(w)
    ref = _unchunked_pipeline(inp, c)
    res, plan = O.mla_prefill(c["q"], c["kv_cache"], c["page_table"], inp["page_size"],
                              c["w_k"], c["w_uv"], c["input_row_offsets"], c["cache_lengths"],
                              w.buffer_token_size, w.max_chunks, inp["scale"])
    assert plan[3] == 0 and (plan[2] >= 0).sum() > 1
    for key, (tok, o, lse) in ref.items():
        np.testing.assert_allclose(res[key][1], o, atol=1e-10)


def test_absorbed_equals_upprojected():
    w = WORKLOADS["tiny_ragged"]
    inp, c = _oracle_inputs(w)
    new, cache = inp["new_lens"], inp["cache_lens"]
    wk = O.decode(c["w_k"], "bf16")
    wuv = O.decode(c["w_uv"], "bf16")
    H = w.H
    # w_uk[h] = W_k,h^T, the absorbed weight of the same projection
    w_uk = np.stack([wk[h * M.DN:(h + 1) * M.DN].T for h in range(H)])
    ctx = O.context_latents(c["kv_cache"], c["page_table"], inp["page_size"], new + cache)
    lat = [O.decode(x, "bf16") for x in ctx]
    q = O.decode(c["q"], "bf16")
    up = _unchunked_pipeline(inp, c, store=False)
    ab = O.attention_absorbed(q, [x[:, :M.R] for x in lat], [x[:, M.R:] for x in lat],
                              w_uk, wuv, new, cache, inp["scale"])
    for key in up:
        np.testing.assert_allclose(ab[key][1], up[key][1], rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(ab[key][2], up[key][2], rtol=1e-12, atol=1e-10)


def _decode_case(seed=3, H=3):
    """A decode-shaped batch: one or two new tokens per sequence over cached
    context, w_uk built from w_k (w_uk[h] = W_k,h^T)."""
    w = scaled(WORKLOADS["tiny_ragged"], H=H, B=3, page_size=8, new_lens=(1, 2, 1),
               cache_lens=(20, 0, 37), seed=seed)
    inp, c = _oracle_inputs(w)
    wk = O.decode(c["w_k"], "bf16")
    w_uk = np.stack([wk[h * M.DN:(h + 1) * M.DN].T for h in range(H)])
    wuv = O.decode(c["w_uv"], "bf16")
    q = O.decode(c["q"], "bf16")
    return inp, c, q, w_uk, wuv


def test_decode_equals_upprojected_attention():
    """The absorbed decode over the paged cache equals up-projecting K and V and
    attending over them (no rounding of K/V on either side)."""
    inp, c, q, w_uk, wuv = _decode_case()
    dec = O.mla_decode(q, c["kv_cache"], c["page_table"], inp["page_size"], w_uk, wuv,
                       c["input_row_offsets"], c["cache_lengths"], inp["scale"], num_partitions=3)
    up = _unchunked_pipeline(inp, c, store=False)
    assert set(dec) == set(up)
    for key in up:
        np.testing.assert_array_equal(dec[key][0], up[key][0])
        np.testing.assert_allclose(dec[key][1], up[key][1], rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(dec[key][2], up[key][2], rtol=1e-12, atol=1e-10)


def test_decode_partition_count_invariant():
    """Any number of key partitions, including more partitions than keys (empty
    ones), gives the same result."""
    inp, c, q, w_uk, wuv = _decode_case(seed=5, H=2)
    args = (q, c["kv_cache"], c["page_table"], inp["page_size"], w_uk, wuv, c["input_row_offsets"],
            c["cache_lengths"], inp["scale"])
    base = O.mla_decode(*args, num_partitions=1)
    for parts in (2, 5, 16, 64):
        got = O.mla_decode(*args, num_partitions=parts)
        for key in base:
            np.testing.assert_allclose(got[key][1], base[key][1], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(got[key][2], base[key][2], rtol=1e-13, atol=1e-13)


def _sparse_args(inp, c, q, w_uk, wuv):
    """Each sequence's whole context as physical cache rows, padded with -1."""
    ps = inp["page_size"]
    L = inp["new_lens"] + inp["cache_lens"]
    stride = int(L.max()) + 3
    idx = np.full((inp["B"], stride), -1, dtype=np.int64)
    for b in range(inp["B"]):
        pos = np.arange(int(L[b]))
        idx[b, :L[b]] = c["page_table"][b, pos // ps] * ps + pos % ps
    return idx, L


def test_sparse_decode_over_the_whole_context_equals_dense_decode():
    """One new token per sequence: listing every context row of the sequence
    gives exactly the dense decode (whose pins tie it to up-projected attention)."""
    w = scaled(WORKLOADS["tiny_ragged"], H=2, B=3, page_size=8, new_lens=(1, 1, 1),
               cache_lens=(20, 0, 37), seed=9)
    inp, c = _oracle_inputs(w)
    wk = O.decode(c["w_k"], "bf16")
    w_uk = np.stack([wk[h * M.DN:(h + 1) * M.DN].T for h in range(2)])
    wuv = O.decode(c["w_uv"], "bf16")
    q = O.decode(c["q"], "bf16")
    idx, L = _sparse_args(inp, c, q, w_uk, wuv)
    dense = O.mla_decode(q, c["kv_cache"], c["page_table"], inp["page_size"], w_uk, wuv,
                         c["input_row_offsets"], c["cache_lengths"], inp["scale"])
    sparse = O.mla_sparse_decode(q, c["kv_cache"], inp["page_size"], w_uk, wuv, c["input_row_offsets"],
                                 idx, L, inp["scale"])
    assert set(dense) == set(sparse)
    for key in dense:
        np.testing.assert_array_equal(sparse[key][0], dense[key][0])
        np.testing.assert_allclose(sparse[key][1], dense[key][1], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sparse[key][2], dense[key][2], rtol=1e-13, atol=1e-13)


def _sparse_case(seed=4):
    inp, c, q, w_uk, wuv = _decode_case(seed=seed, H=2)
    idx, L = _sparse_args(inp, c, q, w_uk, wuv)
    return inp, c, q, w_uk, wuv, idx, L


def test_sparse_decode_is_a_set_and_ignores_entries_past_topk():
    """Permuting the listed rows changes nothing; entries past topk_lengths are
    never read (garbage there changes nothing)."""
    inp, c, q, w_uk, wuv, idx, L = _sparse_case()
    args = (q, c["kv_cache"], inp["page_size"], w_uk, wuv, c["input_row_offsets"])
    base = O.mla_sparse_decode(*args, idx, L, inp["scale"])
    rng = np.random.default_rng(1)
    perm = idx.copy()
    for b in range(idx.shape[0]):
        perm[b, :L[b]] = rng.permutation(idx[b, :L[b]])
        perm[b, L[b]:] = 10 ** 6   # out of range: must not be read
    got = O.mla_sparse_decode(*args, perm, L, inp["scale"])
    for key in base:
        np.testing.assert_allclose(got[key][1], base[key][1], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(got[key][2], base[key][2], rtol=1e-13)


def test_sparse_decode_closed_forms():
    """top-1: the output is w_uv[h] times that row's latent values and the LSE
    is its score; a row listed twice weighs twice (LSE grows by log 2)."""
    inp, c, q, w_uk, wuv, idx, L = _sparse_case(seed=6)
    rows = c["kv_cache"].reshape(-1, 576)
    one = np.ones(inp["B"], dtype=np.int64)
    res = O.mla_sparse_decode(q, c["kv_cache"], inp["page_size"], w_uk, wuv, c["input_row_offsets"],
                              idx, one, inp["scale"])
    for (b, h), (tok, out, lse) in res.items():
        lat = O.decode(rows[idx[b, 0]], "bf16")
        for n, t in enumerate(tok):
            s = inp["scale"] * ((w_uk[h] @ q[t, h, :M.DN]) @ lat[:M.R] + q[t, h, M.DN:] @ lat[M.R:])
            np.testing.assert_allclose(out[n], wuv[h] @ lat[:M.R], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[n], s, rtol=1e-12, atol=1e-13)
    twice = np.concatenate([idx[:, :1], idx[:, :1]], axis=1)
    res2 = O.mla_sparse_decode(q, c["kv_cache"], inp["page_size"], w_uk, wuv, c["input_row_offsets"],
                               twice, None, inp["scale"])
    for key in res:
        np.testing.assert_allclose(res2[key][1], res[key][1], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(res2[key][2], res[key][2] + math.log(2.0), rtol=1e-12)


def test_attention_sink_closed_forms():
    """A sink of -inf changes nothing.  With q = 0 every score is 0, so over n
    rows and a sink s: LSE = log(n + e^s) and out = n / (n + e^s) times w_uv[h]
    applied to the mean latent row."""
    inp, c, q, w_uk, wuv, idx, L = _sparse_case(seed=8)
    args = (c["kv_cache"], inp["page_size"], w_uk, wuv, c["input_row_offsets"], idx, L, inp["scale"])
    base = O.mla_sparse_decode(q, *args)
    none = O.mla_sparse_decode(q, *args, attn_sink=np.full(inp["B"], -np.inf))
    for key in base:
        np.testing.assert_allclose(none[key][1], base[key][1], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(none[key][2], base[key][2], rtol=1e-13)
    sink = np.array([0.5, -1.25, 2.0])
    zq = np.zeros_like(q)
    got = O.mla_sparse_decode(zq, *args, attn_sink=sink)
    rows = c["kv_cache"].reshape(-1, 576)
    for (b, h), (tok, out, lse) in got.items():
        n = int(L[b])
        mean = O.decode(rows[idx[b, :n]], "bf16")[:, :M.R].mean(axis=0)
        frac = n / (n + math.exp(sink[b]))
        for k in range(len(tok)):
            np.testing.assert_allclose(lse[k], math.log(n + math.exp(sink[b])), rtol=1e-12)
            np.testing.assert_allclose(out[k], frac * (wuv[h] @ mean), rtol=1e-10, atol=1e-12)


def test_fp8_pipeline_chunked_equals_unchunked():
    w = scaled(WORKLOADS["longctx_fp8"], H=2, new_lens=(40,), cache_lens=(50,),
               buffer_token_size=48, max_chunks=2, page_size=16)
    inp, c = _oracle_inputs(w)
    assert inp["w_scale"] != 1.0
    ref = _unchunked_pipeline(inp, c, dtype="e4m3")
    res, plan = O.mla_prefill(c["q"], c["kv_cache"], c["page_table"], inp["page_size"],
                              c["w_k"], c["w_uv"], c["input_row_offsets"], c["cache_lengths"],
                              w.buffer_token_size, w.max_chunks, inp["scale"], dtype="e4m3",
                              w_scale=inp["w_scale"])
    for key, (tok, o, lse) in ref.items():
        np.testing.assert_allclose(res[key][1], o, atol=1e-10)
    # K/V were held in e4m3: outputs differ from the unrounded path, but not by much
    raw = _unchunked_pipeline(inp, c, dtype="e4m3", store=False)
    d = max(np.abs(raw[k][1] - ref[k][1]).max() for k in ref)
    assert 1e-4 < d < 0.2


def test_flop_count_tiny():
    # 16*17/2 + 33*40 + 33*34/2 visible pairs, 640 flops per pair per head
    assert M.causal_pairs([16, 33], [0, 40]) == 2017
    assert M.attention_flops([16, 33], [0, 40], 4) == 2 * 4 * 320 * 2017
