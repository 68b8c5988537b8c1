"""The C ABI on the host: the library builds, loads, exports every function
include/mla_prefill.h declares, and rejects bad arguments before touching the
GPU.  CPU only: no call here launches a kernel."""
import ctypes
import os
import re

import pytest

import mla_prefill_attention_plan_gb300 as mla
from mla_prefill_attention_plan_gb300 import build as B

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return mla.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("mla_latent_cache_write", "mla_prefill_plan", "mla_gather_latent", "mla_upproject",
              "mla_prefill_attention", "mla_chunk_cache_rows", "mla_upproject_paged",
              "mla_prefill_attention_paged", "mla_prefill", "mla_prefill_workspace_bytes",
              "mla_status_string"):
        assert n in names


def test_every_entry_point_cites_its_passage():
    """Each declaration in the header is preceded by a comment that names the
    page it follows (a quoted page title) or says it has no counterpart there."""
    import re
    text = open(os.path.join(HEADER_DIR, "mla_prefill.h")).read()
    for m in re.finditer(r"\n[a-z_0-9 \*]*\b(mla_[a-z_0-9]+)\(", text):
        before = text[:m.start()]
        comment = before[before.rfind("/*"):]
        assert comment.startswith("/*") and "*/" in comment, m.group(1)
        assert '"' in comment or "no counterpart" in comment, m.group(1)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # and the binding describes each of them
    assert set(_declared()) == set(mla.SIGNATURES)


def test_abi_version_and_strings(lib):
    assert mla.mla_abi_version() == 2
    # dtype-only answers need no device
    assert mla.mla_attention_kernel(mla.MLA_E4M3) == "e4m3"
    assert mla.mla_attention_kernel(7) is None
    assert "workspace" in mla.status_string(mla.MLA_ERR_WORKSPACE)
    assert "timed out" in mla.status_string(mla.MLA_DEV_TIMEOUT)


def test_host_argument_errors(lib):
    s = 1  # any non-null stream handle: these calls fail before using it
    assert mla.mla_prefill_plan(None, None, None, None, None, 1, 1, 8, None, s) == mla.MLA_ERR_ARG
    assert mla.mla_prefill_plan(16, 16, 16, 16, 16, 1, 1, 0, None, s) == mla.MLA_ERR_ARG
    assert mla.mla_prefill_plan(16, 16, 16, 16, 16, 1, 0, 8, None, s) == mla.MLA_ERR_ARG
    assert mla.mla_gather_latent(16, 16, 16, 16, 1, 16, 1, 16, 16, 16, 0, 1, 8, 7, None, s) == mla.MLA_ERR_DTYPE
    assert mla.mla_gather_latent(17, 16, 16, 16, 1, 16, 1, 16, 16, 16, 0, 1, 8, 0, None, s) == mla.MLA_ERR_ARG
    assert mla.mla_upproject(16, 16, 16, 16, 16, None, 0, 8, 0, 0, stream=s) == mla.MLA_ERR_GEOMETRY
    assert mla.mla_upproject(16, 16, 16, 16, 16, None, 0, 8, 4, 2, stream=s) == mla.MLA_ERR_DTYPE
    # multi-chunk attention needs the merge scratch
    args = [16, None, None, None] + [16] * 9 + [0, 2, 1, 4, 16, 16, 8, 0.1]
    assert mla.mla_prefill_attention(*args, stream=s) == mla.MLA_ERR_ARG
    # chunk index outside the plan
    args = [16, None, 16, 16] + [16] * 9 + [3, 2, 1, 4, 16, 16, 8, 0.1]
    assert mla.mla_prefill_attention(*args, stream=s) == mla.MLA_ERR_ARG


def _caller(fn, ok, names):
    def call(**change):
        a = list(ok)
        for k, v in change.items():
            a[names.index(k)] = v
        return fn(*a, stream=1)   # any non-null handle: these calls fail before using it
    return call


def test_paged_attention_host_argument_errors(lib):
    names = ["out", "lse", "oacc", "lacc", "q", "kn", "v", "kv", "rows", "ncr", "iro", "cl", "bro", "co",
             "bl", "ch", "mc", "B", "H", "mpl", "T", "S", "scale"]
    ok = [16, None, None, None, 16, 16, 16, 16, 16, 64, 16, 16, 16, 16, 16, 0, 1, 1, 4, 16, 16, 8, 0.1]
    call = _caller(mla.mla_prefill_attention_paged, ok, names)
    assert call(kv=None) == mla.MLA_ERR_ARG
    assert call(kv=24) == mla.MLA_ERR_ARG              # misaligned cache
    assert call(rows=None) == mla.MLA_ERR_ARG
    assert call(ncr=0) == mla.MLA_ERR_ARG
    assert call(H=0) == mla.MLA_ERR_GEOMETRY
    assert call(mc=2) == mla.MLA_ERR_ARG               # merge scratch missing
    # the buffered entry point still wants its k_rope buffer
    args = [16, None, None, None, 16, 16, 16, None] + [16] * 5 + [0, 1, 1, 4, 16, 16, 8, 0.1]
    assert mla.mla_prefill_attention(*args, stream=1) == mla.MLA_ERR_ARG


def test_paged_upproject_host_argument_errors(lib):
    names = ["kn", "v", "kv", "rows", "ncr", "bl", "ch", "S", "wk", "wuv", "H", "dt"]
    ok = [16, 16, 16, 16, 64, 16, 0, 8, 16, 16, 2, mla.MLA_BF16]
    call = _caller(mla.mla_upproject_paged, ok, names)
    assert call(kv=None) == mla.MLA_ERR_ARG
    assert call(kv=8) == mla.MLA_ERR_ARG
    assert call(rows=None) == mla.MLA_ERR_ARG
    assert call(bl=None) == mla.MLA_ERR_ARG
    assert call(ncr=0) == mla.MLA_ERR_ARG
    assert call(H=0) == mla.MLA_ERR_GEOMETRY
    assert call(dt=5) == mla.MLA_ERR_DTYPE


def test_chunk_cache_rows_host_argument_errors(lib):
    names = ["rows", "pt", "np", "ps", "mp", "bro", "co", "bl", "mc", "B", "S"]
    ok = [16, 16, 4, 16, 2, 16, 16, 16, 2, 1, 8]
    call = _caller(mla.mla_chunk_cache_rows, ok, names)
    for k in ("rows", "pt", "bro", "co", "bl"):
        assert call(**{k: None}) == mla.MLA_ERR_ARG, k
    for k in ("np", "ps", "mp", "mc", "B", "S"):
        assert call(**{k: 0}) == mla.MLA_ERR_ARG, k
    assert call(np=1 << 20, ps=1 << 11) == mla.MLA_ERR_ARG   # 2^31 cache rows
    assert call(mc=1 << 16) == mla.MLA_ERR_ARG


def test_selftest_host_argument_errors(lib):
    s = 1
    assert mla.mla_selftest_bounded_wait(None, 16, 5_000_000, 2, s) == mla.MLA_ERR_ARG
    assert mla.mla_selftest_bounded_wait(16, None, 5_000_000, 2, s) == mla.MLA_ERR_ARG
    assert mla.mla_selftest_bounded_wait(16, 12, 5_000_000, 2, s) == mla.MLA_ERR_ARG   # misaligned
    assert mla.mla_selftest_bounded_wait(16, 16, 5_000_000, 3, s) == mla.MLA_ERR_ARG
    assert mla.mla_selftest_bounded_wait(16, 16, 10, 1, s) == mla.MLA_ERR_ARG
    assert mla.mla_selftest_bounded_wait(16, 16, 3_000_000_000, 1, s) == mla.MLA_ERR_ARG


def test_cache_write_host_argument_errors(lib):
    s = 1
    # kv_cache, q, kv_latent, gamma, freqs, iro, cache_lengths, page_table, num_pages, page_size,
    # max_pages, B, H, T, max_seq_len, epsilon, kv_inv_scale, dtype
    ok = [16, 16, 16, 16, 16, 16, 16, 16, 4, 16, 2, 1, 2, 8, 64, 1e-6, 1.0, mla.MLA_BF16]

    def call(**change):
        a = list(ok)
        names = ["kv", "q", "lat", "gamma", "freqs", "iro", "cl", "pt", "np", "ps", "mp", "B", "H", "T",
                 "msl", "eps", "inv", "dt"]
        for k, v in change.items():
            a[names.index(k)] = v
        return mla.mla_latent_cache_write(*a, None, s)
    assert call(dt=7) == mla.MLA_ERR_DTYPE
    assert call(kv=None) == mla.MLA_ERR_ARG
    assert call(lat=24) == mla.MLA_ERR_ARG          # misaligned
    assert call(freqs=20) == mla.MLA_ERR_ARG
    assert call(B=0) == mla.MLA_ERR_ARG
    assert call(T=-1) == mla.MLA_ERR_ARG
    assert call(H=0) == mla.MLA_ERR_ARG             # q given without heads
    assert call(msl=0) == mla.MLA_ERR_ARG
    assert call(eps=-1.0) == mla.MLA_ERR_ARG
    assert call(inv=0.0) == mla.MLA_ERR_ARG


def test_workspace_size_and_errors(lib):
    small = mla.mla_prefill_workspace_bytes(2, 4, 49, 1, 32, mla.MLA_BF16)
    big = mla.mla_prefill_workspace_bytes(2, 4, 49, 4, 32, mla.MLA_BF16)
    fp8 = mla.mla_prefill_workspace_bytes(2, 4, 49, 1, 32, mla.MLA_E4M3)
    # one chunk: no merge scratch; more chunks: fp32 O and LSE per (token, head)
    assert big - small >= 49 * 4 * 128 * 4 + 49 * 4 * 4
    assert fp8 < small
    assert mla.mla_prefill_workspace_bytes(2, 0, 49, 1, 32, 0) == 0
    need = big
    common = dict(out=16, lse=None, q=16, input_row_offsets=16, cache_lengths=16, kv_cache=16,
                  page_table=16, num_pages=1, page_size=16, max_pages_per_seq=1, w_k=16, w_uv=16,
                  batch_size=2, num_heads=4, total_q_tokens=49, max_prompt_len=33,
                  buffer_token_size=32, max_chunks=4, scale=0.07, stream=s_handle())
    assert mla.mla_prefill(workspace=None, workspace_bytes=need, **common) == mla.MLA_ERR_WORKSPACE
    assert mla.mla_prefill(workspace=256, workspace_bytes=need - 1, **common) == mla.MLA_ERR_WORKSPACE
    assert mla.mla_prefill(workspace=128, workspace_bytes=need, **common) == mla.MLA_ERR_WORKSPACE


def s_handle():
    return 1


def test_build_flags_target_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    for src in B.SOURCES:
        assert os.path.exists(os.path.join(B.CSRC, src))


def test_product_path_never_touches_the_oracle():
    pkg = os.path.dirname(mla.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
