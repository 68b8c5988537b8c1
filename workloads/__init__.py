"""Seeded synthetic inputs for ragged MLA prefill over a paged latent KV cache.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and lays them out in the tensor shapes
the method consumes; it holds none of the method's arithmetic (no planning, no
gather, no projection, no attention).

Shapes follow the MLA pages:
  * ``q``            [T_q, H, 192]  (128 nope then 64 rope per head)
                     -- mla_prefill_decode_graph_bf16, Args ``q``;
                        flare_mla_prefill_dispatch, Parameters ``q_depth``
  * ``kv_cache``     [num_pages, page_size, 576] (512 latent c_kv, then 64 k_rope)
                     -- flare_mla_prefill_dispatch, Parameters ``cache_depth``
  * ``w_k``          [H*128, 512], ``w_uk`` [H, 512, 128], ``w_uv`` [H, 128, 512]
                     -- mla_prefill_decode_graph_bf16, Args ``w_k``/``w_uk``/``w_uv``
  * ``input_row_offsets`` [B+1] cumulative new-token offsets
                     -- mla_prefill_plan, Args ``input_row_offsets``

The paged cache holds every context token of a sequence, cached tokens first and
then the new tokens, ``cache_len + new_len`` tokens in all.  Pages of a sequence
are listed in ``page_table[b]``; unused entries are -1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

KV_LORA_RANK = 512          # latent width R
QK_NOPE = 128               # dn
QK_ROPE = 64                # dr
V_DIM = 128                 # dv
Q_DEPTH = QK_NOPE + QK_ROPE  # 192
CACHE_DEPTH = KV_LORA_RANK + QK_ROPE  # 576


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: batch geometry, cache paging and dtype."""
    name: str
    B: int
    H: int
    page_size: int
    buffer_token_size: int
    max_chunks: int
    dtype: str = "bf16"                 # "bf16" or "e4m3"
    new_lens: tuple | None = None       # fixed new-token counts, or None for random
    cache_lens: tuple | None = None     # fixed cached-token counts, or None for random
    new_range: tuple = (256, 2048)      # inclusive integer ranges for random lengths
    cache_range: tuple = (0, 8192)
    shuffle_pages: bool = False
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(Q_DEPTH)


# The five workloads: a tiny ragged case, a DeepSeek-V2-Lite-shaped prefill, a
# DeepSeek-V3-shaped prefill, a ragged multi-chunk prefill with cache and a long
# fp8 prefill.  Sizes the pages leave open (buffer size for one-chunk runs, the
# chunk-table height) are chosen to fit exactly as many chunks as the lengths need.
WORKLOADS = {
    "tiny_ragged": Workload("tiny_ragged", B=2, H=4, page_size=16, buffer_token_size=32,
                            max_chunks=4, new_lens=(16, 33), cache_lens=(0, 40)),
    "v2lite_prefill": Workload("v2lite_prefill", B=4, H=16, page_size=128,
                               buffer_token_size=4096, max_chunks=1,
                               new_lens=(1024,) * 4, cache_lens=(0,) * 4),
    "v3_prefill": Workload("v3_prefill", B=1, H=128, page_size=128, buffer_token_size=4096,
                           max_chunks=1, new_lens=(4096,), cache_lens=(0,)),
    "ragged_chunked_cache": Workload("ragged_chunked_cache", B=8, H=128, page_size=128,
                                     buffer_token_size=8192, max_chunks=10,
                                     shuffle_pages=True),
    "longctx_fp8": Workload("longctx_fp8", B=1, H=128, page_size=128,
                            buffer_token_size=16384, max_chunks=2, dtype="e4m3",
                            new_lens=(16384,), cache_lens=(16384,)),
}

# Decode (the absorbed branch of the same graph): a few new tokens per sequence
# over long cached contexts, DeepSeek-V3 dims.  Inputs come from make_inputs
# with with_w_uk=True; the cache holds every context token, new ones included.
DECODE_WORKLOADS = {
    "v3_decode": Workload("v3_decode", B=64, H=128, page_size=128, buffer_token_size=1,
                          max_chunks=1, new_range=(1, 2), cache_range=(4096, 16384),
                          shuffle_pages=True),
    # Sparse decode: each sequence attends to 2048 listed rows of its context
    # (make_sparse_indices), with per-batch sinks (make_attention_sinks).
    "v3_sparse_decode": Workload("v3_sparse_decode", B=64, H=128, page_size=128,
                                 buffer_token_size=1, max_chunks=1, new_range=(1, 1),
                                 cache_range=(4096, 16384), shuffle_pages=True),
}

# Reduced cases of the workloads above, small enough for a full profiler capture
# (a few hundred MB on the device); timed by bench.py, not parity cases.
PROFILE_CASES = {
    "longctx_fp8_4k": Workload("longctx_fp8_4k", B=1, H=128, page_size=128,
                               buffer_token_size=4096, max_chunks=2, dtype="e4m3",
                               new_lens=(4096,), cache_lens=(4096,)),
}


def lengths(w: Workload):
    """Seeded (new_lens, cache_lens) as int64 numpy arrays."""
    rng = np.random.default_rng(w.seed)
    if w.new_lens is not None:
        new = np.asarray(w.new_lens, dtype=np.int64)
    else:
        new = rng.integers(w.new_range[0], w.new_range[1], size=w.B, endpoint=True)
    if w.cache_lens is not None:
        cache = np.asarray(w.cache_lens, dtype=np.int64)
    else:
        cache = rng.integers(w.cache_range[0], w.cache_range[1], size=w.B, endpoint=True)
    assert len(new) == w.B and len(cache) == w.B
    return new.astype(np.int64), cache.astype(np.int64)


def _normal(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def _to_storage(x: torch.Tensor, dtype: str) -> torch.Tensor:
    """Round float32 samples to the storage dtype (torch's round-to-nearest-even)."""
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "e4m3":
        return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    raise ValueError(dtype)


def make_inputs(w: Workload, with_w_uk: bool = False, new_lens=None, cache_lens=None):
    """Build every input tensor of a workload on the CPU.

    Generation order is fixed: lengths, cache lengths, page permutation, q,
    cache, w_k, w_uv (then w_uk, only if asked).  Activations are N(0,1); the
    weights are N(0, 1/sqrt(512)) (standard deviation), so the projected K and V
    come out near N(0,1).  For the e4m3 workload the weights are stored as
    N(0,1) e4m3 values with a per-tensor descale of 1/sqrt(512), and the cache
    descale is 1.
    """
    if new_lens is None or cache_lens is None:
        n_new, n_cache = lengths(w)
    else:
        n_new = np.asarray(new_lens, np.int64)
        n_cache = np.asarray(cache_lens, np.int64)
    B, H, ps = len(n_new), w.H, w.page_size
    total = n_new + n_cache
    iro = np.zeros(B + 1, dtype=np.int64)
    iro[1:] = np.cumsum(n_new)
    T_q = int(iro[-1])

    pages_per_seq = [(int(t) + ps - 1) // ps for t in total]
    num_pages = max(1, sum(pages_per_seq))
    max_pages = max(1, max(pages_per_seq))
    rng = np.random.default_rng(w.seed + 1)
    phys = rng.permutation(num_pages) if w.shuffle_pages else np.arange(num_pages)
    page_table = np.full((B, max_pages), -1, dtype=np.int64)
    k = 0
    for b in range(B):
        for p in range(pages_per_seq[b]):
            page_table[b, p] = phys[k]
            k += 1

    gen = torch.Generator().manual_seed(w.seed)
    q = _to_storage(_normal(gen, (T_q, H, Q_DEPTH)), w.dtype)
    kv_cache = _to_storage(_normal(gen, (num_pages, ps, CACHE_DEPTH)), w.dtype)
    if w.dtype == "bf16":
        w_std, w_descale = 1.0 / math.sqrt(KV_LORA_RANK), 1.0
    else:
        w_std, w_descale = 1.0, 1.0 / math.sqrt(KV_LORA_RANK)
    w_k = _to_storage(_normal(gen, (H * QK_NOPE, KV_LORA_RANK), w_std), w.dtype)
    w_uv = _to_storage(_normal(gen, (H, V_DIM, KV_LORA_RANK), w_std), w.dtype)
    out = dict(
        workload=w, B=B, H=H, T_q=T_q, page_size=ps, num_pages=num_pages,
        max_pages=max_pages, new_lens=n_new, cache_lens=n_cache,
        input_row_offsets=torch.from_numpy(iro.astype(np.int32)),
        cache_lengths=torch.from_numpy(n_cache.astype(np.int32)),
        page_table=torch.from_numpy(page_table.astype(np.int32)),
        q=q, kv_cache=kv_cache, w_k=w_k, w_uv=w_uv,
        scale=w.scale, q_scale=1.0, ckv_scale=1.0, w_scale=w_descale,
        max_prompt_len=int(n_new.max()) if B else 0,
    )
    if with_w_uk:
        out["w_uk"] = _to_storage(_normal(gen, (H, KV_LORA_RANK, QK_NOPE), w_std), w.dtype)
    return out


def make_attention_operands(w: Workload, rows: int, seed_offset: int = 7):
    """Direct K_nope / V / k_rope buffers ([rows,H,128], [rows,H,128], [rows,64]),
    N(0,1) in the workload's dtype, for testing the attention stage on its own.
    For e4m3, V is stored as float16 holding the e4m3-rounded values (the
    layout the up-projection writes for the attention)."""
    gen = torch.Generator().manual_seed(w.seed + seed_offset)
    k_nope = _to_storage(_normal(gen, (rows, w.H, QK_NOPE)), w.dtype)
    v = _to_storage(_normal(gen, (rows, w.H, V_DIM)), w.dtype)
    if w.dtype == "e4m3":
        v = v.to(torch.float16)   # exact
    k_rope = _to_storage(_normal(gen, (rows, QK_ROPE)), w.dtype)
    return k_nope, v, k_rope


def make_cache_write_operands(w: Workload, T_q: int, max_seq_len: int, seed_offset: int = 11):
    """Inputs of the latent-cache write ("mla_prefill_decode_graph_bf16", Args
    freqs_cis, kv_norm_gamma, epsilon): the new tokens' latent rows before
    normalisation ([T_q, 576] bf16, N(0, 2**2): a projection output of
    arbitrary scale), the RMSNorm weights ([512] float32, 1 + N(0, 0.1**2)),
    and a RoPE frequency table ([max_seq_len, 64] float32: for position p and
    pair k the unit complex number at angle p * 10000**(-k/32), stored as
    interleaved (cos, sin) values)."""
    gen = torch.Generator().manual_seed(w.seed + seed_offset)
    kv_latent = _normal(gen, (T_q, CACHE_DEPTH), 2.0).to(torch.bfloat16)
    gamma = 1.0 + _normal(gen, (KV_LORA_RANK,), 0.1)
    pos = np.arange(max_seq_len, dtype=np.float64)[:, None]
    inv_freq = 10000.0 ** (-np.arange(QK_ROPE // 2, dtype=np.float64) / (QK_ROPE // 2))
    ang = pos * inv_freq[None, :]
    freqs = np.empty((max_seq_len, QK_ROPE), dtype=np.float32)
    freqs[:, 0::2] = np.cos(ang)
    freqs[:, 1::2] = np.sin(ang)
    return kv_latent, gamma, torch.from_numpy(freqs)


def make_sparse_indices(inp, topk: int, stride: int | None = None, seed: int = 13, pad: int = -1):
    """Top-k lists for sparse decode ("mla_prefill_decode_graph_bf16", Args
    d_indices, indices_stride, topk_lengths): for each sequence, min(topk, L_b)
    distinct context positions drawn uniformly (seeded), stored as physical
    cache rows page * page_size + slot; entries past the count hold `pad`.
    Returns (indices int32 [B, stride], topk_lengths int32 [B])."""
    rng = np.random.default_rng(seed)
    L = inp["new_lens"] + inp["cache_lens"]
    stride = stride or max(1, topk)
    ps = inp["page_size"]
    pt = inp["page_table"].numpy().astype(np.int64)
    idx = np.full((inp["B"], stride), pad, dtype=np.int64)
    cnt = np.zeros(inp["B"], dtype=np.int64)
    for b in range(inp["B"]):
        k = min(topk, int(L[b]), stride)
        pos = np.sort(rng.choice(int(L[b]), size=k, replace=False))
        idx[b, :k] = pt[b, pos // ps] * ps + pos % ps
        cnt[b] = k
    return torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(cnt.astype(np.int32))


def make_attention_sinks(B: int, seed: int = 17):
    """Per-batch attention sink logits ("attn_sink_ptr"), N(0, 1) float32."""
    gen = torch.Generator().manual_seed(seed)
    return _normal(gen, (B,))


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller test variants)."""
    return dataclasses.replace(w, **changes)
