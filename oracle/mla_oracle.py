"""CPU oracle for ragged MLA prefill over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
Python binding) imports or calls this module; only the tests, the smoke check
and the benchmark's CPU baseline do.  It shares no code with the CUDA path.

Everything is plain numpy in float64, written to be checked against the pages
by eye, with a library matmul as the only borrowed step.  The pages are three
API references from the Modular MAX kernel library:

  * "mla_prefill_plan" -- the chunk plan (Args: buffer_row_offsets,
    cache_offsets, buffer_lengths, input_row_offsets, buffer_token_size);
  * "mla_prefill_decode_graph_bf16" -- the whole BF16 MLA layer (Args: q,
    freqs_cis, kv_norm_gamma, epsilon, w_k, w_uk, w_uv, scale,
    buffer_row_offsets, cache_offsets, buffer_length, num_partitions_in,
    d_indices, indices_stride, topk_lengths, attn_sink_ptr; Parameters:
    kv_input_fn, mask_str, sparse_mla, sparse_indices_stride);
  * "flare_mla_prefill_dispatch" -- prefill attention (Parameters: q_depth,
    cache_depth, kv_num_heads, dtype, output_type; Args: k, v, k_rope,
    valid_length, scale, cache_offsets).

Readings taken where the pages are silent (each one is listed with its reason
in the design notes of the repository):
  * the plan packs all sequences' context tokens (cached first, then new, in
    batch order) into consecutive chunks of ``buffer_token_size`` rows;
  * a cache row is 512 latent values followed by the 64 k_rope values, and a
    query row is 128 nope values followed by 64 rope values;
  * the causal mask lets the new token ``i`` of sequence ``b`` (absolute
    position ``cache_len_b + i``) see context positions ``j <= cache_len_b + i``;
  * LSE is the natural log of the sum of exp of the scaled scores;
  * the latent-cache write normalises the 512 latent values only (the
    weights have kv_lora_rank entries) as x / sqrt(mean(x**2) + epsilon) *
    gamma, and rotates rope values as 32 interleaved (real, imaginary) pairs
    multiplied by the freqs_cis row of the token's absolute position, for the
    latent's k_rope and for every query head's rope part;
  * K and V leave the up-projection in the storage dtype of the attention
    operands (bf16 for the BF16 graph, e4m3 for the fp8 path), rounded to
    nearest even, in the descale domain of the cache;
  * sparse decode: a d_indices entry is a physical cache row (page *
    page_size + slot), the list of batch entry b serves every new token of
    sequence b with no causal limit, and an attention sink is one extra logit
    per batch entry with no value row.
"""
from __future__ import annotations

import math

import numpy as np

R = 512        # kv_lora_rank: latent width
DN = 128       # qk_nope_head_dim
DR = 64        # qk_rope_head_dim
DV = 128       # v_head_dim
DQ = DN + DR   # q_depth, 192
DC = R + DR    # cache_depth, 576

# Device status codes shared by the plan and gather definitions.
STATUS_OK = 0
STATUS_TOO_MANY_CHUNKS = 1
STATUS_BAD_OFFSETS = 2
STATUS_BAD_PAGE = 3


# --------------------------------------------------------------------------
# Number formats (storage types named by flare_mla_prefill_dispatch, "dtype":
# bfloat16 or float8_e4m3fn).  Decoders and encoders are written from the
# format definitions, not taken from a library.
# --------------------------------------------------------------------------

def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64.  bf16 is the top half of an
    IEEE binary32, so widening the bits by 16 zero bits gives the exact value."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even) and
    return them as float64.  bf16 keeps 8 significant bits; below the smallest
    normal (2**-126) the quantum is fixed at 2**-133."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2**e with 0.5 <= |m| < 1
    e = np.maximum(e - 1, -126)              # exponent of the leading bit
    quantum = np.ldexp(1.0, e - 7)
    return np.rint(x / quantum) * quantum    # np.rint rounds half to even


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), round to nearest even."""
    r = round_to_bf16(x).astype(np.float32)  # exact: r has 8 significant bits
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
# no infinities; S.1111.111 is NaN; largest finite value 448 = 1.75 * 2**8;
# exponent field 0 holds subnormals m/8 * 2**-6.
E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = np.ldexp(1.0 + man / 8.0, exp - 7)
    sub = np.ldexp(man / 8.0, -6)
    val = np.where(exp == 0, sub, normal)
    val = np.where((exp == 0xF) & (man == 0x7), np.nan, val)
    return sign * val


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even, saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, e = np.frexp(a)
    e = np.maximum(e - 1, -6)                # subnormal quantum is 2**-9
    quantum = np.ldexp(1.0, e - 3)           # 4 significant bits
    r = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float64 -> E4M3 codes (uint8), round to nearest even, saturating."""
    r = round_to_e4m3(x)
    a = np.abs(r)
    _, e = np.frexp(a)
    e = e - 1
    is_sub = a < 2.0 ** -6
    exp_field = np.where(is_sub, 0, e + 7)
    man = np.where(is_sub, a / 2.0 ** -9, (a / np.ldexp(1.0, e) - 1.0) * 8.0)
    man = np.where(a == 0, 0, man)
    exp_field = np.where(a == 0, 0, exp_field)
    code = (exp_field.astype(np.int64) << 3) | np.rint(man).astype(np.int64)
    code = code | np.where(np.signbit(r), 0x80, 0)
    return code.astype(np.uint8)


def decode(codes: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_decode(codes) if dtype == "bf16" else e4m3_decode(codes)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_to_bf16(x) if dtype == "bf16" else round_to_e4m3(x)


# --------------------------------------------------------------------------
# (0) Latent-cache write -- "mla_prefill_decode_graph_bf16", Args freqs_cis
# ("precomputed RoPE frequency values", [max_seq_len, qk_rope_head_dim]),
# kv_norm_gamma (RMSNorm weights, [kv_lora_rank]), epsilon, kv_collection.
# Upstream of the plan: every new token's latent row is normalised, its rope
# part rotated, and the row stored in the paged cache at the token's position;
# the rope part of every query head is rotated with the same frequencies.
# --------------------------------------------------------------------------

def rms_norm(x, gamma, eps: float):
    """RMSNorm over the last axis: x / sqrt(mean(x**2) + eps) * gamma."""
    x = np.asarray(x, dtype=np.float64)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * np.asarray(gamma, dtype=np.float64)


def rope_rotate(x, freqs):
    """Rotate rope values by a freqs_cis row.  Both hold 32 complex numbers as
    interleaved (real, imaginary) pairs; the result is their complex product,
    laid out the same way."""
    x = np.asarray(x, dtype=np.float64)
    f = np.asarray(freqs, dtype=np.float64)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * (f[..., 0::2] + 1j * f[..., 1::2])
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],), dtype=np.float64)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def latent_cache_write(kv_latent, q, kv_norm_gamma, freqs_cis, input_row_offsets, cache_lengths,
                       page_table, page_size: int, kv_cache_codes, epsilon: float,
                       dtype: str = "bf16", inv_scale: float = 1.0):
    """Write the new tokens' latent rows into the paged cache.

    New token ``i`` of sequence ``b`` (row ``input_row_offsets[b] + i`` of
    ``kv_latent`` and ``q``) sits at context position ``p = cache_lengths[b]
    + i``.  Its 576 latent values are 512 c_kv values, normalised with
    ``rms_norm(c_kv, kv_norm_gamma, epsilon)``, and 64 k_rope values, rotated
    with ``rope_rotate(k_rope, freqs_cis[p])``.  The row, times ``inv_scale``
    and rounded to the cache's storage type, goes to page
    ``page_table[b, p // page_size]``, slot ``p % page_size``; every other cache
    row is left as it was.  The rope part (last 64 values) of every head of
    ``q[row]`` is rotated with the same ``freqs_cis[p]``.

    ``kv_latent`` and ``q`` are values (float), the cache is storage codes.
    Returns (cache codes after the write, rotated q as float64 or None,
    status: 0, STATUS_BAD_OFFSETS for decreasing offsets or a position past
    freqs_cis, STATUS_BAD_PAGE for a missing page).
    """
    lat = np.asarray(kv_latent, dtype=np.float64)
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    cache = np.asarray(cache_lengths, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    freqs = np.asarray(freqs_cis, dtype=np.float64)
    kv = np.array(kv_cache_codes, copy=True)
    q_out = None if q is None else np.array(q, dtype=np.float64, copy=True)
    encode = bf16_encode if dtype == "bf16" else e4m3_encode
    status = STATUS_OK
    for b in range(cache.shape[0]):
        n_new = int(iro[b + 1] - iro[b])
        if n_new < 0:
            status = STATUS_BAD_OFFSETS
            continue
        for i in range(n_new):
            t = int(iro[b]) + i
            p = int(cache[b]) + i
            if p >= freqs.shape[0]:
                status = STATUS_BAD_OFFSETS
                continue
            c_kv = rms_norm(lat[t, :R], kv_norm_gamma, epsilon)
            k_rope = rope_rotate(lat[t, R:], freqs[p])
            if q_out is not None:
                q_out[t, :, DN:] = rope_rotate(q_out[t, :, DN:], freqs[p])
            slot_page = p // page_size
            if slot_page >= pt.shape[1] or pt[b, slot_page] < 0 or pt[b, slot_page] >= kv.shape[0]:
                status = STATUS_BAD_PAGE
                continue
            kv[pt[b, slot_page], p % page_size] = encode(np.concatenate([c_kv, k_rope]) * inv_scale)
    return kv, q_out, status


# --------------------------------------------------------------------------
# (1) The chunk plan -- "mla_prefill_plan".
# --------------------------------------------------------------------------

def prefill_plan(input_row_offsets, cache_lengths, buffer_token_size: int, max_chunks: int):
    """Chunk plan of a ragged batch through a buffer of ``buffer_token_size`` rows.

    Follows the page's description: every sequence has cached tokens and new
    tokens; the total tokens are divided into chunks of ``buffer_token_size``;
    for each chunk the plan records, per sequence, where its rows start in the
    buffer (``buffer_row_offsets [max_chunks, B+1]``) and where they start in
    the cache (``cache_offsets [max_chunks, B]``), and the chunk's total valid
    rows (``buffer_lengths [max_chunks]``, -1 for an unused chunk).

    Returns (buffer_row_offsets, cache_offsets, buffer_lengths, status) as
    int64 arrays and an int status (0 ok, 1 more chunks needed than
    ``max_chunks``, 2 malformed ``input_row_offsets`` or total beyond int32).
    """
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    cache = np.asarray(cache_lengths, dtype=np.int64)
    B = cache.shape[0]
    S = int(buffer_token_size)
    if S <= 0 or max_chunks < 0 or iro.shape[0] != B + 1:
        raise ValueError("bad plan arguments")
    status = STATUS_OK
    new = iro[1:] - iro[:-1]
    if B + 1 > 0 and (iro[0] != 0 or np.any(new < 0)):
        status = STATUS_BAD_OFFSETS
        new = np.maximum(new, 0)
    total = cache + new                         # context tokens per sequence
    # Each sequence's slice of the packed token order.
    seq_start = np.zeros(B + 1, dtype=np.int64)
    seq_start[1:] = np.cumsum(total)
    tot = int(seq_start[B])
    if tot >= 2 ** 31 and status == STATUS_OK:
        status = STATUS_BAD_OFFSETS
    needed = -(-tot // S)
    if needed > max_chunks and status == STATUS_OK:
        status = STATUS_TOO_MANY_CHUNKS

    buffer_row_offsets = np.zeros((max_chunks, B + 1), dtype=np.int64)
    cache_offsets = np.zeros((max_chunks, B), dtype=np.int64)
    buffer_lengths = np.full(max_chunks, -1, dtype=np.int64)
    for c in range(max_chunks):
        win_lo, win_hi = c * S, (c + 1) * S     # this chunk's window of the packed order
        rows = 0
        for b in range(B):
            lo = max(int(seq_start[b]), win_lo)
            hi = min(int(seq_start[b + 1]), win_hi)
            buffer_row_offsets[c, b] = rows
            # Position (within sequence b) of its first token at or after the
            # window start; L_b once the sequence is done, 0 before it starts.
            cache_offsets[c, b] = min(max(win_lo - int(seq_start[b]), 0), int(total[b]))
            rows += max(hi - lo, 0)
        buffer_row_offsets[c, B] = rows
        buffer_lengths[c] = rows if win_lo < tot else -1
    return buffer_row_offsets, cache_offsets, buffer_lengths, status


# --------------------------------------------------------------------------
# (2) Latent gather -- "kv_input_fn" of mla_prefill_decode_graph_bf16 and the
# k_rope operand of flare_mla_prefill_dispatch.
# --------------------------------------------------------------------------

def gather_latent(kv_cache_codes, page_table, page_size: int, plan, chunk: int):
    """Copy chunk ``chunk``'s rows out of the paged cache.

    For each sequence ``b`` and each of its ``n`` rows in the chunk, buffer row
    ``buffer_row_offsets[chunk, b] + t`` receives the cache token at position
    ``cache_offsets[chunk, b] + t`` of sequence ``b``, which lives in page
    ``page_table[b, pos // page_size]`` at slot ``pos % page_size``.  The first
    512 values go to ``c_kv_buf``, the last 64 to ``k_rope_buf``.  Bit copy:
    the inputs are storage codes and so are the outputs.

    Returns (c_kv_buf [n, 512], k_rope_buf [n, 64], status).
    """
    bro, co, bl, _ = plan
    kv = np.asarray(kv_cache_codes)
    pt = np.asarray(page_table, dtype=np.int64)
    num_pages = kv.shape[0]
    n = int(bl[chunk])
    n = max(n, 0)
    c_kv = np.zeros((n, R), dtype=kv.dtype)
    k_rope = np.zeros((n, DR), dtype=kv.dtype)
    status = STATUS_OK
    B = bro.shape[1] - 1
    for b in range(B):
        r0, r1 = int(bro[chunk, b]), int(bro[chunk, b + 1])
        for t in range(r1 - r0):
            pos = int(co[chunk, b]) + t
            slot_page = pos // page_size
            if slot_page >= pt.shape[1] or pt[b, slot_page] < 0 or pt[b, slot_page] >= num_pages:
                status = STATUS_BAD_PAGE
                continue
            row = kv[pt[b, slot_page], pos % page_size]
            c_kv[r0 + t] = row[:R]
            k_rope[r0 + t] = row[R:]
    return c_kv, k_rope, status


def chunk_cache_rows(page_table, page_size: int, num_pages: int, plan, chunk: int,
                     buffer_token_size: int):
    """Where each buffer row of chunk ``chunk`` lives in the paged cache, the
    cache seen as ``num_pages * page_size`` consecutive rows: the lookup of
    ``gather_latent`` without the copy.  Buffer row ``buffer_row_offsets
    [chunk, b] + t`` of sequence ``b`` is context position ``cache_offsets
    [chunk, b] + t``, slot ``pos % page_size`` of page ``page_table[b, pos //
    page_size]``, i.e. row ``page * page_size + pos % page_size``.  Entries
    past the chunk's rows are 0, and so is the entry of a row whose page is
    out of range (status BAD_PAGE).

    Returns (rows [buffer_token_size] int64, status).
    """
    bro, co, bl, _ = plan
    pt = np.asarray(page_table, dtype=np.int64)
    rows = np.zeros(buffer_token_size, dtype=np.int64)
    status = STATUS_OK
    B = bro.shape[1] - 1
    for b in range(B):
        r0, r1 = int(bro[chunk, b]), int(bro[chunk, b + 1])
        for t in range(r1 - r0):
            pos = int(co[chunk, b]) + t
            slot_page = pos // page_size
            if slot_page >= pt.shape[1] or pt[b, slot_page] < 0 or pt[b, slot_page] >= num_pages:
                status = STATUS_BAD_PAGE
                continue
            rows[r0 + t] = pt[b, slot_page] * page_size + pos % page_size
    return rows, status


def context_latents(kv_cache_codes, page_table, page_size: int, total_lens):
    """All context tokens of every sequence, in position order, straight from
    the paged cache (no plan): a list of [L_b, 576] code arrays."""
    kv = np.asarray(kv_cache_codes)
    pt = np.asarray(page_table, dtype=np.int64)
    out = []
    for b, L in enumerate(total_lens):
        pos = np.arange(int(L))
        out.append(kv[pt[b, pos // page_size], pos % page_size])
    return out


# --------------------------------------------------------------------------
# (3) Up-projection -- mla_prefill_decode_graph_bf16, Args w_k and w_uv.
# --------------------------------------------------------------------------

def upproject(c_kv, w_k, w_uv, heads=None, store: str | None = None, inv_scale: float = 1.0):
    """Per-head K_nope and V from the latent.

    ``c_kv`` [rows, 512], ``w_k`` [H*128, 512], ``w_uv`` [H, 128, 512], all
    float64 real values.  For head h:  K_nope[:, h, :] = c_kv @ W_k,h^T with
    W_k,h = w_k[h*128:(h+1)*128], and V[:, h, :] = c_kv @ w_uv[h]^T.
    ``heads`` restricts the heads computed (the output keeps only those, in
    order).  With ``store`` set, each result is multiplied by ``inv_scale``,
    rounded to that storage type and multiplied back (the attention operands'
    dtype and descale).
    """
    c = np.asarray(c_kv, dtype=np.float64)
    H = w_uv.shape[0]
    hs = range(H) if heads is None else heads
    k = np.stack([c @ w_k[h * DN:(h + 1) * DN].T for h in hs], axis=1)
    v = np.stack([c @ w_uv[h].T for h in hs], axis=1)
    if store is not None:
        k = round_to(k * inv_scale, store) / inv_scale
        v = round_to(v * inv_scale, store) / inv_scale
    return k, v


# --------------------------------------------------------------------------
# (4) Causal attention with q_depth 192 -- flare_mla_prefill_dispatch.
# --------------------------------------------------------------------------

def softmax_weights(s):
    """Row softmax of a score matrix where -inf marks a masked entry.  Rows with
    no visible entry get all-zero weights and LSE -inf."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe)
    l = np.sum(p, axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        w = np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[..., 0] > 0, m_safe[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
    return w, lse


def partial_attention(q_nope, q_rope, k_nope, k_rope, v, q_pos, k_pos, scale):
    """Attention of query rows over one set of keys, causal by absolute position.

    q_nope [n,128], q_rope [n,64], k_nope [m,128], k_rope [m,64], v [m,128];
    q_pos [n], k_pos [m] absolute positions.  Score of query i and key j is
    scale * (q_nope_i . k_nope_j + q_rope_i . k_rope_j), visible iff
    k_pos[j] <= q_pos[i].  Returns (O [n,128] normalised, LSE [n]); a row with
    no visible key has O = 0 and LSE = -inf.
    """
    s = scale * (q_nope @ k_nope.T + q_rope @ k_rope.T)
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    s = np.where(visible, s, -np.inf)
    w, lse = softmax_weights(s)
    return w @ v, lse


def merge_partials(o_a, lse_a, o_b, lse_b):
    """Combine two attention results over disjoint key sets: with
    LSE = log(e^LSE_a + e^LSE_b), O = e^(LSE_a-LSE) O_a + e^(LSE_b-LSE) O_b."""
    m = np.maximum(lse_a, lse_b)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    ea = np.exp(lse_a - m_safe)
    eb = np.exp(lse_b - m_safe)
    tot = ea + eb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        wa = np.where(tot > 0, ea / np.where(tot > 0, tot, 1.0), 0.0)
        wb = np.where(tot > 0, eb / np.where(tot > 0, tot, 1.0), 0.0)
    return wa[..., None] * o_a + wb[..., None] * o_b, lse


def attention_reference(q, k_nope_ctx, k_rope_ctx, v_ctx, new_lens, cache_lens, scale,
                        heads=None, rows=None):
    """The definition, unchunked: for new token i of sequence b and head h,
    softmax over every context position j <= cache_len_b + i of
    scale * (q_nope . K_nope_h[j] + q_rope . k_rope[j]), applied to V_h.

    q [T_q, H, 192] float64 (real values); per sequence b: k_nope_ctx[b]
    [L_b, Hs, 128], k_rope_ctx[b] [L_b, 64], v_ctx[b] [L_b, Hs, 128] where Hs
    indexes ``heads`` (all heads when None).  ``rows`` optionally lists, per
    sequence, the new-token indices to evaluate.  Returns dicts keyed by
    (b, head) with (token_indices, O [n,128], LSE [n]).
    """
    H = q.shape[1]
    hs = list(range(H)) if heads is None else list(heads)
    iro = np.concatenate([[0], np.cumsum(new_lens)]).astype(np.int64)
    res = {}
    for b in range(len(new_lens)):
        n = int(new_lens[b])
        idx = np.arange(n) if rows is None else np.asarray(rows[b], dtype=np.int64)
        if idx.size == 0:
            continue
        L = int(cache_lens[b]) + n
        q_pos = int(cache_lens[b]) + idx
        k_pos = np.arange(L)
        for hi, h in enumerate(hs):
            qb = q[iro[b] + idx, h]
            o, lse = partial_attention(qb[:, :DN], qb[:, DN:], k_nope_ctx[b][:, hi],
                                       k_rope_ctx[b], v_ctx[b][:, hi], q_pos, k_pos, scale)
            res[(b, h)] = (iro[b] + idx, o, lse)
    return res


def attention_absorbed(q, c_kv_ctx, k_rope_ctx, w_uk, w_uv, new_lens, cache_lens, scale,
                       heads=None):
    """Absorbed form (mla_prefill_decode_graph_bf16, Args w_uk and w_uv): the
    nope query is projected into latent space by w_uk[h] [512,128], scored
    against the latent c_kv directly, the softmax-weighted latent is projected
    back by w_uv[h] [128,512].  Same result as up-projecting K and V first when
    w_uk[h] = W_k,h^T."""
    H = q.shape[1]
    hs = list(range(H)) if heads is None else list(heads)
    iro = np.concatenate([[0], np.cumsum(new_lens)]).astype(np.int64)
    res = {}
    for b in range(len(new_lens)):
        n = int(new_lens[b])
        if n == 0:
            continue
        L = int(cache_lens[b]) + n
        q_pos = int(cache_lens[b]) + np.arange(n)
        visible = np.arange(L)[None, :] <= q_pos[:, None]
        for h in hs:
            qb = q[iro[b]:iro[b + 1], h]
            q_lat = qb[:, :DN] @ w_uk[h].T               # [n, 512]
            s = scale * (q_lat @ c_kv_ctx[b].T + qb[:, DN:] @ k_rope_ctx[b].T)
            w, lse = softmax_weights(np.where(visible, s, -np.inf))
            o_lat = w @ c_kv_ctx[b]                      # [n, 512]
            res[(b, h)] = (np.arange(iro[b], iro[b + 1]), o_lat @ w_uv[h].T, lse)
    return res


# --------------------------------------------------------------------------
# The whole path, chunk by chunk, as the graph runs it.
# --------------------------------------------------------------------------

def attention_over_chunks(q, operands, plan, input_row_offsets, cache_lengths, scale,
                          heads=None, rows=None):
    """Chunk by chunk, as the prefill graph runs it: for every used chunk c of
    the plan, each sequence's new tokens attend to the sequence's keys in the
    chunk (buffer rows buffer_row_offsets[c,b] .. [c,b+1], at context positions
    cache_offsets[c,b] onward), and the result is merged into the running
    (O, LSE) of every query row.

    q [T_q, H, 192] real values; ``operands(c)`` returns the chunk's buffers
    (k_nope [n, Hs, 128], k_rope [n, 64], v [n, Hs, 128]) as real values, Hs
    indexing ``heads``.  Returns a dict keyed by (b, h) -> (tokens, O, LSE).
    """
    bro, co, bl, _ = plan
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    cache = np.asarray(cache_lengths, dtype=np.int64)
    new = iro[1:] - iro[:-1]
    B = cache.shape[0]
    H = q.shape[1]
    hs = list(range(H)) if heads is None else list(heads)
    sel = [np.arange(int(new[b])) if rows is None else np.asarray(rows[b], np.int64)
           for b in range(B)]
    acc = {}
    for b in range(B):
        for h in hs:
            n = sel[b].size
            acc[(b, h)] = (iro[b] + sel[b], np.zeros((n, DV)), np.full(n, -np.inf))
    for c in range(bl.shape[0]):
        if bl[c] < 0:
            continue
        k_nope, k_rope, v = operands(c)
        for b in range(B):
            r0, r1 = int(bro[c, b]), int(bro[c, b + 1])
            if r1 == r0 or sel[b].size == 0:
                continue
            k_pos = int(co[c, b]) + np.arange(r1 - r0)
            q_pos = int(cache[b]) + sel[b]
            for hi, h in enumerate(hs):
                qb = q[iro[b] + sel[b], h]
                o_c, lse_c = partial_attention(qb[:, :DN], qb[:, DN:], k_nope[r0:r1, hi],
                                               k_rope[r0:r1], v[r0:r1, hi], q_pos, k_pos, scale)
                tok, o_acc, lse_acc = acc[(b, h)]
                o_new, lse_new = merge_partials(o_acc, lse_acc, o_c, lse_c)
                acc[(b, h)] = (tok, o_new, lse_new)
    return acc


def mla_prefill(q_codes, kv_cache_codes, page_table, page_size, w_k_codes, w_uv_codes,
                input_row_offsets, cache_lengths, buffer_token_size, max_chunks, scale,
                dtype="bf16", q_scale=1.0, ckv_scale=1.0, w_scale=1.0,
                heads=None, rows=None):
    """The whole path: plan, then per chunk gather, up-project and attend,
    merging chunk results by LSE (``attention_over_chunks``).

    Inputs are storage codes (uint16 bf16 bits or uint8 e4m3 codes) plus
    per-tensor descales (real = stored * scale).  K and V are held in the
    storage dtype between the projection and the attention, in the cache's
    descale domain.  ``heads``/``rows`` restrict the output to a sample.

    Returns (out dict keyed by (b,h) -> (tokens, O [n,128], LSE [n]), plan).
    """
    plan = prefill_plan(input_row_offsets, cache_lengths, buffer_token_size, max_chunks)
    q = decode(q_codes, dtype) * q_scale
    H = q.shape[1]
    hs = list(range(H)) if heads is None else list(heads)
    w_k = decode(w_k_codes, dtype) * w_scale
    w_uv = decode(w_uv_codes, dtype) * w_scale

    def operands(c):
        c_kv_codes, k_rope_codes, _ = gather_latent(kv_cache_codes, page_table, page_size, plan, c)
        c_kv = decode(c_kv_codes, dtype) * ckv_scale
        k_rope = decode(k_rope_codes, dtype) * ckv_scale
        k_nope, v = upproject(c_kv, w_k, w_uv, heads=hs, store=dtype, inv_scale=1.0 / ckv_scale)
        return k_nope, k_rope, v

    acc = attention_over_chunks(q, operands, plan, input_row_offsets, cache_lengths, scale,
                                heads=hs, rows=rows)
    return acc, plan


# --------------------------------------------------------------------------
# (5) Decode branch -- "mla_prefill_decode_graph_bf16" (dispatches to decode by
# the batch's max sequence length; Args w_uk, w_uv, num_partitions_in).  The
# nope query is absorbed into latent space, attention runs over the 576-wide
# latent rows read straight from the paged cache, the keys are split into
# partitions whose partial results merge by LSE, and the latent result is
# projected back per head.
# --------------------------------------------------------------------------

def mla_decode(q, kv_cache_codes, page_table, page_size: int, w_uk, w_uv, input_row_offsets,
               cache_lengths, scale: float, num_partitions: int = 1, dtype: str = "bf16",
               ckv_scale: float = 1.0):
    """Decode attention in the absorbed form.

    ``q`` [T, H, 192], ``w_uk`` [H, 512, 128] and ``w_uv`` [H, 128, 512] are
    values; the cache is storage codes (real = stored * ``ckv_scale``).  New
    token i of sequence b (row ``input_row_offsets[b] + i``) at position
    p = cache_lengths[b] + i sees context positions 0..p.  Per head,
    q_lat = w_uk[h] q_nope scores the latent rows (score = scale * (q_lat .
    c_kv_j + q_rope . k_rope_j)); the p + 1 keys are cut into
    ``num_partitions`` contiguous ranges of ceil((p + 1) / num_partitions)
    keys (trailing ranges may be empty), each range gives a partial (latent O,
    LSE), and the partials merge in order with ``merge_partials``.  The merged
    latent O is projected by w_uv[h].

    Returns a dict (b, h) -> (tokens, out [n, 128], LSE [n]).
    """
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    cache = np.asarray(cache_lengths, dtype=np.int64)
    L = cache + (iro[1:] - iro[:-1])
    ctx = context_latents(kv_cache_codes, page_table, page_size, L)
    q = np.asarray(q, dtype=np.float64)
    H = q.shape[1]
    res = {}
    for b in range(cache.shape[0]):
        n = int(iro[b + 1] - iro[b])
        if n <= 0:
            continue
        lat = decode(ctx[b], dtype) * ckv_scale
        c_kv, k_rope = lat[:, :R], lat[:, R:]
        for h in range(H):
            out = np.zeros((n, DV))
            lses = np.zeros(n)
            for i in range(n):
                t = int(iro[b]) + i
                keys = int(cache[b]) + i + 1
                q_lat = np.asarray(w_uk[h], dtype=np.float64) @ q[t, h, :DN]
                s = scale * (c_kv[:keys] @ q_lat + k_rope[:keys] @ q[t, h, DN:])
                size = -(-keys // num_partitions)
                o, lse = np.zeros((1, R)), np.array([-np.inf])
                for k in range(num_partitions):
                    lo, hi = k * size, min((k + 1) * size, keys)
                    if lo >= hi:
                        o_k, lse_k = np.zeros((1, R)), np.array([-np.inf])
                    else:
                        w, lse_k = softmax_weights(s[None, lo:hi])
                        o_k = w @ c_kv[lo:hi]
                    o, lse = merge_partials(o, lse, o_k, lse_k)
                out[i] = np.asarray(w_uv[h], dtype=np.float64) @ o[0]
                lses[i] = lse[0]
            res[(b, h)] = (np.arange(iro[b], iro[b + 1]), out, lses)
    return res


# --------------------------------------------------------------------------
# (6) Sparse decode and attention sinks -- "mla_prefill_decode_graph_bf16"
# (Parameters sparse_mla, sparse_indices_stride; Args d_indices, packed int32
# physical KV row indices; indices_stride, the stride between batch rows;
# topk_lengths, the valid top-k count of each batch entry; attn_sink_ptr,
# per-batch attention sink weights).
# --------------------------------------------------------------------------

def mla_sparse_decode(q, kv_cache_codes, page_size: int, w_uk, w_uv, input_row_offsets, indices,
                      topk_lengths, scale: float, attn_sink=None, dtype: str = "bf16",
                      ckv_scale: float = 1.0):
    """Sparse decode in the absorbed form.

    ``indices`` [B, stride] int: physical cache rows, row = page * page_size +
    slot of the cache [num_pages, page_size, 576] viewed as rows; entry e of
    batch row b is used when e < topk_lengths[b] (all ``stride`` when
    ``topk_lengths`` is None).  Every new token of sequence b attends to
    exactly those rows (the list is per batch entry; no causal limit).  For
    head h, q_lat = w_uk[h] q_nope, score_e = scale * (q_lat . c_kv_e +
    q_rope . k_rope_e), out = w_uv[h] (sum_e softmax_e c_kv_e).

    ``attn_sink`` [B] (reading: one logit per batch entry, in the scaled-score
    domain): an extra entry of every softmax of sequence b that has no value
    row, so it only adds e^sink to the denominator; the LSE includes it.

    Returns a dict (b, h) -> (tokens, out [n, 128], LSE [n]).
    """
    iro = np.asarray(input_row_offsets, dtype=np.int64)
    idx = np.asarray(indices, dtype=np.int64)
    B = iro.shape[0] - 1
    stride = idx.shape[1]
    kv = np.asarray(kv_cache_codes)
    rows_all = kv.reshape(-1, kv.shape[-1])
    q = np.asarray(q, dtype=np.float64)
    H = q.shape[1]
    res = {}
    for b in range(B):
        n = int(iro[b + 1] - iro[b])
        if n <= 0:
            continue
        k = stride if topk_lengths is None else max(0, min(int(topk_lengths[b]), stride))
        lat = decode(rows_all[idx[b, :k]], dtype) * ckv_scale
        c_kv, k_rope = lat[:, :R], lat[:, R:]
        for h in range(H):
            out = np.zeros((n, DV))
            lses = np.zeros(n)
            for i in range(n):
                t = int(iro[b]) + i
                q_lat = np.asarray(w_uk[h], dtype=np.float64) @ q[t, h, :DN]
                s = scale * (c_kv @ q_lat + k_rope @ q[t, h, DN:])
                if attn_sink is not None:
                    s = np.concatenate([s, [float(attn_sink[b])]])
                if s.size == 0:   # nothing listed and no sink: no weights, LSE -inf
                    w, lse = np.zeros((1, 0)), np.array([-np.inf])
                else:
                    w, lse = softmax_weights(s[None, :])
                o = w[0, :k] @ c_kv if k > 0 else np.zeros(R)
                out[i] = np.asarray(w_uv[h], dtype=np.float64) @ o
                lses[i] = lse[0]
            res[(b, h)] = (np.arange(iro[b], iro[b + 1]), out, lses)
    return res


def causal_pairs(new_lens, cache_lens) -> int:
    """Number of visible (query, key) pairs: sum over b, i of cache_len_b + i + 1."""
    tot = 0
    for n, c in zip(new_lens, cache_lens):
        n, c = int(n), int(c)
        tot += n * c + n * (n + 1) // 2
    return tot


def attention_flops(new_lens, cache_lens, H) -> int:
    """Causal-effective attention flops: 2*H*(128+64+128) per visible pair."""
    return 2 * H * (DN + DR + DV) * causal_pairs(new_lens, cache_lens)
