"""Planted mistakes in the oracle (CPU only): each plausible slip -- an
off-by-one mask, a dropped rope term, a wrong weight slice, a shifted cache
offset, swapped merge weights -- must make at least one pin fail."""
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as M
import test_oracle_pins as P


def _plant(monkeypatch, name, fn):
    """Replace an oracle function in the module and in the package namespace."""
    monkeypatch.setattr(M, name, fn)
    if hasattr(P.O, name):
        monkeypatch.setattr(P.O, name, fn)


def _must_fail(*pins):
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, "a planted mistake went unnoticed"


def test_strict_causal_mask_is_caught(monkeypatch):
    orig = M.partial_attention

    def strict(q_nope, q_rope, k_nope, k_rope, v, q_pos, k_pos, scale):
        return orig(q_nope, q_rope, k_nope, k_rope, v, np.asarray(q_pos) - 1, k_pos, scale)
    _plant(monkeypatch, "partial_attention", strict)
    _must_fail(P.test_attention_bruteforce_tiny, P.test_attention_closed_forms)


def test_dropped_rope_term_is_caught(monkeypatch):
    orig = M.partial_attention

    def no_rope(q_nope, q_rope, k_nope, k_rope, v, q_pos, k_pos, scale):
        return orig(q_nope, 0 * q_rope, k_nope, k_rope, v, q_pos, k_pos, scale)
    _plant(monkeypatch, "partial_attention", no_rope)
    _must_fail(P.test_attention_bruteforce_tiny)


def test_wrong_weight_slice_is_caught(monkeypatch):
    def bad(c_kv, w_k, w_uv, heads=None, store=None, inv_scale=1.0):
        c = np.asarray(c_kv, dtype=np.float64)
        H = w_uv.shape[0]
        hs = range(H) if heads is None else heads
        k = np.stack([c @ w_k[h::H][:M.DN].T for h in hs], axis=1)     # strided, not blocked
        v = np.stack([c @ w_uv[h].T for h in hs], axis=1)
        return k, v
    _plant(monkeypatch, "upproject", bad)
    _must_fail(P.test_upproject_bruteforce)


def test_transposed_value_weight_is_caught(monkeypatch):
    def bad(c_kv, w_k, w_uv, heads=None, store=None, inv_scale=1.0):
        c = np.asarray(c_kv, dtype=np.float64)
        H = w_uv.shape[0]
        hs = range(H) if heads is None else heads
        k = np.stack([c @ w_k[h * M.DN:(h + 1) * M.DN].T for h in hs], axis=1)
        flat = w_uv.reshape(H * M.DV, M.R)
        v = np.stack([c @ flat[h::H].T for h in hs], axis=1)           # heads interleaved
        return k, v
    _plant(monkeypatch, "upproject", bad)
    _must_fail(P.test_upproject_bruteforce)


def test_shifted_cache_offset_is_caught(monkeypatch):
    orig = M.prefill_plan

    def shifted(*a, **k):
        bro, co, bl, st = orig(*a, **k)
        co = co.copy()
        co[1:] = np.maximum(co[1:] - 1, 0)
        return bro, co, bl, st
    _plant(monkeypatch, "prefill_plan", shifted)
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    _must_fail(lambda: P.test_plan_hand_worked_tiny_ragged(golden),
               P.test_plan_matches_token_walk_random)


def test_swapped_merge_weights_are_caught(monkeypatch):
    orig = M.merge_partials

    def swapped(o_a, lse_a, o_b, lse_b):
        o, lse = orig(o_a, lse_a, o_b, lse_b)
        o2, _ = orig(o_b, lse_a, o_a, lse_b)
        return o2, lse
    _plant(monkeypatch, "merge_partials", swapped)
    _must_fail(P.test_merge_split_equals_one_shot,
               lambda: P.test_chunked_pipeline_equals_unchunked(32))


def test_unscaled_scores_are_caught(monkeypatch):
    orig = M.partial_attention

    def unscaled(q_nope, q_rope, k_nope, k_rope, v, q_pos, k_pos, scale):
        return orig(q_nope, q_rope, k_nope, k_rope, v, q_pos, k_pos, 1.0)
    _plant(monkeypatch, "partial_attention", unscaled)
    _must_fail(P.test_attention_bruteforce_tiny, P.test_attention_closed_forms)


def test_epsilon_outside_the_root_is_caught(monkeypatch):
    def bad(x, gamma, eps):
        x = np.asarray(x, dtype=np.float64)
        return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * np.asarray(gamma)
    _plant(monkeypatch, "rms_norm", bad)
    _must_fail(P.test_rms_norm_closed_forms_and_library)


def test_sum_instead_of_mean_is_caught(monkeypatch):
    def bad(x, gamma, eps):
        x = np.asarray(x, dtype=np.float64)
        return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma)
    _plant(monkeypatch, "rms_norm", bad)
    _must_fail(P.test_rms_norm_closed_forms_and_library, P.test_cache_write_round_trip_through_cache)


def test_conjugate_rotation_is_caught(monkeypatch):
    orig = M.rope_rotate

    def conj(x, freqs):
        f = np.array(freqs, dtype=np.float64, copy=True)
        f[..., 1::2] *= -1
        return orig(x, f)
    _plant(monkeypatch, "rope_rotate", conj)
    _must_fail(P.test_rope_rotation_special_cases)


def test_half_split_rope_layout_is_caught(monkeypatch):
    def half(x, freqs):
        x = np.asarray(x, dtype=np.float64)
        f = np.asarray(freqs, dtype=np.float64)
        z = (x[..., :32] + 1j * x[..., 32:]) * (f[..., 0::2] + 1j * f[..., 1::2])
        return np.concatenate([z.real, z.imag], axis=-1)
    _plant(monkeypatch, "rope_rotate", half)
    _must_fail(P.test_rope_rotation_special_cases)


def test_position_off_by_one_is_caught(monkeypatch):
    orig = M.latent_cache_write

    def shifted(kv_latent, q, gamma, freqs, iro, cache_lengths, *a, **k):
        return orig(kv_latent, q, gamma, np.asarray(freqs)[1:], iro, cache_lengths, *a, **k)
    _plant(monkeypatch, "latent_cache_write", shifted)
    _must_fail(P.test_cache_write_round_trip_through_cache, P.test_cache_write_page_permutation_and_e4m3)


def test_gather_slot_off_by_one_is_caught(monkeypatch):
    """A cache row read one slot later than its position: the rows encode
    (sequence, position, column), so the construction pin sees it."""
    orig = M.gather_latent

    def shifted(kv_cache_codes, page_table, page_size, plan, chunk):
        kv = np.asarray(kv_cache_codes)
        rolled = np.roll(kv.reshape(-1, kv.shape[-1]), -1, axis=0).reshape(kv.shape)
        return orig(rolled, page_table, page_size, plan, chunk)
    _plant(monkeypatch, "gather_latent", shifted)
    _must_fail(P.test_gather_by_construction)


def test_bf16_truncation_is_caught(monkeypatch):
    """Rounding toward zero instead of to nearest even."""
    def trunc(x):
        x = np.asarray(x, dtype=np.float64)
        _, e = np.frexp(x)
        q = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
        return np.trunc(x / q) * q
    monkeypatch.setattr(M, "round_to_bf16", trunc)
    _must_fail(P.test_bf16_codec_against_torch)


def test_e4m3_ties_away_from_zero_is_caught(monkeypatch):
    """Ties rounded away from zero instead of to even."""
    def away(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.minimum(np.abs(x), M.E4M3_MAX)
        _, e = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
        r = np.minimum(np.floor(a / q + 0.5) * q, M.E4M3_MAX)
        return np.copysign(r, x)
    monkeypatch.setattr(M, "round_to_e4m3", away)
    _must_fail(P.test_e4m3_codec_against_torch, P.test_e4m3_spec_values)


def test_log2_lse_is_caught(monkeypatch):
    """The log-sum-exp in base 2 instead of the natural log."""
    orig = M.softmax_weights

    def log2(s):
        w, lse = orig(s)
        return w, lse / math.log(2.0)
    _plant(monkeypatch, "softmax_weights", log2)
    _must_fail(P.test_attention_closed_forms, P.test_merge_split_equals_one_shot)


def test_partials_averaged_instead_of_merged_is_caught(monkeypatch):
    """Partition results averaged instead of weighted by their LSE."""
    def average(o_a, lse_a, o_b, lse_b):
        fa, fb = np.isfinite(lse_a), np.isfinite(lse_b)
        o = np.where((fa & fb)[..., None], 0.5 * (o_a + o_b), np.where(fa[..., None], o_a, o_b))
        return o, np.logaddexp(lse_a, lse_b)
    monkeypatch.setattr(M, "merge_partials", average)
    _must_fail(P.test_decode_partition_count_invariant)


def test_sink_left_out_of_the_output_is_caught(monkeypatch):
    """The sink enters the LSE but the output is normalised over the listed
    rows only (as if the sink had no place in the denominator)."""
    orig = M.mla_sparse_decode

    def bad(q, kv, ps, w_uk, w_uv, iro, idx, topk, scale, attn_sink=None, dtype="bf16", ckv_scale=1.0):
        res = orig(q, kv, ps, w_uk, w_uv, iro, idx, topk, scale, None, dtype, ckv_scale)
        if attn_sink is None:
            return res
        with_sink = orig(q, kv, ps, w_uk, w_uv, iro, idx, topk, scale, attn_sink, dtype, ckv_scale)
        return {k: (v[0], v[1], with_sink[k][2]) for k, v in res.items()}
    _plant(monkeypatch, "mla_sparse_decode", bad)
    _must_fail(P.test_attention_sink_closed_forms)


def test_causal_limit_on_sparse_lists_is_caught(monkeypatch):
    """A causal limit applied to the positions of a sparse list (new token i
    keeping only the first i + 1 entries) instead of using the whole list."""
    orig = M.mla_sparse_decode

    def bad(q, kv, ps, w_uk, w_uv, iro, idx, topk, scale, attn_sink=None, dtype="bf16", ckv_scale=1.0):
        iro = np.asarray(iro)
        res = {}
        for b in range(len(iro) - 1):
            for i in range(int(iro[b + 1] - iro[b])):
                t = int(iro[b]) + i
                sub = np.asarray([0, 1])
                keep = np.asarray(idx)[b:b + 1, :i + 1]
                one = orig(q[t:t + 1], kv, ps, w_uk, w_uv, sub, keep, None, scale,
                           None if attn_sink is None else np.asarray(attn_sink)[b:b + 1], dtype, ckv_scale)
                for (_, h), (_, o, l) in one.items():
                    tok, out, lse = res.get((b, h), (np.arange(iro[b], iro[b + 1]),
                                                     np.zeros((iro[b + 1] - iro[b], M.DV)),
                                                     np.zeros(iro[b + 1] - iro[b])))
                    out[i], lse[i] = o[0], l[0]
                    res[(b, h)] = (tok, out, lse)
        return res
    _plant(monkeypatch, "mla_sparse_decode", bad)
    _must_fail(P.test_sparse_decode_over_the_whole_context_equals_dense_decode,
               P.test_sparse_decode_is_a_set_and_ignores_entries_past_topk)


def test_cache_row_table_slips_are_caught(monkeypatch):
    """Two slips in the cache-row table: the page's first row for every slot
    (the slot within the page dropped), and the buffer row's index used as
    the context position (the chunk's cache offset dropped)."""
    orig = M.chunk_cache_rows

    def page_start_only(page_table, page_size, num_pages, plan, chunk, buffer_token_size):
        rows, st = orig(page_table, page_size, num_pages, plan, chunk, buffer_token_size)
        return rows - rows % page_size, st
    _plant(monkeypatch, "chunk_cache_rows", page_start_only)
    _must_fail(P.test_chunk_cache_rows_by_construction, P.test_chunk_cache_rows_identity_pages)

    def no_cache_offset(page_table, page_size, num_pages, plan, chunk, buffer_token_size):
        bro, co, bl, extra = plan
        return orig(page_table, page_size, num_pages, (bro, np.zeros_like(co), bl, extra), chunk,
                    buffer_token_size)
    _plant(monkeypatch, "chunk_cache_rows", no_cache_offset)
    _must_fail(P.test_chunk_cache_rows_by_construction, P.test_chunk_cache_rows_identity_pages)
