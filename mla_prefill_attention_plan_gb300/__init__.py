"""Python binding of libmla_prefill.so: ragged MLA prefill over a paged latent
KV cache on GB300 (sm_103a).

Argument marshalling only.  Each function has the name and argument order of
the C entry point declared in include/mla_prefill.h; tensors are passed as
device pointers (torch tensors on the GPU, or raw integer addresses), the
stream defaults to torch's current CUDA stream, and the C status code is
returned.  Every stage runs in the library's CUDA kernels; there is no other
implementation behind these names, and loading fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_prefill.so")

MLA_OK = 0
MLA_ERR_ARG = -1
MLA_ERR_GEOMETRY = -2
MLA_ERR_DTYPE = -3
MLA_ERR_LAUNCH = -4
MLA_ERR_WORKSPACE = -5
MLA_DEV_OK = 0
MLA_DEV_TOO_MANY_CHUNKS = 1
MLA_DEV_BAD_OFFSETS = 2
MLA_DEV_BAD_PAGE = 3
MLA_DEV_TIMEOUT = 4
MLA_BF16 = 0
MLA_E4M3 = 1

_P = ctypes.c_void_p
_I = ctypes.c_int32
_U = ctypes.c_uint32
_F = ctypes.c_float
_Z = ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/mla_prefill.h
SIGNATURES = {
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_abi_version": (_I, []),
    "mla_attention_kernel": (ctypes.c_char_p, [_I]),
    "mla_selftest_bounded_wait": (_I, [_P, _P, ctypes.c_int64, _I, _P]),
    "mla_prefill_plan": (_I, [_P, _P, _P, _P, _P, _I, _I, _U, _P, _P]),
    "mla_latent_cache_write": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                    _F, _F, _I, _P, _P]),
    "mla_gather_latent": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _U, _I, _P, _P]),
    "mla_upproject": (_I, [_P, _P, _P, _P, _P, _P, _I, _U, _I, _I, _F, _F, _F, _P, _P]),
    "mla_chunk_cache_rows": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _U, _P, _P]),
    "mla_upproject_paged": (_I, [_P, _P, _P, _P, _I, _P, _I, _U, _P, _P, _I, _I, _F, _F, _F, _P,
                                 _P]),
    "mla_prefill_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _I, _I, _I, _I, _I, _I, _U, _F, _F, _F, _F, _I, _P, _P]),
    "mla_prefill_attention_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                         _I, _I, _I, _I, _I, _I, _U, _F, _F, _F, _F, _I, _P, _P]),
    "mla_prefill_attention_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _I, _I, _I, _I, _I, _I, _U, _F, _F, _F, _F, _I, _P,
                                           _P]),
    "mla_prefill_workspace_bytes": (_Z, [_I, _I, _I, _I, _U, _I]),
    "mla_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _I, _U, _I,
                         _F, _F, _F, _F, _I, _P, _Z, _P, _P]),
    "mla_decode_partitions": (_I, [_I, _I, _I, _I]),
    "mla_decode_workspace_bytes": (_Z, [_I, _I, _I]),
    "mla_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                        _F, _P, _I, _P, _P, _I, _P, _Z, _P, _P]),
}

_lib = None


class MLAError(RuntimeError):
    pass


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise MLAError(f"{path} is missing: build it with "
                           "`python -m mla_prefill_attention_plan_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(code: int) -> str:
    return load().mla_status_string(code).decode()


def check(code: int) -> None:
    if code != MLA_OK:
        raise MLAError(f"{code}: {status_string(code)}")


def mla_abi_version() -> int:
    return load().mla_abi_version()


def mla_attention_kernel(dtype) -> str:
    """Which attention kernel a call with `dtype` launches on the current device."""
    r = load().mla_attention_kernel(dtype)
    return r.decode() if r is not None else None


def mla_selftest_bounded_wait(d_status, d_elapsed_ns, limit_ns, cluster_size, stream=None) -> int:
    """Launch the bounded-wait self-test (see include/mla_prefill.h)."""
    return load().mla_selftest_bounded_wait(_ptr(d_status), _ptr(d_elapsed_ns), int(limit_ns),
                                            cluster_size, _stream(stream))


def mla_prefill_plan(buffer_row_offsets, cache_offsets, buffer_lengths, input_row_offsets,
                     cache_lengths, batch_size, max_chunks, buffer_token_size, d_status=None,
                     stream=None) -> int:
    return load().mla_prefill_plan(_ptr(buffer_row_offsets), _ptr(cache_offsets),
                                   _ptr(buffer_lengths), _ptr(input_row_offsets),
                                   _ptr(cache_lengths), batch_size, max_chunks,
                                   buffer_token_size, _ptr(d_status), _stream(stream))


def mla_latent_cache_write(kv_cache, q, kv_latent, kv_norm_gamma, freqs_cis, input_row_offsets,
                           cache_lengths, page_table, num_pages, page_size, max_pages_per_seq,
                           batch_size, num_heads, total_q_tokens, max_seq_len, epsilon,
                           kv_inv_scale, dtype, d_status=None, stream=None) -> int:
    return load().mla_latent_cache_write(_ptr(kv_cache), _ptr(q), _ptr(kv_latent),
                                         _ptr(kv_norm_gamma), _ptr(freqs_cis),
                                         _ptr(input_row_offsets), _ptr(cache_lengths),
                                         _ptr(page_table), num_pages, page_size,
                                         max_pages_per_seq, batch_size, num_heads,
                                         total_q_tokens, max_seq_len, epsilon, kv_inv_scale,
                                         dtype, _ptr(d_status), _stream(stream))


def mla_gather_latent(c_kv_buf, k_rope_buf, kv_cache, page_table, num_pages, page_size,
                      max_pages_per_seq, buffer_row_offsets, cache_offsets, buffer_lengths, chunk,
                      batch_size, buffer_token_size, dtype, d_status=None, stream=None) -> int:
    return load().mla_gather_latent(_ptr(c_kv_buf), _ptr(k_rope_buf), _ptr(kv_cache),
                                    _ptr(page_table), num_pages, page_size, max_pages_per_seq,
                                    _ptr(buffer_row_offsets), _ptr(cache_offsets),
                                    _ptr(buffer_lengths), chunk, batch_size, buffer_token_size,
                                    dtype, _ptr(d_status), _stream(stream))


def mla_upproject(k_nope, v, c_kv_buf, w_k, w_uv, buffer_lengths, chunk, buffer_token_size,
                  num_heads, dtype, ckv_scale=1.0, w_scale=1.0, kv_out_inv_scale=1.0,
                  d_status=None, stream=None) -> int:
    return load().mla_upproject(_ptr(k_nope), _ptr(v), _ptr(c_kv_buf), _ptr(w_k), _ptr(w_uv),
                                _ptr(buffer_lengths), chunk, buffer_token_size, num_heads, dtype,
                                ckv_scale, w_scale, kv_out_inv_scale, _ptr(d_status),
                                _stream(stream))


def mla_chunk_cache_rows(cache_rows, page_table, num_pages, page_size, max_pages_per_seq,
                         buffer_row_offsets, cache_offsets, buffer_lengths, max_chunks, batch_size,
                         buffer_token_size, d_status=None, stream=None) -> int:
    return load().mla_chunk_cache_rows(_ptr(cache_rows), _ptr(page_table), num_pages, page_size,
                                       max_pages_per_seq, _ptr(buffer_row_offsets),
                                       _ptr(cache_offsets), _ptr(buffer_lengths), max_chunks,
                                       batch_size, buffer_token_size, _ptr(d_status),
                                       _stream(stream))


def mla_upproject_paged(k_nope, v, kv_cache, cache_rows, num_cache_rows, buffer_lengths, chunk,
                        buffer_token_size, w_k, w_uv, num_heads, dtype=MLA_BF16, ckv_scale=1.0,
                        w_scale=1.0, kv_out_inv_scale=1.0, d_status=None, stream=None) -> int:
    return load().mla_upproject_paged(_ptr(k_nope), _ptr(v), _ptr(kv_cache), _ptr(cache_rows),
                                      num_cache_rows, _ptr(buffer_lengths), chunk,
                                      buffer_token_size, _ptr(w_k), _ptr(w_uv), num_heads, dtype,
                                      ckv_scale, w_scale, kv_out_inv_scale, _ptr(d_status),
                                      _stream(stream))


def mla_prefill_attention(out, lse, o_acc, lse_acc, q, k_nope, v, k_rope, input_row_offsets,
                          cache_lengths, buffer_row_offsets, cache_offsets, buffer_lengths, chunk,
                          max_chunks, batch_size, num_heads, max_prompt_len, total_q_tokens,
                          buffer_token_size, scale, q_scale=1.0, k_scale=1.0, v_scale=1.0,
                          dtype=MLA_BF16, d_status=None, stream=None) -> int:
    return load().mla_prefill_attention(
        _ptr(out), _ptr(lse), _ptr(o_acc), _ptr(lse_acc), _ptr(q), _ptr(k_nope), _ptr(v),
        _ptr(k_rope), _ptr(input_row_offsets), _ptr(cache_lengths), _ptr(buffer_row_offsets),
        _ptr(cache_offsets), _ptr(buffer_lengths), chunk, max_chunks, batch_size, num_heads,
        max_prompt_len, total_q_tokens, buffer_token_size, scale, q_scale, k_scale, v_scale,
        dtype, _ptr(d_status), _stream(stream))


def mla_prefill_attention_paged(out, lse, o_acc, lse_acc, q, k_nope, v, kv_cache, cache_rows,
                                num_cache_rows, input_row_offsets, cache_lengths,
                                buffer_row_offsets, cache_offsets, buffer_lengths, chunk,
                                max_chunks, batch_size, num_heads, max_prompt_len, total_q_tokens,
                                buffer_token_size, scale, q_scale=1.0, k_scale=1.0, v_scale=1.0,
                                dtype=MLA_BF16, d_status=None, stream=None) -> int:
    return load().mla_prefill_attention_paged(
        _ptr(out), _ptr(lse), _ptr(o_acc), _ptr(lse_acc), _ptr(q), _ptr(k_nope), _ptr(v),
        _ptr(kv_cache), _ptr(cache_rows), num_cache_rows, _ptr(input_row_offsets),
        _ptr(cache_lengths), _ptr(buffer_row_offsets), _ptr(cache_offsets), _ptr(buffer_lengths),
        chunk, max_chunks, batch_size, num_heads, max_prompt_len, total_q_tokens,
        buffer_token_size, scale, q_scale, k_scale, v_scale, dtype, _ptr(d_status),
        _stream(stream))


MLA_NOALLOC_MAX_ROWS = 32768


def mla_prefill_attention_noalloc(out, lse, q, k_nope, v, k_rope, input_row_offsets,
                                  cache_lengths, buffer_row_offsets, cache_offsets,
                                  buffer_lengths, chunk, max_chunks, batch_size, num_heads,
                                  max_prompt_len, total_q_tokens, buffer_token_size, scale,
                                  q_scale=1.0, k_scale=1.0, v_scale=1.0, dtype=MLA_BF16,
                                  d_status=None, stream=None) -> int:
    """mla_prefill_attention without caller scratch: the cross-chunk merge
    state lives in a fixed array inside the library, for callers that cannot
    allocate device memory.  See include/mla_prefill.h for the limits."""
    return load().mla_prefill_attention_noalloc(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_nope), _ptr(v), _ptr(k_rope),
        _ptr(input_row_offsets), _ptr(cache_lengths), _ptr(buffer_row_offsets),
        _ptr(cache_offsets), _ptr(buffer_lengths), chunk, max_chunks, batch_size, num_heads,
        max_prompt_len, total_q_tokens, buffer_token_size, scale, q_scale, k_scale, v_scale,
        dtype, _ptr(d_status), _stream(stream))


def mla_prefill_workspace_bytes(batch_size, num_heads, total_q_tokens, max_chunks,
                                buffer_token_size, dtype) -> int:
    return load().mla_prefill_workspace_bytes(batch_size, num_heads, total_q_tokens, max_chunks,
                                              buffer_token_size, dtype)


def mla_prefill(out, lse, q, input_row_offsets, cache_lengths, kv_cache, page_table, num_pages,
                page_size, max_pages_per_seq, w_k, w_uv, batch_size, num_heads, total_q_tokens,
                max_prompt_len, buffer_token_size, max_chunks, scale, q_scale=1.0, ckv_scale=1.0,
                w_scale=1.0, dtype=MLA_BF16, workspace=None, workspace_bytes=0, d_status=None,
                stream=None) -> int:
    return load().mla_prefill(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(input_row_offsets), _ptr(cache_lengths),
        _ptr(kv_cache), _ptr(page_table), num_pages, page_size, max_pages_per_seq, _ptr(w_k),
        _ptr(w_uv), batch_size, num_heads, total_q_tokens, max_prompt_len, buffer_token_size,
        max_chunks, scale, q_scale, ckv_scale, w_scale, dtype, _ptr(workspace),
        workspace_bytes, _ptr(d_status), _stream(stream))


def mla_decode_partitions(batch_size, num_heads, max_new_tokens, max_keys) -> int:
    return load().mla_decode_partitions(batch_size, num_heads, max_new_tokens, max_keys)


def mla_decode_workspace_bytes(num_heads, total_q_tokens, num_partitions) -> int:
    return load().mla_decode_workspace_bytes(num_heads, total_q_tokens, num_partitions)


def mla_decode(out, lse, q, input_row_offsets, cache_lengths, kv_cache, page_table, num_pages,
               page_size, max_pages_per_seq, w_uk, w_uv, batch_size, num_heads, total_q_tokens,
               max_new_tokens, max_seq_len, num_partitions, scale, d_indices=None, indices_stride=0,
               topk_lengths=None, attn_sink=None, dtype=MLA_BF16, workspace=None,
               workspace_bytes=0, d_status=None, stream=None) -> int:
    return load().mla_decode(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(input_row_offsets), _ptr(cache_lengths),
        _ptr(kv_cache), _ptr(page_table), num_pages, page_size, max_pages_per_seq, _ptr(w_uk),
        _ptr(w_uv), batch_size, num_heads, total_q_tokens, max_new_tokens, max_seq_len,
        num_partitions, scale,
        _ptr(d_indices), indices_stride, _ptr(topk_lengths), _ptr(attn_sink), dtype,
        _ptr(workspace), workspace_bytes, _ptr(d_status), _stream(stream))


__all__ = [n for n in SIGNATURES] + ["load", "check", "status_string", "MLAError", "LIB_PATH"]
