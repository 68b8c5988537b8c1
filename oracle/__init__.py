"""CPU oracle for ragged MLA prefill (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library and its binding never do.
"""
import numpy as np

from .mla_oracle import *  # noqa: F401,F403
from .mla_oracle import (attention_over_chunks, attention_reference, attention_absorbed,  # noqa: F401
                         chunk_cache_rows, context_latents, latent_cache_write, rms_norm,
                         rope_rotate,
                         decode, gather_latent, merge_partials, mla_decode, mla_prefill,
                         mla_sparse_decode,
                         partial_attention, prefill_plan, upproject)


def codes(t) -> np.ndarray:
    """Storage codes of a CPU tensor: uint16 bits for bfloat16, uint8 codes
    for float8_e4m3fn, the integer values otherwise."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()
