"""Test-side helpers: build small paged caches from dense per-sequence K/V.

This is independent of both the oracle and the library: it places rows with
numpy fancy indexing so that dense library routines (torch's
scaled_dot_product_attention in fp64) can serve as the reference for the
oracle's paged gather.
"""

from __future__ import annotations

import numpy as np
import torch

BS = 16


def paged_from_dense(ks, vs, num_blocks, num_kv_heads, head_dim, rng, dtype=torch.float32,
                     fill=float("nan")):
    """Scatter per-sequence dense K/V ``[L_s, Hkv, d]`` into shuffled blocks.

    Returns (k_cache, v_cache, block_tables) with unused rows set to ``fill``.
    """
    S = len(ks)
    nblk = [(k.shape[0] + BS - 1) // BS for k in ks]
    assert sum(nblk) <= num_blocks
    perm = rng.permutation(num_blocks)
    kc = torch.full((num_blocks, num_kv_heads, BS, head_dim), fill, dtype=dtype)
    vc = torch.full_like(kc, fill)
    width = max(1, max(nblk) if nblk else 1)
    bt = torch.full((S, width), -1, dtype=torch.int32)
    off = 0
    for s in range(S):
        ids = perm[off: off + nblk[s]]
        off += nblk[s]
        bt[s, : nblk[s]] = torch.from_numpy(ids.astype(np.int32))
        L = ks[s].shape[0]
        for t in range(L):
            kc[ids[t // BS], :, t % BS, :] = ks[s][t]
            vc[ids[t // BS], :, t % BS, :] = vs[s][t]
    return kc, vc, bt


def sdpa_rows(q, k, v, scale, mask=None, is_causal=False):
    """torch fp64 SDPA for one sequence, GQA by repeating kv heads.

    q [n, Hq, d], k/v [L, Hkv, d] -> [n, Hq, d].
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    kk = k.double().repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
    vv = v.double().repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
    qq = q.double().transpose(0, 1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qq, kk, vv, attn_mask=mask, is_causal=is_causal, scale=scale)
    return o.transpose(0, 1)
