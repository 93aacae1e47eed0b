"""The roofline's algorithmic counts (`accounting.py`) against brute force:
the causal (query, key) pairs of a chunk counted one by one, the prefill
flops of the mixed-step chunks, and the decode bytes summed token by token
from the per-token ledger (K and V rows of every kv head)."""

import numpy as np
import torch

from paged_kv_cache_297_gb300 import accounting
from paged_kv_cache_297_gb300 import workloads as W


def test_causal_pairs_match_enumeration():
    rng = np.random.Generator(np.random.PCG64(4))
    for _ in range(50):
        prior, n = int(rng.integers(0, 300)), int(rng.integers(0, 200))
        # query j (absolute position prior + j) sees keys 0 .. prior + j
        brute = sum(1 for j in range(n) for k in range(prior + n) if k <= prior + j)
        assert accounting.causal_pairs(prior, n) == brute


def test_prefill_flops_of_the_mixed_step_chunks():
    b = W.make_batch("mixed_step", poison=False)
    cu = b.prefill_cu_q_lens.tolist()
    L = b.prefill_context_lens.tolist()
    assert [cu[i + 1] - cu[i] for i in range(len(L))] == [512, 512]
    assert [L[i] - (cu[i + 1] - cu[i]) for i in range(len(L))] == [0, 3072]
    # chunk of 512 from scratch: 512 * 513 / 2 pairs; after 3072 tokens:
    # 512 * 3072 more; 1,835,520 pairs per head in all
    pairs = 512 * 513 // 2 + (512 * 3072 + 512 * 513 // 2)
    assert pairs == 1_835_520
    Hq, d = b.prefill_q.shape[1], b.prefill_q.shape[2]
    assert accounting.prefill_flops(b.prefill_cu_q_lens, b.prefill_context_lens, Hq, d) == 4 * d * Hq * pairs
    assert 4 * d * Hq * pairs == 30_073_159_680


def test_decode_bytes_sum_the_per_token_ledger():
    lens = torch.tensor([1, 15, 16, 17, 1000], dtype=torch.int32)
    Hq, Hkv, d = 32, 8, 128
    for elem, q_elem in ((2, None), (1, 2)):
        got = accounting.decode_bytes(lens, Hq, Hkv, d, elem, 2, q_elem)
        kv = sum(2 * Hkv * d * elem for L in lens.tolist() for _ in range(L))
        qo = len(lens) * Hq * d * ((q_elem or elem) + 2)
        tables = sum(4 * -(-L // 16) + 4 for L in lens.tolist())
        assert got == {"kv": kv, "q_out": qo, "tables": tables, "total": kv + qo + tables}


def test_append_and_copy_bytes():
    # each appended token: K and V rows read once and written once, one slot id
    assert accounting.append_bytes(3, 8, 128, 2) == 3 * (2 * 2 * 8 * 128 * 2 + 8)
    # each pair: one K and one V block (16 rows of every kv head) read and written
    assert accounting.copy_blocks_bytes(2, 8, 128, 2) == 2 * (2 * 2 * 8 * 16 * 128 * 2 + 16)
