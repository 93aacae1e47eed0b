"""Host block manager (``pkv_bm_*``): allocation, reference counts,
copy-on-write, the prefix index and LRU eviction, then a long random
workload whose block tables, slot mappings and copy pairs drive the oracle's
append and copy: every live sequence must read back exactly the K/V rows of
its own token history through its table.  The last test runs the same flow
through the CUDA kernels.  All but that one run without a GPU."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_297_gb300 as pkv

BS = pkv.BLOCK_SIZE


def _table(bm, sid):
    t, n = bm.block_tables([sid])
    L = int(n[0])
    return [int(b) for b in t[0, : (L + BS - 1) // BS]], L


def test_allocation_slots_and_free():
    bm = pkv.BlockManager(16, 8, prefix_cache=False)
    assert bm.num_free_blocks() == (16, 0)
    assert bm.add_sequence(1, list(range(40))) == 0
    blocks, L = _table(bm, 1)
    assert L == 40 and len(blocks) == 3 and len(set(blocks)) == 3
    assert bm.num_free_blocks() == (13, 0)
    slots = bm.slots(1, 0, 40)
    assert slots.tolist() == [blocks[t // BS] * BS + t % BS for t in range(40)]
    t, _ = bm.block_tables([1])
    assert (t[0, 3:] == -1).all()
    bm.free_sequence(1)
    assert bm.num_free_blocks() == (16, 0)


def test_prefix_index_reuses_full_blocks_only():
    bm = pkv.BlockManager(32, 8)
    prompt = list(range(100, 148)) + [7, 8, 9]          # 3 full blocks + 3 tokens
    assert bm.add_sequence(1, prompt) == 0
    a, _ = _table(bm, 1)
    # the same 48-token prefix, then different tokens
    assert bm.add_sequence(2, prompt[:48] + [1, 2]) == 48
    b, _ = _table(bm, 2)
    assert b[:3] == a[:3] and b[3] != a[3]
    # a difference inside the second block stops the match after the first
    other = prompt[:20] + [0] + prompt[21:48]
    assert bm.add_sequence(3, other) == 16
    c, _ = _table(bm, 3)
    assert c[0] == a[0] and c[1] != a[1]
    # no index: nothing is found
    bm2 = pkv.BlockManager(32, 8, prefix_cache=False)
    bm2.add_sequence(1, prompt)
    assert bm2.add_sequence(2, prompt) == 0


def test_freed_registered_blocks_stay_cached_until_evicted():
    bm = pkv.BlockManager(6, 8)
    p = list(range(64))                                 # 4 full blocks
    bm.add_sequence(1, p)
    bm.free_sequence(1)
    assert bm.num_free_blocks() == (6, 4)               # all available, 4 of them cached
    assert bm.add_sequence(2, p) == 64                  # found again
    assert bm.num_free_blocks() == (2, 0)
    bm.free_sequence(2)
    # a new prompt of 5 blocks takes the 2 free blocks, then evicts the 3
    # least recently used cached ones: only the last cached block survives
    bm.add_sequence(3, list(range(1000, 1080)))
    assert bm.num_free_blocks() == (1, 1)
    bm.free_sequence(3)
    assert bm.add_sequence(4, p) == 0                   # its first block was evicted


def test_fork_then_append_copies_the_shared_partial_block():
    bm = pkv.BlockManager(16, 8)
    bm.add_sequence(1, list(range(20)))                 # block a full, block b with 4 tokens
    a, _ = _table(bm, 1)
    bm.fork(1, 2)
    assert _table(bm, 2)[0] == a
    slots, pairs = bm.append_tokens([2], [99])
    b2, L2 = _table(bm, 2)
    assert L2 == 21 and b2[0] == a[0] and b2[1] != a[1]
    assert pairs.tolist() == [[a[1], b2[1]]]
    assert slots.tolist() == [b2[1] * BS + 4]
    # the parent now holds its partial block alone: written in place
    slots, pairs = bm.append_tokens([1], [98])
    assert pairs.numel() == 0 and slots.tolist() == [a[1] * BS + 4]


def test_full_last_block_gets_a_new_block_without_copy():
    bm = pkv.BlockManager(8, 8)
    bm.add_sequence(1, list(range(32)))
    bm.fork(1, 2)
    slots, pairs = bm.append_tokens([1, 2], [5, 6])
    assert pairs.numel() == 0
    t1, _ = _table(bm, 1)
    t2, _ = _table(bm, 2)
    assert t1[:2] == t2[:2] and t1[2] != t2[2]
    assert slots.tolist() == [t1[2] * BS, t2[2] * BS]


def test_failed_calls_change_nothing():
    bm = pkv.BlockManager(4, 8)
    bm.add_sequence(1, list(range(50)))                 # 4 blocks, none left
    before = (bm.num_free_blocks(), _table(bm, 1))
    with pytest.raises(pkv.PkvError) as e:
        bm.add_sequence(2, [1] * 17)
    assert e.value.code == pkv.ERR_OOB
    bm.fork(1, 3)
    with pytest.raises(pkv.PkvError):
        bm.append_tokens([3, 1], [0, 0])                # two copies needed, none available
    assert (bm.num_free_blocks(), _table(bm, 1)) == before
    for bad in (lambda: bm.fork(9, 10), lambda: bm.fork(1, 3), lambda: bm.free_sequence(42),
                lambda: bm.append_tokens([1, 1], [0, 0]), lambda: bm.slots(1, 40, 20),
                lambda: bm.add_sequence(1, [0])):
        with pytest.raises(pkv.PkvError):
            bad()
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(4, 8).add_sequence(1, [0] * (8 * 16 + 1))   # wider than a table


def _kv_rows(prefix_hashes, H, d, dtype):
    """K/V of tokens given the hash of each token's whole prefix: a model's
    K/V depend on the prefix, so equal prefixes give equal rows."""
    k = torch.empty((len(prefix_hashes), H, d))
    v = torch.empty((len(prefix_hashes), H, d))
    for i, h in enumerate(prefix_hashes):
        g = np.random.Generator(np.random.PCG64(h))
        k[i] = torch.from_numpy(g.standard_normal((H, d)))
        v[i] = torch.from_numpy(g.standard_normal((H, d)))
    return k.to(dtype), v.to(dtype)


def _chain(prev, tok):
    return (prev * 1000003 + int(tok) + 1) % (1 << 61)


def _random_workload(seed, steps, apply_copy, apply_append, NB=96, H=2, d=8, dtype=torch.float32):
    """Drive the manager with prompts over shared prefixes, forks, appends
    and frees; write K/V through the given copy / append functions.
    Returns the manager, the live sequences' token histories and the
    prefix hashes of their tokens."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bm = pkv.BlockManager(NB, 16)
    hist, hashes = {}, {}
    systems = [rng.integers(0, 50, size=int(n)).tolist() for n in (40, 33)]
    nid = 0
    for _ in range(steps):
        op = rng.integers(0, 10)
        live = sorted(hist)
        if op < 3 or not live:                          # new prompt, often over a shared prefix
            base = systems[rng.integers(0, 2)] if rng.random() < 0.7 else []
            toks = base + rng.integers(0, 50, size=int(rng.integers(1, 30))).tolist()
            try:
                cached = bm.add_sequence(nid, toks)
            except pkv.PkvError:
                continue
            hs, h = [], 0
            for t in toks:
                h = _chain(h, t)
                hs.append(h)
            if cached < len(toks):
                k, v = _kv_rows(hs[cached:], H, d, dtype)
                apply_append(k, v, bm.slots(nid, cached, len(toks) - cached))
            hist[nid], hashes[nid] = toks, hs
            nid += 1
        elif op < 5:                                    # fork
            p = live[rng.integers(0, len(live))]
            bm.fork(p, nid)
            hist[nid], hashes[nid] = list(hist[p]), list(hashes[p])
            nid += 1
        elif op < 9:                                    # one decode step for some sequences
            ids = [s for s in live if rng.random() < 0.6 and len(hist[s]) < 16 * 16 - 1]
            if not ids:
                continue
            toks = rng.integers(0, 50, size=len(ids)).tolist()
            try:
                slots, pairs = bm.append_tokens(ids, toks)
            except pkv.PkvError:
                continue
            if pairs.numel():
                apply_copy(pairs)
            hs = [_chain(hashes[s][-1], t) for s, t in zip(ids, toks)]
            k, v = _kv_rows(hs, H, d, dtype)
            apply_append(k, v, slots)
            for s, t, h in zip(ids, toks, hs):
                hist[s].append(t)
                hashes[s].append(h)
        else:                                           # a sequence ends
            s = live[rng.integers(0, len(live))]
            bm.free_sequence(s)
            del hist[s], hashes[s]
    return bm, hist, hashes


def test_random_workload_reads_back_every_history():
    NB, H, d = 96, 2, 8
    kc = torch.full((NB, H, BS, d), float("nan"))
    vc = torch.full((NB, H, BS, d), float("nan"))
    bm, hist, hashes = _random_workload(
        7, 400, lambda pairs: oracle.copy_blocks(kc, vc, pairs),
        lambda k, v, slots: oracle.kv_append(k, v, slots, kc, vc), NB=NB, H=H, d=d)
    assert len(hist) >= 5
    for s, hs in hashes.items():
        blocks, L = _table(bm, s)
        assert L == len(hs)
        k, v = _kv_rows(hs, H, d, torch.float32)
        got_k = torch.stack([kc[blocks[t // BS], :, t % BS] for t in range(L)])
        got_v = torch.stack([vc[blocks[t // BS], :, t % BS] for t in range(L)])
        assert torch.equal(got_k, k) and torch.equal(got_v, v), f"sequence {s}"
    # and the paged oracle over the manager's tables equals attention over the histories
    ids = sorted(hashes)
    tables, lens = bm.block_tables(ids)
    q = torch.randn((len(ids), H, d), generator=torch.Generator().manual_seed(3))
    out = oracle.decode(q, kc, vc, tables, lens, 0.35)
    for i, s in enumerate(ids):
        k, v = _kv_rows(hashes[s], H, d, torch.float32)
        for h in range(H):
            w = torch.softmax((k[:, h].double() @ q[i, h].double()) * 0.35, dim=0)
            assert torch.allclose(out[i, h].double(), w @ v[:, h].double(), atol=1e-12)


@pytest.mark.gpu
def test_random_workload_through_the_kernels():
    NB, H, d = 96, 8, 128
    dev = "cuda"
    kc = torch.full((NB, H, BS, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    kc_o, vc_o = kc.cpu(), vc.cpu()

    def copy(pairs):
        pkv.copy_blocks(pairs.to(dev), kc, vc)
        oracle.copy_blocks(kc_o, vc_o, pairs)

    def append(k, v, slots):
        pkv.kv_append(k.to(dev), v.to(dev), slots.to(dev), kc, vc)
        oracle.kv_append(k, v, slots, kc_o, vc_o)

    bm, hist, hashes = _random_workload(11, 300, copy, append, NB=NB, H=H, d=d, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert torch.equal(kc.cpu().view(torch.int16), kc_o.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), vc_o.view(torch.int16))
    ids = sorted(hashes)
    tables, lens = bm.block_tables(ids)
    q = torch.randn((len(ids), 4 * H, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    ref = oracle.decode(q, kc_o, vc_o, tables, lens, d ** -0.5)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pkv.paged_attention_decode(q.to(dev), kc, vc, tables.to(dev), lens.to(dev), d ** -0.5, out,
                               max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert float((out.cpu().double() - ref).abs().max()) <= 1e-2
