"""Pins for the fp64 oracle: things it must agree with that are not itself.

Each pin targets a plausible mistake:
  * dense library attention (torch SDPA, fp64) on contiguous K/V catches a wrong
    softmax, scale, sign, GQA head map or gather index;
  * closed forms (one token, all-zero keys, zero scale, one dominant key) and
    the ToyKV worked example of chengxuchu PyTorch #47 section 6.1 catch a
    dropped normalisation or max term;
  * bitwise invariance under relabelling physical blocks, and shared vs copied
    prefix blocks, catches any dependence on physical placement;
  * the memory ledger of section 2.3 and the block-table example of the
    caffein.top "Paging" section pin the byte formula and the gather order.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_297_gb300 import accounting
from tests._util import BS, paged_from_dense, sdpa_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(path):
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = [x.strip() for x in line.split("=")]
        out[k] = float(v) if "." in v else int(v)
    return out


def _random_case(seed, S, Hq, Hkv, d, lens, dtype=torch.float32):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    ks = [torch.randn(L, Hkv, d, generator=g).to(dtype) for L in lens]
    vs = [torch.randn(L, Hkv, d, generator=g).to(dtype) for L in lens]
    need = sum((L + BS - 1) // BS for L in lens)
    kc, vc, bt = paged_from_dense(ks, vs, need + 3, Hkv, d, rng, dtype=dtype)
    q = torch.randn(S, Hq, d, generator=g).to(dtype)
    cl = torch.tensor(lens, dtype=torch.int32)
    return q, ks, vs, kc, vc, bt, cl


# ---------------------------------------------------------------- dense library

@pytest.mark.parametrize("S,Hq,Hkv,d,lens,dtype", [
    (3, 4, 4, 8, [1, 17, 40], torch.float32),
    (4, 8, 2, 16, [16, 15, 33, 64], torch.float32),
    (2, 6, 1, 4, [5, 48], torch.bfloat16),
    (5, 8, 8, 64, [1, 2, 31, 32, 100], torch.bfloat16),
])
def test_decode_matches_dense_sdpa(S, Hq, Hkv, d, lens, dtype):
    q, ks, vs, kc, vc, bt, cl = _random_case(7 + S, S, Hq, Hkv, d, lens, dtype)
    scale = 1.0 / math.sqrt(d) * 1.3
    got = oracle.decode(q, kc, vc, bt, cl, scale)
    for s in range(S):
        ref = sdpa_rows(q[s:s + 1], ks[s], vs[s], scale)[0]
        torch.testing.assert_close(got[s], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("priors,chunks,Hq,Hkv,d", [
    ([0, 0], [5, 33], 4, 2, 8),
    ([3, 20, 47], [1, 16, 9], 8, 2, 16),
    ([64], [64], 2, 1, 32),
])
def test_prefill_matches_dense_sdpa(priors, chunks, Hq, Hkv, d):
    lens = [p + n for p, n in zip(priors, chunks)]
    S = len(lens)
    rng = np.random.default_rng(3)
    g = torch.Generator().manual_seed(11)
    ks = [torch.randn(L, Hkv, d, generator=g) for L in lens]
    vs = [torch.randn(L, Hkv, d, generator=g) for L in lens]
    kc, vc, bt = paged_from_dense(ks, vs, sum((L + BS - 1) // BS for L in lens) + 2, Hkv, d, rng)
    cu = torch.tensor([0] + list(np.cumsum(chunks)), dtype=torch.int32)
    q = torch.randn(int(cu[-1]), Hq, d, generator=g)
    scale = 0.3
    got = oracle.prefill_chunk(q, cu, kc, vc, bt, torch.tensor(lens, dtype=torch.int32), scale)
    for s in range(S):
        rows = q[cu[s]:cu[s + 1]]
        if priors[s] == 0:
            # no prior context: the library's own causal flag is the reference
            ref = sdpa_rows(rows, ks[s], vs[s], scale, is_causal=True)
        else:
            pos = torch.arange(chunks[s]) + priors[s]
            mask = torch.arange(lens[s])[None, :] <= pos[:, None]
            ref = sdpa_rows(rows, ks[s], vs[s], scale, mask=mask[None])
        torch.testing.assert_close(got[cu[s]:cu[s + 1]], ref, rtol=0, atol=1e-12)


def test_decode_is_prefill_of_one_token():
    q, ks, vs, kc, vc, bt, cl = _random_case(5, 4, 4, 2, 16, [3, 16, 17, 50])
    dec = oracle.decode(q, kc, vc, bt, cl, 0.25)
    cu = torch.arange(5, dtype=torch.int32)
    pre = oracle.prefill_chunk(q, cu, kc, vc, bt, cl, 0.25)
    assert torch.equal(dec, pre)


# ---------------------------------------------------------------- closed forms

def test_single_token_returns_its_value_row():
    q, ks, vs, kc, vc, bt, cl = _random_case(1, 3, 4, 2, 16, [1, 1, 1])
    got = oracle.decode(q, kc, vc, bt, cl, 0.125)
    for s in range(3):
        ref = vs[s][0].double().repeat_interleave(2, dim=0)
        assert torch.equal(got[s], ref)


def test_zero_keys_or_zero_scale_give_mean_of_values():
    q, ks, vs, kc, vc, bt, cl = _random_case(2, 2, 2, 2, 8, [7, 30])
    for kcache, scale in ((torch.zeros_like(kc), 0.5), (kc, 0.0)):
        got = oracle.decode(q, kcache, vc, bt, cl, scale)
        for s in range(2):
            ref = vs[s].double().mean(dim=0)
            torch.testing.assert_close(got[s], ref, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value_row():
    q, ks, vs, kc, vc, bt, cl = _random_case(4, 1, 1, 1, 8, [37])
    t = 21
    kc2 = kc.clone()
    blk = int(bt[0, t // BS])
    kc2[blk, 0, t % BS, :] = q[0, 0] * 1000.0
    got = oracle.decode(q, kc2, vc, bt, cl, 1.0)
    torch.testing.assert_close(got[0, 0], vs[0][t, 0].double(), rtol=0, atol=1e-12)


def test_empty_context_gives_zero_row():
    q, ks, vs, kc, vc, bt, cl = _random_case(6, 2, 2, 1, 8, [0, 5])
    got = oracle.decode(q, kc, vc, bt, cl, 1.0)
    assert torch.equal(got[0], torch.zeros_like(got[0]))
    assert torch.isfinite(got[1]).all()


def test_toykv_worked_example():
    """chengxuchu PyTorch #47 section 6.1, ToyKV: token i is the one-hot e_i,
    its key is e_i, its value 2 e_i, the query is the newest key and no scale
    is applied.  Step i attends over keys e_0..e_i, so the newest key scores 1
    and the others 0: out_i = 2 * (sum_{j<i} e_j + e * e_i) / (i + e).
    (The page's printed rows disagree with its own code; the code is the
    definition taken here.)"""
    d, e = 4, math.e
    kc = torch.full((1, 1, BS, d), float("nan"))
    vc = torch.full((1, 1, BS, d), float("nan"))
    bt = torch.zeros((1, 1), dtype=torch.int32)
    for i in range(3):
        tok = torch.zeros(d)
        tok[i] = 1.0
        oracle.kv_append(tok.view(1, 1, d), (2 * tok).view(1, 1, d),
                         torch.tensor([i], dtype=torch.int64), kc, vc)
        got = oracle.decode(tok.view(1, 1, d), kc, vc, bt,
                            torch.tensor([i + 1], dtype=torch.int32), 1.0)[0, 0]
        ref = torch.zeros(d, dtype=torch.float64)
        ref[:i] = 2.0 / (i + e)
        ref[i] = 2.0 * e / (i + e)
        torch.testing.assert_close(got, ref, rtol=0, atol=1e-15)
    torch.testing.assert_close(got[:3], torch.tensor([0.424, 0.424, 1.152], dtype=torch.float64),
                               rtol=0, atol=5e-4)


# ---------------------------------------------------------------- invariants

def test_block_relabelling_is_bitwise_invariant():
    q, ks, vs, kc, vc, bt, cl = _random_case(8, 4, 8, 2, 16, [9, 48, 49, 3])
    NB = kc.shape[0]
    pi = torch.from_numpy(np.random.default_rng(0).permutation(NB))
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = torch.where(bt >= 0, pi[bt.clamp(min=0).long()].to(torch.int32), bt)
    a = oracle.decode(q, kc, vc, bt, cl, 0.2)
    b = oracle.decode(q, kc2, vc2, bt2, cl, 0.2)
    assert torch.equal(a, b)


def test_append_to_another_slot_is_bitwise_invariant():
    """The new token written into a copy of the last block (table updated)
    gives the same output as writing it in place."""
    g = torch.Generator().manual_seed(13)
    Hkv, d, NB = 2, 8, 10
    kc = torch.randn(NB, Hkv, BS, d, generator=g)
    vc = torch.randn(NB, Hkv, BS, d, generator=g)
    k = torch.randn(1, Hkv, d, generator=g)
    v = torch.randn(1, Hkv, d, generator=g)
    q = torch.randn(1, 4, d, generator=g)
    bt = torch.tensor([[2, 6, 4]], dtype=torch.int32)
    cl = torch.tensor([40], dtype=torch.int32)               # token 39: block 4, row 7
    kc_a, vc_a = kc.clone(), vc.clone()
    oracle.kv_append(k, v, torch.tensor([4 * BS + 7]), kc_a, vc_a)
    a = oracle.decode(q, kc_a, vc_a, bt, cl, 0.3)
    kc_b, vc_b = kc.clone(), vc.clone()
    oracle.copy_blocks(kc_b, vc_b, torch.tensor([[4, 9]]))
    oracle.kv_append(k, v, torch.tensor([9 * BS + 7]), kc_b, vc_b)
    b = oracle.decode(q, kc_b, vc_b, torch.tensor([[2, 6, 9]], dtype=torch.int32), cl, 0.3)
    assert torch.equal(a, b)


def test_shared_prefix_equals_private_copies():
    g = torch.Generator().manual_seed(9)
    Hkv, d, NB = 2, 8, 12
    kc = torch.randn(NB, Hkv, BS, d, generator=g)
    vc = torch.randn(NB, Hkv, BS, d, generator=g)
    # both sequences share blocks 3 and 5 as a prefix, then private 7 / 8
    shared = torch.tensor([[3, 5, 7], [3, 5, 8]], dtype=torch.int32)
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[[0, 1]] = kc[[3, 5]]
    vc2[[0, 1]] = vc[[3, 5]]
    private = torch.tensor([[3, 5, 7], [0, 1, 8]], dtype=torch.int32)
    q = torch.randn(2, 4, d, generator=g)
    cl = torch.tensor([40, 45], dtype=torch.int32)
    assert torch.equal(oracle.decode(q, kc, vc, shared, cl, 0.3),
                       oracle.decode(q, kc2, vc2, private, cl, 0.3))


# ---------------------------------------------------------------- append / copy

def test_append_then_read_matches_dense():
    """Appending a sequence's tokens one by one at slots taken from its block
    table, then decoding, equals dense attention over those tokens."""
    g = torch.Generator().manual_seed(12)
    Hkv, Hq, d, L = 2, 4, 16, 37
    table = torch.tensor([[6, 2, 9]], dtype=torch.int32)
    kc = torch.full((10, Hkv, BS, d), float("nan"))
    vc = torch.full((10, Hkv, BS, d), float("nan"))
    ks = torch.randn(L, Hkv, d, generator=g)
    vs = torch.randn(L, Hkv, d, generator=g)
    slots = torch.tensor([int(table[0, t // BS]) * BS + t % BS for t in range(L)])
    for t in torch.randperm(L, generator=g).tolist():  # any order of appends
        oracle.kv_append(ks[t:t + 1], vs[t:t + 1], slots[t:t + 1], kc, vc)
    q = torch.randn(1, Hq, d, generator=g)
    got = oracle.decode(q, kc, vc, table, torch.tensor([L], dtype=torch.int32), 0.25)
    torch.testing.assert_close(got[0], sdpa_rows(q, ks, vs, 0.25)[0], rtol=0, atol=1e-12)


def test_append_skips_negative_slots_and_touches_nothing_else():
    g = torch.Generator().manual_seed(13)
    kc = torch.randn(4, 2, BS, 8, generator=g).to(torch.bfloat16)
    vc = torch.randn(4, 2, BS, 8, generator=g).to(torch.bfloat16)
    k = torch.randn(3, 2, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(3, 2, 8, generator=g).to(torch.bfloat16)
    slots = torch.tensor([5, -1, 63])
    k0, v0 = kc.clone(), vc.clone()
    oracle.kv_append(k, v, slots, kc, vc)
    assert torch.equal(kc[0, :, 5], k[0]) and torch.equal(vc[3, :, 15], v[2])
    mask = torch.ones(4, BS, dtype=torch.bool)
    mask[0, 5] = mask[3, 15] = False
    assert torch.equal(kc.permute(0, 2, 1, 3)[mask], k0.permute(0, 2, 1, 3)[mask])
    assert torch.equal(vc.permute(0, 2, 1, 3)[mask], v0.permute(0, 2, 1, 3)[mask])
    with pytest.raises(IndexError):
        oracle.kv_append(k[:1], v[:1], torch.tensor([64]), kc, vc)


def test_copy_blocks_copies_whole_blocks_only():
    g = torch.Generator().manual_seed(14)
    kc = torch.randn(6, 2, BS, 8, generator=g)
    vc = torch.randn(6, 2, BS, 8, generator=g)
    k0, v0 = kc.clone(), vc.clone()
    oracle.copy_blocks(kc, vc, torch.tensor([[1, 4], [2, 0]]))
    assert torch.equal(kc[4], k0[1]) and torch.equal(vc[0], v0[2])
    for b in (1, 2, 3, 5):
        assert torch.equal(kc[b], k0[b]) and torch.equal(vc[b], v0[b])
    q = torch.randn(1, 2, 8, generator=g)
    cl = torch.tensor([20], dtype=torch.int32)
    a = oracle.decode(q, kc, vc, torch.tensor([[3, 1]], dtype=torch.int32), cl, 0.5)
    b = oracle.decode(q, kc, vc, torch.tensor([[3, 4]], dtype=torch.int32), cl, 0.5)
    assert torch.equal(a, b)


def test_bad_block_id_is_reported():
    q, ks, vs, kc, vc, bt, cl = _random_case(15, 1, 1, 1, 8, [20])
    bt2 = bt.clone()
    bt2[0, 1] = kc.shape[0]
    with pytest.raises(IndexError):
        oracle.decode(q, kc, vc, bt2, cl, 1.0)


# ---------------------------------------------------------------- golden fixtures

def test_ledger_worked_example():
    p = _read_kv(os.path.join(GOLDEN, "kv_ledger.txt"))
    nbytes = accounting.kv_cache_bytes(p["layers"], p["batch"], p["kv_heads"],
                                       p["sequence_length"], p["head_dim"],
                                       p["bytes_per_element"])
    assert round(nbytes / 1024 ** 3, 2) == p["printed_gib"]
    # the per-request form of the caffein.top page gives the same total
    per_request = 2 * p["layers"] * p["sequence_length"] * p["kv_heads"] * p["head_dim"] * 2
    assert per_request * p["batch"] == nbytes
    # one layer of the Llama-3-8B-shaped decode: 4096 B per cached token
    cl = torch.tensor([1000, 24], dtype=torch.int32)
    assert accounting.decode_bytes(cl, 32, 8, 128, 2, 2)["kv"] == 1024 * 4096


def test_block_table_example_gathers_in_table_order():
    """caffein.top "Paging": request A's tokens live in blocks 1, 4, 7 and
    request B's in 2, 3.  Reading through those tables must see the tokens in
    that block order: with one dominant key per logical position the output
    is the value row of that position."""
    tables = {}
    for line in open(os.path.join(GOLDEN, "block_table_example.txt")):
        if line.strip() and not line.startswith("#"):
            name, *ids = line.split()
            tables[name] = [int(x) for x in ids]
    d, NB = 8, 8
    kc = torch.zeros(NB, 1, BS, d)
    vc = torch.zeros(NB, 1, BS, d)
    for blk in range(NB):  # value row encodes (block, row)
        for r in range(BS):
            vc[blk, 0, r, 0] = blk
            vc[blk, 0, r, 1] = r
    for name, ids in tables.items():
        bt = torch.tensor([ids], dtype=torch.int32)
        L = len(ids) * BS
        for t in (0, 15, 16, L - 1):
            kk = kc.clone()
            q = torch.zeros(1, 1, d)
            q[0, 0, 2] = 1.0
            kk[ids[t // BS], 0, t % BS, 2] = 1000.0
            out = oracle.decode(q, kk, vc, bt, torch.tensor([L], dtype=torch.int32), 1.0)[0, 0]
            assert round(float(out[0])) == ids[t // BS] and round(float(out[1])) == t % BS


# ------------------------------------------------------------------ fp8 (E4M3) cache

def test_e4m3_codes_decode_like_the_library_format():
    """Every one of the 256 codes widens to torch's float8_e4m3fn value;
    S.1111.111 is NaN (the format has no infinity)."""
    codes = torch.arange(256, dtype=torch.uint8)
    got = oracle.e4m3_decode(codes)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64)
    nan = ref.isnan()
    assert nan.nonzero().flatten().tolist() == [127, 255]
    assert got[nan].isnan().all() and torch.equal(got[~nan], ref[~nan])
    assert float(got[0x7E]) == 448.0 and float(got[0x01]) == 2.0 ** -9 and float(got[0x38]) == 1.0


def test_e4m3_encoding_round_trips_and_matches_the_library_in_range():
    codes = torch.tensor([c for c in range(256) if c not in (127, 255)], dtype=torch.uint8)
    vals = oracle.e4m3_decode(codes).to(torch.float32)
    assert torch.equal(oracle.e4m3_encode(vals), codes)          # -0 -> 0x80 included
    g = torch.Generator().manual_seed(17)
    x = torch.cat([torch.randn(4000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[x.abs() <= 448]
    assert torch.equal(oracle.e4m3_encode(x), x.to(torch.float8_e4m3fn).view(torch.uint8))


def test_e4m3_rounds_ties_to_even_and_saturates():
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (001): even wins;
    # 1.1875 halfway between 1.125 (001) and 1.25 (010); 2^-10 halfway
    # between 0 and the smallest subnormal
    x = torch.tensor([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 449.0, 1e6, -1e6, 464.0])
    assert oracle.e4m3_encode(x).tolist() == [0x38, 0x3A, 0x00, 0x02, 0x7E, 0x7E, 0xFE, 0x7E]


def test_fp8_append_stores_codes_of_the_scaled_rows():
    NB, H, d = 4, 2, 16
    g = torch.Generator().manual_seed(3)
    k = (torch.randn(5, H, d, generator=g) * 40).to(torch.bfloat16)
    v = (torch.randn(5, H, d, generator=g) * 3).to(torch.bfloat16)
    ks, vs = torch.tensor([0.25, 3.0]), torch.tensor([0.125, 0.01])
    slots = torch.tensor([0, 17, -1, 63, 5], dtype=torch.int64)
    kc = torch.full((NB, H, BS, d), 0x55, dtype=torch.uint8)
    vc = kc.clone()
    oracle.kv_append_fp8(k, v, slots, kc, vc, ks, vs)
    touched = torch.zeros(NB * BS, dtype=torch.bool)
    def want(x):  # torch's cast in range; beyond 448 the saturated code
        c = x.to(torch.float8_e4m3fn).view(torch.uint8)
        return torch.where(x.abs() > 448, torch.where(x > 0, 0x7E, 0xFE).to(torch.uint8), c)

    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        touched[s] = True
        for h in range(H):
            assert torch.equal(kc[s // BS, h, s % BS], want(k[i, h].float() / ks[h]))
            assert torch.equal(vc[s // BS, h, s % BS], want(v[i, h].float() / vs[h]))
    rest = ~touched.view(NB, BS)
    assert (kc.permute(0, 2, 1, 3)[rest] == 0x55).all() and (vc.permute(0, 2, 1, 3)[rest] == 0x55).all()


def test_fp8_attention_multiplies_the_per_head_scales_back():
    """An fp8 cache read with per-head power-of-two scales equals the binary32
    cache holding code value x scale exactly."""
    NB, Hkv, Hq, d = 6, 2, 4, 16
    g = torch.Generator().manual_seed(9)
    kc = torch.randint(0, 256, (NB, Hkv, BS, d), dtype=torch.uint8, generator=g)
    vc = torch.randint(0, 256, (NB, Hkv, BS, d), dtype=torch.uint8, generator=g)
    kc[(kc & 0x7F) == 0x7F] = 0x10                           # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    ks, vs = torch.tensor([0.5, 4.0]), torch.tensor([2.0 ** -3, 8.0])
    kf = (oracle.e4m3_decode(kc) * ks.double().view(1, Hkv, 1, 1)).float()
    vf = (oracle.e4m3_decode(vc) * vs.double().view(1, Hkv, 1, 1)).float()
    bt = torch.tensor([[3, 1, 5], [0, 2, 4]], dtype=torch.int32)
    cl = torch.tensor([40, 33], dtype=torch.int32)
    q = torch.randn(2, Hq, d, generator=g) * 0.05
    a = oracle.decode(q, kc, vc, bt, cl, 0.3, ks, vs)
    b = oracle.decode(q, kf, vf, bt, cl, 0.3)
    assert torch.equal(a, b)
