"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Indexing work (append scatter, copy-on-write copy, block-table gather) must be
bit-exact; attention outputs must meet the stated float tolerances.  Every
cache row that holds no token is NaN, so an over-read shows up as a
non-finite output.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_297_gb300 as pkv
from paged_kv_cache_297_gb300 import workloads as W
from tests._steps import assert_bits_equal, assert_parity, gpu_step, oracle_step, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        pkv.get_status()
    yield
    if torch.cuda.is_available():
        pkv.get_status()


def _check_step(b, out_dtype=torch.float32, partition_size=0):
    kc_o, vc_o, out_o, pout_o = oracle_step(b)
    kc_g, vc_g, out_g, pout_g = gpu_step(b, out_dtype=out_dtype, partition_size=partition_size)
    assert_bits_equal(kc_g, kc_o, "k_cache after copy+append")
    assert_bits_equal(vc_g, vc_o, "v_cache after copy+append")
    res = {}
    if b.q.shape[0]:
        res["decode"] = assert_parity(out_g, out_o, b.dtype, "decode")
    if pout_o is not None:
        res["prefill"] = assert_parity(pout_g, pout_o, b.dtype, "prefill")
    assert pkv.get_status() == 0
    return res


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", list(W.SPECS))
def test_workload_parity_fp32_out(name):
    b = W.make_batch(name)
    res = _check_step(b, torch.float32)
    print(name, res)


@pytest.mark.parametrize("name", ["llama3_8b_decode", "long_context", "mixed_step"])
def test_workload_parity_bf16_out(name):
    b = W.make_batch(name)
    _check_step(b, torch.bfloat16)


@pytest.mark.parametrize("name", ["llama3_8b_decode", "long_context"])
def test_workload_parity_smallest_partition(name):
    # the default picks a large partition on these shapes; the smallest one
    # splits every long sequence and exercises the reduction at full size
    b = W.make_batch(name)
    _check_step(b, partition_size=512)


# ------------------------------------------------------------------ edge cases

EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 511, 512, 513, 1023, 1024, 1025, 2047]


@pytest.mark.parametrize("dtype,hq,hkv,d", [
    ("bf16", 32, 8, 128), ("bf16", 64, 8, 128), ("bf16", 8, 8, 64), ("bf16", 16, 1, 128),
    ("bf16", 32, 1, 64), ("bf16", 48, 2, 128), ("f32", 4, 4, 64), ("f32", 16, 4, 128),
])
def test_edge_lengths(dtype, hq, hkv, d):
    b = W.custom_batch(dtype, len(EDGE_LENS), hq, hkv, d, EDGE_LENS, seed=101 + hq + d)
    _check_step(b)


@pytest.mark.parametrize("partition", [16, 64, 112, 512, 4096])
def test_partition_sizes_agree(partition):
    lens = [1, 16, 100, 511, 512, 513, 1500, 4000]
    b = W.custom_batch("bf16", len(lens), 32, 8, 128, lens, seed=202)
    _check_step(b, partition_size=partition)


def test_split_matches_unsplit():
    lens = [3000, 4096, 777, 2049]
    b = W.custom_batch("bf16", len(lens), 32, 8, 128, lens, seed=203)
    _, _, split, _ = gpu_step(b, partition_size=512)
    _, _, whole, _ = gpu_step(b, partition_size=4096)
    assert float((split - whole).abs().max()) <= 2e-3


def test_head_warps_match_split_warps():
    # partitions of at most 512 tokens give each warp a whole (kv head,
    # partition); larger ones split a (kv head, partition) over four warps
    # (160 sequences: enough thread blocks for the head-warp schedule)
    lens = [1, 40, 500, 512, 513, 1000, 1023] * 23
    b = W.custom_batch("bf16", len(lens), 40, 5, 128, lens, seed=207)
    _, _, heads, _ = gpu_step(b, partition_size=512)
    _, _, split, _ = gpu_step(b, partition_size=1024)
    assert float((heads - split).abs().max()) <= 2e-3
    _check_step(b, partition_size=512)
    _check_step(b, partition_size=1024)


def test_default_matches_unsplit():
    lens = [3000, 4096, 777, 2049]
    b = W.custom_batch("bf16", len(lens), 32, 8, 128, lens, seed=206)
    _, _, dflt, _ = gpu_step(b, partition_size=0)
    _, _, whole, _ = gpu_step(b, partition_size=4096)
    assert float((dflt - whole).abs().max()) <= 2e-3


# ------------------------------------------------------------------ batch shapes

def _lens(n, lo, hi, seed):
    import numpy as np
    return np.random.Generator(np.random.PCG64(seed)).integers(lo, hi + 1, n).tolist()


@pytest.mark.parametrize("S,hq,hkv,d,lo,hi,seed", [
    (300, 32, 8, 128, 0, 200, 601),       # many short sequences, some empty
    (1, 32, 8, 128, 65536, 65536, 602),   # one long sequence: 128 partitions of 512
    (2049, 8, 8, 64, 1, 64, 604),         # many tiny sequences, G = 1
    (7, 16, 1, 128, 1000, 9000, 605),     # a group of 16 on one kv head
    (33, 12, 4, 64, 1, 3000, 606),        # group of 3 (rows 3..15 of the tile empty)
])
def test_batch_shapes(S, hq, hkv, d, lo, hi, seed):
    lens = _lens(S, lo, hi, seed)
    b = W.custom_batch("bf16", S, hq, hkv, d, lens, seed=seed)
    _check_step(b)
    _check_step(b, out_dtype=torch.bfloat16)


def test_single_token_context_returns_value_row_exactly():
    b = W.custom_batch("bf16", 6, 32, 8, 128, [1] * 6, seed=204)
    _, _, out, _ = gpu_step(b)
    ref = b.v_new.float().repeat_interleave(4, dim=1)
    assert torch.equal(out.cpu(), ref)


def test_outlier_rows_long_mixed_lengths():
    lens = [40000, 513, 8191, 65536]
    b = W.custom_batch("bf16", len(lens), 64, 8, 128, lens, seed=205, outlier_p=0.01,
                       outlier_scale=20.0)
    _check_step(b)


@pytest.mark.parametrize("priors,chunks,hq,hkv,d", [
    ([0, 5, 100, 16], [1, 17, 64, 200], 32, 8, 128),
    ([0, 3072], [512, 512], 64, 8, 128),
    ([7, 0], [130, 33], 8, 8, 64),
    ([1000], [1], 16, 1, 128),
    # q tiles by TMA for groups that divide the 128-row tile (1, 32), copied
    # by the softmax threads otherwise (12)
    ([50, 0], [200, 129], 8, 8, 128),
    ([0, 900], [40, 300], 32, 1, 128),
    ([0, 300], [77, 260], 24, 2, 128),
    # empty chunks beside a non-empty one (their work items do nothing)
    ([10, 0, 300], [0, 50, 0], 32, 8, 128),
    ([10, 0, 300], [0, 50, 0], 8, 8, 64),
])
def test_prefill_edges(priors, chunks, hq, hkv, d):
    b = W.custom_prefill("bf16", hq, hkv, d, priors, chunks, seed=301 + sum(chunks))
    _check_step(b)


@pytest.mark.parametrize("scale,d", [(30.0, 128), (-30.0, 128), (30.0, 64)])
def test_prefill_late_score_jumps_in_either_key_half(scale, d):
    # Keys scaled x30 at a few positions of later key tiles, in either 64-key
    # half of their tile (positions 300, 700, 900: first half; 500, 1100,
    # 1150: second half): the running maximum of many rows jumps by far more
    # than 8 (log2 units) mid-sequence.  The reference of both threads of a
    # row must move, whichever half holds the jump, and O must be rescaled.
    # The negative scale makes the jumps land on other rows.  A row whose
    # weight then sits on one key must get that key's V: P enters the PV
    # product in bf16, and the row sum must add those same values.  d = 64
    # runs the mma.sync kernel.
    b = W.custom_prefill("bf16", 32, 8, d, [1000, 0], [200, 300], seed=331)
    prior, table = 1000, b.prefill_block_tables
    for pos in (300, 500, 700, 900, 1100, 1150):
        if pos < prior:
            blk = int(table[0, pos // 16])
            b.k_cache[blk, :, pos % 16, :] = (b.k_cache[blk, :, pos % 16, :].float() * scale).to(b.dtype)
        else:  # sequence 0's new tokens come first in k_new
            b.k_new[pos - prior] = (b.k_new[pos - prior].float() * scale).to(b.dtype)
    _check_step(b)


@pytest.mark.parametrize("case", range(8))
def test_decode_random_shapes(case):
    # Seeded random decode batches: group sizes 1-16, head_dim 64 and 128,
    # lengths from 1 token to 20k (outlier rows in some), partitions from 16
    # tokens to adaptive, both output types.
    import random
    rng = random.Random(7200 + case)
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 4, 8, 12, 16])
    d = rng.choice([64, 128])
    S = rng.randint(1, 48)
    hi = rng.choice([600, 5000, 20000])
    lens = [rng.choice([1, rng.randint(16, hi), rng.randint(1, 64)]) for _ in range(S)]
    b = W.custom_batch("bf16", S, hkv * g, hkv, d, lens, seed=rng.randint(1, 10 ** 6),
                       outlier_p=rng.choice([0.0, 0.01]), outlier_scale=20.0)
    _check_step(b, rng.choice([torch.float32, torch.bfloat16]), partition_size=rng.choice([0, 16, 256, 1536]))


@pytest.mark.parametrize("case", range(6))
def test_shared_prefix_random_shapes(case):
    # Seeded random cascade batches: prefix of 1-40 blocks, suffixes of 1 to
    # ~1500 tokens, groups 1-12, appended or fused, adaptive or 256/512-token
    # partitions; caches bit-exact, output within the bf16 bound.
    import random
    rng = random.Random(7300 + case)
    hkv = rng.choice([4, 8])
    g = rng.choice([1, 2, 4, 8, 12])
    S, pb = rng.randint(2, 120), rng.randint(1, 40)
    lo = rng.randint(1, 64)
    b = W.make_batch("shared_prefix_cow", num_seqs=S, ctx=(lo, lo + rng.randint(0, 1500)), prefix_blocks=pb,
                     heads=(hkv * g, hkv))
    kc_o, vc_o, out_o, _ = oracle_step(b)
    t, out = _cascade_step(b, pb * 16, fused=rng.choice([True, False]), partition=rng.choice([0, 256, 512]))
    assert pkv.get_status() == 0
    assert_bits_equal(t["k_cache"], kc_o, "k_cache")
    assert_bits_equal(t["v_cache"], vc_o, "v_cache")
    assert_parity(out, out_o, b.dtype, "cascade decode")


def _random_prefill_case(rng):
    """One seeded random prefill shape: group size, head_dim, priors and chunk
    sizes (empty chunks included), output type, and sometimes keys of the
    first sequence scaled x25 (score jumps in later tiles)."""
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 3, 4, 6, 8, 12, 16])
    d = rng.choice([128, 128, 64])
    nseq = rng.randint(1, 6)
    priors = [rng.choice([0, rng.randint(0, 3000), rng.randint(3000, 6000)]) for _ in range(nseq)]
    chunks = [rng.choice([0, 1, rng.randint(1, 700), rng.randint(700, 1500)]) for _ in range(nseq)]
    if sum(chunks) == 0:
        chunks[0] = rng.randint(1, 300)
    b = W.custom_prefill("bf16", hkv * g, hkv, d, priors, chunks, seed=rng.randint(1, 10 ** 6))
    jump = rng.choice([None, None, 25.0, -25.0])
    if jump is not None:
        L0 = priors[0] + chunks[0]
        for _ in range(4):
            pos = rng.randrange(0, max(1, L0))
            if pos < priors[0]:
                blk = int(b.prefill_block_tables[0, pos // 16])
                b.k_cache[blk, :, pos % 16, :] = (b.k_cache[blk, :, pos % 16, :].float() * jump).to(b.dtype)
            else:
                b.k_new[pos - priors[0]] = (b.k_new[pos - priors[0]].float() * jump).to(b.dtype)
    return b, rng.choice([torch.float32, torch.bfloat16])


@pytest.mark.parametrize("case", range(12))
def test_prefill_random_shapes(case):
    # Seeded random shapes beyond the hand-picked edges: several items per CTA
    # pair, queries that G does not divide into the 128-row tile, empty
    # chunks beside long ones, both kernels, both output types.
    import random
    b, out_dtype = _random_prefill_case(random.Random(7100 + case))
    _check_step(b, out_dtype)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_output_only_16_byte_aligned(out_dtype):
    # the epilogue writes 32 bytes per store only to a 32-byte aligned output
    b = W.custom_prefill("bf16", 32, 8, 128, [0, 700], [300, 200], seed=311)
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    n = b.prefill_q.numel()
    shift = 16 // torch.empty(0, dtype=out_dtype).element_size()
    buf = torch.empty(n + shift, dtype=out_dtype, device="cuda")
    outs = [buf[:n].view(b.prefill_q.shape), buf[shift:].view(b.prefill_q.shape)]
    assert outs[1].data_ptr() % 32 == 16
    res = []
    for out in outs:
        out.fill_(float("nan"))
        pkv.paged_attention_prefill_chunk(t["prefill_q"], t["prefill_cu_q_lens"], t["k_cache"], t["v_cache"],
                                          t["prefill_block_tables"], t["prefill_context_lens"], b.scale, out,
                                          max_q_len=300, max_context_len=900)
        torch.cuda.synchronize()
        res.append(out.clone())
    assert pkv.get_status() == 0
    assert torch.equal(res[0], res[1])


def test_prefill_fp32():
    b = W.custom_prefill("f32", 8, 2, 64, [0, 40], [20, 9], seed=302)
    _check_step(b)


# ------------------------------------------------------------------ fused append + decode

@pytest.mark.parametrize("dtype,hq,hkv,d,lens,partition", [
    ("bf16", 32, 8, 128, [1, 16, 17, 512, 513, 1024, 1025, 3000, 0], 0),
    ("bf16", 32, 8, 128, [1, 16, 17, 512, 513, 1024, 1025, 3000], 512),
    ("bf16", 64, 2, 64, [5, 40, 700], 0),
    ("f32", 16, 4, 128, [1, 33, 600], 256),
    # head-warp schedule (partitions of at most 512 tokens and at least two
    # thread blocks per SM): two chunks of a 24-head group append the same
    # row; three kv heads leave a warp idle
    ("bf16", 48, 2, 128, [1, 17, 300, 512] * 80, 0),
    ("bf16", 12, 3, 128, [5, 200, 600, 1500] * 80, 512),
    ("bf16", 32, 8, 128, [3, 16, 17, 300, 511, 900] * 4, 128),
])
def test_decode_step_equals_append_then_decode(dtype, hq, hkv, d, lens, partition):
    b = W.custom_batch(dtype, len(lens), hq, hkv, d, lens, seed=501 + d + hq)
    # the generator's new tokens sit at position L-1 of each non-empty sequence
    S = len(lens)
    t = to_dev(b)
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    ref = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               b.scale, ref, max_context_len=max(lens), partition_size=partition)
    # new-token rows per sequence (zeros for empty sequences, which append nothing)
    k_new = torch.zeros((S, hkv, d), dtype=b.k_new.dtype, device="cuda")
    v_new = torch.zeros_like(k_new)
    rows = [i for i, L in enumerate(lens) if L > 0]
    k_new[rows] = t["k_new"]
    v_new[rows] = t["v_new"]
    got = torch.empty_like(ref)
    pkv.decode_step(t["q"], k_new, v_new, kc, vc, t["block_tables"], t["context_lens"], b.scale, got,
                    max_context_len=max(lens), partition_size=partition)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert_bits_equal(kc, t["k_cache"], "k_cache")
    assert_bits_equal(vc, t["v_cache"], "v_cache")
    assert torch.equal(got.cpu(), ref.cpu())


@pytest.mark.parametrize("name", ["llama3_8b_decode", "shared_prefix_cow"])
def test_decode_step_workload_parity(name):
    b = W.make_batch(name)
    kc_o, vc_o, out_o, _ = oracle_step(b)
    t = to_dev(b)
    if t["copy_pairs"] is not None and t["copy_pairs"].numel():
        pkv.copy_blocks(t["copy_pairs"], t["k_cache"], t["v_cache"])
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    pkv.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["block_tables"],
                    t["context_lens"], b.scale, out, max_context_len=b.max_context_len)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert_bits_equal(t["k_cache"], kc_o, "k_cache")
    assert_bits_equal(t["v_cache"], vc_o, "v_cache")
    assert_parity(out, out_o, b.dtype, name)


# ------------------------------------------------------------------ invariances (bitwise)

def test_block_relabelling_is_bitwise_invariant_on_gpu():
    b = W.make_batch("llama3_8b_decode", num_seqs=16)
    _, _, out_a, _ = gpu_step(b)
    NB = b.num_blocks
    pi = torch.from_numpy(np.random.default_rng(5).permutation(NB))
    kc = torch.empty_like(b.k_cache)
    vc = torch.empty_like(b.v_cache)
    kc[pi] = b.k_cache
    vc[pi] = b.v_cache
    b.k_cache, b.v_cache = kc, vc
    bt = b.block_tables
    b.block_tables = torch.where(bt >= 0, pi[bt.clamp(min=0).long()].to(torch.int32), bt)
    sm = b.slot_mapping
    b.slot_mapping = pi[sm // 16].to(torch.int64) * 16 + sm % 16
    _, _, out_b, _ = gpu_step(b)
    assert torch.equal(out_a.cpu(), out_b.cpu())


def test_append_to_another_slot_is_bitwise_invariant_on_gpu():
    # each sequence's last block moves to a spare block before the step: its
    # rows are copied there (copy_blocks), the table points at the copy and
    # the new token is appended into the copy; the output must not change
    b = W.make_batch("llama3_8b_decode", num_seqs=16)
    _, _, out_a, _ = gpu_step(b)
    S = b.num_seqs
    L = b.context_lens.long()
    last = (L - 1) // 16
    old = b.block_tables.long().gather(1, last.unsqueeze(1)).squeeze(1)
    used = set(b.block_tables[b.block_tables >= 0].tolist())
    spare = torch.tensor([x for x in range(b.num_blocks) if x not in used][:S], dtype=torch.int64)
    assert spare.numel() == S
    b.copy_pairs = torch.stack([old, spare], dim=1)
    bt = b.block_tables.clone()
    bt[torch.arange(S), last] = spare.to(torch.int32)
    b.block_tables = bt
    b.slot_mapping = spare * 16 + (L - 1) % 16
    _, _, out_b, _ = gpu_step(b)
    assert pkv.get_status() == 0
    assert torch.equal(out_a.cpu(), out_b.cpu())


def test_shared_prefix_equals_private_copies_on_gpu():
    b = W.make_batch("shared_prefix_cow", num_seqs=32)
    _, _, shared, _ = gpu_step(b)
    # give every sequence a private copy of the 128 prefix blocks
    P = b.meta["prefix_blocks"]
    S = b.num_seqs
    prefix = b.block_tables[0, :P].long()
    NB = b.num_blocks
    extra = S * P
    kc = torch.cat([b.k_cache, torch.empty((extra,) + b.k_cache.shape[1:], dtype=b.k_cache.dtype)])
    vc = torch.cat([b.v_cache, torch.empty((extra,) + b.v_cache.shape[1:], dtype=b.v_cache.dtype)])
    bt = b.block_tables.clone()
    for s in range(S):
        ids = torch.arange(NB + s * P, NB + (s + 1) * P)
        kc[ids] = b.k_cache[prefix]
        vc[ids] = b.v_cache[prefix]
        bt[s, :P] = ids.to(torch.int32)
    b.k_cache, b.v_cache, b.block_tables, b.num_blocks = kc, vc, bt, NB + extra
    _, _, private, _ = gpu_step(b)
    assert torch.equal(shared.cpu(), private.cpu())


# ------------------------------------------------------------------ device-side checks

def test_bad_block_id_is_flagged_and_skipped():
    lens = [40, 40]
    b = W.custom_batch("bf16", 2, 8, 2, 128, lens, seed=401, poison=False)
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    bt = t["block_tables"].clone()
    bt[0, 1] = b.num_blocks + 5  # out of range: must be skipped, not read
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], bt, t["context_lens"], b.scale,
                               out, max_context_len=64)
    flags = pkv.get_status()
    assert flags & pkv.STATUS_BITS["bad_block"]
    assert bool(torch.isfinite(out).all())
    # sequence 1 is untouched by the bad id
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, kc, vc)
    ref = oracle.decode(b.q[1:], kc, vc, b.block_tables[1:], b.context_lens[1:], b.scale)
    assert_parity(out[1:], ref, torch.bfloat16, "seq 1")


def test_bad_slot_is_flagged_and_skipped():
    b = W.custom_batch("bf16", 2, 8, 2, 128, [5, 9], seed=402, poison=False)
    t = to_dev(b)
    before = t["k_cache"].clone()
    slots = t["slot_mapping"].clone()
    slots[0] = b.num_blocks * 16 + 3
    slots[1] = -1  # padding: skipped silently
    pkv.kv_append(t["k_new"], t["v_new"], slots, t["k_cache"], t["v_cache"])
    assert pkv.get_status() & pkv.STATUS_BITS["bad_slot"]
    assert torch.equal(before.cpu(), t["k_cache"].cpu())


def test_too_long_context_is_flagged():
    b = W.custom_batch("bf16", 2, 8, 2, 128, [100, 30], seed=403, poison=False)
    t = to_dev(b)
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                               t["context_lens"], b.scale, out, max_context_len=64)
    assert pkv.get_status() & pkv.STATUS_BITS["bad_length"]


def test_bad_copy_pair_is_flagged():
    b = W.custom_batch("bf16", 1, 8, 2, 128, [20], seed=404, poison=False)
    t = to_dev(b)
    before = t["k_cache"].clone()
    pairs = torch.tensor([[0, b.num_blocks]], dtype=torch.int64, device="cuda")
    pkv.copy_blocks(pairs, t["k_cache"], t["v_cache"])
    assert pkv.get_status() & pkv.STATUS_BITS["bad_block"]
    assert torch.equal(before.cpu(), t["k_cache"].cpu())


def test_python_layer_rejects_bad_tensors():
    b = W.custom_batch("bf16", 2, 8, 2, 128, [5, 9], seed=405, poison=False)
    t = to_dev(b)
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        pkv.paged_attention_decode(t["q"].cpu(), t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], b.scale, out)
    with pytest.raises(TypeError):
        pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"].long(),
                                   t["context_lens"], b.scale, out)
    with pytest.raises(pkv.PkvError):
        pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], b.scale, out, partition_size=24)


# ------------------------------------------------------------------ shared-prefix (cascade) decode

def _cascade_step(b, prefix_len, out_dtype=torch.float32, fused=True, partition=0):
    t = to_dev(b)
    if t["copy_pairs"] is not None and t["copy_pairs"].numel():
        pkv.copy_blocks(t["copy_pairs"], t["k_cache"], t["v_cache"])
    if not fused:
        pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    out = torch.empty(b.q.shape, dtype=out_dtype, device="cuda")
    pkv.decode_shared_prefix(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                             b.scale, out, prefix_len, k_new=t["k_new"] if fused else None,
                             v_new=t["v_new"] if fused else None, max_context_len=b.max_context_len,
                             partition_size=partition)
    torch.cuda.synchronize()
    return t, out


def _prefill_call(b, t, out):
    cu = b.prefill_cu_q_lens
    pkv.paged_attention_prefill_chunk(
        t["prefill_q"], t["prefill_cu_q_lens"], t["k_cache"], t["v_cache"], t["prefill_block_tables"],
        t["prefill_context_lens"], b.scale, out, max_q_len=int((cu[1:] - cu[:-1]).max()),
        max_context_len=int(b.prefill_context_lens.max()))


def _replay_checks(call, out, expected, dtype, what, replays=3):
    # capture one call in a CUDA graph (after one plain call: attributes and
    # occupancy queries happen outside the capture), then replay it with the
    # output cleared each time
    call()
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for rep in range(replays):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_status() == 0, (what, rep)
        assert_parity(out, expected, dtype, f"{what}, graph replay {rep}")


def test_prefill_replays_from_a_cuda_graph():
    # A graph replays a launch with the parameters it was captured with, the
    # work counter's launch tag included: every replay must still hand out
    # all of its items (the kernel clears the counter's tags when it ends).
    b = W.custom_prefill("bf16", 32, 8, 128, [0, 3072], [512, 512], seed=37)
    _, _, _, pout_o = oracle_step(b)
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    cu = b.prefill_cu_q_lens
    mq, mc = int((cu[1:] - cu[:-1]).max()), int(b.prefill_context_lens.max())
    ws = torch.empty(max(1, pkv.prefill_workspace_bytes(int(cu.numel()) - 1, b.prefill_q.shape[0], 32, 8, 128,
                                                         mq, mc)), dtype=torch.uint8, device="cuda")
    out = torch.empty(b.prefill_q.shape, dtype=torch.float32, device="cuda")

    def call():
        pkv.paged_attention_prefill_chunk(
            t["prefill_q"], t["prefill_cu_q_lens"], t["k_cache"], t["v_cache"], t["prefill_block_tables"],
            t["prefill_context_lens"], b.scale, out, max_q_len=mq, max_context_len=mc, workspace=ws)

    _replay_checks(call, out, pout_o, b.dtype, "prefill")


def test_shared_prefix_decode_replays_from_a_cuda_graph():
    # 1024 sequences: 4096 query rows per kv head, 128 prefix items, more
    # than one per resident CTA pair, so items also come from the counter
    b = W.make_batch("shared_prefix_cow", num_seqs=1024, ctx=(16, 200), prefix_blocks=8)
    _, _, out_o, _ = oracle_step(b)
    t = to_dev(b)
    pkv.copy_blocks(t["copy_pairs"], t["k_cache"], t["v_cache"])
    S, Hq, d = b.q.shape
    P = 8 * 16
    ws = torch.empty(pkv.decode_shared_prefix_workspace_bytes(S, Hq, d, b.max_context_len, P),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")

    def call():
        # (the fused append writes the same rows on every replay)
        pkv.decode_shared_prefix(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                                 b.scale, out, P, k_new=t["k_new"], v_new=t["v_new"],
                                 max_context_len=b.max_context_len, workspace=ws)

    _replay_checks(call, out, out_o, b.dtype, "cascade decode")


def test_prefill_wait_limit_runs_out_and_is_reported():
    # The tensor-core kernel's waits are bounded in time.  With a bound of 1 ns
    # a wait runs out at once: the launch must stop, record the internal status
    # bit and return (no hang, no fault), and the next launch with the default
    # bound must be correct again.
    b = W.custom_prefill("bf16", 32, 8, 128, [0, 3072], [512, 512], seed=31)
    kc_o, vc_o, _, pout_o = oracle_step(b)
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    out = torch.zeros(b.prefill_q.shape, dtype=torch.float32, device="cuda")
    pkv.set_wait_limit_ns(1)
    try:
        _prefill_call(b, t, out)
        torch.cuda.synchronize()
        status = pkv.get_status()
    finally:
        pkv.set_wait_limit_ns(0)
    assert status & pkv.STATUS_BITS["internal"], status
    out = torch.empty(b.prefill_q.shape, dtype=torch.float32, device="cuda")
    _prefill_call(b, t, out)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert_parity(out, pout_o, b.dtype, "prefill after a run-out launch")


def test_decode_on_a_side_stream_keeps_its_workspace():
    # The binding allocates the split-K workspace on the current stream and
    # the call runs on another one; the current stream then allocates a
    # buffer of the same size and overwrites it while the decode may still be
    # running.  The workspace must not be handed out again before the decode
    # is done with it.
    b = W.make_batch("llama3_8b_decode")
    _, _, out_o, _ = oracle_step(b, prefill=False)
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    out = torch.full(b.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    need = pkv.decode_workspace_bytes(b.q.shape[0], b.q.shape[1], b.q.shape[2], b.max_context_len, 512)
    for _ in range(3):
        pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                                   b.scale, out, max_context_len=b.max_context_len, partition_size=512,
                                   stream=side)
        junk = torch.empty(need, dtype=torch.uint8, device="cuda")
        junk.fill_(0xFF)
        del junk
    torch.cuda.synchronize()
    assert_parity(out, out_o, b.dtype, "decode on a side stream")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_shared_prefix_cascade_workload(out_dtype):
    b = W.make_batch("shared_prefix_cow")
    prefix_len = b.meta["prefix_blocks"] * 16
    kc_o, vc_o, out_o, _ = oracle_step(b)
    t, out = _cascade_step(b, prefix_len, out_dtype)
    assert pkv.get_status() == 0
    assert_bits_equal(t["k_cache"], kc_o, "k_cache")
    assert_bits_equal(t["v_cache"], vc_o, "v_cache")
    assert_parity(out, out_o, b.dtype, "cascade decode")


@pytest.mark.parametrize("num_seqs,prefix_blocks,ctx,fused,partition,heads", [
    (40, 3, (16, 300), True, 0, (32, 8)),       # 48-token prefix (one partial key tile), 160 query rows
    (5, 9, (1, 40), False, 0, (32, 8)),         # tiny suffixes, one row tile, append outside
    (64, 20, (100, 2000), True, 256, (32, 8)),  # long suffixes split in 256-token partitions
    (160, 4, (16, 600), True, 256, (32, 8)),    # head-warp suffix partitions with partials
    (24, 5, (16, 200), True, 0, (64, 8)),       # group of 8: every row of the transposed tile
    (48, 6, (1, 700), True, 0, (8, 4)),         # group of 2
    (20, 7, (10, 500), True, 0, (48, 4)),       # group of 12: the kernel with queries on M
])
def test_shared_prefix_cascade_shapes(num_seqs, prefix_blocks, ctx, fused, partition, heads):
    b = W.make_batch("shared_prefix_cow", num_seqs=num_seqs, ctx=ctx, prefix_blocks=prefix_blocks,
                     heads=heads)
    kc_o, vc_o, out_o, _ = oracle_step(b)
    t, out = _cascade_step(b, prefix_blocks * 16, fused=fused, partition=partition)
    assert pkv.get_status() == 0
    assert_bits_equal(t["k_cache"], kc_o, "k_cache")
    assert_bits_equal(t["v_cache"], vc_o, "v_cache")
    assert_parity(out, out_o, b.dtype, "cascade decode")
