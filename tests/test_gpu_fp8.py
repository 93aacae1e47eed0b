"""fp8 E4M3 KV cache on the GPU against the oracle: the quantising append and
the block copy bit-exact, decode within the bf16 tolerances (the cache values
are exact; the query and the softmax weights enter the products as fp16)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_297_gb300 as pkv
from paged_kv_cache_297_gb300 import workloads as W
from tests._steps import assert_parity, to_dev

pytestmark = pytest.mark.gpu

EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 511, 512, 513, 1023, 1024, 1025, 2047]


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        pkv.get_status()
    yield
    if torch.cuda.is_available():
        pkv.get_status()


def _fp8_step(b, out_dtype=torch.float32, partition_size=0):
    """(oracle output, GPU output, oracle caches, GPU caches) for one
    append + decode step over the fp8 caches of batch b."""
    kc_o, vc_o = b.k_cache.clone(), b.v_cache.clone()
    oracle.kv_append_fp8(b.k_new, b.v_new, b.slot_mapping, kc_o, vc_o, b.k_scale, b.v_scale)
    ref = oracle.decode(b.q, kc_o, vc_o, b.block_tables, b.context_lens, b.scale, b.k_scale, b.v_scale)
    t = to_dev(b)
    ks, vs = b.k_scale.cuda(), b.v_scale.cuda()
    pkv.kv_append_fp8(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"], ks, vs)
    out = torch.empty(b.q.shape, dtype=out_dtype, device="cuda")
    if b.q.shape[0]:
        pkv.paged_attention_decode_fp8(t["q"], t["k_cache"], t["v_cache"], ks, vs, t["block_tables"],
                                       t["context_lens"], b.scale, out, max_context_len=max(1, b.max_context_len),
                                       partition_size=partition_size)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    return ref, out, (kc_o, vc_o), (t["k_cache"].cpu(), t["v_cache"].cpu())


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_fp8_append_is_bit_exact(in_dtype):
    NB, H, d = 40, 8, 128
    g = torch.Generator().manual_seed(21)
    # magnitudes from tiny to past 448 after scaling, so every rounding regime
    # (subnormal, normal, saturated) occurs
    k = (torch.randn(300, H, d, generator=g) * torch.logspace(-4, 2, d)).to(in_dtype)
    v = (torch.randn(300, H, d, generator=g) * 3).to(in_dtype)
    ks = 2.0 ** -3 * (1 + torch.arange(H, dtype=torch.float32) / 3)
    vs = 0.011 * (1 + torch.arange(H, dtype=torch.float32))
    slots = torch.from_numpy(np.random.Generator(np.random.PCG64(5)).permutation(NB * 16)[:300].astype(np.int64))
    slots[::37] = -1
    kc = torch.full((NB, H, 16, d), 0x5A, dtype=torch.uint8)
    vc = kc.clone()
    kc_o, vc_o = kc.clone(), vc.clone()
    oracle.kv_append_fp8(k, v, slots, kc_o, vc_o, ks, vs)
    kc_g, vc_g = kc.cuda(), vc.cuda()
    pkv.kv_append_fp8(k.cuda(), v.cuda(), slots.cuda(), kc_g, vc_g, ks.cuda(), vs.cuda())
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert torch.equal(kc_g.cpu(), kc_o) and torch.equal(vc_g.cpu(), vc_o)
    assert bool((kc_o == 0x7E).any()) and bool((kc_o & 0x78 == 0).any())  # saturated and subnormal codes seen


def test_fp8_copy_blocks_is_bit_exact():
    g = torch.Generator().manual_seed(8)
    kc = torch.randint(0, 256, (24, 8, 16, 128), dtype=torch.uint8, generator=g)
    vc = torch.randint(0, 256, (24, 8, 16, 128), dtype=torch.uint8, generator=g)
    pairs = torch.tensor([[3, 10], [7, 0], [23, 5]], dtype=torch.int64)
    kc_o, vc_o = kc.clone(), vc.clone()
    oracle.copy_blocks(kc_o, vc_o, pairs)
    kc_g, vc_g = kc.cuda(), vc.cuda()
    pkv.copy_blocks(pairs.cuda(), kc_g, vc_g)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert torch.equal(kc_g.cpu(), kc_o) and torch.equal(vc_g.cpu(), vc_o)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_llama3_workload(out_dtype):
    b = W.fp8_batch(W.make_batch("llama3_8b_decode"))
    ref, out, (kc_o, vc_o), (kc_g, vc_g) = _fp8_step(b, out_dtype)
    assert torch.equal(kc_g, kc_o) and torch.equal(vc_g, vc_o)
    assert_parity(out, ref, torch.bfloat16, "fp8 decode")


@pytest.mark.parametrize("partition", [0, 512])
def test_fp8_long_context_workload(partition):
    # 8 sequences of 32k-131k tokens with 1% of K and V rows scaled by 20: the
    # largest softmax weights meet the outlier V rows, and q and P enter the
    # products as fp16; the adaptive partition and 512-token partitions (the
    # longest reduce rows)
    b = W.fp8_batch(W.make_batch("long_context"))
    ref, out, (kc_o, vc_o), (kc_g, vc_g) = _fp8_step(b, partition_size=partition)
    assert torch.equal(kc_g, kc_o) and torch.equal(vc_g, vc_o)
    assert_parity(out, ref, torch.bfloat16, "fp8 long-context decode")


@pytest.mark.parametrize("hq,hkv,partition", [(32, 8, 0), (64, 8, 512), (16, 1, 0), (48, 2, 256)])
def test_fp8_edge_lengths(hq, hkv, partition):
    b = W.fp8_batch(W.custom_batch("bf16", len(EDGE_LENS), hq, hkv, 128, EDGE_LENS, seed=41 + hq))
    ref, out, _, _ = _fp8_step(b, partition_size=partition)
    assert_parity(out, ref, torch.bfloat16, "fp8 decode")


def test_fp8_head_warp_schedule():
    # many short sequences: partitions of at most 512 tokens, one warp per kv head
    lens = np.random.Generator(np.random.PCG64(3)).integers(1, 400, 320).tolist()
    b = W.fp8_batch(W.custom_batch("bf16", len(lens), 32, 8, 128, lens, seed=77))
    ref, out, _, _ = _fp8_step(b)
    assert_parity(out, ref, torch.bfloat16, "fp8 decode")


@pytest.mark.parametrize("case", ["llama3", "edges", "head_warps"])
def test_fp8_decode_step_equals_append_then_decode(case):
    # the fused call writes the same codes as kv_append_fp8 and then reads the
    # same cache: caches and outputs bitwise equal to the two calls
    if case == "llama3":
        b = W.fp8_batch(W.make_batch("llama3_8b_decode"))
    elif case == "edges":
        b = W.fp8_batch(W.custom_batch("bf16", len(EDGE_LENS), 32, 8, 128, EDGE_LENS, seed=43))
    else:
        lens = np.random.Generator(np.random.PCG64(5)).integers(1, 400, 320).tolist()
        b = W.fp8_batch(W.custom_batch("bf16", len(lens), 32, 8, 128, lens, seed=79))
    live = b.context_lens > 0
    mc = max(1, b.max_context_len)
    ta, tb = to_dev(b), to_dev(b)
    ks, vs = b.k_scale.cuda(), b.v_scale.cuda()
    out_a = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    out_b = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    pkv.kv_append_fp8(ta["k_new"], ta["v_new"], ta["slot_mapping"], ta["k_cache"], ta["v_cache"], ks, vs)
    pkv.paged_attention_decode_fp8(ta["q"], ta["k_cache"], ta["v_cache"], ks, vs, ta["block_tables"],
                                   ta["context_lens"], b.scale, out_a, max_context_len=mc)
    # the fused call takes one row per sequence (sequences with L = 0 append nothing)
    S, Hkv, d = b.q.shape[0], b.k_cache.shape[1], b.k_cache.shape[3]
    k_new = torch.zeros((S, Hkv, d), dtype=torch.bfloat16, device="cuda")
    v_new = torch.zeros((S, Hkv, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.nonzero(live).flatten().cuda()
    k_new[idx] = tb["k_new"][: idx.numel()]
    v_new[idx] = tb["v_new"][: idx.numel()]
    pkv.decode_step_fp8(tb["q"], k_new, v_new, tb["k_cache"], tb["v_cache"], ks, vs, tb["block_tables"],
                        tb["context_lens"], b.scale, out_b, max_context_len=mc)
    torch.cuda.synchronize()
    assert pkv.get_status() == 0
    assert torch.equal(ta["k_cache"], tb["k_cache"]) and torch.equal(ta["v_cache"], tb["v_cache"])
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("case", range(6))
def test_fp8_random_shapes(case):
    # Seeded random fp8 batches: groups 1-16, lengths 1 token to 20k,
    # adaptive or fixed partitions, both output types; caches bit-exact.
    import random
    rng = random.Random(7400 + case)
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 4, 8, 12, 16])
    S = rng.randint(1, 48)
    hi = rng.choice([600, 5000, 20000])
    lens = [rng.choice([1, rng.randint(16, hi), rng.randint(1, 64)]) for _ in range(S)]
    b = W.fp8_batch(W.custom_batch("bf16", S, hkv * g, hkv, 128, lens, seed=rng.randint(1, 10 ** 6)))
    ref, out, (kc_o, vc_o), (kc_g, vc_g) = _fp8_step(b, rng.choice([torch.float32, torch.bfloat16]),
                                                       partition_size=rng.choice([0, 256, 512, 1536]))
    assert torch.equal(kc_g, kc_o) and torch.equal(vc_g, vc_o)
    assert_parity(out, ref, torch.bfloat16, "fp8 decode")


def test_fp8_rejects_what_it_does_not_support():
    b = W.fp8_batch(W.custom_batch("bf16", 2, 8, 8, 64, [5, 9], seed=2))
    t = to_dev(b)
    out = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PkvError):   # head_dim 64
        pkv.paged_attention_decode_fp8(t["q"], t["k_cache"], t["v_cache"], b.k_scale.cuda(), b.v_scale.cuda(),
                                       t["block_tables"], t["context_lens"], b.scale, out)
    with pytest.raises(pkv.PkvError):   # the plain append does not quantise
        pkv.kv_append(t["k_new"].to(torch.uint8), t["v_new"].to(torch.uint8), t["slot_mapping"], t["k_cache"],
                      t["v_cache"])
