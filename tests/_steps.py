"""One step of the hot path through the oracle and through the library, on the
same seeded batch, plus the comparison rules the parity tests share."""

from __future__ import annotations

import torch

import oracle
import paged_kv_cache_297_gb300 as pkv

# Parity tolerances: fp32 max abs 1e-4; bf16 (fp32 accumulation) max abs
# 1e-2 and mean abs 1e-3, checked on an fp32 output.  A bf16 output adds its
# own final rounding: |err| <= 1e-2 + 2^-8 |ref|.
TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (1e-2, 1e-3)}


def oracle_step(b, prefill=True):
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    if b.copy_pairs is not None and b.copy_pairs.numel():
        oracle.copy_blocks(kc, vc, b.copy_pairs)
    oracle.kv_append(b.k_new, b.v_new, b.slot_mapping, kc, vc)
    out = oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale) \
        if b.q.shape[0] else torch.zeros(0, dtype=torch.float64)
    pout = None
    if prefill and b.prefill_q is not None:
        pout = oracle.prefill_chunk(b.prefill_q, b.prefill_cu_q_lens, kc, vc,
                                    b.prefill_block_tables, b.prefill_context_lens, b.scale)
    return kc, vc, out, pout


def to_dev(b, dev="cuda"):
    d = {}
    for name in ("k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "q", "block_tables",
                 "context_lens", "copy_pairs", "prefill_q", "prefill_cu_q_lens",
                 "prefill_block_tables", "prefill_context_lens"):
        t = getattr(b, name)
        d[name] = None if t is None else t.to(dev)
    return d


def gpu_step(b, out_dtype=torch.float32, partition_size=0, prefill=True, dev="cuda"):
    t = to_dev(b, dev)
    if t["copy_pairs"] is not None and t["copy_pairs"].numel():
        pkv.copy_blocks(t["copy_pairs"], t["k_cache"], t["v_cache"])
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    out = torch.empty(b.q.shape, dtype=out_dtype, device=dev)
    if b.q.shape[0]:
        pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], b.scale, out,
                                   max_context_len=max(1, b.max_context_len),
                                   partition_size=partition_size)
    pout = None
    if prefill and b.prefill_q is not None:
        pout = torch.empty(b.prefill_q.shape, dtype=out_dtype, device=dev)
        cu = b.prefill_cu_q_lens
        pkv.paged_attention_prefill_chunk(
            t["prefill_q"], t["prefill_cu_q_lens"], t["k_cache"], t["v_cache"],
            t["prefill_block_tables"], t["prefill_context_lens"], b.scale, pout,
            max_q_len=int((cu[1:] - cu[:-1]).max()),
            max_context_len=int(b.prefill_context_lens.max()))
    torch.cuda.synchronize()
    return t["k_cache"], t["v_cache"], out, pout


def bits(t: torch.Tensor) -> torch.Tensor:
    """Bit pattern view (so NaN-poisoned rows compare equal to themselves)."""
    t = t.cpu().contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_bits_equal(a: torch.Tensor, b: torch.Tensor, what: str) -> None:
    eq = bits(a) == bits(b)
    if not bool(eq.all()):
        bad = (~eq).nonzero()[:5].tolist()
        raise AssertionError(f"{what}: {int((~eq).sum())} elements differ, first at {bad}")


def err_stats(got: torch.Tensor, ref: torch.Tensor):
    g = got.detach().float().cpu().double()
    assert bool(torch.isfinite(g).all()), "non-finite output"
    e = (g - ref).abs()
    return float(e.max()) if e.numel() else 0.0, float(e.mean()) if e.numel() else 0.0


def assert_parity(got: torch.Tensor, ref: torch.Tensor, in_dtype: torch.dtype, what: str):
    mx, mean = err_stats(got, ref)
    tmax, tmean = TOL[in_dtype]
    if got.dtype == torch.bfloat16:
        g = got.float().cpu().double()
        bound = 1e-2 + 2.0 ** -8 * ref.abs()
        worst = float(((g - ref).abs() - bound).max()) if g.numel() else -1.0
        assert worst <= 0, f"{what}: bf16 output exceeds 1e-2 + 2^-8|ref| by {worst:.3g}"
        return mx, mean
    assert mx <= tmax, f"{what}: max abs err {mx:.3g} > {tmax}"
    assert mean <= tmean, f"{what}: mean abs err {mean:.3g} > {tmean}"
    return mx, mean
