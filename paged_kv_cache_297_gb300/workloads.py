"""Seeded synthetic inputs for the paged KV-cache paths.

This module only *draws* inputs: shapes, value distributions and structure
(ragged context lengths, shuffled physical block ids, shared prefixes, forks,
prompt chunks).  It holds none of the attention arithmetic, and it is the one
module that both the oracle-side tests and the CUDA path consume.

Cache layout (the reading this library takes of the paged KV cache described in
"Serving deep dive" / "PagedAttention" and the chengxuchu PyTorch #47 page,
section 5.2): K and V are separate tensors of shape
``[num_blocks, num_kv_heads, BLOCK_SIZE, head_dim]``; logical token ``t`` of
sequence ``s`` lives in physical block ``block_tables[s, t // BLOCK_SIZE]`` at
row ``t % BLOCK_SIZE``.  ``slot = block * BLOCK_SIZE + row`` names one row.

Every batch is drawn on the host from a ``numpy`` PCG64 stream seeded with
``20260000 + index`` and materialised as CPU torch tensors, so that the oracle
and the GPU see identical bytes.  Normal draws are chunked over independent
child streams (``SeedSequence.spawn``) so the bytes do not depend on how many
threads generate them.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16  # tokens per block ("usually 16 tokens per block", ainews page)
SEED_BASE = 20260000
_CHUNK = 1 << 22  # elements per independent normal stream


# ----------------------------------------------------------------------------
# workload catalogue
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Spec:
    name: str
    index: int
    dtype: str  # "f32" | "bf16"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx_lo: int = 1
    ctx_hi: int = 1
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    fixed_pool: Optional[int] = None
    description: str = ""


SPECS = {
    "tiny_fp32": Spec(
        "tiny_fp32", 1, "f32", 4, 4, 4, 64, 1, 64, fixed_pool=32,
        description="4 seqs, 4 q = 4 kv heads, d 64, context U[1,64], pool of 32 "
                    "shuffled blocks, N(0,1), scale 1/8, one appended token per seq"),
    "llama3_8b_decode": Spec(
        "llama3_8b_decode", 2, "bf16", 64, 32, 8, 128, 512, 4096,
        description="Llama-3-8B-shaped decode layer: 64 seqs, 32 q / 8 kv heads, d 128, "
                    "context U[512,4096], pool 1.2x need, shuffled, N(0,1)"),
    "long_context": Spec(
        "long_context", 3, "bf16", 8, 64, 8, 128, 32768, 131072,
        outlier_p=0.01, outlier_scale=20.0,
        description="long-context decode: 8 seqs, 64 q / 8 kv heads, d 128, context "
                    "U[32768,131072], 1% of K and V rows scaled x20"),
    "shared_prefix_cow": Spec(
        "shared_prefix_cow", 4, "bf16", 256, 32, 8, 128, 16, 512,
        description="256 seqs share a 2048-token prefix (128 blocks), private suffix "
                    "U[16,512]; 10% of seqs fork mid-block and copy-on-write the partial "
                    "block before the append"),
    "mixed_step": Spec(
        "mixed_step", 5, "bf16", 128, 32, 8, 128, 256, 8192,
        description="128 decode seqs (context U[256,8192]) + 2 prefill chunks of 512 "
                    "tokens with prior context 0 and 3072, one paged cache"),
}

# The workload the headline throughput is quoted on.
HEADLINE = "llama3_8b_decode"


@dataclass
class Batch:
    """One step's worth of synthetic input over one paged cache (host tensors)."""

    spec: Spec
    dtype: torch.dtype
    scale: float
    num_blocks: int
    k_cache: torch.Tensor          # [NB, Hkv, 16, d], state *before* this step
    v_cache: torch.Tensor
    k_new: torch.Tensor            # [T, Hkv, d] tokens appended this step
    v_new: torch.Tensor
    slot_mapping: torch.Tensor     # [T] int64
    # decode part
    q: torch.Tensor                # [S, Hq, d]
    block_tables: torch.Tensor     # [S, max_blocks] int32, -1 past the end
    context_lens: torch.Tensor     # [S] int32, includes the appended token
    # copy-on-write pairs (src, dst) to run before the append, or None
    copy_pairs: Optional[torch.Tensor] = None
    # chunked-prefill part (mixed step only)
    prefill_q: Optional[torch.Tensor] = None            # [sum n, Hq, d]
    prefill_cu_q_lens: Optional[torch.Tensor] = None    # [P+1] int32
    prefill_block_tables: Optional[torch.Tensor] = None  # [P, max_blocks] int32
    prefill_context_lens: Optional[torch.Tensor] = None  # [P] int32
    # fp8 E4M3 caches (k_cache / v_cache are uint8 codes): per kv head scales
    k_scale: Optional[torch.Tensor] = None               # [Hkv] float32
    v_scale: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.numel() else 0


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------

def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _fill_normal(dst: torch.Tensor, seed: int, outlier_p: float = 0.0,
                 outlier_scale: float = 1.0, row: int = 1,
                 threads: Optional[int] = None) -> None:
    """Fill ``dst`` (contiguous, any float dtype) with N(0,1) draws.

    With ``outlier_p > 0`` each run of ``row`` consecutive elements (one K or V
    row of one kv head) is multiplied by ``outlier_scale`` with probability
    ``outlier_p``, after sampling and before rounding to ``dst``'s dtype.
    """
    flat = dst.view(-1)
    n = flat.numel()
    if n == 0:
        return
    chunk = max(row, (_CHUNK // row) * row)
    nchunks = (n + chunk - 1) // chunk
    children = np.random.SeedSequence(seed).spawn(nchunks)

    def work(i: int) -> None:
        a = i * chunk
        b = min(n, a + chunk)
        g = np.random.Generator(np.random.PCG64(children[i]))
        x = g.standard_normal(b - a, dtype=np.float32)
        if outlier_p > 0.0:
            nrow = (b - a) // row
            hit = g.random(nrow) < outlier_p
            x.reshape(nrow, row)[hit] *= np.float32(outlier_scale)
        flat[a:b].copy_(torch.from_numpy(x))

    threads = threads or min(32, os.cpu_count() or 1)
    if nchunks == 1 or threads == 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))


def _poison_value(dtype: torch.dtype) -> float:
    return float("nan")


# ----------------------------------------------------------------------------
# structure helpers (block tables, slots)
# ----------------------------------------------------------------------------

def _slots_of(table_row: np.ndarray, first: int, count: int) -> np.ndarray:
    """Slots of logical tokens [first, first+count) of one sequence."""
    t = np.arange(first, first + count, dtype=np.int64)
    return table_row[t // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + (t % BLOCK_SIZE)


def _make_cache(spec: Spec, num_blocks: int, seed: int, used_slots: np.ndarray,
                poison: bool) -> tuple[torch.Tensor, torch.Tensor]:
    dt = _torch_dtype(spec.dtype)
    shape = (num_blocks, spec.num_kv_heads, BLOCK_SIZE, spec.head_dim)
    k = torch.empty(shape, dtype=dt)
    v = torch.empty(shape, dtype=dt)
    _fill_normal(k, seed * 16 + 1, spec.outlier_p, spec.outlier_scale, spec.head_dim)
    _fill_normal(v, seed * 16 + 2, spec.outlier_p, spec.outlier_scale, spec.head_dim)
    if poison:
        # every row that holds no token of the pre-step state reads as NaN
        unused = np.ones(num_blocks * BLOCK_SIZE, dtype=bool)
        unused[used_slots] = False
        idx = torch.from_numpy(np.nonzero(unused)[0])
        blk, row = idx // BLOCK_SIZE, idx % BLOCK_SIZE
        nan = _poison_value(dt)
        k[blk, :, row, :] = nan
        v[blk, :, row, :] = nan
    return k, v


def _new_tokens(spec: Spec, count: int, seed: int) -> tuple[torch.Tensor, torch.Tensor]:
    dt = _torch_dtype(spec.dtype)
    k = torch.empty((count, spec.num_kv_heads, spec.head_dim), dtype=dt)
    v = torch.empty_like(k)
    _fill_normal(k, seed * 16 + 3, spec.outlier_p, spec.outlier_scale, spec.head_dim)
    _fill_normal(v, seed * 16 + 4, spec.outlier_p, spec.outlier_scale, spec.head_dim)
    return k, v


def _queries(spec: Spec, rows: int, seed: int, salt: int = 5) -> torch.Tensor:
    q = torch.empty((rows, spec.num_q_heads, spec.head_dim), dtype=_torch_dtype(spec.dtype))
    _fill_normal(q, seed * 16 + salt)
    return q


def _tables(lists: list[np.ndarray], width: int) -> torch.Tensor:
    t = np.full((len(lists), max(1, width)), -1, dtype=np.int32)
    for i, row in enumerate(lists):
        t[i, : len(row)] = row
    return torch.from_numpy(t)


# ----------------------------------------------------------------------------
# batch builders
# ----------------------------------------------------------------------------

def _decode_batch(spec: Spec, seed: int, poison: bool, lens: Optional[np.ndarray] = None,
                  pool_factor: float = 1.2) -> Batch:
    rng = np.random.Generator(np.random.PCG64(seed))
    S = spec.num_seqs
    if lens is None:
        lens = rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=S).astype(np.int64)
    lens = np.asarray(lens, dtype=np.int64)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = int(nblk.sum())
    NB = spec.fixed_pool if spec.fixed_pool else max(1, int(math.ceil(pool_factor * need)))
    assert NB >= need
    perm = rng.permutation(NB).astype(np.int32)
    rows, used, new_slots, off = [], [], [], 0
    for s in range(S):
        row = perm[off: off + nblk[s]]
        off += nblk[s]
        rows.append(row)
        L = int(lens[s])
        if L > 0:
            used.append(_slots_of(row, 0, L - 1))
            new_slots.append(_slots_of(row, L - 1, 1))
    used = np.concatenate(used) if used else np.zeros(0, np.int64)
    k_cache, v_cache = _make_cache(spec, NB, seed, used, poison)
    T = len(new_slots)
    k_new, v_new = _new_tokens(spec, T, seed)
    slot_mapping = torch.from_numpy(np.concatenate(new_slots) if new_slots
                                    else np.zeros(0, np.int64))
    width = int(max(1, math.ceil(spec.ctx_hi / BLOCK_SIZE)))
    return Batch(
        spec=spec, dtype=_torch_dtype(spec.dtype), scale=1.0 / math.sqrt(spec.head_dim),
        num_blocks=NB, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=slot_mapping, q=_queries(spec, S, seed),
        block_tables=_tables(rows, max(width, int(nblk.max(initial=1)))),
        context_lens=torch.from_numpy(lens.astype(np.int32)),
        meta={"pool_need": need})


def _shared_prefix_batch(spec: Spec, seed: int, poison: bool,
                         prefix_blocks: int = 128, fork_frac: float = 0.10) -> Batch:
    """256 sequences over one refcounted 2048-token prefix, with forks.

    A fork's child shares *all* of its parent's blocks, including the parent's
    partially filled last block.  Before the step's append the child's shared
    partial block is copied to a fresh block (copy-on-write, ainews page,
    "PagedAttention" paragraph), and the child's table is pointed at the copy;
    ``copy_pairs`` lists those (src, dst) copies.  The copy targets hold NaN
    until the copy runs, so a skipped copy is visible in the child's output.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    S = spec.num_seqs
    P = prefix_blocks * BLOCK_SIZE
    suffix = rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=S).astype(np.int64)
    pre = P + suffix                       # tokens before this step's append
    n_fork = int(round(fork_frac * S))
    order = rng.permutation(S)
    parents = [int(i) for i in order if pre[i] % BLOCK_SIZE != 0][:n_fork]
    rest = [int(i) for i in order if int(i) not in set(parents)]
    children = rest[:n_fork]
    parent_of = dict(zip(children, parents))
    for c, p in parent_of.items():
        pre[c] = pre[p]
    lens = pre + 1

    # block needs: prefix once; private blocks for every non-child; one fresh
    # block for a non-child whose append opens a new block; one CoW block per child
    priv = {}
    for s in range(S):
        if s in parent_of:
            continue
        priv[s] = int((pre[s] + BLOCK_SIZE - 1) // BLOCK_SIZE) - prefix_blocks
    extra = sum(1 for s in range(S) if s not in parent_of and pre[s] % BLOCK_SIZE == 0)
    need = prefix_blocks + sum(priv.values()) + extra + n_fork
    NB = int(math.ceil(1.2 * need))
    perm = rng.permutation(NB).astype(np.int32)
    cur = 0

    def take(n: int) -> np.ndarray:
        nonlocal cur
        out = perm[cur: cur + n]
        cur += n
        return out

    prefix = take(prefix_blocks)
    rows: list[Optional[np.ndarray]] = [None] * S
    for s in range(S):
        if s in parent_of:
            continue
        rows[s] = np.concatenate([prefix, take(priv[s])])
    for s in range(S):
        if s not in parent_of and pre[s] % BLOCK_SIZE == 0:
            rows[s] = np.concatenate([rows[s], take(1)])
    pairs = []
    for c, p in parent_of.items():
        nb = int((pre[p] + BLOCK_SIZE - 1) // BLOCK_SIZE)
        src = rows[p][nb - 1]
        dst = take(1)[0]
        row = rows[p][:nb].copy()
        row[nb - 1] = dst
        rows[c] = row
        pairs.append((int(src), int(dst)))
    # slots holding a pre-step token: the prefix, then each non-child's suffix
    used = [_slots_of(prefix, 0, P)]
    for s in range(S):
        if s in parent_of:
            continue
        used.append(_slots_of(rows[s], P, int(pre[s]) - P))
    used = np.concatenate(used)
    k_cache, v_cache = _make_cache(spec, NB, seed, used, poison)
    new_slots = np.concatenate([_slots_of(rows[s], int(pre[s]), 1) for s in range(S)])
    k_new, v_new = _new_tokens(spec, S, seed)
    width = prefix_blocks + int(math.ceil((spec.ctx_hi + 1) / BLOCK_SIZE))
    return Batch(
        spec=spec, dtype=_torch_dtype(spec.dtype), scale=1.0 / math.sqrt(spec.head_dim),
        num_blocks=NB, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(new_slots), q=_queries(spec, S, seed),
        block_tables=_tables(rows, width),
        context_lens=torch.from_numpy(lens.astype(np.int32)),
        copy_pairs=torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2),
        meta={"pool_need": need, "children": sorted(parent_of), "parent_of": parent_of,
              "prefix_blocks": prefix_blocks,
              "unique_tokens": int(P + sum(int(pre[s]) - P for s in range(S)
                                               if s not in parent_of) + S)})


def _mixed_batch(spec: Spec, seed: int, poison: bool, chunk: int = 512,
                 priors: tuple[int, ...] = (0, 3072)) -> Batch:
    """128 decode sequences plus prompt chunks over one paged cache.

    Each chunk sequence has ``prior`` tokens already cached and appends ``chunk``
    new ones this step (chunked prefill, caffein.top page, "Chunked Prefill");
    its queries sit at absolute positions prior .. prior+chunk-1.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    S = spec.num_seqs
    lens = rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=S).astype(np.int64)
    plens = np.asarray([p + chunk for p in priors], dtype=np.int64)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    pblk = (plens + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = int(nblk.sum() + pblk.sum())
    NB = int(math.ceil(1.2 * need))
    perm = rng.permutation(NB).astype(np.int32)
    off = 0
    rows, prow = [], []
    for s in range(S):
        rows.append(perm[off: off + nblk[s]])
        off += nblk[s]
    for i in range(len(priors)):
        prow.append(perm[off: off + pblk[i]])
        off += pblk[i]
    used = [_slots_of(rows[s], 0, int(lens[s]) - 1) for s in range(S)]
    used += [_slots_of(prow[i], 0, priors[i]) for i in range(len(priors))]
    used = np.concatenate(used)
    k_cache, v_cache = _make_cache(spec, NB, seed, used, poison)
    new_slots = [_slots_of(rows[s], int(lens[s]) - 1, 1) for s in range(S)]
    new_slots += [_slots_of(prow[i], priors[i], chunk) for i in range(len(priors))]
    new_slots = np.concatenate(new_slots)
    k_new, v_new = _new_tokens(spec, len(new_slots), seed)
    cu = np.zeros(len(priors) + 1, dtype=np.int32)
    cu[1:] = np.cumsum([chunk] * len(priors))
    width = int(math.ceil(max(spec.ctx_hi, int(plens.max())) / BLOCK_SIZE))
    return Batch(
        spec=spec, dtype=_torch_dtype(spec.dtype), scale=1.0 / math.sqrt(spec.head_dim),
        num_blocks=NB, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(new_slots), q=_queries(spec, S, seed),
        block_tables=_tables(rows, width),
        context_lens=torch.from_numpy(lens.astype(np.int32)),
        prefill_q=_queries(spec, int(cu[-1]), seed, salt=6),
        prefill_cu_q_lens=torch.from_numpy(cu),
        prefill_block_tables=_tables(prow, width),
        prefill_context_lens=torch.from_numpy(plens.astype(np.int32)),
        meta={"pool_need": need, "chunk": chunk, "priors": list(priors)})


def make_batch(name: str, poison: bool = True, seed: Optional[int] = None, **kw) -> Batch:
    """Draw the named workload.  ``poison`` fills every cache row that holds no
    token with NaN so that any over-read shows up as a non-finite output."""
    spec = SPECS[name]
    if "num_seqs" in kw or "ctx" in kw or "heads" in kw:
        from dataclasses import replace
        ctx = kw.pop("ctx", (spec.ctx_lo, spec.ctx_hi))
        hq, hkv = kw.pop("heads", (spec.num_q_heads, spec.num_kv_heads))
        spec = replace(spec, num_seqs=kw.pop("num_seqs", spec.num_seqs),
                       ctx_lo=ctx[0], ctx_hi=ctx[1], num_q_heads=hq, num_kv_heads=hkv)
    seed = SEED_BASE + spec.index if seed is None else seed
    if name == "shared_prefix_cow":
        b = _shared_prefix_batch(spec, seed, poison, **kw)
    elif name == "mixed_step":
        b = _mixed_batch(spec, seed, poison, **kw)
    else:
        b = _decode_batch(spec, seed, poison, **kw)
    if name == "tiny_fp32":
        b.scale = 1.0 / 8.0
    return b


def custom_batch(dtype: str, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, lens, seed: int, poison: bool = True,
                 pool_factor: float = 1.2, outlier_p: float = 0.0,
                 outlier_scale: float = 1.0) -> Batch:
    """A decode batch with explicit context lengths (edge-case tests)."""
    lens = np.asarray(lens, dtype=np.int64)
    spec = Spec("custom", 0, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim,
                int(lens.min(initial=0)), int(max(1, lens.max(initial=1))),
                outlier_p=outlier_p, outlier_scale=outlier_scale)
    return _decode_batch(spec, seed, poison, lens=lens, pool_factor=pool_factor)


def custom_prefill(dtype: str, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   priors, chunks, seed: int, poison: bool = True) -> Batch:
    """Prompt-chunk sequences with explicit prior lengths and chunk sizes and no
    decode sequences (edge-case tests for the prefill path)."""
    spec = Spec("custom_prefill", 0, dtype, 0, num_q_heads, num_kv_heads, head_dim)
    rng = np.random.Generator(np.random.PCG64(seed))
    priors = [int(p) for p in priors]
    chunks = [int(c) for c in chunks]
    plens = np.asarray([p + c for p, c in zip(priors, chunks)], dtype=np.int64)
    pblk = (plens + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = int(pblk.sum())
    NB = max(1, int(math.ceil(1.2 * need)))
    perm = rng.permutation(NB).astype(np.int32)
    off, prow = 0, []
    for i in range(len(priors)):
        prow.append(perm[off: off + pblk[i]])
        off += pblk[i]
    used = [_slots_of(prow[i], 0, priors[i]) for i in range(len(priors))]
    used = np.concatenate(used) if used else np.zeros(0, np.int64)
    k_cache, v_cache = _make_cache(spec, NB, seed, used, poison)
    new_slots = [_slots_of(prow[i], priors[i], chunks[i]) for i in range(len(priors))]
    new_slots = np.concatenate(new_slots) if new_slots else np.zeros(0, np.int64)
    k_new, v_new = _new_tokens(spec, len(new_slots), seed)
    cu = np.zeros(len(priors) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(chunks)
    width = int(max(1, pblk.max(initial=1)))
    dt = _torch_dtype(dtype)
    return Batch(
        spec=spec, dtype=dt, scale=1.0 / math.sqrt(head_dim), num_blocks=NB,
        k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(new_slots),
        q=torch.zeros((0, num_q_heads, head_dim), dtype=dt),
        block_tables=torch.zeros((0, width), dtype=torch.int32),
        context_lens=torch.zeros(0, dtype=torch.int32),
        prefill_q=_queries(spec, int(cu[-1]), seed, salt=6),
        prefill_cu_q_lens=torch.from_numpy(cu),
        prefill_block_tables=_tables(prow, width),
        prefill_context_lens=torch.from_numpy(plens.astype(np.int32)),
        meta={"pool_need": need})


def fp8_batch(base: Batch, seed: int = 97) -> Batch:
    """The same step over fp8 E4M3 caches: random codes in place of the cache
    values (drawn directly as codes: random sign, exponent field uniform in
    [4, 10], mantissa uniform, so magnitudes 2^-3 .. 2^4 before scaling),
    the NaN code (0x7F) in every row the base batch poisons, and per kv head
    scales 2^-4 (1 + g/8) for K and 2^-3 (1 + g/16) for V.  A row that the
    base batch made an outlier (a row whose largest magnitude exceeds 8, which
    an N(0,1) row of the workloads' sizes practically never does) keeps that
    role: its exponent fields are raised by 4, so its values are 16 times
    larger (magnitudes up to 240, still finite codes).  Queries and the new
    tokens stay bf16 (the append quantises them)."""
    g = torch.Generator().manual_seed(seed)
    NB, H, bs, d = base.k_cache.shape

    def codes(src):
        sign = torch.randint(0, 2, src.shape, generator=g, dtype=torch.int32) << 7
        ex = torch.randint(4, 11, src.shape, generator=g, dtype=torch.int32)
        big = torch.empty(src.shape[:-1] + (1,), dtype=torch.bool)
        for a in range(0, src.shape[0], 4096):  # in slices: the long-context caches hold ~1.6 GB each
            big[a:a + 4096] = src[a:a + 4096].float().abs().amax(dim=-1, keepdim=True) > 8.0  # NaN: False
        ex = torch.where(big, ex + 4, ex) << 3
        man = torch.randint(0, 8, src.shape, generator=g, dtype=torch.int32)
        c = (sign | ex | man).to(torch.uint8)
        c[src.isnan()] = 0x7F
        return c

    out = Batch(**{f.name: getattr(base, f.name) for f in base.__dataclass_fields__.values()})
    out.k_cache, out.v_cache = codes(base.k_cache), codes(base.v_cache)
    out.k_scale = 2.0 ** -4 * (1 + torch.arange(H, dtype=torch.float32) / 8)
    out.v_scale = 2.0 ** -3 * (1 + torch.arange(H, dtype=torch.float32) / 16)
    out.meta = dict(base.meta, fp8=True)
    return out
