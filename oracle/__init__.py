"""fp64 host oracle for the paged KV-cache paths.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may import this package; the library never calls
it and has no fallback onto it.  The arithmetic lives in ``oracle.c``; this
file only marshals torch CPU tensors into it.

Every function takes host tensors in the library's layouts:
``k_cache``/``v_cache`` ``[num_blocks, num_kv_heads, block_size, head_dim]``,
``block_tables`` ``[S, max_blocks]`` int32, ``context_lens`` ``[S]`` int32
(including the token appended this step), ``q`` ``[rows, num_q_heads, head_dim]``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
# A test may point the wrapper at another build of oracle.c (the mutation test
# compiles deliberately broken copies to show that the pins catch them).
_OVERRIDE = os.environ.get("PKV_ORACLE_LIB")
_SRC = os.path.join(_HERE, "oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP, -O2, no architecture flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        if _OVERRIDE:
            lib = ctypes.CDLL(_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_SO)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.oracle_kv_append.argtypes = [P, P, P, I, P, P, I, I, I, I, I]
        lib.oracle_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I]
        lib.oracle_paged_attention.argtypes = [P, I, P, P, I, P, I, P, P, I, I, I, I, I, I,
                                               ctypes.c_double, P, P, P]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_kv_append_fp8.argtypes = [P, P, I, P, I, P, P, I, I, I, I, P, P]
        lib.oracle_threads.restype = I
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_set_threads.restype = None
        _lib = lib
    return _lib


_DT = {torch.float32: 0, torch.bfloat16: 1, torch.uint8: 2}  # uint8: fp8 E4M3 codes


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return t.data_ptr()


def threads() -> int:
    return _load().oracle_threads()


def set_threads(n: int) -> None:
    """Threads for later calls (OpenMP)."""
    _load().oracle_set_threads(int(n))


def kv_append(k, v, slot_mapping, k_cache, v_cache) -> None:
    """In place on the host caches; bit copy of each new token's rows."""
    NB, H, bs, d = k_cache.shape
    rc = _load().oracle_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping.to(torch.int64)),
                                  int(k.shape[0]), _ptr(k_cache), _ptr(v_cache), NB, H, bs, d,
                                  _DT[k_cache.dtype])
    if rc != 0:
        raise IndexError(f"oracle kv_append: slot out of range (rc={rc})")


def copy_blocks(k_cache, v_cache, pairs) -> None:
    NB, H, bs, d = k_cache.shape
    pairs = pairs.to(torch.int64).contiguous()
    rc = _load().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), int(pairs.shape[0]),
                                    NB, H, bs, d, _DT[k_cache.dtype])
    if rc != 0:
        raise IndexError(f"oracle copy_blocks: block id out of range (rc={rc})")


def e4m3_encode(x: torch.Tensor) -> torch.Tensor:
    """E4M3 codes (uint8) of binary32 values: nearest, ties to even, saturating at 448."""
    lib = _load()
    flat = x.to(torch.float32).reshape(-1).tolist()
    return torch.tensor([lib.oracle_e4m3_encode(f) for f in flat], dtype=torch.uint8).reshape(x.shape)


def e4m3_decode(codes: torch.Tensor) -> torch.Tensor:
    """Values (float64) of E4M3 codes, widened exactly."""
    lib = _load()
    table = torch.tensor([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=torch.float64)
    return table[codes.to(torch.uint8).long()]


def kv_append_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> None:
    """In place on uint8 (E4M3) host caches: code of x / scale per kv head."""
    NB, H, bs, d = k_cache.shape
    assert k_cache.dtype == torch.uint8 and v_cache.dtype == torch.uint8
    ks = k_scale.to(torch.float32).contiguous()
    vs = v_scale.to(torch.float32).contiguous()
    k, v = k.contiguous(), v.contiguous()
    rc = _load().oracle_kv_append_fp8(_ptr(k), _ptr(v), _DT[k.dtype],
                                      _ptr(slot_mapping.to(torch.int64)), int(k.shape[0]), _ptr(k_cache),
                                      _ptr(v_cache), NB, H, bs, d, _ptr(ks), _ptr(vs))
    if rc != 0:
        raise IndexError(f"oracle kv_append_fp8: slot out of range (rc={rc})")


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                    cu_q_lens=None, k_scale=None, v_scale=None) -> torch.Tensor:
    """fp64 output ``[rows, Hq, d]``; decode when ``cu_q_lens`` is None.
    ``k_scale``/``v_scale`` (per kv head) multiply the cache values (fp8)."""
    NB, Hkv, bs, d = k_cache.shape
    rows, Hq, dq = q.shape
    assert dq == d
    S = int(context_lens.shape[0])
    out = torch.empty((rows, Hq, d), dtype=torch.float64)
    bt = block_tables.to(torch.int32).contiguous()
    cl = context_lens.to(torch.int32).contiguous()
    cu = None if cu_q_lens is None else cu_q_lens.to(torch.int32).contiguous()
    q = q.contiguous()
    ks = None if k_scale is None else k_scale.to(torch.float32).contiguous()
    vs = None if v_scale is None else v_scale.to(torch.float32).contiguous()
    rc = _load().oracle_paged_attention(
        _ptr(q), _DT[q.dtype], _ptr(k_cache), _ptr(v_cache), _DT[k_cache.dtype],
        _ptr(bt), int(bt.shape[1]), _ptr(cl), _ptr(cu), S, Hq, Hkv, d, bs, NB, float(scale),
        _ptr(ks), _ptr(vs), _ptr(out))
    if rc == -1:
        raise ValueError("oracle paged_attention: bad argument")
    if rc == -2:
        raise IndexError("oracle paged_attention: block id out of range")
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=None, v_scale=None) -> torch.Tensor:
    return paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale, None, k_scale, v_scale)


def prefill_chunk(q, cu_q_lens, k_cache, v_cache, block_tables, context_lens, scale):
    return paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale, cu_q_lens)
