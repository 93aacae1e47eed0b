"""GB300-native paged KV-cache attention.

Thin ctypes binding over ``libpkv.so`` (the C ABI of ``include/pkv.h``).  The
functions here only check and marshal torch tensors (device memory, the current
stream); every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or no GPU is present the calls
raise.

Calls (names follow the C ABI without the ``pkv_`` prefix):
  kv_append(k, v, slot_mapping, k_cache, v_cache)
  copy_blocks(src_dst_pairs, k_cache, v_cache)
  paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out)
  decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out)
  decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                       prefix_len)
  paged_attention_prefill_chunk(q, cu_q_lens, k_cache, v_cache, block_tables,
                                context_lens, scale, out)
  kv_append_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale)
  paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                             context_lens, scale, out)
  get_status()
  BlockManager(num_blocks, max_blocks_per_seq)   (host block allocator, pkv_bm_*)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "BLOCK_SIZE", "DEFAULT_PARTITION", "PkvError", "load", "library_path", "kv_append",
    "copy_blocks", "decode_workspace_bytes", "decode_partition_size", "paged_attention_decode",
    "decode_step", "decode_shared_prefix_workspace_bytes", "decode_shared_prefix",
    "prefill_workspace_bytes", "paged_attention_prefill_chunk", "get_status", "set_wait_limit_ns", "STATUS_BITS",
    "EXPORTED", "kv_append_fp8", "paged_attention_decode_fp8", "check_copy_pairs", "BlockManager",
    "FP8_E4M3",
]

BLOCK_SIZE = 16
DEFAULT_PARTITION = 512
OK, ERR_INVALID, ERR_CUDA, ERR_OOB = 0, 1, 2, 3
F32, BF16, FP8_E4M3 = 0, 1, 2  # FP8_E4M3: a uint8 tensor of E4M3 codes
STATUS_BITS = {"bad_slot": 1, "bad_block": 2, "bad_length": 4, "bad_qlen": 8, "internal": 16}

# every entry point declared in include/pkv.h
EXPORTED = (
    "pkv_kv_append", "pkv_copy_blocks", "pkv_decode_workspace_bytes", "pkv_decode_partition_size",
    "pkv_paged_attention_decode", "pkv_decode_step", "pkv_paged_attention_decode_no_alloc",
    "pkv_decode_shared_prefix_workspace_bytes", "pkv_paged_attention_decode_shared_prefix",
    "pkv_prefill_workspace_bytes",
    "pkv_paged_attention_prefill_chunk", "pkv_get_status", "pkv_set_wait_limit_ns", "pkv_last_error_string",
    "pkv_version",
    "pkv_kv_append_fp8", "pkv_paged_attention_decode_fp8", "pkv_decode_partition_size_fp8", "pkv_decode_step_fp8",
    "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_num_free_blocks", "pkv_bm_add_sequence", "pkv_bm_fork",
    "pkv_bm_append_tokens", "pkv_bm_slots", "pkv_bm_free_sequence", "pkv_bm_block_tables",
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lib = None


class PkvError(RuntimeError):
    """A call of the C ABI returned an error code."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"pkv error {code}: {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load ``libpkv.so`` (built by ``paged_kv_cache_297_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m paged_kv_cache_297_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pkv_kv_append.argtypes = [P, P, P, I, P, P, I, I, I, I, I, P]
    lib.pkv_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I, P]
    lib.pkv_decode_workspace_bytes.argtypes = [I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.pkv_decode_partition_size.argtypes = [I, I, I, I, ctypes.POINTER(I)]
    lib.pkv_decode_partition_size_fp8.argtypes = [I, I, I, I, I, ctypes.POINTER(I)]
    lib.pkv_paged_attention_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, I, I, F, P, I,
                                               I, P, SZ, P]
    lib.pkv_decode_step.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, F, P, I, I, P, SZ, P]
    lib.pkv_paged_attention_decode_no_alloc.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, I,
                                                        I, F, P, I, I, P]
    lib.pkv_decode_shared_prefix_workspace_bytes.argtypes = [I, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.pkv_paged_attention_decode_shared_prefix.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I,
                                                             I, F, P, I, I, P, SZ, P]
    lib.pkv_prefill_workspace_bytes.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.pkv_paged_attention_prefill_chunk.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, I,
                                                      I, F, P, I, I, P, SZ, P]
    lib.pkv_get_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.pkv_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.pkv_last_error_string.argtypes = []
    lib.pkv_version.argtypes = []
    lib.pkv_kv_append_fp8.argtypes = [P, P, I, P, I, P, P, P, P, I, I, I, I, P]
    lib.pkv_paged_attention_decode_fp8.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, F, P, I, P,
                                                   SZ, P]
    lib.pkv_decode_step_fp8.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, F, P, I, P, SZ, P]
    L = ctypes.c_int64
    lib.pkv_bm_create.argtypes = [I, I, I, ctypes.POINTER(P)]
    lib.pkv_bm_destroy.argtypes = [P]
    lib.pkv_bm_num_free_blocks.argtypes = [P, ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.pkv_bm_add_sequence.argtypes = [P, L, P, I, ctypes.POINTER(I)]
    lib.pkv_bm_fork.argtypes = [P, L, L]
    lib.pkv_bm_append_tokens.argtypes = [P, P, I, P, P, P, ctypes.POINTER(I)]
    lib.pkv_bm_slots.argtypes = [P, L, I, I, P]
    lib.pkv_bm_free_sequence.argtypes = [P, L]
    lib.pkv_bm_block_tables.argtypes = [P, P, I, P, I, P]
    for name in EXPORTED:
        getattr(lib, name).restype = I
    lib.pkv_last_error_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != OK:
        msg = load().pkv_last_error_string()
        raise PkvError(rc, msg.decode() if msg else "")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.uint8:
        return FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


# the current stream's handle without building a Stream object (a few
# microseconds less host time per call)
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _RAW_STREAM is not None:
            return _RAW_STREAM(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(need: int, device, stream) -> Optional[torch.Tensor]:
    """A scratch buffer of `need` bytes for one call enqueued on `stream`.

    torch's caching allocator ties a block to the stream current at
    allocation; when the call runs on another stream the block is also
    recorded on that stream, so it is not handed out again (to work on the
    current stream) before the call's kernels are done with it."""
    if need <= 0:
        return None
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    if stream is not None:
        s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(
            stream.cuda_stream if hasattr(stream, "cuda_stream") else stream), device=device)
        if s.cuda_stream != torch.cuda.current_stream(device).cuda_stream:
            ws.record_stream(s)
    return ws


def _cache_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must both be [num_blocks, num_kv_heads, 16, head_dim]")
    NB, H, bs, d = k_cache.shape
    return int(NB), int(H), int(bs), int(d)


def kv_append(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Write token i's K/V rows (``k``/``v`` ``[T, Hkv, d]``) at slot ``slot_mapping[i]``."""
    NB, H, bs, d = _cache_dims(k_cache, v_cache)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (H, d) or k.dtype != k_cache.dtype:
        raise ValueError("k/v must be [T, num_kv_heads, head_dim] in the cache dtype")
    if slot_mapping.shape != (k.shape[0],):
        raise ValueError("slot_mapping must be [T]")
    _check(load().pkv_kv_append(
        _dev(k, "k"), _dev(v, "v"), _dev(slot_mapping, "slot_mapping", torch.int64),
        int(k.shape[0]), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), NB, H, d, bs,
        _dt(k_cache), _stream(stream)))


def check_copy_pairs(src_dst_pairs) -> None:
    """The copy_blocks caller contract, checked on a host copy: destinations
    distinct and none of them a source of the same call (the blocks of one
    call are copied concurrently)."""
    p = src_dst_pairs.detach().to("cpu", torch.int64).view(-1, 2)
    dst = p[:, 1].tolist()
    if len(set(dst)) != len(dst):
        raise ValueError("copy_blocks: a destination block appears twice")
    if set(dst) & set(p[:, 0].tolist()):
        raise ValueError("copy_blocks: a destination block is also a source")


def copy_blocks(src_dst_pairs, k_cache, v_cache, stream=None, check: Optional[bool] = None) -> None:
    """Copy-on-write: block dst of both caches becomes a copy of block src.
    ``check`` (default: the PKV_CHECK_PAIRS environment variable) validates
    the caller contract on a host copy first (a device-to-host copy)."""
    NB, H, bs, d = _cache_dims(k_cache, v_cache)
    if src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")
    if check if check is not None else os.environ.get("PKV_CHECK_PAIRS", "") not in ("", "0"):
        check_copy_pairs(src_dst_pairs)
    _check(load().pkv_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(src_dst_pairs, "src_dst_pairs", torch.int64), int(src_dst_pairs.shape[0]), NB, H, d,
        bs, _dt(k_cache), _stream(stream)))


def decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                           partition_size: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pkv_decode_workspace_bytes(int(num_seqs), int(num_q_heads), int(head_dim),
                                             int(max_context_len), int(partition_size),
                                             ctypes.byref(out)))
    return int(out.value)


def decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size: int = 0) -> int:
    """Split-K partition (tokens) a decode call with these sizes uses on the
    current device; partition_size 0 asks for the adaptive choice."""
    out = ctypes.c_int(0)
    _check(load().pkv_decode_partition_size(int(num_seqs), int(num_kv_heads), int(max_context_len),
                                            int(partition_size), ctypes.byref(out)))
    return int(out.value)


def decode_partition_size_fp8(num_seqs, num_q_heads, num_kv_heads, max_context_len,
                              partition_size: int = 0) -> int:
    """As :func:`decode_partition_size` for :func:`paged_attention_decode_fp8`."""
    out = ctypes.c_int(0)
    _check(load().pkv_decode_partition_size_fp8(int(num_seqs), int(num_q_heads), int(num_kv_heads),
                                                int(max_context_len), int(partition_size), ctypes.byref(out)))
    return int(out.value)


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                           max_context_len: Optional[int] = None, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[s, h] = softmax(scale * q[s, h] . K^T) V over sequence s's cached tokens."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    S, Hq, dq = q.shape
    if dq != d or q.dtype != k_cache.dtype:
        raise ValueError("q must be [S, Hq, head_dim] in the cache dtype")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    mb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_workspace_bytes(S, Hq, d, max_context_len, partition_size)
        workspace = _workspace(need, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_paged_attention_decode(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), mb,
        _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, d, bs, NB,
        int(max_context_len), int(partition_size), float(scale), _dev(out, "out"), _dt(q),
        _dt(out), ws_ptr, ws_bytes, _stream(stream)))
    return out


def kv_append_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None) -> None:
    """Append into fp8 E4M3 caches (uint8 tensors): element x of kv head g is
    stored as the code of x / scale[g] (nearest even, saturated at 448)."""
    NB, H, bs, d = _cache_dims(k_cache, v_cache)
    if k_cache.dtype != torch.uint8:
        raise TypeError("fp8 caches are uint8 tensors of E4M3 codes")
    if k.dim() != 3 or k.shape[1:] != (H, d) or v.shape != k.shape or k.dtype != v.dtype:
        raise ValueError("k/v must be [num_tokens, num_kv_heads, head_dim]")
    for sc, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if sc.shape != (H,):
            raise ValueError(f"{name} must be [num_kv_heads]")
    _check(load().pkv_kv_append_fp8(
        _dev(k, "k"), _dev(v, "v"), _dt(k), _dev(slot_mapping, "slot_mapping", torch.int64), int(k.shape[0]),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(k_scale, "k_scale", torch.float32),
        _dev(v_scale, "v_scale", torch.float32), NB, H, d, bs, _stream(stream)))


def paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                               max_context_len: Optional[int] = None, partition_size: int = 0,
                               workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode with bf16 queries over fp8 E4M3 caches (uint8), cached element x
    of kv head g standing for x * scale[g]."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    S, Hq, dq = q.shape
    if k_cache.dtype != torch.uint8 or q.dtype != torch.bfloat16 or dq != d:
        raise ValueError("q must be bf16 [S, Hq, head_dim] over uint8 (E4M3) caches")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    mb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_workspace_bytes(S, Hq, d, max_context_len, partition_size)
        workspace = _workspace(need, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_paged_attention_decode_fp8(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(block_tables, "block_tables", torch.int32), mb,
        _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, d, bs, NB,
        int(max_context_len), int(partition_size), float(scale), _dev(out, "out"),
        _dt(out), ws_ptr, ws_bytes, _stream(stream)))
    return out


def decode_step_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                    out, max_context_len: Optional[int] = None, partition_size: int = 0,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """:func:`kv_append_fp8` of each sequence's new K/V row (``k_new``/``v_new``
    ``[S, Hkv, 128]`` bf16, at position L-1) fused into
    :func:`paged_attention_decode_fp8`: one launch."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    S, Hq, dq = q.shape
    if k_cache.dtype != torch.uint8 or q.dtype != torch.bfloat16 or dq != d:
        raise ValueError("q must be bf16 [S, Hq, head_dim] over uint8 (E4M3) caches")
    if k_new.shape != (S, Hkv, d) or v_new.shape != k_new.shape or k_new.dtype != torch.bfloat16 \
            or v_new.dtype != torch.bfloat16:
        raise ValueError("k_new/v_new must be bf16 [S, num_kv_heads, head_dim]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    mb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_workspace_bytes(S, Hq, d, max_context_len, partition_size)
        workspace = _workspace(need, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_decode_step_fp8(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(block_tables, "block_tables", torch.int32), mb, _dev(context_lens, "context_lens", torch.int32),
        S, Hq, Hkv, d, bs, NB, int(max_context_len), int(partition_size), float(scale), _dev(out, "out"),
        _dt(out), ws_ptr, ws_bytes, _stream(stream)))
    return out


def decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out,
                max_context_len: Optional[int] = None, partition_size: int = 0,
                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Append each sequence's new K/V (``[S, Hkv, d]``) at position L-1, then
    decode, in one launch; same result as kv_append + paged_attention_decode."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    S, Hq, dq = q.shape
    if dq != d or q.dtype != k_cache.dtype or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, head_dim] in the cache dtype")
    if k_new.shape != (S, Hkv, d) or v_new.shape != k_new.shape or k_new.dtype != k_cache.dtype:
        raise ValueError("k_new/v_new must be [S, num_kv_heads, head_dim] in the cache dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    mb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_workspace_bytes(S, Hq, d, max_context_len, partition_size)
        workspace = _workspace(need, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_decode_step(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables", torch.int32), mb,
        _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, d, bs, NB,
        int(max_context_len), int(partition_size), float(scale), _dev(out, "out"), _dt(q), _dt(out),
        ws_ptr, ws_bytes, _stream(stream)))
    return out


def decode_shared_prefix_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                         prefix_len, partition_size: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pkv_decode_shared_prefix_workspace_bytes(
        int(num_seqs), int(num_q_heads), int(head_dim), int(max_context_len), int(prefix_len),
        int(partition_size), ctypes.byref(out)))
    return int(out.value)


def decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, scale, out, prefix_len: int,
                         k_new=None, v_new=None, max_context_len: Optional[int] = None,
                         partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Decode of a batch whose sequences share their first ``prefix_len``
    tokens (same physical blocks): the prefix once for all queries on the
    tensor cores, each sequence's own tokens by the partitioned kernel, then a
    log-sum-exp merge.  With ``k_new``/``v_new`` (``[S, Hkv, d]``) the new
    tokens are appended at position L-1 first, as in :func:`decode_step`."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    S, Hq, dq = q.shape
    if dq != d or q.dtype != k_cache.dtype or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, head_dim] in the cache dtype")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None and (k_new.shape != (S, Hkv, d) or v_new.shape != k_new.shape
                              or k_new.dtype != k_cache.dtype):
        raise ValueError("k_new/v_new must be [S, num_kv_heads, head_dim] in the cache dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks] and context_lens [S]")
    mb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_shared_prefix_workspace_bytes(S, Hq, d, max_context_len, prefix_len, partition_size)
        workspace = _workspace(need, q.device, stream)
    _check(load().pkv_paged_attention_decode_shared_prefix(
        _dev(q, "q"), None if k_new is None else _dev(k_new, "k_new"),
        None if v_new is None else _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables", torch.int32), mb,
        _dev(context_lens, "context_lens", torch.int32), S, Hq, Hkv, d, bs, NB,
        int(max_context_len), int(prefix_len), int(partition_size), float(scale), _dev(out, "out"),
        _dt(q), _dt(out), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def prefill_workspace_bytes(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_q_len,
                            max_context_len) -> int:
    out = ctypes.c_size_t(0)
    _check(load().pkv_prefill_workspace_bytes(int(num_seqs), int(total_q), int(num_q_heads),
                                              int(num_kv_heads), int(head_dim), int(max_q_len),
                                              int(max_context_len), ctypes.byref(out)))
    return int(out.value)


def paged_attention_prefill_chunk(q, cu_q_lens, k_cache, v_cache, block_tables, context_lens,
                                  scale, out, max_q_len: Optional[int] = None,
                                  max_context_len: Optional[int] = None,
                                  workspace: Optional[torch.Tensor] = None,
                                  stream=None) -> torch.Tensor:
    """Causal attention of each sequence's prompt chunk over its whole cache."""
    NB, Hkv, bs, d = _cache_dims(k_cache, v_cache)
    total_q, Hq, dq = q.shape
    S = int(context_lens.shape[0])
    if dq != d or q.dtype != k_cache.dtype or out.shape != q.shape:
        raise ValueError("q/out must be [total_q, Hq, head_dim] in the cache dtype")
    if cu_q_lens.shape != (S + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("cu_q_lens must be [S+1] and block_tables [S, max_blocks]")
    mb = int(block_tables.shape[1])
    if max_q_len is None:
        max_q_len = total_q
    if max_context_len is None:
        max_context_len = mb * bs
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = prefill_workspace_bytes(S, total_q, Hq, Hkv, d, max_q_len, max_context_len)
        workspace = _workspace(need, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_paged_attention_prefill_chunk(
        _dev(q, "q"), _dev(cu_q_lens, "cu_q_lens", torch.int32), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables", torch.int32), mb,
        _dev(context_lens, "context_lens", torch.int32), S, int(total_q), int(max_q_len),
        int(max_context_len), Hq, Hkv, d, bs, NB, float(scale), _dev(out, "out"), _dt(q),
        _dt(out), ws_ptr, ws_bytes, _stream(stream)))
    return out


def set_wait_limit_ns(ns: int = 0) -> None:
    """Bound on each wait inside the tensor-core kernels, in nanoseconds (0:
    the default, 200 ms); a launch whose wait runs out records the
    ``internal`` status bit and returns with undefined outputs."""
    _check(load().pkv_set_wait_limit_ns(int(ns)))


def get_status(stream=None) -> int:
    """Synchronise the stream, read and clear this device's status word."""
    flags = ctypes.c_uint(0)
    rc = load().pkv_get_status(_stream(stream), ctypes.byref(flags))
    if rc == ERR_CUDA:
        _check(rc)
    return int(flags.value)


class BlockManager:
    """Host block manager (``pkv_bm_*``): physical block allocation with
    reference counts, copy-on-write and a prefix index over full blocks.
    Produces the block tables, context lengths, slot mappings and copy pairs
    that the kernels take.  Host memory only; returns CPU tensors."""

    def __init__(self, num_blocks: int, max_blocks_per_seq: int, prefix_cache: bool = True):
        h = ctypes.c_void_p()
        _check(load().pkv_bm_create(int(num_blocks), int(max_blocks_per_seq), int(bool(prefix_cache)),
                                    ctypes.byref(h)))
        self._h = h
        self.max_blocks_per_seq = int(max_blocks_per_seq)

    def close(self) -> None:
        if self._h:
            _check(load().pkv_bm_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free_blocks(self):
        """(blocks a new allocation could take, of which cached)"""
        f, c = ctypes.c_int(0), ctypes.c_int(0)
        _check(load().pkv_bm_num_free_blocks(self._h, ctypes.byref(f), ctypes.byref(c)))
        return f.value, c.value

    def add_sequence(self, seq_id: int, tokens) -> int:
        """New sequence with prompt ``tokens``; returns how many leading
        tokens were found in the prefix index."""
        t = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
        n = ctypes.c_int(0)
        _check(load().pkv_bm_add_sequence(self._h, int(seq_id), t.data_ptr() if t.numel() else None,
                                          t.numel(), ctypes.byref(n)))
        return n.value

    def fork(self, parent: int, child: int) -> None:
        _check(load().pkv_bm_fork(self._h, int(parent), int(child)))

    def append_tokens(self, seq_ids, tokens):
        """One new token per sequence: returns (slot_mapping int64 [n],
        copy pairs int64 [p, 2]) for copy_blocks then kv_append."""
        ids = torch.as_tensor(seq_ids, dtype=torch.int64).contiguous()
        tok = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
        if ids.shape != tok.shape or ids.dim() != 1:
            raise ValueError("seq_ids and tokens must be 1-D of the same length")
        n = ids.numel()
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty(max(1, 2 * n), dtype=torch.int64)
        np_ = ctypes.c_int(0)
        _check(load().pkv_bm_append_tokens(self._h, ids.data_ptr() if n else None, n,
                                           tok.data_ptr() if n else None, slots.data_ptr(),
                                           pairs.data_ptr(), ctypes.byref(np_)))
        return slots, pairs[: 2 * np_.value].view(-1, 2).clone()

    def slots(self, seq_id: int, first: int, n: int) -> torch.Tensor:
        out = torch.empty(max(1, n), dtype=torch.int64)
        _check(load().pkv_bm_slots(self._h, int(seq_id), int(first), int(n), out.data_ptr()))
        return out[:n]

    def free_sequence(self, seq_id: int) -> None:
        _check(load().pkv_bm_free_sequence(self._h, int(seq_id)))

    def block_tables(self, seq_ids, max_blocks: Optional[int] = None):
        """(block tables int32 [n, max_blocks], context lengths int32 [n])"""
        ids = torch.as_tensor(seq_ids, dtype=torch.int64).contiguous()
        w = int(max_blocks or self.max_blocks_per_seq)
        n = ids.numel()
        tables = torch.empty((max(1, n), w), dtype=torch.int32)
        lens = torch.empty(max(1, n), dtype=torch.int32)
        _check(load().pkv_bm_block_tables(self._h, ids.data_ptr() if n else None, n, tables.data_ptr(), w,
                                          lens.data_ptr()))
        return tables[:n], lens[:n]
