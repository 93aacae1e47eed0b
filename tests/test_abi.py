"""The C ABI without a GPU: the library builds, loads, exports every entry
point that include/pkv.h declares, and rejects bad arguments on the host
before any CUDA call."""

import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_297_gb300 as pkv
from paged_kv_cache_297_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"^(?:int|const char \*)\s*(pkv_\w+)\(", text, re.M)))


def test_header_and_binding_agree():
    assert _declared() == sorted(pkv.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.pkv_version() >= 100


def test_decode_workspace_sizes(lib):
    n = ctypes.c_size_t(0)
    # one partition: no workspace
    assert lib.pkv_decode_workspace_bytes(64, 32, 128, 512, 0, ctypes.byref(n)) == 0
    assert n.value == 0
    # 8 partitions of 512 for 4096 tokens: partial O (d floats) and (m, l) per
    # (seq, q head, partition), each region rounded up to 256 bytes
    assert lib.pkv_decode_workspace_bytes(64, 32, 128, 4096, 0, ctypes.byref(n)) == 0
    rows = 64 * 32 * 8
    r256 = lambda x: (x + 255) // 256 * 256
    assert n.value == r256(rows * 128 * 4) + r256(rows * 2 * 4)
    assert lib.pkv_decode_workspace_bytes(64, 32, 128, 4096, 100, ctypes.byref(n)) == pkv.ERR_INVALID
    assert b"multiple of 16" in lib.pkv_last_error_string()


def test_shared_prefix_workspace_sizes(lib):
    # slot 0 for the shared prefix plus the suffix's 512-token partitions
    # (the most slots any adaptive choice needs), then a 256-byte counter
    r256 = lambda x: (x + 255) // 256 * 256
    for S, Hq, L, P in ((256, 32, 2560, 2048), (8, 64, 100000, 512), (3, 8, 48, 32)):
        parts = 1 + -(-(L - P) // 512)
        rows = S * Hq * parts
        want = (r256(rows * 128 * 4) + r256(rows * 2 * 4) if parts > 1 else 0) + 256
        assert pkv.decode_shared_prefix_workspace_bytes(S, Hq, 128, L, P) == want
    # head_dim 64, no prefix, a prefix not in whole blocks, a prefix past the context
    for bad in ((4, 32, 64, 1000, 48), (4, 32, 128, 1000, 0), (4, 32, 128, 1000, 40), (4, 32, 128, 100, 112)):
        with pytest.raises(pkv.PkvError):
            pkv.decode_shared_prefix_workspace_bytes(*bad)


def test_prefill_workspace_sizes(lib):
    # head_dim 128 (the tcgen05 kernel): one 8-byte work-item counter,
    # rounded to 256 bytes; head_dim 64 needs none
    assert pkv.prefill_workspace_bytes(2, 1024, 32, 8, 128, 512, 3584) == 256
    assert pkv.prefill_workspace_bytes(2, 1024, 8, 8, 64, 512, 3584) == 0
    with pytest.raises(pkv.PkvError):
        pkv.prefill_workspace_bytes(2, 1024, 32, 8, 96, 512, 3584)


def test_decode_partition_choice(lib):
    assert pkv.decode_partition_size(64, 8, 4096, 256) == 256
    # adaptive: the largest partition that still leaves ~4 blocks per SM, for
    # any device of 129..256 SMs (without a device the library assumes 148)
    assert pkv.decode_partition_size(64, 8, 4096) == 1536   # 64x8x2 units
    assert pkv.decode_partition_size(8, 8, 131072) == 3072  # 8x8x22 units
    assert pkv.decode_partition_size(256, 8, 2560) == 3072
    assert pkv.decode_partition_size(4, 4, 64) == pkv.DEFAULT_PARTITION
    assert pkv.decode_partition_size(0, 8, 0) == pkv.DEFAULT_PARTITION
    # the workspace asked for with partition 0 covers whatever is chosen
    for S, hkv, L in [(64, 8, 4096), (8, 8, 131072), (4, 4, 64), (1, 1, 70000)]:
        part = pkv.decode_partition_size(S, hkv, L)
        assert pkv.decode_workspace_bytes(S, 4 * hkv, 128, L, 0) >= \
            pkv.decode_workspace_bytes(S, 4 * hkv, 128, L, part)
    with pytest.raises(pkv.PkvError):
        pkv.decode_partition_size(1, 8, 100, 24)


def test_decode_partition_choice_fp8(lib):
    # the fp8 kernel (four blocks of 4 warps per SM) leaves a batch unsplit
    # when its (sequence, unit) pairs fill 2..4 blocks per SM; with 148 SMs
    # (no device) that is 296..592 units
    assert pkv.decode_partition_size_fp8(64, 32, 8, 4096) == 4096       # 512 units
    assert pkv.decode_partition_size_fp8(64, 32, 8, 4090) == 4096       # rounded up to 16
    assert pkv.decode_partition_size_fp8(8, 64, 8, 131072) == 3072      # 64 units: split
    assert pkv.decode_partition_size_fp8(256, 32, 8, 2560) == 3072      # 2048 units: split
    assert pkv.decode_partition_size_fp8(32, 128, 8, 4096) == 4096      # group 16: 2 units per kv head
    assert pkv.decode_partition_size_fp8(64, 32, 8, 8192) == 8192       # the longest context left unsplit
    assert pkv.decode_partition_size_fp8(64, 32, 8, 8193) == 3072       # longer: split (64x8x2 units)
    assert pkv.decode_partition_size_fp8(64, 32, 8, 4096, 256) == 256   # explicit
    # unsplit needs no workspace; the partition-0 workspace still covers it
    assert pkv.decode_workspace_bytes(64, 32, 128, 4096, 4096) == 0
    with pytest.raises(pkv.PkvError):
        pkv.decode_partition_size_fp8(1, 12, 8, 100)


@pytest.mark.parametrize("bad", ["block_size", "head_dim", "dtype", "heads"])
def test_host_rejects_bad_arguments(lib, bad):
    P = ctypes.c_void_p
    dummy = P(256)  # never dereferenced: rejected before any launch
    args = dict(block_size=16, head_dim=128, dtype=pkv.BF16, hq=32, hkv=8)
    if bad == "block_size":
        args["block_size"] = 32
    elif bad == "head_dim":
        args["head_dim"] = 96
    elif bad == "dtype":
        args["dtype"] = 7
    else:
        args["hq"] = 30
    rc = lib.pkv_paged_attention_decode(
        dummy, dummy, dummy, dummy, 4, dummy, 2, args["hq"], args["hkv"], args["head_dim"],
        args["block_size"], 8, 64, 0, ctypes.c_float(0.1), dummy, args["dtype"], pkv.F32, None,
        0, None)
    assert rc == pkv.ERR_INVALID
    assert lib.pkv_last_error_string()
    if bad in ("block_size", "head_dim", "dtype"):
        # (with valid sizes the append would launch on the dummy pointers)
        rc = lib.pkv_kv_append(dummy, dummy, dummy, 1, dummy, dummy, 8, args["hkv"],
                               args["head_dim"], args["block_size"], args["dtype"], None)
        assert rc == pkv.ERR_INVALID


def test_decode_rejects_small_workspace_and_misalignment(lib):
    P = ctypes.c_void_p
    a = P(4096)
    rc = lib.pkv_paged_attention_decode(a, a, a, a, 256, a, 2, 32, 8, 128, 16, 64, 4096, 0,
                                        ctypes.c_float(0.1), a, pkv.BF16, pkv.F32, a, 16, None)
    assert rc == pkv.ERR_INVALID and b"workspace" in lib.pkv_last_error_string()
    rc = lib.pkv_paged_attention_decode(P(4098), a, a, a, 4, a, 2, 32, 8, 128, 16, 64, 64, 0,
                                        ctypes.c_float(0.1), a, pkv.BF16, pkv.F32, None, 0, None)
    assert rc == pkv.ERR_INVALID and b"aligned" in lib.pkv_last_error_string()


def test_prefill_rejects_wide_groups(lib):
    P = ctypes.c_void_p
    a = P(4096)
    rc = lib.pkv_paged_attention_prefill_chunk(a, a, a, a, a, 4, a, 1, 8, 8, 64, 128, 1, 128, 16,
                                               8, ctypes.c_float(0.1), a, pkv.BF16, pkv.F32, None,
                                               0, None)
    assert rc == pkv.ERR_INVALID


def test_zero_sized_calls_launch_nothing(lib):
    # num_tokens / num_pairs / num_seqs of 0 return OK before any CUDA call
    assert lib.pkv_kv_append(None, None, None, 0, None, None, 0, 8, 128, 16, pkv.BF16, None) == 0
    assert lib.pkv_copy_blocks(None, None, None, 0, 0, 8, 128, 16, pkv.BF16, None) == 0
    assert lib.pkv_paged_attention_decode(None, None, None, None, 0, None, 0, 32, 8, 128, 16, 0, 0,
                                          0, ctypes.c_float(1.0), None, pkv.BF16, pkv.F32, None, 0,
                                          None) == 0


def test_copy_pair_contract_check_on_the_host():
    pkv.check_copy_pairs(torch.tensor([[1, 5], [2, 6], [1, 7]]))
    with pytest.raises(ValueError):
        pkv.check_copy_pairs(torch.tensor([[1, 5], [2, 5]]))   # duplicate destination
    with pytest.raises(ValueError):
        pkv.check_copy_pairs(torch.tensor([[1, 5], [5, 6]]))   # destination also a source
