"""The decode entry point that allocates nothing.

Callers that cannot allocate device memory where they run decode (inside an
allocator or memory-pool hook, or with a device-memory budget fixed up front)
use pkv_paged_attention_decode_no_alloc, whose split-K scratch is a fixed
array inside the library.  These tests call it through the C ABI and check
that it returns what the ordinary entry point (with a caller workspace)
returns, on two calls in a row with different batches, and that sizes beyond
the array are refused.  The file is named to be collected last.
"""

import ctypes

import pytest
import torch

import paged_kv_cache_297_gb300 as pkv
from paged_kv_cache_297_gb300 import workloads as W
from tests._steps import TOL, err_stats, to_dev

pytestmark = pytest.mark.gpu


def _no_alloc(t, b, out, max_ctx):
    lib = pkv.load()
    S, Hq, d = b.q.shape
    NB, Hkv, bs, _ = b.k_cache.shape
    return lib.pkv_paged_attention_decode_no_alloc(
        t["q"].data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(),
        t["block_tables"].data_ptr(), int(b.block_tables.shape[1]), t["context_lens"].data_ptr(),
        S, Hq, Hkv, d, bs, NB, max_ctx, 0, ctypes.c_float(b.scale), out.data_ptr(),
        pkv.BF16 if b.dtype == torch.bfloat16 else pkv.F32, pkv.F32,
        torch.cuda.current_stream().cuda_stream)


def _prepare(b):
    t = to_dev(b)
    pkv.kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    return t


def test_no_alloc_matches_workspace_entry_on_two_calls():
    batches = [W.make_batch("llama3_8b_decode", poison=True),
               W.custom_batch("bf16", 9, 64, 8, 128, [1, 17, 511, 513, 1200, 3000, 4097, 64, 900],
                              seed=77)]
    for b in batches:
        t = _prepare(b)
        max_ctx = b.max_context_len
        ref = torch.empty(b.q.shape, dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                   t["context_lens"], b.scale, ref, max_context_len=max_ctx)
        got = torch.full(b.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        rc = _no_alloc(t, b, got, max_ctx)
        assert rc == pkv.OK, pkv.load().pkv_last_error_string()
        torch.cuda.synchronize()
        assert pkv.get_status() == 0
        mx, mean = err_stats(got, ref.double().cpu())
        tmax, tmean = TOL[b.dtype]
        assert mx <= tmax and mean <= tmean, (mx, mean)


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    lib = pkv.load()
    need = ctypes.c_size_t(0)
    # 8 long sequences x 64 q heads x 256 partitions need far more than 16 MiB
    assert lib.pkv_decode_workspace_bytes(8, 64, 128, 131072, 0, ctypes.byref(need)) == 0
    assert need.value > (16 << 20)
    dummy = ctypes.c_void_p(4096)
    # explicit 512-token partitions: 8 x 64 x 256 partials of 130 floats
    # (68 MB) whatever the device, so the call is refused before any launch
    rc = lib.pkv_paged_attention_decode_no_alloc(dummy, dummy, dummy, dummy, 8192, dummy, 8, 64, 8,
                                                 128, 16, 1, 131072, 512, ctypes.c_float(0.1), dummy,
                                                 pkv.BF16, pkv.F32, None)
    assert rc == pkv.ERR_INVALID
    assert b"static scratch" in lib.pkv_last_error_string()
