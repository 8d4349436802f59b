"""Failure handling, tested without faulting a GPU.

Host side (no GPU): KVS_FAULT_INJECT makes a named entry point return a
chosen error code before it validates or enqueues anything, so a caller's
error paths can be exercised.  Device side (GPU): a test hook withholds one
mbarrier arrive in the pass-1 kernel; its reducers' bounded wait runs out
after a shortened limit, the kernel records KVS_ERR_TIMEOUT and returns, the
merge kernels leave the outputs untouched, and the next normal call on the
same context succeeds.
"""
import os
import subprocess
import sys
import time

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PROBE = r"""
import ctypes, sys
sys.path.insert(0, {root!r})
from kv_cache_compression_flash_b300 import _lib as L
lib = L.lib()
p = ctypes.c_void_p(1 << 20)
s = L.StreamSetC()
print(lib.kvs_allocate_bits(p, p, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None))                 # injected
print(lib.kvs_quantize_pack(p, 8, 64, 128, 0, p, None, ctypes.byref(s), p, 1 << 20, None))   # injected
print(lib.kvs_unit_rms(p, 8, 64, 128, 3, None, p, p, 1 << 20, None))                         # not injected: bad axis
print(lib.kvs_allocate_bits_pools(p, p, -1, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None))       # not injected
print(lib.kvs_gram(p, 8, 100, 64, None, 0, p, p, 1 << 30, None))                              # code 9 ignored
"""


def _probe(spec):
    env = dict(os.environ)
    env["KVS_FAULT_INJECT"] = spec
    out = subprocess.run([sys.executable, "-c", _PROBE.format(root=ROOT)], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    return [int(x) for x in out.stdout.split()]


def test_fault_inject_returns_the_code_before_validation():
    got = _probe("kvs_allocate_bits:5,kvs_quantize_pack:3,not_a_call:4,kvs_gram:9,malformed")
    assert got == [5, 3, 1, 1, 2]


def test_fault_inject_unset_changes_nothing():
    got = _probe("")
    # kvs_allocate_bits with a valid budget goes on to the device (no device here: KVS_ERR_CUDA, or KVS_OK);
    # the others give their own argument errors
    assert got[0] in (0, 4) and got[1:] == [1, 1, 1, 2]


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_survives():
    import oracle as O
    from kv_cache_compression_flash_b300 import _lib as L
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(77)
    Hq, Hkv, W, N, d = 8, 2, 130, 700, 128
    Q = torch.randn(Hq, W, d, generator=g).bfloat16()
    K = torch.randn(Hkv, N, d, generator=g).bfloat16()
    Qd, Kd = Q.to(dev), K.to(dev)
    assert L.device_error() == 0
    out = {"lse": torch.full((Hq, W), float("nan"), device=dev), "w_t": torch.full((Hkv, N), float("nan"), device=dev)}
    L.debug_inject(L.DEBUG_WITHHOLD_LSE_ARRIVE, 20_000_000)          # 20 ms
    try:
        t0 = time.perf_counter()
        L.score_attention(Qd, Kd, mode=L.MODE_LSE | L.MODE_RDKV_WT, out=out)
        err = L.device_error()
        elapsed = time.perf_counter() - t0
    finally:
        L.debug_inject(L.DEBUG_NONE, 0)
    assert err == 5, L.STATUS.get(err, err)                          # KVS_ERR_TIMEOUT
    assert elapsed < 10.0
    assert torch.isnan(out["lse"]).all() and torch.isnan(out["w_t"]).all()   # nothing half-merged was written
    # the same context runs the next call normally
    res = L.score_attention(Qd, Kd, mode=L.MODE_LSE | L.MODE_RDKV_WT)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    ref = O.attention_scores(Q.float().numpy().astype(np.float64), K.float().numpy().astype(np.float64), N - W)
    err_lse = np.abs(res["lse"].cpu().numpy() - ref["lse"])
    assert (err_lse <= 2e-3 * np.maximum(1.0, np.abs(ref["lse"]))).all()
