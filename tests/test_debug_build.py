"""The bounds-checked library (libkvs_debug.so, compiled with KVS_DEBUG).

It checks every data-dependent index the kernels compute (gathered kept
tokens, stream group entries, the kept-token lists of the channel plan)
before the access, records KVS_ERR_BOUNDS and skips the access when one is
out of range.  It stands in for a memory checker.  These tests require that
it exports the same ABI and that on valid inputs it gives the same results as
libkvs.so with the error word still clear.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from kv_cache_compression_flash_b300 import _lib as L
from kv_cache_compression_flash_b300 import synth
from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep

DEBUG_LIB = os.path.join(os.path.dirname(L.LIB_PATH), "libkvs_debug.so")


@pytest.fixture
def debug_lib():
    """Switches the binding to the checked library for one test."""
    assert os.path.exists(DEBUG_LIB), "built by __graft_entry__.build()"
    saved_path, saved_lib = L.LIB_PATH, L._lib
    L.LIB_PATH, L._lib = DEBUG_LIB, None
    try:
        yield L.lib()
    finally:
        L.LIB_PATH, L._lib = saved_path, saved_lib


def test_debug_library_exports_the_abi(debug_lib):
    for name in L.SIGNATURES:
        assert hasattr(debug_lib, name), name
    assert debug_lib.kvs_status_string(7).decode() == "KVS_ERR_BOUNDS"
    assert debug_lib.kvs_version() == ctypes.CDLL(os.path.join(os.path.dirname(DEBUG_LIB), "libkvs.so")).kvs_version()


def _pooled_run(Q, K, V, shape, P):
    Hq, Hkv, N, W, d = shape
    st = RdkvLayerStep(Hq, Hkv, N, W, d, 3, device=Q.device, n_pools=P)
    st.run(Q, K, V)
    torch.cuda.synchronize()
    err = L.device_error()
    return err, {k: v.clone() for k, v in (("w_t", st.out["w_t"]), ("bits_v", st.bits_v), ("bits_k", st.bits_k),
                                           ("v_hat", st.v_hat), ("k_hat", st.k_hat))}


@pytest.mark.gpu
def test_checked_build_matches_on_a_pooled_step():
    wl = synth.WORKLOADS["llama3_8b_layer_n8192_w512"].small(N=700, W=100, Hq=8, Hkv=2)
    P = 3
    dev = torch.device("cuda:0")
    x = synth.make_pools(wl, 0, range(P), device=dev)
    shape = (wl.Hq, wl.Hkv, wl.N, wl.W, wl.d)
    err, ref = _pooled_run(x["Q"], x["K"], x["V"], shape, P)
    assert err == 0
    saved_path, saved_lib = L.LIB_PATH, L._lib
    L.LIB_PATH, L._lib = DEBUG_LIB, None
    try:
        err_d, got = _pooled_run(x["Q"], x["K"], x["V"], shape, P)
    finally:
        L.LIB_PATH, L._lib = saved_path, saved_lib
    assert err_d == 0, L.STATUS.get(err_d, err_d)
    for k in ref:
        assert torch.equal(ref[k], got[k]), k


@pytest.mark.gpu
def test_checked_build_pack_dequant_random_widths(debug_lib):
    rng = np.random.default_rng(5)
    dev = torch.device("cuda:0")
    Hkv, N, d = 3, 1000, 128
    X = torch.from_numpy(rng.standard_normal((Hkv, N, d)).astype(np.float32)).bfloat16().to(dev)
    bits_v = torch.from_numpy(rng.choice([0, 2, 4, 8, 16], size=Hkv * N).astype(np.uint8)).to(dev)
    st = L.Streams(Hkv, N, d, 0, int(bits_v.int().sum()), dev)
    L.quantize_pack(X, 0, bits_v, None, st)
    xh = L.dequantize(st, bits_v, None)
    bits_k = torch.from_numpy(rng.choice([0, 2, 4, 8, 16], size=Hkv * d).astype(np.uint8)).to(dev)
    sk = L.Streams(Hkv, N, d, 1, int(bits_k.int().sum()), dev)
    L.quantize_pack(X, 1, bits_k, bits_v, sk)
    kh = L.dequantize(sk, bits_k, bits_v)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    # evicted tokens and channels come back as zeros, kept ones within half a step
    keep = (bits_v.view(Hkv, N) > 0).cpu()
    assert torch.all(xh.cpu()[~keep] == 0)
    assert torch.isfinite(kh).all()
