"""kvs_allocate_bits_static: bit allocation without any caller-provided device memory.

Some hosts of this library (an inference engine that has already reserved the
device memory for its own pool, a plug-in that is not allowed to allocate)
cannot hand the allocator a workspace.  For them the library keeps one fixed
scratch array of its own.  These tests call that entry point through the C ABI
and require exactly the widths that kvs_allocate_bits gives with an ordinary
workspace, on two calls in a row, so that anything the first call leaves in the
shared array cannot leak into the second.  This file is named to be collected
last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from kv_cache_compression_flash_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _weights(U, seed):
    rng = np.random.default_rng(seed)
    w = (rng.random(U) ** 3 * 10).astype(np.float32)
    s = (rng.random(U) + 0.05).astype(np.float32)
    w[rng.random(U) < 0.05] = 0          # units that are always evicted
    w[::13] = w[7]                       # ties between units
    s[::13] = s[7]
    return torch.from_numpy(w).to(DEV), torch.from_numpy(s).to(DEV)


def _static(w, s, budget, mask):
    bits = torch.full((w.numel(),), 0xEE, dtype=torch.uint8, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.lib().kvs_allocate_bits_static(ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(s.data_ptr()), w.numel(),
                                          budget, mask, ctypes.c_void_p(bits.data_ptr()), stream)
    assert rc == 0, L.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    return bits


# Pools that fit one thread-block cluster's shared memory need no scratch at
# all; these sizes are past that, so both calls run the grid allocator on the
# library's scratch array.
SCRATCH_SIZES = {L.WIDTHS_ALL: (400000, 250000), L.WIDTHS_KEEP_OR_EVICT: (1000000, 700000)}


@pytest.mark.parametrize("mask", [L.WIDTHS_ALL, L.WIDTHS_KEEP_OR_EVICT])
def test_static_scratch_matches_workspace_allocator_twice(mask):
    # the first call is the larger one, so stale scratch would be visible in the second
    big, small = SCRATCH_SIZES[mask]
    for U in (big, small):
        cl, blocks, ws_bytes = L.allocate_plan_info(U, mask)
        # the grid path, whose scratch lives in the library's array, and it fits there
        assert cl == 0 and blocks > 0 and 0 < ws_bytes <= L.lib().kvs_allocate_workspace_size(U)
    for U, seed, avg in ((big, 1, 3.0), (small, 2, 2.5)):
        w, s = _weights(U, seed)
        budget = int(math.floor(avg * U))
        expect = L.allocate_bits(w, s, budget, mask)
        got = _static(w, s, budget, mask)
        assert L.device_error() == 0
        assert torch.equal(got, expect), (U, (got != expect).sum().item())


def test_static_scratch_rejects_bad_sizes():
    p = ctypes.c_void_p(1 << 20)
    assert L.lib().kvs_allocate_bits_static(p, p, -1, 10, L.WIDTHS_ALL, p, None) == 1
    assert L.lib().kvs_allocate_bits_static(p, p, 10, -5, L.WIDTHS_ALL, p, None) == 1
