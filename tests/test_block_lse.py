"""Block LSE through the C ABI vs the oracle   [KVSculpt §2].

The row LSE over the leading keys [0, n_block) of each KV head: the attention
mass of the compression zone when the last N - n_block tokens are retained.
Tolerance as for the scoring passes' LSE (fp32 accumulation of bf16 products,
relative 2e-3 of max(1, |lse|)).
"""
import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL = 2e-3


def close(got, ref):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert (err <= TOL * np.maximum(1.0, np.abs(ref))).all(), f"lse worst error {err.max()}"


CASES = [
    # Hq, Hkv, W, N, d, q_pos0, n_block
    (8, 2, 100, 700, 128, 600, 300),     # every query after the block
    (8, 2, 130, 700, 128, 570, 640),     # the block ends inside the window: causal inside it
    (4, 4, 64, 256, 64, 192, 1),         # one key
    (16, 4, 200, 1000, 64, 800, 777),    # d = 64, G = 4, ragged block end
    (8, 1, 64, 2000, 128, 1936, 1024),   # G = 8, block a whole number of key tiles
    (8, 2, 100, 700, 128, 600, 700),     # the whole cache: the plain row LSE
]


@pytest.mark.parametrize("Hq,Hkv,W,N,d,q_pos0,n_block", CASES)
def test_block_lse_vs_oracle(Hq, Hkv, W, N, d, q_pos0, n_block):
    g = torch.Generator().manual_seed(N + n_block)
    Q = torch.randn(Hq, W, d, generator=g).bfloat16()
    K = torch.randn(Hkv, N, d, generator=g).bfloat16()
    lse = L.block_lse(Q.to(DEV), K.to(DEV), n_block, q_pos0=q_pos0)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    close(lse.cpu().numpy(), O.block_lse(Q.double().numpy(), K.double().numpy(), q_pos0, n_block))
    if n_block == N:
        full = L.score_attention(Q.to(DEV), K.to(DEV), q_pos0=q_pos0, mode=L.MODE_LSE)["lse"]
        assert torch.equal(full.cpu(), lse.cpu())          # the same pass, the same plan


def test_block_lse_long_context_sampled_rows():
    """The long-context layer's compression zone (all but the 4096-token window),
    checked on sampled rows of every head."""
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS["long_context_n131072_w4096"]
    t = synth.make_layer(wl)
    n_block = wl.N - wl.W
    lse = L.block_lse(t["Q"].to(DEV), t["K"].to(DEV), n_block, q_pos0=wl.q_pos0).cpu().numpy()
    assert L.device_error() == 0
    rows = [0, 1, 1234, wl.W - 1]
    Q64 = t["Q"][:, rows].double().numpy()
    K64 = t["K"][:, :n_block].double().numpy()
    for i, r in enumerate(rows):
        ref = O.block_lse(Q64[:, i:i + 1], K64, wl.q_pos0 + r, n_block)[:, 0]
        close(lse[:, r], ref)
