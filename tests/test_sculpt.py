"""KVSculpt's attention targets and closed-form values through the C ABI vs the
oracle   [KVSculpt §2: the compressed pairs of the compression zone are fitted
to the block's attention output and LSE; with the keys fixed, the values are a
ridge least-squares solution].

Tolerances, from the fp32 arithmetic of the kernels (u = 2^-24):
  block attention  a logit q.k/sqrt(d) is a sequential fp32 sum of d bf16
                   products, off by at most about d u S with S = sum_c |q_c k_c|
                   / sqrt(d); a softmax weight inherits that relative error
                   and the running sums add n_vis u, so
                     |dY| <= 2 u (d S + n_vis) max|v|,
                     |dlse| <= 2 u (d S + n_vis) + u |lse|.
  ridge values     A^T A, A^T Y and the logits are fp32 sums over R, R and d
                   terms, the Cholesky solve adds k; to first order the
                   solution moves by the condition number kappa of
                   A^T A + lam I times those relative errors:
                     max|dVc| <= kappa u (R + k + d) max|Vc|.
  kappa is taken from the fp64 matrix of the test's own inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
U = 2.0 ** -24


def logit_scale(Q64, K64):
    """max over query rows and keys of sum_c |q_c k_c| / sqrt(d)."""
    d = Q64.shape[-1]
    Qa = np.abs(Q64.reshape(-1, d))
    return max(float((Qa @ np.abs(Kh).T).max()) for Kh in np.abs(K64)) / math.sqrt(d)


def check_block_attention(Y, lse, Yr, lser, d, S, n_vis, vmax):
    bound = 2 * U * (d * S + n_vis)
    errY = np.abs(np.asarray(Y, np.float64) - Yr).max()
    assert errY <= bound * vmax, f"Y worst error {errY} > {bound * vmax}"
    errL = np.abs(np.asarray(lse, np.float64) - lser)
    assert (errL <= bound + U * np.abs(lser)).all(), f"lse worst error {errL.max()}"


CASES = [
    # Hq, Hkv, W, N, d, q_pos0, n_block
    (8, 2, 100, 700, 128, 600, 300),     # every query after the block
    (8, 2, 130, 700, 128, 570, 640),     # the block ends inside the window: causal inside it
    (4, 4, 64, 256, 64, 192, 1),         # one key: Y is its value row
    (16, 4, 200, 1000, 64, 800, 777),    # d = 64, G = 4, ragged block end
    (8, 1, 37, 2000, 128, 1963, 1025),   # G = 8, ragged window, one key past a chunk of 32
    (8, 2, 100, 700, 128, 600, 700),     # the whole cache: plain causal attention
]


@pytest.mark.parametrize("Hq,Hkv,W,N,d,q_pos0,n_block", CASES)
def test_block_attention_vs_oracle(Hq, Hkv, W, N, d, q_pos0, n_block):
    g = torch.Generator().manual_seed(3 * N + n_block)
    Q = torch.randn(Hq, W, d, generator=g).bfloat16()
    K = torch.randn(Hkv, N, d, generator=g).bfloat16()
    V = torch.randn(Hkv, N, d, generator=g).bfloat16()
    Y, lse = L.block_attention(Q.to(DEV), K.to(DEV), V.to(DEV), n_block, q_pos0=q_pos0)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    Q64, K64, V64 = Q.double().numpy(), K.double().numpy(), V.double().numpy()
    Yr, lser = O.block_attention(Q64, K64, V64, q_pos0, n_block)
    check_block_attention(Y.cpu().numpy(), lse.cpu().numpy(), Yr, lser, d,
                          logit_scale(Q64, K64[:, :n_block]), n_block, np.abs(V64[:, :n_block]).max())
    if n_block == 1:  # one key: its weight is 1 and Y is its value row (to the rounding of 1 / l)
        v0 = V[:, :1].float().repeat_interleave(Hq // Hkv, 0).expand(Hq, W, d).numpy()
        assert np.abs(Y.cpu().numpy() - v0).max() <= 4 * U * np.abs(v0).max()
    # the block LSE kernel (tensor-core logits) agrees within its own tolerance
    lse_only = L.block_lse(Q.to(DEV), K.to(DEV), n_block, q_pos0=q_pos0).cpu().numpy()
    assert (np.abs(lse_only - lse.cpu().numpy()) <= 2e-3 * np.maximum(1.0, np.abs(lser))).all()


def test_block_attention_rising_logits_rescale():
    """Keys scaled up along the block, so a tile's row max keeps passing the
    running max by more than the lazy-rescale margin: both softmax groups
    raise their max and scale their O again and again."""
    Hq, Hkv, W, N, d, q_pos0, n_block = 8, 2, 64, 1200, 128, 1136, 1100
    g = torch.Generator().manual_seed(77)
    Q = torch.randn(Hq, W, d, generator=g).abs().bfloat16()
    ramp = (torch.arange(N, dtype=torch.float32) / N * 6.0).view(1, N, 1)
    K = (torch.randn(Hkv, N, d, generator=g).abs() * ramp).bfloat16()
    V = torch.randn(Hkv, N, d, generator=g).bfloat16()
    Y, lse = L.block_attention(Q.to(DEV), K.to(DEV), V.to(DEV), n_block, q_pos0=q_pos0)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    Q64, K64, V64 = Q.double().numpy(), K.double().numpy(), V.double().numpy()
    Yr, lser = O.block_attention(Q64, K64, V64, q_pos0, n_block)
    # every row's largest logit (log2 units) rises by more than two rescale
    # margins (8 each) from the first key tile to the last
    lg = Q64[0] @ K64[0, :n_block].T / math.sqrt(d) * 1.4426950408889634
    assert (lg[:, 1024:].max(axis=1) - lg[:, :128].max(axis=1)).min() > 16
    S = logit_scale(Q64, K64[:, :n_block])
    check_block_attention(Y.cpu().numpy(), lse.cpu().numpy(), Yr, lser, d, S, n_block,
                          np.abs(V64[:, :n_block]).max())


def test_block_attention_without_lse_and_into_out():
    g = torch.Generator().manual_seed(11)
    Q = torch.randn(8, 64, 128, generator=g).bfloat16().to(DEV)
    K = torch.randn(2, 512, 128, generator=g).bfloat16().to(DEV)
    V = torch.randn(2, 512, 128, generator=g).bfloat16().to(DEV)
    Y1, lse = L.block_attention(Q, K, V, 300)
    out = torch.full((8, 64, 128), float("nan"), device=DEV)
    Y2, none = L.block_attention(Q, K, V, 300, want_lse=False, out=out)
    assert none is None and Y2.data_ptr() == out.data_ptr()
    assert torch.equal(Y1, Y2)                       # deterministic, lse or not


def test_block_attention_llama3_8b_layer_sampled_rows():
    """The 8B-shaped layer's compression zone (all but the 512-token window), on
    sampled rows of every head."""
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS["llama3_8b_layer_n8192_w512"]
    t = synth.make_layer(wl)
    n_block = wl.N - wl.W
    Y, lse = L.block_attention(t["Q"].to(DEV), t["K"].to(DEV), t["V"].to(DEV), n_block, q_pos0=wl.q_pos0)
    Y, lse = Y.cpu().numpy(), lse.cpu().numpy()
    assert L.device_error() == 0
    rows = [0, 1, 255, wl.W - 1]
    Q64 = t["Q"][:, rows].double().numpy()
    K64 = t["K"][:, :n_block].double().numpy()
    V64 = t["V"][:, :n_block].double().numpy()
    S = logit_scale(Q64, K64)
    for i, r in enumerate(rows):
        Yr, lser = O.block_attention(Q64[:, i:i + 1], K64, V64, wl.q_pos0 + r, n_block)
        check_block_attention(Y[:, r:r + 1], lse[:, r:r + 1], Yr, lser, wl.d, S, n_block, np.abs(V64).max())


# ---- ridge values -----------------------------------------------------------

def attention_weights(Qh, Kh):
    """softmax_rows(Qh Kh^T / sqrt(d)) in fp64 (for the tolerance only)."""
    S = Qh @ Kh.T / math.sqrt(Qh.shape[-1])
    A = np.exp(S - S.max(axis=1, keepdims=True))
    return A / A.sum(axis=1, keepdims=True)


def lam_and_kappa(Qt64, Kc64, lam_frac):
    """One lam for every head, lam_frac times the smallest lambda_max(A^T A)
    over the heads (rounded to fp32, as the kernel takes it), and the largest
    condition number of A^T A + lam I over the heads."""
    evs = [np.linalg.eigvalsh(attention_weights(Qh, Kh).T @ attention_weights(Qh, Kh))
           for Qh, Kh in zip(Qt64, Kc64)]
    lam = float(np.float32(lam_frac * min(ev.max() for ev in evs)))
    kappa = max((ev.max() + lam) / (max(ev.min(), 0.0) + lam) for ev in evs)
    return lam, kappa


def check_ridge(Vc, Qt64, Kc64, Y64, lam, kappa):
    R, k, d = Qt64.shape[1], Kc64.shape[1], Qt64.shape[2]
    for h in range(Qt64.shape[0]):
        ref = O.ridge_values(Qt64[h], Kc64[h], Y64[h], lam)
        err = np.abs(np.asarray(Vc[h], np.float64) - ref).max()
        bound = kappa * U * (R + k + d) * np.abs(ref).max()
        assert err <= bound, f"head {h}: Vc worst error {err} > {bound} (kappa {kappa:.3g})"


RIDGE = [
    # Hkv, R, k, d, lam as a fraction of lambda_max(A^T A)
    (2, 160, 48, 128, 0.05),
    (2, 160, 48, 128, 0.002),     # kappa in the hundreds
    (3, 100, 33, 64, 0.05),       # d = 64, ragged tiles everywhere
    (1, 7, 1, 128, 0.1),          # one key: sum(Y) / (R + lam) per channel
    (2, 40, 512, 128, 0.05),      # k at its limit, fewer queries than keys
]


@pytest.mark.parametrize("Hkv,R,k,d,lam_frac", RIDGE)
def test_ridge_values_vs_oracle(Hkv, R, k, d, lam_frac):
    g = torch.Generator().manual_seed(R * 1000 + k)
    Qt = torch.randn(Hkv, R, d, generator=g).bfloat16()
    Kc = torch.randn(Hkv, k, d, generator=g).bfloat16()
    Y = (0.3 * torch.randn(Hkv, R, d, generator=g)).float()
    Qt64, Kc64, Y64 = Qt.double().numpy(), Kc.double().numpy(), Y.double().numpy()
    lam, kappa = lam_and_kappa(Qt64, Kc64, lam_frac)
    Vc = L.ridge_values(Qt.to(DEV), Kc.to(DEV), Y.to(DEV), lam)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    check_ridge(Vc.cpu().numpy(), Qt64, Kc64, Y64, lam, kappa)


def test_ridge_values_nan_key_reports_range():
    """A NaN among one head's compressed keys makes every pivot of that head's
    factorisation NaN: the head's values are 0, KVS_ERR_RANGE is recorded, and
    the other head (its own cluster) is unaffected."""
    Hkv, R, k, d = 2, 40, 64, 128
    g = torch.Generator().manual_seed(5)
    Qt = torch.randn(Hkv, R, d, generator=g).bfloat16()
    Kc = torch.randn(Hkv, k, d, generator=g).bfloat16()
    Y = (0.3 * torch.randn(Hkv, R, d, generator=g)).float()
    Kc[0, 3, 7] = float("nan")
    Qt64, Kc64, Y64 = Qt.double().numpy(), Kc.double().numpy(), Y.double().numpy()
    lam, kappa = lam_and_kappa(Qt64[1:], Kc64[1:], 0.05)
    Vc = L.ridge_values(Qt.to(DEV), Kc.to(DEV), Y.to(DEV), lam)
    torch.cuda.synchronize()
    assert L.device_error() == 3                     # KVS_ERR_RANGE
    out = Vc.cpu().numpy()
    assert (out[0] == 0).all()
    check_ridge(out[1:], Qt64[1:], Kc64[1:], Y64[1:], lam, kappa)


def test_ridge_values_after_block_attention_llama3_8b_layer():
    """The chained path on the 8B-shaped layer: the zone's targets Y from the
    block attention, the compressed keys every 15th key of the zone (512 of
    7680), the training queries the window's 4 x 512 queries per KV head."""
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS["llama3_8b_layer_n8192_w512"]
    t = synth.make_layer(wl)
    n_block = wl.N - wl.W
    Q, K, V = t["Q"].to(DEV), t["K"].to(DEV), t["V"].to(DEV)
    Y, _ = L.block_attention(Q, K, V, n_block, q_pos0=wl.q_pos0, want_lse=False)
    G, R = wl.Hq // wl.Hkv, (wl.Hq // wl.Hkv) * wl.W
    Kc = K[:, :n_block:15][:, :512].contiguous()
    heads = [0, wl.Hkv - 1]
    Qt64 = t["Q"].double().numpy().reshape(wl.Hkv, R, wl.d)[heads]
    Kc64 = Kc.cpu().double().numpy()[heads]
    lam, kappa = lam_and_kappa(Qt64, Kc64, 0.05)    # kappa over the two checked heads
    Vc = L.ridge_values(Q.view(wl.Hkv, R, wl.d), Kc, Y.view(wl.Hkv, R, wl.d), lam)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    # the oracle's targets for the two heads, fed to the oracle's solve
    Y64 = np.empty((len(heads), R, wl.d))
    for i, h in enumerate(heads):
        Yh, _ = O.block_attention(t["Q"][h * G:(h + 1) * G].double().numpy(), t["K"][h:h + 1].double().numpy(),
                                  t["V"][h:h + 1].double().numpy(), wl.q_pos0, n_block)
        Y64[i] = Yh.reshape(R, wl.d)
    # Y's own fp32 error (first bound of the module docstring) moves Vc by at most kappa times it
    S = logit_scale(Qt64, t["K"][heads][:, :n_block].double().numpy())
    y_rel = 2 * U * (wl.d * S + n_block) * float(t["V"].abs().max()) / np.abs(Y64).max()
    k, d = Kc.shape[1], wl.d
    for i, h in enumerate(heads):
        ref = O.ridge_values(Qt64[i], Kc64[i], Y64[i], lam)
        err = np.abs(Vc[h].cpu().numpy().astype(np.float64) - ref).max()
        bound = kappa * (U * (R + k + d) + y_rel) * np.abs(ref).max()
        assert err <= bound, f"head {h}: Vc worst error {err} > {bound} (kappa {kappa:.3g})"
