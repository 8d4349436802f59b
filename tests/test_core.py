"""KV-CoRE Gram accumulation and spectrum through the C ABI vs the oracle
[KV-CoRE §2].

Tolerances.  bf16 products are exact in fp32 and the tensor cores add them in
fp32: a CTA adds its token range into two accumulators (even and odd tiles)
16 tokens per step, and the ranges are added in order, so entry (i, j) of G
is within (range / 32 + ranges) * 2^-24 of its own scale sum_t |x_ti| |x_tj|
in the worst case; the tests allow twice that, at least 1e-5, entry by entry.  The spectrum comes from fp32 Jacobi on that G: an
eigenvalue moves by at most about 1e-6 * |G|_F, so sigma = sqrt(lambda) moves
by at most 1e-6 relative for the large values and by sqrt(1e-6 |G|_F) for the
smallest; the NER is compared within 1e-3 with the rank equal, on data whose
singular values keep a clear margin from the rank threshold.
"""
import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def structured(Hkv, N, seed, ranks=(64,), scale_hi=(1.0, 0.1), low=1e-5):
    """X = Z diag(s) R: s spans scale_hi over the first r channels, then `low`."""
    g = torch.Generator().manual_seed(seed)
    out = []
    for h in range(Hkv):
        r = ranks[h % len(ranks)]
        s = torch.cat([torch.logspace(np.log10(scale_hi[0]), np.log10(scale_hi[1]), r), torch.full((128 - r,), low)])
        Rm, _ = torch.linalg.qr(torch.randn(128, 128, generator=g, dtype=torch.float64))
        Z = torch.randn(N, 128, generator=g, dtype=torch.float64)
        out.append((Z * s.double()) @ Rm.T)
    return torch.stack(out).float().bfloat16()


def gram_rtol(Hkv, N):
    ranges = max(1, min(-(-N // 128), torch.cuda.get_device_properties(0).multi_processor_count // Hkv))
    per = -(-N // ranges)
    return max(1e-5, 2 * (per / 32 + ranges) * 2.0 ** -24)


def check_gram(G, X, keep=None):
    """Every entry within tol * sum_t |x_ti| |x_tj| (the scale of that entry's
    own fp32 sum of exact bf16 products), not a bound shared by the whole matrix."""
    x64 = X.double().numpy()
    ref = O.gram(x64, keep)
    got = G.cpu().numpy().astype(np.float64)
    tol = gram_rtol(x64.shape[0], x64.shape[1])
    for g in range(x64.shape[0]):
        a = np.abs(x64[g] if keep is None else x64[g][keep[g]])
        scale = a.T @ a
        err = np.abs(got[g] - ref[g])
        bad = err > tol * scale + 1e-30
        assert not bad.any(), (g, err[bad].max(), scale[bad].min())


@pytest.mark.parametrize("Hkv,N", [(2, 1000), (1, 1), (3, 129), (8, 4096)])
def test_gram_vs_oracle(Hkv, N):
    g = torch.Generator().manual_seed(N)
    X = (torch.randn(Hkv, N, 128, generator=g) * torch.exp(torch.randn(Hkv, 1, 128, generator=g))).bfloat16()
    G = L.gram(X.to(DEV))
    torch.cuda.synchronize()
    assert L.device_error() == 0
    check_gram(G, X)
    keep = (torch.rand(Hkv, N, generator=g) > 0.4).to(torch.uint8)
    Gk = L.gram(X.to(DEV), keep.to(DEV))
    check_gram(Gk, X, keep.numpy().astype(bool))


def test_gram_accumulates_over_token_blocks():
    g = torch.Generator().manual_seed(5)
    X = torch.randn(2, 700, 128, generator=g).bfloat16()
    G = L.gram(X[:, :300].contiguous().to(DEV))
    L.gram(X[:, 300:].contiguous().to(DEV), out=G, accumulate=True)
    torch.cuda.synchronize()
    check_gram(G, X)


@pytest.mark.parametrize("ranks", [(64,), (128, 20, 1, 100)])
def test_spectrum_and_ner_vs_oracle(ranks):
    Hkv = len(ranks)
    X = structured(Hkv, 3000, seed=sum(ranks), ranks=ranks)
    G = L.gram(X.to(DEV))
    sigma, ner, rank = L.spectrum(G, rtol=1e-3)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    ref_sig = O.spectrum(O.gram(X.double().numpy()))
    for g in range(Hkv):
        s_ref = ref_sig[g]
        smax = s_ref[0]
        # the data keep a clear margin from the rank threshold
        assert not np.any(np.abs(s_ref - 1e-3 * smax) < 0.2 * 1e-3 * smax)
        s = sigma[g].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(s - s_ref) <= 1e-5 * s_ref + np.sqrt(2e-6) * smax), np.abs(s - s_ref).max()
        assert int(rank[g]) == O.numerical_rank(s_ref, 1e-3) == ranks[g]
        assert abs(float(ner[g]) - O.ner(s_ref, 1e-3)) <= 1e-3


def test_spectrum_special_cases():
    G = torch.zeros(2, 128, 128, device=DEV)
    G[1] = torch.eye(128, device=DEV) * 4.0                       # equal singular values 2: NER 1
    sigma, ner, rank = L.spectrum(G)
    torch.cuda.synchronize()
    assert float(ner[0]) == 0.0 and int(rank[0]) == 0 and float(sigma[0].abs().max()) == 0.0
    assert int(rank[1]) == 128 and abs(float(ner[1]) - 1.0) < 1e-5
    assert torch.allclose(sigma[1], torch.full((128,), 2.0, device=DEV))


def test_gram_full_size_properties():
    """The long-context K cache (8 heads x 131 072 tokens): G is symmetric, its
    trace is |X|_F^2 (summed on the host in float64) and it is positive
    semidefinite within the fp32 bound."""
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS["long_context_n131072_w4096"]
    K = synth.make_layer(wl)["K"]
    G = L.gram(K.to(DEV))
    sigma, ner, rank = L.spectrum(G)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    Gc = G.cpu().double()
    k64 = K.double()
    tol = gram_rtol(wl.Hkv, wl.N)
    for g in range(wl.Hkv):
        fro2 = float((k64[g] ** 2).sum())
        assert abs(float(torch.trace(Gc[g])) - fro2) <= tol * fro2
        assert float((Gc[g] - Gc[g].T).abs().max()) <= 1e-6 * fro2
        assert abs(float((sigma[g].double() ** 2).sum().cpu()) - fro2) <= 1e-4 * fro2   # sum sigma^2 = trace
        assert 0 < int(rank[g]) <= 128 and 1.0 / int(rank[g]) - 1e-6 <= float(ner[g]) <= 1.0 + 1e-6
