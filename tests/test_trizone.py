"""TriZone decode attention through the C ABI vs the oracle   [RDKV §2.3].

The oracle dequantises both caches (itself pinned bit-exact against the GPU
pack) and runs plain float64 attention over the kept tokens and the zone C
rows.  Tolerance: the kernel works in fp32 with the logits in the log2
domain and ex2.approx (relative error about 2^-22); a logit carries an
absolute error of about 2^-24 * sum_c |q_c k_c| (under 1e-6 here) and the
output inherits it times max|v|.  The test allows 1e-4 * max|v| on the output
and 1e-4 * max(1, |lse|) on lse: a single misplaced token among a thousand
moves the output by about 1e-3 * |v|, ten times the bound.
"""
import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL = 1e-4


def make_case(Hq, Hkv, N, nc_cap, seed, p_evict=0.3, d=128, kv_widths=(0, 2, 4, 8, 16), qscale=1.0):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    K = (torch.randn(Hkv, N, d, generator=g) * 1.5).bfloat16()
    V = torch.randn(Hkv, N, d, generator=g).bfloat16()
    q = (torch.randn(Hq, d, generator=g) * qscale).bfloat16()
    kn = (torch.randn(Hkv, max(nc_cap, 1), d, generator=g) * 1.5).bfloat16()[:, :nc_cap].contiguous()
    vn = torch.randn(Hkv, max(nc_cap, 1), d, generator=g).bfloat16()[:, :nc_cap].contiguous()
    keep_w = [w for w in kv_widths if w]
    bits_v = np.where(rng.random(Hkv * N) < p_evict, 0, rng.choice(keep_w, size=Hkv * N)).astype(np.uint8)
    bits_k = rng.choice(kv_widths, size=Hkv * d).astype(np.uint8)
    return dict(q=q, K=K, V=V, kn=kn, vn=vn, bits_v=bits_v, bits_k=bits_k)


def gpu_pack(c):
    Hkv, N, d = c["K"].shape
    bv = torch.from_numpy(c["bits_v"]).to(DEV)
    bk = torch.from_numpy(c["bits_k"]).to(DEV)
    sv = L.Streams(Hkv, N, d, 0, int(c["bits_v"].astype(int).sum()), DEV)
    sk = L.Streams(Hkv, N, d, 1, int(c["bits_k"].astype(int).sum()), DEV)
    L.quantize_pack(c["V"].to(DEV), 0, bv, None, sv)
    L.quantize_pack(c["K"].to(DEV), 1, bk, bv, sk)
    idx = L.trizone_index(sk, sv, bv)
    return sk, sv, bv, idx


def oracle_decode(c, nc):
    Hkv, N, d = c["K"].shape
    K64 = c["K"].double().numpy()
    V64 = c["V"].double().numpy()
    keep = (c["bits_v"] > 0).reshape(Hkv, N)
    Kh = O.dequantize(O.quantize_pack(K64, 1, c["bits_k"], keep), K64.shape, 1, c["bits_k"], keep)
    Vh = O.dequantize(O.quantize_pack(V64, 0, c["bits_v"]), V64.shape, 0, c["bits_v"])
    kn = c["kn"][:, :nc].double().numpy() if nc else None
    vn = c["vn"][:, :nc].double().numpy() if nc else None
    return O.trizone_decode(c["q"].double().numpy(), Kh, Vh, keep, kn, vn), Vh


def check(out, lse, ref, vmax):
    ro, rl = ref
    out = out.cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    err = np.abs(out - ro)
    assert err.max() <= TOL * vmax, f"out worst error {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"
    assert np.array_equal(np.isinf(lse), np.isinf(rl))
    f = np.isfinite(rl)
    assert (np.abs(lse[f] - rl[f]) <= TOL * np.maximum(1.0, np.abs(rl[f]))).all(), np.abs(lse[f] - rl[f]).max()


CASES = [
    # Hq, Hkv, N, nc_cap, nc, p_evict
    (8, 2, 300, 0, 0, 0.3),        # G=4, one full chunk and a ragged tail, no zone C
    (4, 4, 1, 0, 0, 0.0),          # one token, G=1
    (4, 2, 1000, 300, 300, 0.5),   # G=2, zone C spans a full chunk and a tail
    (16, 2, 2000, 64, 17, 0.3),    # G=8: two head slices per KV head
    (8, 2, 700, 8, 1, 0.97),       # nearly everything evicted
    (32, 8, 8192, 128, 100, 0.3),  # the layer shape of an 8B-class model
]


@pytest.mark.parametrize("Hq,Hkv,N,nc_cap,nc,p_evict", CASES)
def test_trizone_decode_vs_oracle(Hq, Hkv, N, nc_cap, nc, p_evict):
    c = make_case(Hq, Hkv, N, nc_cap, seed=N + Hq, p_evict=p_evict)
    sk, sv, bv, idx = gpu_pack(c)
    n_new = torch.tensor([nc], dtype=torch.int32, device=DEV)
    kn = c["kn"].to(DEV) if nc_cap else None
    vn = c["vn"].to(DEV) if nc_cap else None
    out, lse = L.trizone_decode(c["q"].to(DEV), sk, sv, idx, kn, vn, n_new if nc_cap else None)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    ref, Vh = oracle_decode(c, nc)
    vmax = max(np.abs(Vh).max(), float(c["vn"].abs().max()) if nc_cap else 0.0)
    check(out, lse, ref, vmax)


def test_trizone_nothing_visible_and_zone_c_only():
    c = make_case(8, 2, 500, 40, 0, p_evict=1.0)
    sk, sv, bv, idx = gpu_pack(c)
    hv = sk.host_view()
    ref = O.quantize_pack(c["K"].double().numpy(), 1, c["bits_k"], np.zeros((2, 500), bool))
    for wd in (2, 4, 8, 16):                          # channels over no kept token: listed, no groups
        assert hv[wd]["n_groups"] == 0 and np.array_equal(hv[wd]["ids"], ref[wd]["ids"])
    n_new = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = L.trizone_decode(c["q"].to(DEV), sk, sv, idx, c["kn"].to(DEV), c["vn"].to(DEV), n_new)
    torch.cuda.synchronize()
    assert (out.cpu() == 0).all() and torch.isinf(lse.cpu()).all() and (lse.cpu() < 0).all()
    n_new.fill_(40)
    out, lse = L.trizone_decode(c["q"].to(DEV), sk, sv, idx, c["kn"].to(DEV), c["vn"].to(DEV), n_new)
    ref, _ = oracle_decode(c, 40)
    check(out, lse, ref, float(c["vn"].abs().max()))
    assert L.device_error() == 0


def test_trizone_widths_16_only_is_dense_attention():
    """Every kept token and channel at width 16: the decode reads the raw bf16
    values, so it must match attention over the bf16 cache itself."""
    c = make_case(8, 2, 600, 0, 0, p_evict=0.2, kv_widths=(0, 16))
    c["bits_k"][:] = 16
    sk, sv, bv, idx = gpu_pack(c)
    out, lse = L.trizone_decode(c["q"].to(DEV), sk, sv, idx)
    keep = (c["bits_v"] > 0).reshape(2, 600)
    ref = O.trizone_decode(c["q"].double().numpy(), c["K"].double().numpy(), c["V"].double().numpy(), keep)
    check(out, lse, ref, float(c["V"].abs().max()))
    assert L.device_error() == 0


def test_trizone_graph_replay_as_zone_c_grows():
    """n_new is read on the device, so one captured graph serves successive
    decode steps while zone C fills."""
    c = make_case(8, 2, 1500, 300, 0, p_evict=0.4)
    sk, sv, bv, idx = gpu_pack(c)
    q, kn, vn = c["q"].to(DEV), c["kn"].to(DEV), c["vn"].to(DEV)
    n_new = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(8, 128, device=DEV)
    lse = torch.empty(8, device=DEV)
    ws = L.Workspace()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.trizone_decode(q, sk, sv, idx, kn, vn, n_new, out=out, lse=lse, ws=ws)   # sizes the workspace
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            L.trizone_decode(q, sk, sv, idx, kn, vn, n_new, out=out, lse=lse, ws=ws)
    vmax = max(float(c["V"].abs().max()), float(c["vn"].abs().max()))
    for nc in (0, 1, 255, 256, 257, 300):
        n_new.fill_(nc)
        gr.replay()
        torch.cuda.synchronize()
        ref, _ = oracle_decode(c, nc)
        check(out, lse, ref, vmax)
    assert L.device_error() == 0


def test_trizone_mismatched_index_is_reported():
    """An index built from widths the V streams were not packed with is
    reported in the error word; the decode stays inside the streams."""
    c = make_case(4, 2, 400, 0, 0, p_evict=0.3)
    sk, sv, bv, idx = gpu_pack(c)
    wrong = torch.from_numpy(np.roll(c["bits_v"], 1)).to(DEV)
    idx2 = L.trizone_index(sk, sv, wrong)
    L.trizone_decode(c["q"].to(DEV), sk, sv, idx2)
    torch.cuda.synchronize()
    assert L.device_error() == 3
