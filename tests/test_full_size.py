"""CUDA path vs the CPU oracle at the workloads' full sizes.

The oracle cannot materialise these attention matrices whole in a test's time,
so each check is one of:
  * sampled outputs the oracle computes exactly (LSE of chosen rows; w_t / s+
    of keys whose every query row is in the oracle's slice; whole KV groups
    split by query head over spawned workers);
  * properties that hold at any size (each softmax row sums to one, so
    sum_t w_t = G * W per KV head; the {0,16} allocation keeps exactly the top
    keys; |x - x_hat| <= s/2 for every packed element);
  * allocation and packing fed seeded weights and widths, compared bit for bit
    (whole pools for allocation, sampled units for packing).
Tolerances are those of test_gpu_parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L
from kv_cache_compression_flash_b300 import synth
from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep

from oracle_jobs import f64, per_head_scores
from test_gpu_parity import _cmp_streams, assert_lse_close, assert_scores_close, gpu_alloc

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL = 2e-3


def check_sampled_lse(lse_gpu, Q, K, G, q_pos0, heads, rows):
    """lse of (head, row) pairs, each from the oracle on that single row."""
    for hd in heads:
        g = hd // G
        Kg = f64(K[g:g + 1])
        for r in rows:
            ref = O.attention_scores(f64(Q[hd:hd + 1, r:r + 1]), Kg, q_pos0 + r)["lse"][0, 0]
            got = float(lse_gpu[hd, r])
            assert abs(got - ref) <= TOL * max(1.0, abs(ref)), (hd, r, got, ref)


def check_tail_keys(gpu, Q, K, G, q_pos0, g, tail, key, **norms):
    """Keys t >= N - tail are seen only by rows at positions >= N - tail, so the
    oracle on that slice of rows gives their exact scores."""
    N = K.shape[1]
    W = Q.shape[1]
    r0 = W - tail
    extra = {}
    if norms:
        extra = {"V": f64(norms["V"][g]), "h": f64(norms["h"][r0:]), "W_O_heads": norms["W_O_heads"]}
    per = per_head_scores(f64(Q[g * G:(g + 1) * G, r0:]), f64(K[g]), q_pos0 + r0, **extra)
    if key == "w_t":
        ref = np.sum([p["w_t"] for p in per], axis=0)
    else:
        ref = np.max([p[key] for p in per], axis=0)
    assert_scores_close(gpu[g, N - tail:], ref[N - tail:], f"{key} tail of group {g}")


def check_pack_sampled(X, axis, bits, keep, streams, units, xhat):
    """Sampled units: stream bytes, scales and dequantised values equal the
    oracle's, each unit packed on its own."""
    Hkv, N, d = X.shape
    hv = streams.host_view()
    for u in units:
        wd = int(bits[u])
        if wd == 0:
            continue
        if axis == 0:
            g, t = divmod(int(u), N)
            Xs = f64(X[g:g + 1, t:t + 1])
            ref = O.quantize_pack(Xs, 0, np.array([wd], np.uint8))
            ref_hat = O.dequantize(ref, Xs.shape, 0, np.array([wd], np.uint8))[0, 0]
            got_hat = xhat[g, t]
        else:
            g, c = divmod(int(u), d)
            Xs = f64(X[g:g + 1])
            bsub = np.zeros(d, np.uint8)
            bsub[c] = wd
            ks = keep[g:g + 1]
            ref = O.quantize_pack(Xs, 1, bsub, ks)
            ref_hat = O.dequantize(ref, Xs.shape, 1, bsub, ks)[0][ks[0], c]
            got_hat = xhat[g, ks[0], c]
        r = ref[wd]
        st = hv[wd]
        j = np.nonzero(st["ids"] == u)[0]
        assert j.size == 1, (u, wd)
        g0 = int(st["group_offsets"][j[0]])
        ng = r["n_groups"]
        assert np.array_equal(st["codes"][g0 * 8 * wd:(g0 + ng) * 8 * wd], r["codes"]), (u, wd)
        if wd != 16:
            assert np.array_equal(st["scales"][g0:g0 + ng], r["scales"]), (u, wd)
        assert np.array_equal(np.asarray(got_hat, np.float32), ref_hat.astype(np.float32)), (u, wd)


def check_roundtrip_bound(X, axis, bits, keep, xhat):
    """Every packed element is within s/2 of its input, s = its group's scale
    <= absmax/qmax (1 + 2^-10) (or one fp16 subnormal step); evicted units and
    dropped tokens dequantise to 0; width 16 is exact."""
    Hkv, N, d = X.shape
    x = X.float()
    b = bits.long()
    if axis == 0:
        xs = [x.reshape(Hkv * N, d)]
        hs = [xhat.reshape(Hkv * N, d)]
        ws = [b.reshape(Hkv * N, 1).expand(Hkv * N, d)]
        kept_all = torch.ones(Hkv, N, dtype=torch.bool, device=X.device)
    else:
        kept_all = keep.reshape(Hkv, N) != 0
        # per head: [d channels, kept tokens] so that a unit is a row
        xs = [x[g][kept_all[g]].T.contiguous() for g in range(Hkv)]
        hs = [xhat[g][kept_all[g]].T.contiguous() for g in range(Hkv)]
        ws = [b.reshape(Hkv, d)[g].reshape(d, 1).expand(d, xs[g].shape[1]) for g in range(Hkv)]
    dropped = ~kept_all
    assert torch.all(xhat[dropped] == 0)
    for xu, hu, wu in zip(xs, hs, ws):
        n = xu.shape[1]
        if n == 0:
            continue
        assert torch.all(hu[wu == 0] == 0)
        assert torch.all(hu[wu == 16] == xu[wu == 16])
        pad = (-n) % 64
        xp = torch.nn.functional.pad(xu.abs(), (0, pad))
        amax = xp.reshape(xu.shape[0], -1, 64).amax(dim=2, keepdim=True).expand(-1, -1, 64)
        amax = amax.reshape(xu.shape[0], -1)[:, :n]
        err = (hu - xu).abs()
        for wd in (2, 4, 8):
            m = wu == wd
            if torch.any(m):
                qmax = 2 ** (wd - 1) - 1
                bound = amax / qmax * (1 + 2.0 ** -10) / 2 + 2.0 ** -25
                assert torch.all(err[m] <= bound[m]), wd


# ---------------------------------------------------------------------------
# KVzip+ over a repeated prompt: N = W = 32768, full causal, hidden 4096
# ---------------------------------------------------------------------------
def test_kvzip_plus_full_size():
    wl = synth.WORKLOADS["kvzip_plus_n32768_d4096"]
    t = synth.make_layer(wl)
    G, d = wl.G, wl.d
    Qd, Kd, Vd, hd, Wod = (t[k].to(DEV) for k in ("Q", "K", "V", "h", "W_O"))
    out = L.score_attention(Qd, Kd, q_pos0=0, mode=L.MODE_LSE | L.MODE_KVZIP_PLUS, V=Vd, h=hd, W_O=Wod)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    lse = out["lse"].cpu().numpy()
    sp = out["s_plus"].cpu().numpy()
    assert np.isfinite(lse).all() and np.isfinite(sp).all() and (sp > 0).all()
    check_sampled_lse(lse, t["Q"], t["K"], G, 0, heads=(0, 13, 31),
                      rows=(0, 1, 127, 128, 129, 4095, 16383, 32766, 32767))
    for g in (0, 7):
        wo_heads = np.stack([f64(t["W_O"][:, (g * G + i) * d:(g * G + i + 1) * d]) for i in range(G)])
        check_tail_keys(sp, t["Q"], t["K"], G, 0, g, 300, "s_plus", V=t["V"], h=t["h"], W_O_heads=wo_heads)
    # every key of KV group 5 against the oracle (the merge over pass 2's splits
    # is covered at a size that splits, in test_gpu_parity.py)
    g = 5
    wo_heads = np.stack([f64(t["W_O"][:, (g * G + i) * d:(g * G + i + 1) * d]) for i in range(G)])
    per = per_head_scores(f64(t["Q"][g * G:(g + 1) * G]), f64(t["K"][g]), 0, V=f64(t["V"][g]), h=f64(t["h"]),
                          W_O_heads=wo_heads, workers=G)
    assert_scores_close(sp[g], np.max([p["s_plus"] for p in per], axis=0), f"s_plus group {g}")
    assert_lse_close(lse[g * G:(g + 1) * G], np.stack([p["lse"] for p in per]))
    # evict the bottom 80%: widths {0,16}, sigma = 1, B = 16 * keep -> exactly the top keys stay
    U = wl.Hkv * wl.N
    B = synth.kvzip_keep_budget(U, wl.evict_fraction)
    bits = L.allocate_bits(out["s_plus"], torch.ones_like(out["s_plus"]), B, L.WIDTHS_KEEP_OR_EVICT)
    torch.cuda.synchronize()
    b = bits.cpu().numpy()
    keep = B // 16
    order = np.lexsort((np.arange(U), -sp.ravel().astype(np.float64)))
    expect = np.zeros(U, np.uint8)
    expect[order[:keep]] = 16
    assert (b == expect).all()
    assert L.device_error() == 0


# ---------------------------------------------------------------------------
# long-context layer: N = 131072, window 4096, budgets 2 / 3 / 4 bits
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def long_layer():
    wl = synth.WORKLOADS["long_context_n131072_w4096"]
    return wl, synth.make_layer(wl)


def test_long_context_scores(long_layer):
    wl, t = long_layer
    G = wl.G
    Q, K, V = (t[k].to(DEV) for k in ("Q", "K", "V"))
    step = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, 3, device=DEV)
    step.run(Q, K, V)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    lse = step.out["lse"].cpu().numpy()
    wt = step.out["w_t"].cpu().numpy()
    # each softmax row sums to one: sum_t w_t = G * W for every KV head
    np.testing.assert_allclose(wt.astype(np.float64).sum(axis=1), G * wl.W, rtol=1e-4)
    check_sampled_lse(lse, t["Q"], t["K"], G, wl.q_pos0, heads=(0, 17, 31), rows=(0, 1, 2047, 4094, 4095))
    check_tail_keys(wt, t["Q"], t["K"], G, wl.q_pos0, 5, 256, "w_t")
    # one whole KV group (sinks, outlier channels, every key) against the oracle
    g = 3
    per = per_head_scores(f64(t["Q"][g * G:(g + 1) * G]), f64(t["K"][g]), wl.q_pos0)
    assert_scores_close(wt[g], np.sum([p["w_t"] for p in per], axis=0), f"w_t group {g}")
    assert_lse_close(lse[g * G:(g + 1) * G], np.stack([p["lse"] for p in per]))
    # w_c and sigma against the oracle at full size
    np.testing.assert_allclose(step.w_c.cpu().numpy(), O.channel_weights(f64(t["Q"]), f64(t["K"])), rtol=TOL)
    np.testing.assert_allclose(step.sig_t.cpu().numpy(), O.unit_rms(f64(t["V"]), 0), rtol=TOL)


@pytest.mark.parametrize("avg_bits", [2, 3, 4])
def test_long_context_alloc_pack(long_layer, avg_bits):
    """Seeded weights shaped like the layer's (heavy-tailed w, RMS-like sigma):
    allocation bit-exact on the whole 1M-unit pool; pack/dequantise bit-exact on
    sampled units and within s/2 everywhere."""
    wl, t = long_layer
    Hkv, N, d = wl.Hkv, wl.N, wl.d
    U = Hkv * N
    rng = np.random.default_rng(1000 + avg_bits)
    w = (np.exp(rng.standard_normal(U) * 2.0) * 1e-3).astype(np.float32)
    w[rng.random(U) < 0.01] = 0
    s = (1.0 + 0.1 * rng.standard_normal(U)).astype(np.float32).clip(0.5)
    B = int(math.floor(avg_bits * U))
    bits_v = O.allocate_bits(w, s, B)
    assert (gpu_alloc(w, s, B) == bits_v).all()
    wc = (np.exp(rng.standard_normal(Hkv * d)) * 10).astype(np.float32)
    sc = (1.0 + rng.random(Hkv * d)).astype(np.float32)
    Bk = int(math.floor(avg_bits * Hkv * d))
    bits_k = O.allocate_bits(wc, sc, Bk)
    assert (gpu_alloc(wc, sc, Bk) == bits_k).all()
    V, K = t["V"].to(DEV), t["K"].to(DEV)
    bv, bk = torch.from_numpy(bits_v).to(DEV), torch.from_numpy(bits_k).to(DEV)
    sv = L.Streams(Hkv, N, d, 0, B, DEV)
    L.quantize_pack(V, 0, bv, None, sv)
    vh = L.dequantize(sv, bv, None)
    sk = L.Streams(Hkv, N, d, 1, Bk, DEV)
    L.quantize_pack(K, 1, bk, bv, sk)
    kh = L.dequantize(sk, bk, bv)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    keep = (bits_v > 0).reshape(Hkv, N)
    units_v = np.concatenate([np.arange(8), rng.choice(U, 200, replace=False), np.arange(U - 8, U)])
    check_pack_sampled(t["V"], 0, bits_v, None, sv, units_v, vh.cpu().numpy())
    check_pack_sampled(t["K"], 1, bits_k, keep, sk, (0, 1, 127, 300, 513, Hkv * d - 1), kh.cpu().numpy())
    check_roundtrip_bound(V, 0, bv, None, vh)
    check_roundtrip_bound(K, 1, bk, bv, kh)


# ---------------------------------------------------------------------------
# full model: 32 layers x 16 sequences, sampled (layer, sequence) pools
# ---------------------------------------------------------------------------
def test_full_model_pooled_layer():
    """One layer of the full-model batch, its 16 sequences as 16 pools of one
    pooled step (inputs drawn on the device): every KV head's weights sum to
    G * W; sampled pools against the oracle on that pool alone, allocation
    and packing fed the oracle's weights bit-exact inside the pooled calls."""
    wl = synth.WORKLOADS["full_model_l32_b16_n16384"]
    layer, P = 31, wl.seqs
    t = synth.make_pools(wl, layer, range(P), device=DEV)
    avg = wl.avg_bits[0]
    step = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, avg, device=DEV, n_pools=P)
    step.run(t["Q"], t["K"], t["V"])
    torch.cuda.synchronize()
    assert L.device_error() == 0
    wt = step.out["w_t"]
    np.testing.assert_allclose(wt.double().sum(dim=1).cpu().numpy(), wl.G * wl.W, rtol=1e-4)
    Hq, Hkv, N, d = wl.Hq, wl.Hkv, wl.N, wl.d
    wv, sv = wt.view(P, -1).clone(), step.sig_t.view(P, -1).clone()
    wk, sk = step.w_c.view(P, -1).clone(), step.sig_c.view(P, -1).clone()
    refs = {}
    for q in (0, P - 1):
        x = [f64(t[k][q * h:(q + 1) * h]) for k, h in (("Q", Hq), ("K", Hkv), ("V", Hkv))]
        ref = O.rdkv_compress(x[0], x[1], x[2], wl.q_pos0, avg)
        refs[q] = ref
        assert_lse_close(step.out["lse"][q * Hq:(q + 1) * Hq].cpu().numpy(), ref["scores"]["lse"])
        assert_scores_close(wt[q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["scores"]["w_t"], f"w_t pool {q}")
        np.testing.assert_allclose(step.w_c[q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["w_c"], rtol=TOL)
        np.testing.assert_allclose(step.sig_t[q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["sigma_t"], rtol=TOL)
        wv[q] = torch.from_numpy(ref["scores"]["w_t"].astype(np.float32).ravel())
        sv[q] = torch.from_numpy(ref["sigma_t"].ravel())
        wk[q] = torch.from_numpy(ref["w_c"].ravel())
        sk[q] = torch.from_numpy(ref["sigma_c"].ravel())
    bits_v = L.allocate_bits_pools(wv, sv, step.B_v)
    bits_k = L.allocate_bits_pools(wk, sk, step.B_k)
    X4 = (P, Hkv, N, d)
    vs = L.Streams(Hkv, N, d, 0, step.B_v, DEV, n_pools=P)
    L.quantize_pack_pools(t["V"].view(X4), 0, bits_v, None, vs)
    ks = L.Streams(Hkv, N, d, 1, step.B_k, DEV, n_pools=P)
    L.quantize_pack_pools(t["K"].view(X4), 1, bits_k, bits_v, ks)
    vh = L.dequantize_pools(vs, bits_v, None)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    for q, ref in refs.items():
        assert (bits_v[q].cpu().numpy() == ref["bits_v"]).all()
        assert (bits_k[q].cpu().numpy() == ref["bits_k"]).all()
        _cmp_streams(vs.pool(q), ref["v_streams"])
        _cmp_streams(ks.pool(q), ref["k_streams"])
        assert np.array_equal(vh[q].cpu().numpy(), O.dequantize(ref["v_streams"], (Hkv, N, d), 0, ref["bits_v"]))
    # the pools the oracle did not see: the pooled calls equal one-pool calls
    for q in (1, 7):
        assert torch.equal(bits_v[q], L.allocate_bits(wv[q], sv[q], step.B_v))
        one = L.Streams(Hkv, N, d, 0, step.B_v, DEV)
        L.quantize_pack(t["V"][q * Hkv:(q + 1) * Hkv], 0, bits_v[q], None, one)
        a, b = one.host_view(), vs.pool(q).host_view()
        for wd in (2, 4, 8, 16):
            assert np.array_equal(a[wd]["codes"], b[wd]["codes"]) and np.array_equal(a[wd]["ids"], b[wd]["ids"])
    assert L.device_error() == 0
