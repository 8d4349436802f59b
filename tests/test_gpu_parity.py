"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Scores and LSE: within the relative 2e-3 the method's accuracy target states
(fp32 accumulation of bf16 products); allocations, packed bytes and the
dequantised values: bit-exact when the GPU is fed the oracle's own weights.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_compression_flash_b300 import _lib as L
from kv_cache_compression_flash_b300 import synth
from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL = 2e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_scores_close(got, ref, what):
    """|g - o| <= 2e-3 * max(|o|, 1e-4 * max|o|) per element; 2e-3 on the vector norm."""
    got = np.asarray(got, dtype=np.float64)
    floor = 1e-4 * np.abs(ref).max()
    bad = np.abs(got - ref) > TOL * np.maximum(np.abs(ref), floor)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at " \
                          f"{np.unravel_index(np.argmax(np.abs(got - ref)), ref.shape)}"
    assert np.linalg.norm(got - ref) <= TOL * np.linalg.norm(ref) + 1e-30


def assert_lse_close(got, ref):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert (err <= TOL * np.maximum(1.0, np.abs(ref))).all(), f"lse worst error {err.max()}"


def rand_layer(Hq, Hkv, W, N, d, seed, scale=1.0, sinks=0):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(Hq, W, d, generator=g) * scale
    K = torch.randn(Hkv, N, d, generator=g) * scale
    V = torch.randn(Hkv, N, d, generator=g)
    if sinks:
        K[:, :sinks] *= 4
    return Q.bfloat16(), K.bfloat16(), V.bfloat16()


SCORE_SHAPES = [
    # Hq, Hkv, W, N, d
    (1, 1, 512, 512, 64),      # single head, every position a query
    (4, 2, 100, 300, 128),     # G=2, ragged key tail, ragged window
    (8, 2, 130, 700, 128),     # G=4, window not a multiple of the 32-row position block
    (4, 4, 1, 1, 64),          # one key, one query
    (2, 1, 1, 129, 128),       # one query row, a key tile plus one
    (16, 4, 200, 1000, 64),    # d=64, G=4
    (8, 1, 64, 2000, 128),     # G=8: two head chunks per group
    (2, 2, 257, 257, 128),     # full causal, G=1, 3 position blocks
]


@pytest.mark.parametrize("shape", SCORE_SHAPES)
def test_scores_rdkv_and_kvzip(shape):
    Hq, Hkv, W, N, d = shape
    Q, K, V = rand_layer(Hq, Hkv, W, N, d, seed=sum(shape), scale=1.5, sinks=2)
    q_pos0 = N - W
    ref = O.attention_scores(f64(Q), f64(K), q_pos0)
    out = L.score_attention(Q.to(DEV), K.to(DEV), q_pos0=q_pos0,
                            mode=L.MODE_LSE | L.MODE_RDKV_WT | L.MODE_KVZIP)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    assert_lse_close(out["lse"].cpu().numpy(), ref["lse"])
    assert_scores_close(out["w_t"].cpu().numpy(), ref["w_t"], "w_t")
    assert_scores_close(out["s_plus"].cpu().numpy(), ref["kvzip"], "kvzip")


@pytest.mark.parametrize("shape", [(4, 2, 100, 300, 128), (8, 2, 96, 96, 64), (4, 1, 70, 333, 128)])
def test_scores_kvzip_plus(shape):
    Hq, Hkv, W, N, d = shape
    D = 256
    Q, K, V = rand_layer(Hq, Hkv, W, N, d, seed=7 + sum(shape))
    g = torch.Generator().manual_seed(99)
    h = (torch.randn(W, D, generator=g) * torch.exp(0.5 * torch.randn(W, 1, generator=g))).bfloat16()
    WO = (torch.randn(D, Hq * d, generator=g) / math.sqrt(D)).bfloat16()
    ref = O.attention_scores(f64(Q), f64(K), N - W, V=f64(V), h=f64(h), W_O=f64(WO))
    out = L.score_attention(Q.to(DEV), K.to(DEV), mode=L.MODE_LSE | L.MODE_KVZIP_PLUS, V=V.to(DEV),
                            h=h.to(DEV), W_O=WO.to(DEV))
    torch.cuda.synchronize()
    assert L.device_error() == 0
    assert_lse_close(out["lse"].cpu().numpy(), ref["lse"])
    assert_scores_close(out["s_plus"].cpu().numpy(), ref["s_plus"], "s_plus")


def test_scores_deterministic():
    Q, K, _ = rand_layer(8, 2, 300, 3000, 128, seed=5)
    Qd, Kd = Q.to(DEV), K.to(DEV)
    a = L.score_attention(Qd, Kd)
    a = {k: v.clone() for k, v in a.items()}
    b = L.score_attention(Qd, Kd)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("shape", [(32, 8, 512, 8192, 128), (1, 1, 512, 512, 64), (8, 2, 130, 700, 128)])
def test_channel_weights_and_rms(shape):
    Hq, Hkv, W, N, d = shape
    Q, K, V = rand_layer(Hq, Hkv, W, N, d, seed=11)
    wc = L.channel_weights(Q.to(DEV), K.to(DEV))
    np.testing.assert_allclose(wc.cpu().numpy(), O.channel_weights(f64(Q), f64(K)), rtol=TOL)
    st = L.unit_rms(V.to(DEV), 0)
    np.testing.assert_allclose(st.cpu().numpy(), O.unit_rms(f64(V), 0), rtol=TOL)
    keep = torch.rand(Hkv, N, generator=torch.Generator().manual_seed(3)) > 0.6
    keep[0] = False
    sc = L.unit_rms(K.to(DEV), 1, keep_bits=keep.to(torch.uint8).reshape(-1).to(DEV))
    np.testing.assert_allclose(sc.cpu().numpy(), O.unit_rms(f64(K), 1, keep.numpy()), rtol=TOL, atol=0)
    # both channel quantities from one read of K: the same sums in the same order
    wc2, sc2 = L.channel_stats(Q.to(DEV), K.to(DEV), keep.to(torch.uint8).reshape(-1).to(DEV))
    assert torch.equal(wc2, wc) and torch.equal(sc2, sc)
    wc3, sc3 = L.channel_stats(Q.to(DEV), K.to(DEV), None)
    assert torch.equal(wc3, wc)
    np.testing.assert_allclose(sc3.cpu().numpy(), O.unit_rms(f64(K), 1), rtol=TOL)


def gpu_alloc(w, s, B, mask=L.WIDTHS_ALL):
    bits = L.allocate_bits(torch.from_numpy(w).to(DEV), torch.from_numpy(s).to(DEV), B, mask)
    torch.cuda.synchronize()
    return bits.cpu().numpy()


MASKS = {(0, 2, 4, 8, 16): L.WIDTHS_ALL, (0, 16): L.WIDTHS_KEEP_OR_EVICT, (0, 4, 16): (1 << 4) | (1 << 16),
         (0, 2, 8): (1 << 2) | (1 << 8)}


@pytest.mark.parametrize("U", [1, 3, 17, 1000, 70000])
@pytest.mark.parametrize("widths", list(MASKS))
def test_allocation_bit_exact(U, widths):
    rng = np.random.default_rng(U + len(widths))
    w = (rng.random(U) ** 3 * 10).astype(np.float32)
    s = (rng.random(U) + 0.05).astype(np.float32)
    w[rng.random(U) < 0.05] = 0                       # zero keys
    w[::11] = w[5 % U]                                # ties
    s[::11] = s[5 % U]
    for avg in (0.0, 0.3, 1.7, 3.0, 4.0, 9.5, 16.0, 20.0):
        B = int(math.floor(avg * U))
        ref = O.allocate_bits(w, s, B, widths)
        got = gpu_alloc(w, s, B, MASKS[widths])
        assert (got == ref).all(), (avg, np.nonzero(got != ref)[0][:10])
    assert L.device_error() == 0


def test_allocation_power_of_two_ties():
    """key_v = 4 key_u makes theta(u, 0) == theta(v, 1): ties across steps."""
    w = np.array([1, 4, 1, 4, 2, 8, 0.5, 16, 1, 4] * 30, dtype=np.float32)
    s = np.ones_like(w)
    for B in range(0, 16 * w.size + 1, 7):
        assert (gpu_alloc(w, s, B) == O.allocate_bits(w, s, B)).all(), B


@pytest.mark.parametrize("U", [5000, 50000, 400000])
def test_allocation_many_equal_keys(U):
    """Thousands of items share one threshold (more than a cluster CTA lists
    for its exact low-half pass), and pools past one cluster's shared memory
    (400 000 units) take the grid path."""
    rng = np.random.default_rng(U)
    w = np.ones(U, np.float32)
    w[rng.random(U) < 0.3] = 4.0                      # theta(u,0) of these == theta(v,1) of the ones
    w[rng.random(U) < 0.01] = 0.0
    s = np.ones(U, np.float32)
    for avg in (0.5, 2.0, 3.3, 7.9):
        B = int(math.floor(avg * U))
        assert (gpu_alloc(w, s, B) == O.allocate_bits(w, s, B)).all(), avg
    assert L.device_error() == 0


def test_allocation_rejects_bad_weights():
    w = np.ones(100, np.float32)
    w[7] = np.nan
    gpu_alloc(w, np.ones(100, np.float32), 300)
    assert L.device_error() == 3


def _cmp_streams(dev_streams, ref):
    got = dev_streams.host_view()
    for wd in (2, 4, 8, 16):
        assert (got[wd]["ids"] == ref[wd]["ids"]).all(), wd
        assert (got[wd]["group_offsets"] == ref[wd]["group_offsets"]).all(), wd
        assert got[wd]["n_groups"] == ref[wd]["n_groups"], wd
        assert np.array_equal(got[wd]["codes"], ref[wd]["codes"]), wd
        if wd != 16:
            assert np.array_equal(got[wd]["scales"], ref[wd]["scales"]), wd


@pytest.mark.parametrize("Hkv,N,d", [(2, 300, 128), (1, 64, 64), (3, 1000, 64), (8, 8192, 128)])
def test_pack_dequant_bit_exact(Hkv, N, d):
    rng = np.random.default_rng(N)
    g = torch.Generator().manual_seed(N)
    X = (torch.randn(Hkv, N, d, generator=g) * torch.exp(torch.randn(Hkv, N, 1, generator=g))).bfloat16()
    X[0, 0, :] = 0                                   # an all-zero group
    Xd = X.to(DEV)
    x64 = f64(X)
    # V: per token
    bits_v = rng.choice([0, 2, 4, 8, 16], size=Hkv * N).astype(np.uint8)
    B_v = int(bits_v.astype(int).sum())
    st = L.Streams(Hkv, N, d, 0, B_v, DEV)
    bv = torch.from_numpy(bits_v).to(DEV)
    L.quantize_pack(Xd, 0, bv, None, st)
    ref_v = O.quantize_pack(x64, 0, bits_v)
    _cmp_streams(st, ref_v)
    xh = L.dequantize(st, bv, None)
    assert np.array_equal(xh.cpu().numpy(), O.dequantize(ref_v, X.shape, 0, bits_v))
    # K: per channel over kept tokens
    keep = (bits_v > 0).reshape(Hkv, N)
    bits_k = rng.choice([0, 2, 4, 8, 16], size=Hkv * d).astype(np.uint8)
    B_k = int(bits_k.astype(int).sum())
    sk = L.Streams(Hkv, N, d, 1, B_k, DEV)
    bk = torch.from_numpy(bits_k).to(DEV)
    L.quantize_pack(Xd, 1, bk, bv, sk)
    ref_k = O.quantize_pack(x64, 1, bits_k, keep)
    _cmp_streams(sk, ref_k)
    kh = L.dequantize(sk, bk, bv)
    assert np.array_equal(kh.cpu().numpy(), O.dequantize(ref_k, X.shape, 1, bits_k, keep))
    assert L.device_error() == 0


QMAX = {2: 1, 4: 7, 8: 127, 16: 7}


def _tie_group(rng, w, n=64):
    """64 bf16-exact values whose group maximum is qmax * s with s a power of two,
    so that x / s lands exactly on half integers for about half of them (ties)."""
    qm = QMAX[w]
    s = 2.0 ** int(rng.integers(-6, 7))
    sign = rng.choice([-1.0, 1.0], size=n)
    tie = (rng.integers(0, qm, size=n) + 0.5) * s                    # (n + 1/2) s: 8 significant bits at most
    grid = 2 ** int(np.floor(np.log2(255 / qm)))                      # qmax * grid < 256: 8 bits
    other = np.floor(rng.random(n) * qm * grid) / grid * s           # on a fine grid below qmax s
    g = np.where(rng.random(n) < 0.5, tie, other) * sign
    g[rng.integers(0, n)] = qm * s * rng.choice([-1.0, 1.0])         # the group maximum
    return g


@pytest.mark.parametrize("d", [64, 128])
def test_pack_exact_ties_bit_exact(d):
    """Elements exactly halfway between two codes, at every width and on both axes:
    each must take the even code, as round-half-even of x / s does."""
    Hkv, N = 2, 640
    rng = np.random.default_rng(11 + d)
    # V (rows): every row of width w is made of tie groups for that width
    bits_v = rng.choice([2, 4, 8, 16], size=Hkv * N).astype(np.uint8)
    X = np.zeros((Hkv, N, d))
    for u in range(Hkv * N):
        for g0 in range(0, d, 64):
            X[u // N, u % N, g0:g0 + 64] = _tie_group(rng, int(bits_v[u]))
    Xt = torch.from_numpy(X).float().bfloat16()
    assert np.array_equal(f64(Xt), X)                                 # every value is bf16-exact
    st = L.Streams(Hkv, N, d, 0, int(bits_v.astype(int).sum()), DEV)
    bv = torch.from_numpy(bits_v).to(DEV)
    L.quantize_pack(Xt.to(DEV), 0, bv, None, st)
    ref_v = O.quantize_pack(X, 0, bits_v)
    _cmp_streams(st, ref_v)
    assert np.array_equal(L.dequantize(st, bv, None).cpu().numpy(), O.dequantize(ref_v, X.shape, 0, bits_v))
    # K (channels over the kept tokens; every token kept): each channel's 64-token groups are tie groups
    bits_k = rng.choice([2, 4, 8, 16], size=Hkv * d).astype(np.uint8)
    Y = np.zeros((Hkv, N, d))
    for h in range(Hkv):
        for c in range(d):
            for t0 in range(0, N, 64):
                Y[h, t0:t0 + 64, c] = _tie_group(rng, int(bits_k[h * d + c]), min(64, N - t0))
    Yt = torch.from_numpy(Y).float().bfloat16()
    assert np.array_equal(f64(Yt), Y)
    keep = np.ones((Hkv, N), dtype=bool)
    sk = L.Streams(Hkv, N, d, 1, int(bits_k.astype(int).sum()), DEV)
    bk = torch.from_numpy(bits_k).to(DEV)
    L.quantize_pack(Yt.to(DEV), 1, bk, bv, sk)
    ref_k = O.quantize_pack(Y, 1, bits_k, keep)
    _cmp_streams(sk, ref_k)
    assert np.array_equal(L.dequantize(sk, bk, bv).cpu().numpy(), O.dequantize(ref_k, Y.shape, 1, bits_k, keep))
    assert L.device_error() == 0


def test_pack_scale_overflow_is_reported():
    X = torch.zeros(1, 64, 64)
    X[0, 3, 5] = 2.0 ** 100
    st = L.Streams(1, 64, 64, 0, 64 * 8, DEV)
    L.quantize_pack(X.bfloat16().to(DEV), 0, torch.full((64,), 8, dtype=torch.uint8, device=DEV), None, st)
    assert L.device_error() == 3


@pytest.mark.parametrize("name", ["single_head_n512_d64", "llama3_8b_layer_n8192_w512"])
def test_pipeline_vs_oracle(name):
    """The whole RDKV pass on the synthetic workload: scores within tolerance;
    allocation and packing bit-exact when fed the oracle's weights."""
    wl = synth.WORKLOADS[name]
    t = synth.make_layer(wl)
    Q, K, V = (t[k].to(DEV) for k in ("Q", "K", "V"))
    avg = wl.avg_bits[0]
    step = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, avg, device=DEV)
    step.run(Q, K, V)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    x = {k: f64(t[k]) for k in ("Q", "K", "V")}
    ref = O.rdkv_compress(x["Q"], x["K"], x["V"], wl.q_pos0, avg)
    assert_lse_close(step.out["lse"].cpu().numpy(), ref["scores"]["lse"])
    assert_scores_close(step.out["w_t"].cpu().numpy(), ref["scores"]["w_t"], "w_t")
    np.testing.assert_allclose(step.w_c.cpu().numpy(), ref["w_c"], rtol=TOL)
    np.testing.assert_allclose(step.sig_t.cpu().numpy(), ref["sigma_t"], rtol=TOL)
    # stage 2/3 fed the oracle's weights
    bits_v = gpu_alloc(ref["scores"]["w_t"].astype(np.float32).ravel(), ref["sigma_t"].ravel(), step.B_v)
    assert (bits_v == ref["bits_v"]).all()
    bits_k = gpu_alloc(ref["w_c"].ravel(), ref["sigma_c"].ravel(), step.B_k)
    assert (bits_k == ref["bits_k"]).all()
    bv, bk = torch.from_numpy(bits_v).to(DEV), torch.from_numpy(bits_k).to(DEV)
    sv = L.Streams(wl.Hkv, wl.N, wl.d, 0, step.B_v, DEV)
    L.quantize_pack(V, 0, bv, None, sv)
    _cmp_streams(sv, ref["v_streams"])
    sk = L.Streams(wl.Hkv, wl.N, wl.d, 1, step.B_k, DEV)
    L.quantize_pack(K, 1, bk, bv, sk)
    _cmp_streams(sk, ref["k_streams"])
    # sigma_c on the oracle's kept set
    sc = L.unit_rms(K, 1, keep_bits=bv)
    np.testing.assert_allclose(sc.cpu().numpy(), ref["sigma_c"], rtol=TOL)
    assert L.device_error() == 0


@pytest.mark.parametrize("Hkv,N", [(1, 1), (2, 7), (8, 8192), (3, 1001)])
def test_threshold_keep_bit_exact(Hkv, N):
    """KVzap threshold + sliding window   [KVzap §2.3], against the oracle."""
    rng = np.random.default_rng(N)
    s = (rng.random((Hkv, N)) ** 3).astype(np.float32)
    s[:, ::5] = np.float32(0.125)                      # ties at tau
    for tau, window, kw in ((0.125, 128, 16), (0.5, 0, 8), (0.0, 3, 2), (2.0, N + 5, 4)):
        got = L.threshold_keep(torch.from_numpy(s).to(DEV), tau, window, kw).cpu().numpy()
        assert np.array_equal(got, O.threshold_keep(s, tau, window, kw)), (tau, window, kw)
    assert L.device_error() == 0
    s[0, 0] = np.nan
    got = L.threshold_keep(torch.from_numpy(s).to(DEV), 0.1, 0, 16).cpu().numpy()
    assert np.array_equal(got, O.threshold_keep(s, 0.1, 0, 16))
    assert L.device_error() == 3


def test_one_graph_step_matches_the_eager_step():
    """The bench's one-graph replay of the whole step gives the eager step's results."""
    wl = synth.WORKLOADS["llama3_8b_layer_n8192_w512"]
    t = synth.make_layer(wl)
    Q, K, V = (t[k].to(DEV) for k in ("Q", "K", "V"))
    a = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, 3, device=DEV)
    a.run(Q, K, V)
    b = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, 3, device=DEV)
    b.capture(Q, K, V)
    b.replay_step()
    torch.cuda.synchronize()
    assert L.device_error() == 0
    assert torch.equal(a.sig_t, b.sig_t) and torch.equal(a.bits_v, b.bits_v) and torch.equal(a.bits_k, b.bits_k)
    assert torch.equal(a.v_hat, b.v_hat) and torch.equal(a.k_hat, b.k_hat)
    assert torch.equal(a.out["w_t"], b.out["w_t"])


def test_scores_kvzip_plus_split_merge():
    """KVzip+ with pass 2 split over several CTAs per key tile: the column max of
    a_{r,t} |h_r| is merged across the splits, and the 1 / |W_O^h v_t| factor
    is applied after it   [KVzap §2.1, KVzip+]."""
    Hq, Hkv, W, N, d, D = 8, 2, 700, 700, 128, 256
    mode = L.MODE_LSE | L.MODE_KVZIP_PLUS
    assert L.score_plan_info(Hq, Hkv, W, N, d, D=D, q_pos0=0, mode=mode)[3] > 1   # the merge runs
    Q, K, V = rand_layer(Hq, Hkv, W, N, d, seed=4242, scale=1.4, sinks=3)
    g = torch.Generator().manual_seed(4243)
    h = (torch.randn(W, D, generator=g) * torch.exp(0.5 * torch.randn(W, 1, generator=g))).bfloat16()
    WO = (torch.randn(D, Hq * d, generator=g) / math.sqrt(D)).bfloat16()
    ref = O.attention_scores(f64(Q), f64(K), 0, V=f64(V), h=f64(h), W_O=f64(WO))
    out = L.score_attention(Q.to(DEV), K.to(DEV), q_pos0=0, mode=mode, V=V.to(DEV), h=h.to(DEV), W_O=WO.to(DEV))
    torch.cuda.synchronize()
    assert L.device_error() == 0
    assert_lse_close(out["lse"].cpu().numpy(), ref["lse"])
    assert_scores_close(out["s_plus"].cpu().numpy(), ref["s_plus"], "s_plus")


# ---------------------------------------------------------------------------
# pooled calls: several (layer, sequence) pools of one shape in one call
# ---------------------------------------------------------------------------
def _pooled_inputs(P, Hq, Hkv, W, N, d, seed):
    parts = [rand_layer(Hq, Hkv, W, N, d, seed=seed + 31 * q, scale=1.3, sinks=2) for q in range(P)]
    return tuple(torch.cat([p[i] for p in parts]).contiguous() for i in range(3))


@pytest.mark.parametrize("P,Hq,Hkv,W,N,d", [(3, 8, 2, 130, 700, 128), (2, 4, 4, 64, 300, 64),
                                            (4, 32, 8, 96, 1000, 128)])
def test_pooled_step_vs_oracle(P, Hq, Hkv, W, N, d):
    """n_pools pools through one pooled step: every pool's scores match the
    oracle on that pool alone; pooled allocation, packing and dequantisation
    fed the oracle's weights and widths are bit-exact per pool."""
    Q, K, V = _pooled_inputs(P, Hq, Hkv, W, N, d, seed=P * 1000 + N)
    avg = 3
    step = RdkvLayerStep(Hq, Hkv, N, W, d, avg, device=DEV, n_pools=P)
    step.run(Q.to(DEV), K.to(DEV), V.to(DEV))
    torch.cuda.synchronize()
    assert L.device_error() == 0
    q_pos0 = N - W
    refs = []
    for q in range(P):
        x = [f64(t[q * h:(q + 1) * h]) for t, h in ((Q, Hq), (K, Hkv), (V, Hkv))]
        ref = O.rdkv_compress(x[0], x[1], x[2], q_pos0, avg)
        refs.append(ref)
        assert_lse_close(step.out["lse"][q * Hq:(q + 1) * Hq].cpu().numpy(), ref["scores"]["lse"])
        assert_scores_close(step.out["w_t"][q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["scores"]["w_t"], f"w_t {q}")
        np.testing.assert_allclose(step.w_c[q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["w_c"], rtol=TOL)
        np.testing.assert_allclose(step.sig_t[q * Hkv:(q + 1) * Hkv].cpu().numpy(), ref["sigma_t"], rtol=TOL)
    # stage 2 and 3 on the oracle's weights, all pools in one call
    wv = torch.from_numpy(np.stack([r["scores"]["w_t"].astype(np.float32).ravel() for r in refs])).to(DEV)
    sv = torch.from_numpy(np.stack([r["sigma_t"].ravel() for r in refs])).to(DEV)
    bits_v = L.allocate_bits_pools(wv, sv, step.B_v)
    wk = torch.from_numpy(np.stack([r["w_c"].ravel() for r in refs])).to(DEV)
    sk = torch.from_numpy(np.stack([r["sigma_c"].ravel() for r in refs])).to(DEV)
    bits_k = L.allocate_bits_pools(wk, sk, step.B_k)
    torch.cuda.synchronize()
    for q, r in enumerate(refs):
        assert (bits_v[q].cpu().numpy() == r["bits_v"]).all(), q
        assert (bits_k[q].cpu().numpy() == r["bits_k"]).all(), q
    Vd, Kd = V.to(DEV).view(P, Hkv, N, d), K.to(DEV).view(P, Hkv, N, d)
    vs = L.Streams(Hkv, N, d, 0, step.B_v, DEV, n_pools=P)
    L.quantize_pack_pools(Vd, 0, bits_v, None, vs)
    ks = L.Streams(Hkv, N, d, 1, step.B_k, DEV, n_pools=P)
    L.quantize_pack_pools(Kd, 1, bits_k, bits_v, ks)
    vh = L.dequantize_pools(vs, bits_v, None)
    kh = L.dequantize_pools(ks, bits_k, bits_v)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    for q, r in enumerate(refs):
        _cmp_streams(vs.pool(q), r["v_streams"])
        _cmp_streams(ks.pool(q), r["k_streams"])
        assert np.array_equal(vh[q].cpu().numpy(), O.dequantize(r["v_streams"], (Hkv, N, d), 0, r["bits_v"]))
        assert np.array_equal(kh[q].cpu().numpy(),
                              O.dequantize(r["k_streams"], (Hkv, N, d), 1, r["bits_k"], r["keep"]))
        # a pool's view reads back through the one-pool call too
        assert np.array_equal(L.dequantize(vs.pool(q), bits_v[q], None).cpu().numpy(), vh[q].cpu().numpy())


@pytest.mark.parametrize("U,P", [(1000, 5), (70000, 3), (400000, 2), (131072, 4), (131072, 16)])
def test_pooled_allocation_matches_single_calls(U, P):
    """allocate_bits_pools equals one allocate_bits call per pool: on the
    cluster path (1000, 70 000 units), and on the side-by-side cooperative grid
    with the thetas cached (400 000 x 2, 131 072 x 4) and recomputed in every
    pass (131 072 x 16: too many blocks for every pool's cache at once)."""
    rng = np.random.default_rng(U + P)
    w = (rng.random((P, U)) ** 3 * 10).astype(np.float32)
    s = (rng.random((P, U)) + 0.05).astype(np.float32)
    w[rng.random((P, U)) < 0.05] = 0
    w[:, ::11] = w[:, 5:6]
    wd, sd = torch.from_numpy(w).to(DEV), torch.from_numpy(s).to(DEV)
    for avg in (0.7, 3.0):
        B = int(math.floor(avg * U))
        got = L.allocate_bits_pools(wd, sd, B)
        for q in range(P):
            assert torch.equal(got[q], L.allocate_bits(wd[q], sd[q], B)), (avg, q)
    # with only one pool's workspace the pools run one after the other, with the same widths
    lib = L.lib()
    small = torch.empty(lib.kvs_allocate_workspace_size(U), dtype=torch.uint8, device=DEV)
    seq = torch.empty(P, U, dtype=torch.uint8, device=DEV)
    B = int(math.floor(2.5 * U))
    rc = lib.kvs_allocate_bits_pools(L._ptr(wd), L._ptr(sd), P, U, B, L.WIDTHS_ALL, L._ptr(seq), L._ptr(small),
                                     small.numel(), L._stream(None))
    assert rc == 0
    assert torch.equal(seq, L.allocate_bits_pools(wd, sd, B))
    assert L.device_error() == 0
