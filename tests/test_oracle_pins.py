"""Pins of the CPU oracle to facts the papers and the mathematics fix.

None of these re-types the oracle's own formula: each compares it with a closed
form, an invariant, a brute-force pure-Python evaluation on tiny inputs, a
different decomposition (SVD, exhaustive search) or a hand-worked example.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    import torch
    return torch.tensor(np.asarray(a, dtype=np.float32)).bfloat16().float().numpy().astype(np.float64)


# ---------------------------------------------------------------- scores ----
@pytest.mark.parametrize("Hq,Hkv,W,N,d", [(4, 2, 7, 19, 16), (1, 1, 5, 5, 8), (8, 2, 33, 40, 32)])
def test_token_weight_mass_equals_rows(Hq, Hkv, W, N, d):
    """Each softmax row sums to one, so sum_t w_t[g] = G * W   [RDKV §2.1]."""
    rng = np.random.default_rng(1)
    Q = rng.standard_normal((Hq, W, d)) * 2
    K = rng.standard_normal((Hkv, N, d)) * 2
    sc = O.attention_scores(Q, K, N - W)
    np.testing.assert_allclose(sc["w_t"].sum(axis=1), (Hq // Hkv) * W, rtol=1e-12)


@pytest.mark.parametrize("q_pos0", [0, 3, 10])
def test_constant_keys_harmonic_closed_form(q_pos0):
    """Equal keys give a_{r,t} = 1/(p_r+1) for t <= p_r, hence
    w_t = G * sum_{r: p_r >= t} 1/(p_r+1) and lse_r = q_r.k/sqrt(d) + ln(p_r+1)."""
    rng = np.random.default_rng(2)
    Hq, Hkv, W, N, d = 6, 2, 5, 16, 8
    N = max(N, q_pos0 + W)
    Q = rng.standard_normal((Hq, W, d))
    k = rng.standard_normal(d)
    K = np.broadcast_to(k, (Hkv, N, d)).copy()
    sc = O.attention_scores(Q, K, q_pos0)
    G = Hq // Hkv
    pos = q_pos0 + np.arange(W)
    for t in range(N):
        expect = G * sum(1.0 / (p + 1) for p in pos if p >= t)
        np.testing.assert_allclose(sc["w_t"][:, t], expect, rtol=1e-12, atol=1e-15)
    lse_expect = Q @ k / math.sqrt(d) + np.log(pos + 1)[None, :]
    np.testing.assert_allclose(sc["lse"], lse_expect, rtol=1e-12)
    # KVzip: every visible column max is the largest 1/(p+1) among rows that see t
    for t in range(N):
        seen = [1.0 / (p + 1) for p in pos if p >= t]
        np.testing.assert_allclose(sc["kvzip"][:, t], max(seen) if seen else 0.0, rtol=1e-12)


def test_single_key():
    """N = 1: every row puts all its mass on key 0; lse equals the logit."""
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((4, 3, 8))
    K = rng.standard_normal((2, 1, 8))
    sc = O.attention_scores(Q, K, 0)
    np.testing.assert_allclose(sc["w_t"], 2 * 3, rtol=1e-14)
    s = np.stack([Q[h] @ K[h // 2, 0] for h in range(4)]) / math.sqrt(8)
    np.testing.assert_allclose(sc["lse"], s, rtol=1e-13)


def _brute_scores(Q, K, V, h, WO, q_pos0):
    """Pure-Python loops, straight from the definitions."""
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    G = Hq // Hkv
    D = h.shape[1]
    lse = [[0.0] * W for _ in range(Hq)]
    wt = [[0.0] * N for _ in range(Hkv)]
    kz = [[0.0] * N for _ in range(Hkv)]
    sp = [[0.0] * N for _ in range(Hkv)]
    hn = [math.sqrt(math.fsum(float(h[r, i]) ** 2 for i in range(D))) for r in range(W)]
    for hd in range(Hq):
        g = hd // G
        vn = []
        for t in range(N):
            acc = []
            for i in range(D):
                acc.append(math.fsum(float(WO[i, hd * d + c]) * float(V[g, t, c]) for c in range(d)) ** 2)
            vn.append(math.sqrt(math.fsum(acc)))
        for r in range(W):
            p = q_pos0 + r
            logits = {t: math.fsum(float(Q[hd, r, c]) * float(K[g, t, c]) for c in range(d)) / math.sqrt(d)
                      for t in range(N) if t <= p}
            mx = max(logits.values())
            l = mx + math.log(math.fsum(math.exp(s - mx) for s in logits.values()))
            lse[hd][r] = l
            for t, s in logits.items():
                a = math.exp(s - l)
                wt[g][t] += a
                kz[g][t] = max(kz[g][t], a)
                sp[g][t] = max(sp[g][t], a / (vn[t] / hn[r]))
    return np.array(lse), np.array(wt), np.array(kz), np.array(sp)


@pytest.mark.parametrize("q_pos0,W,N", [(2, 4, 6), (0, 5, 5), (4, 3, 9)])
def test_scores_brute_force(q_pos0, W, N):
    """LSE [KVSculpt §2], w_t [RDKV §2.1], KVzip and KVzip+ [KVzap §2.1] by brute force."""
    rng = np.random.default_rng(4 + W)
    Hq, Hkv, d, D = 4, 2, 4, 3
    Q = rng.standard_normal((Hq, W, d)) * 1.5
    K = rng.standard_normal((Hkv, N, d)) * 1.5
    V = rng.standard_normal((Hkv, N, d))
    h = rng.standard_normal((W, D)) * np.exp(rng.standard_normal((W, 1)))
    WO = rng.standard_normal((D, Hq * d))
    sc = O.attention_scores(Q, K, q_pos0, V=V, h=h, W_O=WO)
    lse, wt, kz, sp = _brute_scores(Q, K, V, h, WO, q_pos0)
    np.testing.assert_allclose(sc["lse"], lse, rtol=1e-12)
    np.testing.assert_allclose(sc["w_t"], wt, rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(sc["kvzip"], kz, rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(sc["s_plus"], sp, rtol=1e-11, atol=1e-15)


def test_row_chunking_is_invisible():
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((4, 37, 16))
    K = rng.standard_normal((2, 50, 16))
    a = O.attention_scores(Q, K, 13, row_chunk=7)
    b = O.attention_scores(Q, K, 13, row_chunk=1000)
    for k in ("lse", "w_t", "kvzip"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-13)


# ------------------------------------------------------- channel weights ----
def test_channel_weight_is_spectral_norm_of_logit_change():
    """w_c is the spectral norm of the logit deviation when channel c is zeroed
    [RDKV §2.1]; the deviation is a rank-one outer product, so the bound is tight."""
    rng = np.random.default_rng(6)
    Hq, Hkv, W, N, d = 4, 2, 6, 11, 8
    Q = rng.standard_normal((Hq, W, d))
    K = rng.standard_normal((Hkv, N, d))
    wc = O.channel_weights(Q, K)
    G = Hq // Hkv
    for g in range(Hkv):
        Qg = Q[g * G:(g + 1) * G].reshape(G * W, d)
        S = Qg @ K[g].T / math.sqrt(d)
        for c in range(d):
            Kz = K[g].copy()
            Kz[:, c] = 0
            dS = S - Qg @ Kz.T / math.sqrt(d)
            np.testing.assert_allclose(wc[g, c], np.linalg.norm(dS, 2), rtol=1e-10)


# --------------------------------------------------------------- sigma -----
def test_unit_rms_brute_force():
    rng = np.random.default_rng(7)
    X = rng.standard_normal((2, 9, 4))
    keep = rng.random((2, 9)) > 0.4
    keep[1] = False
    s0 = O.unit_rms(X, 0)
    s1 = O.unit_rms(X, 1, keep)
    for g in range(2):
        for t in range(9):
            assert math.isclose(s0[g, t], math.sqrt(math.fsum(X[g, t, c] ** 2 for c in range(4)) / 4), rel_tol=1e-13)
        for c in range(4):
            ts = [t for t in range(9) if keep[g, t]]
            e = math.sqrt(math.fsum(X[g, t, c] ** 2 for t in ts) / len(ts)) if ts else 0.0
            assert math.isclose(s1[g, c], e, rel_tol=1e-13, abs_tol=0.0)


# ---------------------------------------------------------- allocation -----
def test_allocation_hand_examples():
    gold = json.load(open(os.path.join(GOLD, "alloc_hand_examples.json")))
    for case in gold["cases"]:
        got = O.allocate_bits(case["w"], case["sigma"], case["budget"])
        assert got.tolist() == case["bits"], case["why"]


def test_chord_slopes_exact():
    assert O.chord_slopes((0, 2, 4, 8, 16)) == [3 / 8, 3 / 32, 15 / 1024, 255 / 524288]
    assert O.chord_slopes((0, 16)) == [65535 / 1048576]


def _exhaustive(key, widths, B):
    best = None
    for combo in itertools.product(widths, repeat=len(key)):
        if sum(combo) <= B:
            D = sum(k * 2.0 ** (-b) for k, b in zip(key, combo))
            if best is None or D < best[0]:
                best = (D, combo)
    return best


@pytest.mark.parametrize("U", [1, 3, 5, 7])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_allocation_vs_exhaustive(U, seed):
    """Everett: the Lagrangian prefix is optimal at its own rate; the final
    allocation fits B and sits between the exhaustive optimum and the prefix."""
    rng = np.random.default_rng(100 * U + seed)
    w = (rng.random(U) * rng.choice([1, 10, 100], U)).astype(np.float32)
    s = rng.random(U).astype(np.float32) + np.float32(0.1)
    key = (w.astype(np.float64) * s.astype(np.float64)).tolist()
    widths = (0, 2, 4, 8, 16)
    for B in range(0, 16 * U + 3, max(1, U)):
        bits = O.allocate_bits(w, s, B)
        assert int(bits.astype(int).sum()) <= B
        D_final = O.distortion(w, s, bits)
        D_opt, _ = _exhaustive(key, widths, B)
        assert D_final >= D_opt * (1 - 1e-12)
        # the prefix alone: recompute with the fix pass disabled by a budget equal to its own rate
        c = O.chord_slopes(widths)
        items = sorted(((-ck * k, u, j, widths[j + 1] - widths[j])
                        for u, k in enumerate(key) for j, ck in enumerate(c) if ck * k > 0))
        used, lvl = 0, [0] * U
        for _, u, j, cost in items:
            if used + cost > B:
                break
            used += cost
            lvl[u] += 1
        prefix_bits = [widths[l] for l in lvl]
        D_prefix = sum(k * 2.0 ** (-b) for k, b in zip(key, prefix_bits))
        assert D_final <= D_prefix * (1 + 1e-12)
        D_at_rate, _ = _exhaustive(key, widths, used)
        assert math.isclose(D_prefix, D_at_rate, rel_tol=1e-12), (B, prefix_bits)


def test_allocation_extremes():
    rng = np.random.default_rng(8)
    w = rng.random(50).astype(np.float32)
    s = rng.random(50).astype(np.float32) + np.float32(0.01)
    assert (O.allocate_bits(w, s, 0) == 0).all()
    assert (O.allocate_bits(w, s, 16 * 50) == 16).all()
    assert (O.allocate_bits(w, s, 10 ** 9) == 16).all()


def test_allocation_two_widths_is_topk():
    """Widths {0,16}: keep the top-k keys (ties by lower index), k = floor(B/16)."""
    rng = np.random.default_rng(9)
    U = 300
    w = rng.random(U).astype(np.float32)
    w[::7] = w[3]                                     # plenty of ties
    s = np.ones(U, dtype=np.float32)
    for k in (0, 1, 17, 150, 299, 300):
        bits = O.allocate_bits(w, s, 16 * k, widths=(0, 16))
        key = w.astype(np.float64)
        order = sorted(range(U), key=lambda u: (-key[u], u))
        expect = np.zeros(U, dtype=np.uint8)
        expect[order[:k]] = 16
        assert (bits == expect).all()


# --------------------------------------------------------- quantisation ----
def test_quant_hand_examples():
    gold = json.load(open(os.path.join(GOLD, "quant_hand_examples.json")))
    for case in gold["cases"]:
        wd = case["width"]
        x = np.zeros(64)
        x[:len(case["x"])] = case["x"]
        X = x.reshape(1, 1, 64)
        st = O.quantize_pack(X, 0, np.array([wd], np.uint8))[wd]
        expect = np.zeros(case["n_bytes"], np.uint8)
        for k, v in case["bytes_nonzero"].items():
            expect[int(k)] = v
        assert st["codes"].tolist() == expect.tolist(), case["why"]
        if case["scale_bits"] is not None:
            assert st["scales"].tolist() == [case["scale_bits"]], case["why"]
        xh = O.dequantize({w: (st if w == wd else {"ids": np.zeros(0, np.int32)}) for w in (2, 4, 8, 16)},
                          (1, 1, 64), 0, np.array([wd], np.uint8))
        np.testing.assert_array_equal(xh[0, 0, :len(case["x_hat"])], np.float32(case["x_hat"]))


def _unpack_bitloop(blk, wd):
    """Independent unpack: walk the bits one at a time."""
    vals = []
    for e in range(64):
        code = 0
        for b in range(wd):
            bit_index = wd * e + b
            code |= ((int(blk[bit_index // 8]) >> (bit_index % 8)) & 1) << b
        vals.append(code - (1 << wd) if code >= 1 << (wd - 1) else code)
    return vals


@pytest.mark.parametrize("wd", [2, 4, 8])
def test_quant_bounds_and_bit_layout(wd):
    rng = np.random.default_rng(10 + wd)
    X = _bf16(rng.standard_normal((2, 5, 128)) * np.exp(rng.standard_normal((2, 5, 1)) * 3))
    bits = np.full(10, wd, np.uint8)
    st = O.quantize_pack(X, 0, bits)
    qmax = 2 ** (wd - 1) - 1
    s = st[wd]["scales"].view(np.float16).astype(np.float64)
    groups = X.reshape(-1, 64)
    a = np.abs(groups).max(axis=1)
    assert (s * qmax >= a).all()                                              # s >= a/qmax
    prev = np.nextafter(s.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
    assert (prev * qmax < a).all()                                            # s minimal
    for gi in range(groups.shape[0]):
        blk = st[wd]["codes"][gi * 8 * wd:(gi + 1) * 8 * wd]
        q = np.array(_unpack_bitloop(blk, wd))
        assert np.abs(q).max() <= qmax
        xh = q * s[gi]
        assert (np.abs(groups[gi] - xh) <= s[gi] / 2).all()                  # |x - x_hat| <= s/2
    xh = O.dequantize(st, X.shape, 0, bits)
    assert (np.abs(X - xh) <= np.repeat(s, 64).reshape(X.shape) / 2).all()


def test_pack_axis1_kept_tokens_and_padding():
    rng = np.random.default_rng(11)
    X = _bf16(rng.standard_normal((2, 150, 64)))
    keep = rng.random((2, 150)) > 0.3
    bits = rng.choice([0, 2, 4, 8, 16], size=2 * 64).astype(np.uint8)
    st = O.quantize_pack(X, 1, bits, keep)
    xh = O.dequantize(st, X.shape, 1, bits, keep)
    for g in range(2):
        tk = np.nonzero(keep[g])[0]
        ng = -(-tk.size // 64)
        for c in range(64):
            b = int(bits[g * 64 + c])
            col = xh[g, :, c]
            assert (col[~keep[g]] == 0).all()
            if b == 0:
                assert (col == 0).all()
            elif b == 16:
                np.testing.assert_array_equal(col[tk], X[g, tk, c].astype(np.float32))
            else:
                j = list(st[b]["ids"]).index(g * 64 + c)
                g0 = st[b]["group_offsets"][j]
                s = st[b]["scales"][g0:g0 + ng].view(np.float16).astype(np.float64)
                err = np.abs(col[tk] - X[g, tk, c])
                assert (err <= np.repeat(s, 64)[:tk.size] / 2).all()
                last = st[b]["codes"][(g0 + ng - 1) * 8 * b:(g0 + ng) * 8 * b]
                q = _unpack_bitloop(last, b)
                assert all(v == 0 for v in q[tk.size - (ng - 1) * 64:])       # padding codes are 0


def test_zero_group_and_overflow():
    X = np.zeros((1, 1, 64))
    st = O.quantize_pack(X, 0, np.array([4], np.uint8))
    assert st[4]["scales"].tolist() == [0] and not st[4]["codes"].any()
    Y = np.zeros((1, 1, 64))
    Y[0, 0, 0] = 2.0 ** 100                                                   # bf16-exact, beyond fp16 range
    with pytest.raises(OverflowError):
        O.quantize_pack(Y, 0, np.array([8], np.uint8))


# ----------------------------------------------------------------------------
# threshold pruning with a sliding window   [KVzap §2.3]
# ----------------------------------------------------------------------------
def test_threshold_hand_examples(root):
    import json
    cases = json.load(open(os.path.join(root, "tests", "golden", "threshold_hand_examples.json")))["cases"]
    for c in cases:
        got = O.threshold_keep(np.array(c["score"], np.float32), c["tau"], c["window"], c["keep_width"])
        assert got.tolist() == c["bits"], c["why"]


def test_threshold_special_cases():
    rng = np.random.default_rng(3)
    s = rng.random((3, 50)).astype(np.float32)
    assert (O.threshold_keep(s, 2.0, 50) == 16).all()                    # the window covers every token
    assert (O.threshold_keep(s, -np.inf, 0) == 16).all()                 # every finite score passes
    b = O.threshold_keep(s, np.inf, 7)
    assert (b[:, -7:] == 16).all() and (b[:, :-7] == 0).all()            # only the window
    s[0, 3] = np.nan
    assert O.threshold_keep(s, 0.0, 0)[0, 3] == 0                        # NaN never passes
    kept = [int((O.threshold_keep(s, t, 5) > 0).sum()) for t in (0.1, 0.3, 0.6, 0.9)]
    assert kept == sorted(kept, reverse=True)                            # monotone in tau


# ----------------------------------------------------------------------------
# decode attention over the TriZone streams   [RDKV §2.3]
# ----------------------------------------------------------------------------
def _lse_value(s):
    return {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "-inf": -math.inf}[s]


def test_trizone_hand_examples():
    ex = json.load(open(os.path.join(GOLD, "trizone_hand_examples.json")))["examples"]
    for e in ex:
        kn = None if e["k_new"] is None else np.array(e["k_new"], float)
        vn = None if e["v_new"] is None else np.array(e["v_new"], float)
        out, lse = O.trizone_decode(np.array(e["q"], float), np.array(e["K_hat"], float),
                                    np.array(e["V_hat"], float), np.array(e["keep"], bool), kn, vn)
        np.testing.assert_allclose(out, np.array(e["out"], float), rtol=0, atol=1e-13, err_msg=e["name"])
        want = np.array([_lse_value(s) for s in e["lse"]])
        np.testing.assert_array_equal(np.isinf(lse), np.isinf(want))
        fin = np.isfinite(want)
        np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-13, err_msg=e["name"])


def _trizone_case(rng, Hq=4, Hkv=2, N=37, d=8, Nc=3):
    q = rng.standard_normal((Hq, d))
    K = rng.standard_normal((Hkv, N, d))
    V = rng.standard_normal((Hkv, N, d))
    keep = rng.random((Hkv, N)) > 0.4
    kn = rng.standard_normal((Hkv, Nc, d))
    vn = rng.standard_normal((Hkv, Nc, d))
    return q, K, V, keep, kn, vn


def test_trizone_single_visible_token_and_equal_logits():
    rng = np.random.default_rng(21)
    q, K, V, keep, kn, vn = _trizone_case(rng)
    keep1 = np.zeros_like(keep)
    keep1[:, 5] = True
    out, lse = O.trizone_decode(q, K, V, keep1)
    for hd in range(4):
        g = hd // 2
        np.testing.assert_array_equal(out[hd], V[g, 5])                    # softmax of one logit is 1
        assert abs(lse[hd] - K[g, 5] @ q[hd] / math.sqrt(8)) < 1e-13
    out, lse = O.trizone_decode(np.zeros_like(q), K, V, keep, kn, vn)       # every logit 0: the mean
    for hd in range(4):
        g = hd // 2
        rows = np.concatenate([V[g, keep[g]], vn[g]])
        np.testing.assert_allclose(out[hd], rows.mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[hd] - math.log(rows.shape[0])) < 1e-13


def test_trizone_evicted_tokens_have_no_effect():
    rng = np.random.default_rng(22)
    q, K, V, keep, kn, vn = _trizone_case(rng)
    base = O.trizone_decode(q, K, V, keep, kn, vn)
    K2, V2 = K.copy(), V.copy()
    K2[~keep] = 1e3 * np.sign(q[0]).reshape(1, -1)                         # would dominate if visible
    V2[~keep] = 7e5
    got = O.trizone_decode(q, K2, V2, keep, kn, vn)
    np.testing.assert_array_equal(got[0], base[0])
    np.testing.assert_array_equal(got[1], base[1])


def test_trizone_two_part_merge_and_permutation():
    """Attention over A u B equals the log-sum-exp merge of attention over A and
    over B (the split a decode kernel relies on), and a permutation of the old
    tokens changes nothing."""
    rng = np.random.default_rng(23)
    q, K, V, keep, kn, vn = _trizone_case(rng, N=60, Nc=5)
    out, lse = O.trizone_decode(q, K, V, keep, kn, vn)
    oa, la = O.trizone_decode(q, K, V, keep)                               # old tokens only
    ob, lb = O.trizone_decode(q, K, V, np.zeros_like(keep), kn, vn)        # new tokens only
    m = np.maximum(la, lb)
    wa, wb = np.exp(la - m), np.exp(lb - m)
    np.testing.assert_allclose(lse, m + np.log(wa + wb), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, (wa[:, None] * oa + wb[:, None] * ob) / (wa + wb)[:, None], rtol=0, atol=1e-12)
    perm = rng.permutation(60)
    op, lp = O.trizone_decode(q, K[:, perm], V[:, perm], keep[:, perm], kn, vn)
    np.testing.assert_allclose(op, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, lse, rtol=0, atol=1e-12)


def test_trizone_gqa_head_mapping():
    """Query head h reads KV head h // G: with constant V rows per KV head the
    output of head h is that constant."""
    rng = np.random.default_rng(24)
    q, K, V, keep, kn, vn = _trizone_case(rng, Hq=6, Hkv=3)
    for g in range(3):
        V[g] = g + 1.0
        vn[g] = g + 1.0
    out, _ = O.trizone_decode(q, K, V, keep, kn, vn)
    for hd in range(6):
        np.testing.assert_allclose(out[hd], hd // 2 + 1.0, rtol=1e-14)


def test_channels_over_no_kept_token_have_no_groups():
    """Axis 1 with every token evicted: each channel unit holds zero elements,
    so it is listed with no groups and dequantises to zeros."""
    X = np.ones((2, 5, 64))
    keep = np.zeros((2, 5), bool)
    bits = np.array([2, 4, 8, 16] * 32, np.uint8)
    st = O.quantize_pack(X, 1, bits, keep)
    for wd in (2, 4, 8, 16):
        assert st[wd]["n_groups"] == 0 and st[wd]["codes"].size == 0
        assert st[wd]["ids"].size == 32 and (st[wd]["group_offsets"] == 0).all()
    assert not O.dequantize(st, X.shape, 1, bits, keep).any()


# ----------------------------------------------------------------------------
# KV-CoRE: Gram accumulation, spectrum, NER, Eckart-Young error   [KV-CoRE §2]
# ----------------------------------------------------------------------------
def test_gram_blocks_trace_and_svd():
    rng = np.random.default_rng(31)
    X = rng.standard_normal((2, 40, 6)) * np.array([3, 1, 0.5, 0.1, 2, 1])
    keep = rng.random((2, 40)) > 0.3
    G = O.gram(X)
    np.testing.assert_allclose(O.gram(X[:, :17]) + O.gram(X[:, 17:]), G, rtol=1e-12, atol=1e-12)  # token blocks
    for g in range(2):
        assert abs(np.trace(G[g]) - (X[g] ** 2).sum()) < 1e-9                      # trace = |X|_F^2
        sv = np.linalg.svd(X[g], compute_uv=False)                                  # a different decomposition
        np.testing.assert_allclose(O.spectrum(G)[g], sv, rtol=1e-9, atol=1e-9)
        Gk = O.gram(X, keep)[g]
        np.testing.assert_allclose(Gk, X[g, keep[g]].T @ X[g, keep[g]], rtol=1e-12, atol=1e-12)


def test_gram_orthogonal_columns():
    """X = U diag(s) with orthonormal columns U: G = diag(s^2), sigma = s sorted."""
    rng = np.random.default_rng(32)
    U, _ = np.linalg.qr(rng.standard_normal((50, 5)))
    s = np.array([4.0, 0.5, 2.0, 1.0, 3.0])
    G = O.gram((U * s)[None])[0]
    np.testing.assert_allclose(G, np.diag(s ** 2), atol=1e-12)
    np.testing.assert_allclose(O.spectrum(G), np.sort(s)[::-1], rtol=1e-12)


def test_ner_closed_forms_and_bounds():
    assert O.ner([3.0] * 7) == pytest.approx(1.0, abs=1e-15)                       # equal values: erank = r
    # sigma = (2, 1, 1): p = (1/2, 1/4, 1/4), H = (1/2)ln2 + (1/2)ln4 = (3/2)ln2,
    # erank = 2^(3/2), NER = 2^(3/2) / 3 (worked by hand)
    assert O.ner([2.0, 1.0, 1.0]) == pytest.approx(2 ** 1.5 / 3, rel=1e-14)
    eps = 2e-3                                                                      # just above rtol = 1e-3
    assert 1 / 5 <= O.ner([1.0] + [eps] * 4) < 1 / 5 * 1.2                         # one dominant value -> 1/r
    assert O.ner([1.0, 1e-6, 1e-6]) == 1.0                                          # below rtol: rank 1
    assert O.ner([0.0, 0.0]) == 0.0
    rng = np.random.default_rng(33)
    for _ in range(50):
        s = rng.random(16) ** 4
        r = O.numerical_rank(s, 1e-3)
        assert 1 / r - 1e-12 <= O.ner(s) <= 1 + 1e-12


def test_lowrank_error_is_eckart_young():
    rng = np.random.default_rng(34)
    X = rng.standard_normal((30, 8)) @ np.diag([5, 4, 3, 2, 1, 0.5, 0.2, 0.1])
    sig = O.spectrum(O.gram(X[None]))[0]
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    for r in (0, 1, 3, 8):
        Xr = (U[:, :r] * S[:r]) @ Vt[:r]
        assert O.lowrank_error(sig, r) == pytest.approx(((X - Xr) ** 2).sum(), rel=1e-9, abs=1e-9)


# ----------------------------------------------------------------------------
# block LSE   [KVSculpt §2]
# ----------------------------------------------------------------------------
def test_block_lse_closed_forms():
    rng = np.random.default_rng(41)
    Q = rng.standard_normal((4, 6, 8))
    K = rng.standard_normal((2, 20, 8))
    got = O.block_lse(Q, K, 14, 1)                                   # one key: its logit
    for hd in range(4):
        np.testing.assert_allclose(got[hd], Q[hd] @ K[hd // 2, 0] / math.sqrt(8), rtol=1e-13)
    Kc = np.repeat(K[:, :1], 20, axis=1)                              # equal keys: logit + ln(count)
    for q0, nb in ((14, 9), (3, 12), (0, 20)):
        got = O.block_lse(Q, Kc, q0, nb)
        for hd in range(4):
            cnt = np.minimum(nb, q0 + np.arange(6) + 1)
            np.testing.assert_allclose(got[hd], Q[hd] @ Kc[hd // 2, 0] / math.sqrt(8) + np.log(cnt), rtol=1e-13)


def test_block_lse_plus_rest_is_row_lse():
    """exp(block LSE) + the brute-force sum over the visible keys after the block
    = exp(row LSE over the whole prefix)."""
    rng = np.random.default_rng(42)
    Q = rng.standard_normal((2, 5, 4))
    K = rng.standard_normal((1, 11, 4))
    q0, nb = 6, 7
    blk = O.block_lse(Q, K, q0, nb)
    for hd in range(2):
        for r in range(5):
            rest = 0.0
            for t in range(nb, q0 + r + 1):                              # pure-Python sum
                rest += math.exp(sum(Q[hd, r, i] * K[0, t, i] for i in range(4)) / 2.0)
            full = 0.0
            for t in range(0, q0 + r + 1):
                full += math.exp(sum(Q[hd, r, i] * K[0, t, i] for i in range(4)) / 2.0)
            assert math.exp(blk[hd, r]) + rest == pytest.approx(full, rel=1e-12)


# ----------------------------------------------------------------------------
# KVSculpt targets and ridge values   [KVSculpt §2]
# ----------------------------------------------------------------------------
def test_block_attention_closed_forms_and_merge():
    rng = np.random.default_rng(51)
    Q = rng.standard_normal((2, 4, 4))
    K = rng.standard_normal((1, 9, 4))
    V = rng.standard_normal((1, 9, 4))
    Y, lse = O.block_attention(Q, K, V, 5, 1)                       # one key: its value row
    np.testing.assert_allclose(Y, np.broadcast_to(V[0, 0], Y.shape), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, O.block_lse(Q, K, 5, 1), rtol=1e-14)
    Kc = np.repeat(K[:, :1], 9, axis=1)                              # equal keys: mean of the visible rows
    Y, _ = O.block_attention(Q, Kc, V, 2, 7)
    for r in range(4):
        np.testing.assert_allclose(Y[0, r], V[0, :min(7, 3 + r)].mean(axis=0), rtol=1e-13)
    # block [0, 5) merged with the rest of the prefix, by hand, = the whole prefix
    Yb, lb = O.block_attention(Q, K, V, 5, 5)
    Ya, la = O.block_attention(Q, K, V, 5, 9)
    for hd in range(2):
        for r in range(4):
            num = math.exp(lb[hd, r]) * Yb[hd, r]
            den = math.exp(lb[hd, r])
            for t in range(5, 5 + r + 1):
                w = math.exp(float(Q[hd, r] @ K[0, t]) / 2.0)
                num = num + w * V[0, t]
                den += w
            np.testing.assert_allclose(Ya[hd, r], num / den, rtol=1e-12)
            assert la[hd, r] == pytest.approx(math.log(den), rel=1e-12)


def test_ridge_values_pins():
    rng = np.random.default_rng(52)
    Qt = rng.standard_normal((20, 8))
    Y = rng.standard_normal((20, 8))
    one = O.ridge_values(Qt, rng.standard_normal((1, 8)), Y, 0.5)    # one key: softmax is 1 everywhere
    np.testing.assert_allclose(one[0], Y.sum(axis=0) / (20 + 0.5), rtol=1e-13)
    Kc = rng.standard_normal((5, 8)) * 2
    S = Qt @ Kc.T / math.sqrt(8)
    A = np.exp(S - S.max(axis=1, keepdims=True))
    A /= A.sum(axis=1, keepdims=True)
    V_true = rng.standard_normal((5, 8))
    np.testing.assert_allclose(O.ridge_values(Qt, Kc, A @ V_true, 1e-12), V_true, rtol=0, atol=1e-5)  # noiseless
    lam = 0.3
    Vc = O.ridge_values(Qt, Kc, Y, lam)
    grad = A.T @ (A @ Vc - Y) + lam * Vc                              # optimality: the gradient vanishes
    assert np.abs(grad).max() < 1e-12
    for trial in range(5):                                           # and nearby points are no better
        P = Vc + 1e-3 * rng.standard_normal(Vc.shape)
        f = lambda X: ((A @ X - Y) ** 2).sum() + lam * (X ** 2).sum()
        assert f(P) >= f(Vc)


def test_ridge_values_closed_forms():
    """Two closed forms that fix the softmax and its 1/sqrt(d) scale without
    restating them   [KVSculpt §2: ridge values for fixed keys].
    Equal keys: every weight is 1/k, A^T A = (R / k^2) 1 1^T, and every value row
    is sum(Y) / (R + lam k).  Two keys a e and 0 seen by R copies of the unit
    query e: the weights are p = logistic(a / sqrt(d)) and 1 - p, so with
    u = (p, 1 - p) the solution of the rank-one system is u sum(Y)^T / (R |u|^2 + lam)."""
    rng = np.random.default_rng(53)
    R, d, k, lam = 12, 16, 5, 0.7
    Qt = rng.standard_normal((R, d))
    Y = rng.standard_normal((R, d))
    Kc = np.repeat(rng.standard_normal((1, d)), k, axis=0)
    Vc = O.ridge_values(Qt, Kc, Y, lam)
    np.testing.assert_allclose(Vc, np.broadcast_to(Y.sum(axis=0) / (R + lam * k), (k, d)), rtol=1e-12)

    e = np.zeros(d)
    e[3] = 1.0
    a = 2.5
    Qt = np.repeat(e[None, :], R, axis=0)
    Kc = np.stack([a * e, np.zeros(d)])
    p = 1.0 / (1.0 + math.exp(-a / math.sqrt(d)))
    u = np.array([p, 1.0 - p])
    expect = np.outer(u, Y.sum(axis=0)) / (R * (u @ u) + lam)
    np.testing.assert_allclose(O.ridge_values(Qt, Kc, Y, lam), expect, rtol=1e-12)
