"""CPU oracle for KV-cache importance scoring and rate-distortion compression.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain, float64 statement
of what the CUDA library computes.  Only the test-suite, the smoke check and
the CPU-baseline leg of the benchmark may import it; the product path never
does, and it shares no code with the CUDA sources (the two meet only in the
seeded input generator, which holds none of the method's arithmetic).

Sources (web summaries of the papers; sections as printed there):
  [RDKV]      "RDKV - Asignacion de Bits de Tasa-Distorsion para Eviccion y
              Cuantizacion Conjunta de la Cache KV" (gist.science 2605.08317):
              §2.1 token weight w_t and channel weight w_c, the RD objective;
              §2.2 reverse water-filling over {0,2,4,8,16}, stages 1-3;
              §2.3 TriZone streams grouped by width.
  [KVzap]     "KVzap - Poda del KV Cache Rapida, Adaptativa y Fiel"
              (gist.science 2601.07891): §2.1 the KVzip and KVzip+ scores;
              §2.3 threshold pruning with a sliding window.
  [KVSculpt]  "KVSculpt: KV Cache Compression as Distillation"
              (gist.science 2603.27819): §2 loss, the log-sum-exp term.

Conventions (row-major arrays, float64 unless stated):
  Q [Hq, W, d]; K, V [Hkv, N, d]; h [W, D]; W_O [D, Hq*d].
  Query head hd belongs to KV head g = hd // G with G = Hq // Hkv.
  Window row r sits at absolute position p_r = q_pos0 + r and sees keys t <= p_r.
  Logits are s = q.k / sqrt(d).
Every function lists its parity pins (the tests that tie it to something other
than itself) in its docstring.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

WIDTHS = (0, 2, 4, 8, 16)
GROUP = 64


# ----------------------------------------------------------------------------
# O1. attention-derived scores
# ----------------------------------------------------------------------------
def attention_scores(Q, K, q_pos0, *, V=None, h=None, W_O=None, row_chunk=512):
    """Row LSE, RDKV token weight, KVzip and KVzip+ scores, from the materialised
    causal softmax.

    lse[hd, r]  = ln sum_{t <= p_r} exp(s_{r,t})                  [KVSculpt §2, LSE term]
    w_t[g, t]   = sum_{hd in g} sum_{r : p_r >= t} a^hd_{r,t}      [RDKV §2.1, w_t = sum_tau a_{tau,t}]
    kvzip[g, t] = max_{hd in g} max_r a^hd_{r,t}                   [KVzap §2.1, KVzip]
    s_plus[g,t] = max_{hd in g} max_r a^hd_{r,t} * |h_r| / |W_O^hd v_t|   [KVzap §2.1, KVzip+]
    with a = exp(s - lse) and W_O^hd = W_O[:, hd*d:(hd+1)*d].

    Rows are materialised in chunks of `row_chunk` full rows (N wide).
    Pins: sum_t w_t = G*W; constant-key harmonic closed form; N = 1;
    brute-force pure-Python LSE, w_t, KVzip+ on tiny inputs.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    G = Hq // Hkv
    assert G * Hkv == Hq
    inv_sqrt_d = 1.0 / math.sqrt(d)
    want_plus = h is not None
    lse = np.zeros((Hq, W))
    w_t = np.zeros((Hkv, N))
    kvzip = np.zeros((Hkv, N))
    s_plus = np.zeros((Hkv, N)) if want_plus else None
    if want_plus:
        hn = np.linalg.norm(np.asarray(h, dtype=np.float64), axis=1)          # |h_r|, [W]
        V = np.asarray(V, dtype=np.float64)
        W_O = np.asarray(W_O, dtype=np.float64)
    tpos = np.arange(N)
    for hd in range(Hq):
        g = hd // G
        col_max = np.zeros(N)
        col_max_plus = np.zeros(N)
        for r0 in range(0, W, row_chunk):
            r1 = min(W, r0 + row_chunk)
            pos = q_pos0 + np.arange(r0, r1)
            S = (Q[hd, r0:r1] @ K[g].T) * inv_sqrt_d                          # [R, N]
            S[tpos[None, :] > pos[:, None]] = -np.inf
            m = S.max(axis=1)
            l_rows = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
            lse[hd, r0:r1] = l_rows
            A = np.exp(S - l_rows[:, None])                                   # softmax rows
            w_t[g] += A.sum(axis=0)
            col_max = np.maximum(col_max, A.max(axis=0))
            if want_plus:
                col_max_plus = np.maximum(col_max_plus, (A * hn[r0:r1, None]).max(axis=0))
        kvzip[g] = np.maximum(kvzip[g], col_max)
        if want_plus:
            Wh = W_O[:, hd * d:(hd + 1) * d]                                  # [D, d]
            vn = np.empty(N)
            for t0 in range(0, N, 4096):
                t1 = min(N, t0 + 4096)
                vn[t0:t1] = np.linalg.norm(Wh @ V[g, t0:t1].T, axis=0)        # |W_O^hd v_t|
            s_plus[g] = np.maximum(s_plus[g], col_max_plus / vn)
    out = {"lse": lse, "w_t": w_t, "kvzip": kvzip}
    if want_plus:
        out["s_plus"] = s_plus
    return out


# ----------------------------------------------------------------------------
# O2. channel weights
# ----------------------------------------------------------------------------
def channel_weights(Q, K):
    """w_c[g, c] = |Q_{:,c}|_2 |K_{:,c}|_2 / sqrt(d)      [RDKV §2.1, w_c]

    The query column stacks the G heads' W window rows of KV group g; the key
    column spans all N tokens of head g.
    Pin: equals the spectral norm of the logit change when channel c is zeroed
    (rank-one outer product), checked by SVD.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Hq, W, d = Q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    qn = np.sqrt((Q.reshape(Hkv, G * W, d) ** 2).sum(axis=1))
    kn = np.sqrt((K ** 2).sum(axis=1))
    return qn * kn / math.sqrt(d)


# ----------------------------------------------------------------------------
# O3. per-unit sigma
# ----------------------------------------------------------------------------
def unit_rms(X, axis, keep=None):
    """sigma of a unit = root mean square of its values.

    axis 0 (V cache, unit = token):   sigma[g, t] = sqrt(mean_c X[g,t,c]^2)
    axis 1 (K cache, unit = channel): sigma[g, c] = sqrt(mean_{t kept} X[g,t,c]^2),
                                      0 when head g keeps no token.
    sigma_u is the per-unit scale in the RD objective [RDKV §2.1]; stage 3
    restricts the K cache to the tokens kept by stage 2 [RDKV §2.2].
    Pin: brute-force pure-Python RMS.
    """
    X = np.asarray(X, dtype=np.float64)
    if axis == 0:
        return np.sqrt((X ** 2).mean(axis=2))
    Hkv, N, d = X.shape
    if keep is None:
        keep = np.ones((Hkv, N), dtype=bool)
    keep = np.asarray(keep).astype(bool).reshape(Hkv, N)
    out = np.zeros((Hkv, d))
    for g in range(Hkv):
        n = int(keep[g].sum())
        if n:
            out[g] = np.sqrt((X[g, keep[g]] ** 2).sum(axis=0) / n)
    return out


# ----------------------------------------------------------------------------
# O4. Lagrangian multiple-choice-knapsack bit allocation
# ----------------------------------------------------------------------------
def chord_slopes(widths):
    """c_k = (2^-b_k - 2^-b_{k+1}) / (b_{k+1} - b_k), each rounded once to fp64.

    D_u(b) = key_u 2^-b is strictly convex in b, so the Lagrangian argmin of
    D_u(b) + lambda*b climbs the widths in order; c_k*key_u is the multiplier at
    which unit u moves from b_k to b_{k+1}.
    """
    ws = list(widths)
    out = []
    for b0, b1 in zip(ws[:-1], ws[1:]):
        out.append(float((Fraction(1, 2 ** b0) - Fraction(1, 2 ** b1)) / (b1 - b0)))
    return out


def allocate_bits(w, sigma, budget, widths=WIDTHS):
    """min sum_u w_u sigma_u 2^-b_u  s.t.  sum_u b_u <= B,  b_u in widths.

    [RDKV §2.1] objective; [RDKV §2.2] discrete widths {0,2,4,8,16} (0 = evict)
    solved by reverse water-filling / Lagrangian relaxation (MCKP).

    Reading (the summary prints only the objective and the method's name):
      key_u = fl64(w_u) * fl64(sigma_u)                  (exact in fp64)
      upgrade items (u, k): theta = fl64(c_k * key_u), cost b_{k+1} - b_k
      order: theta descending, then u ascending, then k ascending; theta <= 0 never taken
      1. Lagrangian prefix: take items in order while the running cost <= B.
      2. Budget fix: keep scanning; take an item iff it fits the remaining
         budget and its predecessor (u, k-1) was taken.
    Returns uint8 widths.
    Pins: exhaustive MCKP on <= 8 units (Everett: the prefix is optimal at its own
    rate); sum b <= B; B = 0 and B >= max*U; widths {0,16} = top-k by key.
    """
    widths = tuple(int(b) for b in widths)
    assert widths[0] == 0 and all(a < b for a, b in zip(widths[:-1], widths[1:]))
    w = np.asarray(w, dtype=np.float32).astype(np.float64).ravel()
    sigma = np.asarray(sigma, dtype=np.float32).astype(np.float64).ravel()
    U = w.size
    key = w * sigma
    c = chord_slopes(widths)
    Kn = len(c)
    cost = np.array([widths[k + 1] - widths[k] for k in range(Kn)], dtype=np.int64)
    theta = np.stack([ck * key for ck in c], axis=1)                          # [U, Kn]
    uu, kk = np.meshgrid(np.arange(U), np.arange(Kn), indexing="ij")
    th, uu, kk = theta.ravel(), uu.ravel(), kk.ravel()
    pos = th > 0
    th, uu, kk = th[pos], uu[pos], kk[pos]
    order = np.lexsort((kk, uu, -th))
    uu, kk = uu[order], kk[order]
    item_cost = cost[kk]
    level = np.zeros(U, dtype=np.int64)
    B = int(budget)
    # 1. prefix
    cum = np.cumsum(item_cost)
    n_prefix = int(np.searchsorted(cum, B, side="right"))
    np.add.at(level, uu[:n_prefix], 1)
    used = int(cum[n_prefix - 1]) if n_prefix else 0
    # 2. budget fix, scanning on in the same order
    rem = B - used
    min_cost = int(cost.min()) if Kn else 0
    for i in range(n_prefix, uu.size):
        if rem < min_cost:
            break
        u, k = int(uu[i]), int(kk[i])
        if item_cost[i] <= rem and level[u] == k:
            level[u] += 1
            rem -= int(item_cost[i])
    return np.asarray(widths, dtype=np.uint8)[level]


def distortion(w, sigma, bits):
    """sum_u w_u sigma_u 2^-b_u with the same fp64 key as allocate_bits."""
    key = np.asarray(w, np.float32).astype(np.float64) * np.asarray(sigma, np.float32).astype(np.float64)
    return float((key * np.exp2(-np.asarray(bits, dtype=np.float64))).sum())


# ----------------------------------------------------------------------------
# O5. quantise / pack / dequantise
# ----------------------------------------------------------------------------
def _bf16_bits(x64):
    """bf16 bit patterns of float64 values that are exactly bf16."""
    f32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    u32 = f32.view(np.uint32)
    assert not np.any(u32 & 0xFFFF), "input is not bf16-representable"
    return (u32 >> 16).astype(np.uint16)


def fp16_scale_ru(a, qmax):
    """Smallest fp16 s with s * qmax >= a (a >= 0, exact).  inf when none is finite."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = (a / qmax).astype(np.float16)
        low = s.astype(np.float64) * qmax < a
        s[low] = np.nextafter(s[low], np.float16(np.inf))
        prev = np.nextafter(s, np.float16(-np.inf))
        ok_prev = (prev >= 0) & (prev.astype(np.float64) * qmax >= a) & np.isfinite(s)
    s[ok_prev] = prev[ok_prev]
    return s


def _unit_rows(X, axis, keep):
    """Element vectors of every unit, in unit-id order, as (ids, list of 1-D arrays).

    axis 0: unit (g, t), id g*N + t, elements X[g, t, 0..d-1].
    axis 1: unit (g, c), id g*d + c, elements X[g, t, c] over kept t ascending.
    """
    Hkv, N, d = X.shape
    if axis == 0:
        return [X[g, t] for g in range(Hkv) for t in range(N)]
    keep = np.asarray(keep).astype(bool).reshape(Hkv, N)
    rows = []
    for g in range(Hkv):
        Xg = X[g, keep[g]]                                                    # [n_g, d]
        rows.extend(Xg[:, c] for c in range(d))
    return rows


def quantize_pack(X, axis, bits, keep=None):
    """Pack a K or V cache into per-width streams.   [RDKV §2.2 stages 2-3, §2.3 TriZone]

    Unit = token (axis 0, V cache) or channel over kept tokens (axis 1, K cache).
    Group = 64 consecutive elements of a unit; a short last group is padded with
    code 0 and left out of the group's absmax.
    Width b in {2,4,8}: qmax = 2^(b-1) - 1; s = smallest fp16 >= absmax/qmax;
    q = round-half-even(x / s) (s = 0 gives q = 0); code = q in b-bit two's
    complement; element e of a group fills bits [b*e, b*e+b) of the group's
    8b-byte block, least significant first.
    Width 16: the raw bf16 bits, no scale.  Width 0: nothing.
    Streams per width: codes (uint8), scales (fp16 bits as uint16, b < 16),
    ids (int32, ascending unit id), group_offsets (int64 start group of each unit).
    Pins: |x - x_hat| <= s/2; s minimal; independent bit-loop unpack; raw-16 exact.
    """
    X = np.asarray(X, dtype=np.float64)
    bits = np.asarray(bits, dtype=np.uint8).ravel()
    rows = _unit_rows(X, axis, keep)
    assert len(rows) == bits.size
    streams = {}
    for wd in (2, 4, 8, 16):
        ids = np.nonzero(bits == wd)[0]
        codes, scales, offs = [], [], []
        ng_total = 0
        for u in ids:
            x = rows[u]
            n = x.size
            ng = -(-n // GROUP)
            offs.append(ng_total)
            ng_total += ng
            if ng == 0:                                # a channel over no kept token: no groups
                continue
            xp = np.zeros(ng * GROUP)
            xp[:n] = x
            xg = xp.reshape(ng, GROUP)
            if wd == 16:
                codes.append(_bf16_bits(xg).view(np.uint8).ravel())
                continue
            qmax = 2 ** (wd - 1) - 1
            a = np.abs(xg).max(axis=1)                # padding zeros never raise absmax
            s = fp16_scale_ru(a, qmax)
            if not np.all(np.isfinite(s)):
                raise OverflowError("group scale overflows fp16")
            s64 = s.astype(np.float64)
            safe = np.where(s64 > 0, s64, 1.0)
            q = np.where(s64[:, None] > 0, np.rint(xg / safe[:, None]), 0.0).astype(np.int64)
            q.reshape(-1)[n:] = 0                      # padding codes are 0
            code = (q & ((1 << wd) - 1)).astype(np.uint8)
            bitplanes = ((code[:, :, None] >> np.arange(wd)[None, None, :]) & 1).astype(np.uint8)
            codes.append(np.packbits(bitplanes.reshape(ng, -1), axis=1, bitorder="little").ravel())
            scales.append(s.view(np.uint16))
        streams[wd] = {
            "ids": ids.astype(np.int32),
            "group_offsets": np.asarray(offs, dtype=np.int64),
            "n_groups": ng_total,
            "codes": np.concatenate(codes) if codes else np.zeros(0, np.uint8),
            "scales": np.concatenate(scales) if scales else np.zeros(0, np.uint16),
        }
    return streams


def dequantize(streams, shape, axis, bits, keep=None):
    """x_hat = q * s in fp32 (exact: <= 8-bit times 11-bit significands);
    width 16 -> the bf16 value; width 0 and tokens not kept -> 0.   [RDKV §2.3]
    Returns float32 [Hkv, N, d].
    """
    Hkv, N, d = shape
    out = np.zeros(shape, dtype=np.float32)
    bits = np.asarray(bits, dtype=np.uint8).ravel()
    if axis == 1:
        keep = np.asarray(keep).astype(bool).reshape(Hkv, N)
    for wd in (2, 4, 8, 16):
        st = streams[wd]
        for j, u in enumerate(st["ids"]):
            u = int(u)
            if axis == 0:
                g, t = divmod(u, N)
                n = d
            else:
                g, c = divmod(u, d)
                tk = np.nonzero(keep[g])[0]
                n = tk.size
            ng = -(-n // GROUP)
            g0 = int(st["group_offsets"][j])
            blk = st["codes"][g0 * 8 * wd:(g0 + ng) * 8 * wd].reshape(ng, 8 * wd)
            if wd == 16:
                raw = blk.view(np.uint16).reshape(-1)[:n].astype(np.uint32) << 16
                vals = raw.view(np.float32)
            else:
                bitplanes = np.unpackbits(blk, axis=1, bitorder="little").reshape(ng, GROUP, wd)
                code = (bitplanes.astype(np.int64) << np.arange(wd)[None, None, :]).sum(axis=2)
                q = np.where(code >= (1 << (wd - 1)), code - (1 << wd), code)
                s = st["scales"][g0:g0 + ng].view(np.float16).astype(np.float32)
                vals = (q.astype(np.float32) * s[:, None]).reshape(-1)[:n]
            if axis == 0:
                out[g, t, :] = vals
            else:
                out[g, tk, c] = vals
    return out


# ----------------------------------------------------------------------------
# Stages 1-3 for one pool (one layer of one sequence)
# ----------------------------------------------------------------------------
def rdkv_compress(Q, K, V, q_pos0, avg_bits, widths=WIDTHS):
    """Stage 1 weights, stage 2 V allocation, stage 3 K allocation over kept
    tokens, then packing.   [RDKV §2.2]

    Budgets: B_V = floor(avg_bits * Hkv*N), B_K = floor(avg_bits * Hkv*d).
    """
    Hkv, N, d = np.shape(K)
    sc = attention_scores(Q, K, q_pos0)
    w_t = sc["w_t"].astype(np.float32)
    w_c = channel_weights(Q, K).astype(np.float32)
    sig_t = unit_rms(V, 0).astype(np.float32)
    bits_v = allocate_bits(w_t, sig_t, math.floor(avg_bits * Hkv * N), widths)
    keep = (bits_v > 0).reshape(Hkv, N)
    sig_c = unit_rms(K, 1, keep).astype(np.float32)
    bits_k = allocate_bits(w_c, sig_c, math.floor(avg_bits * Hkv * d), widths)
    return {"scores": sc, "w_c": w_c, "sigma_t": sig_t, "sigma_c": sig_c,
            "bits_v": bits_v, "bits_k": bits_k, "keep": keep,
            "v_streams": quantize_pack(V, 0, bits_v),
            "k_streams": quantize_pack(K, 1, bits_k, keep)}


# ----------------------------------------------------------------------------
# O6. threshold pruning with a sliding window
# ----------------------------------------------------------------------------
def threshold_keep(score, tau, window, keep_width=16):
    """KVzap's adaptive eviction [KVzap §2.3]: a token whose score is below the
    fixed threshold tau is dropped, except that the last `window` positions
    are always kept.

    score [Hkv, N] is read as float32 and compared with float32(tau) (the
    comparison the library makes); a NaN score is not >= tau, so it is dropped
    unless the window keeps it.  Returns uint8 widths: keep_width or 0.
    Pins: hand-worked fixture; window >= N keeps all; tau = -inf keeps all
    finite scores; tau = +inf keeps exactly the window.
    """
    score = np.asarray(score, dtype=np.float32)
    Hkv, N = score.shape
    with np.errstate(invalid="ignore"):
        keep = score >= np.float32(tau)
    keep[:, max(0, N - int(window)):] = True
    return np.where(keep, keep_width, 0).astype(np.uint8)


# ----------------------------------------------------------------------------
# O7. decode attention over the TriZone streams
# ----------------------------------------------------------------------------
def trizone_decode(q, K_hat, V_hat, keep, k_new=None, v_new=None):
    """One decode step of attention over a compressed cache.   [RDKV §2.3, TriZone]

    The page's decode kernel computes the logits and the output over three
    zones at once, with dequantisation inside the products:
      zone A + B: the old cache, dequantised (K_hat, V_hat from dequantize();
                  zone B is the width-16 part of V), over the kept tokens only;
      zone C:     k_new, v_new [Hkv, Nc, d], tokens generated since compression,
                  all visible.
    An evicted token (keep false) takes no part in the softmax.  Since fusing
    the dequantisation into the products changes no value, the plain definition
    is attention over the dequantised cache:
      s_t = q_h . k_t / sqrt(d),   lse_h = ln sum_t exp(s_t),
      out_h = sum_t exp(s_t - lse_h) v_t,
    with query head h reading KV head h // G.  No visible token: out = 0 and
    lse = -inf.
    q [Hq, d]; K_hat, V_hat [Hkv, N, d]; keep [Hkv, N].  Returns (out [Hq, d],
    lse [Hq]) in float64.
    Pins: hand-worked fixture; one visible token gives its V row; equal logits
    give the mean of V; evicted tokens have no effect however large their key;
    the two-part log-sum-exp merge; permutation invariance.
    """
    q = np.asarray(q, dtype=np.float64)
    K_hat = np.asarray(K_hat, dtype=np.float64)
    V_hat = np.asarray(V_hat, dtype=np.float64)
    keep = np.asarray(keep).astype(bool)
    Hq, d = q.shape
    Hkv = K_hat.shape[0]
    G = Hq // Hkv
    out = np.zeros((Hq, d))
    lse = np.full(Hq, -np.inf)
    for hd in range(Hq):
        g = hd // G
        keys = [K_hat[g, keep[g]]]
        vals = [V_hat[g, keep[g]]]
        if k_new is not None:
            keys.append(np.asarray(k_new, dtype=np.float64)[g])
            vals.append(np.asarray(v_new, dtype=np.float64)[g])
        Kv = np.concatenate(keys, axis=0)
        Vv = np.concatenate(vals, axis=0)
        if Kv.shape[0] == 0:
            continue
        s = Kv @ q[hd] / math.sqrt(d)
        m = s.max()
        e = np.exp(s - m)
        z = e.sum()
        lse[hd] = m + math.log(z)
        out[hd] = (e @ Vv) / z
    return out, lse


# ----------------------------------------------------------------------------
# O8. KV-CoRE: covariance (Gram) accumulation, spectrum, NER, low-rank error
# ----------------------------------------------------------------------------
def gram(X, keep=None):
    """G[g] = sum_t x_t x_t^T over the tokens t of KV head g (the kept ones when
    keep is given), in float64.   [KV-CoRE §2: the covariance updated token by
    token, from which the singular values and right singular vectors follow]
    X [Hkv, N, d]; keep [Hkv, N] or None.  Returns [Hkv, d, d].
    Pins: a sum over two token blocks equals the sum over all; the trace is the
    squared Frobenius norm; orthogonal columns give a diagonal of their squared
    norms; the eigenvalues are the squared singular values of X (SVD).
    """
    X = np.asarray(X, dtype=np.float64)
    Hkv, N, d = X.shape
    G = np.zeros((Hkv, d, d))
    for g in range(Hkv):
        rows = X[g] if keep is None else X[g, np.asarray(keep, bool)[g]]
        for x in rows:                                  # token by token, as the page describes
            G[g] += np.outer(x, x)
    return G


def spectrum(G):
    """Singular values of X from its Gram matrix: sigma_i = sqrt(max(lambda_i, 0))
    for the eigenvalues lambda_i of G, in descending order.   [KV-CoRE §2]
    The eigenvalues come from LAPACK's symmetric solver (a library primitive)."""
    G = np.asarray(G, dtype=np.float64)
    lam = np.linalg.eigvalsh(G)[..., ::-1]
    return np.sqrt(np.maximum(lam, 0.0))


def numerical_rank(sigma, rtol):
    """Number of singular values above rtol * sigma_max (0 for an all-zero spectrum)."""
    sigma = np.asarray(sigma, dtype=np.float64)
    if sigma.size == 0 or sigma.max() <= 0:
        return 0
    return int((sigma > rtol * sigma.max()).sum())


def ner(sigma, rtol=1e-3):
    """Normalised effective rank   [KV-CoRE §2, NER].

    The page defines NER as the effective rank, computed from the distribution
    of the singular values, divided by the actual rank r, so 1/r <= NER <= 1;
    it prints no formula.  Reading taken: the entropy effective rank over the
    r singular values above rtol * sigma_max,
        p_i = sigma_i / sum_{j<=r} sigma_j,   erank = exp(-sum_i p_i ln p_i),
        NER = erank / r.
    An all-zero spectrum gives 0.  Pins: equal singular values give 1; one
    dominant value gives 1/r in the limit; the bounds hold on random spectra.
    """
    sigma = np.sort(np.asarray(sigma, dtype=np.float64))[::-1]
    r = numerical_rank(sigma, rtol)
    if r == 0:
        return 0.0
    s = sigma[:r]
    p = s / s.sum()
    H = -float(np.sum(p * np.log(p)))
    return math.exp(H) / r


def lowrank_error(sigma, r):
    """Squared Frobenius error of the best rank-r approximation of X:
    sum_{i>r} sigma_i^2.   [KV-CoRE §2, Eckart-Young-Mirsky]"""
    sigma = np.sort(np.asarray(sigma, dtype=np.float64))[::-1]
    return float(np.sum(sigma[r:] ** 2))


# ----------------------------------------------------------------------------
# O9. block LSE (the compression zone's attention mass)
# ----------------------------------------------------------------------------
def block_lse(Q, K, q_pos0, n_block):
    """lse[hd, r] = ln sum_{t < n_block, t <= p_r} exp(q_r . k_t / sqrt(d)),
    p_r = q_pos0 + r.   [KVSculpt §2: the LSE term matches the attention mass
    of the compressed block, the leading zone of the cache]
    Q [Hq, W, d]; K [Hkv, N, d] with 1 <= n_block <= N.  Returns [Hq, W].
    Pins: one key gives its logit; equal keys give logit + ln(count); the
    block LSE and a brute-force sum over the rest of the visible keys add up
    to the full row LSE.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Hq, W, d = Q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    out = np.empty((Hq, W))
    t = np.arange(n_block)
    for hd in range(Hq):
        Kb = K[hd // G, :n_block]
        for r in range(W):
            s = Kb @ Q[hd, r] / math.sqrt(d)
            s = s[t <= q_pos0 + r]
            m = s.max()
            out[hd, r] = m + math.log(np.exp(s - m).sum())
    return out


# ----------------------------------------------------------------------------
# O10. KVSculpt targets and the ridge value solve
# ----------------------------------------------------------------------------
def block_attention(Q, K, V, q_pos0, n_block):
    """Attention output and LSE of the window queries over the leading keys
    [0, n_block) of each head: the targets (Y, lse) that KVSculpt's compressed
    pairs must reproduce for the compression zone.   [KVSculpt §2, loss: MSE of
    the output and the LSE term]
    Y[hd, r] = sum_{t < n_block, t <= p_r} softmax_t(q_r . k_t / sqrt(d)) v_t.
    Returns (Y [Hq, W, d], lse [Hq, W]).
    Pins: one key gives its value row; equal keys give the mean of the visible
    rows; the block and the rest of the prefix merge (by their LSE) into the
    attention over the whole prefix.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, W, d = Q.shape
    G = Hq // K.shape[0]
    Y = np.zeros((Hq, W, d))
    lse = np.empty((Hq, W))
    t = np.arange(n_block)
    for hd in range(Hq):
        Kb, Vb = K[hd // G, :n_block], V[hd // G, :n_block]
        for r in range(W):
            vis = t <= q_pos0 + r
            s = Kb[vis] @ Q[hd, r] / math.sqrt(d)
            m = s.max()
            e = np.exp(s - m)
            lse[hd, r] = m + math.log(e.sum())
            Y[hd, r] = (e @ Vb[vis]) / e.sum()
    return Y, lse


def ridge_values(Qt, Kc, Y, lam):
    """Closed-form values of KVSculpt's alternating solve for fixed keys
    [KVSculpt §2: with the keys fixed, the values are a ridge least-squares
    solution]:
        A = softmax_rows(Qt Kc^T / sqrt(d))             [R, k]
        V_c = argmin |A V - Y|_F^2 + lam |V|_F^2 = (A^T A + lam I)^-1 A^T Y.
    Qt [R, d] training queries, Kc [k, d] compressed keys, Y [R, d] targets,
    lam > 0.  Returns V_c [k, d].  The linear solve is LAPACK's (a library
    primitive).
    Pins: one key gives sum(Y) / (R + lam); k equal keys give sum(Y) /
    (R + lam k) in every row; two keys a e and 0 under copies of the unit query
    e give the rank-one closed form with weights logistic(a / sqrt(d));
    noiseless targets Y = A V are recovered as lam -> 0; the gradient of the
    objective vanishes at V_c.
    """
    Qt = np.asarray(Qt, dtype=np.float64)
    Kc = np.asarray(Kc, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    d = Qt.shape[1]
    S = Qt @ Kc.T / math.sqrt(d)
    S = S - S.max(axis=1, keepdims=True)
    A = np.exp(S)
    A /= A.sum(axis=1, keepdims=True)
    k = Kc.shape[0]
    return np.linalg.solve(A.T @ A + lam * np.eye(k), A.T @ Y)
