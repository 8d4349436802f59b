"""One pass of the RDKV hot path over a batch of (layer, sequence) pools.

Stage 1 weights, stage 2 V allocation, stage 3 K allocation over the kept
tokens, then packing (and optionally dequantisation), each step a call into
libkvs.so.   [RDKV §2.2 pipeline; §2.3 TriZone streams]

A pool is one (layer, sequence) cache with all of its KV heads; the RD
allocation is solved per pool.  n_pools pools of one shape are processed
together: the scoring and norm calls see them as one cache of n_pools * Hkv
KV heads (every quantity they compute is per KV head), the allocation and
packing calls take the pool count and keep each pool's solution and streams
separate.

Buffers are allocated once per shape so a step allocates nothing and can be
replayed from CUDA graphs.
"""
from __future__ import annotations

import math

import torch

from . import _lib as K_


class RdkvLayerStep:
    """Preallocated outputs and workspaces for n_pools pools of one shape.

    Inputs: Q [n_pools*Hq, W, d], K and V [n_pools*Hkv, N, d] (bf16,
    contiguous; pool q's heads are rows q*Hq.. and q*Hkv..).
    run() = score() + rest(): score() computes the row LSE (pass 1) and the
    token weights (pass 2), rest() everything after scoring; pass1() and
    pass2() split the scoring for timing.
    """

    PASS2_MODE = K_.MODE_RDKV_WT | K_.MODE_LSE_GIVEN
    BOTH_MODE = K_.MODE_LSE | K_.MODE_RDKV_WT      # both passes in one call (the merge writes pass 2's offsets)
    SEGMENTS = ("pass1", "pass2", "rest")

    def __init__(self, Hq, Hkv, N, W, d, avg_bits, device="cuda", width_mask=K_.WIDTHS_ALL, dequant=True,
                 n_pools=1):
        self.shape = (Hq, Hkv, N, W, d)
        self.n_pools = P = n_pools
        self.dequant = dequant
        self.width_mask = width_mask
        dev = torch.device(device)
        self.U_v, self.U_k = Hkv * N, Hkv * d
        self.B_v = int(math.floor(avg_bits * self.U_v))
        self.B_k = int(math.floor(avg_bits * self.U_k))
        f32 = dict(dtype=torch.float32, device=dev)
        self.out = {"lse": torch.empty(P * Hq, W, **f32), "w_t": torch.empty(P * Hkv, N, **f32)}
        self.w_c = torch.empty(P * Hkv, d, **f32)
        self.sig_t = torch.empty(P * Hkv, N, **f32)
        self.sig_c = torch.empty(P * Hkv, d, **f32)
        self.bits_v = torch.empty(P * self.U_v, dtype=torch.uint8, device=dev)
        self.bits_k = torch.empty(P * self.U_k, dtype=torch.uint8, device=dev)
        self.v_streams = K_.Streams(Hkv, N, d, 0, self.B_v, dev, n_pools=P)
        self.k_streams = K_.Streams(Hkv, N, d, 1, self.B_k, dev, n_pools=P)
        self.v_hat = torch.empty(P * Hkv, N, d, **f32) if dequant else None
        self.k_hat = torch.empty(P * Hkv, N, d, **f32) if dequant else None
        names = ("score", "score2", "score12", "cw", "rms0", "rms1", "av", "ak", "pv", "pk", "dv", "dk")
        self.ws = {k: K_.Workspace() for k in names}
        # size every workspace now so a step allocates nothing
        L = K_.lib()
        HQ, HKV = P * Hq, P * Hkv
        sizes = {
            "score": L.kvs_score_workspace_size(HQ, HKV, W, N, d, 0, N - W, K_.MODE_LSE),
            "score2": L.kvs_score_workspace_size(HQ, HKV, W, N, d, 0, N - W, self.PASS2_MODE),
            "score12": L.kvs_score_workspace_size(HQ, HKV, W, N, d, 0, N - W, self.BOTH_MODE),
            "cw": L.kvs_channel_weights_workspace_size(HQ, HKV, W, N, d),
            "rms0": 256, "rms1": L.kvs_unit_rms_workspace_size(HKV, N, d, 1),
            "av": L.kvs_allocate_pools_workspace_size(P, self.U_v), "ak": L.kvs_allocate_pools_workspace_size(P, self.U_k),
            "pv": L.kvs_pack_pools_workspace_size(P, Hkv, N, d, 0), "pk": L.kvs_pack_pools_workspace_size(P, Hkv, N, d, 1),
            "dv": L.kvs_pack_pools_workspace_size(P, Hkv, N, d, 0), "dk": L.kvs_pack_pools_workspace_size(P, Hkv, N, d, 1),
        }
        for k, n in sizes.items():
            self.ws[k].get(n, dev)
        self.graphs = None
        self.side_stream = torch.cuda.Stream(device=dev)
        self.v_done = torch.cuda.Event()

    # ---- views --------------------------------------------------------------
    def pool_bits(self):
        """(bits_v [n_pools, U_v], bits_k [n_pools, U_k])."""
        return self.bits_v.view(self.n_pools, self.U_v), self.bits_k.view(self.n_pools, self.U_k)

    def kernel_launches(self) -> int:
        """Kernels one step launches (memset nodes excluded)."""
        Hq, Hkv, N, W, d = self.shape
        P = self.n_pools
        n = K_.score_plan_info(P * Hq, P * Hkv, W, N, d, mode=self.BOTH_MODE)[4]   # the step's one scoring call
        n += 1          # sigma_t
        for U in (self.U_v, self.U_k):   # allocations: one launch for every pool on clusters, else one per pool
            n += 1 if K_.allocate_plan_info(U, self.width_mask)[0] > 0 else P
        n += 1          # w_c and sigma_c (one cluster per KV head)
        n += 2 + 2      # V pack (chunk counts, pack), K pack (plan, pack)
        if self.dequant:
            n += 2 + 2  # V dequant (chunk counts, decode), K dequant (plan, decode + zero)
        return n

    def _flat(self, Q, K, V):
        Hq, Hkv, N, W, d = self.shape
        P = self.n_pools
        return (Q.view(P * Hq, W, d), K.view(P * Hkv, N, d), None if V is None else V.view(P * Hkv, N, d))

    def pass1(self, Q, K, V, stream=None):
        Hq, Hkv, N, W, d = self.shape
        Q, K, V = self._flat(Q, K, V)
        K_.score_attention(Q, K, q_pos0=N - W, mode=K_.MODE_LSE, out=self.out, ws=self.ws["score"], stream=stream)

    def score(self, Q, K, V, stream=None):
        """Both passes in one call (the step); pass1/pass2 split them for timing."""
        Hq, Hkv, N, W, d = self.shape
        Q, K, V = self._flat(Q, K, V)
        K_.score_attention(Q, K, q_pos0=N - W, mode=self.BOTH_MODE, out=self.out, ws=self.ws["score12"],
                           stream=stream)

    def pass2(self, Q, K, V, stream=None):
        Hq, Hkv, N, W, d = self.shape
        Q, K, V = self._flat(Q, K, V)
        K_.score_attention(Q, K, q_pos0=N - W, mode=self.PASS2_MODE, out=self.out, ws=self.ws["score2"],
                           stream=stream)

    def rest(self, Q, K, V, stream=None):
        """Everything after scoring, as two dependent chains on two streams:
        V: sigma_t -> V allocation -> V pack (-> dequant);
        K, after the V widths: w_c and sigma_c (one read of K) -> K
        allocation -> K pack (-> dequant)."""
        Hq, Hkv, N, W, d = self.shape
        P = self.n_pools
        Q, K, V = self._flat(Q, K, V)
        ws = self.ws
        main = stream if stream is not None else torch.cuda.current_stream()
        side = self.side_stream
        K_.unit_rms(V, 0, out=self.sig_t, ws=ws["rms0"], stream=main)
        bits_v, bits_k = self.pool_bits()
        K_.allocate_bits_pools(self.out["w_t"].view(P, self.U_v), self.sig_t.view(P, self.U_v), self.B_v,
                               self.width_mask, out=bits_v, ws=ws["av"], stream=main)
        self.v_done.record(main)
        X4 = (P, Hkv, N, d)
        with torch.cuda.stream(side):
            side.wait_event(self.v_done)
            K_.channel_stats(Q, K, self.bits_v, out_wc=self.w_c, out_sigma=self.sig_c, stream=side)
            K_.allocate_bits_pools(self.w_c.view(P, self.U_k), self.sig_c.view(P, self.U_k), self.B_k,
                                   self.width_mask, out=bits_k, ws=ws["ak"], stream=side)
            K_.quantize_pack_pools(K.view(X4), 1, self.bits_k, self.bits_v, self.k_streams, ws=ws["pk"], stream=side)
            if self.dequant:
                K_.dequantize_pools(self.k_streams, self.bits_k, self.bits_v, out=self.k_hat.view(X4), ws=ws["dk"],
                                    stream=side)
        K_.quantize_pack_pools(V.view(X4), 0, self.bits_v, None, self.v_streams, ws=ws["pv"], stream=main)
        if self.dequant:
            K_.dequantize_pools(self.v_streams, self.bits_v, None, out=self.v_hat.view(X4), ws=ws["dv"], stream=main)
        main.wait_stream(side)

    def run(self, Q, K, V, stream=None):
        self.score(Q, K, V, stream)
        self.rest(Q, K, V, stream)
        return self

    # ---- CUDA graphs: one per segment, so a replay launches no Python -------
    def capture(self, Q, K, V):
        """Records pass1 / pass2 / rest as three CUDA graphs over these buffers."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                self.run(Q, K, V)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graphs = {}
        for name in self.SEGMENTS:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                getattr(self, name)(Q, K, V)
            self.graphs[name] = g
        # the whole step as one graph as well: no launch gap between segments
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            self.run(Q, K, V)
        self.step_graph = g
        torch.cuda.synchronize()
        return self

    def replay_step(self):
        """Replays the whole captured step as one graph."""
        self.step_graph.replay()
        return self

    def replay(self, events=None):
        """Replays the captured step; `events` (4 CUDA events) bracket the segments."""
        if events is not None:
            events[0].record()
        for i, name in enumerate(self.SEGMENTS):
            self.graphs[name].replay()
            if events is not None:
                events[i + 1].record()
        return self


class KvzipStep(RdkvLayerStep):
    """KVzap's eviction pass over one pool: KVzip+ scores, then the bottom
    fraction of tokens evicted and the rest kept at 16 bits   [KVzap §2.1
    score s+, §2.3 eviction by score].

    Inputs as RdkvLayerStep plus h [W, D] and W_O [D, Hq*d] (given to the
    constructor, they stay fixed).  Stage 2 is the allocation over widths
    {0, 16} with sigma = 1 and budget 16 * (U - floor(evict * U)), which keeps
    exactly the top-scoring tokens (ties to the lower unit); the K cache is
    stored for the kept tokens at 16 bits per channel.
    """

    PASS2_MODE = K_.MODE_KVZIP_PLUS | K_.MODE_LSE_GIVEN
    BOTH_MODE = K_.MODE_LSE | K_.MODE_KVZIP_PLUS

    def __init__(self, Hq, Hkv, N, W, d, evict_fraction, h, W_O, device="cuda", dequant=True):
        U = Hkv * N
        keep = U - int(math.floor(evict_fraction * U))
        super().__init__(Hq, Hkv, N, W, d, 16.0 * keep / U, device=device, width_mask=K_.WIDTHS_KEEP_OR_EVICT,
                         dequant=dequant, n_pools=1)
        dev = torch.device(device)
        self.B_v = 16 * keep
        self.B_k = 16 * self.U_k
        self.h, self.W_O = h, W_O
        self.D = h.shape[1]
        self.out["s_plus"] = torch.empty(Hkv, N, dtype=torch.float32, device=dev)
        self.ones = torch.ones(U, dtype=torch.float32, device=dev)
        self.bits_k.fill_(16)                      # kept tokens: every K channel at 16 bits
        self.v_streams = K_.Streams(Hkv, N, d, 0, self.B_v, dev)
        self.k_streams = K_.Streams(Hkv, N, d, 1, self.B_k, dev)
        L = K_.lib()
        for k, mode in (("score", K_.MODE_LSE), ("score2", self.PASS2_MODE), ("score12", self.BOTH_MODE)):
            self.ws[k].get(L.kvs_score_workspace_size(Hq, Hkv, W, N, d, self.D, N - W, mode), dev)

    def kernel_launches(self) -> int:
        Hq, Hkv, N, W, d = self.shape
        n = K_.score_plan_info(Hq, Hkv, W, N, d, D=self.D, mode=self.BOTH_MODE)[4]
        n += 1 if K_.allocate_plan_info(self.U_v, self.width_mask)[0] > 0 else 1
        n += 2 + 2      # V pack (chunk counts, pack), K pack (plan, pack)
        if self.dequant:
            n += 2 + 2  # V dequant (chunk counts, decode), K dequant (plan, decode + zero)
        return n

    def _score(self, Q, K, V, mode, ws, stream):
        Hq, Hkv, N, W, d = self.shape
        K_.score_attention(Q, K, q_pos0=N - W, mode=mode, V=V, h=self.h, W_O=self.W_O, out=self.out, ws=ws,
                           stream=stream)

    def pass1(self, Q, K, V, stream=None):
        self._score(Q, K, V, K_.MODE_LSE, self.ws["score"], stream)

    def pass2(self, Q, K, V, stream=None):
        self._score(Q, K, V, self.PASS2_MODE, self.ws["score2"], stream)

    def score(self, Q, K, V, stream=None):
        self._score(Q, K, V, self.BOTH_MODE, self.ws["score12"], stream)

    def rest(self, Q, K, V, stream=None):
        """Eviction by score (widths {0, 16}), then V rows and K channels of the
        kept tokens packed raw (16 bits) and read back."""
        ws = self.ws
        main = stream if stream is not None else torch.cuda.current_stream()
        K_.allocate_bits(self.out["s_plus"], self.ones, self.B_v, self.width_mask, out=self.bits_v, ws=ws["av"],
                         stream=main)
        K_.quantize_pack(V, 0, self.bits_v, None, self.v_streams, ws=ws["pv"], stream=main)
        K_.quantize_pack(K, 1, self.bits_k, self.bits_v, self.k_streams, ws=ws["pk"], stream=main)
        if self.dequant:
            K_.dequantize(self.v_streams, self.bits_v, None, out=self.v_hat, ws=ws["dv"], stream=main)
            K_.dequantize(self.k_streams, self.bits_k, self.bits_v, out=self.k_hat, ws=ws["dk"], stream=main)
