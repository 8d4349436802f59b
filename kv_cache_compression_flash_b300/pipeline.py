"""One pass of the RDKV hot path over one (layer, sequence) pool.

Stage 1 weights, stage 2 V allocation, stage 3 K allocation over the kept
tokens, then packing (and optionally dequantisation), each step a call into
libkvs.so.   [RDKV §2.2 pipeline; §2.3 TriZone streams]

Buffers are allocated once per shape so a step allocates nothing and can be
replayed from CUDA graphs.
"""
from __future__ import annotations

import math

import torch

from . import _lib as K_


class RdkvLayerStep:
    """Preallocated outputs and workspaces for one pool shape.

    run() = pass1() + pass2() + rest(): pass 1 computes the row LSE, pass 2
    the token weights from it, rest() everything after scoring.
    """

    PASS2_MODE = K_.MODE_RDKV_WT | K_.MODE_LSE_GIVEN
    BOTH_MODE = K_.MODE_LSE | K_.MODE_RDKV_WT      # both passes in one call (the merge writes pass 2's offsets)
    SEGMENTS = ("pass1", "pass2", "rest")

    def __init__(self, Hq, Hkv, N, W, d, avg_bits, device="cuda", width_mask=K_.WIDTHS_ALL, dequant=True):
        self.shape = (Hq, Hkv, N, W, d)
        self.dequant = dequant
        self.width_mask = width_mask
        dev = torch.device(device)
        self.U_v, self.U_k = Hkv * N, Hkv * d
        self.B_v = int(math.floor(avg_bits * self.U_v))
        self.B_k = int(math.floor(avg_bits * self.U_k))
        f32 = dict(dtype=torch.float32, device=dev)
        self.out = {"lse": torch.empty(Hq, W, **f32), "w_t": torch.empty(Hkv, N, **f32)}
        self.w_c = torch.empty(Hkv, d, **f32)
        self.sig_t = torch.empty(Hkv, N, **f32)
        self.sig_c = torch.empty(Hkv, d, **f32)
        self.bits_v = torch.empty(self.U_v, dtype=torch.uint8, device=dev)
        self.bits_k = torch.empty(self.U_k, dtype=torch.uint8, device=dev)
        self.v_streams = K_.Streams(Hkv, N, d, 0, self.B_v, dev)
        self.k_streams = K_.Streams(Hkv, N, d, 1, self.B_k, dev)
        self.v_hat = torch.empty(Hkv, N, d, **f32) if dequant else None
        self.k_hat = torch.empty(Hkv, N, d, **f32) if dequant else None
        names = ("score", "score2", "score12", "cw", "rms0", "rms1", "av", "ak", "pv", "pk", "dv", "dk")
        self.ws = {k: K_.Workspace() for k in names}
        # size every workspace now so a step allocates nothing
        L = K_.lib()
        sizes = {
            "score": L.kvs_score_workspace_size(Hq, Hkv, W, N, d, 0, N - W, K_.MODE_LSE),
            "score2": L.kvs_score_workspace_size(Hq, Hkv, W, N, d, 0, N - W, self.PASS2_MODE),
            "score12": L.kvs_score_workspace_size(Hq, Hkv, W, N, d, 0, N - W, self.BOTH_MODE),
            "cw": L.kvs_channel_weights_workspace_size(Hq, Hkv, W, N, d),
            "rms0": 256, "rms1": L.kvs_unit_rms_workspace_size(Hkv, N, d, 1),
            "av": L.kvs_allocate_workspace_size(self.U_v), "ak": L.kvs_allocate_workspace_size(self.U_k),
            "pv": L.kvs_pack_workspace_size(Hkv, N, d, 0), "pk": L.kvs_pack_workspace_size(Hkv, N, d, 1),
            "dv": L.kvs_pack_workspace_size(Hkv, N, d, 0), "dk": L.kvs_pack_workspace_size(Hkv, N, d, 1),
        }
        for k, n in sizes.items():
            self.ws[k].get(n, dev)
        self.graphs = None
        self.side_stream = torch.cuda.Stream(device=dev)
        self.v_done = torch.cuda.Event()

    def kernel_launches(self) -> int:
        """Kernels one step launches (memset nodes excluded)."""
        Hq, Hkv, N, W, d = self.shape
        n = K_.score_plan_info(Hq, Hkv, W, N, d, mode=self.BOTH_MODE)[4]   # the step's one scoring call
        n += 1          # channel weights (one cluster per KV head)
        n += 1          # sigma_t
        n += 1 + 1      # V allocation, sigma_c
        n += 1          # K allocation
        n += 2 + 2      # V pack (plan, pack), K pack (plan, pack)
        if self.dequant:
            # V dequant (decode + zero); K dequant (decode + zero, planned inside the
            # kernel up to 16 384 tokens, else a plan kernel first)
            n += 1 + (1 if N <= 16384 and Hkv * d < 65536 else 2)
        return n

    def pass1(self, Q, K, V, stream=None):
        Hq, Hkv, N, W, d = self.shape
        K_.score_attention(Q, K, q_pos0=N - W, mode=K_.MODE_LSE, out=self.out, ws=self.ws["score"], stream=stream)

    def score(self, Q, K, V, stream=None):
        """Both passes in one call (the step); pass1/pass2 split them for timing."""
        Hq, Hkv, N, W, d = self.shape
        K_.score_attention(Q, K, q_pos0=N - W, mode=self.BOTH_MODE, out=self.out, ws=self.ws["score12"],
                           stream=stream)

    def pass2(self, Q, K, V, stream=None):
        Hq, Hkv, N, W, d = self.shape
        K_.score_attention(Q, K, q_pos0=N - W, mode=self.PASS2_MODE, out=self.out, ws=self.ws["score2"],
                           stream=stream)

    def rest(self, Q, K, V, stream=None):
        """Everything after scoring, as two dependent chains on two streams:
        V: sigma_t -> V allocation -> V pack (-> dequant);
        K: w_c (from the start), then after the V widths: sigma_c -> K
        allocation -> K pack (-> dequant)."""
        ws = self.ws
        main = stream if stream is not None else torch.cuda.current_stream()
        side = self.side_stream
        side.wait_stream(main)
        with torch.cuda.stream(side):
            K_.channel_weights(Q, K, out=self.w_c, ws=ws["cw"], stream=side)
        K_.unit_rms(V, 0, out=self.sig_t, ws=ws["rms0"], stream=main)
        K_.allocate_bits(self.out["w_t"], self.sig_t, self.B_v, self.width_mask, out=self.bits_v, ws=ws["av"],
                         stream=main)
        self.v_done.record(main)
        with torch.cuda.stream(side):
            side.wait_event(self.v_done)
            K_.unit_rms(K, 1, keep_bits=self.bits_v, out=self.sig_c, ws=ws["rms1"], stream=side)
            K_.allocate_bits(self.w_c, self.sig_c, self.B_k, self.width_mask, out=self.bits_k, ws=ws["ak"],
                             stream=side)
            K_.quantize_pack(K, 1, self.bits_k, self.bits_v, self.k_streams, ws=ws["pk"], stream=side)
            if self.dequant:
                K_.dequantize(self.k_streams, self.bits_k, self.bits_v, out=self.k_hat, ws=ws["dk"], stream=side)
        K_.quantize_pack(V, 0, self.bits_v, None, self.v_streams, ws=ws["pv"], stream=main)
        if self.dequant:
            K_.dequantize(self.v_streams, self.bits_v, None, out=self.v_hat, ws=ws["dv"], stream=main)
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
