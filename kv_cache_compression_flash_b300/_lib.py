"""ctypes binding of libkvs.so (C ABI in include/kvs.h).

Argument marshalling only: every computation runs in the CUDA library.  Torch
supplies device memory (outputs, workspaces, stream buffers) and the current
CUDA stream.  There is no fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int, c_int64, c_size_t, c_uint32, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvs.so")

KVS_OK = 0
STATUS = {0: "KVS_OK", 1: "KVS_ERR_INVALID_ARG", 2: "KVS_ERR_UNSUPPORTED", 3: "KVS_ERR_RANGE",
          4: "KVS_ERR_CUDA", 5: "KVS_ERR_TIMEOUT", 6: "KVS_ERR_WORKSPACE", 7: "KVS_ERR_BOUNDS"}

MODE_LSE = 1
MODE_RDKV_WT = 2
MODE_KVZIP = 4
MODE_KVZIP_PLUS = 8
MODE_LSE_GIVEN = 16

WIDTHS_ALL = (1 << 2) | (1 << 4) | (1 << 8) | (1 << 16)
WIDTHS_KEEP_OR_EVICT = 1 << 16
STREAM_WIDTHS = (2, 4, 8, 16)

# every exported symbol the header declares, with its ctypes signature
SIGNATURES = {
    "kvs_status_string": (c_char_p, [c_int]),
    "kvs_version": (c_int, []),
    "kvs_get_device_error": (c_int, [c_void_p]),
    "kvs_debug_inject": (c_int, [c_uint32, ctypes.c_uint64]),
    "kvs_debug_exp2": (c_int, [c_void_p, c_void_p, c_int64, c_void_p]),
    "kvs_score_workspace_size": (c_size_t, [c_int64] * 7 + [c_uint32]),
    "kvs_score_attention": (c_int, [c_void_p] * 5 + [c_int64] * 7 + [c_uint32] + [c_void_p] * 4 + [c_size_t, c_void_p]),
    "kvs_score_plan_info": (c_int, [c_int64] * 7 + [c_uint32, POINTER(c_int64)]),
    "kvs_channel_weights_workspace_size": (c_size_t, [c_int64] * 5),
    "kvs_channel_weights": (c_int, [c_void_p, c_void_p] + [c_int64] * 5 + [c_void_p, c_void_p, c_size_t, c_void_p]),
    "kvs_channel_stats": (c_int, [c_void_p] * 3 + [c_int64] * 5 + [c_void_p] * 3),
    "kvs_unit_rms_workspace_size": (c_size_t, [c_int64] * 3 + [c_int]),
    "kvs_unit_rms": (c_int, [c_void_p] + [c_int64] * 3 + [c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "kvs_allocate_workspace_size": (c_size_t, [c_int64]),
    "kvs_allocate_pools_workspace_size": (c_size_t, [c_int64, c_int64]),
    "kvs_allocate_bits": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_uint32, c_void_p, c_void_p, c_size_t,
                                  c_void_p]),
    "kvs_allocate_bits_static": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_uint32, c_void_p, c_void_p]),
    "kvs_allocate_bits_pools": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_uint32, c_void_p, c_void_p,
                                        c_size_t, c_void_p]),
    "kvs_allocate_plan_info": (c_int, [c_int64, c_uint32, POINTER(c_int64)]),
    "kvs_pack_capacity": (c_int, [c_int64] * 3 + [c_int, c_int64, POINTER(c_int64), POINTER(c_int64)]),
    "kvs_pack_workspace_size": (c_size_t, [c_int64] * 3 + [c_int]),
    "kvs_quantize_pack": (c_int, [c_void_p] + [c_int64] * 3 + [c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                               c_size_t, c_void_p]),
    "kvs_dequantize": (c_int, [c_void_p] + [c_int64] * 3 + [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                                            c_void_p]),
    "kvs_pack_pools_workspace_size": (c_size_t, [c_int64] * 4 + [c_int]),
    "kvs_quantize_pack_pools": (c_int, [c_void_p] + [c_int64] * 4 + [c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                                     c_size_t, c_void_p]),
    "kvs_dequantize_pools": (c_int, [c_void_p] + [c_int64] * 4 + [c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                                  c_size_t, c_void_p]),
    "kvs_threshold_keep": (c_int, [c_void_p, c_int64, c_int64, ctypes.c_float, c_int64, c_uint32, c_void_p,
                                   c_void_p]),
    "kvs_trizone_index_size": (c_size_t, [c_int64, c_int64]),
    "kvs_trizone_index": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_void_p, c_size_t,
                                  c_void_p]),
    "kvs_trizone_workspace_size": (c_size_t, [c_int64] * 5),
    "kvs_trizone_decode": (c_int, [c_void_p] + [c_int64] * 4 + [c_void_p] * 6 + [c_int64] + [c_void_p] * 3
                           + [c_size_t, c_void_p]),
    "kvs_block_lse_workspace_size": (c_size_t, [c_int64] * 7),
    "kvs_block_lse": (c_int, [c_void_p, c_void_p] + [c_int64] * 7 + [c_void_p, c_void_p, c_size_t, c_void_p]),
    "kvs_gram_workspace_size": (c_size_t, [c_int64] * 3),
    "kvs_gram": (c_int, [c_void_p] + [c_int64] * 3 + [c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "kvs_spectrum": (c_int, [c_void_p, c_int64, c_int64, ctypes.c_float, c_void_p, c_void_p, c_void_p, c_void_p]),
    "kvs_block_attention": (c_int, [c_void_p] * 3 + [c_int64] * 7 + [c_void_p] * 3),
    "kvs_ridge_values_workspace_size": (c_size_t, [c_int64] * 4),
    "kvs_ridge_values": (c_int, [c_void_p] * 3 + [c_int64] * 4 + [ctypes.c_float, c_void_p, c_void_p, c_size_t,
                                                                  c_void_p]),
}


class KvsError(RuntimeError):
    pass


class StreamSetC(ctypes.Structure):
    _fields_ = [("codes", c_void_p * 4), ("scales", c_void_p * 4), ("unit_ids", c_void_p * 4),
                ("group_offsets", c_void_p * 4), ("cap_units", c_int64 * 4), ("cap_groups", c_int64 * 4),
                ("counts", c_void_p)]


_lib = None


def lib():
    """The loaded library (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvsError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != KVS_OK:
        raise KvsError(f"{what}: {STATUS.get(rc, rc)}")


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _bf16(t, name):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise KvsError(f"{name} must be a contiguous bf16 CUDA tensor")
    return t


class Workspace:
    """A growable device scratch buffer (one per caller)."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int, device):
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_default_ws = {}


def _ws(ws, key, nbytes, device):
    if ws is None:
        ws = _default_ws.setdefault(key, Workspace())
    return ws.get(nbytes, device)


DEBUG_NONE = 0
DEBUG_WITHHOLD_LSE_ARRIVE = 1


def debug_inject(fault=DEBUG_NONE, wait_limit_ns=0):
    """Test hook: plant a device fault in later launches and set the wait limit (0 = default)."""
    _check(lib().kvs_debug_inject(fault, wait_limit_ns), "kvs_debug_inject")


def debug_exp2(x, *, stream=None):
    """The library's FMA-pipe 2^x of a float32 CUDA tensor (test hook)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise KvsError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x)
    _check(lib().kvs_debug_exp2(_ptr(x), _ptr(y), x.numel(), _stream(stream)), "kvs_debug_exp2")
    return y


def device_error(stream=None) -> int:
    """Reads and clears the library's device error word (synchronises the stream)."""
    return lib().kvs_get_device_error(_stream(stream))


def score_attention(Q, K, *, q_pos0=None, mode=MODE_LSE | MODE_RDKV_WT, V=None, h=None, W_O=None,
                    out=None, ws=None, stream=None):
    """lse [Hq,W], w_t [Hkv,N], s_plus [Hkv,N] (per mode) from bf16 Q [Hq,W,d], K [Hkv,N,d]."""
    _bf16(Q, "Q"), _bf16(K, "K")
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    q_pos0 = N - W if q_pos0 is None else q_pos0
    D = 0
    if mode & MODE_KVZIP_PLUS:
        _bf16(V, "V"), _bf16(h, "h"), _bf16(W_O, "W_O")
        D = h.shape[1]
    dev = Q.device
    out = {} if out is None else out
    lse = out.get("lse")
    if lse is None and mode & MODE_LSE_GIVEN:
        raise KvsError("MODE_LSE_GIVEN needs out['lse'] as input")
    if lse is None:
        lse = out["lse"] = torch.empty(Hq, W, dtype=torch.float32, device=dev)
    w_t = s_plus = None
    if mode & MODE_RDKV_WT:
        w_t = out.get("w_t")
        if w_t is None:
            w_t = out["w_t"] = torch.empty(Hkv, N, dtype=torch.float32, device=dev)
    if mode & (MODE_KVZIP | MODE_KVZIP_PLUS):
        s_plus = out.get("s_plus")
        if s_plus is None:
            s_plus = out["s_plus"] = torch.empty(Hkv, N, dtype=torch.float32, device=dev)
    L = lib()
    nbytes = L.kvs_score_workspace_size(Hq, Hkv, W, N, d, D, q_pos0, mode)
    if nbytes == 0:
        raise KvsError("kvs_score_workspace_size: unsupported shape or mode")
    buf = _ws(ws, "score", nbytes, dev)
    _check(L.kvs_score_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(h), _ptr(W_O), Hq, Hkv, W, N, d, D, q_pos0,
                                 mode, _ptr(lse), _ptr(w_t), _ptr(s_plus), _ptr(buf), buf.numel(),
                                 _stream(stream)), "kvs_score_attention")
    return out


def score_plan_info(Hq, Hkv, W, N, d, D=0, q_pos0=None, mode=MODE_LSE | MODE_RDKV_WT):
    """(kt_chunk, pass-1 splits, qt_chunk, pass-2 splits, kernels launched) of kvs_score_attention."""
    info = (c_int64 * 5)()
    q_pos0 = N - W if q_pos0 is None else q_pos0
    _check(lib().kvs_score_plan_info(Hq, Hkv, W, N, d, D, q_pos0, mode, info), "kvs_score_plan_info")
    return tuple(info)


def channel_weights(Q, K, *, out=None, ws=None, stream=None):
    _bf16(Q, "Q"), _bf16(K, "K")
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    w_c = out if out is not None else torch.empty(Hkv, d, dtype=torch.float32, device=Q.device)
    L = lib()
    buf = _ws(ws, "cw", L.kvs_channel_weights_workspace_size(Hq, Hkv, W, N, d), Q.device)
    _check(L.kvs_channel_weights(_ptr(Q), _ptr(K), Hq, Hkv, W, N, d, _ptr(w_c), _ptr(buf), buf.numel(),
                                 _stream(stream)), "kvs_channel_weights")
    return w_c


def channel_stats(Q, K, keep_bits=None, *, out_wc=None, out_sigma=None, stream=None):
    """(w_c, sigma_c) float32 [Hkv, d] from one read of K: w_c over every token, sigma_c over the kept ones."""
    _bf16(Q, "Q"), _bf16(K, "K")
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    w_c = out_wc if out_wc is not None else torch.empty(Hkv, d, dtype=torch.float32, device=Q.device)
    sc = out_sigma if out_sigma is not None else torch.empty(Hkv, d, dtype=torch.float32, device=Q.device)
    _check(lib().kvs_channel_stats(_ptr(Q), _ptr(K), _ptr(keep_bits), Hq, Hkv, W, N, d, _ptr(w_c), _ptr(sc),
                                   _stream(stream)), "kvs_channel_stats")
    return w_c, sc


def unit_rms(X, axis, keep_bits=None, *, out=None, ws=None, stream=None):
    _bf16(X, "X")
    Hkv, N, d = X.shape
    shape = (Hkv, N) if axis == 0 else (Hkv, d)
    sigma = out if out is not None else torch.empty(shape, dtype=torch.float32, device=X.device)
    L = lib()
    buf = _ws(ws, "rms", L.kvs_unit_rms_workspace_size(Hkv, N, d, axis), X.device)
    _check(L.kvs_unit_rms(_ptr(X), Hkv, N, d, axis, _ptr(keep_bits), _ptr(sigma), _ptr(buf), buf.numel(),
                          _stream(stream)), "kvs_unit_rms")
    return sigma


def allocate_bits(w, sigma, budget_bits, width_mask=WIDTHS_ALL, *, out=None, ws=None, stream=None):
    w = w.reshape(-1)
    sigma = sigma.reshape(-1)
    if w.dtype != torch.float32 or sigma.dtype != torch.float32 or w.numel() != sigma.numel():
        raise KvsError("w and sigma must be float32 of equal length")
    U = w.numel()
    bits = out if out is not None else torch.empty(U, dtype=torch.uint8, device=w.device)
    L = lib()
    buf = _ws(ws, "alloc", L.kvs_allocate_workspace_size(U), w.device)
    _check(L.kvs_allocate_bits(_ptr(w), _ptr(sigma), U, int(budget_bits), width_mask, _ptr(bits), _ptr(buf),
                               buf.numel(), _stream(stream)), "kvs_allocate_bits")
    return bits


def allocate_bits_pools(w, sigma, budget_bits, width_mask=WIDTHS_ALL, *, out=None, ws=None, stream=None):
    """Widths of n_pools independent pools: w, sigma float32 [n_pools, U] (same budget per pool)."""
    if w.dim() != 2 or w.shape != sigma.shape or w.dtype != torch.float32 or sigma.dtype != torch.float32:
        raise KvsError("w and sigma must be float32 [n_pools, U] of equal shape")
    if not (w.is_contiguous() and sigma.is_contiguous()):
        raise KvsError("w and sigma must be contiguous")
    P, U = w.shape
    bits = out if out is not None else torch.empty(P, U, dtype=torch.uint8, device=w.device)
    L = lib()
    buf = _ws(ws, "alloc", L.kvs_allocate_pools_workspace_size(P, U), w.device)
    _check(L.kvs_allocate_bits_pools(_ptr(w), _ptr(sigma), P, U, int(budget_bits), width_mask, _ptr(bits), _ptr(buf),
                                     buf.numel(), _stream(stream)), "kvs_allocate_bits_pools")
    return bits


def allocate_plan_info(U, width_mask=WIDTHS_ALL):
    """(cluster CTAs or 0, grid blocks or 0, grid workspace bytes) of kvs_allocate_bits for U units."""
    info = (c_int64 * 3)()
    _check(lib().kvs_allocate_plan_info(U, width_mask, info), "kvs_allocate_plan_info")
    return tuple(info)


class Streams:
    """Device buffers of a width-grouped stream set (see kvs_stream_set).

    With n_pools > 1 the set holds that many pools of one shape back to back
    (the layout kvs_quantize_pack_pools writes); pool(q) is a one-pool view."""

    def __init__(self, Hkv, N, d, axis, budget_bits, device, n_pools=1):
        cu = (c_int64 * 4)()
        cg = (c_int64 * 4)()
        _check(lib().kvs_pack_capacity(Hkv, N, d, axis, int(budget_bits), cu, cg), "kvs_pack_capacity")
        self.shape, self.axis, self.n_pools = (Hkv, N, d), axis, n_pools
        self.cap_units, self.cap_groups = list(cu), list(cg)
        P = n_pools
        self.codes, self.scales, self.ids, self.goff = [], [], [], []
        for i, wd in enumerate(STREAM_WIDTHS):
            self.codes.append(torch.empty(max(1, P * cg[i] * 8 * wd), dtype=torch.uint8, device=device))
            self.scales.append(torch.empty(max(1, P * cg[i]), dtype=torch.int16, device=device))
            self.ids.append(torch.empty(max(1, P * cu[i]), dtype=torch.int32, device=device))
            self.goff.append(torch.empty(max(1, P * cu[i]), dtype=torch.int64, device=device))
        self.counts = torch.zeros(8 * P, dtype=torch.int64, device=device)
        self.c = self._struct(0)

    def _struct(self, q):
        c = StreamSetC()
        for i, wd in enumerate(STREAM_WIDTHS):
            c.codes[i] = self.codes[i].data_ptr() + q * self.cap_groups[i] * 8 * wd
            c.scales[i] = self.scales[i].data_ptr() + q * self.cap_groups[i] * 2
            c.unit_ids[i] = self.ids[i].data_ptr() + q * self.cap_units[i] * 4
            c.group_offsets[i] = self.goff[i].data_ptr() + q * self.cap_units[i] * 8
            c.cap_units[i] = self.cap_units[i]
            c.cap_groups[i] = self.cap_groups[i]
        c.counts = self.counts.data_ptr() + q * 64
        return c

    def pool(self, q):
        """A one-pool view of pool q (shares the memory)."""
        if not 0 <= q < self.n_pools:
            raise KvsError("pool index out of range")
        v = object.__new__(Streams)
        v.shape, v.axis, v.n_pools = self.shape, self.axis, 1
        v.cap_units, v.cap_groups = self.cap_units, self.cap_groups
        cu, cg = self.cap_units, self.cap_groups
        v.codes = [self.codes[i][q * cg[i] * 8 * wd:(q + 1) * cg[i] * 8 * wd] if cg[i] else self.codes[i][:1]
                   for i, wd in enumerate(STREAM_WIDTHS)]
        v.scales = [self.scales[i][q * cg[i]:(q + 1) * cg[i]] if cg[i] else self.scales[i][:1] for i in range(4)]
        v.ids = [self.ids[i][q * cu[i]:(q + 1) * cu[i]] if cu[i] else self.ids[i][:1] for i in range(4)]
        v.goff = [self.goff[i][q * cu[i]:(q + 1) * cu[i]] if cu[i] else self.goff[i][:1] for i in range(4)]
        v.counts = self.counts[8 * q:8 * q + 8]
        v.c = self._struct(q)
        v._parent = self
        return v

    def host_view(self):
        """Copy the used part of every stream to host numpy arrays (width -> dict)."""
        if self.n_pools != 1:
            raise KvsError("host_view of a pooled set: take pool(q) first")
        counts = self.counts.cpu().tolist()
        out = {}
        for i, wd in enumerate(STREAM_WIDTHS):
            nu, ng = counts[i], counts[4 + i]
            out[wd] = {
                "ids": self.ids[i][:nu].cpu().numpy(),
                "group_offsets": self.goff[i][:nu].cpu().numpy(),
                "n_groups": ng,
                "codes": self.codes[i][:ng * 8 * wd].cpu().numpy(),
                "scales": self.scales[i][:ng].cpu().numpy().view("uint16") if wd != 16 else None,
            }
        return out


def quantize_pack(X, axis, bits, keep_bits, streams: Streams, *, ws=None, stream=None):
    _bf16(X, "X")
    Hkv, N, d = X.shape
    L = lib()
    buf = _ws(ws, "pack%d" % axis, L.kvs_pack_workspace_size(Hkv, N, d, axis), X.device)
    _check(L.kvs_quantize_pack(_ptr(X), Hkv, N, d, axis, _ptr(bits), _ptr(keep_bits), ctypes.byref(streams.c),
                               _ptr(buf), buf.numel(), _stream(stream)), "kvs_quantize_pack")
    return streams


def dequantize(streams: Streams, bits, keep_bits, *, out=None, ws=None, stream=None):
    Hkv, N, d = streams.shape
    axis = streams.axis
    dev = streams.counts.device
    y = out if out is not None else torch.empty(Hkv, N, d, dtype=torch.float32, device=dev)
    L = lib()
    buf = _ws(ws, "deq%d" % axis, L.kvs_pack_workspace_size(Hkv, N, d, axis), dev)
    _check(L.kvs_dequantize(ctypes.byref(streams.c), Hkv, N, d, axis, _ptr(bits), _ptr(keep_bits), _ptr(y),
                            _ptr(buf), buf.numel(), _stream(stream)), "kvs_dequantize")
    return y


def quantize_pack_pools(X, axis, bits, keep_bits, streams: Streams, *, ws=None, stream=None):
    """X bf16 [n_pools, Hkv, N, d]; bits uint8 [n_pools, U]; keep_bits uint8 [n_pools, Hkv*N] (axis 1)."""
    _bf16(X, "X")
    P, Hkv, N, d = X.shape
    if streams.n_pools != P or tuple(streams.shape) != (Hkv, N, d) or streams.axis != axis:
        raise KvsError("stream set does not match X")
    L = lib()
    buf = _ws(ws, "packp%d" % axis, L.kvs_pack_pools_workspace_size(P, Hkv, N, d, axis), X.device)
    _check(L.kvs_quantize_pack_pools(_ptr(X), P, Hkv, N, d, axis, _ptr(bits), _ptr(keep_bits),
                                     ctypes.byref(streams.c), _ptr(buf), buf.numel(), _stream(stream)),
           "kvs_quantize_pack_pools")
    return streams


def dequantize_pools(streams: Streams, bits, keep_bits, *, out=None, ws=None, stream=None):
    """float32 [n_pools, Hkv, N, d] from a pooled stream set."""
    Hkv, N, d = streams.shape
    P, axis = streams.n_pools, streams.axis
    dev = streams.counts.device
    y = out if out is not None else torch.empty(P, Hkv, N, d, dtype=torch.float32, device=dev)
    L = lib()
    buf = _ws(ws, "deqp%d" % axis, L.kvs_pack_pools_workspace_size(P, Hkv, N, d, axis), dev)
    _check(L.kvs_dequantize_pools(ctypes.byref(streams.c), P, Hkv, N, d, axis, _ptr(bits), _ptr(keep_bits), _ptr(y),
                                  _ptr(buf), buf.numel(), _stream(stream)), "kvs_dequantize_pools")
    return y


def threshold_keep(score, tau, window=128, keep_width=16, *, out=None, stream=None):
    """uint8 widths [Hkv, N]: keep_width where score >= tau or in the last `window` positions, else 0."""
    if score.dtype != torch.float32 or not score.is_cuda or not score.is_contiguous() or score.dim() != 2:
        raise KvsError("score must be a contiguous float32 CUDA tensor [Hkv, N]")
    Hkv, N = score.shape
    bits = out if out is not None else torch.empty(Hkv, N, dtype=torch.uint8, device=score.device)
    _check(lib().kvs_threshold_keep(_ptr(score), Hkv, N, float(tau), int(window), int(keep_width), _ptr(bits),
                                    _stream(stream)), "kvs_threshold_keep")
    return bits


def trizone_index(k_streams: Streams, v_streams: Streams, bits_v, *, out=None, stream=None):
    """The decode lookup of one compressed pool (uint8 device buffer, opaque)."""
    Hkv, N, d = v_streams.shape
    L = lib()
    n = L.kvs_trizone_index_size(Hkv, N)
    idx = out if out is not None else torch.empty(n, dtype=torch.uint8, device=v_streams.counts.device)
    _check(L.kvs_trizone_index(ctypes.byref(k_streams.c), ctypes.byref(v_streams.c), _ptr(bits_v), Hkv, N, d,
                               _ptr(idx), idx.numel(), _stream(stream)), "kvs_trizone_index")
    return idx


def trizone_decode(q, k_streams: Streams, v_streams: Streams, index, k_new=None, v_new=None, n_new=None, *,
                   out=None, lse=None, ws=None, stream=None):
    """One decode step over the compressed pool plus zone C rows: (out [Hq, d] fp32, lse [Hq] fp32).

    k_new, v_new: bf16 [Hkv, nc_cap, d] or None; n_new: device int32 [1] (valid rows)."""
    _bf16(q, "q")
    Hq, d = q.shape
    Hkv, N, _ = v_streams.shape
    nc_cap = 0
    if k_new is not None:
        _bf16(k_new, "k_new")
        _bf16(v_new, "v_new")
        nc_cap = k_new.shape[1]
        if n_new is None or n_new.dtype != torch.int32 or not n_new.is_cuda:
            raise KvsError("n_new must be an int32 CUDA tensor when zone C rows are given")
    L = lib()
    o = out if out is not None else torch.empty(Hq, d, dtype=torch.float32, device=q.device)
    ls = lse if lse is not None else torch.empty(Hq, dtype=torch.float32, device=q.device)
    buf = _ws(ws, "trizone", L.kvs_trizone_workspace_size(Hq, Hkv, N, d, nc_cap), q.device)
    _check(L.kvs_trizone_decode(_ptr(q), Hq, Hkv, N, d, ctypes.byref(k_streams.c), ctypes.byref(v_streams.c),
                                _ptr(index), _ptr(k_new), _ptr(v_new), _ptr(n_new), nc_cap, _ptr(o), _ptr(ls),
                                _ptr(buf), buf.numel(), _stream(stream)), "kvs_trizone_decode")
    return o, ls


def gram(X, keep_bits=None, *, out=None, accumulate=False, ws=None, stream=None):
    """G [Hkv, d, d] float32: sum over tokens of x x^T per KV head (added to `out` when accumulate)."""
    _bf16(X, "X")
    Hkv, N, d = X.shape
    L = lib()
    G = out if out is not None else torch.zeros(Hkv, d, d, dtype=torch.float32, device=X.device)
    buf = _ws(ws, "gram", L.kvs_gram_workspace_size(Hkv, N, d), X.device)
    _check(L.kvs_gram(_ptr(X), Hkv, N, d, _ptr(keep_bits), 1 if accumulate else 0, _ptr(G), _ptr(buf), buf.numel(),
                      _stream(stream)), "kvs_gram")
    return G


def spectrum(G, rtol=1e-3, *, stream=None):
    """(sigma [Hkv, d] descending, ner [Hkv], rank [Hkv] int32) of the Gram matrices G [Hkv, d, d]."""
    if G.dtype != torch.float32 or not G.is_cuda or not G.is_contiguous() or G.dim() != 3:
        raise KvsError("G must be a contiguous float32 CUDA tensor [Hkv, d, d]")
    Hkv, d, _ = G.shape
    sigma = torch.empty(Hkv, d, dtype=torch.float32, device=G.device)
    ner = torch.empty(Hkv, dtype=torch.float32, device=G.device)
    rank = torch.empty(Hkv, dtype=torch.int32, device=G.device)
    _check(lib().kvs_spectrum(_ptr(G), Hkv, d, float(rtol), _ptr(sigma), _ptr(ner), _ptr(rank), _stream(stream)),
           "kvs_spectrum")
    return sigma, ner, rank


def block_lse(Q, K, n_block, *, q_pos0=None, out=None, ws=None, stream=None):
    """Row LSE over keys [0, n_block) of each KV head: float [Hq, W]."""
    _bf16(Q, "Q")
    _bf16(K, "K")
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    if q_pos0 is None:
        q_pos0 = N - W
    L = lib()
    lse = out if out is not None else torch.empty(Hq, W, dtype=torch.float32, device=Q.device)
    n = L.kvs_block_lse_workspace_size(Hq, Hkv, W, N, d, q_pos0, n_block)
    buf = _ws(ws, "block_lse", n, Q.device)
    _check(L.kvs_block_lse(_ptr(Q), _ptr(K), Hq, Hkv, W, N, d, q_pos0, n_block, _ptr(lse), _ptr(buf), buf.numel(),
                           _stream(stream)), "kvs_block_lse")
    return lse


def block_attention(Q, K, V, n_block, *, q_pos0=None, want_lse=True, out=None, stream=None):
    """(Y [Hq, W, d], lse [Hq, W] or None) float32: attention of the window
    queries over keys [0, n_block) of each KV head (causal inside the block)."""
    _bf16(Q, "Q"), _bf16(K, "K"), _bf16(V, "V")
    Hq, W, d = Q.shape
    Hkv, N, _ = K.shape
    if tuple(V.shape) != tuple(K.shape):
        raise KvsError("V must have K's shape")
    if q_pos0 is None:
        q_pos0 = N - W
    Y = out if out is not None else torch.empty(Hq, W, d, dtype=torch.float32, device=Q.device)
    lse = torch.empty(Hq, W, dtype=torch.float32, device=Q.device) if want_lse else None
    _check(lib().kvs_block_attention(_ptr(Q), _ptr(K), _ptr(V), Hq, Hkv, W, N, d, q_pos0, n_block, _ptr(Y), _ptr(lse),
                                     _stream(stream)), "kvs_block_attention")
    return Y, lse


def ridge_values(Qt, Kc, Y, lam, *, out=None, ws=None, stream=None):
    """Vc [Hkv, k, d] float32 = (A^T A + lam I)^-1 A^T Y per KV head, with
    A = softmax(Qt Kc^T / sqrt(d)); Qt bf16 [Hkv, R, d], Kc bf16 [Hkv, k, d],
    Y float32 [Hkv, R, d]."""
    _bf16(Qt, "Qt"), _bf16(Kc, "Kc")
    if Y.dtype != torch.float32 or not Y.is_cuda or not Y.is_contiguous():
        raise KvsError("Y must be a contiguous float32 CUDA tensor")
    Hkv, R, d = Qt.shape
    k = Kc.shape[1]
    if tuple(Kc.shape) != (Hkv, k, d) or tuple(Y.shape) != (Hkv, R, d):
        raise KvsError("Qt [Hkv, R, d], Kc [Hkv, k, d] and Y [Hkv, R, d] must agree")
    L = lib()
    Vc = out if out is not None else torch.empty(Hkv, k, d, dtype=torch.float32, device=Qt.device)
    buf = _ws(ws, "ridge", L.kvs_ridge_values_workspace_size(Hkv, R, k, d), Qt.device)
    _check(L.kvs_ridge_values(_ptr(Qt), _ptr(Kc), _ptr(Y), Hkv, R, k, d, float(lam), _ptr(Vc), _ptr(buf), buf.numel(),
                              _stream(stream)), "kvs_ridge_values")
    return Vc
