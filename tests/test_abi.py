"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from kv_cache_compression_flash_b300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return L.lib()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"binding lacks {n}"


def test_status_strings_and_version(lib):
    assert lib.kvs_version() == 101
    for code, name in L.STATUS.items():
        assert lib.kvs_status_string(code).decode() == name


def _score(lib, **kw):
    a = dict(Q=1 << 20, K=1 << 20, V=None, h=None, W_O=None, Hq=8, Hkv=2, W=16, N=64, d=128, D=0, q_pos0=48,
             mode=L.MODE_LSE | L.MODE_RDKV_WT, lse=1 << 20, w_t=1 << 20, s_plus=None, ws=1 << 20, wsb=1 << 30)
    a.update(kw)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kvs_score_attention(v(a["Q"]), v(a["K"]), v(a["V"]), v(a["h"]), v(a["W_O"]), a["Hq"], a["Hkv"],
                                   a["W"], a["N"], a["d"], a["D"], a["q_pos0"], a["mode"], v(a["lse"]),
                                   v(a["w_t"]), v(a["s_plus"]), v(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=None), 1), (dict(lse=None), 1), (dict(w_t=None), 1),
    (dict(Hq=7), 1), (dict(q_pos0=49), 1), (dict(q_pos0=-1), 1), (dict(N=0), 1), (dict(W=0), 1),
    (dict(d=96), 2), (dict(Hq=12, Hkv=2), 2), (dict(Hq=6, Hkv=2), 2),    # G = 6, G = 3
    (dict(mode=L.MODE_LSE | L.MODE_KVZIP | L.MODE_KVZIP_PLUS, s_plus=1 << 20), 1),
    (dict(mode=L.MODE_LSE | L.MODE_KVZIP_PLUS, s_plus=1 << 20, D=64), 1),   # V, h, W_O missing
    (dict(mode=1 << 9), 1),
    (dict(Q=(1 << 20) + 2), 1),                                             # TMA needs 16-byte alignment
    (dict(wsb=16), 6), (dict(ws=(1 << 20) + 64), 6),
])
def test_score_argument_errors(lib, kw, code):
    assert _score(lib, **kw) == code


def test_workspace_sizes_and_plan(lib):
    assert lib.kvs_score_workspace_size(32, 8, 512, 8192, 128, 0, 7680, 3) > 0
    assert lib.kvs_score_workspace_size(32, 8, 512, 8192, 96, 0, 7680, 3) == 0
    info = L.score_plan_info(32, 8, 512, 8192, 128)
    assert info[0] >= 4 and info[1] >= 1 and info[2] >= 4 and info[3] >= 1 and info[4] >= 3
    assert lib.kvs_allocate_workspace_size(1000) > 0
    assert lib.kvs_allocate_pools_workspace_size(16, 131072) >= lib.kvs_allocate_workspace_size(131072)
    assert lib.kvs_allocate_pools_workspace_size(1, 1000) == lib.kvs_allocate_workspace_size(1000)
    assert lib.kvs_pack_workspace_size(8, 8192, 128, 0) > 0          # token units need no scratch
    assert lib.kvs_pack_workspace_size(8, 8192, 128, 1) >= 8 * 8192 * 4  # kept-token index per head


def test_pack_capacity(lib):
    cu, cg = (ctypes.c_int64 * 4)(), (ctypes.c_int64 * 4)()
    assert lib.kvs_pack_capacity(8, 8192, 128, 0, 3 * 65536, cu, cg) == 0
    assert list(cu) == [65536, 49152, 24576, 12288]
    assert list(cg) == [2 * x for x in cu]
    assert lib.kvs_pack_capacity(8, 8192, 128, 1, 3 * 1024, cu, cg) == 0
    assert list(cu) == [1024, 768, 384, 192]
    assert list(cg) == [x * 128 for x in cu]
    assert lib.kvs_pack_capacity(8, 8192, 96, 0, 10, cu, cg) == 2


def test_alloc_and_pack_argument_errors(lib):
    p = ctypes.c_void_p(1 << 20)
    assert lib.kvs_allocate_bits(p, p, 10, -1, L.WIDTHS_ALL, p, p, 1 << 20, None) == 1
    assert lib.kvs_allocate_bits(p, p, 10, 5, 1 << 3, p, p, 1 << 20, None) == 1       # width 3 is not a width
    assert lib.kvs_allocate_bits(None, p, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None) == 1
    assert lib.kvs_allocate_bits(p, p, 0, 5, L.WIDTHS_ALL, p, p, 1 << 20, None) == 0  # nothing to do
    s = L.StreamSetC()
    assert lib.kvs_quantize_pack(p, 8, 64, 128, 0, p, None, ctypes.byref(s), p, 1 << 20, None) == 1  # no counts
    assert lib.kvs_quantize_pack(p, 8, 64, 128, 2, p, None, ctypes.byref(s), p, 1 << 20, None) == 1  # bad axis
    assert lib.kvs_quantize_pack(p, 8, 64, 96, 0, p, None, ctypes.byref(s), p, 1 << 20, None) == 2
    assert lib.kvs_unit_rms(p, 8, 64, 128, 3, None, p, p, 1 << 20, None) == 1
    # pooled allocation and packing
    assert lib.kvs_allocate_bits_pools(p, p, -1, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None) == 1
    assert lib.kvs_allocate_bits_pools(p, p, 0, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None) == 0   # no pools
    assert lib.kvs_allocate_bits_pools(p, p, 1 << 16, 10, 5, L.WIDTHS_ALL, p, p, 1 << 20, None) == 2
    assert lib.kvs_quantize_pack_pools(p, 0, 8, 64, 128, 0, p, None, ctypes.byref(s), p, 1 << 20, None) == 1
    assert lib.kvs_quantize_pack_pools(p, 2, 8, 64, 96, 0, p, None, ctypes.byref(s), p, 1 << 20, None) == 2
    assert lib.kvs_dequantize_pools(ctypes.byref(s), 3, 8, 64, 128, 2, p, None, p, p, 1 << 20, None) == 1
    assert lib.kvs_pack_pools_workspace_size(4, 8, 8192, 128, 1) >= 4 * 8 * 8192 * 4     # kept-token index per head
    assert lib.kvs_pack_pools_workspace_size(1, 8, 8192, 128, 1) == lib.kvs_pack_workspace_size(8, 8192, 128, 1)
    assert lib.kvs_pack_pools_workspace_size(1 << 16, 1, 64, 128, 0) == 0
    info = (ctypes.c_int64 * 3)()
    assert lib.kvs_allocate_plan_info(-1, L.WIDTHS_ALL, info) == 1
    assert lib.kvs_allocate_plan_info(10, 1 << 3, info) == 1
    assert lib.kvs_allocate_plan_info(0, L.WIDTHS_ALL, info) == 0 and list(info) == [0, 0, 0]
    assert lib.kvs_channel_weights(p, p, 8, 3, 16, 64, 128, p, p, 1 << 20, None) == 1


def test_pack_rejects_token_capacities_without_room_for_their_groups(lib):
    # token units at d = 128 have two groups each: cap_groups < 2 cap_units is refused before any launch
    p = ctypes.c_void_p(1 << 20)
    s = L.StreamSetC()
    for i in range(4):
        s.codes[i] = s.scales[i] = s.unit_ids[i] = s.group_offsets[i] = 1 << 20
        s.cap_units[i], s.cap_groups[i] = 100, 200
    s.counts = 1 << 20
    s.cap_groups[1] = 199
    assert lib.kvs_quantize_pack(p, 8, 64, 128, 0, p, None, ctypes.byref(s), p, 1 << 20, None) == 1
    assert lib.kvs_dequantize(ctypes.byref(s), 8, 64, 128, 0, p, None, p, p, 1 << 20, None) == 1
    # channel units: a group count per unit depends on the kept tokens, so no such rule
    assert lib.kvs_quantize_pack(p, 8, 64, 128, 1, p, None, ctypes.byref(s), p, 1 << 20, None) == 1  # no keep


def test_trizone_sizes_and_argument_errors(lib):
    # header 8 heads x 16 int64 (1 KiB); per 64-token group the first V entry of
    # each width (8 x 129 x 4 int32, padded to 16640 B); one width byte per token
    assert lib.kvs_trizone_index_size(8, 8192) == 1024 + 16640 + 8 * 8192
    # 32 heads x (128 groups of 64 tokens + 1 zone C step of 128) records: max and
    # sum (16512 B each, padded to 16640) and 128 output floats
    assert lib.kvs_trizone_workspace_size(32, 8, 8192, 128, 100) == 2 * 16640 + 32 * 129 * 128 * 4
    assert lib.kvs_trizone_workspace_size(0, 8, 8192, 128, 0) == 0
    p = ctypes.c_void_p(1 << 20)
    s = L.StreamSetC()
    dec = lib.kvs_trizone_decode
    args = [p, 32, 8, 8192, 128, ctypes.byref(s), ctypes.byref(s), p, None, None, None, 0, p, p, p, 1 << 30, None]
    bad = list(args)
    bad[0] = None                                                       # no queries
    assert dec(*bad) == 1
    bad = list(args)
    bad[2] = 5                                                          # Hq not a multiple of Hkv
    assert dec(*bad) == 1
    bad = list(args)
    bad[4] = 64                                                         # only d = 128
    assert dec(*bad) == 2
    bad = list(args)
    bad[1], bad[2] = 24, 8                                              # G = 3
    assert dec(*bad) == 2
    bad = list(args)
    bad[11] = 10                                                        # zone C rows without buffers
    assert dec(*bad) == 1
    bad = list(args)
    bad[15] = 16                                                        # workspace too small
    assert dec(*bad) == 6
    assert lib.kvs_trizone_index(ctypes.byref(s), ctypes.byref(s), p, 8, 8192, 128, p, 1 << 30, None) == 1  # no counts


def test_core_sizes_and_argument_errors(lib):
    assert lib.kvs_gram_workspace_size(8, 8192, 64) == 0                # d = 128 only
    assert lib.kvs_gram_workspace_size(8, 100, 128) == 1 * 8 * 128 * 128 * 4   # one 128-token range per head
    p = ctypes.c_void_p(1 << 20)
    assert lib.kvs_gram(None, 8, 100, 128, None, 0, p, p, 1 << 30, None) == 1
    assert lib.kvs_gram(p, 8, 100, 64, None, 0, p, p, 1 << 30, None) == 2
    assert lib.kvs_gram(p, 8, 100, 128, None, 0, p, p, 16, None) == 6
    assert lib.kvs_spectrum(p, 8, 128, ctypes.c_float(1.5), p, p, p, None) == 1  # rtol outside [0, 1)
    assert lib.kvs_spectrum(p, 8, 64, ctypes.c_float(1e-3), p, p, p, None) == 2


def test_block_lse_argument_errors(lib):
    assert lib.kvs_block_lse_workspace_size(32, 8, 512, 8192, 128, 7680, 7680) > 0
    assert lib.kvs_block_lse_workspace_size(32, 8, 512, 8192, 128, 7680, 0) == 0          # empty block
    assert lib.kvs_block_lse_workspace_size(32, 8, 512, 8192, 128, 7680, 8193) == 0       # past the cache
    p = ctypes.c_void_p(1 << 20)
    assert lib.kvs_block_lse(p, p, 32, 8, 512, 8192, 128, 7680, 0, p, p, 1 << 30, None) == 1
    assert lib.kvs_block_lse(p, p, 32, 8, 512, 8192, 96, 7680, 100, p, p, 1 << 30, None) == 2
    assert lib.kvs_block_lse(p, p, 32, 8, 512, 8192, 128, 7681, 100, p, p, 1 << 30, None) == 1  # window past N


def test_sculpt_sizes_and_argument_errors(lib):
    # A [Hkv, R, k], then A^T A [2, Hkv, k, k] and A^T Y [2, Hkv, k, d] (partial sums over
    # the two halves of R), fp32, each 256-byte aligned
    assert lib.kvs_ridge_values_workspace_size(8, 2048, 256, 128) == 4 * 8 * (2048 * 256 + 2 * 256 * 256
                                                                             + 2 * 256 * 128)
    assert lib.kvs_ridge_values_workspace_size(1, 3, 5, 64) == 256 + 256 + 4 * 2 * 5 * 64
    assert lib.kvs_ridge_values_workspace_size(8, 2048, 513, 128) == 0     # k above 512
    assert lib.kvs_ridge_values_workspace_size(8, 2048, 256, 96) == 0      # d outside {64, 128}
    assert lib.kvs_ridge_values_workspace_size(8, 0, 256, 128) == 0
    p = ctypes.c_void_p(1 << 20)
    lam = ctypes.c_float(0.1)
    rv = lib.kvs_ridge_values
    assert rv(None, p, p, 8, 2048, 256, 128, lam, p, p, 1 << 30, None) == 1
    assert rv(p, p, p, 8, 2048, 256, 128, ctypes.c_float(0.0), p, p, 1 << 30, None) == 1       # lam must be > 0
    assert rv(p, p, p, 8, 2048, 256, 128, ctypes.c_float(float("inf")), p, p, 1 << 30, None) == 1
    assert rv(p, p, p, 8, 2048, 256, 128, ctypes.c_float(float("nan")), p, p, 1 << 30, None) == 1
    assert rv(p, p, p, 8, 2048, 600, 128, lam, p, p, 1 << 30, None) == 2
    assert rv(p, p, p, 8, 2048, 256, 96, lam, p, p, 1 << 30, None) == 2
    assert rv(p, p, p, 8, 2048, 256, 128, lam, p, p, 1024, None) == 6                         # workspace too small
    assert rv(p, p, p, 8, 2048, 256, 128, lam, p, ctypes.c_void_p((1 << 20) + 16), 1 << 30, None) == 6  # misaligned
    assert rv(ctypes.c_void_p((1 << 20) + 2), p, p, 8, 2048, 256, 128, lam, p, p, 1 << 30, None) == 1
    ba = lib.kvs_block_attention
    assert ba(p, p, p, 32, 8, 512, 8192, 128, 7680, 0, p, None, None) == 1        # empty block
    assert ba(p, p, p, 32, 8, 512, 8192, 128, 7680, 8193, p, None, None) == 1     # past the cache
    assert ba(p, p, None, 32, 8, 512, 8192, 128, 7680, 100, p, None, None) == 1   # no V
    assert ba(p, p, p, 32, 8, 512, 8192, 128, 7680, 100, None, None, None) == 1   # no Y
    assert ba(p, p, p, 32, 8, 512, 8192, 96, 7680, 100, p, None, None) == 2
    assert ba(p, p, p, 32, 8, 512, 8192, 128, 7681, 100, p, None, None) == 1      # window past N
