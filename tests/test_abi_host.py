"""Host-only checks of the C ABI (no GPU needed): the library loads, exports
every entry point that include/smoe.h declares, and rejects bad arguments on
the host before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smoe.h")


@pytest.fixture(scope="module")
def lib():
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe
    return smoe


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(smoe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("smoe_route_topk", "smoe_expert_union", "smoe_moe_decode", "smoe_moe_prefill_chunk",
              "smoe_workspace_bytes", "smoe_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in declared_functions():
        assert hasattr(so, n), n
    assert set(declared_functions()) <= set(lib.EXPORTED) | {"smoe_status_string"}


def _layer(lib, D=2048, E=128, K=8, F=768, ptr=1 << 20):
    s = lib.smoe_layer()
    s.d_model, s.n_experts, s.top_k, s.ffn_dim, s.group_size, s.norm_topk_prob = D, E, K, F, 64, 1
    s.rms_eps = 1e-6
    for n in ("router_w", "gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q",
              "down_s", "down_b"):
        setattr(s, n, ptr)
    return s


def test_workspace_bytes_and_shape_checks(lib):
    so = lib._lib
    s = _layer(lib)
    n1 = so.smoe_workspace_bytes(ctypes.byref(s), 1)
    n64 = so.smoe_workspace_bytes(ctypes.byref(s), 64)
    assert 0 < n1 < n64 and n64 % 256 == 0
    assert so.smoe_workspace_bytes(ctypes.byref(s), 65) == 0
    assert so.smoe_workspace_bytes(ctypes.byref(s), 0) == 0
    for bad in (dict(D=2000), dict(F=700), dict(K=0), dict(K=17), dict(E=300), dict(E=4, K=8),
                dict(D=16384), dict(F=4096, K=8)):
        assert so.smoe_workspace_bytes(ctypes.byref(_layer(lib, **bad)), 1) == 0, bad
    g = _layer(lib)
    g.group_size = 32
    assert so.smoe_workspace_bytes(ctypes.byref(g), 1) == 0
    assert so.smoe_workspace_bytes(None, 1) == 0


def test_entry_points_reject_bad_arguments_on_host(lib):
    so = lib._lib
    s = _layer(lib)
    ref = ctypes.byref(s)
    ws = ctypes.c_void_p(1 << 24)
    n = so.smoe_workspace_bytes(ref, 64)
    P = ctypes.c_void_p
    # NULL layer / NULL tensors
    assert so.smoe_moe_decode(None, P(4096), P(8192), None, None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_decode(ref, None, P(8192), None, None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    # misaligned hidden state
    assert so.smoe_moe_decode(ref, P(4098), P(8192), None, None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    # workspace too small / missing / misaligned
    assert so.smoe_moe_decode(ref, P(4096), P(8192), None, None, None, ws, 16, None) == lib.SMOE_ERR_WORKSPACE
    assert so.smoe_moe_decode(ref, P(4096), P(8192), None, None, None, None, n, None) == lib.SMOE_ERR_WORKSPACE
    assert so.smoe_moe_decode(ref, P(4096), P(8192), None, None, None, P((1 << 24) + 8), n, None) == lib.SMOE_ERR_WORKSPACE
    # prefill: T out of range, aliasing
    assert so.smoe_moe_prefill_chunk(ref, P(4096), 0, P(8192), None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_prefill_chunk(ref, P(4096), 65, P(8192), None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_prefill_chunk(ref, P(4096), 4, P(4096), None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    # route: T range, NULL outputs
    assert so.smoe_route_topk(ref, P(4096), 65, P(64), P(128), None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_route_topk(ref, P(4096), 1, None, P(128), None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    # union: sizes
    args = [P(64)] * 2
    outs = [P(256)] * 6
    assert so.smoe_expert_union(*args, 65, 8, 128, *outs, None, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_expert_union(*args, 4, 17, 128, *outs, None, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_expert_union(*args, 4, 8, 257, *outs, None, None) == lib.SMOE_ERR_INVALID_ARG
    # unsupported layer shape
    bad = _layer(lib, D=2000)
    assert so.smoe_moe_decode(ctypes.byref(bad), P(4096), P(8192), None, None, None, ws, n, None) == lib.SMOE_ERR_UNSUPPORTED
    # misaligned codes
    mis = _layer(lib)
    mis.gate_q = (1 << 20) + 4
    assert so.smoe_moe_decode(ctypes.byref(mis), P(4096), P(8192), None, None, None, ws, n, None) == lib.SMOE_ERR_INVALID_ARG


def test_decode_layers_rejects_bad_arguments_on_host(lib):
    so = lib._lib
    P = ctypes.c_void_p
    arr = (lib.smoe_layer * 3)(_layer(lib), _layer(lib), _layer(lib))
    LP = ctypes.POINTER(lib.smoe_layer)
    host = ctypes.cast(arr, LP)
    ws = ctypes.c_void_p(1 << 24)
    n = so.smoe_workspace_bytes(ctypes.byref(arr[0]), 1)
    dev_tab = P(1 << 22)
    call = lambda h, d, nl, x=P(4096), y=P(8192), i=None, w=None, wsp=ws, nb=n: \
        so.smoe_moe_decode_layers(h, d, nl, x, y, i, w, wsp, nb, None)
    assert call(host, dev_tab, 0) == lib.SMOE_ERR_INVALID_ARG            # no layers
    assert call(None, dev_tab, 3) == lib.SMOE_ERR_INVALID_ARG            # no host table
    assert call(host, None, 3) == lib.SMOE_ERR_INVALID_ARG               # no device table
    assert call(host, P((1 << 22) + 4), 3) == lib.SMOE_ERR_INVALID_ARG   # misaligned device table
    assert call(host, dev_tab, 3, x=P(4098)) == lib.SMOE_ERR_INVALID_ARG
    assert call(host, dev_tab, 3, i=P(64)) == lib.SMOE_ERR_INVALID_ARG   # ids without weights
    assert call(host, dev_tab, 3, wsp=None) == lib.SMOE_ERR_WORKSPACE
    assert call(host, dev_tab, 3, nb=16) == lib.SMOE_ERR_WORKSPACE
    arr[2].ffn_dim = 1536                                                 # layers of different shapes
    assert call(host, dev_tab, 3) == lib.SMOE_ERR_INVALID_ARG
    arr[2].ffn_dim = 768
    arr[1].rms_gain = 1 << 20                                             # gain on one layer only
    assert call(host, dev_tab, 3) == lib.SMOE_ERR_INVALID_ARG
    arr[1].rms_gain = None
    arr[1].d_model = 2000                                                 # unsupported layer
    assert call(host, dev_tab, 3) == lib.SMOE_ERR_UNSUPPORTED


def test_dense_matvec_and_quantiser_reject_bad_arguments_on_host(lib):
    so = lib._lib
    P = ctypes.c_void_p
    W, X, Y = P(1 << 20), P(1 << 21), P(1 << 22)
    mv = lambda w=W, x=X, rows=512, cols=4096, y=Y: so.smoe_dense_matvec(w, x, rows, cols, y, None)
    assert mv(w=None) == lib.SMOE_ERR_INVALID_ARG
    assert mv(y=None) == lib.SMOE_ERR_INVALID_ARG
    assert mv(rows=0) == lib.SMOE_ERR_INVALID_ARG
    assert mv(cols=4100) == lib.SMOE_ERR_UNSUPPORTED                      # not a multiple of 8
    assert mv(cols=16384) == lib.SMOE_ERR_UNSUPPORTED                     # beyond 8192
    assert mv(w=P((1 << 20) + 8)) == lib.SMOE_ERR_INVALID_ARG             # w not 16-byte aligned
    assert mv(x=P((1 << 21) + 2)) == lib.SMOE_ERR_INVALID_ARG
    assert mv(y=P((1 << 22) + 2)) == lib.SMOE_ERR_INVALID_ARG
    C, S, B = P(1 << 23), P(1 << 24), P(1 << 25)
    qz = lambda w=W, rows=768, cols=2048, c=C, s=S, b=B: so.smoe_quantize_q4(w, rows, cols, c, s, b, None)
    assert qz(c=None) == lib.SMOE_ERR_INVALID_ARG
    assert qz(rows=0) == lib.SMOE_ERR_INVALID_ARG
    assert qz(cols=2000) == lib.SMOE_ERR_UNSUPPORTED                      # not whole groups of 64
    assert qz(w=P((1 << 20) + 2)) == lib.SMOE_ERR_INVALID_ARG
    assert qz(c=P((1 << 23) + 8)) == lib.SMOE_ERR_INVALID_ARG              # codes not 16-byte aligned
    assert qz(s=P((1 << 24) + 1)) == lib.SMOE_ERR_INVALID_ARG
    q2 = lambda cols=2048, c=C: so.smoe_quantize_q2(W, 768, cols, c, S, B, None)
    assert q2(cols=96) == lib.SMOE_ERR_UNSUPPORTED
    assert q2(c=P((1 << 23) + 4)) == lib.SMOE_ERR_INVALID_ARG
    assert q2(c=None) == lib.SMOE_ERR_INVALID_ARG


def test_layer_code_bits_checked_on_host(lib):
    so = lib._lib
    P = ctypes.c_void_p
    ws = P(1 << 24)
    for bits, want in ((3, lib.SMOE_ERR_UNSUPPORTED), (8, lib.SMOE_ERR_UNSUPPORTED)):
        L = _layer(lib)
        L.code_bits = bits
        assert so.smoe_workspace_bytes(ctypes.byref(L), 1) == 0
        assert so.smoe_moe_decode(ctypes.byref(L), P(4096), P(8192), None, None, None, ws, 1 << 30, None) == want


def test_status_strings(lib):
    for code in range(-6, 1):
        assert lib.smoe_status_string(code).startswith("SMOE_")
    assert "unknown" in lib.smoe_status_string(7)


def test_binding_refuses_host_tensors(lib):
    """The Python binding hands the library device pointers only: a host tensor
    is refused before any call (its address would reach a kernel)."""
    import torch
    with pytest.raises(ValueError, match="device tensors"):
        lib.smoe_dense_matvec(torch.zeros((4, 8), dtype=torch.bfloat16),
                              torch.zeros(8, dtype=torch.bfloat16), torch.zeros(4))
    with pytest.raises(ValueError, match="device tensors"):
        lib.smoe_workspace_init(torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="device tensors"):
        lib._p(torch.zeros(1))
    assert lib._p(None) is None


def test_ffn_decode_and_noalloc_reject_bad_arguments_on_host(lib):
    so = lib._lib
    P = ctypes.c_void_p
    s = _layer(lib)
    ref = ctypes.byref(s)
    ws = ctypes.c_void_p(1 << 24)
    n = so.smoe_workspace_bytes(ref, 1)
    ffn = lambda x=P(4096), idx=P(64), w=P(128), y=P(8192), eo=None, wsp=ws, nb=n, layer=ref: \
        so.smoe_moe_ffn_decode(layer, x, idx, w, y, eo, wsp, nb, None)
    assert ffn(idx=None) == lib.SMOE_ERR_INVALID_ARG          # ids are required
    assert ffn(w=None) == lib.SMOE_ERR_INVALID_ARG            # and their weights
    assert ffn(y=P(8194)) == lib.SMOE_ERR_INVALID_ARG         # misaligned output
    assert ffn(eo=P(4098)) == lib.SMOE_ERR_INVALID_ARG        # misaligned expert outputs
    assert ffn(nb=16) == lib.SMOE_ERR_WORKSPACE
    assert ffn(layer=None) == lib.SMOE_ERR_INVALID_ARG
    nd = so.smoe_moe_decode_noalloc
    assert nd(None, P(4096), P(8192), None, None, None) == lib.SMOE_ERR_INVALID_ARG
    bad = _layer(lib, D=2000)
    assert nd(ctypes.byref(bad), P(4096), P(8192), None, None, None) == lib.SMOE_ERR_UNSUPPORTED
    big = _layer(lib, D=8192)
    big.ffn_dim = 2048
    assert so.smoe_workspace_bytes(ctypes.byref(big), 1) > lib.SMOE_DECODE_NOALLOC_MAX_BYTES
    assert nd(ctypes.byref(big), P(4096), P(8192), None, None, None) == lib.SMOE_ERR_WORKSPACE


def test_prefill_experts_and_status_calls_reject_bad_arguments_on_host(lib):
    so = lib._lib
    s = _layer(lib)
    ref = ctypes.byref(s)
    ws = ctypes.c_void_p(1 << 24)
    n = so.smoe_workspace_bytes(ref, 64)
    P = ctypes.c_void_p
    # the expert outputs are what this entry point is for: NULL or misaligned is refused
    assert so.smoe_moe_prefill_chunk_experts(ref, P(4096), 4, P(8192), None, None, None, ws, n,
                                             None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_prefill_chunk_experts(ref, P(4096), 4, P(8192), None, None, P(1 << 20 | 4),
                                             ws, n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_prefill_chunk_experts(ref, P(4096), 65, P(8192), None, None, P(1 << 20), ws,
                                             n, None) == lib.SMOE_ERR_INVALID_ARG
    assert so.smoe_moe_decode_noalloc_status(None, None) == lib.SMOE_ERR_INVALID_ARG


def test_grid_wait_limit_round_trip(lib):
    """The grid-barrier wait limit is plain host state: default 200 ms, set and
    read back, restored."""
    default = lib.smoe_get_grid_wait_limit()
    assert default == 200_000_000
    try:
        for v in (0, 1, 5_000_000, 2 ** 63):
            lib.smoe_set_grid_wait_limit(v)
            assert lib.smoe_get_grid_wait_limit() == v
    finally:
        lib.smoe_set_grid_wait_limit(default)
    assert lib.smoe_get_grid_wait_limit() == default
