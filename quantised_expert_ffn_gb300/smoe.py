"""Thin ctypes binding of libsmoe.so (the C ABI in include/smoe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch tensors already on the GPU; their data pointers
and the current CUDA stream are handed to the C entry points of the same
names.  There is no fallback: if libsmoe.so is missing or fails to load, the
import of this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmoe.so")

SMOE_OK = 0
SMOE_ERR_INVALID_ARG = -1
SMOE_ERR_UNSUPPORTED = -2
SMOE_ERR_WORKSPACE = -3
SMOE_ERR_CUDA = -4
SMOE_ERR_TIMEOUT = -5
SMOE_ERR_DEVICE = -6
SMOE_ERR_RANGE = -7


class SmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = f" [{smoe_last_cuda_error()}]" if status == SMOE_ERR_CUDA else ""
        super().__init__(f"{where}: {smoe_status_string(status)} ({status}){extra}")


class smoe_layer(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int),
        ("n_experts", ctypes.c_int),
        ("top_k", ctypes.c_int),
        ("ffn_dim", ctypes.c_int),
        ("group_size", ctypes.c_int),
        ("norm_topk_prob", ctypes.c_int),
        ("rms_eps", ctypes.c_float),
        ("rms_gain", ctypes.c_void_p),
        ("router_w", ctypes.c_void_p),
        ("gate_q", ctypes.c_void_p),
        ("gate_s", ctypes.c_void_p),
        ("gate_b", ctypes.c_void_p),
        ("up_q", ctypes.c_void_p),
        ("up_s", ctypes.c_void_p),
        ("up_b", ctypes.c_void_p),
        ("down_q", ctypes.c_void_p),
        ("down_s", ctypes.c_void_p),
        ("down_b", ctypes.c_void_p),
        ("code_bits", ctypes.c_int),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsmoe.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    LP = ctypes.POINTER(smoe_layer)
    sig = {
        "smoe_workspace_bytes": (Z, [LP, I]),
        "smoe_workspace_init": (I, [P, Z, P]),
        "smoe_read_device_status": (I, [P, ctypes.POINTER(ctypes.c_int32), P]),
        "smoe_route_topk": (I, [LP, P, I, P, P, P, P, P, Z, P]),
        "smoe_expert_union": (I, [P, P, I, I, I, P, P, P, P, P, P, P, P]),
        "smoe_moe_decode": (I, [LP, P, P, P, P, P, P, Z, P]),
        "smoe_moe_ffn_decode": (I, [LP, P, P, P, P, P, P, Z, P]),
        "smoe_moe_prefill_chunk": (I, [LP, P, I, P, P, P, P, Z, P]),
        "smoe_moe_prefill_chunk_experts": (I, [LP, P, I, P, P, P, P, P, Z, P]),
        "smoe_status_string": (ctypes.c_char_p, [I]),
        "smoe_moe_decode_noalloc": (I, [LP, P, P, P, P, P]),
        "smoe_moe_decode_noalloc_status": (I, [ctypes.POINTER(ctypes.c_int32), P]),
        "smoe_moe_decode_layers": (I, [LP, P, I, P, P, P, P, P, Z, P]),
        "smoe_last_cuda_error": (ctypes.c_char_p, []),
        "smoe_dense_matvec": (I, [P, P, I, I, P, P]),
        "smoe_quantize_q4": (I, [P, I, I, P, P, P, P]),
        "smoe_quantize_q2": (I, [P, I, I, P, P, P, P]),
        "smoe_set_grid_wait_limit": (I, [ctypes.c_ulonglong]),
        "smoe_get_grid_wait_limit": (ctypes.c_ulonglong, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("smoe_workspace_bytes", "smoe_workspace_init", "smoe_read_device_status",
            "smoe_route_topk", "smoe_expert_union", "smoe_moe_decode", "smoe_moe_ffn_decode",
            "smoe_moe_prefill_chunk", "smoe_moe_prefill_chunk_experts", "smoe_status_string", "smoe_moe_decode_noalloc",
            "smoe_moe_decode_noalloc_status",
            "smoe_last_cuda_error", "smoe_moe_decode_layers", "smoe_dense_matvec", "smoe_quantize_q4",
            "smoe_quantize_q2", "smoe_set_grid_wait_limit", "smoe_get_grid_wait_limit")


def _dev_ptr(t: torch.Tensor, what: str = "tensor") -> int:
    """Address of a contiguous CUDA tensor.  A host tensor is refused here: its
    address would reach the kernels as a device pointer."""
    if not t.is_cuda:
        raise ValueError(f"libsmoe takes device tensors; {what} is on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"libsmoe takes contiguous (row-major) tensors; {what} is not")
    return t.data_ptr()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(_dev_ptr(t))


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != SMOE_OK:
        raise SmoeError(status, where)


def smoe_last_cuda_error() -> str:
    return _lib.smoe_last_cuda_error().decode()


def smoe_set_grid_wait_limit(limit_ns: int):
    """Limit (ns) of each grid-barrier wait of the one-kernel decode, process-wide."""
    _check(_lib.smoe_set_grid_wait_limit(int(limit_ns)), "smoe_set_grid_wait_limit")


def smoe_get_grid_wait_limit() -> int:
    return int(_lib.smoe_get_grid_wait_limit())


def smoe_status_string(status: int) -> str:
    return _lib.smoe_status_string(int(status)).decode()


class Layer:
    """A smoe_layer over device tensors (keeps the tensors alive).

    `w` is any object with the attributes of synth.LayerWeights."""

    def __init__(self, w):
        self.w = w
        self._keep = w.tensors()
        s = smoe_layer()
        s.d_model, s.n_experts, s.top_k, s.ffn_dim = w.d_model, w.n_experts, w.top_k, w.ffn_dim
        s.group_size = 64
        s.norm_topk_prob = int(bool(w.norm_topk_prob))
        s.rms_eps = float(w.rms_eps)
        s.rms_gain = None if w.rms_gain is None else _dev_ptr(w.rms_gain, "rms_gain")
        s.code_bits = int(getattr(w, "code_bits", 4))
        for n in ("router_w", "gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q",
                  "down_s", "down_b"):
            setattr(s, n, _dev_ptr(getattr(w, n), n))
        self.s = s
        self.ref = ctypes.byref(s)


def smoe_workspace_bytes(layer: Layer, max_tokens: int) -> int:
    return int(_lib.smoe_workspace_bytes(layer.ref, int(max_tokens)))


def workspace(layer: Layer, max_tokens: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace tensor for `layer` (torch owns the memory)."""
    n = smoe_workspace_bytes(layer, max_tokens)
    if n == 0:
        raise SmoeError(SMOE_ERR_UNSUPPORTED, "smoe_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def smoe_workspace_init(ws: torch.Tensor, stream=None):
    _check(_lib.smoe_workspace_init(_p(ws), ws.numel(), _stream(stream)), "smoe_workspace_init")


def smoe_read_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(_lib.smoe_read_device_status(_p(ws), ctypes.byref(out), _stream(stream)),
           "smoe_read_device_status")
    return int(out.value)


def smoe_route_topk(layer: Layer, x, T, idx, w, logits=None, xn=None, ws=None, stream=None):
    _check(_lib.smoe_route_topk(layer.ref, _p(x), int(T), _p(idx), _p(w), _p(logits), _p(xn),
                                _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "smoe_route_topk")


def smoe_expert_union(idx, w, T, k, E, union_ids, n_union, offsets, bucket_tok, bucket_rank,
                      bucket_w, status_dev=None, stream=None):
    _check(_lib.smoe_expert_union(_p(idx), _p(w), int(T), int(k), int(E), _p(union_ids),
                                  _p(n_union), _p(offsets), _p(bucket_tok), _p(bucket_rank),
                                  _p(bucket_w), _p(status_dev), _stream(stream)),
           "smoe_expert_union")


def smoe_moe_decode(layer: Layer, x, y, idx_out=None, w_out=None, expert_out=None, ws=None,
                    stream=None):
    _check(_lib.smoe_moe_decode(layer.ref, _p(x), _p(y), _p(idx_out), _p(w_out), _p(expert_out),
                                _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "smoe_moe_decode")


def smoe_moe_ffn_decode(layer: Layer, x, idx, w, y, expert_out=None, ws=None, stream=None):
    _check(_lib.smoe_moe_ffn_decode(layer.ref, _p(x), _p(idx), _p(w), _p(y), _p(expert_out),
                                    _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "smoe_moe_ffn_decode")


def smoe_moe_prefill_chunk(layer: Layer, x, T, y, idx_out=None, w_out=None, ws=None, stream=None):
    _check(_lib.smoe_moe_prefill_chunk(layer.ref, _p(x), int(T), _p(y), _p(idx_out), _p(w_out),
                                       _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "smoe_moe_prefill_chunk")


def smoe_moe_prefill_chunk_experts(layer: Layer, x, T, y, expert_out, idx_out=None, w_out=None,
                                   ws=None, stream=None):
    """smoe_moe_prefill_chunk plus the unweighted expert outputs, fp32 [T, k, D]."""
    _check(_lib.smoe_moe_prefill_chunk_experts(layer.ref, _p(x), int(T), _p(y), _p(idx_out), _p(w_out),
                                               _p(expert_out), _p(ws), 0 if ws is None else ws.numel(),
                                               _stream(stream)),
           "smoe_moe_prefill_chunk_experts")


def smoe_dense_matvec(w, x, y, stream=None):
    """y = w @ x: w bf16 [rows, cols], x bf16 [cols], y fp32 [rows] (device tensors)."""
    rows, cols = w.shape
    _check(_lib.smoe_dense_matvec(_p(w), _p(x), int(rows), int(cols), _p(y), _stream(stream)),
           "smoe_dense_matvec")


def smoe_quantize_q4(w, codes, scale, bias, stream=None):
    """SMOE-Q4 of bf16 weights w [..., cols]: codes uint8 [..., cols/2], scale and
    bias bf16 [..., cols/64] (device tensors; leading dimensions flattened into rows)."""
    cols = w.shape[-1]
    rows = w.numel() // cols
    _check(_lib.smoe_quantize_q4(_p(w), int(rows), int(cols), _p(codes), _p(scale), _p(bias),
                                 _stream(stream)),
           "smoe_quantize_q4")


def smoe_quantize_q2(w, codes, scale, bias, stream=None):
    """SMOE-Q2 of bf16 weights w [..., cols]: codes uint8 [..., cols/4], scale and
    bias bf16 [..., cols/64]."""
    cols = w.shape[-1]
    rows = w.numel() // cols
    _check(_lib.smoe_quantize_q2(_p(w), int(rows), int(cols), _p(codes), _p(scale), _p(bias),
                                 _stream(stream)),
           "smoe_quantize_q2")


SMOE_DECODE_NOALLOC_MAX_BYTES = 512 * 1024


def smoe_moe_decode_noalloc(layer: Layer, x, y, idx_out=None, w_out=None, stream=None):
    """Decode one token with the library's fixed device scratch instead of a
    workspace (for callers that cannot allocate device memory, e.g. latency-bound
    serving loops or plug-ins whose host owns the device memory); see include/smoe.h."""
    _check(_lib.smoe_moe_decode_noalloc(layer.ref, _p(x), _p(y), _p(idx_out), _p(w_out),
                                        _stream(stream)), "smoe_moe_decode_noalloc")


def smoe_moe_decode_noalloc_status(stream=None) -> int:
    """Status word the last smoe_moe_decode_noalloc call on this device left
    (0 or a negative smoe status); synchronises the stream."""
    out = ctypes.c_int32(0)
    _check(_lib.smoe_moe_decode_noalloc_status(ctypes.byref(out), _stream(stream)),
           "smoe_moe_decode_noalloc_status")
    return int(out.value)


class LayerTable:
    """Host array of smoe_layer structs for a list of Layer objects, and its
    device copy (what smoe_moe_decode_layers reads on the GPU)."""

    def __init__(self, layers, device="cuda"):
        self.layers = list(layers)
        n = len(self.layers)
        self.host = (smoe_layer * n)(*[L.s for L in self.layers])
        raw = bytes(memoryview(self.host).cast("B"))
        self.dev = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)
        self.n = n


def smoe_moe_decode_layers(table: LayerTable, x, y, idx_out=None, w_out=None, ws=None, stream=None):
    """One decode token through every layer of `table` in one kernel launch."""
    _check(_lib.smoe_moe_decode_layers(ctypes.cast(table.host, ctypes.POINTER(smoe_layer)), _p(table.dev),
                                       int(table.n), _p(x), _p(y), _p(idx_out), _p(w_out), _p(ws),
                                       0 if ws is None else ws.numel(), _stream(stream)),
           "smoe_moe_decode_layers")
