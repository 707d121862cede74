"""Python face of the CPU oracle (``smoe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
does.  It shares nothing with the CUDA library: bf16 values travel as raw
``uint16`` bit patterns and Q4 codes as ``uint8`` bytes, in the storage layout
the C file documents.

``build()`` compiles ``smoe_oracle.c`` with gcc (``-O2 -ffp-contract=off
-fopenmp``) into ``liborc.so`` beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smoe_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (plain C, fp64, no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
    return _lib


class _Layer(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int),
        ("n_experts", ctypes.c_int),
        ("top_k", ctypes.c_int),
        ("ffn_dim", ctypes.c_int),
        ("group_size", ctypes.c_int),
        ("norm_topk_prob", ctypes.c_int),
        ("rms_eps", ctypes.c_double),
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


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


@dataclass
class OracleLayer:
    """One layer's parameters as host arrays (bf16 as uint16 bits).

    Shapes: router_w [E, D]; gate_q/up_q [E, F, D/2]; gate_s/gate_b/up_s/up_b
    [E, F, D/64]; down_q [E, D, F/2]; down_s/down_b [E, D, F/64]; rms_gain [D]
    or None (no RMSNorm).  With code_bits = 2 (SMOE-Q2) the code arrays are
    [E, F, D/4] and [E, D, F/4].
    """
    d_model: int
    n_experts: int
    top_k: int
    ffn_dim: int
    router_w: np.ndarray
    gate_q: np.ndarray
    gate_s: np.ndarray
    gate_b: np.ndarray
    up_q: np.ndarray
    up_s: np.ndarray
    up_b: np.ndarray
    down_q: np.ndarray
    down_s: np.ndarray
    down_b: np.ndarray
    rms_gain: Optional[np.ndarray] = None
    rms_eps: float = 1e-6
    norm_topk_prob: bool = True
    group_size: int = 64
    code_bits: int = 4

    def __post_init__(self):
        u16, u8 = np.uint16, np.uint8
        for name in ("router_w", "gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b"):
            setattr(self, name, _c(getattr(self, name), u16))
        for name in ("gate_q", "up_q", "down_q"):
            setattr(self, name, _c(getattr(self, name), u8))
        if self.rms_gain is not None:
            self.rms_gain = _c(self.rms_gain, u16)
        D, E, F, G = self.d_model, self.n_experts, self.ffn_dim, self.group_size
        assert self.code_bits in (2, 4)
        per_byte = 8 // self.code_bits
        assert self.router_w.shape == (E, D)
        assert self.gate_q.shape == (E, F, D // per_byte) and self.up_q.shape == (E, F, D // per_byte)
        assert self.gate_s.shape == (E, F, D // G) and self.up_b.shape == (E, F, D // G)
        assert self.down_q.shape == (E, D, F // per_byte) and self.down_s.shape == (E, D, F // G)
        self._s = _Layer(D, E, self.top_k, F, G, int(self.norm_topk_prob), float(self.rms_eps),
                         _ptr(self.rms_gain), _ptr(self.router_w),
                         _ptr(self.gate_q), _ptr(self.gate_s), _ptr(self.gate_b),
                         _ptr(self.up_q), _ptr(self.up_s), _ptr(self.up_b),
                         _ptr(self.down_q), _ptr(self.down_s), _ptr(self.down_b), int(self.code_bits))

    @property
    def ref(self):
        return ctypes.byref(self._s)


def layer_from_weights(W) -> OracleLayer:
    """An OracleLayer on the very bytes of a seeded layer (an object with the
    attributes of the input generator's LayerWeights, tensors on any device):
    bf16 tensors become uint16 bit patterns, codes uint8, all on the host."""
    import torch

    def host(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    return OracleLayer(
        d_model=W.d_model, n_experts=W.n_experts, top_k=W.top_k, ffn_dim=W.ffn_dim,
        router_w=host(W.router_w), gate_q=host(W.gate_q), gate_s=host(W.gate_s),
        gate_b=host(W.gate_b), up_q=host(W.up_q), up_s=host(W.up_s), up_b=host(W.up_b),
        down_q=host(W.down_q), down_s=host(W.down_s), down_b=host(W.down_b),
        rms_gain=None if W.rms_gain is None else host(W.rms_gain), rms_eps=W.rms_eps,
        norm_topk_prob=W.norm_topk_prob, code_bits=getattr(W, "code_bits", 4))


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (the upper half of a binary32)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """float64 -> bf16 bits, round to nearest, ties to even (one rounding)."""
    lib = _load()
    lib.orc_f64_to_bf16.restype = ctypes.c_uint16
    lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat, of = v.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        of[i] = lib.orc_f64_to_bf16(float(flat[i]))
    return out


def q4_weight(q, s, b, row, cols, col, group=64) -> float:
    lib = _load()
    lib.orc_q4_weight.restype = ctypes.c_double
    lib.orc_q4_weight.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_long] * 4
    q, s, b = _c(q, np.uint8), _c(s, np.uint16), _c(b, np.uint16)
    return lib.orc_q4_weight(_ptr(q), _ptr(s), _ptr(b), row, cols, group, col)


def q2_weight(q, s, b, row, cols, col, group=64) -> float:
    lib = _load()
    lib.orc_q2_weight.restype = ctypes.c_double
    lib.orc_q2_weight.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_long] * 4
    q, s, b = _c(q, np.uint8), _c(s, np.uint16), _c(b, np.uint16)
    return lib.orc_q2_weight(_ptr(q), _ptr(s), _ptr(b), row, cols, group, col)


def rmsnorm(L: OracleLayer, r) -> np.ndarray:
    lib = _load()
    r = _c(r, np.uint16)
    xn = np.empty(L.d_model, dtype=np.uint16)
    lib.orc_rmsnorm(L.ref, _ptr(r), _ptr(xn))
    return xn


def router_logits(L: OracleLayer, xn) -> np.ndarray:
    lib = _load()
    xn = _c(xn, np.uint16)
    out = np.empty(L.n_experts, dtype=np.float64)
    lib.orc_router_logits(L.ref, _ptr(xn), _ptr(out))
    return out


def topk(logits, k: int) -> np.ndarray:
    lib = _load()
    logits = _c(logits, np.float64)
    idx = np.empty(k, dtype=np.int32)
    lib.orc_topk(_ptr(logits), ctypes.c_int(logits.size), ctypes.c_int(k), _ptr(idx))
    return idx


def mix_weights(logits, idx, norm_topk_prob: bool = True) -> np.ndarray:
    lib = _load()
    logits, idx = _c(logits, np.float64), _c(idx, np.int32)
    w = np.empty(idx.size, dtype=np.float64)
    lib.orc_mix_weights(_ptr(logits), ctypes.c_int(logits.size), _ptr(idx),
                        ctypes.c_int(idx.size), ctypes.c_int(int(norm_topk_prob)), _ptr(w))
    return w


def expert_ffn(L: OracleLayer, e: int, xn):
    """(o [D], h [F]) of expert e on the normed input xn (bf16 bits)."""
    lib = _load()
    xn = _c(xn, np.uint16)
    o = np.empty(L.d_model, dtype=np.float64)
    h = np.empty(L.ffn_dim, dtype=np.float64)
    lib.orc_expert_ffn(L.ref, ctypes.c_int(e), _ptr(xn), _ptr(o), _ptr(h))
    return o, h


def moe_token(L: OracleLayer, r) -> dict:
    """One token through the layer: y (fp64), y_bf16, idx, w, logits, xn, expert_out."""
    lib = _load()
    r = _c(r, np.uint16)
    D, E, K = L.d_model, L.n_experts, L.top_k
    y = np.empty(D, np.float64)
    yb = np.empty(D, np.uint16)
    idx = np.empty(K, np.int32)
    w = np.empty(K, np.float64)
    logits = np.empty(E, np.float64)
    xn = np.empty(D, np.uint16)
    eo = np.empty((K, D), np.float64)
    lib.orc_moe_token(L.ref, _ptr(r), _ptr(y), _ptr(yb), _ptr(idx), _ptr(w), _ptr(logits),
                      _ptr(xn), _ptr(eo))
    return dict(y=y, y_bf16=yb, idx=idx, w=w, logits=logits, xn=xn, expert_out=eo)


def moe_tokens(L: OracleLayer, r) -> dict:
    """T independent tokens [T, D] (decode steps), host threads over tokens."""
    lib = _load()
    r = _c(r, np.uint16)
    T, D = r.shape
    K = L.top_k
    y = np.empty((T, D), np.float64)
    yb = np.empty((T, D), np.uint16)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    lib.orc_moe_tokens(L.ref, _ptr(r), ctypes.c_int(T), _ptr(y), _ptr(yb), _ptr(idx), _ptr(w))
    return dict(y=y, y_bf16=yb, idx=idx, w=w)


def moe_tokens_experts(L: OracleLayer, r) -> dict:
    """moe_tokens plus every token's unweighted expert outputs, expert_out [T, K, D]."""
    lib = _load()
    r = _c(r, np.uint16)
    T, D = r.shape
    K = L.top_k
    y = np.empty((T, D), np.float64)
    yb = np.empty((T, D), np.uint16)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    eo = np.empty((T, K, D), np.float64)
    lib.orc_moe_tokens_experts(L.ref, _ptr(r), ctypes.c_int(T), _ptr(y), _ptr(yb), _ptr(idx),
                               _ptr(w), _ptr(eo))
    return dict(y=y, y_bf16=yb, idx=idx, w=w, expert_out=eo)


def expert_union(idx, E: int) -> dict:
    """Union (ascending ids, -1 padded to E), offsets [E+1], buckets; 'bad' counts ids out of range."""
    lib = _load()
    idx = _c(idx, np.int32)
    T, k = idx.shape
    union_ids = np.empty(E, np.int32)
    n_union = np.zeros(1, np.int32)
    offsets = np.empty(E + 1, np.int32)
    bt = np.full(T * k, -1, np.int32)
    br = np.full(T * k, -1, np.int32)
    bad = lib.orc_expert_union(_ptr(idx), ctypes.c_int(T), ctypes.c_int(k), ctypes.c_int(E),
                               _ptr(union_ids), _ptr(n_union), _ptr(offsets), _ptr(bt), _ptr(br))
    return dict(union_ids=union_ids, n_union=int(n_union[0]), offsets=offsets,
                bucket_tok=bt, bucket_rank=br, bad=int(bad))


def prefill_chunk(L: OracleLayer, r) -> dict:
    """One chunk of T tokens [T, D] through the layer, via the expert union."""
    lib = _load()
    r = _c(r, np.uint16)
    T, D = r.shape
    E, K = L.n_experts, L.top_k
    y = np.empty((T, D), np.float64)
    yb = np.empty((T, D), np.uint16)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    union_ids = np.empty(E, np.int32)
    n_union = np.zeros(1, np.int32)
    offsets = np.empty(E + 1, np.int32)
    bt = np.full(T * K, -1, np.int32)
    br = np.full(T * K, -1, np.int32)
    lib.orc_moe_prefill_chunk(L.ref, _ptr(r), ctypes.c_int(T), _ptr(y), _ptr(yb), _ptr(idx),
                              _ptr(w), _ptr(union_ids), _ptr(n_union), _ptr(offsets), _ptr(bt),
                              _ptr(br))
    return dict(y=y, y_bf16=yb, idx=idx, w=w, union_ids=union_ids, n_union=int(n_union[0]),
                offsets=offsets, bucket_tok=bt, bucket_rank=br)


def omp_threads() -> int:
    """Threads the oracle's parallel loop uses (OMP_NUM_THREADS, else all host cores)."""
    v = os.environ.get("OMP_NUM_THREADS")
    if v and v.isdigit():
        return int(v)
    return len(os.sched_getaffinity(0))


def dense_matvec(w, x) -> np.ndarray:
    """y = W x in fp64; W bf16 bits [rows, cols], x bf16 bits [cols]."""
    lib = _load()
    w, x = _c(w, np.uint16), _c(x, np.uint16)
    rows, cols = w.shape
    assert x.shape == (cols,)
    y = np.empty(rows, dtype=np.float64)
    lib.orc_dense_matvec.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long, ctypes.c_long,
                                     ctypes.c_void_p]
    lib.orc_dense_matvec(_ptr(w), _ptr(x), rows, cols, _ptr(y))
    return y


def quantize_q4(w):
    """SMOE-Q4 codes, scales and biases of bf16 weights [rows, cols] (cols % 64 == 0)."""
    lib = _load()
    w = _c(w, np.uint16)
    rows, cols = w.shape
    assert cols % 64 == 0
    codes = np.empty((rows, cols // 2), dtype=np.uint8)
    scale = np.empty((rows, cols // 64), dtype=np.uint16)
    bias = np.empty((rows, cols // 64), dtype=np.uint16)
    lib.orc_quantize_q4.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_long] + [ctypes.c_void_p] * 3
    lib.orc_quantize_q4(_ptr(w), rows, cols, _ptr(codes), _ptr(scale), _ptr(bias))
    return codes, scale, bias


def quantize_q2(w):
    """SMOE-Q2 codes ([rows, cols/4]), scales and biases of bf16 weights [rows, cols]."""
    lib = _load()
    w = _c(w, np.uint16)
    rows, cols = w.shape
    assert cols % 64 == 0
    codes = np.empty((rows, cols // 4), dtype=np.uint8)
    scale = np.empty((rows, cols // 64), dtype=np.uint16)
    bias = np.empty((rows, cols // 64), dtype=np.uint16)
    lib.orc_quantize_q2.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_long] + [ctypes.c_void_p] * 3
    lib.orc_quantize_q2(_ptr(w), rows, cols, _ptr(codes), _ptr(scale), _ptr(bias))
    return codes, scale, bias
