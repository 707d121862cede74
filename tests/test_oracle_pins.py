"""Pins for the CPU oracle: each test checks it against something other than
itself -- hand-derived closed forms, textbook/library routines (numpy matmul,
argsort, scipy softmax/expit, torch's own fp32->bf16 rounding and rms_norm),
invariants and brute force on tiny inputs -- so that a dropped term, a wrong
sign or index, a swapped nibble or a transposed operand fails one of them."""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from quantised_expert_ffn_gb300 import synth
from tests.util import bf16_f64, bits, oracle_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_hand_cases(oracle_mod):
    f = oracle_mod.f64_to_bf16
    cases = {
        1.0: 0x3F80,
        -2.0: 0xC000,
        1.0 + 2.0 ** -8: 0x3F80,                  # tie -> even (down)
        1.0 + 3 * 2.0 ** -8: 0x3F82,              # tie -> even (up)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,     # just above the tie: one rounding, up
        2.0 ** -130: 0x0008,                      # subnormal: 8 * 2^-133
        3.5e38: 0x7F80,                           # overflow -> inf
        0.0: 0x0000,
    }
    for v, b in cases.items():
        assert int(f(v)) == b, (v, hex(int(f(v))), hex(b))


def test_bf16_rounding_matches_torch_on_fp32(oracle_mod):
    g = torch.Generator().manual_seed(5)
    v = torch.randn(4000, generator=g) * torch.exp(torch.randn(4000, generator=g) * 8)
    ours = oracle_mod.f64_to_bf16(v.double().numpy())
    theirs = bits(v.to(torch.bfloat16))
    assert np.array_equal(ours, theirs)


def test_bf16_round_trip_all_finite(oracle_mod):
    pats = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    vals = bf16_f64(pats)
    keep = np.isfinite(vals)
    back = oracle_mod.f64_to_bf16(vals[keep])
    # +0/-0 both fine; everything else must come back bit-identical
    assert np.array_equal(back, pats[keep])


# ---------------------------------------------------------------- Q4 layout / dequant

def _zero_layer(D=128, F=64, E=2, K=1, seed=0):
    """A layer whose every weight is exactly 0 (codes 8, bias = -8 * scale)."""
    W = synth.layer_weights(D, E, F, K, seed=seed)
    for n in ("gate_q", "up_q", "down_q"):
        getattr(W, n).fill_(0x88)
    return W


def test_zero_weights_give_identity(oracle_mod):
    """q = 8 with bias = -8 s gives w = 0 exactly, so y = r bit-exactly."""
    W = _zero_layer(K=2, E=4)
    L = oracle_layer(W)
    r = bits(synth.hidden(1, 128, seed=3))[0]
    out = oracle_mod.moe_token(L, r)
    assert np.array_equal(out["y_bf16"], r)
    assert np.all(out["expert_out"] == 0.0)


def _set_code(q, row, col, code):
    byte = q[row, col // 2]
    if col % 2 == 0:
        q[row, col // 2] = (byte & 0xF0) | code
    else:
        q[row, col // 2] = (byte & 0x0F) | (code << 4)


@pytest.mark.parametrize("d0,j0,d1", [(70, 5, 33), (71, 6, 32), (0, 0, 127), (127, 63, 1)])
def test_single_code_pins_layout(oracle_mod, d0, j0, d1):
    """One code moved off 8 in gate (row j0, col d0) and in down (row d1, col j0):
    g is zero except g[j0] = s_g * x[d0]; o is zero except o[d1] = s_d * h[j0].
    Distinct scales per group make a wrong group, nibble or transposition show."""
    D, F = 128, 64
    W = _zero_layer(D=D, F=F, E=1, K=1)
    # distinct exact scales per (row, group), bias = -8 s keeps w = 0 elsewhere
    gs = (torch.arange(F * D // 64, dtype=torch.float32).reshape(1, F, D // 64) + 1) / 256
    W.gate_s = gs.to(torch.bfloat16)
    W.gate_b = (W.gate_s.float() * -8).to(torch.bfloat16)
    W.up_s = torch.zeros_like(W.up_s)
    W.up_b = torch.full_like(W.up_b, 1 / 64)          # constant up matrix
    ds = (torch.arange(D * F // 64, dtype=torch.float32).reshape(1, D, F // 64) + 3) / 512
    W.down_s = ds.to(torch.bfloat16)
    W.down_b = (W.down_s.float() * -8).to(torch.bfloat16)
    _set_code(W.gate_q[0], j0, d0, 9)
    _set_code(W.down_q[0], d1, j0, 11)
    L = oracle_layer(W)
    x = bits(synth.hidden(1, D, seed=11))[0]
    xf = bf16_f64(x)
    o, h = oracle_mod.expert_ffn(L, 0, x)
    s_g = float(W.gate_s[0, j0, d0 // 64])
    g = s_g * 1 * xf[d0]
    u = xf.sum() / 64
    hj = g * scipy.special.expit(g) * u
    assert np.count_nonzero(h) == 1 and h[j0] == pytest.approx(hj, rel=1e-13)
    s_d = float(W.down_s[0, d1, j0 // 64])
    assert np.count_nonzero(o) == 1 and o[d1] == pytest.approx(3 * s_d * hj, rel=1e-13)


def _numpy_dequant(q, s, b):
    """Independent unpack of the documented Q4 layout with numpy."""
    lo = (q & 0x0F).astype(np.float64)
    hi = (q >> 4).astype(np.float64)
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    return codes * np.repeat(bf16_f64(s), 64, axis=1) + np.repeat(bf16_f64(b), 64, axis=1)


def test_expert_ffn_matches_numpy_matmul(oracle_mod):
    """Brute force on a tiny layer: numpy fp64 matmul of the dequantised matrices."""
    D, F, E = 128, 128, 3
    W = synth.layer_weights(D, E, F, 2, seed=21)
    # a general (not -8 s) bias, so that the affine term is exercised
    W.gate_b = (torch.randn(W.gate_b.shape) * 0.01).to(torch.bfloat16)
    W.down_b = (torch.randn(W.down_b.shape) * 0.01).to(torch.bfloat16)
    L = oracle_layer(W)
    x = bits(synth.hidden(1, D, seed=4))[0]
    xf = bf16_f64(x)
    for e in range(E):
        Wg = _numpy_dequant(L.gate_q[e], L.gate_s[e], L.gate_b[e])
        Wu = _numpy_dequant(L.up_q[e], L.up_s[e], L.up_b[e])
        Wd = _numpy_dequant(L.down_q[e], L.down_s[e], L.down_b[e])
        g, u = Wg @ xf, Wu @ xf
        h_ref = g * scipy.special.expit(g) * u
        o_ref = Wd @ h_ref
        o, h = oracle_mod.expert_ffn(L, e, x)
        np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-14)


def test_silu_closed_forms(oracle_mod):
    """Constant matrices reduce the FFN to scalars: g = cg * sum x, u = cu * sum x,
    o = cd * F * SiLU(g) * u.  At g = 0 the output is 0; at large |g| SiLU is g or 0."""
    D, F = 64, 64
    x = np.full(D, 0x3F80, np.uint16)                 # ones: sum x = 64
    for cg, expect in [(0.0, lambda g, u: 0.0),
                       (0.5, lambda g, u: g * u),     # g = 32: sigma(32) = 1 - 1.3e-14
                       (-0.5, lambda g, u: 0.0)]:     # g = -32: g*sigma(g) = -4e-13
        W = synth.layer_weights(D, 1, F, 1, seed=1)
        for n in ("gate_s", "up_s", "down_s"):
            setattr(W, n, torch.zeros_like(getattr(W, n)))
        W.gate_b = torch.full_like(W.gate_b, cg)
        W.up_b = torch.full_like(W.up_b, 1 / 64)
        W.down_b = torch.full_like(W.down_b, 1 / 64)
        o, h = oracle_mod.expert_ffn(oracle_layer(W), 0, x)
        g, u = 64 * cg, 1.0
        np.testing.assert_allclose(h, expect(g, u), rtol=1e-12, atol=1e-11)
        np.testing.assert_allclose(o, F / 64 * expect(g, u), rtol=1e-12, atol=1e-11)


# ---------------------------------------------------------------- router, top-k, weights

def test_router_logits_match_numpy(oracle_mod):
    W = synth.layer_weights(256, 16, 64, 4, seed=8)
    L = oracle_layer(W)
    x = bits(synth.hidden(1, 256, seed=9))[0]
    ref = bf16_f64(L.router_w) @ bf16_f64(x)
    np.testing.assert_allclose(oracle_mod.router_logits(L, x), ref, rtol=1e-13, atol=1e-15)


def test_topk_matches_full_sort_with_ties(oracle_mod):
    rng = np.random.default_rng(3)
    for trial in range(50):
        E = int(rng.integers(1, 160))
        k = int(rng.integers(1, E + 1))
        logits = np.round(rng.normal(size=E), 1)      # many exact ties
        key32 = logits.astype(np.float32)
        ref = np.lexsort((np.arange(E), -key32))[:k]
        assert np.array_equal(oracle_mod.topk(logits, k), ref)


def test_topk_k_equals_e_is_permutation(oracle_mod):
    logits = np.random.default_rng(0).normal(size=33)
    idx = oracle_mod.topk(logits, 33)
    assert sorted(idx.tolist()) == list(range(33))
    assert np.all(np.diff(logits[idx]) <= 0)


def test_topk_decides_in_fp32(oracle_mod):
    """Two logits that differ only below fp32 resolution tie; the lower id wins."""
    logits = np.array([1.0, 1.0 + 2.0 ** -40, 0.5])
    assert oracle_mod.topk(logits, 1)[0] == 0


def test_mix_weights(oracle_mod):
    rng = np.random.default_rng(1)
    logits = rng.normal(size=128) * 2
    idx = oracle_mod.topk(logits, 8)
    w = oracle_mod.mix_weights(logits, idx, True)
    assert abs(w.sum() - 1.0) < 8 * 2.0 ** -24
    assert np.all(np.diff(w) <= 0)
    np.testing.assert_allclose(w, scipy.special.softmax(logits[idx]), rtol=1e-13)
    w_all = oracle_mod.mix_weights(logits, idx, False)
    np.testing.assert_allclose(w_all, scipy.special.softmax(logits)[idx], rtol=1e-13)
    full = oracle_mod.topk(logits, 128)
    np.testing.assert_allclose(oracle_mod.mix_weights(logits, full, True),
                               scipy.special.softmax(logits)[full], rtol=1e-13)


def test_single_expert_layer(oracle_mod):
    """E = 1, k = 1: w = 1 and y = r + FFN(r)."""
    W = synth.layer_weights(64, 1, 64, 1, seed=2)
    L = oracle_layer(W)
    r = bits(synth.hidden(1, 64, seed=7))[0]
    out = oracle_mod.moe_token(L, r)
    assert out["idx"].tolist() == [0] and out["w"][0] == 1.0
    o, _ = oracle_mod.expert_ffn(L, 0, r)
    np.testing.assert_array_equal(out["y"], bf16_f64(r) + o)


def test_rmsnorm_matches_torch(oracle_mod):
    D = 256
    W = synth.layer_weights(D, 4, 64, 2, seed=3, rms_norm=True)
    W.rms_gain = (1 + 0.1 * torch.randn(D, generator=torch.Generator().manual_seed(1))).to(
        torch.bfloat16)
    L = oracle_layer(W)
    r = synth.hidden(1, D, seed=12)[0] * 3
    ref = torch.nn.functional.rms_norm(r.double(), (D,), W.rms_gain.double(), eps=1e-6)
    assert np.array_equal(oracle_mod.rmsnorm(L, bits(r)), oracle_mod.f64_to_bf16(ref.numpy()))


# ---------------------------------------------------------------- union and buckets

def _brute_union(idx, E):
    buckets = {}
    for t, row in enumerate(idx):
        for i, e in enumerate(row):
            buckets.setdefault(int(e), []).append((t, i))
    return buckets


@pytest.mark.parametrize("T,k,E,seed", [(1, 8, 128, 0), (45, 8, 128, 1), (64, 8, 128, 2),
                                        (7, 3, 5, 3), (64, 8, 16, 4)])
def test_union_matches_python_dict(oracle_mod, T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    u = oracle_mod.expert_union(idx, E)
    ref = _brute_union(idx, E)
    assert u["n_union"] == len(ref)
    assert u["union_ids"][:u["n_union"]].tolist() == sorted(ref)
    assert np.all(u["union_ids"][u["n_union"]:] == -1)
    for n, e in enumerate(sorted(ref)):
        lo, hi = u["offsets"][n], u["offsets"][n + 1]
        got = list(zip(u["bucket_tok"][lo:hi].tolist(), u["bucket_rank"][lo:hi].tolist()))
        assert got == ref[e]
    assert np.all(u["offsets"][u["n_union"]:] == T * k)


def test_union_degenerate_cases(oracle_mod):
    same = np.tile(np.arange(8, dtype=np.int32)[::-1], (64, 1))
    assert oracle_mod.expert_union(same, 128)["n_union"] == 8
    distinct = np.arange(128, dtype=np.int32).reshape(16, 8)
    assert oracle_mod.expert_union(distinct, 128)["n_union"] == 128
    few = np.arange(24, dtype=np.int32).reshape(3, 8)
    assert oracle_mod.expert_union(few, 128)["n_union"] == 24


def test_union_skips_out_of_range(oracle_mod):
    idx = np.array([[0, 5, 200], [-1, 5, 3]], np.int32)
    u = oracle_mod.expert_union(idx, 8)
    assert u["bad"] == 2 and u["n_union"] == 3
    assert u["union_ids"][:3].tolist() == [0, 3, 5]


# ---------------------------------------------------------------- chunk vs per-token

def test_prefill_chunk_equals_per_token_bit_exact(oracle_mod):
    W = synth.layer_weights(128, 16, 64, 4, seed=30, rms_norm=True)
    L = oracle_layer(W)
    r = bits(synth.hidden(9, 128, seed=31))
    chunk = oracle_mod.prefill_chunk(L, r)
    for t in range(9):
        tok = oracle_mod.moe_token(L, r[t])
        assert np.array_equal(chunk["idx"][t], tok["idx"])
        assert np.array_equal(chunk["w"][t], tok["w"])
        assert np.array_equal(chunk["y"][t], tok["y"])
        assert np.array_equal(chunk["y_bf16"][t], tok["y_bf16"])
    batch = oracle_mod.moe_tokens(L, r)
    assert np.array_equal(batch["y"], chunk["y"])


# ---------------------------------------------------------------- hand-worked fixture

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *rest = line.split()
                vals[key] = rest
    return vals


def test_hand_worked_layer(oracle_mod):
    g = _read_golden("hand_worked_constant_experts.txt")
    D, F, E, K = (int(g[k][0]) for k in ("D", "F", "E", "K"))
    W = synth.layer_weights(D, E, F, K, seed=0)
    v = [float(a) for a in g["router_v"]]
    W.router_w = torch.tensor([[ve / 64] * D for ve in v]).to(torch.bfloat16)
    for mat, key in (("gate", "const_gate"), ("up", "const_up"), ("down", "const_down")):
        s = getattr(W, mat + "_s")
        setattr(W, mat + "_s", torch.zeros_like(s))
        c = torch.tensor([float(a) for a in g[key]]).view(E, 1, 1).expand_as(s)
        setattr(W, mat + "_b", c.to(torch.bfloat16).contiguous())
    out = oracle_mod.moe_token(oracle_layer(W), np.full(D, 0x3F80, np.uint16))
    assert out["idx"].tolist() == [int(a) for a in g["expect_idx"]]
    np.testing.assert_allclose(out["w"], [float(a) for a in g["expect_w"]], rtol=1e-15)
    np.testing.assert_allclose(out["expert_out"][:, 0], [float(a) for a in g["expect_o"]],
                               rtol=1e-14)
    np.testing.assert_allclose(out["y"], float(g["expect_y"][0]), rtol=1e-15)
    assert np.all(out["y_bf16"] == int(g["expect_y_bf16"][0], 16))


# ---------------------------------------------------------------- dense bf16 matvec

def _bf16_bits(v):
    return bits(torch.tensor(np.asarray(v, dtype=np.float32)).to(torch.bfloat16))


def test_dense_matvec_one_hot_rows_pick_inputs(oracle_mod):
    """Row r of W is one-hot at column (7 r + 3) mod cols: y[r] = x[that column]
    exactly (a transposed operand or a shifted index fails)."""
    rows, cols = 37, 24
    W = np.zeros((rows, cols), dtype=np.float32)
    pick = (7 * np.arange(rows) + 3) % cols
    W[np.arange(rows), pick] = 1.0
    x = np.linspace(-3.0, 5.0, cols).astype(np.float32)
    xb = _bf16_bits(x)
    y = oracle_mod.dense_matvec(_bf16_bits(W), xb)
    assert np.array_equal(y, bf16_f64(xb)[pick])


def test_dense_matvec_closed_form(oracle_mod):
    """W[r][c] = r + 1 (every column), x[c] = c: y[r] = (r + 1) * cols (cols - 1) / 2."""
    rows, cols = 5, 64
    W = np.repeat(np.arange(1, rows + 1, dtype=np.float32)[:, None], cols, axis=1)
    x = np.arange(cols, dtype=np.float32)
    y = oracle_mod.dense_matvec(_bf16_bits(W), _bf16_bits(x))
    assert np.array_equal(y, (np.arange(1, rows + 1) * cols * (cols - 1) / 2).astype(np.float64))


def test_dense_matvec_matches_numpy_matmul(oracle_mod):
    g = torch.Generator().manual_seed(21)
    W = bits(torch.randn(33, 200, generator=g).to(torch.bfloat16))
    x = bits(torch.randn(200, generator=g).to(torch.bfloat16))
    ref = bf16_f64(W) @ bf16_f64(x)
    y = oracle_mod.dense_matvec(W, x)
    scale = np.abs(bf16_f64(W)) @ np.abs(bf16_f64(x))
    assert np.all(np.abs(y - ref) <= 1e-13 * scale)


# ---------------------------------------------------------------- SMOE-Q4 quantiser

def _codes_of(codes_row):
    """Unpack one row of Q4 codes: element 2j is the low nibble of byte j."""
    c = np.asarray(codes_row, dtype=np.uint8)
    return np.stack([c & 0x0F, c >> 4], axis=-1).reshape(-1)


def test_quantize_ladder_is_exact(oracle_mod):
    """A group holding 1 + 0.5 k (k = 0..15, four times) has min 1, max 8.5:
    scale 0.5, bias 1 and codes k, all exact; a second group shifted by -4."""
    k = np.arange(64) % 16
    W = np.stack([np.concatenate([1.0 + 0.5 * k, -3.0 + 0.5 * k])]).astype(np.float32)
    codes, scale, bias = oracle_mod.quantize_q4(_bf16_bits(W))
    assert np.array_equal(bf16_f64(scale), [[0.5, 0.5]])
    assert np.array_equal(bf16_f64(bias), [[1.0, -3.0]])
    assert np.array_equal(_codes_of(codes[0]), np.concatenate([k, k]))


def test_quantize_constant_group(oracle_mod):
    """Equal weights: scale 0, every code 0, bias = the weight (a zero range
    never divides)."""
    W = np.full((2, 64), -1.25, dtype=np.float32)
    W[1] = 0.0
    codes, scale, bias = oracle_mod.quantize_q4(_bf16_bits(W))
    assert np.all(scale == 0) and np.all(codes == 0)
    assert np.array_equal(bf16_f64(bias)[:, 0], [-1.25, 0.0])
    assert bias[1, 0] == 0x0000                    # +0, not -0


def test_quantize_rounds_halves_to_even(oracle_mod):
    """min 0, max 15 gives scale 1: 2.5 -> 2, 3.5 -> 4, 4.5 -> 4, 14.5 -> 14."""
    W = np.zeros((1, 64), dtype=np.float32)
    W[0, 1] = 15.0
    W[0, 2:6] = [2.5, 3.5, 4.5, 14.5]
    codes, scale, bias = oracle_mod.quantize_q4(_bf16_bits(W))
    assert bf16_f64(scale)[0, 0] == 1.0 and bf16_f64(bias)[0, 0] == 0.0
    assert list(_codes_of(codes[0])[:6]) == [0, 15, 2, 4, 4, 14]


def test_quantize_round_trip_error_bound(oracle_mod):
    """Random groups: every weight decodes to within half a (rounded) scale
    step plus binary32 slack, the least weight decodes exactly, and the codes
    are the nearest of the 16 levels wherever that level is within [0, 15]."""
    g = torch.Generator().manual_seed(8)
    W = torch.randn(12, 256, generator=g) * torch.exp(torch.randn(12, 1, generator=g))
    Wb = bits(W.to(torch.bfloat16))
    codes, scale, bias = oracle_mod.quantize_q4(Wb)
    w = bf16_f64(Wb).reshape(12, 4, 64)
    s = bf16_f64(scale)[:, :, None]
    b = bf16_f64(bias)[:, :, None]
    q = np.stack([_codes_of(codes[r]) for r in range(12)]).reshape(12, 4, 64).astype(np.float64)
    dec = s * q + b
    assert np.all(np.abs(dec - w) <= s * (0.5 + 2.0 ** -16))
    assert np.array_equal(b[:, :, 0], w.min(axis=2))
    levels = s * np.arange(16)[None, None, :] + b              # [12, 4, 16]
    best = np.abs(w[..., None] - levels[:, :, None, :]).argmin(axis=-1)
    gap = np.abs(w[..., None] - levels[:, :, None, :])
    gap.sort(axis=-1)
    clear = gap[..., 1] - gap[..., 0] > 1e-6 * s               # no near-tie
    assert np.array_equal(q[clear], best[clear])


def _exact_group(wbits, levels):
    """Brute force of the quantiser's reading on one group of 64 bf16 weights,
    with exact rationals: scale = bf16 of the binary32 ((mx - mn) + 0) / levels
    (numpy binary32 arithmetic, torch's bf16 rounding), bias = mn, and each code
    the level index k in 0..levels minimising |w - (mn + scale k)|, the even k
    on a tie.  Returns (codes, scale bits, bias bits)."""
    from fractions import Fraction
    wf = bf16_f64(wbits).astype(np.float32)
    mn, mx = np.float32(wf.min()), np.float32(wf.max())
    quot = np.float32(np.float32(np.float32(mx - mn) + np.float32(0.0)) / np.float32(levels))
    sb = int(_bf16_bits([quot])[0])
    s = Fraction(float(bf16_f64(np.array([sb], np.uint16))[0]))
    m = Fraction(float(mn))
    codes = []
    for w in wf:
        if s == 0:
            codes.append(0)
            continue
        d = Fraction(float(w)) - m
        codes.append(min(range(levels + 1), key=lambda k: (abs(d - s * k), k % 2)))
    return np.array(codes), sb, int(_bf16_bits([mn + np.float32(0.0)])[0])


def _check_against_exact(oracle_mod, W, bits_=4):
    rows, cols = W.shape
    quant = oracle_mod.quantize_q4 if bits_ == 4 else oracle_mod.quantize_q2
    codes, scale, bias = quant(W)
    for r in range(rows):
        if bits_ == 4:
            got = _codes_of(codes[r])
        else:
            got = np.stack([(codes[r] >> (2 * j)) & 3 for j in range(4)], -1).reshape(-1)
        for g in range(cols // 64):
            c, sb, bb = _exact_group(W[r, 64 * g:64 * g + 64], (1 << bits_) - 1)
            assert scale[r, g] == sb and bias[r, g] == bb, (r, g)
            assert np.array_equal(got[64 * g:64 * g + 64], c), (r, g, got[64 * g:64 * g + 64], c)


def test_quantize_matches_exact_rational_brute_force(oracle_mod):
    """Random groups of very different magnitudes, groups with weights near
    zero next to a large minimum, and groups built with exact ties: every
    scale, bias and code equals the exact-rational brute force."""
    g = torch.Generator().manual_seed(21)
    W = torch.randn(6, 256, generator=g) * torch.exp(2 * torch.randn(6, 1, generator=g))
    W[0, :64] *= torch.rand(64, generator=g) ** 8            # many weights near 0
    W[1, 5] = -1.0                                           # a large minimum ...
    W[1, 6:12] = torch.tensor([1e-9, -1e-9, 2e-7, -3e-8, 0.0, 1e-20])   # ... with tiny weights
    Wb = bits(W.to(torch.bfloat16))
    # a tie group: min 0, max 15 * 0.375 (scale 0.375), weights on every midpoint
    Wb[2, 64:128] = _bf16_bits([0.0, 15 * 0.375] + [0.375 * (k % 15 + 0.5) for k in range(62)])
    _check_against_exact(oracle_mod, Wb, 4)
    _check_against_exact(oracle_mod, Wb, 2)


def test_quantize_tie_with_scale_not_a_power_of_two(oracle_mod):
    """(w - mn) / scale = 17/2 exactly with scale = 85 * 2^-16: the nearest
    level, halves to even, is 8.  Multiplying by the rounded binary32
    reciprocal of the scale instead gives 9, so a quantiser that divides that
    way fails here."""
    mn, mx, w = -155 * 2.0 ** -14, 164 * 2.0 ** -14, 205 * 2.0 ** -17
    W = np.zeros((1, 64), dtype=np.float32)
    W[0, :3] = [mn, mx, w]
    W[0, 3:] = 0.0
    codes, scale, bias = oracle_mod.quantize_q4(_bf16_bits(W))
    s = bf16_f64(scale)[0, 0]
    assert s == 85 * 2.0 ** -16 and bf16_f64(bias)[0, 0] == mn
    assert (w - mn) / s == 8.5
    assert _codes_of(codes[0])[2] == 8
    r = np.float32(1.0) / np.float32(s)                     # the reciprocal rule disagrees
    assert np.rint(np.float64(np.float32(w - mn)) * np.float64(r)) == 9
    _check_against_exact(oracle_mod, _bf16_bits(W), 4)


def test_quantize_needs_the_exact_difference(oracle_mod):
    """mn = -0.09375, max 0.84375: scale 1/16 and -mn = 1.5 scales exactly, so
    w = +2^-100 lies just above the midpoint (code 2) and w = -2^-100 just
    below it (code 1).  In binary64 (and binary32) w - mn rounds onto the
    midpoint itself; only the exact difference tells the two apart."""
    W = np.zeros((1, 64), dtype=np.float32)
    W[0, :4] = [-0.09375, 0.84375, 2.0 ** -100, -(2.0 ** -100)]
    W[0, 4:] = -0.09375
    codes, scale, bias = oracle_mod.quantize_q4(_bf16_bits(W))
    assert bf16_f64(scale)[0, 0] == 0.0625
    assert np.float64(2.0 ** -100) + 0.09375 == 0.09375      # the rounded difference ties
    assert list(_codes_of(codes[0])[:4]) == [0, 15, 2, 1]
    _check_against_exact(oracle_mod, _bf16_bits(W), 4)


def test_quantize_scale_below_binary32_normal_range(oracle_mod):
    """A group whose scale is below 2^-126 (bf16 subnormal range): min 0,
    max 15 * 2^-130; halves 2.5 and 3.5 scales round to 2 and 4, and random
    weights in range match the exact brute force."""
    s = 2.0 ** -130
    W = np.zeros((2, 64), dtype=np.float32)
    W[0, :6] = [0.0, 15 * s, 2.5 * s, 3.5 * s, 7 * s, 14.5 * s]
    g = np.random.default_rng(3)
    W[1] = (g.integers(0, 61, 64) * 2.0 ** -135).astype(np.float32)
    Wb = _bf16_bits(W)
    codes, scale, bias = oracle_mod.quantize_q4(Wb)
    assert bf16_f64(scale)[0, 0] == s
    assert list(_codes_of(codes[0])[:6]) == [0, 15, 2, 4, 7, 14]
    _check_against_exact(oracle_mod, Wb, 4)
    _check_against_exact(oracle_mod, Wb, 2)


# ---------------------------------------------------------------- SMOE-Q2 layout

def _set_code2(q, row, col, code):
    sh = 2 * (col % 4)
    q[row, col // 4] = (int(q[row, col // 4]) & ~(3 << sh) & 0xFF) | (code << sh)


def test_q2_single_code_pins_layout(oracle_mod):
    """SMOE-Q2: every code 2 with bias -2 s gives w = 0; one code moved to 3 in
    gate (row 6, col 71) and to 0 in down (row 33, col 6): g is zero except
    g[6] = s_g x[71], o zero except o[33] = -2 s_d h[6].  Distinct scales per
    group and the 2-bit position (col % 4 = 3, then 2) make a wrong group,
    shift or transposition show."""
    D, F = 128, 64
    W = synth.layer_weights(D, 1, F, 1, seed=0, code_bits=2)
    for n in ("gate_q", "up_q", "down_q"):
        getattr(W, n).fill_(0xAA)                      # every code 2
    gs = (torch.arange(F * D // 64, dtype=torch.float32).reshape(1, F, D // 64) + 1) / 256
    W.gate_s = gs.to(torch.bfloat16)
    W.gate_b = (W.gate_s.float() * -2).to(torch.bfloat16)
    W.up_s = torch.zeros_like(W.up_s)
    W.up_b = torch.full_like(W.up_b, 1 / 64)
    ds = (torch.arange(D * F // 64, dtype=torch.float32).reshape(1, D, F // 64) + 3) / 512
    W.down_s = ds.to(torch.bfloat16)
    W.down_b = (W.down_s.float() * -2).to(torch.bfloat16)
    j0, d0, d1 = 6, 71, 33
    _set_code2(W.gate_q[0], j0, d0, 3)
    _set_code2(W.down_q[0], d1, j0, 0)
    L = oracle_layer(W)
    assert L.code_bits == 2
    x = bits(synth.hidden(1, D, seed=11))[0]
    xf = bf16_f64(x)
    o, h = oracle_mod.expert_ffn(L, 0, x)
    g = float(W.gate_s[0, j0, d0 // 64]) * xf[d0]
    hj = g * scipy.special.expit(g) * (xf.sum() / 64)
    assert np.count_nonzero(h) == 1 and h[j0] == pytest.approx(hj, rel=1e-13)
    s_d = float(W.down_s[0, d1, j0 // 64])
    assert np.count_nonzero(o) == 1 and o[d1] == pytest.approx(-2 * s_d * hj, rel=1e-13)


def _numpy_dequant_q2(q, s, b):
    """Independent unpack of the documented Q2 layout with numpy."""
    codes = np.stack([(q >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(q.shape[0], -1)
    return codes.astype(np.float64) * np.repeat(bf16_f64(s), 64, axis=1) + np.repeat(bf16_f64(b), 64, axis=1)


def test_q2_expert_ffn_matches_numpy_matmul(oracle_mod):
    D, F, E = 128, 192, 2
    W = synth.layer_weights(D, E, F, 2, seed=22, code_bits=2)
    W.up_b = (torch.randn(W.up_b.shape) * 0.01).to(torch.bfloat16)
    W.down_b = (torch.randn(W.down_b.shape) * 0.01).to(torch.bfloat16)
    L = oracle_layer(W)
    x = bits(synth.hidden(1, D, seed=5))[0]
    xf = bf16_f64(x)
    for e in range(E):
        Wg = _numpy_dequant_q2(L.gate_q[e], L.gate_s[e], L.gate_b[e])
        Wu = _numpy_dequant_q2(L.up_q[e], L.up_s[e], L.up_b[e])
        Wd = _numpy_dequant_q2(L.down_q[e], L.down_s[e], L.down_b[e])
        g, u = Wg @ xf, Wu @ xf
        h_ref = g * scipy.special.expit(g) * u
        o, h = oracle_mod.expert_ffn(L, e, x)
        np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(o, Wd @ h_ref, rtol=1e-11, atol=1e-14)


def test_q2_weight_reads_the_documented_bits(oracle_mod):
    """Byte 0b11_10_01_00 holds codes 0, 1, 2, 3 for columns 0..3."""
    q = np.array([[0b11100100] + [0] * 15], dtype=np.uint8)
    s = _bf16_bits([[1.0]])
    b = _bf16_bits([[0.5]])
    assert [oracle_mod.q2_weight(q, s, b, 0, 64, c) for c in range(4)] == [0.5, 1.5, 2.5, 3.5]


def test_quantize_q2_ladder_and_ties(oracle_mod):
    """Q2: a group of 1 + 0.25 k (k = 0..3) has scale 0.25, bias 1, codes k; a
    group with min 0, max 3 and halves 0.5, 1.5, 2.5 rounds them to 0, 2, 2."""
    k = np.arange(64) % 4
    W = np.zeros((2, 64), dtype=np.float32)
    W[0] = 1.0 + 0.25 * k
    W[1, 1] = 3.0
    W[1, 2:5] = [0.5, 1.5, 2.5]
    codes, scale, bias = oracle_mod.quantize_q2(_bf16_bits(W))
    assert np.array_equal(bf16_f64(scale)[:, 0], [0.25, 1.0])
    assert np.array_equal(bf16_f64(bias)[:, 0], [1.0, 0.0])
    unpack = lambda row: np.stack([(codes[row] >> (2 * j)) & 3 for j in range(4)], -1).reshape(-1)
    assert np.array_equal(unpack(0), k)
    assert list(unpack(1)[:5]) == [0, 3, 0, 2, 2]
