"""GPU parity of the dense bf16 matvec and the SMOE-Q4 quantiser, called
through the C ABI, against the CPU oracle on the same seeded bytes.

Bars: the quantiser's codes, scales and biases bit-exact (both sides take
every rounding decision in binary32 with the same operations); the matvec
within its fp32 summation bound, |y - y_ref| <= 2^-18 * sum_c |w x| per row
(the kernel's longest chain of dependent fp32 additions per row is well under
64 steps of relative error 2^-24)."""
import numpy as np
import pytest
import torch

from quantised_expert_ffn_gb300 import synth
from tests.util import bf16_f64, bits, from_bits, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smoe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe as m
    return m


@pytest.fixture(scope="module")
def orc():
    from oracle import oracle
    oracle.build()
    return oracle


def _check_matvec(orc, W, x, y, rows_idx=None):
    Wn = bits(W) if rows_idx is None else bits(W[rows_idx])
    yn = host(y) if rows_idx is None else host(y)[rows_idx]
    xn = bits(x)
    ref = orc.dense_matvec(Wn, xn)
    bound = 2.0 ** -18 * (np.abs(bf16_f64(Wn)) @ np.abs(bf16_f64(xn))) + 1e-30
    err = np.abs(yn.astype(np.float64) - ref)
    assert np.all(err <= bound), (float((err / bound).max()), int((err / bound).argmax()))


# (rows, cols): one row; ragged chunk split (33 chunks over 8 warps); the K/V
# projection (512 x 4096, one row per CTA step); 30B Q (4096 x 2048, four rows
# per step); 235B O (4096 x 8192, four chunks per lane); ragged row blocks; wide
# rows at four rows per step (two chunks per lane) and two rows (four chunks)
@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 264), (512, 4096), (4096, 2048), (4096, 8192),
                                       (3001, 1032), (2437, 4096), (2500, 8192)])
def test_dense_matvec_against_oracle(smoe, orc, rows, cols):
    W = synth.dense_weights((rows, cols), seed=rows * 7 + cols, device="cuda")
    x = synth.hidden(1, cols, seed=cols, device="cuda")[0]
    y = torch.full((rows,), float("nan"), device="cuda")
    smoe.smoe_dense_matvec(W, x, y)
    torch.cuda.synchronize()
    _check_matvec(orc, W, x, y)


def test_dense_matvec_lm_head_full_size(smoe, orc):
    """The LM head shape (151,936 x 4096, 1.24 GB of bf16), as the benchmark runs
    it: 96 sampled rows (both ends and spread between) against the oracle,
    every row finite."""
    rows, cols = 151936, 4096
    W = synth.dense_weights((rows, cols), seed=3, device="cuda")
    x = synth.hidden(1, cols, seed=4, device="cuda")[0]
    y = torch.full((rows,), float("nan"), device="cuda")
    smoe.smoe_dense_matvec(W, x, y)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y).all())
    idx = np.unique(np.concatenate([np.arange(8), rows - 1 - np.arange(8),
                                    np.random.default_rng(0).integers(0, rows, 80)]))
    _check_matvec(orc, W, x, y, rows_idx=idx)


def test_dense_matvec_zero_and_one_hot(smoe):
    """A zero matrix gives exact zeros; a one-hot row gives the picked input exactly."""
    rows, cols = 96, 512
    W = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    pick = (torch.arange(rows, device="cuda") * 37 + 5) % cols
    W[torch.arange(rows, device="cuda"), pick] = 1.0
    x = synth.hidden(1, cols, seed=9, device="cuda")[0]
    y = torch.empty(rows, device="cuda")
    smoe.smoe_dense_matvec(W, x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, x[pick].float())
    smoe.smoe_dense_matvec(torch.zeros_like(W), x, y)
    torch.cuda.synchronize()
    assert bool((y == 0).all())


def _quantize(smoe, W):
    cols = W.shape[-1]
    lead = W.shape[:-1]
    codes = torch.full(lead + (cols // 2,), 0xAA, dtype=torch.uint8, device="cuda")
    scale = torch.full(lead + (cols // 64,), -7.0, dtype=torch.bfloat16, device="cuda")
    bias = torch.full(lead + (cols // 64,), -7.0, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_quantize_q4(W, codes, scale, bias)
    torch.cuda.synchronize()
    return codes, scale, bias


def _special_groups(W):
    """Plant the degenerate groups: constant, all zero with a -0, a ladder with
    exact halves, one huge outlier."""
    W = W.clone()
    r = W.view(-1, W.shape[-1])
    if r.shape[1] >= 256 and r.shape[0] >= 2:
        r[0, 0:64] = -1.25
        r[0, 64:128] = 0.0
        r[0, 64 + 5] = -0.0
        lad = torch.arange(64, device=W.device) % 16
        r[0, 128:192] = (lad * 1.0).to(torch.bfloat16)
        r[0, 128 + 3] = 2.5
        r[0, 128 + 4] = 3.5
        r[1, 200] = 3.0e4
        if r.shape[1] >= 320:                              # scale below binary32's normal range
            r[1, 256:320] = torch.linspace(0.0, 1.5e-38, 64, device=W.device).to(torch.bfloat16)
    return W


@pytest.mark.parametrize("shape,spread", [((1, 64), 0.0), ((3, 192), 0.0), ((5, 4096), 4.0),
                                          ((768, 2048), 0.0), ((8, 768, 2048), 2.0),
                                          ((2048, 1536), 0.0)])
def test_quantize_q4_bit_exact(smoe, orc, shape, spread):
    W = _special_groups(synth.dense_weights(shape, seed=sum(shape), device="cuda", row_spread=spread))
    codes, scale, bias = _quantize(smoe, W)
    cols = shape[-1]
    c_ref, s_ref, b_ref = orc.quantize_q4(bits(W).reshape(-1, cols))
    assert np.array_equal(host(codes).reshape(-1, cols // 2), c_ref)
    assert np.array_equal(host(scale).reshape(-1, cols // 64), s_ref)
    assert np.array_equal(host(bias).reshape(-1, cols // 64), b_ref)


def adversarial_groups(n_groups, seed):
    """bf16 weights [n_groups, 64] built to sit on or next to the midpoints
    between quantisation levels: exact ties with scales that are not powers of
    two (the 17/2 case among them), weights of magnitude 2^-100 .. 2^-1 beside
    a minimum of -0.09375 whose scale 1/16 puts it on a midpoint, groups whose
    scale is below 2^-126, groups of weights near 2^124 (scale above 2^120),
    and random groups of very different magnitudes."""
    g = np.random.default_rng(seed)
    out = np.zeros((n_groups, 64), dtype=np.float32)
    for i in range(n_groups):
        kind = i % 6
        if kind == 0:                                      # ties at mn + s (k + 1/2)
            s = np.float32(g.integers(129, 256)) * np.float32(2.0 ** int(g.integers(-20, 0)))
            mn = np.float32(-g.integers(1, 256) * 2.0 ** int(g.integers(-16, -4)))
            v = mn + s * (g.integers(0, 15, 64) + 0.5)
            v[0], v[1] = mn, mn + 15 * s
            out[i] = v
        elif kind == 1:                                    # tiny weights beside a midpoint minimum
            out[i] = g.choice([-1, 1], 64) * 2.0 ** -g.integers(1, 120, 64).astype(np.float64)
            out[i, 0], out[i, 1] = -0.09375, 0.84375
        elif kind == 2:                                    # scale below 2^-126
            out[i] = g.integers(0, 61, 64) * 2.0 ** -135
        elif kind == 3:                                    # scale above 2^120
            out[i] = g.standard_normal(64) * 2.0 ** 123
        elif kind == 4:
            out[i, :3] = [-155 * 2.0 ** -14, 164 * 2.0 ** -14, 205 * 2.0 ** -17]   # (w - mn) / s = 17/2
            out[i, 3:] = g.standard_normal(61) * 0.004
        else:
            out[i] = g.standard_normal(64) * np.exp(3 * g.standard_normal())
    return bits(torch.from_numpy(out).to(torch.bfloat16))


@pytest.mark.parametrize("code_bits", [4, 2])
def test_quantize_adversarial_groups_bit_exact(smoe, orc, code_bits):
    """Both quantisers on groups planted on and next to the midpoints between
    levels (where a quotient with any rounding error picks the wrong code):
    codes, scales and biases equal the oracle's exact nearest-level codes."""
    Wb = adversarial_groups(6 * 512, seed=code_bits).reshape(-1, 512)
    W = from_bits(Wb).cuda()
    rows, cols = Wb.shape
    codes = torch.empty((rows, cols * code_bits // 8), dtype=torch.uint8, device="cuda")
    scale = torch.empty((rows, cols // 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.empty_like(scale)
    (smoe.smoe_quantize_q4 if code_bits == 4 else smoe.smoe_quantize_q2)(W, codes, scale, bias)
    torch.cuda.synchronize()
    c_ref, s_ref, b_ref = (orc.quantize_q4 if code_bits == 4 else orc.quantize_q2)(Wb)
    assert np.array_equal(host(scale), s_ref) and np.array_equal(host(bias), b_ref)
    assert np.array_equal(host(codes), c_ref)


def all_tie_groups(n_groups, levels, seed):
    """bf16 weights [n_groups, 64] of which 62 per group sit exactly on a
    midpoint mn + s (k + 1/2) between two of the `levels` + 1 levels, the other
    two being the group's least and greatest weight (mn and mn + levels * s).
    s = c * 2^e with c odd and below 8, so the quantiser's scale
    bf16((mx - mn) / levels) is s itself and every quotient is an exact
    half; each such code is decided by the halves-to-even rule alone."""
    g = np.random.default_rng(seed)
    out = np.zeros((n_groups, 64), dtype=np.float64)
    for i in range(n_groups):
        e = int(g.integers(-30, 10))
        s = int(g.choice([1, 3, 5, 7])) * 2.0 ** e
        mn = -int(g.integers(0, 64)) * 2.0 ** (e - 1)
        v = mn + s * (g.integers(0, levels, 64) + 0.5)
        v[0], v[1] = mn, mn + levels * s
        out[i] = g.permutation(v)
    w = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(w.double().numpy(), out)            # every value exact in bf16
    return bits(w)


@pytest.mark.parametrize("code_bits", [4, 2])
@pytest.mark.parametrize("rows,cols", [(37, 576), (1024, 512)])
def test_quantize_all_tie_groups_bit_exact(smoe, orc, code_bits, rows, cols):
    """Every group of every warp step holds 62 exact ties, so every lane queues
    the most bytes a group can need re-deciding and the queue flushes many
    times within each step; 333 groups leave a partial last step.  Codes,
    scales and biases equal the oracle's."""
    levels = 15 if code_bits == 4 else 3
    Wb = all_tie_groups(rows * cols // 64, levels, seed=rows + code_bits).reshape(rows, cols)
    W = from_bits(Wb).cuda()
    codes = torch.empty((rows, cols * code_bits // 8), dtype=torch.uint8, device="cuda")
    scale = torch.empty((rows, cols // 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.empty_like(scale)
    (smoe.smoe_quantize_q4 if code_bits == 4 else smoe.smoe_quantize_q2)(W, codes, scale, bias)
    torch.cuda.synchronize()
    c_ref, s_ref, b_ref = (orc.quantize_q4 if code_bits == 4 else orc.quantize_q2)(Wb)
    assert np.array_equal(host(scale), s_ref) and np.array_equal(host(bias), b_ref)
    assert np.array_equal(host(codes), c_ref)


def test_quantize_q4_full_layer_tensor(smoe, orc):
    """A 30B layer's gate tensor (128 x 768 x 2048 bf16, 402 MB), as the
    benchmark runs it: 64 sampled rows bit-exact against the oracle, and the
    round trip of every weight within half a scale step."""
    E, F, D = 128, 768, 2048
    W = synth.dense_weights((E, F, D), seed=11, device="cuda")
    codes, scale, bias = _quantize(smoe, W)
    rows = np.random.default_rng(1).integers(0, E * F, 64)
    Wr = bits(W.view(E * F, D)[torch.from_numpy(rows).cuda()])
    c_ref, s_ref, b_ref = orc.quantize_q4(Wr)
    assert np.array_equal(host(codes.view(E * F, D // 2))[rows], c_ref)
    assert np.array_equal(host(scale.view(E * F, D // 64))[rows], s_ref)
    assert np.array_equal(host(bias.view(E * F, D // 64))[rows], b_ref)
    # round trip on the device, every weight
    c = codes.view(E * F, D // 2)
    q = torch.stack([c & 0x0F, c >> 4], dim=-1).view(E * F, D // 64, 64).float()
    s = scale.view(E * F, D // 64, 1).float()
    b = bias.view(E * F, D // 64, 1).float()
    err = (s * q + b - W.view(E * F, D // 64, 64).float()).abs()
    assert bool((err <= s * (0.5 + 2.0 ** -16)).all())
