"""The prefill chunk's expert FFN outputs, slot by slot, against the oracle.

smoe_moe_prefill_chunk_experts returns o[t][i], the unweighted output of
expert idx[t][i] for token t, as the chunk's grouped GEMMs (one read of each
union expert) computed it.  Each is compared with the oracle's o for the same
token and expert: max over (t, i) of ||gpu - oracle|| / ||oracle|| <= 2e-3, so
an error in the tensor-core FFN cannot hide behind the residual (which
dominates y).  Cases: the 30B and 235B shapes, SMOE-Q4 and SMOE-Q2, chunks of
1, 45 and 64 tokens (independent, or sharing a direction so the union holds
~60-100 experts), a Zipf(1.2)-skewed chunk, and a chunk whose tokens all
route alike (every bucket full), a ragged shape (6 and 10 groups: scales read
group by group, an odd count of down tiles) and the largest layer taken;
then weights written by the library's own
quantiser (biases at the group minimum, not -8 s; some groups with scales
below fp16's normal range) through decode and prefill; the fp16 range
bound of the tensor-core path; and one chunk five times through the same
workspace, bit-identical each time (units are claimed dynamically)."""
import os

import numpy as np
import pytest
import torch

from quantised_expert_ffn_gb300 import synth
from tests.util import (bf16_f64, bits, from_bits, host, margin_tokens, max_row_rel_l2, oracle_layer,
                        rel_l2, zipf_chunk)

pytestmark = pytest.mark.gpu
TOL = 2e-3      # fp32 expert outputs vs the oracle; bf16 residuals vs the oracle's bf16 y
SIMT = os.environ.get("SMOE_PREFILL_PATH") == "simt"     # the CUDA-core engine (fp32, Q4 only)

# k384: D/64 = 6 and F/64 = 10 groups (scales read group by group, not 8 at a
# time; 3 and 5 two-group stages) and an odd count of 128-row down tiles (one
# tile per unit); max: the largest layer the library takes (d_model 8192,
# 256 experts, top-16).
SHAPES = {"30b": (2048, 128, 8, 768), "235b": (4096, 128, 8, 1536), "k384": (384, 32, 4, 640),
          "max": (8192, 256, 16, 1024)}
ALPHA = {"30b": 0.7, "235b": 0.6}


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


def dev(a):
    if a.dtype == np.uint16:
        return from_bits(a).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_prefill(smoe, L, x, T, K, D):
    ws = smoe.workspace(L, T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    eo = torch.full((T, K, D), float("nan"), dtype=torch.float32, device="cuda")
    smoe.smoe_moe_prefill_chunk_experts(L, dev(x), T, y, eo, idx, w, ws)
    torch.cuda.synchronize()
    return dict(y=y, idx=idx, w=w, eo=eo, status=smoe.smoe_read_device_status(ws), ws=ws)


def slot_errors(eo_gpu, eo_ref):
    T, K, D = eo_ref.shape
    return np.array([[rel_l2(eo_gpu[t, i], eo_ref[t, i]) for i in range(K)] for t in range(T)])


CASES = [("30b", 4, 1, "indep"), ("30b", 4, 45, "corr"), ("30b", 4, 64, "corr"),
         ("235b", 4, 1, "indep"), ("235b", 4, 45, "corr"), ("235b", 4, 64, "corr"),
         ("30b", 2, 1, "indep"), ("30b", 2, 64, "corr"), ("235b", 2, 45, "corr"),
         ("30b", 4, 64, "zipf"), ("30b", 2, 64, "zipf"),
         ("30b", 4, 64, "one_bucket"), ("235b", 2, 64, "one_bucket"),
         ("k384", 4, 45, "indep"), ("k384", 2, 64, "indep"), ("max", 4, 8, "indep"), ("max", 2, 8, "indep")]


@pytest.mark.parametrize("name,code_bits,T,kind", CASES)
def test_prefill_expert_outputs_per_slot(smoe, orc, name, code_bits, T, kind):
    if SIMT and code_bits == 2:
        pytest.skip("the CUDA-core prefill engine takes SMOE-Q4 only")
    D, E, K, F = SHAPES[name]
    W = synth.layer_weights(D, E, F, K, seed=500 + code_bits, device="cuda", rms_norm=True,
                            code_bits=code_bits)
    OL = oracle_layer(W)
    L = smoe.Layer(W)
    if kind == "indep":
        x = margin_tokens(OL, T, seed=600 + T)
    elif kind == "corr":
        x = margin_tokens(OL, T, seed=610 + T, alpha=ALPHA[name])
    elif kind == "zipf":
        got = zipf_chunk(orc, OL, W.router_w, T=T, seed=31)
        assert got is not None, "no bias scale gave a 30-60 token bucket"
        x, sizes = got
        assert sizes.max() >= 30
    else:
        x = np.repeat(margin_tokens(OL, 1, seed=620), T, axis=0)
    r = run_prefill(smoe, L, x, T, K, D)
    assert r["status"] == 0
    ref = orc.moe_tokens_experts(OL, x)
    assert np.array_equal(host(r["idx"]), ref["idx"])
    np.testing.assert_allclose(host(r["w"]), ref["w"], rtol=2e-5)
    err = slot_errors(host(r["eo"]), ref["expert_out"])
    assert err.max() <= TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))
    assert max_row_rel_l2(bf16_f64(host(r["y"])), bf16_f64(ref["y_bf16"])) <= TOL
    if kind == "one_bucket":
        assert len(np.unique(host(r["idx"]))) == K
    # the residual output is the one smoe_moe_prefill_chunk gives, bit for bit
    y2 = torch.empty_like(r["y"])
    smoe.smoe_moe_prefill_chunk(L, dev(x), T, y2, ws=r["ws"])
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int16), r["y"].view(torch.int16))


def quantised_layer(smoe, D, E, F, K, code_bits, seed):
    """A layer whose gate, up and down matrices are bf16 N(0, 0.02^2) weights
    quantised by the library (bias = group minimum, scale = range / levels);
    every 7th row of each matrix scaled by 1e-4 first, so its groups' scales
    fall below 6.1e-5 (fp16 subnormal on the tensor-core path)."""
    W = synth.layer_weights(D, E, F, K, seed=seed, device="cuda", rms_norm=True, code_bits=code_bits)
    quant = smoe.smoe_quantize_q4 if code_bits == 4 else smoe.smoe_quantize_q2
    for n, shape in (("gate", (E, F, D)), ("up", (E, F, D)), ("down", (E, D, F))):
        wb = synth.dense_weights(shape, seed=seed + len(n), device="cuda")
        wb[:, ::7, :] = (wb[:, ::7, :].float() * 1e-4).to(torch.bfloat16)
        quant(wb, getattr(W, n + "_q"), getattr(W, n + "_s"), getattr(W, n + "_b"))
    torch.cuda.synchronize()
    s = W.gate_s.float()
    assert bool((s[:, ::7] < 6.1e-5).all()) and bool((s[:, 1::7] > 1e-4).all())
    assert not bool((W.gate_b.float() == -8 * s).all())          # general biases
    return W


@pytest.mark.parametrize("name,code_bits", [("30b", 4), ("235b", 4), ("30b", 2)])
def test_quantised_weights_through_decode_and_prefill(smoe, orc, name, code_bits):
    if SIMT and code_bits == 2:
        pytest.skip("the CUDA-core prefill engine takes SMOE-Q4 only")
    D, E, K, F = SHAPES[name]
    W = quantised_layer(smoe, D, E, F, K, code_bits, seed=700)
    OL = oracle_layer(W)
    L = smoe.Layer(W)
    T = 45
    x = margin_tokens(OL, T, seed=701, alpha=ALPHA[name])
    ref = orc.moe_tokens_experts(OL, x)
    # prefill: every slot's expert output
    r = run_prefill(smoe, L, x, T, K, D)
    assert r["status"] == 0
    assert np.array_equal(host(r["idx"]), ref["idx"])
    err = slot_errors(host(r["eo"]), ref["expert_out"])
    assert err.max() <= TOL, err.max()
    assert max_row_rel_l2(bf16_f64(host(r["y"])), bf16_f64(ref["y_bf16"])) <= TOL
    # decode: every expert output of a few tokens
    ws1 = smoe.workspace(L, 1)
    for t in range(0, T, 11):
        y = torch.empty(D, dtype=torch.bfloat16, device="cuda")
        idx = torch.empty(K, dtype=torch.int32, device="cuda")
        eo = torch.empty((K, D), dtype=torch.float32, device="cuda")
        smoe.smoe_moe_decode(L, dev(x[t]), y, idx, None, eo, ws1)
        torch.cuda.synchronize()
        assert np.array_equal(host(idx), ref["idx"][t])
        e = max(rel_l2(host(eo)[i], ref["expert_out"][t, i]) for i in range(K))
        assert e <= TOL, (t, e)
        assert rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"][t])) <= TOL
    assert smoe.smoe_read_device_status(ws1) == 0


def test_prefill_reports_values_beyond_fp16(smoe, orc):
    """The tensor-core prefill carries weights, inputs and h in fp16: a group
    whose levels reach past 65504, or an input above it, sets SMOE_ERR_RANGE;
    decode (fp32) computes the same layer within the bar."""
    if SIMT:
        pytest.skip("the CUDA-core prefill engine has no fp16 bound")
    D, E, K, F = 2048, 16, 4, 256
    W = synth.layer_weights(D, E, F, K, seed=800, device="cuda", rms_norm=True)
    W.down_b[:, :, 0] = 7.0e4                          # first group of every down row, all experts
    OL = oracle_layer(W)
    L = smoe.Layer(W)
    x = margin_tokens(OL, 8, seed=801)
    r = run_prefill(smoe, L, x, 8, K, D)
    assert r["status"] == smoe.SMOE_ERR_RANGE
    ref = orc.moe_tokens_experts(OL, x)
    ws1 = smoe.workspace(L, 1)
    y = torch.empty(D, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_moe_decode(L, dev(x[0]), y, ws=ws1)
    torch.cuda.synchronize()
    assert smoe.smoe_read_device_status(ws1) == 0
    assert rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"][0])) <= TOL
    # an input beyond fp16's range (no RMSNorm before the router and FFN)
    W2 = synth.layer_weights(D, E, F, K, seed=802, device="cuda", rms_norm=False)
    L2 = smoe.Layer(W2)
    x2 = bits(synth.hidden(4, D, seed=803))
    x2[1, 17] = bits(torch.tensor([1.0e5], dtype=torch.bfloat16))[0]
    r2 = run_prefill(smoe, L2, x2, 4, K, D)
    assert r2["status"] == smoe.SMOE_ERR_RANGE
    # in range again: a clean workspace reads 0
    r3 = run_prefill(smoe, L2, bits(synth.hidden(4, D, seed=804)), 4, K, D)
    assert r3["status"] == 0


@pytest.mark.parametrize("name,code_bits", [("235b", 4), ("30b", 4), ("30b", 2)])
def test_prefill_repeats_bit_identical(smoe, orc, name, code_bits):
    """The tensor-core kernels take their units from a device counter, so which
    CTA computes which unit differs from call to call; each unit's arithmetic
    does not depend on it.  The same chunk through the same workspace, five
    times in a row: ids, weights, per-slot expert outputs and y equal bit for
    bit every time, and the status word stays 0 (the counters are reset by
    each call)."""
    D, E, K, F = SHAPES[name]
    W = synth.layer_weights(D, E, F, K, seed=900 + code_bits, device="cuda", rms_norm=True,
                            code_bits=code_bits)
    OL = oracle_layer(W)
    L = smoe.Layer(W)
    x = margin_tokens(OL, 64, seed=901, alpha=ALPHA[name])
    ws = smoe.workspace(L, 64)
    first = None
    for _ in range(5):
        y = torch.empty((64, D), dtype=torch.bfloat16, device="cuda")
        idx = torch.empty((64, K), dtype=torch.int32, device="cuda")
        w = torch.empty((64, K), dtype=torch.float32, device="cuda")
        eo = torch.full((64, K, D), float("nan"), dtype=torch.float32, device="cuda")
        smoe.smoe_moe_prefill_chunk_experts(L, dev(x), 64, y, eo, idx, w, ws)
        torch.cuda.synchronize()
        assert smoe.smoe_read_device_status(ws) == 0
        got = (host(idx), host(w).view(np.int32), host(eo).view(np.int32), host(y).view(np.int16))
        if first is None:
            first = got
            continue
        for a, b in zip(first, got):
            assert np.array_equal(a, b)
