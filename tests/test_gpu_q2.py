"""GPU parity of SMOE-Q2 (2-bit codes, the pages' Q2 vault): the one-kernel
decode, the FFN with given ids, the one-launch stack, and the Q2 quantiser,
through the C ABI against the CPU oracle on the same seeded bytes.  Bars as
for SMOE-Q4: ids bit-exact, values within 2e-3 relative L2, quantiser bytes
bit-exact."""
import numpy as np
import pytest
import torch

from quantised_expert_ffn_gb300 import synth
from tests.util import bf16_f64, bits, from_bits, host, margin_tokens, max_row_rel_l2, oracle_layer, rel_l2

pytestmark = pytest.mark.gpu
TOL = 2e-3      # fp32 expert outputs vs the oracle; bf16 residuals vs the oracle's bf16 y

SHAPES = {"30b": (2048, 128, 8, 768), "235b": (4096, 128, 8, 1536), "f1536": (1536, 64, 6, 384),
          "f512": (512, 16, 4, 128), "one": (512, 1, 1, 128)}


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


def q2_layer(name, seed=1337):
    D, E, K, F = SHAPES[name]
    W = synth.layer_weights(D, E, F, K, seed=seed, device="cuda", rms_norm=True, code_bits=2)
    return W, oracle_layer(W)


def dev(a):
    return from_bits(a).cuda()


@pytest.mark.parametrize("name,ntok", [("30b", 4), ("235b", 2), ("f1536", 3), ("f512", 3), ("one", 2)])
def test_q2_decode_against_oracle(smoe, orc, name, ntok):
    W, OL = q2_layer(name)
    D, K = W.d_model, W.top_k
    assert OL.code_bits == 2 and W.gate_q.shape[-1] == D // 4
    x = margin_tokens(OL, ntok, seed=200 + ntok)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, 1)
    for t in range(ntok):
        xt = dev(x[t])
        y = torch.empty_like(xt)
        idx = torch.empty(K, dtype=torch.int32, device="cuda")
        w = torch.empty(K, dtype=torch.float32, device="cuda")
        eo = torch.empty((K, D), dtype=torch.float32, device="cuda")
        smoe.smoe_moe_decode(L, xt, y, idx, w, eo, ws)
        torch.cuda.synchronize()
        ref = orc.moe_token(OL, x[t])
        assert np.array_equal(host(idx), ref["idx"])
        np.testing.assert_allclose(host(w), ref["w"], rtol=2e-5)
        assert max_row_rel_l2(host(eo), ref["expert_out"]) <= TOL
        assert rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"])) <= TOL
    assert smoe.smoe_read_device_status(ws) == 0


@pytest.mark.parametrize("name", ["30b", "235b"])
def test_q2_ffn_given_ids(smoe, orc, name):
    W, OL = q2_layer(name, seed=7)
    D, E, K = W.d_model, W.n_experts, W.top_k
    rng = np.random.default_rng(5)
    x = bits(synth.hidden(1, D, seed=32))[0]
    idx = rng.choice(E, K, replace=False).astype(np.int32)
    w = rng.uniform(0.05, 1.0, K).astype(np.float32)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, 1)
    y = torch.empty(D, dtype=torch.bfloat16, device="cuda")
    eo = torch.empty((K, D), dtype=torch.float32, device="cuda")
    smoe.smoe_moe_ffn_decode(L, dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), y, eo, ws)
    torch.cuda.synchronize()
    xn = orc.rmsnorm(OL, x)
    o = np.stack([orc.expert_ffn(OL, int(e), xn)[0] for e in idx])
    assert max_row_rel_l2(host(eo), o) <= TOL
    y_ref = bf16_f64(x) + (w.astype(np.float64)[:, None] * o).sum(0)
    assert rel_l2(bf16_f64(host(y)), y_ref) <= TOL
    assert smoe.smoe_read_device_status(ws) == 0


@pytest.mark.parametrize("name,n", [("30b", 3), ("f512", 3)])
def test_q2_decode_layers_equals_chained(smoe, name, n):
    D, E, K, F = SHAPES[name]
    Ls = [smoe.Layer(synth.layer_weights(D, E, F, K, seed=600 + i, device="cuda", rms_norm=True, code_bits=2))
          for i in range(n)]
    table = smoe.LayerTable(Ls)
    ws = smoe.workspace(Ls[0], 1)
    x = synth.hidden(1, D, seed=15, device="cuda")[0]
    y = torch.empty_like(x)
    idx = torch.empty((n, K), dtype=torch.int32, device="cuda")
    w = torch.empty((n, K), dtype=torch.float32, device="cuda")
    smoe.smoe_moe_decode_layers(table, x, y, idx, w, ws)
    cur = x.clone()
    for i, L in enumerate(Ls):
        nxt = torch.empty_like(cur)
        ii = torch.empty(K, dtype=torch.int32, device="cuda")
        wi = torch.empty(K, dtype=torch.float32, device="cuda")
        smoe.smoe_moe_decode(L, cur, nxt, ii, wi, ws=ws)
        assert torch.equal(ii, idx[i]) and torch.equal(wi, w[i]), i
        cur = nxt
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), cur.view(torch.int16))
    assert smoe.smoe_read_device_status(ws) == 0


@pytest.mark.parametrize("name,T,alpha", [("f512", 8, None), ("30b", 45, None), ("235b", 64, 0.7),
                                          ("f1536", 5, None)])
def test_q2_prefill_chunk_against_oracle(smoe, orc, name, T, alpha):
    """Q2 prefill on the tensor cores (the Q2 dequant feeds A in the Q4 element
    order): ids bit-exact, values within 2e-3 of the oracle."""
    W, OL = q2_layer(name, seed=11)
    K = W.top_k
    x = margin_tokens(OL, T, seed=300 + T, alpha=alpha)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, T)
    y = torch.empty((T, W.d_model), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    smoe.smoe_moe_prefill_chunk(L, from_bits(x).cuda(), T, y, idx, w, ws)
    torch.cuda.synchronize()
    assert smoe.smoe_read_device_status(ws) == 0
    ref = orc.moe_tokens(OL, x)
    assert np.array_equal(host(idx), ref["idx"])
    np.testing.assert_allclose(host(w), ref["w"], rtol=2e-5)
    assert max_row_rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"])) <= TOL


def test_q2_unsupported_calls_return_status(smoe):
    """Q2 outside its kernels' plans -- prefill with d_model 192 (not a
    multiple of the 128-row tensor-core tile), decode with d_model 128 --
    returns SMOE_ERR_UNSUPPORTED and enqueues nothing; a stack mixing Q2 and
    Q4 layers is an invalid argument."""
    W, _ = q2_layer("f512")
    L = smoe.Layer(W)
    x = synth.hidden(4, 512, seed=1, device="cuda")
    Wo = synth.layer_weights(192, 24, 320, 3, seed=5, device="cuda", rms_norm=True, code_bits=2)
    Lo = smoe.Layer(Wo)
    xo = synth.hidden(4, 192, seed=1, device="cuda")
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_moe_prefill_chunk(Lo, xo, 4, torch.empty_like(xo), ws=smoe.workspace(Lo, 4))
    assert e.value.status == smoe.SMOE_ERR_UNSUPPORTED
    Wt = synth.layer_weights(128, 16, 128, 4, seed=2, device="cuda", rms_norm=True, code_bits=2)
    Lt = smoe.Layer(Wt)
    xt = synth.hidden(1, 128, seed=1, device="cuda")[0]
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_moe_decode(Lt, xt, torch.empty_like(xt), ws=smoe.workspace(Lt, 1))
    assert e.value.status == smoe.SMOE_ERR_UNSUPPORTED
    W4 = synth.layer_weights(512, 16, 128, 4, seed=3, device="cuda", rms_norm=True)
    table = smoe.LayerTable([L, smoe.Layer(W4)])
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_moe_decode_layers(table, x[0], torch.empty_like(x[0]), ws=smoe.workspace(L, 1))
    assert e.value.status == smoe.SMOE_ERR_INVALID_ARG


def _quantize_q2(smoe, W):
    cols = W.shape[-1]
    lead = W.shape[:-1]
    codes = torch.full(lead + (cols // 4,), 0xAA, dtype=torch.uint8, device="cuda")
    scale = torch.full(lead + (cols // 64,), -7.0, dtype=torch.bfloat16, device="cuda")
    bias = torch.full(lead + (cols // 64,), -7.0, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_quantize_q2(W, codes, scale, bias)
    torch.cuda.synchronize()
    return codes, scale, bias


@pytest.mark.parametrize("shape,spread", [((1, 64), 0.0), ((3, 192), 0.0), ((5, 4096), 4.0),
                                          ((8, 768, 2048), 2.0)])
def test_quantize_q2_bit_exact(smoe, orc, shape, spread):
    W = synth.dense_weights(shape, seed=sum(shape) + 1, device="cuda", row_spread=spread)
    r = W.view(-1, shape[-1])
    if r.shape[1] >= 256 and r.shape[0] >= 2:       # constant, +-0, exact halves, tiny-scale groups
        r[0, 0:64] = 0.75
        r[0, 64:128] = 0.0
        r[0, 69] = -0.0
        r[0, 128:192] = (torch.arange(64, device="cuda") % 4).to(torch.bfloat16)
        r[0, 130:133] = torch.tensor([0.5, 1.5, 2.5], device="cuda").to(torch.bfloat16)
        r[1, 192:256] = torch.linspace(0.0, 1.5e-38, 64, device="cuda").to(torch.bfloat16)
    codes, scale, bias = _quantize_q2(smoe, W)
    cols = shape[-1]
    c_ref, s_ref, b_ref = orc.quantize_q2(bits(W).reshape(-1, cols))
    assert np.array_equal(host(codes).reshape(-1, cols // 4), c_ref)
    assert np.array_equal(host(scale).reshape(-1, cols // 64), s_ref)
    assert np.array_equal(host(bias).reshape(-1, cols // 64), b_ref)


def test_quantise_then_decode_q2(smoe, orc):
    """bf16 expert weights quantised to SMOE-Q2 on the GPU, then decoded by the
    one-kernel Q2 decode: the oracle, given the GPU's quantised bytes (checked
    bit-exact first), agrees with the decode."""
    D, E, K, F = 2048, 16, 4, 768
    g = synth.dense_weights((E, F, D), seed=41, device="cuda")
    u = synth.dense_weights((E, F, D), seed=42, device="cuda")
    d = synth.dense_weights((E, D, F), seed=43, device="cuda")
    W = synth.layer_weights(D, E, F, K, seed=44, device="cuda", rms_norm=True, code_bits=2)
    W.gate_q, W.gate_s, W.gate_b = _quantize_q2(smoe, g)
    W.up_q, W.up_s, W.up_b = _quantize_q2(smoe, u)
    W.down_q, W.down_s, W.down_b = _quantize_q2(smoe, d)
    c_ref, s_ref, b_ref = orc.quantize_q2(bits(d).reshape(-1, F))
    assert np.array_equal(host(W.down_q).reshape(-1, F // 4), c_ref)
    assert np.array_equal(host(W.down_s).reshape(-1, F // 64), s_ref)
    OL = oracle_layer(W)
    x = margin_tokens(OL, 2, seed=9)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, 1)
    for t in range(2):
        y = torch.empty(D, dtype=torch.bfloat16, device="cuda")
        idx = torch.empty(K, dtype=torch.int32, device="cuda")
        smoe.smoe_moe_decode(L, dev(x[t]), y, idx, ws=ws)
        torch.cuda.synchronize()
        ref = orc.moe_token(OL, x[t])
        assert np.array_equal(host(idx), ref["idx"])
        assert rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"])) <= TOL


def _margin_ok(orc, OL, r, Wabs, K):
    xn = orc.rmsnorm(OL, r)
    lg = orc.router_logits(OL, xn)
    tau = 64 * 2.0 ** -24 * float((Wabs @ np.abs(bf16_f64(xn))).max())
    top = np.sort(lg)[::-1][:K + 1]
    return bool(np.all(top[:-1] - top[1:] >= 10 * tau))


def test_q2_skewed_prefill_chunk(smoe, orc):
    """SMOE-Q2 prefill of a Zipf(1.2)-biased 64-token chunk whose largest bucket
    holds 30-60 tokens (N up to 64 on the tensor cores) against the oracle."""
    W, OL = q2_layer("30b", seed=23)
    D, E, K = W.d_model, W.n_experts, W.top_k
    Wabs = np.abs(bf16_f64(OL.router_w))
    L = smoe.Layer(W)
    chosen = None
    for scale in (1.0, 1.5, 2.0, 3.0, 4.0, 6.0):
        cand = bits(synth.zipf_bias_hidden(256, W.router_w.float(), 1.2, scale, seed=33))
        keep = [r for r in cand if _margin_ok(orc, OL, r, Wabs, K)][:64]
        if len(keep) < 64:
            continue
        x = np.stack(keep)
        idx_ref = np.stack([orc.topk(orc.router_logits(OL, orc.rmsnorm(OL, r)), K) for r in x])
        sizes = np.bincount(idx_ref.ravel(), minlength=E)
        if 30 <= sizes.max() <= 60:
            chosen = (x, sizes)
            break
    assert chosen is not None, "no bias scale gave a 30-60 token bucket"
    x, sizes = chosen
    ws = smoe.workspace(L, 64)
    y = torch.empty((64, D), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((64, K), dtype=torch.int32, device="cuda")
    smoe.smoe_moe_prefill_chunk(L, from_bits(x).cuda(), 64, y, idx, None, ws)
    torch.cuda.synchronize()
    assert smoe.smoe_read_device_status(ws) == 0
    ref = orc.moe_tokens(OL, x)
    assert np.array_equal(host(idx), ref["idx"])
    assert max_row_rel_l2(bf16_f64(host(y)), bf16_f64(ref["y_bf16"])) <= TOL


def test_q2_ffn_repeated_ids(smoe, orc):
    """SMOE-Q2 FFN with the same expert in several slots."""
    W, OL = q2_layer("f1536", seed=29)
    D, E, K = W.d_model, W.n_experts, W.top_k
    rng = np.random.default_rng(6)
    x = bits(synth.hidden(1, D, seed=34))[0]
    idx = rng.choice(E, K, replace=True).astype(np.int32)
    idx[1] = idx[0]
    idx[3] = idx[0]
    w = rng.uniform(0.05, 1.0, K).astype(np.float32)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, 1)
    y = torch.empty(D, dtype=torch.bfloat16, device="cuda")
    eo = torch.empty((K, D), dtype=torch.float32, device="cuda")
    smoe.smoe_moe_ffn_decode(L, from_bits(x).cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), y, eo, ws)
    torch.cuda.synchronize()
    xn = orc.rmsnorm(OL, x)
    o = np.stack([orc.expert_ffn(OL, int(e), xn)[0] for e in idx])
    assert max_row_rel_l2(host(eo), o) <= TOL
    assert rel_l2(bf16_f64(host(y)), bf16_f64(x) + (w.astype(np.float64)[:, None] * o).sum(0)) <= TOL
