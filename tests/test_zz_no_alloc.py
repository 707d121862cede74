"""smoe_moe_decode_noalloc: decode without a workspace, for callers that cannot
allocate device memory (latency-bound serving loops, services whose device
memory is fixed at start-up, plug-ins whose host owns the device memory).  Its output must match the
workspace entry point's, call after call: the fixed scratch keeps the previous
call's contents, so two calls in a row are checked.  This file is collected
last so that a failure here comes after every other test has run."""
import numpy as np
import pytest
import torch

from quantised_expert_ffn_gb300 import synth
from tests.util import bf16_f64, host, rel_l2

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def smoe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe as m
    return m


@pytest.mark.parametrize("D,E,K,F", [(2048, 128, 8, 768), (4096, 128, 8, 1536), (128, 16, 4, 128)])
def test_noalloc_matches_workspace_decode_twice(smoe, D, E, K, F):
    """Same kernels, same arithmetic: the output, ids and weights equal the
    workspace call's bit for bit, on two calls in a row, and the fixed
    scratch's status word reads 0 after each."""
    W = synth.layer_weights(D, E, F, K, seed=4242, device="cuda", rms_norm=True)
    L = smoe.Layer(W)
    assert smoe.smoe_workspace_bytes(L, 1) <= smoe.SMOE_DECODE_NOALLOC_MAX_BYTES
    ws = smoe.workspace(L, 1)
    xs = synth.hidden(2, D, seed=99, device="cuda")
    for t in range(2):                                   # two calls in a row
        y_ref = torch.empty_like(xs[t])
        idx_ref = torch.empty(K, dtype=torch.int32, device="cuda")
        w_ref = torch.empty(K, dtype=torch.float32, device="cuda")
        smoe.smoe_moe_decode(L, xs[t], y_ref, idx_ref, w_ref, None, ws)
        y = torch.empty_like(xs[t])
        idx = torch.full((K,), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros(K, dtype=torch.float32, device="cuda")
        smoe.smoe_moe_decode_noalloc(L, xs[t], y, idx, w)
        assert smoe.smoe_moe_decode_noalloc_status() == 0
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref)
        assert torch.equal(w, w_ref)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        assert rel_l2(bf16_f64(host(y)), bf16_f64(host(y_ref))) <= TOL
    assert smoe.smoe_read_device_status(ws) == 0


def test_noalloc_rejects_layers_beyond_its_scratch(smoe):
    W = synth.layer_weights(8192, 16, 2048, 8, seed=1, device="cuda")
    L = smoe.Layer(W)
    assert smoe.smoe_workspace_bytes(L, 1) > smoe.SMOE_DECODE_NOALLOC_MAX_BYTES
    x = torch.zeros(8192, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_moe_decode_noalloc(L, x, torch.empty_like(x))
    assert e.value.status == smoe.SMOE_ERR_WORKSPACE


def test_noalloc_status_reports_a_device_error_and_the_next_call_clears_it(smoe):
    """A device-side error of a no-workspace call is readable afterwards through
    smoe_moe_decode_noalloc_status: with the grid-barrier wait limit at 0 the
    call's barriers give up (SMOE_ERR_TIMEOUT); with the limit restored the
    next call clears the word and equals the workspace call bit for bit."""
    W = synth.layer_weights(512, 16, 128, 4, seed=5, device="cuda", rms_norm=True)
    L = smoe.Layer(W)
    x = synth.hidden(1, 512, seed=6, device="cuda")[0]
    y = torch.empty_like(x)
    default = smoe.smoe_get_grid_wait_limit()
    try:
        smoe.smoe_set_grid_wait_limit(0)
        for _ in range(20):             # a call whose barriers all happen to pass at once reads 0
            smoe.smoe_moe_decode_noalloc(L, x, y)
            st = smoe.smoe_moe_decode_noalloc_status()
            if st != 0:
                break
        assert st == smoe.SMOE_ERR_TIMEOUT
    finally:
        smoe.smoe_set_grid_wait_limit(default)
    smoe.smoe_moe_decode_noalloc(L, x, y)
    assert smoe.smoe_moe_decode_noalloc_status() == 0
    y_ref = torch.empty_like(x)
    smoe.smoe_moe_decode(L, x, y_ref, ws=smoe.workspace(L, 1))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_q2_layer(smoe):
    """An SMOE-Q2 layer through the fixed scratch equals the workspace call."""
    W = synth.layer_weights(2048, 128, 768, 8, seed=4343, device="cuda", rms_norm=True, code_bits=2)
    L = smoe.Layer(W)
    ws = smoe.workspace(L, 1)
    x = synth.hidden(1, 2048, seed=98, device="cuda")[0]
    y_ref, y = torch.empty_like(x), torch.empty_like(x)
    smoe.smoe_moe_decode(L, x, y_ref, ws=ws)
    smoe.smoe_moe_decode_noalloc(L, x, y)
    assert smoe.smoe_moe_decode_noalloc_status() == 0
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
