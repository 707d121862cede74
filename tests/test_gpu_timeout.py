"""The one-kernel decode's grid barriers: the timeout path and co-residency.

A grid-wide barrier is a global-memory poll bounded in time; the host sets
that bound (smoe_set_grid_wait_limit).  With the bound at 0 every barrier that
has to wait gives up at once: the call must return, leave SMOE_ERR_TIMEOUT in
the device status word and leave the GPU usable -- the next call on a cleared
workspace is correct again.  The kernel is a cooperative launch, so two
persistent decodes enqueued on two unordered streams never run interleaved
(which would leave each one's barriers waiting on CTAs that cannot start)."""
import pytest
import torch

from quantised_expert_ffn_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smoe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe as m
    return m


def _stack(smoe, n, D, E, K, F, seed):
    W = [synth.layer_weights(D, E, F, K, seed=seed + i, device="cuda", rms_norm=True) for i in range(n)]
    L = [smoe.Layer(w) for w in W]
    return W, L, smoe.LayerTable(L, "cuda")


def test_zero_grid_wait_limit_reports_timeout_then_recovers(smoe):
    W, L, table = _stack(smoe, 6, 512, 16, 4, 128, seed=70)
    x = synth.hidden(1, 512, seed=71, device="cuda")[0]
    ws = smoe.workspace(L[0], 1)
    y_ref = torch.empty_like(x)
    smoe.smoe_moe_decode_layers(table, x, y_ref, ws=ws)
    assert smoe.smoe_read_device_status(ws) == 0
    default = smoe.smoe_get_grid_wait_limit()
    assert default == 200_000_000
    y = torch.empty_like(x)
    try:
        smoe.smoe_set_grid_wait_limit(0)
        for _ in range(3):                                   # 18 barriers per call, none may wait
            smoe.smoe_moe_decode_layers(table, x, y, ws=ws)
        torch.cuda.synchronize()
    finally:
        smoe.smoe_set_grid_wait_limit(default)
    assert smoe.smoe_read_device_status(ws) == smoe.SMOE_ERR_TIMEOUT
    smoe.smoe_workspace_init(ws)                             # clears the status word
    smoe.smoe_moe_decode_layers(table, x, y, ws=ws)
    assert smoe.smoe_read_device_status(ws) == 0
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    # the single-layer entry point as well
    y1_ref, y1 = torch.empty_like(x), torch.empty_like(x)
    smoe.smoe_moe_decode(L[0], x, y1_ref, ws=ws)
    smoe.smoe_moe_decode(L[0], x, y1, ws=ws)
    assert smoe.smoe_read_device_status(ws) == 0
    assert torch.equal(y1.view(torch.int16), y1_ref.view(torch.int16))


def test_two_streams_of_persistent_decodes_stay_correct(smoe):
    """Two 30B-shaped decode stacks on two streams with no ordering between
    them, each launch occupying one CTA per SM: with a cooperative launch one
    grid waits for the other; both results equal their one-stream runs and
    no barrier times out."""
    _, La, ta = _stack(smoe, 3, 2048, 128, 8, 768, seed=80)
    _, Lb, tb = _stack(smoe, 3, 2048, 128, 8, 768, seed=90)
    xs = synth.hidden(8, 2048, seed=81, device="cuda")
    wsa, wsb = smoe.workspace(La[0], 1), smoe.workspace(Lb[0], 1)
    ref_a = torch.empty_like(xs)
    ref_b = torch.empty_like(xs)
    for t in range(8):
        smoe.smoe_moe_decode_layers(ta, xs[t], ref_a[t], ws=wsa)
        smoe.smoe_moe_decode_layers(tb, xs[t], ref_b[t], ws=wsb)
    torch.cuda.synchronize()
    ya, yb = torch.empty_like(xs), torch.empty_like(xs)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(4):
        for t in range(8):
            smoe.smoe_moe_decode_layers(ta, xs[t], ya[t], ws=wsa, stream=sa)
            smoe.smoe_moe_decode_layers(tb, xs[t], yb[t], ws=wsb, stream=sb)
    torch.cuda.synchronize()
    assert smoe.smoe_read_device_status(wsa) == 0
    assert smoe.smoe_read_device_status(wsb) == 0
    assert torch.equal(ya.view(torch.int16), ref_a.view(torch.int16))
    assert torch.equal(yb.view(torch.int16), ref_b.view(torch.int16))
