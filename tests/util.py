"""Helpers shared by the tests: moving the seeded inputs between torch and the
oracle's numpy view (bf16 as uint16 bits)."""
import numpy as np
import torch

from oracle.oracle import layer_from_weights as oracle_layer  # noqa: F401  (re-exported)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host numpy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return bits(t)
    return t.detach().cpu().contiguous().numpy()


def bf16_f64(a: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
            np.float64)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_row_rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64).reshape(np.shape(b)[0], -1)
    b = np.asarray(b, np.float64).reshape(np.shape(b)[0], -1)
    return max(rel_l2(a[i], b[i]) for i in range(b.shape[0]))


def margin_tokens(OL, n, seed, *, alpha=None, tau_factor=10.0, max_tries=50):
    """n hidden states (bf16 [n, D], host) whose oracle routing has every
    adjacent gap among ranks 1..k+1 at least tau_factor * tau, with
    tau = 64 * 2^-24 * max_e sum_d |Wr[e][d] xn[d]| (so the GPU's fp32 logits
    rank the same experts in the same order).  Candidates come from the seeded
    generator (independent, or sharing a direction when alpha is given)."""
    from oracle import oracle
    from quantised_expert_ffn_gb300 import synth
    D, k = OL.d_model, OL.top_k
    Wabs = np.abs(bf16_f64(OL.router_w))
    keep = []
    for attempt in range(max_tries):
        if alpha is None:
            cand = bits(synth.hidden(2 * n, D, seed=seed * 7919 + attempt))
        else:
            cand = bits(synth.correlated_hidden(2 * n, D, alpha, seed=seed * 7919 + attempt))
        for r in cand:
            xn = oracle.rmsnorm(OL, r)
            lg = oracle.router_logits(OL, xn)
            tau = 64 * 2.0 ** -24 * float((Wabs @ np.abs(bf16_f64(xn))).max())
            top = np.sort(lg)[::-1][:k + 1]
            if top.size < 2 or np.all(top[:-1] - top[1:] >= tau_factor * tau):
                keep.append(r)
                if len(keep) == n:
                    return np.stack(keep)
    raise RuntimeError("could not draw enough tokens with routing margins")


def margin_ok(orc, OL, x_row, Wabs, K, factor=10.0):
    """Whether the oracle's top-(K+1) adjacent logit gaps of one token are all
    at least factor * tau (see margin_tokens); also returns the logits."""
    xn = orc.rmsnorm(OL, x_row)
    lg = orc.router_logits(OL, xn)
    tau = 64 * 2.0 ** -24 * float((Wabs @ np.abs(bf16_f64(xn))).max())
    top = np.sort(lg)[::-1][:K + 1]
    return bool(np.all(top[:-1] - top[1:] >= factor * tau)), lg


def zipf_chunk(orc, OL, router_w, T=64, seed=31):
    """T hidden states (bf16 bits [T, D]) whose router logits carry a Zipf(1.2)
    bias over a seeded expert permutation, drawn with routing margins, at the
    first bias scale whose largest bucket holds 30-60 tokens.  Returns
    (x, bucket sizes) or None."""
    from quantised_expert_ffn_gb300 import synth
    K, E = OL.top_k, OL.n_experts
    Wabs = np.abs(bf16_f64(OL.router_w))
    for scale in (1.0, 1.5, 2.0, 3.0, 4.0, 6.0):
        cand = bits(synth.zipf_bias_hidden(4 * T, router_w.float(), 1.2, scale, seed=seed))
        keep = []
        for r in cand:
            if margin_ok(orc, OL, r, Wabs, K)[0]:
                keep.append(r)
            if len(keep) == T:
                break
        if len(keep) < T:
            continue
        x = np.stack(keep)
        idx_ref = np.stack([orc.topk(orc.router_logits(OL, orc.rmsnorm(OL, r)), K) for r in x])
        sizes = np.bincount(idx_ref.ravel(), minlength=E)
        if 30 <= sizes.max() <= 60:
            return x, sizes
    return None
