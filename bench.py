"""Benchmark of the routed-MoE hot path on one GB300 (or N replicas).

Headline workload: a 30B-shaped 48-layer MoE decode stack at batch 1
(d_model 2048, 128 experts, top-8, ffn 768, SMOE-Q4 group 64, RMSNorm before
every router), 256 seeded N(0,1) start states.  One step = one decode token
through all 48 layers (router + top-k + fused Q4 expert FFN + weighted
residual sum, per layer), replayed from a CUDA graph; inputs are resident in
HBM and each token reads 1.04 GB of distinct expert weights, more than L2.

The JSON line also carries: the roofline of the step's one kernel (the decode
launch over 48 layers: algorithmic bytes over its CUDA-event time, ncu DRAM
traffic from profiles/ while the kernel's sources match the capture), the
expert FFN alone per call, the end-to-end rate through the C ABI with host
buffers, clocks sampled during the timed region, the oracle's CPU rate, the
SMOE-Q2 decode stack, a 30B-shaped prefill (SMOE-Q4 and SMOE-Q2), the dense
bf16 matvec on the trunk's projection shapes and the LM head, the Q4 and Q2
quantisers, a 235B-shaped 94-layer decode (per-token and per-layer time) and
a 235B-shaped layer-major prefill (prompts of 45, 512 and 4096 tokens in
chunks of 64, tokens correlated so a chunk's union holds ~60-100 experts).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (the only other implementation of
this path) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = ("MoE decode tokens/s (b=1) + expert-FFN effective HBM GB/s vs peak; prefill tok/s")
D30, E, K, F30, L30 = 2048, 128, 8, 768, 48
D235, F235, L235 = 4096, 1536, 94
E30Q = (E, F30, D30)                      # a 30B layer's gate tensor, [E][F][D]
SEED = 1337
PER_LAYER = False   # --per-layer: decode through one smoe_moe_decode call per layer

# sources of the kernel the roofline reports (the fused decode kernel)
FFN_SOURCES = ["quantised_expert_ffn_gb300/csrc/decode_fused.cu",
               "quantised_expert_ffn_gb300/csrc/common.cuh",
               "quantised_expert_ffn_gb300/csrc/kernels.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def expert_bytes(D, F, code_bits=4):
    # codes + bf16 scale + bf16 bias for gate, up (F x D) and down (D x F)
    per_matrix = D * F * code_bits // 8 + 2 * 2 * (D * F // 64)
    return 3 * per_matrix


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_from_profile(name, source_files, key="traffic_bytes_per_layer"):
    """DRAM bytes recorded under `key` in profiles/<name>.md, if the kernels it
    was taken on are unchanged (sha256 of their sources' code, comments
    stripped, matches the digest recorded with the capture)."""
    path = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(key + r":\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]{16,64})", txt)
    if not m or not h:
        return None
    if not source_digest(source_files).startswith(h.group(1)):
        return None
    return float(m.group(1))


def _code_only(text):
    """Source text without comments and blank space: the digest then changes
    when the code changes, not when a comment does."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def source_digest(source_files):
    cur = hashlib.sha256()
    for f in source_files:
        cur.update(_code_only(open(os.path.join(ROOT, f)).read()).encode())
    return cur.hexdigest()


def replica_rate(units_per_rank, elapsed_ms, device=None):
    """Whole-job rate of N independent replicas: every rank processed
    units_per_rank units; the job took the slowest rank's time (max over ranks,
    one all-reduce that is timing only, not data path).  Returns (rate in
    units/s, job ms).  Without an initialised process group: one replica."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n = dist.get_world_size()
        ms = float(t.item())
    else:
        n, ms = 1, float(elapsed_ms)
    return units_per_rank * n / (ms / 1e3), ms


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- our arm

class DecodeStack:
    """A stack of decode layers driven through the C ABI (one shared workspace)."""

    def __init__(self, smoe, synth, n_layers, D, F, seed, dev, code_bits=4):
        self.smoe = smoe
        self.W = [synth.layer_weights(D, E, F, K, seed=seed * 1000 + i, device=dev, rms_norm=True,
                                      code_bits=code_bits)
                  for i in range(n_layers)]
        self.L = [smoe.Layer(w) for w in self.W]
        self.table = smoe.LayerTable(self.L, dev)
        self.ws = smoe.workspace(self.L[0], 64)
        self.D, self.F, self.n = D, F, n_layers
        self.bufs = [torch.empty(D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.per_layer = PER_LAYER

    def token(self, x_in, y_out):
        """One token through all layers: one launch (smoe_moe_decode_layers), or
        with --per-layer one smoe_moe_decode call per layer (ping-pong buffers)."""
        if not self.per_layer:
            self.smoe.smoe_moe_decode_layers(self.table, x_in, y_out, ws=self.ws)
            return
        cur = x_in
        for i, L in enumerate(self.L):
            nxt = y_out if i == self.n - 1 else self.bufs[i % 2]
            self.smoe.smoe_moe_decode(L, cur, nxt, ws=self.ws)
            cur = nxt


def capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm (module loads, attributes) outside the graph
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_decode(stack, states, steps, warmup, batch):
    """Device-timed decode: graph of `batch` tokens (each from its own start
    state) replayed until `steps` tokens ran; returns (ms per token, total ms)."""
    D = stack.D
    x_in = torch.empty((batch, D), dtype=torch.bfloat16, device=states.device)
    y_out = torch.empty((batch, D), dtype=torch.bfloat16, device=states.device)

    def run():
        for t in range(batch):
            stack.token(x_in[t], y_out[t])

    g = capture(run)
    n_states = states.shape[0]
    reps = steps // batch
    for r in range(max(1, (warmup + batch - 1) // batch)):
        x_in.copy_(states[(r * batch) % n_states:(r * batch) % n_states + batch])
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for r in range(reps):
        base = (r * batch) % n_states
        x_in.copy_(states[base:base + batch])
        g.replay()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    return ms / (reps * batch), ms


def time_e2e(stack, states_host, steps, warmup):
    """End to end: per token, H2D of its start state from pinned memory, the
    48-layer decode, D2H of the output -- all inside the timed region."""
    dev = stack.bufs[0].device
    D = stack.D
    x_dev = torch.empty(D, dtype=torch.bfloat16, device=dev)
    y_dev = torch.empty(D, dtype=torch.bfloat16, device=dev)
    y_host = torch.empty((steps, D), dtype=torch.bfloat16).pin_memory()
    g = capture(lambda: stack.token(x_dev, y_dev))
    n = states_host.shape[0]
    for t in range(warmup):
        x_dev.copy_(states_host[t % n], non_blocking=True)
        g.replay()
        y_host[t % steps].copy_(y_dev, non_blocking=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for t in range(steps):
        x_dev.copy_(states_host[t % n], non_blocking=True)
        g.replay()
        y_host[t].copy_(y_dev, non_blocking=True)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return steps / dt, D * 2, D * 2


def time_ffn(stack, states, n_tokens):
    """Average duration of the expert FFN call (gate/up + down/combine kernels)
    per layer, CUDA events on the launching stream, over n_tokens x layers."""
    smoe = stack.smoe
    dev = states.device
    idx = torch.empty(K, dtype=torch.int32, device=dev)
    w = torch.empty(K, dtype=torch.float32, device=dev)
    evs = []
    stream = torch.cuda.current_stream()
    for t in range(n_tokens):
        cur = states[t % states.shape[0]].clone()
        nxt = torch.empty_like(cur)
        for L in stack.L:
            smoe.smoe_route_topk(L, cur, 1, idx, w, ws=stack.ws)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            smoe.smoe_moe_ffn_decode(L, cur, idx, w, nxt, ws=stack.ws)
            b.record(stream)
            evs.append((a, b))
            cur, nxt = nxt, cur
    torch.cuda.synchronize()
    durs = [a.elapsed_time(b) for a, b in evs]
    return sum(durs) / len(durs)


def calibrate_alpha(smoe, synth, L0, dev, lo=0.0, hi=0.95, target=(60, 100)):
    """Shared-direction weight alpha so that a 64-token chunk's layer-0 union
    lands in [60, 100] experts (bisection on the GPU router)."""
    idx = torch.empty((64, K), dtype=torch.int32, device=dev)
    w = torch.empty((64, K), dtype=torch.float32, device=dev)
    ws = smoe.workspace(L0, 64)
    u = 0
    for _ in range(20):
        a = 0.5 * (lo + hi)
        x = synth.correlated_hidden(64, L0.w.d_model, a, seed=SEED, device=dev)
        smoe.smoe_route_topk(L0, x, 64, idx, w, ws=ws)
        u = int(torch.unique(idx).numel())
        if target[0] <= u <= target[1]:
            return a, u
        if u > target[1]:
            lo = a
        else:
            hi = a
    return a, u


def union_sizes(idx):
    """Distinct experts per row of idx [..., T, K] (the chunk's union size)."""
    flat = idx.reshape(-1, idx.shape[-2] * idx.shape[-1])
    srt, _ = torch.sort(flat, dim=1)
    return 1 + (srt[:, 1:] != srt[:, :-1]).sum(dim=1).reshape(idx.shape[:-2])


def time_prefill(stack, smoe, synth, dev, prompt_lens, alpha, hbm_peak=None, code_bits=4):
    """Layer-major prefill over the stack: each 64-token chunk goes through all
    layers (per layer: route, union, grouped FFN, combine), replayed from CUDA
    graphs.  After the timed replays, one untimed pass records every layer's
    top-k ids per chunk, from which the union sizes U follow; the algorithmic
    bytes are sum over chunks and layers of U x expert bytes + router bytes."""
    res = {}
    T = 64
    ws = stack.ws
    xa = torch.empty((T, stack.D), dtype=torch.bfloat16, device=dev)
    bufs = [torch.empty((T, stack.D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)

    def chunk(t, idx_all=None):
        cur = xa[:t]
        for i, L in enumerate(stack.L):
            nxt = bufs[i % 2][:t]
            io = idx[:t] if i == 0 else None
            if idx_all is not None:
                io = idx_all[i, :t]
            smoe.smoe_moe_prefill_chunk(L, cur, t, nxt, idx_out=io, ws=ws)
            cur = nxt

    graphs = {T: capture(lambda: chunk(T))}
    eb = expert_bytes(stack.D, stack.F, code_bits)
    rb = E * stack.D * 2
    for n in prompt_lens:
        x = synth.correlated_hidden(n, stack.D, alpha, seed=SEED + n, device=dev)
        tail = n % T
        if tail and tail not in graphs:
            graphs[tail] = capture(lambda: chunk(tail))
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for c0 in range(0, n, T):
            t = min(T, n - c0)
            xa[:t].copy_(x[c0:c0 + t])
            graphs[t].replay()
        ev1.record()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        # untimed pass: every layer's ids for every chunk -> union sizes
        us = []
        idx_all = torch.empty((stack.n, T, K), dtype=torch.int32, device=dev)
        for c0 in range(0, n, T):
            t = min(T, n - c0)
            xa[:t].copy_(x[c0:c0 + t])
            chunk(t, idx_all)
            us.append(union_sizes(idx_all[:, :t]))
        U = torch.stack(us).cpu()                          # [chunks, layers]
        nbytes = int(U.sum()) * eb + U.numel() * rb
        gbs = nbytes / (ms / 1e3) / 1e9
        res[str(n)] = {"ms": round(ms, 3), "tok_s": round(n / ms * 1e3, 1), "chunks": (n + T - 1) // T,
                       "union_mean": round(float(U.float().mean()), 2), "union_min": int(U.min()),
                       "union_max": int(U.max()), "union_layer0": [int(u) for u in U[:, 0]][:8],
                       "bytes": nbytes, "gbs": round(gbs, 1)}
        if hbm_peak:
            res[str(n)]["frac"] = round(gbs / hbm_peak, 4)
    return res


def time_skewed(stack, smoe, synth, dev, hbm_peak, alpha):
    """The skewed-routing workload on the 30B shape.  Prefill: 16 chunks of 64
    tokens whose layer-0 router logits carry a Zipf(1.2) bias over a seeded
    expert permutation (x_t = z_t + pinv(Wr) b, the bias scale raised until the
    largest bucket of a chunk holds 30-60 tokens), through layer 0 -- the layer
    the bias is realised at -- beside 16 chunks whose tokens share a direction
    (alpha as calibrated for the 60-100 expert unions) through the same layer;
    each set replayed from one CUDA graph.  Hot experts of the Zipf chunks recur
    from chunk to chunk, so L2 may keep them: the GB/s are algorithmic bytes
    over time, not DRAM traffic.  Decode: a stream whose consecutive tokens
    share about 46 % of their layer-0 experts (x_{s+1} = rho x_s + sqrt(1 -
    rho^2) z), through the 48-layer stack."""
    L0, W0 = stack.L[0], stack.W[0]
    T, NCH = 64, 16
    ws = smoe.workspace(L0, T)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    scale = None
    for sc in (1.0, 1.5, 2.0, 3.0, 4.0, 6.0):
        x = synth.zipf_bias_hidden(T, W0.router_w.float(), 1.2, sc, seed=SEED)
        smoe.smoe_route_topk(L0, x, T, idx, w, ws=ws)
        if 30 <= int(torch.bincount(idx.flatten().long(), minlength=E).max()) <= 60:
            scale = sc
            break
    out = {"zipf_s": 1.2, "bias_scale": scale}
    eb, rb = expert_bytes(stack.D, stack.F), E * stack.D * 2
    sets = {"zipf": torch.stack([synth.zipf_bias_hidden(T, W0.router_w.float(), 1.2, scale or 6.0,
                                                        seed=SEED + c) for c in range(NCH)]),
            "uniform": torch.stack([synth.correlated_hidden(T, stack.D, alpha, seed=SEED + 100 + c,
                                                            device=dev) for c in range(NCH)])}
    for name, xs in sets.items():
        ys = torch.empty_like(xs)
        ids = torch.empty((NCH, T, K), dtype=torch.int32, device=dev)

        def run():
            for c in range(NCH):
                smoe.smoe_moe_prefill_chunk(L0, xs[c], T, ys[c], idx_out=ids[c], ws=ws)

        g = capture(run)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = 8
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * NCH)
        U = union_sizes(ids)
        bmax = [int(torch.bincount(ids[c].flatten().long(), minlength=E).max()) for c in range(NCH)]
        nb = float(U.float().mean()) * eb + rb
        out[name] = {"us_per_chunk": round(ms * 1e3, 2), "tok_s": round(T / ms * 1e3, 1),
                     "union_mean": round(float(U.float().mean()), 2),
                     "largest_bucket_mean": round(sum(bmax) / NCH, 2), "largest_bucket_max": max(bmax),
                     "bytes_per_chunk": int(nb), "gbs": round(nb / (ms / 1e3) / 1e9, 1),
                     "frac": round(nb / (ms / 1e3) / 1e9 / hbm_peak, 4)}
        del g
    # decode stream with ~46 % adjacent overlap at layer 0 (rho picked on the GPU router)
    best = None
    i1 = torch.empty((64, K), dtype=torch.int32, device=dev)
    w1 = torch.empty((64, K), dtype=torch.float32, device=dev)
    for rho in (0.5, 0.6, 0.7, 0.75, 0.8, 0.85, 0.9):
        st = synth.overlap_stream(64, stack.D, rho, seed=SEED + 7, device=dev)
        smoe.smoe_route_topk(L0, st, 64, i1, w1, ws=ws)
        a = i1.cpu().tolist()
        ov = sum(len(set(p) & set(q)) / K for p, q in zip(a[:-1], a[1:])) / 63
        if best is None or abs(ov - 0.46) < abs(best[1] - 0.46):
            best = (rho, ov)
    rho, ov = best
    stream = synth.overlap_stream(256, stack.D, rho, seed=SEED + 8, device=dev)
    ms_tok, _ = time_decode(stack, stream, 256, 16, 16)        # tokens in stream order
    out["decode_stream"] = {"rho": rho, "layer0_adjacent_overlap": round(ov, 3),
                            "tok_s": round(1e3 / ms_tok, 2), "ms_per_token": round(ms_tok, 4)}
    return out


def near_tie_count(stack, smoe, states, n_tokens):
    """Routing near-ties that n_tokens decode tokens meet through the stack: a
    (token, layer) where two adjacent logits among the top k+1 lie within
    tau = 64 * 2^-24 * max_e sum_d |Wr[e][d] xn[d]| (the GPU's fp32 logits and
    normed input), where fp32 and fp64 may rank experts differently."""
    dev = states.device
    idx = torch.empty(K, dtype=torch.int32, device=dev)
    w = torch.empty(K, dtype=torch.float32, device=dev)
    lg = torch.empty(E, dtype=torch.float32, device=dev)
    xn = torch.empty(stack.D, dtype=torch.bfloat16, device=dev)
    count = 0
    for t in range(n_tokens):
        cur = states[t].clone()
        nxt = torch.empty_like(cur)
        for Wl, L in zip(stack.W, stack.L):
            smoe.smoe_route_topk(L, cur, 1, idx, w, logits=lg, xn=xn, ws=stack.ws)
            tau = 64 * 2.0 ** -24 * float((Wl.router_w.double().abs() @ xn.double().abs()).max())
            top = torch.topk(lg.double(), K + 1).values
            count += int(bool(((top[:-1] - top[1:]) < tau).any()))
            smoe.smoe_moe_decode(L, cur, nxt, ws=stack.ws)
            cur, nxt = nxt, cur
    torch.cuda.synchronize()
    return {"tokens": n_tokens, "layers": stack.n, "token_layers_with_near_tie": count}


def time_dense(smoe, synth, dev, hbm_peak):
    """The dense bf16 matvec on decode's projection shapes (Qwen3-235B: K/V
    512 x 4096, Q 8192 x 4096, O 4096 x 8192; the LM head 151,936 x 4096) and
    the Q4 quantiser on a 30B layer's gate tensor.  Small matrices rotate over
    enough copies that the weights of consecutive calls exceed L2."""
    out = {}
    shapes = {"kv_proj_512x4096": (512, 4096), "q_proj_8192x4096": (8192, 4096),
              "o_proj_4096x8192": (4096, 8192), "lm_head_151936x4096": (151936, 4096)}
    for name, (rows, cols) in shapes.items():
        nbytes = rows * cols * 2
        copies = max(1, -(-(256 << 20) // nbytes)) if nbytes < (256 << 20) else 1
        Ws = [synth.dense_weights((rows, cols), seed=SEED + i, device=dev) for i in range(copies)]
        x = synth.hidden(1, cols, seed=SEED, device=dev)[0]
        y = torch.empty(rows, dtype=torch.float32, device=dev)
        calls = max(8, copies)                 # one graph: back-to-back calls over the copies

        def run():
            for i in range(calls):
                smoe.smoe_dense_matvec(Ws[i % copies], x, y)

        g = capture(run)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(3, 64 // calls)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * calls)
        del g
        gbs = (nbytes + cols * 2 + rows * 4) / (us / 1e6) / 1e9
        out[name] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                     "weight_copies": copies}
        del Ws
        torch.cuda.empty_cache()
    dense = {"kernel": "k_dense_matvec (bf16 weights, fp32 sums), one launch per call",
             "timing": "CUDA graph of back-to-back calls (programmatic dependent launches), per call",
             "shapes": out}
    E, F, D = E30Q
    W = synth.dense_weights((E, F, D), seed=SEED, device=dev)
    codes = torch.empty((E, F, D // 2), dtype=torch.uint8, device=dev)
    scale = torch.empty((E, F, D // 64), dtype=torch.bfloat16, device=dev)
    bias = torch.empty_like(scale)
    for _ in range(3):
        smoe.smoe_quantize_q4(W, codes, scale, bias)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        smoe.smoe_quantize_q4(W, codes, scale, bias)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nb = W.numel() * 2 + codes.numel() + scale.numel() * 4
    quant = {"kernel": "k_quantize<4>", "workload": f"30B layer gate tensor {E}x{F}x{D} bf16 -> SMOE-Q4",
             "ms": round(ms, 4), "gbs": round(nb / (ms / 1e3) / 1e9, 1),
             "frac": round(nb / (ms / 1e3) / 1e9 / hbm_peak, 4), "bytes": nb}
    codes2 = torch.empty((E, F, D // 4), dtype=torch.uint8, device=dev)
    for _ in range(3):
        smoe.smoe_quantize_q2(W, codes2, scale, bias)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        smoe.smoe_quantize_q2(W, codes2, scale, bias)
    e1.record()
    torch.cuda.synchronize()
    ms2 = e0.elapsed_time(e1) / reps
    nb2 = W.numel() * 2 + codes2.numel() + scale.numel() * 4
    quant["q2"] = {"kernel": "k_quantize<2>", "ms": round(ms2, 4), "gbs": round(nb2 / (ms2 / 1e3) / 1e9, 1),
                   "frac": round(nb2 / (ms2 / 1e3) / 1e9 / hbm_peak, 4), "bytes": nb2}
    del W, codes, codes2, scale, bias
    torch.cuda.empty_cache()
    return dense, quant


def cpu_baseline_oracle(stack, states, n_tokens, n_layers):
    """The oracle (as it stands) on n_tokens decode tokens through the first
    n_layers of the same stack, tokens in parallel on the host cores; the rate
    is scaled to the full stack depth."""
    import numpy as np
    from oracle import oracle
    oracle.build()
    OL = [oracle.layer_from_weights(w) for w in stack.W[:n_layers]]
    x = states[:n_tokens].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    cur = x
    for L in OL:
        out = oracle.moe_tokens(L, cur)
        cur = out["y_bf16"]
    dt = time.perf_counter() - t0
    per_token_full = dt / n_tokens * (stack.n / n_layers)
    return {"value": round(1.0 / per_token_full, 4), "unit": "tok/s", "cores": oracle.omp_threads(),
            "kind": "oracle",
            "sample": f"{n_tokens} tokens x first {n_layers} of {stack.n} layers "
                      f"({dt:.1f} s wall), rate scaled to {stack.n} layers"}


def profile_case(args):
    """Small case for ncu captures: an N-layer 30B-shaped stack (a few GB),
    a few decode tokens and one 64-token prefill chunk through each layer,
    launched directly (no graph).  Prints no JSON line."""
    dev = torch.device("cuda", 0)
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe, synth
    n = args.profile_layers
    shape = (D235, F235) if args.profile_shape == "235b" else (D30, F30)
    stack = DecodeStack(smoe, synth, n, shape[0], shape[1], SEED, dev)
    states = synth.hidden(8, shape[0], seed=SEED, device=dev)
    y = torch.empty(shape[0], dtype=torch.bfloat16, device=dev)
    idx = torch.empty(K, dtype=torch.int32, device=dev)
    w = torch.empty(K, dtype=torch.float32, device=dev)
    for L in stack.L:   # expert FFN calls first (decode FFN kernel launches 0..n-1)
        smoe.smoe_route_topk(L, states[0], 1, idx, w, ws=stack.ws)
        smoe.smoe_moe_ffn_decode(L, states[0], idx, w, y, ws=stack.ws)
    for t in range(4):
        stack.token(states[t], y)
    x64 = synth.correlated_hidden(64, shape[0], 0.6, seed=SEED, device=dev)
    y64 = torch.empty_like(x64)
    for L in stack.L:
        smoe.smoe_moe_prefill_chunk(L, x64, 64, y64, ws=stack.ws)
    torch.cuda.synchronize()
    log(f"[bench] profile case done: {n} layers of {shape}")


def profile_dense():
    """Small case for ncu captures of the dense kernels: each matvec shape once
    (K/V, Q, O projections, the LM head) and the quantiser on one 30B gate
    tensor.  Prints no JSON line."""
    dev = torch.device("cuda", 0)
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe, synth
    for rows, cols in ((512, 4096), (8192, 4096), (4096, 8192), (151936, 4096)):
        W = synth.dense_weights((rows, cols), seed=SEED, device=dev)
        x = synth.hidden(1, cols, seed=SEED, device=dev)[0]
        y = torch.empty(rows, dtype=torch.float32, device=dev)
        smoe.smoe_dense_matvec(W, x, y)
        torch.cuda.synchronize()
        del W
    E_, F_, D_ = E30Q
    W = synth.dense_weights((E_, F_, D_), seed=SEED, device=dev)
    codes = torch.empty((E_, F_, D_ // 2), dtype=torch.uint8, device=dev)
    scale = torch.empty((E_, F_, D_ // 64), dtype=torch.bfloat16, device=dev)
    smoe.smoe_quantize_q4(W, codes, scale, torch.empty_like(scale))
    torch.cuda.synchronize()
    log("[bench] dense profile case done")


def our_arm(args):
    ws_, rank, local = dist_env()
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        torch.cuda.set_device(local)
    dev = torch.device("cuda", local if ws_ > 1 else 0)
    torch.cuda.set_device(dev)
    from quantised_expert_ffn_gb300 import build
    build.build()
    from quantised_expert_ffn_gb300 import smoe, synth

    hbm_peak, peak_kind = peaks()
    log(f"[bench] building 30B stack ({L30} layers)")
    stack = DecodeStack(smoe, synth, L30, D30, F30, SEED, dev)
    states = synth.hidden(256, D30, seed=SEED, device=dev)
    batch = 16 if args.steps % 16 == 0 else (8 if args.steps % 8 == 0 else 1)

    # ---- headline: device-timed decode, clocks sampled during the timed region
    time_decode(stack, states, batch, batch, batch)   # compile graph paths once
    with Clocks(dev.index) as ck:
        ms_tok, ms_total = time_decode(stack, states, args.steps, args.warmup, batch)
    clocks = ck.summary()
    value, ms_total = replica_rate(args.steps, ms_total, dev if ws_ > 1 else None)
    ms_tok = ms_total / args.steps
    bytes_token = L30 * (K * expert_bytes(D30, F30) + E * D30 * 2)

    line = {"metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_tok, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random SMOE-Q4 weights and N(0,1) start states)",
            "config": {"workload": "30B-shaped 48-layer MoE decode stack, batch 1 (d_model 2048, "
                                   "128 experts, top-8, ffn 768, SMOE-Q4 group 64, RMSNorm)",
                       "layers": L30, "global_batch": 1, "start_states": 256,
                       "l2": "inputs larger than L2: each token reads "
                             f"{bytes_token / 1e9:.2f} GB of distinct weights",
                       "parallelism": "replicas" if ws_ > 1 else "single GPU",
                       "graph_tokens": batch},
            "effective_gbs_per_token": round(bytes_token / (ms_tok / 1e3) / 1e9, 1),
            "clocks": clocks,
            "gpu_launches": args.steps * (L30 if PER_LAYER else 1)}
    line["config"]["decode_launches_per_token"] = L30 if PER_LAYER else 1

    if rank == 0:
        # ---- roofline of the dominant kernel: the decode step's one launch per
        # token (all 48 layers), timed by the graph replays above
        achieved = bytes_token / (ms_tok / 1e3) / 1e9
        traffic = traffic_from_profile("decode_stack_30b", FFN_SOURCES)
        if traffic is not None:
            traffic = round(traffic * L30, 0)      # profiled per layer; traffic grows with layers
        kname = ("k_decode_layer, one launch per layer (route + gate/up + down + residual)" if PER_LAYER
                 else "k_decode_layer, one launch per token over 48 layers (route + gate/up + down + residual)")
        line["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                            "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                            "traffic": traffic, "peak_kind": peak_kind, "kernel": kname,
                            "bytes_per_launch": bytes_token // (L30 if PER_LAYER else 1),
                            "ms_per_launch": round(ms_tok / (L30 if PER_LAYER else 1), 5)}
        # ---- the expert FFN call alone (FFN-only variant, ids given), per layer
        ffn_ms = time_ffn(stack, states, 8)
        ffn_bytes = K * expert_bytes(D30, F30)
        line["ffn_call"] = {"kernel": "k_decode_layer (FFN only: gate/up + down + residual), 8 experts",
                            "bytes": ffn_bytes, "ms": round(ffn_ms, 5),
                            "gbs": round(ffn_bytes / (ffn_ms / 1e3) / 1e9, 1),
                            "frac": round(ffn_bytes / (ffn_ms / 1e3) / 1e9 / hbm_peak, 4)}
        # ---- end to end through the C ABI with host buffers
        states_host = states[:64].cpu().pin_memory()
        e2e, bi, bo = time_e2e(stack, states_host, args.steps, max(3, args.warmup))
        line["e2e"] = {"value": round(e2e, 2), "unit": "tok/s", "h2d_bytes_per_step": bi,
                       "d2h_bytes_per_step": bo}
        if ws_ == 1 and not args.no_cpu:
            log("[bench] timing the oracle on the host cores")
            line["cpu_baseline"] = cpu_baseline_oracle(stack, states, args.cpu_tokens,
                                                       args.cpu_layers)
    pre30 = None
    if rank == 0 and ws_ == 1:
        # prefill on the 30B shape, SMOE-Q4 here and SMOE-Q2 below (same prompts, same router draw)
        alpha30, u30 = calibrate_alpha(smoe, synth, stack.L[0], dev)
        pre30 = {"alpha": round(alpha30, 4), "layer0_union_64tok": u30,
                 "q4": time_prefill(stack, smoe, synth, dev, [512, 4096], alpha30, hbm_peak)}
        log("[bench] skewed routing (Zipf chunks, overlapping decode stream)")
        line["skewed_routing"] = dict(
            workload="30B shape: 16 Zipf(1.2)-biased 64-token chunks through layer 0 beside 16 "
                     "direction-sharing chunks; a 46 %-overlap decode stream through 48 layers",
            **time_skewed(stack, smoe, synth, dev, hbm_peak, alpha30))
        line["near_ties"] = near_tie_count(stack, smoe, states, 8)
    del stack
    torch.cuda.empty_cache()

    if rank == 0 and ws_ == 1:
        log(f"[bench] building 30B SMOE-Q2 stack ({L30} layers)")
        q2 = DecodeStack(smoe, synth, L30, D30, F30, SEED + 2, dev, code_bits=2)
        msq2, _ = time_decode(q2, states, 256, 16, 16)
        bq2 = L30 * (K * expert_bytes(D30, F30, 2) + E * D30 * 2)
        line["decode_q2"] = {"workload": "30B-shaped 48-layer decode stack with SMOE-Q2 experts (2-bit "
                                         "codes, same groups), batch 1, 256 tokens",
                             "tok_s": round(1e3 / msq2, 2), "ms_per_token": round(msq2, 4),
                             "us_per_layer": round(msq2 * 1e3 / L30, 2),
                             "effective_gbs": round(bq2 / (msq2 / 1e3) / 1e9, 1),
                             "bytes_per_token": bq2}
        alpha_q2, u_q2 = calibrate_alpha(smoe, synth, q2.L[0], dev)
        pre30["q2"] = time_prefill(q2, smoe, synth, dev, [512, 4096], alpha_q2, hbm_peak, code_bits=2)
        pre30["q2_alpha"], pre30["q2_layer0_union_64tok"] = round(alpha_q2, 4), u_q2
        line["prefill_30b"] = dict(workload="30B-shaped 48-layer layer-major prefill, chunks of 64, "
                                            "SMOE-Q4 and SMOE-Q2 stacks", **pre30)
        line["prefill_30b"]["roofline_4096"] = {
            "bound": "hbm", "bytes": "sum over chunks and layers of union size x expert bytes + router bytes",
            "q4_frac": pre30["q4"]["4096"]["frac"], "q2_frac": pre30["q2"]["4096"]["frac"]}
        del q2
        torch.cuda.empty_cache()
        log("[bench] dense matvec and quantiser")
        line["dense_matvec"], line["quantize_q4"] = time_dense(smoe, synth, dev, hbm_peak)

    if rank == 0 and ws_ == 1 and not args.no_235b:
        log(f"[bench] building 235B stack ({L235} layers, ~128 GB)")
        big = DecodeStack(smoe, synth, L235, D235, F235, SEED + 1, dev)
        st235 = synth.hidden(128, D235, seed=SEED + 1, device=dev)
        ms235, _ = time_decode(big, st235, 128, 16, 16)
        b235 = L235 * (K * expert_bytes(D235, F235) + E * D235 * 2)
        ach235 = b235 / (ms235 / 1e3) / 1e9
        ffn235 = time_ffn(big, st235, 4)
        fb235 = K * expert_bytes(D235, F235)
        line["decode_235b"] = {"workload": "235B-shaped 94-layer MoE decode, batch 1 (d_model "
                                           "4096, ffn 1536), 128 tokens",
                               "tok_s": round(1e3 / ms235, 2), "ms_per_token": round(ms235, 4),
                               "us_per_layer": round(ms235 * 1e3 / L235, 2),
                               "effective_gbs": round(ach235, 1),
                               "roofline": {"bound": "hbm", "achieved": round(ach235, 1), "peak": hbm_peak,
                                            "unit": "GB/s", "frac": round(ach235 / hbm_peak, 4),
                                            "kernel": "k_decode_layer, one launch per token over 94 layers",
                                            "bytes_per_launch": b235, "ms_per_launch": round(ms235, 5)},
                               "ffn_call": {"kernel": "k_decode_layer (FFN only), 8 experts of 10,616,832 B",
                                            "bytes": fb235, "ms": round(ffn235, 5),
                                            "gbs": round(fb235 / (ffn235 / 1e3) / 1e9, 1),
                                            "frac": round(fb235 / (ffn235 / 1e3) / 1e9 / hbm_peak, 4)}}
        alpha, u0 = calibrate_alpha(smoe, synth, big.L[0], dev)
        pre = time_prefill(big, smoe, synth, dev, [45, 512, 4096], alpha, hbm_peak)
        line["prefill"] = {"workload": "235B-shaped 94-layer layer-major prefill, chunks of 64",
                           "alpha": round(alpha, 4), "layer0_union_64tok": u0, "prompts": pre,
                           "tok_s_4096": pre["4096"]["tok_s"],
                           "roofline_4096": {"bound": "hbm", "achieved": pre["4096"]["gbs"], "peak": hbm_peak,
                                             "unit": "GB/s", "frac": pre["4096"]["frac"],
                                             "bytes": pre["4096"]["bytes"],
                                             "bytes_rule": "sum over chunks and layers of union size x "
                                                           "10,616,832 B + router 1,048,576 B",
                                             "time": "whole chunk path (route, union, gather, gate/up and "
                                                     "down grouped GEMMs, combine), CUDA events around "
                                                     "graph replays"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_ > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def reference_arm(args):
    """The CPU oracle timed as it stands, on a bounded sample of the headline
    workload (30B-shaped 48-layer decode, same seeded weights)."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    from oracle import oracle
    from quantised_expert_ffn_gb300 import synth
    oracle.build()
    # bounded run: past 128 steps (warm-up included) fewer layers per step, never fewer
    # tokens (the tokens are what the oracle spreads over the host cores)
    n_layers = args.cpu_layers
    if args.steps + args.warmup > 128:
        n_layers = max(1, n_layers * 128 // (args.steps + args.warmup))
    W = [synth.layer_weights(D30, E, F30, K, seed=SEED * 1000 + i, device="cpu", rms_norm=True)
         for i in range(n_layers)]
    OL = [oracle.layer_from_weights(w) for w in W]
    states = synth.hidden(256, D30, seed=SEED, device="cpu")
    x_all = states.contiguous().view(torch.int16).numpy().view(np.uint16)
    ntok = args.cpu_tokens

    def step(i):
        cur = x_all[(i * ntok) % 256:(i * ntok) % 256 + ntok]
        for L in OL:
            cur = oracle.moe_tokens(L, cur)["y_bf16"]

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    per_token_full = dt / (args.steps * ntok) * (L30 / n_layers)
    value = 1.0 / per_token_full
    sample = (f"{ntok} tokens x first {n_layers} of {L30} layers per step, rate scaled to "
              f"{L30} layers")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s",
            "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_token_full * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random SMOE-Q4 weights and N(0,1) start states)",
            "config": {"workload": "30B-shaped 48-layer MoE decode stack, batch 1 (d_model 2048, "
                                   "128 experts, top-8, ffn 768, SMOE-Q4 group 64, RMSNorm)",
                       "layers": L30, "global_batch": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "tok/s",
                             "cores": oracle.omp_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=16)
    ap.add_argument("--cpu-layers", type=int, default=4)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--per-layer", action="store_true",
                    help="decode with one launch per layer instead of one per token")
    ap.add_argument("--no-235b", action="store_true")
    ap.add_argument("--profile-layers", type=int, default=0,
                    help="run only the small ncu case with this many layers")
    ap.add_argument("--profile-shape", default="30b", choices=["30b", "235b"])
    ap.add_argument("--profile-dense", action="store_true",
                    help="run the dense matvec shapes and the quantiser once (for ncu), no JSON line")
    args = ap.parse_args()
    global PER_LAYER
    PER_LAYER = args.per_layer
    if args.profile_layers:
        profile_case(args)
        return
    if args.profile_dense:
        profile_dense()
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if args.steps > 4 and "--steps" not in " ".join(sys.argv):
            args.steps = 2
        reference_arm(args)
    else:
        our_arm(args)


if __name__ == "__main__":
    main()
