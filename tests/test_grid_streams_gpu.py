"""Launch-shape and stream properties of libfattn on the GPU: grids beyond
65535 CTAs (every kernel indexes (batch, head) through a one-dimensional
grid), and calls on two streams at once giving exactly the results of the
same calls run one after the other (the library keeps no per-call state
outside the caller's buffers)."""
import numpy as np
import pytest
import torch

import fp8_bound
import oracle
import oracle.fp8 as ofp8
from exact_attention_93_gb300 import fattn, workloads as W

pytestmark = pytest.mark.gpu


def test_more_than_65535_ctas_forward_and_backward():
    # B * H = 66000 slices of N = 3: 66000 CTAs in every backward tile kernel; the
    # forward's 66000 work units run on resident CTAs, about 434 each
    w = W.custom(2, 33000, 3, 64, "bf16", causal=True, seed=41)
    inputs = W.make_inputs(w)
    g = {k: v.cuda() for k, v in inputs.items()}
    o = torch.empty_like(g["q"])
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, True)
    out = {}
    for det in (False, True):
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        fattn.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, w.scale, True, det)
        out[det] = (dq, dk, dv)
    torch.cuda.synchronize()
    assert fattn.fa_device_error() == fattn.FA_OK
    # the first, a middle and the last slice against the oracle
    for b, h in ((0, 0), (1, 16500), (1, 32999)):
        ref = oracle.attention_head(inputs["q"][b, h], inputs["k"][b, h], inputs["v"][b, h],
                                    w.scale, True, dout=inputs["do"][b, h])
        assert np.max(np.abs(o[b, h].float().cpu().numpy() - ref["o"])) < 1e-2
        assert np.max(np.abs(lse[b, h].cpu().numpy() - ref["lse"])) < 1e-3
        for det in (False, True):
            for name, t in zip(("dq", "dk", "dv"), out[det]):
                r = ref[name]
                err = np.max(np.abs(t[b, h].float().cpu().numpy() - r))
                assert err <= 2e-2 * max(np.max(np.abs(r)), 1e-2), (name, det, b, h)


def test_fp8_forward_with_more_than_65535_ctas():
    w = W.custom(1, 66000, 2, 128, "bf16", causal=False, seed=42, backward=False)
    d = W.make_fp8_inputs(w)
    q8, k8, v8 = (d[n].cuda() for n in ("q8", "k8", "v8"))
    o = torch.empty(w.B, w.H, w.N, w.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd_fp8(q8, k8, v8, o, lse, None, None, w.B, w.H, w.N, w.D, w.scale, False,
                     d["descale_q"].cuda(), d["descale_k"].cuda(), d["descale_v"].cuda())
    torch.cuda.synchronize()
    # the last slice against the oracle, with the e4m3 bound of the parity tests
    q, k, v = ofp8.dequantise(d["q8"][:, -1:], d["k8"][:, -1:], d["v8"][:, -1:],
                              d["descale_q"][:, -1:], d["descale_k"][:, -1:], d["descale_v"][:, -1:])
    rows = np.arange(w.N)
    ref = oracle.attention_head(q[0, 0], k[0, 0], v[0, 0], w.scale, False, rows=rows,
                                want_probs=True)
    fp8_bound.check_head(o[0, -1].float().cpu().numpy(), lse[0, -1].cpu().numpy(), ref,
                         q[0, 0], k[0, 0], v[0, 0], w.scale, rows, label="last slice")


def test_two_streams_at_once_match_sequential_calls():
    shapes = [W.custom(1, 4, 1000, 128, "bf16", causal=True, seed=43),
              W.custom(2, 3, 700, 64, "fp16", causal=False, seed=44)]
    data = []
    for w in shapes:
        g = {k: v.cuda() for k, v in W.make_inputs(w).items()}
        bufs = {"o": torch.empty_like(g["q"]),
                "lse": torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda"),
                "dq": torch.empty_like(g["q"]), "dk": torch.empty_like(g["q"]),
                "dv": torch.empty_like(g["q"]),
                "ws": fattn.alloc_workspace(w.B, w.H, w.N, w.D, True)}
        data.append((w, g, bufs))

    def run(w, g, b, stream):
        fattn.fa_fwd(g["q"], g["k"], g["v"], b["o"], b["lse"], w.scale, w.causal, stream=stream)
        fattn.fa_bwd(g["q"], g["k"], g["v"], b["o"], b["lse"], g["do"], b["dq"], b["dk"],
                     b["dv"], w.scale, w.causal, True, b["ws"], stream=stream)

    for w, g, b in data:  # one after the other, deterministic backward
        run(w, g, b, None)
    torch.cuda.synchronize()
    seq = [{k: v.clone() for k, v in b.items() if k != "ws"} for _, _, b in data]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for (w, g, b), s in zip(data, streams):
            for k, v in b.items():
                if k != "ws":
                    v.zero_()
        torch.cuda.synchronize()
        for (w, g, b), s in zip(data, streams):
            run(w, g, b, s)
        torch.cuda.synchronize()
        for (_, _, b), ref in zip(data, seq):
            for k, v in ref.items():
                assert torch.equal(b[k], v), k
    assert fattn.fa_device_error() == fattn.FA_OK


def test_cuda_graph_replay_matches_eager_calls():
    # A forward + deterministic backward captured once in a CUDA graph and
    # replayed (the way a training loop hides launch costs at short lengths)
    # gives bit for bit the results of the same calls made one by one; the
    # forward kernel's launch allows overlap with the preceding kernel, which
    # a graph keeps as a programmatic edge.
    w = W.custom(4, 12, 1024, 64, "bf16", causal=True, seed=43)
    g = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    ws = fattn.alloc_workspace(w.B, w.H, w.N, w.D, True)
    outs = {}
    for name in ("eager", "graph"):
        o = torch.empty_like(g["q"])
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))

        def step(stream=None):
            fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, True, stream=stream)
            fattn.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, w.scale, True,
                         True, ws, stream=stream)

        if name == "eager":
            step()
        else:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                step(s)  # first calls set kernel attributes outside the capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                step(torch.cuda.current_stream())
            for t in (o, lse, dq, dk, dv):
                t.zero_()
            graph.replay()
            graph.replay()
        torch.cuda.synchronize()
        outs[name] = (o, lse, dq, dk, dv)
    for a, b in zip(outs["eager"], outs["graph"]):
        assert torch.equal(a, b)
    assert fattn.fa_device_error() == fattn.FA_OK
