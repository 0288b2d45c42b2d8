"""Host logic of the seeded workload generator (no GPU, no oracle)."""
import numpy as np
import torch

from exact_attention_93_gb300 import workloads as W


def test_five_workloads_with_their_shapes():
    got = {n: (w.B, w.H, w.N, w.D, w.dtype, w.causal, w.seed, w.backward) for n, w in W.WORKLOADS.items()}
    assert got == {
        "tiny": (1, 2, 128, 64, "bf16", False, 0, True),
        "long4k_fwd": (2, 8, 4096, 128, "bf16", False, 1, False),
        "gpt2_causal": (8, 12, 1024, 64, "bf16", True, 2, True),
        "bert_fp16": (32, 16, 512, 64, "fp16", False, 3, True),
        "long64k_causal": (1, 8, 65536, 128, "bf16", True, 4, True),
    }
    assert W.ORDER == list(W.WORKLOADS)


def test_flop_counts():
    w = W.WORKLOADS["long4k_fwd"]
    assert w.fwd_flops() == 4 * 2 * 8 * 4096 ** 2 * 128
    c = W.WORKLOADS["long64k_causal"]
    assert c.fwd_flops() == 2 * 8 * 65536 ** 2 * 128
    assert c.bwd_flops() == 2.5 * c.fwd_flops()


def test_inputs_are_seeded_and_in_the_right_dtype():
    w = W.WORKLOADS["tiny"]
    a, b = W.make_inputs(w), W.make_inputs(w)
    assert set(a) == {"q", "k", "v", "do"}
    for key in a:
        assert a[key].dtype == torch.bfloat16 and a[key].shape == (1, 2, 128, 64)
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["q"], a["k"])
    # draw order: q first, from the workload's seed
    g = torch.Generator().manual_seed(0)
    assert torch.equal(a["q"], torch.randn((1, 2, 128, 64), generator=g).to(torch.bfloat16))
    f = W.make_inputs(W.custom(1, 1, 64, 64, dtype="fp16", seed=3, do_std=0.1))
    assert f["do"].dtype == torch.float16
    assert 0.05 < f["do"].float().std().item() < 0.15


def test_sampled_rows():
    w = W.WORKLOADS["long64k_causal"]
    r = W.sampled_rows(w, 0, 3)
    assert r[0] == 0 and r[-1] == w.N - 1
    assert len(r) == 258 and np.all(np.diff(r) > 0)
    assert np.array_equal(r, W.sampled_rows(w, 0, 3))
    assert not np.array_equal(r, W.sampled_rows(w, 0, 4))
    assert np.array_equal(W.sampled_rows(W.WORKLOADS["tiny"], 0, 0), np.arange(128))
    assert np.array_equal(W.tail_rows(w), np.arange(w.N - 128, w.N))
