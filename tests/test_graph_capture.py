"""The layer forward captured into a CUDA graph and replayed.

A serving loop captures the forward once and replays it on new inputs
written into the same buffers.  Every launch of the forward is stream
ordered, takes its arguments by value and allocates nothing, so the
captured graph must reproduce the eager results bit for bit (same kernels,
same inputs, same order of operations) for the top-1 layer and its
variants.
"""
import pytest
import torch

from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, d, F, N, cf, mode, extra forward arguments
    ("top1-token-order", 2048, 256, 512, 32, 1.0, 0, {}),
    ("top1-gate-priority", 2048, 256, 512, 32, 1.0, 1, {}),
    ("top2", 2048, 256, 512, 32, 1.0, 0, {"top_k": 2, "renormalize": 1}),
    ("expanded-drop", 2048, 256, 512, 32, 0.8, 0, {"expand": 2}),
    ("decode-shape", 64, 512, 1024, 8, 2.0, 0, {}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_graph_replay_matches_eager(lib, case):
    name, T, d, F, N, cf, mode, kw = case
    w = Workload(name, T, d, F, N, cf, "bf16", 0.3, zipf_s=1.1, zipf_lambda=0.6)
    inp = make_inputs(w, seed=3, device="cuda")
    x = inp.x.clone()
    ws = lib.workspace(lib.switch_moe_workspace_bytes(
        lib.make_params(T, d, F, N, cf, mode, 1, lib.BF16, 0, kw.get("expand", 1),
                        kw.get("top_k", 1), kw.get("renormalize", 0))), "cuda")
    out = lib.switch_moe_forward(x, inp.W_g, inp.W1, inp.W2, cf, mode, 1, b_g=inp.b_g, ws=ws,
                                 **kw)   # eager, also the first call (attributes, tensor maps)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lib.switch_moe_forward(x, inp.W_g, inp.W1, inp.W2, cf, mode, 1, b_g=inp.b_g, ws=ws,
                                   out=out, stream=s, **kw)
    torch.cuda.synchronize()
    gen = torch.Generator(device="cuda").manual_seed(11)
    for rep in range(3):   # new inputs into the captured buffer, replay, compare
        x.copy_(torch.randn(x.shape, generator=gen, device="cuda").to(x.dtype))
        g.replay()
        torch.cuda.synchronize()
        assert lib.switch_moe_sync_status() == 0
        got = [t.clone() for t in out]
        ref = lib.switch_moe_forward(x, inp.W_g, inp.W1, inp.W2, cf, mode, 1, b_g=inp.b_g,
                                     **kw)
        torch.cuda.synchronize()
        for f, a, b in zip(out._fields, got, ref):
            assert torch.equal(a, b), f"{name} replay {rep}: {f} differs from the eager run"
