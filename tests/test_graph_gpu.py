"""The C ABI inside CUDA graphs: every entry point only enqueues work on the
stream it is given (no synchronisation, no allocation), so a forward, a
backward and an FP8 forward captured into one graph and replayed give the same
bits as eager calls."""
import pytest
import torch

import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_capture_and_replay_matches_eager():
    B, H, N, d = 1, 2, 333, 128
    w = wl.WORKLOADS["fwdbwd_4k_d128"]
    inp = wl.make_inputs(w, B=B, H=H, N=N, d=d, seed=41)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    words = wl.sign_bits(42)

    # eager reference
    o_e, lse_e = fa.forward(q, k, v, causal=True)
    g_e = fa.backward(q, k, v, o_e, lse_e, do, causal=True)
    o8_e, lse8_e = fa.forward_fp8(q, k, v, signs=words, causal=True)
    fa.sync_status()

    # static buffers for the graph
    o, lse = torch.empty_like(o_e), torch.empty_like(lse_e)
    dq, dk, dv = (torch.empty_like(t) for t in g_e)
    ws = fa.alloc_workspace(B, H, N, d, DEV)
    ws8 = torch.empty(fa.fp8_workspace_bytes(B, H, N), dtype=torch.uint8, device=DEV)
    o8, lse8 = torch.empty_like(o8_e), torch.empty_like(lse8_e)

    def run():
        fa.forward(q, k, v, causal=True, out=o, lse=lse)
        fa.backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
        fa.quantize_fp8(q, k, v, signs=words, workspace=ws8)
        fa.forward_fp8_quantized(ws8, B, H, N, causal=True, out=o8, lse=lse8)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for t in (o, lse, dq, dk, dv, o8, lse8):
        t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    fa.sync_status()

    assert torch.equal(o, o_e) and torch.equal(lse, lse_e)
    for got, ref in zip((dq, dk, dv), g_e):
        assert torch.equal(got, ref)
    assert torch.equal(o8, o8_e) and torch.equal(lse8, lse8_e)
