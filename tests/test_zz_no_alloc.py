"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Checked through the
C ABI against fa_bwd with a caller-allocated workspace, on two calls in a row.

This file is collected last on purpose, so a failure here leaves every other
test already run; it also passes on its own in a fresh process."""
import math

import pytest
import torch

import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl
from parity import GRAD_REL, grad_rel, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_matches_fa_bwd_on_two_calls(d, causal):
    B, H, N = 1, 4, 1000
    scale = 1.0 / math.sqrt(d)
    inp = wl.make_inputs(wl.WORKLOADS["fwdbwd_4k_d128"], B=B, H=H, N=N, d=d, seed=31 + d)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    ref = fa.backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    h = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, H, N, d, scale, int(causal), h)
        assert rc == fa.FA_OK, fa.status_string(rc)
        assert fa.fa_sync_status(h) == fa.FA_OK
        for got, want, name in ((dq, ref[0], "dq"), (dk, ref[1], "dk"), (dv, ref[2], "dv")):
            rel = grad_rel(to_np(got), to_np(want))
            assert rel <= GRAD_REL, f"call {call}: {name} differs from fa_bwd by {rel:.3e}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # D for 1 * 512 * 32769 > 2^24 rows needs more than 64 MiB (d = 64 keeps the
    # shape itself under 2^31 elements); the sizes are rejected before any
    # pointer is touched.
    fake = 0x100000
    rc = fa.fa_bwd_noalloc(*([fake] * 9), 1, 512, 32769, 64, 0.125, 1,
                           torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_WORKSPACE
