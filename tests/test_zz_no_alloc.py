"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (code running inside an allocator's callbacks, services with a fixed
device-memory footprint, plug-ins whose host owns every allocation).  Its
scratch is one fixed array inside the library, shared by every call on a
device and keeping the previous call's contents.

Checked through the C ABI against fa_bwd with a caller-allocated workspace:
both run the same deterministic kernels on the same inputs, so the gradients
must be bitwise equal, on consecutive calls whose sizes change (a larger N
between two calls of the same size, then a smaller one), which moves where
the row statistics and the work counters sit in the shared array.

This file is collected last on purpose, so a failure here leaves every other
test already run; it also passes on its own in a fresh process."""
import math

import pytest
import torch

import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def case(H, N, d, causal, seed):
    scale = 1.0 / math.sqrt(d)
    inp = wl.make_inputs(wl.WORKLOADS["fwdbwd_4k_d128"], B=1, H=H, N=N, d=d, seed=seed)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    ref = fa.backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    fa.sync_status()
    return (q, k, v, o, lse, do), ref, scale


def noalloc(tensors, H, N, d, scale, causal):
    q, k, v, o, lse, do = tensors
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    h = torch.cuda.current_stream().cuda_stream
    rc = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, H, N, d,
                           scale, int(causal), h)
    assert rc == fa.FA_OK, fa.status_string(rc)
    assert fa.fa_sync_status(h) == fa.FA_OK
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_equals_fa_bwd_on_consecutive_calls(d, causal):
    small = case(4, 1000, d, causal, seed=31 + d)
    large = case(3, 2900, d, causal, seed=41 + d)
    tiny = case(2, 200, d, causal, seed=51 + d)
    # same size twice, then larger, then smaller: every call against fa_bwd
    for step, (tensors, ref, scale), (H, N) in (
            (0, small, (4, 1000)), (1, small, (4, 1000)), (2, large, (3, 2900)),
            (3, small, (4, 1000)), (4, tiny, (2, 200))):
        got = noalloc(tensors, H, N, d, scale, causal)
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            assert torch.equal(g, r), f"call {step} (H={H} N={N}): {name} differs from fa_bwd"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # the scratch holds 2^23 padded rows: one more 128-row tile is refused
    # before any pointer is touched
    h = torch.cuda.current_stream().cuda_stream
    fake = 0x100000
    assert fa.fa_bwd_noalloc(*([fake] * 9), 1, 64, 131073, 64, 0.125, 1, h) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_noalloc(*([fake] * 9), 1, 512, 32769, 64, 0.125, 1, h) == fa.FA_ERR_WORKSPACE
    assert fa.fa_sync_status(h) == fa.FA_OK
