"""Failure detection without a GPU fault.

A test build of the library (FA_FAULT_INJECT=1, wait limit 0.2 s) never issues
the K/V copies of the forward or the Q/dO copies of the backward, so a bounded
mbarrier wait inside the kernel runs out.  The kernel must record
FA_ERR_DEVICE_TIMEOUT in the device status word, leave cleanly (TMEM freed,
copies drained), and the CUDA context must stay usable: afterwards the normal
library still computes correct results on the same device."""
import ctypes
import math
import os
import time

import numpy as np
import pytest
import torch

import oracle
import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import build as fa_build
from exact_tiled_attention_05_gb300 import workloads as wl
from parity import bits, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fault_lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("fault_build")
    path = fa_build.build(force=True, lib_path=str(d / "libfa_fault.so"), build_dir=str(d),
                          extra_flags=["-DFA_FAULT_INJECT=1", "-DFA_WAIT_TIMEOUT_NS=200000000ull"])
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P]
    lib.fa_fwd_ws.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P, Z, P]
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P]
    lib.fa_sync_status.argtypes = [P]
    for f in (lib.fa_fwd, lib.fa_fwd_ws, lib.fa_bwd, lib.fa_sync_status):
        f.restype = I
    return lib


def _inputs(N, d, seed):
    return wl.make_inputs(wl.WORKLOADS["fwdbwd_4k_d128"], B=1, H=1, N=N, d=d, seed=seed)


def _normal_library_still_works():
    inp = _inputs(300, 64, 5)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=True)
    fa.sync_status()
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 1 / math.sqrt(64), True)
    check_o(to_np(o).reshape(o_ref.shape), o_ref, "after timeout")
    check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "after timeout")


@pytest.mark.parametrize("persistent", [True, False])
def test_forward_wait_runs_out_and_reports(fault_lib, persistent):
    inp = _inputs(200, 128, 1)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 1, 200, dtype=torch.float32, device=DEV)
    h = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    if persistent:  # fa_fwd_ws: one CTA per SM with a work counter
        ws = torch.empty(256, dtype=torch.uint8, device=DEV)
        rc = fault_lib.fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 1, 1, 200, 128, 0.088, 1, ws.data_ptr(),
                                 ws.numel(), h)
    else:
        rc = fault_lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 1, 200, 128, 0.088, 1, h)
    assert rc == fa.FA_OK  # the launch itself succeeds
    assert fault_lib.fa_sync_status(h) == fa.FA_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30
    assert fault_lib.fa_sync_status(h) == fa.FA_OK  # reading clears the word
    assert torch.count_nonzero(o).item() == 0  # nothing was written
    _normal_library_still_works()


def test_backward_wait_runs_out_and_reports(fault_lib):
    N, d = 128, 64
    inp = _inputs(N, d, 2)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=False)
    fa.sync_status()
    dq, dk, dv = (torch.zeros_like(q) for _ in range(3))
    ws = fa.alloc_workspace(1, 1, N, d, DEV)
    h = torch.cuda.current_stream().cuda_stream
    rc = fault_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          1, 1, N, d, 0.125, 0, ws.data_ptr(), ws.numel(), h)
    assert rc == fa.FA_OK
    assert fault_lib.fa_sync_status(h) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fault_lib.fa_sync_status(h) == fa.FA_OK
    assert torch.count_nonzero(dk).item() == 0 and torch.count_nonzero(dv).item() == 0
    _normal_library_still_works()
