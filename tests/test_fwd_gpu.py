"""Forward pass on the GPU, through the C ABI, against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl
from parity import (bf16_half_ulp, bits, check_lse, check_o, check_o_beyond_rounding, o_report,
                    to_np, with_guard)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
_cache = {}


def run_fwd(inp, causal, scale=None):
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    fa.sync_status()
    return o, lse


def workload_run(name, causal):
    key = (name, causal)
    if key not in _cache:
        w = wl.WORKLOADS[name]
        inp = wl.make_inputs(w)
        o, lse = run_fwd(inp, causal, w.scale)
        _cache[key] = (w, inp, o.cpu(), lse.cpu())
    return _cache[key]


# ---------------------------------------------------------------------------
# the worked example from the pages, through the kernel
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
def test_worked_example_three_scores(d):
    """scores [0, ln2, ln3], V = [1, 2, 4]: O = 17/6 and lse = ln 6 for every row
    ("07 GPU、资源估算与 FlashAttention" §7.8)."""
    inp = wl.worked_example_inputs(d=d)
    o, lse = run_fwd(inp, causal=False, scale=1.0)
    o = to_np(o)[0, 0]
    lse = to_np(lse)[0, 0]
    assert np.all(np.abs(o[:, 0] - 17.0 / 6.0) <= 1e-2)
    assert np.all(o[:, 1:] == 0.0)
    assert np.all(np.abs(lse - math.log(6.0)) <= 1e-3)
    # and the oracle on the very same bf16 inputs agrees
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 1.0, False)
    check_o(o, o_ref[0], "worked example")
    check_lse(lse, l_ref[0], "worked example")


# ---------------------------------------------------------------------------
# the workloads, element by element
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_single_head_256(causal):
    w, inp, o, lse = workload_run("single_head_256", causal)
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), w.scale, causal)
    check_o(to_np(o).reshape(o_ref.shape), o_ref, "single head 256")
    check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "single head 256")


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_2k_d64_all_heads(causal):
    w, inp, o, lse = workload_run("fwd_2k_d64", causal)
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), w.scale, causal)
    check_o(to_np(o).reshape(o_ref.shape), o_ref, "fwd 2k d64")
    check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "fwd 2k d64")


def test_fwd_8k_d128_kx3_all_heads():
    """The forward-gate workload (B=2 H=16 N=8192 d=128, K x3, causal) in full:
    every one of the 32 x 8192 rows of O and lse against the oracle."""
    w, inp, o, lse = workload_run("fwd_8k_d128_kx3", True)
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), w.scale, True)
    o = to_np(o).reshape(o_ref.shape)
    check_o(o, o_ref, "8k kx3 all heads")
    check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "8k kx3 all heads")
    print("8k kx3 all heads:", o_report(o, o_ref))


def test_fwd_32k_d128_sampled_rows():
    """Long context: 512 seeded rows per head (rows 0 and N-1 always)."""
    w = wl.WORKLOADS["fwd_32k_d128"]
    inp = wl.make_inputs(w)
    o, lse = run_fwd(inp, True, w.scale)
    o = to_np(o).reshape(w.BH, w.N, w.d)
    lse = to_np(lse).reshape(w.BH, w.N)
    rows = wl.sampled_rows(w)
    assert rows.shape == (w.BH, 512)
    o_ref, l_ref = oracle.fwd_rows(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), w.scale,
                                   True, rows)
    check_o(np.take_along_axis(o, rows[:, :, None], axis=1), o_ref, "32k sampled rows")
    check_lse(np.take_along_axis(lse, rows, axis=1), l_ref, "32k sampled rows")
    # causal row 0 is exactly V[0]
    v0 = inp["v"][0, :, 0, :].double().numpy()
    assert np.array_equal(o[:, 0, :], v0)


@pytest.mark.parametrize("causal", [True, False])
def test_fwd_one_million_keys_sampled_rows(causal):
    """N = 2^20, d = 128, one head: 8192 query tiles, up to 8192 key tiles per
    row block.  32 seeded rows (with 0, 1, 127, 128 and N-1) against the oracle."""
    N, d = 1 << 20, 128
    inp = wl.make_inputs(wl.WORKLOADS["fwd_32k_d128"], B=1, H=1, N=N, d=d, seed=90 + causal)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(inp, causal, scale)
    rng = np.random.default_rng(91)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.choice(N, 27, replace=False)]))[None, :]
    idx = torch.as_tensor(rows[0], device=o.device)
    o_s = to_np(o.reshape(N, d)[idx])[None]
    l_s = to_np(lse.reshape(N)[idx])[None]
    o_ref, l_ref = oracle.fwd_rows(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), scale, causal, rows)
    # rows 0 and 1 see one and two keys: the limits apply beyond the output rounding
    check_o_beyond_rounding(o_s, o_ref, f"N=2^20 causal={causal}")
    check_lse(l_s, l_ref, f"N=2^20 causal={causal}")
    if causal:  # row 0 is exactly V[0]
        assert np.array_equal(o_s[0, 0], inp["v"][0, 0, 0].double().numpy())


# ---------------------------------------------------------------------------
# ragged and degenerate shapes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 3, 64, 127, 128, 129, 255, 256, 257, 300, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(N, d, causal):
    w = wl.WORKLOADS["single_head_256"]
    inp = wl.make_inputs(w, B=2, H=3, N=N, d=d, seed=1000 + N + d)
    o, lse = run_fwd(inp, causal, 1.0 / math.sqrt(d))
    o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 1.0 / math.sqrt(d),
                              causal)
    check_o_beyond_rounding(to_np(o).reshape(o_ref.shape), o_ref, f"N={N} d={d}")
    check_lse(to_np(lse).reshape(l_ref.shape), l_ref, f"N={N} d={d}")


def test_many_heads_short_rows():
    w = wl.WORKLOADS["single_head_256"]
    inp = wl.make_inputs(w, B=16, H=40, N=96, d=128, seed=5)
    for causal in (False, True):
        o, lse = run_fwd(inp, causal, 0.1)
        o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 0.1, causal)
        check_o_beyond_rounding(to_np(o).reshape(o_ref.shape), o_ref, "many heads")
        check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "many heads")


@pytest.mark.parametrize("B,H,N,d", [
    (2, 24, 300, 128), (2, 24, 1000, 64), (2, 8, 4096, 128),   # static table, up to 512 items
    (2, 16, 8192, 128), (1, 32, 32768, 64),                    # static table, 1024 / 4096 items
    (1, 9000, 128, 64),                                        # 9000 items: round robin
])
@pytest.mark.parametrize("causal", [False, True])
def test_static_schedule_matches_work_counter(B, H, N, d, causal):
    """fa_fwd (no workspace) runs one CTA per SM over a static schedule (a
    greedy longest-first table in the launch parameters, or round robin past
    8192 items); fa_fwd_ws hands the items out from a counter.  Every item is
    computed by the same code in the same order whichever CTA takes it, so O
    and lse are bitwise equal: a missing or misrouted item would show."""
    inp = wl.make_inputs(wl.WORKLOADS["single_head_256"], B=B, H=H, N=N, d=d, seed=N + d + causal)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=causal)
    o2, l2 = fa.forward(q, k, v, causal=causal, workspace=False)
    fa.sync_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    if B * H > 1000:  # the round-robin case: a few heads against the oracle too
        heads = [0, 4499, B * H - 1]
        o_ref, l_ref = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 1 / math.sqrt(d),
                                  causal, heads=heads)
        check_o_beyond_rounding(to_np(o2).reshape(B * H, N, d)[heads], o_ref, "round robin")
        check_lse(to_np(l2).reshape(B * H, N)[heads], l_ref, "round robin")


def test_persistent_calls_on_two_streams():
    """Two persistent forwards at once on two streams, each with its own work
    counter: the same bits as the calls one after the other."""
    w = wl.WORKLOADS["single_head_256"]
    a_in = wl.make_inputs(w, B=2, H=24, N=1000, d=128, seed=61)
    b_in = wl.make_inputs(w, B=2, H=24, N=1000, d=128, seed=62)
    qa, ka, va = (a_in[n].to(DEV) for n in ("q", "k", "v"))
    qb, kb, vb = (b_in[n].to(DEV) for n in ("q", "k", "v"))
    oa_ref, la_ref = fa.forward(qa, ka, va, causal=True)
    ob_ref, lb_ref = fa.forward(qb, kb, vb, causal=True)
    fa.sync_status()
    wsa, wsb = (torch.empty(256, dtype=torch.uint8, device=DEV) for _ in range(2))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    oa, la = fa.forward(qa, ka, va, causal=True, workspace=wsa, stream=sa)
    ob, lb = fa.forward(qb, kb, vb, causal=True, workspace=wsb, stream=sb)
    sa.synchronize()
    sb.synchronize()
    fa.sync_status()
    assert torch.equal(oa, oa_ref) and torch.equal(la, la_ref)
    assert torch.equal(ob, ob_ref) and torch.equal(lb, lb_ref)


def test_large_scores_dynamic_range():
    """Scores of magnitude ~100: the running max moves by far more than the
    rescale threshold, many times per row."""
    g = torch.Generator().manual_seed(3)
    B, H, N, d = 1, 4, 1024, 128
    q = (torch.randn(B, H, N, d, generator=g) * 4).to(torch.bfloat16)
    k = (torch.randn(B, H, N, d, generator=g) * 4).to(torch.bfloat16)
    # keys get larger along the sequence so the max keeps rising
    ramp = torch.linspace(0.2, 3.0, N).view(1, 1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    inp = {"q": q, "k": k, "v": v}
    for causal in (False, True):
        o, lse = run_fwd(inp, causal, 1.0 / math.sqrt(d))
        o_ref, l_ref = oracle.fwd(bits(q), bits(k), bits(v), 1.0 / math.sqrt(d), causal)
        check_o_beyond_rounding(to_np(o).reshape(o_ref.shape), o_ref, "dynamic range")
        check_lse(to_np(lse).reshape(l_ref.shape), l_ref, "dynamic range")


# ---------------------------------------------------------------------------
# invariants at full size
# ---------------------------------------------------------------------------

def test_causal_row0_equals_v0_full_size():
    w, inp, o, lse = workload_run("fwd_8k_d128_kx3", True)
    assert torch.equal(o[:, :, 0, :], inp["v"][:, :, 0, :])


def test_constant_values_give_constant_output():
    w = wl.WORKLOADS["fwd_2k_d64"]
    inp = wl.make_inputs(w)
    c = torch.randn(w.B, w.H, 1, w.d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    inp["v"] = c.expand(w.B, w.H, w.N, w.d).contiguous()
    for causal in (False, True):
        o, _ = run_fwd(inp, causal, w.scale)
        # the weights sum to one up to fp32/bf16 rounding: O is V within one bf16 ulp
        err = (o.cpu().double() - inp["v"].double()).abs()
        ulp = 2.0 * torch.from_numpy(bf16_half_ulp(inp["v"].double().numpy()))
        assert bool((err <= ulp).all()), f"max err {err.max().item()}"


def test_key_value_permutation_invariance():
    w = wl.WORKLOADS["fwd_2k_d64"]
    inp = wl.make_inputs(w, B=1, H=4)
    perm = torch.randperm(w.N, generator=torch.Generator().manual_seed(4))
    o1, l1 = run_fwd(inp, False, w.scale)
    inp2 = dict(inp, k=inp["k"][:, :, perm].contiguous(), v=inp["v"][:, :, perm].contiguous())
    o2, l2 = run_fwd(inp2, False, w.scale)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


# ---------------------------------------------------------------------------
# API behaviour on the device
# ---------------------------------------------------------------------------

def test_guard_bands_untouched():
    B, H, N, d = 2, 2, 300, 128
    inp = wl.make_inputs(wl.WORKLOADS["single_head_256"], B=B, H=H, N=N, d=d, seed=8)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o, chk_o = with_guard((B, H, N, d), torch.bfloat16, DEV)
    lse, chk_l = with_guard((B, H, N), torch.float32, DEV)
    for causal in (False, True):
        fa.forward(q, k, v, causal=causal, out=o, lse=lse)
        fa.sync_status()
        chk_o()
        chk_l()


def test_non_default_stream_and_repeat_determinism():
    w = wl.WORKLOADS["fwd_2k_d64"]
    inp = wl.make_inputs(w, B=1, H=8)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = fa.forward(q, k, v, causal=True)
        o2, l2 = fa.forward(q, k, v, causal=True)
    fa.sync_status(s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_device_argument_errors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 1, 128, dtype=torch.float32, device=DEV)
    h = torch.cuda.current_stream().cuda_stream
    rc = fa.fa_fwd(q.data_ptr() + 2, q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(),
                   1, 1, 128, 64, 0.125, 0, h)
    assert rc == fa.FA_ERR_MISALIGNED
    assert fa.fa_sync_status(h) == fa.FA_OK
