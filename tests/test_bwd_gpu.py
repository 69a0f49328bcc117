"""Backward pass on the GPU, through the C ABI, against the fp64 oracle.

The GPU backward consumes the GPU forward's own bf16 O and fp32 lse; the oracle
uses its own fp64 forward.  Gradients are compared per tensor with
max|err| / max|ref| <= 2e-2."""
import math

import numpy as np
import pytest
import torch

import oracle
import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl
from parity import bits, check_grad, check_lse, check_o, grad_rel, to_np, with_guard

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def gpu_fwd_bwd(inp, causal, scale):
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    fa.sync_status()
    return o, lse, dq, dk, dv


def small_inputs(B, H, N, d, seed):
    w = wl.WORKLOADS["fwdbwd_4k_d128"]
    return wl.make_inputs(w, B=B, H=H, N=N, d=d, seed=seed)


@pytest.mark.parametrize("N", [1, 3, 64, 128, 200, 256, 384, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_small_full_compare(N, d, causal):
    B, H = 1, 3
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=2000 + N + d + causal)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale, causal)
    for got, ref, name in ((dq, g[0], "dq"), (dk, g[1], "dk"), (dv, g[2], "dv")):
        check_grad(to_np(got).reshape(ref.shape), ref, f"{name} N={N} d={d} causal={causal}")


def test_fwdbwd_4k_d128_all_heads():
    """The fwd+bwd workload (B=4 H=16 N=4096 d=128, causal) in full: O, lse,
    dQ, dK and dV of all 64 heads against the oracle, element by element."""
    w = wl.WORKLOADS["fwdbwd_4k_d128"]
    inp = wl.make_inputs(w)
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp, True, w.scale)
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), w.scale, True)
    rels = {}
    for got, ref, name in ((dq, g[0], "dq"), (dk, g[1], "dk"), (dv, g[2], "dv")):
        rels[name] = check_grad(to_np(got).reshape(ref.shape), ref, f"{name} all heads")
    print("fwdbwd 4k relative errors:", rels)
    # the forward output of this workload also meets the forward gates
    check_o(to_np(o).reshape(g[3].shape), g[3], "fwdbwd 4k O")
    check_lse(to_np(lse).reshape(g[4].shape), g[4], "fwdbwd 4k lse")


def test_stage_entry_points_match_fa_bwd():
    B, H, N, d = 2, 2, 640, 128
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=7)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    dq1, dk1, dv1 = fa.backward(q, k, v, o, lse, do, causal=True)
    ws = fa.alloc_workspace(B, H, N, d, DEV)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    h = torch.cuda.current_stream().cuda_stream
    assert fa.fa_bwd_prep(o.data_ptr(), do.data_ptr(), lse.data_ptr(), B, H, N, d, ws.data_ptr(),
                          ws.numel(), h) == 0
    assert fa.fa_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(),
                          dk2.data_ptr(), dv2.data_ptr(), B, H, N, d, scale, 1, ws.data_ptr(),
                          ws.numel(), h) == 0
    assert fa.fa_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(),
                        dq2.data_ptr(), B, H, N, d, scale, 1, ws.data_ptr(), ws.numel(), h) == 0
    fa.sync_status()
    # dQ, dK and dV are each accumulated on chip in a fixed order: bitwise equal
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


@pytest.mark.parametrize("N,d", [(128, 128), (256, 128), (200, 128), (128, 64), (256, 64), (200, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_many_short_items_per_cta(N, d, causal):
    """400 heads of one or two 128-row tiles (N = 200: the second one ragged): the
    persistent dK/dV and dQ kernels (one CTA per SM) each run several short work
    items back to back, so item hand-over, the rings that run on across items
    and the per-item barriers are exercised many times per CTA."""
    B, H = 2, 200
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=3000 + N + d + causal)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
    heads = list(range(0, B * H, 7)) + [B * H - 1]
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale, causal,
                   heads=heads)
    for got, ref, name in ((dq, g[0], "dq"), (dk, g[1], "dk"), (dv, g[2], "dv")):
        check_grad(to_np(got).reshape(B * H, N, d)[heads], ref, f"{name} N={N} d={d} causal={causal}")


def test_main_and_dq_concurrently_on_two_streams():
    """After prep, the dK/dV and dQ stages on two streams at once (each takes its
    work items from its own counter in the workspace): bitwise equal to fa_bwd."""
    B, H, N, d = 4, 16, 1024, 128
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=11)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    dq1, dk1, dv1 = fa.backward(q, k, v, o, lse, do, causal=True)
    ws = fa.alloc_workspace(B, H, N, d, DEV)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    main = torch.cuda.current_stream()
    assert fa.fa_bwd_prep(o.data_ptr(), do.data_ptr(), lse.data_ptr(), B, H, N, d, ws.data_ptr(),
                          ws.numel(), main.cuda_stream) == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(main)
    s2.wait_stream(main)
    assert fa.fa_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(),
                          dk2.data_ptr(), dv2.data_ptr(), B, H, N, d, scale, 1, ws.data_ptr(),
                          ws.numel(), s1.cuda_stream) == 0
    assert fa.fa_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(),
                        dq2.data_ptr(), B, H, N, d, scale, 1, ws.data_ptr(), ws.numel(),
                        s2.cuda_stream) == 0
    main.wait_stream(s1)
    main.wait_stream(s2)
    fa.sync_status()
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


def test_guard_bands_and_workspace_reuse():
    B, H, N, d = 1, 3, 300, 64
    inp = small_inputs(B, H, N, d, seed=9)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=False)
    bufs = [with_guard((B, H, N, d), torch.bfloat16, DEV) for _ in range(3)]
    ws = fa.alloc_workspace(B, H, N, d, DEV)
    ws.fill_(0x7F)  # garbage in the workspace must not matter
    outs = []
    for _ in range(2):
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=False, dq=bufs[0][0], dk=bufs[1][0],
                                 dv=bufs[2][0], workspace=ws)
        fa.sync_status()
        outs.append((dq.clone(), dk.clone(), dv.clone()))
        for _, chk in bufs:
            chk()
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]),
                   1.0 / math.sqrt(d), False)
    for got, ref in zip(outs[1], g[:3]):
        check_grad(to_np(got).reshape(ref.shape), ref, "guarded")


def test_fwd_2k_d64_backward_both_modes():
    """d = 64 at the size of the d = 64 forward workload (dO drawn with the same
    recipe): all 64 heads of dQ, dK and dV against the oracle, both masks."""
    w = wl.WORKLOADS["fwd_2k_d64"]
    inp = wl.make_inputs(w)
    inp["do"] = wl.random_bf16(w.shape(), seed=w.seed + 100)
    for causal in (False, True):
        o, lse, dq, dk, dv = gpu_fwd_bwd(inp, causal, w.scale)
        g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), w.scale,
                       causal)
        for got, ref, name in ((dq, g[0], "dq"), (dk, g[1], "dk"), (dv, g[2], "dv")):
            check_grad(to_np(got).reshape(ref.shape), ref, f"{name} 2k d64 causal={causal}")


def test_autograd_wrapper_matches_oracle():
    """attention() under torch.autograd: O and the gradients of sum(dO * O)."""
    B, H, N, d = 1, 2, 333, 128
    inp = small_inputs(B, H, N, d, seed=77)
    q, k, v = (inp[n].to(DEV).requires_grad_(True) for n in ("q", "k", "v"))
    do = inp["do"].to(DEV)
    o = fa.attention(q, k, v, causal=True)
    o.backward(do)
    fa.sync_status()
    scale = 1.0 / math.sqrt(d)
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale, True)
    err = np.abs(to_np(o).reshape(g[3].shape) - g[3])
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    for got, ref, name in ((q.grad, g[0], "dq"), (k.grad, g[1], "dk"), (v.grad, g[2], "dv")):
        check_grad(to_np(got).reshape(ref.shape), ref, f"autograd {name}")


def test_entry_points_from_a_fresh_host_thread():
    """Every entry point called first on a thread that has made no CUDA call
    (autograd runs the backward on such a worker thread): the library makes
    the device's context current itself before encoding its tensor maps."""
    import threading
    B, H, N, d = 1, 2, 333, 128
    inp = small_inputs(B, H, N, d, seed=78)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    o_ref, lse_ref = fa.forward(q, k, v, causal=True)
    g_ref = fa.backward(q, k, v, o_ref, lse_ref, do, causal=True)
    words = wl.sign_bits(5)
    o8_ref = fa.forward_fp8(q, k, v, signs=words, causal=True)[0]
    fa.sync_status()
    torch.cuda.synchronize()
    out = {}

    def work(name):
        try:
            if name == "fwd":
                out[name] = fa.forward(q, k, v, causal=True)
            elif name == "bwd":
                out[name] = fa.backward(q, k, v, o_ref, lse_ref, do, causal=True)
            else:
                out[name] = fa.forward_fp8(q, k, v, signs=words, causal=True)
            torch.cuda.synchronize()
        except Exception as e:  # reported below, in the test's own thread
            out[name] = e

    for name in ("fwd", "bwd", "fp8"):
        t = threading.Thread(target=work, args=(name,))
        t.start()
        t.join()
        assert not isinstance(out[name], Exception), f"{name}: {out[name]!r}"
    fa.sync_status()
    assert torch.equal(out["fwd"][0], o_ref) and torch.equal(out["fwd"][1], lse_ref)
    for a_, b_ in zip(out["bwd"], g_ref):
        assert torch.equal(a_, b_)
    assert torch.equal(out["fp8"][0], o8_ref)


def test_more_heads_than_a_grid_dimension():
    """B*H = 100000 heads of N = 200 (past the 65535 limit of a launch grid's y
    and z dimensions; every kernel here takes its work items on x or from a
    counter).  61 seeded heads (a prime, so a wrong head index lands on another
    pattern) tile all heads on the device: O, lse, dQ, dK and dV of every head
    must equal its base head's bit for bit, and the base heads must match the
    oracle."""
    nb, N, d, B, H = 61, 200, 64, 4, 25000
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(1, nb, N, d, seed=4242)
    reps = -(-(B * H) // nb)
    big = {n: inp[n].to(DEV).repeat(1, reps, 1, 1)[:, :B * H].reshape(B, H, N, d).contiguous()
           for n in ("q", "k", "v", "do")}
    o, lse = fa.forward(big["q"], big["k"], big["v"], scale=scale, causal=True)
    dq, dk, dv = fa.backward(big["q"], big["k"], big["v"], o, lse, big["do"], scale=scale, causal=True)
    fa.sync_status()
    del big
    base = torch.arange(B * H, device=DEV) % nb
    outs = {"o": o.reshape(B * H, N, d), "lse": lse.reshape(B * H, N), "dq": dq.reshape(B * H, N, d),
            "dk": dk.reshape(B * H, N, d), "dv": dv.reshape(B * H, N, d)}
    for name, t in outs.items():
        assert torch.equal(t, t[:nb][base]), f"{name}: a head differs from its base head"
    g = oracle.bwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale, True)
    for name, ref in (("dq", g[0]), ("dk", g[1]), ("dv", g[2])):
        check_grad(to_np(outs[name][:nb]), ref, f"{name}, 100000 heads")
    err = np.abs(to_np(outs["o"][:nb]) - g[3])
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(to_np(outs["lse"][:nb]) - g[4]).max() <= 1e-3


def sampled_key_rows(N, BH, count, lo, seed):
    """count distinct key rows per head from [lo, N), N - 1 and lo always in."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(BH):
        r = rng.choice(np.arange(lo + 1, N - 1), count - 2, replace=False)
        out.append(np.sort(np.concatenate([[lo, N - 1], r])))
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (64, True), (128, False)])
def test_long_sequence_sampled_rows_and_invariants(d, causal):
    """N = 2^17 (1024 key and query tiles per head).  Element by element against
    the oracle's sampled-row backward: dQ on 64 seeded query rows per head (rows
    0 and N - 1 among them); dK and dV, when causal, on 32 seeded key rows per
    head from the last 8192 keys (each sums over the query rows that see it,
    so the oracle needs those rows' statistics: the tail keeps that to the last
    8192 rows; the non-causal key rows are checked at N = 2^15 below).  On every
    key row and column, the identities that hold at any size: sum_j dK_j = 0
    (each row of dS sums to zero) and sum_j dV_j = sum_i dO_i (each row of P
    sums to one)."""
    B, H, N = 1, 2, 1 << 17
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=5000 + d + causal)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, causal, scale)
    dq_n = to_np(dq).reshape(B * H, N, d)
    dk_n = to_np(dk).reshape(B * H, N, d)
    dv_n = to_np(dv).reshape(B * H, N, d)
    qrows = sampled_key_rows(N, B * H, 64, 0, seed=6000 + d + causal)
    krows = sampled_key_rows(N, B * H, 32, N - 8192, seed=6100 + d) if causal else None
    g = oracle.bwd_rows(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale,
                        causal, qrows=qrows, krows=krows)
    take = lambda a, r: np.take_along_axis(a, r[:, :, None], axis=1)
    check_grad(take(dq_n, qrows), g[0], f"dq sampled rows N=2^17 d={d}")
    if causal:
        check_grad(take(dk_n, krows), g[1], f"dk sampled key rows N=2^17 d={d}")
        check_grad(take(dv_n, krows), g[2], f"dv sampled key rows N=2^17 d={d}")
    sk = np.abs(dk_n.sum(axis=1)) / np.maximum(np.abs(dk_n).sum(axis=1), 1e-30)
    assert sk.max() <= 1e-2, f"sum_j dK_j not ~0: {sk.max()}"
    do_n = inp["do"].double().numpy().reshape(B * H, N, d)
    sv = np.abs(dv_n.sum(axis=1) - do_n.sum(axis=1)) / np.maximum(np.abs(dv_n).sum(axis=1), 1e-30)
    assert sv.max() <= 1e-2, f"sum_j dV_j != sum_i dO_i: {sv.max()}"


def test_long_sequence_non_causal_key_rows():
    """Non-causal key rows sum over every query row, so the oracle needs the
    whole head's statistics: at N = 2^15 (256 tiles, d = 64, two heads), dK
    and dV on 32 seeded key rows per head (0 and N - 1 among them) and dQ on
    32 seeded query rows, element by element."""
    B, H, N, d = 1, 2, 1 << 15, 64
    scale = 1.0 / math.sqrt(d)
    inp = small_inputs(B, H, N, d, seed=5200)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, False, scale)
    krows = sampled_key_rows(N, B * H, 32, 0, seed=6200)
    qrows = sampled_key_rows(N, B * H, 32, 0, seed=6300)
    g = oracle.bwd_rows(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), bits(inp["do"]), scale,
                        False, qrows=qrows, krows=krows)
    take = lambda t, r: np.take_along_axis(to_np(t).reshape(B * H, N, d), r[:, :, None], axis=1)
    check_grad(take(dq, qrows), g[0], "dq sampled rows N=2^15")
    check_grad(take(dk, krows), g[1], "dk sampled key rows N=2^15")
    check_grad(take(dv, krows), g[2], "dv sampled key rows N=2^15")


def test_largest_accepted_size():
    """The largest inputs the boundary takes: B·H·N·d = 16 · (2^20 - 64) · 128 =
    2^31 - 2^17 elements (2^31 is refused), causal, with a ragged last tile.
    Forward O and lse and backward dQ on 16 seeded rows of the first and the
    last head (rows 0 and N - 1 among them) against the oracle, element by
    element; on every head the identities sum_j dK_j = 0 and
    sum_j dV_j = sum_i dO_i, summed in fp64 on the device."""
    B, H, N, d = 1, 16, (1 << 20) - 64, 128
    assert B * H * N * d < (1 << 31) <= B * H * (N + 64) * d
    scale = 1.0 / math.sqrt(d)
    inp = wl.make_inputs_device(B, H, N, d, seed=7000, device=DEV)
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp, True, scale)
    heads = [0, H - 1]
    rows = sampled_key_rows(N, len(heads), 16, 0, seed=7100)
    sel = lambda t: bits(t[:, heads])
    take = lambda t, width: np.stack([to_np(t.reshape(B * H, N, width)[h][torch.as_tensor(r, device=DEV)])
                                      for h, r in zip(heads, rows)])
    o_ref, l_ref = oracle.fwd_rows(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), scale, True, rows)
    check_o(take(o, d), o_ref, "largest size O")
    check_lse(take(lse, 1)[..., 0], l_ref, "largest size lse")
    g = oracle.bwd_rows(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["do"]), scale, True,
                        qrows=rows)
    check_grad(take(dq, d), g[0], "largest size dq")
    sk = (torch.sum(dk, dim=2, dtype=torch.float64).abs() /
          torch.sum(dk.abs(), dim=2, dtype=torch.float64).clamp_min(1e-30))
    assert sk.max().item() <= 1e-2, f"sum_j dK_j not ~0: {sk.max().item()}"
    sv = ((torch.sum(dv, dim=2, dtype=torch.float64) - torch.sum(inp["do"], dim=2, dtype=torch.float64)).abs() /
          torch.sum(dv.abs(), dim=2, dtype=torch.float64).clamp_min(1e-30))
    assert sv.max().item() <= 1e-2, f"sum_j dV_j != sum_i dO_i: {sv.max().item()}"


def test_backward_bitwise_repeatable_back_to_back():
    """16 forward + backward passes of the fwd+bwd workload enqueued back to back
    on one stream (fresh output buffers each, no host synchronisation between
    them): every pass's dQ, dK and dV equal the first pass's bit for bit.  The
    dK/dV kernel's dO ring slots also hold each tile's D, which its compute
    threads read in the dS phase; a slot may be refilled only after both the dV
    product and those reads (releasing it after dV alone let dK pick up the
    next tile's D, now and then, with back-to-back launches)."""
    w = wl.WORKLOADS["fwdbwd_4k_d128"]
    inp = wl.make_inputs(w)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    ws = fa.alloc_workspace(w.B, w.H, w.N, w.d, DEV)
    outs = []
    for _ in range(16):
        o, lse = fa.forward(q, k, v, causal=True)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        fa.backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
        outs.append((dq, dk, dv))
    fa.sync_status()
    for n, (dq, dk, dv) in enumerate(outs[1:], 1):
        for got, ref, name in ((dq, outs[0][0], "dq"), (dk, outs[0][1], "dk"), (dv, outs[0][2], "dv")):
            if not torch.equal(got, ref):
                heads = torch.nonzero((got != ref).reshape(w.BH, -1).any(dim=1)).flatten().tolist()
                raise AssertionError(f"pass {n}: {name} differs from the first pass in heads {heads[:10]}")
