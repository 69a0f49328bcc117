"""FP8 forward on the GPU, through the C ABI, against the CPU oracle.

"FlashAttention 1–4" §"FlashAttention-3", paragraph "FP8 with block quantization
and incoherent processing".  The oracle computes the quantization exactly, in
fp64 (rotation, tile amax, x * 448 / amax rounded to E4M3); the checks:
  * every E4M3 code of the quantizer is the correctly rounded code of the exact
    value, except where the float32 error band of the value straddles a
    rounding boundary (either neighbour accepted, the cases counted); every
    fp32 scale lies within its float32 tolerance of amax / 448;
  * O of the FP8 forward against exact attention on the ORIGINAL bf16 inputs:
    RMSE <= 2 x the method's own error (exact attention on the exactly rounded
    codes) + the rms bf16 output rounding, and every element within 2 x that
    ideal error's maximum + half a bf16 ulp; lse within 1e-3 of exact
    attention on the codes;
  * diagnostic: O against exact attention on the oracle's codes within the
    bound on rounding P to E4M3 plus the slack of the band cases;
  * on inputs with simulated outlier features, block quantization plus the
    random-sign Hadamard rotation has a lower RMSE against exact attention on
    the original inputs than per-tensor scaling without rotation.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import workloads as wl
from parity import bf16_half_ulp, bits, check_lse, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
D = 128


def f32_of(t):
    """bf16 tensor [B,H,N,d] -> exact float32 numpy [BH,N,d]."""
    return (bits(t).astype(np.uint32) << 16).view(np.float32)


def key_of_index(i):
    """Key order of V^T within a 128-key tile (the layout fa.h documents):
    i = 64 h + 16 x + 2 w + e holds key 64 h + 8 w + 2 x + e."""
    h, x, w, e = i // 64, (i // 16) % 4, (i // 2) % 8, i % 2
    return 64 * h + 8 * w + 2 * x + e


PERM = np.array([key_of_index(i) for i in range(128)])


def run_quant(inp, signs_seed=11, rotate=True, per_tensor=False):
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    B, H, N, _ = q.shape
    words = wl.sign_bits(signs_seed)
    ws = fa.quantize_fp8(q, k, v, signs=words, rotate=rotate, per_tensor=per_tensor)
    fa.sync_status()
    return ws, words


def oracle_quant(inp, words, rotate, per_tensor):
    signs = ofp8.signs_from_bits(words, D)
    return ofp8.quantize_qkv(f32_of(inp["q"]), f32_of(inp["k"]), f32_of(inp["v"]), signs,
                             rotate=rotate, per_tensor=per_tensor)


def check_codes(got, ref, name):
    ok, n_band, n_bad = ofp8.codes_within_band(got, ref)
    assert ok, f"{name}: {n_bad} codes are neither the exact rounding nor a band neighbour"
    return n_band


def check_scales(got, ref, name):
    ok, worst = ofp8.scales_within_tolerance(got, ref)
    assert ok, f"{name}: a scale is {worst:.2f} x its float32 tolerance from amax / 448"


def exact_attention(inp, causal, rows=None):
    """Exact attention (fp64 oracle) on the original bf16 inputs: (o, lse)."""
    q, k, v = bits(inp["q"]), bits(inp["k"]), bits(inp["v"])
    if rows is None:
        return oracle.fwd(q, k, v, 1.0 / math.sqrt(D), causal)
    return oracle.fwd_rows(q, k, v, 1.0 / math.sqrt(D), causal, rows)


def check_budget(o, lse, exact, quant, causal, what, rows=None):
    """The FP8 gates against exact attention on the original inputs: O within
    its RMSE and element-wise budgets, lse within its budget."""
    o_exact, lse_exact = exact
    ideal = ofp8.ideal_fp8_error(o_exact, quant, 1.0 / math.sqrt(D), causal, rows=rows,
                                 lse_exact=lse_exact)
    rmse_b, max_b = ofp8.fp8_budget(o_exact, ideal)
    err = np.abs(o - o_exact)
    rmse = float(np.sqrt((err ** 2).mean()))
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    assert rmse <= rmse_b, f"{what}: RMSE {rmse:.3e} over the budget {rmse_b:.3e} (ideal {ideal[0]:.3e})"
    worst = (err - max_b).max()
    assert worst <= 0, (f"{what}: max err {err.max():.3e} over its budget by {worst:.3e} "
                        f"(ideal max {ideal[1]:.3e})")
    if lse is not None:
        lerr = np.abs(lse - lse_exact).max()
        assert lerr <= ofp8.fp8_lse_budget(ideal[2]), (
            f"{what}: lse max err {lerr:.3e} over its budget (ideal {ideal[2]:.3e})")
    return rmse, ideal


def check_diagnostic(o, lse, quant, causal, what, rows=None):
    """O within the P-rounding bound (plus band slack, bf16 rounding and fp32
    score arithmetic) of exact attention on the oracle's codes, the typical
    error well inside it; lse within 1e-3 plus the band cases' largest score
    change of the same attention's lse."""
    scale = 1.0 / math.sqrt(D)
    bound, o_ref, lse_ref = ofp8.p_rounding_bound(quant, scale, causal, rows=rows)
    slack = (ofp8.band_slack(quant, scale, causal, rows=rows) + bf16_half_ulp(o_ref)
             + 1e-4 * np.abs(o_ref) + 1e-6)
    err = np.abs(o - o_ref)
    excess = err - (bound + slack)
    assert excess.max() <= 0, (
        f"{what}: max err {err.max():.3e} exceeds the P-rounding bound by {excess.max():.3e}")
    assert err.mean() <= 0.5 * bound.mean() + 1e-6
    if lse is not None:
        lerr = np.abs(lse - lse_ref)
        ds = ofp8.band_score_slack(quant, scale, causal, rows=rows)
        assert np.isfinite(lse).all(), f"{what}: non-finite lse"
        assert (lerr - ds).max() <= 1e-3, (
            f"{what}: lse max err {lerr.max():.3e}, beyond the band slack by {(lerr - ds).max():.3e}")


QUANT_CASES = [
    # (B, H, N, rotate, per_tensor)
    (1, 1, 1, True, False),
    (1, 2, 127, True, False),
    (2, 2, 300, True, False),
    (1, 3, 1000, False, False),
    (2, 1, 513, True, True),
    (1, 2, 256, False, True),
]


def check_workspace(views, ref, B, H, N):
    """Codes (un-permuting V^T), padding, scales, vmax and fold of a filled
    FP8 workspace against the oracle's exact quantization.  Returns the number
    of band cases."""
    T = (N + 127) // 128
    npad = 128 * T
    n_band = 0
    for name, key in (("q8", "q"), ("k8", "k")):
        got = views[name]
        n_band += check_codes(got[:, :N], ref[key], name)
        assert not got[:, N:].any(), f"{name} padding rows are not zero"
    vt = views["vt8"].reshape(B * H, D, T, 128)
    v_rows = np.empty((B * H, T, 128, D), np.uint8)
    v_rows[:, :, PERM, :] = vt.transpose(0, 2, 3, 1)
    v_rows = v_rows.reshape(B * H, npad, D)
    n_band += check_codes(v_rows[:, :N], ref["v"], "vt8")
    assert not v_rows[:, N:].any(), "vt8 padding keys are not zero"
    for name, key in (("sq", "q"), ("sk", "k"), ("sv", "v")):
        check_scales(views[name], ref[key], name)
    # vmax = the head's largest V scale; fold = sv / vmax: a float32 rounding
    # of the exact ratio of tile maxima (and of that largest scale)
    amax = ref["v"]["amax"]
    vmax_exact = amax.max(axis=1) / 448.0
    assert np.all(np.abs(views["vmax"] - vmax_exact) <= 2 * ofp8.U32 * vmax_exact)
    fold_exact = amax / amax.max(axis=1, keepdims=True)
    assert np.all(np.abs(views["vfold"] - fold_exact) <= 4 * ofp8.U32 * fold_exact)
    return n_band


@pytest.mark.parametrize("B,H,N,rotate,per_tensor", QUANT_CASES)
def test_quantizer_codes_and_scales(B, H, N, rotate, per_tensor):
    inp = wl.outlier_inputs(B, H, N, D, seed=100 + N, kind="entries")
    ws, words = run_quant(inp, rotate=rotate, per_tensor=per_tensor)
    views = {n: t.cpu().numpy() for n, t in fa.fp8_workspace_views(ws, B, H, N).items()}
    ref = oracle_quant(inp, words, rotate, per_tensor)
    n_band = check_workspace(views, ref, B, H, N)
    print(f"\nB={B} H={H} N={N} rotate={rotate} per_tensor={per_tensor}: "
          f"{n_band} of {3 * B * H * N * D} codes in a straddling band")


def fp8_case(B, H, N, causal, rotate=True, per_tensor=False, seed=0, kind="entries"):
    inp = wl.outlier_inputs(B, H, N, D, seed=seed, kind=kind)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    words = wl.sign_bits(seed + 1)
    o, lse = fa.forward_fp8(q, k, v, signs=words, causal=causal, rotate=rotate,
                            per_tensor=per_tensor)
    fa.sync_status()
    return inp, words, to_np(o).reshape(B * H, N, D), to_np(lse).reshape(B * H, N)


PARITY_CASES = [
    # (B, H, N, causal, rotate, per_tensor)
    (1, 1, 1, False, True, False),
    (1, 1, 1, True, True, False),
    (1, 2, 200, False, True, False),
    (1, 2, 200, True, True, False),
    (2, 1, 640, True, True, False),
    (1, 2, 1000, False, False, False),
    (1, 1, 1357, True, True, True),
    (1, 2, 2048, True, True, False),
    # more work items than SMs: several waves of CTAs, one item each
    (4, 100, 256, True, True, False),
    (2, 80, 384, False, True, False),  # the second Q tile of every second item is past N
]


@pytest.mark.parametrize("B,H,N,causal,rotate,per_tensor", PARITY_CASES)
def test_fp8_forward_parity(B, H, N, causal, rotate, per_tensor):
    inp, words, o, lse = fp8_case(B, H, N, causal, rotate, per_tensor, seed=N)
    quant = oracle_quant(inp, words, rotate, per_tensor)
    what = f"fp8 B={B} H={H} N={N} causal={causal} rotate={rotate} per_tensor={per_tensor}"
    rmse, ideal = check_budget(o, lse, exact_attention(inp, causal), quant, causal, what)
    check_diagnostic(o, lse, quant, causal, what)
    print(f"\n{what}: RMSE vs exact attention {rmse:.3e} (method's own {ideal[0]:.3e})")


def test_fp8_full_size_sampled_rows():
    """The workload and launch the bench times (B=2 H=16 N=8192 d=128, K x3,
    causal, rotation on, per-tile scales): codes and scales bit-exact in full,
    O within the P-rounding bound and lse within 1e-3 on 64 sampled query rows
    per head (rows 0 and N-1 included)."""
    w = wl.WORKLOADS["fwd_8k_d128_kx3"]
    inp = wl.make_inputs(w)
    words = wl.sign_bits(w.seed + 7)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    ws = fa.quantize_fp8(q, k, v, signs=words)
    o, lse = fa.forward_fp8_quantized(ws, w.B, w.H, w.N, causal=True)
    fa.sync_status()
    views = {n: t.cpu().numpy() for n, t in fa.fp8_workspace_views(ws, w.B, w.H, w.N).items()}
    del q, k, v, ws
    quant = oracle_quant(inp, words, True, False)
    n_band = check_workspace(views, quant, w.B, w.H, w.N)
    rows = wl.sampled_rows(w, count=64)
    o = to_np(o).reshape(w.BH, w.N, D)
    lse = to_np(lse).reshape(w.BH, w.N)
    got = np.stack([o[b][rows[b]] for b in range(w.BH)])
    got_l = np.stack([lse[b][rows[b]] for b in range(w.BH)])
    rmse, ideal = check_budget(got, got_l, exact_attention(inp, True, rows), quant, True,
                               "fp8 full size", rows=rows)
    check_diagnostic(got, got_l, quant, True, "fp8 full size", rows=rows)
    print(f"\nfp8 full size: {n_band} band codes; RMSE vs exact attention {rmse:.3e} "
          f"(method's own {ideal[0]:.3e})")


def test_fp8_single_key_is_exact_value():
    """N = 1: the one weight is 1, so O is V's only row as its E4M3 code times
    its scale (the largest weight is corrected in the row sum), and lse is the
    score of the dequantized q . k."""
    inp = wl.outlier_inputs(1, 4, 1, D, seed=5, kind="entries")
    words = wl.sign_bits(6)
    o = fa.forward_fp8(*(inp[n].to(DEV) for n in ("q", "k", "v")), signs=words)[0]
    fa.sync_status()
    quant = oracle_quant(inp, words, True, False)
    vd = ofp8.dequantize_tiles(*ofp8.codes_and_scales(quant)["v"])
    got = to_np(o).reshape(4, 1, D)
    slack = ofp8.band_slack(quant, 1.0 / math.sqrt(D), False)
    assert np.all(np.abs(got - vd) <= bf16_half_ulp(vd) + 1e-6 * np.abs(vd) + slack)


def test_fp8_argument_errors():
    B, H, N = 1, 1, 64
    q = torch.zeros(B, H, N, D, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(fa.fp8_workspace_bytes(B, H, N), dtype=torch.uint8, device=DEV)
    p = q.data_ptr()
    sw = fa.sign_words([0, 0, 0, 0])
    s = fa._stream_handle()
    assert fa.fa_fp8_workspace_size(B, H, N, 64) == 0
    assert fa.fa_fp8_quantize(p, p, p, B, H, N, 64, sw, 1, ws.data_ptr(), ws.numel(), s) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fp8_quantize(p, p, p, B, H, N, D, None, 1, ws.data_ptr(), ws.numel(), s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fp8_quantize(p, p, p, B, H, N, D, sw, 4, ws.data_ptr(), ws.numel(), s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fp8_quantize(p, p, p, B, H, N, D, sw, 1, ws.data_ptr(), ws.numel() - 1, s) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fp8_quantize(p, p, p, B, H, N, D, sw, 1, ws.data_ptr() + 16, ws.numel() - 16, s) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fp8_quantize(p + 2, p, p, B, H, N, D, sw, 1, ws.data_ptr(), ws.numel(), s) == fa.FA_ERR_MISALIGNED
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    assert fa.fa_fwd_fp8(ws.data_ptr(), ws.numel(), p, lse.data_ptr(), B, H, N, D, 0.0, 0, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_fp8(ws.data_ptr(), ws.numel(), p, lse.data_ptr(), B, H, N, D, 0.1, 2, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_fp8(ws.data_ptr(), 100, p, lse.data_ptr(), B, H, N, D, 0.1, 0, s) == fa.FA_ERR_WORKSPACE
    assert fa.fa_sync_status(s) == fa.FA_OK


# ---------------------------------------------------------------------------
# RMSE study: simulated outlier features
# ---------------------------------------------------------------------------

def rmse_modes(kind, B=1, H=4, N=2048, causal=True, seed=21):
    """RMSE of O against exact attention on the original inputs for the four
    quantization modes and the bf16 kernel; every FP8 mode also meets its own
    budget (twice the error of exact attention on its exactly rounded codes)."""
    inp = wl.outlier_inputs(B, H, N, D, seed=seed, kind=kind)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    exact = exact_attention(inp, causal)
    o_ref = exact[0]
    words = wl.sign_bits(seed + 1)
    out, ideal = {}, {}
    for name, rot, pt in (("tile+rotate", True, False), ("tile", False, False),
                          ("tensor+rotate", True, True), ("tensor", False, True)):
        o = to_np(fa.forward_fp8(q, k, v, signs=words, causal=causal, rotate=rot,
                                 per_tensor=pt)[0]).reshape(o_ref.shape)
        quant = oracle_quant(inp, words, rot, pt)
        out[name], ideal[name] = check_budget(o, None, exact, quant, causal, f"'{kind}' {name}")
    o16 = fa.forward(q, k, v, causal=causal)[0]
    out["bf16"] = float(np.sqrt(((to_np(o16).reshape(o_ref.shape) - o_ref) ** 2).mean()))
    fa.sync_status()
    return out, ideal


@pytest.mark.parametrize("kind", ["entries", "channels"])
def test_rmse_outliers(kind):
    r, ideal = rmse_modes(kind)
    print(f"\nRMSE vs exact attention, outliers '{kind}': " +
          ", ".join(f"{k} {v:.3e}" for k, v in r.items()) +
          "; method's own: " + ", ".join(f"{k} {v[0]:.3e}" for k, v in ideal.items()) +
          f"; per-tensor / (per-tile + rotation) = {r['tensor'] / r['tile+rotate']:.2f}")
    assert r["tile+rotate"] < r["tensor"]
    assert r["bf16"] < r["tile+rotate"]


def test_fp8_largest_head_count():
    """B*H = 65535, the most heads the FP8 path takes (the quantizers put heads
    on the launch grid's y dimension).  61 seeded heads (a prime, so a wrong
    head index lands on another pattern) tile all 65535 on the device: every
    head's codes-based output must equal its base head's bit for bit, and the
    base heads must meet the oracle's P-rounding bound."""
    nb, N, B, H = 61, 128, 5, 13107
    scale = 1.0 / math.sqrt(D)
    inp = wl.outlier_inputs(1, nb, N, D, seed=77)
    reps = -(-(B * H) // nb)
    big = {n: inp[n].to(DEV).repeat(1, reps, 1, 1)[:, :B * H].reshape(B, H, N, D).contiguous()
           for n in ("q", "k", "v")}
    words = wl.sign_bits(78)
    o, lse = fa.forward_fp8(big["q"], big["k"], big["v"], signs=words, causal=True)
    fa.sync_status()
    del big
    o = o.reshape(B * H, N, D)
    lse = lse.reshape(B * H, N)
    base = torch.arange(B * H, device=DEV) % nb
    assert torch.equal(o, o[:nb][base]) and torch.equal(lse, lse[:nb][base])
    quant = oracle_quant(inp, words, True, False)
    got, got_l = to_np(o[:nb]), to_np(lse[:nb])
    check_budget(got, got_l, exact_attention(inp, True), quant, True, "fp8, 65535 heads")
    check_diagnostic(got, got_l, quant, True, "fp8, 65535 heads")
