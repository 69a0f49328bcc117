"""FP8 forward on the GPU, through the C ABI, against the CPU oracle.

"FlashAttention 1–4" §"FlashAttention-3", paragraph "FP8 with block quantization
and incoherent processing".  Three checks:
  * the quantizer's E4M3 codes and fp32 scales equal the oracle's bit for bit
    (both take every rounding decision in fp32);
  * O of the FP8 forward differs from exact attention on the dequantized codes
    by no more than the oracle's bound on rounding P to E4M3, and lse (fp32 P)
    matches within 1e-3;
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


QUANT_CASES = [
    # (B, H, N, rotate, per_tensor)
    (1, 1, 1, True, False),
    (1, 2, 127, True, False),
    (2, 2, 300, True, False),
    (1, 3, 1000, False, False),
    (2, 1, 513, True, True),
    (1, 2, 256, False, True),
]


@pytest.mark.parametrize("B,H,N,rotate,per_tensor", QUANT_CASES)
def test_quantizer_bit_exact(B, H, N, rotate, per_tensor):
    inp = wl.outlier_inputs(B, H, N, D, seed=100 + N, kind="entries")
    ws, words = run_quant(inp, rotate=rotate, per_tensor=per_tensor)
    views = {n: t.cpu().numpy() for n, t in fa.fp8_workspace_views(ws, B, H, N).items()}
    ref = oracle_quant(inp, words, rotate, per_tensor)
    T = (N + 127) // 128
    npad = 128 * T
    for name, key in (("q8", "q"), ("k8", "k")):
        got = views[name]
        assert np.array_equal(got[:, :N], ref[key][0]), f"{name} codes differ"
        assert not got[:, N:].any(), f"{name} padding rows are not zero"
    # V^T: un-permute the keys of every tile
    vt = views["vt8"].reshape(B * H, D, T, 128)
    v_rows = np.empty((B * H, T, 128, D), np.uint8)
    v_rows[:, :, PERM, :] = vt.transpose(0, 2, 3, 1)
    v_rows = v_rows.reshape(B * H, npad, D)
    assert np.array_equal(v_rows[:, :N], ref["v"][0]), "vt8 codes differ"
    assert not v_rows[:, N:].any(), "vt8 padding keys are not zero"
    for name, key in (("sq", "q"), ("sk", "k"), ("sv", "v")):
        assert np.array_equal(views[name].view(np.uint32), ref[key][1].view(np.uint32)), \
            f"{name} scales differ"
    sv = ref["v"][1]
    vmax = sv.max(axis=1)
    assert np.array_equal(views["vmax"], vmax)
    assert np.array_equal(views["vfold"], (sv / vmax[:, None]).astype(np.float32))


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
    scale = 1.0 / math.sqrt(D)
    inp, words, o, lse = fp8_case(B, H, N, causal, rotate, per_tensor, seed=N)
    quant = oracle_quant(inp, words, rotate, per_tensor)
    bound, o_ref, _ = ofp8.p_rounding_bound(quant, scale, causal)
    _, lse_ref = ofp8.attention_on_codes(quant, scale, causal)
    # rounding of the bf16 output, plus fp32 scores / ex2 (relative 1e-4 of the
    # bound's scale is far above their ~1e-6)
    slack = bf16_half_ulp(o_ref) + 1e-4 * np.abs(o_ref) + 1e-6
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all()
    excess = err - (bound + slack)
    assert excess.max() <= 0, (
        f"max err {err.max():.3e} exceeds the P-rounding bound by {excess.max():.3e}; "
        f"rms err {np.sqrt((err ** 2).mean()):.3e}, mean bound {bound.mean():.3e}")
    # the bound is a worst case; the typical error must sit well inside it
    assert err.mean() <= 0.5 * bound.mean() + 1e-6
    check_lse(lse, lse_ref, f"fp8 lse B={B} H={H} N={N} causal={causal}")


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
    assert np.array_equal(views["q8"], quant["q"][0]) and np.array_equal(views["k8"], quant["k"][0])
    for name, key in (("sq", "q"), ("sk", "k"), ("sv", "v")):
        assert np.array_equal(views[name].view(np.uint32), quant[key][1].view(np.uint32))
    T = w.N // 128
    vt = views["vt8"].reshape(w.BH, D, T, 128).transpose(0, 2, 3, 1)
    assert np.array_equal(vt[:, :, np.argsort(PERM), :].reshape(w.BH, w.N, D), quant["v"][0])
    rows = wl.sampled_rows(w, count=64)
    bound, o_ref, lse_ref = ofp8.p_rounding_bound(quant, w.scale, True, rows=rows)
    o = to_np(o).reshape(w.BH, w.N, D)
    lse = to_np(lse).reshape(w.BH, w.N)
    got = np.stack([o[b][rows[b]] for b in range(w.BH)])
    got_l = np.stack([lse[b][rows[b]] for b in range(w.BH)])
    err = np.abs(got - o_ref)
    slack = bf16_half_ulp(o_ref) + 1e-4 * np.abs(o_ref) + 1e-6
    assert (err - bound - slack).max() <= 0, f"max err {err.max():.3e}"
    assert err.mean() <= 0.5 * bound.mean() + 1e-6
    check_lse(got_l, lse_ref, "fp8 full size lse")


def test_fp8_single_key_is_exact_value():
    """N = 1: the one weight is 1, so O is V's only row as its E4M3 code times
    its scale (the largest weight is corrected in the row sum), and lse is the
    score of the dequantized q . k."""
    inp = wl.outlier_inputs(1, 4, 1, D, seed=5, kind="entries")
    words = wl.sign_bits(6)
    o = fa.forward_fp8(*(inp[n].to(DEV) for n in ("q", "k", "v")), signs=words)[0]
    fa.sync_status()
    quant = oracle_quant(inp, words, True, False)
    vd = ofp8.dequantize_tiles(*quant["v"])
    got = to_np(o).reshape(4, 1, D)
    assert np.all(np.abs(got - vd) <= bf16_half_ulp(vd) + 1e-6 * np.abs(vd))


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
    inp = wl.outlier_inputs(B, H, N, D, seed=seed, kind=kind)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o_ref, _ = oracle.fwd(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), 1.0 / math.sqrt(D), causal)
    words = wl.sign_bits(seed + 1)
    out = {}
    for name, rot, pt in (("tile+rotate", True, False), ("tile", False, False),
                          ("tensor+rotate", True, True), ("tensor", False, True)):
        o = fa.forward_fp8(q, k, v, signs=words, causal=causal, rotate=rot, per_tensor=pt)[0]
        out[name] = float(np.sqrt(((to_np(o).reshape(o_ref.shape) - o_ref) ** 2).mean()))
    o16 = fa.forward(q, k, v, causal=causal)[0]
    out["bf16"] = float(np.sqrt(((to_np(o16).reshape(o_ref.shape) - o_ref) ** 2).mean()))
    fa.sync_status()
    return out


@pytest.mark.parametrize("kind", ["entries", "channels"])
def test_rmse_outliers(kind):
    r = rmse_modes(kind)
    print(f"\nRMSE vs exact attention, outliers '{kind}': " +
          ", ".join(f"{k} {v:.3e}" for k, v in r.items()) +
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
    bound, o_ref, _ = ofp8.p_rounding_bound(quant, scale, True)
    _, lse_ref = ofp8.attention_on_codes(quant, scale, True)
    got = to_np(o[:nb])
    slack = bf16_half_ulp(o_ref) + 1e-4 * np.abs(o_ref) + 1e-6
    assert (np.abs(got - o_ref) - (bound + slack)).max() <= 0
    check_lse(to_np(lse[:nb]), lse_ref, "fp8 lse, 65535 heads")
