"""Pins of the FP8 oracle (oracle/fp8.py) against what the pages and the
mathematics fix: the E4M3 grid, the Sylvester Hadamard matrix, the rotation
M = diag(s) H / sqrt(d) ("FlashAttention 1–4" §"FlashAttention-3", FP8 with
block quantization and incoherent processing), per-tile scaling, and the
bound on rounding P.  A few tests plant a mistake in a copy of an oracle
function and check that a pin catches it."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split(":", 1)
                out[key.strip()] = float(val)
    return out


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------

def finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def test_e4m3_decode_matches_torch_float8():
    c = finite_codes()
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_decode(c), ref)


def test_e4m3_round_matches_torch_float8():
    r = np.random.default_rng(0)
    x = np.concatenate([
        r.standard_normal(20000) * 10.0 ** r.uniform(-4, 2.7, 20000),
        fp8.e4m3_decode(finite_codes()),                   # grid points
        (fp8.e4m3_decode(finite_codes())[:-1] + fp8.e4m3_decode(finite_codes())[1:]) / 2,
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(x), ref)


@pytest.mark.parametrize("x,want", [
    (448.0, 448.0),                 # largest finite value
    (464.0, 448.0),                 # saturates (no infinity in E4M3)
    (1e6, 448.0),
    (-500.0, -448.0),
    (2.0 ** -9, 2.0 ** -9),         # smallest subnormal
    (2.0 ** -10, 0.0),              # tie between 0 and 2^-9: even (0)
    (3 * 2.0 ** -10, 2.0 ** -8),    # tie between 2^-9 and 2^-8: even (2 * 2^-9)
    (1.0625, 1.0),                  # tie between 1 and 1.125: even mantissa
    (1.1875, 1.25),                 # tie between 1.125 and 1.25: even mantissa
    (2.0 ** -6, 2.0 ** -6),         # smallest normal
    (0.0, 0.0),
])
def test_e4m3_round_closed_forms(x, want):
    assert fp8.e4m3_round(np.array([x]))[0] == want


def test_e4m3_encode_decode_round_trip():
    c = finite_codes()
    v = fp8.e4m3_decode(c)
    back = fp8.e4m3_encode(v)
    zero_neg = (c == 0x80)          # -0 encodes as 0x80 too
    assert np.array_equal(back[~zero_neg], c[~zero_neg])
    assert fp8.e4m3_encode(np.array([448.0]))[0] == 0x7E


# ---------------------------------------------------------------------------
# Hadamard rotation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_is_scipy_sylvester(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    assert np.array_equal(fp8.hadamard(d), scipy_linalg.hadamard(d))
    h = fp8.hadamard(d)
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_hadamard_recursion():
    h4, h8 = fp8.hadamard(4), fp8.hadamard(8)
    assert np.array_equal(h8, np.block([[h4, h4], [h4, -h4]]))


def test_signs_from_bits():
    words = np.array([0b101, 0, 0, 1 << 31], np.uint32)
    s = fp8.signs_from_bits(words, 128)
    neg = np.flatnonzero(s < 0)
    assert list(neg) == [0, 2, 127]


def test_rotation_signs_come_first():
    """M = diag(s) H / sqrt(d): the first basis vector goes to s_0 / sqrt(d)
    times a constant vector (row 0 of H is all ones).  Applying the signs after
    H instead would give s_j / sqrt(d), not constant."""
    d = 16
    s = np.where(np.arange(d) % 3 == 0, -1.0, 1.0)
    y = fp8.rotate(np.eye(d)[:1], s)[0]
    assert np.allclose(y, np.full(d, s[0] / math.sqrt(d)), rtol=0, atol=1e-15)
    y32 = fp8.rotate_f32(np.eye(d)[:1], s)[0]
    assert np.all(y32 == np.float32(s[0] / math.sqrt(d)))


def test_rotation_is_orthogonal_and_keeps_scores():
    r = np.random.default_rng(1)
    d = 128
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    m = fp8.rotate(np.eye(d), s)
    assert np.abs(m @ m.T - np.eye(d)).max() < 1e-13
    q, k = r.standard_normal((50, d)), r.standard_normal((70, d))
    assert np.abs(fp8.rotate(q, s) @ fp8.rotate(k, s).T - q @ k.T).max() < 1e-11


def test_rotate_f32_matches_fp64_rotation():
    r = np.random.default_rng(2)
    d = 128
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    x = (r.standard_normal((200, d)) * 3).astype(np.float32)
    y64 = fp8.rotate(x.astype(np.float64), s)
    y32 = fp8.rotate_f32(x, s).astype(np.float64)
    # seven butterfly levels and one scaling, each rounding to fp32
    tol = 8 * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) / math.sqrt(d)
    assert np.all(np.abs(y32 - y64) <= tol)


def test_spike_spreads_evenly():
    """A single outlier c e_i becomes a vector of entries +-c / sqrt(d)."""
    d = 8
    s = np.array([1, -1, -1, 1, 1, 1, -1, 1], dtype=np.float64)
    for i in range(d):
        y = fp8.rotate(8.0 * np.eye(d)[i:i + 1], s)[0]
        assert np.allclose(np.abs(y), 8.0 / math.sqrt(d), rtol=0, atol=1e-14)


def test_page_toy_vector():
    """The page's toy: one outlier 8.0 among 8 entries, length 8.03, largest
    entry 3.1 after the rotation.  Any such vector keeps its length, and its
    rotated maximum lies between the length / sqrt(8) (mean square) and
    (8 + sum of the seven small magnitudes) / sqrt(8); the page's 3.1 is inside."""
    g = load_golden("incoherent_toy_8.txt")
    d, out, rmax, length = int(g["d"]), g["outlier"], g["rotated_max"], g["length"]
    small = math.sqrt(length ** 2 - out ** 2)
    lo, hi = length / math.sqrt(d), (out + math.sqrt(d - 1) * small) / math.sqrt(d)
    assert lo <= rmax <= hi
    r = np.random.default_rng(3)
    hits = 0
    for _ in range(2000):
        x = r.standard_normal(d)
        x[0] = 0.0
        x *= small / np.linalg.norm(x)
        x[0] = out
        s = np.where(r.random(d) < 0.5, -1.0, 1.0)
        y = fp8.rotate(x[None], s)[0]
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
        assert lo - 1e-12 <= np.abs(y).max() <= hi + 1e-12
        hits += abs(np.abs(y).max() - rmax) < 0.05
    assert hits > 0   # the page's value is reached by such vectors


# ---------------------------------------------------------------------------
# block quantization
# ---------------------------------------------------------------------------

def test_tile_max_maps_to_448():
    r = np.random.default_rng(4)
    x = r.standard_normal((2, 300, 16)).astype(np.float32)
    codes, scales = fp8.quantize_tiles(x)
    for b in range(2):
        for t in range(3):
            blk = x[b, 128 * t:128 * (t + 1)]
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            assert fp8.e4m3_decode(codes[b, 128 * t:128 * (t + 1)][i]) == math.copysign(448.0, blk[i])
            assert scales[b, t] == np.float32(np.abs(blk).max()) / np.float32(448.0)


def test_quantization_error_is_half_ulp():
    r = np.random.default_rng(5)
    x = (r.standard_normal((1, 256, 32)) * 4).astype(np.float32)
    codes, scales = fp8.quantize_tiles(x)
    deq = fp8.dequantize_tiles(codes, scales)
    y = x.astype(np.float64) / np.repeat(scales.astype(np.float64), 128, axis=1)[:, :, None]
    # (codes are taken from x * (448 / amax) in fp32, y up to two fp32 roundings)
    bound = np.maximum(2.0 ** -4 * np.abs(y), 2.0 ** -10)   # in code units
    err = np.abs(deq - x) / np.repeat(scales.astype(np.float64), 128, axis=1)[:, :, None]
    assert np.all(err <= bound * (1 + 1e-6) + 4 * 2.0 ** -24 * np.abs(y))


def test_tiles_are_independent_and_per_tensor_is_global():
    r = np.random.default_rng(6)
    x = r.standard_normal((1, 256, 8)).astype(np.float32)
    y = x.copy()
    y[0, 5, 3] = 1000.0                          # an outlier in tile 0 only
    cx, sx = fp8.quantize_tiles(x)
    cy, sy = fp8.quantize_tiles(y)
    assert np.array_equal(cx[:, 128:], cy[:, 128:]) and sx[0, 1] == sy[0, 1]
    assert sy[0, 0] == np.float32(1000.0) / np.float32(448.0)
    ct, st = fp8.quantize_tiles(y, per_tensor=True)
    assert np.all(st == np.float32(1000.0) / np.float32(448.0))
    assert not np.array_equal(ct[:, 128:], cy[:, 128:])


def test_zero_tile_scale_is_one():
    codes, scales = fp8.quantize_tiles(np.zeros((1, 130, 4), np.float32))
    assert np.all(scales == 1.0) and not codes.any()


def test_attention_on_grid_values_is_lossless():
    """Entries already on the E4M3 grid, with 448 in every tile so that every
    scale is 1: quantization is exact, and attention on the codes equals the
    exact attention of the inputs."""
    r = np.random.default_rng(7)
    grid = fp8.e4m3_decode(finite_codes())
    grid = grid[np.abs(grid) <= 4]
    BH, N, d = 2, 200, 8
    x = {n: r.choice(grid, (BH, N, d)) for n in "qkv"}
    for n in "qkv":
        x[n][:, 0, 0] = 448.0
        x[n][:, 128, 0] = 448.0
    quant = fp8.quantize_qkv(x["q"], x["k"], x["v"], rotate=False)
    for n in "qkv":
        assert np.all(quant[n][1] == 1.0)
    o, lse = fp8.attention_on_codes(quant, 0.01, True)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], 0.01, True)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_rotation_leaves_attention_on_unquantized_values():
    """(QM)(KM)^T = QK^T: attention of the rotated fp64 Q, K equals that of Q, K."""
    r = np.random.default_rng(8)
    BH, N, d = 1, 50, 16
    q, k, v = (r.standard_normal((BH, N, d)) for _ in range(3))
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    o1, l1 = oracle.fwd(fp8.rotate(q, s), fp8.rotate(k, s), v, 0.25, False)
    o0, l0 = oracle.fwd(q, k, v, 0.25, False)
    assert np.abs(o1 - o0).max() < 1e-12 and np.abs(l1 - l0).max() < 1e-12


# ---------------------------------------------------------------------------
# the P-rounding bound
# ---------------------------------------------------------------------------

def emulate_p_rounding(quant, scale, causal, tile=128):
    """P rounded as the bound describes (fp64 p against the row max, y = p c_j
    rounded to E4M3, the largest weight of each tile corrected in the row sum)."""
    qd, kd, vd = fp8.dequantized_qkv(quant, tile)
    sv = quant["v"][1].astype(np.float64)
    c = fp8.P_SCALE * sv / sv.max(axis=1, keepdims=True)
    BH, N, d = qd.shape
    jt = np.arange(N) // tile
    out = np.empty((BH, N, d))
    for b in range(BH):
        s = scale * qd[b] @ kd[b].T
        if causal:
            s = np.where(np.arange(N)[None] <= np.arange(N)[:, None], s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ck = c[b][jt][None, :]
        pr = fp8.e4m3_round(p * ck) / ck
        l = p.sum(axis=1)
        for j in range(c.shape[1]):
            cols = jt == j
            pj = p[:, cols]
            i = pj.argmax(axis=1)
            pm = pj[np.arange(N), i]
            l = l + np.where(pm > 0, fp8.e4m3_round(pm * c[b, j]) / c[b, j] - pm, 0.0)
        out[b] = (pr @ vd[b]) / l[:, None]
    return out


@pytest.mark.parametrize("N,causal,vscale", [(300, True, 1.0), (260, False, 1.0), (200, True, 0.01)])
def test_p_rounding_bound_holds(N, causal, vscale):
    r = np.random.default_rng(N)
    BH, d = 2, 16
    q, k = (r.standard_normal((BH, N, d)).astype(np.float32) * 2 for _ in range(2))
    v = r.standard_normal((BH, N, d)).astype(np.float32)
    v[:, 128:] *= vscale                         # small V tiles: small fold, subnormal P
    quant = fp8.quantize_qkv(q, k, v, rotate=False)
    bound, o_codes, lse_codes = fp8.p_rounding_bound(quant, 0.5, causal)
    o_codes2, lse2 = fp8.attention_on_codes(quant, 0.5, causal)
    assert np.abs(o_codes - o_codes2).max() < 1e-12
    assert np.abs(lse_codes - lse2).max() < 1e-12
    rows = np.array([[0, 7, N - 1], [1, N // 2, N - 2]])
    b_s, o_s, l_s = fp8.p_rounding_bound(quant, 0.5, causal, rows=rows)
    for h in range(2):
        assert np.abs(o_s[h] - o_codes[h][rows[h]]).max() < 1e-12
        assert np.abs(b_s[h] - bound[h][rows[h]]).max() < 1e-12
        assert np.abs(l_s[h] - lse_codes[h][rows[h]]).max() < 1e-12
    em = emulate_p_rounding(quant, 0.5, causal)
    err = np.abs(em - o_codes)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err.max() > 0.05 * bound.max()        # the bound is not vacuous by orders of magnitude


# ---------------------------------------------------------------------------
# planted mistakes: a wrong oracle must fail a pin
# ---------------------------------------------------------------------------

def test_planted_signs_after_hadamard_is_caught():
    def bad_rotate(x, signs):
        d = x.shape[-1]
        return (np.asarray(x, np.float64) @ fp8.hadamard(d)) * signs / math.sqrt(d)
    d = 16
    s = np.where(np.arange(d) % 3 == 0, -1.0, 1.0)
    y = bad_rotate(np.eye(d)[:1], s)[0]
    assert not np.allclose(y, np.full(d, s[0] / math.sqrt(d)))


def test_planted_ties_away_from_zero_is_caught():
    def bad_round(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
        step = np.exp2(e - 3)
        return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), x)
    assert bad_round(np.array([1.0625]))[0] != 1.0      # the tie pin rejects it


def test_planted_wrong_scale_is_caught():
    r = np.random.default_rng(9)
    x = r.standard_normal((1, 128, 8)).astype(np.float32)
    amax = np.float32(np.abs(x).max())
    bad_scale = amax / np.float32(240.0)                 # E4M3's other maximum convention
    code = fp8.e4m3_round(np.array([amax / bad_scale]))[0]
    assert code != 448.0                                 # the max-to-448 pin rejects it
