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


def test_rotation_is_orthogonal_and_keeps_scores():
    r = np.random.default_rng(1)
    d = 128
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    m = fp8.rotate(np.eye(d), s)
    assert np.abs(m @ m.T - np.eye(d)).max() < 1e-13
    q, k = r.standard_normal((50, d)), r.standard_normal((70, d))
    assert np.abs(fp8.rotate(q, s) @ fp8.rotate(k, s).T - q @ k.T).max() < 1e-11


# Two float32 fast Walsh-Hadamard transforms written here, in the test, with
# different operation orders (butterfly distance rising or falling; the
# normalisation as a product with float32(1/sqrt(d)) or as a quotient by
# float32(sqrt(d))), and two ways to form the code-unit value (x * (448/A) or
# x / (A/448)).  The oracle's bands must hold every such evaluation.

def fwht32(x, signs, rising=True, divide=False):
    v = np.asarray(x, np.float32) * np.asarray(signs, np.float32)
    d = v.shape[-1]
    hs = [1 << i for i in range(int(math.log2(d)))]
    for h in (hs if rising else hs[::-1]):
        v = v.reshape(v.shape[:-1] + (d // (2 * h), 2, h))
        a, b = v[..., 0, :].copy(), v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        v = v.reshape(v.shape[:-3] + (d,))
    if divide:
        return (v / np.float32(math.sqrt(d))).astype(np.float32)
    return (v * np.float32(1.0 / math.sqrt(d))).astype(np.float32)


def codes32(y, tile=128, per_tensor=False, quotient=False):
    """float32 block quantization of float32 values y [BH, N, d]."""
    y = np.asarray(y, np.float32)
    BH, N, d = y.shape
    nt = (N + tile - 1) // tile
    codes = np.zeros(y.shape, np.uint8)
    scales = np.ones((BH, nt), np.float32)
    whole = np.abs(y).max()
    for t in range(nt):
        blk = y[:, t * tile:(t + 1) * tile]
        amax = np.full(BH, whole, np.float32) if per_tensor else np.abs(blk).reshape(BH, -1).max(axis=1)
        sc = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        scales[:, t] = sc
        if quotient:
            tv = (blk / sc[:, None, None]).astype(np.float32)
        else:
            f = np.where(amax > 0, np.float32(448.0) / np.where(amax > 0, amax, 1), 1).astype(np.float32)
            tv = (blk * f[:, None, None]).astype(np.float32)
        codes[:, t * tile:(t + 1) * tile] = fp8.e4m3_encode(fp8.e4m3_round(tv))
    return codes, scales


@pytest.mark.parametrize("rising,divide", [(True, False), (False, True)])
def test_fwht_error_bound_holds(rising, divide):
    """Every entry of a float32 FWHT lies within fwht_f32_error_bound of the
    fp64 rotation, for either butterfly order and normalisation, on inputs
    with large outliers; the bound is not vacuous (the worst entry uses a
    visible part of it)."""
    r = np.random.default_rng(2)
    d = 128
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    x = (r.standard_normal((400, d)) * 3).astype(np.float32)
    x[r.random(x.shape) < 0.01] *= 40
    y64 = fp8.rotate(x.astype(np.float64), s)
    y32 = fwht32(x, s, rising, divide).astype(np.float64)
    tol = fp8.fwht_f32_error_bound(x)
    ratio = np.abs(y32 - y64) / tol
    assert ratio.max() <= 1.0
    assert ratio.max() > 0.02


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
            blk = x[b, 128 * t:128 * (t + 1)].astype(np.float64)
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            assert fp8.e4m3_decode(codes[b, 128 * t:128 * (t + 1)][i]) == math.copysign(448.0, blk[i])
            assert scales[b, t] == np.abs(blk).max() / 448.0


def test_quantization_error_is_half_ulp():
    """|code * scale - x| is at most half an E4M3 step of x / scale (2^-4
    relative in the normal range, 2^-10 below 2^-6), up to the fp64 rounding
    of the two products."""
    r = np.random.default_rng(5)
    x = (r.standard_normal((1, 256, 32)) * 4).astype(np.float32).astype(np.float64)
    x[0, 3, :8] = np.ldexp(1.0, -np.arange(8) - 4) * x[0, 3, :8]   # tiny values: subnormal codes
    codes, scales = fp8.quantize_tiles(x)
    sc = np.repeat(scales, 128, axis=1)[:, :, None]
    y = x / sc
    bound = np.maximum(2.0 ** -4 * np.abs(y), 2.0 ** -10)   # in code units
    err = np.abs(fp8.dequantize_tiles(codes, scales) - x) / sc
    assert np.all(err <= bound * (1 + 1e-12))
    # exactly half a grid step at most, and some values sit almost that far
    half_step = fp8.e4m3_step(y) / 2
    assert np.all(err <= half_step * (1 + 1e-12))
    assert (err / half_step).max() > 0.99


def test_tiles_are_independent_and_per_tensor_is_global():
    r = np.random.default_rng(6)
    x = r.standard_normal((1, 256, 8)).astype(np.float32)
    y = x.copy()
    y[0, 5, 3] = 1000.0                          # an outlier in tile 0 only
    cx, sx = fp8.quantize_tiles(x)
    cy, sy = fp8.quantize_tiles(y)
    assert np.array_equal(cx[:, 128:], cy[:, 128:]) and sx[0, 1] == sy[0, 1]
    assert sy[0, 0] == 1000.0 / 448.0
    ct, st = fp8.quantize_tiles(y, per_tensor=True)
    assert np.all(st == 1000.0 / 448.0)
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
        assert np.all(quant[n]["scales"] == 1.0)
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
    sv = quant["v"]["scales"].astype(np.float64)
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
# the float32 bands of the codes and scales
# ---------------------------------------------------------------------------

def band_inputs(seed, BH=2, N=300, d=128):
    """Random rows with outliers and a row of tiny values, plus, in every
    128-row tile, 40 rows whose ROTATED values sit on E4M3 rounding midpoints
    (with the tile's amax held at 448 so that code units are values): drawn
    as midpoints, rotated back, rounded to float32.  Those rows' exact targets
    lie within about one float32 rounding of a midpoint, so the code depends
    on the float32 rotation's own error."""
    r = np.random.default_rng(seed)
    x = (r.standard_normal((BH, N, d)) * 2).astype(np.float32)
    x[r.random(x.shape) < 0.002] *= 30                       # outliers
    x[:, 5, :] *= np.float32(2.0 ** -12)                     # a row of tiny values (subnormal codes)
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    grid = fp8.e4m3_decode(np.arange(0x38, 0x7E, dtype=np.uint8))   # 1 .. 416
    mids = (grid[:-1] + grid[1:]) / 2
    for t0 in range(0, N, 128):
        rows = min(40, N - t0 - 10)
        if rows <= 0:
            continue
        y = r.choice(mids, (BH, rows, d)) * np.where(r.random((BH, rows, d)) < 0.5, -1, 1)
        y[:, 0, 0] = 448.0                                    # holds the amax at 448 (exactly)
        m = fp8.rotate(np.eye(d), s)                          # rows of M
        x[:, t0 + 10:t0 + 10 + rows, :] = (y @ m.T).astype(np.float32)
    return x, s


@pytest.mark.parametrize("rising,divide,quotient,per_tensor", [
    (True, False, False, False), (False, True, True, False), (True, True, False, True),
    (False, False, True, True)])
def test_float32_quantizers_fall_within_the_bands(rising, divide, quotient, per_tensor):
    """Four float32 quantizers with different operation orders (written in this
    test): every code within codes_within_band, every scale within
    scales_within_tolerance; some codes need the band (they differ from the
    exact rounding), so the band is doing work."""
    x, s = band_inputs(10 + rising + 2 * divide)
    ref = fp8.quantize_reference(x, s, True, per_tensor=per_tensor)
    c32, s32 = codes32(fwht32(x, s, rising, divide), per_tensor=per_tensor, quotient=quotient)
    ok, n_band, n_bad = fp8.codes_within_band(c32, ref)
    assert ok, f"{n_bad} codes outside the band"
    differ = fp8.e4m3_decode(c32) != fp8.e4m3_round(ref["target"])
    assert differ.sum() > 0 and n_band >= differ.sum()
    ok_s, worst = fp8.scales_within_tolerance(s32, ref)
    assert ok_s, f"scale error {worst:.2f} x the tolerance"
    # without the rotation the band is a few float32 roundings of |t| wide
    ref_v = fp8.quantize_reference(x, None, False, per_tensor=per_tensor)
    cv, sv = codes32(x, per_tensor=per_tensor, quotient=quotient)
    assert fp8.codes_within_band(cv, ref_v)[0]
    assert fp8.scales_within_tolerance(sv, ref_v)[0]


def test_band_rejects_a_code_one_step_off():
    """A code one E4M3 step from the exact rounding where the band does not
    straddle a boundary is rejected; so is a scale off by more than its
    tolerance."""
    x, s = band_inputs(20)
    ref = fp8.quantize_reference(x, s, True)
    t, b = ref["target"], ref["band"]
    clear = (fp8.e4m3_round(t - b) == fp8.e4m3_round(t + b)) & (np.abs(t) > 1) & (np.abs(t) < 400)
    idx = np.argwhere(clear)[7]
    bad = ref["codes"].copy()
    bad[tuple(idx)] += 1                                      # next code up in magnitude
    assert fp8.codes_within_band(ref["codes"], ref)[0]
    ok, _, n_bad = fp8.codes_within_band(bad, ref)
    assert not ok and n_bad == 1
    sc = ref["scales"].copy()
    sc[0, 0] += 3 * ref["scale_tol"][0, 0]
    assert not fp8.scales_within_tolerance(sc, ref)[0]


def test_band_accepts_both_neighbours_at_a_tie():
    """A value whose code-unit target is exactly a rounding midpoint (1.0625,
    between 1 and 1.125): with a non-zero band both neighbours are accepted;
    everywhere else only the exact rounding."""
    x = np.zeros((1, 128, 4))
    x[0, 0, 0] = 448.0                                         # amax = 448: code units = values
    x[0, 1, 0] = 1.0625
    x[0, 2, 0] = 1.03
    ref = fp8.quantize_reference(x, None, False)
    assert ref["target"][0, 1, 0] == 1.0625 and ref["band"][0, 1, 0] > 0
    for v in (1.0, 1.125):
        c = ref["codes"].copy()
        c[0, 1, 0] = fp8.e4m3_encode(np.array([v]))[0]
        assert fp8.codes_within_band(c, ref)[0]
    c = ref["codes"].copy()
    c[0, 2, 0] = fp8.e4m3_encode(np.array([1.125]))[0]        # 1.03 rounds to 1 only
    assert not fp8.codes_within_band(c, ref)[0]


def test_band_slack_covers_neighbour_codes():
    """Flipping every straddling code of Q, K and V to its other neighbour
    changes attention on the codes by no more than band_slack."""
    r = np.random.default_rng(30)
    BH, N, d = 1, 200, 128
    q, k, v = ((r.standard_normal((BH, N, d)) * 2).astype(np.float32) for _ in range(3))
    for t in (q, k):
        t[r.random(t.shape) < 0.003] *= 30
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    quant = fp8.quantize_qkv(q, k, v, s)
    flipped = {}
    n_flip = 0
    for n in "qkv":
        ref = quant[n]
        t, b = ref["target"], ref["band"]
        lo, hi = fp8.e4m3_round(t - b), fp8.e4m3_round(t + b)
        exact = fp8.e4m3_round(t)
        other = np.where(exact == lo, hi, lo)
        amb = lo != hi
        n_flip += int(amb.sum())
        flipped[n] = dict(ref, codes=np.where(amb, fp8.e4m3_encode(other), ref["codes"]).astype(np.uint8))
    assert n_flip > 0
    o0, l0 = fp8.attention_on_codes(quant, 0.09, True)
    o1, l1 = fp8.attention_on_codes(flipped, 0.09, True)
    slack = fp8.band_slack(quant, 0.09, True)
    assert np.all(np.abs(o1 - o0) <= slack * (1 + 1e-9) + 1e-15)
    assert (np.abs(o1 - o0)).max() > 0
    # and lse moves by no more than the largest score change of its row
    ds = fp8.band_score_slack(quant, 0.09, True)
    assert np.all(np.abs(l1 - l0) <= ds * (1 + 1e-9) + 1e-15)
    assert (np.abs(l1 - l0)).max() > 0


def test_budget_of_exact_codes_is_met_by_exact_codes():
    """The error budget against exact attention, fed the method's own ideal
    error, holds for attention on the exactly rounded codes (by a factor of
    two) and fails for codes of a coarser format (one mantissa bit fewer)."""
    r = np.random.default_rng(31)
    BH, N, d = 2, 256, 128
    q, k, v = ((r.standard_normal((BH, N, d))).astype(np.float32) for _ in range(3))
    s = np.where(r.random(d) < 0.5, -1.0, 1.0)
    o_ex, _ = oracle.fwd(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                         d ** -0.5, True)
    quant = fp8.quantize_qkv(q, k, v, s)
    ideal = fp8.ideal_fp8_error(o_ex, quant, d ** -0.5, True)
    rmse_b, max_b = fp8.fp8_budget(o_ex, ideal)
    o_c, _ = fp8.attention_on_codes(quant, d ** -0.5, True)
    err = np.abs(o_c - o_ex)
    assert np.sqrt((err ** 2).mean()) <= rmse_b / 2 + 1e-15 and np.all(err <= max_b)
    # codes with two mantissa bits: the same inputs miss the budget
    coarse = {}
    for n in "qkv":
        vals = fp8.e4m3_decode(quant[n]["codes"])
        step = fp8.e4m3_step(vals) * 2
        coarse[n] = dict(quant[n], codes=fp8.e4m3_encode(np.clip(np.round(vals / step) * step, -448, 448)))
    o_2, _ = fp8.attention_on_codes(coarse, d ** -0.5, True)
    assert np.sqrt(((o_2 - o_ex) ** 2).mean()) > rmse_b


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


def test_planted_narrow_band_is_caught(monkeypatch):
    """A band without the rotation's error term (a plausible slip in the error
    analysis: only the roundings of the code-unit product counted) leaves
    float32 codes outside it: the float32 quantizer pin catches it."""
    monkeypatch.setattr(fp8, "fwht_f32_error_bound", lambda x: np.zeros(x.shape[:-1] + (1,)))
    with pytest.raises(AssertionError):
        test_float32_quantizers_fall_within_the_bands(True, False, False, False)
