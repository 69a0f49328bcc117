"""FP8 attention references -- TEST INFRASTRUCTURE ONLY (tests and bench's
reference leg load this module; the library never does).

What the FP8 forward computes, restated from "FlashAttention 1–4: How
IO-Awareness Reshaped the Attention Kernel" §"FlashAttention-3", paragraph
"FP8 with block quantization and incoherent processing":

* block quantization: one FP8 scale per tile instead of one per tensor;
* incoherent processing: Q and K are multiplied by the same random orthogonal
  matrix M before quantizing, so (QM)(KM)^T = QK^T; M is a Hadamard transform
  with random sign flips, O(d log d) per row.

Definitions here, all in fp64 (the exact values of the method; nothing below
follows any implementation's float32 operation order):

* ``hadamard(d)``: the Sylvester matrix, H[i, j] = (-1)^popcount(i & j).
* ``rotate(x, signs)``: (x * signs) @ H / sqrt(d), the orthogonal M = diag(s) H / sqrt(d).
* ``e4m3_round(x)``: round-to-nearest-even onto the E4M3 grid (1 sign bit,
  4 exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite
  448, subnormals in steps of 2^-9), values beyond 448 saturate to 448.
* ``quantize_tiles``: per 128-row tile, A = max |x| over the tile, scale =
  A / 448 and code = e4m3_round(x * 448 / A).  (The page fixes one scale per
  tile; how a value becomes a code it leaves open: the reading here maps the
  tile's amax onto E4M3's largest value 448.)

A float32 implementation cannot reach these exact values: its rotation and its
products round.  ``quantize_reference`` therefore also returns, per element, a
band around the exact code-unit value x * 448 / A that holds every float32
evaluation of the same definition whose rotation is a fast Walsh-Hadamard
transform (log2(d) levels of a + b / a - b, then one multiplication by
float32(1 / sqrt(d)); the page's O(d log d) rotation) and whose code value is
formed with at most two more float32 roundings (a quotient or a reciprocal and
a product).  ``codes_within_band`` accepts an implementation's code when it is
the correctly rounded E4M3 of the exact value, or, only where the band
straddles an E4M3 rounding boundary, either neighbour; it counts those cases.
Scales are checked the same way (``scales_within_tolerance``).

``attention_on_codes`` is exact attention (``oracle.fwd``, fp64) on the
dequantized codes.  ``ideal_fp8_error`` is the error that exact E4M3 rounding
of the block-quantized (and rotated) inputs causes against exact attention on
the original inputs: the method's own accuracy, against which the FP8 path's
error budget is stated.  ``p_rounding_bound`` is a diagnostic: per output
element, the largest change that rounding the probabilities P to E4M3 can make
under the reading the library documents (P * fold_j * 16 rounded to nearest
E4M3, fp32 row sums, the largest weight of every tile corrected in the row
sum); ``band_slack`` bounds the further change that the band cases' one-step
code differences can make.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
U32 = 2.0 ** -24          # unit roundoff of float32 (round to nearest)


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), entries +-1."""
    assert d > 0 and d & (d - 1) == 0
    i = np.arange(d)
    pop = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pop % 2 == 0, 1.0, -1.0)


def signs_from_bits(bits: np.ndarray, d: int) -> np.ndarray:
    """+-1 vector of length d from a little-endian bit mask (uint32 words):
    bit j set means s_j = -1."""
    words = np.asarray(bits, dtype=np.uint64)
    j = np.arange(d)
    b = (words[j // 32] >> (j % 32).astype(np.uint64)) & np.uint64(1)
    return np.where(b == 1, -1.0, 1.0)


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x @ M with M = diag(signs) H / sqrt(d): orthogonal, fp64."""
    d = x.shape[-1]
    return (np.asarray(x, np.float64) * signs) @ hadamard(d) / math.sqrt(d)


def fwht_f32_error_bound(x: np.ndarray) -> np.ndarray:
    """Per row of x [..., d] (values exact in float32), a bound on
    |y32 - y| for every entry of the row, where y = rotate(x, s) and y32 is any
    float32 fast Walsh-Hadamard transform of the sign-flipped row (log2(d)
    levels of sums and differences, each rounding once) followed by one product
    with float32(1 / sqrt(d)).  Each output is a sum of the d terms +-x_j
    formed by an addition tree of depth L = log2(d), so its error is at most
    gamma_L * sum_j |x_j| (gamma_L = L u / (1 - L u)); the constant and the
    product add two more roundings: (L + 3) u sum_j |x_j| / sqrt(d) covers all
    of it (u = 2^-24).  Returns [..., 1]."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    L = int(round(math.log2(d)))
    return (L + 3) * U32 * np.abs(x).sum(axis=-1, keepdims=True) / math.sqrt(d)


def _binade(a: np.ndarray) -> np.ndarray:
    """floor(log2 a) for a > 0, exactly, as int32 (frexp: a = m 2^e with m in
    [0.5, 1)); -1 where a == 0."""
    return np.frexp(a)[1] - np.int32(1)


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.clip(_binade(a), -6, 8)        # below 2^-6: the subnormal step 2^-9
    step = np.ldexp(1.0, e - np.int32(3))
    q = np.round(a / step) * step         # numpy rounds halves to even (exact: step is a power of 2)
    return np.copysign(np.minimum(q, E4M3_MAX), x)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E4M3 byte (0x7f / 0xff, the NaN codes, are not produced)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = c & 0x7
    val = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(ex - 7.0))
    return sign * val


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """E4M3 byte of each value (must already lie on the grid, |x| <= 448):
    its magnitude in steps of 2^-9 below 2^-6 (exponent field 0), otherwise
    exponent field e + 7 and mantissa (a / 2^e - 1) * 8."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0)
    sub = a < 2.0 ** -6
    e = np.maximum(_binade(a), np.int32(-6))
    man = np.round((np.ldexp(a, -e) - 1.0) * 8).astype(np.int32)
    code = np.where(sub, np.round(a * 2.0 ** 9).astype(np.int32), ((e + 7) << 3) | man)
    return (code | sign).astype(np.uint8)


def e4m3_step(x: np.ndarray) -> np.ndarray:
    """Spacing of the E4M3 grid at |x| (the step up from |x|'s binade bottom)."""
    e = np.clip(_binade(np.abs(np.asarray(x, np.float64))), -6, 8)
    return np.ldexp(1.0, e - np.int32(3))


def _tile_amax(x: np.ndarray, tile: int, per_tensor: bool) -> np.ndarray:
    """max |x| per 128-row tile [BH, T] (the whole tensor's max in every entry
    when per_tensor)."""
    BH, N, d = x.shape
    nt = (N + tile - 1) // tile
    if per_tensor:
        return np.full((BH, nt), np.abs(x).max() if x.size else 0.0)
    amax = np.zeros((BH, nt))
    for t in range(nt):
        amax[:, t] = np.abs(x[:, t * tile:(t + 1) * tile, :]).reshape(BH, -1).max(axis=1)
    return amax


def quantize_tiles(x: np.ndarray, tile: int = 128, per_tensor: bool = False):
    """Per-tile scale and E4M3 codes of x [BH, N, d], in fp64: A = max |x| over
    the tile's rows (the whole tensor when per_tensor), scale = A / 448 and
    code = e4m3_round(x * 448 / A); scale 1 and code 0 for an all-zero tile.
    Returns (codes uint8 [BH, N, d], scales float64 [BH, ceil(N/tile)])."""
    x = np.asarray(x, np.float64)
    BH, N, d = x.shape
    amax = _tile_amax(x, tile, per_tensor)
    scales = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    rows = np.repeat(np.where(amax > 0, E4M3_MAX / np.where(amax > 0, amax, 1.0), 1.0),
                     tile, axis=1)[:, :N]
    codes = e4m3_encode(e4m3_round(x * rows[:, :, None]))
    return codes, scales


def dequantize_tiles(codes: np.ndarray, scales: np.ndarray, tile: int = 128) -> np.ndarray:
    """codes * scale of their tile, fp64 [BH, N, d]."""
    v = e4m3_decode(codes)
    BH, N, d = v.shape
    sc = np.repeat(np.asarray(scales, np.float64), tile, axis=1)[:, :N]
    return v * sc[:, :, None]


def quantize_reference(x, signs=None, rotate_rows: bool = False, tile: int = 128,
                       per_tensor: bool = False):
    """The quantization of one input tensor x [BH, N, d] (values exact in
    float32, such as bf16), exactly, plus the room a float32 evaluation has.

    y = rotate(x, signs) when rotate_rows, else x; A = tile amax of y;
    target t = y * 448 / A (code units, fp64); codes = e4m3_round(t).
    With E the per-row rotation error bound (``fwht_f32_error_bound``; 0
    without rotation) and E_A its largest value over the tile (|A32 - A| <=
    E_A for the float32 amax A32), a float32 evaluation's code-unit value lies
    within
        band = (448 E + |t| E_A) / (A - E_A) + 3 u |t|
    of t (3 u: the two roundings of 448 / A32 and the product, with room), and
    its scale A32 / 448, rounded, within
        scale_tol = (E_A + u (A + E_A)) / 448
    of A / 448.  Returns a dict with codes, scales (fp64), target, band,
    scale_tol ([BH, T])."""
    x = np.asarray(x, np.float64)
    BH, N, d = x.shape
    y = rotate(x, signs) if rotate_rows else x
    err = fwht_f32_error_bound(x) if rotate_rows else np.zeros((BH, N, 1))
    codes, scales = quantize_tiles(y, tile, per_tensor)
    amax = _tile_amax(y, tile, per_tensor)
    if per_tensor:
        e_a = np.full(amax.shape, err.max() if err.size else 0.0)
    else:
        e_a = _tile_amax(err, tile, False)
    rows = lambda a: np.repeat(a, tile, axis=1)[:, :N, None]
    A, EA = rows(amax), rows(e_a)
    safe = np.where(A > 0, A, 1.0)
    target = np.where(A > 0, y * E4M3_MAX / safe, 0.0)
    band = np.where(A > 0, (E4M3_MAX * err + np.abs(target) * EA) / np.maximum(safe - EA, 1e-300)
                    + 3 * U32 * np.abs(target), 0.0)
    scale_tol = (e_a + U32 * (amax + e_a)) / E4M3_MAX
    return {"codes": codes, "scales": scales, "target": target, "band": band,
            "scale_tol": scale_tol, "amax": amax}


def codes_within_band(got_codes: np.ndarray, ref: dict):
    """Checks an implementation's E4M3 codes [BH, N, d] against
    ``quantize_reference``: every code must decode to e4m3_round(target),
    except where target - band and target + band round to different E4M3
    values (the band straddles a rounding boundary); there either of the two
    is accepted.  Returns (ok: bool, n_band: int, n_bad: int)."""
    v = e4m3_decode(got_codes)
    t, b = ref["target"], ref["band"]
    exact = e4m3_round(t)
    lo, hi = e4m3_round(t - b), e4m3_round(t + b)
    ambiguous = lo != hi
    ok_elem = np.where(ambiguous, (v == lo) | (v == hi), v == exact)
    n_bad = int((~ok_elem).sum())
    return n_bad == 0, int(ambiguous.sum()), n_bad


def scales_within_tolerance(got_scales: np.ndarray, ref: dict):
    """|scale32 - A / 448| <= scale_tol for every tile.  Returns (ok, worst ratio)."""
    err = np.abs(np.asarray(got_scales, np.float64) - ref["scales"])
    tol = np.where(ref["amax"] > 0, ref["scale_tol"], 0.0)
    ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= tol)), float(ratio.max() if ratio.size else 0.0)


def quantize_qkv(q, k, v, signs=None, rotate: bool = True, per_tensor: bool = False,
                 tile: int = 128):
    """The quantization step for attention inputs [BH, N, d]: Q and K rows
    rotated by diag(signs) H / sqrt(d) when ``rotate``, V never; each tensor
    then quantized per tile (``quantize_reference``).  Returns {name: ref dict}
    for q, k, v; ``codes_and_scales`` gives the plain (codes, scales) pairs."""
    return {"q": quantize_reference(q, signs, rotate, tile, per_tensor),
            "k": quantize_reference(k, signs, rotate, tile, per_tensor),
            "v": quantize_reference(v, None, False, tile, per_tensor)}


def codes_and_scales(quant):
    """{name: (codes, scales)} of a ``quantize_qkv`` result."""
    return {n: (r["codes"], r["scales"]) if isinstance(r, dict) else r for n, r in quant.items()}


def dequantized_qkv(quant, tile: int = 128):
    """fp64 values code * scale of the three quantized tensors."""
    cs = codes_and_scales(quant)
    return tuple(dequantize_tiles(*cs[n], tile=tile) for n in ("q", "k", "v"))


def attention_on_codes(quant, scale: float, causal: bool, tile: int = 128):
    """Exact attention (fp64, by definition) on the dequantized Q, K, V.
    Returns (o [BH, N, d], lse [BH, N])."""
    from . import fwd
    qd, kd, vd = dequantized_qkv(quant, tile)
    return fwd(np.ascontiguousarray(qd), np.ascontiguousarray(kd), np.ascontiguousarray(vd),
               scale, causal)


def attention_on_codes_rows(quant, scale: float, causal: bool, rows, tile: int = 128):
    """``attention_on_codes`` for selected query rows [BH, R] only."""
    from . import fwd_rows
    qd, kd, vd = dequantized_qkv(quant, tile)
    return fwd_rows(np.ascontiguousarray(qd), np.ascontiguousarray(kd), np.ascontiguousarray(vd),
                    scale, causal, rows)


def ideal_fp8_error(o_exact: np.ndarray, quant, scale: float, causal: bool, tile: int = 128,
                    rows=None, lse_exact=None):
    """The method's own FP8 error: exact attention on the exactly rounded codes
    (``attention_on_codes``) against exact attention on the original inputs
    (o_exact, [BH, N, d], or [BH, R, d] for the query rows ``rows``).
    Returns (rmse, max |err|), and max |lse error| third when lse_exact
    (the exact attention's lse, [BH, N] or [BH, R]) is given."""
    if rows is None:
        o_codes, lse_codes = attention_on_codes(quant, scale, causal, tile)
    else:
        o_codes, lse_codes = attention_on_codes_rows(quant, scale, causal, rows, tile)
    err = np.abs(o_codes - o_exact)
    out = (float(np.sqrt((err ** 2).mean())), float(err.max()))
    if lse_exact is not None:
        out += (float(np.abs(lse_codes - lse_exact).max()),)
    return out


def fp8_budget(o_exact: np.ndarray, ideal):
    """The FP8 forward's accuracy budget against exact attention on the
    original inputs, from the method's own error ``ideal`` = (rmse, max) of
    exact attention on exactly rounded codes: the FP8 path also rounds the
    probabilities to E4M3 (3 mantissa bits, like V) and works in float32, so
    it may double that error; the bf16 rounding of the output comes on top.
        rmse <= 2 ideal_rmse + rms(half_ulp_bf16(O))
        max  <= 2 ideal_max  + half_ulp_bf16(O)    (element by element)
    Returns (rmse_budget, per-element max budget [same shape as o_exact])."""
    a = np.maximum(np.abs(o_exact), np.finfo(np.float32).tiny)
    half = np.ldexp(1.0, (np.floor(np.log2(a)) - 8).astype(np.int64))
    return 2.0 * ideal[0] + float(np.sqrt((half ** 2).mean())), 2.0 * ideal[1] + half


def fp8_lse_budget(ideal_lse_max: float) -> float:
    """The FP8 forward's lse budget against exact attention on the original
    inputs: its probabilities are not rounded for the row sums, so only the
    quantized scores move lse; 2 x the method's own largest lse error plus
    the 1e-3 of the bf16 path's lse gate."""
    return 2.0 * ideal_lse_max + 1e-3


# E4M3 rounding of a probability y = P * c: |e4m3(y) - y| <= max(2^-4 y, 2^-10)
# (half an ulp: 2^-4 relative in the normal range, half the subnormal step 2^-9
# below 2^-6).
_HALF_ULP_REL = 2.0 ** -4
_HALF_SUB_STEP = 2.0 ** -10
P_SCALE = 16.0


def _vscales(quant):
    r = quant["v"]
    return (r["scales"] if isinstance(r, dict) else r[1]).astype(np.float64)


def p_rounding_bound(quant, scale: float, causal: bool, tile: int = 128, rows=None):
    """Diagnostic: per output element, the largest |O_fp8 - O_codes| that
    rounding P to E4M3 can cause, O_codes = ``attention_on_codes``.

    With p_k = exp(s_k - m) (m the row max), the weight of key k in tile j is
    rounded as y = p_k * c_j with c_j = 16 * sv_j / max_t sv_t (any running max
    at or below m only shrinks the subnormal term, so m gives the bound):
        |dP_k| <= max(2^-4 p_k, 2^-10 / c_j).
    The row sum l = sum p_k is corrected by the rounding of the largest weight
    of every tile, |lc| <= LC = sum_j max(2^-4 max_j p, 2^-10 / c_j), so
        |O_fp8 - O_codes| <= (sum_k |dP_k| |v_k| + |O_codes| LC) / (l - LC).
    rows: optional int array [BH, R] of query rows to evaluate (all rows when
    None).  Returns (bound, o_codes, lse_codes), [BH, R, d], [BH, R, d], [BH, R]."""
    qd, kd, vd = dequantized_qkv(quant, tile)
    sv = _vscales(quant)
    BH, N, d = qd.shape
    c = P_SCALE * sv / sv.max(axis=1, keepdims=True)            # [BH, T]
    key_tile = np.arange(N) // tile
    if rows is None:
        rows = np.tile(np.arange(N), (BH, 1))
    rows = np.asarray(rows, np.int64)
    R = rows.shape[1]
    bound = np.empty((BH, R, d))
    o_ref = np.empty((BH, R, d))
    lse = np.empty((BH, R))
    for b in range(BH):
        s = scale * (qd[b][rows[b]] @ kd[b].T)                   # [R, N]
        if causal:
            s = np.where(np.arange(N)[None, :] <= rows[b][:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1)
        ck = c[b][key_tile]                                      # [N] per key
        dp = np.maximum(_HALF_ULP_REL * p, _HALF_SUB_STEP / ck[None, :])
        dp = np.where(p > 0, dp, 0.0)                            # masked keys carry no weight
        lc = np.zeros(R)
        for j in range(c.shape[1]):
            cols = key_tile == j
            pj = p[:, cols]
            vis = (pj > 0).any(axis=1)
            lc += np.where(vis, np.maximum(_HALF_ULP_REL * pj.max(axis=1),
                                           _HALF_SUB_STEP / c[b, j]), 0.0)
        o = (p @ vd[b]) / l[:, None]
        o_ref[b] = o
        lse[b] = m[:, 0] + np.log(l)
        bound[b] = (dp @ np.abs(vd[b]) + np.abs(o) * lc[:, None]) / (l - lc)[:, None]
    return bound, o_ref, lse


def band_score_slack(quant, scale: float, causal: bool, tile: int = 128, rows=None):
    """Per query row, the largest change of any visible score s_ij that the band
    cases' neighbouring codes can cause, max_j ds_ij (see ``band_slack``); an
    lse moves by no more than that.  Returns [BH, R]."""
    return _band_terms(quant, scale, causal, tile, rows)[0]


def _band_terms(quant, scale, causal, tile, rows):
    qd, kd, vd = dequantized_qkv(quant, tile)
    BH, N, d = qd.shape

    def steps(name):
        r = quant[name]
        t, b = r["target"], r["band"]
        amb = e4m3_round(t - b) != e4m3_round(t + b)
        sc = np.repeat(r["scales"] + r["scale_tol"], tile, axis=1)[:, :N, None]
        return np.where(amb, e4m3_step(np.abs(t) + b) * sc, 0.0)

    uq, uk, uv = steps("q"), steps("k"), steps("v")
    if rows is None:
        rows = np.tile(np.arange(N), (BH, 1))
    rows = np.asarray(rows, np.int64)
    dmax_all = np.empty((BH, rows.shape[1]))
    out = np.empty((BH, rows.shape[1], d))
    for b in range(BH):
        qa = np.abs(qd[b][rows[b]]) + uq[b][rows[b]]
        ka = np.abs(kd[b]) + uk[b]
        ds = scale * (uq[b][rows[b]] @ ka.T + qa @ uk[b].T)     # [R, N]
        s = scale * (qd[b][rows[b]] @ kd[b].T)
        vis = np.ones_like(s, dtype=bool)
        if causal:
            vis = np.arange(N)[None, :] <= rows[b][:, None]
        s = np.where(vis, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        o = p @ vd[b]
        dmax = np.where(vis, ds, 0.0).max(axis=1)                # [R]
        growth = np.exp(2 * dmax) - 1.0
        spread = np.stack([np.where(vis[i][:, None], np.abs(vd[b] - o[i][None, :]), 0.0).max(axis=0)
                           for i in range(len(rows[b]))])       # [R, d]
        dmax_all[b] = dmax
        out[b] = growth[:, None] * spread + (p @ uv[b]) * (1.0 + growth[:, None])
    return dmax_all, out


def band_slack(quant, scale: float, causal: bool, tile: int = 128, rows=None):
    """Diagnostic companion of ``p_rounding_bound``: where an element's band
    straddles a rounding boundary, an implementation may hold the neighbouring
    code, one E4M3 step (times the tile scale, widened by the scale tolerance)
    away from the exact code.  Per query row i this moves each score by at most
    ds_ij = scale (sum_c U_q[i,c] |k_jc| + |q_ic| U_k[j,c]) (U: those steps,
    0 elsewhere; |q|, |k| widened by U), so the weights change by at most a
    factor exp(+-2 max_j ds_ij), and O moves by at most
    (exp(2 max_j ds_ij) - 1) max_j |v_j - O_i| + exp(2 max_j ds_ij) sum_j P_ij U_v[j].
    Returns [BH, R, d] (all rows when rows is None)."""
    return _band_terms(quant, scale, causal, tile, rows)[1]
