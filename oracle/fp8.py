"""FP8 attention references -- TEST INFRASTRUCTURE ONLY (tests and bench's
reference leg load this module; the library never does).

What the FP8 forward computes, restated from "FlashAttention 1–4: How
IO-Awareness Reshaped the Attention Kernel" §"FlashAttention-3", paragraph
"FP8 with block quantization and incoherent processing":

* block quantization: one FP8 scale per tile instead of one per tensor;
* incoherent processing: Q and K are multiplied by the same random orthogonal
  matrix M before quantizing, so (QM)(KM)^T = QK^T; M is a Hadamard transform
  with random sign flips, O(d log d) per row.

Definitions here (fp64 unless stated):

* ``hadamard(d)``: the Sylvester matrix, H[i, j] = (-1)^popcount(i & j).
* ``rotate(x, signs)``: (x * signs) @ H / sqrt(d), the orthogonal M = diag(s) H / sqrt(d).
* ``e4m3_round(x)``: round-to-nearest-even onto the E4M3 grid (1 sign bit,
  4 exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite
  448, subnormals in steps of 2^-9), values beyond 448 saturate to 448.
* ``quantize_tiles``: per 128-row tile, scale = amax / 448 and codes =
  e4m3_round(x * (448 / amax)); dequantized value = code * scale.  (The page
  fixes one scale per tile; how a value becomes a code it leaves open: the
  reading here maps the tile's amax onto E4M3's largest value 448.)

``attention_on_codes`` is the attention the FP8 path approximates: the exact
definition (``oracle.fwd``, fp64) applied to the dequantized codes.  The kernel
also rounds the probabilities P to E4M3 before the P V product (the page says
the path runs in FP8 but not how P is scaled); ``p_rounding_bound`` gives, per
output element, the largest change that rounding can make under the reading
the library documents (P * fold_j * 16 rounded to nearest E4M3, fp32 row sums,
the largest weight of every tile corrected in the row sum), and is the parity
tolerance of the GPU tests.

``rotate_f32`` restates the rotation as the butterfly network the kernel runs,
in float32 with the same operation order, so that the kernel's FP8 codes can
be compared bit for bit (both sides take the rounding decision in fp32).  It is
pinned against ``rotate`` (fp64) and against ``scipy.linalg.hadamard`` by the
tests.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


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


def rotate_f32(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """The same rotation as the kernel's float32 butterflies: element j of a
    row is multiplied by s_j, then for h = 1, 2, 4, .., d/2 every pair
    (a, b) = (v[i], v[i + h]) with i & h == 0 becomes (a + b, a - b), and the
    result is multiplied by float32(1 / sqrt(d))."""
    v = np.asarray(x, np.float32) * np.asarray(signs, np.float32)
    d = v.shape[-1]
    h = 1
    while h < d:
        v = v.reshape(v.shape[:-1] + (d // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        v = v.reshape(v.shape[:-3] + (d,))
        h *= 2
    return v * np.float32(1.0 / math.sqrt(d))


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.where(nz, np.floor(np.log2(np.where(nz, a, 1.0))), 0.0)
    e = np.clip(e, -6, 8)                 # below 2^-6: the subnormal step 2^-9
    step = np.exp2(e - 3)
    q = np.round(a / step) * step         # numpy rounds halves to even
    out = np.where(nz, np.minimum(q, E4M3_MAX), 0.0)
    return np.copysign(out, x)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E4M3 byte (0x7f / 0xff, the NaN codes, are not produced)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = c & 0x7
    val = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(ex - 7.0))
    return sign * val


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """E4M3 byte of each value (must already lie on the grid, |x| <= 448)."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0)
    code = np.zeros(a.shape, np.int64)
    sub = a < 2.0 ** -6
    code = np.where(sub, np.round(a / 2.0 ** -9).astype(np.int64), code)
    e = np.floor(np.log2(np.where(sub, 1.0, a))).astype(np.int64)
    man = np.round((np.where(sub, 1.0, a) / np.exp2(e) - 1.0) * 8).astype(np.int64)
    code = np.where(sub, code, ((e + 7) << 3) | man)
    return (code | sign).astype(np.uint8)


def _scale_of(amax):
    """fp32 scale amax / 448, or 1 where amax is 0."""
    amax = np.asarray(amax, np.float32)
    return np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)


def _factor_of(amax):
    """fp32 factor 448 / amax that maps the tile onto E4M3's range, 1 where amax is 0."""
    amax = np.asarray(amax, np.float32)
    safe = np.where(amax > 0, amax, np.float32(1.0)).astype(np.float32)
    return np.where(amax > 0, np.float32(E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)


def quantize_tiles(x: np.ndarray, tile: int = 128, per_tensor: bool = False):
    """Per-tile scale and E4M3 codes of x [BH, N, d] in float32 arithmetic:
    amax over the tile's rows (rows past N count as 0), scale = amax / 448 and
    code = e4m3(x * (448 / amax)) (scale and factor 1 when the tile is all
    zero), so that code * scale ~ x.  per_tensor: amax over the whole tensor
    instead, the same scale for every tile.
    Returns (codes uint8 [BH, N, d], scales float32 [BH, ceil(N/tile)])."""
    x = np.asarray(x, np.float32)
    BH, N, d = x.shape
    nt = (N + tile - 1) // tile
    scales = np.ones((BH, nt), np.float32)
    codes = np.zeros((BH, N, d), np.uint8)
    whole = np.abs(x).max() if per_tensor else None
    for t in range(nt):
        blk = x[:, t * tile:(t + 1) * tile, :]
        if per_tensor:
            amax = np.full(BH, whole, np.float32)
        else:
            amax = np.abs(blk).reshape(BH, -1).max(axis=1).astype(np.float32)
        scales[:, t] = _scale_of(amax)
        y = (blk * _factor_of(amax)[:, None, None]).astype(np.float32)
        codes[:, t * tile:(t + 1) * tile, :] = e4m3_encode(e4m3_round(y))
    return codes, scales


def dequantize_tiles(codes: np.ndarray, scales: np.ndarray, tile: int = 128) -> np.ndarray:
    """codes * scale of their tile, fp64 [BH, N, d]."""
    v = e4m3_decode(codes)
    BH, N, d = v.shape
    sc = np.repeat(np.asarray(scales, np.float64), tile, axis=1)[:, :N]
    return v * sc[:, :, None]


def quantize_qkv(q, k, v, signs=None, rotate: bool = True, per_tensor: bool = False,
                 tile: int = 128):
    """The quantization step for attention inputs [BH, N, d] (float32-exact
    inputs such as bf16): Q and K rows rotated by diag(signs) H / sqrt(d)
    (float32 butterflies) when ``rotate``, V never; then ``quantize_tiles``.
    Returns {name: (codes, scales)} for q, k, v."""
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    if rotate:
        q = rotate_f32(q, signs)
        k = rotate_f32(k, signs)
    return {"q": quantize_tiles(q, tile, per_tensor),
            "k": quantize_tiles(k, tile, per_tensor),
            "v": quantize_tiles(v, tile, per_tensor)}


def dequantized_qkv(quant, tile: int = 128):
    """fp64 values code * scale of the three quantized tensors."""
    return tuple(dequantize_tiles(*quant[n], tile=tile) for n in ("q", "k", "v"))


def attention_on_codes(quant, scale: float, causal: bool, tile: int = 128):
    """Exact attention (fp64, by definition) on the dequantized Q, K, V.
    Returns (o [BH, N, d], lse [BH, N])."""
    from . import fwd
    qd, kd, vd = dequantized_qkv(quant, tile)
    return fwd(np.ascontiguousarray(qd), np.ascontiguousarray(kd), np.ascontiguousarray(vd),
               scale, causal)


# E4M3 rounding of a probability y = P * c: |e4m3(y) - y| <= max(2^-4 y, 2^-10)
# (half an ulp: 2^-4 relative in the normal range, half the subnormal step 2^-9
# below 2^-6).
_HALF_ULP_REL = 2.0 ** -4
_HALF_SUB_STEP = 2.0 ** -10
P_SCALE = 16.0


def p_rounding_bound(quant, scale: float, causal: bool, tile: int = 128, rows=None):
    """Per output element, the largest |O_fp8 - O_codes| that rounding P to
    E4M3 can cause, O_codes = ``attention_on_codes``.

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
    sv = quant["v"][1].astype(np.float64)
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
