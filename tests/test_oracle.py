"""Pins for the fp64 CPU oracle (no GPU).

Each pin checks the oracle against something other than itself: values printed
on the pages (``tests/golden``), closed forms, invariants of softmax attention,
library routines on special cases, brute force on tiny inputs and finite
differences.  The planted-mistake tests at the end compile edited copies of the
oracle and show that each plausible slip is caught by at least one pin.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import oracle as orc_mod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TIGHT = 1e-12


# ---------------------------------------------------------------------------
# golden fixture parsing
# ---------------------------------------------------------------------------

def _value(tok):
    """'ln3' -> log 3, '17/6' -> 17/6, '1.37' -> 1.37."""
    if tok.startswith("ln"):
        return math.log(float(tok[2:]))
    if "/" in tok:
        a, b = tok.split("/")
        return float(a) / float(b)
    return float(tok)


def load_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            out[key.strip()] = [_value(t) for t in rest.split()]
    return out


def _attn_inputs_from_scores(scores, values, q_scale=1.0):
    """d = 1 inputs whose scores are exactly the given numbers: Q = q_scale,
    K_j = s_j (so q k_j * (1/q_scale) = s_j), one identical query per key."""
    n = len(scores)
    q = np.full((1, n, 1), q_scale, dtype=np.float64)
    k = np.asarray(scores, dtype=np.float64).reshape(1, n, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, n, -1)
    return q, k, v


def _rng_inputs(seed, BH=2, N=9, d=4, scale_k=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((BH, N, d))
    k = r.standard_normal((BH, N, d)) * scale_k
    v = r.standard_normal((BH, N, d))
    return q, k, v


# ---------------------------------------------------------------------------
# pins (each raises AssertionError when the oracle disagrees)
# ---------------------------------------------------------------------------

def pin_three_score_online():
    g = load_golden("online_softmax_3score.txt")
    s, v = g["scores"], g["values"]
    # first block of two scores
    m1, l1, u1 = oracle.online_row(s[:2], v[:2], block=2)
    assert abs(m1 - g["block1_m"][0]) < TIGHT
    assert abs(l1 - g["block1_l"][0]) < TIGHT
    assert abs(u1[0] - g["block1_u"][0]) < TIGHT
    assert abs(math.exp(m1 - g["block2_m"][0]) - g["block2_factor"][0]) < TIGHT
    # the whole row split 2 + 1, and every other split, give the same state
    for block in (1, 2, 3):
        m, l, u = oracle.online_row(s, v, block=block)
        assert abs(m - g["block2_m"][0]) < TIGHT
        assert abs(l - g["block2_l"][0]) < TIGHT
        assert abs(u[0] - g["block2_u"][0]) < TIGHT
        assert abs(u[0] / l - g["output"][0]) < TIGHT


def pin_three_score_attention():
    """The same example through the attention entry points (d = 1 inputs, scale 1
    and scale 1/2 with Q doubled), and the softmax row itself via V = identity."""
    g = load_golden("online_softmax_3score.txt")
    s, vals = g["scores"], g["values"]
    for qs, scale in ((1.0, 1.0), (2.0, 0.5)):
        q, k, v = _attn_inputs_from_scores(s, vals, q_scale=qs)
        o, lse = oracle.fwd(q, k, v, scale, False)
        assert np.all(np.abs(o[0, :, 0] - g["output"][0]) < TIGHT)
        assert np.all(np.abs(lse[0] - math.log(6.0)) < TIGHT)
        ob, lb = oracle.fwd_blockwise(q, k, v, scale, False, 1, 2)
        assert np.all(np.abs(ob[0, :, 0] - g["output"][0]) < TIGHT)
        assert np.all(np.abs(lb[0] - math.log(6.0)) < TIGHT)
    # V = I_3 makes O the probability row
    q = np.zeros((1, 3, 3)); q[0, :, 0] = 1.0
    k = np.zeros((1, 3, 3)); k[0, :, 0] = s
    v = np.eye(3).reshape(1, 3, 3)
    o, _ = oracle.fwd(q, k, v, 1.0, False)
    assert np.all(np.abs(o[0] - np.asarray(g["softmax"])[None, :]) < TIGHT)


def pin_six_score_online():
    g = load_golden("online_softmax_6score.txt")
    s = g["scores"]
    b = int(g["block"][0])
    dec = int(g["decimals"][0])
    for nb, (m_ref, l_ref) in enumerate(zip(g["m_after_block"], g["l_after_block"]), start=1):
        m, l, _ = oracle.online_row(s[: nb * b], None, block=b)
        assert abs(m - m_ref) < TIGHT
        assert round(l, dec) == pytest.approx(l_ref, abs=1e-9)
    # closed form of the final sum and the printed rescale factor
    m, l, _ = oracle.online_row(s, None, block=b)
    exact = 1 + math.exp(-1) + math.exp(-2) + 2 * math.exp(-3) + math.exp(-4)
    assert abs(l - exact) < TIGHT
    assert round(math.exp(2 - 4), dec) == g["rescale_factor_block2"][0]


def pin_large_dynamic_range():
    """10,000 N(0,1)*30 scores in blocks of 128 against scipy's logsumexp and
    softmax (the self-check of "CS336 Lecture 5 notes" §11.3)."""
    x = np.random.default_rng(11).standard_normal(10000) * 30
    m, l, _ = oracle.online_row(x, None, block=128)
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-9
    assert np.max(np.abs(np.exp(x - m) / l - scipy.special.softmax(x))) < 1e-12


def pin_probability_rows():
    """V = identity turns O into P: every row is a probability vector and equals
    scipy's softmax of the scores; lse equals scipy's logsumexp."""
    N = 7
    q, k, _ = _rng_inputs(3, BH=2, N=N, d=N, scale_k=2.0)
    v = np.tile(np.eye(N), (2, 1, 1))
    scale = 0.7
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, scale, causal)
        assert np.all(o >= 0)
        assert np.max(np.abs(o.sum(-1) - 1.0)) < TIGHT
        for bh in range(2):
            for i in range(N):
                nk = i + 1 if causal else N
                s = np.array([scale * np.dot(q[bh, i], k[bh, j]) for j in range(nk)])
                assert np.max(np.abs(o[bh, i, :nk] - scipy.special.softmax(s))) < TIGHT
                assert np.all(o[bh, i, nk:] == 0.0)
                assert abs(lse[bh, i] - scipy.special.logsumexp(s)) < 1e-10


def pin_two_keys_logistic():
    """Two keys: P = (sigmoid(a - b), sigmoid(b - a)), a closed form."""
    q = np.array([[[1.0, 0.0]]]).repeat(2, axis=1)
    a, b = 0.3, -1.1
    k = np.array([[[a, 0.0], [b, 0.0]]])
    v = np.array([[[2.0, -1.0], [5.0, 3.0]]])
    o, lse = oracle.fwd(q, k, v, 1.0, False)
    p0 = 1.0 / (1.0 + math.exp(b - a))
    expect = p0 * v[0, 0] + (1 - p0) * v[0, 1]
    assert np.max(np.abs(o[0, 0] - expect)) < TIGHT
    assert abs(lse[0, 0] - (a + math.log1p(math.exp(b - a)))) < TIGHT
    o, lse = oracle.fwd(q, k, v, 1.0, True)
    assert np.all(o[0, 0] == v[0, 0])  # causal row 0 sees only key 0
    assert np.max(np.abs(o[0, 1] - expect)) < TIGHT


def pin_causal_row0_and_zero_keys():
    q, k, v = _rng_inputs(5, BH=3, N=11, d=6)
    o, lse = oracle.fwd(q, k, v, 0.4, True)
    assert np.array_equal(o[:, 0, :], v[:, 0, :])  # exactly V[0]
    assert np.max(np.abs(lse[:, 0] - 0.4 * np.einsum("bc,bc->b", q[:, 0], k[:, 0]))) < TIGHT
    kz = np.zeros_like(k)
    o, lse = oracle.fwd(q, kz, v, 0.4, False)
    assert np.max(np.abs(o - v.mean(axis=1, keepdims=True))) < TIGHT
    assert np.max(np.abs(lse - math.log(11))) < TIGHT
    o, lse = oracle.fwd(q, kz, v, 0.4, True)
    for i in range(11):
        assert np.max(np.abs(o[:, i] - v[:, : i + 1].mean(axis=1))) < TIGHT
        assert np.max(np.abs(lse[:, i] - math.log(i + 1))) < TIGHT


def pin_shift_and_affine_invariance():
    """Adding one vector u to every key shifts row i's scores by scale q_i.u, so O
    is unchanged and lse moves by that amount; V -> a V + w gives O -> a O + w."""
    q, k, v = _rng_inputs(7, BH=2, N=10, d=5)
    scale = 0.45
    u = np.array([0.5, -1.0, 2.0, 0.25, -0.75])
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, scale, causal)
        o2, lse2 = oracle.fwd(q, k + u, v, scale, causal)
        assert np.max(np.abs(o2 - o)) < 1e-11
        assert np.max(np.abs(lse2 - (lse + scale * q @ u))) < 1e-11
        w = np.array([1.0, -2.0, 0.5, 3.0, -0.25])
        o3, lse3 = oracle.fwd(q, k, 2.5 * v + w, scale, causal)
        assert np.max(np.abs(o3 - (2.5 * o + w))) < 1e-11
        assert np.max(np.abs(lse3 - lse)) < TIGHT


def pin_permutations():
    """Non-causal: permuting keys together with values leaves O unchanged;
    permuting queries permutes the output rows."""
    q, k, v = _rng_inputs(9, BH=1, N=8, d=3)
    o, lse = oracle.fwd(q, k, v, 0.8, False)
    perm = np.random.default_rng(1).permutation(8)
    o2, lse2 = oracle.fwd(q, k[:, perm], v[:, perm], 0.8, False)
    assert np.max(np.abs(o2 - o)) < TIGHT and np.max(np.abs(lse2 - lse)) < TIGHT
    o3, lse3 = oracle.fwd(q[:, perm], k, v, 0.8, False)
    assert np.max(np.abs(o3 - o[:, perm])) < TIGHT


def pin_blockwise_equals_full():
    """Brute force: the tiled online recurrence equals the one-shot row for
    every block size, with and without the causal mask."""
    q, k, v = _rng_inputs(13, BH=2, N=13, d=5, scale_k=3.0)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, 0.6, causal)
        for bq, bk in ((1, 1), (2, 3), (4, 5), (13, 13), (16, 2), (3, 16)):
            ob, lb = oracle.fwd_blockwise(q, k, v, 0.6, causal, bq, bk)
            assert np.max(np.abs(ob - o)) < 1e-12
            assert np.max(np.abs(lb - lse)) < 1e-12


def _fd_grads(q, k, v, do, scale, causal, h=1e-6):
    """Central differences of f = sum(dO * O) with respect to Q, K and V."""
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [t.copy() for t in base]
            minus = [t.copy() for t in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fp = np.sum(do * oracle.fwd(*plus, scale, causal)[0])
            fm = np.sum(do * oracle.fwd(*minus, scale, causal)[0])
            g[idx] = (fp - fm) / (2 * h)
        grads.append(g)
    return grads


def pin_backward_finite_differences():
    q, k, v = _rng_inputs(17, BH=1, N=5, d=3, scale_k=1.5)
    do = np.random.default_rng(18).standard_normal(q.shape)
    scale = 0.9
    for causal in (False, True):
        dq, dk, dv, _, _ = oracle.bwd(q, k, v, do, scale, causal)
        fq, fk, fv = _fd_grads(q, k, v, do, scale, causal)
        for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
            assert np.max(np.abs(got - ref)) < 1e-7 * max(1.0, np.max(np.abs(ref)))


def pin_backward_invariants():
    """sum_j dS_ij = 0 makes sum_j dK_j = 0; rows of P summing to 1 make
    sum_j dV_j = sum_i dO_i."""
    q, k, v = _rng_inputs(21, BH=3, N=12, d=4)
    do = np.random.default_rng(22).standard_normal(q.shape)
    for causal in (False, True):
        dq, dk, dv, o, lse = oracle.bwd(q, k, v, do, 0.5, causal)
        assert np.max(np.abs(dk.sum(axis=1))) < 1e-12
        assert np.max(np.abs(dv.sum(axis=1) - do.sum(axis=1))) < 1e-12
        of, lf = oracle.fwd(q, k, v, 0.5, causal)
        assert np.max(np.abs(o - of)) < TIGHT and np.max(np.abs(lse - lf)) < TIGHT


def pin_backward_rows_finite_differences():
    """The sampled-row backward against central differences of sum(dO * O):
    dQ of selected query rows, dK and dV of selected key rows (two heads, so a
    statistic left over from the previous head would show)."""
    q, k, v = _rng_inputs(19, BH=2, N=7, d=3, scale_k=1.5)
    do = np.random.default_rng(20).standard_normal(q.shape)
    scale = 0.8
    qrows = np.array([[6, 0, 3], [2, 5, 1]], dtype=np.int64)
    krows = np.array([[4, 1], [0, 6]], dtype=np.int64)
    for causal in (False, True):
        dq, dk, dv = oracle.bwd_rows(q, k, v, do, scale, causal, qrows=qrows, krows=krows)
        for bh in range(2):
            fq, fk, fv = _fd_grads(q[bh:bh + 1], k[bh:bh + 1], v[bh:bh + 1], do[bh:bh + 1],
                                   scale, causal)
            tol = 1e-7 * max(1.0, np.max(np.abs(fq)), np.max(np.abs(fk)), np.max(np.abs(fv)))
            assert np.max(np.abs(dq[bh] - fq[0][qrows[bh]])) < tol
            assert np.max(np.abs(dk[bh] - fk[0][krows[bh]])) < tol
            assert np.max(np.abs(dv[bh] - fv[0][krows[bh]])) < tol


def pin_backward_rows_equal_whole():
    """The sampled-row backward gives the whole-head backward's values for the
    same rows, bit for bit (the same row and column passes), with only query
    rows, only key rows, or both asked for."""
    q, k, v = _rng_inputs(23, BH=3, N=19, d=4, scale_k=2.0)
    do = np.random.default_rng(24).standard_normal(q.shape)
    rng = np.random.default_rng(25)
    qrows = np.stack([rng.choice(19, 5, replace=False) for _ in range(3)])
    krows = np.stack([rng.choice(19, 4, replace=False) for _ in range(3)])
    for causal in (False, True):
        dq, dk, dv, _, _ = oracle.bwd(q, k, v, do, 0.6, causal)
        rq, rk, rv = oracle.bwd_rows(q, k, v, do, 0.6, causal, qrows=qrows, krows=krows)
        oq, _, _ = oracle.bwd_rows(q, k, v, do, 0.6, causal, qrows=qrows)
        _, ok, ov = oracle.bwd_rows(q, k, v, do, 0.6, causal, krows=krows)
        for bh in range(3):
            assert np.array_equal(rq[bh], dq[bh][qrows[bh]]) and np.array_equal(oq, rq)
            assert np.array_equal(rk[bh], dk[bh][krows[bh]]) and np.array_equal(ok, rk)
            assert np.array_equal(rv[bh], dv[bh][krows[bh]]) and np.array_equal(ov, rv)


PINS = [
    pin_three_score_online, pin_three_score_attention, pin_six_score_online,
    pin_large_dynamic_range, pin_probability_rows, pin_two_keys_logistic,
    pin_causal_row0_and_zero_keys, pin_shift_and_affine_invariance, pin_permutations,
    pin_blockwise_equals_full, pin_backward_finite_differences, pin_backward_invariants,
    pin_backward_rows_finite_differences, pin_backward_rows_equal_whole,
]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# further checks of the oracle's plumbing
# ---------------------------------------------------------------------------

def test_backward_matches_torch_autograd():
    """Independent cross-check: torch.autograd in fp64 on CPU."""
    torch = pytest.importorskip("torch")
    q, k, v = _rng_inputs(31, BH=2, N=10, d=4)
    do = np.random.default_rng(32).standard_normal(q.shape)
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        s = 0.7 * tq @ tk.transpose(-1, -2)
        if causal:
            mask = torch.triu(torch.ones(10, 10, dtype=torch.bool), diagonal=1)
            s = s.masked_fill(mask, float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv
        o.backward(torch.tensor(do))
        dq, dk, dv, _, _ = oracle.bwd(q, k, v, do, 0.7, causal)
        assert np.max(np.abs(dq - tq.grad.numpy())) < 1e-12
        assert np.max(np.abs(dk - tk.grad.numpy())) < 1e-12
        assert np.max(np.abs(dv - tv.grad.numpy())) < 1e-12


def test_bf16_inputs_widen_exactly():
    torch = pytest.importorskip("torch")
    from exact_tiled_attention_05_gb300 import workloads
    t = workloads.random_bf16((1, 2, 16, 8), seed=5, scale=3.0)
    bits = workloads.bf16_bits(t)
    f64 = t.to(torch.float64).reshape(2, 16, 8).numpy()
    o1, l1 = oracle.fwd(bits, bits, bits, 0.3, True)
    o2, l2 = oracle.fwd(f64, f64, f64, 0.3, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_rows_and_heads_selection():
    q, k, v = _rng_inputs(41, BH=3, N=20, d=5)
    o, lse = oracle.fwd(q, k, v, 0.5, True)
    rows = np.array([[0, 5, 19], [1, 2, 3], [19, 18, 0]], dtype=np.int64)
    orows, lrows = oracle.fwd_rows(q, k, v, 0.5, True, rows)
    for bh in range(3):
        assert np.array_equal(orows[bh], o[bh, rows[bh]])
        assert np.array_equal(lrows[bh], lse[bh, rows[bh]])
    oh, lh = oracle.fwd(q, k, v, 0.5, True, heads=[2, 0])
    assert np.array_equal(oh[0], o[2]) and np.array_equal(lh[1], lse[0])
    do = np.random.default_rng(3).standard_normal(q.shape)
    full = oracle.bwd(q, k, v, do, 0.5, True)
    part = oracle.bwd(q, k, v, do, 0.5, True, heads=[1])
    for a, b in zip(full, part):
        assert np.array_equal(a[1], b[0])


def test_threads_do_not_change_results():
    q, k, v = _rng_inputs(43, BH=4, N=33, d=7)
    a = oracle.fwd(q, k, v, 0.5, False, nthreads=1)
    b = oracle.fwd(q, k, v, 0.5, False, nthreads=8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_arguments_are_rejected():
    q, k, v = _rng_inputs(1, BH=1, N=4, d=2)
    with pytest.raises(RuntimeError):
        oracle.fwd_rows(q, k, v, 1.0, False, np.array([[7]]))
    with pytest.raises(RuntimeError):
        oracle.fwd(q, k, v, 1.0, False, heads=[3])
    with pytest.raises(TypeError):
        oracle.fwd(q.astype(np.float32), k, v, 1.0, False)


# ---------------------------------------------------------------------------
# planted mistakes: each edited oracle must fail at least one pin
# ---------------------------------------------------------------------------

MUTATIONS = {
    "softmax_without_max_in_lse": ("return m + log(l);", "return log(l);"),
    "unnormalised_probabilities": ("for (long j = 0; j < nk; ++j) p[j] /= l;", ""),
    "scale_dropped": ("s[j] = scale * dot(qi, h->k + j * d, d);",
                      "s[j] = dot(qi, h->k + j * d, d);"),
    "q_k_transposed": ("s[j] = scale * dot(qi, h->k + j * d, d);",
                       "s[j] = scale * dot(h->q + j * d, h->k + i * d, d);"),
    "causal_one_key_too_many": ("return causal ? i + 1 : N;", "return causal ? (i + 2 < N ? i + 2 : N) : N;"),
    "online_alpha_sign": ("double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);\n        double ref",
                          "double alpha = (m == -INFINITY) ? 0.0 : exp(m_new - m);\n        double ref"),
    "online_no_rescale_of_sum": ("        l *= alpha;\n        for (long c = 0; c < dv; ++c) u_out[c] *= alpha;",
                                 "        for (long c = 0; c < dv; ++c) u_out[c] *= alpha;"),
    "blockwise_wrong_value_row": ("const double* vj = h->v + (j0 + t) * d;",
                                  "const double* vj = h->v + (j0 + t + (t + 1 < nb)) * d;"),
    "bwd_dS_sign": ("double dS = Pij * (dP - c->D[i]);", "double dS = Pij * (dP + c->D[i]);"),
    "bwd_dq_uses_q": ("const double* kj = c->h->k + j * d;\n        for (long cc = 0; cc < d; ++cc) dqi[cc]",
                      "const double* kj = c->h->q + j * d;\n        for (long cc = 0; cc < d; ++cc) dqi[cc]"),
    "bwd_dv_uses_dS": ("dvj[cc] += Pij * doi[cc];", "dvj[cc] += dS * doi[cc];"),
    "bwd_D_from_v": ("double Di = dot(doi, orow, d);", "double Di = dot(doi, c->h->v + i * d, d);"),
    "bwd_dk_missing_scale": ("dkj[cc] += c->scale * dS * qi[cc];", "dkj[cc] += dS * qi[cc];"),
    "bwd_rows_noncausal_stats_from_first_key": ("        if (nk > 0 && !causal) first = 0;\n", ""),
    "bwd_rows_stats_one_row_late": ("for (long i = first; i < N; ++i) need[n_need++] = i;",
                                    "for (long i = first + 1; i < N; ++i) need[n_need++] = i;"),
    "bwd_rows_dq_copied_from_wrong_row": (
        "memcpy(dq_rows + (bh * nq + t) * d, c.dq + qrows[bh * nq + t] * d,",
        "memcpy(dq_rows + (bh * nq + t) * d, c.dq + qrows[bh * nq] * d,"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(orc_mod.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    lib = orc_mod.compile_variant(src.replace(old, new), str(tmp_path / f"lib_{name}.so"))
    failed = []
    with orc_mod.use_library(lib):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, RuntimeError, FloatingPointError):
                failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
