"""The software exp2's cubic: the coefficients in the kernel header are the
ones the committed fitting script produces, and its error bound holds."""
import os
import re
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_05_gb300", "csrc")


def test_header_coefficients_match_the_fit():
    out = subprocess.run([sys.executable, os.path.join(CSRC, "fit_exp2_poly.py")],
                         capture_output=True, text=True, check=True).stdout
    fitted = [float(x) for x in re.findall(r"c\d = np\.float32\(([-0-9.e]+)\)", out)]
    assert len(fitted) == 4
    hdr = open(os.path.join(CSRC, "ptx.cuh")).read()
    body = hdr[hdr.index("exp2_fma_pair"):]
    used = [float(x) for x in re.findall(r"f2_pack\(([0-9.]+)f, \1f\)", body)[:4]]
    # Horner order in the header: c3, c2, c1, c0
    assert np.allclose(used, fitted[::-1], rtol=0, atol=1e-7), (used, fitted)
    err = float(re.search(r"max relative error: ([0-9.e-]+) \(fp64\)", out).group(1))
    assert err < 2e-4


def test_emulation_matches_exp2_on_the_cpu():
    """The same bit manipulation in numpy float32: 2^x within 1.2e-4 relative."""
    c = np.float32([1.0, 0.6933686, 0.24221784, 0.054592825])
    x = np.linspace(-124.9, 8.0, 100001).astype(np.float32)
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic)).astype(np.float32)
    p = c[3]
    for k in (2, 1, 0):
        p = (p * f + c[k]).astype(np.float32)
    j = t.view(np.int32) - np.int32(0x4B400000)
    r = (p.view(np.int32) + (j << 23)).view(np.float32)
    rel = np.abs(r.astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.2e-4
