"""The C ABI without a GPU: the library loads, exports every function that
include/fa.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import exact_tiled_attention_05_gb300 as fa
from exact_tiled_attention_05_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(fa_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert n in fa.EXPORTED


def test_status_strings(lib):
    for code, name in ((0, "FA_OK"), (1, "FA_ERR_INVALID_ARG"), (6, "FA_ERR_DEVICE_TIMEOUT")):
        assert fa.fa_status_string(code).decode() == name
    assert fa.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"
    assert fa.fa_version() >= 100


def test_workspace_size(lib):
    B, H, N, d = 2, 3, 100, 64
    r256 = lambda x: (x + 255) // 256 * 256
    npad = B * H * ((N + 127) // 128) * 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) == 2 * r256(npad * 4) + 256  # D, -lse*log2(e), counter
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0


def test_fp8_workspace_size_limits(lib):
    """The FP8 path takes d = 128 only, at most 65535 heads (B*H) and fewer
    than 2^31 code bytes per tensor; outside that the size is 0 and the calls
    refuse the shape before any launch."""
    assert fa.fa_fp8_workspace_size(1, 65535, 128, 128) > 0
    assert fa.fa_fp8_workspace_size(1, 65536, 128, 128) == 0
    assert fa.fa_fp8_workspace_size(256, 256, 1, 128) == 0
    assert fa.fa_fp8_workspace_size(1, 1, 128, 64) == 0
    assert fa.fa_fp8_workspace_size(1, 1, 1 << 24, 128) == 0  # 2^24 rows x 128 bytes = 2^31
    assert fa.fa_fp8_workspace_size(1, 1, (1 << 24) - 128, 128) > 0
    big = 1 << 40
    assert fa.fa_fp8_quantize(FAKE, FAKE, FAKE, 1, 65536, 128, 128, None, 0, FAKE, big, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_fp8(FAKE, big, FAKE, FAKE, 1, 65536, 128, 128, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED


FAKE = 0x100000  # 16-byte aligned, never dereferenced: validation fails first


def test_fwd_argument_errors(lib):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64,
                scale=0.125, causal=0, ws=None, ws_bytes=0, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        if a["ws"] is None:
            return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                             a["d"], a["scale"], a["causal"], a["stream"])
        return fa.fa_fwd_ws(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                            a["d"], a["scale"], a["causal"], a["ws"], a["ws_bytes"], a["stream"])

    assert call(q=None) == fa.FA_ERR_INVALID_ARG
    assert call(lse=None) == fa.FA_ERR_INVALID_ARG
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    assert call(B=-1) == fa.FA_ERR_INVALID_ARG
    assert call(causal=2) == fa.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(d=256) == fa.FA_ERR_UNSUPPORTED
    assert call(B=1 << 12, H=1 << 12, N=1 << 8) == fa.FA_ERR_INVALID_ARG  # >= 2^31 elements
    assert call(B=1, H=16, N=1 << 20, d=128) == fa.FA_ERR_INVALID_ARG  # exactly 2^31 elements
    assert call(q=FAKE + 8) == fa.FA_ERR_MISALIGNED
    assert call(o=FAKE + 2) == fa.FA_ERR_MISALIGNED
    assert call(lse=FAKE + 2) == fa.FA_ERR_MISALIGNED
    # the optional work-counter workspace: 256-byte aligned, at least the size asked for
    assert fa.fa_fwd_workspace_size(1, 1, 128, 64) == 256
    assert fa.fa_fwd_workspace_size(0, 1, 128, 64) == 0
    assert call(ws=FAKE + 16, ws_bytes=256) == fa.FA_ERR_WORKSPACE
    assert call(ws=FAKE, ws_bytes=255) == fa.FA_ERR_WORKSPACE
    assert call(ws=FAKE, ws_bytes=256, q=None) == fa.FA_ERR_INVALID_ARG  # checked before the workspace


def test_bwd_argument_errors(lib):
    ws = fa.fa_bwd_workspace_size(1, 1, 128, 64)
    base = [FAKE] * 9 + [1, 1, 128, 64, 0.125, 1, FAKE, ws, None]

    def call(i=None, val=None):
        a = list(base)
        if i is not None:
            a[i] = val
        return fa.fa_bwd(*a)

    assert call(0, None) == fa.FA_ERR_INVALID_ARG
    assert call(8, None) == fa.FA_ERR_INVALID_ARG
    assert call(12, 80) == fa.FA_ERR_UNSUPPORTED
    assert call(15, None) == fa.FA_ERR_WORKSPACE
    assert call(15, FAKE + 16) == fa.FA_ERR_WORKSPACE  # not 256-byte aligned
    assert call(16, ws - 1) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_prep(None, FAKE, FAKE, 1, 1, 128, 64, FAKE, ws, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_prep(FAKE, FAKE, None, 1, 1, 128, 64, FAKE, ws, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 64, 0.125, 1, FAKE, ws,
                        None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_main(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.125, 1,
                          FAKE, 16, None) == fa.FA_ERR_WORKSPACE


def test_library_is_the_in_tree_build(lib):
    assert os.path.dirname(fa.LIB_PATH) == os.path.join(ROOT, "exact_tiled_attention_05_gb300")


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(RuntimeError):
        fa.load_library(str(tmp_path / "nope.so"))


def test_noalloc_argument_checks_and_scratch_limit(lib):
    """fa_bwd_noalloc checks its arguments in fa_bwd's order before touching the
    device: bad pointers and shapes first, then its fixed scratch limit (2^23
    padded rows, 64 MiB of row statistics + 256 bytes), then alignment.  A
    misaligned pointer marks a size as accepted without any launch."""
    def call(B, H, N, d, q=FAKE, scale=0.125, causal=1):
        return fa.fa_bwd_noalloc(q, *([FAKE] * 8), B, H, N, d, scale, causal, None)

    assert call(1, 1, 128, 64, q=None) == fa.FA_ERR_INVALID_ARG
    assert call(1, 1, 0, 64) == fa.FA_ERR_INVALID_ARG
    assert call(1, 1, 128, 64, causal=2) == fa.FA_ERR_INVALID_ARG
    assert call(1, 1, 128, 64, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    # the shape errors come first, even for sizes beyond the scratch
    assert call(1, 64, 1 << 20, 96) == fa.FA_ERR_UNSUPPORTED
    assert call(1 << 12, 1 << 12, 1 << 8, 128) == fa.FA_ERR_INVALID_ARG  # >= 2^31 elements
    # the limit itself: B*H*ceil(N/128)*128 <= 2^23 rows
    assert fa.fa_bwd_workspace_size(1, 64, 131072, 64) == (64 << 20) + 256
    assert call(1, 64, 131072, 64, q=FAKE + 2) == fa.FA_ERR_MISALIGNED   # accepted size
    assert call(1, 64, 131073, 64, q=FAKE + 2) == fa.FA_ERR_WORKSPACE    # one row over
    assert call(1, 64, 131073, 64) == fa.FA_ERR_WORKSPACE
    assert call(2, 32, 131072, 64, q=FAKE + 2) == fa.FA_ERR_MISALIGNED
    assert call(1, 65, 131072, 64) == fa.FA_ERR_WORKSPACE
