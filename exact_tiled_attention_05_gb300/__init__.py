"""GB300 (sm_103a) exact tiled attention: Python binding of libfa.so.

The functions with ``fa_`` names are one-to-one ctypes wrappers of the C ABI in
``include/fa.h`` (raw pointers and sizes).  ``forward`` / ``backward`` marshal
torch tensors into those calls; every step of the computation runs in the CUDA
kernels of libfa.so.  torch supplies only device memory and the current stream.
There is no fallback: if libfa.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_CUDA = 5
FA_ERR_DEVICE_TIMEOUT = 6

EXPORTED = (
    "fa_fwd", "fa_fwd_ws", "fa_fwd_workspace_size", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_prep", "fa_bwd_main",
    "fa_bwd_dq", "fa_bwd_noalloc", "fa_fp8_workspace_size", "fa_fp8_quantize", "fa_fwd_fp8",
    "fa_sync_status", "fa_status_string", "fa_version",
)

FA_FP8_ROTATE = 1
FA_FP8_PER_TENSOR = 2

_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what} failed: {status_string(code)} ({code})")


def load_library(path: str = LIB_PATH):
    """Load libfa.so and declare the C signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libfa.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "fa_fwd": ([P, P, P, P, P, I, I, I, I, F, I, P], I),
        "fa_fwd_ws": ([P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
        "fa_fwd_workspace_size": ([I, I, I, I], Z),
        "fa_bwd_workspace_size": ([I, I, I, I], Z),
        "fa_bwd": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
        "fa_bwd_prep": ([P, P, P, I, I, I, I, P, Z, P], I),
        "fa_bwd_main": ([P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
        "fa_bwd_dq": ([P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
        "fa_bwd_noalloc": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P], I),
        "fa_fp8_workspace_size": ([I, I, I, I], Z),
        "fa_fp8_quantize": ([P, P, P, I, I, I, I, P, I, P, Z, P], I),
        "fa_fwd_fp8": ([P, Z, P, P, I, I, I, I, F, I, P], I),
        "fa_sync_status": ([P], I),
        "fa_status_string": ([I], ctypes.c_char_p),
        "fa_version": ([], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# one-to-one wrappers of the C ABI (pointers as Python ints)
# ---------------------------------------------------------------------------

def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return load_library().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_ws(q, k, v, o, lse, B, H, N, d, scale, causal, ws, ws_bytes, stream):
    return load_library().fa_fwd_ws(q, k, v, o, lse, B, H, N, d, scale, causal, ws, ws_bytes,
                                    stream)


def fa_fwd_workspace_size(B, H, N, d):
    return load_library().fa_fwd_workspace_size(B, H, N, d)


def fa_bwd_workspace_size(B, H, N, d):
    return load_library().fa_bwd_workspace_size(B, H, N, d)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes, stream):
    return load_library().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal,
                                 ws, ws_bytes, stream)


def fa_bwd_prep(o, dout, lse, B, H, N, d, ws, ws_bytes, stream):
    return load_library().fa_bwd_prep(o, dout, lse, B, H, N, d, ws, ws_bytes, stream)


def fa_bwd_main(q, k, v, lse, dout, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes, stream):
    return load_library().fa_bwd_main(q, k, v, lse, dout, dk, dv, B, H, N, d, scale, causal,
                                      ws, ws_bytes, stream)


def fa_bwd_dq(q, k, v, lse, dout, dq, B, H, N, d, scale, causal, ws, ws_bytes, stream):
    return load_library().fa_bwd_dq(q, k, v, lse, dout, dq, B, H, N, d, scale, causal, ws,
                                    ws_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, stream):
    """fa_bwd without a workspace argument, for callers that cannot allocate
    device memory: the scratch is a fixed array (64 MiB + 256 bytes) inside the
    library."""
    return load_library().fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale,
                                         causal, stream)


def fa_fp8_workspace_size(B, H, N, d):
    return load_library().fa_fp8_workspace_size(B, H, N, d)


def fa_fp8_quantize(q, k, v, B, H, N, d, signs, flags, ws, ws_bytes, stream):
    """signs: a ctypes array of four c_uint32 (or None without FA_FP8_ROTATE)."""
    return load_library().fa_fp8_quantize(q, k, v, B, H, N, d, signs, flags, ws, ws_bytes, stream)


def fa_fwd_fp8(ws, ws_bytes, o, lse, B, H, N, d, scale, causal, stream):
    return load_library().fa_fwd_fp8(ws, ws_bytes, o, lse, B, H, N, d, scale, causal, stream)


def fa_sync_status(stream):
    return load_library().fa_sync_status(stream)


def fa_status_string(code):
    return load_library().fa_status_string(code)


def fa_version():
    return load_library().fa_version()


def status_string(code: int) -> str:
    try:
        return fa_status_string(code).decode()
    except Exception:  # library not loadable: still name the code
        return str(code)


def _check(rc: int, what: str):
    if rc != FA_OK:
        raise FAError(rc, what)


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _keep_for_stream(t, stream):
    """A scratch tensor allocated here and used by work enqueued on `stream`:
    keep the caching allocator from reusing its memory until that work is done."""
    if stream is not None:
        t.record_stream(stream)


def _check_qkv(*ts):
    torch = _torch()
    ref = ts[0]
    if ref.dim() != 4:
        raise ValueError("tensors are [B, H, N, d]")
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous bf16 CUDA tensors")
        if t.shape != ref.shape or t.device != ref.device:
            raise ValueError("tensors must share shape and device")
    return tuple(ref.shape)


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, workspace=None, stream=None):
    """O, lse = attention(q, k, v).  q, k, v: bf16 [B, H, N, d] on the GPU.
    Returns (o bf16 [B,H,N,d], lse fp32 [B,H,N]).  Runs fa_fwd_ws: `workspace`
    (uint8 CUDA tensor of fa_fwd_workspace_size bytes) holds the kernel's work
    counter, and one is allocated when none is given.  workspace=False runs
    fa_fwd instead (no workspace: a static schedule of the same items, same
    results)."""
    torch = _torch()
    B, H, N, d = _check_qkv(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv(q, out)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    if workspace is None:
        workspace = torch.empty(int(fa_fwd_workspace_size(B, H, N, d)), dtype=torch.uint8,
                                device=q.device)
        _keep_for_stream(workspace, stream)
    if workspace is False:
        rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, H, N, d, scale, int(bool(causal)), _stream_handle(stream))
    else:
        rc = fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, N, d, scale, int(bool(causal)), workspace.data_ptr(), workspace.numel(),
                       _stream_handle(stream))
    _check(rc, "fa_fwd")
    return out, lse


def workspace_bytes(B, H, N, d) -> int:
    return int(fa_bwd_workspace_size(B, H, N, d))


def alloc_workspace(B, H, N, d, device):
    torch = _torch()
    return torch.empty(workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)


def backward(q, k, v, o, lse, dout, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """dq, dk, dv of attention given the forward's o and lse and dL/dO."""
    torch = _torch()
    B, H, N, d = _check_qkv(q, k, v, o, dout)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_qkv(q, dq, dk, dv)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    if workspace is None:
        workspace = alloc_workspace(B, H, N, d, q.device)
        _keep_for_stream(workspace, stream)
    rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                B, H, N, d, scale, int(bool(causal)), workspace.data_ptr(), workspace.numel(),
                _stream_handle(stream))
    _check(rc, "fa_bwd")
    return dq, dk, dv


def sync_status(stream=None):
    """Synchronise the stream and raise if a kernel reported a device timeout."""
    _check(fa_sync_status(_stream_handle(stream)), "device status")


# ---------------------------------------------------------------------------
# FP8 forward
# ---------------------------------------------------------------------------

def fp8_workspace_bytes(B, H, N, d=128) -> int:
    return int(fa_fp8_workspace_size(B, H, N, d))


def _r256(x: int) -> int:
    return (x + 255) & ~255


def fp8_workspace_views(ws, B, H, N):
    """Typed views of an FP8 workspace (uint8 CUDA tensor) in the layout fa.h
    documents: q8, k8 [BH, npad, 128] and vt8 [BH, 128, npad] (uint8 E4M3 codes),
    sq, sk, sv, vfold [BH, T], vmax [BH] and amax [3] (fp32)."""
    torch = _torch()
    BH, T = B * H, (N + 127) // 128
    npad = 128 * T
    codes = _r256(BH * npad * 128)
    per_tile = _r256(BH * T * 4)
    off = 0
    out = {}
    for name in ("q8", "k8", "vt8"):
        out[name] = ws[off:off + BH * npad * 128]
        off += codes
    out["q8"] = out["q8"].view(BH, npad, 128)
    out["k8"] = out["k8"].view(BH, npad, 128)
    out["vt8"] = out["vt8"].view(BH, 128, npad)
    for name in ("sq", "sk", "sv", "vfold"):
        out[name] = ws[off:off + BH * T * 4].view(torch.float32).view(BH, T)
        off += per_tile
    out["vmax"] = ws[off:off + BH * 4].view(torch.float32)
    off += _r256(BH * 4)
    out["amax"] = ws[off:off + 12].view(torch.float32)
    return out


def sign_words(bits):
    """Four uint32 words (bit j set: s_j = -1) as the ctypes array fa_fp8_quantize takes."""
    words = [int(x) & 0xFFFFFFFF for x in bits]
    if len(words) != 4:
        raise ValueError("signs are four 32-bit words (head dimension 128)")
    return (ctypes.c_uint32 * 4)(*words)


def quantize_fp8(q, k, v, signs=None, rotate=True, per_tensor=False, workspace=None, stream=None):
    """Fill an FP8 workspace from bf16 q, k, v [B, H, N, 128].  signs: four
    uint32 words of random sign bits (required when rotate).  Returns the
    workspace (uint8 CUDA tensor)."""
    torch = _torch()
    B, H, N, d = _check_qkv(q, k, v)
    nbytes = fp8_workspace_bytes(B, H, N, d)
    if nbytes == 0:
        raise ValueError("the FP8 forward takes head dimension 128, B*H <= 65535 and "
                         "B*H*ceil(N/128)*128*128 < 2^31 only")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    flags = (FA_FP8_ROTATE if rotate else 0) | (FA_FP8_PER_TENSOR if per_tensor else 0)
    if rotate and signs is None:
        raise ValueError("rotate=True needs the random sign words")
    sw = sign_words(signs) if rotate else None
    rc = fa_fp8_quantize(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, N, d, sw, flags,
                         workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(rc, "fa_fp8_quantize")
    return workspace


def forward_fp8_quantized(workspace, B, H, N, scale=None, causal=False, out=None, lse=None,
                          device=None, stream=None):
    """Attention from a filled FP8 workspace.  Returns (o bf16, lse fp32)."""
    torch = _torch()
    d = 128
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    device = workspace.device if device is None else device
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or tuple(out.shape) != (B, H, N, d):
        raise ValueError("out must be contiguous bf16 [B, H, N, 128]")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    rc = fa_fwd_fp8(workspace.data_ptr(), workspace.numel(), out.data_ptr(), lse.data_ptr(),
                    B, H, N, d, scale, int(bool(causal)), _stream_handle(stream))
    _check(rc, "fa_fwd_fp8")
    return out, lse


def forward_fp8(q, k, v, signs=None, scale=None, causal=False, rotate=True, per_tensor=False,
                workspace=None, out=None, lse=None, stream=None):
    """FP8 attention: quantize (optionally rotating Q and K), then the FP8
    forward.  Returns (o bf16 [B,H,N,128], lse fp32 [B,H,N])."""
    B, H, N, d = _check_qkv(q, k, v)
    ws = quantize_fp8(q, k, v, signs=signs, rotate=rotate, per_tensor=per_tensor,
                      workspace=workspace, stream=stream)
    return forward_fp8_quantized(ws, B, H, N, scale=scale, causal=causal, out=out, lse=lse,
                                 device=q.device, stream=stream)


# ---------------------------------------------------------------------------
# autograd
# ---------------------------------------------------------------------------

def _make_function():
    torch = _torch()

    class _Attention(torch.autograd.Function):
        """Exact attention with the fused forward and the recompute backward.
        Saves q, k, v, o (bf16) and lse (fp32) for the backward."""

        @staticmethod
        def forward(ctx, q, k, v, scale, causal):
            o, lse = forward(q, k, v, scale=scale, causal=causal)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.scale, ctx.causal = scale, causal
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = backward(q, k, v, o, lse, do.contiguous(), scale=ctx.scale,
                                  causal=ctx.causal)
            return dq, dk, dv, None, None

    return _Attention


_attention_fn = None


def attention(q, k, v, scale=None, causal=False):
    """Differentiable exact attention: O = softmax(scale q k^T [+ causal mask]) v.
    q, k, v: contiguous bf16 CUDA tensors [B, H, N, d], d in {64, 128}."""
    global _attention_fn
    if _attention_fn is None:
        _attention_fn = _make_function()
    d = q.shape[-1]
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    return _attention_fn.apply(q, k, v, s, bool(causal))
