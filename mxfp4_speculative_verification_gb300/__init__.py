"""Python binding of libmxs: MXFP4 speculative verification on GB300 (sm_103a).

The calls of the C ABI (``include/mxs.h``) under the same names:

* :func:`mxfp4_pack` -- real weights -> E2M1 nibbles + E8M0 scales;
* :func:`mxfp4_verify_gemm` -- Y = X . dequant(W)^T, bf16 X, fp32 Y (also
  grouped, without workspace, and :func:`nvfp4_verify_gemm` on NVFP4 weights);
* :func:`spec_accept` -- acceptance, residual / bonus sampling, emission
  (also :func:`spec_accept_logits` from logits under temperature / top-k /
  top-p, and :func:`spec_sampling_law` for the law itself);
* :func:`mxfp4_kv_append`, :func:`spec_kv_commit`, :func:`mxfp4_kv_dequant` --
  the MX-FP4 KV cache of the verification block.

This module only marshals arguments: it checks dtypes, shapes and devices,
allocates the output tensors with torch, and passes raw device pointers and
the current CUDA stream to the library.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU fallback.  If ``libmxs.so`` is
missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import torch

from . import _build

__all__ = ["build", "lib", "mxfp4_pack", "mxfp4_verify_gemm", "mxfp4_verify_gemm_workspace_size",
           "mxfp4_verify_gemm_grouped", "mxfp4_verify_gemm_grouped_workspace_size", "GroupedGemm",
           "mxfp4_verify_gemm_noalloc", "mxfp4_verify_gemm_w4a4", "mxfp4_verify_gemm_w4a4_workspace_size",
           "nvfp4_verify_gemm", "nvfp4_verify_gemm_workspace_size",
           "spec_accept", "mxfp4_kv_append", "spec_kv_commit", "mxfp4_kv_dequant", "spec_sampling_law", "spec_accept_logits",
           "spec_accept_logits_workspace_size", "hbm_read_probe", "hbm_copy_probe", "MxsError",
           "DEV_FLAGS",
           "declared_symbols"]

MXS_F32, MXS_BF16 = 0, 1
DEV_FLAGS = {
    "BAD_DRAFT": 0x1, "ZERO_Q": 0x2, "ZERO_RESIDUAL": 0x4, "NO_LAW": 0x8,
    "NEAR_EDGE": 0x10, "NONFINITE": 0x20, "TIMEOUT": 0x40, "KV_FULL": 0x80,
}

_lib = None


class MxsError(RuntimeError):
    pass


def build(force: bool = False) -> Path:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def declared_symbols() -> list[str]:
    """Function names declared in include/mxs.h."""
    text = (_build.INCLUDE / "mxs.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                      text, flags=re.M)


def lib():
    """The loaded libmxs.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _build.LIB.exists():
        raise MxsError(f"{_build.LIB} is not built; run mxfp4_speculative_verification_gb300.build()")
    L = ctypes.CDLL(str(_build.LIB))
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    L.mxfp4_pack.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp]
    L.mxfp4_pack.restype = i32
    L.mxfp4_verify_gemm_workspace_size.argtypes = [i64, i64, i64]
    L.mxfp4_verify_gemm_workspace_size.restype = sz
    L.mxfp4_verify_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, sz, vp, vp]
    L.mxfp4_verify_gemm.restype = i32
    L.mxfp4_verify_gemm_w4a4_workspace_size.argtypes = [i64, i64, i64]
    L.mxfp4_verify_gemm_w4a4_workspace_size.restype = sz
    L.mxfp4_verify_gemm_w4a4.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, sz, vp, vp]
    L.mxfp4_verify_gemm_w4a4.restype = i32
    L.nvfp4_verify_gemm_workspace_size.argtypes = [i64, i64, i64]
    L.nvfp4_verify_gemm_workspace_size.restype = sz
    L.nvfp4_verify_gemm.argtypes = [vp, vp, vp, ctypes.c_float, vp, i64, i64, i64, vp, sz, vp, vp]
    L.nvfp4_verify_gemm.restype = i32
    L.mxfp4_kv_append.argtypes = [vp, i32, i64, i64, i64, vp, vp, i64, vp, vp, vp]
    L.mxfp4_kv_append.restype = i32
    L.spec_kv_commit.argtypes = [vp, vp, i64, i64, vp]
    L.spec_kv_commit.restype = i32
    L.mxfp4_kv_dequant.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp]
    L.mxfp4_kv_dequant.restype = i32
    L.mxfp4_verify_gemm_grouped_workspace_size.argtypes = [vp, i32, i64]
    L.mxfp4_verify_gemm_grouped_workspace_size.restype = sz
    L.mxfp4_verify_gemm_grouped.argtypes = [vp, i32, i64, vp, sz, vp, vp]
    L.mxfp4_verify_gemm_grouped.restype = i32
    L.mxfp4_verify_gemm_grouped_w4a4_workspace_size.argtypes = [vp, i32, i64]
    L.mxfp4_verify_gemm_grouped_w4a4_workspace_size.restype = sz
    L.mxfp4_verify_gemm_grouped_w4a4.argtypes = [vp, i32, i64, vp, sz, vp, vp]
    L.mxfp4_verify_gemm_grouped_w4a4.restype = i32
    L.spec_accept.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp]
    L.spec_accept.restype = i32
    L.spec_sampling_law.argtypes = [vp, i64, i64, vp, vp, vp, vp]
    L.spec_sampling_law.restype = i32
    L.spec_accept_logits_workspace_size.argtypes = [i64, i64]
    L.spec_accept_logits_workspace_size.restype = sz
    L.spec_accept_logits.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, sz, vp, vp, vp, vp, vp]
    L.spec_accept_logits.restype = i32
    L.mxs_hbm_read_probe.argtypes = [vp, sz, vp, vp]
    L.mxs_hbm_read_probe.restype = i32
    L.mxs_hbm_copy_probe.argtypes = [vp, vp, sz, vp]
    L.mxs_hbm_copy_probe.restype = i32
    L.mxs_status_string.argtypes = [i32]
    L.mxs_status_string.restype = ctypes.c_char_p
    L.mxs_version.argtypes = []
    L.mxs_version.restype = i32
    _lib = L
    return L


def _check(status: int) -> None:
    if status != 0:
        raise MxsError(lib().mxs_status_string(status).decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(*ts: torch.Tensor) -> torch.device:
    dev = ts[0].device
    for t in ts:
        if t is None:
            continue
        if t.device.type != "cuda" or t.device != dev:
            raise MxsError("all tensors must live on the same CUDA device")
        if not t.is_contiguous():
            raise MxsError("tensors must be contiguous")
    return dev


# ---------------------------------------------------------------- pack
def mxfp4_pack(w: torch.Tensor, *, nibbles: torch.Tensor | None = None,
               scales: torch.Tensor | None = None, dev_status: torch.Tensor | None = None):
    """Pack W [N, K] (fp32 or bf16, K % 32 == 0) into (nibbles [N, K/2], scales [N, K/32])."""
    if w.dim() != 2:
        raise MxsError("w must be 2-D [N, K]")
    N, K = w.shape
    if w.dtype == torch.float32:
        dt = MXS_F32
    elif w.dtype == torch.bfloat16:
        dt = MXS_BF16
    else:
        raise MxsError("w must be float32 or bfloat16")
    if K % 32 != 0:
        raise MxsError("K must be a multiple of 32")
    for name, t, shape in (("nibbles", nibbles, (N, K // 2)), ("scales", scales, (N, K // 32))):
        if t is not None and (t.dtype != torch.uint8 or tuple(t.shape) != shape):
            raise MxsError(f"{name} must be a uint8 tensor of shape {list(shape)}")
    _check_status(dev_status)
    if nibbles is None:
        nibbles = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 32), dtype=torch.uint8, device=w.device)
    dev = _need_cuda(w, nibbles, scales, dev_status)
    _check(lib().mxfp4_pack(_ptr(w), dt, N, K, _ptr(nibbles), _ptr(scales), _ptr(dev_status),
                            _stream(dev)))
    return nibbles, scales


# ---------------------------------------------------------------- GEMM
_workspaces: dict = {}


def mxfp4_verify_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().mxfp4_verify_gemm_workspace_size(M, N, K))


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _gemm_shapes(x: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor,
                 out: torch.Tensor | None, dev_status: torch.Tensor | None, block: int = 32):
    """Check the GEMM operands (the C side cannot see buffer extents); returns
    (M, N, K).  block: elements per scale byte (32 MXFP4, 16 NVFP4)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise MxsError("x must be a 2-D bfloat16 tensor [M, K]")
    if nibbles.dtype != torch.uint8 or scales.dtype != torch.uint8 or nibbles.dim() != 2:
        raise MxsError("nibbles and scales must be 2-D uint8 tensors")
    M, K = x.shape
    N = nibbles.shape[0]
    if K % 32 != 0 or nibbles.shape != (N, K // 2) or scales.shape != (N, K // block):
        raise MxsError(f"W shapes must be [N, K/2] and [N, K/{block}] with K % 32 == 0")
    if out is not None and (out.dtype != torch.float32 or tuple(out.shape) != (M, N)):
        raise MxsError("out must be a float32 tensor [M, N]")
    _check_status(dev_status)
    return M, N, K


def _check_status(dev_status: torch.Tensor | None) -> None:
    if dev_status is not None and (dev_status.dtype != torch.int32 or dev_status.numel() < 1):
        raise MxsError("dev_status must be an int32 tensor of at least one element")


def mxfp4_verify_gemm(x: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor, *,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      dev_status: torch.Tensor | None = None) -> torch.Tensor:
    """Y[M, N] (fp32) = X[M, K] (bf16) . dequant(W)^T for MXFP4 W ([N, K/2] + [N, K/32])."""
    M, N, K = _gemm_shapes(x, nibbles, scales, out, dev_status)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise MxsError("workspace must be a uint8 tensor")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    dev = _need_cuda(x, nibbles, scales, out, workspace, dev_status)
    need = mxfp4_verify_gemm_workspace_size(M, N, K)
    if need == 0:
        raise MxsError("unsupported GEMM shape")
    if workspace is None:
        workspace = _workspace(dev, need)
    _check(lib().mxfp4_verify_gemm(_ptr(x), _ptr(nibbles), _ptr(scales), _ptr(out), M, N, K,
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(dev_status), _stream(dev)))
    return out


def mxfp4_verify_gemm_w4a4_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().mxfp4_verify_gemm_w4a4_workspace_size(M, N, K))


def mxfp4_verify_gemm_w4a4(x: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor, *,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           dev_status: torch.Tensor | None = None) -> torch.Tensor:
    """W4A4: Y[M, N] (fp32) = q(X) . dequant(W)^T, q = X quantised to MX-FP4 by the pack rule."""
    M, N, K = _gemm_shapes(x, nibbles, scales, out, dev_status)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise MxsError("workspace must be a uint8 tensor")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    dev = _need_cuda(x, nibbles, scales, out, workspace, dev_status)
    need = mxfp4_verify_gemm_w4a4_workspace_size(M, N, K)
    if need == 0:
        raise MxsError("unsupported GEMM shape")
    if workspace is None:
        workspace = _workspace(dev, need)
    _check(lib().mxfp4_verify_gemm_w4a4(_ptr(x), _ptr(nibbles), _ptr(scales), _ptr(out), M, N, K,
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _ptr(dev_status), _stream(dev)))
    return out


def nvfp4_verify_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_verify_gemm_workspace_size(M, N, K))


def nvfp4_verify_gemm(x: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor, global_scale: float = 1.0,
                      *, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      dev_status: torch.Tensor | None = None) -> torch.Tensor:
    """Y[M, N] (fp32) = global_scale * X[M, K] (bf16) . dequant(W)^T for NVFP4 W
    ([N, K/2] E2M1 nibbles + [N, K/16] E4M3 scale bytes)."""
    M, N, K = _gemm_shapes(x, nibbles, scales, out, dev_status, block=16)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise MxsError("workspace must be a uint8 tensor")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    dev = _need_cuda(x, nibbles, scales, out, workspace, dev_status)
    need = nvfp4_verify_gemm_workspace_size(M, N, K)
    if need == 0:
        raise MxsError("unsupported GEMM shape")
    if workspace is None:
        workspace = _workspace(dev, need)
    _check(lib().nvfp4_verify_gemm(_ptr(x), _ptr(nibbles), _ptr(scales), float(global_scale), _ptr(out), M, N, K,
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(dev_status), _stream(dev)))
    return out


def _kv_cache_shapes(nibbles: torch.Tensor, scales: torch.Tensor, lens: torch.Tensor):
    """(B, L, W) of an MX-FP4 KV cache, checked."""
    if nibbles.dtype != torch.uint8 or scales.dtype != torch.uint8 or nibbles.dim() != 3:
        raise MxsError("cache nibbles and scales must be 3-D uint8 tensors [B, L, W/2] and [B, L, W/32]")
    B, L, half = nibbles.shape
    W = 2 * half
    if W % 32 != 0 or W < 32 or tuple(scales.shape) != (B, L, W // 32):
        raise MxsError("cache shapes must be [B, L, W/2] and [B, L, W/32] with W % 32 == 0")
    if lens.dtype != torch.int32 or tuple(lens.shape) != (B,):
        raise MxsError("lens must be an int32 tensor [B]")
    return B, L, W


def mxfp4_kv_append(kv: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor, lens: torch.Tensor, *,
                    dev_status: torch.Tensor | None = None) -> None:
    """Pack kv [B, T, W] (fp32 or bf16) into the cache at positions lens[b] + t."""
    B, L, W = _kv_cache_shapes(nibbles, scales, lens)
    if kv.dim() != 3 or kv.shape[0] != B or kv.shape[2] != W:
        raise MxsError("kv must be [B, T, W] matching the cache")
    if kv.dtype == torch.float32:
        dt = MXS_F32
    elif kv.dtype == torch.bfloat16:
        dt = MXS_BF16
    else:
        raise MxsError("kv must be float32 or bfloat16")
    _check_status(dev_status)
    dev = _need_cuda(kv, nibbles, scales, lens, dev_status)
    _check(lib().mxfp4_kv_append(_ptr(kv), dt, B, kv.shape[1], W, _ptr(nibbles), _ptr(scales), L, _ptr(lens),
                                 _ptr(dev_status), _stream(dev)))


def spec_kv_commit(lens: torch.Tensor, n_emitted: torch.Tensor, L: int) -> None:
    """lens[b] <- min(lens[b] + n_emitted[b], L) in place (the rejected suffix is discarded)."""
    if lens.dtype != torch.int32 or n_emitted.dtype != torch.int32 or lens.dim() != 1 \
            or tuple(n_emitted.shape) != tuple(lens.shape):
        raise MxsError("lens and n_emitted must be int32 tensors [B]")
    dev = _need_cuda(lens, n_emitted)
    _check(lib().spec_kv_commit(_ptr(lens), _ptr(n_emitted), lens.shape[0], int(L), _stream(dev)))


def mxfp4_kv_dequant(nibbles: torch.Tensor, scales: torch.Tensor, lens: torch.Tensor, *,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """The decoded cache [B, L, W] (fp32), zero past each sequence's length."""
    B, L, W = _kv_cache_shapes(nibbles, scales, lens)
    if out is None:
        out = torch.empty((B, L, W), dtype=torch.float32, device=nibbles.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (B, L, W):
        raise MxsError("out must be a float32 tensor [B, L, W]")
    dev = _need_cuda(nibbles, scales, lens, out)
    _check(lib().mxfp4_kv_dequant(_ptr(nibbles), _ptr(scales), B, L, W, _ptr(lens), _ptr(out), _stream(dev)))
    return out


class GemmProblem(ctypes.Structure):
    """C layout of mxs_gemm_problem."""
    _fields_ = [("x", ctypes.c_void_p), ("nibbles", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


def _problem_array(problems):
    arr = (GemmProblem * len(problems))()
    M = None
    for i, (x, nib, sc, y) in enumerate(problems):
        if x.dtype != torch.bfloat16 or nib.dtype != torch.uint8 or sc.dtype != torch.uint8 \
                or y.dtype != torch.float32:
            raise MxsError("grouped problem dtypes: x bf16, nibbles/scales uint8, y fp32")
        m, K = x.shape
        N = nib.shape[0]
        if nib.shape != (N, K // 2) or sc.shape != (N, K // 32) or y.shape != (m, N):
            raise MxsError("grouped problem shapes: x [M,K], nibbles [N,K/2], scales [N,K/32], y [M,N]")
        if M is None:
            M = m
        elif m != M:
            raise MxsError("all grouped problems must share M")
        arr[i] = GemmProblem(x.data_ptr(), nib.data_ptr(), sc.data_ptr(), y.data_ptr(), N, K)
    return arr, M


def _grouped_fns(w4a4: bool):
    L = lib()
    if w4a4:
        return L.mxfp4_verify_gemm_grouped_w4a4_workspace_size, L.mxfp4_verify_gemm_grouped_w4a4
    return L.mxfp4_verify_gemm_grouped_workspace_size, L.mxfp4_verify_gemm_grouped


_GROUPED_LIMITS = "unsupported grouped GEMM (need 1 <= M <= 65536, K % 512 == 0, aligned W)"


def mxfp4_verify_gemm_grouped_workspace_size(problems, *, w4a4: bool = False) -> int:
    arr, M = _problem_array(problems)
    return int(_grouped_fns(w4a4)[0](arr, len(problems), M))


class GroupedGemm:
    """mxfp4_verify_gemm_grouped bound to its tensors: the problems are checked
    and their table built once, and each call is one C-ABI call on the current
    stream.  For a stack called every step (checking 129 problems in Python
    takes about 0.4 ms of host time).  The plan keeps its tensors alive; it
    reads whatever they hold at each call (in-place updates of x are the way to
    feed new inputs).  Without a workspace it owns one of its own.  With
    w4a4=True it binds mxfp4_verify_gemm_grouped_w4a4 (X quantised to MX-FP4)."""

    def __init__(self, problems, *, workspace: torch.Tensor | None = None, w4a4: bool = False):
        if not problems:
            raise MxsError("a grouped GEMM needs at least one problem")
        self._arr, self._M = _problem_array(problems)
        self._n = len(problems)
        self._tensors = [t for p in problems for t in p]
        self._dev = _need_cuda(*self._tensors, workspace)
        size_fn, self._fn = _grouped_fns(w4a4)
        need = int(size_fn(self._arr, self._n, self._M))
        if need == 0:
            raise MxsError(_GROUPED_LIMITS)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=self._dev)
        elif workspace.dtype != torch.uint8 or workspace.numel() < need:
            raise MxsError(f"workspace must be a uint8 tensor of at least {need} bytes")
        self._ws = workspace

    def __call__(self, *, dev_status: torch.Tensor | None = None) -> None:
        _check_status(dev_status)
        if dev_status is not None:
            _need_cuda(self._ws, dev_status)
        _check(self._fn(self._arr, self._n, self._M, _ptr(self._ws), self._ws.numel(), _ptr(dev_status),
                        _stream(self._dev)))


def mxfp4_verify_gemm_grouped(problems, *, workspace: torch.Tensor | None = None,
                              dev_status: torch.Tensor | None = None, w4a4: bool = False) -> None:
    """Independent GEMMs sharing M: problems is a list of (x, nibbles, scales, y)
    device tensors; each y [M, N] is written with X . dequant(W)^T (w4a4=True:
    with X quantised to MX-FP4 by the pack rule, mxfp4_verify_gemm_grouped_w4a4)."""
    if not problems:
        return
    arr, M = _problem_array(problems)
    dev = _need_cuda(*[t for p in problems for t in p], workspace, dev_status)
    size_fn, fn = _grouped_fns(w4a4)
    need = int(size_fn(arr, len(problems), M))
    if need == 0:
        raise MxsError(_GROUPED_LIMITS)
    if workspace is None:
        workspace = _workspace(dev, need)
    _check(fn(arr, len(problems), M, _ptr(workspace), workspace.numel() * workspace.element_size(),
              _ptr(dev_status), _stream(dev)))


# ---------------------------------------------------------- acceptance
def spec_accept(p: torch.Tensor, q: torch.Tensor, draft: torch.Tensor, u: torch.Tensor, *,
                out_tokens: torch.Tensor | None = None, n_emitted: torch.Tensor | None = None,
                row_flags: torch.Tensor | None = None, dev_status: torch.Tensor | None = None):
    """Speculative acceptance for B rows.

    p [B, K+1, V] fp32, q [B, K, V] fp32, draft [B, K] int32, u [B, K+1] fp32.
    Returns (out_tokens [B, K+1] int32, n_emitted [B] int32).
    """
    if p.dtype != torch.float32 or q.dtype != torch.float32 or u.dtype != torch.float32:
        raise MxsError("p, q and u must be float32")
    if draft.dtype != torch.int32:
        raise MxsError("draft must be int32")
    if p.dim() != 3:
        raise MxsError("p must be 3-D [B, K+1, V]")
    B, K1, V = p.shape
    K = K1 - 1
    if q.shape != (B, K, V) or draft.shape != (B, K) or u.shape != (B, K + 1):
        raise MxsError("shape mismatch: p [B,K+1,V], q [B,K,V], draft [B,K], u [B,K+1]")
    for name, t, shape in (("out_tokens", out_tokens, (B, K + 1)), ("n_emitted", n_emitted, (B,)),
                           ("row_flags", row_flags, (B,))):
        if t is not None and (t.dtype != torch.int32 or tuple(t.shape) != shape):
            raise MxsError(f"{name} must be an int32 tensor of shape {list(shape)}")
    _check_status(dev_status)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=p.device)
    if n_emitted is None:
        n_emitted = torch.empty((B,), dtype=torch.int32, device=p.device)
    dev = _need_cuda(p, q, draft, u, out_tokens, n_emitted, row_flags, dev_status)
    _check(lib().spec_accept(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), B, K, V, _ptr(out_tokens),
                             _ptr(n_emitted), _ptr(row_flags), _ptr(dev_status), _stream(dev)))
    return out_tokens, n_emitted


class _Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


def _sampling(temperature: float, top_k: int, top_p: float) -> _Sampling:
    if not (temperature > 0.0) or top_k < 0 or not (0.0 < top_p <= 1.0):
        raise MxsError("need temperature > 0, top_k >= 0, 0 < top_p <= 1")
    return _Sampling(float(temperature), int(min(top_k, 2**31 - 1)), float(top_p))


def spec_sampling_law(logits: torch.Tensor, *, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                      out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None) -> torch.Tensor:
    """Transformed laws (temperature, top-k, top-p) of logit rows [..., V] fp32."""
    if logits.dtype != torch.float32 or logits.dim() < 1:
        raise MxsError("logits must be a float32 tensor [..., V]")
    if not logits.is_contiguous():
        raise MxsError("logits must be contiguous")
    V = logits.shape[-1]
    R = logits.numel() // max(V, 1)
    if out is None:
        out = torch.empty_like(logits)
    elif out.dtype != torch.float32 or out.shape != logits.shape or not out.is_contiguous():
        raise MxsError("out must be a contiguous float32 tensor shaped like logits")
    _check_status(dev_status)
    s = _sampling(temperature, top_k, top_p)
    dev = _need_cuda(logits, out, dev_status)
    _check(lib().spec_sampling_law(_ptr(logits), R, V, ctypes.addressof(s), _ptr(out), _ptr(dev_status),
                                   _stream(dev)))
    return out


def spec_accept_logits_workspace_size(B: int, K: int) -> int:
    return int(lib().spec_accept_logits_workspace_size(B, K))


def spec_accept_logits(target_logits: torch.Tensor, draft_logits: torch.Tensor, draft: torch.Tensor,
                       u: torch.Tensor, *, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                       workspace: torch.Tensor | None = None, out_tokens: torch.Tensor | None = None,
                       n_emitted: torch.Tensor | None = None, row_flags: torch.Tensor | None = None,
                       dev_status: torch.Tensor | None = None):
    """Speculative acceptance on the transformed laws of logits.

    target_logits [B, K+1, V] fp32, draft_logits [B, K, V] fp32, draft [B, K] int32,
    u [B, K+1] fp32.  Returns (out_tokens [B, K+1] int32, n_emitted [B] int32).
    """
    if target_logits.dtype != torch.float32 or draft_logits.dtype != torch.float32 or u.dtype != torch.float32:
        raise MxsError("logits and u must be float32")
    if draft.dtype != torch.int32:
        raise MxsError("draft must be int32")
    if target_logits.dim() != 3:
        raise MxsError("target_logits must be 3-D [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if draft_logits.shape != (B, K, V) or draft.shape != (B, K) or u.shape != (B, K + 1):
        raise MxsError("shape mismatch: target [B,K+1,V], draft logits [B,K,V], draft [B,K], u [B,K+1]")
    for t in (target_logits, draft_logits, draft, u):
        if not t.is_contiguous():
            raise MxsError("inputs must be contiguous")
    for name, t, shape in (("out_tokens", out_tokens, (B, K + 1)), ("n_emitted", n_emitted, (B,)),
                           ("row_flags", row_flags, (B,))):
        if t is not None and (t.dtype != torch.int32 or tuple(t.shape) != shape):
            raise MxsError(f"{name} must be an int32 tensor of shape {list(shape)}")
    _check_status(dev_status)
    s = _sampling(temperature, top_k, top_p)
    need = spec_accept_logits_workspace_size(B, K)
    if workspace is None:
        workspace = _workspace(target_logits.device, need)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=target_logits.device)
    if n_emitted is None:
        n_emitted = torch.empty((B,), dtype=torch.int32, device=target_logits.device)
    dev = _need_cuda(target_logits, draft_logits, draft, u, workspace, out_tokens, n_emitted, row_flags,
                     dev_status)
    _check(lib().spec_accept_logits(_ptr(target_logits), _ptr(draft_logits), _ptr(draft), _ptr(u), B, K, V,
                                    ctypes.addressof(s), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(out_tokens),
                                    _ptr(n_emitted), _ptr(row_flags), _ptr(dev_status), _stream(dev)))
    return out_tokens, n_emitted


def hbm_read_probe(src: torch.Tensor, sink: torch.Tensor) -> None:
    """Stream ``src`` once (read-only HBM roofline measurement)."""
    dev = _need_cuda(src, sink)
    _check(lib().mxs_hbm_read_probe(_ptr(src), src.numel() * src.element_size() // 16 * 16,
                                    _ptr(sink), _stream(dev)))


def hbm_copy_probe(dst: torch.Tensor, src: torch.Tensor) -> None:
    """Copy ``src`` into ``dst`` with the library's copy kernel (read + write HBM roofline)."""
    nbytes = src.numel() * src.element_size() // 16 * 16
    if dst.numel() * dst.element_size() < nbytes:
        raise MxsError("dst is smaller than src")
    dev = _need_cuda(dst, src)
    _check(lib().mxs_hbm_copy_probe(_ptr(dst), _ptr(src), nbytes, _stream(dev)))


# ------------------------------------------------------- no-allocation GEMM
def mxfp4_verify_gemm_noalloc(x: torch.Tensor, nibbles: torch.Tensor, scales: torch.Tensor, *,
                              out: torch.Tensor | None = None,
                              dev_status: torch.Tensor | None = None) -> torch.Tensor:
    """mxfp4_verify_gemm without a workspace, for callers that cannot allocate
    device memory (e.g. a plugin whose host framework owns every device
    allocation).  The library's fixed 16 MiB device scratch is used instead;
    calls must not overlap on the GPU.  ``out`` should be preallocated by such
    callers (it is allocated here only when omitted)."""
    M, N, K = _gemm_shapes(x, nibbles, scales, out, dev_status)
    L = lib()
    fn = L.mxfp4_verify_gemm_noalloc
    if fn.restype is not ctypes.c_int32:
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        fn.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp]
        fn.restype = ctypes.c_int32
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    dev = _need_cuda(x, nibbles, scales, out, dev_status)
    _check(fn(_ptr(x), _ptr(nibbles), _ptr(scales), _ptr(out), M, N, K, _ptr(dev_status),
              _stream(dev)))
    return out
