"""Plain CPU oracle for the MXFP4 speculative-verification hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The CUDA
product path never imports, loads or calls it, and the two share no code: the
oracle's arithmetic lives in ``mxs_oracle.c`` (plain C, double precision,
written from the pages' definitions), and this module only marshals numpy
arrays into it.

What each entry point follows (page title, section):

* ``e2m1_value`` / ``e8m0_value`` / ``dequant`` -- "Module 11. Speculative
  Decoding and Quantization", §12 (E2M1 bit layout and magnitudes, E8M0 power
  of two, 32-element MX blocks); "Next-Gen Speculative Decoding and FP4
  Quantization ...", section "Microscaling FP4 (MX-FP4) Integration" (packed
  [rows, K/2] nibbles and [rows, K/32] scales).
* ``gemm`` -- the definition Y[m,n] = sum_k x[m,k] * w[n,k], summed in double.
* ``pack`` -- Module 11 §12-§13 (one power-of-two scale per block, nearest grid
  value, zero block gets scale 1).
* ``gemm_w4a4`` -- Module 11 §12 (W4A4: activations in MX-FP4 as well):
  X quantised by ``pack``'s rule, then the plain definition on the quantised
  values.
* ``spec_accept`` -- Module 11 §4 (left-to-right acceptance, residual
  norm((p-q)+), bonus token) and §5 (strict "draw < acceptance", acceptance 0
  where q = 0).
* ``e4m3_value`` / ``nvfp4_dequant`` / ``nvfp4_gemm`` -- Module 11 §12 (NVFP4:
  16 E2M1 values per E4M3 scale, one FP32 scale per tensor).
* ``sampling_law`` -- Module 11 §4 (the laws acceptance uses are the ones
  tokens are actually sampled from: temperature, then top-k, then top-p, on
  the target and the draft alike).
* ``kv_append`` / ``kv_commit`` / ``kv_dequant`` -- the MX-FP4 KV cache of
  "Next-Gen Speculative Decoding and FP4 Quantization ..." (pipeline diagram,
  "Benchmarks and Real-World Impact" item 2) and Module 11 §4 (the unaccepted
  suffix and its cache entries are discarded).

Every function is pinned by ``tests/test_oracle_*.py`` against values the pages
print, closed forms, invariants and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "mxs_oracle.c"
_LIB_PATH = _HERE / "libmxs_oracle.so"
_lib = None

ROW_BAD_DRAFT = 1
ROW_ZERO_Q = 2
ROW_ZERO_RESIDUAL = 4
ROW_NONFINITE = 8


def build(force: bool = False) -> Path:
    """Compile ``mxs_oracle.c`` with the host C compiler (gcc)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", "-o", str(tmp), str(_SRC), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(str(_LIB_PATH))
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.mxs_oracle_e2m1_value.argtypes = [ctypes.c_int]
    lib.mxs_oracle_e2m1_value.restype = ctypes.c_double
    lib.mxs_oracle_e8m0_value.argtypes = [ctypes.c_int]
    lib.mxs_oracle_e8m0_value.restype = ctypes.c_double
    lib.mxs_oracle_dequant.argtypes = [p, p, i64, i64, p]
    lib.mxs_oracle_dequant.restype = ctypes.c_int
    lib.mxs_oracle_gemm.argtypes = [p, p, p, i64, i64, i64, p, ctypes.c_int]
    lib.mxs_oracle_gemm.restype = ctypes.c_int
    lib.mxs_oracle_pack.argtypes = [p, i64, i64, p, p]
    lib.mxs_oracle_pack.restype = ctypes.c_int
    lib.mxs_oracle_e4m3_value.argtypes = [ctypes.c_int]
    lib.mxs_oracle_e4m3_value.restype = ctypes.c_double
    lib.mxs_oracle_nvfp4_dequant.argtypes = [p, p, ctypes.c_double, i64, i64, p]
    lib.mxs_oracle_nvfp4_dequant.restype = ctypes.c_int
    lib.mxs_oracle_nvfp4_gemm.argtypes = [p, p, p, ctypes.c_double, i64, i64, i64, p]
    lib.mxs_oracle_nvfp4_gemm.restype = ctypes.c_int
    lib.mxs_oracle_sampling_law.argtypes = [p, i64, i64, ctypes.c_double, i64, ctypes.c_double, p, p, p]
    lib.mxs_oracle_sampling_law.restype = ctypes.c_int
    lib.mxs_oracle_kv_append.argtypes = [p, i64, i64, i64, p, p, i64, p, p]
    lib.mxs_oracle_kv_append.restype = ctypes.c_int
    lib.mxs_oracle_kv_commit.argtypes = [p, p, i64, i64]
    lib.mxs_oracle_kv_commit.restype = ctypes.c_int
    lib.mxs_oracle_kv_dequant.argtypes = [p, p, i64, i64, i64, p, p]
    lib.mxs_oracle_kv_dequant.restype = ctypes.c_int
    for name in ("mxs_oracle_spec_accept", "mxs_oracle_spec_accept_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [p, p, p, p, i64, i64, i64, p, p, p, p, ctypes.c_int]
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1_value(code: int) -> float:
    return _load().mxs_oracle_e2m1_value(int(code))


def e8m0_value(e: int) -> float:
    return _load().mxs_oracle_e8m0_value(int(e))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 = top half of fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dequant(nibbles: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed MXFP4 [N, K/2] + [N, K/32] -> float64 [N, K]."""
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    N, half = nib.shape
    K = 2 * half
    assert sc.shape == (N, K // 32)
    w = np.empty((N, K), dtype=np.float64)
    rc = _load().mxs_oracle_dequant(_ptr(nib), _ptr(sc), N, K, _ptr(w))
    if rc:
        raise ValueError(f"oracle dequant failed ({rc})")
    return w


def gemm(x_bf16_bits: np.ndarray, nibbles: np.ndarray, scales: np.ndarray,
         nthreads: int | None = None) -> np.ndarray:
    """Y[M, N] (float64) = X (bf16 bit patterns [M, K]) . dequant(W)^T."""
    x = _c(x_bf16_bits, np.uint16)
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    M, K = x.shape
    N = nib.shape[0]
    assert nib.shape == (N, K // 2) and sc.shape == (N, K // 32)
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().mxs_oracle_gemm(_ptr(x), _ptr(nib), _ptr(sc), M, N, K, _ptr(y),
                                 nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle gemm failed ({rc})")
    return y


def pack(w: np.ndarray, *, dtype: str = "f32") -> tuple[np.ndarray, np.ndarray, bool]:
    """Quantise [N, K] weights to (nibbles [N,K/2], scales [N,K/32], all_finite).

    ``w`` is float32 values (dtype="f32") or bf16 bit patterns as uint16
    (dtype="bf16"); both convert to float64 exactly before packing.
    """
    if dtype == "f32":
        wd = np.ascontiguousarray(w, dtype=np.float32).astype(np.float64)
    elif dtype == "bf16":
        wd = bf16_bits_to_f64(w)
    else:
        raise ValueError(dtype)
    wd = np.ascontiguousarray(wd)
    N, K = wd.shape
    nib = np.zeros((N, K // 2), dtype=np.uint8)
    sc = np.zeros((N, K // 32), dtype=np.uint8)
    rc = _load().mxs_oracle_pack(_ptr(wd), N, K, _ptr(nib), _ptr(sc))
    if rc not in (0, 4):
        raise ValueError(f"oracle pack failed ({rc})")
    return nib, sc, rc == 0


def gemm_w4a4(x_bf16_bits: np.ndarray, nibbles: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y[M, N] (float64) = dequant(pack(X)) . dequant(W)^T: both operands MX-FP4.

    X (bf16 bit patterns [M, K]) is quantised block by block by the same rule
    as ``pack``; a row holding a non-finite value, and a weight row with a NaN
    scale (E8M0 byte 255), give NaN outputs.
    """
    x = _c(x_bf16_bits, np.uint16)
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    M, K = x.shape
    N = nib.shape[0]
    assert nib.shape == (N, K // 2) and sc.shape == (N, K // 32)
    xn, xs, _ = pack(x, dtype="bf16")
    xq = dequant(xn, xs)
    w = dequant(nib, sc)
    bad_x = np.any(xs == 255, axis=1)
    bad_w = np.any(sc == 255, axis=1)
    xq[bad_x] = 0.0
    w[bad_w] = 0.0
    y = xq @ w.T
    y[bad_x, :] = np.nan
    y[:, bad_w] = np.nan
    return y


def spec_accept(p: np.ndarray, q: np.ndarray, draft: np.ndarray, u: np.ndarray,
                nthreads: int | None = None, *, f64: bool = False):
    """Acceptance + residual/bonus sampling for B rows.

    p [B, K+1, V], q [B, K, V], draft [B, K] int32, u [B, K+1].
    Returns (tokens [B, K+1] int32 padded with -1, n_emitted [B] int32,
    row_flags [B] int32, edge_dist [B] float64) where edge_dist is the distance
    of u[b, K] from the nearer edge of the chosen inverse-CDF bin.
    """
    dt = np.float64 if f64 else np.float32
    p = _c(p, dt)
    q = _c(q, dt)
    u = _c(u, dt)
    draft = _c(draft, np.int32)
    B, K1, V = p.shape
    K = K1 - 1
    assert q.shape == (B, K, V) and draft.shape == (B, K) and u.shape == (B, K + 1)
    tokens = np.empty((B, K + 1), dtype=np.int32)
    n_emitted = np.empty(B, dtype=np.int32)
    flags = np.empty(B, dtype=np.int32)
    edge = np.empty(B, dtype=np.float64)
    fn = _load().mxs_oracle_spec_accept_f64 if f64 else _load().mxs_oracle_spec_accept
    rc = fn(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), B, K, V, _ptr(tokens),
            _ptr(n_emitted), _ptr(flags), _ptr(edge), nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle spec_accept failed ({rc})")
    return tokens, n_emitted, flags, edge


def sampling_law(logits: np.ndarray, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0):
    """Transformed laws of logit rows [..., V] (fp32): temperature, top-k, top-p.

    Returns (probs float64 [..., V], cut_margin float64 [...], kept int64 [...]):
    cut_margin is the distance of top_p from the cumulative mass at the two
    positions that decide the top-p cut (inf when top-p keeps everything), kept
    the number of tokens of positive probability (0: the row has no law).
    """
    lg = _c(logits, np.float32)
    shape = lg.shape
    V = shape[-1]
    R = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    lg = lg.reshape(R, V)
    probs = np.empty((R, V), dtype=np.float64)
    margin = np.empty(R, dtype=np.float64)
    kept = np.empty(R, dtype=np.int64)
    rc = _load().mxs_oracle_sampling_law(_ptr(lg), R, V, float(temperature), int(top_k), float(top_p),
                                         _ptr(probs), _ptr(margin), _ptr(kept))
    if rc:
        raise ValueError(f"oracle sampling_law failed ({rc})")
    return probs.reshape(shape), margin.reshape(shape[:-1]), kept.reshape(shape[:-1])


def e4m3_value(code: int) -> float:
    return _load().mxs_oracle_e4m3_value(int(code))


def nvfp4_dequant(nibbles: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """NVFP4 [N, K/2] nibbles + [N, K/16] E4M3 scales + FP32 tensor scale -> float64 [N, K]."""
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    N, half = nib.shape
    K = 2 * half
    assert sc.shape == (N, K // 16)
    w = np.empty((N, K), dtype=np.float64)
    if _load().mxs_oracle_nvfp4_dequant(_ptr(nib), _ptr(sc), float(global_scale), N, K, _ptr(w)):
        raise ValueError("oracle nvfp4_dequant failed")
    return w


def nvfp4_gemm(x_bf16_bits: np.ndarray, nibbles: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """Y[M, N] (float64) = X (bf16 bits [M, K]) . nvfp4_dequant(W)^T."""
    x = _c(x_bf16_bits, np.uint16)
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    M, K = x.shape
    N = nib.shape[0]
    assert nib.shape == (N, K // 2) and sc.shape == (N, K // 16)
    y = np.empty((M, N), dtype=np.float64)
    if _load().mxs_oracle_nvfp4_gemm(_ptr(x), _ptr(nib), _ptr(sc), float(global_scale), M, N, K, _ptr(y)):
        raise ValueError("oracle nvfp4_gemm failed")
    return y


def kv_append(kv: np.ndarray, nibbles: np.ndarray, scales: np.ndarray, lens: np.ndarray, *,
              dtype: str = "f32") -> int:
    """Quantise rows kv [B, T, W] into the cache (nibbles [B, L, W/2], scales
    [B, L, W/32], updated in place) at positions lens[b] + t.  Returns the
    number of rows that fell at or beyond L and were not written."""
    if dtype == "f32":
        kd = np.ascontiguousarray(kv, dtype=np.float32).astype(np.float64)
    elif dtype == "bf16":
        kd = bf16_bits_to_f64(kv)
    else:
        raise ValueError(dtype)
    kd = np.ascontiguousarray(kd)
    B, T, W = kd.shape
    L = nibbles.shape[1]
    assert nibbles.shape == (B, L, W // 2) and scales.shape == (B, L, W // 32)
    assert nibbles.flags.c_contiguous and scales.flags.c_contiguous
    assert nibbles.dtype == np.uint8 and scales.dtype == np.uint8
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    full = np.zeros(1, dtype=np.int64)
    rc = _load().mxs_oracle_kv_append(_ptr(kd), B, T, W, _ptr(nibbles), _ptr(scales), L, _ptr(ln), _ptr(full))
    if rc not in (0, 4):
        raise ValueError(f"oracle kv_append failed ({rc})")
    return int(full[0])


def kv_commit(lens: np.ndarray, n_emitted: np.ndarray, L: int) -> np.ndarray:
    """New committed lengths: min(lens + max(n_emitted, 0), L)."""
    ln = np.array(lens, dtype=np.int32, copy=True)
    ne = np.ascontiguousarray(n_emitted, dtype=np.int32)
    rc = _load().mxs_oracle_kv_commit(_ptr(ln), _ptr(ne), ln.size, int(L))
    if rc:
        raise ValueError(f"oracle kv_commit failed ({rc})")
    return ln


def kv_dequant(nibbles: np.ndarray, scales: np.ndarray, lens: np.ndarray) -> np.ndarray:
    """Decoded cache [B, L, W] (float64), zero past each sequence's length."""
    nib = _c(nibbles, np.uint8)
    sc = _c(scales, np.uint8)
    B, L, half = nib.shape
    W = 2 * half
    assert sc.shape == (B, L, W // 32)
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.empty((B, L, W), dtype=np.float64)
    rc = _load().mxs_oracle_kv_dequant(_ptr(nib), _ptr(sc), B, L, W, _ptr(ln), _ptr(out))
    if rc:
        raise ValueError(f"oracle kv_dequant failed ({rc})")
    return out
