"""CPU oracle for C = epilogue(A . B) -- TEST INFRASTRUCTURE ONLY.

A plain fp64 statement of the tiled tensor-core matrix multiply-accumulate,
written in C (``oracle.c``) and loaded with ctypes.  Only the tests, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may use
it; the product path never imports it and shares no code with it.

Citations (page title and section):
  * gizml:tile, "Tile.dot": [M,K]·[K,N] -> [M,N] in F32 (here fp64).
  * gizml:tile, "In.at" / "Out.put": out-of-range reads are 0, out-of-range
    writes do not happen.
  * gizml:tile, "Tile.run" example, "Tile.relu", "Tile.add": the fused ReLU and
    the broadcast per-column bias.
  * gizml:tile, "Tile.to": one final round to the storage type (RNE).
  * gizml:tile, "Program.fold": an empty K range returns the init (zeros,
    or the residual R when one is given).
  * d4r, rrswin_enc2_epilogues.md, "Shape of the whole MLP band": the
    back-projection's MMA takes the previous accumulator as its C input,
    D = A . B + C -- the residual R added to the sum before bias and ReLU.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# The oracle's own type codes (must match the #defines in oracle.c only).
_DT = {"f32": ord("S"), "f16": ord("H"), "bf16": ord("B"), "e4m3": ord("E")}
_EPI = {"none": ord("n"), "relu": ord("r"), "bias_relu": ord("b")}
_NP_BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no GPU)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        lib.orc_decode.restype = ctypes.c_double
        lib.orc_decode.argtypes = [i32, ctypes.c_uint32]
        lib.orc_encode.restype = ctypes.c_uint32
        lib.orc_encode.argtypes = [i32, ctypes.c_double]
        lib.orc_gemm.restype = i32
        lib.orc_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, vp, i32, vp, i64, dp, dp, i32]
        lib.orc_gemm_residual.restype = i32
        lib.orc_gemm_residual.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i32, i64, i32, i32, vp, i32, vp, i64,
                                          dp, dp, i32]
        lib.orc_gemm_residual_at.restype = i32
        lib.orc_gemm_residual_at.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i32, i64, i32, i32, vp, i32, i64,
                                             vp, vp, vp, dp, dp, i32]
        lib.orc_gemm_at.restype = i32
        lib.orc_gemm_at.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, vp, i32, i64, vp, vp, vp, dp, dp,
                                    i32]
        lib.orc_gemm_qb.restype = i32
        lib.orc_gemm_qb.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, vp, i32, vp, i32, vp, i64, dp, dp, i32]
        lib.orc_decode_array.restype = None
        lib.orc_decode_array.argtypes = [i32, vp, i64, dp]
        lib.orc_encode_array.restype = None
        lib.orc_encode_array.argtypes = [i32, dp, i64, vp]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns (uint16 / uint32) of storage type ``dtype`` -> float64 values."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=_NP_BITS[dtype])
    out = np.empty(b.shape, dtype=np.float64)
    lib.orc_decode_array(_DT[dtype], _ptr(b), b.size, _ptr(out))
    return out


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values -> bit patterns of ``dtype``, round to nearest even."""
    lib = _load()
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=_NP_BITS[dtype])
    lib.orc_encode_array(_DT[dtype], _ptr(v), v.size, _ptr(out))
    return out


def _check_operands(A_bits, B_bits, in_dtype):
    if A_bits.ndim != 2 or B_bits.ndim != 2:
        raise ValueError("A and B must be 2-D bit arrays")
    want = _NP_BITS[in_dtype]
    if A_bits.dtype != want or B_bits.dtype != want:
        raise ValueError(f"A and B hold {in_dtype} patterns ({np.dtype(want).name})")
    for X in (A_bits, B_bits):
        if X.size > 0 and X.shape[1] > 1 and X.strides[1] != X.itemsize:
            raise ValueError("rows of A and B must be contiguous")


def _ld(X) -> int:
    """Row pitch in elements (a degenerate array gets its width)."""
    return max(X.strides[0] // X.itemsize, X.shape[1]) if X.size > 0 and X.shape[0] > 1 else X.shape[1]


def _residual(R_bits, r_dtype, N):
    if R_bits is None:
        return None, _DT["f32"], 0
    if r_dtype is None:
        raise ValueError("r_dtype is required with a residual")
    R = np.asarray(R_bits)
    if R.dtype != _NP_BITS[r_dtype] or R.ndim != 2 or (R.shape[1] > 1 and R.strides[1] != R.itemsize):
        raise ValueError("R must be a row-major bit matrix of r_dtype")
    ldr = max(R.strides[0] // R.itemsize, R.shape[1]) if R.shape[0] > 1 else R.shape[1]
    return R, _DT[r_dtype], ldr


def gemm(A_bits: np.ndarray, B_bits: np.ndarray, in_dtype: str, out_dtype: str, epilogue: str = "none",
         bias: np.ndarray | None = None, K: int | None = None, N: int | None = None, threads: int | None = None,
         C_init: np.ndarray | None = None, R_bits: np.ndarray | None = None, r_dtype: str | None = None):
    """Full product.  A_bits is M x lda (uint16), B_bits is K x ldb (uint16);
    the logical K and N default to the arrays' widths (pass them to leave
    ld padding unread).  R_bits (M x ldr, of storage type r_dtype) is an
    optional residual added to the sum before bias and ReLU.  Returns
    (C_bits, C_exact, S): C_bits is M x ldc in the output's bit type (ldc =
    C_init's width, whose padding is kept untouched; else N), C_exact the
    fp64 value before the final rounding and S the sum of |a_ik b_kj|, both
    M x N."""
    _check_operands(A_bits, B_bits, in_dtype)
    M = A_bits.shape[0]
    K = A_bits.shape[1] if K is None else int(K)
    N = B_bits.shape[1] if N is None else int(N)
    if B_bits.shape[0] < K:
        raise ValueError("B has fewer than K rows")
    lda = _ld(A_bits)
    ldb = _ld(B_bits)
    if C_init is None:
        C = np.zeros((M, N), dtype=_NP_BITS[out_dtype])
    else:
        C = np.array(C_init, dtype=_NP_BITS[out_dtype], copy=True, order="C")
    ldc = C.shape[1] if C.ndim == 2 else N
    exact = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    R, rdt, ldr = _residual(R_bits, r_dtype, N)
    rc = _load().orc_gemm_residual(M, N, K, _ptr(A_bits), lda, _ptr(B_bits), ldb, _ptr(R), rdt, ldr, _DT[in_dtype],
                                   _EPI[epilogue], _ptr(b), _DT[out_dtype], _ptr(C), ldc, _ptr(exact), _ptr(S),
                                   _threads(threads))
    if rc != 0:
        raise ValueError(f"orc_gemm rejected its arguments (rc={rc})")
    return C, exact, S


def gemm_qb(A_bits: np.ndarray, Q: np.ndarray, scale: np.ndarray, in_dtype: str, out_dtype: str,
            epilogue: str = "none", bias: np.ndarray | None = None, K: int | None = None, N: int | None = None,
            threads: int | None = None):
    """Product with an integer-coded B (Tolk.Stage, "Decoded panels on the
    host"): Q holds int8 codes (K x ldq), ``scale`` one fp32 value per
    column, and b_kj = scale_j * q_kj.  A_bits is M x lda of ``in_dtype``.
    Returns (C_bits, C_exact, S) as ``gemm`` does (C dense M x N)."""
    if A_bits.ndim != 2 or Q.ndim != 2:
        raise ValueError("A and Q must be 2-D")
    if A_bits.dtype != _NP_BITS[in_dtype] or Q.dtype != np.int8:
        raise ValueError(f"A holds {in_dtype} patterns and Q int8 codes")
    for X in (A_bits, Q):
        if X.size > 0 and X.shape[1] > 1 and X.strides[1] != X.itemsize:
            raise ValueError("rows of A and Q must be contiguous")
    M = A_bits.shape[0]
    K = A_bits.shape[1] if K is None else int(K)
    N = Q.shape[1] if N is None else int(N)
    if Q.shape[0] < K:
        raise ValueError("Q has fewer than K rows")
    s = np.ascontiguousarray(scale, dtype=np.float32)
    if s.size < N:
        raise ValueError("scale has fewer than N values")
    C = np.zeros((M, N), dtype=_NP_BITS[out_dtype])
    exact = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = _load().orc_gemm_qb(M, N, K, _ptr(A_bits), _ld(A_bits), _DT[in_dtype], _ptr(Q), _ld(Q), _ptr(s),
                             _EPI[epilogue], _ptr(b), _DT[out_dtype], _ptr(C), N, _ptr(exact), _ptr(S),
                             _threads(threads))
    if rc != 0:
        raise ValueError(f"orc_gemm_qb rejected its arguments (rc={rc})")
    return C, exact, S


def gemm_at(A_bits: np.ndarray, B_bits: np.ndarray, rows, cols, in_dtype: str, out_dtype: str,
            epilogue: str = "none", bias: np.ndarray | None = None, K: int | None = None, N: int | None = None,
            threads: int | None = None, R_bits: np.ndarray | None = None, r_dtype: str | None = None):
    """The same definition at the positions (rows[t], cols[t]) only.
    Returns (C_bits, C_exact, S) as 1-D arrays over t."""
    _check_operands(A_bits, B_bits, in_dtype)
    M = A_bits.shape[0]
    K = A_bits.shape[1] if K is None else int(K)
    N = B_bits.shape[1] if N is None else int(N)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    n = r.size
    bits = np.empty(n, dtype=np.uint32)
    exact = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    R, rdt, ldr = _residual(R_bits, r_dtype, N)
    rc = _load().orc_gemm_residual_at(M, N, K, _ptr(A_bits), _ld(A_bits), _ptr(B_bits), _ld(B_bits), _ptr(R), rdt,
                                      ldr, _DT[in_dtype], _EPI[epilogue], _ptr(b), _DT[out_dtype], n, _ptr(r),
                                      _ptr(c), _ptr(bits), _ptr(exact), _ptr(S), _threads(threads))
    if rc != 0:
        raise ValueError(f"orc_gemm_at rejected its arguments (rc={rc})")
    return bits.astype(_NP_BITS[out_dtype]), exact, S


def ulp(values: np.ndarray, dtype: str) -> np.ndarray:
    """One unit in the last place of each (finite) value in storage type
    ``dtype``: 2^(max(floor(log2|v|), emin) - fraction bits)."""
    fbits, emin = {"f32": (23, -126), "f16": (10, -14), "bf16": (7, -126)}[dtype]
    v = np.abs(np.asarray(values, dtype=np.float64))
    _, ex = np.frexp(v)                    # v = m * 2^ex, m in [0.5, 1): floor(log2 v) = ex - 1
    e = np.maximum(np.where(v > 0, ex - 1, emin), emin)
    return np.ldexp(1.0, (e - fbits).astype(np.int64))


def tolerance(S: np.ndarray, C_ref_value: np.ndarray, out_dtype: str, added=None) -> np.ndarray:
    """The parity bound: 1e-3 * sum|a b| + 1e-5, plus one ulp of the rounded
    reference for 16-bit outputs.  `added` (|R| + |bias| per element) covers
    the fp32 additions of a residual and a bias to the fp32 accumulator: each
    rounds by at most half an fp32 ulp of its result, which is within
    2^-24 * (|sum| + |R| + |bias|); the |sum| part lies inside 1e-3 * S, the
    rest is 2^-23 * added."""
    tol = 1e-3 * np.asarray(S, dtype=np.float64) + 1e-5
    if added is not None:
        tol = tol + 2.0 ** -23 * np.abs(np.asarray(added, dtype=np.float64))
    if out_dtype in ("f16", "bf16"):
        tol = tol + ulp(C_ref_value, out_dtype)
    return tol
