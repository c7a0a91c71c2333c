"""GB300 (sm_103a) tensor-core GEMM, C = epilogue(A . B), through the C ABI of
``libstage_gemm.so`` (declared in ``include/stage_gemm.h``).

This module only marshals arguments: every step of the product runs in the
CUDA kernels of the library.  PyTorch supplies device memory and streams.
There is no fallback: if the library is missing, loading raises.

    import torch, tensor_core_gemm_tma_gb300 as sg
    C = sg.stage_gemm(A, B, out_dtype=torch.float16, epilogue="relu")

The operation follows gizml:tile ("Tile.dot", "Tile.run", "In.at",
"Out.put", "Tile.to", "Program.stages") and Tolk.Stage (staged operands,
zero-filling gates, bit-identical results at every stage count).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LIB_PATH = _build.LIB

# Storage-type and epilogue codes of the C ABI.
SG_F32, SG_F16, SG_BF16, SG_E4M3 = 0, 1, 2, 3
EPILOGUES = {"none": 0, "relu": 1, "bias_relu": 2}
SG_MAX_STAGES = 8

ERRORS = {
    -1: "SG_ERR_ARG", -2: "SG_ERR_DTYPE", -3: "SG_ERR_STAGES", -4: "SG_ERR_ALIAS",
    -5: "SG_ERR_ALIGN", -6: "SG_ERR_ARCH", -7: "SG_ERR_CUDA", -8: "SG_ERR_TIMEOUT", -9: "SG_ERR_CONFIG",
}


class SgError(RuntimeError):
    """A negative return code of the C ABI."""

    def __init__(self, code: int, text: str):
        super().__init__(f"{ERRORS.get(code, code)}: {text}")
        self.code = code


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "block_m", "block_n", "block_k", "stages", "max_stages", "tiles", "grid", "threads", "smem_bytes",
        "tmem_columns", "tma_store", "cluster_m", "pair_mma", "group_m", "mode", "ring_group", "tail_units")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class Config(ctypes.Structure):
    """sg_config: an explicit launch configuration (0 = the planner's choice
    for that field).  block_n 128/192/256/512; mode 1 (one CTA per tile), 3
    (CTA pairs with the paired MMA, each CTA owning 128 x block_n), 4
    (resident B) or 6 (CTA pairs over 256 x 512 tiles held as two 256-column
    accumulators; block_n 512); stages 1..8; group_m 1..64; tail_split -1
    (never) or 0/1 (default)."""
    _fields_ = [(n, ctypes.c_int32) for n in ("block_n", "mode", "stages", "group_m", "tail_split")]


def _config(config):
    if config is None:
        return None
    if isinstance(config, Config):
        return config
    unknown = set(config) - {n for n, _ in Config._fields_}
    if unknown:
        raise ValueError(f"unknown configuration fields {sorted(unknown)}")
    return Config(**{k: int(v) for k, v in config.items()})


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libstage_gemm.so (built by ``__graft_entry__.build()`` or
    ``tensor_core_gemm_tma_gb300._build.build()``).  Raises if it is absent."""
    global _lib
    if _lib is not None and path is None:  # the loaded library: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built; run __graft_entry__.build() (nvcc, sm_103a) first")
        lib = ctypes.CDLL(p)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.sg_gemm.restype = i32
        lib.sg_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp, i32, vp]
        lib.sg_gemm_residual.restype = i32
        lib.sg_gemm_residual.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp, i32, vp]
        lib.sg_gemm_qb.restype = i32
        lib.sg_gemm_qb.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, vp, i64, i32, i32, i32, vp, i32, vp]
        lib.sg_gemm_host.restype = i32
        lib.sg_gemm_host.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp, i32, vp]
        lib.sg_plan.restype = i32
        lib.sg_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, i64, vp, ctypes.POINTER(PlanInfo)]
        lib.sg_gemm_ex.restype = i32
        lib.sg_gemm_ex.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp,
                                   ctypes.POINTER(Config), vp]
        lib.sg_plan_ex.restype = i32
        lib.sg_plan_ex.argtypes = [i64, i64, i64, i32, i32, i32, i64, vp, ctypes.POINTER(Config),
                                   ctypes.POINTER(PlanInfo)]
        lib.sg_device_status.restype = i32
        lib.sg_device_status.argtypes = [vp]
        lib.sg_set_wait_limit_ns.restype = None
        lib.sg_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.sg_get_wait_limit_ns.restype = ctypes.c_uint64
        lib.sg_get_wait_limit_ns.argtypes = []
        lib.sg_strerror.restype = ctypes.c_char_p
        lib.sg_strerror.argtypes = [i32]
        lib.sg_version.restype = i32
        lib.sg_version.argtypes = []
        lib.sg_tune.restype = i32
        lib.sg_tune.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp, vp,
                                ctypes.POINTER(PlanInfo), ctypes.POINTER(ctypes.c_float)]
        lib.sg_tune_clear.restype = i32
        lib.sg_tune_clear.argtypes = []
        lib.sg_tune_count.restype = i32
        lib.sg_tune_count.argtypes = []
        lib.sg_test_set_skip_load.restype = i32
        lib.sg_test_set_skip_load.argtypes = [i64]
        lib.sg_test_set_tile_n.restype = i32
        lib.sg_test_set_tile_n.argtypes = [i32]
        lib.sg_test_set_cluster.restype = i32
        lib.sg_test_set_cluster.argtypes = [i32]
        lib.sg_test_set_tail_split.restype = i32
        lib.sg_test_set_tail_split.argtypes = [i32]
        if path is None:
            _lib = lib
        return lib


def strerror(code: int) -> str:
    return load_library().sg_strerror(int(code)).decode()


def _check(rc: int):
    if rc != 0:
        raise SgError(rc, strerror(rc))


def _torch():
    import torch
    return torch


_DTYPE_CODES = None


def dtype_code(dt) -> int:
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        torch = _torch()
        codes = {torch.float32: SG_F32, torch.float16: SG_F16, torch.bfloat16: SG_BF16}
        if hasattr(torch, "float8_e4m3fn"):
            codes[torch.float8_e4m3fn] = SG_E4M3
        _DTYPE_CODES = codes
    code = _DTYPE_CODES.get(dt)
    if code is None:
        raise ValueError(f"unsupported dtype {dt}")
    return code


def _stream_ptr(stream, device):
    torch = _torch()
    if stream is None:
        # the current stream's handle without building a Stream object (the
        # slowest part of a small call); the public route otherwise
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            idx = device.index if getattr(device, "index", None) is not None else torch.cuda.current_device()
            return ctypes.c_void_p(raw(idx))
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _row_pitch(t) -> int:
    """Leading dimension (elements) of a 2-D tensor with unit column stride."""
    if t.dim() != 2:
        raise ValueError("operands must be 2-D")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError("operands must be row-major (unit stride along columns)")
    return max(t.stride(0), t.size(1)) if t.size(0) > 1 else t.size(1)


def gemm_raw(M: int, N: int, K: int, A_ptr: int, lda: int, B_ptr: int, ldb: int, C_ptr: int, ldc: int,
             in_dtype: int, out_dtype: int, epilogue: int, bias_ptr: int | None, stages: int, stream_ptr: int) -> int:
    """The C ABI call itself, on raw pointers; returns its code."""
    return load_library().sg_gemm(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, in_dtype, out_dtype, epilogue,
                                  bias_ptr, stages, stream_ptr)


def stage_gemm(A, B, out_dtype=None, epilogue: str = "none", bias=None, stages: int = 0, out=None, stream=None,
               residual=None, config=None):
    """C = epilogue(A @ B [+ residual]) on A's CUDA device, queued on
    ``stream`` (default: the current stream).  A (M x K) and B (K x N) are
    row-major fp16 or bf16 CUDA tensors of one dtype; ``out_dtype`` is
    float32 (default), float16 or bfloat16; ``bias`` is an fp32 CUDA vector
    of N values for ``epilogue="bias_relu"``; ``residual`` is an M x N
    row-major tensor of the output dtype added to the accumulator before the
    bias and the ReLU (it may be ``out`` itself); ``stages`` is the operand
    ring depth (0: the largest that fits).  ``out`` may be a preallocated
    row-major M x N view (its padding columns are never written).
    ``config`` (a dict of sg_config fields or a ``Config``) fixes the launch
    configuration through sg_gemm_ex: e.g. ``{"block_n": 128, "mode": 3}``
    runs 128 x 128 output tiles per CTA, CTA pairs sharing B; a field the
    problem cannot take raises SG_ERR_CONFIG.  Every configuration gives the
    same bits."""
    torch = _torch()
    if A.device.type != "cuda" or B.device.type != "cuda":
        raise ValueError("A and B must be CUDA tensors")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    elif out_dtype is not None and out.dtype != out_dtype:
        raise ValueError("out has a different dtype from out_dtype")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be M x N")
    if epilogue not in EPILOGUES:
        raise ValueError(f"epilogue must be one of {sorted(EPILOGUES)}")
    bptr = None
    if bias is not None:
        if bias.dtype != torch.float32 or bias.device != A.device or bias.numel() != N or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32 CUDA vector of N values")
        bptr = bias.data_ptr()
    if residual is not None:
        if residual.dtype != out.dtype or tuple(residual.shape) != (M, N) or residual.device != A.device:
            raise ValueError("residual must be an M x N CUDA tensor of the output dtype")
    if config is not None:
        cfg = _config(config)
        if stages:
            cfg.stages = int(stages)
        rptr, ldr = (None, 0) if residual is None else (residual.data_ptr(), _row_pitch(residual))
        rc = load_library().sg_gemm_ex(
            M, N, K, A.data_ptr(), _row_pitch(A), B.data_ptr(), _row_pitch(B), rptr, ldr, out.data_ptr(),
            _row_pitch(out), dtype_code(A.dtype), dtype_code(out.dtype), EPILOGUES[epilogue], bptr,
            ctypes.byref(cfg), _stream_ptr(stream, A.device).value)
    elif residual is not None:
        rc = load_library().sg_gemm_residual(
            M, N, K, A.data_ptr(), _row_pitch(A), B.data_ptr(), _row_pitch(B), residual.data_ptr(),
            _row_pitch(residual), out.data_ptr(), _row_pitch(out), dtype_code(A.dtype), dtype_code(out.dtype),
            EPILOGUES[epilogue], bptr, int(stages), _stream_ptr(stream, A.device).value)
    else:
        rc = gemm_raw(M, N, K, A.data_ptr(), _row_pitch(A), B.data_ptr(), _row_pitch(B), out.data_ptr(),
                      _row_pitch(out), dtype_code(A.dtype), dtype_code(out.dtype), EPILOGUES[epilogue], bptr,
                      int(stages), _stream_ptr(stream, A.device).value)
    _check(rc)
    return out


def stage_gemm_qb(A, Bq, b_scale, out_dtype=None, epilogue: str = "none", bias=None, stages: int = 0, out=None,
                  stream=None):
    """C = epilogue(A @ (Bq * b_scale)) with an integer-coded B: ``Bq`` an
    int8 CUDA tensor of codes (K x N, K <= 128, N <= 512), ``b_scale`` an
    fp32 CUDA vector of N per-column scales; A fp16 or bf16.  Each CTA
    decodes B once into shared memory and every row tile reads it back."""
    torch = _torch()
    if A.device.type != "cuda" or Bq.device.type != "cuda" or b_scale.device.type != "cuda":
        raise ValueError("A, Bq and b_scale must be CUDA tensors")
    if Bq.dtype != torch.int8:
        raise ValueError("Bq must hold int8 codes")
    M, K = A.shape
    K2, N = Bq.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if b_scale.dtype != torch.float32 or b_scale.numel() != N or not b_scale.is_contiguous():
        raise ValueError("b_scale must be a contiguous fp32 vector of N values")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    elif out_dtype is not None and out.dtype != out_dtype:
        raise ValueError("out has a different dtype from out_dtype")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be M x N")
    if epilogue not in EPILOGUES:
        raise ValueError(f"epilogue must be one of {sorted(EPILOGUES)}")
    bptr = None
    if bias is not None:
        if bias.dtype != torch.float32 or bias.device != A.device or bias.numel() != N or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32 CUDA vector of N values")
        bptr = bias.data_ptr()
    rc = load_library().sg_gemm_qb(M, N, K, A.data_ptr(), _row_pitch(A), Bq.data_ptr(), _row_pitch(Bq),
                                   b_scale.data_ptr(), out.data_ptr(), _row_pitch(out), dtype_code(A.dtype),
                                   dtype_code(out.dtype), EPILOGUES[epilogue], bptr, int(stages),
                                   _stream_ptr(stream, A.device).value)
    _check(rc)
    return out


def stage_gemm_host(A_host, B_host, out_dtype=None, epilogue: str = "none", bias_host=None, stages: int = 0,
                    device=None, stream=None, out_host=None, residual_host=None):
    """C = epilogue(A @ B [+ residual]) on HOST tensors through the C ABI's
    host-buffer call (sg_gemm_host): the library copies bias and B in, then
    A (and the residual) in row chunks whose GEMMs run on ``stream`` as the
    rows arrive, and copies each chunk of C back into ``out_host`` while
    later chunks compute.  Asynchronous: synchronise ``stream`` before
    reading ``out_host``, and keep the host tensors alive until then.
    Page-locked (pinned) host tensors let the copies overlap the GEMMs.
    ``out_host`` defaults to a new pinned M x N tensor of ``out_dtype``
    (float32 if not given).  Returns ``out_host``."""
    torch = _torch()
    dev = torch.device(device or "cuda")
    for t in (A_host, B_host):
        if t.device.type != "cpu":
            raise ValueError("A_host and B_host must be CPU tensors")
    if A_host.dtype != B_host.dtype:
        raise ValueError("A and B must have the same dtype")
    M, K = A_host.shape
    K2, N = B_host.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out_host is None:
        out_host = torch.empty((M, N), dtype=out_dtype or torch.float32, pin_memory=True)
    elif out_dtype is not None and out_host.dtype != out_dtype:
        raise ValueError("out_host has a different dtype from out_dtype")
    if out_host.device.type != "cpu" or tuple(out_host.shape) != (M, N):
        raise ValueError("out_host must be an M x N CPU tensor")
    if epilogue not in EPILOGUES:
        raise ValueError(f"epilogue must be one of {sorted(EPILOGUES)}")
    bptr = None
    if bias_host is not None:
        if (bias_host.dtype != torch.float32 or bias_host.device.type != "cpu" or bias_host.numel() != N
                or not bias_host.is_contiguous()):
            raise ValueError("bias_host must be a contiguous fp32 CPU vector of N values")
        bptr = bias_host.data_ptr()
    rptr, ldr = None, 0
    if residual_host is not None:
        if (residual_host.dtype != out_host.dtype or tuple(residual_host.shape) != (M, N)
                or residual_host.device.type != "cpu"):
            raise ValueError("residual_host must be an M x N CPU tensor of the output dtype")
        rptr, ldr = residual_host.data_ptr(), _row_pitch(residual_host)
    with torch.cuda.device(dev):
        rc = load_library().sg_gemm_host(
            M, N, K, A_host.data_ptr(), _row_pitch(A_host), B_host.data_ptr(), _row_pitch(B_host), rptr, ldr,
            out_host.data_ptr(), _row_pitch(out_host), dtype_code(A_host.dtype), dtype_code(out_host.dtype),
            EPILOGUES[epilogue], bptr, int(stages), _stream_ptr(stream, dev).value)
    _check(rc)
    return out_host


def plan(M: int, N: int, K: int, in_dtype, out_dtype, epilogue: str = "none", stages: int = 0, ldc: int | None = None,
         C_ptr: int = 0, config=None) -> dict:
    """The launch configuration ``stage_gemm`` would use (tile, stages, grid,
    shared memory), under ``config`` if given (sg_plan_ex).  Needs a CUDA
    device."""
    info = PlanInfo()
    ldc = N if ldc is None else ldc
    if config is not None:
        cfg = _config(config)
        if stages:
            cfg.stages = int(stages)
        rc = load_library().sg_plan_ex(M, N, K, dtype_code(in_dtype), dtype_code(out_dtype), EPILOGUES[epilogue],
                                       ldc, C_ptr, ctypes.byref(cfg), ctypes.byref(info))
    else:
        rc = load_library().sg_plan(M, N, K, dtype_code(in_dtype), dtype_code(out_dtype), EPILOGUES[epilogue],
                                    int(stages), ldc, C_ptr, ctypes.byref(info))
    _check(rc)
    return info.as_dict()


def tune(A, B, out_dtype=None, epilogue: str = "none", bias=None, out=None, stream=None):
    """Measure every launch configuration that fits C = epilogue(A @ B) on
    these operands and keep the fastest for later calls with the same
    shapes, types and layouts (gizml:tile, "tune").  Returns (plan dict,
    milliseconds per call).  Every configuration computes the same bits."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    info = PlanInfo()
    ms = ctypes.c_float(0.0)
    bptr = None if bias is None else bias.data_ptr()
    rc = load_library().sg_tune(M, N, K, A.data_ptr(), _row_pitch(A), B.data_ptr(), _row_pitch(B), out.data_ptr(),
                                _row_pitch(out), dtype_code(A.dtype), dtype_code(out.dtype), EPILOGUES[epilogue], bptr,
                                _stream_ptr(stream, A.device).value, ctypes.byref(info), ctypes.byref(ms))
    _check(rc)
    return info.as_dict(), float(ms.value)


def tune_clear() -> int:
    return int(load_library().sg_tune_clear())


def tune_count() -> int:
    return int(load_library().sg_tune_count())


def device_status(stream=None) -> int:
    """Synchronises ``stream`` and returns 0, or SG_ERR_TIMEOUT (-8) when a
    kernel of the library gave up on a device-side wait since the last call."""
    torch = _torch()
    return load_library().sg_device_status(_stream_ptr(stream, torch.device("cuda")).value)


def set_wait_limit_ns(ns: int):
    load_library().sg_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    return int(load_library().sg_get_wait_limit_ns())


def version() -> int:
    return int(load_library().sg_version())
