"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the CPU oracle on the same seeded bits and compare element by element within
the stated bound |C_gpu - C_ref| <= 1e-3 * sum_k |a_ik b_kj| + 1e-5, plus one
ulp of C_ref for fp16 / bf16 outputs."""
from __future__ import annotations

import contextlib
import numpy as np

import gemm_inputs
import oracle

TORCH_DT = None


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
            "e4m3": torch.float8_e4m3fn}[name]


def bits_dtype(name):
    return {"f32": np.uint32, "e4m3": np.uint8}.get(name, np.uint16)


def decode_np(bits: np.ndarray, name: str) -> np.ndarray:
    """Library decode of output bits (independent of the oracle's decoder)."""
    if name == "f32":
        return bits.view(np.float32).astype(np.float64)
    if name == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_device_bits(bits: np.ndarray, name: str, device):
    """A uint16/uint32 numpy matrix -> CUDA tensor of the storage dtype with
    the same bits."""
    import torch
    if name == "f32":
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int32))
    elif name == "e4m3":
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8))
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch_dtype(name))


def from_device_bits(t, name: str) -> np.ndarray:
    import torch
    if name == "f32":
        return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(a_bits, b_bits, M, N, K, in_dt, out_dt, epi="none", bias=None, stages=0, ldc=None, canary=None,
            device="cuda"):
    """a_bits: M x lda, b_bits: K x ldb (numpy uint16); returns the M x ldc
    output bit matrix (padding included)."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    dev = torch.device(device)
    A = to_device_bits(a_bits, in_dt, dev)[:, :K] if M > 0 else to_device_bits(a_bits, in_dt, dev)
    B = to_device_bits(b_bits, in_dt, dev)[:, :N] if K > 0 else to_device_bits(b_bits, in_dt, dev)
    ldc = N if ldc is None else ldc
    cbits = np.full((M, ldc), canary if canary is not None else 0, dtype=bits_dtype(out_dt))
    Cfull = to_device_bits(cbits, out_dt, dev)
    C = Cfull[:, :N]
    bias_d = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).to(dev)
    lda = a_bits.shape[1] if a_bits.ndim == 2 else K
    ldb = b_bits.shape[1] if b_bits.ndim == 2 else N
    rc = sg.gemm_raw(M, N, K, A.data_ptr(), max(lda, K), B.data_ptr(), max(ldb, N), C.data_ptr(), ldc,
                     sg.dtype_code(torch_dtype(in_dt)), sg.dtype_code(torch_dtype(out_dt)), sg.EPILOGUES[epi],
                     None if bias_d is None else bias_d.data_ptr(), stages,
                     torch.cuda.current_stream(dev).cuda_stream)
    if rc != 0:
        raise sg.SgError(rc, sg.strerror(rc))
    st = sg.device_status()
    assert st == 0, f"device status {st}"
    return from_device_bits(Cfull, out_dt)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, S: np.ndarray, out_dt: str, what: str = ""):
    got = decode_np(got_bits, out_dt)
    ref = decode_np(ref_bits, out_dt)
    tol = oracle.tolerance(S, ref, out_dt)
    finite = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), finite), f"{what}: non-finite pattern differs"
    err = np.where(finite, np.abs(got - ref), 0.0)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"got {got[bad][:5]} ref {ref[bad][:5]} tol {tol[bad][:5]}")
    return float(err.max()) if err.size else 0.0


NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}


def seeded_case(M, N, K, in_dt, seed, dist=("normal", 0.0, 1.0), lda=None, ldb=None, pad_bits=None):
    """Seeded operands with optional ld padding filled with `pad_bits` (a NaN
    of the storage type by default: padding must never be read)."""
    pad_bits = NAN_BITS[in_dt] if pad_bits is None else pad_bits
    a = gemm_inputs.matrix_bits(seed, 0, M, K, dist, in_dt)
    b = gemm_inputs.matrix_bits(seed, 1, K, N, dist, in_dt)
    if lda is not None and lda > K:
        ap = np.full((M, lda), pad_bits, a.dtype)
        ap[:, :K] = a
        a = ap
    if ldb is not None and ldb > N:
        bp = np.full((K, ldb), pad_bits, b.dtype)
        bp[:, :N] = b
        b = bp
    return a, b


@contextlib.contextmanager
def repack(on):
    """Within the block, operands (and residuals) without a TMA-legal layout
    are copied to 16-byte pitches before the launch (on=1, the library's
    default) or staged by element loads (on=0)."""
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    assert lib.sg_test_set_repack(int(on)) == 0
    try:
        yield
    finally:
        lib.sg_test_set_repack(1)
