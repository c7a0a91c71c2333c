"""Operands without a TMA-legal layout (a base off a 16-byte boundary, or a
row pitch that is not a multiple of 16 bytes) are either copied to 16-byte
pitches before the launch (the device entry points' default) or staged by
element loads of the producer warp into the same swizzled layout, with 0
written where the index is out of range (Tolk.Stage: a failing gate copies
0; sg_gemm_noalloc always takes this path).  Staging moves values and never
rounds them, so C must be bit-identical between the two and to the TMA path
on the same values, and within the parity bound of the oracle."""
import numpy as np
import pytest

import oracle
from parity_util import compare, from_device_bits, repack, run_gpu, seeded_case, to_device_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()


@pytest.mark.parametrize("M,N,K", [(1000, 1000, 999), (257, 129, 130), (64, 33, 7), (130, 1, 200), (1, 77, 95)])
def test_dense_odd_pitches(M, N, K):
    """Dense row-major operands whose pitch (K or N elements) breaks the TMA rule."""
    a, b = seeded_case(M, N, K, "f16", seed=M + N + K)
    with repack(1):
        got = run_gpu(a, b, M, N, K, "f16", "f32", "relu")
    with repack(0):
        elem = run_gpu(a, b, M, N, K, "f16", "f32", "relu")
    assert np.array_equal(got, elem)
    ref, _, S = oracle.gemm(a, b, "f16", "f32", "relu")
    compare(got, ref, S, "f32", f"dense {M}x{N}x{K}")


def _raw(A_ptr, lda, B_ptr, ldb, M, N, K, in_dt, out_dt, C, stages=0):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    codes = {"f32": 0, "f16": 1, "bf16": 2}
    rc = sg.gemm_raw(M, N, K, A_ptr, lda, B_ptr, ldb, C.data_ptr(), N, codes[in_dt], codes[out_dt], 0, None,
                     stages, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    assert sg.device_status() == 0


@pytest.mark.parametrize("in_dt", ["f16", "bf16"])
def test_offset_views_bit_identical_to_tma(in_dt):
    """The same values from a 16-byte-aligned buffer (TMA) and from buffers
    shifted by one element (element loads): identical bits."""
    import torch
    M, N, K = 515, 392, 328
    a, b = seeded_case(M, N, K, in_dt, seed=51, dist=("uniform", -1.0, 1.0))
    dev = torch.device("cuda")
    A = to_device_bits(a, in_dt, dev)
    B = to_device_bits(b, in_dt, dev)
    C_tma = torch.empty(M, N, dtype=torch.float32, device=dev)
    _raw(A.data_ptr(), K, B.data_ptr(), N, M, N, K, in_dt, "f32", C_tma)
    # one-element offsets: base 2 bytes past a 16-byte boundary, same pitch
    a_off = np.zeros((M, K + 8), np.uint16)
    a_off[:, 1:K + 1] = a
    b_off = np.zeros((K, N + 8), np.uint16)
    b_off[:, 1:N + 1] = b
    A2 = to_device_bits(a_off, in_dt, dev)
    B2 = to_device_bits(b_off, in_dt, dev)
    for which in ("A", "B", "AB"):
        for on in (1, 0):  # copied to 16-byte pitches, then staged by element loads
            C = torch.empty(M, N, dtype=torch.float32, device=dev)
            ap, lda = (A2.data_ptr() + 2, K + 8) if "A" in which else (A.data_ptr(), K)
            bp, ldb = (B2.data_ptr() + 2, N + 8) if "B" in which else (B.data_ptr(), N)
            with repack(on):
                _raw(ap, lda, bp, ldb, M, N, K, in_dt, "f32", C)
            assert torch.equal(C.view(torch.int32), C_tma.view(torch.int32)), (which, on)
    ref, _, S = oracle.gemm(a, b, in_dt, "f32")
    compare(from_device_bits(C_tma, "f32"), ref, S, "f32", "tma")


def test_element_path_stage_counts_bit_identical():
    import torch
    M, N, K = 300, 200, 333
    a, b = seeded_case(M, N, K, "bf16", seed=52)
    with repack(0):
        outs = [run_gpu(a, b, M, N, K, "bf16", "bf16", stages=s) for s in (1, 2, 3, 6)]
    with repack(1):
        outs.append(run_gpu(a, b, M, N, K, "bf16", "bf16"))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ref, _, S = oracle.gemm(a, b, "bf16", "bf16")
    compare(outs[0], ref, S, "bf16", "element path")


def test_element_path_nan_padding_never_read():
    """Odd pitch plus NaN in the padding: the padding must not be read."""
    M, N, K = 140, 90, 70
    a, b = seeded_case(M, N, K, "f16", seed=53, lda=73, ldb=93)
    with repack(0):
        got = run_gpu(a, b, M, N, K, "f16", "f16", "bias_relu", np.linspace(-1, 1, N).astype(np.float32))
    with repack(1):
        copied = run_gpu(a, b, M, N, K, "f16", "f16", "bias_relu", np.linspace(-1, 1, N).astype(np.float32))
    assert np.array_equal(got, copied)
    assert np.all(np.isfinite(got.view(np.float16)))
    ref, _, S = oracle.gemm(a, b, "f16", "f16", "bias_relu", np.linspace(-1, 1, N).astype(np.float32), K=K, N=N)
    compare(got, ref, S, "f16", "element nan padding")


@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("epi", ["none", "relu", "bias_relu"])
def test_c_without_tma_layout_bit_identical(out_dt, epi):
    """A C whose pitch breaks the TMA rule (N + 1 elements) is computed into a
    16-byte-pitch buffer and copied out (the default), or written row by row
    from the staging buffer (element path): either way the same bits as the
    TMA store of a dense C, nothing past N or M written (a canary fills the
    padding column), for ragged M and N."""
    M, N, K = 333, 200, 96
    a, b = seeded_case(M, N, K, "f16", seed=54)
    bias = np.linspace(-1, 1, N).astype(np.float32) if epi == "bias_relu" else None
    dense = run_gpu(a, b, M, N, K, "f16", out_dt, epi, bias)
    canary = 0x7F7F7F7F if out_dt == "f32" else 0x7E7E
    for on in (1, 0):
        with repack(on):
            odd = run_gpu(a, b, M, N, K, "f16", out_dt, epi, bias, ldc=N + 1, canary=canary)
        assert np.array_equal(odd[:, :N], dense), on
        assert np.all(odd[:, N] == canary), on
    ref, _, S = oracle.gemm(a, b, "f16", out_dt, epi, bias, K=K, N=N)
    compare(odd[:, :N], ref, S, out_dt, f"element-stored C {out_dt} {epi}")
