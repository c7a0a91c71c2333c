"""The host-buffer entry point (sg_gemm_host): chunked copies around the
same GEMM.  Its C must have the bits the device entry point gives on the
same operands (the chunks are row ranges of one product), for every chunk
count, pitched and pageable host buffers, bias, residual (also in place),
FP8 operands and K = 0; one case is also checked against the oracle."""
import os

import numpy as np
import pytest

import oracle
from parity_util import compare, seeded_case, torch_dtype

pytestmark = pytest.mark.gpu


def _host(bits, dt, pinned=True, cols=None):
    """CPU tensor of storage type `dt` holding `bits` (optionally a column
    view of the first `cols` columns, leaving the pitch)."""
    import torch
    view = {"f32": np.int32, "e4m3": np.uint8}.get(dt, np.int16)
    t = torch.from_numpy(np.ascontiguousarray(bits).view(view)).view(torch_dtype(dt))
    if pinned:
        t = t.pin_memory()
    return t if cols is None else t[:, :cols]


def _device_ref(A, B, out_dt, epilogue="none", bias=None, residual=None):
    """The device entry point on copies of the same host operands."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    return sg.stage_gemm(A.cuda(), B.cuda(), out_dtype=torch_dtype(out_dt), epilogue=epilogue,
                         bias=None if bias is None else bias.cuda(),
                         residual=None if residual is None else residual.cuda()).cpu()


def _bits(t):
    import torch
    return t.contiguous().view({1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()]).numpy()


@pytest.fixture
def chunks():
    """Sets STAGE_GEMM_HOST_CHUNKS for one test (read at every call)."""
    old = os.environ.get("STAGE_GEMM_HOST_CHUNKS")

    def set_(n):
        os.environ["STAGE_GEMM_HOST_CHUNKS"] = str(n)
    yield set_
    if old is None:
        os.environ.pop("STAGE_GEMM_HOST_CHUNKS", None)
    else:
        os.environ["STAGE_GEMM_HOST_CHUNKS"] = old


@pytest.mark.parametrize("n_chunks", [1, 3, 7, 64])
def test_chunk_counts_bit_identical(chunks, n_chunks):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 1300, 520, 264                    # ragged rows, 264 = 4 K chunks + 8
    a, b = seeded_case(M, N, K, "f16", seed=61)
    A, B = _host(a, "f16"), _host(b, "f16")
    ref = _device_ref(A, B, "f32", "relu")
    chunks(n_chunks)
    C = sg.stage_gemm_host(A, B, out_dtype=torch.float32, epilogue="relu")
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C), _bits(ref))


def test_pitched_and_pageable_buffers(chunks):
    """Host A and B with row padding (NaN, never read), a C view whose pad
    columns must stay untouched, pageable memory, bias + ReLU, bf16 out."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 777, 300, 200
    a, b = seeded_case(M, N, K, "bf16", seed=62, lda=212, ldb=310)
    A = _host(a, "bf16", pinned=False, cols=K)
    B = _host(b, "bf16", pinned=False, cols=N)
    bias = torch.linspace(-0.5, 0.5, N, dtype=torch.float32)
    Cfull = torch.full((M, N + 12), 7.0, dtype=torch.bfloat16)
    C = Cfull[:, :N]
    chunks(4)
    sg.stage_gemm_host(A, B, epilogue="bias_relu", bias_host=bias, out_host=C)
    torch.cuda.synchronize()
    ref = _device_ref(A.contiguous(), B.contiguous(), "bf16", "bias_relu", bias=bias)
    assert np.array_equal(_bits(C), _bits(ref))
    assert torch.all(Cfull[:, N:] == 7.0)


@pytest.mark.parametrize("in_place", [False, True])
def test_residual(chunks, in_place):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 1030, 96, 384
    a, b = seeded_case(M, N, K, "f16", seed=63)
    A, B = _host(a, "f16"), _host(b, "f16")
    r = torch.randn(M, N, generator=torch.Generator().manual_seed(5)).to(torch.float16)
    ref = _device_ref(A, B, "f16", residual=r)
    chunks(5)
    if in_place:
        C = r.clone().pin_memory()
        sg.stage_gemm_host(A, B, out_host=C, residual_host=C)
    else:
        C = sg.stage_gemm_host(A, B, out_dtype=torch.float16, residual_host=r.pin_memory())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C), _bits(ref))


def test_fp8_operands(chunks):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 600, 256, 320
    a, b = seeded_case(M, N, K, "e4m3", seed=64, dist=("uniform", -2.0, 2.0))
    A, B = _host(a, "e4m3"), _host(b, "e4m3")
    ref = _device_ref(A, B, "bf16")
    chunks(3)
    C = sg.stage_gemm_host(A, B, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C), _bits(ref))


def test_k_zero_bias():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N = 300, 130
    A = torch.empty((M, 0), dtype=torch.float16)
    B = torch.empty((0, N), dtype=torch.float16)
    bias = torch.linspace(-1.0, 1.0, N, dtype=torch.float32)
    C = sg.stage_gemm_host(A, B, out_dtype=torch.float32, epilogue="bias_relu", bias_host=bias)
    torch.cuda.synchronize()
    assert torch.equal(C, torch.relu(bias).expand(M, N))


def test_side_stream_and_oracle(chunks):
    """Queued on a side stream: `stream` waits for every copy and GEMM, so
    synchronising it is enough; the result matches the fp64 oracle."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 900, 640, 512
    a, b = seeded_case(M, N, K, "f16", seed=65)
    A, B = _host(a, "f16"), _host(b, "f16")
    s = torch.cuda.Stream()
    chunks(3)
    C = sg.stage_gemm_host(A, B, out_dtype=torch.float32, stream=s)
    s.synchronize()
    ref, _, S = oracle.gemm(a, b, "f16", "f32")
    compare(C.view(torch.int32).numpy().view(np.uint32), ref, S, "f32", "host entry")
    assert sg.device_status(s) == 0
