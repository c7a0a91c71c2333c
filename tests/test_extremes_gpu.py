"""Sizes at the edges of the index arithmetic, against the oracle on
sampled elements: a K loop of 2048 chunks (the operand ring wraps around
hundreds of times; every stage count must give the same bits), a C of a
million columns (4096+ column tiles), and an A of more than 2^32 elements
(64-bit offsets through TMA and through element loads).  Operands are drawn
on the device from a seeded generator; only the sampled rows and columns
come back to the host for the oracle."""
import numpy as np
import pytest

import oracle
from parity_util import compare

pytestmark = pytest.mark.gpu


def _dev_matrix(rows, cols, dtype, seed, ld=None):
    """rows x cols values N(0,1) rounded to `dtype`, in a rows x ld buffer
    (padding NaN, never read); returns the rows x cols view."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    ld = ld or cols
    buf = torch.full((rows, ld), float("nan"), dtype=dtype, device="cuda")
    step = max(1, (1 << 26) // max(cols, 1))        # row blocks of ~64M values
    for r in range(0, rows, step):
        n = min(step, rows - r)
        buf[r:r + n, :cols] = torch.randn((n, cols), generator=g, device="cuda").to(dtype)
    return buf[:, :cols]


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_sampled(A, B, C, rows, cols, in_dt, out_dt, epi="none"):
    """Oracle on the sampled (rows[t], cols[t]) pairs, from host copies of
    just those rows of A and columns of B."""
    import torch
    ur, ri = np.unique(rows, return_inverse=True)
    uc, ci = np.unique(cols, return_inverse=True)
    a = _bits(A[torch.from_numpy(ur).cuda()])
    b = _bits(B[:, torch.from_numpy(uc).cuda()])
    ref, _, S = oracle.gemm_at(a, b, ri, ci, in_dt, out_dt, epi)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    gbits = got.view(torch.int32 if out_dt == "f32" else torch.int16).cpu().numpy()
    gbits = gbits.view(np.uint32) if out_dt == "f32" else gbits.view(np.uint16)
    compare(gbits, ref, S, out_dt, "sampled")


def test_long_k_ring_wraps():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 256, 256, 131072                      # 2048 K chunks
    A = _dev_matrix(M, K, torch.bfloat16, 1)
    B = _dev_matrix(K, N, torch.bfloat16, 2)
    C = sg.stage_gemm(A, B, out_dtype=torch.float32)
    C1 = sg.stage_gemm(A, B, out_dtype=torch.float32, stages=1)
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    assert torch.equal(C.view(torch.int32), C1.view(torch.int32))
    rng = np.random.default_rng(5)
    rows = np.concatenate([rng.integers(0, M, 600), [0, M - 1, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 600), [0, 0, N - 1]])
    _check_sampled(A, B, C, rows, cols, "bf16", "f32")


def test_million_columns():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 200, (1 << 20) + 40, 72                # ragged in M, N and K
    A = _dev_matrix(M, K, torch.float16, 3, ld=80)
    B = _dev_matrix(K, N, torch.float16, 4)
    C = sg.stage_gemm(A, B, out_dtype=torch.float16, epilogue="relu")
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    rng = np.random.default_rng(6)
    rows = np.concatenate([rng.integers(0, M, 3000), np.full(64, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 3000), np.arange(N - 64, N)])
    _check_sampled(A, B, C, rows, cols, "f16", "f16", "relu")


@pytest.mark.parametrize("lda", [1032, 1033])      # TMA-legal pitch / element-load staging
def test_a_beyond_2_pow_32_elements(lda):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = (1 << 22) + 5, 128, 1030              # A spans (M - 1) * lda + K > 2^32 elements
    assert (M - 1) * lda + K > (1 << 32)
    A = _dev_matrix(M, K, torch.float16, 7, ld=lda)
    B = _dev_matrix(K, N, torch.float16, 8)
    C = sg.stage_gemm(A, B, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    rng = np.random.default_rng(9)
    rows = np.concatenate([rng.integers(0, M, 1500), np.full(N, M - 1), np.full(8, (1 << 22) - 1)])
    cols = np.concatenate([rng.integers(0, N, 1500), np.arange(N), rng.integers(0, N, 8)])
    _check_sampled(A, B, C, rows, cols, "f16", "f16")
    del A, B, C
    torch.cuda.empty_cache()
