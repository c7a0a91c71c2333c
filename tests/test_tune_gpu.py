"""gizml:tile, "tune": each configuration is measured once and the fastest
is cached; every configuration must compute the same result.  sg_tune times
the configurations that fit, later calls use the choice, and C does not
change by a single bit."""
import numpy as np
import pytest

import oracle
from parity_util import compare, from_device_bits, seeded_case, to_device_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    sg.tune_clear()
    yield
    sg.tune_clear()


@pytest.mark.parametrize("M,N,K,in_dt,out_dt,epi", [
    (2048, 2048, 1024, "bf16", "bf16", "none"),
    (20000, 384, 96, "f16", "f16", "relu"),
    (1000, 1000, 1000, "f16", "f32", "none"),
])
def test_tune_then_gemm_bit_identical(M, N, K, in_dt, out_dt, epi):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    a, b = seeded_case(M, N, K, in_dt, seed=61)
    A = to_device_bits(a, in_dt, "cuda")
    B = to_device_bits(b, in_dt, "cuda")
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out_dt]
    before = sg.stage_gemm(A, B, out_dtype=tdt, epilogue=epi)
    plan0 = sg.plan(M, N, K, A.dtype, tdt, epi)
    best, ms = sg.tune(A, B, out_dtype=tdt, epilogue=epi)
    assert ms > 0 and sg.tune_count() == 1
    plan1 = sg.plan(M, N, K, A.dtype, tdt, epi)
    for k in ("block_n", "stages", "cluster_m", "pair_mma", "group_m"):
        assert plan1[k] == best[k], (k, plan1, best)
    after = sg.stage_gemm(A, B, out_dtype=tdt, epilogue=epi)
    assert sg.device_status() == 0
    assert torch.equal(before.view(torch.int16 if out_dt != "f32" else torch.int32),
                       after.view(torch.int16 if out_dt != "f32" else torch.int32)), (plan0, best)
    if M * N * K <= 1 << 31:
        ref, _, S = oracle.gemm(a, b, in_dt, out_dt, epi)
        compare(from_device_bits(after, out_dt), ref, S, out_dt, "tuned")
    assert sg.tune_clear() == 1 and sg.tune_count() == 0
