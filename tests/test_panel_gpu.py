"""Mode 4, the resident B (Tolk.Stage's "decoded panels": an operand's panel
staged once and read back by every trip of the other output loop): each CTA
keeps all of a small B in shared memory and streams only A.  The same MMAs
in the same K order, so C must be bit-identical to the single-CTA mode, for
ragged shapes, every output type, the residual and FP8."""
import numpy as np
import pytest

import oracle
from parity_util import compare, run_gpu, seeded_case
from test_residual_gpu import _rbits, check, run_residual

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()


def _forced(mode, fn):
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    try:
        assert lib.sg_test_set_cluster(mode) == 0
        return fn()
    finally:
        lib.sg_test_set_cluster(0)


def _plan(M, N, K, ind, outd):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}
    return sg.plan(M, N, K, t[ind], t[outd])


@pytest.mark.parametrize("M,N,K", [(300, 100, 16), (1000, 384, 96), (777, 512, 128), (5000, 200, 72), (129, 1, 8),
                                   (40000, 384, 96)])
@pytest.mark.parametrize("out_dt", ["f32", "f16"])
def test_panel_bit_identical_to_single_cta(M, N, K, out_dt):
    a, b = seeded_case(M, N, K, "f16", seed=M + N + K, lda=(K + 7) // 8 * 8, ldb=(N + 7) // 8 * 8)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    p4 = _forced(4, lambda: _plan(M, N, K, "f16", out_dt))
    assert p4["block_n"] == 128 and p4["tiles"] == (M + 127) // 128 and p4["mode"] == 4
    got4 = _forced(4, lambda: run_gpu(a, b, M, N, K, "f16", out_dt, "bias_relu", bias))
    got1 = _forced(1, lambda: run_gpu(a, b, M, N, K, "f16", out_dt, "bias_relu", bias))
    assert np.array_equal(got4, got1)
    ref, _, S = oracle.gemm(a, b, "f16", out_dt, "bias_relu", bias, K=K, N=N)
    compare(got4, ref, S, out_dt, f"panel {M}x{N}x{K}")


def test_panel_stage_counts_bit_identical():
    M, N, K = 3000, 384, 96
    a, b = seeded_case(M, N, K, "bf16", seed=111)
    outs = [_forced(4, lambda s=s: run_gpu(a, b, M, N, K, "bf16", "bf16", stages=s)) for s in (1, 2, 3)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_panel_residual():
    M, N, K = 2000, 96, 128
    a, b = seeded_case(M, N, K, "f16", seed=112)
    r = _rbits(M, N, "f16", 112)
    got4 = _forced(4, lambda: run_residual(a, b, r, M, N, K, "f16", "f16"))
    got1 = _forced(1, lambda: run_residual(a, b, r, M, N, K, "f16", "f16"))
    assert np.array_equal(got4, got1)
    check(got4, a, b, r, "f16", "f16", what="panel residual")


def test_panel_fp8():
    M, N, K = 2500, 384, 200
    a, b = seeded_case(M, N, K, "e4m3", seed=113, dist=("normal", 0.0, 2.0), lda=208, ldb=384)
    p4 = _forced(4, lambda: _plan(M, N, K, "e4m3", "f16"))
    assert p4["block_k"] == 128
    got4 = _forced(4, lambda: run_gpu(a, b, M, N, K, "e4m3", "f16", "relu"))
    got1 = _forced(1, lambda: run_gpu(a, b, M, N, K, "e4m3", "f16", "relu"))
    assert np.array_equal(got4, got1)
    ref, _, S = oracle.gemm(a, b, "e4m3", "f16", "relu", K=K)
    compare(got4, ref, S, "f16", "panel fp8")


def test_panel_is_the_default_for_the_skinny_projection():
    p = _plan(518400, 384, 96, "f16", "f16")
    assert p["tiles"] == 4050 and p["block_n"] == 128 and p["mode"] == 4


@pytest.mark.parametrize("in_dt,out_dt,M,N,K", [("e4m3", "bf16", 2500, 384, 200), ("f16", "f32", 1500, 300, 96),
                                                ("bf16", "bf16", 700, 130, 64)])
def test_panel_bias_from_shared_memory(in_dt, out_dt, M, N, K):
    """Mode 4 stages the biases in shared memory once per CTA (zero past N)
    and adds them per chunk from there: the same fp32 additions as the
    single-CTA mode's reads from global memory, so the same bits."""
    dist = ("normal", 0.0, 2.0) if in_dt == "e4m3" else ("normal", 0.0, 1.0)
    a, b = seeded_case(M, N, K, in_dt, seed=114 + N, dist=dist)
    bias = np.linspace(-2, 2, N).astype(np.float32)
    assert _forced(4, lambda: _plan(M, N, K, in_dt, out_dt))["mode"] == 4
    got4 = _forced(4, lambda: run_gpu(a, b, M, N, K, in_dt, out_dt, "bias_relu", bias))
    got1 = _forced(1, lambda: run_gpu(a, b, M, N, K, in_dt, out_dt, "bias_relu", bias))
    assert np.array_equal(got4, got1)
    ref, _, S = oracle.gemm(a, b, in_dt, out_dt, "bias_relu", bias, K=K, N=N)
    compare(got4, ref, S, out_dt, f"panel bias {in_dt} {M}x{N}x{K}")


def test_panel_residual_with_bias():
    M, N, K = 2000, 200, 96
    a, b = seeded_case(M, N, K, "f16", seed=115)
    r = _rbits(M, N, "f16", 115)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    got4 = _forced(4, lambda: run_residual(a, b, r, M, N, K, "f16", "f16", "bias_relu", bias))
    got1 = _forced(1, lambda: run_residual(a, b, r, M, N, K, "f16", "f16", "bias_relu", bias))
    assert np.array_equal(got4, got1)
    check(got4, a, b, r, "f16", "f16", "bias_relu", bias, what="panel residual + bias")


def test_panel_plan_counts_the_staged_biases():
    """With a bias, mode 4's shared memory also holds the N biases (fp32,
    whole 128-column blocks): the projection's plan grows by 3 x 128 x 4
    bytes and keeps its 3 ring slots."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    plain = sg.plan(518400, 384, 96, torch.float16, torch.float16, "relu")
    biased = sg.plan(518400, 384, 96, torch.float16, torch.float16, "bias_relu")
    assert plain["mode"] == biased["mode"] == 4
    assert biased["smem_bytes"] == plain["smem_bytes"] + 3 * 128 * 4
    assert biased["stages"] == plain["stages"] == 3


def test_panel_k_zero_gives_relu_bias():
    """Program.fold: with K = 0 no MMA runs and every element is the
    epilogue of zero: relu(bias[col]), read from the biases mode 4 staged in
    shared memory (N = 296: the last 128-column block is ragged)."""
    M, N = 1000, 296
    bias = np.linspace(-3, 3, N).astype(np.float32)
    a = np.zeros((M, 8), np.uint16)
    b = np.zeros((8, N), np.uint16)
    assert _forced(4, lambda: _plan(M, N, 0, "f16", "f16"))["mode"] == 4
    got = _forced(4, lambda: run_gpu(a, b, M, N, 0, "f16", "f16", "bias_relu", bias))
    want = np.tile(np.maximum(bias.astype(np.float64), 0), (M, 1))
    assert np.array_equal(got, want.astype(np.float16).view(np.uint16))
