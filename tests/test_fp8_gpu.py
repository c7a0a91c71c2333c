"""FP8 E4M3 operands (gizml:tile's "FP8" storage type) on the tensor cores
(tcgen05 kind::f8f6f4), fp32 accumulate: parity with the oracle within the
stated bound, K tails, every stage count, tile width and kernel mode giving
the same bits, element-load staging bit-identical to TMA, the residual, and
the full-size 8192^3 workload on sampled positions."""
import numpy as np
import pytest

import gemm_inputs
import oracle
from parity_util import compare, run_gpu, seeded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()


def _case(M, N, K, seed, lda=None, ldb=None):
    return seeded_case(M, N, K, "e4m3", seed=seed, dist=("normal", 0.0, 2.0), lda=lda, ldb=ldb)


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (7, 9, 32), (128, 128, 128), (129, 257, 300), (300, 200, 1000),
                                   (1000, 1000, 999 + 17)])
def test_fp8_small_shapes(M, N, K):
    lda = (K + 15) // 16 * 16
    ldb = (N + 15) // 16 * 16
    a, b = _case(M, N, K, seed=M + N + K, lda=lda, ldb=ldb)
    got = run_gpu(a, b, M, N, K, "e4m3", "f32")
    ref, _, S = oracle.gemm(a, b, "e4m3", "f32", K=K, N=N)
    compare(got, ref, S, "f32", f"e4m3 {M}x{N}x{K}")


@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("epi", ["none", "relu", "bias_relu"])
def test_fp8_outputs_and_epilogues(out_dt, epi):
    M, N, K = 333, 384, 272
    a, b = _case(M, N, K, seed=101)
    bias = np.linspace(-3, 3, N).astype(np.float32) if epi == "bias_relu" else None
    got = run_gpu(a, b, M, N, K, "e4m3", out_dt, epi, bias)
    ref, _, S = oracle.gemm(a, b, "e4m3", out_dt, epi, bias)
    compare(got, ref, S, out_dt, f"e4m3 -> {out_dt} {epi}")


def test_fp8_stages_widths_modes_bit_identical():
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 1130, 1024, 640
    a, b = _case(M, N, K, seed=102)
    outs = {}
    try:
        for bn, modes in ((128, (1,)), (256, (1, 3))):
            assert lib.sg_test_set_tile_n(bn) == 0
            for mode in modes:
                assert lib.sg_test_set_cluster(mode) == 0
                for st in (1, 2, 4):
                    outs[(bn, mode, st)] = run_gpu(a, b, M, N, K, "e4m3", "bf16", stages=st)
    finally:
        lib.sg_test_set_cluster(0)
        lib.sg_test_set_tile_n(0)
    first = outs[(128, 1, 1)]
    for k, o in outs.items():
        assert np.array_equal(o, first), k
    ref, _, S = oracle.gemm(a, b, "e4m3", "bf16")
    compare(first, ref, S, "bf16", "e4m3 modes")


def test_fp8_element_loads_bit_identical_to_tma():
    """Odd pitches (not multiples of 16 bytes) are staged by element loads."""
    M, N, K = 257, 300, 333
    a, b = _case(M, N, K, seed=103)                      # dense: pitches 333 and 300 bytes
    got = run_gpu(a, b, M, N, K, "e4m3", "f32")
    a2, b2 = _case(M, N, K, seed=103, lda=336, ldb=304)  # 16-byte pitches: TMA
    got2 = run_gpu(a2, b2, M, N, K, "e4m3", "f32")
    assert np.array_equal(got, got2)
    ref, _, S = oracle.gemm(a, b, "e4m3", "f32")
    compare(got, ref, S, "f32", "e4m3 element loads")


def test_fp8_nan_padding_never_read():
    M, N, K = 140, 128, 200
    a, b = _case(M, N, K, seed=104, lda=208, ldb=144)   # E4M3 NaN in the padding
    got = run_gpu(a, b, M, N, K, "e4m3", "f16", "relu")
    assert np.all(np.isfinite(got.view(np.float16)))
    ref, _, S = oracle.gemm(a, b, "e4m3", "f16", "relu", K=K, N=N)
    compare(got, ref, S, "f16", "e4m3 nan padding")


def test_fp8_square8192_sampled():
    w = gemm_inputs.WORKLOADS["square8192_e4m3"]
    a, b = w.a_bits(), w.b_bits()
    got = run_gpu(a, b, w.M, w.N, w.K, w.in_dtype, w.out_dtype)
    rng = np.random.default_rng(w.seed)
    rows = np.concatenate([rng.integers(0, w.M, 4096), np.full(w.N, w.M - 1), np.arange(w.M)])
    cols = np.concatenate([rng.integers(0, w.N, 4096), np.arange(w.N), np.full(w.M, w.N - 1)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, "e4m3", "bf16")
    compare(got[rows, cols], ref, S, "bf16", "square8192_e4m3")


def test_fp8_wide_tiles_bit_identical():
    """FP8 operands in 256 x 512 paired tiles of two accumulators (mode 6; a
    B box is 128 FP8 columns, so each CTA stages one box per accumulator):
    the bits of the 256 x 256 paired tiles and of single CTAs, at every
    depth, with a split tail."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    from parity_util import from_device_bits, to_device_bits
    M, N, K = 2500, 4736, 640                     # FP8 rows of 4736 bytes: TMA-legal
    a, b = _case(M, N, K, seed=103)
    dev = torch.device("cuda")
    A = to_device_bits(a, "e4m3", dev)
    B = to_device_bits(b, "e4m3", dev)
    assert sg.plan(M, N, K, torch.float8_e4m3fn, torch.bfloat16, config={"block_n": 512})["tail_units"] > 0

    def run(cfg):
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        sg.stage_gemm(A, B, out=C, config=cfg)
        assert sg.device_status() == 0
        return from_device_bits(C, "bf16")
    ref = run({"block_n": 256, "mode": 3})
    assert np.array_equal(run({"block_n": 256, "mode": 1}), ref)
    for s in (1, 2, 4):
        assert np.array_equal(run({"block_n": 512, "mode": 6, "stages": s}), ref), s
    rng = np.random.default_rng(7)
    rows = np.concatenate([rng.integers(0, M, 3000), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 3000), np.arange(N)])
    r, _, S = oracle.gemm_at(a, b, rows, cols, "e4m3", "bf16")
    compare(ref[rows, cols], r, S, "bf16", "fp8 wide")
