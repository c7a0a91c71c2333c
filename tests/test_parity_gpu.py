"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs, element by element within
|C_gpu - C_ref| <= 1e-3 * sum_k |a_ik b_kj| + 1e-5 (+ 1 ulp of C_ref for
fp16/bf16 output).  The five workloads run at their full sizes with the
launch configuration the benchmark uses (stages = 0: the deepest ring);
the oracle checks every element where it finishes in seconds, and sampled
positions (plus whole edge rows and columns) where it does not."""
import numpy as np
import pytest

import gemm_inputs
import oracle
from parity_util import compare, run_gpu, seeded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    sg.load_library()
    torch.cuda.set_device(0)
    yield


def _full_workload(name):
    w = gemm_inputs.WORKLOADS[name]
    a, b, bias = w.a_bits(), w.b_bits(), w.bias()
    got = run_gpu(a, b, w.M, w.N, w.K, w.in_dtype, w.out_dtype, w.epilogue, bias)
    ref, exact, S = oracle.gemm(a, b, w.in_dtype, w.out_dtype, w.epilogue, bias)
    return compare(got, ref, S, w.out_dtype, name)


def test_square256_f16_full():
    _full_workload("square256_f16")


def test_ragged1000_f16_full():
    _full_workload("ragged1000_f16")


def test_relu4096_f16_full():
    _full_workload("relu4096_f16")


def _sampled_workload(name, n_random=4096, edge_rows=(), edge_cols=()):
    w = gemm_inputs.WORKLOADS[name]
    a, b, bias = w.a_bits(), w.b_bits(), w.bias()
    got = run_gpu(a, b, w.M, w.N, w.K, w.in_dtype, w.out_dtype, w.epilogue, bias)
    rng = np.random.default_rng(w.seed)
    rows = [rng.integers(0, w.M, n_random)]
    cols = [rng.integers(0, w.N, n_random)]
    for r in edge_rows:
        rows.append(np.full(w.N, r))
        cols.append(np.arange(w.N))
    for c in edge_cols:
        rows.append(np.arange(w.M))
        cols.append(np.full(w.M, c))
    rows = np.concatenate(rows)
    cols = np.concatenate(cols)
    ref, exact, S = oracle.gemm_at(a, b, rows, cols, w.in_dtype, w.out_dtype, w.epilogue, bias)
    return compare(got[rows, cols], ref, S, w.out_dtype, name)


def test_square8192_bf16_sampled():
    # 4096 random elements, row 0 and column 0, and every element of the last
    # row tile and the last column tile (256 = one paired tile's rows and columns)
    edge = (0,) + tuple(range(8192 - 256, 8192))
    _sampled_workload("square8192_bf16", edge_rows=edge, edge_cols=edge)


def test_swin4k_proj_f16_sampled():
    w = gemm_inputs.WORKLOADS["swin4k_proj_f16"]
    _sampled_workload("swin4k_proj_f16", n_random=8192, edge_rows=tuple(range(w.M - 130, w.M)) + (0, 1),
                      edge_cols=(0, 383))


SMALL = [(1, 1, 8), (1, 8, 1), (7, 9, 16), (128, 128, 64), (129, 65, 72), (255, 257, 200), (64, 300, 8),
         (300, 64, 136), (1000, 8, 40), (8, 1000, 1000), (130, 130, 1024)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_small_shapes_f16_f32(M, N, K):
    a, b = seeded_case(M, N, K, "f16", seed=M * 7 + N * 3 + K, lda=(K + 7) // 8 * 8, ldb=(N + 7) // 8 * 8)
    got = run_gpu(a, b, M, N, K, "f16", "f32")
    ref, _, S = oracle.gemm(a, b, "f16", "f32", K=K, N=N)
    compare(got, ref, S, "f32", f"{M}x{N}x{K}")


@pytest.mark.parametrize("in_dt", ["f16", "bf16"])
@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("epi", ["none", "relu", "bias_relu"])
def test_dtype_epilogue_grid(in_dt, out_dt, epi):
    M, N, K = 333, 300, 200
    a, b = seeded_case(M, N, K, in_dt, seed=5, lda=208, ldb=304)
    bias = None
    if epi == "bias_relu":
        bias = gemm_inputs.to_storage_bits(gemm_inputs.draw(5, 2, N, ("normal", 0.0, 3.0)), "f32").view(np.float32)
    got = run_gpu(a, b, M, N, K, in_dt, out_dt, epi, bias)
    ref, _, S = oracle.gemm(a, b, in_dt, out_dt, epi, bias, K=K, N=N)
    compare(got, ref, S, out_dt, f"{in_dt}->{out_dt} {epi}")


@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
def test_c_padding_canaries_untouched(out_dt):
    """Out.put: nothing outside M x N is written (ldc padding keeps its bits)."""
    M, N, K = 200, 136, 96
    ldc = 136 + 24
    canary = 0x7F7F7F7F if out_dt == "f32" else 0x7BAD
    a, b = seeded_case(M, N, K, "f16", seed=11)
    got = run_gpu(a, b, M, N, K, "f16", out_dt, ldc=ldc, canary=canary)
    assert np.all(got[:, N:] == canary)
    ref, _, S = oracle.gemm(a, b, "f16", out_dt)
    compare(got[:, :N], ref, S, out_dt, "canary")


def test_nan_in_operand_padding_is_never_read():
    """In.at / Tolk.Stage gates: out-of-range operand elements read as 0."""
    M, N, K = 150, 100, 70
    a, b = seeded_case(M, N, K, "f16", seed=12, lda=96, ldb=128)   # NaN in the padding
    got = run_gpu(a, b, M, N, K, "f16", "f32")
    assert np.all(np.isfinite(got.view(np.float32)))
    ref, _, S = oracle.gemm(a, b, "f16", "f32", K=K, N=N)
    compare(got, ref, S, "f32", "nan-padding")


@pytest.mark.parametrize("epi", ["none", "relu", "bias_relu"])
def test_k_zero_writes_epilogue_of_zero(epi):
    """Program.fold: an empty K range leaves the zeros it starts from."""
    M, N = 130, 72
    bias = np.linspace(-2, 2, N).astype(np.float32) if epi == "bias_relu" else None
    a = np.zeros((M, 8), np.uint16)
    b = np.zeros((8, N), np.uint16)
    got = run_gpu(a, b, M, N, 0, "f16", "f16", epi, bias)
    want = np.zeros((M, N)) if bias is None else np.tile(np.maximum(bias.astype(np.float64), 0), (M, 1))
    # one rounding of the fp32 value to the fp16 output (Tile.to)
    assert np.array_equal(got, want.astype(np.float16).view(np.uint16))


def test_empty_m_or_n_is_noop():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    A = torch.zeros(0, 64, dtype=torch.float16, device="cuda")
    B = torch.zeros(64, 32, dtype=torch.float16, device="cuda")
    C = sg.stage_gemm(A, B)
    assert C.shape == (0, 32)
    A = torch.zeros(16, 64, dtype=torch.float16, device="cuda")
    B = torch.zeros(64, 0, dtype=torch.float16, device="cuda")
    assert sg.stage_gemm(A, B).shape == (16, 0)


@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
def test_unaligned_c_uses_masked_stores(out_dt):
    """An ldc whose byte pitch is not a multiple of 16 cannot use TMA stores;
    the masked element-store epilogue must give the same values."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 190, 150, 64
    ldc = 151
    p = sg.plan(M, N, K, torch.float16, {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out_dt],
                ldc=ldc, C_ptr=0)
    assert p["tma_store"] == 0
    a, b = seeded_case(M, N, K, "f16", seed=13, ldb=152)
    canary = 0x7F7F7F7F if out_dt == "f32" else 0x7BAD
    got = run_gpu(a, b, M, N, K, "f16", out_dt, ldc=ldc, canary=canary)
    assert np.all(got[:, N:] == canary)
    ref, _, S = oracle.gemm(a, b, "f16", out_dt, N=N)
    compare(got[:, :N], ref, S, out_dt, "masked")


def test_torch_api_matches_raw_path():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 256, 384, 192
    a, b = seeded_case(M, N, K, "bf16", seed=14)
    A = torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    B = torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    C = sg.stage_gemm(A, B, out_dtype=torch.bfloat16, epilogue="relu")
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, _, S = oracle.gemm(a, b, "bf16", "bf16", "relu")
    compare(got, ref, S, "bf16", "torch-api")
    # end-to-end host path
    Ah, Bh = A.cpu().pin_memory(), B.cpu().pin_memory()  # alive until the stream has finished with them
    Ch = sg.stage_gemm_host(Ah, Bh, out_dtype=torch.bfloat16, epilogue="relu")
    torch.cuda.synchronize()
    assert torch.equal(Ch.view(torch.int16), C.cpu().view(torch.int16))
