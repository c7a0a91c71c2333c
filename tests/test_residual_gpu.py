"""C = epilogue(A . B + R): the residual as the accumulator's seed, the
back-projection of the Swin-layer MLP band (d4r, rrswin_enc2_epilogues.md,
"Shape of the whole MLP band"; gizml:tile, "Program.fold" with a non-zero
init).  Parity with the oracle, in place (R = C), R loaded by TMA or by
element loads (bit-identical), K = 0, stage counts, and the full-size
back-projection workload on sampled positions."""
import numpy as np
import pytest

import gemm_inputs
import oracle
from parity_util import bits_dtype, decode_np, from_device_bits, repack, seeded_case, to_device_bits

pytestmark = pytest.mark.gpu

CODES = {"f32": 0, "f16": 1, "bf16": 2}
EPI = {"none": 0, "relu": 1, "bias_relu": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()


def _rbits(M, N, out_dt, seed, ld=None, scale=2.0):
    ld = N if ld is None else ld
    r = gemm_inputs.to_storage_bits(gemm_inputs.draw(seed, 3, M * N, ("normal", 0.0, scale)), out_dt).reshape(M, N)
    if ld > N:
        rp = np.zeros((M, ld), r.dtype)
        rp[:, :N] = r
        r = rp
    return r


def run_residual(a, b, r, M, N, K, in_dt, out_dt, epi="none", bias=None, stages=0, in_place=False, r_offset=0):
    """r: M x ldr bits; r_offset shifts R by whole elements inside a larger
    buffer (an R whose base is not 16-byte aligned is read by element loads)."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    dev = torch.device("cuda")
    A = to_device_bits(a, in_dt, dev)
    B = to_device_bits(b, in_dt, dev)
    ldr = r.shape[1]
    esz = 4 if out_dt == "f32" else 2
    if in_place:
        C = to_device_bits(np.ascontiguousarray(r), out_dt, dev)
        Rp, Cp, ldc = C.data_ptr(), C.data_ptr(), ldr
    else:
        rbuf = np.zeros(r.size + 16, bits_dtype(out_dt))
        rbuf[r_offset:r_offset + r.size] = r.ravel()
        Rdev = to_device_bits(rbuf, out_dt, dev)
        Rp = Rdev.data_ptr() + r_offset * esz
        C = to_device_bits(np.zeros((M, N), bits_dtype(out_dt)), out_dt, dev)
        Cp, ldc = C.data_ptr(), N
    bias_d = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).to(dev)
    rc = sg.load_library().sg_gemm_residual(M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], Rp, ldr,
                                            Cp, ldc, CODES[in_dt], CODES[out_dt], EPI[epi],
                                            None if bias_d is None else bias_d.data_ptr(), stages,
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    assert sg.device_status() == 0
    out = from_device_bits(C, out_dt)
    return out[:, :N] if in_place else out


def check(got, a, b, r, in_dt, out_dt, epi="none", bias=None, K=None, N=None, what=""):
    ref, exact, S = oracle.gemm(a, b, in_dt, out_dt, epi, bias, K=K, N=N, R_bits=r, r_dtype=out_dt)
    Nn = ref.shape[1]
    rv = np.abs(decode_np(np.ascontiguousarray(r[:, :Nn]), out_dt))
    added = rv + (0.0 if bias is None else np.abs(bias.astype(np.float64)))
    g = decode_np(got, out_dt)
    rr = decode_np(ref, out_dt)
    tol = oracle.tolerance(S, rr, out_dt, added=added)
    err = np.abs(g - rr)
    assert np.all(err <= tol), f"{what}: {int((err > tol).sum())} outside tolerance, max {err.max()}"


@pytest.mark.parametrize("in_dt,out_dt,epi", [("f16", "f16", "none"), ("bf16", "f32", "relu"),
                                                ("f16", "bf16", "bias_relu"), ("bf16", "bf16", "none")])
def test_residual_parity(in_dt, out_dt, epi):
    M, N, K = 333, 200, 264
    a, b = seeded_case(M, N, K, in_dt, seed=81)
    r = _rbits(M, N, out_dt, 81)
    bias = np.linspace(-1, 1, N).astype(np.float32) if epi == "bias_relu" else None
    got = run_residual(a, b, r, M, N, K, in_dt, out_dt, epi, bias)
    check(got, a, b, r, in_dt, out_dt, epi, bias, what=f"{in_dt}->{out_dt} {epi}")


@pytest.mark.parametrize("out_dt", ["f32", "f16"])
def test_residual_in_place(out_dt):
    """R = C (same pointer and pitch): x <- A.B + x."""
    M, N, K = 300, 256, 128
    a, b = seeded_case(M, N, K, "f16", seed=82)
    r = _rbits(M, N, out_dt, 82)
    got = run_residual(a, b, r, M, N, K, "f16", out_dt, in_place=True)
    check(got, a, b, r, "f16", out_dt, what="in place")


@pytest.mark.parametrize("out_dt", ["f16", "f32"])
def test_residual_element_loads_bit_identical(out_dt):
    """An R off a 16-byte boundary or with an odd pitch, copied to a 16-byte
    pitch or read by element loads: the same bits as the TMA-staged
    residual."""
    M, N, K = 260, 136, 192
    a, b = seeded_case(M, N, K, "f16", seed=83)
    r = _rbits(M, N, out_dt, 83)
    tma = run_residual(a, b, r, M, N, K, "f16", out_dt)
    r_odd = _rbits(M, N, out_dt, 83, ld=N + 1)
    for on in (1, 0):  # copied to a 16-byte pitch, then read by element loads
        with repack(on):
            off = run_residual(a, b, r, M, N, K, "f16", out_dt, r_offset=1)
            odd = run_residual(a, b, r_odd, M, N, K, "f16", out_dt)
        assert np.array_equal(tma, off) and np.array_equal(tma, odd), on
    check(tma, a, b, r, "f16", out_dt, what="tma residual")


def test_residual_k_zero_is_epilogue_of_r():
    M, N = 140, 100
    a = np.zeros((M, 8), np.uint16)
    b = np.zeros((8, N), np.uint16)
    r = _rbits(M, N, "f16", 84)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    got = run_residual(a, b, r, M, N, 0, "f16", "f16", "bias_relu", bias)
    check(got, a, b, r, "f16", "f16", "bias_relu", bias, K=0, what="K=0")
    got2 = run_residual(a, b, r, M, N, 0, "f16", "f16")
    assert np.array_equal(got2, r)


def test_residual_stage_counts_bit_identical():
    M, N, K = 600, 96, 384
    a, b = seeded_case(M, N, K, "f16", seed=85)
    r = _rbits(M, N, "f16", 85)
    outs = [run_residual(a, b, r, M, N, K, "f16", "f16", stages=s) for s in (1, 2, 4, 6)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    check(outs[0], a, b, r, "f16", "f16", what="stages")


def test_backproj_workload_sampled():
    w = gemm_inputs.WORKLOADS["swin4k_backproj_f16"]
    a, b, r = w.a_bits(), w.b_bits(), w.r_bits()
    got = run_residual(a, b, r, w.M, w.N, w.K, w.in_dtype, w.out_dtype, w.epilogue)
    rng = np.random.default_rng(w.seed)
    rows = np.concatenate([rng.integers(0, w.M, 8192), np.repeat(np.arange(w.M - 130, w.M), w.N)])
    cols = np.concatenate([rng.integers(0, w.N, 8192), np.tile(np.arange(w.N), 130)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, "f16", "f16", R_bits=r, r_dtype="f16")
    g = decode_np(got[rows, cols], "f16")
    rr = decode_np(ref, "f16")
    tol = oracle.tolerance(S, rr, "f16", added=np.abs(decode_np(r[rows, cols], "f16")))
    assert np.all(np.abs(g - rr) <= tol)


@pytest.mark.parametrize("out_dt", ["f16", "f32"])
def test_residual_wide_tiles_bit_identical(out_dt):
    """The residual through every paired form: 256 x 256 tiles (mode 3) and
    256 x 512 tiles of two accumulators (mode 6), in place and not, give the
    single-CTA bits."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    from parity_util import torch_dtype
    M, N, K = 1130, 1304, 520
    a, b = seeded_case(M, N, K, "f16", seed=61)
    r = _rbits(M, N, out_dt, seed=62)
    dev = torch.device("cuda")
    A = to_device_bits(a, "f16", dev)
    B = to_device_bits(b, "f16", dev)
    outs = {}
    for name, cfg in (("single", {"block_n": 256, "mode": 1}), ("pair", {"block_n": 256, "mode": 3}),
                      ("wide", {"block_n": 512, "mode": 6})):
        R = to_device_bits(r, out_dt, dev)
        C = torch.empty((M, N), dtype=torch_dtype(out_dt), device=dev)
        sg.stage_gemm(A, B, epilogue="relu", out=C, residual=R, config=cfg)
        outs[name] = from_device_bits(C, out_dt)
        sg.stage_gemm(A, B, epilogue="relu", out=R, residual=R, config=cfg)   # in place
        outs[name + " in place"] = from_device_bits(R, out_dt)
        assert sg.device_status() == 0
    for k, o in outs.items():
        assert np.array_equal(o, outs["single"]), k
    check(outs["wide"], a, b, r, "f16", out_dt, "relu", what="residual wide")
