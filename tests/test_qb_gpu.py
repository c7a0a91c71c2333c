"""Mode 5: an integer-coded B (int8 codes, one fp32 scale per column)
decoded once per CTA into the resident shared-memory panel and read back by
every row tile (Tolk.Stage, "Decoded panels on the host", taken on the GPU).
Parity with the oracle's gemm_qb on ragged and full-size shapes; with scale
1 the decoded panel must give exactly the bits of mode 4 on B = the codes as
16-bit values (the same MMAs in the same K order)."""
import numpy as np
import pytest

import oracle
from parity_util import compare, from_device_bits, repack, seeded_case, to_device_bits, torch_dtype

pytestmark = pytest.mark.gpu


def _codes(K, N, seed, ld=None):
    rng = np.random.default_rng(seed)
    q = rng.integers(-128, 128, (K, ld or N), dtype=np.int16).astype(np.int8)
    s = (rng.uniform(0.5, 2.0, N) / 127.0).astype(np.float32)
    return q, s


def _run(a_bits, q, s, M, N, K, in_dt, out_dt, epi="none", bias=None, ldc=None, canary=0):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    A = to_device_bits(a_bits, in_dt, "cuda")[:, :K] if K > 0 else torch.empty((M, 0), dtype=torch_dtype(in_dt),
                                                                                device="cuda")
    Q = torch.from_numpy(np.ascontiguousarray(q)).cuda()[:, :N] if K > 0 else torch.empty((0, N), dtype=torch.int8,
                                                                                            device="cuda")
    S = torch.from_numpy(s).cuda()
    ldc = ldc or N
    Cfull = to_device_bits(np.full((M, ldc), canary, dtype=np.uint32 if out_dt == "f32" else np.uint16), out_dt,
                           "cuda")
    b = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).cuda()
    sg.stage_gemm_qb(A, Q, S, epilogue=epi, bias=b, out=Cfull[:, :N])
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    return from_device_bits(Cfull, out_dt)


CASES = [
    # M, N, K, in, out, epilogue
    (1000, 384, 96, "f16", "f16", "bias_relu"),   # the projection's panel, ragged M
    (300, 200, 72, "bf16", "f32", "none"),         # ragged N (2 column blocks) and K (2nd chunk partial)
    (2048, 512, 128, "f16", "bf16", "relu"),       # the largest panel: 2 K chunks x 4 column blocks
    (50, 64, 16, "f16", "f32", "none"),            # one tile, one K step
    (700, 129, 65, "bf16", "bf16", "bias_relu"),   # one column and one K element past a block
]


@pytest.mark.parametrize("M,N,K,ind,outd,epi", CASES)
def test_parity_with_oracle(M, N, K, ind, outd, epi):
    # A's pitch padded (NaN, never read) to a whole number of 16 bytes: mode 5 stages A by TMA (an odd pitch
    # would be copied to one first)
    a, _ = seeded_case(M, 1, K, ind, seed=70 + M % 13, lda=-(-K // 8) * 8)
    q, s = _codes(K, N, seed=K + N)
    bias = np.linspace(-0.5, 0.5, N).astype(np.float32) if epi == "bias_relu" else None
    got = _run(a, q, s, M, N, K, ind, outd, epi, bias)
    ref, _, S = oracle.gemm_qb(a, q, s, ind, outd, epi, bias=bias, K=K)
    compare(got, ref, S, outd, f"qb {M}x{N}x{K}")


def test_padding_untouched_and_codes_pitch():
    """Codes with a row pitch > N (their padding never read: it holds codes
    that would change C) and a C view whose padding keeps its canary."""
    M, N, K = 400, 160, 100
    a, _ = seeded_case(M, 1, K, "f16", seed=75, lda=104)
    q, s = _codes(K, N, seed=76, ld=N + 24)
    q[:, N:] = 127
    got = _run(a, q, s, M, N, K, "f16", "f32", ldc=N + 8, canary=0x7FC00001)
    assert np.all(got[:, N:] == 0x7FC00001)
    ref, _, S = oracle.gemm_qb(a, q, s, "f16", "f32", K=K, N=N)
    compare(got[:, :N], ref, S, "f32", "qb pitches")


def test_scale_one_matches_mode4_bits():
    """Scale 1: the decoded panel holds exactly what mode 4 stages from B =
    fp16(codes), so C must have mode 4's bits."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 1500, 384, 96
    a, _ = seeded_case(M, 1, K, "f16", seed=77)
    q, _ = _codes(K, N, seed=78)
    one = np.ones(N, dtype=np.float32)
    got = _run(a, q, one, M, N, K, "f16", "f16", "relu")
    A = to_device_bits(a, "f16", "cuda")
    B = torch.from_numpy(q.astype(np.float16)).cuda()
    lib = sg.load_library()
    try:
        assert lib.sg_test_set_cluster(4) == 0
        assert sg.plan(M, N, K, torch.float16, torch.float16)["mode"] == 4
        C = sg.stage_gemm(A, B, out_dtype=torch.float16, epilogue="relu")
    finally:
        lib.sg_test_set_cluster(0)
    torch.cuda.synchronize()
    assert np.array_equal(got, from_device_bits(C, "f16"))


def test_scale_is_per_column():
    """Doubling one column's scale doubles exactly that column (fp32 out)."""
    M, N, K = 256, 256, 64
    a, _ = seeded_case(M, 1, K, "bf16", seed=79)
    q, s = _codes(K, N, seed=80)
    c1 = _run(a, q, s, M, N, K, "bf16", "f32").view(np.float32)
    s2 = s.copy()
    s2[37] *= 2
    c2 = _run(a, q, s2, M, N, K, "bf16", "f32").view(np.float32)
    assert np.array_equal(c2[:, 37], 2 * c1[:, 37])
    assert np.array_equal(np.delete(c2, 37, axis=1), np.delete(c1, 37, axis=1))


def test_k_zero_gives_relu_bias():
    M, N = 300, 200
    bias = np.linspace(-1.0, 1.0, N).astype(np.float32)
    s = np.ones(N, dtype=np.float32)
    got = _run(None, np.zeros((0, N), np.int8), s, M, N, 0, "f16", "f32", "bias_relu", bias)
    assert np.array_equal(got.view(np.float32), np.broadcast_to(np.maximum(bias, 0), (M, N)))


def test_full_size_projection_sampled():
    """The projection shape (M = 518400 tokens, K = 96, N = 384) with int8
    weights: sampled rows, including the last row tile, against the oracle."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    import gemm_inputs
    w = gemm_inputs.WORKLOADS["swin4k_proj_i8w"]
    M, N, K = w.M, w.N, w.K
    a, (q, s), bias = w.a_bits(), w.b_codes(), w.bias()
    got = _run(a, q, s, M, N, K, "f16", "f16", "bias_relu", bias)
    rng = np.random.default_rng(82)
    rows = np.unique(np.concatenate([rng.integers(0, M, 1500), np.arange(M - 128, M)]))
    ref, _, S = oracle.gemm_qb(np.ascontiguousarray(a[rows]), q, s, "f16", "f16", "bias_relu", bias=bias)
    compare(got[rows], ref, S, "f16", "qb full size")
    del got
    torch.cuda.empty_cache()
    assert sg.device_status() == 0


def test_panel_limits_and_types_rejected():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    A = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    S = torch.ones(600, dtype=torch.float32, device="cuda")
    Q = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    # A's pitch (100 halves) is not a whole number of 16 bytes: it is copied to a 16-byte pitch first and gives
    # the bits of a dense A; staged by element loads instead (the copy switched off) the decoded panel cannot
    # take it
    A_odd = torch.randn((256, 100), device="cuda").half()[:, :64]
    Qr = torch.randint(-8, 8, (64, 64), dtype=torch.int8, device="cuda")
    with repack(1):
        got = sg.stage_gemm_qb(A_odd, Qr, S[:64])
    assert torch.equal(got, sg.stage_gemm_qb(A_odd.contiguous(), Qr, S[:64]))
    with repack(0):
        with pytest.raises(sg.SgError) as e:
            sg.stage_gemm_qb(A_odd, Q, S[:64])
    assert e.value.code == -1
    for K, N in ((136, 128), (128, 520)):      # past 2 K chunks / 4 column blocks
        Q = torch.zeros((K, N), dtype=torch.int8, device="cuda")
        with pytest.raises(sg.SgError) as e:
            sg.stage_gemm_qb(A[:, :K], Q, S[:N])
        assert e.value.code == -1
    Q = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    with pytest.raises(sg.SgError) as e:
        sg.stage_gemm_qb(A[:, :64].to(torch.float8_e4m3fn), Q, S[:64])
    assert e.value.code == -2
