"""Pins for the CPU oracle, against things other than itself: values worked
by hand from the IEEE 754 / bfloat16 bit layouts and from the definition of
the matrix product (tests/golden), library routines (numpy's binary16 and
binary32 conversions, numpy integer and float64 matrix products, torch's
bfloat16 cast on ties it rounds exactly), closed forms (identity,
permutation, rank-1, epilogue identities) and invariants (zero-fill, empty K,
thread-count independence).  CPU only."""
import os

import numpy as np
import pytest

import gemm_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ formats

def _read_formats():
    rows = []
    with open(os.path.join(GOLDEN, "float_formats.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            dt, bits, mant, e = line.split()
            rows.append((dt, int(bits, 16), int(mant), int(e)))
    return rows


def test_decode_golden(oracle_mod):
    rows = _read_formats()
    assert len(rows) >= 20
    for dt, bits, mant, e in rows:
        arr = np.array([bits], dtype={"f32": np.uint32, "e4m3": np.uint8}.get(dt, np.uint16))
        got = oracle_mod.decode(arr, dt)[0]
        want = float(np.ldexp(float(mant), e))
        assert got == want, (dt, hex(bits), got, want)
        if mant == 0:
            assert np.signbit(got) == bool(bits >> (31 if dt == "f32" else 15))


def test_encode_golden_roundtrip(oracle_mod):
    for dt, bits, mant, e in _read_formats():
        if dt == "e4m3":
            continue  # an operand type only: the oracle never encodes it
        got = oracle_mod.encode(np.array([np.ldexp(float(mant), e)]), dt)[0]
        assert int(got) == bits, (dt, hex(bits), hex(int(got)))


def test_decode_all_fp16_vs_numpy(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_all_bf16_vs_float32_upper_half(oracle_mod):
    # bfloat16 is the upper half of a binary32 pattern.
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.decode(bits, "bf16")
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_fp32_vs_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    bits[:6] = [0, 0x80000000, 1, 0x7F800000, 0xFF800000, 0x7FC00000]
    ours = oracle_mod.decode(bits, "f32")
    ref = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _fp16_midpoints():
    # all finite positive fp16 values, and the midpoint between neighbours
    v = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2.0          # exact in fp64
    return v, mids


def test_encode_fp16_vs_numpy_rne(oracle_mod):
    v, mids = _fp16_midpoints()
    rng = np.random.default_rng(11)
    x = np.concatenate([
        v, -v, mids, -mids,
        mids + 1e-12 * np.abs(mids), mids - 1e-12 * np.abs(mids),
        rng.normal(0, 1, 50000), rng.normal(0, 3e4, 50000), rng.normal(0, 1e-6, 50000),
        [65504.0, 65519.99, 65520.0, 65536.0, 1e10, -65520.0, np.inf, -np.inf, 0.0, -0.0, 2.0 ** -25,
         3 * 2.0 ** -26],
    ])
    ours = oracle_mod.encode(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_fp16_ties_go_to_even(oracle_mod):
    # 1 + 2^-11 lies halfway between 1 (even) and 1 + 2^-10 (odd)
    assert oracle_mod.encode(np.array([1 + 2.0 ** -11]), "f16")[0] == 0x3C00
    # 1 + 3 * 2^-11 lies halfway between 1 + 2^-10 (odd) and 1 + 2^-9 (even)
    assert oracle_mod.encode(np.array([1 + 3 * 2.0 ** -11]), "f16")[0] == 0x3C02
    # 65520 is halfway between 65504 (odd) and 65536 (overflow): infinity
    assert oracle_mod.encode(np.array([65520.0]), "f16")[0] == 0x7C00
    # half of the smallest subnormal rounds to 0 (even); 3/2 of it to 2 ulps
    assert oracle_mod.encode(np.array([2.0 ** -25]), "f16")[0] == 0x0000
    assert oracle_mod.encode(np.array([3 * 2.0 ** -25]), "f16")[0] == 0x0002


def test_encode_fp32_vs_numpy(oracle_mod):
    rng = np.random.default_rng(3)
    f = rng.integers(0, 0x7F800000, size=100000, dtype=np.int64).astype(np.uint32).view(np.float32)
    f64 = f.astype(np.float64)
    nxt = np.nextafter(f, np.float32(np.inf)).astype(np.float64)
    mids = (f64 + nxt) / 2.0
    x = np.concatenate([f64, -f64, mids, -mids, rng.normal(0, 1, 100000),
                        np.ldexp(rng.normal(0, 1, 20000), -140), [3.5e38, 3.4028235677973366e38, 1e39]])
    ours = oracle_mod.encode(x, "f32")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).view(np.uint32)
    assert np.array_equal(ours, ref)


def test_encode_bf16_vs_torch_on_float32_inputs(oracle_mod):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    # float32 inputs, so torch's float32 -> bfloat16 cast rounds them exactly once
    f = rng.integers(0, 0x7F7F0000, size=200000, dtype=np.int64).astype(np.uint32)
    ties = (f & np.uint32(0xFFFF0000)) | np.uint32(0x8000)          # exact midpoints
    x = np.concatenate([f.view(np.float32), ties.view(np.float32)]).astype(np.float64)
    x = np.concatenate([x, -x])
    ours = oracle_mod.encode(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_bf16_overflow_and_subnormal(oracle_mod):
    big = np.ldexp(255.5, 120)             # halfway between max finite (odd) and 2^128
    assert oracle_mod.encode(np.array([big]), "bf16")[0] == 0x7F80
    assert oracle_mod.encode(np.array([np.ldexp(255.49, 120)]), "bf16")[0] == 0x7F7F
    assert oracle_mod.encode(np.array([np.ldexp(1.0, -134)]), "bf16")[0] == 0x0000   # tie -> even 0
    assert oracle_mod.encode(np.array([np.ldexp(3.0, -134)]), "bf16")[0] == 0x0002   # tie -> even 2
    assert oracle_mod.encode(np.array([np.nan]), "bf16")[0] & 0x7FFF > 0x7F80


# ------------------------------------------------------------ products

def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _read_products():
    cases = []
    with open(os.path.join(GOLDEN, "small_products.txt")) as f:
        lines = [ln.split("#")[0].strip() for ln in f]
    lines = [ln for ln in lines if ln]
    i = 0
    while i < len(lines):
        _, name, M, N, K, epi = lines[i].split()
        M, N, K = int(M), int(N), int(K)
        i += 1
        A = np.array([[float(t) for t in lines[i + r].split()] for r in range(M)])
        i += M
        B = np.array([[float(t) for t in lines[i + r].split()] for r in range(K)])
        i += K
        bias = None if lines[i] == "-" else np.array([float(t) for t in lines[i].split()], dtype=np.float32)
        i += 1
        C = np.array([[float(t) for t in lines[i + r].split()] for r in range(M)])
        i += M
        cases.append((name, A, B, bias, epi, C))
    return cases


def test_small_products_golden(oracle_mod):
    cases = _read_products()
    assert len(cases) == 5
    torch = pytest.importorskip("torch")
    for name, A, B, bias, epi, C in cases:
        for out in ("f32", "f16", "bf16"):
            Cb, exact, _ = oracle_mod.gemm(_f16(A), _f16(B), "f16", out, epi, bias)
            assert np.array_equal(exact, C), name
            # the golden values are exact in binary32; round them with library casts
            if out == "f32":
                want = C.astype(np.float32).view(np.uint32)
            elif out == "f16":
                want = C.astype(np.float16).view(np.uint16)
            else:
                want = torch.from_numpy(C.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
                want = want.view(np.uint16)
            assert np.array_equal(Cb, want), (name, out)
    # 154.5 is a bfloat16 tie (9 significant bits): to even, 154
    Cb, _, _ = oracle_mod.gemm(_f16(cases[2][1]), _f16(cases[2][2]), "f16", "bf16", "bias_relu", cases[2][3])
    assert oracle_mod.decode(Cb, "bf16")[1, 1] == 154.0


def test_identity_exact(oracle_mod):
    rng = np.random.default_rng(1)
    for dt in ("f16", "bf16"):
        K = 77
        A = gemm_inputs.to_storage_bits(rng.normal(0, 10, (50, K)), dt)
        I = gemm_inputs.to_storage_bits(np.eye(K), dt)
        C, exact, _ = oracle_mod.gemm(A, I, dt, "f32")
        assert np.array_equal(exact, oracle_mod.decode(A, dt))
        assert np.array_equal(C.view(np.float32).astype(np.float64), oracle_mod.decode(A, dt))
        B = gemm_inputs.to_storage_bits(rng.normal(0, 10, (K, 31)), dt)
        C2, exact2, _ = oracle_mod.gemm(I, B, dt, dt)
        assert np.array_equal(C2, B)       # a 16-bit value rounds to itself


def test_permutation_exact(oracle_mod):
    rng = np.random.default_rng(2)
    K, N = 40, 23
    perm = rng.permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0
    B = _f16(rng.uniform(-1, 1, (K, N)))
    C, exact, _ = oracle_mod.gemm(_f16(P), B, "f16", "f16")
    assert np.array_equal(C, B[perm])
    # and on the right: A . P permutes A's columns by the inverse permutation
    A = _f16(rng.uniform(-1, 1, (13, K)))
    C, _, _ = oracle_mod.gemm(A, _f16(P), "f16", "f16")
    inv = np.argsort(perm)
    assert np.array_equal(C, A[:, inv])


def test_rank1_closed_form(oracle_mod):
    rng = np.random.default_rng(4)
    M, N, K = 19, 33, 100
    u = rng.integers(-16, 17, M) / 8.0      # dyadic, exact in fp16
    w = rng.integers(-16, 17, N) / 4.0
    A = _f16(np.outer(u, np.ones(K)))
    B = _f16(np.outer(np.ones(K), w))
    _, exact, S = oracle_mod.gemm(A, B, "f16", "f32")
    assert np.array_equal(exact, K * np.outer(u, w))
    assert np.array_equal(S, K * np.abs(np.outer(u, w)))


def test_integer_inputs_bitwise_vs_int64_matmul(oracle_mod):
    rng = np.random.default_rng(6)
    for (M, N, K) in [(37, 29, 2048), (64, 64, 1), (5, 200, 333)]:
        Ai = rng.integers(-4, 5, (M, K))
        Bi = rng.integers(-4, 5, (K, N))
        ref = Ai @ Bi                          # exact integer product (numpy int64)
        for dt in ("f16", "bf16"):
            A = gemm_inputs.to_storage_bits(Ai.astype(np.float64), dt)
            B = gemm_inputs.to_storage_bits(Bi.astype(np.float64), dt)
            C, exact, S = oracle_mod.gemm(A, B, dt, "f32")
            assert np.array_equal(exact, ref.astype(np.float64))
            assert np.array_equal(C.view(np.float32), ref.astype(np.float32))
            assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 17, 3), (17, 1, 5), (3, 4, 17), (16, 16, 16), (17, 13, 11),
                                   (9, 2, 15), (7, 7, 1)])
def test_brute_force_tiny_vs_float64_matmul(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * 10000 + N * 100 + K)
    for dt in ("f16", "bf16"):
        A = gemm_inputs.to_storage_bits(rng.normal(0, 1, (M, K)), dt)
        B = gemm_inputs.to_storage_bits(rng.normal(0, 1, (K, N)), dt)
        Ad = oracle_mod.decode(A, dt)
        Bd = oracle_mod.decode(B, dt)
        # independent decode for fp16: numpy's binary16
        if dt == "f16":
            assert np.array_equal(Ad, A.view(np.float16).astype(np.float64))
        ref = Ad @ Bd
        _, exact, S = oracle_mod.gemm(A, B, dt, "f32")
        np.testing.assert_allclose(exact, ref, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(S, np.abs(Ad) @ np.abs(Bd), rtol=1e-13, atol=1e-13)


def test_ragged_1000_vs_float64_matmul(oracle_mod):
    w = gemm_inputs.WORKLOADS["ragged1000_f16"]
    A, B = w.a_bits(), w.b_bits()
    C, exact, S = oracle_mod.gemm(A, B, "f16", "f32")
    ref = A.view(np.float16).astype(np.float64) @ B.view(np.float16).astype(np.float64)
    np.testing.assert_allclose(exact, ref, rtol=1e-12, atol=1e-12)
    # the fp32 result is the RNE rounding of the fp64 value
    assert np.array_equal(C, exact.astype(np.float32).view(np.uint32))


def test_zero_fill_padding_and_canaries(oracle_mod):
    """Reading out of range = reading 0 (In.at); ld padding is never read;
    nothing outside M x N is written (Out.put)."""
    rng = np.random.default_rng(8)
    M, N, K = 45, 70, 83
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    C0, e0, _ = oracle_mod.gemm(A, B, "f16", "f32")
    # 1) zero-padded to tile multiples: the same values in the logical box
    Ap = np.zeros((128, 128), np.uint16)
    Ap[:M, :K] = A
    Bp = np.zeros((128, 128), np.uint16)
    Bp[:K, :N] = B
    C1, e1, _ = oracle_mod.gemm(Ap, Bp, "f16", "f32")
    assert np.array_equal(e1[:M, :N], e0)
    assert np.array_equal(C1[:M, :N], C0)
    assert np.all(e1[M:, :] == 0) and np.all(e1[:, N:] == 0)
    # 2) NaN in the ld padding of A and B is never read
    An = np.full((M, K + 9), 0x7E00, np.uint16)
    An[:, :K] = A
    Bn = np.full((K + 4, N + 6), 0x7E00, np.uint16)
    Bn[:K, :N] = B
    C2, e2, _ = oracle_mod.gemm(An, Bn, "f16", "f32", K=K, N=N)
    assert np.array_equal(e2, e0) and np.array_equal(C2, C0)
    # 3) C padding columns (ldc > N) keep their canary
    canary = np.full((M, N + 5), 0xDEADBEEF, np.uint32)
    C3, _, _ = oracle_mod.gemm(A, B, "f16", "f32", C_init=canary)
    assert np.all(C3[:, N:] == 0xDEADBEEF)
    assert np.array_equal(C3[:, :N], C0)


def test_epilogue_closed_forms(oracle_mod):
    rng = np.random.default_rng(9)
    M, N, K = 31, 41, 57
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    bias = rng.normal(0, 2, N).astype(np.float32)
    _, none, S = oracle_mod.gemm(A, B, "f16", "f32")
    _, relu, S2 = oracle_mod.gemm(A, B, "f16", "f32", "relu")
    assert np.array_equal(relu, np.maximum(none, 0.0))
    assert np.array_equal(S, S2)
    _, br, _ = oracle_mod.gemm(A, B, "f16", "f32", "bias_relu", bias)
    assert np.array_equal(br, np.maximum(none + bias.astype(np.float64), 0.0))
    # A = 0: relu(bias) in every row
    Z = np.zeros((M, K), np.uint16)
    Cb, ez, _ = oracle_mod.gemm(Z, B, "f16", "f16", "bias_relu", bias)
    assert np.array_equal(ez, np.tile(np.maximum(bias.astype(np.float64), 0), (M, 1)))
    assert np.array_equal(Cb, np.tile(np.maximum(bias, 0).astype(np.float16).view(np.uint16), (M, 1)))
    # relu never yields -0
    Cr, _, _ = oracle_mod.gemm(A, B, "f16", "f32", "relu")
    assert not np.any(Cr == 0x80000000)


def test_empty_k_returns_init(oracle_mod):
    """K = 0: an empty fold returns its init (zeros), then the epilogue."""
    M, N = 6, 9
    A = np.zeros((M, 0), np.uint16)
    B = np.zeros((0, N), np.uint16)
    bias = np.linspace(-2, 2, N).astype(np.float32)
    for epi, b in (("none", None), ("relu", None), ("bias_relu", bias)):
        C, exact, S = oracle_mod.gemm(A, B, "f16", "f32", epi, b)
        want = np.zeros((M, N)) if b is None else np.tile(np.maximum(b.astype(np.float64), 0), (M, 1))
        assert np.array_equal(exact, want)
        assert np.all(S == 0)


def test_gemm_at_matches_full(oracle_mod):
    rng = np.random.default_rng(10)
    M, N, K = 90, 75, 130
    for dt, out, epi in (("f16", "f32", "none"), ("bf16", "bf16", "relu"), ("f16", "f16", "bias_relu")):
        A = gemm_inputs.to_storage_bits(rng.normal(0, 1, (M, K)), dt)
        B = gemm_inputs.to_storage_bits(rng.normal(0, 1, (K, N)), dt)
        bias = rng.normal(0, 1, N).astype(np.float32) if epi == "bias_relu" else None
        C, exact, S = oracle_mod.gemm(A, B, dt, out, epi, bias)
        rows = rng.integers(0, M, 500)
        cols = rng.integers(0, N, 500)
        cb, ce, cs = oracle_mod.gemm_at(A, B, rows, cols, dt, out, epi, bias)
        assert np.array_equal(cb, C[rows, cols])
        assert np.array_equal(ce, exact[rows, cols])
        assert np.array_equal(cs, S[rows, cols])


def test_thread_count_independent(oracle_mod):
    w = gemm_inputs.WORKLOADS["square256_f16"]
    A, B = w.a_bits(), w.b_bits()
    r1 = oracle_mod.gemm(A, B, "f16", "f32", threads=1)
    r7 = oracle_mod.gemm(A, B, "f16", "f32", threads=7)
    for x, y in zip(r1, r7):
        assert np.array_equal(x, y)


def test_rejects_bad_arguments(oracle_mod):
    A = np.zeros((4, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.gemm(A, A, "f16", "f32", "bias_relu", None)
    with pytest.raises(ValueError):
        oracle_mod.gemm(A, A, "f16", "f32", "none", np.zeros(4, np.float32))


def test_tolerance_helpers(oracle_mod):
    assert oracle_mod.ulp(np.array([1.0]), "f16")[0] == 2.0 ** -10
    assert oracle_mod.ulp(np.array([1.5]), "bf16")[0] == 2.0 ** -7
    assert oracle_mod.ulp(np.array([0.0]), "f16")[0] == 2.0 ** -24
    assert oracle_mod.ulp(np.array([65504.0]), "f16")[0] == 32.0
    t = oracle_mod.tolerance(np.array([10.0]), np.array([2.0]), "f16")
    assert t[0] == pytest.approx(1e-2 + 1e-5 + 2.0 ** -9)


# ------------------------------------------------------------ residual

def _read_residual_products():
    cases = []
    with open(os.path.join(GOLDEN, "residual_products.txt")) as f:
        lines = [ln.split("#")[0].strip() for ln in f]
    lines = [ln for ln in lines if ln]
    i = 0
    while i < len(lines):
        _, name, M, N, K, epi = lines[i].split()
        M, N, K = int(M), int(N), int(K)
        i += 1
        rows = lambda n: np.array([[float(t) for t in lines[i + r].split()] for r in range(n)])
        A = rows(M); i += M
        B = rows(K); i += K
        bias = None if lines[i] == "-" else np.array([float(t) for t in lines[i].split()], dtype=np.float32)
        i += 1
        R = rows(M); i += M
        C = rows(M); i += M
        cases.append((name, A, B, bias, epi, R, C))
    return cases


def test_residual_golden(oracle_mod):
    cases = _read_residual_products()
    assert len(cases) == 3
    for name, A, B, bias, epi, R, C in cases:
        for rdt in ("f16", "f32"):
            Rb = R.astype(np.float16).view(np.uint16) if rdt == "f16" else R.astype(np.float32).view(np.uint32)
            Cb, exact, _ = oracle_mod.gemm(_f16(A), _f16(B), "f16", "f32", epi, bias, R_bits=Rb, r_dtype=rdt)
            assert np.array_equal(exact, C), (name, rdt, exact)
            assert np.array_equal(Cb, C.astype(np.float32).view(np.uint32)), name


def test_residual_zero_is_plain_product(oracle_mod):
    rng = np.random.default_rng(70)
    M, N, K = 33, 21, 40
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    C0, e0, S0 = oracle_mod.gemm(A, B, "f16", "f16", "relu")
    C1, e1, S1 = oracle_mod.gemm(A, B, "f16", "f16", "relu", R_bits=np.zeros((M, N), np.uint16), r_dtype="f16")
    assert np.array_equal(C0, C1) and np.array_equal(e0, e1) and np.array_equal(S0, S1)


def test_residual_adds_after_the_sum(oracle_mod):
    """exact(A, B, R) = exact(A, B) + R, bitwise in fp64 (the fold's init is
    added once to the finished sum), and the epilogue comes after it."""
    rng = np.random.default_rng(71)
    M, N, K = 29, 37, 50
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    R = rng.normal(0, 3, (M, N)).astype(np.float32)
    _, none, S = oracle_mod.gemm(A, B, "f16", "f32")
    _, er, Sr = oracle_mod.gemm(A, B, "f16", "f32", R_bits=R.view(np.uint32), r_dtype="f32")
    assert np.array_equal(er, none + R.astype(np.float64)) and np.array_equal(S, Sr)
    bias = rng.normal(0, 1, N).astype(np.float32)
    _, ebr, _ = oracle_mod.gemm(A, B, "f16", "f32", "bias_relu", bias, R_bits=R.view(np.uint32), r_dtype="f32")
    assert np.array_equal(ebr, np.maximum(none + R.astype(np.float64) + bias.astype(np.float64), 0.0))


def test_residual_with_zero_operand_and_empty_k(oracle_mod):
    rng = np.random.default_rng(72)
    M, N = 17, 23
    R = rng.normal(0, 10, (M, N)).astype(np.float16).view(np.uint16)
    for K in (0, 19):
        A = np.zeros((M, K), np.uint16)
        B = _f16(rng.normal(0, 1, (K, N)))
        C, exact, S = oracle_mod.gemm(A, B, "f16", "f16", R_bits=R, r_dtype="f16", K=K, N=N)
        assert np.array_equal(C, R)                # one rounding of an fp16 value is itself
        assert np.all(S == 0)


def test_residual_integer_exact(oracle_mod):
    rng = np.random.default_rng(73)
    M, N, K = 31, 17, 384
    Ai = rng.integers(-4, 5, (M, K))
    Bi = rng.integers(-4, 5, (K, N))
    Ri = rng.integers(-1000, 1001, (M, N))
    C, exact, _ = oracle_mod.gemm(_f16(Ai), _f16(Bi), "f16", "f32", R_bits=Ri.astype(np.float32).view(np.uint32),
                                  r_dtype="f32")
    assert np.array_equal(exact, (Ai @ Bi + Ri).astype(np.float64))


def test_residual_at_matches_full(oracle_mod):
    rng = np.random.default_rng(74)
    M, N, K = 60, 44, 70
    A = _f16(rng.normal(0, 1, (M, K)))
    B = _f16(rng.normal(0, 1, (K, N)))
    R = _f16(rng.normal(0, 1, (M, N + 5)))       # padded residual rows
    C, exact, S = oracle_mod.gemm(A, B, "f16", "bf16", "relu", R_bits=R, r_dtype="f16", N=N)
    rows = rng.integers(0, M, 300)
    cols = rng.integers(0, N, 300)
    cb, ce, cs = oracle_mod.gemm_at(A, B, rows, cols, "f16", "bf16", "relu", R_bits=R, r_dtype="f16", N=N)
    assert np.array_equal(cb, C[rows, cols]) and np.array_equal(ce, exact[rows, cols])


def test_tolerance_added_term(oracle_mod):
    t0 = oracle_mod.tolerance(np.array([0.0]), np.array([1.0]), "f32")
    t1 = oracle_mod.tolerance(np.array([0.0]), np.array([1.0]), "f32", added=np.array([2.0 ** 20]))
    assert t1[0] - t0[0] == pytest.approx(2.0 ** -3)


# ------------------------------------------------------------ FP8 E4M3

def test_decode_all_e4m3_vs_torch(oracle_mod):
    torch = pytest.importorskip("torch")
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ours = oracle_mod.decode(bits, "e4m3")
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _e4m3(x):
    return gemm_inputs.to_storage_bits(np.asarray(x, dtype=np.float64), "e4m3")


def test_e4m3_integer_inputs_exact(oracle_mod):
    rng = np.random.default_rng(90)
    M, N, K = 23, 31, 512
    Ai = rng.integers(-8, 9, (M, K))        # every integer in [-16, 16] is exact in E4M3
    Bi = rng.integers(-8, 9, (K, N))
    C, exact, S = oracle_mod.gemm(_e4m3(Ai), _e4m3(Bi), "e4m3", "f32")
    assert np.array_equal(exact, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 33), (17, 16, 64), (9, 40, 130)])
def test_e4m3_brute_force_vs_float64_matmul(oracle_mod, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = _e4m3(rng.normal(0, 2, (M, K)))
    B = _e4m3(rng.normal(0, 2, (K, N)))
    Ad, Bd = oracle_mod.decode(A, "e4m3"), oracle_mod.decode(B, "e4m3")
    _, exact, _ = oracle_mod.gemm(A, B, "e4m3", "f32")
    np.testing.assert_allclose(exact, Ad @ Bd, rtol=1e-13, atol=1e-13)


def test_e4m3_identity_exact(oracle_mod):
    rng = np.random.default_rng(91)
    A = _e4m3(rng.normal(0, 10, (20, 48)))
    C, exact, _ = oracle_mod.gemm(A, _e4m3(np.eye(48)), "e4m3", "f32")
    assert np.array_equal(exact, oracle_mod.decode(A, "e4m3"))
