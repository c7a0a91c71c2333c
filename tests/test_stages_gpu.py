"""Staging moves values and never rounds them (Tolk.Stage, module overview;
gizml:tile, "tune": every configuration computes the same result): C is
bit-identical for every ring depth, and repeated runs are bit-identical
(a race on a ring slot would show up as differing bits)."""
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


def _plan(M, N, K, ind, outd, stages=0):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    return sg.plan(M, N, K, t[ind], t[outd], stages=stages)


def test_stage_counts_bit_identical_bn128():
    w = gemm_inputs.WORKLOADS["ragged1000_f16"]
    a, b = w.a_bits(), w.b_bits()
    p = _plan(w.M, w.N, w.K, "f16", "f32")
    assert p["block_n"] == 128 and p["max_stages"] >= 4
    outs = {s: run_gpu(a, b, w.M, w.N, w.K, "f16", "f32", stages=s) for s in range(1, p["max_stages"] + 1)}
    outs[0] = run_gpu(a, b, w.M, w.N, w.K, "f16", "f32", stages=0)
    for s, o in outs.items():
        assert np.array_equal(o, outs[1]), f"stages={s} differs from stages=1"
    ref, _, S = oracle.gemm(a, b, "f16", "f32")
    compare(outs[1], ref, S, "f32", "stages")


def test_stage_counts_bit_identical_bn256():
    M, N, K = 2560, 2048, 520          # enough tiles for the 256-wide tile; ragged K
    a, b = seeded_case(M, N, K, "bf16", seed=21, dist=("uniform", -1.0, 1.0))
    p = _plan(M, N, K, "bf16", "bf16")
    assert p["block_n"] == 256 and p["max_stages"] >= 4  # the planner's own choice here
    outs = [run_gpu(a, b, M, N, K, "bf16", "bf16", stages=s) for s in (1, 2, 3, 4)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    rng = np.random.default_rng(3)
    rows = np.concatenate([rng.integers(0, M, 3000), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 3000), np.arange(N)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, "bf16", "bf16")
    compare(outs[0][rows, cols], ref, S, "bf16", "bn256")


def test_repeated_runs_bit_identical():
    M, N, K = 1536, 1280, 768
    a, b = seeded_case(M, N, K, "f16", seed=22)
    first = run_gpu(a, b, M, N, K, "f16", "f16", "relu")
    for _ in range(3):
        assert np.array_equal(run_gpu(a, b, M, N, K, "f16", "f16", "relu"), first)


def test_stage_count_rejected_when_too_deep():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    p = _plan(2560, 2048, 512, "bf16", "bf16")
    if p["max_stages"] >= 8:
        pytest.skip("every stage count fits")
    A = torch.zeros(2560, 512, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(512, 2048, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sg.SgError) as e:
        sg.stage_gemm(A, B, out_dtype=torch.bfloat16, stages=p["max_stages"] + 1)
    assert e.value.code == -3


def test_tile_widths_bit_identical():
    """gizml:tile, "tune": every configuration computes the same result.  The
    128-, 192- and 256-column tiles sum the same products in the same K
    order, so their outputs must agree bit for bit."""
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 1100, 1152, 300
    a, b = seeded_case(M, N, K, "f16", seed=23, lda=304)
    outs = {}
    try:
        for bn in (128, 192, 256):
            assert lib.sg_test_set_tile_n(bn) == 0
            assert _plan(M, N, K, "f16", "f16")["block_n"] == bn
            outs[bn] = run_gpu(a, b, M, N, K, "f16", "f16", "relu")
    finally:
        lib.sg_test_set_tile_n(0)
    assert np.array_equal(outs[128], outs[192]) and np.array_equal(outs[128], outs[256])
    ref, _, S = oracle.gemm(a, b, "f16", "f16", "relu", K=K)
    compare(outs[128], ref, S, "f16", "tile widths")


def test_stage_counts_bit_identical_bn192():
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 700, 576, 200
    a, b = seeded_case(M, N, K, "bf16", seed=24, lda=208)
    try:
        assert lib.sg_test_set_tile_n(192) == 0
        p = _plan(M, N, K, "bf16", "f32")
        assert p["block_n"] == 192 and p["max_stages"] >= 3
        outs = [run_gpu(a, b, M, N, K, "bf16", "f32", stages=s) for s in range(1, p["max_stages"] + 1)]
    finally:
        lib.sg_test_set_tile_n(0)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ref, _, S = oracle.gemm(a, b, "bf16", "f32", K=K)
    compare(outs[0], ref, S, "f32", "bn192")


def test_planner_tile_widths():
    """The planner's width choice counts whole waves of tiles: 2048^3 fills
    fewer SMs with 256-wide tiles than with 128-wide ones, but 128-wide tiles
    stage twice the operand bytes per product, so 256 (paired) wins; 8192^3
    with a long K loop takes the paired 256 x 512 tiles (mode 6), 4096^3 and
    an fp32 output keep the 256-column pairs; a 1000^3 problem fits in one
    wave either way and keeps 128; a short K loop keeps 128 for the
    epilogue's sake."""
    p = _plan(2048, 2048, 2048, "f16", "f16")
    assert p["block_n"] == 256 and p["pair_mma"] == 1
    p = _plan(8192, 8192, 8192, "bf16", "bf16")
    assert p["block_n"] == 512 and p["mode"] == 6 and p["pair_mma"] == 1
    p = _plan(4096, 4096, 4096, "f16", "f16")
    assert p["block_n"] == 256 and p["mode"] == 3
    p = _plan(8192, 8192, 8192, "bf16", "f32")
    assert p["block_n"] == 256 and p["mode"] == 3
    assert _plan(1000, 1000, 1000, "f16", "f16")["block_n"] == 128
    assert _plan(8192, 8192, 256, "f16", "f16")["block_n"] == 128


def test_paired_mma_small():
    """The paired MMA (two CTAs, one 256-row tile) on a small case: every
    row block pairing, a ragged K tail and an odd number of row blocks."""
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 300, 256, 200
    a, b = seeded_case(M, N, K, "f16", seed=26, lda=208)
    try:
        assert lib.sg_test_set_cluster(3) == 0
        p = _plan(M, N, K, "f16", "f32")
        assert p["pair_mma"] == 1 and p["cluster_m"] == 2
        got = run_gpu(a, b, M, N, K, "f16", "f32")
    finally:
        lib.sg_test_set_cluster(0)
    ref, _, S = oracle.gemm(a, b, "f16", "f32", K=K)
    compare(got, ref, S, "f32", "paired small")


@pytest.mark.parametrize("bn", [128, 256])
def test_cluster_modes_bit_identical(bn):
    """Computing 256-row tiles with the paired MMA (mode 3) changes only who
    copies and who issues: C must be bit-identical to the single-CTA path
    (mode 1), at every stage count, including an odd number of row blocks
    (the last cluster's second CTA owns rows wholly below M)."""
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    N, K = 1024, 640
    outs = {}
    try:
        assert lib.sg_test_set_tile_n(bn) == 0
        for m in (1000, 1130):          # 8 row blocks (ragged), 9 (odd)
            a, b = seeded_case(m, N, K, "bf16", seed=25 + m, dist=("uniform", -1.0, 1.0))
            for mode in (1, 3):
                assert lib.sg_test_set_cluster(mode) == 0
                p = _plan(m, N, K, "bf16", "bf16")
                assert p["block_n"] == bn and p["cluster_m"] == (1 if mode == 1 else 2)
                assert p["pair_mma"] == (1 if mode == 3 else 0)
                for st in sorted({1, 2, p["max_stages"]}):
                    outs[(m, mode, st)] = run_gpu(a, b, m, N, K, "bf16", "bf16", stages=st)
            rng = np.random.default_rng(m)
            rows = np.concatenate([rng.integers(0, m, 2000), np.full(N, m - 1)])
            cols = np.concatenate([rng.integers(0, N, 2000), np.arange(N)])
            ref, _, S = oracle.gemm_at(a, b, rows, cols, "bf16", "bf16")
            for mode in (1, 3):
                compare(outs[(m, mode, 1)][rows, cols], ref, S, "bf16", f"mode {mode} m={m}")
    finally:
        lib.sg_test_set_cluster(0)
        lib.sg_test_set_tile_n(0)
    for (m, mode, st), o in outs.items():
        assert np.array_equal(o, outs[(m, 1, 1)]), (m, mode, st)


@pytest.mark.parametrize("mode", [1, 3])
def test_paired_slots_odd_chunk_count(mode):
    """With 6 or 8 ring slots and both operands copied by TMA, slots are
    filled and consumed in pairs on one pair of barriers.  An odd number of
    K chunks leaves each tile's last pair half used, and the next tile's
    chunks start on the following pair; C must keep the single-slot bits
    (the same MMAs in the same K order) in every kernel mode."""
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 1300, 1100, 9 * 64 - 3                 # 9 K chunks, the last one ragged
    a, b = seeded_case(M, N, K, "f16", seed=27 + mode, lda=576)
    try:
        assert lib.sg_test_set_cluster(mode) == 0
        assert lib.sg_test_set_tile_n(128) == 0
        p = _plan(M, N, K, "f16", "f32")
        assert p["mode"] == mode and p["max_stages"] >= 6
        grouped = {s: _plan(M, N, K, "f16", "f32", stages=s)["ring_group"] for s in range(1, p["max_stages"] + 1)}
        assert grouped[6] == 2 and grouped[5] == 1 and grouped[4] == 1 and grouped[1] == 1
        outs = {s: run_gpu(a, b, M, N, K, "f16", "f32", stages=s) for s in (1, 5, 6)}
    finally:
        lib.sg_test_set_cluster(0)
        lib.sg_test_set_tile_n(0)
    assert np.array_equal(outs[6], outs[1]) and np.array_equal(outs[5], outs[1])
    rng = np.random.default_rng(mode)
    rows = np.concatenate([rng.integers(0, M, 2000), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 2000), np.arange(N)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, "f16", "f32", K=K)
    compare(outs[6][rows, cols], ref, S, "f32", f"paired slots, mode {mode}")


def test_paired_slots_only_with_tma_operands():
    """Element-load staging (an A pitch that TMA cannot take) and the
    resident-B mode keep one barrier pair per slot."""
    import tensor_core_gemm_tma_gb300 as sg
    assert _plan(4096, 4096, 4096, "bf16", "bf16")["ring_group"] == 2
    assert _plan(40000, 384, 96, "f16", "f16")["ring_group"] == 1      # mode 4
    lib = sg.load_library()
    M, N, K = 600, 500, 1000
    a, b = seeded_case(M, N, K, "f16", seed=31, lda=1001)               # 2002-byte rows: element loads
    try:
        assert lib.sg_test_set_tile_n(128) == 0                           # a 6-slot ring
        assert _plan(M, N, K, "f16", "f32")["max_stages"] >= 6
        out = run_gpu(a, b, M, N, K, "f16", "f32")
    finally:
        lib.sg_test_set_tile_n(0)
    ref, _, S = oracle.gemm(a, b, "f16", "f32", K=K)
    compare(out, ref, S, "f32", "element loads, 6 slots")


def _cfg_run(a, b, M, N, K, ind, outd, epi, cfg, bias=None):
    """run_gpu through sg_gemm_ex under the configuration `cfg`."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    from parity_util import from_device_bits, to_device_bits, torch_dtype
    dev = torch.device("cuda")
    A = to_device_bits(a, ind, dev)[:, :K]
    B = to_device_bits(b, ind, dev)[:, :N]
    C = torch.empty((M, N), dtype=torch_dtype(outd), device=dev)
    bias_d = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).to(dev)
    sg.stage_gemm(A, B, epilogue=epi, bias=bias_d, out=C, config=cfg)
    assert sg.device_status() == 0
    return from_device_bits(C, outd)


WIDE_CASES = [
    # M, N, K, in, out, epilogue (B pitches TMA-legal: the paired forms need TMA operands): odd row
    # blocks, N ragged inside a tile's second accumulator, ragged K
    (1130, 1304, 9 * 64 - 3, "bf16", "bf16", "none"),
    (1130, 1304, 9 * 64 - 3, "f16", "f32", "relu"),
    # 10 x 10 wide tiles over 76 clusters (the last column block 96 wide: its second accumulator wholly
    # past N); the last 24 tiles run as 48 half units (one accumulator each)
    (2500, 4704, 300, "f16", "f16", "bias_relu"),
]


@pytest.mark.parametrize("M,N,K,ind,outd,epi", WIDE_CASES)
def test_wide_tiles_bit_identical(M, N, K, ind, outd, epi):
    """Mode 6 (a CTA pair computes a 256 x 512 tile as two 256-column
    accumulators, each CTA staging A once for both) issues, for every output
    element, the same MMAs in the same K order as the paired 256 x 256 tiles
    (mode 3) and the single-CTA tiles (mode 1): C must be bit-identical at
    every ring depth, with the split tail on and off."""
    a, b = seeded_case(M, N, K, ind, seed=51, lda=(K + 7) // 8 * 8)
    bias = np.linspace(-2, 2, N).astype(np.float32) if epi == "bias_relu" else None
    p = _plan(M, N, K, ind, outd)
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    pw = sg.plan(M, N, K, t[ind], t[outd], epi, config={"block_n": 512, "mode": 6})
    assert pw["mode"] == 6 and pw["block_n"] == 512 and pw["pair_mma"] == 1 and pw["cluster_m"] == 2
    assert pw["max_stages"] == 4 and pw["ring_group"] == 1
    if M == 2500:
        assert pw["tail_units"] > 0
    ref = _cfg_run(a, b, M, N, K, ind, outd, epi, {"block_n": 256, "mode": 3}, bias)
    assert np.array_equal(_cfg_run(a, b, M, N, K, ind, outd, epi, {"block_n": 256, "mode": 1}, bias), ref)
    for s in (1, 2, 3, 4):
        got = _cfg_run(a, b, M, N, K, ind, outd, epi, {"block_n": 512, "mode": 6, "stages": s}, bias)
        assert np.array_equal(got, ref), f"mode 6, stages={s}"
    got = _cfg_run(a, b, M, N, K, ind, outd, epi, {"block_n": 512, "tail_split": -1}, bias)
    assert np.array_equal(got, ref), "mode 6 without the split tail"
    rng = np.random.default_rng(M)
    rows = np.concatenate([rng.integers(0, M, 3000), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 3000), np.arange(N)])
    r, _, S = oracle.gemm_at(a, b, rows, cols, ind, outd, epi, bias, K=K)
    compare(ref[rows, cols], r, S, outd, f"wide tiles {ind}->{outd} {epi}")
    assert p["block_m"] == 128
