"""Split tail: when the last wave of 256-column tiles would fill at most half
of the clusters, each of its tiles runs as two 128-column units.  Every
output element is still computed by one unit, summing the same products in
the same K order (gizml:tile, "tune": every configuration computes the same
result), so C must be bit-identical with the split on and off, in every
kernel mode, with ragged edges, epilogues and a residual."""
import numpy as np
import pytest

import oracle
from parity_util import compare, run_gpu, seeded_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()


def _plan(M, N, K, ind, outd):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    t = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}
    return sg.plan(M, N, K, t[ind], t[outd])


class _Hooks:
    """Forces a kernel mode and the 256-column tile; restores both."""

    def __init__(self, mode, split):
        import tensor_core_gemm_tma_gb300 as sg
        self.lib = sg.load_library()
        self.mode, self.split = mode, split

    def __enter__(self):
        assert self.lib.sg_test_set_cluster(self.mode) == 0
        assert self.lib.sg_test_set_tile_n(256) == 0
        assert self.lib.sg_test_set_tail_split(self.split) == 0
        return self

    def __exit__(self, *exc):
        self.lib.sg_test_set_cluster(0)
        self.lib.sg_test_set_tile_n(0)
        self.lib.sg_test_set_tail_split(1)
        return False


CASES = [
    # M, N, K, in, out, epilogue, mode
    (2500, 2300, 300, "f16", "f32", "none", 1),       # 20 x 9 tiles over 152 CTAs: 28 split, ragged M, N, K
    (2500, 2300, 300, "bf16", "bf16", "relu", 1),     # single CTAs, bf16 with ReLU: 28 split
    (2500, 2300, 300, "f16", "f16", "bias_relu", 3),  # paired MMA, 256-row tiles: 14 split
    (2560, 2048, 1024, "bf16", "f32", "none", 3),     # whole tiles: 10 x 8 = 80 over 76 clusters, 4 split
]


@pytest.mark.parametrize("M,N,K,ind,outd,epi,mode", CASES)
def test_split_equals_unsplit(M, N, K, ind, outd, epi, mode):
    a, b = seeded_case(M, N, K, ind, seed=60 + mode + K % 5, lda=-(-K // 8) * 8)
    bias = np.linspace(-1.0, 1.0, N).astype(np.float32) if epi == "bias_relu" else None
    outs = {}
    for split in (1, 0):
        with _Hooks(mode, split):
            p = _plan(M, N, K, ind, outd)
            assert p["mode"] == mode and p["block_n"] == 256
            cm = p["cluster_m"]
            tiles = p["tiles"]
            clusters = 152 // cm
            tail = tiles % clusters
            if split:
                assert 0 < 2 * tail <= clusters and p["tail_units"] == 2 * tail
                assert p["grid"] == clusters * cm
            else:
                assert p["tail_units"] == 0
            outs[split] = run_gpu(a, b, M, N, K, ind, outd, epi, bias)
    assert np.array_equal(outs[1], outs[0]), "the split tail changed C"
    rng = np.random.default_rng(M + K)
    rows = np.concatenate([rng.integers(0, M, 2500), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 2500), np.arange(N)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, ind, outd, epi, bias=bias, K=K)
    compare(outs[1][rows, cols], ref, S, outd, f"split tail, mode {mode}")


def test_split_with_residual():
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    M, N, K = 2500, 2300, 200
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    A = torch.randn((M, K), generator=g, device="cuda").half()
    B = torch.randn((K, N), generator=g, device="cuda").half()
    R = torch.randn((M, N), generator=g, device="cuda").half()
    outs = []
    for split in (1, 0):
        with _Hooks(3, split):
            assert (_plan(M, N, K, "f16", "f16")["tail_units"] > 0) == bool(split)
            outs.append(sg.stage_gemm(A, B, out_dtype=torch.float16, epilogue="relu", residual=R))
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_split_only_where_it_pays():
    """No split for a last wave over half the clusters, for FP8 operands in
    256-column tiles (a half tile would not be whole 128-column boxes per
    CTA), for 128-column tiles, or for the resident-B mode; 256 x 512 tiles
    (mode 6) split into 256-column halves."""
    p = _plan(8192, 8192, 8192, "bf16", "f32")             # 1024 tiles: 36 over 13 full waves of 76
    assert p["block_n"] == 256 and p["mode"] == 3 and p["tail_units"] == 72
    p = _plan(16384, 8192, 4096, "f16", "f16")              # 1024 wide tiles: 36 over 13 full waves
    assert p["block_n"] == 512 and p["mode"] == 6 and p["tail_units"] == 72
    assert _plan(8192, 8192, 8192, "bf16", "bf16")["tail_units"] == 0   # 512 wide tiles: 56 left
    assert _plan(4096, 4096, 4096, "f16", "f16")["tail_units"] == 56   # 256 tiles: 28 left
    assert _plan(8192, 8192, 8192, "e4m3", "bf16")["tail_units"] == 0
    assert _plan(40000, 384, 96, "f16", "f16")["tail_units"] == 0      # mode 4
    assert _plan(1000, 1000, 1000, "f16", "f32")["tail_units"] == 0    # one wave
    assert _plan(8192, 8192, 256, "f16", "f16")["tail_units"] == 0     # 128-column tiles (short K)


def test_full_size_square8192_split_sampled():
    """The 8192^3 bf16 product in paired 256 x 256 tiles (split tail) on the
    last rows and columns, where the half-width units land, against the
    oracle."""
    import gemm_inputs
    w = gemm_inputs.WORKLOADS["square8192_bf16"]
    a, b = w.a_bits(), w.b_bits()
    with _Hooks(3, 1):
        assert _plan(w.M, w.N, w.K, "bf16", "bf16")["tail_units"] > 0
        got = run_gpu(a, b, w.M, w.N, w.K, "bf16", "bf16")
    rng = np.random.default_rng(11)
    rows = np.concatenate([rng.integers(w.M - 1024, w.M, 2000), rng.integers(0, w.M, 500)])
    cols = np.concatenate([rng.integers(w.N - 2048, w.N, 2000), rng.integers(0, w.N, 500)])
    ref, _, S = oracle.gemm_at(a, b, rows, cols, "bf16", "bf16")
    compare(got[rows, cols], ref, S, "bf16", "8192 split tail")
