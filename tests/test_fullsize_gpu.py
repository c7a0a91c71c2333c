"""Full-size invariants at the workloads' own sizes and launch shapes.

* Staging moves values and never rounds them (Tolk.Stage, module overview),
  so the ring depth cannot change C: the 8192^3 bf16 product in the
  benchmark's launch shape (paired 256 x 512 tiles of two accumulators, 4
  slots, 6.7 waves) and in the paired 256 x 256 form (6 slots on 3 barrier
  pairs, a split last wave, 13.5 waves) must give the same bits at every
  depth; so must the skinny-K projection's resident-B kernel at 1, 2 and 3
  slots, and the 4096^3 ReLU product.  Many wraps of the ring over many
  tiles per CTA are exactly where a slot race would show.
* gizml:tile's fused example computes relu(A.B) over 128 x 128 output tiles,
  and "tune" says every configuration computes the same result: the 4096^3
  ReLU product with 128 x 128 tiles (one CTA per tile, or CTA pairs whose
  CTAs each own one 128 x 128 tile and share B) must match the oracle at
  every element and equal the planner's wider paired tiles bit for bit.

Bitwise comparisons run on the device (torch.equal); the oracle checks every
element where it finishes in seconds (4096^3) and sampled positions plus
whole edge rows and columns where it does not."""
import numpy as np
import pytest

import gemm_inputs
import oracle
from parity_util import compare, from_device_bits, to_device_bits

pytestmark = pytest.mark.gpu

TILE_128 = [{"block_n": 128, "mode": 1}, {"block_n": 128, "mode": 3}]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    sg.load_library()
    torch.cuda.set_device(0)
    yield


def _operands(w):
    import torch
    dev = torch.device("cuda")
    a, b, bias = w.a_bits(), w.b_bits(), w.bias()
    A = to_device_bits(a, w.in_dtype, dev)
    B = to_device_bits(b, w.in_dtype, dev)
    bias_d = None if bias is None else torch.from_numpy(bias.copy()).to(dev)
    return (a, b, bias), (A, B, bias_d)


def _run(w, dev_ops, stages=0, config=None):
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    A, B, bias = dev_ops
    C = torch.empty((w.M, w.N), dtype={"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[
        w.out_dtype], device=A.device)
    sg.stage_gemm(A, B, epilogue=w.epilogue, bias=bias, stages=stages, out=C, config=config)
    assert sg.device_status() == 0
    return C


def _plan(w, stages=0, config=None):
    import tensor_core_gemm_tma_gb300 as sg
    from parity_util import torch_dtype
    return sg.plan(w.M, w.N, w.K, torch_dtype(w.in_dtype), torch_dtype(w.out_dtype), w.epilogue, stages,
                   config=config)


def _sample(w, n_random, edge_rows=(), edge_cols=()):
    rng = np.random.default_rng(w.seed + 17)
    rows = [rng.integers(0, w.M, n_random)]
    cols = [rng.integers(0, w.N, n_random)]
    for r in edge_rows:
        rows.append(np.full(w.N, r))
        cols.append(np.arange(w.N))
    for c in edge_cols:
        rows.append(np.arange(w.M))
        cols.append(np.full(w.M, c))
    return np.concatenate(rows), np.concatenate(cols)


def _sampled_check(w, host_ops, C, rows, cols, what):
    a, b, bias = host_ops
    got = from_device_bits(C, w.out_dtype)[rows, cols]
    ref, _, S = oracle.gemm_at(a, b, rows, cols, w.in_dtype, w.out_dtype, w.epilogue, bias)
    compare(got, ref, S, w.out_dtype, what)


def test_square8192_bf16_stage_counts_bit_identical():
    import torch
    w = gemm_inputs.WORKLOADS["square8192_bf16"]
    host_ops, dev_ops = _operands(w)
    p = _plan(w)
    # the benchmark's launch shape: paired 256 x 512 tiles (mode 6), 4 slots
    assert p["pair_mma"] == 1 and p["block_n"] == 512 and p["mode"] == 6 and p["stages"] == 4
    ref = _run(w, dev_ops, stages=0)
    for s in (1, 2, 3):
        assert torch.equal(_run(w, dev_ops, stages=s), ref), f"stages={s} differs from the 4-slot ring"
    # paired 256 x 256 tiles: 6 slots in 3 barrier pairs, a split last wave
    pair = {"block_n": 256, "mode": 3}
    p3 = _plan(w, config=pair)
    assert p3["stages"] == 6 and p3["ring_group"] == 2 and p3["tail_units"] > 0
    for s in (0, 1, 2, 4):
        assert torch.equal(_run(w, dev_ops, config=dict(pair, stages=s)), ref), f"256x256, stages={s}"
    edge = (0,) + tuple(range(w.M - 256, w.M))
    rows, cols = _sample(w, 4096, edge_rows=edge, edge_cols=edge)
    _sampled_check(w, host_ops, ref, rows, cols, "square8192_bf16, 6 slots")


def test_swin4k_proj_f16_resident_b_stage_counts_bit_identical():
    import torch
    w = gemm_inputs.WORKLOADS["swin4k_proj_f16"]
    host_ops, dev_ops = _operands(w)
    p = _plan(w)
    assert p["mode"] == 4 and p["max_stages"] >= 3
    ref = _run(w, dev_ops, stages=0)
    for s in (1, 2, 3):
        assert _plan(w, s, config={"mode": 4})["mode"] == 4
        assert torch.equal(_run(w, dev_ops, config={"mode": 4, "stages": s}), ref), f"mode 4, stages={s}"
    # the single-CTA tiles (B re-read per tile) give the same bits too
    assert torch.equal(_run(w, dev_ops, config={"mode": 1, "block_n": 128}), ref)
    rows, cols = _sample(w, 8192, edge_rows=tuple(range(w.M - 130, w.M)) + (0, 1), edge_cols=(0, w.N - 1))
    _sampled_check(w, host_ops, ref, rows, cols, "swin4k_proj_f16, resident B")


def test_relu4096_f16_stage_counts_bit_identical():
    import torch
    w = gemm_inputs.WORKLOADS["relu4096_f16"]
    _, dev_ops = _operands(w)
    ref = _run(w, dev_ops)
    for s in (1, 2, 4):
        assert torch.equal(_run(w, dev_ops, stages=s), ref), f"stages={s}"


@pytest.fixture(scope="module")
def relu4096_oracle():
    w = gemm_inputs.WORKLOADS["relu4096_f16"]
    a, b = w.a_bits(), w.b_bits()
    ref, _, S = oracle.gemm(a, b, w.in_dtype, w.out_dtype, w.epilogue)
    return ref, S


@pytest.mark.parametrize("cfg", TILE_128, ids=["single_cta_128x128", "cta_pair_128x128_each"])
def test_relu4096_f16_128x128_tiles_full(cfg, relu4096_oracle):
    """The fused example's tiling at full size: every element against the
    oracle, and the same bits as the planner's (wider, paired) tiles, at the
    default depth and at 1, 2 and 4 slots."""
    import torch
    w = gemm_inputs.WORKLOADS["relu4096_f16"]
    _, dev_ops = _operands(w)
    p = _plan(w, config=cfg)
    assert p["block_n"] == 128 and p["mode"] == cfg["mode"] and p["block_m"] == 128
    assert p["pair_mma"] == (1 if cfg["mode"] == 3 else 0)
    planner = _run(w, dev_ops)
    assert _plan(w)["block_n"] > 128
    got = _run(w, dev_ops, config=cfg)
    ref, S = relu4096_oracle
    compare(from_device_bits(got, w.out_dtype), ref, S, w.out_dtype, f"relu4096 {cfg}")
    assert torch.equal(got, planner), f"{cfg} differs from the planner's tiles"
    for s in (1, 2, 4):
        assert torch.equal(_run(w, dev_ops, config=dict(cfg, stages=s)), planner), f"{cfg}, stages={s}"


def test_config_rejects_what_the_problem_cannot_take():
    """sg_gemm_ex honours a configuration exactly or refuses it: the paired
    MMA needs whole B boxes per CTA (not 192 columns, not 128 FP8 columns),
    the resident B needs a small B."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    A = torch.zeros((512, 512), dtype=torch.float16, device="cuda")
    B = torch.zeros((512, 512), dtype=torch.float16, device="cuda")
    for cfg in ({"block_n": 192, "mode": 3}, {"mode": 4}, {"block_n": 256, "mode": 4}, {"block_n": 256, "mode": 6},
                {"block_n": 512, "mode": 3}, {"block_n": 512, "mode": 1}):
        with pytest.raises(sg.SgError) as e:
            sg.stage_gemm(A, B, config=cfg)
        assert e.value.code == -9, cfg
        with pytest.raises(sg.SgError):
            sg.plan(512, 512, 512, torch.float16, torch.float32, config=cfg)
    A8 = torch.zeros((512, 512), dtype=torch.float8_e4m3fn, device="cuda")
    B8 = torch.zeros((512, 512), dtype=torch.float8_e4m3fn, device="cuda")
    for cfg in ({"block_n": 128, "mode": 3}, {"block_n": 192}):
        with pytest.raises(sg.SgError) as e:
            sg.stage_gemm(A8, B8, out_dtype=torch.bfloat16, config=cfg)
        assert e.value.code == -9, cfg
    torch.cuda.synchronize()
    assert sg.device_status() == 0


@pytest.mark.parametrize("name", ["square8192_bf16", "square8192_e4m3", "relu4096_f16"])
def test_wide_tiles_full_size_bit_identical(name):
    """256 x 512 paired tiles of two accumulators (mode 6) at the workloads'
    full sizes, at the deepest ring and at 2 slots: the bits of the paired
    256 x 256 tiles."""
    import torch
    w = gemm_inputs.WORKLOADS[name]
    host_ops, dev_ops = _operands(w)
    ref = _run(w, dev_ops, config={"block_n": 256, "mode": 3})
    assert _plan(w, config={"block_n": 512})["mode"] == 6
    for s in (0, 2):
        assert torch.equal(_run(w, dev_ops, config={"block_n": 512, "mode": 6, "stages": s}), ref), f"stages={s}"
    if name == "square8192_bf16":
        edge = (0,) + tuple(range(w.M - 256, w.M))
        rows, cols = _sample(w, 4096, edge_rows=edge, edge_cols=edge)
        _sampled_check(w, host_ops, ref, rows, cols, name)
