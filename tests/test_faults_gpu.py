"""Failure detection without a GPU fault: a copy that never happens makes
the MMA issuer's bounded wait run out; the kernel records the timeout,
every role drains its own work and exits (in the cluster modes both CTAs
of a pair meet at the final cluster barrier), the host reads
SG_ERR_TIMEOUT, and the context stays usable for the next, correct call."""
import numpy as np
import pytest

import oracle
from parity_util import compare, run_gpu, seeded_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [1, 3, 6])
def test_skipped_copy_times_out_and_context_survives(mode):
    import torch
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 1024, 512, 512
    a, b = seeded_case(M, N, K, "f16", seed=31)
    A = torch.from_numpy(a.view(np.int16)).cuda().view(torch.float16)
    B = torch.from_numpy(b.view(np.int16)).cuda().view(torch.float16)
    old = sg.get_wait_limit_ns()
    try:
        assert lib.sg_test_set_cluster(mode) == 0
        assert lib.sg_test_set_tile_n(256) == 0
        p = sg.plan(M, N, K, torch.float16, torch.float32)
        assert p["cluster_m"] == (1 if mode == 1 else 2) and p["pair_mma"] == (0 if mode == 1 else 1)
        assert p["mode"] == mode
        sg.set_wait_limit_ns(50_000_000)          # 50 ms
        lib.sg_test_set_skip_load(1)
        sg.stage_gemm(A, B)                       # the launch itself succeeds
        assert sg.device_status() == -8           # SG_ERR_TIMEOUT, reported asynchronously
        assert sg.device_status() == 0            # the record is cleared once read
    finally:
        lib.sg_test_set_skip_load(-1)
        sg.set_wait_limit_ns(old)
        lib.sg_test_set_cluster(0)
        lib.sg_test_set_tile_n(0)
    got = run_gpu(a, b, M, N, K, "f16", "f32")
    ref, _, S = oracle.gemm(a, b, "f16", "f32")
    compare(got, ref, S, "f32", f"after-timeout mode {mode}")


@pytest.mark.parametrize("coded", [False, True])
def test_resident_panel_timeout_and_context_survives(coded):
    """Modes 4 (resident B) and 5 (decoded panel): a skipped A copy (each CTA
    has at least two row tiles, so its second fill exists) makes the MMA
    issuer's wait run out; the CTA drains its copies (and, in mode 4, the
    resident B's), SG_ERR_TIMEOUT is read, and the next call is correct."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    lib = sg.load_library()
    M, N, K = 40000, 384, 96                     # 313 row tiles over 152 CTAs
    a, b = seeded_case(M, N, K, "f16", seed=32)
    A = torch.from_numpy(a.view(np.int16)).cuda().view(torch.float16)
    Bf = torch.from_numpy(b.view(np.int16)).cuda().view(torch.float16)
    rng = np.random.default_rng(33)
    q = rng.integers(-127, 128, (K, N), dtype=np.int16).astype(np.int8)
    Q = torch.from_numpy(q).cuda()
    S = torch.full((N,), 0.01, dtype=torch.float32, device="cuda")

    def call():
        return sg.stage_gemm_qb(A, Q, S) if coded else sg.stage_gemm(A, Bf)
    old = sg.get_wait_limit_ns()
    try:
        assert lib.sg_test_set_cluster(0 if coded else 4) == 0
        if not coded:
            assert sg.plan(M, N, K, torch.float16, torch.float32)["mode"] == 4
        sg.set_wait_limit_ns(50_000_000)          # 50 ms
        lib.sg_test_set_skip_load(1)
        call()
        assert sg.device_status() == -8
        assert sg.device_status() == 0
    finally:
        lib.sg_test_set_skip_load(-1)
        sg.set_wait_limit_ns(old)
        lib.sg_test_set_cluster(0)
    C = call()
    torch.cuda.synchronize()
    assert sg.device_status() == 0
    rows = np.arange(0, M, 97)
    got = C.view(torch.int32).cpu().numpy().view(np.uint32)[rows]
    if coded:
        ref, _, Sx = oracle.gemm_qb(np.ascontiguousarray(a[rows]), q, np.full(N, 0.01, np.float32), "f16", "f32")
    else:
        ref, _, Sx = oracle.gemm(np.ascontiguousarray(a[rows]), b, "f16", "f32")
    compare(got, ref, Sx, "f32", f"after-timeout {'mode 5' if coded else 'mode 4'}")
