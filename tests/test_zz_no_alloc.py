"""sg_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(allocator callbacks, runtimes that own every device allocation, processes
that must not grow their device footprint).  Its only scratch, the device
status word, lives in a static device array instead of library-allocated
memory.  Called through the C ABI, its output must match the regular entry
point's within the parity tolerance, on two calls in a row.  This file is
collected last so that a failure here cannot hide the other tests."""
import ctypes

import numpy as np
import pytest

import oracle
from parity_util import compare, from_device_bits, run_gpu, seeded_case, to_device_bits

pytestmark = pytest.mark.gpu


def _noalloc_lib():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    sg.load_library()
    lib = ctypes.CDLL(sg.LIB_PATH)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.sg_gemm_noalloc.restype = i32
    lib.sg_gemm_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, vp, i32, vp]
    lib.sg_gemm_noalloc_status.restype = i32
    lib.sg_gemm_noalloc_status.argtypes = [vp]
    return lib


@pytest.mark.parametrize("M,N,K,in_dt,out_dt,epi", [
    (1000, 1000, 1000, "f16", "f32", "none"),
    (2560, 2048, 520, "bf16", "bf16", "relu"),
])
def test_noalloc_matches_sg_gemm_twice(M, N, K, in_dt, out_dt, epi):
    import torch
    lib = _noalloc_lib()
    a, b = seeded_case(M, N, K, in_dt, seed=41, lda=(K + 7) // 8 * 8)
    bias = None
    expected = run_gpu(a, b, M, N, K, in_dt, out_dt, epi, bias)   # the existing entry point
    ref, _, S = oracle.gemm(a, b, in_dt, out_dt, epi, bias, K=K)
    dev = torch.device("cuda")
    A = to_device_bits(a, in_dt, dev)
    B = to_device_bits(b, in_dt, dev)
    codes = {"f32": 0, "f16": 1, "bf16": 2}
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call in range(2):
        C = to_device_bits(np.zeros((M, N), np.uint32 if out_dt == "f32" else np.uint16), out_dt, dev)
        rc = lib.sg_gemm_noalloc(M, N, K, A.data_ptr(), a.shape[1], B.data_ptr(), b.shape[1], C.data_ptr(), N,
                                 codes[in_dt], codes[out_dt], {"none": 0, "relu": 1, "bias_relu": 2}[epi], None, 0,
                                 stream)
        assert rc == 0, f"call {call}: rc {rc}"
        assert lib.sg_gemm_noalloc_status(stream) == 0
        got = from_device_bits(C, out_dt)
        compare(got, expected, S, out_dt, f"noalloc vs sg_gemm, call {call}")
        compare(got, ref, S, out_dt, f"noalloc vs oracle, call {call}")
        # the same plan and kernel as sg_gemm: the same bits, not only within tolerance
        assert np.array_equal(got, expected), f"call {call}: bits differ from sg_gemm"


def test_noalloc_status_records_a_timeout_and_is_cleared():
    """The status word in the static array records a device-side wait that
    gave up (a K chunk whose copy a test hook skips, with a 50 ms limit),
    and the next call clears it before its kernel runs: a clean call then
    reports 0 and matches the oracle."""
    import torch
    import tensor_core_gemm_tma_gb300 as sg
    lib = _noalloc_lib()
    M, N, K = 1024, 512, 512
    a, b = seeded_case(M, N, K, "f16", seed=43)
    dev = torch.device("cuda")
    A = to_device_bits(a, "f16", dev)
    B = to_device_bits(b, "f16", dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    hooks = sg.load_library()
    old = sg.get_wait_limit_ns()
    try:
        sg.set_wait_limit_ns(50_000_000)
        hooks.sg_test_set_skip_load(1)
        assert lib.sg_gemm_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, 1, 0, 0, None, 0,
                                   stream) == 0
        assert lib.sg_gemm_noalloc_status(stream) == -8      # SG_ERR_TIMEOUT, from the static array
    finally:
        hooks.sg_test_set_skip_load(-1)
        sg.set_wait_limit_ns(old)
    assert lib.sg_gemm_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, 1, 0, 0, None, 0,
                               stream) == 0
    assert lib.sg_gemm_noalloc_status(stream) == 0
    ref, _, S = oracle.gemm(a, b, "f16", "f32")
    compare(from_device_bits(C, "f32"), ref, S, "f32", "noalloc after a timeout")


def test_noalloc_rejects_like_sg_gemm():
    """Host-side checks are sg_gemm's.  Only arguments that are rejected on
    the host before any CUDA call are used here (the pointers are not real
    device memory): an A that is not aligned to its 2-byte elements, an
    unknown epilogue, a negative size."""
    lib = _noalloc_lib()
    assert lib.sg_gemm_noalloc(64, 64, 64, 0x10001, 64, 0x20000, 64, 0x400000, 64, 1, 0, 0, None, 0, None) == -5
    assert lib.sg_gemm_noalloc(64, 64, 64, 0x10000, 64, 0x20000, 64, 0x400000, 64, 1, 0, 9, None, 0, None) == -2
    assert lib.sg_gemm_noalloc(-1, 64, 64, 0x10000, 64, 0x20000, 64, 0x400000, 64, 1, 0, 0, None, 0, None) == -1
    # a C off its 4-byte fp32 elements
    assert lib.sg_gemm_noalloc(64, 64, 64, 0x10000, 64, 0x20000, 64, 0x400002, 64, 1, 0, 0, None, 0, None) == -5
