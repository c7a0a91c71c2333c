"""CUDA graphs instead of a tracing compiler: after a warm-up call (which
does the per-device set-up: device attributes, the status word, kernel
attributes), stage_gemm calls are plain stream work -- tensor maps and
parameters travel in the kernel's arguments -- so a chain of them can be
captured once and replayed on new inputs written in place.  Replays must
give the same bits as eager calls."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_capture_and_replay_chain():
    import torch
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    dev = torch.device("cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    M, N, K = 2048, 1536, 1024
    A = torch.randn(M, K, device=dev, dtype=torch.bfloat16, generator=g)
    B = torch.randn(K, N, device=dev, dtype=torch.bfloat16, generator=g)
    W = torch.randn(N, 384, device=dev, dtype=torch.bfloat16, generator=g)
    bias = torch.randn(384, device=dev, generator=g)
    R = torch.randn(M, 384, device=dev, dtype=torch.bfloat16, generator=g)
    H = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
    Y = torch.empty(M, 384, device=dev, dtype=torch.bfloat16)
    Z = torch.empty(M, 384, device=dev, dtype=torch.bfloat16)

    def chain():
        sg.stage_gemm(A, B, epilogue="relu", out=H)                       # paired-MMA size
        sg.stage_gemm(H, W, epilogue="bias_relu", bias=bias, out=Y)        # resident-B size
        sg.stage_gemm(H, W, out=Z, residual=R)                             # residual

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()                                                            # warm-up: set-up happens here
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for it in range(3):
        A.copy_(torch.randn(M, K, device=dev, dtype=torch.bfloat16, generator=g))
        graph.replay()
        torch.cuda.synchronize()
        got = (H.clone(), Y.clone(), Z.clone())
        chain()                                                            # eager, same inputs
        torch.cuda.synchronize()
        for x, y in zip(got, (H, Y, Z)):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), it
    assert sg.device_status() == 0


def test_capture_with_copied_operands():
    """An A view whose pitch breaks the TMA rule and a C view with an odd
    pitch: under capture the 16-byte-pitch copies, the kernel and the copy
    out become graph nodes (the buffer from the capture's own pool), and
    replays give the bits of eager calls; C's padding keeps its values."""
    import torch
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as sg
    dev = torch.device("cuda")
    g = torch.Generator(device="cuda").manual_seed(6)
    M, N, K = 1000, 300, 200
    A_full = torch.randn(M, K + 3, device=dev, dtype=torch.float16, generator=g)
    A = A_full[:, :K]                                                  # pitch 203 halves
    B = torch.randn(K, N, device=dev, dtype=torch.float16, generator=g)
    C_full = torch.full((M, N + 1), 7.0, device=dev, dtype=torch.float16)
    C = C_full[:, :N]                                                  # pitch 301 halves

    def call():
        sg.stage_gemm(A, B, epilogue="relu", out=C)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for it in range(3):
        A_full.copy_(torch.randn(M, K + 3, device=dev, dtype=torch.float16, generator=g))
        graph.replay()
        torch.cuda.synchronize()
        got = C.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(got, C), f"replay {it}"
        assert bool((C_full[:, N] == 7.0).all())
    assert sg.device_status() == 0
