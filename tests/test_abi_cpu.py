"""The C ABI library without a GPU: it builds, loads, exports every function
the headers declare, and rejects bad arguments on the host before any CUDA
call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("stage_gemm.h", "stage_gemm_testing.h")]


@pytest.fixture(scope="module")
def sg():
    from tensor_core_gemm_tma_gb300 import _build
    _build.build()
    import tensor_core_gemm_tma_gb300 as mod
    mod.load_library()
    return mod


def _declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(sg_[a-z_0-9]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_headers_declare_the_api():
    names = _declared_functions()
    for n in ("sg_gemm", "sg_plan", "sg_device_status", "sg_strerror", "sg_version", "sg_set_wait_limit_ns",
              "sg_get_wait_limit_ns", "sg_test_set_skip_load"):
        assert n in names


def test_library_exports_every_declared_symbol(sg):
    lib = ctypes.CDLL(sg.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_version_and_strerror(sg):
    assert sg.version() == 120
    for code in range(0, -10, -1):
        txt = sg.strerror(code)
        assert txt and txt != "unknown error code"
    assert sg.strerror(-99) == "unknown error code"


def test_header_codes_match_binding():
    text = open(HEADERS[0]).read()
    codes = dict(re.findall(r"(SG_ERR_[A-Z]+)\s*=\s*(-\d+)", text))
    import tensor_core_gemm_tma_gb300 as mod
    for v, name in mod.ERRORS.items():
        assert int(codes[name]) == v
    assert re.search(r"SG_F16 = 1", text) and re.search(r"SG_BF16 = 2", text) and re.search(r"SG_F32 = 0", text)
    assert re.search(r"#define SG_MAX_STAGES 8", text)


# Pointers below are not device memory: every call here must be rejected on
# the host before any CUDA call.  So that a change of the rules can never
# turn one into a launch on these addresses, the calls only run where no GPU
# is present (this is the CPU suite).
def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


needs_no_gpu = pytest.mark.skipif(not _no_gpu(), reason="fake-pointer rejection tests run only without a GPU")

P16 = 0x10000      # 16-byte aligned fake addresses
P16B = 0x900000
PC = 0x4000000


def call(sg, M=64, N=64, K=64, A=P16, lda=None, B=P16B, ldb=None, C=PC, ldc=None, ind=1, outd=0, epi=0,
         bias=None, stages=0):
    return sg.gemm_raw(M, N, K, A, K if lda is None else lda, B, N if ldb is None else ldb, C,
                       N if ldc is None else ldc, ind, outd, epi, bias, stages, None)


@needs_no_gpu
def test_empty_problem_is_a_noop(sg):
    assert call(sg, M=0) == 0
    assert call(sg, N=0) == 0
    assert call(sg, M=0, N=0, K=0, A=None, B=None, C=None) == 0


@needs_no_gpu
def test_rejects_bad_sizes_and_pitches(sg):
    assert call(sg, M=-1) == -1
    assert call(sg, K=-5) == -1
    assert call(sg, lda=63) == -1
    assert call(sg, ldb=10) == -1
    assert call(sg, ldc=63) == -1
    assert call(sg, M=1 << 31) == -1
    assert call(sg, A=None) == -1
    assert call(sg, C=None) == -1


@needs_no_gpu
def test_rejects_bad_types_and_epilogues(sg):
    assert call(sg, ind=0) == -2           # fp32 operands are not supported
    assert call(sg, outd=7) == -2
    assert call(sg, epi=3) == -2
    assert call(sg, epi=2, bias=None) == -1
    assert call(sg, epi=0, bias=0x7000000) == -1


@needs_no_gpu
def test_rejects_bad_stage_counts(sg):
    assert call(sg, stages=-1) == -3
    assert call(sg, stages=9) == -3


@needs_no_gpu
def test_rejects_aliasing(sg):
    # C overlapping A, B or bias (Tolk.Uniform precondition: written
    # parameters do not overlap the others)
    assert call(sg, C=P16 + 64) == -4
    assert call(sg, C=P16B) == -4
    assert call(sg, epi=2, bias=PC + 128) == -4


@needs_no_gpu
def test_rejects_element_misalignment(sg):
    # 16-bit operands must sit on 2-byte boundaries (coarser misalignment is
    # staged by element loads and needs a GPU, so it is tested there)
    assert call(sg, A=P16 + 1) == -5
    assert call(sg, B=P16B + 3) == -5


@needs_no_gpu
def test_rejects_c_and_bias_misalignment(sg):
    # C off its own elements (4 bytes for fp32, 2 for fp16) and a bias off
    # 4 bytes would make the masked element stores / scalar bias loads fault
    # on the GPU: rejected on the host
    assert call(sg, C=PC + 2, outd=0) == -5
    assert call(sg, C=PC + 1, outd=1) == -5
    assert call(sg, epi=2, bias=0x7000002) == -5


@needs_no_gpu
def test_config_entry_rejects_bad_configs(sg):
    """sg_gemm_ex checks its configuration on the host before anything else:
    unknown tile widths, modes (2 is not a mode), raster groups and tail
    settings are SG_ERR_CONFIG, an out-of-range depth SG_ERR_STAGES; with a
    valid configuration the ordinary argument checks follow."""
    lib = sg.load_library()

    def ex(cfg, M=64, C=PC, lda=64, outd=0):
        return lib.sg_gemm_ex(M, 64, 64, P16, lda, P16B, 64, None, 0, C, 64, 1, outd, 0, None,
                              ctypes.byref(sg.Config(**cfg)), None)

    assert ex({"block_n": 64}) == -9
    assert ex({"block_n": 320}) == -9
    assert ex({"mode": 2}) == -9
    assert ex({"mode": 5}) == -9
    assert ex({"group_m": 65}) == -9
    assert ex({"tail_split": 2}) == -9
    assert ex({"stages": 9}) == -3
    assert ex({"block_n": 128, "mode": 3}, M=0) == 0          # empty: a no-op
    assert ex({"block_n": 128, "mode": 3}, lda=63) == -1      # then sg_gemm's checks
    assert ex({"block_n": 128, "mode": 3}, C=PC + 2) == -5
    with pytest.raises(ValueError):
        sg._config({"tile": 128})


@needs_no_gpu
def test_host_entry_rejects_bad_args(sg):
    """sg_gemm_host applies sg_gemm's checks and the residual's to the host
    ranges before any CUDA call."""
    f = sg.load_library().sg_gemm_host

    def call(M=64, N=64, K=64, A=P16, lda=64, B=P16B, ldb=64, R=None, ldr=0, C=PC, ldc=64, ind=1, outd=1, epi=0,
             bias=None):
        return f(M, N, K, A, lda, B, ldb, R, ldr, C, ldc, ind, outd, epi, bias, 0, None)

    assert call(M=0, A=None, B=None, C=None) == 0          # empty: a no-op
    assert call(lda=63) == -1
    assert call(ind=0) == -2                                # fp32 operands
    assert call(epi=2) == -1                                # bias missing
    assert call(C=P16 + 64) == -4                           # C overlaps A
    assert call(R=0x5000000, ldr=10) == -1                  # ldr < N
    assert call(R=PC + 1, ldr=64) == -5                     # residual not aligned to its 2-byte elements
    assert call(R=PC + 2, ldr=64) == -4                     # residual partly overlapping C
