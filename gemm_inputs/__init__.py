"""Seeded synthetic inputs for the GEMM workloads.

This module only makes inputs: it holds none of the product's arithmetic and
none of the oracle's.  Both the CUDA path's tests/benchmark and the oracle
draw their operands from here, so the two sides see the same bits.

Generator (counter-based, so any element can be drawn independently):
  * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014; the constants of Vigna's public-domain
    splitmix64.c).  Stream ``s`` of seed ``seed`` starts from the state
    ``x0 = seed * 2^8 + s`` and element ``i`` is ``mix(x0 + (i + 1) * golden)``,
    exactly the i-th output of a SplitMix64 generator seeded with x0.
  * Uniform[-1, 1): u = (bits >> 11) * 2^-53 in [0, 1), value = 2u - 1.
  * Normal(mu, sigma): Box-Muller on draw pairs (2i, 2i+1):
    r = sqrt(-2 ln(1 - u0)); z_2i = r cos(2 pi u1), z_2i+1 = r sin(2 pi u1).
  * Values are computed in float64 and rounded to nearest-even into the
    storage type: fp16 directly; bf16 through binary32 (float64 -> float32
    RNE, then float32 -> bf16 RNE on the bit pattern); fp32 bias directly.

Streams: A = 0, B = 1, bias = 2, residual = 3.  Workload w (1..7) uses seed
1000 + w.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_A, STREAM_B, STREAM_BIAS, STREAM_RESIDUAL = 0, 1, 2, 3


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(state0: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of SplitMix64 seeded with ``state0``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = np.uint64(state0 & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        return _mix(z)


def _state0(seed: int, stream: int) -> int:
    return ((seed << 8) + stream) & 0xFFFFFFFFFFFFFFFF


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    bits = splitmix64(_state0(seed, stream), start, count)
    return (bits >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def draw(seed: int, stream: int, n: int, dist: tuple) -> np.ndarray:
    """n float64 values of distribution ``dist``: ("uniform", lo, hi) or
    ("normal", mean, std)."""
    out = np.empty(n, dtype=np.float64)
    kind = dist[0]
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        if kind == "uniform":
            lo, hi = dist[1], dist[2]
            u = uniform01(seed, stream, c0, c1 - c0)
            out[c0:c1] = lo + (hi - lo) * u
        elif kind == "normal":
            mu, sd = dist[1], dist[2]
            p0 = c0 // 2                      # first pair touched by this chunk
            p1 = (c1 + 1) // 2
            u = uniform01(seed, stream, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
            r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
            t = 2.0 * np.pi * u[:, 1]
            z = np.empty(2 * (p1 - p0), dtype=np.float64)
            z[0::2] = r * np.cos(t)
            z[1::2] = r * np.sin(t)
            out[c0:c1] = mu + sd * z[c0 - 2 * p0:c1 - 2 * p0]
        else:
            raise ValueError(f"unknown distribution {dist!r}")
    return out


def to_storage_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> bit patterns of the storage type (uint16 for fp16/bf16,
    uint32 for fp32, uint8 for e4m3), round to nearest even (e4m3 saturates
    at +-448 first)."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32)
    if dtype == "e4m3":
        # OCP FP8 E4M3: saturate to the largest finite value (+-448), then
        # round to nearest even on the 3-bit fraction (quantum 2^(e-3) for
        # |x| in [2^e, 2^(e+1)), 2^-9 below the smallest normal 2^-6)
        a = np.minimum(np.abs(x), 448.0)
        sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
        _, ex = np.frexp(a)                    # a = m * 2^ex, m in [0.5, 1)
        e = np.maximum(ex - 1, -6)             # exponent of the binade (clamped to the subnormal range)
        q = np.ldexp(1.0, (e - 3).astype(np.int64))
        m = np.rint(a / q)                     # np.rint rounds half to even
        carry = m >= 16.0
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 8.0, m)
        normal = m >= 8.0
        enc = np.where(normal, ((e + 7).astype(np.int64) << 3) | (m.astype(np.int64) - 8), m.astype(np.int64))
        enc = np.where(a == 0, 0, enc)
        return (enc.astype(np.uint8) | sign).astype(np.uint8)
    if dtype == "bf16":
        f = x.astype(np.float32).view(np.uint32)
        nan = (f & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        # no overflow: the largest non-NaN pattern, 0xFF800000, plus 0x8000 fits
        rounded = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        if nan.any():
            rounded = np.where(nan, (f >> np.uint32(16)) | np.uint32(0x40), rounded)
        return rounded.astype(np.uint16)
    raise ValueError(dtype)


def matrix_bits(seed: int, stream: int, rows: int, cols: int, dist: tuple, dtype: str,
                ld: int | None = None) -> np.ndarray:
    """A rows x ld bit matrix (uint16, or uint8 for e4m3) whose first
    ``cols`` columns hold the seeded values (row-major draw order); padding
    columns are zero."""
    ld = cols if ld is None else ld
    vals = to_storage_bits(draw(seed, stream, rows * cols, dist), dtype).reshape(rows, cols)
    if ld == cols:
        return vals
    out = np.zeros((rows, ld), dtype=vals.dtype)
    out[:, :cols] = vals
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic GEMM configuration: C = epilogue(A . B)."""
    name: str
    M: int
    N: int
    K: int
    in_dtype: str
    out_dtype: str
    epilogue: str
    dist_a: tuple
    dist_b: tuple
    dist_bias: tuple | None
    seed: int
    description: str
    dist_r: tuple | None = None   # residual R (M x N, output type), if the workload has one
    b_coded: bool = False         # B given as int8 codes with one fp32 scale per column

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Each operand read once and C written once (bias included)."""
        out_size = {"f32": 4, "f16": 2, "bf16": 2}[self.out_dtype]
        in_size = 1 if self.in_dtype == "e4m3" else 2
        b_bytes = (self.K * self.N + 4 * self.N) if self.b_coded else in_size * self.K * self.N
        b = in_size * self.M * self.K + b_bytes + out_size * self.M * self.N
        if self.epilogue == "bias_relu":
            b += 4 * self.N
        if self.dist_r is not None:
            b += out_size * self.M * self.N
        return b

    def a_bits(self, ld: int | None = None) -> np.ndarray:
        return matrix_bits(self.seed, STREAM_A, self.M, self.K, self.dist_a, self.in_dtype, ld)

    def b_bits(self, ld: int | None = None) -> np.ndarray:
        return matrix_bits(self.seed, STREAM_B, self.K, self.N, self.dist_b, self.in_dtype, ld)

    def b_codes(self) -> tuple[np.ndarray, np.ndarray]:
        """B as int8 codes (K x N) and one fp32 scale per column: B's seeded
        values quantised per column, symmetric over 127 levels each side
        (s_j = max_k |w_kj| / 127, q_kj = w_kj / s_j rounded to nearest even),
        the usual form of quantised weights."""
        w = draw(self.seed, STREAM_B, self.K * self.N, self.dist_b).reshape(self.K, self.N)
        amax = np.abs(w).max(axis=0)
        s = (np.where(amax > 0, amax, 1.0) / 127.0).astype(np.float32)
        q = np.clip(np.rint(w / s.astype(np.float64)), -127, 127).astype(np.int8)
        return q, s

    def r_bits(self) -> np.ndarray | None:
        """The residual's bit patterns (M x N, the output's storage type)."""
        if self.dist_r is None:
            return None
        return to_storage_bits(draw(self.seed, STREAM_RESIDUAL, self.M * self.N, self.dist_r),
                               self.out_dtype).reshape(self.M, self.N)

    def bias(self) -> np.ndarray | None:
        if self.dist_bias is None:
            return None
        return to_storage_bits(draw(self.seed, STREAM_BIAS, self.N, self.dist_bias), "f32").view(np.float32)


WORKLOADS = {
    "square256_f16": Workload(
        "square256_f16", 256, 256, 256, "f16", "f32", "none",
        ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), None, 1001,
        "fp16 M=N=K=256, uniform[-1,1), fp32 accumulate and output, no epilogue"),
    "ragged1000_f16": Workload(
        "ragged1000_f16", 1000, 1000, 1000, "f16", "f32", "none",
        ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), None, 1002,
        "ragged fp16 M=N=K=1000, N(0,1), fp32 accumulate and output (zero-fill of out-of-range elements)"),
    "square8192_bf16": Workload(
        "square8192_bf16", 8192, 8192, 8192, "bf16", "bf16", "none",
        ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), None, 1003,
        "bf16 M=N=K=8192, uniform[-1,1), fp32 accumulate, bf16 output, no epilogue"),
    "square8192_e4m3": Workload(
        "square8192_e4m3", 8192, 8192, 8192, "e4m3", "bf16", "none",
        ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), None, 1007,
        "FP8 E4M3 M=N=K=8192, uniform[-1,1) rounded to E4M3, fp32 accumulate, bf16 output, no epilogue"),
    "relu4096_f16": Workload(
        "relu4096_f16", 4096, 4096, 4096, "f16", "f16", "relu",
        ("normal", 0.0, 1.0 / 64.0), ("normal", 0.0, 1.0 / 64.0), None, 1004,
        "fused C = relu(A.B), fp16 M=N=K=4096, N(0, 1/sqrt(K)), fp32 accumulate, fp16 output"),
    "swin4k_proj_f16": Workload(
        "swin4k_proj_f16", 518400, 384, 96, "f16", "f16", "bias_relu",
        ("normal", 0.0, 1.0), ("normal", 0.0, 0.1), ("normal", 0.0, 0.1), 1005,
        "skinny-K token projection, 3840x2160 frame in 4x4 patches: M=518400 tokens, K=96 -> N=384, "
        "C = relu(A.W + b), fp16 in/out, fp32 bias"),
    "swin4k_backproj_f16": Workload(
        "swin4k_backproj_f16", 518400, 96, 384, "f16", "f16", "none",
        ("normal", 0.0, 1.0), ("normal", 0.0, 0.05), None, 1006,
        "skinny-N back-projection of the Swin MLP band on a 3840x2160 frame in 4x4 patches: M=518400 tokens, "
        "K=384 -> N=96, C = A.W + R with the residual R as the accumulator's seed, fp16 in/out",
        dist_r=("normal", 0.0, 1.0)),
    "swin4k_proj_i8w": Workload(
        "swin4k_proj_i8w", 518400, 384, 96, "f16", "f16", "bias_relu",
        ("normal", 0.0, 1.0), ("normal", 0.0, 0.1), ("normal", 0.0, 0.1), 1008,
        "the skinny-K token projection with int8-coded weights (per-column scales): M=518400 tokens, K=96 -> "
        "N=384, C = relu(A.(Q.diag(s)) + b), fp16 activations and output, B decoded once per CTA into a "
        "shared-memory panel", b_coded=True),
}

# The five workloads in the order they are listed for this path.
WORKLOAD_ORDER = ["square256_f16", "ragged1000_f16", "square8192_bf16", "relu4096_f16", "swin4k_proj_f16"]
