"""The seeded input generator: its SplitMix64 against the published
reference outputs, determinism, element-addressability and the moments of
the workloads' distributions.  CPU only."""
import numpy as np

import gemm_inputs as gi


def test_splitmix64_reference_outputs():
    # First outputs of the reference splitmix64.c seeded with 1234567.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [int(x) for x in gi.splitmix64(1234567, 0, 5)] == want


def test_counter_based_slices_agree():
    full = gi.splitmix64(99, 0, 1000)
    assert np.array_equal(gi.splitmix64(99, 500, 100), full[500:600])
    a = gi.draw(5, 1, 10001, ("normal", 0.0, 1.0))
    b = gi.draw(5, 1, 10001, ("normal", 0.0, 1.0))
    assert np.array_equal(a, b)


def test_chunk_boundaries_do_not_change_values(monkeypatch):
    ref = gi.draw(7, 0, 5003, ("normal", 1.0, 2.0))
    monkeypatch.setattr(gi, "_CHUNK", 1024)
    assert np.array_equal(gi.draw(7, 0, 5003, ("normal", 1.0, 2.0)), ref)
    u_ref = gi.draw(7, 2, 3001, ("uniform", -1.0, 1.0))
    monkeypatch.setattr(gi, "_CHUNK", 512)
    assert np.array_equal(gi.draw(7, 2, 3001, ("uniform", -1.0, 1.0)), u_ref)


def test_distribution_moments():
    u = gi.draw(1, 0, 400000, ("uniform", -1.0, 1.0))
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1.0 / 3.0) < 0.01
    z = gi.draw(1, 1, 400000, ("normal", 0.0, 0.1))
    assert abs(z.mean()) < 0.001 and abs(z.std() - 0.1) < 0.001


def test_streams_and_seeds_differ():
    a = gi.draw(1001, 0, 100, ("uniform", -1, 1))
    b = gi.draw(1001, 1, 100, ("uniform", -1, 1))
    c = gi.draw(1002, 0, 100, ("uniform", -1, 1))
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_bf16_storage_rounding_is_rne_of_float32():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625])
    bits = gi.to_storage_bits(x, "bf16")
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4049]


def test_workload_table():
    w = gi.WORKLOADS["swin4k_proj_f16"]
    assert (w.M, w.N, w.K) == (3840 * 2160 // 16, 384, 96)
    assert w.algorithmic_bytes == 497_739_264
    assert gi.WORKLOADS["square8192_bf16"].flops == 2 * 8192 ** 3
    assert [gi.WORKLOADS[n].seed for n in gi.WORKLOAD_ORDER] == [1001, 1002, 1003, 1004, 1005]
    a = gi.WORKLOADS["ragged1000_f16"].a_bits(ld=1008)
    assert a.shape == (1000, 1008) and np.all(a[:, 1000:] == 0)
    assert np.array_equal(a[:, :1000], gi.WORKLOADS["ragged1000_f16"].a_bits())


def test_e4m3_storage_rounding():
    torch = __import__("pytest").importorskip("torch")
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 50, 20000), rng.normal(0, 0.01, 20000), [0.0, -0.0, 448.0, -448.0,
                        2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 2.0 ** -6]])
    ours = gi.to_storage_bits(x, "e4m3")
    within = np.abs(x) <= 448.0
    # inside the finite range torch's float32 -> e4m3fn cast rounds to nearest even
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours[within], ref[within])
    # beyond it the generator saturates (torch would give NaN)
    big = gi.to_storage_bits(np.array([449.0, 1e6, -1e6, 500.0]), "e4m3")
    assert list(big) == [0x7E, 0x7E, 0xFE, 0x7E]
    # ties to even: 1.0625 is halfway between 1 (even) and 1.125; 1.1875 between 1.125 and 1.25 (even)
    assert list(gi.to_storage_bits(np.array([1.0625, 1.1875]), "e4m3")) == [0x38, 0x3A]
