"""The seeded input generator (host side)."""
import numpy as np

from kv_cache_decode_gqa_gb300 import inputs as I


def test_splitmix64_published_vectors():
    # SplitMix64 seeded with 0: its first three outputs
    got = [int(x) for x in I.draws(0, np.arange(3))]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_draws_are_counter_based():
    key = I.stream_key(20262, 3, 1)
    a = I.draws(key, np.arange(1000))
    b = I.draws(key, np.arange(500, 1000))
    assert np.array_equal(a[500:], b)
    assert I.stream_key(20262, 3, 1) != I.stream_key(20262, 3, 2)


def test_normal_table():
    t = I.normal_bf16_table()
    import oracle
    v = oracle.bf16_bits_to_f64(t)
    assert t.shape == (65536,)
    assert np.all(np.diff(v) >= 0)
    assert abs(v.mean()) < 1e-3 and abs(v.std() - 1) < 5e-3
    assert np.array_equal(v, -v[::-1])


def test_host_fill_offsets():
    t = I.normal_bf16_table()
    key = I.stream_key(1, 2)
    whole = I.host_tensor(t, key, (4, 100))
    part = I.host_tensor(t, key, (100,), offset=200)
    assert np.array_equal(whole[2], part)


def test_fp8_code_table_has_no_nan_or_zero():
    c = I.fp8_code_table()
    assert np.all((c & 0x7F) != 0x7F) and np.all((c & 0x7F) != 0)
    assert len(set(c.tolist())) == 128


def test_permutation_and_ints():
    p = I.permutation(I.stream_key(5), 1000)
    assert sorted(p.tolist()) == list(range(1000))
    L = I.uniform_int(I.stream_key(6), 5000, 1024, 8192)
    assert L.min() >= 1024 and L.max() <= 8192
    u = I.uniform01_f32(I.stream_key(7), 1000)
    assert u.dtype == np.float32 and u.min() >= 0 and u.max() < 1
