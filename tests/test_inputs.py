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


def test_mxfp4_input_tables():
    """MXFP4 inputs: code bytes are all 256 values (two random E2M1 codes
    each); group scales decode (with the oracle's E4M3 table) to exactly the
    16 values 1/8 .. 15/32, each 16 times, where amax / 6 of 16 N(0,1)
    values falls for about 92 % of groups."""
    import numpy as np
    import oracle
    from kv_cache_decode_gqa_gb300 import inputs as I
    assert sorted(I.byte_table().tolist()) == list(range(256))
    vals = oracle.e4m3_codes_to_f64(I.mxfp4_scale_table())
    want = sorted({e * (1 + m / 8) for e in (1 / 8, 1 / 4) for m in range(8)})
    assert len(want) == 16 and want[0] == 1 / 8 and want[-1] == 15 / 32
    u, counts = np.unique(vals, return_counts=True)
    assert u.tolist() == want and set(counts.tolist()) == {16}
    amax6 = np.abs(np.random.default_rng(5).standard_normal((100_000, 16))
                   ).max(axis=1) / 6
    inside = np.mean((amax6 >= 1 / 8) & (amax6 <= 15 / 32))
    assert 0.91 < inside < 0.94


def test_fp8_cache_codes_cover_eighth_to_thirty():
    import numpy as np
    import oracle
    from kv_cache_decode_gqa_gb300 import inputs as I
    mag = np.abs(oracle.e4m3_codes_to_f64(I.fp8_code_table()))
    assert mag.min() == 1 / 8 and mag.max() == 30.0


def test_workload_recipe_ranges():
    """fp8 scales in [1/16, 1/8) with inv_scale their fp32 reciprocal;
    Llama-3.1-70B cached lengths in [1024, 8192]; indexer weights in
    [0, 1)."""
    import numpy as np
    from kv_cache_decode_gqa_gb300 import workloads as W
    s = W.config("llama31_70b_gqa_fp8")
    for layer in (0, 79):
        for t in (W.T_KSCALE, W.T_VSCALE):
            sc, inv = W.host_scales(s, layer, t)
            assert sc.dtype == np.float32 and sc.shape == (8,)
            assert np.all((sc >= 1 / 16) & (sc < 1 / 8))
            assert np.array_equal(inv, np.float32(1) / sc)
    lens = W.config("llama31_70b_gqa").lengths
    assert len(lens) == 32 and min(lens) >= 1024 and max(lens) <= 8192
    assert len(set(lens)) > 16                        # a real length mix
    sp = W.config("sparse")
    w = W.host_weights(sp, 0)
    assert w.shape == (sp.batch, sp.idx_heads)
    assert np.all((w >= 0) & (w < 1))
