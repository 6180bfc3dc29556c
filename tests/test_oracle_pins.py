"""Pins of the fp64 oracle against things other than itself: the pages'
figures (tests/golden/page_figures.json), hand-worked examples, closed forms,
brute force in plain Python, library conversions, and invariants of the
mathematics. A plausible mistake in the oracle (a dropped scale, a transposed
operand, a wrong head-to-group map, a tie broken the wrong way, an off-by-one
length) fails at least one test here; test_oracle_mutants.py plants such
mistakes to check that.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _bf16_bits(x):
    """float64 array -> bf16 bit patterns (library rounding, torch CPU)."""
    t = torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bf16_round(x):
    return O.bf16_bits_to_f64(_bf16_bits(x))


# ---------------------------------------------------------------------------
# element formats
# ---------------------------------------------------------------------------
def test_bf16_closed_form():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x8000, 0x4049],
                    dtype=np.uint16)
    v = O.bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0
    assert v[2] == 2.0 ** -133                     # smallest subnormal
    assert np.isinf(v[3]) and v[3] > 0
    assert v[4] == 0.0 and np.signbit(v[4])
    assert v[5] == 3.140625


def test_bf16_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=20000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # drop inf / NaN
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double()
    assert np.array_equal(O.bf16_bits_to_f64(bits), ref.numpy())


def test_e4m3_closed_form(golden_dir):
    g = _load(golden_dir, "page_figures.json")["e4m3_max"]
    t = O.e4m3_value_table()
    assert t[0x7E] == g["value"] == 448.0
    assert t[0x7E] * 6 == g["fp4_bound"]
    assert t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9                     # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6                     # smallest normal
    assert t[0x38] == 1.0
    assert t[0x00] == 0.0 and t[0x80] == 0.0 and np.signbit(t[0x80])
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254
    pos = t[:127]
    assert np.all(np.diff(pos) > 0)                 # codes ordered by value


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    mine = O.e4m3_codes_to_f64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[fin], mine[fin])


def test_e4m3_encode_round_trip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F],
                     dtype=np.uint8)
    vals = O.e4m3_codes_to_f64(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode_f32(vals), codes)


def test_e4m3_encode_midpoints_ties_to_even():
    t = O.e4m3_value_table()[:127]
    for c in range(126):
        mid = np.float32((t[c] + t[c + 1]) / 2)     # exact in fp32
        assert float(mid) == (t[c] + t[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert O.e4m3_encode_f32(np.array([mid]))[0] == want, c
        assert O.e4m3_encode_f32(np.array([-mid]))[0] == (want | 0x80), c
        up = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
        dn = np.nextafter(mid, np.float32(0), dtype=np.float32)
        assert O.e4m3_encode_f32(np.array([up]))[0] == c + 1
        assert O.e4m3_encode_f32(np.array([dn]))[0] == c


def test_e4m3_encode_saturates_and_edges():
    x = np.array([448.0, 449.0, 464.0, 500.0, 1e30, np.inf, -np.inf, -1e9,
                  2.0 ** -10, 2.0 ** -10 * 1.0001, 3 * 2.0 ** -10, -1e-30,
                  0.0, np.nan], dtype=np.float32)
    got = O.e4m3_encode_f32(x)
    want = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE,
            0x00, 0x01, 0x02, 0x80, 0x00, 0x7F]
    assert got.tolist() == want


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(50000) * 30,
                        rng.standard_normal(20000) * 0.01,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(O.e4m3_encode_f32(x), ref.numpy())


# ---------------------------------------------------------------------------
# attention at one position
# ---------------------------------------------------------------------------
def test_worked_examples(golden_dir):
    for case in _load(golden_dir, "worked_attention.json")["cases"]:
        out, lse = O.attend(np.array(case["q"]), np.array(case["K"]),
                            np.array(case["V"]), case["scale"])
        np.testing.assert_allclose(out, case["out"], rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse, case["lse"], rtol=0, atol=1e-12,
                                   err_msg=case["name"])


def _brute_attend(q, K, V, scale):
    """Plain-Python loops: one head, one position."""
    T = len(K)
    s = [scale * sum(q[i] * K[t][i] for i in range(len(q))) for t in range(T)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    out = [sum(e[t] * V[t][j] for t in range(T)) / z for j in range(len(V[0]))]
    return out, m + math.log(z)


def test_attend_brute_force():
    rng = np.random.default_rng(3)
    for T in (1, 2, 5, 9):
        for d in (1, 3, 4):
            q = rng.standard_normal((2, d))
            K = rng.standard_normal((T, d))
            V = rng.standard_normal((T, d + 1))
            out, lse = O.attend(q, K, V, 0.37)
            for h in range(2):
                bo, bl = _brute_attend(q[h].tolist(), K.tolist(), V.tolist(),
                                       0.37)
                np.testing.assert_allclose(out[h], bo, atol=1e-12)
                assert abs(lse[h] - bl) < 1e-12


def test_weights_sum_to_one_and_identity_values():
    rng = np.random.default_rng(4)
    T = 37
    S = rng.standard_normal((3, T)) * 4
    w, _ = O.attend_scores(S, np.eye(T))            # out = the weights
    assert np.all(w >= 0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-14)
    # weights are proportional to exp(score)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], np.exp(S[:, 1:] - S[:, :1]),
                               rtol=1e-12)


def test_empty_prefix():
    out, lse = O.attend(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def _causal_full(Q, K, V):
    """Causal self-attention for every position at once, with an explicit
    -inf mask over future positions (no cache), written independently of
    the oracle. Q [T][n_h][d], K, V [T][n_kv][d]."""
    T, n_h, d = Q.shape
    g = n_h // K.shape[1]
    mask = np.triu(np.full((T, T), -np.inf), k=1)
    out = np.zeros((T, n_h, d))
    for h in range(n_h):
        kv = h // g
        S = Q[:, h, :] @ K[:, kv, :].T / math.sqrt(d) + mask
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ V[:, kv, :]
    return out


@pytest.mark.parametrize("n_h,n_kv", [(4, 4), (8, 2), (6, 1)])
def test_cached_decode_equals_full_recompute(n_h, n_kv):
    """KV cache, 'A cache you keep ...': k_i, v_i depend on h_i alone and
    causality fixes h_i, so attending over cached k, v at the last position
    equals recomputing causal attention over the whole sequence. The
    projections k = W_K h, v = W_V h are stored in bf16, and the recompute
    uses those stored values too."""
    rng = np.random.default_rng(5)
    T, d_model, d, bs = 23, 16, 8, 4
    H = rng.standard_normal((T, d_model))
    Wq = rng.standard_normal((d_model, n_h * d)) / 4
    Wk = rng.standard_normal((d_model, n_kv * d)) / 4
    Wv = rng.standard_normal((d_model, n_kv * d)) / 4
    Q = (H @ Wq).reshape(T, n_h, d)
    K = _bf16_round((H @ Wk).reshape(T, n_kv, d))
    V = _bf16_round((H @ Wv).reshape(T, n_kv, d))
    full = _causal_full(Q, K, V)
    nb = (T + bs - 1) // bs
    perm = rng.permutation(nb + 3)[:nb]
    k_raw = np.zeros((nb + 3, n_kv, bs, d), dtype=np.uint16)
    v_raw = np.zeros_like(k_raw)
    for t in range(T):
        k_raw[perm[t // bs], :, t % bs, :] = _bf16_bits(K[t])
        v_raw[perm[t // bs], :, t % bs, :] = _bf16_bits(V[t])
    for t_last in (0, 5, T - 1):
        out, _ = O.gqa_decode(Q[t_last][None], k_raw, v_raw, perm[None],
                              [t_last + 1], bs)
        np.testing.assert_allclose(out[0], full[t_last], atol=1e-12)


# ---------------------------------------------------------------------------
# paging and grouped heads
# ---------------------------------------------------------------------------
def _random_paged(rng, B, n_kv, d, bs, lens, spare=2, dtype=np.uint16):
    nbs = [(L + bs - 1) // bs for L in lens]
    nb = sum(nbs) + spare
    perm = rng.permutation(nb)
    mb = max(max(nbs), 1)
    bt = np.full((B, mb), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        bt[b, :nbs[b]] = perm[k:k + nbs[b]]
        k += nbs[b]
    if dtype == np.uint16:
        kr = _bf16_bits(rng.standard_normal((nb, n_kv, bs, d)))
        vr = _bf16_bits(rng.standard_normal((nb, n_kv, bs, d)))
    else:
        kr = rng.integers(0, 256, (nb, n_kv, bs, d)).astype(np.uint8)
        kr[(kr & 0x7F) == 0x7F] = 0x11
        vr = rng.integers(0, 256, (nb, n_kv, bs, d)).astype(np.uint8)
        vr[(vr & 0x7F) == 0x7F] = 0x22
    return kr, vr, bt


def _contiguous_copy(raw, bt, lens, bs):
    """Same sequences, one contiguous block per sequence."""
    B = len(lens)
    cap = max(max(lens), 1)
    out = np.zeros((B, raw.shape[1], cap, raw.shape[3]), dtype=raw.dtype)
    for b in range(B):
        for t in range(lens[b]):
            out[b, :, t, :] = raw[bt[b, t // bs], :, t % bs, :]
    return out


def test_paging_is_transparent():
    rng = np.random.default_rng(6)
    lens = [1, 15, 16, 17, 40]
    B, n_kv, d, bs, n_h = len(lens), 2, 8, 16, 4
    kr, vr, bt = _random_paged(rng, B, n_kv, d, bs, lens)
    q = rng.standard_normal((B, n_h, d))
    o1, l1 = O.gqa_decode(q, kr, vr, bt, lens, bs)
    cap = max(lens)
    kc = _contiguous_copy(kr, bt, lens, bs)
    vc = _contiguous_copy(vr, bt, lens, bs)
    o2, l2 = O.gqa_decode(q, kc, vc, np.arange(B)[:, None], lens, cap)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_gqa_equals_mha_on_repeated_heads():
    """KV cache, 'Fewer KV heads ...': GQA partitions the query heads into
    groups sharing one KV head; it is exactly MHA over the KV heads repeated
    per group (query head h reads KV head h // g)."""
    rng = np.random.default_rng(7)
    lens = [5, 33, 64]
    B, n_kv, g, d, bs = 3, 2, 4, 16, 16
    kr, vr, bt = _random_paged(rng, B, n_kv, d, bs, lens)
    q = rng.standard_normal((B, n_kv * g, d))
    o1, l1 = O.gqa_decode(q, kr, vr, bt, lens, bs)
    o2, l2 = O.gqa_decode(q, np.repeat(kr, g, axis=1), np.repeat(vr, g, axis=1),
                          bt, lens, bs)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_mha_brute_force_per_head():
    rng = np.random.default_rng(8)
    lens = [3, 7]
    B, n_kv, d, bs = 2, 3, 4, 4
    kr, vr, bt = _random_paged(rng, B, n_kv, d, bs, lens)
    q = rng.standard_normal((B, n_kv, d))
    out, lse = O.gqa_decode(q, kr, vr, bt, lens, bs, scale=0.5)
    for b in range(B):
        for h in range(n_kv):
            K = [O.bf16_bits_to_f64(kr[bt[b, t // bs], h, t % bs]).tolist()
                 for t in range(lens[b])]
            V = [O.bf16_bits_to_f64(vr[bt[b, t // bs], h, t % bs]).tolist()
                 for t in range(lens[b])]
            bo, bl = _brute_attend(q[b, h].tolist(), K, V, 0.5)
            np.testing.assert_allclose(out[b, h], bo, atol=1e-12)
            assert abs(lse[b, h] - bl) < 1e-12


def test_default_scale_is_inverse_sqrt_head_dim():
    rng = np.random.default_rng(9)
    kr, vr, bt = _random_paged(rng, 1, 1, 16, 8, [11])
    q = rng.standard_normal((1, 2, 16))
    a = O.gqa_decode(q, kr, vr, bt, [11], 8)
    b = O.gqa_decode(q, kr, vr, bt, [11], 8, scale=0.25)
    np.testing.assert_allclose(a[0], b[0], atol=0)


def test_fp8_cache_is_scaled_codes():
    rng = np.random.default_rng(10)
    lens = [9, 20]
    kr, vr, bt = _random_paged(rng, 2, 2, 8, 8, lens, dtype=np.uint8)
    ks = np.array([0.5, 0.125], dtype=np.float32)
    vs = np.array([2.0, 0.25], dtype=np.float32)
    q = rng.standard_normal((2, 4, 8))
    o1, l1 = O.gqa_decode(q, kr, vr, bt, lens, 8, dtype="fp8", k_scale=ks,
                          v_scale=vs)
    # the same values stored as exact bf16 (each code * power-of-two scale
    # has <= 4 significant bits, so bf16 holds it exactly)
    kv = O.e4m3_codes_to_f64(kr) * ks[None, :, None, None].astype(np.float64)
    vv = O.e4m3_codes_to_f64(vr) * vs[None, :, None, None].astype(np.float64)
    o2, l2 = O.gqa_decode(q, _bf16_bits(kv), _bf16_bits(vv), bt, lens, 8)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------
def test_append_bf16_writes_one_slot():
    rng = np.random.default_rng(11)
    lens = [3, 16, 30]
    kr, _, bt = _random_paged(rng, 3, 2, 8, 16, [L + 1 for L in lens])
    new = _bf16_bits(rng.standard_normal((3, 2, 8)))
    out = O.kv_append(kr, bt, lens, new, 16)
    changed = np.argwhere(np.any(out != kr, axis=3))
    for b, L in enumerate(lens):
        assert np.array_equal(out[bt[b, L // 16], :, L % 16, :], new[b])
    assert len(changed) <= 3 * 2                    # nothing else moved
    mask = np.ones(kr.shape[:3], dtype=bool)
    for b, L in enumerate(lens):
        mask[bt[b, L // 16], :, L % 16] = False
    assert np.array_equal(out[mask], kr[mask])


def test_append_fp8_codes():
    rng = np.random.default_rng(12)
    kr, _, bt = _random_paged(rng, 2, 2, 8, 8, [5, 9], dtype=np.uint8)
    new_f = rng.standard_normal((2, 2, 8)) * 3
    new = _bf16_bits(new_f)
    inv = np.array([8.0, 1 / 0.07], dtype=np.float32)
    out = O.kv_append(kr, bt, [4, 8], new, 8, dtype="fp8", inv_scale=inv)
    for b, p in enumerate([4, 8]):
        x = O.bf16_bits_to_f64(new[b]).astype(np.float32)
        y = x * inv[:, None]                         # float32 products
        ref = torch.from_numpy(np.ascontiguousarray(y)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(out[bt[b, p // 8], :, p % 8, :], ref)


# ---------------------------------------------------------------------------
# latent cache
# ---------------------------------------------------------------------------
def test_mla_absorbed_equals_explicit():
    """KV cache, 'Caching a compressed latent ...': folding W_UK into the
    query gives the same scores as decompressing per-head keys, and the
    value up-projection can be applied after the weighted sum."""
    rng = np.random.default_rng(13)
    n_h, d_c, d_r, d_nope, d_v, bs = 3, 16, 4, 6, 5, 8
    T = 19
    c = _bf16_round(rng.standard_normal((T, d_c)))
    kr = _bf16_round(rng.standard_normal((T, d_r)))
    W_uk = rng.standard_normal((n_h, d_c, d_nope)) / 3
    W_uv = rng.standard_normal((n_h, d_c, d_v)) / 3
    q_nope = rng.standard_normal((n_h, d_nope))
    q_rope = rng.standard_normal((n_h, d_r))
    scale = 1 / math.sqrt(d_c + d_r)
    # explicit: per-head keys [W_uk^T c | k_rope], values W_uv^T c
    explicit = np.zeros((n_h, d_v))
    for h in range(n_h):
        Kh = np.concatenate([c @ W_uk[h], kr], axis=1)
        Vh = c @ W_uv[h]
        qh = np.concatenate([q_nope[h], q_rope[h]])
        explicit[h] = O.attend(qh[None], Kh, Vh, scale)[0][0]
    # absorbed: q_lat = W_uk q_nope, attend over [c | k_rope], out in latent
    q_lat = np.einsum("hcn,hn->hc", W_uk, q_nope)
    nb = (T + bs - 1) // bs
    lat = np.zeros((nb, 1, bs, d_c + d_r), dtype=np.uint16)
    rows = _bf16_bits(np.concatenate([c, kr], axis=1))
    for t in range(T):
        lat[t // bs, 0, t % bs] = rows[t]
    q = np.concatenate([q_lat, q_rope], axis=1)[None]
    out_lat, _ = O.mla_decode(q, lat, np.arange(nb)[None], [T], bs, d_c=d_c,
                              scale=scale)
    absorbed = np.einsum("hcv,hc->hv", W_uv, out_lat[0])
    np.testing.assert_allclose(absorbed, explicit, atol=1e-12)


def test_mla_is_mqa_with_shared_row():
    rng = np.random.default_rng(14)
    d_c, d_r, bs, n_h = 8, 4, 4, 5
    lens = [6, 13]
    kr, _, bt = _random_paged(rng, 2, 1, d_c + d_r, bs, lens)
    q = rng.standard_normal((2, n_h, d_c + d_r))
    o1, l1 = O.mla_decode(q, kr, bt, lens, bs, d_c=d_c)
    vr = kr.copy()
    vr[..., d_c:] = 0                                 # values: c only
    o2, l2 = O.gqa_decode(q, kr, vr, bt, lens, bs)
    np.testing.assert_allclose(o1, o2[..., :d_c], atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


# ---------------------------------------------------------------------------
# indexer and top-k
# ---------------------------------------------------------------------------
def test_indexer_brute_force():
    rng = np.random.default_rng(15)
    lens = [1, 9, 25]
    kr, _, bt = _random_paged(rng, 3, 1, 6, 8, lens)
    qI = rng.standard_normal((3, 4, 6))
    w = rng.uniform(0, 1, (3, 4))
    sc = O.indexer_scores(qI, w, kr, bt, lens, 8)
    for b, L in enumerate(lens):
        assert sc[b].shape == (L,)
        for t in range(L):
            k = O.bf16_bits_to_f64(kr[bt[b, t // 8], 0, t % 8]).tolist()
            want = 0.0
            for j in range(4):
                dot = sum(qI[b, j, i] * k[i] for i in range(6))
                want += w[b, j] * (dot if dot > 0 else 0.0)
            assert abs(sc[b][t] - want) < 1e-12


def test_indexer_exact_arithmetic_values():
    """q, k in {a/8}, w in {1..4}: every score is a multiple of 2^-6 and the
    fp64 sum is exact; checked against integer arithmetic."""
    rng = np.random.default_rng(16)
    T, d, bs = 40, 64, 16
    ka = rng.integers(-7, 9, (T, d))
    qa = rng.integers(-7, 9, (1, 4, d))
    w = rng.integers(1, 5, (1, 4)).astype(np.float64)
    nb = (T + bs - 1) // bs
    raw = np.zeros((nb, 1, bs, d), dtype=np.uint16)
    bits = _bf16_bits(ka / 8.0)
    for t in range(T):
        raw[t // bs, 0, t % bs] = bits[t]
    sc = O.indexer_scores(qa / 8.0, w, raw, np.arange(nb)[None], [T], bs)[0]
    dots = ka @ qa[0].T                                # integers * 64
    want = (np.maximum(dots, 0) * w[0]).sum(axis=1) / 64.0
    assert np.array_equal(sc, want)


def test_topk_golden(golden_dir):
    for case in _load(golden_dir, "topk_ties.json")["cases"]:
        got = O.topk_select(np.array(case["scores"], dtype=np.float64),
                            case["k"])
        assert got.tolist() == case["indices"], case["why"]


def test_topk_brute_force():
    rng = np.random.default_rng(17)
    for T in (1, 7, 100, 513):
        s = np.round(rng.standard_normal(T) * 3) / 2     # many ties
        for k in (1, 5, 64, 600):
            want = sorted(sorted(range(T), key=lambda t: (-s[t], t))[:k])
            want += [-1] * (k - len(want))
            assert O.topk_select(s, k).tolist() == want


def test_topk_all_equal_takes_lowest():
    assert O.topk_select(np.zeros(10), 3).tolist() == [0, 1, 2]


def test_sparse_all_positions_equals_dense():
    rng = np.random.default_rng(18)
    lens = [10, 40]
    kr, vr, bt = _random_paged(rng, 2, 1, 16, 8, lens)
    q = rng.standard_normal((2, 4, 16))
    idx = np.full((2, 48), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        idx[b, :L] = np.arange(L)
    o1, l1 = O.sparse_decode(q, kr, vr, bt, lens, 8, idx)
    o2, l2 = O.gqa_decode(q, kr, vr, bt, lens, 8)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_sparse_subset_equals_dense_over_subset():
    rng = np.random.default_rng(19)
    L, bs, d = 50, 8, 8
    kr, vr, bt = _random_paged(rng, 1, 1, d, bs, [L])
    q = rng.standard_normal((1, 3, d))
    sel = np.sort(rng.choice(L, 12, replace=False))
    idx = np.concatenate([sel, [-1, -1, L + 5]]).astype(np.int32)[None]
    o1, l1 = O.sparse_decode(q, kr, vr, bt, [L], bs, idx, scale=0.3)
    K = np.stack([O.bf16_bits_to_f64(kr[bt[0, t // bs], 0, t % bs])
                  for t in sel])
    V = np.stack([O.bf16_bits_to_f64(vr[bt[0, t // bs], 0, t % bs])
                  for t in sel])
    o2, l2 = O.attend(q[0], K, V, 0.3)
    np.testing.assert_allclose(o1[0], o2, atol=1e-13)
    np.testing.assert_allclose(l1[0], l2, atol=1e-13)


def test_schedule_reuse_and_reindex():
    rng = np.random.default_rng(20)
    lens = [30, 70]
    bs, k = 8, 16
    kr, vr, bt = _random_paged(rng, 2, 1, 16, bs, lens)
    ir, _, _ = _random_paged(np.random.default_rng(21), 2, 1, 8, bs, lens)
    ir = ir[:kr.shape[0]] if ir.shape[0] >= kr.shape[0] else None
    assert ir is not None
    modes = ["full", "reuse", "reindex", "reuse"]
    q = [rng.standard_normal((2, 4, 16)) for _ in modes]
    qI = [rng.standard_normal((2, 4, 8)) for _ in modes]
    w = [rng.uniform(0, 1, (2, 4)) for _ in modes]
    outs, _, sel = O.sparse_schedule(modes, q, qI, w, kr, vr, ir, bt, lens, bs,
                                     k)
    i0, _ = O.indexer_topk(qI[0], w[0], ir, bt, lens, bs, k)
    i2, _ = O.indexer_topk(qI[2], w[2], ir, bt, lens, bs, k)
    assert np.array_equal(sel[0], i0) and np.array_equal(sel[1], i0)
    assert np.array_equal(sel[2], i2) and np.array_equal(sel[3], i2)
    o1, _ = O.sparse_decode(q[1], kr, vr, bt, lens, bs, i0)
    np.testing.assert_allclose(outs[1], o1, atol=0)
    with pytest.raises(ValueError):
        O.sparse_schedule(["reuse"], q, qI, w, kr, vr, ir, bt, lens, bs, k)


# ---------------------------------------------------------------------------
# split-K merge
# ---------------------------------------------------------------------------
def test_split_merge_equals_unsplit():
    rng = np.random.default_rng(22)
    T, d = 200, 16
    q = rng.standard_normal((4, d)) * 2
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    ref = O.attend(q, K, V, 0.25)
    for bounds in ([0, T], [0, 1, T], [0, 64, 128, 192, T],
                   [0, 0, 50, 50, 199, T], [0, 7, 13, 150, T]):
        out, lse = O.split_decode(q, K, V, 0.25, bounds)
        np.testing.assert_allclose(out, ref[0], atol=1e-12)
        np.testing.assert_allclose(lse, ref[1], atol=1e-12)


def test_merge_of_only_empty_parts():
    out, lse = O.lse_merge([(np.zeros((2, 3)), np.full(2, -np.inf))] * 3)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------------------
# size accounting (page figures)
# ---------------------------------------------------------------------------
def test_bytes_per_token_llama31_70b(golden_dir):
    g = _load(golden_dir, "page_figures.json")["llama31_70b_bytes_per_token"]
    f = g["factors"]
    assert O.bytes_per_token(f["n_l"], f["n_kv"], f["d_h"], f["b"]) == g["value"]
    assert g["value"] == 320 * 1024


def test_llama2_7b_cache_about_2gb(golden_dir):
    g = _load(golden_dir, "page_figures.json")["llama2_7b_4096_cache"]
    f = g["factors"]
    n = O.cache_bytes(f["n_l"], f["n_kv"], f["d_h"], f["b"], f["B"], f["L"])
    assert n == 2147483648
    assert abs(n - g["approx_bytes"]) / g["approx_bytes"] < g["rel_tol"]


def test_paged_waste_bound(golden_dir):
    g = _load(golden_dir, "page_figures.json")["paged_waste"]
    bs, Lbar = g["block_size"], g["mean_len"]
    rng = np.random.default_rng(23)
    for _ in range(20):
        lens = rng.integers(1, 2 * Lbar, 64)
        waste = O.paged_waste_slots(lens, bs)
        assert np.all((waste >= 0) & (waste <= bs - 1))
        assert waste.sum() <= len(lens) * (bs - 1)
    assert (bs - 1) / Lbar < g["bound_fraction_below"]
    assert O.paged_waste_slots([16, 17, 1], 16).tolist() == [0, 15, 15]


# ---------------------------------------------------------------------------
# fp4 E2M1 and MXFP4 rows ("890 bytes a token ...", section 6)
# ---------------------------------------------------------------------------
# The OCP Microscaling Formats specification lists the FP4 (E2M1)
# magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7), sign in bit 3.
_OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_are_the_ocp_list():
    t = O.e2m1_value_table()
    assert list(t[:8]) == _OCP_E2M1
    assert list(t[8:]) == [-v for v in _OCP_E2M1]
    assert math.copysign(1.0, t[8]) == -1.0           # code 8 is -0


def test_e2m1_encode_round_trip_all_codes():
    t = O.e2m1_value_table().astype(np.float32)
    assert np.array_equal(O.e2m1_encode_f32(t), np.arange(16, dtype=np.uint8))


def test_e2m1_encode_midpoints_ties_to_even():
    # each midpoint goes to the neighbour whose mantissa bit is 0
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, code in cases.items():
        assert O.e2m1_encode_f32(np.float32(x)) == code, x
        assert O.e2m1_encode_f32(np.float32(-x)) == code | 8, -x
        up = np.nextafter(np.float32(x), np.float32(10))
        dn = np.nextafter(np.float32(x), np.float32(0))
        lo = max(c for c in range(8) if _OCP_E2M1[c] < x)
        hi = min(c for c in range(8) if _OCP_E2M1[c] > x)
        assert O.e2m1_encode_f32(up) == hi and O.e2m1_encode_f32(dn) == lo


def test_e2m1_encode_saturates_and_signs():
    x = np.array([6.0, 6.5, 1e30, np.inf, -7.0, -np.inf, 0.0, -0.0, -0.1,
                  0.1], dtype=np.float32)
    assert list(O.e2m1_encode_f32(x)) == [7, 7, 7, 7, 15, 15, 0, 8, 8, 0]


def test_e2m1_encode_is_nearest_brute_force():
    rng = np.random.default_rng(40)
    x = (rng.standard_normal(4000) * 3).astype(np.float32)
    got = O.e2m1_codes_to_f64(O.e2m1_encode_f32(x))
    for xi, gi in zip(x.astype(np.float64), got):
        a = min(abs(xi), 6.0)
        best = min(abs(a - v) for v in _OCP_E2M1)
        assert abs(abs(gi) - a) == best
        assert gi == 0 or math.copysign(1, gi) == math.copysign(1, xi)


def _mxfp4_groups(codes, scales):
    """Hand-built rows: 16-channel groups of code values times a scale."""
    vals = []
    for g, s in enumerate(scales):
        vals += [O.e2m1_value_table()[c] * s for c in codes[16 * g:16 * g + 16]]
    return np.array(vals)


def test_mxfp4_scaled_grid_round_trips():
    # a group whose largest magnitude is 6 s, s an E4M3 value, stores s and
    # the codes themselves; every such value is exact in bf16
    rng = np.random.default_rng(41)
    e4 = O.e4m3_value_table()
    normal = [c for c in range(0x08, 0x7F) if 6 * e4[c] <= 448 * 6]
    for _ in range(50):
        scodes = rng.choice(normal, 8)
        codes = rng.integers(0, 16, 128)
        for g in range(8):
            codes[16 * g + rng.integers(16)] = 7 | (8 * rng.integers(2))
        x = _mxfp4_groups(codes, e4[scodes])
        row = O.mxfp4_encode_rows(_bf16_bits(x))
        assert row.shape == (O.mxfp4_row_bytes(128),) == (72,)
        assert np.array_equal(row[64:], scodes.astype(np.uint8))
        # channel 2j in the low nibble, 2j+1 in the high one
        lo, hi = row[:64] & 0xF, row[:64] >> 4
        c = codes.astype(np.uint8)
        zero = O.e2m1_value_table()[c] == 0          # +-0 may swap sign
        assert np.array_equal(np.where(zero[0::2], 0, lo),
                              np.where(zero[0::2], 0, c[0::2]))
        assert np.array_equal(np.where(zero[1::2], 0, hi),
                              np.where(zero[1::2], 0, c[1::2]))
        assert np.array_equal(O.mxfp4_rows_to_f64(row, 128), x)


def test_mxfp4_bound_is_2688(golden_dir):
    fig = _load(golden_dir, "page_figures.json")["e4m3_max"]
    e2, e4 = O.e2m1_value_table(), O.e4m3_value_table()
    assert np.nanmax(np.abs(np.outer(e2, e4))) == fig["fp4_bound"]
    x = np.zeros(32)
    x[3], x[20] = 3000.0, -1e5                 # both groups saturate
    got = O.mxfp4_rows_to_f64(O.mxfp4_encode_rows(_bf16_bits(x)), 32)
    assert got[3] == fig["fp4_bound"] and got[20] == -fig["fp4_bound"]


def test_mxfp4_error_within_one_scale():
    # |x - dequant(x)| <= s: the grid's largest gap is 2 (4 to 6), and a
    # scale rounded down by at most 2^-4 relative overshoots 6 by < 0.4 s
    rng = np.random.default_rng(42)
    x = rng.standard_normal((300, 64)) * np.exp(rng.uniform(-3, 3, (300, 1)))
    x[7] = 0.0
    bits = _bf16_bits(x)
    xb = O.bf16_bits_to_f64(bits)
    rows = O.mxfp4_encode_rows(bits)
    got = O.mxfp4_rows_to_f64(rows, 64)
    s = np.repeat(O.e4m3_codes_to_f64(rows[:, 32:]), 16, axis=1)
    assert np.all(np.abs(xb - got) <= s)
    assert np.all(got[7] == 0)
    amax = np.abs(xb).reshape(300, 4, 16).max(axis=2)
    ok = amax[[i for i in range(300) if i != 7]] / 6
    sc = O.e4m3_codes_to_f64(rows[:, 32:])[[i for i in range(300) if i != 7]]
    assert np.all(np.abs(sc - ok) <= ok * 2.0 ** -4)   # E4M3 rounding


def test_mxfp4_size_against_fp8(golden_dir):
    fig = _load(golden_dir, "page_figures.json")["fp4_vs_fp8_size"]
    saving = 1 - O.mxfp4_row_bytes(128) / 128
    assert abs(saving - fig["value"]) <= fig["abs_tol"]


def test_mxfp4_cache_decodes_as_bf16_values():
    # an MXFP4 cache attends like a bf16 cache holding its decoded values
    # (each is a code times an E4M3 value: <= 5 significant bits, in range)
    rng = np.random.default_rng(43)
    lens = [9, 20]
    kb, vb, bt = _random_paged(rng, 2, 2, 32, 8, lens)
    kr, vr = O.mxfp4_encode_rows(kb), O.mxfp4_encode_rows(vb)
    q = rng.standard_normal((2, 4, 32))
    o1, l1 = O.gqa_decode(q, kr, vr, bt, lens, 8, dtype="mxfp4")
    kv = _bf16_bits(O.mxfp4_rows_to_f64(kr, 32))
    vv = _bf16_bits(O.mxfp4_rows_to_f64(vr, 32))
    assert np.array_equal(O.bf16_bits_to_f64(kv), O.mxfp4_rows_to_f64(kr, 32))
    o2, l2 = O.gqa_decode(q, kv, vv, bt, lens, 8)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_append_mxfp4_writes_one_encoded_row():
    rng = np.random.default_rng(44)
    kb, _, bt = _random_paged(rng, 2, 2, 32, 8, [5, 9])
    kr = O.mxfp4_encode_rows(kb)
    new = _bf16_bits(rng.standard_normal((2, 2, 32)) * 5)
    out = O.kv_append(kr, bt, [4, 8], new, 8, dtype="mxfp4")
    for b, p in enumerate([4, 8]):
        assert np.array_equal(out[bt[b, p // 8], :, p % 8, :],
                              O.mxfp4_encode_rows(new[b]))
    assert np.count_nonzero(np.any(out != kr, axis=3)) <= 4


# ---------------------------------------------------------------------------
# hierarchical indexer pool ("890 bytes a token ...", section 4)
# ---------------------------------------------------------------------------
def test_pool_capacity_is_the_page_figure(golden_dir):
    fig = _load(golden_dir, "page_figures.json")["indexer_pool"]
    assert O.POOL_CAP == fig["blocks"]
    assert O.POOL_BLOCK == fig["positions_per_block"]
    assert O.POOL_CAP * O.POOL_BLOCK == fig["candidates"] == 16384


def test_pool_is_the_set_of_selected_blocks():
    rng = np.random.default_rng(60)
    lens = [1000, 37, 0, 5000]
    idx = np.full((4, 300), -1, dtype=np.int64)
    for b, L in enumerate(lens):
        n = min(L, int(rng.integers(0, 300)))
        if n:
            idx[b, :n] = np.sort(rng.choice(L + 40, n, replace=False))
    pools = O.indexer_pool(idx, lens)
    for b, L in enumerate(lens):
        want = sorted({int(t) // 8 for t in idx[b] if 0 <= t < L})
        assert list(pools[b]) == want
        cand = O.pool_positions(pools[b], L)
        assert list(cand) == [p for p in range(L) if p // 8 in set(want)]
        for t in idx[b]:                      # every selection is a candidate
            if 0 <= t < L:
                assert t in set(cand)


def test_pool_cap_keeps_the_lowest_blocks():
    idx = np.arange(0, 8 * 3000, 8)[None, :]             # 3000 blocks
    pools = O.indexer_pool(idx, [8 * 3000])
    assert list(pools[0]) == list(range(2048))


def _pool_case(seed, lens, k_full, bs=8, d=8):
    rng = np.random.default_rng(seed)
    ir, _, bt = _random_paged(rng, len(lens), 1, d, bs, lens)
    qI = rng.standard_normal((len(lens), 2, d))
    w = rng.uniform(0, 1, (len(lens), 2))
    full, _ = O.indexer_topk(qI, w, ir, bt, lens, bs, k_full)
    return ir, bt, qI, w, full


def test_topk_in_full_pool_equals_full_topk():
    lens = [50, 123]
    ir, bt, qI, w, _ = _pool_case(61, lens, 4)
    pools = [np.arange((L + 7) // 8) for L in lens]      # every block
    a, _ = O.indexer_topk_in_pool(qI, w, ir, bt, lens, 8, pools, 9)
    b, _ = O.indexer_topk(qI, w, ir, bt, lens, 8, 9)
    assert np.array_equal(a, b)


def test_topk_in_pool_brute_force():
    lens = [90, 200, 13]
    ir, bt, qI, w, full = _pool_case(62, lens, 6)
    pools = O.indexer_pool(full, lens)
    got, cand = O.indexer_topk_in_pool(qI, w, ir, bt, lens, 8, pools, 10)
    scores = O.indexer_scores(qI, w, ir, bt, lens, 8)
    for b, L in enumerate(lens):
        blocks = set(int(t) // 8 for t in full[b] if t >= 0)
        c = [t for t in range(L) if t // 8 in blocks]      # plain loops
        best = sorted(c, key=lambda t: (-scores[b][t], t))[:10]
        want = sorted(best) + [-1] * (10 - len(best))
        assert list(got[b]) == want
        assert all(t == -1 or t // 8 in blocks for t in got[b])


def test_schedule_with_pool():
    rng = np.random.default_rng(63)
    lens = [70, 150]
    bs, k, kp = 8, 12, 5
    kr, vr, bt = _random_paged(rng, 2, 1, 16, bs, lens)
    ir, _, _ = _random_paged(np.random.default_rng(64), 2, 1, 8, bs, lens)
    ir = ir[:kr.shape[0]]
    modes = ["full", "reuse", "reindex", "reindex"]
    q = [rng.standard_normal((2, 4, 16)) for _ in modes]
    qI = [rng.standard_normal((2, 4, 8)) for _ in modes]
    w = [rng.uniform(0, 1, (2, 4)) for _ in modes]
    _, _, sel = O.sparse_schedule(modes, q, qI, w, kr, vr, ir, bt, lens, bs,
                                  k, pool_k=kp)
    i0, _ = O.indexer_topk(qI[0], w[0], ir, bt, lens, bs, k)
    pools = O.indexer_pool(i0, lens)
    assert np.array_equal(sel[0], i0) and np.array_equal(sel[1], i0)
    for layer in (2, 3):
        want, _ = O.indexer_topk_in_pool(qI[layer], w[layer], ir, bt, lens,
                                         bs, pools, kp)
        assert np.array_equal(sel[layer], want)
        assert sel[layer].shape == (2, kp)


# ---------------------------------------------------------------------------
# sliding window ("890 bytes a token ...", section 7)
# ---------------------------------------------------------------------------
def test_window_is_attention_over_the_last_w_positions():
    rng = np.random.default_rng(80)
    lens = [1, 7, 40, 130]
    kr, vr, bt = _random_paged(rng, 4, 2, 8, 8, lens)
    q = rng.standard_normal((4, 4, 8))
    W, starts = 16, [0, 3, 30, 2]
    got, lse = O.gqa_decode(q, kr, vr, bt, lens, 8, window=W,
                            window_start=starts)
    for b, T in enumerate(lens):
        lo = max(starts[b], T - W)
        K = O.bf16_bits_to_f64(kr[bt[b, np.arange(lo, T) // 8], :,
                                  np.arange(lo, T) % 8, :])
        V = O.bf16_bits_to_f64(vr[bt[b, np.arange(lo, T) // 8], :,
                                  np.arange(lo, T) % 8, :])
        for h in range(4):
            kv = h // 2                               # group of 2
            s = (K[:, kv, :] @ q[b, h]) / math.sqrt(8)
            wgt = np.exp(s - s.max())
            ref = (wgt / wgt.sum()) @ V[:, kv, :]
            np.testing.assert_allclose(got[b, h], ref, atol=1e-12)
    # a window at least the length is plain decode
    full, _ = O.gqa_decode(q, kr, vr, bt, lens, 8)
    w_all, _ = O.gqa_decode(q, kr, vr, bt, lens, 8, window=200)
    np.testing.assert_allclose(w_all, full, atol=0)


# ---------------------------------------------------------------------------
# copy-on-write prefix sharing ("KV cache", "The allocator, not the
# algorithm")
# ---------------------------------------------------------------------------
def test_cow_fork_shares_and_append_copies_once():
    pool = O.CowPool(10)
    a = pool.new_sequence("a", 3, payload=["a0", "a1", "a2"])
    assert a == [0, 1, 2] and pool.free_blocks() == list(range(3, 10))
    pool.fork("a", "b")                          # a prefix shared, no copy
    assert [pool.refcount(x) for x in a] == [2, 2, 2]
    assert pool.blocks_used() == 3
    # b appends into its last block (slot 2 * 16 + 5): one copy, to block 3
    cp = pool.prepare_append("b", 2 * 16 + 5, 16)
    assert cp == (2, 3)
    assert pool.tables["a"] == [0, 1, 2] and pool.tables["b"] == [0, 1, 3]
    assert pool.data[3] == "a2" and pool.data[2] == "a2"   # a's view kept
    assert pool.refcount(2) == 1 and pool.refcount(3) == 1
    # the same append again: the block is private now
    assert pool.prepare_append("b", 2 * 16 + 6, 16) is None
    # a new block past the table: fresh, nothing to copy
    assert pool.prepare_append("a", 3 * 16, 16) is None
    assert pool.tables["a"][3] == 4
    pool.drop("a")
    assert pool.refcount(2) == 0 and 2 in pool.free_blocks()
    assert pool.refcount(0) == 1                 # still held by b


def test_cow_refcounts_are_table_counts():
    rng = np.random.default_rng(90)
    pool = O.CowPool(64)
    names = []
    for step in range(200):
        op = rng.integers(4)
        if op == 0 or not names:
            n = f"s{step}"
            try:
                pool.new_sequence(n, int(rng.integers(1, 4)))
                names.append(n)
            except MemoryError:
                pass
        elif op == 1:
            n = f"f{step}"
            pool.fork(names[rng.integers(len(names))], n)
            names.append(n)
        elif op == 2:
            n = names[rng.integers(len(names))]
            try:
                pool.prepare_append(n, int(rng.integers(0, 6 * 8)), 8)
            except MemoryError:
                pass
        else:
            pool.drop(names.pop(rng.integers(len(names))))
        counts = {}
        for t in pool.tables.values():
            for b in t:
                if b >= 0:
                    counts[b] = counts.get(b, 0) + 1
        for b in range(64):
            assert pool.refcount(b) == counts.get(b, 0)
        assert len(pool.free_blocks()) == 64 - len(counts)


def test_cow_unshared_blocks_meet_the_waste_bound(golden_dir):
    g = _load(golden_dir, "page_figures.json")["paged_waste"]
    bs, Lbar = g["block_size"], g["mean_len"]
    rng = np.random.default_rng(91)
    lens = rng.integers(1, 2 * Lbar, 64)
    pool = O.CowPool(int(sum(lens)) // bs + 200)
    for i, L in enumerate(lens):                 # append token by token
        pool.tables[f"s{i}"] = []
        for p in range(int(L)):
            pool.prepare_append(f"s{i}", p, bs)
    used = pool.blocks_used()
    assert used == O.blocks_for_lengths(lens, bs)
    waste = used * bs - int(sum(lens))
    assert waste == int(O.paged_waste_slots(lens, bs).sum())
    assert waste <= len(lens) * (bs - 1)
