"""Plant plausible mistakes in the oracle (on the CPU, one at a time) and
check that the pins in test_oracle_pins.py catch each of them."""
import numpy as np
import pytest

import oracle
import oracle.attention as OA
import tests.test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(oracle, name, fn)
    monkeypatch.setattr(OA, name, fn)


def _fails(test, *args):
    with pytest.raises(AssertionError):
        test(*args)


def test_dropped_scale_is_caught(monkeypatch, golden_dir):
    orig = OA.attend
    _patch(monkeypatch, "attend", lambda q, K, V, s: orig(q, K, V, 1.0))
    _fails(P.test_worked_examples, golden_dir)


def test_values_swapped_for_keys_is_caught(monkeypatch, golden_dir):
    orig = OA.attend
    _patch(monkeypatch, "attend", lambda q, K, V, s: orig(q, K, K, s)
           if K.shape == V.shape else orig(q, K, V, s))
    _fails(P.test_worked_examples, golden_dir)


def test_wrong_group_map_is_caught(monkeypatch):
    orig = OA.gqa_decode

    def mutant(q, k_raw, v_raw, *a, **kw):
        # query head h reads KV head h % n_kv instead of h // g
        n_h, n_kv = q.shape[1], k_raw.shape[1]
        g = n_h // n_kv
        perm = np.array([(h % n_kv) * g + h // n_kv for h in range(n_h)])
        out, lse = orig(q[:, perm], k_raw, v_raw, *a, **kw)
        inv = np.argsort(perm)
        return out[:, inv], lse[:, inv]
    _patch(monkeypatch, "gqa_decode", mutant)
    _fails(P.test_gqa_equals_mha_on_repeated_heads)


def test_off_by_one_length_is_caught(monkeypatch):
    orig = OA.gqa_decode

    def mutant(q, k_raw, v_raw, bt, seq_lens, *a, **kw):
        return orig(q, k_raw, v_raw, bt, np.maximum(np.asarray(seq_lens) - 1,
                                                     1), *a, **kw)
    _patch(monkeypatch, "gqa_decode", mutant)
    _fails(P.test_cached_decode_equals_full_recompute, 4, 4)


def test_ties_to_higher_index_are_caught(monkeypatch, golden_dir):
    orig = OA.topk_select

    def mutant(s, k):
        s = np.asarray(s, dtype=np.float64)
        T = s.shape[0]
        r = orig(s[::-1], k)
        return np.array(sorted(T - 1 - i for i in r if i >= 0)
                        + [-1] * int((r < 0).sum()), dtype=np.int32)
    _patch(monkeypatch, "topk_select", mutant)
    _fails(P.test_topk_golden, golden_dir)


def test_dropped_rope_term_is_caught(monkeypatch):
    orig = OA.mla_decode

    def mutant(q, lat_raw, bt, seq_lens, bs, d_c=512, scale=None):
        q = np.array(q, dtype=np.float64)
        q[..., d_c:] = 0
        return orig(q, lat_raw, bt, seq_lens, bs, d_c=d_c, scale=scale)
    _patch(monkeypatch, "mla_decode", mutant)
    _fails(P.test_mla_absorbed_equals_explicit)


def test_missing_relu_is_caught(monkeypatch):
    orig = OA.indexer_scores

    def mutant(q_idx, w, idx_raw, bt, seq_lens, bs):
        # plain weighted sum of dot products, without the ReLU
        out = []
        for b in range(len(seq_lens)):
            pos = np.arange(int(seq_lens[b]))
            Kx = oracle.bf16_bits_to_f64(OA.gather_rows(idx_raw, bt[b], pos,
                                                        bs))[0]
            out.append((Kx @ np.asarray(q_idx[b]).T) @ np.asarray(w[b]))
        return out
    assert orig is not mutant
    _patch(monkeypatch, "indexer_scores", mutant)
    _fails(P.test_indexer_brute_force)


def test_merge_without_rescale_is_caught(monkeypatch):
    def mutant(parts):
        outs = np.stack([o for o, _ in parts])
        lses = np.stack([l for _, l in parts])
        return outs.mean(axis=0), lses.max(axis=0)
    _patch(monkeypatch, "lse_merge", mutant)
    _fails(P.test_split_merge_equals_unsplit)


def test_fp8_ties_away_from_zero_are_caught(monkeypatch):
    import oracle.numerics as ON
    orig = ON.e4m3_encode_f32

    def mutant(x):
        x = np.asarray(x, dtype=np.float32)
        bumped = np.nextafter(x, np.float32(np.inf) * np.sign(x),
                              dtype=np.float32)
        return orig(np.where(x != 0, bumped, x))
    monkeypatch.setattr(oracle, "e4m3_encode_f32", mutant)
    _fails(P.test_e4m3_encode_midpoints_ties_to_even)


def test_fp4_ties_away_from_zero_are_caught(monkeypatch):
    import oracle.numerics as ON
    orig = ON.e2m1_encode_f32

    def mutant(x):
        x = np.asarray(x, dtype=np.float32)
        bumped = np.nextafter(x, np.float32(np.inf) * np.sign(x),
                              dtype=np.float32)
        return orig(np.where(x != 0, bumped, x))
    monkeypatch.setattr(oracle, "e2m1_encode_f32", mutant)
    monkeypatch.setattr(ON, "e2m1_encode_f32", mutant)
    _fails(P.test_e2m1_encode_midpoints_ties_to_even)


def test_fp4_sign_dropped_is_caught(monkeypatch):
    import oracle.numerics as ON
    orig = ON.e2m1_encode_f32
    mutant = lambda x: orig(np.abs(np.asarray(x, dtype=np.float32)))
    monkeypatch.setattr(oracle, "e2m1_encode_f32", mutant)
    monkeypatch.setattr(ON, "e2m1_encode_f32", mutant)
    _fails(P.test_e2m1_encode_saturates_and_signs)


def test_fp4_nibbles_swapped_is_caught(monkeypatch):
    # encoder and decoder agree with each other, but not with the layout
    import oracle.numerics as ON
    enc, dec = ON.mxfp4_encode_rows, ON.mxfp4_rows_to_f64

    def swap(row, d):
        row = np.array(row, dtype=np.uint8)
        c = row[..., :d // 2]
        row[..., :d // 2] = (c >> 4) | ((c & 0xF) << 4)
        return row
    monkeypatch.setattr(oracle, "mxfp4_encode_rows",
                        lambda bits: swap(enc(bits), np.shape(bits)[-1]))
    monkeypatch.setattr(oracle, "mxfp4_rows_to_f64",
                        lambda raw, d: dec(swap(raw, d), d))
    _fails(P.test_mxfp4_scaled_grid_round_trips)


def test_fp4_scale_from_amax_over_4_is_caught(monkeypatch):
    import oracle.numerics as ON

    def mutant(bits):
        x = ON.bf16_bits_to_f64(bits).astype(np.float32)
        d = x.shape[-1]
        g = x.reshape(x.shape[:-1] + (d // 16, 16))
        amax = np.fmax.reduce(np.abs(g), axis=-1).astype(np.float32)
        sc = ON.e4m3_encode_f32((amax / np.float32(4.0)).astype(np.float32))
        s = ON.e4m3_codes_to_f64(sc).astype(np.float32)[..., None]
        q = (g / np.where(s > 0, s, np.float32(1))).astype(np.float32)
        codes = np.where(s > 0, ON.e2m1_encode_f32(q), 0).astype(np.uint8)
        codes = codes.reshape(x.shape)
        packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
        return np.concatenate([packed, sc], axis=-1)
    monkeypatch.setattr(oracle, "mxfp4_encode_rows", mutant)
    _fails(P.test_mxfp4_scaled_grid_round_trips)


def test_pool_of_16_position_blocks_is_caught(monkeypatch):
    def mutant(indices, seq_lens, cap=2048):
        return [np.unique(np.asarray(r)[(np.asarray(r) >= 0)
                                        & (np.asarray(r) < L)] // 16)[:cap]
                for r, L in zip(indices, seq_lens)]
    _patch(monkeypatch, "indexer_pool", mutant)
    _fails(P.test_pool_is_the_set_of_selected_blocks)


def test_reindex_ignoring_the_pool_is_caught(monkeypatch):
    def mutant(q_idx, w, idx_raw, bt, seq_lens, bs, pools, k):
        return OA.indexer_topk(q_idx, w, idx_raw, bt, seq_lens, bs, k)
    _patch(monkeypatch, "indexer_topk_in_pool", mutant)
    _fails(P.test_topk_in_pool_brute_force)


def test_window_one_position_too_wide_is_caught(monkeypatch):
    orig = OA.gqa_decode

    def mutant(*a, window=0, **kw):
        return orig(*a, window=window + 1 if window else 0, **kw)
    _patch(monkeypatch, "gqa_decode", mutant)
    _fails(P.test_window_is_attention_over_the_last_w_positions)


def test_append_into_a_shared_block_without_copy_is_caught(monkeypatch):
    def mutant(self, name, pos, block_size):
        table = self.tables[name]
        lb = pos // block_size
        while len(table) <= lb:
            table.append(-1)
        if table[lb] < 0:
            table[lb] = self.free_blocks()[0]
        return None                              # writes in place
    monkeypatch.setattr(oracle.CowPool, "prepare_append", mutant)
    _fails(P.test_cow_fork_shares_and_append_copies_once)


def test_fork_that_copies_is_caught(monkeypatch):
    def mutant(self, src, name):
        self.new_sequence(name, len(self.tables[src]))
    monkeypatch.setattr(oracle.CowPool, "fork", mutant)
    _fails(P.test_cow_fork_shares_and_append_copies_once)
