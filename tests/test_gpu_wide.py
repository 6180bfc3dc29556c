"""GPU parity of the 64-head-tile kernels through the C ABI: latent (MLA)
decode and top-k sparse (gather) decode, against the fp64 oracle."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import kv_cache_decode_gqa_gb300 as K  # noqa: E402
from kv_cache_decode_gqa_gb300 import inputs as I  # noqa: E402
from kv_cache_decode_gqa_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    K.device_error()
    yield
    assert K.device_error() == 0


# ---------------------------------------------------------------------------
# latent (MLA) decode
# ---------------------------------------------------------------------------
MLA_CASES = [
    # n_h, block_size, cached lengths
    (64, 64, [0, 31, 32, 33, 500]),
    (128, 16, [1, 95, 1000]),
    (128, 128, [2047]),
]


@pytest.mark.parametrize("case", MLA_CASES, ids=["h64", "h128_bs16",
                                                 "h128_bs128"])
def test_mla_small(case):
    n_h, bs, lengths = case
    s = W.config("mla", batch=len(lengths), lengths=lengths, n_h=n_h,
                 block_size=bs)
    wl = W.DeviceWorkload(s)
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, f"mla {case}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"mla {case}")


def test_mla_full_size_sampled():
    s = W.config("mla")
    wl = W.DeviceWorkload(s)
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    seqs = [0, 41, 63]
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0, seqs=seqs)
    H.assert_close(H.to_np_bf16(out)[seqs], ref, "mla full")
    H.assert_lse_close(lse.cpu().numpy()[seqs], ref_lse, "mla full")


# ---------------------------------------------------------------------------
# sparse (gather) decode
# ---------------------------------------------------------------------------
def _index_lists(shape, k, seed):
    """Seeded selections: ascending positions, -1 padding when the
    sequence is shorter than k, and a few lists in scrambled order."""
    out = np.full((shape.batch, k), -1, dtype=np.int32)
    for b, T in enumerate(shape.seq_lens):
        n = min(k, T)
        perm = I.permutation(I.stream_key(seed, b), T)[:n]
        sel = np.sort(perm) if b % 2 == 0 else perm
        out[b, :n] = sel
    return out


def _sparse_oracle(shape, paging, layer_q, idx, seqs, host_rows,
                   seq_lens=None):
    """Oracle over a compact cache of only the selected rows (`seq_lens`:
    the visible lengths, if not the workload's)."""
    q = oracle.bf16_bits_to_f64(layer_q)[seqs]
    lens = shape.seq_lens if seq_lens is None else seq_lens
    outs, lses = [], []
    for j, b in enumerate(seqs):
        sel = idx[b]
        valid = sel[(sel >= 0) & (sel < lens[b])]
        kr, vr = host_rows(b, valid)
        n = len(valid)
        bt = np.arange(n, dtype=np.int64)[None, :] if n else np.zeros((1, 1),
                                                                     np.int64)
        o, l = oracle.sparse_decode(q[j:j + 1], kr, vr, bt, [n], 1,
                                    np.arange(n)[None, :])
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


def _row_source(shape, paging, knew, vnew):
    """Host K and V rows (after this step's append) of chosen positions,
    as [n][1][1][512] caches (block size 1)."""
    def rows(b, positions):
        positions = np.asarray(positions, dtype=np.int64)
        blk = paging.table[b][positions // shape.block_size].astype(np.uint64)
        slot = (positions % shape.block_size).astype(np.uint64)
        base = (blk * np.uint64(shape.block_size) + slot) * np.uint64(512)
        flat = base[:, None] + np.arange(512, dtype=np.uint64)[None, :]
        tab = I.normal_bf16_table()
        kr = I.host_fill(tab, W._key(shape, 0, W.T_K), flat.reshape(-1))
        vr = I.host_fill(tab, W._key(shape, 0, W.T_V), flat.reshape(-1))
        kr = kr.reshape(-1, 1, 1, 512)
        vr = vr.reshape(-1, 1, 1, 512)
        newpos = shape.lengths[b]
        hit = positions == newpos
        kr[hit, 0, 0] = knew[b, 0]
        vr[hit, 0, 0] = vnew[b, 0]
        return kr, vr
    return rows


SPARSE_CASES = [
    # cached lengths, k, block size
    ([10, 100, 700], 64, 64),
    ([31, 64, 2000], 256, 16),
    ([5000], 2048, 64),
]


@pytest.mark.parametrize("case", SPARSE_CASES, ids=["k64", "k256_bs16",
                                                    "k2048"])
def test_sparse_small(case):
    lengths, k, bs = case
    s = W.config("sparse", batch=len(lengths), lengths=lengths, topk=k,
                 block_size=bs, n_layers=1, modes=["full"])
    wl = W.DeviceWorkload(s)
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    idx = _index_lists(s, k, 77)
    out, lse = K.sparse_decode(c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                               torch.from_numpy(idx).cuda(), wl.q[0])
    torch.cuda.synchronize()
    knew = H.host_bits(s, 0, W.T_KNEW, (s.batch, 1, 512))
    vnew = H.host_bits(s, 0, W.T_VNEW, (s.batch, 1, 512))
    qbits = H.host_bits(s, 0, W.T_Q, (s.batch, s.n_h, 512))
    seqs = list(range(s.batch))
    ref, ref_lse = _sparse_oracle(s, wl.paging, qbits, idx, seqs,
                                  _row_source(s, wl.paging, knew, vnew))
    H.assert_close(H.to_np_bf16(out), ref, f"sparse {case}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"sparse {case}")


def _sparse_case(lengths, k, bs, n_h=64, seed=77, idx=None, lens=None):
    """Sparse decode of a small workload (every output compared with the
    oracle); `lens` overrides the visible lengths."""
    s = W.config("sparse", batch=len(lengths), lengths=lengths, topk=k,
                 block_size=bs, n_layers=1, modes=["full"], n_h=n_h)
    wl = W.DeviceWorkload(s)
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    if idx is None:
        idx = _index_lists(s, k, seed)
    seq_lens = wl.seq_lens if lens is None else torch.tensor(
        lens, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_decode(c, wl.block_table, seq_lens, wl.max_seq_len,
                               torch.from_numpy(idx).cuda(), wl.q[0])
    torch.cuda.synchronize()
    knew = H.host_bits(s, 0, W.T_KNEW, (s.batch, 1, 512))
    vnew = H.host_bits(s, 0, W.T_VNEW, (s.batch, 1, 512))
    qbits = H.host_bits(s, 0, W.T_Q, (s.batch, s.n_h, 512))
    seqs = list(range(s.batch))
    ref, ref_lse = _sparse_oracle(s, wl.paging, qbits, idx, seqs,
                                  _row_source(s, wl.paging, knew, vnew),
                                  seq_lens=lens)
    return out, lse, ref, ref_lse


# The tensor-core gather kernel's work split: S CTAs per (sequence, 64-head
# tile). Two head tiles; a k that is no multiple of anything; k smaller
# than the CTAs of a unit (most CTAs get no entry); several 128-entry
# chunks per CTA (the online rescale across chunks, forced with a small CTA
# count); the most CTAs per unit (32, the workspace merge of 32 parts,
# forced with a large CTA count); one CTA per unit (outputs written
# directly).
@pytest.mark.parametrize("lengths,k,bs,n_h,ctas", [
    ([300, 1200, 9], 1000, 64, 128, 0),
    ([40, 3], 5, 16, 64, 0),
    ([6000], 5000, 64, 64, 8),
    ([3000, 2500], 2048, 32, 64, 1024),
    ([9000, 100, 4000, 2], 3000, 64, 64, 4),
    ([9000, 100, 4000, 2], 3000, 64, 64, 16),
], ids=["h128_k1000", "k5", "chunks_per_cta", "splits_max", "b4_s1",
        "b4_s4"])
def test_sparse_work_splits(lengths, k, bs, n_h, ctas):
    K.set_tuning(decode_ctas=ctas)
    try:
        out, lse, ref, ref_lse = _sparse_case(lengths, k, bs, n_h)
    finally:
        K.set_tuning()
    H.assert_close(H.to_np_bf16(out), ref, f"sparse {lengths} k={k}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"sparse {lengths} lse")


def test_sparse_repeats_and_empty_sequence():
    """A list naming some positions twice (each copy counts, as in the
    oracle), and a sequence with nothing visible (out = 0, lse = -inf)."""
    s_len = [500, 300, 50]
    k = 256
    idx = np.full((3, k), -1, dtype=np.int32)
    rng = np.random.default_rng(5)
    idx[0] = rng.integers(0, 501, k)            # with repeats
    idx[1, :100] = np.arange(100) * 3
    idx[2, :40] = np.arange(40)
    lens = [501, 301, 0]                        # sequence 2: nothing visible
    out, lse, ref, ref_lse = _sparse_case(s_len, k, 64, idx=idx, lens=lens)
    H.assert_close(H.to_np_bf16(out), ref, "repeats / empty")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, "repeats / empty lse")
    assert np.all(H.to_np_bf16(out)[2] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[2]))
    K.device_error()     # entries of sequence 2 are past its length: flagged


def test_sparse_full_size_sampled():
    s = W.config("sparse")
    wl = W.DeviceWorkload(s, layers=[0])
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    idx = _index_lists(s, s.topk, 91)
    out, lse = K.sparse_decode(c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                               torch.from_numpy(idx).cuda(), wl.q[0])
    torch.cuda.synchronize()
    knew = H.host_bits(s, 0, W.T_KNEW, (s.batch, 1, 512))
    vnew = H.host_bits(s, 0, W.T_VNEW, (s.batch, 1, 512))
    qbits = H.host_bits(s, 0, W.T_Q, (s.batch, s.n_h, 512))
    seqs = [0, 5, 7]
    ref, ref_lse = _sparse_oracle(s, wl.paging, qbits, idx, seqs,
                                  _row_source(s, wl.paging, knew, vnew))
    H.assert_close(H.to_np_bf16(out)[seqs], ref, "sparse full")
    H.assert_lse_close(lse.cpu().numpy()[seqs], ref_lse, "sparse full")


def test_sparse_index_past_length_is_flagged():
    s = W.config("sparse", batch=1, lengths=[100], topk=32, n_layers=1,
                 modes=["full"])
    wl = W.DeviceWorkload(s)
    idx = torch.arange(32, dtype=torch.int32, device="cuda")[None, :] * 4
    K.sparse_decode(wl.caches[0], wl.block_table, wl.seq_lens,
                    wl.max_seq_len, idx, wl.q[0])
    assert K.device_error() & 8          # KVD_DEVERR_INDEX (entries >= 101)
