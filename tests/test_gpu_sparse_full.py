"""The top-k sparse workload's whole 8-layer schedule at full size (B = 8
sequences of 131,072 cached positions, k = 2,048, Full / Reuse x3 /
Reindex x4 over one shared main cache and one shared indexer cache,
"890 bytes a token ...", section 3), run through
schedule.sparse_schedule_step as the bench runs it, and checked layer by
layer:

  * the indices each scoring layer attended to equal the oracle's selection
    rule (top k by score, equal scores to the lower position, ascending)
    applied to the scores the GPU computed for that layer, for every
    sequence (bit-exact), and a Reuse layer attends to the indices of the
    layer before it;
  * one sampled sequence's outputs and log-sum-exps per layer equal the
    fp64 oracle's sparse decode over those indices, at the stated tolerance.

Only the selected rows of the sampled sequence are generated on the host
(the input generator gives any element from its flat physical index)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import kv_cache_decode_gqa_gb300 as K  # noqa: E402
from kv_cache_decode_gqa_gb300 import inputs as I  # noqa: E402
from kv_cache_decode_gqa_gb300 import schedule as S  # noqa: E402
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


def _selected_rows(s, pg, b, positions, tensor, new_bits):
    """bf16 bits [len(positions)][d] of sequence b's rows at `positions`
    of the shared main cache (tensor T_K or T_V), the appended row taken
    from this step's new key / value."""
    d = s.head_dim
    pos = np.asarray(positions, dtype=np.int64)
    blk = pg.table[b][pos // s.block_size].astype(np.uint64)
    row = blk * np.uint64(s.block_size) + (pos % s.block_size).astype(
        np.uint64)
    flat = (row[:, None] * np.uint64(d) + np.arange(d, dtype=np.uint64))
    bits = I.host_fill(I.normal_bf16_table(), W._key(s, 0, tensor),
                       flat.reshape(-1)).reshape(len(pos), d)
    bits = bits.astype(np.uint16)
    bits[pos == s.lengths[b]] = new_bits
    return bits


@pytest.mark.parametrize("pooled", [False, True], ids=["sparse", "pool"])
def test_full_size_schedule(pooled):
    s = W.config("sparse_pool" if pooled else "sparse")
    wl = W.DeviceWorkload(s)
    L = len(s.modes)
    dev = "cuda"
    outs = [torch.empty((s.batch, s.n_h, s.head_dim), dtype=torch.bfloat16,
                        device=dev) for _ in range(L)]
    lses = [torch.empty((s.batch, s.n_h), dtype=torch.float32, device=dev)
            for _ in range(L)]
    idxs = [torch.empty((s.batch, s.pool_k if pooled and m == "reindex"
                         else s.topk), dtype=torch.int32, device=dev)
            for m in s.modes]
    used = S.sparse_schedule_step(
        s.modes, wl.caches[0], wl.idx_cache, wl.block_table, wl.pos,
        wl.seq_lens, wl.max_seq_len, [wl.q[l] for l in range(L)], wl.q_idx,
        wl.w, s.topk, outs, idxs, k_new=wl.k_new[0], v_new=wl.v_new[0],
        idx_k_new=wl.idx_k_new, lses=lses, pool_k=s.pool_k)
    torch.cuda.synchronize()
    used = [u.cpu().numpy() for u in used]

    # indices: the oracle's rule on the GPU's own scores, every sequence
    pool = pool_n = None
    for l, mode in enumerate(s.modes):
        if mode == "reuse":
            assert np.array_equal(used[l], used[l - 1]), f"layer {l}"
            continue
        if mode == "reindex" and pooled:
            sc = torch.empty((s.batch, K.POOL_BLOCKS * K.POOL_BLOCK),
                             dtype=torch.float32, device=dev)
            idx2, _ = K.indexer_topk_pool(
                wl.idx_cache, wl.block_table, wl.seq_lens, wl.max_seq_len,
                wl.q_idx[l], wl.w[l], pool, pool_n, s.pool_k, scores=sc)
            torch.cuda.synchronize()
            sc = sc.cpu().numpy()
            pl, pn = pool.cpu().numpy(), pool_n.cpu().numpy()
            for b in range(s.batch):
                cand = (pl[b, :pn[b], None] * 8 + np.arange(8)).reshape(-1)
                sel = oracle.topk_select(sc[b, :cand.size], s.pool_k)
                want = np.where(sel >= 0, cand[np.maximum(sel, 0)], -1)
                assert np.array_equal(used[l][b], want), (l, b)
        else:
            sc = torch.empty((s.batch, wl.max_seq_len), dtype=torch.float32,
                             device=dev)
            idx2, _ = K.indexer_topk(wl.idx_cache, wl.block_table,
                                     wl.seq_lens, wl.max_seq_len, wl.q_idx[l],
                                     wl.w[l], s.topk, scores=sc)
            torch.cuda.synchronize()
            sc = sc.cpu().numpy()
            for b in range(s.batch):
                want = oracle.topk_select(sc[b, :s.seq_lens[b]], s.topk)
                assert np.array_equal(used[l][b], want), (l, b)
            if mode == "full" and pooled and pool is None:
                pool, pool_n = K.indexer_pool(wl.block_table, wl.seq_lens,
                                              wl.max_seq_len, idx2)
        assert np.array_equal(idx2.cpu().numpy(), used[l]), f"layer {l}"

    # outputs of one sampled sequence, every layer, against the oracle
    b = 5
    T = s.seq_lens[b]
    kn = W.host_bf16(s, 0, W.T_KNEW, (s.batch, 1, s.head_dim))[b, 0]
    vn = W.host_bf16(s, 0, W.T_VNEW, (s.batch, 1, s.head_dim))[b, 0]
    for l in range(L):
        sel = used[l][b]
        pos = np.unique(sel[(sel >= 0) & (sel < T)])
        kr = _selected_rows(s, wl.paging, b, pos, W.T_K, kn)
        vr = _selected_rows(s, wl.paging, b, pos, W.T_V, vn)
        # a compact cache of the selected rows: position pos[i] in row i
        table = np.zeros((1, T), dtype=np.int64)
        table[0, pos] = np.arange(pos.size)
        q = oracle.bf16_bits_to_f64(W.host_bf16(
            s, l, W.T_Q, (s.batch, s.n_h, s.head_dim)))[[b]]
        ref, ref_lse = oracle.sparse_decode(
            q, kr[:, None, None, :], vr[:, None, None, :], table, [T], 1,
            sel[None, :])
        H.assert_close(H.to_np_bf16(outs[l])[[b]], ref, f"layer {l}")
        H.assert_lse_close(lses[l].cpu().numpy()[[b]], ref_lse, f"lse {l}")
