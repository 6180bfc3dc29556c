"""GPU parity of the indexer scores, the top-k selection and the static
Full / Reuse / Reindex schedule, through the C ABI.

Top-k indices are checked bit-exactly in two ways: (i) the oracle's
selection rule applied to the scores the GPU computed must give exactly
the GPU's indices (every shape, full size included); (ii) on an
exact-arithmetic input set (indexer queries and keys in {a/8}, weights in
{1,2,3,4}) every fp32 score is exact, so the GPU's indices must equal the
fp64 oracle's, heavy ties included."""
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


def _shape(lengths, k, bs=64, heads=4, modes=("full",)):
    return W.config("sparse", batch=len(lengths), lengths=list(lengths),
                    topk=k, block_size=bs, idx_heads=heads,
                    n_layers=len(modes), modes=list(modes))


def _exact_inputs(wl, s, layer_keys):
    """Replace the indexer cache, queries and weights by the exact set."""
    tab = I.eighths_bf16_table()
    I.device_fill(wl.idx_cache.k, tab, W._key(s, 0, W.T_IDXK))
    for layer in layer_keys:
        q = I.host_tensor(tab, W._key(s, layer, W.T_QIDX),
                          (s.batch, s.idx_heads, s.idx_dim))
        wl.q_idx[layer] = torch.from_numpy(q.view(np.int16)).view(
            torch.bfloat16).cuda()
        wi = I.uniform_int(W._key(s, layer, W.T_W), s.batch * s.idx_heads, 1, 4)
        wl.w[layer] = torch.from_numpy(
            wi.reshape(s.batch, s.idx_heads).astype(np.float32)).cuda()
    return tab


def _host_idx_cache(s, pg, table):
    return W.host_cache_full(s, pg, 0, W.T_IDXK, width=s.idx_dim, n_kv=1,
                             table=table)


def _run_indexer(wl, layer, scores=True):
    s = wl.shape
    sc = torch.empty((s.batch, max(wl.max_seq_len, 1)), dtype=torch.float32,
                     device="cuda") if scores else None
    idx, sc = K.indexer_topk(wl.idx_cache, wl.block_table, wl.seq_lens,
                             wl.max_seq_len, wl.q_idx[layer], wl.w[layer],
                             s.topk, scores=sc)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), None if sc is None else sc.cpu().numpy()


CASES = [
    # cached lengths, k, block size, indexer heads
    ([5, 63, 64, 200], 64, 64, 4),       # T < k, T == k, T > k
    ([1000, 4000], 256, 16, 4),
    ([3000], 2048, 64, 8),
    ([700, 1500], 100, 32, 1),
    # block sizes below 8 (a 64-entry slice spans more block pieces than a
    # lane resolves ahead) and not powers of two
    ([2000, 130], 100, 1, 4),
    ([500, 1900], 64, 3, 2),
    ([3000, 77], 256, 48, 3),
]


@pytest.mark.parametrize("case", CASES, ids=["small", "bs16", "k2048",
                                             "one_head", "bs1", "bs3",
                                             "bs48"])
def test_scores_and_selection(case):
    lengths, k, bs, heads = case
    s = _shape(lengths, k, bs, heads)
    wl = W.DeviceWorkload(s)
    idx, sc = _run_indexer(wl, 0)
    # scores vs the fp64 oracle
    tab = I.normal_bf16_table()
    ir = _host_idx_cache(s, wl.paging, tab)
    qI = oracle.bf16_bits_to_f64(W.host_bf16(s, 0, W.T_QIDX,
                                             (s.batch, heads, s.idx_dim)))
    w = W.host_weights(s, 0).astype(np.float64)
    ref = oracle.indexer_scores(qI, w, ir, wl.paging.table, s.seq_lens, bs)
    for b, T in enumerate(s.seq_lens):
        np.testing.assert_allclose(sc[b, :T], ref[b], rtol=1e-5, atol=1e-4)
        # (i) the selection the GPU's own scores define, exactly
        want = oracle.topk_select(sc[b, :T].astype(np.float64), k)
        assert np.array_equal(idx[b], want), f"row {b}"


def test_exact_arithmetic_set_matches_fp64_oracle():
    s = _shape([5000, 2000, 64], 512, 64, 4)
    wl = W.DeviceWorkload(s)
    tab = _exact_inputs(wl, s, [0])
    idx, sc = _run_indexer(wl, 0)
    ir = _host_idx_cache(s, wl.paging, tab)
    qI = oracle.bf16_bits_to_f64(I.host_tensor(tab, W._key(s, 0, W.T_QIDX),
                                               (s.batch, 4, 64)))
    w = wl.w[0].cpu().numpy().astype(np.float64)
    ref_idx, ref_sc = oracle.indexer_topk(qI, w, ir, wl.paging.table,
                                          s.seq_lens, 64, 512)
    for b, T in enumerate(s.seq_lens):
        assert np.array_equal(sc[b, :T].astype(np.float64), ref_sc[b])
    assert np.array_equal(idx, ref_idx)
    # the set really has ties at the selection boundary
    b0 = ref_sc[0]
    kth = np.sort(b0)[-512]
    assert (b0 == kth).sum() > 1


def test_full_size_indexer():
    s = W.config("sparse")
    wl = W.DeviceWorkload(s, layers=[0])
    idx, sc = _run_indexer(wl, 0)
    T = s.seq_lens[0]
    for b in range(s.batch):
        want = oracle.topk_select(sc[b, :T].astype(np.float64), s.topk)
        assert np.array_equal(idx[b], want), f"row {b}"
    # sampled sequence: scores against the fp64 oracle
    b = 3
    ir, bt = W.host_cache_compact(s, wl.paging, 0, W.T_IDXK, [b],
                                  width=s.idx_dim, n_kv=1,
                                  table=I.normal_bf16_table())
    qI = oracle.bf16_bits_to_f64(W.host_bf16(s, 0, W.T_QIDX,
                                             (s.batch, 4, 64)))[[b]]
    w = W.host_weights(s, 0)[[b]].astype(np.float64)
    ref = oracle.indexer_scores(qI, w, ir, bt, [T], s.block_size)[0]
    np.testing.assert_allclose(sc[b, :T], ref, rtol=1e-5, atol=1e-4)


def test_many_ragged_sequences():
    """70 sequences of 0 .. 3,000 visible positions (some empty), block
    size 16, two indexer heads: every sequence's scores against the fp64
    oracle and its selection against the oracle's rule on those scores.
    Slices of many sequences share a CTA's run here."""
    rng = np.random.default_rng(71)
    lengths = [int(x) for x in rng.integers(0, 3000, 70)]
    s = _shape(lengths, 128, 16, 2)
    wl = W.DeviceWorkload(s)
    vis = list(s.seq_lens)
    for b in (0, 7, 8, 9, 40, 69):         # empty sequences
        vis[b] = 0
    wl.seq_lens.copy_(torch.tensor(vis, dtype=torch.int32))
    idx, sc = _run_indexer(wl, 0)
    tab = I.normal_bf16_table()
    ir = _host_idx_cache(s, wl.paging, tab)
    qI = oracle.bf16_bits_to_f64(W.host_bf16(s, 0, W.T_QIDX,
                                             (s.batch, 2, s.idx_dim)))
    w = W.host_weights(s, 0).astype(np.float64)
    ref = oracle.indexer_scores(qI, w, ir, wl.paging.table, vis, 16)
    for b, T in enumerate(vis):
        np.testing.assert_allclose(sc[b, :T], ref[b], rtol=1e-5, atol=1e-4)
        want = oracle.topk_select(sc[b, :T].astype(np.float64), 128)
        assert np.array_equal(idx[b], want), f"row {b}"


@pytest.mark.parametrize("kind", ["all_zero", "few_above"])
def test_selection_with_heavy_ties(kind):
    """Long sequences whose scores are mostly 0, so that the bin of the
    k-th largest score holds far more keys than a CTA collects as
    candidates and the selection takes its cluster-wide passes: "all_zero"
    (an all-zero indexer cache: every score 0, the first k positions win)
    and "few_above" (1,000 positions a sequence get key dim 0 in
    {1/8 .. 1}, scores relu(k_t0) with ties among them; the rest of the k
    come from the lowest zero-score positions). The short sequence in the
    same launch takes the candidate path."""
    lengths = [131071, 60000, 3000]
    s = _shape(lengths, 2048, 64, 4)
    wl = W.DeviceWorkload(s)
    kc = wl.idx_cache.k
    kc.zero_()
    if kind == "few_above":
        rng = np.random.default_rng(72)
        for b, T in enumerate(s.seq_lens):
            pos = rng.choice(T, size=1000, replace=False)
            blk = wl.paging.table[b][pos // 64].astype(np.int64)
            vals = torch.from_numpy(rng.integers(1, 9, pos.size) / 8.0)
            kc[torch.from_numpy(blk).cuda(), 0,
               torch.from_numpy(pos % 64).cuda(), 0] = vals.to(
                   torch.bfloat16).cuda()
    q = torch.zeros_like(wl.q_idx[0])
    q[:, 0, 0] = 1.0
    w = torch.zeros_like(wl.w[0])
    w[:, 0] = 1.0
    wl.q_idx[0] = q
    wl.w[0] = w
    idx, sc = _run_indexer(wl, 0)
    ir = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    ref_idx, ref_sc = oracle.indexer_topk(
        q.float().cpu().numpy().astype(np.float64),
        w.cpu().numpy().astype(np.float64), ir, wl.paging.table, s.seq_lens,
        64, 2048)
    for b, T in enumerate(s.seq_lens):
        assert np.array_equal(sc[b, :T].astype(np.float64), ref_sc[b])
        assert (ref_sc[b] == 0).sum() > (8 * 4096 if b == 0 else 0)
    assert np.array_equal(idx, ref_idx)
    if kind == "all_zero":
        assert np.array_equal(idx[0], np.arange(2048))


@pytest.mark.parametrize("flags", [1, 3], ids=["stable", "prefix_ready"])
def test_seqs_flags_after_an_append(flags):
    """kvd_indexer_topk with KVD_SEQS_STABLE (plan made while the kernel
    before finishes) and KVD_SEQS_PREFIX_READY (cached rows copied then
    too), launched right after the append of this step's indexer keys: the
    scores, the newest position's included, equal the fp64 oracle's on the
    appended cache, and the selection is the oracle's rule on them."""
    s = _shape([20000, 3000, 64, 700], 512, 64, 4)
    wl = W.DeviceWorkload(s)
    sc = torch.empty((s.batch, wl.max_seq_len), dtype=torch.float32,
                     device="cuda")
    for _ in range(2):                     # the append runs first each time
        K.kv_append(wl.idx_cache, wl.block_table, wl.pos, wl.idx_k_new)
        idx, _ = K.indexer_topk(wl.idx_cache, wl.block_table, wl.seq_lens,
                                wl.max_seq_len, wl.q_idx[0], wl.w[0], s.topk,
                                scores=sc, seqs_flags=flags)
    torch.cuda.synchronize()
    idx, scn = idx.cpu().numpy(), sc.cpu().numpy()
    ir = _host_idx_cache(s, wl.paging, I.normal_bf16_table())
    xn = W.host_bf16(s, 0, W.T_IDXKNEW, (s.batch, 1, 64))
    ir = oracle.kv_append(ir, wl.paging.table, s.lengths, xn, s.block_size)
    qI = oracle.bf16_bits_to_f64(W.host_bf16(s, 0, W.T_QIDX,
                                             (s.batch, 4, s.idx_dim)))
    w = W.host_weights(s, 0).astype(np.float64)
    ref = oracle.indexer_scores(qI, w, ir, wl.paging.table, s.seq_lens, 64)
    for b, T in enumerate(s.seq_lens):
        np.testing.assert_allclose(scn[b, :T], ref[b], rtol=1e-5, atol=1e-4)
        want = oracle.topk_select(scn[b, :T].astype(np.float64), s.topk)
        assert np.array_equal(idx[b], want), f"row {b}"


def test_schedule_matches_oracle():
    """Full, Reuse x3, Reindex x4 over one main cache and one indexer
    cache (exact indexer inputs, so the selections are identical)."""
    modes = W.SPARSE_MODES
    s = _shape([3000, 900], 128, 64, 4, modes)
    wl = W.DeviceWorkload(s)
    tab = _exact_inputs(wl, s, [l for l, m in enumerate(modes)
                                if m != "reuse"])
    outs = [torch.empty((s.batch, s.n_h, 512), dtype=torch.bfloat16,
                        device="cuda") for _ in modes]
    lses = [torch.empty((s.batch, s.n_h), dtype=torch.float32, device="cuda")
            for _ in modes]
    idxs = [torch.empty((s.batch, s.topk), dtype=torch.int32, device="cuda")
            for _ in modes]
    used = S.sparse_schedule_step(
        modes, wl.caches[0], wl.idx_cache, wl.block_table, wl.pos,
        wl.seq_lens, wl.max_seq_len, [wl.q[l] for l in range(len(modes))],
        wl.q_idx, wl.w, s.topk, outs, idxs, k_new=wl.k_new[0],
        v_new=wl.v_new[0], idx_k_new=wl.idx_k_new, lses=lses)
    torch.cuda.synchronize()
    # oracle: append the new token to the three caches, then the schedule
    pg = wl.paging
    kr = W.host_cache_full(s, pg, 0, W.T_K, n_kv=1)
    vr = W.host_cache_full(s, pg, 0, W.T_V, n_kv=1)
    ir = _host_idx_cache(s, pg, tab)
    kn = W.host_bf16(s, 0, W.T_KNEW, (s.batch, 1, 512))
    vn = W.host_bf16(s, 0, W.T_VNEW, (s.batch, 1, 512))
    xn = W.host_bf16(s, 0, W.T_IDXKNEW, (s.batch, 1, 64))
    kr = oracle.kv_append(kr, pg.table, s.lengths, kn, s.block_size)
    vr = oracle.kv_append(vr, pg.table, s.lengths, vn, s.block_size)
    ir = oracle.kv_append(ir, pg.table, s.lengths, xn, s.block_size)
    qs = [oracle.bf16_bits_to_f64(W.host_bf16(s, l, W.T_Q,
                                              (s.batch, s.n_h, 512)))
          for l in range(len(modes))]
    qIs = [None if m == "reuse" else oracle.bf16_bits_to_f64(
        I.host_tensor(tab, W._key(s, l, W.T_QIDX), (s.batch, 4, 64)))
        for l, m in enumerate(modes)]
    ws = [None if m == "reuse" else wl.w[l].cpu().numpy().astype(np.float64)
          for l, m in enumerate(modes)]
    r_out, r_lse, r_idx = oracle.sparse_schedule(
        modes, qs, qIs, ws, kr, vr, ir, pg.table, s.seq_lens, s.block_size,
        s.topk)
    for l in range(len(modes)):
        assert np.array_equal(used[l].cpu().numpy(), r_idx[l]), f"layer {l}"
        H.assert_close(H.to_np_bf16(outs[l]), r_out[l], f"layer {l}")
        H.assert_lse_close(lses[l].cpu().numpy(), r_lse[l], f"layer {l}")


# ---------------------------------------------------------------------------
# hierarchical indexer pool
# ---------------------------------------------------------------------------
def _gpu_pool(wl, idx_t):
    pool, pool_n = K.indexer_pool(wl.block_table, wl.seq_lens,
                                  wl.max_seq_len, idx_t)
    torch.cuda.synchronize()
    return pool.cpu().numpy(), pool_n.cpu().numpy()


def _check_pool(pool, pool_n, want):
    for b, w in enumerate(want):
        assert pool_n[b] == len(w), (b, pool_n[b], len(w))
        assert np.array_equal(pool[b, :len(w)], w), b


def test_pool_matches_oracle():
    s = _shape([5, 700, 3000, 64], 256, 64, 4)
    wl = W.DeviceWorkload(s)
    idx, _ = _run_indexer(wl, 0, scores=False)
    pool, pool_n = _gpu_pool(wl, torch.from_numpy(idx).cuda())
    _check_pool(pool, pool_n, oracle.indexer_pool(idx, s.seq_lens))
    # any order, repeats and -1 entries
    rng = np.random.default_rng(70)
    sel = np.full((4, 300), -1, dtype=np.int32)
    for b, T in enumerate(s.seq_lens):
        n = min(T, 250)
        sel[b, :n] = rng.integers(0, T, n)        # unsorted, repeats
    rng.shuffle(sel, axis=1)
    pool, pool_n = _gpu_pool(wl, torch.from_numpy(sel).cuda())
    _check_pool(pool, pool_n, oracle.indexer_pool(sel, s.seq_lens))


def test_pool_keeps_the_lowest_2048_blocks():
    s = _shape([30000], 16, 64, 1)
    wl = W.DeviceWorkload(s)
    sel = (np.arange(3500, dtype=np.int32) * 8 + 3)[None, :]   # 3500 blocks
    pool, pool_n = _gpu_pool(wl, torch.from_numpy(sel).cuda())
    assert pool_n[0] == 2048 and np.array_equal(pool[0], np.arange(2048))


def _run_pool_topk(wl, layer, pool_t, pool_n_t, k):
    s = wl.shape
    sc = torch.empty((s.batch, K.POOL_BLOCKS * K.POOL_BLOCK),
                     dtype=torch.float32, device="cuda")
    idx, sc = K.indexer_topk_pool(wl.idx_cache, wl.block_table, wl.seq_lens,
                                  wl.max_seq_len, wl.q_idx[layer],
                                  wl.w[layer], pool_t, pool_n_t, k, scores=sc)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


def _pool_rule_check(idx, sc, pools, lens, k):
    """(i): the oracle's rule on the GPU's candidate scores, exactly."""
    for b, T in enumerate(lens):
        pos = oracle.pool_positions(pools[b], T)
        cand = sc[b, :len(pos)].astype(np.float64)
        sel = oracle.topk_select(cand, k)
        want = np.where(sel >= 0, pos[np.maximum(sel, 0)], -1)
        assert np.array_equal(idx[b], want), f"row {b}"
        assert np.all(sc[b, len(pos):8 * len(pools[b])] == -np.inf)


@pytest.mark.parametrize("lengths,k_full,k,bs", [
    ([5, 63, 300, 2000], 64, 32, 64),      # T < k, pools smaller than k
    ([4000, 1500], 256, 100, 16),
    ([20000], 2048, 512, 64)])
def test_pool_selection(lengths, k_full, k, bs):
    s = _shape(lengths, k_full, bs, 4, modes=("full", "reindex"))
    wl = W.DeviceWorkload(s)
    full, _ = _run_indexer(wl, 0, scores=False)
    pool_t, pool_n_t = K.indexer_pool(wl.block_table, wl.seq_lens,
                                      wl.max_seq_len,
                                      torch.from_numpy(full).cuda())
    idx, sc = _run_pool_topk(wl, 1, pool_t, pool_n_t, k)
    pools = oracle.indexer_pool(full, s.seq_lens)
    _pool_rule_check(idx, sc, pools, s.seq_lens, k)
    # candidate scores against the fp64 oracle
    ir = _host_idx_cache(s, wl.paging, I.normal_bf16_table())
    qI = oracle.bf16_bits_to_f64(W.host_bf16(s, 1, W.T_QIDX,
                                             (s.batch, 4, s.idx_dim)))
    w = W.host_weights(s, 1).astype(np.float64)
    _, cand = oracle.indexer_topk_in_pool(qI, w, ir, wl.paging.table,
                                          s.seq_lens, bs, pools, k)
    for b in range(s.batch):
        np.testing.assert_allclose(sc[b, :len(cand[b])], cand[b], rtol=1e-5,
                                   atol=1e-4)


def test_pool_selection_exact_set_matches_fp64_oracle():
    s = _shape([6000, 900], 512, 64, 4, modes=("full", "reindex"))
    wl = W.DeviceWorkload(s)
    tab = _exact_inputs(wl, s, [0, 1])
    full, _ = _run_indexer(wl, 0, scores=False)
    pool_t, pool_n_t = K.indexer_pool(wl.block_table, wl.seq_lens,
                                      wl.max_seq_len,
                                      torch.from_numpy(full).cuda())
    idx, _ = _run_pool_topk(wl, 1, pool_t, pool_n_t, 128)
    ir = _host_idx_cache(s, wl.paging, tab)
    qs = [oracle.bf16_bits_to_f64(I.host_tensor(tab, W._key(s, l, W.T_QIDX),
                                                (s.batch, 4, 64)))
          for l in (0, 1)]
    ws = [wl.w[l].cpu().numpy().astype(np.float64) for l in (0, 1)]
    ref_full, _ = oracle.indexer_topk(qs[0], ws[0], ir, wl.paging.table,
                                      s.seq_lens, 64, 512)
    assert np.array_equal(full, ref_full)
    ref, _ = oracle.indexer_topk_in_pool(
        qs[1], ws[1], ir, wl.paging.table, s.seq_lens, 64,
        oracle.indexer_pool(ref_full, s.seq_lens), 128)
    assert np.array_equal(idx, ref)


def test_schedule_with_pool_matches_oracle():
    """Full, Reuse, Reindex x2 with a pool (Reindex layers pick 48 inside
    the Full layer's pool), exact indexer inputs."""
    modes = ["full", "reuse", "reindex", "reindex"]
    kp = 48
    s = _shape([3000, 900], 128, 64, 4, modes)
    wl = W.DeviceWorkload(s)
    tab = _exact_inputs(wl, s, [0, 2, 3])
    outs = [torch.empty((s.batch, s.n_h, 512), dtype=torch.bfloat16,
                        device="cuda") for _ in modes]
    idxs = [torch.empty((s.batch, kp if m == "reindex" else s.topk),
                        dtype=torch.int32, device="cuda") for m in modes]
    used = S.sparse_schedule_step(
        modes, wl.caches[0], wl.idx_cache, wl.block_table, wl.pos,
        wl.seq_lens, wl.max_seq_len, [wl.q[l] for l in range(len(modes))],
        wl.q_idx, wl.w, s.topk, outs, idxs, pool_k=kp)
    torch.cuda.synchronize()
    pg = wl.paging
    kr = W.host_cache_full(s, pg, 0, W.T_K, n_kv=1)
    vr = W.host_cache_full(s, pg, 0, W.T_V, n_kv=1)
    ir = _host_idx_cache(s, pg, tab)
    qs = [oracle.bf16_bits_to_f64(W.host_bf16(s, l, W.T_Q,
                                              (s.batch, s.n_h, 512)))
          for l in range(len(modes))]
    qIs = [None if m == "reuse" else oracle.bf16_bits_to_f64(
        I.host_tensor(tab, W._key(s, l, W.T_QIDX), (s.batch, 4, 64)))
        for l, m in enumerate(modes)]
    ws = [None if m == "reuse" else wl.w[l].cpu().numpy().astype(np.float64)
          for l, m in enumerate(modes)]
    # no append in this step: the caches as drawn, the same visible lengths
    r_out, _, r_idx = oracle.sparse_schedule(
        modes, qs, qIs, ws, kr, vr, ir, pg.table, s.seq_lens, s.block_size,
        s.topk, pool_k=kp)
    for l in range(len(modes)):
        assert np.array_equal(used[l].cpu().numpy(), r_idx[l]), f"layer {l}"
        H.assert_close(H.to_np_bf16(outs[l]), r_out[l], f"layer {l}")


def test_full_size_pool():
    s = W.config("sparse")
    wl = W.DeviceWorkload(s, layers=[0, 4])
    full, _ = _run_indexer(wl, 0, scores=False)
    pool_t, pool_n_t = K.indexer_pool(wl.block_table, wl.seq_lens,
                                      wl.max_seq_len,
                                      torch.from_numpy(full).cuda())
    idx, sc = _run_pool_topk(wl, 4, pool_t, pool_n_t, 512)
    pools = oracle.indexer_pool(full, s.seq_lens)
    _check_pool(pool_t.cpu().numpy(), pool_n_t.cpu().numpy(), pools)
    _pool_rule_check(idx, sc, pools, s.seq_lens, 512)
