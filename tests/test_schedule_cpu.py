"""The sparse path's static layer schedule as host logic: which C-ABI call
each layer makes, with which index set, in what order ("890 bytes a token
...", sections 3 and 4). The kernels are replaced by recorders, so this runs
without a GPU; the GPU tests check the same schedule's numbers."""
import pytest

from kv_cache_decode_gqa_gb300 import schedule as S
from kv_cache_decode_gqa_gb300 import workloads as W


class _Recorder:
    def __init__(self, monkeypatch):
        self.calls = []
        for name in ("kv_append", "indexer_topk", "indexer_pool",
                     "indexer_topk_pool", "sparse_decode"):
            monkeypatch.setattr(S, name, self._make(name))

    def _make(self, name):
        def call(*args, **kw):
            self.calls.append((name, args, kw))
            if name == "indexer_pool":
                return "POOL", "POOL_N"
        return call

    def names(self):
        return [c[0] for c in self.calls]


def _step(modes, **kw):
    L = len(modes)
    return S.sparse_schedule_step(
        modes, "cache", "idx_cache", "bt", "pos", "lens", 99,
        q=[f"q{l}" for l in range(L)], q_idx=[f"qi{l}" for l in range(L)],
        w=[f"w{l}" for l in range(L)], k=2048,
        outs=[f"out{l}" for l in range(L)],
        indices=[f"ind{l}" for l in range(L)], **kw)


def test_workload_schedule_is_one_full_three_reuse_four_reindex():
    assert W.config("sparse").modes == ["full"] + ["reuse"] * 3 + \
        ["reindex"] * 4


def test_full_reuse_reindex_calls(monkeypatch):
    rec = _Recorder(monkeypatch)
    modes = W.config("sparse").modes
    used = _step(modes, k_new="kn", v_new="vn", idx_k_new="ikn")
    # the new token goes into the main and the indexer caches first
    assert rec.names()[:2] == ["kv_append", "kv_append"]
    assert rec.calls[0][1][:5] == ("cache", "bt", "pos", "kn", "vn")
    assert rec.calls[1][1][:4] == ("idx_cache", "bt", "pos", "ikn")
    # 5 selections (Full + 4 Reindex), 8 gathers, nothing else
    assert rec.names()[2:] == (["indexer_topk", "sparse_decode"]
                               + ["sparse_decode"] * 3
                               + ["indexer_topk", "sparse_decode"] * 4)
    # Reuse layers attend to the Full layer's selection
    assert used == ["ind0"] * 4 + ["ind4", "ind5", "ind6", "ind7"]
    gathers = [c for c in rec.calls if c[0] == "sparse_decode"]
    for layer, (_, args, kw) in enumerate(gathers):
        assert args[4] == used[layer] and args[5] == f"q{layer}"
        assert kw["out"] == f"out{layer}"
    # each selection scores with its own layer's indexer query and weights
    sel = [c for c in rec.calls if c[0] == "indexer_topk"]
    assert [(c[1][4], c[1][5], c[1][6]) for c in sel] == \
        [("qi0", "w0", 2048)] + [(f"qi{l}", f"w{l}", 2048) for l in (4, 5, 6, 7)]


def test_pool_schedule(monkeypatch):
    rec = _Recorder(monkeypatch)
    modes = W.config("sparse").modes
    used = _step(modes, pool_k=512)
    # the Full layer publishes the pool once; Reindex layers select inside it
    assert rec.names() == (["indexer_topk", "indexer_pool", "sparse_decode"]
                           + ["sparse_decode"] * 3
                           + ["indexer_topk_pool", "sparse_decode"] * 4)
    assert rec.calls[1][1][3] == "ind0"            # the pool of layer 0's pick
    for c in rec.calls:
        if c[0] == "indexer_topk_pool":
            assert c[1][6:9] == ("POOL", "POOL_N", 512)
    assert used == ["ind0"] * 4 + ["ind4", "ind5", "ind6", "ind7"]


def test_reindex_before_any_full_layer_scores_the_whole_context(monkeypatch):
    rec = _Recorder(monkeypatch)
    _step(["reindex", "reuse", "full", "reindex"], pool_k=512)
    # no pool exists until the Full layer at 2: the first Reindex selects
    # over everything, the one after the Full layer inside the pool
    assert rec.names() == ["indexer_topk", "sparse_decode", "sparse_decode",
                           "indexer_topk", "indexer_pool", "sparse_decode",
                           "indexer_topk_pool", "sparse_decode"]


def test_bad_schedules_are_refused(monkeypatch):
    _Recorder(monkeypatch)
    with pytest.raises(ValueError, match="first layer"):
        _step(["reuse", "full"])
    with pytest.raises(ValueError, match="unknown layer mode"):
        _step(["full", "skip"])
