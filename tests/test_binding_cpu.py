"""The Python binding fails loudly instead of computing anywhere else: host
(CPU) tensors are refused before the library is called, and a missing
libkvd.so is an error, not a fallback."""
import pytest
import torch

import kv_cache_decode_gqa_gb300 as K
from kv_cache_decode_gqa_gb300 import _native as N


def _host_inputs():
    i32 = dict(dtype=torch.int32)
    bf = dict(dtype=torch.bfloat16)
    cache = K.PagedCache(torch.zeros((2, 2, 16, 64), **bf),
                         torch.zeros((2, 2, 16, 64), **bf), 16, 2, 64)
    lat = K.PagedCache(torch.zeros((2, 1, 16, 576), **bf), None, 16, 1, 576)
    idx = K.PagedCache(torch.zeros((2, 1, 16, 64), **bf), None, 16, 1, 64)
    sp = K.PagedCache(torch.zeros((2, 1, 16, 512), **bf),
                      torch.zeros((2, 1, 16, 512), **bf), 16, 1, 512)
    return dict(
        cache=cache, lat=lat, idx=idx, sp=sp,
        bt=torch.zeros((1, 2), **i32), lens=torch.ones(1, **i32),
        pos=torch.zeros(1, **i32), knew=torch.zeros((1, 2, 64), **bf),
        q=torch.zeros((1, 4, 64), **bf), qlat=torch.zeros((1, 64, 576), **bf),
        qidx=torch.zeros((1, 4, 64), **bf), w=torch.ones((1, 4)),
        qsp=torch.zeros((1, 64, 512), **bf), ind=torch.zeros((1, 8), **i32))


CALLS = {
    "kv_append": lambda a: K.kv_append(a["cache"], a["bt"], a["pos"],
                                       a["knew"], a["knew"]),
    "gqa_decode": lambda a: K.gqa_decode(a["cache"], a["bt"], a["lens"], 32,
                                         a["q"]),
    "gqa_append_decode": lambda a: K.gqa_append_decode(
        a["cache"], a["bt"], a["lens"], 32, a["pos"], a["knew"], a["knew"],
        a["q"]),
    "mla_decode": lambda a: K.mla_decode(a["lat"], a["bt"], a["lens"], 32,
                                         a["qlat"]),
    "indexer_topk": lambda a: K.indexer_topk(a["idx"], a["bt"], a["lens"], 32,
                                             a["qidx"], a["w"], 8),
    "indexer_pool": lambda a: K.indexer_pool(a["bt"], a["lens"], 32,
                                             a["ind"]),
    "sparse_decode": lambda a: K.sparse_decode(a["sp"], a["bt"], a["lens"],
                                               32, a["ind"], a["qsp"]),
    "copy_blocks": lambda a: K.copy_blocks(a["cache"], a["pos"], a["pos"]),
    "workspace_size": lambda a: K.workspace_size(
        K.OP_GQA_DECODE, a["cache"], a["bt"], a["lens"], 32, 4),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name, monkeypatch):
    # the refusal must come before any library call
    def no_library():
        raise AssertionError("the library was called with host tensors")
    monkeypatch.setattr(K, "lib", no_library)
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name](_host_inputs())


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(N, "LIB_PATH", str(tmp_path / "libkvd.so"))
    monkeypatch.setattr(N, "_lib", None)
    with pytest.raises(RuntimeError, match="is not built"):
        N.lib()
