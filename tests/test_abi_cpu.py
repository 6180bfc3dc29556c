"""The C ABI without a GPU: the library loads, exports every function
include/kvd.h declares, and rejects bad arguments on the host before any
CUDA call. Fake, aligned pointers stand in for device buffers; every call
here fails validation (or has nothing to do) before it could launch, so the
fakes are never dereferenced, on a GPU machine either."""
import ctypes
import os

import pytest

from kv_cache_decode_gqa_gb300 import _native as N

FAKE = 0x10000          # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(N.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return N.lib()


def _cache(**kw):
    c = N.KvdCache(FAKE, FAKE + 0x100000, 10, 64, 8, 128, 0, 0, None, None,
                   None, None)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _seqs(**kw):
    s = N.KvdSeqs(FAKE + 0x200000, FAKE + 0x300000, 4, 16, 1000, 0)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_set_tuning_validation(lib):
    assert lib.kvd_set_tuning(-1, 0) == 2
    assert b"decode_ctas" in lib.kvd_last_error()
    assert lib.kvd_set_tuning(0, 0) == 0


def test_exports_every_declared_function(lib):
    names = N.header_functions()
    assert len(names) == 26
    for name in names:
        assert hasattr(lib, name), name
    assert lib.kvd_version() == 1


def test_bytes_per_token(lib):
    assert lib.kvd_bytes_per_token(80, 8, 128, 2) == 327680
    assert lib.kvd_bytes_per_token(32, 32, 128, 2) * 4096 == 2147483648
    assert lib.kvd_bytes_per_token(-1, 8, 128, 2) == 0


def test_status_strings(lib):
    assert lib.kvd_status_string(0) == b"KVD_OK"
    assert lib.kvd_status_string(5) == b"KVD_ERR_WORKSPACE"


def _gqa(lib, c, s, n_h=64, q=FAKE, out=FAKE):
    return lib.kvd_gqa_decode(ctypes.byref(c), ctypes.byref(s), q, n_h, 0.0,
                              out, None, None, 0, None)


def test_gqa_validation(lib):
    assert _gqa(lib, _cache(k=None), _seqs()) == 1
    assert b"cache->k" in lib.kvd_last_error()
    assert _gqa(lib, _cache(v=None), _seqs()) == 1
    assert _gqa(lib, _cache(), _seqs(), q=None) == 1
    assert _gqa(lib, _cache(), _seqs(), n_h=60) == 2      # not a multiple
    assert _gqa(lib, _cache(), _seqs(), n_h=8 * 32) == 3  # group 32
    assert _gqa(lib, _cache(head_dim=96), _seqs(), n_h=8) == 3
    assert _gqa(lib, _cache(dtype=7), _seqs()) == 3
    assert _gqa(lib, _cache(k=FAKE + 8), _seqs()) == 2    # misaligned
    assert _gqa(lib, _cache(), _seqs(max_seq_len=64 * 16 + 1)) == 4
    assert b"capacity" in lib.kvd_last_error()
    assert _gqa(lib, _cache(), _seqs(batch=-1)) == 2
    assert _gqa(lib, _cache(), _seqs(batch=1025)) == 3    # over 1024 a call
    assert b"1024" in lib.kvd_last_error()
    assert _gqa(lib, _cache(dtype=1), _seqs()) == 1       # fp8 needs scales
    assert _gqa(lib, _cache(), _seqs(batch=0)) == 0       # nothing to do
    assert _gqa(lib, _cache(), _seqs(flags=4)) == 2       # unknown flag bit
    assert b"flags" in lib.kvd_last_error()
    assert _gqa(lib, _cache(), _seqs(flags=2)) == 2       # PREFIX_READY alone
    assert b"KVD_SEQS_STABLE" in lib.kvd_last_error()
    assert _gqa(lib, _cache(), _seqs(batch=0, flags=1)) == 0  # STABLE is known
    assert _gqa(lib, _cache(), _seqs(batch=0, flags=3)) == 0  # and both


def _append_decode(lib, c, s, pos=FAKE, k_new=FAKE, v_new=FAKE):
    return lib.kvd_gqa_append_decode(ctypes.byref(c), ctypes.byref(s), pos,
                                     k_new, v_new, FAKE, 64, 0.0, FAKE, None,
                                     None, 0, None)


def test_append_decode_validation(lib):
    assert _append_decode(lib, _cache(), _seqs(), pos=None) == 1
    assert b"pos" in lib.kvd_last_error()
    assert _append_decode(lib, _cache(), _seqs(), v_new=None) == 1
    assert _append_decode(lib, _cache(), _seqs(), k_new=FAKE + 4) == 2
    assert _append_decode(lib, _cache(dtype=1, k_scale=FAKE, v_scale=FAKE),
                          _seqs()) == 1                   # no inverse scales
    assert _append_decode(lib, _cache(), _seqs(batch=0), pos=None) == 0


def test_append_validation(lib):
    c = _cache()
    f = lib.kvd_kv_append
    assert f(ctypes.byref(c), FAKE, 16, FAKE, 4, FAKE, None, None) == 1
    assert f(ctypes.byref(c), FAKE, 0, FAKE, 4, FAKE, FAKE, None) == 2
    assert f(ctypes.byref(_cache(head_dim=4)), FAKE, 16, FAKE, 4, FAKE, FAKE,
             None) == 2
    assert f(ctypes.byref(c), FAKE, 16, FAKE, 4, FAKE + 2, FAKE, None) == 2
    assert f(ctypes.byref(_cache(dtype=1)), FAKE, 16, FAKE, 4, FAKE, FAKE,
             None) == 1
    assert f(ctypes.byref(c), FAKE, 16, FAKE, 0, None, None, None) == 0


def test_mla_sparse_indexer_validation(lib):
    lat = _cache(v=None, n_kv=1, head_dim=576)
    s = _seqs()
    m = lib.kvd_mla_decode
    assert m(ctypes.byref(lat), 256, ctypes.byref(s), FAKE, 128, 0.0, FAKE,
             None, None, 0, None) == 3
    assert m(ctypes.byref(lat), 512, ctypes.byref(s), FAKE, 100, 0.0, FAKE,
             None, None, 0, None) == 3
    sp = _cache(n_kv=1, head_dim=512)
    f = lib.kvd_sparse_decode
    assert f(ctypes.byref(sp), ctypes.byref(s), None, 2048, FAKE, 64, 0.0,
             FAKE, None, None, 0, None) == 1
    assert f(ctypes.byref(sp), ctypes.byref(s), FAKE, 0, FAKE, 64, 0.0,
             FAKE, None, None, 0, None) == 2
    assert f(ctypes.byref(_cache(n_kv=2, head_dim=512)), ctypes.byref(s),
             FAKE, 2048, FAKE, 64, 0.0, FAKE, None, None, 0, None) == 3
    big = _seqs(batch=257)                    # over 256 sequences a call
    assert m(ctypes.byref(lat), 512, ctypes.byref(big), FAKE, 128, 0.0, FAKE,
             None, None, 0, None) == 3
    assert b"256" in lib.kvd_last_error()
    assert f(ctypes.byref(sp), ctypes.byref(big), FAKE, 2048, FAKE, 64, 0.0,
             FAKE, None, None, 0, None) == 3
    assert b"256" in lib.kvd_last_error()
    ix = _cache(v=None, n_kv=1, head_dim=64)
    g = lib.kvd_indexer_topk
    assert g(ctypes.byref(ix), ctypes.byref(s), FAKE, 4, FAKE, 0, FAKE, None,
             None, 0, None) == 3
    assert g(ctypes.byref(ix), ctypes.byref(s), FAKE, 9, FAKE, 16, FAKE, None,
             None, 0, None) == 3
    assert g(ctypes.byref(ix), ctypes.byref(s), None, 4, FAKE, 16, FAKE, None,
             None, 0, None) == 1


def test_no_gpu_means_cuda_error_not_crash(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    size = ctypes.c_size_t(0)
    st = lib.kvd_workspace_size(0, ctypes.byref(_cache()),
                                ctypes.byref(_seqs()), 64, 0,
                                ctypes.byref(size))
    assert st == 6


def test_mxfp4_cache_validation(lib):
    """MXFP4 caches: head_dim 128 and an even block size; decoded on the
    CUDA-core kernel, so query groups of 1, 2 or 4 only; the latent,
    sparse and indexer calls take bf16 caches only."""
    s = _seqs()
    c = _cache(dtype=2, head_dim=64)
    assert _gqa(lib, c, s, n_h=8) == 3                 # head_dim 64
    c = _cache(dtype=2, block_size=63)
    assert _gqa(lib, c, s, n_h=8) == 2                 # odd block size
    c = _cache(dtype=2)                                # n_kv 8, d 128
    assert _gqa(lib, c, s, n_h=64) == 3                # group 8: no MMA
    assert _gqa(lib, c, s, n_h=64, q=None) == 3
    c = _cache(dtype=3)
    assert _gqa(lib, c, s, n_h=8) == 3                 # unknown dtype
    lat = _cache(dtype=2, n_kv=1, head_dim=576, v=None)
    assert lib.kvd_mla_decode(ctypes.byref(lat), 512, ctypes.byref(s), FAKE,
                              128, 0.0, FAKE, None, None, 0, None) == 3


def test_pool_validation(lib):
    s = _seqs()
    # k < 1, a NULL output, an overlong max_seq_len: rejected on the host
    assert lib.kvd_indexer_pool(ctypes.byref(s), FAKE, 0, FAKE, FAKE,
                                None) == 2
    assert lib.kvd_indexer_pool(ctypes.byref(s), FAKE, 8, None, FAKE,
                                None) == 1
    assert lib.kvd_indexer_pool(ctypes.byref(_seqs(max_seq_len=60000000)),
                                FAKE, 8, FAKE, FAKE, None) == 3
    c = _cache(n_kv=1, head_dim=64, v=None, block_size=12)
    s12 = _seqs(max_blocks_per_seq=100)
    assert lib.kvd_indexer_topk_pool(ctypes.byref(c), ctypes.byref(s12), FAKE,
                                     4, FAKE, FAKE, FAKE, 16, FAKE, None,
                                     None, 0, None) == 3   # block_size % 8
    c = _cache(n_kv=1, head_dim=64, v=None)
    assert lib.kvd_indexer_topk_pool(ctypes.byref(c), ctypes.byref(s), FAKE,
                                     4, FAKE, None, FAKE, 16, FAKE, None,
                                     None, 0, None) == 1   # no pool
