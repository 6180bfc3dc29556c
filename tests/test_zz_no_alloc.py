"""kvd_gqa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (for example a plug-in inside a host program that
owns all device allocations, or a path that must not call cudaMalloc). It
uses the library's own static scratch array instead of a caller-provided
workspace. These tests call it through the C ABI and check it against
kvd_gqa_decode with a caller-provided workspace, on two calls in a row (the
array keeps the previous call's contents), and check that shapes needing
more scratch than the array holds are refused before anything runs.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import kv_cache_decode_gqa_gb300 as K  # noqa: E402
from kv_cache_decode_gqa_gb300 import _native as N  # noqa: E402
from kv_cache_decode_gqa_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402

SCRATCH_BYTES = 16 << 20      # KVD_NOALLOC_SCRATCH_BYTES in include/kvd.h


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    K.device_error()
    yield
    assert K.device_error() == 0


def _call_noalloc(cache, block_table, seq_lens, max_seq_len, q, out, lse):
    c = cache.struct()
    s = N.KvdSeqs(block_table.data_ptr(), seq_lens.data_ptr(),
                  block_table.shape[0], block_table.shape[1], max_seq_len, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return N.lib().kvd_gqa_decode_noalloc(
        ctypes.byref(c), ctypes.byref(s), ctypes.c_void_p(q.data_ptr()),
        q.shape[1], 0.0, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), stream)


CASES = [
    # n_h, n_kv, head_dim, block_size, cached lengths, dtype
    (32, 32, 128, 64, [4096], "bf16"),
    (16, 4, 128, 64, [1500, 37, 700], "bf16"),
    (8, 2, 64, 16, [100, 256], "fp8"),
]


@pytest.mark.parametrize("case", CASES, ids=["mha", "gqa4", "gqa4_fp8"])
def test_noalloc_matches_workspace_entry_point(case):
    n_h, n_kv, d, bs, lengths, dtype = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, n_h=n_h, n_kv=n_kv, head_dim=d, block_size=bs,
                 dtype=dtype)
    wl = W.DeviceWorkload(s, layers=[0])
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    ref_out, ref_lse = K.gqa_decode(c, wl.block_table, wl.seq_lens,
                                    wl.max_seq_len, wl.q[0])
    torch.cuda.synchronize()
    ref_o = H.to_np_bf16(ref_out)
    ref_l = ref_lse.cpu().numpy()
    for _ in range(2):                     # two calls in a row
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _call_noalloc(c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                           wl.q[0], out, lse)
        N.check(st)
        torch.cuda.synchronize()
        H.assert_close(H.to_np_bf16(out), ref_o, "noalloc vs workspace")
        H.assert_lse_close(lse.cpu().numpy(), ref_l, "noalloc lse")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    """A launch of 200,000 CTAs (forced with kvd_set_tuning) over 32 heads
    of 128 needs ~200 MB of partials: more than the static array. The call
    must return KVD_ERR_WORKSPACE and launch nothing: the outputs, filled
    with NaN before the call, stay NaN, where a decode of this cache (one
    nonzero row per sequence) would have written numbers."""
    B, n_h, d, bs, T = 8, 32, 128, 64, 65536
    dev = "cuda"
    k = torch.zeros((2, n_h, bs, d), dtype=torch.bfloat16, device=dev)
    v = torch.ones((2, n_h, bs, d), dtype=torch.bfloat16, device=dev)
    cache = K.PagedCache(k, v, bs, n_h, d)
    bt = torch.zeros((B, T // bs), dtype=torch.int32, device=dev)
    lens = torch.ones(B, dtype=torch.int32, device=dev)
    q = torch.ones((B, n_h, d), dtype=torch.bfloat16, device=dev)
    out = torch.full((B, n_h, d), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((B, n_h), float("nan"), dtype=torch.float32, device=dev)
    K.set_tuning(decode_ctas=200000)
    try:
        need = K.workspace_size(K.OP_GQA_DECODE, cache, bt, lens, T, n_h)
        assert need > SCRATCH_BYTES
        st = _call_noalloc(cache, bt, lens, T, q, out, lse)
        msg = N.lib().kvd_last_error()
    finally:
        K.set_tuning()
    assert st == 5                                  # KVD_ERR_WORKSPACE
    assert b"static array" in msg
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all().item()    # nothing ran
    assert torch.isnan(lse).all().item()
