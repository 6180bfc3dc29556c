"""GPU parity of copy-on-write prefix sharing: a sequence forked from
another shares its blocks; its append into the shared last block first
copies that block on the device (kvd_copy_blocks); both sequences then
decode exactly as the oracle decodes two unshared caches."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import kv_cache_decode_gqa_gb300 as K  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    K.device_error()
    yield
    assert K.device_error() == 0


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_fork_append_decode(dtype):
    nb, n_kv, d, bs, L = 24, 2, 128, 16, 37
    g = torch.Generator().manual_seed(7)
    if dtype == "bf16":
        k = torch.randn(nb, n_kv, bs, d, generator=g).to(torch.bfloat16)
        v = torch.randn(nb, n_kv, bs, d, generator=g).to(torch.bfloat16)
        scales = {}
    else:   # fp8 codes of moderate magnitude, unit scales
        k = (torch.randint(0x20, 0x48, (nb, n_kv, bs, d), generator=g) |
             (torch.randint(0, 2, (nb, n_kv, bs, d), generator=g) << 7)
             ).to(torch.uint8)
        v = (torch.randint(0x20, 0x48, (nb, n_kv, bs, d), generator=g) |
             (torch.randint(0, 2, (nb, n_kv, bs, d), generator=g) << 7)
             ).to(torch.uint8)
        one = torch.ones(n_kv, device="cuda")
        scales = dict(k_scale=one, v_scale=one, k_inv_scale=one,
                      v_inv_scale=one)
    if dtype == "bf16":
        host_k, host_v = _bits(k), _bits(v)
    else:
        host_k, host_v = k.numpy().copy(), v.numpy().copy()
    c = K.PagedCache(k.cuda(), v.cuda(), bs, n_kv, d, dtype, **scales)
    pool = K.BlockPool(nb)
    M = 4
    ta = np.full((1, M), -1, dtype=np.int32)
    ta[0, :3] = pool.alloc(3)                      # A holds 37 tokens
    pool.share(ta[0, :3])                          # B forks A
    tb = ta.copy()
    src, dst = pool.prepare_append(tb, [L], bs)    # B writes into block 2
    assert list(src) == [2] and list(dst) == [3]
    K.copy_blocks(c, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    new = torch.randn(2, n_kv, d, generator=g).to(torch.bfloat16)
    K.kv_append(c, torch.from_numpy(tb).cuda(),
                torch.tensor([L], dtype=torch.int32, device="cuda"),
                new[1:2].cuda(), new[1:2].cuda() * 2)
    sa, _ = pool.prepare_append(ta, [L], bs)       # A's block is private now
    assert len(sa) == 0
    K.kv_append(c, torch.from_numpy(ta).cuda(),
                torch.tensor([L], dtype=torch.int32, device="cuda"),
                new[0:1].cuda(), new[0:1].cuda() * 2)
    table = torch.from_numpy(np.concatenate([ta, tb])).cuda()
    lens = torch.tensor([L + 1, L + 1], dtype=torch.int32, device="cuda")
    q = torch.randn(2, 4 * n_kv, d, generator=g).to(torch.bfloat16)
    out, lse = K.gqa_decode(c, table, lens, L + 1, q.cuda())
    torch.cuda.synchronize()
    # oracle: the same copy and appends on the host arrays
    for s_, d_ in zip(src, dst):
        host_k[d_], host_v[d_] = host_k[s_], host_v[s_]
    tab = np.concatenate([ta, tb]).astype(np.int64)
    nk, nv = _bits(new), _bits((new * 2).to(torch.bfloat16))
    kw = {}
    if dtype == "fp8":
        inv = np.ones(n_kv, dtype=np.float32)
        kw = dict(dtype="fp8", inv_scale=inv)
    host_k = oracle.kv_append(host_k, tab, [L, L], nk, bs, **kw)
    host_v = oracle.kv_append(host_v, tab, [L, L], nv, bs, **kw)
    got_k = c.k.cpu()
    got_k = _bits(got_k) if dtype == "bf16" else got_k.numpy()
    assert np.array_equal(got_k, host_k)
    dk = {} if dtype == "bf16" else dict(dtype="fp8", k_scale=np.ones(n_kv),
                                         v_scale=np.ones(n_kv))
    ref, ref_lse = oracle.gqa_decode(oracle.bf16_bits_to_f64(_bits(q)), host_k,
                                     host_v, tab, [L + 1, L + 1], bs, **dk)
    H.assert_close(H.to_np_bf16(out), ref, f"cow/{dtype}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"cow/{dtype}")
    # the two sequences now differ only in their last row
    assert not np.allclose(H.to_np_bf16(out)[0], H.to_np_bf16(out)[1])
