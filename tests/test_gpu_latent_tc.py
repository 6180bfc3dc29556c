"""GPU parity of the tensor-core (tcgen05) latent decode through the C ABI,
against the fp64 oracle: ragged tails and empty sequences, two head tiles,
launches cut so that units split between CTAs and CTAs hold several units,
sharper scores whose maximum keeps growing along the sequence (so heads
rescale their output rows mid-unit), and the CUDA-core latent kernel on the
same inputs."""
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


def make_case(n_h, block_size, lengths, seed, q_mult=1.0, ramp=0.0):
    """Seeded latent cache (N(0,1) rows, optionally growing with position
    by a factor 1 + ramp * t / L) in shuffled blocks, and N(0, q_mult^2)
    queries, all rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    L = max(max(lengths), 1)
    nbps = (L + block_size - 1) // block_size
    num_blocks = B * nbps + 3
    table = torch.randperm(num_blocks, generator=g)[:B * nbps].reshape(
        B, nbps).to(torch.int32)
    cache = torch.randn(num_blocks, 1, block_size, 576, generator=g)
    if ramp:
        for b in range(B):
            for j in range(nbps):
                t = j * block_size + torch.arange(block_size)
                cache[table[b, j], 0] *= (1 + ramp * t / L)[:, None]
    cache = cache.to(torch.bfloat16)
    q = (torch.randn(B, n_h, 576, generator=g) * q_mult).to(torch.bfloat16)
    return cache, table, torch.tensor(lengths, dtype=torch.int32), q


def run_case(n_h, block_size, lengths, seed, **kw):
    cache, table, lens, q = make_case(n_h, block_size, lengths, seed, **kw)
    c = K.PagedCache(k=cache.cuda(), v=None, block_size=block_size, n_kv=1,
                     head_dim=576)
    out, lse = K.mla_decode(c, table.cuda(), lens.cuda(), max(lengths),
                            q.cuda(), d_c=512)
    torch.cuda.synchronize()
    raw = cache.view(torch.int16).numpy().view(np.uint16)
    ref, ref_lse = oracle.mla_decode(q.float().numpy(), raw, table.numpy(),
                                     lens.numpy(), block_size)
    return H.to_np_bf16(out), lse.cpu().numpy(), ref, ref_lse


CASES = [
    # n_h, block_size, lengths, seed, kwargs, forced CTA count
    (128, 64, [0, 1, 63, 64, 65, 500, 1000], 1, {}, None),
    (256, 64, [100, 3000], 2, {}, None),
    (128, 64, [700, 50, 1500, 9, 0, 2100], 3, {}, 8),   # 2 lanes
    (128, 128, [4000, 33], 4, {}, 12),                  # 3 lanes
    (128, 128, [3000, 1200], 5, {"q_mult": 1.5, "ramp": 0.5}, None),
    (128, 64, [2500], 6, {"q_mult": 2.0, "ramp": 0.25}, 4),  # 1 lane
]


@pytest.mark.parametrize("case", CASES, ids=["tails", "h256", "split2",
                                             "split3", "peaked",
                                             "peaked_1lane"])
def test_latent_tc(case):
    n_h, bs, lengths, seed, kw, ctas = case
    K.set_tuning(decode_ctas=ctas or 0)
    try:
        out, lse, ref, ref_lse = run_case(n_h, bs, lengths, seed, **kw)
    finally:
        K.set_tuning()
    H.assert_close(out, ref, f"latent tc {case}")
    H.assert_lse_close(lse, ref_lse, f"latent tc {case}")


def test_latent_tc_matches_cuda_core_kernel():
    """Both latent kernels on the same inputs: each within the tolerance of
    the oracle, and of each other."""
    args = (128, 64, [1234, 77, 4096], 7)
    out_tc, lse_tc, ref, ref_lse = run_case(*args)
    K.set_tuning(mla_cuda_cores=True)
    try:
        out_cc, lse_cc, _, _ = run_case(*args)
    finally:
        K.set_tuning()
    H.assert_close(out_tc, ref, "tc")
    H.assert_close(out_cc, ref, "cuda cores")
    H.assert_close(out_tc, out_cc, "tc vs cuda cores")
    H.assert_lse_close(lse_tc, ref_lse, "tc lse")
    H.assert_lse_close(lse_cc, ref_lse, "cuda cores lse")
