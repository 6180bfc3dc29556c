"""GPU parity of kv_append and gqa_decode against the fp64 oracle, through
the C ABI. Small shapes compare every output element; the full-size
workloads compare sampled sequences in the launch configuration the bench
times."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import kv_cache_decode_gqa_gb300 as K  # noqa: E402
from kv_cache_decode_gqa_gb300 import workloads as W  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    K.device_error()            # clear the error word
    yield
    assert K.device_error() == 0


def _cache_bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def _host_bytes(a):
    return np.ascontiguousarray(a).view(np.uint8)


# ---------------------------------------------------------------------------
# append: whole-cache byte equality, canary blocks included
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("bs,lengths", [(16, [0, 15, 16, 47]),
                                        (64, [63, 64, 200])])
def test_append_bitexact(dtype, bs, lengths):
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, dtype=dtype, n_h=16, n_kv=2)
    wl = W.DeviceWorkload(s, layers=[0])
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    torch.cuda.synchronize()
    kr = W.host_cache_full(s, wl.paging, 0, W.T_K)
    vr = W.host_cache_full(s, wl.paging, 0, W.T_V)
    kn = H.host_bits(s, 0, W.T_KNEW, (s.batch, s.n_kv, s.head_dim))
    vn = H.host_bits(s, 0, W.T_VNEW, (s.batch, s.n_kv, s.head_dim))
    bt = wl.paging.table
    if dtype == "fp8":
        _, kinv, _, vinv = H.host_scales(s, 0)
        kr = oracle.kv_append(kr, bt, s.lengths, kn, bs, "fp8", kinv)
        vr = oracle.kv_append(vr, bt, s.lengths, vn, bs, "fp8", vinv)
    elif dtype == "mxfp4":
        kr = oracle.kv_append(kr, bt, s.lengths, kn, bs, "mxfp4")
        vr = oracle.kv_append(vr, bt, s.lengths, vn, bs, "mxfp4")
    else:
        kr = oracle.kv_append(kr, bt, s.lengths, kn, bs)
        vr = oracle.kv_append(vr, bt, s.lengths, vn, bs)
    assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr))
    assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr))


def test_append_fp8_rounding_edges():
    """Midpoints between adjacent E4M3 values (ties to even), values past
    448 (saturate), subnormals and signed zeros, with inv_scale = 1 and a
    non-power-of-two inv_scale."""
    t = oracle.e4m3_value_table()[:127]
    mids = (t[:-1] + t[1:]) / 2
    vals = np.concatenate([mids, -mids, t, -t,
                           [448.0, 464.0, 480.0, 12288.0, -12288.0, 2.0 ** -10,
                            3 * 2.0 ** -10, -2.0 ** -11, 0.0, -0.0]])
    n_kv, d = 1, 64
    rows = (len(vals) + d - 1) // d
    vals = np.concatenate([vals, np.zeros(rows * d - len(vals))])
    bits = torch.tensor(vals).to(torch.bfloat16)
    assert np.array_equal(bits.double().numpy(), vals)   # all exact in bf16
    for inv in (1.0, 1.0 / 0.07):
        inv32 = np.float32(inv)
        cache = torch.zeros((rows + 1, n_kv, 1, d), dtype=torch.uint8,
                            device="cuda")
        c = K.PagedCache(cache, None, 1, n_kv, d, "fp8",
                         k_scale=torch.ones(1, device="cuda"),
                         k_inv_scale=torch.full((1,), float(inv32),
                                                device="cuda"))
        bt = torch.arange(rows, dtype=torch.int32,
                          device="cuda").reshape(rows, 1) + 1
        pos = torch.zeros(rows, dtype=torch.int32, device="cuda")
        k_new = bits.reshape(rows, 1, d).cuda()
        K.kv_append(c, bt, pos, k_new)
        torch.cuda.synchronize()
        got = cache.cpu().numpy()[1:, 0, 0, :].reshape(-1)
        x = vals.astype(np.float32) * inv32
        want = oracle.e4m3_encode_f32(x.astype(np.float32))
        assert np.array_equal(got, want), np.nonzero(got != want)
        assert np.all(cache.cpu().numpy()[0] == 0)        # untouched block


def test_append_mxfp4_rounding_edges():
    """MXFP4 rows through kv_append, against the oracle's encoder: groups
    whose scale is exactly 1 (amax 6) holding every E2M1 midpoint and its
    neighbours (ties to even), groups that saturate (amax/6 rounding down,
    amax past 2688), all-zero and tiny groups (scale 0: zero codes), signed
    zeros, and N(0,1) groups of every magnitude."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]

    def bf16_neighbours(m):  # the adjacent bf16 values above and below m
        e = np.floor(np.log2(m))
        below = 2.0 ** (e - 8) if m == 2.0 ** e else 2.0 ** (e - 7)
        return m + 2.0 ** (e - 7), m - below
    groups = []
    for m in mids:
        up, dn = bf16_neighbours(m)
        g = [6.0, m, -m, up, dn, -0.0, 0.0, -6.0, m / 2, -m / 2, 3 * m, -up,
             -dn, -4.0, 2.0, 1.0]
        groups.append(g)
    groups.append([7.0] + [6.5, -6.9, 1.0, 0.3] + [0.0] * 11)   # scale 1.125
    groups.append([3000.0, -1e5] + [1.0] * 14)                  # > 2688
    groups.append([0.0] * 16)
    groups.append([2.0 ** -13, -2.0 ** -12] + [0.0] * 14)       # scale -> 0
    groups.append([-0.0] * 8 + [1e-3] * 8)
    rng = np.random.default_rng(50)
    for e in range(-12, 12, 3):
        groups.append(list(rng.standard_normal(16) * 2.0 ** e))
    vals = np.array(groups, dtype=np.float64).reshape(-1)
    d = 128
    rows = (len(vals) + d - 1) // d
    vals = np.concatenate([vals, np.zeros(rows * d - len(vals))])
    bits = torch.tensor(vals).to(torch.bfloat16)
    assert np.array_equal(bits.double().numpy()[:7 * 16],
                          vals[:7 * 16])              # exact in bf16
    cache = torch.zeros((rows + 1, 1, 2, 72), dtype=torch.uint8,
                        device="cuda")
    c = K.PagedCache(cache, None, 2, 1, d, "mxfp4")
    bt = torch.arange(rows, dtype=torch.int32, device="cuda").reshape(rows, 1)
    bt = bt + 1
    pos = torch.ones(rows, dtype=torch.int32, device="cuda")   # slot 1
    k_new = bits.reshape(rows, 1, d).cuda()
    K.kv_append(c, bt, pos, k_new)
    torch.cuda.synchronize()
    got = cache.cpu().numpy()
    want = oracle.mxfp4_encode_rows(
        bits.view(torch.int16).numpy().view(np.uint16).reshape(rows, d))
    assert np.array_equal(got[1:, 0, 1, :], want), np.argwhere(
        got[1:, 0, 1, :] != want)
    assert np.all(got[0] == 0) and np.all(got[1:, 0, 0, :] == 0)


# ---------------------------------------------------------------------------
# dense decode, every element
# ---------------------------------------------------------------------------
DENSE_CASES = [
    # name, n_h, n_kv, d, block_size, cached lengths
    ("mha_d128", 4, 4, 128, 64, [0, 1, 63, 64, 200, 1000]),
    ("gqa2_d128", 8, 4, 128, 16, [5, 130, 511]),
    ("gqa4_d64", 8, 2, 64, 64, [100, 256, 777]),
    ("gqa4_d128_bs32", 16, 4, 128, 32, [31, 32, 33, 1500]),
    ("mha_d64_bs320", 2, 2, 64, 320, [1, 319, 600]),
    # head groups per copy: 2 (bf16, d 128) and 4 (fp8, or d 64)
    ("mha_d64_bs64", 8, 8, 64, 64, [0, 64, 65, 900]),
    ("gqa2_d128_bs64", 8, 4, 128, 64, [1, 200, 1000]),
    # tensor-core path: query groups of 8 and 16
    ("gqa8_bs64", 16, 2, 128, 64, [0, 1, 63, 64, 65, 500]),
    ("gqa16_bs16", 32, 2, 128, 16, [3, 100, 257]),
    ("gqa8_bs128", 8, 1, 128, 128, [129, 1000]),
    ("gqa8_bs32", 64, 8, 128, 32, [31, 700]),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("case", DENSE_CASES, ids=[c[0] for c in DENSE_CASES])
def test_gqa_decode_small(case, dtype):
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=d)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/{dtype}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/{dtype}")


# More than 64 sequences: the split merge then takes its full-size partition
# table (batches up to 64 take a small one); both kernels, with split units
# and one-token sequences.
@pytest.mark.parametrize("n_h,n_kv", [(4, 4), (16, 2)], ids=["mha", "gqa8"])
def test_gqa_decode_batch_over_64(n_h, n_kv):
    lengths = [int(x) for x in np.random.default_rng(96).integers(1, 300, 96)]
    lengths[5] = lengths[50] = 0
    s = W.config("llama31_70b_gqa", batch=96, lengths=lengths, n_layers=1,
                 block_size=64, dtype="bf16", n_h=n_h, n_kv=n_kv,
                 head_dim=128)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, f"batch96/{n_h}x{n_kv}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"batch96/{n_h}x{n_kv}")


# The largest batch a dense call takes (1024 sequences): the partition scan
# at its full width, in both kernels and the merge.
@pytest.mark.parametrize("n_h,n_kv", [(2, 2), (16, 2)], ids=["mha", "gqa8"])
def test_gqa_decode_max_batch(n_h, n_kv):
    lengths = [int(x) for x in np.random.default_rng(1024).integers(0, 130,
                                                                    1024)]
    s = W.config("llama31_70b_gqa", batch=1024, lengths=lengths, n_layers=1,
                 block_size=64, dtype="bf16", n_h=n_h, n_kv=n_kv,
                 head_dim=128)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, f"batch1024/{n_h}x{n_kv}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"batch1024/{n_h}x{n_kv}")


# MXFP4 caches: head_dim 128, query groups of 1, 2 or 4 (CUDA-core kernel)
MXFP4_CASES = [c for c in DENSE_CASES if c[3] == 128 and c[1] // c[2] <= 4]


@pytest.mark.parametrize("case", MXFP4_CASES, ids=[c[0] for c in MXFP4_CASES])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_gqa_decode_mxfp4(case, fused):
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama2_7b_mha_mxfp4", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, n_h=n_h, n_kv=n_kv)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0, fused=fused)
    torch.cuda.synchronize()
    ref, ref_lse, (kr, vr) = H.oracle_dense_step(s, wl.paging, 0)
    c = wl.caches[0]
    assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr)), name
    assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr)), name
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/mxfp4")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/mxfp4")


@pytest.mark.parametrize("case", [c for c in DENSE_CASES if c[0] in
                                  ("mha_d128", "gqa2_d128_bs64", "gqa8_bs64")],
                         ids=lambda c: c[0])
def test_gqa_decode_stable_seqs_flag(case):
    """KVD_SEQS_STABLE moves the plan before the predecessor's completion;
    results are those of the default order."""
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, n_h=n_h, n_kv=n_kv, head_dim=d)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0, seqs_flags=K.SEQS_STABLE)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/stable")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/stable")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("case", [c for c in DENSE_CASES if c[0] in
                                  ("mha_d128", "gqa2_d128", "gqa2_d128_bs64",
                                   "mha_d64_bs64", "gqa8_bs64", "gqa16_bs16",
                                   "gqa8_bs32")],
                         ids=lambda c: c[0])
def test_gqa_decode_prefix_ready_flag(case, fused, dtype):
    """KVD_SEQS_PREFIX_READY lets the first chunks of cached rows be copied
    before the preceding kernel (here the append, or nothing) completes;
    the chunk holding the newest position waits. Results and cache bytes
    are those of the default order."""
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=d)
    wl = W.DeviceWorkload(s, layers=[0])
    flags = K.SEQS_STABLE | K.SEQS_PREFIX_READY
    out, lse = H.device_step(wl, 0, fused=fused, seqs_flags=flags)
    torch.cuda.synchronize()
    ref, ref_lse, (kr, vr) = H.oracle_dense_step(s, wl.paging, 0)
    c = wl.caches[0]
    assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr)), name
    assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr)), name
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/{dtype}/ready")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/ready")


def test_prefix_ready_needs_stable_flag():
    s = W.config("llama31_70b_gqa", batch=2, lengths=[10, 20], n_layers=1,
                 n_h=8, n_kv=8)
    wl = W.DeviceWorkload(s, layers=[0])
    with pytest.raises(K.KvdError) as e:
        K.gqa_decode(wl.caches[0], wl.block_table, wl.seq_lens,
                     s.max_seq_len, wl.q[0], seqs_flags=K.SEQS_PREFIX_READY)
    assert e.value.status == 2


# Split units with many parts: a forced CTA count far above the units puts
# up to ~40 CTAs on one unit, so the last to arrive merges them with lane
# quads (more than 8 parts), in both kernels and in the fused call.
@pytest.mark.parametrize("n_h,n_kv,dtype", [(2, 2, "bf16"), (4, 1, "fp8"),
                                            (8, 1, "bf16"), (16, 1, "fp8")],
                         ids=["mha", "gqa4_fp8", "gqa8", "gqa16_fp8"])
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_many_part_split_merge(n_h, n_kv, dtype, fused):
    lengths = [2500, 3, 700]
    s = W.config("llama31_70b_gqa", batch=3, lengths=lengths, n_layers=1,
                 block_size=64, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=128)
    wl = W.DeviceWorkload(s, layers=[0])
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    K.set_tuning(decode_ctas=57)
    try:
        # twice: the second call finds the counters the first left at zero
        # (its append rewrites the same rows)
        for _ in range(2):
            out, lse = H.device_step(wl, 0, fused=fused,
                                     seqs_flags=K.SEQS_STABLE)
            torch.cuda.synchronize()
            H.assert_close(H.to_np_bf16(out), ref, f"parts {n_h}x{n_kv}")
            H.assert_lse_close(lse.cpu().numpy(), ref_lse, "parts lse")
    finally:
        K.set_tuning()


# A step as a serving loop issues it: several layers back to back, each the
# fused append + decode with both flags, captured in a CUDA graph and
# replayed, every layer sharing ONE workspace (so a layer's kernel starts
# while the previous layer's still runs, over the same counters and
# partials). Each layer's output against the oracle after two replays (the
# second replay re-appends the same rows, so the results are the same).
@pytest.mark.parametrize("name,n_h,n_kv,dtype,lengths", [
    ("mha", 16, 16, "bf16", [3000, 1, 900]),
    ("gqa8", 32, 4, "bf16", [5000, 64, 2100, 17]),
    ("gqa8_fp8", 32, 4, "fp8", [4100, 640, 2000]),
], ids=["mha", "gqa8", "gqa8_fp8"])
def test_layer_chain_in_graph_shared_workspace(name, n_h, n_kv, dtype,
                                               lengths):
    layers = [0, 1, 2, 3]
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=4, block_size=64, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=128)
    wl = W.DeviceWorkload(s, layers=layers)
    need = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                            wl.seq_lens, wl.max_seq_len, n_h)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    outs = {l: torch.empty((s.batch, n_h, 128), dtype=torch.bfloat16,
                           device="cuda") for l in layers}
    lses = {l: torch.empty((s.batch, n_h), dtype=torch.float32,
                           device="cuda") for l in layers}
    flags = K.SEQS_STABLE | K.SEQS_PREFIX_READY

    def step():
        for l in layers:
            K.gqa_append_decode(wl.caches[l], wl.block_table, wl.seq_lens,
                                wl.max_seq_len, wl.pos, wl.k_new[l],
                                wl.v_new[l], wl.q[l], out=outs[l],
                                lse=lses[l], workspace=ws, seqs_flags=flags)
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for l in layers:
        ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, l)
        H.assert_close(H.to_np_bf16(outs[l]), ref, f"{name} layer {l}")
        H.assert_lse_close(lses[l].cpu().numpy(), ref_lse, f"{name} {l}")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("case", DENSE_CASES, ids=[c[0] for c in DENSE_CASES])
def test_append_decode_fused(case, dtype):
    """kvd_gqa_append_decode: the cache bytes of kv_append (every block,
    canaries included) and the outputs of the decode that follows it."""
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=d)
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0, fused=True)
    torch.cuda.synchronize()
    ref, ref_lse, (kr, vr) = H.oracle_dense_step(s, wl.paging, 0)
    c = wl.caches[0]
    assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr)), name
    assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr)), name
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/{dtype}/fused")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/{dtype}/fused")


def test_append_decode_unread_rows_and_bad_positions():
    """Rows no chunk reads (an empty sequence, a slot at the visible length)
    are written all the same; a position out of range is skipped and
    flagged, as kv_append does."""
    s = W.config("llama2_7b_mha", batch=4, lengths=[0, 100, 5, 40],
                 n_layers=1, n_h=4, n_kv=4)
    wl = W.DeviceWorkload(s, layers=[0])
    c = wl.caches[0]
    lens = torch.tensor([0, 100, 6, 41], dtype=torch.int32, device="cuda")
    pos = wl.pos.clone()
    pos[3] = -1                                   # out of range: skipped
    out, lse = K.gqa_append_decode(c, wl.block_table, lens, s.max_seq_len,
                                   pos, wl.k_new[0], wl.v_new[0], wl.q[0])
    torch.cuda.synchronize()
    assert K.device_error() == K.DEVERR_POS
    kr = W.host_cache_full(s, wl.paging, 0, W.T_K)
    vr = W.host_cache_full(s, wl.paging, 0, W.T_V)
    kn = H.host_bits(s, 0, W.T_KNEW, (s.batch, s.n_kv, s.head_dim))
    vn = H.host_bits(s, 0, W.T_VNEW, (s.batch, s.n_kv, s.head_dim))
    bt = wl.paging.table
    # the oracle appends sequences 0..2 only (sequence 3's slot is invalid)
    kr = oracle.kv_append(kr, bt[:3], [0, 100, 5], kn[:3], s.block_size)
    vr = oracle.kv_append(vr, bt[:3], [0, 100, 5], vn[:3], s.block_size)
    assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr))
    assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr))
    q = oracle.bf16_bits_to_f64(H.host_bits(s, 0, W.T_Q,
                                            (s.batch, s.n_h, s.head_dim)))
    ref, ref_lse = oracle.gqa_decode(q, kr, vr, bt, [0, 100, 6, 41],
                                     s.block_size)
    H.assert_close(H.to_np_bf16(out), ref, "unread rows")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, "unread rows")


def test_tiny_config_full():
    s = W.config("tiny_gqa")
    wl = W.DeviceWorkload(s)
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, "tiny_gqa")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, "tiny_gqa")


def test_empty_and_peaked_sequences():
    """seq_len 0 gives out = 0, lse = -inf; a query 64x larger makes the
    softmax nearly one-hot (checks the running-max rescaling)."""
    s = W.config("llama2_7b_mha", batch=3, lengths=[70, 300, 5], n_layers=1,
                 n_h=4, n_kv=4)
    wl = W.DeviceWorkload(s, layers=[0])
    c = wl.caches[0]
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
    q = (wl.q[0].float() * 64).to(torch.bfloat16)
    lens = torch.tensor([0, 301, 6], dtype=torch.int32, device="cuda")
    out, lse = K.gqa_decode(c, wl.block_table, lens, s.max_seq_len, q)
    torch.cuda.synchronize()
    _, _, (kr, vr) = H.oracle_dense_step(s, wl.paging, 0)
    qh = oracle.bf16_bits_to_f64(
        q.view(torch.int16).cpu().numpy().view(np.uint16))
    ref, ref_lse = oracle.gqa_decode(qh, kr, vr, wl.paging.table, [0, 301, 6],
                                     s.block_size)
    H.assert_close(H.to_np_bf16(out), ref, "peaked")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, "peaked")
    assert np.all(H.to_np_bf16(out)[0] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[0]))


def test_bad_block_id_is_flagged_not_faulted():
    s = W.config("llama2_7b_mha", batch=1, lengths=[100], n_layers=1, n_h=2,
                 n_kv=2)
    wl = W.DeviceWorkload(s, layers=[0])
    bt = wl.block_table.clone()
    bt[0, 1] = 1 << 30
    K.gqa_decode(wl.caches[0], bt, wl.seq_lens, s.max_seq_len, wl.q[0])
    assert K.device_error() & 1            # KVD_DEVERR_BLOCK
    bt[0, 1] = -5
    pos = torch.tensor([64], dtype=torch.int32, device="cuda")
    K.kv_append(wl.caches[0], bt, pos, wl.k_new[0], wl.v_new[0])
    assert K.device_error() & 1
    assert K.device_error() == 0           # cleared by the read


def test_workspace_errors():
    # two sequences: the stream-K split, whose partials need the workspace
    # (a single one would take the cluster merge, which needs none)
    s = W.config("llama2_7b_mha", batch=2, lengths=[4000, 3000], n_layers=1,
                 n_h=2, n_kv=2)
    wl = W.DeviceWorkload(s, layers=[0])
    need = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                            wl.seq_lens, s.max_seq_len, 2)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KvdError) as e:
        K.gqa_decode(wl.caches[0], wl.block_table, wl.seq_lens, s.max_seq_len,
                     wl.q[0], workspace=small)
    assert e.value.status == 5


# ---------------------------------------------------------------------------
# full-size workloads, sampled sequences, the bench's launch configuration
# ---------------------------------------------------------------------------
BENCH_FLAGS = K.SEQS_STABLE | K.SEQS_PREFIX_READY
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_llama2_7b_full_size_sampled_layers(fused):
    s = W.config("llama2_7b_mha")
    wl = W.DeviceWorkload(s, layers=[0, 31])
    for layer in (0, 31):
        out, lse = H.device_step(wl, layer, fused=fused,
                                 seqs_flags=BENCH_FLAGS if fused else 0)
        torch.cuda.synchronize()
        ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, layer, seqs=[0])
        H.assert_close(H.to_np_bf16(out), ref, f"llama2 layer {layer}")
        H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"layer {layer}")


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_llama2_7b_mxfp4_full_size_sampled_layers(fused):
    s = W.config("llama2_7b_mha_mxfp4")
    wl = W.DeviceWorkload(s, layers=[0, 31])
    for layer in (0, 31):
        out, lse = H.device_step(wl, layer, fused=fused,
                                 seqs_flags=K.SEQS_STABLE if fused else 0)
        torch.cuda.synchronize()
        ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, layer, seqs=[0])
        H.assert_close(H.to_np_bf16(out), ref, f"mxfp4 layer {layer}")
        H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"mxfp4 {layer}")


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("name", ["llama31_70b_gqa", "llama31_70b_gqa_fp8"])
def test_llama31_70b_full_size_sampled(name, fused):
    s = W.config(name)
    wl = W.DeviceWorkload(s, layers=[0])
    try:
        out, lse = H.device_step(wl, 0, fused=fused,
                                 seqs_flags=BENCH_FLAGS if fused else 0)
    except K.KvdError as e:
        if e.status == 3:
            pytest.skip(f"{name}: kernel not built yet")
        raise
    torch.cuda.synchronize()
    seqs = [0, int(np.argmax(s.lengths)), int(np.argmin(s.lengths)), 31]
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0, seqs=seqs)
    H.assert_close(H.to_np_bf16(out)[seqs], ref, name)
    H.assert_lse_close(lse.cpu().numpy()[seqs], ref_lse, name)


# ---------------------------------------------------------------------------
# sliding window ("890 bytes a token ...", section 7: n_win = 128)
# ---------------------------------------------------------------------------
WINDOW_CASES = [c for c in DENSE_CASES if c[0] in
                ("mha_d128", "gqa2_d128", "gqa4_d64", "gqa8_bs64",
                 "gqa16_bs16", "gqa2_d128_bs64")]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[c[0] for c in
                                                    WINDOW_CASES])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("window,starts,fused", [
    (128, False, False), (100, True, True), (1, False, True)],
    ids=["w128", "w100_starts_fused", "w1_fused"])
def test_window_decode(case, dtype, window, starts, fused):
    name, n_h, n_kv, d, bs, lengths = case
    s = W.config("llama31_70b_gqa", batch=len(lengths), lengths=lengths,
                 n_layers=1, block_size=bs, dtype=dtype, n_h=n_h, n_kv=n_kv,
                 head_dim=d)
    wl = W.DeviceWorkload(s, layers=[0])
    st = None
    if starts:   # replay starts: none, inside the window, past it
        st_host = [(L // 3) if i % 2 else max(0, L - 20)
                   for i, L in enumerate(s.seq_lens)]
        st = torch.tensor(st_host, dtype=torch.int32, device="cuda")
    out, lse = H.device_step(wl, 0, fused=fused, window=window,
                             window_start=st)
    torch.cuda.synchronize()
    ref, ref_lse, (kr, vr) = H.oracle_dense_step(
        s, wl.paging, 0, window=window,
        window_start=None if st is None else st.cpu().numpy())
    if fused:
        c = wl.caches[0]
        assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr)), name
        assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr)), name
    H.assert_close(H.to_np_bf16(out), ref, f"{name}/{dtype}/w{window}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"{name}/w{window}")


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_window_full_size_fp8(fused):
    """The pages' sliding-window cache: fp8, n_win = 128, on the
    Llama-3.1-70B shape."""
    s = W.config("llama31_70b_gqa_fp8")
    wl = W.DeviceWorkload(s, layers=[0])
    out, lse = H.device_step(wl, 0, fused=fused, window=128,
                             seqs_flags=K.SEQS_STABLE if fused else 0)
    torch.cuda.synchronize()
    seqs = [0, int(np.argmax(s.lengths)), 31]
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0, seqs=seqs,
                                          window=128)
    H.assert_close(H.to_np_bf16(out)[seqs], ref, "window full size")
    H.assert_lse_close(lse.cpu().numpy()[seqs], ref_lse, "window full size")


# ---------------------------------------------------------------------------
# whole-unit launches: when every (sequence, head group) unit is short (a
# window of <= 192 positions, or contexts of <= 256) and they fit in one
# wave, each runs whole on one CTA -- no partials, so no workspace and no
# merge launch; otherwise the stream-K split and its merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("n_h,n_kv,batch,longest,window,whole", [
    (8, 2, 6, 1000, 128, True),    # the window bounds every unit
    (8, 2, 6, 250, 0, True),       # short contexts (and empty sequences)
    (16, 2, 5, 250, 0, True),      # tensor-core kernel (group 8)
    (8, 2, 6, 1000, 0, False),     # long units: split and merged
    (16, 2, 5, 1000, 192, True),   # the longest window it takes
    (16, 2, 5, 1000, 193, False),
], ids=["window128", "short", "short_g8", "long", "window192", "window193"])
def test_whole_unit_plan(dtype, n_h, n_kv, batch, longest, window, whole):
    lengths = [max(0, longest - 97 * i) for i in range(batch)]
    s = W.config("llama31_70b_gqa", batch=batch, lengths=lengths, n_layers=1,
                 block_size=64, dtype=dtype, n_h=n_h, n_kv=n_kv, head_dim=128)
    wl = W.DeviceWorkload(s, layers=[0])
    ws = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                          wl.seq_lens, wl.max_seq_len, n_h, window=window)
    assert (ws == 0) == whole, ws
    out, lse = H.device_step(wl, 0, window=window)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0, window=window)
    H.assert_close(H.to_np_bf16(out), ref, f"whole={whole}/{dtype}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"whole={whole}/{dtype}")


def test_whole_unit_plan_needs_one_wave():
    """More units than SMs (bf16 MHA, two kv heads a unit): the split plan,
    although every unit is short."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch = sms // 16 + 2       # 16 units a sequence: more than one wave
    s = W.config("llama2_7b_mha", batch=batch, lengths=[100] * batch,
                 n_layers=1)
    wl = W.DeviceWorkload(s, layers=[0])
    ws = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                          wl.seq_lens, wl.max_seq_len, s.n_h)
    assert ws > 0
    out, lse = H.device_step(wl, 0)
    torch.cuda.synchronize()
    ref, ref_lse, _ = H.oracle_dense_step(s, wl.paging, 0)
    H.assert_close(H.to_np_bf16(out), ref, "one wave")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, "one wave")


# ---------------------------------------------------------------------------
# cluster merge: one sequence with query groups of 1 (the CUDA-core kernel)
# runs each unit as a cluster of CTAs whose parts merge in distributed
# shared memory -- no workspace, no merge launch; parts with no chunk
# (fewer chunks than CTAs) hand over empty partials
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("n_kv,length,fused", [
    (32, 300, False),    # 5 chunks: some of a unit's CTAs have none
    (32, 1000, True),
    (8, 4095, False),    # few units: too few SMs for clusters
    (32, 4095, True),
], ids=["n32_l300", "n32_l1000_fused", "n8_l4095", "n32_l4095_fused"])
def test_cluster_merge_single_sequence(dtype, n_kv, length, fused):
    s = W.config("llama2_7b_mha", batch=1, lengths=[length], n_layers=1,
                 n_h=n_kv, n_kv=n_kv, dtype=dtype)
    wl = W.DeviceWorkload(s, layers=[0])
    ws = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                          wl.seq_lens, wl.max_seq_len, s.n_h)
    # clusters for units of 2 heads (bf16) that fill most SMs (16 units);
    # 4-head units (fp8, MXFP4) and 8 kv heads keep the split and its merge
    cluster = dtype == "bf16" and n_kv == 32
    assert (ws == 0) == cluster, ws  # the cluster plan holds no partials
    out, lse = H.device_step(wl, 0, fused=fused)
    torch.cuda.synchronize()
    ref, ref_lse, (kr, vr) = H.oracle_dense_step(s, wl.paging, 0)
    if fused:
        c = wl.caches[0]
        assert np.array_equal(_cache_bytes(c.k), _host_bytes(kr))
        assert np.array_equal(_cache_bytes(c.v), _host_bytes(vr))
    H.assert_close(H.to_np_bf16(out), ref, f"cluster/{dtype}/{length}")
    H.assert_lse_close(lse.cpu().numpy(), ref_lse, f"cluster/{dtype}/{length}")


def test_cluster_merge_not_for_two_sequences():
    """Two sequences (units of different lengths): the stream-K split."""
    s = W.config("llama2_7b_mha", batch=2, lengths=[1000, 3000], n_layers=1)
    wl = W.DeviceWorkload(s, layers=[0])
    ws = K.workspace_size(K.OP_GQA_DECODE, wl.caches[0], wl.block_table,
                          wl.seq_lens, wl.max_seq_len, s.n_h)
    assert ws > 0
