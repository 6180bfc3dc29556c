"""Helpers for the GPU parity tests: run a workload step through the C ABI
and compute the oracle's answer for the same seeded inputs."""
import numpy as np

import oracle
from kv_cache_decode_gqa_gb300 import workloads as W

# The stated float tolerance: over a whole output tensor, max-abs <= 1e-2
# and relative L2 (||gpu - oracle|| / ||oracle||) <= 5e-3, bf16 outputs with
# fp32 accumulation.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def to_np_bf16(t):
    """torch bf16 CUDA tensor -> float64 numpy."""
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(
        np.uint16)
    return oracle.bf16_bits_to_f64(bits)


def assert_close(gpu, ref, what="", max_abs=MAX_ABS, rel_l2=REL_L2):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    ma = float(err.max()) if err.size else 0.0
    nr = float(np.linalg.norm(ref))
    rl = float(np.linalg.norm(gpu - ref) / nr) if nr > 0 else ma
    assert ma <= max_abs, f"{what}: max-abs {ma:.3e} > {max_abs}"
    assert rl <= rel_l2, f"{what}: rel-L2 {rl:.3e} > {rel_l2}"
    return ma, rl


def assert_lse_close(gpu_lse, ref_lse, what=""):
    g = np.asarray(gpu_lse, dtype=np.float64)
    r = np.asarray(ref_lse, dtype=np.float64)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: -inf pattern differs"
    if fin.any():
        err = np.abs(g[fin] - r[fin])
        assert err.max() <= 1e-3 * max(1.0, np.abs(r[fin]).max()), \
            f"{what}: lse error {err.max():.3e}"


def host_bits(shape, layer, tensor, dims):
    return W.host_bf16(shape, layer, tensor, dims)


def host_scales(shape, layer):
    ks, kinv = W.host_scales(shape, layer, W.T_KSCALE)
    vs, vinv = W.host_scales(shape, layer, W.T_VSCALE)
    return ks, kinv, vs, vinv


def oracle_dense_step(shape, paging, layer, seqs=None, window=0,
                      window_start=None):
    """Oracle output of one append + decode step of a GQA / MLA workload
    layer, for all sequences (small shapes) or the sampled ``seqs``.
    Returns (out [n][n_h][dv], lse [n][n_h], appended caches)."""
    s = shape
    all_seqs = list(range(s.batch)) if seqs is None else list(seqs)
    q = oracle.bf16_bits_to_f64(host_bits(s, layer, W.T_Q,
                                          (s.batch, s.n_h, s.head_dim)))
    knew = host_bits(s, layer, W.T_KNEW, (s.batch, s.n_kv, s.head_dim))
    vnew = host_bits(s, layer, W.T_VNEW, (s.batch, s.n_kv, s.head_dim))
    if seqs is None:
        kr = W.host_cache_full(s, paging, layer, W.T_K)
        vr = W.host_cache_full(s, paging, layer, W.T_V) if s.has_v else None
        bt = paging.table.astype(np.int64)
    else:
        kr, bt = W.host_cache_compact(s, paging, layer, W.T_K, all_seqs)
        vr = (W.host_cache_compact(s, paging, layer, W.T_V, all_seqs)[0]
              if s.has_v else None)
    pos = [s.lengths[b] for b in all_seqs]
    lens = [s.seq_lens[b] for b in all_seqs]
    kn, vn = knew[all_seqs], vnew[all_seqs]
    ws_sel = (None if window_start is None
              else [int(window_start[b]) for b in all_seqs])
    if s.dtype == "mxfp4":
        kr = oracle.kv_append(kr, bt, pos, kn, s.block_size, "mxfp4")
        vr = oracle.kv_append(vr, bt, pos, vn, s.block_size, "mxfp4")
        out, lse = oracle.gqa_decode(q[all_seqs], kr, vr, bt, lens,
                                     s.block_size, dtype="mxfp4",
                                     window=window, window_start=ws_sel)
    elif s.dtype == "fp8":
        ks, kinv, vs, vinv = host_scales(s, layer)
        kr = oracle.kv_append(kr, bt, pos, kn, s.block_size, "fp8", kinv)
        vr = oracle.kv_append(vr, bt, pos, vn, s.block_size, "fp8", vinv)
        out, lse = oracle.gqa_decode(q[all_seqs], kr, vr, bt, lens,
                                     s.block_size, dtype="fp8", k_scale=ks,
                                     v_scale=vs, window=window,
                                     window_start=ws_sel)
    elif s.kind == "mla":
        kr = oracle.kv_append(kr, bt, pos, kn, s.block_size)
        out, lse = oracle.mla_decode(q[all_seqs], kr, bt, lens, s.block_size,
                                     d_c=s.d_c)
    else:
        kr = oracle.kv_append(kr, bt, pos, kn, s.block_size)
        vr = oracle.kv_append(vr, bt, pos, vn, s.block_size)
        out, lse = oracle.gqa_decode(q[all_seqs], kr, vr, bt, lens,
                                     s.block_size, window=window,
                                     window_start=ws_sel)
    return out, lse, (kr, vr)


def device_step(wl, layer, lse=True, seqs_flags=0, fused=False, window=0,
                window_start=None):
    """kv_append then the layer's decode through the C ABI (or, fused, the
    single kvd_gqa_append_decode call)."""
    import kv_cache_decode_gqa_gb300 as K
    s = wl.shape
    c = wl.caches[layer]
    if fused:
        return K.gqa_append_decode(c, wl.block_table, wl.seq_lens,
                                   wl.max_seq_len, wl.pos, wl.k_new[layer],
                                   wl.v_new[layer], wl.q[layer], want_lse=lse,
                                   seqs_flags=seqs_flags, window=window,
                                   window_start=window_start)
    K.kv_append(c, wl.block_table, wl.pos, wl.k_new[layer],
                wl.v_new.get(layer))
    if s.kind == "mla":
        return K.mla_decode(c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                            wl.q[layer], d_c=s.d_c, want_lse=lse)
    return K.gqa_decode(c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                        wl.q[layer], want_lse=lse, seqs_flags=seqs_flags,
                        window=window, window_start=window_start)
