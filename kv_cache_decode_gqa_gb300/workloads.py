"""The decode workloads, as seeded synthetic inputs on the device plus the
matching host arrays for the oracle.

Shapes (cached lengths are BEFORE this step's append):
  tiny_gqa          B=2, n_h=8, n_kv=2, d=64, L = 100 and 256, 1 layer,
                    one contiguous block per sequence
  llama2_7b_mha     B=1, n_h=n_kv=32, d=128, L=4096, 32 layers, 64-token blocks
                    (Llama-2-7B: the transcript's "about two gigabytes")
  llama31_70b_gqa   B=32, n_h=64, n_kv=8, d=128, L_b = 1024 + draw mod 7169,
                    80 layers, 64-token blocks; "_fp8": E4M3 cache with one
                    scale per (layer, kv head) for K and for V
  llama2_7b_mha_mxfp4  the Llama-2 shape over an MXFP4 cache (E2M1 codes, an
                    E4M3 scale per 16 channels: 72 bytes per row)
  llama31_70b_gqa_fp8_swa  the Llama-3.1 fp8 shape as sliding-window layers:
                    each query attends to the last 128 positions
  mla               B=64, n_h=128, latent 512 + rope 64, L=32768, 1 layer
  sparse            B=8, L=131072, main cache n_kv=1, d=512 (K and V), indexer
                    keys d=64, 4 indexer heads, k=2048, n_h=64, 8 layers:
                    Full, Reuse x3, Reindex x4
  sparse_pool       the same with the hierarchical indexer: the Full layer's
                    2048 positions publish their 8-position blocks as a pool
                    (at most 2,048 blocks), Reindex layers pick 512 inside it

Every tensor is a stream of the SplitMix64 generator in ``inputs`` keyed by
(20260 + config id, layer, tensor id). Cache values are N(0,1) bf16 (fp8
caches: random E4M3 codes, magnitudes 1/8..30, and per-head scales in
[1/16, 1/8); MXFP4 caches: uniform random code bytes and group scales
1/8 .. 15/32, so values are about N(0,1)-sized); indexer weights are
U(0,1). Physical blocks are a seeded
permutation of the pool, so no sequence is stored contiguously (except in
tiny_gqa), and two spare blocks per cache stay unused as canaries.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from . import inputs as I

SEED_BASE = 20260

# tensor ids of the generator streams
T_K, T_V, T_Q, T_KNEW, T_VNEW, T_QIDX, T_W, T_IDXK, T_LEN, T_PERM, \
    T_KSCALE, T_VSCALE, T_IDXKNEW, T_KGSCALE, T_VGSCALE = range(15)
# the group-scale streams of an MXFP4 cache's K and V
_GROUP_SCALE = {T_K: T_KGSCALE, T_V: T_VGSCALE}

SPARSE_MODES = ["full", "reuse", "reuse", "reuse",
                "reindex", "reindex", "reindex", "reindex"]


@dataclass
class Shape:
    name: str
    config_id: int
    batch: int
    n_h: int
    n_kv: int
    head_dim: int          # cached row width (576 for the latent cache)
    n_layers: int
    block_size: int
    lengths: List[int]     # cached lengths before the append
    dtype: str = "bf16"
    kind: str = "gqa"      # "gqa" | "mla" | "sparse"
    d_c: int = 512         # mla: latent width (values)
    contiguous: bool = False
    # sparse
    idx_dim: int = 64
    idx_heads: int = 4
    topk: int = 2048
    modes: List[str] = field(default_factory=list)
    pool_k: Optional[int] = None   # hierarchical indexer: Reindex top-k
    window: int = 0                # sliding window (0: every position)

    @property
    def dv(self):
        return self.d_c if self.kind == "mla" else self.head_dim

    @property
    def seq_lens(self):
        return [L + 1 for L in self.lengths]

    @property
    def max_seq_len(self):
        return max(self.seq_lens) if self.lengths else 0

    @property
    def has_v(self):
        return self.kind != "mla"

    @property
    def elem_bytes(self):
        """Cache bytes per element (MXFP4: 9/16, codes and scales)."""
        return {"fp8": 1, "mxfp4": 9 / 16}.get(self.dtype, 2)


def config(name, **over):
    """A named workload; keyword arguments override fields (tests use this
    for smaller shapes with the same structure)."""
    if name == "tiny_gqa":
        s = Shape("tiny_gqa", 1, 2, 8, 2, 64, 1, 320, [100, 256],
                  contiguous=True)
    elif name == "llama2_7b_mha":
        s = Shape("llama2_7b_mha", 2, 1, 32, 32, 128, 32, 64, [4096])
    elif name == "llama2_7b_mha_mxfp4":
        s = Shape(name, 6, 1, 32, 32, 128, 32, 64, [4096], dtype="mxfp4")
    elif name in ("llama31_70b_gqa", "llama31_70b_gqa_fp8",
                  "llama31_70b_gqa_fp8_swa"):
        lens = I.uniform_int(I.stream_key(SEED_BASE + 3, 0, T_LEN), 32, 1024,
                             8192).tolist()
        s = Shape(name, 3, 32, 64, 8, 128, 80, 64, lens,
                  dtype="bf16" if name == "llama31_70b_gqa" else "fp8",
                  window=128 if name.endswith("swa") else 0)
    elif name == "mla":
        s = Shape("mla", 4, 64, 128, 1, 576, 1, 64, [32768] * 64, kind="mla")
    elif name == "sparse":
        s = Shape("sparse", 5, 8, 64, 1, 512, 8, 64, [131072] * 8,
                  kind="sparse", modes=list(SPARSE_MODES))
    elif name == "sparse_pool":
        s = Shape("sparse_pool", 7, 8, 64, 1, 512, 8, 64, [131072] * 8,
                  kind="sparse", modes=list(SPARSE_MODES), pool_k=512)
    else:
        raise KeyError(name)
    for k, v in over.items():
        setattr(s, k, v)
    if "lengths" in over or "batch" in over:
        if len(s.lengths) != s.batch:
            raise ValueError("lengths must have one entry per sequence")
    return s


CONFIGS = ["tiny_gqa", "llama2_7b_mha", "llama2_7b_mha_mxfp4",
           "llama31_70b_gqa", "llama31_70b_gqa_fp8", "llama31_70b_gqa_fp8_swa",
           "mla", "sparse", "sparse_pool"]


# ---------------------------------------------------------------------------
# paging
# ---------------------------------------------------------------------------
class Paging:
    """Physical block assignment: sequence b owns ceil((L_b + 1) / bs) blocks
    (room for this step's append), drawn from a seeded permutation of a pool
    with two spare blocks left over."""

    def __init__(self, shape: Shape, spare=2):
        bs = shape.block_size
        self.counts = [(L + 1 + bs - 1) // bs for L in shape.lengths]
        self.max_blocks = max(max(self.counts, default=1), 1)
        self.num_blocks = sum(self.counts) + spare
        if shape.contiguous:
            perm = np.arange(self.num_blocks)
        else:
            perm = I.permutation(I.stream_key(SEED_BASE + shape.config_id, 0,
                                              T_PERM), self.num_blocks)
        self.table = np.zeros((shape.batch, self.max_blocks), dtype=np.int32)
        off = 0
        for b, n in enumerate(self.counts):
            self.table[b, :n] = perm[off:off + n]
            self.table[b, n:] = perm[off + n - 1] if n else 0
            off += n
        self.spare = perm[off:].astype(np.int64)


def _key(shape, layer, tensor):
    return I.stream_key(SEED_BASE + shape.config_id, layer, tensor)


def cache_table(shape):
    return I.fp8_code_table() if shape.dtype == "fp8" else I.normal_bf16_table()


def host_bf16(shape, layer, tensor, dims):
    """bf16 bit patterns (uint16) of a small per-step tensor."""
    return I.host_tensor(I.normal_bf16_table(), _key(shape, layer, tensor),
                         tuple(dims))


def host_scales(shape, layer, tensor):
    """fp8 per-kv-head scale in [1/16, 1/8) and its fp32 reciprocal."""
    u = I.uniform01_f32(_key(shape, layer, tensor), shape.n_kv)
    scale = (np.float32(0.0625) * (np.float32(1) + u)).astype(np.float32)
    inv = (np.float32(1) / scale).astype(np.float32)
    return scale, inv


def host_weights(shape, layer):
    """Indexer head weights, U(0,1) fp32 [batch][idx_heads]."""
    return I.uniform01_f32(_key(shape, layer, T_W),
                           shape.batch * shape.idx_heads).reshape(
        shape.batch, shape.idx_heads)


def cache_dims(shape, paging, width=None, n_kv=None):
    return (paging.num_blocks, shape.n_kv if n_kv is None else n_kv,
            shape.block_size, shape.head_dim if width is None else width)


def _mxfp4_parts(shape, tensor):
    """An MXFP4 cache is drawn as two streams, concatenated per row: the
    code bytes (d/2 wide) and the group scales (d/16 wide)."""
    d = shape.head_dim
    return ((d // 2, I.byte_table(), tensor),
            (d // 16, I.mxfp4_scale_table(), _GROUP_SCALE[tensor]))


def host_cache_full(shape, paging, layer, tensor, width=None, n_kv=None,
                    table=None):
    """The whole physical cache array on the host (small shapes only)."""
    if shape.dtype == "mxfp4" and width is None and table is None:
        return np.concatenate(
            [host_cache_full(shape, paging, layer, t, w, n_kv, tab)
             for w, tab, t in _mxfp4_parts(shape, tensor)], axis=-1)
    dims = cache_dims(shape, paging, width, n_kv)
    tab = cache_table(shape) if table is None else table
    return I.host_tensor(tab, _key(shape, layer, tensor), dims)


def host_cache_compact(shape, paging, layer, tensor, seqs, width=None,
                       n_kv=None, table=None):
    """Host copy of only the blocks the sequences ``seqs`` use, as a compact
    cache plus a remapped block table (for sampled parity at full size).
    Returns (raw [n][n_kv][bs][w], block_table [len(seqs)][max_blocks])."""
    if shape.dtype == "mxfp4" and width is None and table is None:
        parts = [host_cache_compact(shape, paging, layer, t, seqs, w, n_kv,
                                    tab)
                 for w, tab, t in _mxfp4_parts(shape, tensor)]
        return np.concatenate([p[0] for p in parts], axis=-1), parts[0][1]
    dims = cache_dims(shape, paging, width, n_kv)
    per_block = int(np.prod(dims[1:]))
    tab = cache_table(shape) if table is None else table
    blocks, tables = [], []
    for b in seqs:
        n = paging.counts[b]
        phys = paging.table[b, :n].astype(np.int64)
        tables.append(np.arange(len(blocks), len(blocks) + n))
        blocks.extend(phys.tolist())
    idx = (np.asarray(blocks, dtype=np.uint64)[:, None] * np.uint64(per_block)
           + np.arange(per_block, dtype=np.uint64)[None, :])
    raw = I.host_fill(tab, _key(shape, layer, tensor), idx.reshape(-1))
    raw = raw.reshape((len(blocks),) + tuple(dims[1:]))
    mb = max(len(t) for t in tables)
    bt = np.zeros((len(seqs), mb), dtype=np.int64)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
        bt[i, len(t):] = t[-1]
    return raw, bt


# ---------------------------------------------------------------------------
# device instances
# ---------------------------------------------------------------------------
class DeviceWorkload:
    """All device tensors of a workload: per-layer caches and per-step inputs.

    Layers with a shared cache (the sparse schedule) hold one cache object.
    """

    def __init__(self, shape: Shape, device="cuda", layers=None):
        import torch
        from . import PagedCache
        self.shape = s = shape
        self.paging = pg = Paging(s)
        self.device = device
        self.layers = list(range(s.n_layers)) if layers is None else layers
        dev = torch.device(device)
        self.block_table = torch.from_numpy(pg.table).to(dev)
        self.pos = torch.tensor(s.lengths, dtype=torch.int32, device=dev)
        self.seq_lens = torch.tensor(s.seq_lens, dtype=torch.int32, device=dev)
        self.max_seq_len = s.max_seq_len
        cdt = torch.bfloat16 if s.dtype == "bf16" else torch.uint8
        tab = cache_table(s)

        def dev_cache(layer, tensor, width, n_kv):
            if s.dtype == "mxfp4" and width is None:
                parts = []
                for w, ptab, t in _mxfp4_parts(s, tensor):
                    x = torch.empty(cache_dims(s, pg, w, n_kv),
                                    dtype=torch.uint8, device=dev)
                    I.device_fill(x, ptab, _key(s, layer, t))
                    parts.append(x)
                return torch.cat(parts, dim=-1).contiguous()
            t = torch.empty(cache_dims(s, pg, width, n_kv), dtype=cdt,
                            device=dev)
            I.device_fill(t, tab, _key(s, layer, tensor))
            return t

        def dev_bf16(layer, tensor, dims):
            h = host_bf16(s, layer, tensor, dims)
            return torch.from_numpy(h.view(np.int16)).view(
                torch.bfloat16).to(dev)

        self.caches, self.q, self.k_new, self.v_new = {}, {}, {}, {}
        self.idx_cache, self.q_idx, self.w, self.idx_k_new = None, {}, {}, None
        if s.kind == "sparse":
            c = PagedCache(dev_cache(0, T_K, None, 1), dev_cache(0, T_V, None, 1),
                           s.block_size, 1, s.head_dim)
            self.idx_cache = PagedCache(
                self._idx_cache_tensor(dev), None, s.block_size, 1, s.idx_dim)
            for layer in self.layers:
                self.caches[layer] = c
                self.q[layer] = dev_bf16(layer, T_Q, (s.batch, s.n_h,
                                                      s.head_dim))
                if s.modes[layer] != "reuse":
                    self.q_idx[layer] = dev_bf16(layer, T_QIDX,
                                                 (s.batch, s.idx_heads,
                                                  s.idx_dim))
                    self.w[layer] = torch.from_numpy(
                        host_weights(s, layer)).to(dev)
            self.k_new[0] = dev_bf16(0, T_KNEW, (s.batch, 1, s.head_dim))
            self.v_new[0] = dev_bf16(0, T_VNEW, (s.batch, 1, s.head_dim))
            self.idx_k_new = dev_bf16(0, T_IDXKNEW, (s.batch, 1, s.idx_dim))
            return
        for layer in self.layers:
            k = dev_cache(layer, T_K, None, None)
            v = dev_cache(layer, T_V, None, None) if s.has_v else None
            scales = {}
            if s.dtype == "fp8":
                ks, kinv = host_scales(s, layer, T_KSCALE)
                vs, vinv = host_scales(s, layer, T_VSCALE)
                for n, a in (("k_scale", ks), ("k_inv_scale", kinv),
                             ("v_scale", vs), ("v_inv_scale", vinv)):
                    scales[n] = torch.from_numpy(a).to(dev)
            self.caches[layer] = PagedCache(k, v, s.block_size, s.n_kv,
                                            s.head_dim, s.dtype, **scales)
            self.q[layer] = dev_bf16(layer, T_Q, (s.batch, s.n_h, s.head_dim))
            self.k_new[layer] = dev_bf16(layer, T_KNEW,
                                         (s.batch, s.n_kv, s.head_dim))
            if s.has_v:
                self.v_new[layer] = dev_bf16(layer, T_VNEW,
                                             (s.batch, s.n_kv, s.head_dim))

    def _idx_cache_tensor(self, dev):
        import torch
        s, pg = self.shape, self.paging
        t = torch.empty(cache_dims(s, pg, s.idx_dim, 1), dtype=torch.bfloat16,
                        device=dev)
        I.device_fill(t, I.normal_bf16_table(), _key(s, 0, T_IDXK))
        return t
