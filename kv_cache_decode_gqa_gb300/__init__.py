"""kv_cache_decode_gqa_gb300: Python binding of libkvd.so.

The functions here only marshal arguments: they take torch CUDA tensors,
pass their device pointers and the current CUDA stream to the C ABI
(include/kvd.h), and allocate outputs / workspace with torch when the caller
does not pass them. Every step of the computation runs in the library's
CUDA kernels; there is no other path.

Cache layout (per layer): K and V tensors [num_blocks][n_kv][block_size]
[head_dim] of bf16 (torch.bfloat16) or fp8-e4m3 codes (torch.uint8), or
[num_blocks][n_kv][block_size][head_dim/2 + head_dim/16] bytes of MXFP4 rows
(torch.uint8; include/kvd.h gives the row format).
"""
import ctypes
from dataclasses import dataclass
from typing import Optional

from . import _native
from ._native import KvdError, check, lib

__all__ = ["PagedCache", "kv_append", "gqa_decode", "mla_decode",
           "indexer_topk", "indexer_pool", "indexer_topk_pool",
           "BlockPool", "copy_blocks",
           "sparse_decode", "workspace_size",
           "bytes_per_token", "device_error", "launch_count", "set_tuning",
           "KvdError",
           "OP_GQA_DECODE", "OP_MLA_DECODE", "OP_INDEXER_TOPK",
           "OP_SPARSE_DECODE"]

BF16 = 0
FP8_E4M3 = 1
MXFP4 = 2
_DTYPES = {"bf16": BF16, "fp8": FP8_E4M3, "mxfp4": MXFP4}
OP_GQA_DECODE = 0
OP_MLA_DECODE = 1
OP_INDEXER_TOPK = 2
OP_SPARSE_DECODE = 3
OP_INDEXER_TOPK_POOL = 4
POOL_BLOCKS = 2048   # KVD_POOL_BLOCKS
POOL_BLOCK = 8       # KVD_POOL_BLOCK


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype=None, numel=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return t


@dataclass
class PagedCache:
    """One layer's paged cache. ``v`` is None for a K-only cache."""
    k: "torch.Tensor"
    v: Optional["torch.Tensor"]
    block_size: int
    n_kv: int
    head_dim: int
    dtype: str = "bf16"          # "bf16" | "fp8" | "mxfp4"
    k_scale: Optional["torch.Tensor"] = None      # fp32 [n_kv]
    v_scale: Optional["torch.Tensor"] = None
    k_inv_scale: Optional["torch.Tensor"] = None
    v_inv_scale: Optional["torch.Tensor"] = None

    @property
    def num_blocks(self):
        return self.k.shape[0]

    def struct(self):
        import torch
        want = torch.bfloat16 if self.dtype == "bf16" else torch.uint8
        _need(self.k, "cache.k", want)
        if self.v is not None:
            _need(self.v, "cache.v", want, self.k.numel())
        row = (self.head_dim // 2 + self.head_dim // 16
               if self.dtype == "mxfp4" else self.head_dim)
        shape = (self.num_blocks, self.n_kv, self.block_size, row)
        if tuple(self.k.shape) != shape:
            raise ValueError(f"cache.k shape {tuple(self.k.shape)} != {shape}")
        for n in ("k_scale", "v_scale", "k_inv_scale", "v_inv_scale"):
            t = getattr(self, n)
            if t is not None:
                _need(t, n, torch.float32, self.n_kv)
        return _native.KvdCache(
            _ptr(self.k), _ptr(self.v), self.num_blocks, self.block_size,
            self.n_kv, self.head_dim, _DTYPES[self.dtype],
            0, _ptr(self.k_scale), _ptr(self.v_scale), _ptr(self.k_inv_scale),
            _ptr(self.v_inv_scale))


SEQS_STABLE = 1  # KVD_SEQS_STABLE
SEQS_PREFIX_READY = 2  # KVD_SEQS_PREFIX_READY (with SEQS_STABLE)


def _seqs(block_table, seq_lens, max_seq_len, flags=0, window=0,
          window_start=None):
    import torch
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != seq_lens.numel():
        raise ValueError("block_table must be [batch][max_blocks_per_seq]")
    if window_start is not None:
        _need(window_start, "window_start", torch.int32, seq_lens.numel())
    return _native.KvdSeqs(_ptr(block_table), _ptr(seq_lens),
                           block_table.shape[0], block_table.shape[1],
                           int(max_seq_len), int(flags), int(window),
                           _ptr(window_start))


def workspace_size(op, cache, block_table, seq_lens, max_seq_len, n_h, k=0,
                   window=0):
    """Workspace bytes of a call (kvd_workspace_size); a GQA decode's window
    is part of its plan (short windows need none)."""
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len, window=window)
    out = ctypes.c_size_t(0)
    check(lib().kvd_workspace_size(op, ctypes.byref(c), ctypes.byref(s), n_h,
                                   k, ctypes.byref(out)))
    return out.value


def _workspace(op, cache, block_table, seq_lens, max_seq_len, n_h, k,
               workspace, window=0):
    import torch
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8)
        return workspace
    n = workspace_size(op, cache, block_table, seq_lens, max_seq_len, n_h, k,
                       window)
    # every partial a call keeps here is written before it is read
    return torch.empty(max(n, 256), dtype=torch.uint8,
                       device=block_table.device)


def kv_append(cache, block_table, pos, k_new, v_new=None, stream=None):
    """Write k_new (and v_new) [batch][n_kv][head_dim] bf16 at slot pos[b]."""
    import torch
    c = cache.struct()
    _need(block_table, "block_table", torch.int32)
    _need(pos, "pos", torch.int32)
    _need(k_new, "k_new", torch.bfloat16)
    if v_new is not None:
        _need(v_new, "v_new", torch.bfloat16, k_new.numel())
    check(lib().kvd_kv_append(ctypes.byref(c), _ptr(block_table),
                              block_table.shape[1], _ptr(pos), pos.numel(),
                              _ptr(k_new), _ptr(v_new), _stream(stream)))


def _outputs(q, n_h, dv, out, lse, want_lse):
    import torch
    B = q.shape[0]
    if out is None:
        out = torch.empty((B, n_h, dv), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, B * n_h * dv)
    if lse is None and want_lse:
        lse = torch.empty((B, n_h), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, B * n_h)
    return out, lse


def gqa_decode(cache, block_table, seq_lens, max_seq_len, q, scale=None,
               out=None, lse=None, workspace=None, want_lse=True,
               stream=None, seqs_flags=0, window=0, window_start=None):
    """GQA/MHA decode: q [batch][n_h][head_dim] bf16 -> (out, lse).
    seqs_flags: 0 or SEQS_STABLE (see KVD_SEQS_STABLE in kvd.h). window W >
    0: sliding-window decode over positions [max(s_b, len_b - W), len_b),
    s_b = window_start[b] (int32 device tensor) or 0."""
    import torch
    _need(q, "q", torch.bfloat16)
    n_h = q.shape[1]
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len, seqs_flags, window,
              window_start)
    out, lse = _outputs(q, n_h, cache.head_dim, out, lse, want_lse)
    ws = _workspace(OP_GQA_DECODE, cache, block_table, seq_lens, max_seq_len,
                    n_h, 0, workspace, window)
    check(lib().kvd_gqa_decode(ctypes.byref(c), ctypes.byref(s), _ptr(q), n_h,
                               float(scale or 0.0), _ptr(out), _ptr(lse),
                               _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def gqa_append_decode(cache, block_table, seq_lens, max_seq_len, pos, k_new,
                      v_new, q, scale=None, out=None, lse=None,
                      workspace=None, want_lse=True, stream=None,
                      seqs_flags=0, window=0, window_start=None):
    """kv_append then gqa_decode in one pass (kvd_gqa_append_decode);
    window / window_start as for gqa_decode."""
    import torch
    _need(q, "q", torch.bfloat16)
    _need(pos, "pos", torch.int32)
    _need(k_new, "k_new", torch.bfloat16)
    _need(v_new, "v_new", torch.bfloat16)
    n_h = q.shape[1]
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len, seqs_flags, window,
              window_start)
    out, lse = _outputs(q, n_h, cache.head_dim, out, lse, want_lse)
    ws = _workspace(OP_GQA_DECODE, cache, block_table, seq_lens, max_seq_len,
                    n_h, 0, workspace, window)
    check(lib().kvd_gqa_append_decode(
        ctypes.byref(c), ctypes.byref(s), _ptr(pos), _ptr(k_new), _ptr(v_new),
        _ptr(q), n_h, float(scale or 0.0), _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out, lse


def mla_decode(cache, block_table, seq_lens, max_seq_len, q, d_c=512,
               scale=None, out=None, lse=None, workspace=None, want_lse=True,
               stream=None):
    """Latent-cache decode: q [batch][n_h][d_c + d_rope] -> out [..][d_c]."""
    import torch
    _need(q, "q", torch.bfloat16)
    n_h = q.shape[1]
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len)
    out, lse = _outputs(q, n_h, d_c, out, lse, want_lse)
    ws = _workspace(OP_MLA_DECODE, cache, block_table, seq_lens, max_seq_len,
                    n_h, 0, workspace)
    check(lib().kvd_mla_decode(ctypes.byref(c), d_c, ctypes.byref(s), _ptr(q),
                               n_h, float(scale or 0.0), _ptr(out), _ptr(lse),
                               _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def indexer_topk(cache, block_table, seq_lens, max_seq_len, q_idx, w, k,
                 indices=None, scores=None, workspace=None, stream=None,
                 seqs_flags=0):
    """Indexer scores + top-k: returns (indices [batch][k] int32, scores).
    seqs_flags: SEQS_STABLE [| SEQS_PREFIX_READY] (see kvd_seqs)."""
    import torch
    _need(q_idx, "q_idx", torch.bfloat16)
    _need(w, "w", torch.float32, q_idx.shape[0] * q_idx.shape[1])
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len, seqs_flags)
    B = q_idx.shape[0]
    if indices is None:
        indices = torch.empty((B, k), dtype=torch.int32, device=q_idx.device)
    _need(indices, "indices", torch.int32, B * k)
    if scores is not None:
        _need(scores, "scores", torch.float32, B * max(max_seq_len, 1))
        ws = None
    else:
        ws = _workspace(OP_INDEXER_TOPK, cache, block_table, seq_lens,
                        max_seq_len, q_idx.shape[1], k, workspace)
    check(lib().kvd_indexer_topk(ctypes.byref(c), ctypes.byref(s),
                                 _ptr(q_idx), q_idx.shape[1], _ptr(w), k,
                                 _ptr(indices), _ptr(scores), _ptr(ws),
                                 0 if ws is None else ws.numel(),
                                 _stream(stream)))
    return indices, scores


def indexer_pool(block_table, seq_lens, max_seq_len, indices, pool=None,
                 pool_n=None, stream=None):
    """The hierarchical indexer's pool of a selection indices [batch][k]:
    returns (pool [batch][POOL_BLOCKS] ascending 8-position block ids,
    pool_n [batch] their counts)."""
    import torch
    _need(indices, "indices", torch.int32)
    B, k = indices.shape
    s = _seqs(block_table, seq_lens, max_seq_len)
    if pool is None:
        pool = torch.empty((B, POOL_BLOCKS), dtype=torch.int32,
                           device=indices.device)
    if pool_n is None:
        pool_n = torch.empty((B,), dtype=torch.int32, device=indices.device)
    _need(pool, "pool", torch.int32, B * POOL_BLOCKS)
    _need(pool_n, "pool_n", torch.int32, B)
    check(lib().kvd_indexer_pool(ctypes.byref(s), _ptr(indices), k,
                                 _ptr(pool), _ptr(pool_n), _stream(stream)))
    return pool, pool_n


def indexer_topk_pool(cache, block_table, seq_lens, max_seq_len, q_idx, w,
                      pool, pool_n, k, indices=None, scores=None,
                      workspace=None, stream=None):
    """A Reindex layer over a pool: indexer scores of the pool's candidates
    and their top k. Returns (indices [batch][k] int32, scores)."""
    import torch
    _need(q_idx, "q_idx", torch.bfloat16)
    _need(w, "w", torch.float32, q_idx.shape[0] * q_idx.shape[1])
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len)
    B = q_idx.shape[0]
    _need(pool, "pool", torch.int32, B * POOL_BLOCKS)
    _need(pool_n, "pool_n", torch.int32, B)
    if indices is None:
        indices = torch.empty((B, k), dtype=torch.int32, device=q_idx.device)
    _need(indices, "indices", torch.int32, B * k)
    if scores is not None:
        _need(scores, "scores", torch.float32, B * POOL_BLOCKS * POOL_BLOCK)
        ws = None
    else:
        ws = _workspace(OP_INDEXER_TOPK_POOL, cache, block_table, seq_lens,
                        max_seq_len, q_idx.shape[1], k, workspace)
    check(lib().kvd_indexer_topk_pool(ctypes.byref(c), ctypes.byref(s),
                                      _ptr(q_idx), q_idx.shape[1], _ptr(w),
                                      _ptr(pool), _ptr(pool_n), k,
                                      _ptr(indices), _ptr(scores), _ptr(ws),
                                      0 if ws is None else ws.numel(),
                                      _stream(stream)))
    return indices, scores


def sparse_decode(cache, block_table, seq_lens, max_seq_len, indices, q,
                  scale=None, out=None, lse=None, workspace=None,
                  want_lse=True, stream=None):
    """Decode over the positions in indices [batch][k] (-1 = skip)."""
    import torch
    _need(q, "q", torch.bfloat16)
    _need(indices, "indices", torch.int32)
    n_h = q.shape[1]
    k = indices.shape[1]
    c = cache.struct()
    s = _seqs(block_table, seq_lens, max_seq_len)
    out, lse = _outputs(q, n_h, cache.head_dim, out, lse, want_lse)
    ws = _workspace(OP_SPARSE_DECODE, cache, block_table, seq_lens,
                    max_seq_len, n_h, k, workspace)
    check(lib().kvd_sparse_decode(ctypes.byref(c), ctypes.byref(s),
                                  _ptr(indices), k, _ptr(q), n_h,
                                  float(scale or 0.0), _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


class BlockPool:
    """The library's copy-on-write block pool (kvd_block_pool_*): host
    reference counts of num_blocks physical blocks. Block tables and id
    lists are host numpy int32 arrays."""

    def __init__(self, num_blocks):
        h = ctypes.c_void_p()
        check(lib().kvd_block_pool_create(int(num_blocks), ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            lib().kvd_block_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ids(blocks):
        import numpy as np
        a = np.ascontiguousarray(blocks, dtype=np.int32)
        return a, a.ctypes.data

    def free_count(self):
        return int(lib().kvd_block_pool_free_count(self._h))

    def refcount(self, block):
        return int(lib().kvd_block_pool_refcount(self._h, int(block)))

    def alloc(self, n):
        import numpy as np
        out = np.empty(int(n), dtype=np.int32)
        check(lib().kvd_block_pool_alloc(self._h, int(n), out.ctypes.data))
        return out

    def share(self, blocks):
        a, p = self._ids(blocks)
        check(lib().kvd_block_pool_share(self._h, p, a.size))

    def release(self, blocks):
        a, p = self._ids(blocks)
        check(lib().kvd_block_pool_release(self._h, p, a.size))

    def prepare_append(self, block_table, pos, block_size):
        """block_table: host int32 [batch][max_blocks], updated in place;
        pos: host int32 [batch]. Returns (src, dst) block ids of the copies
        to make before appending."""
        import numpy as np
        assert block_table.dtype == np.int32 and block_table.flags.c_contiguous
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        B, M = block_table.shape
        src = np.empty(max(B, 1), dtype=np.int32)
        dst = np.empty(max(B, 1), dtype=np.int32)
        n = ctypes.c_int32(0)
        check(lib().kvd_block_pool_prepare_append(
            self._h, block_table.ctypes.data, B, M, pos.ctypes.data,
            int(block_size), src.ctypes.data, dst.ctypes.data,
            ctypes.byref(n)))
        return src[:n.value].copy(), dst[:n.value].copy()


def copy_blocks(cache, src, dst, stream=None):
    """Whole blocks dst[i] := src[i] of the cache's K and V (device int32
    tensors)."""
    import torch
    _need(src, "src", torch.int32)
    _need(dst, "dst", torch.int32, src.numel())
    c = cache.struct()
    check(lib().kvd_copy_blocks(ctypes.byref(c), _ptr(src), _ptr(dst),
                                src.numel(), _stream(stream)))


def bytes_per_token(n_l, n_kv, d_h, elem_bytes):
    return int(lib().kvd_bytes_per_token(n_l, n_kv, d_h, elem_bytes))


# device error bits (KVD_DEVERR_* in kvd.h)
DEVERR_BLOCK, DEVERR_POS, DEVERR_TIMEOUT, DEVERR_INDEX, DEVERR_LEN = (
    1, 2, 4, 8, 16)


def set_tuning(decode_ctas=0, mla_cuda_cores=False):
    """Process-wide launch overrides (kvd_set_tuning): decode_ctas > 0
    forces the CTAs of every decode launch; mla_cuda_cores runs the latent
    decode on its CUDA-core kernel."""
    check(lib().kvd_set_tuning(int(decode_ctas), int(bool(mla_cuda_cores))))


def launch_count():
    """Kernels the library has launched in this process (a launch captured
    into a CUDA graph counts once, when captured)."""
    return int(lib().kvd_launch_count())


def device_error():
    """Synchronise, then read and clear the device error word."""
    code = ctypes.c_int32(0)
    check(lib().kvd_device_error(ctypes.byref(code)))
    return code.value
