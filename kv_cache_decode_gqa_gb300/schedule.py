"""Static layer schedule of the top-k sparse path ("890 bytes a token ...",
section 3): every layer is statically Full, Reindex or Reuse. Full and
Reindex layers score the shared indexer key cache with their own indexer
query and pick a fresh top-k; a Reuse layer attends to the selection of the
most recent layer that made one. Every layer attends with its own query
over the shared main K/V cache.

With a pool size (section 4, the hierarchical indexer), the first Full
layer's selection also publishes a candidate pool (its 8-position blocks,
at most 2,048), and every later Reindex layer picks its own top-``pool_k``
from the pool instead of the whole context.

Host orchestration only: each step is one call of the C ABI (kv_append,
indexer_topk, indexer_pool, indexer_topk_pool, sparse_decode), all on the
caller's stream.
"""
from . import (indexer_pool, indexer_topk, indexer_topk_pool, kv_append,
               sparse_decode)

MODES = ("full", "reindex", "reuse")


def sparse_schedule_step(modes, cache, idx_cache, block_table, pos, seq_lens,
                         max_seq_len, q, q_idx, w, k, outs, indices,
                         k_new=None, v_new=None, idx_k_new=None,
                         workspaces=None, topk_workspace=None, lses=None,
                         pool_k=None, pool=None, pool_n=None,
                         pool_workspace=None, stream=None, seqs_flags=0):
    """One decode step through a static schedule.

    modes[l] in MODES (the first layer may not be "reuse"); q[l], q_idx[l],
    w[l], outs[l], indices[l]: per-layer tensors (q_idx / w only for layers
    that score). If k_new / v_new / idx_k_new are given, the step first
    appends the new token to the shared caches at ``pos`` (a Full layer's
    own key and value). With ``pool_k``, Reindex layers select
    ``pool_k`` positions inside the first Full layer's pool (``pool`` /
    ``pool_n``: optional buffers; ``indices[l]`` of those layers then hold
    ``pool_k`` entries). ``seqs_flags`` (SEQS_STABLE, SEQS_PREFIX_READY)
    passes to the indexer calls. Returns the index tensor each layer
    attended to.
    """
    if modes and modes[0] == "reuse":
        raise ValueError("the first layer must pick its own top-k")
    if k_new is not None:
        kv_append(cache, block_table, pos, k_new, v_new, stream=stream)
    if idx_k_new is not None:
        kv_append(idx_cache, block_table, pos, idx_k_new, stream=stream)
    used = []
    current = None
    pooled = False
    for layer, mode in enumerate(modes):
        if mode not in MODES:
            raise ValueError(f"unknown layer mode {mode!r}")
        if mode == "reindex" and pooled:
            current = indices[layer]
            indexer_topk_pool(idx_cache, block_table, seq_lens, max_seq_len,
                              q_idx[layer], w[layer], pool, pool_n, pool_k,
                              indices=current, workspace=pool_workspace,
                              stream=stream)
        elif mode != "reuse":
            current = indices[layer]
            indexer_topk(idx_cache, block_table, seq_lens, max_seq_len,
                         q_idx[layer], w[layer], k, indices=current,
                         workspace=topk_workspace, stream=stream,
                         seqs_flags=seqs_flags)
            if mode == "full" and pool_k is not None and not pooled:
                pool, pool_n = indexer_pool(block_table, seq_lens,
                                            max_seq_len, current, pool=pool,
                                            pool_n=pool_n, stream=stream)
                pooled = True
        sparse_decode(cache, block_table, seq_lens, max_seq_len, current,
                      q[layer], out=outs[layer],
                      lse=None if lses is None else lses[layer],
                      want_lse=lses is not None,
                      workspace=None if workspaces is None
                      else workspaces[layer], stream=stream)
        used.append(current)
    return used
