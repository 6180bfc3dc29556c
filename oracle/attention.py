"""Decode attention over a paged KV cache, written out plainly in fp64.

TEST INFRASTRUCTURE (see the package docstring): imported only by the tests,
the smoke check and the benchmark's CPU-baseline / reference leg.

Pages this follows (cited by page title and section):
  [KV]  "KV cache" (this.guide)
  [POD] "My Weird Prompts" episode 640482 (podcast transcript)
  [890] "890 bytes a token: DeepSeek's KV cache trick, and the eval it should
        make you write"

Parity status (each function is pinned in tests/test_oracle_pins.py):
  attend / attend_scores ........ pinned (hand-worked example, brute force,
                                  cached = full causal recompute, T=1,
                                  identical keys, weights sum to 1)
  gather_* / kv_append .......... pinned (contiguous vs permuted tables,
                                  byte copy, fp8 encoder pins)
  gqa_decode .................... pinned (MHA special case, repeat-interleave;
                                  window = the last W rows, W >= T = full)
  mla_decode .................... pinned (absorbed = explicit decompression)
  indexer_scores ................ pinned (brute-force loops, exact-arithmetic set)
  topk_select / indexer_topk .... pinned (sorted() brute force, ties, k >= T)
  sparse_decode ................. pinned (all positions = dense; subset = dense
                                  over the subset)
  lse_merge / split_decode ...... pinned (any split = unsplit)
  bytes_per_token / cache_bytes / paged_waste_slots ... pinned (page figures)
  sparse_schedule ............... pinned through its parts (Reuse = earlier
                                  indices; Reindex = own scores; with a pool:
                                  Reindex picks inside the pool)
  indexer_pool / pool_positions /
  indexer_topk_in_pool .......... pinned (set brute force, the cap, the
                                  page's 16,384 figure, full pool = full
                                  top-k, plain-loop top-k over candidates)
"""
import math

import numpy as np

from .numerics import (bf16_bits_to_f64, e4m3_codes_to_f64, e4m3_encode_f32,
                       mxfp4_encode_rows, mxfp4_rows_to_f64)


# ---------------------------------------------------------------------------
# storage decoding
# ---------------------------------------------------------------------------
def decode_rows(raw, dtype, scale=None, d=None):
    """Raw cache rows [n_kv, T, row] -> float64 [n_kv, T, d].

    bf16 rows are exact. fp8 rows are the E4M3 code value times the fp32
    per-(kv head) scale, also exact in fp64 ([KV] "Fewer bits per number":
    the cache holds fewer bits per number; the scale restores the range).
    mxfp4 rows ([890] section 6) are E2M1 code values times their 16-channel
    group's E4M3 scale, exact in fp64; ``d`` is the row's channel count.
    """
    if dtype == "bf16":
        return bf16_bits_to_f64(raw)
    if dtype == "fp8":
        vals = e4m3_codes_to_f64(raw)
        s = np.asarray(scale, dtype=np.float32).astype(np.float64)
        return vals * s[:, None, None]
    if dtype == "mxfp4":
        return mxfp4_rows_to_f64(raw, d)
    raise ValueError(f"unknown cache dtype {dtype!r}")


# ---------------------------------------------------------------------------
# paging ([KV] "The allocator, not the algorithm"; [POD] on PagedAttention)
# ---------------------------------------------------------------------------
def gather_positions(block_table_row, positions, block_size):
    """Logical token positions -> (physical block, slot inside the block).

    A sequence's logical position t lives in the block its block table names
    for logical block t // block_size, at slot t % block_size.
    """
    positions = np.asarray(positions, dtype=np.int64)
    table = np.asarray(block_table_row, dtype=np.int64)
    return table[positions // block_size], positions % block_size


def gather_rows(raw, block_table_row, positions, block_size):
    """Rows of a cache stored as [num_blocks][n_kv][block_size][d] for the
    given logical positions, returned as [n_kv][len(positions)][d] (the
    per-layer [n_kv, L, d_h] tensor of [KV] "Two tensors per layer")."""
    blk, slot = gather_positions(block_table_row, positions, block_size)
    return np.ascontiguousarray(raw[blk, :, slot, :].transpose(1, 0, 2))


def kv_append(raw, block_table, pos, new_rows, block_size, dtype="bf16",
              inv_scale=None):
    """Write one new token per sequence into the cache (returns a new array).

    [POD]: each decode step appends the new token's key and value, so the
    cache grows by one entry per layer per token. ``new_rows`` is
    [B][n_kv][d] bf16 bits; ``pos[b]`` is the slot index (the cached length
    before the append).

    fp8: the stored code is E4M3(round-to-nearest-even, saturating) of the
    fp32 product x * inv_scale[kv_head], with x the bf16 input widened to fp32
    and the product rounded once to fp32. mxfp4: the row's MXFP4 encoding
    (numerics.mxfp4_encode_rows); ``raw``'s last axis is the row's bytes.
    """
    out = raw.copy()
    new_rows = np.asarray(new_rows, dtype=np.uint16)
    for b, p in enumerate(np.asarray(pos, dtype=np.int64)):
        blk, slot = gather_positions(block_table[b], [p], block_size)
        if dtype == "bf16":
            out[blk[0], :, slot[0], :] = new_rows[b]
        elif dtype == "fp8":
            x = bf16_bits_to_f64(new_rows[b]).astype(np.float32)
            inv = np.asarray(inv_scale, dtype=np.float32)[:, None]
            y = (x * inv).astype(np.float32)          # one fp32 rounding
            out[blk[0], :, slot[0], :] = e4m3_encode_f32(y)
        elif dtype == "mxfp4":
            out[blk[0], :, slot[0], :] = mxfp4_encode_rows(new_rows[b])
        else:
            raise ValueError(dtype)
    return out


# ---------------------------------------------------------------------------
# attention at one position ([KV] "A cache you keep because attention looks
# backwards": o_t = softmax(q_t K^T / sqrt(d_h) + M) V over positions <= t)
# ---------------------------------------------------------------------------
def attend_scores(S, V):
    """Softmax over the last axis of the scaled scores ``S`` [n_q][T], then
    the weighted sum of the rows of ``V`` [T][d_v].

    Returns (out [n_q][d_v], lse [n_q]) with lse = log sum_t exp(S_t), the
    natural-log normaliser. T = 0 gives out = 0 and lse = -inf.
    """
    S = np.asarray(S, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n_q, T = S.shape
    if T == 0:
        return np.zeros((n_q, V.shape[1])), np.full(n_q, -np.inf)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    out = (P @ V) / l
    lse = m[:, 0] + np.log(l[:, 0])
    return out, lse


def attend(q, K, V, scale):
    """softmax(scale * q K^T) V for query rows q [n_q][d_k] against the keys
    K [T][d_k] and values V [T][d_v] of one KV head."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    return attend_scores(scale * (q @ K.T), V)


# ---------------------------------------------------------------------------
# grouped-query decode ([KV] "Fewer KV heads, held at the same quality";
# [POD] on MQA / GQA). Query head h reads KV head h // (n_h / n_kv).
# ---------------------------------------------------------------------------
def gqa_decode(q, k_raw, v_raw, block_table, seq_lens, block_size,
               scale=None, dtype="bf16", k_scale=None, v_scale=None,
               window=0, window_start=None):
    """One decode step of GQA/MHA attention for every sequence.

    window W > 0 ([890] section 7, SWA bounded replay: a query at position
    i attends to keys in [max(s, i - W + 1), i]; at decode i = seq_len - 1):
    sequence b attends to positions [max(s_b, seq_len - W), seq_len), s_b =
    window_start[b] or 0.

    q: [B][n_h][d] float64. k_raw / v_raw: cache storage
    [num_blocks][n_kv][block_size][row] (row = d elements, or an MXFP4 row's
    bytes). seq_lens[b] = visible length (after the append). Returns out
    [B][n_h][d], lse [B][n_h].
    """
    q = np.asarray(q, dtype=np.float64)
    B, n_h, d = q.shape
    n_kv = k_raw.shape[1]
    g = n_h // n_kv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, n_h, d))
    lse = np.zeros((B, n_h))
    for b in range(B):
        T = int(seq_lens[b])
        lo = 0 if window_start is None else int(window_start[b])
        if window:
            lo = max(lo, T - int(window))
        pos = np.arange(min(max(lo, 0), T), T)
        K = decode_rows(gather_rows(k_raw, block_table[b], pos, block_size),
                        dtype, k_scale, d)
        V = decode_rows(gather_rows(v_raw, block_table[b], pos, block_size),
                        dtype, v_scale, d)
        for kv in range(n_kv):
            heads = slice(kv * g, (kv + 1) * g)
            out[b, heads], lse[b, heads] = attend(q[b, heads], K[kv], V[kv],
                                                  scale)
    return out, lse


# ---------------------------------------------------------------------------
# latent cache ([KV] "Caching a compressed latent instead of the keys", the
# MLA footnote of "Where the memory actually goes": a 512-dim latent plus a
# 64-dim shared positional key per token and layer)
# ---------------------------------------------------------------------------
def mla_decode(q, lat_raw, block_table, seq_lens, block_size, d_c=512,
               scale=None):
    """Absorbed-query MLA decode.

    Each cached row is [c (d_c) | k_rope (d_r)]. A query row is
    [q_lat (d_c) | q_rope (d_r)], with the key up-projection already folded
    into q_lat. Score = scale * (q_lat . c_t + q_rope . k_rope_t);
    out = softmax(scores) . c (the value side stays in latent space).
    q: [B][n_h][d_c + d_r]; lat_raw: [num_blocks][1][block_size][d_c + d_r].
    """
    q = np.asarray(q, dtype=np.float64)
    B, n_h, d_row = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d_row)
    out = np.zeros((B, n_h, d_c))
    lse = np.zeros((B, n_h))
    for b in range(B):
        pos = np.arange(int(seq_lens[b]))
        R = bf16_bits_to_f64(gather_rows(lat_raw, block_table[b], pos,
                                         block_size))[0]
        c, k_rope = R[:, :d_c], R[:, d_c:]
        q_lat, q_rope = q[b, :, :d_c], q[b, :, d_c:]
        S = scale * (q_lat @ c.T + q_rope @ k_rope.T)
        out[b], lse[b] = attend_scores(S, c)
    return out, lse


# ---------------------------------------------------------------------------
# top-k sparse path ([POD] on DeepSeek Sparse Attention: a lightning indexer
# scores the prefix and a top-k subset, k = 2048, is read; [890] section 3 on
# Full / Reindex / Reuse layers)
# ---------------------------------------------------------------------------
def indexer_scores(q_idx, w, idx_raw, block_table, seq_lens, block_size):
    """s_t = sum_j w_j * max(0, q_j . k_t) for every visible position t.

    q_idx: [B][H_I][d_I] float64, w: [B][H_I], idx_raw: K-only cache
    [num_blocks][1][block_size][d_I]. Returns a list of B arrays [T_b].
    """
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    scores = []
    for b in range(q_idx.shape[0]):
        pos = np.arange(int(seq_lens[b]))
        Kx = bf16_bits_to_f64(gather_rows(idx_raw, block_table[b], pos,
                                          block_size))[0]
        dots = Kx @ q_idx[b].T                      # [T][H_I]
        scores.append(np.maximum(dots, 0.0) @ w[b])
    return scores


def topk_select(s, k):
    """The k positions with the largest scores; equal scores go to the lower
    position; returned in ascending position order, padded with -1 when
    fewer than k positions exist."""
    s = np.asarray(s, dtype=np.float64)
    T = s.shape[0]
    order = np.lexsort((np.arange(T), -s))         # score desc, index asc
    chosen = np.sort(order[:min(k, T)])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.shape[0]] = chosen
    return out


def indexer_topk(q_idx, w, idx_raw, block_table, seq_lens, block_size, k):
    """Indexer scores, then top-k per sequence. Returns (indices [B][k],
    scores list)."""
    scores = indexer_scores(q_idx, w, idx_raw, block_table, seq_lens,
                            block_size)
    idx = np.stack([topk_select(s, k) for s in scores])
    return idx, scores


def sparse_decode(q, k_raw, v_raw, block_table, seq_lens, block_size,
                  indices, scale=None):
    """GQA decode restricted to the selected positions of each sequence.

    Entries < 0 (padding) and >= seq_len are skipped.
    """
    q = np.asarray(q, dtype=np.float64)
    B, n_h, d = q.shape
    n_kv = k_raw.shape[1]
    g = n_h // n_kv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, n_h, v_raw.shape[3]))
    lse = np.zeros((B, n_h))
    for b in range(B):
        sel = np.asarray(indices[b], dtype=np.int64)
        sel = sel[(sel >= 0) & (sel < int(seq_lens[b]))]
        K = bf16_bits_to_f64(gather_rows(k_raw, block_table[b], sel,
                                         block_size))
        V = bf16_bits_to_f64(gather_rows(v_raw, block_table[b], sel,
                                         block_size))
        for kv in range(n_kv):
            heads = slice(kv * g, (kv + 1) * g)
            out[b, heads], lse[b, heads] = attend(q[b, heads], K[kv], V[kv],
                                                  scale)
    return out, lse


# ---------------------------------------------------------------------------
# hierarchical indexer ([890] section 4: the first Full layer publishes the
# blocks its selection came from as a candidate pool, capped at 2,048 blocks
# of 8 positions; later Reindex layers pick their own top-k only from the
# pool. [POD]: "two thousand forty-eight blocks times eight positions,
# sixteen thousand three hundred eighty-four candidates")
# ---------------------------------------------------------------------------
POOL_BLOCK = 8      # positions per pool block
POOL_CAP = 2048     # blocks a pool holds


def indexer_pool(indices, seq_lens, cap=POOL_CAP):
    """The pool a Full layer publishes, per sequence: the ascending ids of
    the 8-position blocks (position // 8) that hold its selected positions,
    entries < 0 or >= seq_len ignored, at most ``cap`` of them (the lowest:
    a reading, the pages give only the cap). Returns a list of int64
    arrays."""
    pools = []
    for b, row in enumerate(np.asarray(indices, dtype=np.int64)):
        ok = row[(row >= 0) & (row < int(seq_lens[b]))]
        pools.append(np.unique(ok // POOL_BLOCK)[:cap])
    return pools


def pool_positions(pool_blocks, seq_len):
    """The candidates of a pool: every position of its blocks that is
    visible (< seq_len), ascending."""
    blocks = np.asarray(pool_blocks, dtype=np.int64)
    pos = (blocks[:, None] * POOL_BLOCK + np.arange(POOL_BLOCK)).reshape(-1)
    return pos[pos < int(seq_len)]


def indexer_topk_in_pool(q_idx, w, idx_raw, block_table, seq_lens,
                         block_size, pools, k):
    """A Reindex layer over a pool: the indexer score of each candidate,
    then the k largest among the candidates (equal scores to the lower
    position), as positions in ascending order, -1 padded. Returns
    (indices [B][k], list of candidate-score arrays)."""
    full = indexer_scores(q_idx, w, idx_raw, block_table, seq_lens,
                          block_size)
    idx, cand = [], []
    for b, s in enumerate(full):
        pos = pool_positions(pools[b], seq_lens[b])
        sel = topk_select(s[pos], k)
        idx.append(np.where(sel >= 0, pos[np.maximum(sel, 0)], -1))
        cand.append(s[pos])
    return np.stack(idx).astype(np.int32), cand


def sparse_schedule(modes, q, q_idx, w, k_raw, v_raw, idx_raw, block_table,
                    seq_lens, block_size, k, scale=None, pool_k=None):
    """A static layer schedule over one shared main cache and one shared
    indexer cache ([890] section 3: Full and Reindex layers score and pick
    their own top-k; a Reuse layer attends to the most recent selection).
    With ``pool_k`` ([890] section 4), the first Full layer's selection
    publishes a pool and every Reindex layer picks its top-``pool_k`` from
    that pool.

    modes: sequence of "full" | "reindex" | "reuse" (the first must not be
    "reuse"); q[l], q_idx[l], w[l]: per-layer inputs. Returns
    (outs, lses, indices) lists over layers.
    """
    outs, lses, sel = [], [], []
    current = None
    pools = None
    for layer, mode in enumerate(modes):
        if mode == "reindex" and pool_k is not None and pools is not None:
            current, _ = indexer_topk_in_pool(q_idx[layer], w[layer], idx_raw,
                                              block_table, seq_lens,
                                              block_size, pools, pool_k)
        elif mode in ("full", "reindex"):
            current, _ = indexer_topk(q_idx[layer], w[layer], idx_raw,
                                      block_table, seq_lens, block_size, k)
            if mode == "full" and pool_k is not None and pools is None:
                pools = indexer_pool(current, seq_lens)
        elif mode != "reuse" or current is None:
            raise ValueError(f"bad schedule at layer {layer}: {mode}")
        o, l = sparse_decode(q[layer], k_raw, v_raw, block_table, seq_lens,
                             block_size, current, scale)
        outs.append(o)
        lses.append(l)
        sel.append(current)
    return outs, lses, sel


# ---------------------------------------------------------------------------
# split-K merge: attention over a union of disjoint position sets, from the
# per-set normalised outputs and log-sum-exps (exact up to rounding, as
# FlashAttention is exact: [POD] on FlashAttention)
# ---------------------------------------------------------------------------
def lse_merge(parts):
    """parts: list of (out_s [n][d], lse_s [n]) over disjoint position sets.

    out = sum_s exp(lse_s - M) out_s / sum_s exp(lse_s - M), M = max_s lse_s;
    lse = M + log sum_s exp(lse_s - M). Empty sets (lse = -inf) add nothing.
    """
    outs = np.stack([np.asarray(o, dtype=np.float64) for o, _ in parts])
    lses = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])
    M = lses.max(axis=0)
    safe_M = np.where(np.isfinite(M), M, 0.0)
    wts = np.where(np.isfinite(lses), np.exp(lses - safe_M), 0.0)
    tot = wts.sum(axis=0)
    out = np.where(tot[:, None] > 0,
                   (wts[:, :, None] * outs).sum(axis=0)
                   / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
    lse = np.where(tot > 0, safe_M + np.log(np.where(tot > 0, tot, 1.0)),
                   -np.inf)
    return out, lse


def split_decode(q, K, V, scale, boundaries):
    """attend() over the position ranges [b_i, b_{i+1}) separately, then
    lse_merge(): the flash-decoding split of one head group."""
    parts = []
    for lo, hi in zip(boundaries[:-1], boundaries[1:]):
        parts.append(attend(q, K[lo:hi], V[lo:hi], scale))
    return lse_merge(parts)


# ---------------------------------------------------------------------------
# size accounting ([KV] "The size formula"; "The allocator, not the
# algorithm")
# ---------------------------------------------------------------------------
def bytes_per_token(n_l, n_kv, d_h, b):
    """Cache bytes per token: two tensors (K and V) x layers x KV heads x
    head dim x bytes per element."""
    return 2 * n_l * n_kv * d_h * b


def cache_bytes(n_l, n_kv, d_h, b, B, L):
    """Whole-cache bytes for B sequences of length L."""
    return bytes_per_token(n_l, n_kv, d_h, b) * B * L


def paged_waste_slots(lengths, block_size):
    """Unused slots in each sequence's final block when every sequence holds
    ceil(L / block_size) whole blocks."""
    lengths = np.asarray(lengths, dtype=np.int64)
    blocks = (lengths + block_size - 1) // block_size
    return blocks * block_size - lengths
