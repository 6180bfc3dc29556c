"""Seeded synthetic inputs, identical on the host and on the GPU.

Every element is drawn by a counter-based generator: SplitMix64 (Steele,
Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA
2014). The i-th draw of a stream with 64-bit key ``key`` is
``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` where ``mix`` is the SplitMix64
finaliser. The top bits of a draw index a small table of values that the
host builds once (for N(0,1): the bf16-rounded inverse normal CDF at
65,536 evenly spaced probabilities). The GPU fill kernel (libkvd_inputs.so,
csrc/inputs_fill.cu) implements the same draw, so a multi-gigabyte cache can
be filled on the device and any part of it regenerated on the host,
byte for byte.

This module holds no part of the decode arithmetic. Both the CUDA path and
the oracle take its arrays as plain inputs.
"""
import statistics

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1


def _mix_int(z):
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed, *labels):
    """64-bit key of the stream named by (seed, labels...)."""
    k = _mix_int(int(seed) + GAMMA)
    for lab in labels:
        k = _mix_int(k + (int(lab) + 1) * GAMMA)
    return k


def draws(key, idx):
    """SplitMix64 draw number ``idx`` (uint64 array) of stream ``key``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


# ---------------------------------------------------------------------------
# value tables (indexed by the top bits of a draw)
# ---------------------------------------------------------------------------
_TABLES = {}


def normal_bf16_table():
    """65,536 bf16 bit patterns: N(0,1) quantiles at (j + 0.5) / 65536."""
    if "normal" not in _TABLES:
        import torch
        nd = statistics.NormalDist()
        vals = [nd.inv_cdf((j + 0.5) / 65536.0) for j in range(65536)]
        t = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)
        _TABLES["normal"] = t.view(torch.int16).numpy().view(np.uint16).copy()
    return _TABLES["normal"]


def eighths_bf16_table():
    """16 bf16 bit patterns: a/8 for a = -7..8 (exact in bf16). Products and
    sums of these stay exact in fp32 for the indexer's dot products."""
    if "eighths" not in _TABLES:
        import torch
        vals = [a / 8.0 for a in range(-7, 9)]
        t = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)
        _TABLES["eighths"] = t.view(torch.int16).numpy().view(np.uint16).copy()
    return _TABLES["eighths"]


def fp8_code_table():
    """256 E4M3 codes with random sign, exponent field 4..11 and any
    mantissa: magnitudes 1/8 .. 30, never NaN or zero."""
    if "fp8" not in _TABLES:
        j = np.arange(256, dtype=np.uint32)
        codes = (j & 0x80) | ((4 + ((j >> 3) & 7)) << 3) | (j & 7)
        _TABLES["fp8"] = codes.astype(np.uint8)
    return _TABLES["fp8"]


def byte_table():
    """The 256 byte values: uniform random bytes (the code bytes of an
    MXFP4 row, two random E2M1 codes each)."""
    if "byte" not in _TABLES:
        _TABLES["byte"] = np.arange(256, dtype=np.uint8)
    return _TABLES["byte"]


def mxfp4_scale_table():
    """256 E4M3 codes of the 16 values 1/8 .. 15/32 (exponent field 4 or
    5, any mantissa), each 16 times: positive group scales where amax / 6
    of 16 N(0,1) values falls for about 92 % of groups (median 0.34)."""
    if "mxscale" not in _TABLES:
        j = np.arange(256, dtype=np.uint32)
        codes = ((4 + ((j >> 3) & 1)) << 3) | (j & 7)
        _TABLES["mxscale"] = codes.astype(np.uint8)
    return _TABLES["mxscale"]


def table_bits(table):
    n = int(table.shape[0])
    bits = n.bit_length() - 1
    assert (1 << bits) == n, "table length must be a power of two"
    return bits


def host_fill(table, key, idx):
    """Host values of draws ``idx`` of stream ``key`` looked up in ``table``."""
    bits = table_bits(table)
    sel = draws(key, idx) >> np.uint64(64 - bits)
    return table[sel.astype(np.int64)]


def host_tensor(table, key, shape, offset=0):
    n = int(np.prod(shape)) if len(shape) else 1
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    return host_fill(table, key, idx).reshape(shape)


# ---------------------------------------------------------------------------
# scalar-per-element helpers
# ---------------------------------------------------------------------------
def uniform01_f32(key, n):
    """n float32 values in [0, 1): the top 24 bits of each draw / 2^24."""
    d = draws(key, np.arange(n, dtype=np.uint64)) >> np.uint64(40)
    return (d.astype(np.float64) / float(1 << 24)).astype(np.float32)


def uniform_int(key, n, lo, hi):
    """n integers in [lo, hi] (inclusive): lo + draw mod (hi - lo + 1)."""
    d = draws(key, np.arange(n, dtype=np.uint64))
    return (lo + (d % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


def permutation(key, n):
    """A seeded permutation of range(n): positions sorted by their draw."""
    d = draws(key, np.arange(n, dtype=np.uint64))
    return np.argsort(d, kind="stable").astype(np.int64)


# ---------------------------------------------------------------------------
# device side
# ---------------------------------------------------------------------------
def device_fill(tensor, table, key, offset=0, stream=None):
    """Fill a contiguous CUDA tensor (2-byte or 1-byte elements) with draws
    ``offset .. offset + numel`` of stream ``key`` looked up in ``table``,
    on the GPU, with the same bytes host_fill() gives."""
    import torch
    from ._native import inputs_lib
    lib = inputs_lib()
    assert tensor.is_cuda and tensor.is_contiguous()
    esize = tensor.element_size()
    assert esize == table.dtype.itemsize, "table / tensor element size differ"
    dev_table = torch.from_numpy(table.view(np.uint8).copy()).to(tensor.device)
    if stream is None:
        stream = torch.cuda.current_stream(tensor.device).cuda_stream
    rc = lib.kvdi_fill_table(tensor.data_ptr(), tensor.numel(), esize,
                             key, offset, dev_table.data_ptr(),
                             table_bits(table), stream)
    if rc != 0:
        raise RuntimeError(f"kvdi_fill_table failed with code {rc}")
    # keep the table alive until the fill has run
    torch.cuda.current_stream(tensor.device).synchronize()
    return tensor
