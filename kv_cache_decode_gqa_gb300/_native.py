"""ctypes view of libkvd.so (include/kvd.h) and libkvd_inputs.so.

The libraries are built in-tree by build.py (``__graft_entry__.build()``).
Loading fails loudly if they are missing: there is no other implementation
of these calls.
"""
import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libkvd.so")
INPUTS_LIB_PATH = os.path.join(PKG, "libkvd_inputs.so")
HEADER = os.path.join(ROOT, "include", "kvd.h")

c_void_p = ctypes.c_void_p
c_int32 = ctypes.c_int32
c_size_t = ctypes.c_size_t
c_float = ctypes.c_float


class KvdCache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p),
                ("num_blocks", c_int32), ("block_size", c_int32),
                ("n_kv", c_int32), ("head_dim", c_int32),
                ("dtype", c_int32), ("reserved", c_int32),
                ("k_scale", c_void_p), ("v_scale", c_void_p),
                ("k_inv_scale", c_void_p), ("v_inv_scale", c_void_p)]


class KvdSeqs(ctypes.Structure):
    _fields_ = [("block_table", c_void_p), ("seq_lens", c_void_p),
                ("batch", c_int32), ("max_blocks_per_seq", c_int32),
                ("max_seq_len", c_int32), ("flags", c_int32),
                ("window", c_int32), ("window_start", c_void_p)]


STATUS = {0: "KVD_OK", 1: "KVD_ERR_NULL", 2: "KVD_ERR_SHAPE",
          3: "KVD_ERR_UNSUPPORTED", 4: "KVD_ERR_CAPACITY",
          5: "KVD_ERR_WORKSPACE", 6: "KVD_ERR_CUDA"}

_PCACHE = ctypes.POINTER(KvdCache)
_PSEQS = ctypes.POINTER(KvdSeqs)

_SIGS = {
    "kvd_version": (c_int32, []),
    "kvd_launch_count": (ctypes.c_uint64, []),
    "kvd_set_tuning": (c_int32, [c_int32, c_int32]),
    "kvd_last_error": (ctypes.c_char_p, []),
    "kvd_status_string": (ctypes.c_char_p, [c_int32]),
    "kvd_bytes_per_token": (ctypes.c_uint64, [c_int32] * 4),
    "kvd_device_error": (c_int32, [ctypes.POINTER(c_int32)]),
    "kvd_kv_append": (c_int32, [_PCACHE, c_void_p, c_int32, c_void_p, c_int32,
                                c_void_p, c_void_p, c_void_p]),
    "kvd_gqa_decode": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_int32, c_float,
                                 c_void_p, c_void_p, c_void_p, c_size_t,
                                 c_void_p]),
    "kvd_gqa_append_decode": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_int32, c_float,
                                        c_void_p, c_void_p, c_void_p,
                                        c_size_t, c_void_p]),
    "kvd_gqa_decode_noalloc": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_int32,
                                         c_float, c_void_p, c_void_p,
                                         c_void_p]),
    "kvd_mla_decode": (c_int32, [_PCACHE, c_int32, _PSEQS, c_void_p, c_int32,
                                 c_float, c_void_p, c_void_p, c_void_p,
                                 c_size_t, c_void_p]),
    "kvd_indexer_topk": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_int32,
                                   c_void_p, c_int32, c_void_p, c_void_p,
                                   c_void_p, c_size_t, c_void_p]),
    "kvd_indexer_pool": (c_int32, [_PSEQS, c_void_p, c_int32, c_void_p,
                                   c_void_p, c_void_p]),
    "kvd_indexer_topk_pool": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_int32,
                                        c_void_p, c_void_p, c_void_p, c_int32,
                                        c_void_p, c_void_p, c_void_p,
                                        c_size_t, c_void_p]),
    "kvd_sparse_decode": (c_int32, [_PCACHE, _PSEQS, c_void_p, c_int32,
                                    c_void_p, c_int32, c_float, c_void_p,
                                    c_void_p, c_void_p, c_size_t, c_void_p]),
    "kvd_block_pool_create": (c_int32, [c_int32, ctypes.POINTER(c_void_p)]),
    "kvd_block_pool_destroy": (None, [c_void_p]),
    "kvd_block_pool_free_count": (c_int32, [c_void_p]),
    "kvd_block_pool_refcount": (c_int32, [c_void_p, c_int32]),
    "kvd_block_pool_alloc": (c_int32, [c_void_p, c_int32, c_void_p]),
    "kvd_block_pool_share": (c_int32, [c_void_p, c_void_p, c_int32]),
    "kvd_block_pool_release": (c_int32, [c_void_p, c_void_p, c_int32]),
    "kvd_block_pool_prepare_append": (c_int32, [c_void_p, c_void_p, c_int32,
                                                c_int32, c_void_p, c_int32,
                                                c_void_p, c_void_p,
                                                ctypes.POINTER(c_int32)]),
    "kvd_copy_blocks": (c_int32, [_PCACHE, c_void_p, c_void_p, c_int32,
                                  c_void_p]),
    "kvd_workspace_size": (c_int32, [c_int32, _PCACHE, _PSEQS, c_int32,
                                     c_int32, ctypes.POINTER(c_size_t)]),
}

_lock = threading.Lock()
_lib = None
_inputs_lib = None


class KvdError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{name}: {message}")


def lib():
    """The loaded libkvd.so with argument types set."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def inputs_lib():
    global _inputs_lib
    with _lock:
        if _inputs_lib is None:
            if not os.path.exists(INPUTS_LIB_PATH):
                raise RuntimeError(f"{INPUTS_LIB_PATH} is not built")
            L = ctypes.CDLL(INPUTS_LIB_PATH)
            L.kvdi_fill_table.restype = c_int32
            L.kvdi_fill_table.argtypes = [c_void_p, ctypes.c_uint64, c_int32,
                                          ctypes.c_uint64, ctypes.c_uint64,
                                          c_void_p, c_int32, c_void_p]
            _inputs_lib = L
    return _inputs_lib


def check(status):
    if status != 0:
        msg = lib().kvd_last_error().decode(errors="replace")
        raise KvdError(status, msg)


def header_functions():
    """Names of the functions include/kvd.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvd_[a-z_0-9]+)\s*\(", text)))
