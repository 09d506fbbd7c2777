"""ctypes binding of libgk.so: the C ABI of include/gk.h under the same names.

Argument marshalling only.  Device buffers are passed as torch CUDA tensors (or
raw integer addresses); every computation runs in the library's kernels.  A
missing or unloadable library raises at import of the first call, never falls
back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# GK_LIB_PATH selects another build of the same library (the sanitizer build in the tests)
LIB_PATH = os.environ.get("GK_LIB_PATH") or os.path.join(_HERE, "libgk.so")

GK_OK = 0
GK_ERR_INVALID = 1
GK_ERR_OOM = 2
GK_ERR_HOT_FULL = 3
GK_ERR_CUDA = 4
GK_ERR_DEVICE_BOUNDS = 5
GK_ERR_TIMEOUT = 6
GK_ERR_UNSUPPORTED = 7
GK_BACKEND_DENSE = 0
GK_BACKEND_CASCADE = 1

c_i32, c_i64, c_u64, c_dbl, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p


class GkError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"gk status {status}: {message}")
        self.status = status


class gk_pool_config(ctypes.Structure):
    _fields_ = [("num_layers", c_i32), ("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
                ("hot_tokens", c_i64), ("cold_slots", c_i64), ("cold_page_size", c_i32), ("reserved0", c_i32),
                ("seed", c_u64), ("hot_k", c_vp), ("hot_v", c_vp), ("cold_k", c_vp), ("cold_v", c_vp)]


class gk_batch(ctypes.Structure):
    _fields_ = [("num_requests", c_i32), ("max_blocks", c_i32),
                ("prefix_hot_base", ctypes.POINTER(c_i64)), ("prefix_len", ctypes.POINTER(c_i32)),
                ("suffix_len", ctypes.POINTER(c_i32)), ("d_block_table", c_vp), ("d_q", c_vp),
                ("d_out", c_vp), ("d_lse", c_vp), ("d_new_k", c_vp), ("d_new_v", c_vp)]


class gk_plan_summary(ctypes.Structure):
    _fields_ = [("num_requests", c_i32), ("num_groups", c_i32), ("max_m_eff", c_i32), ("prefix_ctas", c_i32),
                ("suffix_ctas", c_i32), ("dense_ctas", c_i32), ("num_partials", c_i32), ("dense_merge", c_i32),
                ("prefix_bytes", c_i64), ("prefix_flops", c_i64), ("suffix_bytes", c_i64), ("dense_bytes", c_i64),
                ("cascade_split", c_i32), ("prefix_tiles_per_item", c_i32), ("prefix_kernel", c_i32),
                ("prefix_rows_per_item", c_i32), ("prefix_row_groups", c_i32), ("prefix_ctas_gather", c_i32),
                ("sm_slots", c_i32)]


class gk_cost_model(ctypes.Structure):
    _fields_ = [("c_flat_us", c_dbl), ("bw_flat_gbs", c_dbl), ("c_cascade_us", c_dbl), ("bw_prefix_gbs", c_dbl),
                ("bw_suffix_gbs", c_dbl), ("c_merge_us", c_dbl), ("prefix_tile_us", c_dbl), ("prefix_item_us", c_dbl),
                ("gather_sm_gbs", c_dbl), ("c_gather_us", c_dbl), ("prefix_tile_split_us", c_dbl),
                ("warp_tile_us", c_dbl), ("warp_group_us", c_dbl), ("warp_item_us", c_dbl),
                ("warp_split_ratio", c_dbl), ("prefix_cta_ramp_us", c_dbl), ("prefix_cta_gather_ratio", c_dbl),
                ("c_merge_state_us", c_dbl), ("prefix_item_split_us", c_dbl), ("warp_item_split_us", c_dbl),
                ("prefix_item_crowd_us", c_dbl), ("split_gather_ratio_tensor", c_dbl), ("c_gather_split_us", c_dbl),
                ("split_tensor_us", c_dbl)]


P = ctypes.POINTER
_SIGS = {
    "gk_pool_create": (c_i32, [P(gk_pool_config), P(c_vp)]),
    "gk_pool_destroy": (None, [c_vp]),
    "gk_last_error": (ctypes.c_char_p, [c_vp]),
    "gk_status_string": (ctypes.c_char_p, [c_i32]),
    "gk_prefix_alloc": (c_i32, [c_vp, c_i64, P(c_i64)]),
    "gk_prefix_release": (c_i32, [c_vp, c_i64]),
    "gk_hot_stats": (c_i32, [c_vp, P(c_i64), P(c_i64), P(c_i64)]),
    "gk_prefix_acquire": (c_i32, [c_vp, c_u64, c_i64, P(c_i64), P(c_i32)]),
    "gk_prefix_unref": (c_i32, [c_vp, c_u64]),
    "gk_hot_cache_stats": (c_i32, [c_vp, P(c_i64), P(c_i64), P(c_i64)]),
    "gk_seq_create_cached": (c_i32, [c_vp, c_i32, c_vp, P(c_i32), P(c_i64)]),
    "gk_seq_cache_blocks": (c_i32, [c_vp, c_i32, c_i32, c_vp, P(c_i32)]),
    "gk_cold_cache_stats": (c_i32, [c_vp, P(c_i64), P(c_i64)]),
    "gk_seq_create": (c_i32, [c_vp, P(c_i32)]),
    "gk_seq_fork": (c_i32, [c_vp, c_i32, P(c_i32)]),
    "gk_seq_release": (c_i32, [c_vp, c_i32]),
    "gk_seq_table": (c_i32, [c_vp, c_i32, P(P(c_i32)), P(c_i32), P(c_i64)]),
    "gk_seq_append_slots": (c_i32, [c_vp, c_i32, P(c_i32), P(c_i64), P(c_i32), P(c_i32), P(c_i32)]),
    "gk_seq_tables": (c_i32, [c_vp, c_i32, P(c_i32), c_i32, P(c_i32), P(c_i32)]),
    "gk_cold_stats": (c_i32, [c_vp, P(c_i64), P(c_i64)]),
    "gk_block_refcount": (c_i32, [c_vp, c_i32, P(c_i32)]),
    "gk_append_kv": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_vp]),
    "gk_write_prefix_kv": (c_i32, [c_vp, c_vp, c_i32, c_i64, c_i64, c_i64, c_i64, c_vp, c_vp]),
    "gk_plan_build": (c_i32, [c_vp, P(gk_batch), c_vp, P(c_vp)]),
    "gk_plan_update": (c_i32, [c_vp, P(gk_batch), c_vp]),
    "gk_plan_destroy": (None, [c_vp]),
    "gk_plan_info": (c_i32, [c_vp, P(gk_plan_summary)]),
    "gk_plan_segments": (c_i32, [c_vp, c_i32, P(c_i32), P(c_i32), c_vp, c_vp]),
    "gk_decode_dense": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_decode_cascade": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_decode_dense_static": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch)]),
    "gk_cascade_levels": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_cascade_prefix": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_cascade_suffix": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_cascade_merge": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp]),
    "gk_dispatch": (c_i32, [c_vp, c_vp, P(c_i32), P(c_dbl), P(c_dbl)]),
    "gk_cost_model_set": (c_i32, [c_vp, P(gk_cost_model)]),
    "gk_cost_model_get": (c_i32, [c_vp, P(gk_cost_model)]),
    "gk_cost_model_load": (c_i32, [c_vp, ctypes.c_char_p]),
    "gk_pool_set_cascade_mode": (c_i32, [c_vp, c_i32, c_i32]),
    "gk_pool_set_gather_partition": (c_i32, [c_vp, c_i32]),
    "gk_pool_set_prefix_kernel": (c_i32, [c_vp, c_i32]),
    "gk_pool_set_sm_speeds": (c_i32, [c_vp, P(ctypes.c_float), c_i32]),
    "gk_pool_get_sm_speeds": (c_i32, [c_vp, P(ctypes.c_float), P(c_i32)]),
    "gk_sm_speeds_measure": (c_i32, [c_vp, c_vp, c_i32, P(gk_batch), c_vp, c_i32, P(ctypes.c_float)]),
    "gk_calibrate": (c_i32, [c_vp, c_vp, ctypes.c_char_p]),
    "gk_device_error": (c_i32, [c_vp, c_vp, P(c_i32)]),
}

_lib = None


def lib():
    """The loaded libgk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() (or python paged_kv_cache_pool_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    """Device address of a torch tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st, pool=None):
    if st != GK_OK:
        msg = lib().gk_last_error(pool).decode() if pool else ""
        if not msg:
            msg = lib().gk_status_string(st).decode()
        raise GkError(st, msg)


def _i64p(a):
    return a.ctypes.data_as(P(c_i64))


def _i32p(a):
    return a.ctypes.data_as(P(c_i32))


# ---- pool ----------------------------------------------------------------------
def gk_pool_create(num_layers, num_q_heads, num_kv_heads, head_dim, hot_tokens, cold_slots, cold_page_size,
                   seed=0, hot_k=None, hot_v=None, cold_k=None, cold_v=None):
    cfg = gk_pool_config(num_layers, num_q_heads, num_kv_heads, head_dim, hot_tokens, cold_slots, cold_page_size, 0,
                         seed, _ptr(hot_k), _ptr(hot_v), _ptr(cold_k), _ptr(cold_v))
    out = c_vp()
    _check(lib().gk_pool_create(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def gk_pool_destroy(pool):
    lib().gk_pool_destroy(pool)


def gk_last_error(pool):
    return lib().gk_last_error(pool).decode()


def gk_status_string(status):
    return lib().gk_status_string(status).decode()


# ---- HOT pool --------------------------------------------------------------------
def gk_prefix_alloc(pool, prefix_len):
    base = c_i64()
    _check(lib().gk_prefix_alloc(pool, prefix_len, ctypes.byref(base)), pool)
    return base.value


def gk_prefix_release(pool, hot_base):
    _check(lib().gk_prefix_release(pool, hot_base), pool)


def gk_hot_stats(pool):
    a, b, c = c_i64(), c_i64(), c_i64()
    _check(lib().gk_hot_stats(pool, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), pool)
    return a.value, b.value, c.value


def gk_prefix_acquire(pool, key, prefix_len):
    """-> (hot_base, hit): a reference on the cached slab of key, allocated (evicting idle slabs) on a miss."""
    base, hit = c_i64(), c_i32()
    _check(lib().gk_prefix_acquire(pool, int(key) & ((1 << 64) - 1), int(prefix_len), ctypes.byref(base),
                                   ctypes.byref(hit)), pool)
    return base.value, bool(hit.value)


def gk_prefix_unref(pool, key):
    _check(lib().gk_prefix_unref(pool, int(key) & ((1 << 64) - 1)), pool)


def gk_hot_cache_stats(pool):
    """-> (cached slabs, idle slabs, tokens held by idle slabs)."""
    a, b, c = c_i64(), c_i64(), c_i64()
    _check(lib().gk_hot_cache_stats(pool, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), pool)
    return a.value, b.value, c.value


# ---- COLD block manager ----------------------------------------------------------
def gk_seq_create(pool):
    s = c_i32()
    _check(lib().gk_seq_create(pool, ctypes.byref(s)), pool)
    return s.value


def gk_seq_fork(pool, parent):
    s = c_i32()
    _check(lib().gk_seq_fork(pool, parent, ctypes.byref(s)), pool)
    return s.value


def gk_seq_release(pool, seq):
    _check(lib().gk_seq_release(pool, seq), pool)


def gk_seq_table(pool, seq):
    """-> (block table as a numpy int32 copy, length in tokens)."""
    t = P(c_i32)()
    nb, ln = c_i32(), c_i64()
    _check(lib().gk_seq_table(pool, seq, ctypes.byref(t), ctypes.byref(nb), ctypes.byref(ln)), pool)
    arr = np.ctypeslib.as_array(t, shape=(nb.value,)).copy() if nb.value else np.zeros(0, np.int32)
    return arr, ln.value


def gk_seq_append_slots(pool, seqs):
    """-> (slot_mapping int64 [n], cow_pairs int32 [n_cow, 2]).  Raises GkError(GK_ERR_OOM) with .n_done set."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int32)
    n = len(seqs)
    slots = np.empty(n, dtype=np.int64)
    cow = np.empty(2 * max(n, 1), dtype=np.int32)
    ncow, ndone = c_i32(), c_i32()
    st = lib().gk_seq_append_slots(pool, n, _i32p(seqs), _i64p(slots), ctypes.byref(ncow), _i32p(cow),
                                   ctypes.byref(ndone))
    if st != GK_OK:
        err = GkError(st, gk_last_error(pool))
        err.n_done = ndone.value
        err.slots = slots[:ndone.value]
        err.cow_pairs = cow[:2 * ncow.value].reshape(-1, 2)
        raise err
    return slots, cow[:2 * ncow.value].reshape(-1, 2).copy()


def gk_seq_tables(pool, seqs, max_blocks, table_out=None, len_out=None):
    """Fill (or allocate) int32 [n, max_blocks] tables and int32 [n] lengths; returns both."""
    seqs = np.ascontiguousarray(seqs, dtype=np.int32)
    n = len(seqs)
    if table_out is None:
        table_out = np.empty((n, max_blocks), dtype=np.int32)
    if len_out is None:
        len_out = np.empty(n, dtype=np.int32)
    assert table_out.dtype == np.int32 and table_out.flags.c_contiguous and table_out.size >= n * max_blocks
    _check(lib().gk_seq_tables(pool, n, _i32p(seqs), max_blocks, _i32p(table_out), _i32p(len_out)), pool)
    return table_out, len_out


def gk_seq_create_cached(pool, tokens):
    """-> (seq, n_cached): a new sequence starting with the longest cached chain of tokens' full blocks."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    s, n = c_i32(), c_i64()
    _check(lib().gk_seq_create_cached(pool, len(t), t.ctypes.data_as(c_vp), ctypes.byref(s), ctypes.byref(n)), pool)
    return s.value, n.value


def gk_seq_cache_blocks(pool, seq, tokens):
    """Cache seq's full blocks covering tokens; -> blocks newly cached."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    n = c_i32()
    _check(lib().gk_seq_cache_blocks(pool, int(seq), len(t), t.ctypes.data_as(c_vp), ctypes.byref(n)), pool)
    return n.value


def gk_cold_cache_stats(pool):
    """-> (cached blocks, evictable blocks)."""
    a, b = c_i64(), c_i64()
    _check(lib().gk_cold_cache_stats(pool, ctypes.byref(a), ctypes.byref(b)), pool)
    return a.value, b.value


def gk_cold_stats(pool):
    a, b = c_i64(), c_i64()
    _check(lib().gk_cold_stats(pool, ctypes.byref(a), ctypes.byref(b)), pool)
    return a.value, b.value


def gk_block_refcount(pool, block):
    r = c_i32()
    _check(lib().gk_block_refcount(pool, block, ctypes.byref(r)), pool)
    return r.value


# ---- device work -------------------------------------------------------------------
def gk_append_kv(pool, stream, layer, d_slot_mapping, d_k, d_v, d_cow_pairs=None, n=None, n_cow=None):
    n = d_slot_mapping.numel() if n is None else n
    n_cow = (0 if d_cow_pairs is None else d_cow_pairs.numel() // 2) if n_cow is None else n_cow
    _check(lib().gk_append_kv(pool, _stream(stream), layer, n, _ptr(d_slot_mapping), _ptr(d_k), _ptr(d_v), n_cow,
                              _ptr(d_cow_pairs) if n_cow else None), pool)


def gk_write_prefix_kv(pool, stream, layer, hot_base, prefix_len, t0, d_k, d_v, n=None):
    n = d_k.shape[0] if n is None else n
    _check(lib().gk_write_prefix_kv(pool, _stream(stream), layer, hot_base, prefix_len, t0, n, _ptr(d_k), _ptr(d_v)),
           pool)


class Batch:
    """Keeps the host arrays of a gk_batch alive; .set_layer() swaps the per-layer device pointers."""

    def __init__(self, prefix_hot_base, prefix_len, suffix_len, d_block_table=None, max_blocks=0, d_q=None,
                 d_out=None, d_lse=None):
        self.prefix_hot_base = np.ascontiguousarray(prefix_hot_base, dtype=np.int64)
        self.prefix_len = np.ascontiguousarray(prefix_len, dtype=np.int32)
        self.suffix_len = np.ascontiguousarray(suffix_len, dtype=np.int32)
        self.c = gk_batch(len(self.prefix_len), max_blocks, _i64p(self.prefix_hot_base), _i32p(self.prefix_len),
                          _i32p(self.suffix_len), _ptr(d_block_table), _ptr(d_q), _ptr(d_out), _ptr(d_lse), None, None)

    def set_device(self, d_block_table=None, max_blocks=None, d_q=None, d_out=None, d_lse=None, d_new_k=None,
                   d_new_v=None):
        """d_lse, d_new_k and d_new_v are set on every call (None clears them: no LSE
        output, no fused append); the others keep their value when None."""
        if d_block_table is not None:
            self.c.d_block_table = _ptr(d_block_table)
        if max_blocks is not None:
            self.c.max_blocks = max_blocks
        if d_q is not None:
            self.c.d_q = _ptr(d_q)
        if d_out is not None:
            self.c.d_out = _ptr(d_out)
        self.c.d_lse = _ptr(d_lse)
        self.c.d_new_k = _ptr(d_new_k)
        self.c.d_new_v = _ptr(d_new_v)
        return self


def gk_plan_build(pool, batch, stream=None):
    out = c_vp()
    _check(lib().gk_plan_build(pool, ctypes.byref(batch.c), _stream(stream), ctypes.byref(out)), pool)
    return out.value


def gk_plan_update(pool, plan, batch, stream=None):
    _check(lib().gk_plan_update(plan, ctypes.byref(batch.c), _stream(stream)), pool)


def gk_plan_destroy(plan):
    lib().gk_plan_destroy(plan)


def gk_plan_info(plan):
    s = gk_plan_summary()
    _check(lib().gk_plan_info(plan, ctypes.byref(s)))
    return {name: getattr(s, name) for name, _ in gk_plan_summary._fields_}


def gk_plan_segments(plan, dense=False):
    """(begin [n_ctas + 1], segs [n_segs, 4] = request, t0, t1, entry): the plan's gather partition."""
    n_ctas, n_segs = c_i32(), c_i32()
    _check(lib().gk_plan_segments(plan, int(bool(dense)), ctypes.byref(n_ctas), ctypes.byref(n_segs), None, None))
    begin = np.zeros(n_ctas.value + 1, dtype=np.int32)
    segs = np.zeros((n_segs.value, 4), dtype=np.int32)
    _check(lib().gk_plan_segments(plan, int(bool(dense)), ctypes.byref(n_ctas), ctypes.byref(n_segs),
                                  begin.ctypes.data_as(c_vp), segs.ctypes.data_as(c_vp)))
    return begin, segs


def gk_decode_dense(pool, stream, layer, batch, plan):
    _check(lib().gk_decode_dense(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_decode_cascade(pool, stream, layer, batch, plan):
    _check(lib().gk_decode_cascade(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_decode_dense_static(pool, stream, layer, batch):
    _check(lib().gk_decode_dense_static(pool, _stream(stream), layer, ctypes.byref(batch.c)), pool)


def gk_cascade_levels(pool, stream, layer, batch, plan):
    _check(lib().gk_cascade_levels(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_cascade_prefix(pool, stream, layer, batch, plan):
    _check(lib().gk_cascade_prefix(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_cascade_suffix(pool, stream, layer, batch, plan):
    _check(lib().gk_cascade_suffix(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_cascade_merge(pool, stream, layer, batch, plan):
    _check(lib().gk_cascade_merge(pool, _stream(stream), layer, ctypes.byref(batch.c), plan), pool)


def gk_dispatch(pool, plan):
    """-> (GK_BACKEND_*, predicted dense us, predicted cascade us)."""
    ch, td, tc = c_i32(), c_dbl(), c_dbl()
    _check(lib().gk_dispatch(pool, plan, ctypes.byref(ch), ctypes.byref(td), ctypes.byref(tc)), pool)
    return ch.value, td.value, tc.value


def gk_cost_model_get(pool):
    cm = gk_cost_model()
    _check(lib().gk_cost_model_get(pool, ctypes.byref(cm)), pool)
    return {k: getattr(cm, k) for k in COST_MODEL_KEYS}


COST_MODEL_KEYS = ("c_flat_us", "bw_flat_gbs", "c_cascade_us", "bw_prefix_gbs", "bw_suffix_gbs", "c_merge_us",
                   "prefix_tile_us", "prefix_item_us", "gather_sm_gbs", "c_gather_us", "prefix_tile_split_us",
                   "warp_tile_us", "warp_group_us", "warp_item_us", "warp_split_ratio", "prefix_cta_ramp_us",
                   "prefix_cta_gather_ratio", "c_merge_state_us", "prefix_item_split_us", "warp_item_split_us",
                   "prefix_item_crowd_us", "split_gather_ratio_tensor", "c_gather_split_us",
                   "split_tensor_us")


def gk_cost_model_set(pool, cm: dict):
    c = gk_cost_model()
    for k in COST_MODEL_KEYS:
        setattr(c, k, float(cm[k]))
    _check(lib().gk_cost_model_set(pool, ctypes.byref(c)), pool)


GK_CASCADE_AUTO, GK_CASCADE_SEQUENTIAL, GK_CASCADE_SPLIT = 0, 1, 2


def gk_pool_set_cascade_mode(pool, mode, tiles_per_item=0):
    _check(lib().gk_pool_set_cascade_mode(pool, int(mode), int(tiles_per_item)), pool)


GK_PARTITION_STREAM, GK_PARTITION_PER_REQUEST = 0, 1


def gk_pool_set_gather_partition(pool, partition):
    _check(lib().gk_pool_set_gather_partition(pool, int(partition)), pool)


GK_PREFIX_AUTO, GK_PREFIX_TENSOR, GK_PREFIX_WARP = 0, 1, 2


def gk_pool_set_prefix_kernel(pool, kernel):
    _check(lib().gk_pool_set_prefix_kernel(pool, int(kernel)), pool)


def gk_pool_set_sm_speeds(pool, speeds):
    """speeds: one per SM of the device, or None / empty to clear."""
    if speeds is None or len(speeds) == 0:
        _check(lib().gk_pool_set_sm_speeds(pool, None, 0), pool)
        return
    a = np.ascontiguousarray(speeds, dtype=np.float32)
    _check(lib().gk_pool_set_sm_speeds(pool, a.ctypes.data_as(P(ctypes.c_float)), len(a)), pool)


def gk_pool_get_sm_speeds(pool):
    n = c_i32()
    _check(lib().gk_pool_get_sm_speeds(pool, None, ctypes.byref(n)), pool)
    a = np.zeros(n.value, np.float32)
    if n.value:
        _check(lib().gk_pool_get_sm_speeds(pool, a.ctypes.data_as(P(ctypes.c_float)), ctypes.byref(n)), pool)
    return a


def gk_sm_speeds_measure(pool, stream, layer, batch, plan, reps=5):
    """-> the measured per-SM speeds (installed in the pool)."""
    n = c_i32()
    _check(lib().gk_pool_get_sm_speeds(pool, None, ctypes.byref(n)), pool)
    _check(lib().gk_sm_speeds_measure(pool, _stream(stream), layer, ctypes.byref(batch.c), plan, reps, None), pool)
    return gk_pool_get_sm_speeds(pool)


def gk_calibrate(pool, stream=None, json_out=None):
    _check(lib().gk_calibrate(pool, _stream(stream), json_out.encode() if json_out else None), pool)


def gk_cost_model_load(pool, json_text: str):
    _check(lib().gk_cost_model_load(pool, json_text.encode()), pool)


def gk_device_error(pool, stream=None):
    code = c_i32()
    _check(lib().gk_device_error(pool, _stream(stream), ctypes.byref(code)), pool)
    return code.value
