"""Python binding of libpie_attn.so (ctypes): the C ABI of pie_attn.h under the
same names, argument marshalling only.  Every step of the attention path runs
in the library's CUDA kernels; there is no other implementation behind these
calls, and importing this module fails loudly when the library is missing.

Out-parameters become return values and a negative status raises PieError.
Device pointers may be given as torch tensors (their data_ptr()) or ints.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpie_attn.so")

PIE_OK = 0
PIE_ERR_INVALID = -1
PIE_ERR_BAD_HANDLE = -2
PIE_ERR_NO_PAGES = -3
PIE_ERR_RANGE = -4
PIE_ERR_CUDA = -5
PIE_ERR_STATE = -6
PIE_KV_BF16 = 0
PIE_KV_E4M3 = 1

EXPORTS = [
    "pie_ctx_create", "pie_ctx_destroy", "pie_last_error", "pie_ws_create", "pie_ws_destroy",
    "pie_ws_fork", "pie_ws_freeze", "pie_ws_rollback", "pie_ws_match_prefix", "pie_ws_info",
    "pie_ws_page_table", "pie_page_refcount", "pie_free_pages", "pie_batch_begin", "pie_batch_rows",
    "pie_batch_slots", "pie_kv_append", "pie_attend", "pie_batch_end", "pie_batch_plan_info",
    "pie_batch_items", "pie_ctx_check", "pie_attend_decode_noalloc", "pie_selftest_wait_timeout",
    "pie_kv_append_rope", "pie_rope_table", "pie_selftest_fail_next_begin", "pie_ctx_set_merge_mode",
]
PIE_NOALLOC_SCRATCH_BYTES = 16 << 20


class PieError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class pie_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("free_list", ctypes.POINTER(ctypes.c_int32)),
        ("k_scale", ctypes.POINTER(ctypes.c_float)), ("v_scale", ctypes.POINTER(ctypes.c_float)),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("stream", ctypes.c_void_p),
        ("logit_softcap", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("rope_max_positions", ctypes.c_int32),
    ]


class pie_decode_args(ctypes.Structure):
    _fields_ = [
        ("num_rows", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("num_layers", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("layer", ctypes.c_int32), ("max_pages_per_row", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("stream", ctypes.c_void_p),
    ]


class pie_seg(ctypes.Structure):
    _fields_ = [("ws", ctypes.c_int32), ("n_new", ctypes.c_int32), ("token_ids", ctypes.POINTER(ctypes.c_int32))]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with paged_kv_attention_working_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, V = ctypes.POINTER, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    sig = {
        "pie_ctx_create": [P(pie_config), P(V)],
        "pie_ctx_destroy": [V],
        "pie_ws_create": [V, P(I)],
        "pie_ws_destroy": [V, I],
        "pie_ws_fork": [V, I, P(I)],
        "pie_ws_freeze": [V, I, I],
        "pie_ws_rollback": [V, I, I],
        "pie_ws_match_prefix": [V, I, P(I), I, P(I)],
        "pie_ws_info": [V, I, P(I), P(I), P(I)],
        "pie_ws_page_table": [V, I, P(I), I, P(I)],
        "pie_page_refcount": [V, I, P(I)],
        "pie_free_pages": [V, P(I)],
        "pie_batch_begin": [V, P(pie_seg), I, P(V)],
        "pie_batch_rows": [V, P(I)],
        "pie_batch_slots": [V, P(I), P(I)],
        "pie_kv_append": [V, V, I, V, V],
        "pie_kv_append_rope": [V, V, I, V, V, V, V],
        "pie_rope_table": [F, I, I, P(F)],
        "pie_attend": [V, V, I, V, V, V],
        "pie_batch_end": [V, V],
        "pie_batch_plan_info": [V, P(I)],
        "pie_batch_items": [V, I, P(I), I, P(I)],
        "pie_ctx_check": [V, P(I)],
        "pie_attend_decode_noalloc": [P(pie_decode_args)],
        "pie_selftest_wait_timeout": [V, I],
        "pie_selftest_fail_next_begin": [V],
        "pie_ctx_set_merge_mode": [V, I],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int32
    lib.pie_last_error.argtypes = [V]
    lib.pie_last_error.restype = ctypes.c_char_p
    return lib


lib = _load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _i32_array(values):
    if values is None:
        return None
    vals = [int(v) for v in values]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def _check(ctx, st: int, what: str) -> None:
    if st != PIE_OK:
        msg = lib.pie_last_error(ctx).decode() if ctx else what
        raise PieError(st, f"{what}: {msg}")


# ------------------------------------------------------------------ context
def pie_ctx_create(num_layers, num_q_heads, num_kv_heads, head_dim, num_pages, kv_dtype=PIE_KV_BF16,
                   free_list=None, k_scale=None, v_scale=None, k_pool=None, v_pool=None, stream=None,
                   num_sms=0, page_size=16, logit_softcap=0.0, rope_theta=0.0, rope_max_positions=0):
    """Returns an opaque context handle (int).  k_pool/v_pool None = plan-only."""
    keep = []
    cfg = pie_config()
    cfg.num_layers, cfg.num_q_heads, cfg.num_kv_heads = num_layers, num_q_heads, num_kv_heads
    cfg.head_dim, cfg.page_size, cfg.kv_dtype = head_dim, page_size, kv_dtype
    cfg.num_pages, cfg.num_sms = num_pages, num_sms
    if free_list is not None:
        arr = _i32_array(free_list)
        keep.append(arr)
        cfg.free_list = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
    for field, vals in (("k_scale", k_scale), ("v_scale", v_scale)):
        if vals is not None:
            flat = [float(x) for x in __import__("numpy").asarray(vals, dtype="float32").reshape(-1)]
            arr = (ctypes.c_float * len(flat))(*flat)
            keep.append(arr)
            setattr(cfg, field, ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)))
    cfg.k_pool, cfg.v_pool = _ptr(k_pool), _ptr(v_pool)
    cfg.stream = _ptr(stream)
    cfg.logit_softcap = logit_softcap
    cfg.rope_theta, cfg.rope_max_positions = rope_theta, rope_max_positions
    out = ctypes.c_void_p()
    st = lib.pie_ctx_create(ctypes.byref(cfg), ctypes.byref(out))
    if st != PIE_OK:
        raise PieError(st, "pie_ctx_create: invalid configuration or CUDA failure")
    return out.value


def pie_ctx_destroy(ctx) -> None:
    _check(None, lib.pie_ctx_destroy(ctx), "pie_ctx_destroy")


def pie_last_error(ctx) -> str:
    return lib.pie_last_error(ctx).decode()


def pie_ctx_check(ctx) -> int:
    v = ctypes.c_int32()
    _check(ctx, lib.pie_ctx_check(ctx, ctypes.byref(v)), "pie_ctx_check")
    return v.value


def pie_ctx_set_merge_mode(ctx, mode) -> None:
    """0: split rows merged by a merge launch (the default); 1: inside the
    decode launches when no tensor-core item is split."""
    _check(ctx, lib.pie_ctx_set_merge_mode(ctx, mode), "pie_ctx_set_merge_mode")


def pie_selftest_wait_timeout(ctx, polls) -> None:
    _check(ctx, lib.pie_selftest_wait_timeout(ctx, polls), "pie_selftest_wait_timeout")


def pie_selftest_fail_next_begin(ctx) -> None:
    _check(ctx, lib.pie_selftest_fail_next_begin(ctx), "pie_selftest_fail_next_begin")


# ------------------------------------------------------------- working sets
def pie_ws_create(ctx) -> int:
    h = ctypes.c_int32()
    _check(ctx, lib.pie_ws_create(ctx, ctypes.byref(h)), "pie_ws_create")
    return h.value


def pie_ws_destroy(ctx, ws) -> None:
    _check(ctx, lib.pie_ws_destroy(ctx, ws), "pie_ws_destroy")


def pie_ws_fork(ctx, parent) -> int:
    h = ctypes.c_int32()
    _check(ctx, lib.pie_ws_fork(ctx, parent, ctypes.byref(h)), "pie_ws_fork")
    return h.value


def pie_ws_freeze(ctx, ws, n=-1) -> None:
    _check(ctx, lib.pie_ws_freeze(ctx, ws, n), "pie_ws_freeze")


def pie_ws_rollback(ctx, ws, n) -> None:
    _check(ctx, lib.pie_ws_rollback(ctx, ws, n), "pie_ws_rollback")


def pie_ws_match_prefix(ctx, ws, token_ids) -> int:
    toks = _i32_array(token_ids)
    n = ctypes.c_int32()
    _check(ctx, lib.pie_ws_match_prefix(ctx, ws, toks, len(token_ids), ctypes.byref(n)), "pie_ws_match_prefix")
    return n.value


def pie_ws_info(ctx, ws):
    a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(ctx, lib.pie_ws_info(ctx, ws, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "pie_ws_info")
    return a.value, b.value, c.value


def pie_ws_page_table(ctx, ws) -> list:
    n = ctypes.c_int32()
    _check(ctx, lib.pie_ws_page_table(ctx, ws, None, 0, ctypes.byref(n)), "pie_ws_page_table")
    buf = (ctypes.c_int32 * max(1, n.value))()
    _check(ctx, lib.pie_ws_page_table(ctx, ws, buf, n.value, ctypes.byref(n)), "pie_ws_page_table")
    return list(buf[: n.value])


def pie_page_refcount(ctx, page) -> int:
    v = ctypes.c_int32()
    _check(ctx, lib.pie_page_refcount(ctx, page, ctypes.byref(v)), "pie_page_refcount")
    return v.value


def pie_free_pages(ctx) -> int:
    v = ctypes.c_int32()
    _check(ctx, lib.pie_free_pages(ctx, ctypes.byref(v)), "pie_free_pages")
    return v.value


# -------------------------------------------------------------------- passes
def pie_batch_begin(ctx, segs):
    """segs: iterable of (ws, n_new, token_ids or None).  Returns a batch handle."""
    segs = list(segs)
    arr = (pie_seg * max(1, len(segs)))()
    keep = []
    for i, (ws, n_new, toks) in enumerate(segs):
        arr[i].ws, arr[i].n_new = ws, n_new
        if toks is not None:
            t = _i32_array(toks)
            keep.append(t)
            arr[i].token_ids = ctypes.cast(t, ctypes.POINTER(ctypes.c_int32))
    out = ctypes.c_void_p()
    _check(ctx, lib.pie_batch_begin(ctx, arr, len(segs), ctypes.byref(out)), "pie_batch_begin")
    return out.value


def pie_batch_rows(batch) -> int:
    v = ctypes.c_int32()
    _check(None, lib.pie_batch_rows(batch, ctypes.byref(v)), "pie_batch_rows")
    return v.value


def pie_batch_slots(batch):
    n = pie_batch_rows(batch)
    pos, slot = (ctypes.c_int32 * max(1, n))(), (ctypes.c_int32 * max(1, n))()
    _check(None, lib.pie_batch_slots(batch, pos, slot), "pie_batch_slots")
    return list(pos[:n]), list(slot[:n])


def pie_batch_plan_info(batch):
    info = (ctypes.c_int32 * 5)()
    _check(None, lib.pie_batch_plan_info(batch, info), "pie_batch_plan_info")
    return {"decode_items": info[0], "prefill_items": info[1], "merge_rows": info[2], "copies": info[3],
            "merge_launch": info[4]}


def pie_batch_items(batch, kind):
    n = ctypes.c_int32()
    _check(None, lib.pie_batch_items(batch, kind, None, 0, ctypes.byref(n)), "pie_batch_items")
    buf = (ctypes.c_int32 * max(1, 8 * n.value))()
    _check(None, lib.pie_batch_items(batch, kind, buf, n.value, ctypes.byref(n)), "pie_batch_items")
    keys = ("pages_off", "n_pages", "key_base", "rows_off", "n_rows", "part", "n_keys", "direct_rows")
    return [dict(zip(keys, buf[8 * i: 8 * i + 8])) for i in range(n.value)]


def pie_kv_append(ctx, batch, layer, k, v) -> None:
    _check(ctx, lib.pie_kv_append(ctx, batch, layer, _ptr(k), _ptr(v)), "pie_kv_append")


def pie_kv_append_rope(ctx, batch, layer, k, v, q=None, q_out=None) -> None:
    _check(ctx, lib.pie_kv_append_rope(ctx, batch, layer, _ptr(k), _ptr(v), _ptr(q), _ptr(q_out)),
           "pie_kv_append_rope")


def pie_rope_table(theta, head_dim, positions):
    """The library's rotary table as a float32 numpy array [positions, head_dim/2, 2]."""
    import numpy as np

    out = np.empty((positions, head_dim // 2, 2), dtype=np.float32)
    _check(None, lib.pie_rope_table(theta, head_dim, positions,
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), "pie_rope_table")
    return out


def pie_attend(ctx, batch, layer, q, out, lse=None) -> None:
    _check(ctx, lib.pie_attend(ctx, batch, layer, _ptr(q), _ptr(out), _ptr(lse)), "pie_attend")


def pie_batch_end(ctx, batch) -> None:
    _check(ctx, lib.pie_batch_end(ctx, batch), "pie_batch_end")


def pie_attend_decode_noalloc(num_rows, num_q_heads, num_kv_heads, head_dim, num_layers, num_pages, layer,
                              max_pages_per_row, q, k_pool, v_pool, block_table, seq_lens, out, lse=None,
                              stream=None) -> None:
    """Decode attention with no device allocation (scratch in a library-owned
    file-scope device array); see pie_attn.h."""
    a = pie_decode_args()
    a.num_rows, a.num_q_heads, a.num_kv_heads, a.head_dim = num_rows, num_q_heads, num_kv_heads, head_dim
    a.num_layers, a.num_pages, a.layer, a.max_pages_per_row = num_layers, num_pages, layer, max_pages_per_row
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.block_table, a.seq_lens = _ptr(block_table), _ptr(seq_lens)
    a.out, a.lse, a.stream = _ptr(out), _ptr(lse), _ptr(stream)
    _check(None, lib.pie_attend_decode_noalloc(ctypes.byref(a)), "pie_attend_decode_noalloc")
