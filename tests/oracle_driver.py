"""Runs a synthetic workload's operation script against the CPU oracle."""
from __future__ import annotations

import numpy as np

from oracle import attention, kvstore, rope


def make_store(w, with_pool=True, page_size=None, free_list="seeded"):
    ks, vs = w.scales()
    fl = w.free_list() if free_list == "seeded" else free_list
    return kvstore.KVStore(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim,
                           w.num_pages, kv_dtype=w.kv_dtype,
                           page_size=page_size or w.page_size, free_list=fl,
                           k_scale=ks, v_scale=vs, with_pool=with_pool)


def run(w, layers=None, with_pool=True, compute=True, store=None, on_pass=None, kv_layers=None):
    """Execute every op.  Returns (store, handles, passes) where passes is a
    list of dicts {segs, pass, out[layer], lse[layer]} for attending passes.
    layers: layers attended (default all); kv_layers: layers whose K/V are
    appended (default all)."""
    store = store or make_store(w, with_pool=with_pool)
    layers = range(w.num_layers) if layers is None else layers
    kv_layers = range(w.num_layers) if kv_layers is None else kv_layers
    handles = {}
    passes = []
    for op in w.ops:
        kind = op[0]
        if kind == "create":
            handles[op[1]] = store.ws_create()
        elif kind == "fork":
            handles[op[2]] = store.ws_fork(handles[op[1]])
        elif kind == "freeze":
            store.ws_freeze(handles[op[1]], op[2])
        elif kind == "rollback":
            store.ws_rollback(handles[op[1]], op[2])
        elif kind == "destroy":
            store.ws_destroy(handles.pop(op[1]))
        elif kind == "match":
            store.ws_match_prefix(handles[op[1]], w.tok_stream(op[2]))
        elif kind == "pass":
            segs, attend = op[1], op[2]
            pas = store.begin([(handles[s[0]], s[1], w.gather_tok(s[4])) for s in segs])
            rec = {"segs": segs, "pass": pas, "out": {}, "lse": {}}
            if with_pool:
                if w.rope_theta:
                    tab = rope.table(w.rope_theta, w.head_dim, max(pas.rows_pos, default=0) + 1)
                for layer in (kv_layers if compute else ()):
                    k, v, q = w.pass_inputs(segs, layer, attend and layer in layers)
                    if w.rope_theta and len(pas.rows_pos):
                        k = rope.apply(k, pas.rows_pos, tab)
                        if q is not None:
                            q = rope.apply(q, pas.rows_pos, tab)
                            rec.setdefault("q_rot", {})[layer] = q
                    store.kv_append(pas, layer, k, v)
                    if attend and layer in layers:
                        o, l = attention.attend_pass(store, pas, layer, kvstore.bf16_bits_to_f64(q),
                                                    w.logit_softcap)
                        rec["out"][layer], rec["lse"][layer] = o, l
            if on_pass is not None:
                on_pass(store, handles, rec)
            if attend:
                passes.append(rec)
        else:
            raise ValueError(kind)
    return store, handles, passes
