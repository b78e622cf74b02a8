"""The C++ host core (through the C ABI, plan-only contexts, no GPU) against
the oracle's working-set model: bit-exact page tables, reference counts,
slot maps and error statuses; plus the planner's work decomposition."""
import os
import re

import numpy as np
import pytest

import oracle_driver
from oracle import kvstore
from oracle.kvstore import OracleError
from paged_kv_attention_working_gb300 import pie
from paged_kv_attention_working_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "pie_attn.h")).read()
    declared = set(re.findall(r"^\s*(?:pie_status|const char\*)\s+(pie_\w+)\s*\(", header, re.M))
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(pie.lib, name), name
    assert declared <= set(pie.EXPORTS) | {"pie_last_error"}


class Twin:
    """Same operations on the oracle model and on a plan-only library context."""

    def __init__(self, P, free_list, hq=4, hkv=2, d=64):
        self.o = kvstore.KVStore(1, hq, hkv, d, P, free_list=free_list, with_pool=False)
        self.c = pie.pie_ctx_create(1, hq, hkv, d, P, free_list=free_list, num_sms=152)

    def call(self, name, *args):
        err_o = err_c = None
        try:
            ro = getattr(self.o, name)(*args)
        except OracleError as e:
            err_o, ro = e.status, None
        cargs = [self.c] + list(args)
        try:
            if name == "begin":
                b = pie.pie_batch_begin(self.c, args[0])
                rc = pie.pie_batch_slots(b)
                pie.pie_batch_end(self.c, b)
            else:
                rc = getattr(pie, "pie_" + name)(*cargs)
        except pie.PieError as e:
            err_c, rc = e.status, None
        assert err_o == err_c, (name, args, err_o, err_c)
        if name == "begin" and ro is not None:
            assert (ro.rows_pos, ro.rows_slot) == tuple(rc)
        elif name in ("ws_create", "ws_fork", "ws_match_prefix") and ro is not None:
            assert ro == rc
        return ro

    def compare(self):
        assert pie.pie_free_pages(self.c) == len(self.o.free)
        for p in range(self.o.P):
            assert pie.pie_page_refcount(self.c, p) == self.o.refcount[p], p
        for h in self.o.ws:
            assert pie.pie_ws_page_table(self.c, h) == self.o.ws_page_table(h)
            assert pie.pie_ws_info(self.c, h) == self.o.ws_info(h)

    def close(self):
        pie.pie_ctx_destroy(self.c)


def test_random_operation_sequences_bit_exact():
    rng = np.random.default_rng(2024)
    for trial in range(25):
        P = int(rng.integers(4, 48))
        t = Twin(P, rng.permutation(P).tolist())
        live = []
        for step in range(80):
            op = int(rng.integers(0, 8))
            if op == 0 or not live:
                live.append(t.call("ws_create"))
            elif op == 1:
                h = t.call("ws_fork", live[rng.integers(len(live))])
                if h is not None:
                    live.append(h)
            elif op in (2, 7):
                segs = []
                for h in rng.permutation(live)[: rng.integers(1, len(live) + 1)]:
                    n = int(rng.integers(0, 40))
                    toks = rng.integers(0, 2, n).tolist() if rng.random() < 0.7 else None
                    segs.append((int(h), n, toks))
                if rng.random() < 0.05 and segs:
                    segs.append(segs[0])          # duplicate working set: rejected
                t.call("begin", segs)
            elif op == 3:
                t.call("ws_freeze", live[rng.integers(len(live))], int(rng.integers(-1, 30)))
            elif op == 4:
                t.call("ws_rollback", live[rng.integers(len(live))], int(rng.integers(0, 20)))
            elif op == 5:
                h = live.pop(rng.integers(len(live)))
                t.call("ws_destroy", h)
            elif op == 6:
                h = t.call("ws_create")
                live.append(h)
                t.call("ws_match_prefix", h, rng.integers(0, 2, int(rng.integers(0, 70))).tolist())
            t.compare()
        t.call("ws_destroy", 10 ** 6)            # bad handle on both sides
        t.close()


def test_failed_begin_leaves_host_state_unchanged():
    """A pass whose device half fails (a CUDA failure faked on the host at
    the plan upload, after the slots were reserved) gives PIE_ERR_CUDA and
    undoes its reservation: page tables, reference counts, the free stack's
    order (the next allocations match the oracle's) and the lengths are as
    before, and no batch stays open."""
    rng = np.random.default_rng(77)
    for trial in range(12):
        P = int(rng.integers(8, 48))
        t = Twin(P, rng.permutation(P).tolist())
        live = [t.call("ws_create") for _ in range(3)]
        for step in range(60):
            op = int(rng.integers(0, 5))
            segs = []
            for h in rng.permutation(live)[: rng.integers(1, len(live) + 1)]:
                n = int(rng.integers(0, 24))
                segs.append((int(h), n, rng.integers(0, 2, n).tolist() if rng.random() < 0.5 else None))
            if op == 0:
                pie.pie_selftest_fail_next_begin(t.c)
                with pytest.raises(pie.PieError) as e:
                    pie.pie_batch_begin(t.c, segs)
                # a pass the pool cannot cover fails before it reserves anything
                assert e.value.status in (pie.PIE_ERR_CUDA, pie.PIE_ERR_NO_PAGES)
                if e.value.status == pie.PIE_ERR_NO_PAGES:
                    # the injected failure is still pending: an empty pass takes it
                    with pytest.raises(pie.PieError) as e:
                        pie.pie_batch_begin(t.c, [])
                    assert e.value.status == pie.PIE_ERR_CUDA
            elif op == 1:
                t.call("begin", segs)
            elif op == 2:
                h = t.call("ws_fork", live[rng.integers(len(live))])
                if h is not None:
                    live.append(h)
            elif op == 3:
                t.call("ws_freeze", live[rng.integers(len(live))], int(rng.integers(-1, 30)))
            else:
                t.call("ws_rollback", live[rng.integers(len(live))], int(rng.integers(0, 20)))
            t.compare()
        t.close()


def test_block_offsets_match_hand_worked_header_examples():
    """The oracle's byte placement inside a page block against offsets worked
    by hand from the layout the header states (panels of 128 bytes per key,
    2048 bytes per panel, 16-byte chunk c of slot s at s*128 + 16*(c ^ s%8))."""
    bf16 = kvstore.block_offsets(16, 128, 2)        # 256 bytes per key: two panels
    # slot 3, dim 70 -> bytes 140, 141: panel 1, chunk 0 (stored at chunk 3), byte 12
    assert bf16[3, 140] == 2048 + 3 * 128 + 16 * 3 + 12 == 2492
    assert bf16[3, 141] == 2493
    # slot 0 is stored unswizzled: byte b of panel 0 at b
    assert list(bf16[0, :128]) == list(range(128))
    # slot 9, byte 17 (dim 8): panel 0, chunk 1 -> chunk 1 ^ 1 = 0, byte 1
    assert bf16[9, 17] == 9 * 128 + 0 + 1 == 1153
    # slot 15, last byte (dim 127, high byte): panel 1, chunk 7 -> 7 ^ 7 = 0, byte 15
    assert bf16[15, 255] == 2048 + 15 * 128 + 15 == 3983
    e4 = kvstore.block_offsets(16, 128, 1)           # 128 bytes per key: one panel
    # slot 6, dim 100: chunk 6 -> 6 ^ 6 = 0, byte 4
    assert e4[6, 100] == 6 * 128 + 4 == 772
    # slot 13, dim 33: chunk 2 -> 2 ^ 5 = 7, byte 1
    assert e4[13, 33] == 13 * 128 + 112 + 1 == 1777
    d64 = kvstore.block_offsets(16, 64, 2)           # 128 bytes per key
    assert d64[2, 127] == 2 * 128 + 16 * (7 ^ 2) + 15 == 351
    # every block byte is used exactly once
    for offs in (bf16, e4, d64):
        assert sorted(offs.reshape(-1).tolist()) == list(range(offs.size))


@pytest.mark.parametrize("name", list(wl.FULL) + list(wl.EXTRA))
def test_workload_scripts_bit_exact(name):
    w = wl.reduced(name)
    c = pie.pie_ctx_create(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_pages,
                           kv_dtype=w.kv_dtype, free_list=w.free_list().tolist(),
                           k_scale=w.scales()[0], v_scale=w.scales()[1])
    handles = {}
    store = oracle_driver.make_store(w, with_pool=False)
    ohandles = {}
    for op in w.ops:
        k = op[0]
        if k == "create":
            handles[op[1]] = pie.pie_ws_create(c)
            ohandles[op[1]] = store.ws_create()
        elif k == "fork":
            handles[op[2]] = pie.pie_ws_fork(c, handles[op[1]])
            ohandles[op[2]] = store.ws_fork(ohandles[op[1]])
        elif k == "freeze":
            pie.pie_ws_freeze(c, handles[op[1]], op[2])
            store.ws_freeze(ohandles[op[1]], op[2])
        elif k == "rollback":
            pie.pie_ws_rollback(c, handles[op[1]], op[2])
            store.ws_rollback(ohandles[op[1]], op[2])
        elif k == "match":
            toks = w.tok_stream(op[2]).tolist()
            assert pie.pie_ws_match_prefix(c, handles[op[1]], toks) == store.ws_match_prefix(ohandles[op[1]], toks)
        elif k == "pass":
            pas = store.begin([(ohandles[s[0]], s[1], w.gather_tok(s[4])) for s in op[1]])
            b = pie.pie_batch_begin(c, [(handles[s[0]], s[1], w.gather_tok(s[4])) for s in op[1]])
            assert pie.pie_batch_slots(b) == (pas.rows_pos, pas.rows_slot)
            assert pie.pie_batch_plan_info(b)["copies"] == len(pas.cow)
            pie.pie_batch_end(c, b)
    for name_, h in handles.items():
        assert pie.pie_ws_page_table(c, h) == store.ws_page_table(ohandles[name_])
    for p in range(w.num_pages):
        assert pie.pie_page_refcount(c, p) == store.refcount[p]
    pie.pie_ctx_destroy(c)


def _run_plan(w, upto_pass):
    """Executes a workload on a plan-only context up to its upto_pass-th pass
    and returns (ctx, handles, batch) with that pass's batch open."""
    c = pie.pie_ctx_create(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_pages,
                           kv_dtype=w.kv_dtype, free_list=w.free_list().tolist(),
                           k_scale=w.scales()[0], v_scale=w.scales()[1], num_sms=152)
    hs = {}
    n = 0
    for op in w.ops:
        k = op[0]
        if k == "create":
            hs[op[1]] = pie.pie_ws_create(c)
        elif k == "fork":
            hs[op[2]] = pie.pie_ws_fork(c, hs[op[1]])
        elif k == "freeze":
            pie.pie_ws_freeze(c, hs[op[1]], op[2])
        elif k == "rollback":
            pie.pie_ws_rollback(c, hs[op[1]], op[2])
        elif k == "match":
            pie.pie_ws_match_prefix(c, hs[op[1]], w.tok_stream(op[2]).tolist())
        elif k == "pass":
            b = pie.pie_batch_begin(c, [(hs[s[0]], s[1], w.gather_tok(s[4])) for s in op[1]])
            if n == upto_pass:
                return c, hs, b
            pie.pie_batch_end(c, b)
            n += 1
    raise AssertionError("pass not found")


def _coverage(c, b, w, hs, segs):
    """Per row: list of (kind, item) covering it; checks each row's keys
    0..pos are covered exactly once."""
    import itertools
    pos, _ = pie.pie_batch_slots(b)
    rows_ws = list(itertools.chain.from_iterable([s[0]] * s[1] for s in segs))
    # reconstruct row lists: identity for private items, group lists after
    items = [(0, it) for it in pie.pie_batch_items(b, 0)] + [(1, it) for it in pie.pie_batch_items(b, 1)]
    return pos, rows_ws, items


def test_plan_fork_group_reads_shared_pages_once():
    w = wl.fork_spec(name="fork_plan", seed=3, prompt=4096, n_forks=10, suffix_hi=256, unshared=False)
    c, hs, b = _run_plan(w, 2)          # the drafts pass: 10 forks x 4 drafts
    info = pie.pie_batch_plan_info(b)
    pre = pie.pie_batch_items(b, 1)
    dec = pie.pie_batch_items(b, 0)
    # 40 rows x 4 query heads per KV head = 160 > 64: shared prefix on the tensor-core kernel,
    # in two balanced row tiles of 20 rows (one 128-row Q tile each), KV split across items;
    # every shared page in exactly one item per row tile
    shared = [it for it in pre if it["key_base"] < 4096 and it["n_rows"] == 20]
    tiles = sorted({it["rows_off"] for it in shared})
    assert len(tiles) == 2
    for t in tiles:
        mine = sorted((it["key_base"], it["n_pages"]) for it in shared if it["rows_off"] == t)
        assert mine[0][0] == 0 and sum(n for _, n in mine) == 4096 // 16
        for (a, n), (b2, _) in zip(mine, mine[1:]):
            assert a + 16 * n == b2
    # private parts: one decode item (4 drafts x 4 heads = 16) per fork
    assert len([it for it in dec if it["n_rows"] == 4]) >= 10
    assert info["merge_rows"] == 40
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_nested_forks_read_each_shared_run_once():
    """A fork of a fork: the prompt's pages are in shared items over all 7
    leaves' 28 rows, the first fork's own frozen pages in shared items over
    its 4 sub-forks' 16 rows only, each page of each run in exactly one item
    per row tile; every leaf's remaining pages are private."""
    w = wl.reduced("nested_fork")
    c, hs, b = _run_plan(w, 3)              # the drafts pass
    pre, dec = pie.pie_batch_items(b, 1), pie.pie_batch_items(b, 0)
    prompt_pages = 300 // 16                 # full pages of the prompt (18)
    sub_pages = (300 + 70) // 16 - prompt_pages   # the first fork's full pages past the prompt (5)
    top = [it for it in pre if it["n_rows"] == 28]
    assert sorted((it["key_base"], it["n_pages"]) for it in top)[0][0] == 0
    assert sum(it["n_pages"] for it in top) == prompt_pages
    sub = [it for it in dec if it["n_rows"] == 16]
    assert sum(it["n_pages"] for it in sub) == sub_pages
    assert min(it["key_base"] for it in sub) == 16 * prompt_pages
    # every leaf row has the prompt's parts, the sub-forks' rows also the sub-run's
    info = pie.pie_batch_plan_info(b)
    assert info["merge_rows"] == 28
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_drafts_of_large_head_groups_still_share():
    """Four drafts at 32 query heads per KV head (128 rows x heads) join the
    fork group: the prompt is read once per pass, not once per fork."""
    w = wl.reduced("fork_spec_mqa_g32")
    c, hs, b = _run_plan(w, 2)
    pre = pie.pie_batch_items(b, 1)
    prompt_pages = 400 // 16
    shared = [it for it in pre if it["key_base"] < 16 * prompt_pages]
    tiles = sorted({it["rows_off"] for it in shared})
    # 40 rows x 32 heads = 1280: ten row tiles of 4 rows (one Q tile each), each over the whole prompt
    assert len(tiles) == 10 and all(it["n_rows"] == 4 for it in shared)
    for t in tiles:
        assert sum(it["n_pages"] for it in shared if it["rows_off"] == t) == prompt_pages
    assert pie.pie_batch_plan_info(b)["merge_rows"] == 40
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_dedup_groups_on_decode_kernel():
    w = wl.llama70b_fp8(n_ws=16, ctx_lo=2048, ctx_hi=4096, prefix_groups=2)
    c, hs, b = _run_plan(w, 2)
    dec = pie.pie_batch_items(b, 0)
    shared = [it for it in dec if it["n_rows"] == 8]
    # 8 rows x 8 heads = 64 = four M tiles in one CTA: each shared page once per group
    assert sum(it["n_pages"] for it in shared) == 2 * (2048 // 16)
    assert pie.pie_batch_plan_info(b)["prefill_items"] == 0
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_puts_wide_decode_items_first():
    """Decode items of more than 32 rows x query heads (the dedup groups'
    64-wide shared items) come first, each kind longest first: pie_attend
    launches the two kinds separately (two N tiles per warp for the wide
    ones) and relies on this order."""
    w = wl.llama70b_fp8(n_ws=16, ctx_lo=2048, ctx_hi=4096, prefix_groups=2)
    c, hs, b = _run_plan(w, 2)
    G = w.num_q_heads // w.num_kv_heads
    dec = pie.pie_batch_items(b, 0)
    wide = [it["n_rows"] * G > 32 for it in dec]
    n_wide = sum(wide)
    assert n_wide > 0 and all(wide[:n_wide]) and not any(wide[n_wide:])
    for part in (dec[:n_wide], dec[n_wide:]):
        pages = [it["n_pages"] for it in part]
        assert pages == sorted(pages, reverse=True)
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_splits_cover_every_key_once():
    w = wl.decode_batch(name="split_plan", seed=7, n_ws=64, num_layers=1)
    c, hs, b = _run_plan(w, 1)
    dec = pie.pie_batch_items(b, 0)
    pos, _ = pie.pie_batch_slots(b)
    per_row = {}
    for it in dec:
        assert it["n_rows"] == 1
        per_row.setdefault(it["rows_off"], []).append((it["key_base"], it["n_pages"], it["part"]))
    for r, lst in per_row.items():
        lst.sort()
        assert lst[0][0] == 0
        for (a, n, _), (b2, _, _) in zip(lst, lst[1:]):
            assert a + 16 * n == b2
        last = lst[-1]
        assert last[0] + 16 * last[1] >= pos[r] + 1 > last[0] + 16 * (last[1] - 1)
        parts = sorted(p for _, _, p in lst)
        assert parts == ([-1] if len(lst) == 1 else list(range(len(lst))))
    assert len(dec) > 64
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_only_context_rejects_device_calls():
    c = pie.pie_ctx_create(1, 4, 2, 64, 8)
    h = pie.pie_ws_create(c)
    b = pie.pie_batch_begin(c, [(h, 3, None)])
    with pytest.raises(pie.PieError) as e:
        pie.pie_kv_append(c, b, 0, 0, 0)
    assert e.value.status == pie.PIE_ERR_STATE
    with pytest.raises(pie.PieError) as e:
        pie.pie_ws_create(c)                 # batch open
    assert e.value.status == pie.PIE_ERR_STATE
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_merge_mode_takes_the_two_documented_values():
    c = pie.pie_ctx_create(1, 4, 2, 64, 8)
    for mode in (0, 1):
        pie.pie_ctx_set_merge_mode(c, mode)
    for mode in (-1, 2):
        with pytest.raises(pie.PieError) as e:
            pie.pie_ctx_set_merge_mode(c, mode)
        assert e.value.status == pie.PIE_ERR_INVALID
    pie.pie_ctx_destroy(c)


def test_invalid_configurations_rejected():
    with pytest.raises(pie.PieError):
        pie.pie_ctx_create(1, 6, 4, 64, 8)           # Hq not a multiple of Hkv
    with pytest.raises(pie.PieError):
        pie.pie_ctx_create(1, 4, 2, 96, 8)           # unsupported head_dim
    with pytest.raises(pie.PieError):
        pie.pie_ctx_create(1, 4, 2, 128, 8, kv_dtype=pie.PIE_KV_E4M3)   # e4m3 without scales
    with pytest.raises(pie.PieError):
        pie.pie_ctx_create(1, 4, 2, 64, 4, free_list=[0, 1, 1, 2])      # not a permutation
    for cap in (-1.0, float("inf"), float("nan")):
        with pytest.raises(pie.PieError):
            pie.pie_ctx_create(1, 4, 2, 64, 8, logit_softcap=cap)       # soft cap must be finite, >= 0
    for theta, npos in ((-1.0, 16), (1.0, 16), (float("inf"), 16), (float("nan"), 16), (10000.0, 0)):
        with pytest.raises(pie.PieError):
            pie.pie_ctx_create(1, 4, 2, 64, 8, rope_theta=theta, rope_max_positions=npos)


@pytest.mark.parametrize("theta,d,positions", [(500000.0, 128, 33000), (10000.0, 64, 4096), (1234.5, 128, 2000)])
def test_rope_table_matches_oracle_bit_for_bit(theta, d, positions):
    from oracle import rope
    np.testing.assert_array_equal(pie.pie_rope_table(theta, d, positions), rope.table(theta, d, positions))


def test_rope_append_on_a_plan_only_context_is_a_state_error():
    c = pie.pie_ctx_create(1, 4, 2, 64, 8, rope_theta=10000.0, rope_max_positions=20)
    h = pie.pie_ws_create(c)
    b = pie.pie_batch_begin(c, [(h, 21, None)])
    with pytest.raises(pie.PieError) as e:
        pie.pie_kv_append_rope(c, b, 0, 16, 16)   # aligned stand-ins, never dereferenced
    assert e.value.status == pie.PIE_ERR_STATE
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_prefill_chunks_never_join_groups():
    """A pass that appends long chunks to sets sharing a prefix plans every
    row with one part (no partial results to merge)."""
    w = wl.llama70b_fp8(n_ws=16, ctx_lo=2048, ctx_hi=4096, prefix_groups=2)
    c, hs, b = _run_plan(w, 1)          # the fill pass after match_prefix
    info = pie.pie_batch_plan_info(b)
    assert info["merge_rows"] == 0 and info["prefill_items"] > 0
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)


def test_plan_marks_consecutive_rows_direct():
    """Items whose rows are consecutive batch rows carry the direct flag and
    index the identity prefix of the row list: a segment's private items,
    and a fork group whose members sit next to each other in the pass.  A
    group split by another segment keeps its own row list."""
    cfg = dict(num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=64, num_pages=64)
    for order, consecutive in (("ffu", True), ("fuf", False)):
        c = pie.pie_ctx_create(**cfg)
        prompt = pie.pie_ws_create(c)
        b = pie.pie_batch_begin(c, [(prompt, 64, None)])
        pie.pie_batch_end(c, b)
        pie.pie_ws_freeze(c, prompt)
        f1, f2 = pie.pie_ws_fork(c, prompt), pie.pie_ws_fork(c, prompt)
        u = pie.pie_ws_create(c)
        ws = {"f": [f1, f2], "u": [u]}
        segs = [(ws[k].pop(0), 3, None) for k in order]
        b = pie.pie_batch_begin(c, segs)
        items = pie.pie_batch_items(b, 0) + pie.pie_batch_items(b, 1)
        shared = [it for it in items if it["n_rows"] == 6]
        assert shared, "the fork group's prompt pages form a shared item"
        for it in shared:
            assert it["direct_rows"] == (1 if consecutive else 0)
            if consecutive:
                assert it["rows_off"] == 0        # rows 0..5, the identity prefix
            else:
                assert it["rows_off"] >= 9        # a list of its own after the 9 batch rows
        for it in items:
            if it["n_rows"] == 3:                  # private items: each segment's own rows
                assert it["direct_rows"] == 1 and it["rows_off"] % 3 == 0
        pie.pie_batch_end(c, b)
        pie.pie_ctx_destroy(c)


def test_misaligned_pointers_are_rejected_before_any_launch():
    """K, V, Q and outputs move in 16-byte vectors and bulk copies: a call
    given a misaligned pointer fails with PIE_ERR_INVALID before it checks
    anything that would need a GPU (here a plan-only context, whose
    well-aligned calls fail with PIE_ERR_STATE instead)."""
    import ctypes
    c = pie.pie_ctx_create(1, 8, 2, 64, 16)
    ws = pie.pie_ws_create(c)
    b = pie.pie_batch_begin(c, [(ws, 3, None)])
    lib = pie.lib
    odd, ok = 0x1008, 0x1000          # never dereferenced: the calls return first
    assert lib.pie_attend(c, b, 0, odd, ok, None) == pie.PIE_ERR_INVALID
    assert lib.pie_attend(c, b, 0, ok, odd, None) == pie.PIE_ERR_INVALID
    assert lib.pie_attend(c, b, 0, ok, ok, ctypes.c_void_p(0x1002)) == pie.PIE_ERR_INVALID
    assert lib.pie_attend(c, b, 0, ok, ok, None) == pie.PIE_ERR_STATE
    assert lib.pie_kv_append(c, b, 0, odd, ok) == pie.PIE_ERR_INVALID
    assert lib.pie_kv_append(c, b, 0, ok, ok) == pie.PIE_ERR_STATE
    assert lib.pie_kv_append_rope(c, b, 0, ok, ok, odd, ok) == pie.PIE_ERR_INVALID
    pie.pie_batch_end(c, b)
    pie.pie_ctx_destroy(c)
