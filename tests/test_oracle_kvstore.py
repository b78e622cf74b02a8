"""Pins of the oracle's working-set state machine: a hand-worked scenario,
dedup, transactional failure and invariants under random operation
sequences."""
import copy

import numpy as np
import pytest

from oracle import kvstore
from oracle.kvstore import OracleError


def _store(P=8, free_list=(5, 2, 7, 0, 1, 3, 6, 4), page_size=4):
    return kvstore.KVStore(1, 2, 1, 64, P, page_size=page_size, free_list=list(free_list))


def test_hand_worked_scenario():
    st = _store()
    a = st.ws_create()
    assert a == 1
    p = st.begin([(a, 6, None)])
    # free stack pops 5 then 2 (first entries of the given order)
    assert st.ws_page_table(a) == [5, 2]
    assert p.rows_slot == [20, 21, 22, 23, 8, 9] and p.rows_pos == [0, 1, 2, 3, 4, 5]
    st.ws_freeze(a, 5)
    assert st.ws_info(a) == (6, 5, 2)
    b = st.ws_fork(a)
    # the child holds the 5 frozen tokens: pages 5 and 2 (the partial tail), shared
    assert st.ws_info(b) == (5, 5, 2)
    assert st.refcount[5] == 2 and st.refcount[2] == 2
    p = st.begin([(b, 2, None)])
    # b writes into its shared tail page 2 -> copy-on-write into the next free page, 7
    assert p.cow == [(2, 7)]
    assert st.ws_page_table(b) == [5, 7] and st.refcount[2] == 1 and st.refcount[7] == 1
    assert p.rows_slot == [29, 30]
    st.ws_rollback(a, 1)
    assert st.ws_info(a) == (5, 5, 2)
    with pytest.raises(OracleError) as e:
        st.ws_rollback(a, 1)
    assert e.value.status == kvstore.ERR_RANGE
    p = st.begin([(a, 4, None), (b, 1, None)])
    # a: positions 5..7 fill page 2 (no longer shared), position 8 takes page 0
    assert st.ws_page_table(a) == [5, 2, 0]
    assert p.rows_slot == [9, 10, 11, 0, 31]
    assert p.cow == []
    st.ws_destroy(a)
    # release order: page 0, page 2 (both freed), page 5 (still held by b)
    assert st.free[-2:] == [0, 2] and st.refcount[5] == 1
    c = st.ws_create()
    st.begin([(c, 1, None)])
    assert c == 3 and st.ws_page_table(c) == [2]
    st.check_invariants()


def test_fork_and_rollback_release_order():
    st = _store(P=10, free_list=range(10))
    a = st.ws_create()
    st.begin([(a, 10, None)])            # pages 0, 1, 2
    st.ws_freeze(a, 4)
    b = st.ws_fork(a)                    # shares page 0 only (4 frozen tokens = 1 full page)
    assert st.ws_page_table(b) == [0]
    st.ws_rollback(a, 6)                 # drops tokens 4..9 -> releases pages 2 then 1
    assert st.free[-2:] == [2, 1]
    assert st.ws_page_table(a) == [0] and st.refcount[0] == 2
    st.check_invariants()


def test_dedup_match_prefix():
    st = _store(P=12, free_list=range(12))
    a = st.ws_create()
    toks = list(range(100, 110))
    st.begin([(a, 10, toks)])            # pages 0, 1, 2
    st.ws_freeze(a)
    # fully frozen pages 0 and 1 are registered; page 2 (2 tokens) is not
    assert set(st.page_key) == {0, 1}
    b = st.ws_create()
    assert st.ws_match_prefix(b, toks + [7]) == 8
    assert st.ws_page_table(b) == [0, 1] and st.refcount[0] == 2 and st.refcount[1] == 2
    assert st.ws_info(b) == (8, 8, 2)
    c = st.ws_create()
    other = toks[:4] + [1, 2, 3, 4]
    assert st.ws_match_prefix(c, other) == 4
    d = st.ws_create()
    assert st.ws_match_prefix(d, [9] * 4 + toks[4:8]) == 0   # same page tokens, other parent
    with pytest.raises(OracleError):
        st.ws_match_prefix(b, toks)      # not empty
    for h in (a, b, c):
        st.ws_destroy(h)
    assert st.page_key == {} and st.dedup == {}
    e = st.ws_create()
    assert st.ws_match_prefix(e, toks) == 0
    st.check_invariants()


def test_freeze_registers_only_a_chain_from_the_root():
    st = _store(P=12, free_list=range(12))
    a = st.ws_create()
    st.begin([(a, 4, None)])
    st.begin([(a, 4, [1, 2, 3, 4])])
    st.ws_freeze(a)
    # page 0 has unknown tokens, so page 1 cannot be reached from the root
    assert st.page_key == {}


def test_pool_exhaustion_changes_nothing():
    st = _store(P=4, free_list=range(4))
    a = st.ws_create()
    b = st.ws_create()
    st.begin([(a, 5, None)])             # 2 pages
    before = copy.deepcopy((st.free, st.refcount, st.ws))
    with pytest.raises(OracleError) as e:
        st.begin([(b, 4, None), (a, 8, None)])   # needs 1 + 2 > 2 free
    assert e.value.status == kvstore.ERR_NO_PAGES
    assert (st.free, st.refcount, st.ws) == before


def test_duplicate_segment_rejected():
    st = _store()
    a = st.ws_create()
    with pytest.raises(OracleError):
        st.begin([(a, 1, None), (a, 1, None)])


def test_random_operation_sequences_keep_invariants():
    rng = np.random.default_rng(123)
    for trial in range(30):
        P = int(rng.integers(6, 40))
        st = kvstore.KVStore(1, 2, 1, 64, P, page_size=4,
                             free_list=rng.permutation(P).tolist(), with_pool=False)
        live = []
        for step in range(60):
            op = rng.integers(0, 7)
            try:
                if op == 0 or not live:
                    live.append(st.ws_create())
                elif op == 1:
                    live.append(st.ws_fork(live[rng.integers(len(live))]))
                elif op == 2:
                    segs = []
                    for h in rng.permutation(live)[: rng.integers(1, len(live) + 1)]:
                        n = int(rng.integers(0, 9))
                        segs.append((int(h), n, rng.integers(0, 3, n).tolist()))
                    st.begin(segs)
                elif op == 3:
                    h = live[rng.integers(len(live))]
                    st.ws_freeze(h, int(rng.integers(-1, 5)))
                elif op == 4:
                    h = live[rng.integers(len(live))]
                    st.ws_rollback(h, int(rng.integers(0, 4)))
                elif op == 5:
                    h = live.pop(rng.integers(len(live)))
                    st.ws_destroy(h)
                elif op == 6:
                    h = st.ws_create()
                    live.append(h)
                    st.ws_match_prefix(h, rng.integers(0, 3, int(rng.integers(0, 13))).tolist())
            except OracleError:
                pass
            st.check_invariants()
