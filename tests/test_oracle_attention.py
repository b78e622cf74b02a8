"""Pins of the oracle's attention: brute force, PyTorch SDPA in float64,
closed forms and working-set invariants."""
import math

import numpy as np
import pytest
import torch

import oracle_driver
from oracle import attention, kvstore
from paged_kv_attention_working_gb300 import workloads as wl


def brute_force_row(q, k, v, pos):
    """Pure-Python loops, no numpy arithmetic. q [Hq][d]; k, v [n][Hkv][d]."""
    hq, d, hkv = len(q), len(q[0]), len(k[0])
    g = hq // hkv
    out, lse = [], []
    for h in range(hq):
        kv = h // g
        scores = []
        for j in range(pos + 1):
            acc = 0.0
            for i in range(d):
                acc += q[h][i] * k[j][kv][i]
            scores.append(acc / math.sqrt(d))
        m = max(scores)
        w = [math.exp(s - m) for s in scores]
        tot = sum(w)
        out.append([sum(w[j] * v[j][kv][i] for j in range(pos + 1)) / tot for i in range(d)])
        lse.append(m + math.log(tot))
    return out, lse


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 8, 13), (8, 2, 16, 5), (6, 3, 4, 21), (2, 2, 8, 1)])
def test_attend_row_matches_brute_force(hq, hkv, d, n):
    rng = np.random.default_rng(hq * 100 + n)
    q = rng.standard_normal((hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    for pos in (0, n // 2, n - 1):
        o, lse = attention.attend_row(q, k, v, pos)
        bo, bl = brute_force_row(q.tolist(), k.tolist(), v.tolist(), pos)
        np.testing.assert_allclose(o, np.array(bo), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-13)


def _chunk_store(n_ctx, n_new, hq=8, hkv=2, d=64, page_size=16, seed=0, free_list=None):
    """One working set with n_ctx frozen tokens plus a chunk of n_new rows."""
    rng = np.random.default_rng(seed)
    n = n_ctx + n_new
    kb = wl.bf16_round(rng.standard_normal((n, hkv, d)).astype(np.float32))
    vb = wl.bf16_round(rng.standard_normal((n, hkv, d)).astype(np.float32))
    qb = wl.bf16_round(rng.standard_normal((n_new, hq, d)).astype(np.float32))
    pages = -(-n // page_size) + 2
    st = kvstore.KVStore(1, hq, hkv, d, pages, page_size=page_size, free_list=free_list)
    h = st.ws_create()
    if n_ctx:
        p0 = st.begin([(h, n_ctx, None)])
        st.kv_append(p0, 0, kb[:n_ctx], vb[:n_ctx])
        st.ws_freeze(h)
    p1 = st.begin([(h, n_new, None)])
    st.kv_append(p1, 0, kb[n_ctx:], vb[n_ctx:])
    o, lse = attention.attend_pass(st, p1, 0, kvstore.bf16_bits_to_f64(qb))
    return o, lse, kb, vb, qb


def test_prefill_chunk_matches_torch_sdpa_float64():
    n_ctx, n_new, hq, hkv, d = 37, 29, 8, 2, 64
    o, lse, kb, vb, qb = _chunk_store(n_ctx, n_new, hq, hkv, d, seed=3)
    k = torch.from_numpy(kvstore.bf16_bits_to_f64(kb)).permute(1, 0, 2)   # [Hkv, n, d]
    v = torch.from_numpy(kvstore.bf16_bits_to_f64(vb)).permute(1, 0, 2)
    q = torch.from_numpy(kvstore.bf16_bits_to_f64(qb)).permute(1, 0, 2)   # [Hq, n_new, d]
    k = k.repeat_interleave(hq // hkv, dim=0)
    v = v.repeat_interleave(hq // hkv, dim=0)
    n = n_ctx + n_new
    qpos = torch.arange(n_ctx, n)[:, None]
    mask = torch.arange(n)[None, :] <= qpos                              # [n_new, n]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
    # lse: log-sum-exp of the masked, scaled logits
    s = torch.einsum("hqd,hkd->hqk", q, k) / math.sqrt(d)
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).T.numpy(), rtol=1e-12, atol=1e-12)


def test_single_key_returns_v_exactly():
    o, lse, kb, vb, qb = _chunk_store(0, 1, seed=5)
    v = kvstore.bf16_bits_to_f64(vb)[0]
    for h in range(8):
        np.testing.assert_array_equal(o[0, h], v[h // 4])


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, 16))
    k = np.repeat(rng.standard_normal((1, 2, 16)), 11, axis=0)
    v = rng.standard_normal((11, 2, 16))
    o, _ = attention.attend_row(q, k, v, 10)
    for h in range(4):
        np.testing.assert_allclose(o[h], v[:, h // 2].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_output_is_convex_combination_of_values():
    o, lse, kb, vb, qb = _chunk_store(50, 20, seed=11)
    v = kvstore.bf16_bits_to_f64(vb)
    for r in range(20):
        vis = v[:50 + r + 1]
        for h in range(8):
            lo, hi = vis[:, h // 4].min(0), vis[:, h // 4].max(0)
            assert np.all(o[r, h] >= lo - 1e-12) and np.all(o[r, h] <= hi + 1e-12)


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_page_size_does_not_change_result(page_size):
    base, base_lse, *_ = _chunk_store(45, 21, page_size=16, seed=21)
    o, lse, *_ = _chunk_store(45, 21, page_size=page_size, seed=21)
    np.testing.assert_array_equal(o, base)
    np.testing.assert_array_equal(lse, base_lse)


def test_physical_page_permutation_does_not_change_result():
    base, *_ = _chunk_store(70, 9, seed=31)
    pages = -(-79 // 16) + 2
    perm = np.random.default_rng(1).permutation(pages)
    o, *_ = _chunk_store(70, 9, seed=31, free_list=perm)
    np.testing.assert_array_equal(o, base)


def _rows_by_ws(rec, name):
    return [i for i, s in enumerate(_expand(rec)) if s == name]


def _expand(rec):
    names = []
    for s in rec["segs"]:
        names += [s[0]] * s[1]
    return names


def test_fork_attends_like_unshared_copy_and_rollback_reappend():
    w = wl.fork_spec(name="fork_pin", seed=77, prompt=70, n_forks=3, suffix_hi=20, hq=8, hkv=2, d=64)
    store, handles, passes = oracle_driver.run(w)
    drafts_fork, reappend, drafts_copy = passes
    # forks share the prompt pages; unshared copies share nothing with them
    assert store.refcount[store.ws_page_table(handles["f0"])[0]] == 4
    assert store.refcount[store.ws_page_table(handles["u0"])[0]] == 1
    np.testing.assert_array_equal(drafts_fork["out"][0], drafts_copy["out"][0])
    np.testing.assert_array_equal(drafts_fork["lse"][0], drafts_copy["lse"][0])
    # rollback of the last 2 drafts then re-append == never rolled back
    for i in range(3):
        rows = [r for r, n in enumerate(_expand(drafts_fork)) if n == f"f{i}"][2:]
        rrows = [r for r, n in enumerate(_expand(reappend)) if n == f"f{i}"]
        np.testing.assert_array_equal(drafts_fork["out"][0][rows], reappend["out"][0][rrows])


def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible slip in the oracle's arithmetic fails a pin above."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((6, 2, 8))
    v = rng.standard_normal((6, 2, 8))
    bo, _ = brute_force_row(q.tolist(), k.tolist(), v.tolist(), 5)

    def no_scale(q, k, v, softcap=0.0):
        s = np.asarray(k) @ np.asarray(q)
        e = np.exp(s - s.max())
        return (e @ np.asarray(v)) / e.sum(), 0.0

    def wrong_group(q_row, k_ctx, v_ctx, pos):
        hq = q_row.shape[0]
        o = np.empty_like(q_row)
        for h in range(hq):
            o[h], _ = attention.softmax_attention(q_row[h], k_ctx[:pos + 1, h % 2], v_ctx[:pos + 1, h % 2])
        return o, None

    def reversed_keys(q, k, v, softcap=0.0):
        # weights paired with the values in reverse order (an index mistake)
        s = (np.asarray(k) @ np.asarray(q)) / np.sqrt(len(q))
        e = np.exp(s - s.max())
        return (e[::-1] @ np.asarray(v)) / e.sum(), 0.0

    monkeypatch.setattr(attention, "softmax_attention", no_scale)
    assert not np.allclose(attention.attend_row(q, k, v, 5)[0], bo)
    monkeypatch.undo()
    assert not np.allclose(wrong_group(q, k, v, 5)[0], bo)
    monkeypatch.setattr(attention, "softmax_attention", reversed_keys)
    with pytest.raises(AssertionError):
        np.testing.assert_allclose(attention.attend_row(q, k, v, 5)[0], bo)


# ---------------------------------------------------------------- logit soft cap
# The pages name ``logit_softcap`` without a formula; the oracle reads it as
# s <- c * tanh(s / c) on the scaled scores.  These pins come from limits and
# one exactly solvable case, not from the formula restated.

def test_softcap_large_cap_is_no_cap():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal(16), rng.standard_normal((9, 16)), rng.standard_normal((9, 16))
    o0, l0 = attention.softmax_attention(q, k, v)
    o1, l1 = attention.softmax_attention(q, k, v, softcap=1e7)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    assert abs(l1 - l0) < 1e-12


def test_softcap_vanishing_cap_gives_mean_of_values():
    """|capped score| <= c, so as c -> 0 every visible key weighs the same."""
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal(8) * 4, rng.standard_normal((7, 8)), rng.standard_normal((7, 8))
    c = 1e-9
    o, lse = attention.softmax_attention(q, k, v, softcap=c)
    np.testing.assert_allclose(o, v.mean(axis=0), rtol=0, atol=1e-8)
    assert abs(lse - math.log(7)) < 1e-8


def test_softcap_exact_case():
    """d = 4 (scale 1/2), cap 2: a key with q.k = 2 ln 3 has scaled score ln 3,
    capped to 2 tanh(ln 3 / 2) = 1 exactly; a zero key scores 0.  So the
    weights are (1, e) / (1 + e) and lse = ln(1 + e)."""
    q = np.array([2 * math.log(3), 0, 0, 0])
    k = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    v = np.array([[1.0, 2, 3, 4], [-1.0, 0, 5, 2]])
    o, lse = attention.softmax_attention(q, k, v, softcap=2.0)
    e = math.e
    np.testing.assert_allclose(o, (v[0] + e * v[1]) / (1 + e), rtol=1e-14, atol=1e-14)
    assert abs(lse - math.log(1 + e)) < 1e-14
    # the cap must act on the scaled score: capping q.k before the 1/sqrt(d)
    # would give tanh(ln 3) = 0.8, and capping without the outer c would give 0.5
    for wrong in (0.8, 0.5):
        assert abs(lse - math.log(1 + math.exp(wrong))) > 1e-3


def test_softcap_reaches_rows_of_a_pass():
    """Every row of a pass (context plus a causal chunk) takes the cap: with a
    vanishing cap each row is the mean of the values it may see."""
    rng = np.random.default_rng(9)
    hq, hkv, d, n_ctx, n_new = 4, 2, 64, 20, 6
    kb = wl.bf16_round(rng.standard_normal((n_ctx + n_new, hkv, d)).astype(np.float32))
    vb = wl.bf16_round(rng.standard_normal((n_ctx + n_new, hkv, d)).astype(np.float32))
    qb = wl.bf16_round(rng.standard_normal((n_new, hq, d)).astype(np.float32))
    st = kvstore.KVStore(1, hq, hkv, d, 4)
    h = st.ws_create()
    p0 = st.begin([(h, n_ctx, None)])
    st.kv_append(p0, 0, kb[:n_ctx], vb[:n_ctx])
    p1 = st.begin([(h, n_new, None)])
    st.kv_append(p1, 0, kb[n_ctx:], vb[n_ctx:])
    o, _ = attention.attend_pass(st, p1, 0, kvstore.bf16_bits_to_f64(qb), softcap=1e-9)
    v = kvstore.bf16_bits_to_f64(vb)
    for r, pos in enumerate(p1.rows_pos):
        for hh in range(hq):
            np.testing.assert_allclose(o[r, hh], v[:pos + 1, hh // 2].mean(axis=0), rtol=0, atol=1e-7)
