"""GPU parity at the full sizes of the five workloads (and of the fork and
mixed workloads with e4m3 KV), in the launch configuration the benchmark
times (the whole batch in one pie_batch / pie_attend per layer).

The oracle cannot hold every working set of the larger workloads, so a few
working sets are sampled: their K/V/Q (and, for fork / dedup groups, the
whole group's) come from the exact seeded streams, the others' from random
device data that no checked row can see.  The oracle runs the same operation
script restricted to the sampled sets; their appended bytes must match
bit for bit and their rows within the tolerance of the reduced-size tests.
"""
import numpy as np
import pytest
import torch

import gpu_driver
import oracle_driver
from oracle import kvstore
from paged_kv_attention_working_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = {wl.KV_BF16: 2e-2, wl.KV_E4M3: 5e-2}
LSE_ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _involved(op):
    k = op[0]
    if k == "fork":
        return [op[1], op[2]]
    if k == "pass":
        return [s[0] for s in op[1]]
    return [op[1]]


def sub_workload(w, names):
    """The same script restricted to the named working sets."""
    names = set(names)
    ops = []
    for op in w.ops:
        if op[0] == "pass":
            segs = [s for s in op[1] if s[0] in names]
            if segs:
                ops.append(("pass", segs, op[2]))
        elif all(n in names for n in _involved(op)):
            ops.append(op)
    sub = wl.Workload(w.name + "_sub", w.seed, w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim,
                      w.kv_dtype, 0, ops, dict(w.kv_streams), dict(w.q_streams), dict(w.tok_streams))
    sub.logit_softcap, sub.rope_theta, sub.rope_positions = w.logit_softcap, w.rope_theta, w.rope_positions
    # pages needed: replay on a page-count-only store and keep the peak
    big = 1 << 20
    st = kvstore.KVStore(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim, big, with_pool=False)
    peak = [0]

    def note(store, handles, rec):
        peak[0] = max(peak[0], big - len(store.free))

    sub.num_pages = big
    oracle_driver.run(sub, with_pool=False, store=st, on_pass=note)
    sub.num_pages = peak[0] + 16
    return sub


def exact_source(w, exact, seed=7):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)

    def src(segs, layer, want):
        ks, vs, qs = [], [], []
        for s in segs:
            if s[1] == 0:
                continue
            if s[0] in exact:
                k, v = w.gather_kv(s[2], layer)
                ks.append(gpu_driver.to_dev_bf16(k))
                vs.append(gpu_driver.to_dev_bf16(v))
                if want:
                    qs.append(gpu_driver.to_dev_bf16(w.gather_q(s[3], layer)))
            else:
                shape = (s[1], w.num_kv_heads, w.head_dim)
                ks.append(torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16))
                vs.append(torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16))
                if want:
                    qs.append(torch.randn((s[1], w.num_q_heads, w.head_dim), generator=gen,
                                          device="cuda").to(torch.bfloat16))
        return torch.cat(ks), torch.cat(vs), (torch.cat(qs) if want else None)

    return src


def row_ranges(segs):
    out, r = {}, 0
    for s in segs:
        out[s[0]] = (r, r + s[1])
        r += s[1]
    return out


def check(w, names, layers, rows_of=None, merge_mode=0):
    """Runs w on the GPU (names exact) and the restricted script on the
    oracle; compares pool bytes and attention rows of the named sets.
    Returns the device passes' plan summaries."""
    from paged_kv_attention_working_gb300 import pie
    sub = sub_workload(w, names)
    store, ohandles, ref_passes = oracle_driver.run(sub, layers=layers, kv_layers=layers)
    g = gpu_driver.DeviceRun(w)
    pie.pie_ctx_set_merge_mode(g.ctx, merge_mode)
    passes = g.run(layers=layers, kv_source=exact_source(w, set(names)))
    # appended bytes, page by page in logical order, valid slots only
    esize = 2 if w.kv_dtype == wl.KV_BF16 else 1
    offs = kvstore.block_offsets(16, w.head_dim, esize)
    shape = (w.num_layers, w.num_pages, w.num_kv_heads, g.block)
    kp, vp = g.kpool.view(shape), g.vpool.view(shape)
    for n in names:
        n_tok = pie.pie_ws_info(g.ctx, g.handles[n])[0]
        gpages = pie.pie_ws_page_table(g.ctx, g.handles[n])
        opages = store.ws_page_table(ohandles[n])
        for layer in layers:
            gi = torch.tensor(gpages, device="cuda")
            gk, gv = kp[layer][gi].cpu().numpy(), vp[layer][gi].cpu().numpy()
            ok_, ov_ = store.pool[0, layer][opages], store.pool[1, layer][opages]
            for pos in range(n_tok):
                i, s = divmod(pos, 16)
                np.testing.assert_array_equal(gk[i, :, offs[s]], ok_[i, :, offs[s]], err_msg=f"{n} K pos {pos}")
                np.testing.assert_array_equal(gv[i, :, offs[s]], ov_[i, :, offs[s]], err_msg=f"{n} V pos {pos}")
    assert len(passes) == len(ref_passes)
    for got, ref in zip(passes, ref_passes):
        gr, orr = row_ranges(got["segs"]), row_ranges(ref["segs"])
        for n in names:
            if n not in orr:
                continue
            (a, b), (c, d) = gr[n], orr[n]
            sel = slice(None) if rows_of is None else rows_of(n, b - a)
            for layer in layers:
                o = got["out"][layer][a:b].float().cpu().numpy()[sel]
                r = ref["out"][layer][c:d][sel]
                err = np.abs(o - r)
                bad = err > ATOL[w.kv_dtype] + RTOL * np.abs(r)
                assert not bad.any(), f"{n} layer {layer}: {int(bad.sum())} bad, max abs {err.max():.3g}"
                lse = got["lse"][layer][a:b].cpu().numpy()[sel]
                assert np.abs(lse - ref["lse"][layer][c:d][sel]).max() <= LSE_ATOL, f"{n} lse layer {layer}"
    g.close()
    return [p["plan"] for p in passes]


def test_llama8b_decode_full():
    w = wl.llama8b_decode()
    order = np.argsort(w.ctx)
    names = [f"w{order[0]}", f"w{order[len(order) // 2]}", f"w{order[-1]}"]
    check(w, names, layers=[0, w.num_layers - 1])


@pytest.mark.parametrize("kv_dtype", [wl.KV_BF16, wl.KV_E4M3])
def test_fork_spec_full(kv_dtype):
    w = wl.fork_spec(kv_dtype=kv_dtype)
    names = ["root"] + [f"f{i}" for i in range(10)] + [f"u{i}" for i in range(10)]
    check(w, names, layers=[0])


@pytest.mark.parametrize("kv_dtype", [wl.KV_BF16, wl.KV_E4M3])
def test_mixed_batch_full(kv_dtype):
    w = wl.mixed_batch(kv_dtype=kv_dtype)
    chunks = list(np.argsort(w.chunks))
    names = [f"c{chunks[0]}", f"c{chunks[-1]}", "d0", "d77"]
    rng = np.random.default_rng(0)

    def rows_of(n, count):
        if count <= 64:
            return slice(None)
        pick = np.unique(np.concatenate([np.arange(8), np.arange(count - 8, count), rng.integers(0, count, 48)]))
        return pick

    check(w, names, layers=[0], rows_of=rows_of)


def test_llama70b_fp8_full():
    w = wl.llama70b_fp8()
    names = [f"w{i}" for i in range(248, 256)]  # the last dedup group (prefix writer + 7 matches)
    check(w, names, layers=[0])


def test_mixed_batch_full_softcap():
    w = wl.mixed_batch()
    w.logit_softcap = 5.0
    chunks = list(np.argsort(w.chunks))
    names = [f"c{chunks[-1]}", "d5"]
    rng = np.random.default_rng(1)

    def rows_of(n, count):
        if count <= 64:
            return slice(None)
        return np.unique(np.concatenate([np.arange(8), np.arange(count - 8, count), rng.integers(0, count, 48)]))

    check(w, names, layers=[0], rows_of=rows_of)


def test_llama8b_decode_full_rope():
    w = wl.llama8b_decode()
    w.rope_theta = 500000.0
    w.rope_positions = max(w.ctx) + 2
    order = np.argsort(w.ctx)
    names = [f"w{order[0]}", f"w{order[-1]}"]
    check(w, names, layers=[0])


@pytest.mark.parametrize("name", ["llama8b_decode", "llama70b_fp8"])
def test_decode_full_merged_inside_the_decode_launch(name):
    """Merge mode 1 at the benchmark's sizes: the decode kernels merge the
    split rows themselves (per (row, query head) part counters: 64 x 32 and
    256 x 64 of them, over several waves of CTAs; for the 70B batch the wide
    and narrow launches count into the same counters), with no merge launch.
    The 8B batch attends two layers of the pass, so the counters must be back
    at zero after the first."""
    w = getattr(wl, name)()
    if name == "llama8b_decode":
        order = np.argsort(w.ctx)
        names, layers = [f"w{order[0]}", f"w{order[len(order) // 2]}", f"w{order[-1]}"], [0, w.num_layers - 1]
    else:
        names, layers = [f"w{i}" for i in range(248, 256)], [0]
    plans = check(w, names, layers=layers, merge_mode=1)
    decode_passes = [p for p in plans if p["merge_rows"]]
    assert decode_passes and not any(p["merge_launch"] for p in decode_passes)
