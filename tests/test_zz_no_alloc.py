"""Decode attention through the entry point that allocates nothing
(pie_attend_decode_noalloc), checked against the CPU oracle and against
pie_attend on the same pools.

That entry point serves callers that cannot call cudaMalloc -- engines that
reserved device memory for their own allocator, loops that cannot take the
synchronisation an allocation may imply, plug-ins whose host forbids foreign
allocations.  Its split partials live in a library-owned device array that
every call reuses, so it is called twice in a row here: the second call must
not depend on what the first one left behind.

Each case first runs its workload through the library (which fills the
pools) and through the oracle: the pools must agree bit for bit, so the
oracle's outputs are the exact reference for what the entry point reads.
Tolerances are those of the other parity tests (bf16 KV: |g - r| <= 2e-2 +
1e-2 |r|; LSE within 2e-3).
"""
import numpy as np
import pytest
import torch

import gpu_driver
import oracle_driver
from paged_kv_attention_working_gb300 import pie
from paged_kv_attention_working_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL, ATOL, LSE_ATOL = 1e-2, 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _close(got, ref, atol, rtol, what):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside tolerance, max abs {err.max():.3g}"


@pytest.mark.parametrize("name,kw", [
    ("llama8b_small", dict(name="na8b", seed=21, n_ws=6, ctx_lo=200, ctx_hi=1500, num_layers=2)),
    ("many_rows", dict(name="narows", seed=22, n_ws=48, ctx_lo=1, ctx_hi=700, num_layers=1)),
    ("d64", dict(name="na64", seed=23, n_ws=5, ctx_lo=30, ctx_hi=400, num_layers=1, hq=8, hkv=2, d=64)),
    # two rows: the entry point splits them into about 60 parts each (empty
    # ones for the shorter row), which the merge takes 32 at a time
    ("two_long_rows", dict(name="na2", seed=24, n_ws=2, ctx_lo=2500, ctx_hi=3000, num_layers=1)),
    # one KV head for 64 query heads: four MMA row tiles per row
    ("mqa_g64", dict(name="namqa", seed=25, n_ws=4, ctx_lo=100, ctx_hi=900, num_layers=1, hq=64, hkv=1)),
])
def test_noalloc_decode_matches_oracle_and_attend_on_two_calls(name, kw):
    w = wl.decode_batch(**kw)
    store, _, ref_passes = oracle_driver.run(w)
    g = gpu_driver.DeviceRun(w)
    passes = g.run()
    kp, vp = g.pools()
    np.testing.assert_array_equal(kp, store.pool[0])
    np.testing.assert_array_equal(vp, store.pool[1])
    dec, ref_dec = passes[-1], ref_passes[-1]
    segs = dec["segs"]
    handles = [g.handles[s[0]] for s in segs]
    tables = [pie.pie_ws_page_table(g.ctx, h) for h in handles]
    lens = [pie.pie_ws_info(g.ctx, h)[0] for h in handles]
    max_pages = max(len(t) for t in tables)
    bt = np.zeros((len(tables), max_pages), dtype=np.int32)
    for i, t in enumerate(tables):
        bt[i, : len(t)] = t
    bt_d = torch.from_numpy(bt).cuda()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    n = len(handles)
    for layer, attend_out in dec["out"].items():
        q = gpu_driver.to_dev_bf16(w.pass_inputs(segs, layer, True)[2])
        oracle_out, oracle_lse = ref_dec["out"][layer], ref_dec["lse"][layer]
        attend = attend_out.float().cpu().numpy()
        attend_lse = dec["lse"][layer].cpu().numpy()
        for call in range(2):
            out = torch.full((n, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
            lse = torch.full((n, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
            pie.pie_attend_decode_noalloc(n, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_layers, w.num_pages,
                                          layer, max_pages, q, g.kpool, g.vpool, bt_d, lens_d, out, lse, stream)
            torch.cuda.synchronize()
            o, l_ = out.float().cpu().numpy(), lse.cpu().numpy()
            _close(o, oracle_out, ATOL, RTOL, f"{name} layer {layer} call {call} vs oracle")
            _close(l_, oracle_lse, LSE_ATOL, 0.0, f"{name} lse layer {layer} call {call} vs oracle")
            _close(o, attend, ATOL, RTOL, f"{name} layer {layer} call {call} vs pie_attend")
            _close(l_, attend_lse, LSE_ATOL, 0.0, f"{name} lse layer {layer} call {call} vs pie_attend")
    g.close()


def test_noalloc_rejects_work_beyond_its_scratch():
    # one row alone needs about 32 + 28 bytes; this many rows overflow 16 MiB
    rows = pie.PIE_NOALLOC_SCRATCH_BYTES // 40
    with pytest.raises(pie.PieError) as e:
        # aligned stand-in pointers: the call returns before it touches any
        pie.pie_attend_decode_noalloc(rows, 32, 8, 128, 1, 16, 0, 1, 16, 16, 16, 16, 16, 16)
    assert e.value.status == pie.PIE_ERR_RANGE
