"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Bit-exact for the appended KV bytes (the whole pools, bf16 and e4m3);
attention outputs elementwise within |g - r| <= atol + rtol |r| with
rtol 1e-2 and atol 2e-2 (bf16 KV) or 5e-2 (e4m3 KV), and the LSE within
2e-3 absolute.  The output tolerance covers bf16 rounding of the output
(2^-9 relative), bf16 rounding of the softmax weights fed to the tensor
cores (2^-9 relative per weight) and fp32 accumulation over up to ~10^4
keys; for e4m3 the scores and weights are the same computation on the
dequantised values, so only the f16 weight rounding (2^-11) changes.
"""
import numpy as np
import pytest
import torch

import gpu_driver
import oracle_driver
from oracle import e4m3
from paged_kv_attention_working_gb300 import pie
from paged_kv_attention_working_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = {wl.KV_BF16: 2e-2, wl.KV_E4M3: 5e-2}
LSE_ATOL = 2e-3


def assert_close(got, ref, atol, rtol, what):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max abs {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _parity(name, num_sms=0, before=None):
    """Runs reduced workload `name` on the device and the oracle and compares
    pools, outputs and LSE; before(ctx) runs first.  Returns the device
    passes' plan summaries."""
    w = wl.reduced(name)
    store, handles, ref_passes = oracle_driver.run(w)
    g = gpu_driver.DeviceRun(w, num_sms=num_sms)
    if before is not None:
        before(g.ctx)
    passes = g.run()
    kp, vp = g.pools()
    np.testing.assert_array_equal(kp, store.pool[0])
    np.testing.assert_array_equal(vp, store.pool[1])
    assert len(passes) == len(ref_passes)
    for got, ref in zip(passes, ref_passes):
        for layer, qr in got.get("q_rot", {}).items():   # rotated Q, bit for bit
            np.testing.assert_array_equal(qr.view(torch.int16).cpu().numpy().view(np.uint16), ref["q_rot"][layer])
        for layer, out in got["out"].items():
            o = out.float().cpu().numpy()
            assert_close(o, ref["out"][layer], ATOL[w.kv_dtype], RTOL, f"{name} out layer {layer}")
            lse = got["lse"][layer].cpu().numpy()
            assert_close(lse, ref["lse"][layer], LSE_ATOL, 0.0, f"{name} lse layer {layer}")
    g.close()
    return [p["plan"] for p in passes]


@pytest.mark.parametrize("name", list(wl.FULL) + list(wl.EXTRA))
def test_reduced_workload_parity(name):
    _parity(name)


# A context planned for 2 SMs: the planner then splits the KV runs far less
# (decode items of many more pages, shared runs in one item per row tile),
# and every tensor-core launch spans several waves.
@pytest.mark.parametrize("name", ["mixed_batch", "mixed_batch_e4m3", "mixed_batch_d64", "mixed_batch_mha",
                                  "mixed_batch_g8", "mixed_batch_g16", "mixed_batch_mqa_g32", "mixed_batch_mqa_g64",
                                  "mixed_batch_d64_mqa_g16", "mixed_batch_softcap", "fork_spec", "edge_batch",
                                  "interleaved_forks"])
def test_reduced_workload_parity_few_sms(name):
    _parity(name, num_sms=2)


# Workloads whose split rows come from decode items only (one per kernel
# variant: bf16 and e4m3 pages, d 64, wide fork / dedup items, G 64), plus
# the fork workload, which runs passes with split tensor-core items (merge
# launch) and then decode-only passes.
MERGE_CASES = ["llama8b_decode", "llama70b_fp8", "mixed_batch_e4m3", "mixed_batch_d64", "edge_batch",
               "mixed_batch_mqa_g64", "fork_spec"]


@pytest.mark.parametrize("name", MERGE_CASES)
def test_split_rows_merged_inside_the_decode_launch(name):
    """Mode 1: rows split over decode items only are combined by the decode
    kernels themselves (per (row, query head) a count of stored parts; the
    CTA that stores the last part merges them and resets the count), with no
    merge launch; passes with a split tensor-core item still take one.
    Consecutive attends (two layers, or several passes) must each leave the
    counts at zero, and a kernel error report first makes the next pass clear
    them.  Against the oracle."""
    def setup(ctx):
        pie.pie_ctx_set_merge_mode(ctx, 1)
        pie.pie_selftest_wait_timeout(ctx, 64)
        assert pie.pie_ctx_check(ctx) == 1

    merged = [p for p in _parity(name, before=setup) if p["merge_rows"]]
    assert any(not p["merge_launch"] for p in merged)
    if name == "fork_spec":  # its first passes split the shared prompt's tensor-core items
        assert any(p["merge_launch"] for p in merged)


@pytest.mark.parametrize("name", ["llama70b_fp8", "fork_spec"])
def test_split_rows_merged_by_a_merge_launch_by_default(name):
    """Mode 0, the default: every pass with split rows ends with a merge
    launch (set explicitly here after mode 1, to check the switch back)."""
    def setup(ctx):
        pie.pie_ctx_set_merge_mode(ctx, 1)
        pie.pie_ctx_set_merge_mode(ctx, 0)

    merged = [p for p in _parity(name, before=setup) if p["merge_rows"]]
    assert merged and all(p["merge_launch"] for p in merged)


@pytest.mark.parametrize("scale", [5.0 / 448.0, 0.37, 1.0])
def test_e4m3_append_matches_codec_over_all_bf16(scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    bits = bits[~np.isnan(vals)]
    n = -(-bits.size // 128)
    k = np.zeros(n * 128, dtype=np.uint16)
    k[: bits.size] = bits
    k = k.reshape(n, 1, 128)
    w = wl.Workload("e4m3_all", 0, 1, 1, 1, 128, wl.KV_E4M3, -(-n // 16) + 1, [])
    g = gpu_driver.DeviceRun(w)
    pie.pie_ctx_destroy(g.ctx)
    g.ctx = pie.pie_ctx_create(1, 1, 1, 128, w.num_pages, kv_dtype=pie.PIE_KV_E4M3, k_scale=[scale],
                               v_scale=[scale], k_pool=g.kpool, v_pool=g.vpool,
                               stream=torch.cuda.current_stream().cuda_stream)
    h = pie.pie_ws_create(g.ctx)
    b = pie.pie_batch_begin(g.ctx, [(h, n, None)])
    pos, slot = pie.pie_batch_slots(b)
    kd = gpu_driver.to_dev_bf16(k)
    pie.pie_kv_append(g.ctx, b, 0, kd, kd)
    pie.pie_batch_end(g.ctx, b)
    kp, vp = g.pools()
    from oracle import kvstore
    offs = kvstore.block_offsets(16, 128, 1)
    got = np.stack([kp[0, s // 16, 0][offs[s % 16]] for s in slot]).reshape(-1)[: bits.size]
    ref = e4m3.quantize((bits.astype(np.uint32) << 16).view(np.float32), scale)
    np.testing.assert_array_equal(got, ref)
    g.close()


def test_pool_exhaustion_leaves_state_and_device_unchanged():
    w = wl.tiny_decode()
    g = gpu_driver.DeviceRun(w)
    h = pie.pie_ws_create(g.ctx)
    with pytest.raises(pie.PieError) as e:
        pie.pie_batch_begin(g.ctx, [(h, 16 * (w.num_pages + 1), None)])
    assert e.value.status == pie.PIE_ERR_NO_PAGES
    assert pie.pie_free_pages(g.ctx) == w.num_pages
    assert pie.pie_ws_info(g.ctx, h) == (0, 0, 0)
    g.close()


def test_empty_batch_is_a_no_op():
    w = wl.tiny_decode()
    g = gpu_driver.DeviceRun(w)
    h = pie.pie_ws_create(g.ctx)
    b = pie.pie_batch_begin(g.ctx, [(h, 0, None)])
    assert pie.pie_batch_rows(b) == 0
    pie.pie_kv_append(g.ctx, b, 0, None, None)
    pie.pie_attend(g.ctx, b, 0, None, None)
    pie.pie_batch_end(g.ctx, b)
    assert pie.pie_ctx_check(g.ctx) == 0
    g.close()


def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A kernel wait that can never complete ends after its poll limit, sets
    the error bit the host reads, and leaves the context usable."""
    w = wl.tiny_decode()
    g = gpu_driver.DeviceRun(w)
    assert pie.pie_ctx_check(g.ctx) == 0
    pie.pie_selftest_wait_timeout(g.ctx, 1000)
    assert pie.pie_ctx_check(g.ctx) == 1
    assert pie.pie_ctx_check(g.ctx) == 0          # read and cleared
    passes = g.run()                               # the full workload still runs and checks clean
    assert passes and pie.pie_ctx_check(g.ctx) == 0
    g.close()


def test_rope_append_rejects_positions_past_the_table():
    """A row at or past rope_max_positions is a range error with nothing
    launched, and a context without a rotary table refuses the call."""
    w = wl.tiny_decode()
    g = gpu_driver.DeviceRun(w)
    pie.pie_ctx_destroy(g.ctx)
    g.ctx = pie.pie_ctx_create(1, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_pages, k_pool=g.kpool,
                               v_pool=g.vpool, stream=torch.cuda.current_stream().cuda_stream,
                               rope_theta=10000.0, rope_max_positions=20)
    h = pie.pie_ws_create(g.ctx)
    b = pie.pie_batch_begin(g.ctx, [(h, 21, None)])
    k = torch.zeros((21, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pie.PieError) as e:
        pie.pie_kv_append_rope(g.ctx, b, 0, k, k)
    assert e.value.status == pie.PIE_ERR_RANGE
    pie.pie_batch_end(g.ctx, b)
    assert not g.kpool.any()
    g.close()
    g2 = gpu_driver.DeviceRun(w)
    h = pie.pie_ws_create(g2.ctx)
    b = pie.pie_batch_begin(g2.ctx, [(h, 1, None)])
    with pytest.raises(pie.PieError) as e:
        pie.pie_kv_append_rope(g2.ctx, b, 0, k, k)
    assert e.value.status == pie.PIE_ERR_STATE
    pie.pie_batch_end(g2.ctx, b)
    g2.close()
