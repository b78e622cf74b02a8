"""The per-layer calls of a pass (pie_kv_append, pie_kv_append_rope,
pie_attend) only enqueue kernels on the context's stream, so a caller can
capture a whole pass into a CUDA graph once the plan is uploaded
(pie_batch_begin) and replay it.  The replay must give the same bytes as
the eager calls."""
import numpy as np
import pytest
import torch

import gpu_driver
from paged_kv_attention_working_gb300 import pie
from paged_kv_attention_working_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", ["llama8b_decode", "mixed_batch", "fork_spec_e4m3", "mixed_batch_rope"])
def test_pass_replays_from_a_cuda_graph(name):
    w = wl.reduced(name)
    s = torch.cuda.Stream()
    esize = 2 if w.kv_dtype == wl.KV_BF16 else 1
    n = w.num_layers * w.num_pages * w.num_kv_heads * 16 * w.head_dim * esize
    kpool = torch.zeros(n, dtype=torch.uint8, device="cuda")
    vpool = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ks, vs = w.scales()
    ctx = pie.pie_ctx_create(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_pages,
                             kv_dtype=w.kv_dtype, free_list=w.free_list().tolist(), k_scale=ks, v_scale=vs,
                             k_pool=kpool, v_pool=vpool, stream=s.cuda_stream, logit_softcap=w.logit_softcap,
                             rope_theta=w.rope_theta, rope_max_positions=w.rope_positions)
    hs = {}
    last = max(i for i, op in enumerate(w.ops) if op[0] == "pass" and op[2])
    with torch.cuda.stream(s):
        for op in w.ops[:last]:
            k = op[0]
            if k == "create":
                hs[op[1]] = pie.pie_ws_create(ctx)
            elif k == "fork":
                hs[op[2]] = pie.pie_ws_fork(ctx, hs[op[1]])
            elif k == "freeze":
                pie.pie_ws_freeze(ctx, hs[op[1]], op[2])
            elif k == "rollback":
                pie.pie_ws_rollback(ctx, hs[op[1]], op[2])
            elif k == "match":
                pie.pie_ws_match_prefix(ctx, hs[op[1]], w.tok_stream(op[2]).tolist())
            elif k == "pass":
                b = pie.pie_batch_begin(ctx, [(hs[g[0]], g[1], w.gather_tok(g[4])) for g in op[1]])
                for layer in range(w.num_layers):
                    kk, vv, _ = w.pass_inputs(op[1], layer, False)
                    kd, vd = gpu_driver.to_dev_bf16(kk), gpu_driver.to_dev_bf16(vv)
                    if w.rope_theta:
                        pie.pie_kv_append_rope(ctx, b, layer, kd, vd)
                    else:
                        pie.pie_kv_append(ctx, b, layer, kd, vd)
                pie.pie_batch_end(ctx, b)
        segs = w.ops[last][1]
        b = pie.pie_batch_begin(ctx, [(hs[g[0]], g[1], w.gather_tok(g[4])) for g in segs])
        rows = pie.pie_batch_rows(b)
        ins = []
        for layer in range(w.num_layers):
            kk, vv, qq = w.pass_inputs(segs, layer, True)
            ins.append((gpu_driver.to_dev_bf16(kk), gpu_driver.to_dev_bf16(vv), gpu_driver.to_dev_bf16(qq)))
        outs = [(torch.empty((rows, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda"),
                 torch.empty((rows, w.num_q_heads), dtype=torch.float32, device="cuda"),
                 torch.empty((rows, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda"))
                for _ in range(w.num_layers)]

        def run_pass():
            for layer, ((kd, vd, qd), (o, l, qr)) in enumerate(zip(ins, outs)):
                if w.rope_theta:
                    pie.pie_kv_append_rope(ctx, b, layer, kd, vd, qd, qr)
                    pie.pie_attend(ctx, b, layer, qr, o, l)
                else:
                    pie.pie_kv_append(ctx, b, layer, kd, vd)
                    pie.pie_attend(ctx, b, layer, qd, o, l)

        run_pass()  # eager (also sets the kernels' attributes before any capture)
    s.synchronize()
    eager = [(o.clone(), l.clone()) for o, l, _ in outs]
    for o, l, _ in outs:
        o.zero_()
        l.zero_()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_pass()
    for _ in range(2):
        g.replay()
    s.synchronize()
    for (o, l, _), (oe, le) in zip(outs, eager):
        assert torch.equal(o.view(torch.int16), oe.view(torch.int16))
        assert torch.equal(l, le)
    assert pie.pie_ctx_check(ctx) == 0
    pie.pie_batch_end(ctx, b)
    pie.pie_ctx_destroy(ctx)
    del kpool, vpool
