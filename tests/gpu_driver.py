"""Runs a synthetic workload's operation script through the CUDA library's
C ABI (via the Python binding) on the current CUDA device."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_attention_working_gb300 import pie


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to("cuda").view(torch.bfloat16)


class DeviceRun:
    def __init__(self, w, device="cuda", num_sms=0):
        self.w = w
        esize = 2 if w.kv_dtype == pie.PIE_KV_BF16 else 1
        self.block = 16 * w.head_dim * esize
        n = w.num_layers * w.num_pages * w.num_kv_heads * self.block
        self.kpool = torch.zeros(n, dtype=torch.uint8, device=device)
        self.vpool = torch.zeros(n, dtype=torch.uint8, device=device)
        ks, vs = w.scales()
        self.stream = torch.cuda.current_stream()
        self.ctx = pie.pie_ctx_create(w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_pages,
                                      kv_dtype=w.kv_dtype, free_list=w.free_list().tolist(), k_scale=ks,
                                      v_scale=vs, k_pool=self.kpool, v_pool=self.vpool,
                                      stream=self.stream.cuda_stream, logit_softcap=w.logit_softcap,
                                      rope_theta=w.rope_theta, rope_max_positions=w.rope_positions,
                                      num_sms=num_sms)
        self.handles = {}

    def run(self, layers=None, kv_source=None):
        """Executes every op.  kv_source(segs, layer) may supply device K, V (and
        Q) instead of the exact numpy streams.  Returns the attending passes as
        dicts {segs, out[layer], lse[layer], plan}."""
        w = self.w
        layers = range(w.num_layers) if layers is None else layers
        passes = []
        for op in w.ops:
            k = op[0]
            if k == "create":
                self.handles[op[1]] = pie.pie_ws_create(self.ctx)
            elif k == "fork":
                self.handles[op[2]] = pie.pie_ws_fork(self.ctx, self.handles[op[1]])
            elif k == "freeze":
                pie.pie_ws_freeze(self.ctx, self.handles[op[1]], op[2])
            elif k == "rollback":
                pie.pie_ws_rollback(self.ctx, self.handles[op[1]], op[2])
            elif k == "destroy":
                pie.pie_ws_destroy(self.ctx, self.handles.pop(op[1]))
            elif k == "match":
                pie.pie_ws_match_prefix(self.ctx, self.handles[op[1]], w.tok_stream(op[2]).tolist())
            elif k == "pass":
                segs, attend = op[1], op[2]
                b = pie.pie_batch_begin(self.ctx, [(self.handles[s[0]], s[1], w.gather_tok(s[4])) for s in segs])
                n = pie.pie_batch_rows(b)
                rec = {"segs": segs, "out": {}, "lse": {}, "plan": pie.pie_batch_plan_info(b)}
                for layer in range(w.num_layers):
                    want = attend and layer in layers
                    if kv_source is not None:
                        kd, vd, qd = kv_source(segs, layer, want)
                    else:
                        kk, vv, qq = w.pass_inputs(segs, layer, want)
                        kd, vd = to_dev_bf16(kk), to_dev_bf16(vv)
                        qd = to_dev_bf16(qq) if want else None
                    if w.rope_theta:
                        # rotary embedding fused into the append; Q is rotated
                        # into a new buffer that the attention then reads
                        qr = torch.empty_like(qd) if want else None
                        pie.pie_kv_append_rope(self.ctx, b, layer, kd, vd, qd if want else None, qr)
                        if want:
                            rec.setdefault("q_rot", {})[layer] = qr
                            qd = qr
                    else:
                        pie.pie_kv_append(self.ctx, b, layer, kd, vd)
                    if want:
                        out = torch.empty((n, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
                        lse = torch.empty((n, w.num_q_heads), dtype=torch.float32, device="cuda")
                        pie.pie_attend(self.ctx, b, layer, qd, out, lse)
                        rec["out"][layer] = out
                        rec["lse"][layer] = lse
                pie.pie_batch_end(self.ctx, b)
                if attend:
                    passes.append(rec)
        flags = pie.pie_ctx_check(self.ctx)
        assert flags == 0, f"kernel error flags {flags}"
        return passes

    def pools(self):
        shape = (self.w.num_layers, self.w.num_pages, self.w.num_kv_heads, self.block)
        return (self.kpool.cpu().numpy().reshape(shape), self.vpool.cpu().numpy().reshape(shape))

    def close(self):
        pie.pie_ctx_destroy(self.ctx)
