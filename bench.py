"""Benchmark of batched passes over paged KV working sets.

Headline workload: Llama-3.1-8B-shaped decode batch -- 64 working sets with
contexts uniform in [512, 8192] (seeded), 32 query / 8 KV heads, head_dim 128,
bf16 KV in 16-token pages, 32 layers of independent random K/V.  One step is
one whole pass through the hot path: pie_batch_begin (slot reservation,
plan, upload), then for each of the 32 layers pie_kv_append of the new
token's K/V and pie_attend of its 32 query heads, pie_batch_end, and a
rollback of the speculative token (host) so every step sees the same state.

Metric: decode attend KV GB/s = algorithmic K/V bytes the attention reads
(every valid key once per working set, K and V) / step time; plus query
rows/s.  Inputs (KV cache, Q/K/V of the step) are resident in HBM; the KV
read per layer (~1.1 GB) is far larger than L2, so no flush is needed.

The same JSON line carries, under "workloads", the other timed workloads,
each with its own timing, roofline and clock record: the fork / speculative
pass (a 4096-token prompt shared by 10 forks), the mixed continuous batch
(prefill chunks on the tensor cores plus decode rows; bf16 and e4m3 KV) and
the Llama-3.3-70B-shaped long-context decode with e4m3 KV and dedup groups.
--workload X runs one of them alone as the headline; --only-headline skips
the others.

--impl reference times the CPU oracle instead (bounded sample).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def kernel_sources_sha(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_attention_working_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic(key, files, algorithmic):
    """DRAM bytes per launch (read + write) of a kernel from the ncu capture
    recorded in profiles/traffic.json, scaled by algorithmic work when the
    capture ran a smaller case of the same workload; None when the kernel's
    sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(key)
    if not rec or rec.get("source_sha256") != kernel_sources_sha(files):
        return None
    return rec["dram_bytes_per_launch"] * algorithmic / rec["algorithmic_per_launch"]


def _measured(keys):
    """A number from MEASURED_PEAKS.json (first of keys present; a nested
    {"value": ...} is unwrapped), or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    for k in keys:
        v = d.get(k)
        if isinstance(v, dict):
            v = v.get("value")
        if isinstance(v, (int, float)) and v > 0:
            return float(v)
    return None


def peaks():
    """HBM copy bandwidth (GB/s) for the roofline, measured when available."""
    hbm = _measured(("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"))
    return (hbm, "measured") if hbm else (FALLBACK_HBM_GBS, "fallback")


def tensor_peak():
    """Dense bf16 tensor throughput (TFLOP/s), the burst figure (a prefill
    launch is timed on its own), measured when available."""
    t = _measured(("bf16_tflops", "bf16_TFLOPs"))
    return (t, "measured") if t else (FALLBACK_BF16_TFLOPS, "fallback")


class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        """Summary of the samples taken between wall-clock t_begin and t_end."""
        if self.proc is None:
            self.f.close()
            os.unlink(self.f.name)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait()
        self.f.seek(0)
        rows = [[x.strip() for x in r.split(",")] for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        import datetime

        def ts(r):
            try:
                return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None

        inside = [r for r in rows if len(r) > 9 and ts(r) is not None and t_begin - 0.25 <= ts(r) <= t_end + 0.25]
        num = lambda x: x.replace(".", "").isdigit()
        sm = [float(r[2]) for r in inside if num(r[2])]
        mx = [float(r[3]) for r in inside if num(r[3])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for i, n in enumerate(names):
                if r[6 + i] == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def allmax(world, x):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle leg
class OracleSample:
    """The oracle's attention on a bounded sample of the workload: the decode
    rows of the first working sets of one layer (their real context lengths),
    each in an oracle store built once; only attend_pass is timed."""

    def __init__(self, w, max_rows=64):
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from oracle import kvstore
        from paged_kv_attention_working_gb300.workloads import bf16_round

        self.w = w
        self.kvstore = kvstore
        rng = np.random.default_rng(0)
        self.items = []
        self.max_rows = max_rows
        self.rng, self.bf16_round = rng, bf16_round

    def _item(self, i):
        w, kvstore = self.w, self.kvstore
        while len(self.items) <= i:
            c = w.ctx[len(self.items)]
            n = c + 1
            st = kvstore.KVStore(1, w.num_q_heads, w.num_kv_heads, w.head_dim, -(-n // 16) + 1)
            h = st.ws_create()
            shape = (n, w.num_kv_heads, w.head_dim)
            k = self.bf16_round(self.rng.standard_normal(shape, dtype=np.float32))
            v = self.bf16_round(self.rng.standard_normal(shape, dtype=np.float32))
            q = self.bf16_round(self.rng.standard_normal((1, w.num_q_heads, w.head_dim), dtype=np.float32))
            p = st.begin([(h, n, None)])
            st.kv_append(p, 0, k, v)
            self.items.append((st, kvstore.Pass([h], [n - 1], [p.rows_slot[-1]], []),
                               kvstore.bf16_bits_to_f64(q), c))
        return self.items[i]

    def run(self, seconds):
        """Returns (KV GB/s, rows/s, description, cores, elapsed)."""
        from oracle import attention

        esize = 2 if self.w.kv_dtype == 0 else 1
        kv_bytes = rows = 0
        elapsed = 0.0
        used = []
        for i in range(min(self.max_rows, len(self.w.ctx))):
            st, pas, q, c = self._item(i)
            t0 = time.perf_counter()
            attention.attend_pass(st, pas, 0, q)
            elapsed += time.perf_counter() - t0
            kv_bytes += (c + 1) * self.w.num_kv_heads * self.w.head_dim * esize * 2
            rows += 1
            used.append(c)
            if elapsed > seconds:
                break
        cores = len(os.sched_getaffinity(0))
        desc = (f"oracle attend_pass (float64 numpy, page gather + exact softmax) on {rows} decode rows "
                f"(contexts {used[:4]}{'...' if len(used) > 4 else ''}) of one layer of the workload; "
                f"numpy default BLAS threading")
        return kv_bytes / elapsed / 1e9, rows / elapsed, desc, cores, elapsed


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    per_step, gbs_l, rps_l = [], [], []
    desc = cores = None
    sample = OracleSample(w)
    step_s = max(0.2, args.ref_seconds / max(1, args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        gbs, rps, desc, cores, el = sample.run(step_s)
        if i >= args.warmup:
            per_step.append(el)
            gbs_l.append(gbs)
            rps_l.append(rps)
    gbs, rps = statistics.median(gbs_l), statistics.median(rps_l)
    line = {"impl": "reference", "metric": "decode attend KV GB/s", "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(per_step), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(args, w, world),
            "rows_per_s": rps,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_attend_bytes(w):
    """Algorithmic bytes of one decode attend launch (one layer) of a decode
    workload: K and V of every visible key once per working set (the keys a
    dedup group shares once per group: w.shared_keys counts the copies
    beyond the first), Q and O, the LSE and the page ids.  Returns (K/V
    bytes, whole launch)."""
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    esize = 2 if w.kv_dtype == 0 else 1
    n_rows = len(w.ctx)
    shared = getattr(w, "shared_keys", 0)
    keys = sum(c + 1 for c in w.ctx) - shared
    pages = sum(-(-(c + 1) // 16) for c in w.ctx) - shared // 16
    kv = keys * Hkv * D * esize * 2
    return kv, kv + 2 * n_rows * Hq * D * 2 + n_rows * Hq * 4 + 4 * pages


def decode_config(args, w, world):
    """The config of a decode workload's line, the same for the GPU arm and
    the oracle arm."""
    kv, _ = decode_attend_bytes(w)
    return {"workload": w.name, "n_ws": len(w.ctx), "contexts": "uniform [%d, %d] seeded" % w.ctx_range,
            "layers": w.num_layers, "hq": w.num_q_heads, "hkv": w.num_kv_heads, "head_dim": w.head_dim,
            "kv_dtype": "bf16" if w.kv_dtype == 0 else "e4m3", "page_size": 16,
            "l2": "inputs larger than L2 (%.1f GB of K/V per layer)" % (kv / 1e9),
            "logit_softcap": args.logit_softcap, "rope_theta": args.rope_theta, "merge_mode": args.merge_mode,
            "parallelism": f"replicas x{world}"}


def prefill_chunk_flops(w, chunk_segs):
    """Causal-exact flops of the mixed batch's prefill chunks: 4*d per
    (query head, visible key) pair; a chunk of n rows on c cached tokens has
    n*c + n(n+1)/2 such pairs per head."""
    return sum(4 * w.head_dim * w.num_q_heads * (s[1] * c0 + s[1] * (s[1] + 1) // 2)
               for s, c0 in zip(chunk_segs, w.chunk_ctx))


def append_roofline(nbytes, avg_ms, peak, peak_src, kernel):
    """Roofline of one kv_append launch: algorithmic bytes (each new row's K
    and V read as bf16 and written in the pool's element type; with the
    rotary embedding also Q read and written and the (cos, sin) pairs) over
    the event-timed launch."""
    gbs = nbytes / (avg_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "bytes_per_launch": nbytes, "avg_launch_ms": avg_ms,
            "achieved": gbs, "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": gbs / peak}


def llama70b_workload(n_ws):
    """The 70B-shaped FP8 decode batch, n_ws working sets in dedup groups of
    8 sharing a 2048-token prefix."""
    from paged_kv_attention_working_gb300 import workloads as wl

    w = wl.llama70b_fp8(n_ws=n_ws, prefix_groups=n_ws // 8)
    w.shared_keys = (n_ws - n_ws // 8) * 2048   # shared keys beyond their first copy in each group
    return w


# ----------------------------------------------------------------- GPU leg
def run_gpu(args, w, world, rank, local, e2e=True):
    import torch

    from paged_kv_attention_working_gb300 import pie

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    L, Hq, Hkv, D = w.num_layers, w.num_q_heads, w.num_kv_heads, w.head_dim
    esize = 2 if w.kv_dtype == 0 else 1
    block = 16 * D * esize
    pool_bytes = L * w.num_pages * Hkv * block
    kpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    vpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    ks, vs = w.scales()
    ctx = pie.pie_ctx_create(L, Hq, Hkv, D, w.num_pages, kv_dtype=w.kv_dtype, free_list=w.free_list().tolist(),
                             k_scale=ks, v_scale=vs, k_pool=kpool, v_pool=vpool, stream=stream.cuda_stream,
                             logit_softcap=args.logit_softcap, rope_theta=args.rope_theta,
                             rope_max_positions=(max(w.ctx) + 2) if args.rope_theta else 0)
    pie.pie_ctx_set_merge_mode(ctx, args.merge_mode)
    # set-up: every operation of the workload before its final (decode) pass,
    # with random bf16 K/V generated on the device
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    hs = {}
    last_pass = max(i for i, op in enumerate(w.ops) if op[0] == "pass")
    for op in w.ops[:last_pass]:
        kind = op[0]
        if kind == "create":
            hs[op[1]] = pie.pie_ws_create(ctx)
        elif kind == "freeze":
            pie.pie_ws_freeze(ctx, hs[op[1]], op[2])
        elif kind == "match":
            pie.pie_ws_match_prefix(ctx, hs[op[1]], w.tok_stream(op[2]).tolist())
        elif kind == "pass":
            b = pie.pie_batch_begin(ctx, [(hs[sg[0]], sg[1], w.gather_tok(sg[4])) for sg in op[1]])
            n_fill = pie.pie_batch_rows(b)
            for layer in range(L):
                k = torch.randn((n_fill, Hkv, D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                v = torch.randn((n_fill, Hkv, D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                pie.pie_kv_append(ctx, b, layer, k, v)
                del k, v
            pie.pie_batch_end(ctx, b)
        else:
            raise ValueError(kind)
    torch.cuda.synchronize(dev)
    names = [sg[0] for sg in w.ops[last_pass][1]]
    n_rows = len(names)
    q = torch.randn((L, n_rows, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
    kn = torch.randn((L, n_rows, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
    vn = torch.randn((L, n_rows, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty((L, n_rows, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((L, n_rows, Hq), dtype=torch.float32, device=dev)
    segs = [(hs[n], 1, None) for n in names]

    assert n_rows == len(w.ctx)
    kv_bytes_layer, attend_bytes = decode_attend_bytes(w)
    append_bytes = n_rows * Hkv * D * (2 + esize) * 2
    if args.rope_theta:
        qr = torch.empty_like(q)
        append_bytes += 2 * n_rows * Hq * D * 2 + n_rows * D * 4   # Q in and out, the rows' (cos, sin)

    info = {}

    def step(ev=None, host=None):
        if host is not None:
            qh, kh, vh, oh = host
            q.copy_(qh, non_blocking=True)
            kn.copy_(kh, non_blocking=True)
            vn.copy_(vh, non_blocking=True)
        bb = pie.pie_batch_begin(ctx, segs)
        if not info:
            info.update(pie.pie_batch_plan_info(bb))
            # decode items wider than 32 rows x heads (dedup groups) run in a
            # launch of their own beside the others
            info["wide_decode_items"] = sum(it["n_rows"] * (Hq // Hkv) > 32 for it in pie.pie_batch_items(bb, 0))
        for layer in range(L):
            if ev is not None:
                ev[layer][0].record(stream)
            if args.rope_theta:
                pie.pie_kv_append_rope(ctx, bb, layer, kn[layer], vn[layer], q[layer], qr[layer])
            else:
                pie.pie_kv_append(ctx, bb, layer, kn[layer], vn[layer])
            if ev is not None:
                ev[layer][1].record(stream)
            pie.pie_attend(ctx, bb, layer, qr[layer] if args.rope_theta else q[layer], out[layer], lse[layer])
            if ev is not None:
                ev[layer][2].record(stream)
        pie.pie_batch_end(ctx, bb)
        if host is not None:
            oh.copy_(out, non_blocking=True)
        for n in names:
            pie.pie_ws_rollback(ctx, hs[n], 1)

    clocks = Clocks(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert pie.pie_ctx_check(ctx) == 0
    time.sleep(0.5)  # let the clock sampler start before the timed region

    # ---- device-resident timing
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(args.steps):
        step(events[s])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    barrier(world)
    ms = t0.elapsed_time(t1) / args.steps
    ms = allmax(world, ms)
    attend_ms = [e1.elapsed_time(e2) for st in events for _, e1, e2 in st]
    append_ms = [e0.elapsed_time(e1) for st in events for e0, e1, _ in st]
    attend_avg = statistics.mean(attend_ms)
    append_avg = statistics.mean(append_ms)
    assert pie.pie_ctx_check(ctx) == 0

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e_res = None
    if e2e:
        host = (q.cpu().pin_memory(), kn.cpu().pin_memory(), vn.cpu().pin_memory(),
                torch.empty(out.shape, dtype=out.dtype).pin_memory())
        step(host=host)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(args.steps):
            step(host=host)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = allmax(world, e0.elapsed_time(e1) / args.steps)
        h2d = sum(t.numel() * t.element_size() for t in host[:3])
        d2h = host[3].numel() * host[3].element_size()
        e2e_res = {"value": world * kv_bytes_layer * L / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                   "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    hbm_peak, peak_src = peaks()
    kv_step = kv_bytes_layer * L
    value = world * kv_step / (ms * 1e-3) / 1e9
    achieved = attend_bytes / (attend_avg * 1e-3) / 1e9
    # append, tensor-core items, narrow and wide decode items, merge
    launches_per_layer = (1 + (info["prefill_items"] > 0) + (info["decode_items"] > info["wide_decode_items"])
                          + (info["wide_decode_items"] > 0) + info["merge_launch"])
    result = {
        "metric": "decode attend KV GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == 0 else "e4m3 KV, bf16 Q/O",
        "data": "synthetic",
        "config": decode_config(args, w, world),
        "rows_per_s": world * n_rows / (ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (+merge) per pie_attend",
                     "achieved": achieved, "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": traffic(f"decode_kernel {w.name}", ["decode.cu", "ptx.cuh"], attend_bytes),
                     "algorithmic_bytes_per_launch": attend_bytes, "avg_launch_ms": attend_avg},
        "append": append_roofline(append_bytes, append_avg, hbm_peak, peak_src,
                                  "kv_append_rope" if args.rope_theta else
                                  ("kv_append_bf16" if w.kv_dtype == 0 else "kv_append_e4m3")),
        "e2e": e2e_res,
        "gpu_launches": args.steps * L * launches_per_layer,
        "clocks": clk,
    }
    pie.pie_ctx_destroy(ctx)
    return result


def run_fork(args, world, rank, local):
    """Fork / speculative decoding: a 4096-token prompt forked into 10 working
    sets, each with its own frozen suffix, then one pass of 4 draft tokens per
    fork (40 query rows, causal among each fork's drafts), every layer, rolled
    back after each step.  The shared prompt pages are read once per pass; the
    line also reports what the same reads would cost if every fork read the
    prompt itself."""
    import torch

    from paged_kv_attention_working_gb300 import pie
    from paged_kv_attention_working_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    L = args.layers
    w = wl.fork_spec(num_layers=L, unshared=False)
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    pool_bytes = L * w.num_pages * Hkv * 16 * D * 2
    kpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    vpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    ctx = pie.pie_ctx_create(L, Hq, Hkv, D, w.num_pages, free_list=w.free_list().tolist(), k_pool=kpool,
                             v_pool=vpool, stream=stream.cuda_stream, logit_softcap=args.logit_softcap)
    pie.pie_ctx_set_merge_mode(ctx, args.merge_mode)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000 + rank)
    hs = {}
    first_attend = min(i for i, op in enumerate(w.ops) if op[0] == "pass" and op[2])
    for op in w.ops[:first_attend]:
        if op[0] == "create":
            hs[op[1]] = pie.pie_ws_create(ctx)
        elif op[0] == "fork":
            hs[op[2]] = pie.pie_ws_fork(ctx, hs[op[1]])
        elif op[0] == "freeze":
            pie.pie_ws_freeze(ctx, hs[op[1]], op[2])
        elif op[0] == "pass":
            b = pie.pie_batch_begin(ctx, [(hs[sg[0]], sg[1], None) for sg in op[1]])
            n = pie.pie_batch_rows(b)
            for layer in range(L):
                k = torch.randn((n, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
                pie.pie_kv_append(ctx, b, layer, k, k)
            pie.pie_batch_end(ctx, b)
    segs = [(hs[sg[0]], sg[1], None) for sg in w.ops[first_attend][1]]
    drafts = segs[0][1]
    rows = sum(sg[1] for sg in segs)
    q = torch.randn((L, rows, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
    kv = torch.randn((L, rows, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty((L, rows, Hq, D), dtype=torch.bfloat16, device=dev)
    prompt = w.kv_streams["prompt"]
    # keys read per layer: the shared prompt once, each fork's suffix and
    # drafts (every draft row sees the drafts before it; the bytes count each
    # key once per fork)
    private = sum(s + drafts for s in w.suffix)
    kv_bytes_layer = (prompt + private) * Hkv * D * 2 * 2
    unshared_layer = (len(segs) * prompt + private) * Hkv * D * 2 * 2

    # The layers' device pointers are taken once, as a caller of the C
    # functions holds them: indexing a torch tensor costs a few microseconds
    # of host time per call on a GB300 node's Arm cores, and with four of
    # them per layer the pass (about 20 us of GPU time per layer) waited on
    # the host instead of the GPU.
    ptrs = [(kv[layer].data_ptr(), q[layer].data_ptr(), out[layer].data_ptr()) for layer in range(L)]

    def step(ev=None):
        bb = pie.pie_batch_begin(ctx, segs)
        info.update(pie.pie_batch_plan_info(bb))
        for layer, (kvp, qp, outp) in enumerate(ptrs):
            if ev is not None:
                ev[layer][0].record(stream)
            pie.pie_kv_append(ctx, bb, layer, kvp, kvp)
            if ev is not None:
                ev[layer][1].record(stream)
            pie.pie_attend(ctx, bb, layer, qp, outp)
            if ev is not None:
                ev[layer][2].record(stream)
        pie.pie_batch_end(ctx, bb)
        for sg in segs:
            pie.pie_ws_rollback(ctx, sg[0], drafts)

    info = {}
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = Clocks(local)
    clocks.start()
    wall0 = time.time()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    ms = allmax(world, t0.elapsed_time(t1) / args.steps)
    assert pie.pie_ctx_check(ctx) == 0
    # the per-layer split, from separately timed steps (events between the
    # calls add a little time of their own, so these are not the step time)
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
              for _ in range(min(args.steps, 10))]
    for ev in events:
        step(ev)
    torch.cuda.synchronize(dev)
    append_us = 1e3 * statistics.mean(e0.elapsed_time(e1) for st in events for e0, e1, _ in st)
    attend_us = 1e3 * statistics.mean(e1.elapsed_time(e2) for st in events for _, e1, e2 in st)
    hbm, src = peaks()
    value = world * kv_bytes_layer * L / (ms * 1e-3) / 1e9
    res = {"metric": "fork decode attend KV GB/s (shared prompt read once per pass)", "value": value, "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": "fork_spec", "prompt": prompt, "forks": len(segs), "drafts": drafts,
                      "suffix_tokens": w.suffix, "layers": L, "hq": Hq, "hkv": Hkv, "head_dim": D,
                      "l2": "32 layers of K/V (about 0.7 GB per step), larger than L2"},
           "clocks": clk,
           "rows_per_s": world * rows / (ms * 1e-3),
           "unshared_equivalent_GBps": world * unshared_layer * L / (ms * 1e-3) / 1e9,
           "per_layer_us": {"pass": 1e3 * ms / L, "append": append_us, "attend": attend_us},
           "plan": info,
           "roofline": {"bound": "hbm", "kernel": "whole fork pass (append, shared prompt once per pass, "
                                                  "private suffixes and drafts, merge)",
                        "achieved": value, "peak": hbm, "peak_source": src, "unit": "GB/s", "frac": value / hbm,
                        "traffic": None, "algorithmic_bytes_per_layer": kv_bytes_layer}}
    pie.pie_ctx_destroy(ctx)
    return res


def run_mixed(args, w, world, rank, local):
    """Mixed continuous batch (16 prefill chunks + 128 decode rows, one
    pie_attend): times the whole step, and the chunks alone (the tensor-core
    prefill kernel alone, every row written directly) for its TFLOP/s."""
    import torch

    from paged_kv_attention_working_gb300 import pie

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    esize = 2 if w.kv_dtype == 0 else 1
    block = 16 * D * esize
    pool_bytes = w.num_layers * w.num_pages * Hkv * block
    kpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    vpool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
    ks, vs = w.scales()
    ctx = pie.pie_ctx_create(w.num_layers, Hq, Hkv, D, w.num_pages, kv_dtype=w.kv_dtype,
                             free_list=w.free_list().tolist(), k_scale=ks, v_scale=vs,
                             k_pool=kpool, v_pool=vpool, stream=stream.cuda_stream,
                             logit_softcap=args.logit_softcap)
    pie.pie_ctx_set_merge_mode(ctx, args.merge_mode)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + rank)
    hs = {}
    for op in w.ops:
        if op[0] == "create":
            hs[op[1]] = pie.pie_ws_create(ctx)
    fill = [op for op in w.ops if op[0] == "pass"][0][1]
    main_segs = [op for op in w.ops if op[0] == "pass"][1][1]
    b = pie.pie_batch_begin(ctx, [(hs[s[0]], s[1], None) for s in fill])
    n = pie.pie_batch_rows(b)
    k = torch.randn((n, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
    pie.pie_kv_append(ctx, b, 0, k, k)
    pie.pie_batch_end(ctx, b)
    del k
    for name in hs:
        pie.pie_ws_freeze(ctx, hs[name], -1)

    def make(segs):
        rows = sum(s[1] for s in segs)
        q = torch.randn((rows, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
        kv = torch.randn((rows, Hkv, D), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((rows, Hq, D), dtype=torch.bfloat16, device=dev)
        return q, kv, out

    chunk_segs = [s for s in main_segs if s[0].startswith("c")]
    flops = prefill_chunk_flops(w, chunk_segs)
    dec_keys = sum(c + 1 for c in w.decode_ctx)

    # written before every timed attend so that no K/V stays in L2 (129 MB)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(segs, tensors, steps):
        """Median event-timed attend and append of `steps` passes, L2 flushed
        before each."""
        q, kv, out = tensors
        evs = []
        for i in range(args.warmup + steps):
            bb = pie.pie_batch_begin(ctx, [(hs[s[0]], s[1], None) for s in segs])
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            flush.zero_()
            e[2].record(stream)
            pie.pie_kv_append(ctx, bb, 0, kv, kv)
            e[3].record(stream)
            flush.zero_()
            e[0].record(stream)
            pie.pie_attend(ctx, bb, 0, q, out)
            e[1].record(stream)
            pie.pie_batch_end(ctx, bb)
            for s in segs:
                pie.pie_ws_rollback(ctx, hs[s[0]], s[1])
            if i >= args.warmup:
                evs.append(e)
        torch.cuda.synchronize(dev)
        assert pie.pie_ctx_check(ctx) == 0
        return (statistics.median(e[0].elapsed_time(e[1]) for e in evs),
                statistics.median(e[2].elapsed_time(e[3]) for e in evs))

    clocks = Clocks(local)
    clocks.start()
    wall0 = time.time()
    t_chunks, _ = timed(chunk_segs, make(chunk_segs), args.steps)
    t_mixed, t_append = timed(main_segs, make(main_segs), args.steps)
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    # K/V bytes one attend reads (each key once per working set)
    chunk_kv = sum(c0 + s[1] for s, c0 in zip(chunk_segs, w.chunk_ctx)) * Hkv * D * esize * 2
    tflops = flops / (t_chunks * 1e-3) / 1e12
    peak, src = tensor_peak()
    hbm, hsrc = peaks()
    mixed_rows = sum(s[1] for s in main_segs)
    res = {"metric": "prefill attend TFLOP/s (causal-exact flops)", "value": tflops, "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_mixed,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16" if w.kv_dtype == 0 else "e4m3 KV as f16 operands, f16 Q/P, fp32 accumulate",
           "data": "synthetic",
           "config": {"workload": w.name, "kv_dtype": "bf16" if w.kv_dtype == 0 else "e4m3",
                      "logit_softcap": args.logit_softcap,
                      "chunks": len(chunk_segs), "chunk_rows": sum(s[1] for s in chunk_segs),
                      "decode_rows": len(w.decode_ctx), "hq": Hq, "hkv": Hkv, "head_dim": D, "layers": 1,
                      "l2": f"flushed (256 MB written) before each timed attend; the chunks read "
                            f"{chunk_kv / 1e6:.0f} MB of K/V per attend and the whole step "
                            f"{(chunk_kv + dec_keys * Hkv * D * esize * 2) / 1e6:.0f} MB"},
           "clocks": clk,
           "roofline": {"bound": "tensor", "kernel": "prefill_kernel (chunks-only attend)", "achieved": tflops,
                        "peak": peak, "peak_source": src, "unit": "TFLOP/s", "frac": tflops / peak,
                        "traffic": traffic(f"prefill_kernel {w.name}", ["prefill.cu", "ptx.cuh", "tcgen05.cuh"],
                                           flops),
                        "flops_per_launch": flops, "avg_launch_ms": t_chunks},
           "mixed_step": {"attend_ms": t_mixed, "rows": mixed_rows,
                          "rows_per_s": mixed_rows / (t_mixed * 1e-3),
                          "decode_kv_bytes": dec_keys * Hkv * D * esize * 2},
           "append": append_roofline(mixed_rows * Hkv * D * (2 + esize) * 2, t_append, hbm, hsrc,
                                     "kv_append_bf16" if w.kv_dtype == 0 else "kv_append_e4m3")}
    pie.pie_ctx_destroy(ctx)
    return res


def slim(res):
    """A leg's result as a sub-object of the headline line (the keys the
    headline already states are dropped)."""
    drop = ("n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data")
    return {k: v for k, v in res.items() if k not in drop}


def other_workloads(args, world, rank, local):
    """The fork pass, the mixed batch (bf16 and e4m3 KV) and the 70B-shaped
    FP8 decode, one after the other, each with its own timing and clocks."""
    import torch

    from paged_kv_attention_working_gb300 import workloads as wl

    out = {}
    out["fork_spec"] = run_fork(args, world, rank, local)
    torch.cuda.empty_cache()
    for name, kv in (("mixed_batch", wl.KV_BF16), ("mixed_batch_e4m3", wl.KV_E4M3)):
        out[name] = run_mixed(args, wl.mixed_batch(name=name, kv_dtype=kv), world, rank, local)
        torch.cuda.empty_cache()
    out["llama70b_fp8"] = run_gpu(args, llama70b_workload(256), world, rank, local, e2e=False)
    torch.cuda.empty_cache()
    return {k: slim(v) for k, v in out.items()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-seconds", type=float, default=20.0,
                    help="CPU seconds of oracle work (whole reference run, or the cpu_baseline sample)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="llama8b_decode",
                    choices=["llama8b_decode", "mixed_batch", "mixed_batch_e4m3", "llama70b_fp8", "fork_spec"])
    ap.add_argument("--n-ws", type=int, default=0,
                    help="working sets of the e4m3 workload (0 = the full 256; fewer only for profiling)")
    ap.add_argument("--logit-softcap", type=float, default=0.0,
                    help="logit soft cap c of the attention scores (0 = none)")
    ap.add_argument("--rope-theta", type=float, default=0.0,
                    help="rotary base: K and Q rotated in the append (pie_kv_append_rope); 0 = plain append")
    ap.add_argument("--layers", type=int, default=32,
                    help="layers of the workload (32 = the full Llama-3.1-8B shape; fewer only for profiling)")
    ap.add_argument("--merge-mode", type=int, default=0, choices=[0, 1],
                    help="how split rows are combined (pie_ctx_set_merge_mode): 0 = a merge launch, "
                         "1 = inside the decode launches when no tensor-core item is split")
    ap.add_argument("--only-headline", action="store_true",
                    help="time the headline workload alone (no fork / mixed / 70B sub-objects)")
    args = ap.parse_args()
    from paged_kv_attention_working_gb300 import workloads as wl

    world, rank, local = dist_init()
    if args.workload == "fork_spec":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the decode workloads; "
                                  "the fork pass is timed on the GPU only"}), flush=True)
            return
        res = run_fork(args, world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.workload.startswith("mixed_batch"):
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the decode workloads; "
                                  "the mixed batch is timed on the GPU only"}), flush=True)
            return
        kv = wl.KV_E4M3 if args.workload.endswith("e4m3") else wl.KV_BF16
        res = run_mixed(args, wl.mixed_batch(name=args.workload, kv_dtype=kv), world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.workload == "llama70b_fp8":
        w = llama70b_workload(args.n_ws or 256)
    else:
        w = wl.llama8b_decode(num_layers=args.layers)
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return
    result = run_gpu(args, w, world, rank, local)
    if args.workload == "llama8b_decode" and not args.only_headline:
        import torch

        torch.cuda.empty_cache()
        result["workloads"] = other_workloads(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            gbs, rps, desc, cores, _ = OracleSample(w).run(args.ref_seconds)
            result["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                      "sample": desc, "rows_per_s": rps}
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
