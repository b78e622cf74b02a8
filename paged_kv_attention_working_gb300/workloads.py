"""Seeded synthetic workloads for paged-KV attention over working sets.

This module makes INPUTS only: working-set shapes, operation scripts, token
ids, free-page orders, FP8 scales and bf16 query/key/value draws.  It holds
none of the attention or allocator arithmetic, and it is the only code that
both the CPU oracle's tests and the CUDA path's tests and benchmark share.

Value recipe: numpy ``PCG64`` seeded by a ``SeedSequence`` of
(workload seed, stream id, layer, K/V/Q), fp32 draws of N(0, 1) rounded to
bf16 (round to nearest even).  Token ids are uniform in [0, 128256) (the
Llama 3 vocabulary size in "Write a model in Poem", section 1).  The free-page
order is a seeded permutation.  FP8 scales are per (layer, KV head):
``(4 + u) / 448`` with u uniform in [0, 1), so that about 4 to 5 standard
deviations map to the largest E4M3 value.

A workload is a list of operations on named working sets:

    ("create", name)                 ("fork", parent, name)
    ("freeze", name, n)              ("rollback", name, n)
    ("match", name, token_stream)    ("destroy", name)
    ("pass", segs, attend)

where each seg of a pass is ``(name, n_new, kv_pieces, q_pieces, tok_pieces)``
and a piece is ``(stream, start, count)``: the K/V (or Q, or token ids) of a
segment are the concatenation of slices of named streams, so that forks and
their unshared copies, or a rollback and its re-append, feed the same values.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

KV_BF16 = 0
KV_E4M3 = 1
VOCAB = 128256


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _stream_id(name: str) -> int:
    return int.from_bytes(hashlib.sha256(name.encode()).digest()[:4], "little")


def rng_for(seed: int, *key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


@dataclass
class Workload:
    name: str
    seed: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: int
    num_pages: int
    ops: list
    kv_streams: dict = field(default_factory=dict)     # name -> length
    q_streams: dict = field(default_factory=dict)      # name -> length
    tok_streams: dict = field(default_factory=dict)    # name -> length
    page_size: int = 16
    logit_softcap: float = 0.0     # > 0: scores capped at c * tanh(s / c)
    rope_theta: float = 0.0        # > 0: K (and Q) rotated by position before the append
    rope_positions: int = 0        # positions the rotary table covers
    _cache: dict = field(default_factory=dict, repr=False)

    # --------------------------------------------------------------- inputs
    def free_list(self) -> np.ndarray:
        return rng_for(self.seed, 100).permutation(self.num_pages).astype(np.int32)

    def scales(self):
        if self.kv_dtype != KV_E4M3:
            return None, None
        r = rng_for(self.seed, 200)
        shape = (self.num_layers, self.num_kv_heads)
        k = ((4.0 + r.random(shape)) / 448.0).astype(np.float32)
        v = ((4.0 + r.random(shape)) / 448.0).astype(np.float32)
        return k, v

    def kv_stream(self, name: str, layer: int):
        """(K, V) bf16 bits, each [length, Hkv, d]."""
        key = ("kv", name, layer)
        if key not in self._cache:
            n = self.kv_streams[name]
            shape = (n, self.num_kv_heads, self.head_dim)
            sid = _stream_id(name)
            k = bf16_round(rng_for(self.seed, sid, layer, 0).standard_normal(shape, dtype=np.float32))
            v = bf16_round(rng_for(self.seed, sid, layer, 1).standard_normal(shape, dtype=np.float32))
            self._cache[key] = (k, v)
        return self._cache[key]

    def q_stream(self, name: str, layer: int) -> np.ndarray:
        key = ("q", name, layer)
        if key not in self._cache:
            n = self.q_streams[name]
            shape = (n, self.num_q_heads, self.head_dim)
            r = rng_for(self.seed, _stream_id(name), layer, 2)
            self._cache[key] = bf16_round(r.standard_normal(shape, dtype=np.float32))
        return self._cache[key]

    def tok_stream(self, name: str) -> np.ndarray:
        key = ("tok", name)
        if key not in self._cache:
            r = rng_for(self.seed, _stream_id(name), 3)
            self._cache[key] = r.integers(0, VOCAB, self.tok_streams[name]).astype(np.int32)
        return self._cache[key]

    def gather_kv(self, pieces, layer: int):
        ks, vs = [], []
        for stream, start, count in pieces:
            k, v = self.kv_stream(stream, layer)
            ks.append(k[start:start + count])
            vs.append(v[start:start + count])
        return np.concatenate(ks), np.concatenate(vs)

    def gather_q(self, pieces, layer: int) -> np.ndarray:
        return np.concatenate([self.q_stream(s, layer)[a:a + c] for s, a, c in pieces])

    def gather_tok(self, pieces):
        if pieces is None:
            return None
        return np.concatenate([self.tok_stream(s)[a:a + c] for s, a, c in pieces])

    def pass_inputs(self, segs, layer: int, attend: bool):
        """Concatenated K, V (and Q) bf16 bits of a pass, in segment order."""
        live = [s for s in segs if s[1] > 0]
        k, v = zip(*(self.gather_kv(s[2], layer) for s in live)) if live else ((), ())
        kk = np.concatenate(k) if k else np.zeros((0, self.num_kv_heads, self.head_dim), np.uint16)
        vv = np.concatenate(v) if v else np.zeros((0, self.num_kv_heads, self.head_dim), np.uint16)
        q = None
        if attend:
            qs = [self.gather_q(s[3], layer) for s in live]
            q = np.concatenate(qs) if qs else np.zeros((0, self.num_q_heads, self.head_dim), np.uint16)
        return kk, vv, q


def _pages_for(lengths, page_size=16):
    return int(sum(-(-n // page_size) for n in lengths))


# ---------------------------------------------------------------- builders
def tiny_decode() -> Workload:
    """4 working sets, contexts {17, 33, 64, 100}; 8 query / 2 KV heads, d 64;
    one layer; one decode token each, appended then attended."""
    ctx = [17, 33, 64, 100]
    ops = []
    w = Workload("tiny_decode", 1, 1, 8, 2, 64, KV_BF16, 40, ops)
    for i, n in enumerate(ctx):
        ops.append(("create", f"w{i}"))
        w.kv_streams[f"ctx{i}"] = n + 1
        w.q_streams[f"q{i}"] = 1
    ops.append(("pass", [(f"w{i}", n, [(f"ctx{i}", 0, n)], None, None) for i, n in enumerate(ctx)], False))
    ops += [("freeze", f"w{i}", -1) for i in range(len(ctx))]
    ops.append(("pass", [(f"w{i}", 1, [(f"ctx{i}", n, 1)], [(f"q{i}", 0, 1)], None)
                         for i, n in enumerate(ctx)], True))
    return w


def decode_batch(name="llama8b_decode", seed=2, n_ws=64, ctx_lo=512, ctx_hi=8192,
                 num_layers=32, hq=32, hkv=8, d=128, kv_dtype=KV_BF16,
                 prefix_groups=0, prefix_len=0, slack_pages=64) -> Workload:
    """Decode batch: n_ws working sets with contexts uniform in [ctx_lo, ctx_hi];
    one new token each.  With prefix_groups > 0 the sets form that many equal
    groups; in each, the first member writes and freezes a shared prefix of
    prefix_len tokens (with token ids) and the others take it by match_prefix."""
    r = rng_for(seed, 0)
    ctx = r.integers(ctx_lo, ctx_hi + 1, n_ws).tolist()
    ops = []
    w = Workload(name, seed, num_layers, hq, hkv, d, kv_dtype, 0, ops)
    gsize = n_ws // prefix_groups if prefix_groups else 0
    for i in range(n_ws):
        ops.append(("create", f"w{i}"))
        w.q_streams[f"q{i}"] = 1
    fill = []
    if prefix_groups:
        first = []
        for g in range(prefix_groups):
            w.kv_streams[f"pre{g}"] = prefix_len
            w.tok_streams[f"pretok{g}"] = prefix_len
            first.append((f"w{g * gsize}", prefix_len, [(f"pre{g}", 0, prefix_len)], None,
                          [(f"pretok{g}", 0, prefix_len)]))
        ops.append(("pass", first, False))
        ops += [("freeze", f"w{g * gsize}", -1) for g in range(prefix_groups)]
        for i in range(n_ws):
            if i % gsize:
                ops.append(("match", f"w{i}", f"pretok{i // gsize}"))
    for i in range(n_ws):
        own = ctx[i] - (prefix_len if prefix_groups else 0)
        w.kv_streams[f"ctx{i}"] = own + 1
        if own > 0:
            fill.append((f"w{i}", own, [(f"ctx{i}", 0, own)], None, None))
    ops.append(("pass", fill, False))
    ops += [("freeze", f"w{i}", -1) for i in range(n_ws)]
    own = [c - (prefix_len if prefix_groups else 0) for c in ctx]
    ops.append(("pass", [(f"w{i}", 1, [(f"ctx{i}", own[i], 1)], [(f"q{i}", 0, 1)], None)
                         for i in range(n_ws)], True))
    unique = _pages_for([c + 1 for c in ctx])
    if prefix_groups:
        unique -= (n_ws - prefix_groups) * (prefix_len // 16)
    w.num_pages = unique + slack_pages
    w.ctx = ctx
    w.ctx_range = (ctx_lo, ctx_hi)
    return w


def llama8b_decode(**kw) -> Workload:
    """Llama-3.1-8B-shaped decode batch: 32 q / 8 KV heads, d 128, bf16,
    64 working sets with contexts uniform in [512, 8192], 32 layers."""
    return decode_batch(**kw)


def llama70b_fp8(**kw) -> Workload:
    """Llama-3.3-70B-shaped long-context decode with e4m3 KV: 64 q / 8 KV
    heads, d 128, 256 working sets with contexts uniform in [2048, 32768],
    groups of 8 sharing a deduplicated 2048-token prefix; one layer."""
    args = dict(name="llama70b_fp8", seed=5, n_ws=256, ctx_lo=2048, ctx_hi=32768,
                num_layers=1, hq=64, hkv=8, d=128, kv_dtype=KV_E4M3,
                prefix_groups=32, prefix_len=2048)
    args.update(kw)
    return decode_batch(**args)


def fork_spec(name="fork_spec", seed=3, prompt=4096, n_forks=10, suffix_hi=256, drafts=4,
              rollback=2, num_layers=1, hq=32, hkv=8, d=128, unshared=True, kv_dtype=KV_BF16) -> Workload:
    """One frozen prompt forked into n_forks working sets; each adds a frozen
    suffix of 1..suffix_hi tokens and `drafts` speculative tokens that are
    attended causally; then `rollback` drafts are dropped and re-appended
    with the same values and attended again.  With `unshared`, the same
    tokens are also built as independent copies that share nothing."""
    r = rng_for(seed, 0)
    suffix = r.integers(1, suffix_hi + 1, n_forks).tolist()
    ops = []
    w = Workload(name, seed, num_layers, hq, hkv, d, kv_dtype, 0, ops)
    w.kv_streams["prompt"] = prompt
    for i in range(n_forks):
        w.kv_streams[f"suf{i}"] = suffix[i]
        w.kv_streams[f"draft{i}"] = drafts
        w.q_streams[f"dq{i}"] = drafts
    ops.append(("create", "root"))
    ops.append(("pass", [("root", prompt, [("prompt", 0, prompt)], None, None)], False))
    ops.append(("freeze", "root", -1))
    names = [f"f{i}" for i in range(n_forks)]
    for n in names:
        ops.append(("fork", "root", n))
    ops.append(("pass", [(names[i], suffix[i], [(f"suf{i}", 0, suffix[i])], None, None)
                         for i in range(n_forks)], False))
    ops += [("freeze", n, -1) for n in names]
    ops.append(("pass", [(names[i], drafts, [(f"draft{i}", 0, drafts)], [(f"dq{i}", 0, drafts)], None)
                         for i in range(n_forks)], True))
    ops += [("rollback", n, rollback) for n in names]
    keep = drafts - rollback
    ops.append(("pass", [(names[i], rollback, [(f"draft{i}", keep, rollback)],
                          [(f"dq{i}", keep, rollback)], None) for i in range(n_forks)], True))
    pages = _pages_for([prompt]) + _pages_for([prompt + s + drafts for s in suffix]) - n_forks * (prompt // 16)
    if unshared:
        copies = [f"u{i}" for i in range(n_forks)]
        ops += [("create", c) for c in copies]
        ops.append(("pass", [(copies[i], prompt + suffix[i],
                              [("prompt", 0, prompt), (f"suf{i}", 0, suffix[i])], None, None)
                             for i in range(n_forks)], False))
        ops += [("freeze", c, -1) for c in copies]
        ops.append(("pass", [(copies[i], drafts, [(f"draft{i}", 0, drafts)], [(f"dq{i}", 0, drafts)], None)
                             for i in range(n_forks)], True))
        pages += _pages_for([prompt + s + drafts for s in suffix])
    w.num_pages = pages + n_forks * 2 + 16
    w.suffix = suffix
    return w


def nested_fork(name="nested_fork", seed=60, prompt=300, n_forks=4, sub_suffix=70, n_sub=4, suffix_hi=40,
                drafts=4, num_layers=1, hq=32, hkv=8, d=128, kv_dtype=KV_BF16) -> Workload:
    """A fork of a fork: a frozen prompt forked into n_forks working sets;
    the first fork freezes a suffix of sub_suffix tokens and is forked again
    into n_sub working sets.  Every leaf (the other forks and the sub-forks)
    then freezes its own suffix of 1..suffix_hi tokens and attends a pass of
    `drafts` speculative tokens.  The prompt is shared by every leaf; the
    first fork's suffix by the sub-forks only."""
    r = rng_for(seed, 0)
    leaves = [f"a{i}" for i in range(1, n_forks)] + [f"b{i}" for i in range(n_sub)]
    suffix = dict(zip(leaves, r.integers(1, suffix_hi + 1, len(leaves)).tolist()))
    ops = []
    w = Workload(name, seed, num_layers, hq, hkv, d, kv_dtype, 0, ops)
    w.kv_streams["prompt"] = prompt
    w.kv_streams["a0suf"] = sub_suffix
    ops.append(("create", "root"))
    ops.append(("pass", [("root", prompt, [("prompt", 0, prompt)], None, None)], False))
    ops.append(("freeze", "root", -1))
    ops += [("fork", "root", f"a{i}") for i in range(n_forks)]
    ops.append(("pass", [("a0", sub_suffix, [("a0suf", 0, sub_suffix)], None, None)], False))
    ops.append(("freeze", "a0", -1))
    ops += [("fork", "a0", f"b{i}") for i in range(n_sub)]
    for n in leaves:
        w.kv_streams[f"suf_{n}"] = suffix[n]
        w.kv_streams[f"draft_{n}"] = drafts
        w.q_streams[f"dq_{n}"] = drafts
    ops.append(("pass", [(n, suffix[n], [(f"suf_{n}", 0, suffix[n])], None, None) for n in leaves], False))
    ops += [("freeze", n, -1) for n in leaves]
    ops.append(("pass", [(n, drafts, [(f"draft_{n}", 0, drafts)], [(f"dq_{n}", 0, drafts)], None) for n in leaves],
                True))
    w.num_pages = (_pages_for([prompt]) + _pages_for([prompt + sub_suffix])
                   + _pages_for([prompt + sub_suffix + suffix[n] + drafts for n in leaves]) + 32)
    w.suffix = suffix
    return w


def interleaved_forks(name="interleaved_forks", seed=70, prompt_a=300, prompt_b=200, n_forks=3, drafts_a=8,
                      drafts_b=2, suffix_hi=40, num_layers=1, hq=32, hkv=8, d=128, kv_dtype=KV_BF16) -> Workload:
    """Two frozen prompts, each forked into n_forks working sets that freeze
    their own suffixes of 1..suffix_hi tokens; the drafts pass then lists the
    forks alternately (a0, b0, a1, b1, ...), so neither fork group's rows are
    consecutive batch rows.  Group a (n_forks x drafts_a rows) is sized for
    the tensor-core kernel, group b (n_forks x drafts_b rows) for the decode
    kernel's shared items."""
    r = rng_for(seed, 0)
    a = [f"a{i}" for i in range(n_forks)]
    b = [f"b{i}" for i in range(n_forks)]
    leaves = [x for pair in zip(a, b) for x in pair]
    suffix = dict(zip(leaves, r.integers(1, suffix_hi + 1, len(leaves)).tolist()))
    drafts = {n: (drafts_a if n in a else drafts_b) for n in leaves}
    ops = []
    w = Workload(name, seed, num_layers, hq, hkv, d, kv_dtype, 0, ops)
    for root, n_tok in (("pa", prompt_a), ("pb", prompt_b)):
        w.kv_streams[root] = n_tok
        ops.append(("create", root))
        ops.append(("pass", [(root, n_tok, [(root, 0, n_tok)], None, None)], False))
        ops.append(("freeze", root, -1))
    ops += [("fork", "pa", n) for n in a] + [("fork", "pb", n) for n in b]
    for n in leaves:
        w.kv_streams[f"suf_{n}"] = suffix[n]
        w.q_streams[f"sq_{n}"] = suffix[n]
        w.kv_streams[f"draft_{n}"] = drafts[n]
        w.q_streams[f"dq_{n}"] = drafts[n]
    # both passes attend: the suffixes' rows also read their prompt through
    # the groups' own row lists
    ops.append(("pass", [(n, suffix[n], [(f"suf_{n}", 0, suffix[n])], [(f"sq_{n}", 0, suffix[n])], None)
                         for n in leaves], True))
    ops += [("freeze", n, -1) for n in leaves]
    ops.append(("pass", [(n, drafts[n], [(f"draft_{n}", 0, drafts[n])], [(f"dq_{n}", 0, drafts[n])], None)
                         for n in leaves], True))
    w.num_pages = (_pages_for([prompt_a, prompt_b])
                   + _pages_for([(prompt_a if n in a else prompt_b) + suffix[n] + drafts[n] for n in leaves]) + 32)
    w.suffix = suffix
    return w


def mixed_batch(name="mixed_batch", seed=4, n_chunks=16, chunk_lo=512, chunk_hi=2048,
                ctx_lo=0, ctx_hi=4096, n_decode=128, dec_lo=1, dec_hi=4096,
                num_layers=1, hq=32, hkv=8, d=128, kv_dtype=KV_BF16) -> Workload:
    """Mixed continuous batch: n_chunks prefill chunks of chunk_lo..chunk_hi new
    tokens on existing contexts of ctx_lo..ctx_hi tokens, plus n_decode
    single-token rows on contexts of dec_lo..dec_hi tokens, one attend call."""
    r = rng_for(seed, 0)
    chunk = r.integers(chunk_lo, chunk_hi + 1, n_chunks).tolist()
    cctx = r.integers(ctx_lo, ctx_hi + 1, n_chunks).tolist()
    dctx = r.integers(dec_lo, dec_hi + 1, n_decode).tolist()
    ops = []
    w = Workload(name, seed, num_layers, hq, hkv, d, kv_dtype, 0, ops)
    fill, main = [], []
    for i in range(n_chunks):
        ops.append(("create", f"c{i}"))
        w.kv_streams[f"cctx{i}"] = cctx[i] + chunk[i]
        w.q_streams[f"cq{i}"] = chunk[i]
        if cctx[i]:
            fill.append((f"c{i}", cctx[i], [(f"cctx{i}", 0, cctx[i])], None, None))
        main.append((f"c{i}", chunk[i], [(f"cctx{i}", cctx[i], chunk[i])], [(f"cq{i}", 0, chunk[i])], None))
    for i in range(n_decode):
        ops.append(("create", f"d{i}"))
        w.kv_streams[f"dctx{i}"] = dctx[i] + 1
        w.q_streams[f"dq{i}"] = 1
        fill.append((f"d{i}", dctx[i], [(f"dctx{i}", 0, dctx[i])], None, None))
        main.append((f"d{i}", 1, [(f"dctx{i}", dctx[i], 1)], [(f"dq{i}", 0, 1)], None))
    ops.append(("pass", fill, False))
    ops += [("freeze", f"c{i}", -1) for i in range(n_chunks)]
    ops += [("freeze", f"d{i}", -1) for i in range(n_decode)]
    ops.append(("pass", main, True))
    w.num_pages = _pages_for([a + b for a, b in zip(cctx, chunk)]) + _pages_for([c + 1 for c in dctx]) + 32
    w.chunks, w.chunk_ctx, w.decode_ctx = chunk, cctx, dctx
    return w


def edge_batch(name="edge_batch", seed=30, kv_dtype=KV_BF16, hq=32, hkv=8, d=128,
               chunks=((1, 0), (16, 0), (17, 15), (255, 1), (256, 16), (257, 4095), (128, 128), (2, 4094)),
               decodes=(0, 1, 15, 16, 17, 127, 128, 129), idle_ctx=40) -> Workload:
    """One pass of ragged edges: prefill chunks of (new tokens, context) at
    page (16) and row-tile boundaries, single-token rows on contexts around
    page and key-tile (128) boundaries -- context 0 sees only its own key --
    and a working set in the pass with no new tokens."""
    ops = []
    w = Workload(name, seed, 1, hq, hkv, d, kv_dtype, 0, ops)
    fill, main = [], []
    lengths = []
    for i, (n, c) in enumerate(chunks):
        ops.append(("create", f"c{i}"))
        w.kv_streams[f"cctx{i}"] = c + n
        w.q_streams[f"cq{i}"] = n
        if c:
            fill.append((f"c{i}", c, [(f"cctx{i}", 0, c)], None, None))
        main.append((f"c{i}", n, [(f"cctx{i}", c, n)], [(f"cq{i}", 0, n)], None))
        lengths.append(c + n)
    for i, c in enumerate(decodes):
        ops.append(("create", f"d{i}"))
        w.kv_streams[f"dctx{i}"] = c + 1
        w.q_streams[f"dq{i}"] = 1
        if c:
            fill.append((f"d{i}", c, [(f"dctx{i}", 0, c)], None, None))
        main.append((f"d{i}", 1, [(f"dctx{i}", c, 1)], [(f"dq{i}", 0, 1)], None))
        lengths.append(c + 1)
    ops.append(("create", "idle"))
    w.kv_streams["idle"] = idle_ctx
    fill.append(("idle", idle_ctx, [("idle", 0, idle_ctx)], None, None))
    main.append(("idle", 0, [], [], None))
    lengths.append(idle_ctx)
    ops.append(("pass", fill, False))
    ops += [("freeze", f"c{i}", -1) for i in range(len(chunks))]
    ops += [("freeze", f"d{i}", -1) for i in range(len(decodes))]
    ops.append(("pass", main, True))
    w.num_pages = _pages_for(lengths) + 16
    return w


# The five workloads at full size.  The parity tests also run oracle-sized
# reductions of the decode, fork, mixed and 70B-shaped ones (see reduced),
# plus variants with e4m3 KV, a logit soft cap, the fused rotary embedding
# and other head shapes.
FULL = {
    "tiny_decode": tiny_decode,
    "llama8b_decode": llama8b_decode,
    "fork_spec": fork_spec,
    "mixed_batch": mixed_batch,
    "llama70b_fp8": llama70b_fp8,
}

# Reduced-only variants: the same structure with e4m3 KV, and with a logit
# soft cap of 3 (small enough that the cap bends N(0,1) scores visibly).
# Variants with the rotary embedding fused into the append (Llama-3 base
# 500000) take the same inputs rotated by position.
EXTRA = ("fork_spec_e4m3", "mixed_batch_e4m3", "mixed_batch_softcap", "mixed_batch_e4m3_softcap",
         "llama70b_fp8_softcap", "tiny_decode_softcap", "fork_spec_softcap",
         "mixed_batch_rope", "llama70b_fp8_rope", "fork_spec_rope", "tiny_decode_rope",
         "mixed_batch_d64", "mixed_batch_d64_softcap", "mixed_batch_g8", "mixed_batch_e4m3_g8", "mixed_batch_mha",
         "edge_batch", "edge_batch_e4m3",
         "mixed_batch_g16", "mixed_batch_e4m3_g16", "mixed_batch_mqa_g32", "mixed_batch_mqa_g64",
         "mixed_batch_e4m3_mqa_g64", "mixed_batch_d64_mqa_g16", "fork_spec_g16", "fork_spec_mqa_g32",
         "llama70b_fp8_g16", "llama70b_fp8_mqa_g32", "nested_fork", "nested_fork_e4m3",
         "interleaved_forks", "interleaved_forks_e4m3")
SOFTCAP_TEST = 3.0
ROPE_THETA = 500000.0


def reduced(name: str) -> Workload:
    """Oracle-sized variant of a full workload: same structure and head shapes,
    fewer working sets and shorter contexts, still several pages, splits and
    MMA tiles long with ragged tails."""
    if name.endswith("_rope"):
        w = reduced(name[: -len("_rope")])
        w.name += "_rope"
        w.rope_theta = ROPE_THETA
        w.rope_positions = 16 * w.num_pages
        return w
    if name.endswith("_softcap"):
        w = reduced(name[: -len("_softcap")])
        w.name += "_softcap"
        w.logit_softcap = SOFTCAP_TEST
        return w
    if name == "tiny_decode":
        return tiny_decode()
    if name == "llama8b_decode":
        return decode_batch(name="llama8b_decode_small", seed=12, n_ws=6, ctx_lo=200, ctx_hi=1500,
                            num_layers=2)
    if name == "fork_spec":
        return fork_spec(name="fork_spec_small", seed=13, prompt=600, n_forks=10, suffix_hi=40)
    if name == "mixed_batch":
        return mixed_batch(name="mixed_batch_small", seed=14, n_chunks=3, chunk_lo=100, chunk_hi=300,
                           ctx_lo=0, ctx_hi=400, n_decode=5, dec_lo=1, dec_hi=400)
    if name == "fork_spec_e4m3":
        return fork_spec(name="fork_spec_e4m3_small", seed=16, prompt=600, n_forks=10, suffix_hi=40,
                         kv_dtype=KV_E4M3)
    if name == "mixed_batch_e4m3":
        return mixed_batch(name="mixed_batch_e4m3_small", seed=17, n_chunks=3, chunk_lo=100, chunk_hi=300,
                           ctx_lo=0, ctx_hi=400, n_decode=5, dec_lo=1, dec_hi=400, kv_dtype=KV_E4M3)
    # head shapes beyond the five workloads': d = 64 (both kernels), eight query
    # heads per KV head on the tensor-core kernel, and one (plain multi-head)
    if name == "mixed_batch_d64":
        return mixed_batch(name="mixed_batch_d64_small", seed=19, n_chunks=3, chunk_lo=100, chunk_hi=300,
                           ctx_lo=0, ctx_hi=400, n_decode=5, dec_lo=1, dec_hi=400, hq=8, hkv=2, d=64)
    if name in ("mixed_batch_g8", "mixed_batch_e4m3_g8"):
        e4 = name == "mixed_batch_e4m3_g8"
        return mixed_batch(name=name + "_small", seed=20 + e4, n_chunks=3, chunk_lo=40, chunk_hi=120,
                           ctx_lo=0, ctx_hi=400, n_decode=5, dec_lo=1, dec_hi=400, hq=64, hkv=8, d=128,
                           kv_dtype=KV_E4M3 if e4 else KV_BF16)
    if name == "mixed_batch_mha":
        return mixed_batch(name="mixed_batch_mha_small", seed=22, n_chunks=3, chunk_lo=100, chunk_hi=300,
                           ctx_lo=0, ctx_hi=400, n_decode=5, dec_lo=1, dec_hi=400, hq=8, hkv=8, d=128)
    # larger head groups: G = 16, 32, 64 query heads per KV head, with one KV
    # head (multi-query attention) for G = 32 and 64.  Decode rows then fill
    # 1, 2 or 4 MMA row tiles of the decode kernel, and a tensor-core row
    # tile holds 16, 8 or 4 rows.
    if name in ("mixed_batch_g16", "mixed_batch_e4m3_g16", "mixed_batch_mqa_g32", "mixed_batch_mqa_g64",
                "mixed_batch_e4m3_mqa_g64", "mixed_batch_d64_mqa_g16"):
        hq, hkv, d = {"mixed_batch_g16": (32, 2, 128), "mixed_batch_e4m3_g16": (32, 2, 128),
                      "mixed_batch_mqa_g32": (32, 1, 128), "mixed_batch_mqa_g64": (64, 1, 128),
                      "mixed_batch_e4m3_mqa_g64": (64, 1, 128), "mixed_batch_d64_mqa_g16": (16, 1, 64)}[name]
        e4 = "e4m3" in name
        seed = 40 + sorted(EXTRA).index(name)
        return mixed_batch(name=name + "_small", seed=seed, n_chunks=3, chunk_lo=30, chunk_hi=90,
                           ctx_lo=0, ctx_hi=300, n_decode=5, dec_lo=1, dec_hi=400, hq=hq, hkv=hkv, d=d,
                           kv_dtype=KV_E4M3 if e4 else KV_BF16)
    if name == "fork_spec_g16":
        # shared prompt: 40 rows x 16 heads on the tensor-core kernel (three
        # row tiles); each fork's drafts: 4 x 16 = 64, the decode kernel's
        # largest item
        return fork_spec(name="fork_spec_g16_small", seed=50, prompt=400, n_forks=10, suffix_hi=40,
                         hq=32, hkv=2)
    if name == "fork_spec_mqa_g32":
        # 4 drafts x 32 heads = 128: the forks' private pages also go to the
        # tensor-core kernel
        return fork_spec(name="fork_spec_mqa_g32_small", seed=51, prompt=400, n_forks=10, suffix_hi=40,
                         hq=32, hkv=1)
    if name == "llama70b_fp8_g16":
        # dedup groups of 4 rows x 16 heads = 64 on the decode kernel's shared items
        return decode_batch(name="llama70b_fp8_g16_small", seed=52, n_ws=8, ctx_lo=300, ctx_hi=1200,
                            num_layers=1, hq=32, hkv=2, d=128, kv_dtype=KV_E4M3, prefix_groups=2, prefix_len=160)
    if name == "llama70b_fp8_mqa_g32":
        # dedup groups of 2 rows x 32 heads = 64, one KV head
        return decode_batch(name="llama70b_fp8_mqa_g32_small", seed=53, n_ws=8, ctx_lo=300, ctx_hi=1200,
                            num_layers=1, hq=32, hkv=1, d=128, kv_dtype=KV_E4M3, prefix_groups=4,
                            prefix_len=160)
    if name in ("nested_fork", "nested_fork_e4m3"):
        # the prompt's run: 7 leaves x 4 drafts x 4 heads on the tensor-core
        # kernel; the first fork's suffix: 4 sub-forks x 4 x 4 = 64 on the
        # decode kernel
        return nested_fork(name=name + "_small", seed=60 + (name == "nested_fork_e4m3"),
                           kv_dtype=KV_E4M3 if name.endswith("e4m3") else KV_BF16)
    if name in ("interleaved_forks", "interleaved_forks_e4m3"):
        # two fork groups listed alternately: the first (3 forks x 8 drafts x 4
        # heads = 96) on the tensor-core kernel, the second (3 x 2 x 4 = 24) on
        # the decode kernel, both through their own row lists
        e4 = name.endswith("e4m3")
        return interleaved_forks(name=name + "_small", seed=70 + e4, kv_dtype=KV_E4M3 if e4 else KV_BF16)
    if name == "edge_batch":
        return edge_batch()
    if name == "edge_batch_e4m3":
        return edge_batch(name="edge_batch_e4m3", seed=31, kv_dtype=KV_E4M3)
    if name == "llama70b_fp8":
        return decode_batch(name="llama70b_fp8_small", seed=15, n_ws=8, ctx_lo=300, ctx_hi=1200,
                            num_layers=1, hq=64, hkv=8, d=128, kv_dtype=KV_E4M3,
                            prefix_groups=2, prefix_len=160)
    raise KeyError(name)
