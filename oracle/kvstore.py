"""Working sets over a paged KV store (test infrastructure; see the package docstring).

Follows "How Pie thinks", section 4 "Working sets": a working set holds one
sequence's KV state as a frozen prefix (committed tokens that never change)
plus a writable buffer (uncommitted tokens that may be rolled back); ``fork``
makes a new working set that shares the frozen prefix without copying it;
frozen state is deduplicated across requests so that a working set whose
prefix was already computed reuses those pages.  The KV space itself is one K
and one V region per layer, split by KV head ("Write a model in Poem",
section 4 "State (caches)"), written by ``ops.attn.kv_append`` ("Poem ops").

Where the pages leave a step open this module takes the following readings
(each mirrored, in its own code, by the C++ host core):

* pages hold ``page_size`` consecutive token positions of one working set,
  for every layer and KV head; logical page i holds positions
  [i*page_size, (i+1)*page_size);
* free pages form a LIFO stack; its initial order is an input (the caller
  passes a permutation; the first entry is allocated first); ``alloc`` pops,
  ``release`` pushes;
* a page's reference count is the number of working-set page tables holding
  it; the dedup table holds no reference and drops a page's entry when the
  page is freed;
* ``fork`` gives the child the parent's frozen tokens only: the full frozen
  pages and, if the frozen count is not a page multiple, the partial frozen
  tail page, all shared (refcount + 1);
* a write into a page whose refcount is above 1 first copies it (lazy
  copy-on-write): a fresh page is allocated, the whole page block is copied
  for every layer, head, K and V, and the working set's table points at the
  copy;
* ``freeze(n)`` commits the first n writable tokens (all when n < 0); every
  page that becomes fully frozen, whose token ids are all known, and whose
  predecessor page is registered (or that is page 0) is registered in the
  dedup table under the key (predecessor page id or -1, its token ids),
  unless that key is already present; the key carries the predecessor page,
  so a match is exact and never aliases on a hash collision;
* ``match_prefix`` applies to an empty working set only: it walks full pages
  of the given token ids from the root of the dedup table and shares every
  matched page (the matched tokens become frozen);
* ``rollback(n)`` drops the last n writable tokens (error when n exceeds the
  writable count) and releases emptied pages from the highest logical page
  down; ``destroy`` releases all pages the same way;
* a pass (``begin``) reserves slots segment by segment and, within a segment,
  token by token: the copy-on-write page first (if any), then a fresh page at
  every page boundary; if the free stack cannot cover the whole pass the call
  fails and nothing changes.

Pool byte layout (the contract the CUDA library writes, stated in its header
too): per layer and K/V a ``[num_pages][num_kv_heads][block]`` array of
bytes, ``block = page_size * head_dim * esize``; a block is cut along the
head dimension into panels of 128 bytes per key; panel p occupies bytes
[p*page_size*128, (p+1)*page_size*128); within a panel, key slot s's 16-byte
chunk c is stored at byte ``s*128 + 16*(c ^ (s % 8))``.  bf16 elements are
stored as their two little-endian bytes; e4m3 elements as
``e4m3.quantize(x, scale[layer, kv_head])``.

Parity: bit-exact against the C++ host core (page tables, refcounts, slot
maps) and against the GPU pool bytes.  Pinned by invariants (conservation of
references, LIFO order, writable pages unshared), a hand-worked scenario and
brute-force replay of random operation sequences in the tests.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import e4m3

OK = 0
ERR_INVALID = -1
ERR_BAD_HANDLE = -2
ERR_NO_PAGES = -3
ERR_RANGE = -4
ERR_STATE = -6

KV_BF16 = 0
KV_E4M3 = 1


class OracleError(Exception):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def block_offsets(page_size: int, head_dim: int, esize: int) -> np.ndarray:
    """offsets[s, b]: where byte b of key slot s's head vector lives in a block."""
    row = head_dim * esize
    if row % 128:
        raise OracleError(ERR_INVALID, "head_dim * element size must be a multiple of 128 bytes")
    out = np.empty((page_size, row), dtype=np.int64)
    for s in range(page_size):
        for b in range(row):
            panel, within = divmod(b, 128)
            chunk, byte = divmod(within, 16)
            out[s, b] = panel * page_size * 128 + s * 128 + 16 * (chunk ^ (s % 8)) + byte
    return out


@dataclass
class WorkingSet:
    tokens: list = field(default_factory=list)   # token ids, -1 = unknown
    n_frozen: int = 0
    pages: list = field(default_factory=list)

    @property
    def n_tokens(self) -> int:
        return len(self.tokens)


@dataclass
class Pass:
    """Result of ``begin``: one query row per new token, in segment order."""
    rows_ws: list            # working-set handle of each row
    rows_pos: list           # position of each row
    rows_slot: list          # page * page_size + slot of each row
    cow: list                # (src page, dst page) copies done at begin


class KVStore:
    def __init__(self, num_layers: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, num_pages: int, kv_dtype: int = KV_BF16,
                 page_size: int = 16, free_list=None, k_scale=None, v_scale=None,
                 with_pool: bool = True):
        if num_q_heads % num_kv_heads:
            raise OracleError(ERR_INVALID, "query heads must be a multiple of KV heads")
        self.L, self.Hq, self.Hkv, self.d = num_layers, num_q_heads, num_kv_heads, head_dim
        self.P, self.S, self.kv_dtype = num_pages, page_size, kv_dtype
        self.esize = 2 if kv_dtype == KV_BF16 else 1
        order = list(range(num_pages)) if free_list is None else [int(p) for p in free_list]
        if sorted(order) != list(range(num_pages)):
            raise OracleError(ERR_INVALID, "free list must be a permutation of the pages")
        self.free = list(reversed(order))       # top of the stack = last element
        self.refcount = [0] * num_pages
        self.dedup = {}                          # (parent page, tokens) -> page
        self.page_key = {}                       # page -> its dedup key
        self.ws = {}
        self.next_ws = 1
        if kv_dtype == KV_E4M3:
            self.k_scale = np.asarray(k_scale, dtype=np.float32).reshape(num_layers, num_kv_heads)
            self.v_scale = np.asarray(v_scale, dtype=np.float32).reshape(num_layers, num_kv_heads)
        self.block = page_size * head_dim * self.esize
        self.offsets = block_offsets(page_size, head_dim, self.esize)
        self.pool = None
        if with_pool:
            shape = (2, num_layers, num_pages, num_kv_heads, self.block)
            self.pool = np.zeros(shape, dtype=np.uint8)   # [K|V, layer, page, head, bytes]

    # ---------------------------------------------------------------- pages
    def _alloc(self) -> int:
        page = self.free.pop()
        self.refcount[page] = 1
        return page

    def _release(self, page: int) -> None:
        self.refcount[page] -= 1
        assert self.refcount[page] >= 0
        if self.refcount[page] == 0:
            key = self.page_key.pop(page, None)
            if key is not None:
                del self.dedup[key]
            self.free.append(page)

    def _release_from(self, w: WorkingSet, keep_pages: int) -> None:
        while len(w.pages) > keep_pages:
            self._release(w.pages.pop())

    def _get(self, h: int) -> WorkingSet:
        if h not in self.ws:
            raise OracleError(ERR_BAD_HANDLE, f"no working set {h}")
        return self.ws[h]

    # -------------------------------------------------------- working sets
    def ws_create(self) -> int:
        h = self.next_ws
        self.next_ws += 1
        self.ws[h] = WorkingSet()
        return h

    def ws_destroy(self, h: int) -> None:
        w = self._get(h)
        self._release_from(w, 0)
        del self.ws[h]

    def ws_fork(self, parent: int) -> int:
        p = self._get(parent)
        child = WorkingSet()
        nf = p.n_frozen
        child.tokens = list(p.tokens[:nf])
        child.n_frozen = nf
        child.pages = list(p.pages[:_cdiv(nf, self.S)])
        for page in child.pages:
            self.refcount[page] += 1
        h = self.next_ws
        self.next_ws += 1
        self.ws[h] = child
        return h

    def ws_freeze(self, h: int, n: int = -1) -> None:
        w = self._get(h)
        writable = w.n_tokens - w.n_frozen
        if n < 0:
            n = writable
        if n > writable:
            raise OracleError(ERR_RANGE, "freeze beyond the writable buffer")
        old_full = w.n_frozen // self.S
        w.n_frozen += n
        for i in range(old_full, w.n_frozen // self.S):
            page = w.pages[i]
            toks = tuple(w.tokens[i * self.S:(i + 1) * self.S])
            if page in self.page_key or min(toks) < 0:
                continue
            parent = -1 if i == 0 else w.pages[i - 1]
            if i > 0 and parent not in self.page_key:
                continue
            key = (parent, toks)
            if key not in self.dedup:
                self.dedup[key] = page
                self.page_key[page] = key

    def ws_rollback(self, h: int, n: int) -> None:
        w = self._get(h)
        if n < 0 or n > w.n_tokens - w.n_frozen:
            raise OracleError(ERR_RANGE, "rollback beyond the writable buffer")
        del w.tokens[w.n_tokens - n:]
        self._release_from(w, _cdiv(w.n_tokens, self.S))

    def ws_match_prefix(self, h: int, token_ids) -> int:
        w = self._get(h)
        if w.n_tokens:
            raise OracleError(ERR_STATE, "match_prefix needs an empty working set")
        toks = [int(t) for t in token_ids]
        parent = -1
        matched = 0
        while (matched + 1) * self.S <= len(toks):
            key = (parent, tuple(toks[matched * self.S:(matched + 1) * self.S]))
            page = self.dedup.get(key)
            if page is None:
                break
            w.pages.append(page)
            self.refcount[page] += 1
            parent = page
            matched += 1
        w.tokens = toks[:matched * self.S]
        w.n_frozen = matched * self.S
        return matched * self.S

    def ws_info(self, h: int):
        w = self._get(h)
        return w.n_tokens, w.n_frozen, len(w.pages)

    def ws_page_table(self, h: int) -> list:
        return list(self._get(h).pages)

    # ---------------------------------------------------------------- pass
    def begin(self, segs) -> Pass:
        """segs: sequence of (ws handle, n_new, token ids or None)."""
        seen = set()
        need = 0
        for h, n_new, toks in segs:
            w = self._get(h)
            if h in seen:
                raise OracleError(ERR_INVALID, "working set twice in one pass")
            seen.add(h)
            if n_new < 0 or (toks is not None and len(toks) != n_new):
                raise OracleError(ERR_INVALID, "bad segment")
            if n_new == 0:
                continue
            n0 = w.n_tokens
            need += _cdiv(n0 + n_new, self.S) - _cdiv(n0, self.S)
            if n0 % self.S and self.refcount[w.pages[n0 // self.S]] > 1:
                need += 1
        if need > len(self.free):
            raise OracleError(ERR_NO_PAGES, "page pool exhausted")
        rows_ws, rows_pos, rows_slot, cow = [], [], [], []
        for h, n_new, toks in segs:
            w = self.ws[h]
            n0 = w.n_tokens
            if n_new and n0 % self.S:
                tail = w.pages[n0 // self.S]
                if self.refcount[tail] > 1:
                    fresh = self._alloc()
                    if self.pool is not None:
                        self.pool[:, :, fresh] = self.pool[:, :, tail]
                    self.refcount[tail] -= 1
                    w.pages[n0 // self.S] = fresh
                    cow.append((tail, fresh))
            for t in range(n_new):
                pos = n0 + t
                if pos % self.S == 0:
                    w.pages.append(self._alloc())
                rows_ws.append(h)
                rows_pos.append(pos)
                rows_slot.append(w.pages[pos // self.S] * self.S + pos % self.S)
            w.tokens.extend([-1] * n_new if toks is None else [int(t) for t in toks])
        return Pass(rows_ws, rows_pos, rows_slot, cow)

    # ------------------------------------------------------------ KV bytes
    def _encode(self, x_bits: np.ndarray, layer: int, kv: int) -> np.ndarray:
        """[n, Hkv, d] bf16 bits -> [n, Hkv, d*esize] stored bytes."""
        x_bits = np.asarray(x_bits, dtype=np.uint16)
        if self.kv_dtype == KV_BF16:
            return x_bits.astype("<u2").view(np.uint8).reshape(x_bits.shape[0], self.Hkv, -1)
        scale = (self.k_scale if kv == 0 else self.v_scale)[layer]
        x = bf16_bits_to_f64(x_bits).astype(np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        for h in range(self.Hkv):
            out[:, h, :] = e4m3.quantize(x[:, h, :], float(scale[h]))
        return out

    def kv_append(self, pas: Pass, layer: int, k_bits: np.ndarray, v_bits: np.ndarray) -> None:
        """ops.attn.kv_append: write row r's K and V at its reserved slot."""
        slots = np.asarray(pas.rows_slot, dtype=np.int64)
        if slots.size == 0:
            return
        pages, s = slots // self.S, slots % self.S
        for kv, x in ((0, k_bits), (1, v_bits)):
            data = self._encode(x, layer, kv)                  # [n, Hkv, bytes]
            for h in range(self.Hkv):
                # row r's bytes go to offsets[s_r] of block (layer, page_r, h)
                self.pool[kv, layer, pages[:, None], h, self.offsets[s]] = data[:, h, :]

    def read_kv(self, h: int, layer: int, upto: int):
        """Contiguous K, V [upto, Hkv, d] float64 of working set h's first tokens."""
        w = self._get(h)
        pos = np.arange(upto)
        pages = np.asarray(w.pages, dtype=np.int64)[pos // self.S]
        offs = self.offsets[pos % self.S]                       # [upto, bytes]
        out = []
        for kv in (0, 1):
            # raw[p, h, b] = pool[kv, layer, page(p), h, offs[p, b]]
            raw = self.pool[kv, layer][pages[:, None, None], np.arange(self.Hkv)[None, :, None], offs[:, None, :]]
            if self.kv_dtype == KV_BF16:
                vals = bf16_bits_to_f64(np.ascontiguousarray(raw).view("<u2"))
            else:
                scale = (self.k_scale if kv == 0 else self.v_scale)[layer]
                vals = np.stack([e4m3.dequantize(raw[:, hh, :], float(scale[hh]))
                                 for hh in range(self.Hkv)], axis=1)
            out.append(vals)
        return out[0], out[1]

    # --------------------------------------------------------- invariants
    def check_invariants(self) -> None:
        held = [0] * self.P
        for w in self.ws.values():
            assert len(w.pages) == _cdiv(w.n_tokens, self.S)
            assert 0 <= w.n_frozen <= w.n_tokens
            for p in w.pages:
                held[p] += 1
        assert held == self.refcount, "refcount != number of tables holding the page"
        free = set(self.free)
        assert len(free) == len(self.free), "page on the free stack twice"
        for p in range(self.P):
            assert (p in free) == (self.refcount[p] == 0)
        for w in self.ws.values():
            # pages that hold only writable tokens are never shared
            for i in range(_cdiv(w.n_frozen, self.S), len(w.pages)):
                assert self.refcount[w.pages[i]] == 1, "writable page shared"
        for key, page in self.dedup.items():
            assert self.page_key[page] == key and self.refcount[page] > 0
