"""Row-list model of the KV cache sequence operations and the state bytes.

Test infrastructure only; see oracle/__init__.py.

A sequence is an ordered list of rows.  Each row has an int32 position and,
per layer, one stored K head-row and one stored V head-row per KV head
(q8_0: 32-code blocks with an fp16 scale; f16: halves).  The operations are
the llama.cpp-style sequence ops the cold store is assembled from
(Plan: lossless long context - derived hot/cold sizing + host-RAM KV cold
store, section llama - KV-byte offload: MemorySeqCopy, MemorySeqRemove,
MemorySeqAdd, StateSeqGetData/SetData; the evict order is copy to a scratch
sequence, export, drop the scratch, remove and slide; the admit order is
import into a scratch sequence, copy to the tail of sequence 0, fix the
positions):

  append(layer, seq, pos0, k, v)  quantise and add rows (per layer; the first
                                  layer to reach new positions creates them)
  seq_rm(seq, p0, p1)             drop rows with p0 <= pos < p1
  seq_cp(src, dst, p0, p1)        copy those rows (all layers) to the end of dst
  seq_add(seq, p0, p1, delta)     pos += delta on those rows and rotate their K
                                  by delta (OpenVINO - KV-byte offload: shifted
                                  imports rotate RoPE-positioned keys by the
                                  position delta)
  state_get / state_set           export / import a position range as bytes

Ranges are half-open; p0 < 0 means 0 and p1 < 0 means no upper bound.
A shift that would make a position negative is rejected (ValueError).

State byte format (version 1, little endian), all sections padded with zeros
to a multiple of 16 bytes:
  header 64 B: u32 magic 0x3143564B, u32 version 1, u32 n_layer,
               u32 n_head_kv, u32 head_dim, u32 type_k, u32 type_v,
               u32 n_tok, u64 payload_bytes, 24 zero bytes
  positions:   int32 pos[n_tok] (row order), padded
  payload:     for each layer: the K section, then the V section;
               q8_0 section = codes int8 [Hk][n_tok][D] (padded),
                              then scales u16 [Hk][n_tok][D/32] (padded)
               q4_0 section = packed codes u8 [Hk][n_tok][D/2] (padded),
                              then scales u16 [Hk][n_tok][D/32] (padded)
               f16 section  = halves u16 [Hk][n_tok][D] (padded)
"""
from __future__ import annotations

import struct

import numpy as np

from . import numerics as L

STATE_MAGIC = 0x3143564B
STATE_VERSION = 1
HEADER_BYTES = 64
INT32_MAX = 2**31 - 1


def _pad16(n: int) -> int:
    return (n + 15) // 16 * 16


def section_bytes(type_: int, n_tok: int, Hk: int, D: int) -> int:
    if type_ == L.Q8_0:
        return _pad16(Hk * n_tok * D) + _pad16(Hk * n_tok * (D // 32) * 2)
    if type_ == L.Q4_0:
        return _pad16(Hk * n_tok * (D // 2)) + _pad16(Hk * n_tok * (D // 32) * 2)
    return _pad16(Hk * n_tok * D * 2)


def state_size(n_layer, Hk, D, type_k, type_v, n_tok) -> int:
    payload = n_layer * (section_bytes(type_k, n_tok, Hk, D) + section_bytes(type_v, n_tok, Hk, D))
    return HEADER_BYTES + _pad16(4 * n_tok) + payload


def _norm_range(p0: int, p1: int) -> tuple[int, int]:
    return (0 if p0 < 0 else p0), (INT32_MAX + 1 if p1 < 0 else p1)


class _Tensor:
    """One layer's K or V rows: q8_0 (codes, scales), q4_0 (packed codes,
    scales; V only) or f16 (halves, None)."""

    def __init__(self, type_: int, Hk: int, D: int):
        self.type = type_
        if type_ == L.Q8_0:
            self.a = np.zeros((0, Hk, D), np.int8)
            self.s = np.zeros((0, Hk, D // 32), np.uint16)
        elif type_ == L.Q4_0:
            self.a = np.zeros((0, Hk, D // 2), np.uint8)
            self.s = np.zeros((0, Hk, D // 32), np.uint16)
        else:
            self.a = np.zeros((0, Hk, D), np.uint16)
            self.s = None

    def __len__(self):
        return self.a.shape[0]

    def take(self, idx) -> "_Tensor":
        t = object.__new__(_Tensor)
        t.type, t.a = self.type, self.a[idx].copy()
        t.s = None if self.s is None else self.s[idx].copy()
        return t

    def extend(self, other: "_Tensor"):
        self.a = np.concatenate([self.a, other.a])
        if self.s is not None:
            self.s = np.concatenate([self.s, other.s])

    def encode(self, x: np.ndarray) -> "_Tensor":
        """fp32 rows [n][Hk][D] -> stored form."""
        t = object.__new__(_Tensor)
        t.type = self.type
        if self.type == L.Q8_0:
            t.a, t.s = L.q8_0_quantize(x)
        elif self.type == L.Q4_0:
            t.a, t.s = L.q4_0_quantize(x)
        else:
            t.a, t.s = L.f32_to_f16(x), None
        return t


class _Seq:
    def __init__(self, n_layer, Hk, D, type_k, type_v):
        self.pos = np.zeros(0, np.int32)
        self.K = [_Tensor(type_k, Hk, D) for _ in range(n_layer)]
        self.V = [_Tensor(type_v, Hk, D) for _ in range(n_layer)]

    def synced(self) -> bool:
        return all(len(t) == len(self.pos) for t in self.K + self.V)


class OracleCache:
    def __init__(self, n_layer, n_head, n_head_kv, head_dim, type_k=L.Q8_0, type_v=L.Q8_0,
                 rope_base=10000.0, rope_mode=0):
        assert n_head % n_head_kv == 0 and head_dim % 32 == 0
        assert type_k != L.Q4_0, "q4_0 is a V type (the keys are rotated and requantised by seq_add)"
        self.n_layer, self.H, self.Hk, self.D = n_layer, n_head, n_head_kv, head_dim
        self.type_k, self.type_v = type_k, type_v
        self.rope_base, self.rope_mode = float(rope_base), int(rope_mode)
        self.seqs: dict[int, _Seq] = {}

    def _seq(self, s: int) -> _Seq:
        if s not in self.seqs:
            self.seqs[s] = _Seq(self.n_layer, self.Hk, self.D, self.type_k, self.type_v)
        return self.seqs[s]

    def n_tokens(self, s: int) -> int:
        return len(self.seqs[s].pos) if s in self.seqs else 0

    def positions(self, s: int) -> np.ndarray:
        return self._seq(s).pos.copy()

    # -- append ------------------------------------------------------------
    def append(self, layer: int, s: int, pos0: int, k: np.ndarray, v: np.ndarray):
        q = self._seq(s)
        k = np.asarray(k, np.float32).reshape(-1, self.Hk, self.D)
        v = np.asarray(v, np.float32).reshape(-1, self.Hk, self.D)
        n = k.shape[0]
        new_pos = np.arange(pos0, pos0 + n, dtype=np.int64)
        fill = len(q.K[layer])
        if fill == len(q.pos):
            q.pos = np.concatenate([q.pos, new_pos.astype(np.int32)])
        elif fill + n > len(q.pos) or not np.array_equal(q.pos[fill:fill + n], new_pos):
            raise ValueError("append does not match the rows other layers created")
        q.K[layer].extend(q.K[layer].encode(k))
        q.V[layer].extend(q.V[layer].encode(v))

    # -- sequence ops ------------------------------------------------------
    def _sel(self, q: _Seq, p0: int, p1: int) -> np.ndarray:
        p0, p1 = _norm_range(p0, p1)
        pos = q.pos.astype(np.int64)
        return (pos >= p0) & (pos < p1)

    def seq_rm(self, s: int, p0: int, p1: int):
        q = self._seq(s)
        if not q.synced():
            raise ValueError("layers not in sync")
        keep = ~self._sel(q, p0, p1)
        q.pos = q.pos[keep]
        q.K = [t.take(keep) for t in q.K]
        q.V = [t.take(keep) for t in q.V]

    def seq_cp(self, src: int, dst: int, p0: int, p1: int):
        if src == dst:
            return
        a, b = self._seq(src), self._seq(dst)
        if not (a.synced() and b.synced()):
            raise ValueError("layers not in sync")
        sel = self._sel(a, p0, p1)
        b.pos = np.concatenate([b.pos, a.pos[sel]])
        for l in range(self.n_layer):
            b.K[l].extend(a.K[l].take(sel))
            b.V[l].extend(a.V[l].take(sel))

    def seq_add(self, s: int, p0: int, p1: int, delta: int):
        q = self._seq(s)
        if not q.synced():
            raise ValueError("layers not in sync")
        sel = self._sel(q, p0, p1)
        if delta == 0 or not sel.any():
            return
        newpos = q.pos[sel].astype(np.int64) + delta
        if newpos.min() < 0 or newpos.max() > INT32_MAX:
            raise ValueError("shift out of range")
        q.pos = q.pos.copy()
        q.pos[sel] = newpos.astype(np.int32)
        for t in q.K:
            if t.type == L.Q8_0:
                c, sc = L.rope_shift_q8_0(t.a[sel], t.s[sel], self.rope_mode, self.rope_base, delta)
                t.a[sel], t.s[sel] = c, sc
            else:
                t.a[sel] = L.rope_shift_f16(t.a[sel], self.rope_mode, self.rope_base, delta)

    # -- KeyDiff retention-aware context shift ----------------------------
    def key_scores(self, s: int, layer: int) -> np.ndarray:
        """KeyDiff score of every row of sequence s in `layer`, rows in
        position order ("F5 - Advanced KV Cache Techniques", M1: the per-position
        score over a representative layer)."""
        q = self._seq(s)
        order = np.argsort(q.pos, kind="stable")
        K = q.K[layer]
        if len(K) == 0:
            return np.zeros(0)
        return L.keydiff_scores(K.type, K.a, K.s)[order]

    def evict_window(self, s: int, layer: int, n_keep: int, n_discard: int, n_recent: int) -> int:
        """Remove the width-n_discard window of position-ordered rows with the
        smallest score sum inside [n_keep, n - n_recent), then slide the later
        positions down over the gap (seq_rm + seq_add).  Returns the first
        removed position, or -1 when no window fits (nothing changes)."""
        q = self._seq(s)
        sc = self.key_scores(s, layer)
        n = len(sc)
        w = L.min_window(sc, n_keep, n - n_recent, n_discard)
        if w < 0:
            return -1
        pos = np.sort(q.pos)
        p0, p1 = int(pos[w]), int(pos[w + n_discard - 1]) + 1
        self.seq_rm(s, p0, p1)
        self.seq_add(s, p1, -1, -(p1 - p0))
        return p0

    # -- attention ---------------------------------------------------------
    def attn(self, layer: int, seq_ids, q: np.ndarray, kq_scale: float, heads=None) -> np.ndarray:
        """q fp32 [n_seq][H][D] -> fp64 [n_seq][H][D]."""
        q = np.asarray(q, np.float32).reshape(len(seq_ids), self.H, self.D)
        out = np.zeros(q.shape, np.float64)
        for i, s in enumerate(seq_ids):
            sq = self._seq(s)
            K, V = sq.K[layer], sq.V[layer]
            out[i] = L.attn(q[i], K.type, K.a, K.s, V.type, V.a, V.s, kq_scale, heads)
        return out

    # -- state bytes -------------------------------------------------------
    def state_get(self, s: int, p0: int, p1: int) -> bytes:
        q = self._seq(s)
        if not q.synced():
            raise ValueError("layers not in sync")
        sel = self._sel(q, p0, p1)
        n = int(sel.sum())
        payload = self.n_layer * (section_bytes(self.type_k, n, self.Hk, self.D)
                                  + section_bytes(self.type_v, n, self.Hk, self.D))
        out = bytearray()
        out += struct.pack("<8IQ", STATE_MAGIC, STATE_VERSION, self.n_layer, self.Hk, self.D,
                           self.type_k, self.type_v, n, payload)
        out += bytes(HEADER_BYTES - len(out))
        pos = q.pos[sel].astype("<i4").tobytes()
        out += pos + bytes(_pad16(len(pos)) - len(pos))
        for l in range(self.n_layer):
            for t in (q.K[l], q.V[l]):
                sub = t.take(sel)
                for arr in ((sub.a, sub.s) if sub.s is not None else (sub.a,)):
                    # stored [n][Hk][...] -> exported head-major [Hk][n][...]
                    b = np.ascontiguousarray(arr.transpose(1, 0, 2)).astype(
                        arr.dtype.newbyteorder("<")).tobytes()
                    out += b + bytes(_pad16(len(b)) - len(b))
        return bytes(out)

    def parse_state(self, blob: bytes):
        """Validate a blob against this cache's geometry; return (pos, K, V)."""
        if len(blob) < HEADER_BYTES:
            raise ValueError("short header")
        magic, ver, nl, hk, d, tk, tv, n, payload = struct.unpack_from("<8IQ", blob, 0)
        if magic != STATE_MAGIC or ver != STATE_VERSION:
            raise ValueError("bad magic/version")
        if (nl, hk, d, tk, tv) != (self.n_layer, self.Hk, self.D, self.type_k, self.type_v):
            raise ValueError("geometry mismatch")
        want = state_size(nl, hk, d, tk, tv, n)
        if payload != want - HEADER_BYTES - _pad16(4 * n) or len(blob) < want:
            raise ValueError("bad length")
        off = HEADER_BYTES
        pos = np.frombuffer(blob, "<i4", n, off).astype(np.int32)
        off += _pad16(4 * n)
        K, V = [], []
        for l in range(nl):
            for dst, type_ in ((K, tk), (V, tv)):
                t = object.__new__(_Tensor)
                t.type = type_
                if type_ in (L.Q8_0, L.Q4_0):
                    w, dt = (d, np.int8) if type_ == L.Q8_0 else (d // 2, np.uint8)
                    a = np.frombuffer(blob, dt, hk * n * w, off).reshape(hk, n, w)
                    off += _pad16(hk * n * w)
                    sc = np.frombuffer(blob, "<u2", hk * n * (d // 32), off).reshape(hk, n, d // 32)
                    off += _pad16(hk * n * (d // 32) * 2)
                    t.a = np.ascontiguousarray(a.transpose(1, 0, 2))
                    t.s = np.ascontiguousarray(sc.transpose(1, 0, 2)).astype(np.uint16)
                else:
                    a = np.frombuffer(blob, "<u2", hk * n * d, off).reshape(hk, n, d)
                    off += _pad16(hk * n * d * 2)
                    t.a = np.ascontiguousarray(a.transpose(1, 0, 2)).astype(np.uint16)
                    t.s = None
                dst.append(t)
        return pos, K, V

    def state_set(self, s: int, blob: bytes) -> int:
        pos, K, V = self.parse_state(blob)
        q = self._seq(s)
        if not q.synced():
            raise ValueError("layers not in sync")
        q.pos = np.concatenate([q.pos, pos])
        for l in range(self.n_layer):
            q.K[l].extend(K[l])
            q.V[l].extend(V[l])
        return state_size(self.n_layer, self.Hk, self.D, self.type_k, self.type_v, len(pos))


class ColdStore:
    """Host-RAM cold store of evicted ranges (Plan: lossless long context,
    #3 Host-RAM KV cold store + retrieval, section llama - KV-byte offload).

    Evict: copy the range to a scratch sequence, export it as state bytes,
    keep them under the range's token hash with its cache class, drop the
    scratch, then remove the range and slide the later rows down.  The store
    is bounded in tokens; when a block does not fit, blocks are dropped by
    class (the more evictable first: a larger class number here) and least
    recently stored first within a class, but never a block less evictable
    than the new one: then the new block is not kept (the pages: lossy only
    at the cold tier, only for the most evictable classes).  Admit (append
    mode): import the bytes into the scratch sequence, shift them so that the
    first row follows the sequence's last position, copy them into the
    sequence, drop the scratch.  A block lives in one tier, so an admitted
    block leaves the store; a miss changes nothing (the caller recomputes).
    """

    def __init__(self, budget_tokens: int):
        if budget_tokens < 1:
            raise ValueError("budget must be positive")
        self.budget = int(budget_tokens)
        self.blocks = []  # dicts: key, cls, n, first, stamp, blob
        self.clock = 0
        self.stats = {"stored": 0, "rejected": 0, "dropped": 0, "hits": 0, "misses": 0}
        # restore cost samples (rows, microseconds) and an optional model set by the caller
        self.samples = []
        self.model_set = None

    @staticmethod
    def fit_restore_model(samples):
        """Least-squares line through (rows, us) samples: (fixed_us, per_token_us);
        one distinct size only: a line through 0; no samples: None
        (Plan: lossless long context, #3: bulk restore beats re-prefill for large
        blocks, recompute wins for small ones)."""
        if not samples:
            return None
        x = np.array([s[0] for s in samples], np.float64)
        y = np.array([s[1] for s in samples], np.float64)
        n = float(len(x))
        sx, sy, sxx, sxy = x.sum(), y.sum(), (x * x).sum(), (x * y).sum()
        den = n * sxx - sx * sx
        if len(x) >= 2 and den > 1e-9 * n * sxx:
            b = (n * sxy - sx * sy) / den
            return (sy - b * sx) / n, b
        return 0.0, sy / sx

    def plan_admit(self, key: int, recompute_fixed_us: float, recompute_us_per_token: float, model=None):
        """(restore, restore_us, n_tok): restore when the model's estimate of
        restoring the block is below recomputing it; absent block: (0, 0, 0);
        no model: (1, -1, n), the stored bytes first."""
        b = self.find(key)
        if b is None:
            return 0, 0.0, 0
        m = model if model is not None else (self.model_set or self.fit_restore_model(self.samples))
        if m is None:
            return 1, -1.0, b["n"]
        us = m[0] + m[1] * b["n"]
        return int(us < recompute_fixed_us + recompute_us_per_token * b["n"]), us, b["n"]

    @property
    def tokens(self) -> int:
        return sum(b["n"] for b in self.blocks)

    def find(self, key: int):
        for b in self.blocks:
            if b["key"] == key:
                return b
        return None

    def victims(self, n: int, cls: int):
        """Blocks to drop so that n tokens of class cls fit, in drop order, or
        None when they cannot make room."""
        if n > self.budget:
            return None
        cand = sorted((b for b in self.blocks if b["cls"] >= cls), key=lambda b: (-b["cls"], b["stamp"]))
        used, out = self.tokens, []
        for b in cand:
            if used + n <= self.budget:
                break
            out.append(b)
            used -= b["n"]
        return out if used + n <= self.budget else None

    def evict(self, cache: "OracleCache", seq: int, scratch: int, p0: int, p1: int, key: int, cls: int):
        """Returns (stored, n_tok)."""
        q = cache._seq(seq)
        if cache.n_tokens(scratch) != 0:
            raise ValueError("scratch sequence not empty")
        sel = (q.pos >= p0) & (q.pos < p1)
        n = int(sel.sum())
        if n == 0:
            return 0, 0
        first = int(q.pos[sel].min())
        old = self.find(key)
        if old is not None:
            self.blocks.remove(old)
        vict = self.victims(n, cls)
        stored = 0
        if vict is not None:
            cache.seq_cp(seq, scratch, p0, p1)
            blob = cache.state_get(scratch, -1, -1)
            cache.seq_rm(scratch, -1, -1)
            for b in vict:
                self.blocks.remove(b)
                self.stats["dropped"] += 1
            self.clock += 1
            self.blocks.append({"key": key, "cls": cls, "n": n, "first": first, "stamp": self.clock, "blob": blob})
            self.stats["stored"] += 1
            stored = 1
        else:
            self.stats["rejected"] += 1
        cache.seq_rm(seq, p0, p1)
        cache.seq_add(seq, p1, -1, -(p1 - p0))
        return stored, n

    def admit(self, cache: "OracleCache", seq: int, scratch: int, key: int):
        """Returns (hit, n_tok)."""
        if cache.n_tokens(scratch) != 0:
            raise ValueError("scratch sequence not empty")
        b = self.find(key)
        if b is None:
            self.stats["misses"] += 1
            return 0, 0
        pos = cache.positions(seq)
        tail = int(pos.max()) + 1 if len(pos) else 0
        cache.state_set(scratch, b["blob"])
        if tail != b["first"]:
            cache.seq_add(scratch, -1, -1, tail - b["first"])
        cache.seq_cp(scratch, seq, -1, -1)
        cache.seq_rm(scratch, -1, -1)
        self.blocks.remove(b)
        self.stats["hits"] += 1
        return 1, b["n"]
