"""Thin ctypes binding of libkvc.so (include/kvc.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Device arguments accept torch CUDA tensors (their data_ptr is
passed) or raw integer addresses; `stream` defaults to torch's current
stream on the context's device.  Non-zero statuses raise KvcError.

The library must be built (kv_cache_decode_flash_gb300/build.py, or
__graft_entry__.build()); loading fails loudly when it is missing: there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvc.so")

KVC_OK, KVC_EINVAL, KVC_ENOMEM, KVC_ENOSPC, KVC_ERANGE = 0, -1, -2, -3, -4
KVC_EFORMAT, KVC_ECUDA, KVC_ETIMEDOUT, KVC_EINTERNAL = -5, -6, -7, -8
KVC_F16, KVC_Q4_0, KVC_Q8_0 = 1, 2, 8
KVC_DEVICE, KVC_HOST_PINNED, KVC_SPLIT_HEADS = 0, 1, 2
KVC_ROPE_NEOX, KVC_ROPE_NORM = 0, 1


class kvc_params(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layer", "n_head", "n_head_kv", "head_dim", "n_ctx", "n_seq_max",
                                          "type_k", "type_v")] + [("rope_base", C.c_float)] + [
        (n, C.c_int32) for n in ("rope_mode", "residency", "device", "page_rows", "gpu_heads")]


class kvc_stats(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("ring_engaged", "ring_declined", "ring_slots", "transfer_stream")] + [
        (n, C.c_int64) for n in ("slot_bytes", "ring_bytes", "ordered_bytes", "deliveries_early",
                                 "deliveries_ordered", "bytes_delivered", "pages_total", "pages_free",
                                 "device_bytes", "host_pinned_bytes")] + [
        (n, C.c_int32) for n in ("rolling", "tile_rows")] + [("tiles_delivered", C.c_int64)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class kvc_cold_stats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("budget_tokens", "tokens", "bytes")] + [
        (n, C.c_int32) for n in ("blocks", "pad")] + [
        (n, C.c_int64) for n in ("stored", "rejected", "dropped", "hits", "misses")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_ if n != "pad"}


class KvcError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s (%d): %s" % (_status_str(status), status, msg))
        self.status = status


_lib = None


def load():
    """Load libkvc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libkvc.so is not built (run __graft_entry__.build()); there is no CPU fallback")
    L = C.CDLL(LIB_PATH)
    p, i32, sz = C.c_void_p, C.c_int, C.c_size_t
    sig = {
        "kvc_params_init": (None, [C.POINTER(kvc_params)]),
        "kvc_create": (i32, [C.POINTER(kvc_params), C.POINTER(p)]),
        "kvc_destroy": (None, [p]),
        "kvc_last_error": (C.c_char_p, [p]),
        "kvc_status_str": (C.c_char_p, [i32]),
        "kvc_append": (i32, [p, i32, i32, i32, i32, p, p, p]),
        "kvc_attn_decode": (i32, [p, i32, i32, p, p, p, C.c_float, p]),
        "kvc_decode_step": (i32, [p, i32, i32, p, p, p, p, p, p, C.c_float, p]),
        "kvc_seq_rm": (i32, [p, i32, i32, i32]),
        "kvc_seq_cp": (i32, [p, i32, i32, i32, i32]),
        "kvc_seq_add": (i32, [p, i32, i32, i32, i32]),
        "kvc_state_get": (i32, [p, i32, i32, i32, p, sz, C.POINTER(sz)]),
        "kvc_state_set": (i32, [p, i32, p, sz, C.POINTER(sz)]),
        "kvc_seq_key_scores": (i32, [p, i32, i32, p, C.c_int32, C.POINTER(C.c_int32)]),
        "kvc_seq_evict_window": (i32, [p, i32, i32, i32, i32, i32, C.POINTER(C.c_int32)]),
        "kvc_pipeline_depth": (i32, [p, i32]),
        "kvc_pipeline_budget": (i32, [p, sz]),
        "kvc_seq_n_tokens": (i32, [p, i32, C.POINTER(C.c_int32)]),
        "kvc_seq_positions": (i32, [p, i32, p, C.c_int32, C.POINTER(C.c_int32)]),
        "kvc_get_stats": (i32, [p, C.POINTER(kvc_stats)]),
        "kvc_set_chunk_rows": (i32, [p, i32]),
        "kvc_trace_start": (i32, [p, i32]),
        "kvc_trace_stop": (i32, [p]),
        "kvc_trace_read": (i32, [p, p, i32, C.POINTER(C.c_int)]),
        "kvc_debug_chunk_plan": (i32, [i32, i32, i32, i32, i32, i32, i32, i32, p, C.POINTER(C.c_int32),
                                       C.POINTER(C.c_int32)]),
        "kvc_debug_chunk_plan_seq": (i32, [i32, i32, i32, i32, i32, i32, i32, i32, p, p, C.POINTER(C.c_int32)]),
        "kvc_debug_select_rows": (i32, [p, i32, i32, i32, i32, p, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                        C.POINTER(C.c_int32)]),
        "kvc_set_timeout_ms": (i32, [p, i32]),
        "kvc_debug_fail_alloc_after": (i32, [p, i32]),
        "kvc_check_device_error": (i32, [p, C.POINTER(C.c_uint32)]),
        "kvc_cold_create": (i32, [C.c_int64, C.POINTER(p)]),
        "kvc_cold_destroy": (None, [p]),
        "kvc_cold_last_error": (C.c_char_p, [p]),
        "kvc_cold_evict": (i32, [p, p, i32, i32, i32, i32, C.c_uint64, i32, C.POINTER(C.c_int),
                                 C.POINTER(C.c_int32)]),
        "kvc_cold_admit": (i32, [p, p, i32, i32, C.c_uint64, C.POINTER(C.c_int), C.POINTER(C.c_int32)]),
        "kvc_cold_find": (i32, [p, C.c_uint64, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
        "kvc_cold_restore_model": (i32, [p, C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
        "kvc_cold_set_restore_model": (i32, [p, C.c_double, C.c_double]),
        "kvc_cold_plan_admit": (i32, [p, C.c_uint64, C.c_double, C.c_double, C.POINTER(C.c_int),
                                      C.POINTER(C.c_double), C.POINTER(C.c_int32)]),
        "kvc_cold_get_stats": (i32, [p, C.POINTER(kvc_cold_stats)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _status_str(s: int) -> str:
    try:
        return load().kvc_status_str(s).decode()
    except Exception:  # pragma: no cover - only used for messages
        return "status"


def _check(ctx, status: int):
    if status != KVC_OK:
        msg = load().kvc_last_error(ctx).decode() if ctx else ""
        raise KvcError(status, msg)


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError("expected a tensor or an address")


def _stream(stream, device: int):
    if stream is None:
        import torch

        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kvc_params_init() -> kvc_params:
    p = kvc_params()
    load().kvc_params_init(C.byref(p))
    return p


def kvc_create(params: kvc_params) -> int:
    ctx = C.c_void_p()
    _check(None, load().kvc_create(C.byref(params), C.byref(ctx)))
    return ctx.value


def kvc_destroy(ctx: int) -> None:
    if ctx:
        load().kvc_destroy(ctx)


def kvc_last_error(ctx: int) -> str:
    return load().kvc_last_error(ctx).decode()


def kvc_append(ctx, layer, seq, pos0, n_tok, k, v, stream=None, device=0):
    _check(ctx, load().kvc_append(ctx, layer, seq, pos0, n_tok, _addr(k), _addr(v), _stream(stream, device)))


def kvc_attn_decode(ctx, layer, seq_ids, q, out, kq_scale, stream=None, device=0):
    ids = (C.c_int32 * len(seq_ids))(*[int(s) for s in seq_ids])
    _check(ctx, load().kvc_attn_decode(ctx, layer, len(seq_ids), ids, _addr(q), _addr(out), float(kq_scale),
                                       _stream(stream, device)))


def kvc_decode_step(ctx, layer, seq_ids, pos, k, v, q, out, kq_scale, stream=None, device=0):
    if len(pos) != len(seq_ids):
        raise ValueError("one position per sequence")
    ids = (C.c_int32 * len(seq_ids))(*[int(s) for s in seq_ids])
    ps = (C.c_int32 * len(pos))(*[int(x) for x in pos])
    _check(ctx, load().kvc_decode_step(ctx, layer, len(seq_ids), ids, ps, _addr(k), _addr(v), _addr(q), _addr(out),
                                       float(kq_scale), _stream(stream, device)))


class kvc_trace_event(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layer", C.c_int32), ("bytes", C.c_int64), ("t0_us", C.c_double),
                ("t1_us", C.c_double)]


def kvc_trace_start(ctx, max_records: int):
    _check(ctx, load().kvc_trace_start(ctx, int(max_records)))


def kvc_trace_stop(ctx):
    _check(ctx, load().kvc_trace_stop(ctx))


def kvc_trace_read(ctx) -> list:
    """[(kind, layer, bytes, t0_us, t1_us)] of the host transport's recorded
    deliveries (kind 0) and attention launches (kind 1)."""
    n = C.c_int(0)
    _check(ctx, load().kvc_trace_read(ctx, None, 0, C.byref(n)))
    buf = (kvc_trace_event * max(1, n.value))()
    _check(ctx, load().kvc_trace_read(ctx, buf, n.value, C.byref(n)))
    return [(e.kind, e.layer, e.bytes, e.t0_us, e.t1_us) for e in buf[: n.value]]


def kvc_seq_rm(ctx, seq, p0, p1):
    _check(ctx, load().kvc_seq_rm(ctx, seq, p0, p1))


def kvc_seq_cp(ctx, src, dst, p0, p1):
    _check(ctx, load().kvc_seq_cp(ctx, src, dst, p0, p1))


def kvc_seq_add(ctx, seq, p0, p1, delta):
    _check(ctx, load().kvc_seq_add(ctx, seq, p0, p1, delta))


def kvc_state_size(ctx, seq, p0, p1) -> int:
    n = C.c_size_t()
    _check(ctx, load().kvc_state_get(ctx, seq, p0, p1, None, 0, C.byref(n)))
    return n.value


def kvc_state_get(ctx, seq, p0, p1, dst=None) -> bytes | int:
    """Export to `dst` (a writable buffer: bytearray, numpy array, pinned
    tensor or address with enough room); with dst None, return new bytes."""
    n = C.c_size_t()
    if dst is None:
        size = kvc_state_size(ctx, seq, p0, p1)
        buf = (C.c_uint8 * size)()
        _check(ctx, load().kvc_state_get(ctx, seq, p0, p1, C.addressof(buf), size, C.byref(n)))
        return bytes(buf)
    addr, cap = _host_buffer(dst)
    _check(ctx, load().kvc_state_get(ctx, seq, p0, p1, addr, cap, C.byref(n)))
    return n.value


def kvc_state_set(ctx, seq, src, n=None) -> int:
    if isinstance(src, (bytes, bytearray)):
        buf = (C.c_uint8 * len(src)).from_buffer_copy(src) if isinstance(src, bytes) else \
            (C.c_uint8 * len(src)).from_buffer(src)
        addr, size = C.addressof(buf), len(src)
    else:
        addr, size = _host_buffer(src)
    if n is not None:
        size = n
    got = C.c_size_t()
    _check(ctx, load().kvc_state_set(ctx, seq, addr, size, C.byref(got)))
    return got.value


def _host_buffer(b):
    if isinstance(b, tuple):
        return b
    if isinstance(b, bytearray):
        arr = (C.c_uint8 * len(b)).from_buffer(b)
        return C.addressof(arr), len(b)
    if hasattr(b, "data_ptr"):
        return b.data_ptr(), b.numel() * b.element_size()
    if hasattr(b, "ctypes"):
        return b.ctypes.data, b.nbytes
    raise TypeError("expected a host buffer")


def kvc_seq_key_scores(ctx, seq, layer=-1):
    """KeyDiff score of every row of `seq` in `layer` (position order), fp32."""
    import numpy as np

    n = C.c_int32()
    _check(ctx, load().kvc_seq_key_scores(ctx, seq, layer, None, 0, C.byref(n)))
    out = np.zeros(n.value, np.float32)
    if n.value:
        _check(ctx, load().kvc_seq_key_scores(ctx, seq, layer, out.ctypes.data, n.value, C.byref(n)))
    return out


def kvc_seq_evict_window(ctx, seq, layer, n_keep, n_discard, n_recent) -> int:
    """Retention-aware context shift; returns the first removed position or -1."""
    p0 = C.c_int32()
    _check(ctx, load().kvc_seq_evict_window(ctx, seq, layer, n_keep, n_discard, n_recent, C.byref(p0)))
    return p0.value


def kvc_pipeline_depth(ctx, n):
    _check(ctx, load().kvc_pipeline_depth(ctx, n))


def kvc_pipeline_budget(ctx, nbytes):
    _check(ctx, load().kvc_pipeline_budget(ctx, nbytes))


def kvc_seq_n_tokens(ctx, seq) -> int:
    n = C.c_int32()
    _check(ctx, load().kvc_seq_n_tokens(ctx, seq, C.byref(n)))
    return n.value


def kvc_seq_positions(ctx, seq):
    import numpy as np

    n = C.c_int32()
    _check(ctx, load().kvc_seq_positions(ctx, seq, None, 0, C.byref(n)))
    out = np.zeros(n.value, np.int32)
    _check(ctx, load().kvc_seq_positions(ctx, seq, out.ctypes.data, n.value, C.byref(n)))
    return out


def kvc_get_stats(ctx) -> dict:
    s = kvc_stats()
    _check(ctx, load().kvc_get_stats(ctx, C.byref(s)))
    return s.as_dict()


def kvc_set_chunk_rows(ctx, rows):
    _check(ctx, load().kvc_set_chunk_rows(ctx, rows))


def kvc_set_timeout_ms(ctx, ms):
    _check(ctx, load().kvc_set_timeout_ms(ctx, ms))


def kvc_debug_chunk_plan(type_, head_dim, n_head, n_head_kv, sms, occ, occ2, rows):
    """The split-K plan (chunk rows, configuration) of an attention launch over
    sequences of `rows` rows, without a context or a GPU."""
    arr = (C.c_int32 * len(rows))(*[int(r) for r in rows])
    cr, cfg = C.c_int32(), C.c_int32()
    st = load().kvc_debug_chunk_plan(type_, head_dim, n_head, n_head_kv, sms, occ, occ2, len(rows), arr,
                                     C.byref(cr), C.byref(cfg))
    if st != KVC_OK:
        raise KvcError(st, "bad chunk-plan arguments")
    return cr.value, cfg.value


def kvc_debug_chunk_plan_seq(type_, head_dim, n_head, n_head_kv, sms, occ, occ2, rows):
    """Each sequence's rows per chunk and the configuration of an attention
    launch over sequences of `rows` rows, without a context or a GPU."""
    arr = (C.c_int32 * len(rows))(*[int(r) for r in rows])
    out = (C.c_int32 * len(rows))()
    cfg = C.c_int32()
    st = load().kvc_debug_chunk_plan_seq(type_, head_dim, n_head, n_head_kv, sms, occ, occ2, len(rows), arr, out,
                                         C.byref(cfg))
    if st != KVC_OK:
        raise KvcError(st, "bad chunk-plan arguments")
    return list(out), cfg.value


def kvc_debug_select_rows(pos, p0, p1, linear=False):
    """The rows a sequence operation selects for positions [p0, p1) of a
    sequence holding `pos`, without a context or a GPU: (rows, first,
    contiguous)."""
    n = len(pos)
    arr = (C.c_int32 * max(n, 1))(*[int(x) for x in pos])
    out = (C.c_int64 * max(n, 1))()
    cnt, first, contig = C.c_int64(), C.c_int64(), C.c_int32()
    st = load().kvc_debug_select_rows(arr, n, 1 if linear else 0, int(p0), int(p1), out, C.byref(cnt),
                                      C.byref(first), C.byref(contig))
    if st != KVC_OK:
        raise KvcError(st, "bad row-selection arguments")
    return list(out[:cnt.value]), first.value, bool(contig.value)


def kvc_debug_fail_alloc_after(ctx, n):
    _check(ctx, load().kvc_debug_fail_alloc_after(ctx, n))


def kvc_check_device_error(ctx) -> int:
    w = C.c_uint32()
    _check(ctx, load().kvc_check_device_error(ctx, C.byref(w)))
    return w.value


class KVCache:
    """Owns one context; methods forward to the functions above."""

    def __init__(self, n_layer, n_head, n_head_kv, head_dim, n_ctx, n_seq_max=1, type_k=KVC_Q8_0,
                 type_v=KVC_Q8_0, rope_base=10000.0, rope_mode=KVC_ROPE_NEOX, residency=KVC_DEVICE, device=0,
                 page_rows=0, gpu_heads=0):
        p = kvc_params_init()
        p.n_layer, p.n_head, p.n_head_kv, p.head_dim = n_layer, n_head, n_head_kv, head_dim
        p.n_ctx, p.n_seq_max, p.type_k, p.type_v = n_ctx, n_seq_max, type_k, type_v
        p.rope_base, p.rope_mode, p.residency, p.device, p.page_rows = rope_base, rope_mode, residency, device, page_rows
        p.gpu_heads = gpu_heads
        self.params = p
        self.device = device
        self.ctx = kvc_create(p)

    def close(self):
        if self.ctx:
            kvc_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, layer, seq, pos0, k, v, stream=None):
        kvc_append(self.ctx, layer, seq, pos0, int(k.shape[0]), k, v, stream, self.device)

    def attn_decode(self, layer, seq_ids, q, out, kq_scale, stream=None):
        kvc_attn_decode(self.ctx, layer, seq_ids, q, out, kq_scale, stream, self.device)

    def decode_step(self, layer, seq_ids, pos, k, v, q, out, kq_scale, stream=None):
        """Append one token per sequence (k, v: [n_seq][n_head_kv][head_dim] fp32 on the
        device, at positions pos) and attend with q ([n_seq][n_head][head_dim]) into out;
        one launch on device-resident contexts (kvc_decode_step)."""
        kvc_decode_step(self.ctx, layer, seq_ids, pos, k, v, q, out, kq_scale, stream, self.device)

    def seq_rm(self, seq, p0, p1):
        kvc_seq_rm(self.ctx, seq, p0, p1)

    def seq_cp(self, src, dst, p0, p1):
        kvc_seq_cp(self.ctx, src, dst, p0, p1)

    def seq_add(self, seq, p0, p1, delta):
        kvc_seq_add(self.ctx, seq, p0, p1, delta)

    def state_get(self, seq, p0, p1, dst=None):
        return kvc_state_get(self.ctx, seq, p0, p1, dst)

    def state_set(self, seq, src, n=None):
        return kvc_state_set(self.ctx, seq, src, n)

    def key_scores(self, seq, layer=-1):
        return kvc_seq_key_scores(self.ctx, seq, layer)

    def evict_window(self, seq, layer, n_keep, n_discard, n_recent):
        return kvc_seq_evict_window(self.ctx, seq, layer, n_keep, n_discard, n_recent)

    def n_tokens(self, seq):
        return kvc_seq_n_tokens(self.ctx, seq)

    def positions(self, seq):
        return kvc_seq_positions(self.ctx, seq)

    def stats(self):
        return kvc_get_stats(self.ctx)


# ------------------------------------------------------------ cold store --
def _check_cold(store, ctx, status: int):
    if status != KVC_OK:
        msg = load().kvc_cold_last_error(store).decode() if store else ""
        if ctx:
            detail = load().kvc_last_error(ctx).decode()
            if detail:
                msg = "%s (context: %s)" % (msg, detail)
        raise KvcError(status, msg)


def kvc_cold_create(budget_tokens: int) -> int:
    h = C.c_void_p()
    _check_cold(None, None, load().kvc_cold_create(int(budget_tokens), C.byref(h)))
    return h.value


def kvc_cold_destroy(store: int) -> None:
    if store:
        load().kvc_cold_destroy(store)


def kvc_cold_evict(ctx, store, seq, scratch, p0, p1, key, cls):
    """Returns (stored, n_tok)."""
    stored, n = C.c_int(), C.c_int32()
    _check_cold(store, ctx, load().kvc_cold_evict(ctx, store, seq, scratch, p0, p1, C.c_uint64(key), cls,
                                                  C.byref(stored), C.byref(n)))
    return stored.value, n.value


def kvc_cold_admit(ctx, store, seq, scratch, key):
    """Returns (hit, n_tok)."""
    hit, n = C.c_int(), C.c_int32()
    _check_cold(store, ctx, load().kvc_cold_admit(ctx, store, seq, scratch, C.c_uint64(key), C.byref(hit),
                                                  C.byref(n)))
    return hit.value, n.value


def kvc_cold_find(store, key):
    """Returns (n_tok, cls); (0, -1) when absent."""
    n, cls = C.c_int32(), C.c_int32()
    _check_cold(store, None, load().kvc_cold_find(store, C.c_uint64(key), C.byref(n), C.byref(cls)))
    return n.value, cls.value


def kvc_cold_restore_model(store):
    """(fixed_us, per_token_us, samples) of the store's restore cost model."""
    f, t, n = C.c_double(), C.c_double(), C.c_int64()
    _check_cold(store, None, load().kvc_cold_restore_model(store, C.byref(f), C.byref(t), C.byref(n)))
    return f.value, t.value, n.value


def kvc_cold_set_restore_model(store, fixed_us, per_token_us):
    _check_cold(store, None, load().kvc_cold_set_restore_model(store, float(fixed_us), float(per_token_us)))


def kvc_cold_plan_admit(store, key, recompute_fixed_us, recompute_us_per_token):
    """(restore, restore_us, n_tok) for the block under key: restore 1 when the
    model's restore estimate is below the caller's recompute cost."""
    r, us, n = C.c_int(), C.c_double(), C.c_int32()
    _check_cold(store, None, load().kvc_cold_plan_admit(store, C.c_uint64(key), float(recompute_fixed_us),
                                                         float(recompute_us_per_token), C.byref(r), C.byref(us),
                                                         C.byref(n)))
    return r.value, us.value, n.value


def kvc_cold_get_stats(store) -> dict:
    st = kvc_cold_stats()
    _check_cold(store, None, load().kvc_cold_get_stats(store, C.byref(st)))
    return st.as_dict()


class ColdStore:
    """Owns one cold store; evict / admit take the KVCache they act on."""

    def __init__(self, budget_tokens):
        self.handle = kvc_cold_create(budget_tokens)

    def close(self):
        if self.handle:
            kvc_cold_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def evict(self, cache, seq, scratch, p0, p1, key, cls):
        return kvc_cold_evict(cache.ctx, self.handle, seq, scratch, p0, p1, key, cls)

    def admit(self, cache, seq, scratch, key):
        return kvc_cold_admit(cache.ctx, self.handle, seq, scratch, key)

    def find(self, key):
        return kvc_cold_find(self.handle, key)

    def stats(self):
        return kvc_cold_get_stats(self.handle)

    def restore_model(self):
        return kvc_cold_restore_model(self.handle)

    def set_restore_model(self, fixed_us, per_token_us):
        kvc_cold_set_restore_model(self.handle, fixed_us, per_token_us)

    def plan_admit(self, key, recompute_fixed_us, recompute_us_per_token):
        return kvc_cold_plan_admit(self.handle, key, recompute_fixed_us, recompute_us_per_token)
