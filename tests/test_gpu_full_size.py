"""Parity at the full configuration sizes, in the launch configuration the
benchmark times.

Every cache here has the shape and size the benchmark builds: 64 layers,
40/8 heads, head size 128, RoPE base 1e6, K/V drawn from N(0, 0.5^2), the
same capacity, page size and append chunking, so every kernel launch has
the geometry the benchmark times.  Inputs come from the seeded generator
(kv_cache_decode_flash_gb300.synth), drawn once on the device with the
benchmark's streams.  The layers (or sequences) whose outputs are compared
are copied to the host exactly as drawn and handed to the oracle, so both
sides start from the same fp32 values and the oracle sees nothing the CUDA
path computed.  The oracle computes the sampled outputs one at a time (a
layer, a set of query heads, a range of rows); properties that hold at any
size (ordered and pipelined outputs byte-identical, positions after the
churn, the state byte round trip) are checked on everything.

Tolerances are the ones of the other parity tests: attention max abs 1e-3
and relative L2 1e-4; requantised q8_0 K after a shift codes within +-1 and
scales within 1 fp16 ulp; V and unshifted K bit-exact; KeyDiff scores 1e-4.
"""
import os
from concurrent.futures import ThreadPoolExecutor
from ctypes import byref as C_byref, c_uint32 as C_uint32

import numpy as np
import pytest

import oracle
from kv_cache_decode_flash_gb300 import synth
from twin import assert_attn_close

pytestmark = pytest.mark.gpu

Q8, F16, Q4 = oracle.Q8_0, oracle.F16, oracle.Q4_0
H, HK, D, L = 40, 8, 128, 64
SIGMA = 0.5
BASE = 1e6
SCORE_TOL = 1e-4
# one query head per KV group, at every offset within a group of 5
SAMPLED_HEADS = tuple(5 * g + g % 5 for g in range(HK))


def _env():
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    return torch, kvc, torch.device("cuda:0")


def _draw(torch, dev, kind, layer, extra, m, hk=HK, sigma=SIGMA):
    return synth.normal_torch(0, synth.stream_id(kind, layer, extra), m * hk * D, sigma, dev).view(m, hk, D)


def _fill(caches, torch, dev, n, chunk, keep=()):
    """Rows [0, n) of every layer of sequence 0, appended in `chunk`-row
    pieces with the benchmark's streams, to every cache in `caches`.
    Returns {layer: (k, v)}: fp32 host copies of the layers in `keep`."""
    host = {}
    for l in range(L):
        ks, vs = [], []
        for p0 in range(0, n, chunk):
            m = min(chunk, n - p0)
            k, v = _draw(torch, dev, "k", l, p0, m), _draw(torch, dev, "v", l, p0, m)
            for c in caches:
                c.append(l, 0, p0, k, v)
            if l in keep:
                ks.append(k.cpu().numpy())
                vs.append(v.cpu().numpy())
        if l in keep:
            host[l] = (np.concatenate(ks), np.concatenate(vs))
    torch.cuda.synchronize()
    return host


def _stored(type_, x):
    """The oracle's stored form of fp32 rows [n][Hk][D]."""
    if type_ == Q8:
        return oracle.q8_0_quantize(x)
    if type_ == Q4:
        return oracle.q4_0_quantize(x)
    return oracle.f32_to_f16(x), None


def _oracle_attn(q, type_, k, v, kq_scale, heads, type_v=None):
    """Oracle outputs fp64 [H][D] of the listed query heads (zero elsewhere),
    one host thread per head."""
    tv = type_ if type_v is None else type_v
    kc, ks = _stored(type_, k)
    vc, vs = _stored(tv, v)
    scale = float(np.float32(kq_scale))
    one = lambda h: oracle.attn(q, type_, kc, ks, tv, vc, vs, scale, heads=(h, h + 1))
    with ThreadPoolExecutor(max(1, min(len(heads), os.cpu_count() or 1))) as ex:
        return sum(ex.map(one, heads))


def _oracle_attn_stored(q, kc, ks, vc, vs, kq_scale, heads):
    """Oracle outputs fp64 [H][D] over stored q8_0 rows, listed heads only."""
    scale = float(np.float32(kq_scale))
    one = lambda h: oracle.attn(q, Q8, kc, ks, Q8, vc, vs, scale, heads=(h, h + 1))
    with ThreadPoolExecutor(max(1, min(len(heads), os.cpu_count() or 1))) as ex:
        return sum(ex.map(one, heads))


def _close_on_heads(got, want, heads, what):
    idx = list(heads)
    assert_attn_close(got[idx].astype(np.float64), want[idx], what)


# ------------------------------------------------- device-resident decode --
@pytest.mark.parametrize("type_", [Q8, F16])
@pytest.mark.parametrize("n", [4096, 16384])
def test_full_device_resident_decode_step(type_, n):
    """One decode step of the 64-layer stack at n_kv = n (append row n-1,
    then attention, per layer), as the benchmark's step; layers 0, 31 and 63
    checked on all 40 query heads."""
    torch, kvc, dev = _env()
    sampled = (0, 31, 63)
    scale = float(1.0 / np.sqrt(D))
    cache = kvc.KVCache(L, H, HK, D, n + 256, 1, type_, type_, BASE, 0, kvc.KVC_DEVICE, 0)
    try:
        host = _fill([cache], torch, dev, n - 1, 4096, keep=sampled)
        q = synth.normal_torch(0, synth.stream_id("q", 0, n), L * H * D, 1.0, dev).view(L, 1, H, D)
        kn = _draw(torch, dev, "knew", 0, n, L).view(L, 1, HK, D)
        vn = _draw(torch, dev, "vnew", 0, n, L).view(L, 1, HK, D)
        out = torch.empty_like(q)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            for l in range(L):
                cache.append(l, 0, n - 1, kn[l], vn[l], stream=s)
                cache.attn_decode(l, [0], q[l], out[l], scale, stream=s)
        s.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        qh, knh, vnh = q.cpu().numpy(), kn.cpu().numpy(), vn.cpu().numpy()
        for l in sampled:
            k = np.concatenate([host[l][0], knh[l]])
            v = np.concatenate([host[l][1], vnh[l]])
            want = _oracle_attn(qh[l, 0], type_, k, v, scale, range(H))
            _close_on_heads(got[l, 0], want, range(H), "layer %d at n %d" % (l, n))
    finally:
        cache.close()


@pytest.mark.parametrize("type_,type_v", [(Q8, Q8), (F16, F16), (Q8, Q4)])
def test_full_fused_decode_step_graph_replay(type_, type_v):
    """The benchmark's step exactly as it times it: n_kv 16384, 64 layers,
    one fused kvc_decode_step launch per layer (row n-1 quantised inside the
    attention launch), run once eagerly, then captured as a CUDA graph and
    replayed three times (each replay rewrites row n-1).  The eager step and
    every replay give the same bits; layers 0, 31 and 63 of the last replay
    against the oracle on all 40 query heads.  Also the asymmetric cache
    (q8_0 K, q4_0 V)."""
    torch, kvc, dev = _env()
    n = 16384
    sampled = (0, 31, 63)
    scale = float(1.0 / np.sqrt(D))
    cache = kvc.KVCache(L, H, HK, D, n + 256, 1, type_, type_v, BASE, 0, kvc.KVC_DEVICE, 0)
    try:
        host = _fill([cache], torch, dev, n - 1, 4096, keep=sampled)
        q = synth.normal_torch(0, synth.stream_id("q", 0, n + 7), L * H * D, 1.0, dev).view(L, 1, H, D)
        kn = _draw(torch, dev, "knew", 0, n + 7, L).view(L, 1, HK, D)
        vn = _draw(torch, dev, "vnew", 0, n + 7, L).view(L, 1, HK, D)
        out = torch.empty_like(q)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            for l in range(L):
                cache.decode_step(l, [0], [n - 1], kn[l], vn[l], q[l], out[l], scale, stream=s)
        s.synchronize()
        eager = out.clone()
        cache.seq_rm(0, n - 1, -1)  # the captured step re-appends row n-1 (the pages stay)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for l in range(L):
                cache.decode_step(l, [0], [n - 1], kn[l], vn[l], q[l], out[l], scale,
                                  stream=torch.cuda.current_stream())
        for rep in range(3):
            out.fill_(float("nan"))
            with torch.cuda.stream(s):
                gr.replay()
            s.synchronize()
            assert torch.equal(out, eager), "replay %d differs from the eager step" % rep
        word = C_uint32()
        kvc.load().kvc_check_device_error(cache.ctx, C_byref(word))
        assert word.value == 0, "device error word %#x" % word.value
        got = out.cpu().numpy()
        qh, knh, vnh = q.cpu().numpy(), kn.cpu().numpy(), vn.cpu().numpy()
        for l in sampled:
            k = np.concatenate([host[l][0], knh[l]])
            v = np.concatenate([host[l][1], vnh[l]])
            want = _oracle_attn(qh[l, 0], type_, k, v, scale, range(H), type_v)
            _close_on_heads(got[l, 0], want, range(H), "fused step, graph replay, layer %d" % l)
        del gr
    finally:
        cache.close()


# ---------------------------------------------- long-context attention --
@pytest.mark.parametrize("n", [65536, 262144])
def test_full_long_context_attention(n):
    """The benchmark's long-context attention rows (q8_0, 40/8 heads): at
    65536 rows one wave of long chunks, at 262144 rows the configuration with
    two CTAs per SM (its work exceeds one wave of the other at the longest
    chunks) and a merge of the split-K partials in several rounds; layer 1 of
    two against the oracle on one query head per KV group."""
    torch, kvc, dev = _env()
    scale = float(1.0 / np.sqrt(D))
    Lr = 2
    cache = kvc.KVCache(Lr, H, HK, D, n + 64, 1, Q8, Q8, BASE)
    try:
        host = {}
        for l in range(Lr):
            ks, vs = [], []
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k, v = _draw(torch, dev, "k", l, p0, m), _draw(torch, dev, "v", l, p0, m)
                cache.append(l, 0, p0, k, v)
                if l == 1:
                    ks.append(k.cpu().numpy())
                    vs.append(v.cpu().numpy())
            if l == 1:
                host = (np.concatenate(ks), np.concatenate(vs))
        q = synth.normal_torch(0, synth.stream_id("q", 1, n), Lr * H * D, 1.0, dev).view(Lr, H, D)
        out = torch.empty_like(q)
        for l in range(Lr):
            cache.attn_decode(l, [0], q[l:l + 1], out[l:l + 1], scale)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        want = _oracle_attn(q.cpu().numpy()[1], Q8, host[0], host[1], scale, SAMPLED_HEADS)
        _close_on_heads(got[1], want, SAMPLED_HEADS, "n %d" % n)
    finally:
        cache.close()


# ------------------------------------------------- host-resident decode --
def _host_step(torch, dev, caches, pos, step, scale):
    """Append row `pos` and attend, every layer, on every cache; returns the
    outputs [cache][L][H][D] and the step's new rows and queries."""
    q = synth.normal_torch(0, synth.stream_id("q", 0, 1000 + step), L * H * D, 1.0, dev).view(L, 1, H, D)
    kn = _draw(torch, dev, "knew", 0, pos, L).view(L, 1, HK, D)
    vn = _draw(torch, dev, "vnew", 0, pos, L).view(L, 1, HK, D)
    outs = []
    for c in caches:
        out = torch.empty_like(q)
        for l in range(L):
            c.append(l, 0, pos, kn[l], vn[l])
            c.attn_decode(l, [0], q[l], out[l], scale)
        outs.append(out)
    torch.cuda.synchronize()
    return [o.cpu().numpy()[:, 0] for o in outs], q.cpu().numpy()[:, 0], kn.cpu().numpy()[:, 0], vn.cpu().numpy()[:, 0]


def test_full_host_resident_32k_pipelined_equals_ordered():
    """n_kv 32768, 64 layers in pinned host memory: an ordered cache and a
    second cache that runs the ring at depth 1 and 4 (512 MiB) and rolling
    tiles (128 MiB) produce byte-identical outputs on every layer, step by
    step; layer 63 of the first step is checked against the oracle."""
    torch, kvc, dev = _env()
    n = 32768
    scale = float(1.0 / np.sqrt(D))
    a = kvc.KVCache(L, H, HK, D, n + 256, 1, Q8, Q8, BASE, 0, kvc.KVC_HOST_PINNED)
    b = kvc.KVCache(L, H, HK, D, n + 256, 1, Q8, Q8, BASE, 0, kvc.KVC_HOST_PINNED)
    try:
        host = _fill([a, b], torch, dev, n - 1, 8192, keep=(63,))
        kvc.kvc_pipeline_depth(a.ctx, 0)
        pos = n - 1
        for step, (depth, budget, rolling) in enumerate(((1, 512 << 20, 0), (4, 512 << 20, 0), (1, 128 << 20, 1),
                                                         (4, 128 << 20, 1))):
            kvc.kvc_pipeline_depth(b.ctx, depth)
            kvc.kvc_pipeline_budget(b.ctx, budget)
            (oa, ob), qh, knh, vnh = _host_step(torch, dev, [a, b], pos, step, scale)
            st = b.stats()
            assert st["ring_engaged"] > 0 and st["rolling"] == rolling, (depth, budget, st)
            assert np.array_equal(oa.view(np.uint32), ob.view(np.uint32)), (depth, budget)
            if step == 0:
                k = np.concatenate([host[63][0], knh[63][None]])
                v = np.concatenate([host[63][1], vnh[63][None]])
                want = _oracle_attn(qh[63], Q8, k, v, scale, SAMPLED_HEADS)
                _close_on_heads(oa[63], want, SAMPLED_HEADS, "host-resident 32k, layer 63")
            pos += 1
    finally:
        a.close()
        b.close()


def test_full_host_resident_128k_rolling_and_ordered_vs_oracle():
    """n_kv 131072, 64 layers in pinned host memory: rolling tiles at depth 4
    (512 MiB), then ordered; each step's layer 63 against the oracle on one
    query head per KV group."""
    torch, kvc, dev = _env()
    n = 131072
    scale = float(1.0 / np.sqrt(D))
    c = kvc.KVCache(L, H, HK, D, n + 256, 1, Q8, Q8, BASE, 0, kvc.KVC_HOST_PINNED)
    try:
        host = _fill([c], torch, dev, n - 1, 8192, keep=(63,))
        k, v = host[63]
        pos = n - 1
        for step, (depth, budget, rolling) in enumerate(((4, 512 << 20, 1), (0, 512 << 20, 0))):
            kvc.kvc_pipeline_depth(c.ctx, depth)
            kvc.kvc_pipeline_budget(c.ctx, budget)
            (o,), qh, knh, vnh = _host_step(torch, dev, [c], pos, step, scale)
            if depth:  # at depth 0 the ordered path runs and an earlier ring may stay allocated
                assert c.stats()["rolling"] == rolling
            k = np.concatenate([k, knh[63][None]])
            v = np.concatenate([v, vnh[63][None]])
            want = _oracle_attn(qh[63], Q8, k, v, scale, SAMPLED_HEADS)
            _close_on_heads(o[63], want, SAMPLED_HEADS, "host-resident 128k, depth %d, layer 63" % depth)
            pos += 1
    finally:
        c.close()


# ------------------------------------------------------ batched ragged --
@pytest.mark.parametrize("type_", [Q8, F16])
def test_full_ragged_batch(type_):
    """32 sequences, lengths uniform in [1024, 32768] (the benchmark's
    draw), 32/8 heads, one layer, one attention call over the whole batch;
    the shortest, the longest and two other sequences against the oracle on
    all 32 query heads."""
    torch, kvc, dev = _env()
    Hq = 32
    lens = synth.randint(0, synth.stream_id("len"), 32, 1024, 32768).tolist()
    sampled = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 7, 19})
    cache = kvc.KVCache(1, Hq, HK, D, sum(lens) + 32 * 256, 32, type_, type_, BASE)
    try:
        host = {}
        for sidx, n in enumerate(lens):
            ks, vs = [], []
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = _draw(torch, dev, "k", 0, sidx * 4096 + p0 // 8192, m, sigma=1.0)
                v = _draw(torch, dev, "v", 0, sidx * 4096 + p0 // 8192, m, sigma=1.0)
                cache.append(0, sidx, p0, k, v)
                if sidx in sampled:
                    ks.append(k.cpu().numpy())
                    vs.append(v.cpu().numpy())
            if sidx in sampled:
                host[sidx] = (np.concatenate(ks), np.concatenate(vs))
        q = synth.normal_torch(0, synth.stream_id("q", 0, 77), 32 * Hq * D, 1.0, dev).view(32, Hq, D)
        o = torch.empty_like(q)
        cache.attn_decode(0, list(range(32)), q, o, 0.088)
        torch.cuda.synchronize()
        got, qh = o.cpu().numpy(), q.cpu().numpy()
        assert np.isfinite(got).all()
        for sidx in sampled:
            want = _oracle_attn(qh[sidx], type_, host[sidx][0], host[sidx][1], 0.088, range(Hq))
            _close_on_heads(got[sidx], want, range(Hq), "sequence %d (%d rows)" % (sidx, lens[sidx]))
    finally:
        cache.close()


# ------------------------------------------------------ cold-store churn --
def _layer_rows(parser, blob, layer):
    """Positions and layer `layer`'s K/V tensors of a 64-layer state blob."""
    pos, K, V = parser.parse_state(bytes(blob))
    return pos, K[layer], V[layer]


def _compare_shifted(gpu, ref, what):
    """GPU (pos, K, V) against the oracle's: positions and V exact; K codes
    within +-1 and scales within 1 fp16 ulp (requantised after a shift)."""
    (pg, Kg, Vg), (po, Ko, Vo) = gpu, ref
    assert np.array_equal(pg, po), what
    assert np.array_equal(Vg.a, Vo.a) and np.array_equal(Vg.s, Vo.s), what
    assert np.abs(Kg.a.astype(int) - Ko.a.astype(int)).max() <= 1, what
    assert np.abs(Kg.s.astype(int) - Ko.s.astype(int)).max() <= 1, what


def _layer_of_state(blob, n, layer, hk=HK, d=D):
    """Layer `layer`'s q8_0 K and V of a 64-layer state blob of n rows, as the
    oracle stores them: codes int8 [n][Hk][D], scales u16 [n][Hk][D/32]."""
    pad = lambda x: (x + 15) // 16 * 16
    codes, scl = pad(hk * n * d), pad(hk * n * (d // 32) * 2)
    off = 64 + pad(4 * n) + layer * 2 * (codes + scl)
    out = []
    for _ in range(2):  # K then V
        c = np.frombuffer(blob, np.int8, hk * n * d, off).reshape(hk, n, d)
        sc = np.frombuffer(blob, "<u2", hk * n * (d // 32), off + codes).reshape(hk, n, d // 32)
        out.append((np.ascontiguousarray(c.transpose(1, 0, 2)), np.ascontiguousarray(sc.transpose(1, 0, 2))))
        off += codes + scl
    return out


def _export_layer(cache, kvc, torch, n, layer, piece=16384):
    """K and V of one layer of sequence 0 (positions 0..n-1), exported in
    pieces of `piece` positions through the state format."""
    size = kvc.kvc_state_size(cache.ctx, 0, 0, piece)
    buf = torch.empty(size, dtype=torch.uint8, pin_memory=True)
    parts = []
    for p0 in range(0, n, piece):
        cache.state_get(0, p0, p0 + piece, buf)
        blob = buf.numpy().tobytes()
        cnt = int(np.frombuffer(blob, "<u4", 1, 28)[0])  # header: rows in the blob
        parts.append(_layer_of_state(blob, cnt, layer))
    kc = np.concatenate([p[0][0] for p in parts])
    ks = np.concatenate([p[0][1] for p in parts])
    vc = np.concatenate([p[1][0] for p in parts])
    vs = np.concatenate([p[1][1] for p in parts])
    return kc, ks, vc, vs


def test_full_cold_store_churn():
    """131072-token q8_0 cache, 64 layers, 64 cycles of: copy the oldest
    8192 rows to a scratch sequence, export them, drop the scratch, remove
    them and slide the rest down; import into the scratch, shift it to the
    tail, copy it in, drop the scratch; one decode step.  Every cycle:
    positions 0..n-1, and layer 32's decode output bitwise equal to a second
    launch of that layer; first and last cycle: export -> import -> export is
    byte-exact.  After the first cycle, layer 32 is checked against the
    oracle running the same operations (the exported block bit-exact; slid
    and re-admitted rows within the shift tolerances), and so is its decode
    output (one query head per KV group).  Every 16 cycles the decode output
    is checked against the oracle's attention over the rows the cache holds
    then: requantisation after each shift is lossy, so two caches evolved
    independently drift apart by more than the attention tolerance after
    many cycles, and each cycle's shifts are compared one op at a time."""
    torch, kvc, dev = _env()
    n, blk, cycles, lay = 131072, 8192, 64, 32
    cache = kvc.KVCache(L, H, HK, D, n + 2 * blk + 512, 2, Q8, Q8, BASE)
    parser = oracle.OracleCache(L, H, HK, D, Q8, Q8, BASE, 0)
    ref = oracle.OracleCache(1, H, HK, D, Q8, Q8, BASE, 0)
    try:
        host = _fill([cache], torch, dev, n, 8192, keep=(lay,))
        ref.append(0, 0, 0, *host.pop(lay))
        size = kvc.kvc_state_size(cache.ctx, 0, 0, blk)
        blob = torch.empty(size, dtype=torch.uint8, pin_memory=True)
        again = torch.empty(size, dtype=torch.uint8, pin_memory=True)
        q = synth.normal_torch(0, synth.stream_id("q", 0, 5), L * H * D, 1.0, dev).view(L, 1, H, D)
        o = torch.empty_like(q)
        o2 = torch.empty_like(q[0])
        qh = q.cpu().numpy()[lay, 0]
        for c in range(cycles):
            cache.seq_cp(0, 1, 0, blk)
            cache.state_get(1, -1, -1, blob)
            cache.seq_rm(1, -1, -1)
            cache.seq_rm(0, 0, blk)
            cache.seq_add(0, blk, n, -blk)
            cache.state_set(1, blob)
            if c in (0, cycles - 1):
                cache.state_get(1, -1, -1, again)
                assert torch.equal(blob, again), "state round trip, cycle %d" % c
            cache.seq_add(1, -1, -1, n - blk)
            cache.seq_cp(1, 0, -1, -1)
            cache.seq_rm(1, -1, -1)
            for l in range(L):
                cache.attn_decode(l, [0], q[l], o[l], 0.088)
            cache.attn_decode(lay, [0], q[lay], o2, 0.088)
            torch.cuda.synchronize()
            assert torch.equal(o[lay], o2), "decode of layer %d not repeatable, cycle %d" % (lay, c)
            assert torch.isfinite(o).all(), "cycle %d" % c
            word = C_uint32()
            kvc.load().kvc_check_device_error(cache.ctx, C_byref(word))
            assert word.value == 0, "device error word %#x after the decode of cycle %d" % (word.value, c)
            assert np.array_equal(np.sort(cache.positions(0)), np.arange(n)), "positions, cycle %d" % c
            if c == 0:
                ref.seq_cp(0, 1, 0, blk)
                ref_blob = ref.state_get(1, -1, -1)
                pg, Kg, Vg = _layer_rows(parser, blob.numpy(), lay)
                po, Ko, Vo = ref.parse_state(ref_blob)
                assert np.array_equal(pg, po)
                assert np.array_equal(Kg.a, Ko[0].a) and np.array_equal(Kg.s, Ko[0].s)
                assert np.array_equal(Vg.a, Vo[0].a) and np.array_equal(Vg.s, Vo[0].s)
                ref.seq_rm(1, -1, -1)
                ref.seq_rm(0, 0, blk)
                ref.seq_add(0, blk, n, -blk)
                ref.state_set(1, ref_blob)
                ref.seq_add(1, -1, -1, n - blk)
                ref.seq_cp(1, 0, -1, -1)
                ref.seq_rm(1, -1, -1)
                for p0, p1 in ((0, 4096), (n - blk - 4096, n - blk), (n - blk, n)):
                    gpu = _layer_rows(parser, cache.state_get(0, p0, p1), lay)
                    po, Ko, Vo = ref.parse_state(ref.state_get(0, p0, p1))
                    _compare_shifted(gpu, (po, Ko[0], Vo[0]), "rows [%d, %d)" % (p0, p1))
                want = ref.attn(0, [0], qh[None], 0.088)[0]
                got = o[lay, 0].cpu().numpy().astype(np.float64)
                for g in SAMPLED_HEADS:
                    assert_attn_close(got[g:g + 1], want[g:g + 1], "cycle 0 decode, head %d" % g)
            if c % 16 == 15:
                kc, ks, vc, vs = _export_layer(cache, kvc, torch, n, lay)
                assert kc.shape[0] == n
                want = _oracle_attn_stored(qh, kc, ks, vc, vs, 0.088, SAMPLED_HEADS)
                _close_on_heads(o[lay, 0].cpu().numpy(), want, SAMPLED_HEADS, "cycle %d decode" % c)
    finally:
        cache.close()


# ---------------------------------------------------------------- KeyDiff --
def test_full_keydiff_scores_and_window():
    """KeyDiff over a 131072-token q8_0 cache of 64 layers (the default
    layer, 32), then the retention-aware shift with n_keep 4, n_discard
    8192, n_recent 1024, as the benchmark runs them: every score against
    the oracle; the chosen window's oracle score sum within the score
    tolerance of the oracle's minimum; positions and layer 32's rows around
    the gap and at the tail against the oracle removing the same window."""
    torch, kvc, dev = _env()
    n, lay, keep, wd, recent = 131072, 32, 4, 8192, 1024
    cache = kvc.KVCache(L, H, HK, D, n + 512, 1, Q8, Q8, BASE)
    parser = oracle.OracleCache(L, H, HK, D, Q8, Q8, BASE, 0)
    ref = oracle.OracleCache(1, H, HK, D, Q8, Q8, BASE, 0)
    try:
        host = _fill([cache], torch, dev, n, 8192, keep=(lay,))
        ref.append(0, 0, 0, *host.pop(lay))
        got = cache.key_scores(0, -1).astype(np.float64)
        want = ref.key_scores(0, 0)
        assert got.shape == want.shape == (n,)
        assert np.abs(got - want).max() <= SCORE_TOL, np.abs(got - want).max()
        p0 = cache.evict_window(0, -1, keep, wd, recent)
        w_o = oracle.min_window(want, keep, n - recent, wd)
        assert keep <= p0 <= n - recent - wd
        pre = np.concatenate([[0.0], np.cumsum(want)])
        assert (pre[p0 + wd] - pre[p0]) - (pre[w_o + wd] - pre[w_o]) <= 2 * wd * SCORE_TOL, (p0, w_o)
        ref.seq_rm(0, p0, p0 + wd)
        ref.seq_add(0, p0 + wd, -1, -wd)
        assert np.array_equal(cache.positions(0), np.arange(n - wd))
        for a, b in ((max(0, p0 - 2048), p0 + 2048), (n - wd - 4096, n - wd)):
            gpu = _layer_rows(parser, cache.state_get(0, a, b), lay)
            po, Ko, Vo = ref.parse_state(ref.state_get(0, a, b))
            _compare_shifted(gpu, (po, Ko[0], Vo[0]), "rows [%d, %d)" % (a, b))
    finally:
        cache.close()
