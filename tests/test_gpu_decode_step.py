"""The fused decode step (kvc_decode_step) against the two calls it stands for
(kvc_append of each sequence's token, then kvc_attn_decode) and the oracle.

Bit-exact: outputs and stored rows (state bytes) of the fused step equal those
of the two calls; the stored rows equal the oracle's quantisation.  Tolerance
against the oracle: attention max abs 1e-3 and relative L2 1e-4.  Steps are
enqueued back to back on one stream without synchronising, so each launch
overlaps the one before it as in a model's decode loop.
"""
import numpy as np
import pytest

import oracle
from twin import kv_inputs, q_inputs, assert_attn_close

pytestmark = pytest.mark.gpu

Q8, F16 = oracle.Q8_0, oracle.F16


def _pair(L, H, Hk, D, n_ctx, n_seq_max, type_, page_rows, chunk):
    from kv_cache_decode_flash_gb300 import kvc

    a = kvc.KVCache(L, H, Hk, D, n_ctx, n_seq_max, type_, type_, 1e4, 0, kvc.KVC_DEVICE, 0, page_rows)
    b = kvc.KVCache(L, H, Hk, D, n_ctx, n_seq_max, type_, type_, 1e4, 0, kvc.KVC_DEVICE, 0, page_rows)
    if chunk:
        kvc.kvc_set_chunk_rows(a.ctx, chunk)
        kvc.kvc_set_chunk_rows(b.ctx, chunk)
    return a, b


def _run_steps(a, b, ref, L, H, Hk, D, seqs, lens, steps, seed, scale, check_every=1):
    """Prefill `lens` rows per sequence, then `steps` decode steps over all
    layers; returns the fused and two-call outputs [step][layer] and the
    oracle's for the checked steps."""
    import torch

    dev = torch.device("cuda:0")
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    for s, n in zip(seqs, lens):
        if n:
            for l in range(L):
                k, v = kv_inputs(seed, l, n, Hk, D, pos0=1000003 * s)
                a.append(l, s, 0, T(k), T(v))
                b.append(l, s, 0, T(k), T(v))
                ref.append(l, s, 0, k, v)
    ns = len(seqs)
    inputs = []
    for t in range(steps):
        per_layer = []
        for l in range(L):
            kv = [kv_inputs(seed + 1, l, 1, Hk, D, pos0=1000003 * s + lens[i] + t) for i, s in enumerate(seqs)]
            k = np.concatenate([x[0] for x in kv])
            v = np.concatenate([x[1] for x in kv])
            q = q_inputs(seed + 2, l, ns, H, D, extra=t)
            per_layer.append((k, v, q))
        inputs.append(per_layer)
    dk = [[(T(k), T(v), T(q)) for (k, v, q) in step] for step in inputs]
    oa = torch.empty(steps, L, ns, H, D, device=dev)
    ob = torch.empty_like(oa)
    torch.cuda.synchronize()
    for t in range(steps):
        pos = [lens[i] + t for i in range(ns)]
        for l in range(L):
            k, v, q = dk[t][l]
            a.decode_step(l, seqs, pos, k, v, q, oa[t, l], scale)
    for t in range(steps):
        for l in range(L):
            k, v, q = dk[t][l]
            for i, s in enumerate(seqs):
                b.append(l, s, lens[i] + t, k[i:i + 1], v[i:i + 1])
            b.attn_decode(l, seqs, q, ob[t, l], scale)
    torch.cuda.synchronize()
    want = {}
    for t in range(steps):
        for l in range(L):
            k, v, q = inputs[t][l]
            for i, s in enumerate(seqs):
                ref.append(l, s, lens[i] + t, k[i:i + 1], v[i:i + 1])
            if t % check_every == 0 or t == steps - 1:
                want[(t, l)] = ref.attn(l, list(seqs), q, float(np.float32(scale)))
    return oa.cpu().numpy(), ob.cpu().numpy(), want


def _check(a, b, ref, seqs, oa, ob, want):
    assert np.array_equal(oa, ob), "fused step differs from append + attention"
    for (t, l), w in want.items():
        assert_attn_close(oa[t, l].astype(np.float64), w, "step %d layer %d" % (t, l))
    for s in seqs:
        ga, gb = a.state_get(s, -1, -1), b.state_get(s, -1, -1)
        assert ga == gb, "stored rows differ (sequence %d)" % s
        assert ga == ref.state_get(s, -1, -1), "stored rows differ from the oracle (sequence %d)" % s


@pytest.mark.parametrize("type_,D,page_rows,chunk", [(Q8, 128, 0, 0), (F16, 128, 0, 0), (Q8, 64, 16, 0),
                                                     (F16, 64, 16, 32), (Q8, 128, 32, 16), (Q8, 128, 64, 48)])
def test_decode_step_matches_two_calls_and_oracle(type_, D, page_rows, chunk):
    """Pages of 16 to 256 rows (a page is allocated inside many steps), forced
    chunks of 16 to 48 rows (the new row at every tile and chunk position)."""
    L, H, Hk = 2, (40 if D == 128 else 8), (8 if D == 128 else 2)
    a, b = _pair(L, H, Hk, D, 1200, 1, type_, page_rows, chunk)
    ref = oracle.OracleCache(L, H, Hk, D, type_, type_, 1e4, 0)
    try:
        oa, ob, want = _run_steps(a, b, ref, L, H, Hk, D, [0], [301], 40, 31, 0.088, check_every=7)
        _check(a, b, ref, [0], oa, ob, want)
        assert a.n_tokens(0) == 341 and np.array_equal(a.positions(0), np.arange(341))
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("type_", [Q8, F16])
def test_decode_step_one_layer_back_to_back(type_):
    """One layer: every launch attends over the row the launch before it
    stored (the next launch may start before that row is written, so it must
    not read it before its wait).  Starts from an empty sequence."""
    a, b = _pair(1, 8, 2, 64, 600, 1, type_, 16, 0)
    ref = oracle.OracleCache(1, 8, 2, 64, type_, type_, 1e4, 0)
    try:
        oa, ob, want = _run_steps(a, b, ref, 1, 8, 2, 64, [0], [0], 200, 41, 0.125, check_every=9)
        _check(a, b, ref, [0], oa, ob, want)
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("type_", [Q8, F16])
def test_decode_step_ragged_batch(type_):
    """Sequences of 0 to 2100 rows (one empty before the step) in one call,
    addressed in a permuted order."""
    lens = [1000, 0, 15, 16, 17, 255, 2100]
    seqs = [6, 1, 0, 3, 2, 5, 4]
    L, H, Hk, D = 2, 32, 8, 128
    a, b = _pair(L, H, Hk, D, sum(lens) + 400, 7, type_, 128, 0)
    ref = oracle.OracleCache(L, H, Hk, D, type_, type_, 1e4, 0)
    try:
        oa, ob, want = _run_steps(a, b, ref, L, H, Hk, D, seqs, lens, 5, 51, 0.0884, check_every=2)
        _check(a, b, ref, seqs, oa, ob, want)
    finally:
        a.close()
        b.close()


def test_decode_step_many_sequences_multiple_launches():
    """70 sequences: more than one launch carries them."""
    n_seq = 70
    seqs = list(range(n_seq))
    lens = [5 + (s * 7) % 33 for s in seqs]
    a, b = _pair(1, 8, 2, 64, sum(lens) + 70 * 40, n_seq, Q8, 16, 0)
    ref = oracle.OracleCache(1, 8, 2, 64, Q8, Q8, 1e4, 0)
    try:
        oa, ob, want = _run_steps(a, b, ref, 1, 8, 2, 64, seqs, lens, 3, 61, 0.125)
        _check(a, b, ref, seqs, oa, ob, want)
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("residency", ["host", "split"])
def test_decode_step_host_and_split_contexts(residency):
    """Host-resident and split contexts run the two calls: the same bytes as
    calling them, through the staging ring."""
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    L, H, Hk, D, n = 3, 40, 8, 128, 700
    dev = torch.device("cuda:0")
    res = kvc.KVC_HOST_PINNED if residency == "host" else kvc.KVC_SPLIT_HEADS
    G = 0 if residency == "host" else 3
    outs = []
    for fused in (True, False):
        c = kvc.KVCache(L, H, Hk, D, n + 16, 1, Q8, Q8, 1e4, 0, res, 0, 0, G)
        try:
            for l in range(L):
                c.append(l, 0, 0, *[torch.from_numpy(x).to(dev) for x in kv_inputs(71, l, n, Hk, D)])
            got = []
            for t in range(3):
                for l in range(L):
                    k, v = [torch.from_numpy(x).to(dev) for x in kv_inputs(72, l, 1, Hk, D, pos0=n + t)]
                    q = torch.from_numpy(q_inputs(73, l, 1, H, D, extra=t)).to(dev)
                    o = torch.empty_like(q)
                    if fused:
                        c.decode_step(l, [0], [n + t], k, v, q, o, 0.0884)
                    else:
                        c.append(l, 0, n + t, k, v)
                        c.attn_decode(l, [0], q, o, 0.0884)
                    got.append(o.cpu().numpy())
            assert c.n_tokens(0) == n + 3
            outs.append(np.stack(got))
        finally:
            c.close()
    assert np.array_equal(outs[0], outs[1])


def test_decode_step_rejects_bad_calls_without_change():
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    dev = torch.device("cuda:0")
    # 2 layers, pages of 16 rows: 64 / 16 + 2 = 6 pages in all
    c = kvc.KVCache(2, 8, 2, 64, 64, 2, Q8, Q8, 1e4, 0, kvc.KVC_DEVICE, 0, 16)
    try:
        for s, n in ((0, 16), (1, 64)):  # 1 + 4 pages: one left
            for l in range(2):
                c.append(l, s, 0, *[torch.from_numpy(x).to(dev) for x in kv_inputs(81, l, n, 2, 64, pos0=s)])
        k = torch.zeros(2, 2, 64, device=dev)
        v = torch.zeros_like(k)
        q = torch.zeros(2, 8, 64, device=dev)
        o = torch.empty_like(q)
        torch.cuda.synchronize()
        before = [c.state_get(s, -1, -1) for s in (0, 1)]

        def rejected(status, fn):
            with pytest.raises(kvc.KvcError) as e:
                fn()
            assert e.value.status == status
            torch.cuda.synchronize()
            assert [c.state_get(s, -1, -1) for s in (0, 1)] == before
            assert (c.n_tokens(0), c.n_tokens(1)) == (16, 64)

        one = (k[:1], v[:1], q[:1], o[:1])
        rejected(kvc.KVC_EINVAL, lambda: c.decode_step(0, [0, 0], [16, 17], k, v, q, o, 0.1))  # duplicate id
        rejected(kvc.KVC_EINVAL, lambda: c.decode_step(0, [0, 2], [16, 64], k, v, q, o, 0.1))  # id out of range
        rejected(kvc.KVC_EINVAL, lambda: c.decode_step(2, [0], [16], *one, 0.1))  # layer out of range
        rejected(kvc.KVC_EINVAL, lambda: c.decode_step(0, [0], [16], k[:1], v[:1], q[:1], q[:1], 0.1))  # alias
        rejected(kvc.KVC_EINVAL, lambda: c.decode_step(0, [0], [16], *one, float("nan")))
        rejected(kvc.KVC_ERANGE, lambda: c.decode_step(0, [0], [-1], *one, 0.1))
        # each sequence needs a new page and one is free: nothing is taken
        rejected(kvc.KVC_ENOSPC, lambda: c.decode_step(0, [1, 0], [64, 16], k, v, q, o, 0.1))
        with pytest.raises(ValueError):
            c.decode_step(0, [0, 1], [16], k, v, q, o, 0.1)
        # the free page serves sequence 0; layer 1 must then append the position layer 0 created
        c.decode_step(0, [0], [16], *one, 0.1)
        with pytest.raises(kvc.KvcError) as e:
            c.decode_step(1, [0], [17], *one, 0.1)
        assert e.value.status == kvc.KVC_EINVAL
        c.decode_step(1, [0], [16], *one, 0.1)
        torch.cuda.synchronize()
        assert c.n_tokens(0) == 17 and c.n_tokens(1) == 64
        assert kvc.kvc_check_device_error(c.ctx) == 0
    finally:
        c.close()


def test_decode_step_in_cuda_graph():
    """A captured step of 4 layers (the row re-appended at the same position on
    every replay, the rows before it untouched) gives the eager step's bytes."""
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    L, H, Hk, D, n = 4, 40, 8, 128, 3000
    dev = torch.device("cuda:0")
    c = kvc.KVCache(L, H, Hk, D, n + 64, 1, Q8, Q8, 1e4, 0, kvc.KVC_DEVICE, 0, 0)
    try:
        for l in range(L):
            c.append(l, 0, 0, *[torch.from_numpy(x).to(dev) for x in kv_inputs(91, l, n - 1, Hk, D)])
        kn = [[torch.from_numpy(x).to(dev) for x in kv_inputs(92, l, 1, Hk, D, pos0=n)] for l in range(L)]
        qs = [torch.from_numpy(q_inputs(93, l, 1, H, D)).to(dev) for l in range(L)]
        eager = torch.empty(L, 1, H, D, device=dev)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for l in range(L):
                c.decode_step(l, [0], [n - 1], kn[l][0], kn[l][1], qs[l], eager[l], 0.0884, stream=s)
        s.synchronize()
        state = c.state_get(0, -1, -1)
        c.seq_rm(0, n - 1, -1)
        out = torch.zeros_like(eager)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for l in range(L):
                c.decode_step(l, [0], [n - 1], kn[l][0], kn[l][1], qs[l], out[l], 0.0884,
                              stream=torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, eager)
            out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert c.state_get(0, -1, -1) == state
        assert kvc.kvc_check_device_error(c.ctx) == 0
    finally:
        c.close()
