"""The asymmetric cache (q8_0 K, q4_0 V: "F5 - Advanced KV Cache Techniques",
section M6 - PolyKV, "-ctk q8_0 -ctv q4_0") through the C ABI against the
oracle.

Bit-exact: stored q4_0 V bytes after append (and after the fused decode step)
equal the oracle's quantisation, and the hand-derived golden blocks; seq_cp /
seq_rm / state export and import as state bytes; V bytes are untouched by a
RoPE shift.  Tolerance: attention max abs 1e-3 and relative L2 1e-4.
"""
import numpy as np
import pytest

import oracle
from golden_io import q4_0_blocks
from twin import Twin, assert_attn_close, kv_inputs, q_inputs

pytestmark = pytest.mark.gpu

Q8, Q4 = oracle.Q8_0, oracle.Q4_0


def _twin(L, H, Hk, n_ctx, n_seq_max=1, page_rows=0):
    return Twin(L, H, Hk, 128, n_ctx, n_seq_max=n_seq_max, type_=Q8, type_v=Q4, page_rows=page_rows)


def test_q4_0_append_bit_exact():
    tw = _twin(2, 8, 2, 1000, page_rows=64)
    try:
        for l in range(2):
            k, v = kv_inputs(31, l, 300, 2, 128)
            tw.append(l, 0, 0, k, v)
        for l in range(2):
            k, v = kv_inputs(32, l, 77, 2, 128, pos0=300)
            tw.append(l, 0, 300, k, v)
        assert tw.gpu.state_get(0, -1, -1) == tw.ref.state_get(0, -1, -1)
    finally:
        tw.close()


def test_q4_0_golden_blocks_through_the_append_kernel():
    """The hand-derived blocks as V rows (four blocks per 128-value head-row):
    the stored bytes and scales are the fixture's."""
    import torch

    blocks = q4_0_blocks()
    rows = [np.concatenate([blocks[(r + j) % len(blocks)][1] for j in range(4)]) for r in range(len(blocks))]
    v = np.stack(rows).astype(np.float32).reshape(len(rows), 1, 128)
    k = np.zeros_like(v)
    tw = Twin(1, 4, 1, 128, 64, type_=Q8, type_v=Q4)
    try:
        dev = torch.device("cuda:0")
        tw.gpu.append(0, 0, 0, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev))
        _, _, V = tw.ref.parse_state(tw.gpu.state_get(0, -1, -1))
        for r in range(len(rows)):
            for j in range(4):
                _, _, _, packed, scale = blocks[(r + j) % len(blocks)]
                assert V[0].a[r, 0, 16 * j:16 * j + 16].tobytes() == packed.tobytes(), (r, j)
                assert int(V[0].s[r, 0, j]) == scale, (r, j)
    finally:
        tw.close()


@pytest.mark.parametrize("n", [1, 17, 555, 1000, 5000])
def test_q4_0_attention_vs_oracle(n):
    tw = _twin(1, 40, 8, n + 64)
    try:
        tw.fill(0, n, seed=33, sigma=0.5)
        q = q_inputs(33, 0, 1, 40, 128)
        scale = float(np.float32(1 / np.sqrt(128)))
        got, want = tw.attn(0, [0], q, scale)
        assert_attn_close(got, want, "n %d" % n)
        again, _ = tw.attn(0, [0], q, scale)
        assert np.array_equal(got, again)
    finally:
        tw.close()


@pytest.mark.parametrize("r", [3, 4, 5, 8])
def test_q4_0_group_sizes_and_chunks(r):
    tw = _twin(1, 2 * r, 2, 1100)
    try:
        tw.fill(0, 1000, seed=34)
        q = q_inputs(34, 0, 1, 2 * r, 128)
        for C in (32, 128, 256, 1008, 0):
            tw.kvc.kvc_set_chunk_rows(tw.gpu.ctx, C)
            got, want = tw.attn(0, [0], q, 0.088)
            assert_attn_close(got, want, "r %d chunk %d" % (r, C))
    finally:
        tw.close()


def test_q4_0_ragged_batch():
    lens = [0, 1, 15, 16, 17, 255, 256, 257, 1000, 2100]
    tw = _twin(1, 32, 8, sum(lens) + 64, n_seq_max=len(lens), page_rows=128)
    try:
        for s, n in enumerate(lens):
            if n:
                tw.fill(s, n, seed=35)
        q = q_inputs(35, 0, len(lens), 32, 128)
        got, want = tw.attn(0, list(range(len(lens))), q, 0.0884)
        assert_attn_close(got, want, "ragged batch")
        assert np.all(got[0] == 0)
    finally:
        tw.close()


def test_q4_0_decode_step_equals_two_calls_and_oracle():
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    L, H, Hk, D, n = 2, 40, 8, 128, 700
    dev = torch.device("cuda:0")
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    a = kvc.KVCache(L, H, Hk, D, n + 64, 1, Q8, Q4, 1e4, 0, kvc.KVC_DEVICE, 0, 64)
    b = kvc.KVCache(L, H, Hk, D, n + 64, 1, Q8, Q4, 1e4, 0, kvc.KVC_DEVICE, 0, 64)
    ref = oracle.OracleCache(L, H, Hk, D, Q8, Q4, 1e4, 0)
    try:
        for l in range(L):
            k, v = kv_inputs(36, l, n, Hk, D)
            for c in (a, b):
                c.append(l, 0, 0, T(k), T(v))
            ref.append(l, 0, 0, k, v)
        s = torch.cuda.Stream(device=dev)
        oa = torch.empty(3, L, 1, H, D, device=dev)
        ob = torch.empty_like(oa)
        qs, news = [], []
        with torch.cuda.stream(s):
            for t in range(3):
                for l in range(L):
                    k, v = kv_inputs(37, l, 1, Hk, D, pos0=n + t)
                    q = q_inputs(38, l, 1, H, D, extra=t)
                    qs.append(q)
                    news.append((l, k, v))
                    a.decode_step(l, [0], [n + t], T(k), T(v), T(q), oa[t, l], 0.088, stream=s)
                    b.append(l, 0, n + t, T(k), T(v), stream=s)
                    b.attn_decode(l, [0], T(q), ob[t, l], 0.088, stream=s)
        s.synchronize()
        assert torch.equal(oa, ob)
        assert a.state_get(0, -1, -1) == b.state_get(0, -1, -1)
        i = 0
        for t in range(3):
            for l in range(L):
                _, k, v = news[i]
                ref.append(l, 0, n + t, k, v)
                want = ref.attn(l, [0], qs[i], 0.088)
                assert_attn_close(oa[t, l].cpu().numpy().astype(np.float64), want, "step %d layer %d" % (t, l))
                i += 1
        assert a.state_get(0, -1, -1) == ref.state_get(0, -1, -1)
    finally:
        a.close()
        b.close()


def test_q4_0_seq_ops_state_and_shift():
    tw = _twin(2, 8, 2, 2048, n_seq_max=3, page_rows=32)
    try:
        tw.fill(0, 500, seed=39)
        for op in [("cp", 0, 1, 40, 300), ("rm", 0, 100, 150), ("rm", 0, 0, 37), ("cp", 1, 2, -1, -1)]:
            getattr(tw.gpu, "seq_" + op[0])(*op[1:])
            getattr(tw.ref, "seq_" + op[0])(*op[1:])
            for s in range(3):
                assert tw.gpu.state_get(s, -1, -1) == tw.ref.state_get(s, -1, -1), op
        blob = tw.gpu.state_get(0, 200, 400)
        assert blob == tw.ref.state_get(0, 200, 400)
        tw.gpu.state_set(2, blob)
        tw.ref.state_set(2, blob)
        assert tw.gpu.state_get(2, -1, -1) == tw.ref.state_get(2, -1, -1)
        # a RoPE shift requantises K only: the V sections stay bit for bit
        before = tw.ref.parse_state(tw.gpu.state_get(0, -1, -1))
        tw.gpu.seq_add(0, 150, -1, -30)
        tw.ref.seq_add(0, 150, -1, -30)
        after = tw.ref.parse_state(tw.gpu.state_get(0, -1, -1))
        for l in range(2):
            assert np.array_equal(before[2][l].a, after[2][l].a) and np.array_equal(before[2][l].s, after[2][l].s)
        _, Ko, _ = tw.ref.parse_state(tw.ref.state_get(0, -1, -1))
        for l in range(2):
            assert np.abs(after[1][l].a.astype(int) - Ko[l].a.astype(int)).max() <= 1
            assert np.abs(after[1][l].s.astype(int) - Ko[l].s.astype(int)).max() <= 1
        q = q_inputs(39, 1, 1, 8, 128)
        got, want = tw.attn(1, [2], q, 0.125)
        assert_attn_close(got, want, "copied and imported rows")
    finally:
        tw.close()


def test_q4_0_host_resident_ordered_and_pipelined_vs_oracle():
    from kv_cache_decode_flash_gb300 import kvc

    n = 3000
    tw = Twin(4, 40, 8, 128, n + 64, type_=Q8, type_v=Q4, residency=kvc.KVC_HOST_PINNED)
    try:
        tw.fill(0, n, seed=40, sigma=0.5)
        q = q_inputs(40, 3, 1, 40, 128)
        kvc.kvc_pipeline_depth(tw.gpu.ctx, 0)
        got0, want = tw.attn(3, [0], q, 0.088)
        assert_attn_close(got0, want, "ordered")
        kvc.kvc_pipeline_depth(tw.gpu.ctx, 1)
        kvc.kvc_pipeline_budget(tw.gpu.ctx, 512 << 20)
        got1, _ = tw.attn(3, [0], q, 0.088)
        assert np.array_equal(got0, got1)
    finally:
        tw.close()


def test_q4_0_rejected_combinations():
    from kv_cache_decode_flash_gb300 import kvc

    for tk, tv, D in ((Q4, Q4, 128), (oracle.F16, Q4, 128), (Q8, Q4, 64)):
        with pytest.raises(kvc.KvcError):
            kvc.KVCache(1, 8, 2, D, 64, 1, tk, tv)
