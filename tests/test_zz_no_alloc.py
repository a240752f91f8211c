"""kvc_attn_decode_static: decode attention that allocates nothing.

It serves callers that cannot let a library allocate device memory (runtimes
that hand out all device memory from their own arena, latency-critical paths
that cannot take an allocation's synchronisation).  The test builds a cache
through the usual context, exports one layer's K/V as state bytes, uploads
that layer into buffers the test owns (the head-major layout the entry point
takes), and checks two consecutive calls of the no-alloc entry point against
the oracle run on the same fp32 inputs, within the attention tolerances of
the other GPU tests, and against kvc_attn_decode.  Around the second call
the device's free memory must not change.  An empty sequence gives zeros,
and sizes whose partials do not fit the fixed work space are rejected.
This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
from twin import TOL_MAX_ABS, assert_attn_close, kv_inputs, q_inputs

pytestmark = pytest.mark.gpu


def _sections(blob, Hk, D, type_, n):
    """Split a one-layer state blob into its K and V sections (bytes)."""
    pad = lambda x: (x + 15) // 16 * 16
    off = 64 + pad(4 * n)
    out = []
    for _ in range(2):  # K then V
        if type_ == oracle.Q8_0:
            data = blob[off:off + pad(Hk * n * D)]
            off += pad(Hk * n * D)
            sc = blob[off:off + pad(Hk * n * (D // 32) * 2)]
            off += pad(Hk * n * (D // 32) * 2)
        else:
            data = blob[off:off + pad(Hk * n * D * 2)]
            off += pad(Hk * n * D * 2)
            sc = None
        out.append((data, sc))
    return out


def _entry():
    from kv_cache_decode_flash_gb300 import kvc

    f = kvc.load().kvc_attn_decode_static
    f.restype = C.c_int
    f.argtypes = [C.c_int] * 5 + [C.c_void_p] * 6 + [C.c_float, C.c_void_p]
    return f


@pytest.mark.parametrize("type_,n", [(oracle.Q8_0, 5000), (oracle.F16, 3001), (oracle.Q8_0, 1)])
def test_no_alloc_entry_matches_oracle(type_, n):
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    H, Hk, D = 40, 8, 128
    dev = torch.device("cuda:0")
    cache = kvc.KVCache(1, H, Hk, D, n + 64, 1, type_, type_, 1e6)
    try:
        k, v = kv_inputs(21, 0, n, Hk, D, sigma=0.5)
        qh = q_inputs(21, 0, 1, H, D)
        scale = float(1 / np.sqrt(D))
        ref = oracle.OracleCache(1, H, Hk, D, type_, type_, 1e6)
        ref.append(0, 0, 0, k, v)
        want = ref.attn(0, [0], qh, float(np.float32(scale)))

        cache.append(0, 0, 0, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev))
        q = torch.from_numpy(qh).to(dev)
        via_ctx = torch.empty_like(q)
        cache.attn_decode(0, [0], q, via_ctx, scale)
        torch.cuda.synchronize()
        (kd, ks), (vd, vs) = _sections(cache.state_get(0, -1, -1), Hk, D, type_, n)
        buf = lambda b: torch.frombuffer(bytearray(b), dtype=torch.uint8).to(dev) if b is not None else None
        kt, kst, vt, vst = buf(kd), buf(ks), buf(vd), buf(vs)
        ptr = lambda t: t.data_ptr() if t is not None else None
        f = _entry()
        stream = torch.cuda.current_stream().cuda_stream
        outs = [torch.full_like(q, float("nan")) for _ in range(2)]
        torch.cuda.synchronize()
        for call in range(2):  # the work space keeps the previous call's contents
            free0 = torch.cuda.mem_get_info()[0]
            rc = f(type_, H, Hk, D, n, ptr(kt), ptr(kst), ptr(vt), ptr(vst), q.data_ptr(), outs[call].data_ptr(),
                   scale, stream)
            assert rc == kvc.KVC_OK, rc
            torch.cuda.synchronize()
            if call == 1:  # the first call may load the library's device code; later ones take nothing
                assert torch.cuda.mem_get_info()[0] == free0
            got = outs[call].cpu().numpy().astype(np.float64)
            assert_attn_close(got, want, "no-alloc call %d" % call)
        # two calls in a row give the same bits, and agree with the context path
        assert torch.equal(outs[0], outs[1])
        err = (outs[1] - via_ctx).abs().max().item()
        assert err <= TOL_MAX_ABS, err
    finally:
        cache.close()


def test_no_alloc_empty_sequence_gives_zeros():
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    H, Hk, D = 40, 8, 128
    dev = torch.device("cuda:0")
    q = torch.from_numpy(q_inputs(3, 0, 1, H, D)).to(dev)
    f = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    for type_ in (oracle.Q8_0, oracle.F16):
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            rc = f(type_, H, Hk, D, 0, None, None, None, None, q.data_ptr(), out.data_ptr(), 0.088, stream)
            assert rc == kvc.KVC_OK, rc
            torch.cuda.synchronize()
            assert torch.count_nonzero(out).item() == 0


def test_no_alloc_rejects_partials_beyond_the_work_space():
    """Group size 5 runs the group-size-8 kernel instance, whose partials are
    larger: a length whose group-5 partials would fit but whose launched
    partials do not (about 320 chunks per KV head here, against the 251 the
    8 MiB work space holds) is rejected.  The buffers are real, so the call
    would read inside them even if the check were missing."""
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    H, Hk, D, n = 40, 8, 128, 2_500_000
    dev = torch.device("cuda:0")
    kt = torch.empty(Hk * n * D, dtype=torch.uint8, device=dev)
    vt = torch.empty_like(kt)
    kst = torch.empty(Hk * n * (D // 32) * 2 + 16, dtype=torch.uint8, device=dev)
    vst = torch.empty_like(kst)
    q = torch.from_numpy(q_inputs(5, 0, 1, H, D)).to(dev)
    out = torch.zeros_like(q)
    f = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(oracle.Q8_0, H, Hk, D, n, kt.data_ptr(), kst.data_ptr(), vt.data_ptr(), vst.data_ptr(), q.data_ptr(),
           out.data_ptr(), 0.088, stream)
    assert rc == kvc.KVC_ERANGE, rc
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing was launched
    del kt, vt, kst, vst
    torch.cuda.empty_cache()
