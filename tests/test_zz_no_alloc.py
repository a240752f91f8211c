"""kvc_attn_decode_static: decode attention that allocates nothing.

It serves callers that cannot let a library allocate device memory (runtimes
that hand out all device memory from their own arena, latency-critical paths
that cannot take an allocation's synchronisation).  The test builds a cache
through the usual context, exports one layer's K/V as state bytes, uploads
that layer into buffers the test owns (the head-major layout the entry point
takes), and checks two consecutive calls of the no-alloc entry point against
kvc_attn_decode on the same rows, within the attention tolerances used by
the other GPU tests.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
from twin import TOL_MAX_ABS, TOL_REL_L2, kv_inputs, q_inputs

pytestmark = pytest.mark.gpu


def _sections(blob, H, Hk, D, type_, n):
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


@pytest.mark.parametrize("type_,n", [(oracle.Q8_0, 5000), (oracle.F16, 3001), (oracle.Q8_0, 1)])
def test_no_alloc_entry_matches_kvc_attn_decode(type_, n):
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    H, Hk, D = 40, 8, 128
    dev = torch.device("cuda:0")
    cache = kvc.KVCache(1, H, Hk, D, n + 64, 1, type_, type_, 1e6)
    try:
        k, v = kv_inputs(21, 0, n, Hk, D, sigma=0.5)
        cache.append(0, 0, 0, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev))
        q = torch.from_numpy(q_inputs(21, 0, 1, H, D)).to(dev)
        ref = torch.empty_like(q)
        scale = float(1 / np.sqrt(D))
        cache.attn_decode(0, [0], q, ref, scale)
        torch.cuda.synchronize()
        (kd, ks), (vd, vs) = _sections(cache.state_get(0, -1, -1), H, Hk, D, type_, n)
        buf = lambda b: torch.frombuffer(bytearray(b), dtype=torch.uint8).to(dev) if b is not None else None
        kt, kst, vt, vst = buf(kd), buf(ks), buf(vd), buf(vs)
        ptr = lambda t: t.data_ptr() if t is not None else None
        f = kvc.load().kvc_attn_decode_static
        f.restype = C.c_int
        f.argtypes = [C.c_int] * 5 + [C.c_void_p] * 6 + [C.c_float, C.c_void_p]
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):  # the work space keeps the previous call's contents
            out = torch.full_like(q, float("nan"))
            rc = f(type_, H, Hk, D, n, ptr(kt), ptr(kst), ptr(vt), ptr(vst), q.data_ptr(), out.data_ptr(), scale,
                   stream)
            assert rc == kvc.KVC_OK, rc
            torch.cuda.synchronize()
            a, b = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
            err = np.abs(a - b).max()
            rel = np.linalg.norm(a - b) / np.linalg.norm(b)
            assert err <= TOL_MAX_ABS and rel <= TOL_REL_L2, (call, err, rel)
        # sizes beyond the fixed work space are rejected, not truncated
        rc = f(type_, H, Hk, D, 1 << 27, ptr(kt), ptr(kst), ptr(vt), ptr(vst), q.data_ptr(), out.data_ptr(),
               scale, stream)
        assert rc == kvc.KVC_ERANGE
    finally:
        cache.close()
