"""Quantise-on-append at the edges of its arithmetic, through the append
kernel and through the fused decode step, compared byte for byte with the
oracle's state bytes.

fp16 (round to nearest even, IEEE-754 binary16): ties between neighbours,
subnormals and their ties, the largest finite value, values that round to it
or overflow to infinity, signed zero.  q8_0 (d = max|x| / 127, codes
round-half-away(x * (1/d)), fp16(d)): an all-zero block, blocks whose
products x * (1/d) are exact halves, a scale that underflows fp16, a scale
that overflows it, a lone non-zero element, mixed signs of equal magnitude.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

Q8, F16 = oracle.Q8_0, oracle.F16


def _f16_edges() -> np.ndarray:
    e = [0.0, -0.0, 1.0, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 1.0 - 2.0**-12, 2.0 - 2.0**-11,
         2.0**-24, 1.5 * 2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25,
         2.0**-14 - 2.0**-24, 65504.0, 65519.0, 65519.996, 65520.0, 65536.0, 1e6, 3.4e38,
         -65504.0, -65520.0, -1e6, -2.0**-25, -1.5 * 2.0**-24, 0.1, -0.1, 1.0 / 3.0, 1024.5, 2049.0]
    return np.float32(e)


def _q8_edge_blocks() -> np.ndarray:
    """Blocks of 32 values, one per row of the result."""
    blocks = []
    blocks.append(np.zeros(32))                                       # d = 0: codes 0, scale 0
    b = np.zeros(32)
    b[0] = 127.0                                                      # d = 1, 1/d = 1: exact halves
    b[1:12] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5, 63.5, -63.5, 0.49999997]
    blocks.append(b)
    b = np.zeros(32)
    b[5] = -254.0                                                     # d = 2: x * 0.5 ties at odd x
    b[6:14] = [1.0, 3.0, -5.0, 7.0, 253.0, -253.0, 0.999, 1.001]
    blocks.append(b)
    blocks.append(np.full(32, 1e-30))                                 # fp16(d) underflows to 0
    b = np.linspace(-1e7, 1e7, 32)                                    # fp16(d) overflows to inf
    blocks.append(b)
    b = np.zeros(32)
    b[31] = -3.0e-3                                                   # a lone element
    blocks.append(b)
    b = np.tile([0.75, -0.75], 16)                                    # equal magnitudes, both signs
    blocks.append(b)
    b = np.arange(32) - 15.5                                          # every code distinct
    blocks.append(b)
    return np.float32(np.array(blocks))


def _rows(type_, Hk, D, n):
    """n rows of [Hk][D] fp32 values that cover the edge cases."""
    if type_ == F16:
        e = _f16_edges()
        flat = np.resize(np.concatenate([e, -e[::-1]]), n * Hk * D)
    else:
        blk = _q8_edge_blocks().reshape(-1)
        flat = np.resize(blk, n * Hk * D)
    return np.ascontiguousarray(flat.reshape(n, Hk, D), np.float32)


@pytest.mark.parametrize("type_,D", [(F16, 64), (F16, 128), (Q8, 64), (Q8, 128)])
def test_append_and_fused_step_store_the_oracle_bytes(type_, D):
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    dev = torch.device("cuda:0")
    Hk, H, L, n = 2, 8, 2, 24
    k = _rows(type_, Hk, D, n)
    v = np.ascontiguousarray(k[::-1])
    ref = oracle.OracleCache(L, H, Hk, D, type_, type_, 1e4, 0)
    gpu = kvc.KVCache(L, H, Hk, D, 64, 1, type_, type_, 1e4, 0, kvc.KVC_DEVICE, 0, 16)
    try:
        # rows 0..n-2 through the append kernel, the last through the fused step
        for l in range(L):
            kd, vd = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
            gpu.append(l, 0, 0, kd[: n - 1], vd[: n - 1])
            q = torch.zeros(1, H, D, device=dev)
            o = torch.empty_like(q)
            gpu.decode_step(l, [0], [n - 1], kd[n - 1:], vd[n - 1:], q, o, 0.125)
            ref.append(l, 0, 0, k, v)
        torch.cuda.synchronize()
        assert gpu.state_get(0, -1, -1) == ref.state_get(0, -1, -1)
        assert kvc.kvc_check_device_error(gpu.ctx) == 0
    finally:
        gpu.close()
