"""A GPU cache (through the C ABI) and the oracle, fed the same seeded inputs.

Inputs come from kv_cache_decode_flash_gb300.synth (numpy); the oracle never
sees anything the CUDA path produced.
"""
import numpy as np

import oracle
from kv_cache_decode_flash_gb300 import synth

TOL_MAX_ABS = 1e-3  # attention tolerances stated for the decode path
TOL_REL_L2 = 1e-4


def kv_inputs(seed, layer, n, Hk, D, pos0=0, sigma=1.0, tag=""):
    """fp32 K and V rows [n][Hk][D] of one layer; `pos0` offsets the stream so
    that later appends draw fresh numbers."""
    kind_k, kind_v = ("knew", "vnew") if tag else ("k", "v")
    extra = pos0
    k = synth.normal(seed, synth.stream_id(kind_k, layer, extra), n * Hk * D, sigma).reshape(n, Hk, D)
    v = synth.normal(seed, synth.stream_id(kind_v, layer, extra), n * Hk * D, sigma).reshape(n, Hk, D)
    return k, v


def q_inputs(seed, layer, n_seq, H, D, extra=0):
    return synth.normal(seed, synth.stream_id("q", layer, extra), n_seq * H * D).reshape(n_seq, H, D)


class Twin:
    def __init__(self, n_layer, H, Hk, D, n_ctx, n_seq_max=1, type_=8, rope_base=10000.0, rope_mode=0,
                 page_rows=0, residency=0, type_v=None):
        import torch

        from kv_cache_decode_flash_gb300 import kvc

        self.torch, self.kvc = torch, kvc
        self.dev = torch.device("cuda:0")
        self.H, self.Hk, self.D, self.L = H, Hk, D, n_layer
        tv = type_ if type_v is None else type_v
        self.gpu = kvc.KVCache(n_layer, H, Hk, D, n_ctx, n_seq_max, type_, tv, rope_base, rope_mode,
                               residency, 0, page_rows)
        self.ref = oracle.OracleCache(n_layer, H, Hk, D, type_, tv, rope_base, rope_mode)

    def close(self):
        self.gpu.close()

    def append(self, layer, seq, pos0, k, v):
        t = self.torch
        self.gpu.append(layer, seq, pos0, t.from_numpy(np.ascontiguousarray(k)).to(self.dev),
                        t.from_numpy(np.ascontiguousarray(v)).to(self.dev))
        self.ref.append(layer, seq, pos0, k, v)

    def fill(self, seq, n, seed=0, pos0=0, sigma=1.0):
        for l in range(self.L):
            k, v = kv_inputs(seed, l, n, self.Hk, self.D, pos0=pos0 + 1000003 * seq, sigma=sigma)
            self.append(l, seq, pos0, k, v)

    def attn(self, layer, seq_ids, q, kq_scale, heads=None):
        t = self.torch
        qd = t.from_numpy(np.ascontiguousarray(q, np.float32)).to(self.dev)
        out = t.empty_like(qd)
        self.gpu.attn_decode(layer, list(seq_ids), qd, out, kq_scale)
        t.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        want = self.ref.attn(layer, list(seq_ids), q, float(np.float32(kq_scale)), heads)
        return got, want


def attn_errors(got, want):
    err = float(np.abs(got - want).max())
    den = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))
    return err, rel


def assert_attn_close(got, want, what=""):
    err, rel = attn_errors(got, want)
    assert err <= TOL_MAX_ABS and rel <= TOL_REL_L2, "%s: max abs %.3g, rel L2 %.3g" % (what, err, rel)
    return err, rel
