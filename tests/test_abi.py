"""The C-ABI library loads and exports every function include/kvc.h declares
(no compute calls: this runs without a GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("kvc_create", "kvc_destroy", "kvc_append", "kvc_attn_decode", "kvc_seq_rm", "kvc_seq_cp",
              "kvc_seq_add", "kvc_state_get", "kvc_state_set", "kvc_pipeline_depth", "kvc_pipeline_budget"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from kv_cache_decode_flash_gb300 import build, kvc

    build.build()
    L = kvc.load()
    missing = [n for n in declared() if not hasattr(L, n)]
    assert not missing, missing


def test_params_init_and_status_strings():
    from kv_cache_decode_flash_gb300 import kvc

    p = kvc.kvc_params_init()
    assert (p.n_layer, p.n_head, p.n_head_kv, p.head_dim, p.n_ctx) == (1, 8, 2, 64, 512)
    assert (p.type_k, p.type_v, p.residency, p.rope_mode) == (kvc.KVC_Q8_0, kvc.KVC_Q8_0, 0, 0)
    assert kvc.load().kvc_status_str(kvc.KVC_EFORMAT) == b"bad state format"


def test_create_rejects_bad_geometry_without_touching_a_gpu():
    from kv_cache_decode_flash_gb300 import kvc

    # q4_0 is a V type (with q8_0 K and head_dim 128; the default head_dim is 64)
    for field, val in (("head_dim", 96), ("n_head", 7), ("page_rows", 20), ("type_k", 3), ("type_k", 2),
                       ("type_v", 2)):
        p = kvc.kvc_params_init()
        setattr(p, field, val)
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_create(p)
        assert e.value.status == kvc.KVC_EINVAL, field
    # split residency: gpu_heads must leave at least one KV head on each side; one sequence
    for gpu_heads, n_seq in ((0, 1), (2, 1), (5, 1), (1, 2)):
        p = kvc.kvc_params_init()
        p.residency, p.gpu_heads, p.n_seq_max = kvc.KVC_SPLIT_HEADS, gpu_heads, n_seq
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_create(p)
        assert e.value.status == kvc.KVC_EINVAL, (gpu_heads, n_seq)


def test_cold_store_restore_model_calls_without_a_gpu():
    from kv_cache_decode_flash_gb300 import kvc

    s = kvc.ColdStore(1000)
    try:
        assert s.restore_model() == (0.0, 0.0, 0)
        assert s.plan_admit(123, 0.0, 10.0) == (0, 0.0, 0)  # nothing stored under the key: recompute
        s.set_restore_model(1500.0, 0.9)
        assert s.restore_model() == (1500.0, 0.9, 0)
        with pytest.raises(kvc.KvcError):
            s.set_restore_model(-1.0, 0.5)
        s.set_restore_model(0.0, -1.0)  # back to the (empty) fitted model
        assert s.restore_model() == (0.0, 0.0, 0)
    finally:
        s.close()
