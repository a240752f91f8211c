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


def test_row_selection_matches_a_plain_filter():
    """The sequence operations' row selection (by arithmetic when the positions
    are consecutive, else by one counting pass and an index list) against a
    plain filter over the positions, on consecutive, gapped, duplicated and
    shuffled positions."""
    import numpy as np

    from kv_cache_decode_flash_gb300 import kvc

    rng = np.random.default_rng(7)
    cases = [np.arange(0, 300), np.arange(1000, 1513), np.arange(0)]
    g = np.arange(0, 400)
    g[150:] += 50  # a gap
    cases.append(g)
    d = np.concatenate([np.arange(0, 200), np.arange(50, 250)])  # duplicates after a shift
    cases.append(d)
    cases.append(rng.permutation(500))
    cases.append(np.sort(rng.choice(5000, 700, replace=False)))
    for pos in cases:
        linear = len(pos) > 0 and bool(np.all(pos == pos[0] + np.arange(len(pos))))
        top = int(pos.max()) + 3 if len(pos) else 10
        ranges = [(-1, -1), (0, 1), (5, 5)] + [tuple(sorted(rng.integers(-1, top, 2))) for _ in range(40)]
        for p0, p1 in ranges:
            a = 0 if p0 < 0 else p0
            b = 2**31 if p1 < 0 else p1
            want = np.nonzero((pos >= a) & (pos < b))[0].tolist()
            for lin in ([False, True] if linear else [False]):
                rows, first, contig = kvc.kvc_debug_select_rows(pos.tolist(), p0, p1, linear=lin)
                assert rows == want, (pos[:5], p0, p1, lin)
                assert first == (want[0] if want else 0)
                assert contig == (not want or want == list(range(want[0], want[0] + len(want))))
    # a false "consecutive" statement is rejected
    with pytest.raises(kvc.KvcError):
        kvc.kvc_debug_select_rows([0, 1, 3], -1, -1, linear=True)
