"""The split-K chunk planner (host logic, no GPU): whole waves of chunks of
at most 8000 rows, the SM reserve for short chunks, the switch to two CTAs per
SM for long launches, and argument checks.  GB300 figures: 152 SMs, one
attention CTA per SM in configuration 0, two in configuration 1 (q8_0)."""
import random

import pytest

from kv_cache_decode_flash_gb300 import kvc

SMS, OCC, OCC2 = 152, 1, 2
Q8, F16 = kvc.KVC_Q8_0, kvc.KVC_F16


def plan(rows, type_=Q8, D=128, H=40, Hk=8, sms=SMS, occ=OCC, occ2=None):
    if occ2 is None:
        occ2 = OCC2 if type_ == Q8 else 0
    return kvc.kvc_debug_chunk_plan(type_, D, H, Hk, sms, occ, occ2, rows)


def ctas(rows, C, Hk=8):
    return Hk * sum(max(1, -(-r // C)) for r in rows)


def test_decode_16k_leaves_the_merging_ctas_their_sms():
    # 16384 rows x 8 KV heads: 144 slots (8 SMs left to the previous launch's last CTAs) give
    # 18 chunks of 911 rows; whole 128-row tiles make that 16 chunks of 1024 rows, 128 CTAs
    C, cfg = plan([16384])
    assert (C, cfg) == (1024, 0)
    assert ctas([16384], C) == 128


@pytest.mark.parametrize("n", [1000, 4096, 6144, 16384, 65536, 131072])
def test_single_sequence_chunks_are_whole_tiles(n):
    C, cfg = plan([n])
    assert C % 128 == 0 or C == 8000
    # no more chunks than rows-per-slot chunks (16-row multiples) would give
    slots = SMS * OCC
    if 8 * 8 <= slots and n * 8 <= (slots - 8) * 4096:
        slots -= 8  # the SMs left to the previous launch's last CTAs
    raw = -(-n * 8 // slots)
    assert -(-n // C) <= -(-n // ((raw + 15) // 16 * 16))


def test_long_single_sequence_fills_one_wave():
    C, cfg = plan([131072])        # 1,048,576 row-heads: one wave of one CTA per SM
    assert (C, cfg) == (6912, 0) and ctas([131072], C) == 152
    C, cfg = plan([262144])        # above one wave of 8000-row chunks: two CTAs per SM
    assert (C, cfg) == (6912, 1) and ctas([262144], C) == 304


def test_f16_has_one_configuration():
    for n in (4096, 262144, 1 << 20):
        assert plan([n], type_=F16)[1] == 0


@pytest.mark.parametrize("seed", range(5))
def test_invariants_on_random_batches(seed):
    rng = random.Random(seed)
    for _ in range(200):
        n_seq = rng.choice([1, 1, 2, 7, 32, 64])
        rows = [rng.choice([0, 1, rng.randint(1, 40000), rng.randint(1, 600000)]) for _ in range(n_seq)]
        D = rng.choice([64, 128])
        Hk = rng.choice([1, 2, 4, 8])
        H = Hk * rng.choice([1, 3, 4, 5, 8])
        type_ = rng.choice([Q8, F16])
        C, cfg = plan(rows, type_=type_, D=D, H=H, Hk=Hk)
        assert C % 16 == 0 and 64 <= C <= 8000
        assert cfg in (0, 1) and (type_ == Q8 or cfg == 0)
        work = max(sum(rows) * Hk, 1)
        assert cfg == (1 if type_ == Q8 and work > SMS * OCC * 8000 else 0)
        if n_seq == 1 and rows[0] > 0:
            slots = SMS * (OCC2 if cfg else OCC)
            waves = -(-work // (slots * 8000))
            assert ctas(rows, C, Hk) <= waves * slots  # whole waves


def test_rejects_bad_arguments():
    for args in [(Q8, 96, 40, 8, SMS, 1, 2, [10]), (Q8, 128, 41, 8, SMS, 1, 2, [10]),
                 (Q8, 128, 72, 8, SMS, 1, 2, [10]), (F16, 128, 40, 8, SMS, 1, 2, [10]),
                 (Q8, 128, 40, 8, 0, 1, 2, [10]), (Q8, 128, 40, 8, SMS, 1, 2, [-1]), (7, 128, 40, 8, SMS, 1, 2, [10])]:
        with pytest.raises(kvc.KvcError):
            kvc.kvc_debug_chunk_plan(*args)


def plan_seq(rows, type_=Q8, D=128, H=40, Hk=8, sms=SMS, occ=OCC, occ2=None):
    if occ2 is None:
        occ2 = OCC2 if type_ == Q8 else 0
    return kvc.kvc_debug_chunk_plan_seq(type_, D, H, Hk, sms, occ, occ2, rows)


def test_single_sequence_keeps_the_one_length():
    for n in (4096, 16384, 65536, 262144):
        assert plan_seq([n])[0] == [plan([n])[0]]


@pytest.mark.parametrize("seed", range(5))
def test_batches_cut_every_sequence_into_equal_chunks_in_whole_waves(seed):
    rng = random.Random(100 + seed)
    for _ in range(200):
        n_seq = rng.choice([2, 7, 32, 64])
        rows = [rng.choice([0, 1, rng.randint(1, 40000), rng.randint(1, 600000)]) for _ in range(n_seq)]
        type_ = rng.choice([Q8, F16])
        Hk = rng.choice([1, 2, 4, 8])
        H = Hk * rng.choice([1, 4, 5, 8])
        cs, cfg = plan_seq(rows, type_=type_, H=H, Hk=Hk)
        uniform, cfg_u = plan(rows, type_=type_, H=H, Hk=Hk)
        assert cfg == cfg_u
        slots = SMS * (OCC2 if cfg else OCC)
        total = 0
        for r, c in zip(rows, cs):
            assert c % 16 == 0 and 16 <= c <= 8000
            k = max(1, -(-r // c))
            total += k
            if k > 1:
                # equal chunks: the last one is within 16 rows of a full share, none shorter than 64 rows
                assert r - (k - 1) * c > 0 and c >= 64
                assert (k - 1) * c < r <= k * c
        # no more CTAs than one uniform length at the plan's longest chunk would launch
        assert total * Hk <= ctas(rows, max(cs), Hk)


def test_ragged_benchmark_batch_plan():
    # the benchmark's batch: 32 sequences, lengths uniform in [1024, 32768] (seed 0), 32/8 heads:
    # three whole waves of two CTAs per SM (912 CTAs), every sequence in equal chunks of at most
    # 4816 rows (measured 0.204 ms against 0.224 ms for the uniform length)
    from kv_cache_decode_flash_gb300 import synth

    rows = [int(x) for x in synth.randint(0, synth.stream_id("len"), 32, 1024, 32768)]
    cs, cfg = plan_seq(rows, H=32, Hk=8)
    assert cfg == 1
    total = 8 * sum(max(1, -(-r // c)) for r, c in zip(rows, cs))
    assert total == 3 * SMS * OCC2 and max(cs) == 4816
    assert all(max(1, -(-r // c)) * c - r < 16 * max(1, -(-r // c)) for r, c in zip(rows, cs))
