"""The tensor-core kernels' barrier protocols, checked on the CPU under random interleavings
(protocol_model.py says what is modelled and checked). compute-sanitizer's race and barrier
checks are not available on this machine; this stands in for them at the level of the protocol.
Each check is run on its own deliberate mistakes too, to show the model would catch them."""

import random

import pytest

from protocol_model import ProtocolError, decode_ring, varlen_lone, varlen_pair

# the decode kernel's rings: (stages, producer warps, consumer warps, early release)
DECODE_RINGS = [(8, 2, 4, False),   # bf16, head_dim 128: 8 stages of 8 KiB
                (16, 4, 4, True),   # int8 / E4M3 codes, head_dim 128: 16 stages of 4 KiB
                (4, 2, 4, False),   # bf16, head_dim 256
                (16, 2, 4, False),  # bf16, head_dim 64
                (8, 4, 4, True)]    # 8-bit codes, head_dim 256


@pytest.mark.parametrize("stages,producers,consumers,early", DECODE_RINGS)
def test_decode_ring_protocol(stages, producers, consumers, early):
    rng = random.Random(stages * 100 + producers)
    for trial in range(150):
        chunks = rng.choice([0, 1, 2, stages - 1, stages, stages + 1, rng.randint(1, 6 * stages)])
        decode_ring(chunks, stages, producers, consumers, seed=trial, release_early=early)


def test_varlen_pair_protocol():
    rng = random.Random(7)
    cases = [(1, 0), (1, 1), (1, 2), (2, 2), (2, 3), (3, 0), (5, 5), (5, 7)]
    cases += [(a, rng.choice([0, a, a + 1, a + 2])) for a in (rng.randint(1, 9) for _ in range(40))]
    for trial, (nA, nB) in enumerate(cases):
        for seed in range(25):
            varlen_pair(nA, nB, seed=trial * 1000 + seed)


@pytest.mark.parametrize("lead", [0, 1])
def test_varlen_lone_protocol(lead):
    # lead 1: the kernel's order, K copies one tile ahead of V copies; lead 0 also holds
    for nA in list(range(1, 12)) + [17, 32]:
        for seed in range(40):
            varlen_lone(nA, seed=nA * 1000 + seed, lead=lead)


def _caught(fn, *args, **kw):
    for seed in range(300):
        try:
            fn(*args, seed=seed, **kw)
        except ProtocolError:
            return True
    return False


def test_model_catches_a_stage_refilled_by_two_producers():
    # 8 stages for 3 producers: a stage's chunks go to different producers in turn, whose parity
    # waits on its release barrier then race (the kernel asserts stages % producers == 0)
    assert _caught(decode_ring, 60, 8, 3, 4)


def test_model_catches_a_stage_drained_by_two_consumers():
    # 6 stages for 4 consumers: the same race on the fill barrier (stages % consumers == 0)
    assert _caught(decode_ring, 40, 6, 2, 4)


def test_model_catches_a_release_nobody_waits_for():
    # releasing every ring stage after its last use leaves commits landing after the CTA left
    assert _caught(varlen_pair, 3, 3, conditional_release=False)


def test_model_catches_a_wrong_score_phase():
    assert _caught(varlen_pair, 4, 4, score_phase_offset=1)


def test_model_catches_a_lone_tile_merging_without_the_named_barrier():
    assert _caught(varlen_lone, 6, merge_wait=False)

