"""The tensor-core kernels' barrier protocols, checked on the host.

Every configuration the library picks (w4a16_tc_config, no GPU involved)
must satisfy the ring invariants that keep each mbarrier parity wait on the
phase it means, and a discrete-event model of the protocol
(tests/pipeline_model.py) must run those configurations to the end under
random interleavings without a wait passing on a wrong phase or a deadlock.
The CTA-pair kernel's model adds the persistent loop: several output tiles
per cluster, one accumulator handed between the MMA thread and the
epilogues. The models are themselves checked on configurations that break
the invariants: they must catch them (a four-group kernel with three
activation slots, a code ring that is not a multiple of the groups, fewer
dequantized slots than groups in the persistent loop).
"""
import itertools

import pytest

import bit_weight_only_g128_gb300 as w4
from bit_weight_only_g128_gb300 import build as wbuild
from pipeline_model import simulate, simulate_persistent

SHAPES_K = [64, 128, 192, 256, 1088, 4096, 5120, 8192, 11008, 13824, 28672]
ROWS = [17, 20, 32, 33, 48, 49, 64, 80, 96, 100, 112, 128, 144, 160, 176, 192, 208, 224, 240,
        256, 300, 512, 4096]


@pytest.fixture(scope="module")
def configs():
    wbuild.build()
    seen = {}
    for K, M in itertools.product(SHAPES_K, ROWS):
        for group in sorted({64, 128, K}):
            if K % group:
                continue
            cfg = w4.tc_config(M, K, group)
            seen[(M, K, group)] = cfg
    return seen


def test_token_tile_and_stage_atoms(configs):
    for (M, K, group), c in configs.items():
        assert c["token_tile"] == (256 if M >= 256 else (M + 15) // 16 * 16)
        assert c["stage_atoms"] == (2 if K % 128 == 0 and group % 128 == 0 else 1)
        assert c["ctas_per_sm"] == (2 if c["token_tile"] <= 64 else 1)


def test_ring_invariants(configs):
    for key, c in configs.items():
        assert 1 <= c["dq_slots"] <= c["act_slots"], key
        assert c["act_slots"] >= c["dequant_groups"], key
        assert c["code_slots"] % c["dequant_groups"] == 0, key
        assert c["dequant_groups"] in (2, 4), key
        limit = (113 if c["ctas_per_sm"] == 2 else 227) * 1024
        assert c["smem_bytes"] <= limit, key
        # the dequantized ring and the accumulator share the tensor memory
        tmem = 256 if c["ctas_per_sm"] == 2 else 512
        acc = (c["token_tile"] + 31) // 32 * 32
        assert acc + c["dq_slots"] * 32 * c["stage_atoms"] <= tmem, key


def test_protocol_model_runs_every_configuration(configs):
    rings = sorted({(c["code_slots"], c["act_slots"], c["dq_slots"], c["dequant_groups"],
                     c["stage_atoms"] > 2) for c in configs.values()})
    for code, act, dq, groups, slot_first in rings:
        for nk in (1, groups + 1, 3 * max(code, act) + 5):
            for seed in range(12):
                assert simulate(nk, code, act, dq, groups, seed, slot_first=slot_first) == "ok", \
                    (code, act, dq, groups, nk, seed)


@pytest.mark.parametrize("code,act,dq,groups", [(4, 3, 3, 4), (6, 5, 5, 4), (2, 2, 2, 4)])
def test_protocol_model_catches_broken_rings(code, act, dq, groups):
    failures = 0
    for seed in range(60):
        try:
            res = simulate(32, code, act, dq, groups, seed)
        except AssertionError:
            res = "wrong phase"
        failures += res != "ok"
    assert failures > 0


def test_tc_config_rejects_bad_arguments():
    wbuild.build()
    with pytest.raises(w4.W4A16Error):
        w4.tc_config(0, 4096, 128)
    with pytest.raises(w4.W4A16Error):
        w4.tc_config(64, 100, 128)


@pytest.fixture(scope="module")
def pair_configs():
    wbuild.build()
    seen = {}
    for K, M in itertools.product(SHAPES_K, [256, 300, 512, 4096]):
        for group in sorted({64, 128, K}):
            if K % group:
                continue
            seen[(M, K, group)] = w4.tc_config(M, K, group, pair=True)
    return seen


def test_pair_ring_invariants(pair_configs):
    for key, c in pair_configs.items():
        assert c["token_tile"] == 256, key
        assert c["stage_atoms"] == (2 if key[1] % 128 == 0 and key[2] % 128 == 0 else 1), key
        # the persistent loop also needs dq_slots >= dequant_groups
        assert c["dequant_groups"] <= c["dq_slots"] <= c["act_slots"], key
        assert c["code_slots"] % c["dequant_groups"] == 0, key
        assert c["smem_bytes"] <= 227 * 1024, key
        assert c["token_tile"] + c["dq_slots"] * 32 * c["stage_atoms"] <= 512, key


def test_pair_protocol_model_runs_every_configuration(pair_configs):
    rings = sorted({(c["code_slots"], c["act_slots"], c["dq_slots"], c["dequant_groups"])
                    for c in pair_configs.values()})
    for code, act, dq, groups in rings:
        for ntiles, nk in ((1, 5), (3, 1), (4, groups - 1), (3, 2 * max(code, act) + 3)):
            for seed in range(8):
                assert simulate_persistent(ntiles, nk, code, act, dq, groups, seed) == "ok", \
                    (code, act, dq, groups, ntiles, nk, seed)


@pytest.mark.parametrize("code,act,dq,groups", [(8, 5, 3, 4), (8, 5, 2, 4)])
def test_pair_protocol_model_catches_short_dq_ring(code, act, dq, groups):
    failures = 0
    for seed in range(20):
        try:
            res = simulate_persistent(4, 16, code, act, dq, groups, seed)
        except AssertionError:
            res = "wrong phase"
        failures += res != "ok"
    assert failures > 0
