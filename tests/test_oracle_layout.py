"""Pins for the oracle's FlatParameter layout (not gpu).

Layout is integer work: every check is exact.
"""

import json
import os

import numpy as np
import pytest

import synth_inputs as si
from conftest import GOLDEN


def _units(sizes):
    return list(sizes), list(range(len(sizes)))


def test_printed_padding_examples(oracle_lib):
    spec = json.load(open(os.path.join(GOLDEN, "pages_layout.json")))
    for ex in spec["examples"]:
        numel, unit = _units(ex["unit_numel"])
        lay = oracle_lib.layout(numel, unit, ex["n"], stage=3)
        assert list(lay.unit_padded) == ex["padded"], ex["cite"]
        assert list(lay.unit_padded - lay.unit_numel) == ex["pad"], ex["cite"]
        if "shard" in ex:
            assert list(lay.unit_shard) == ex["shard"], ex["cite"]
        if "psi" in ex:
            assert int(lay.unit_numel.sum()) == ex["psi"], ex["cite"]
        if "psi_padded" in ex:
            assert lay.total_padded == ex["psi_padded"], ex["cite"]
        if "pad_owner_rank" in ex:
            # the pad elements sit at the end of the unit: which rank's shard holds them
            first_pad = int(lay.unit_base[0] + lay.unit_numel[0])
            owner = (first_pad - int(lay.unit_base[0])) // int(lay.unit_shard[0])
            assert owner == ex["pad_owner_rank"], ex["cite"]


def test_brute_force_tiny(oracle_lib):
    # padded = the smallest multiple of N not below numel, found by counting up.
    for n in range(1, 17):
        for numel in range(0, 41):
            padded = numel
            while padded % n:
                padded += 1
            lay = oracle_lib.layout([numel], [0], n, stage=1)
            assert lay.unit_padded[0] == padded
            assert lay.unit_shard[0] * n == padded
            assert 0 <= padded - numel <= n - 1  # the pad bound of §5.2


def test_bases_offsets_and_shards_tile(oracle_lib):
    rng = np.random.default_rng(7)
    for trial in range(50):
        n_params = int(rng.integers(1, 12))
        numel = rng.integers(0, 300, n_params).tolist()
        unit = np.sort(rng.integers(0, 4, n_params)).tolist()
        n = int(rng.integers(1, 17))
        lay = oracle_lib.layout(numel, unit, n, stage=2)
        n_units = max(unit) + 1
        # bases are the running sum of padded sizes
        run = 0
        for i in range(n_units):
            assert lay.unit_base[i] == run
            run += lay.unit_padded[i]
        assert lay.total_padded == run
        # params sit back to back inside their unit, in caller order
        cursor = {}
        for p in range(n_params):
            u = unit[p]
            expect = cursor.get(u, int(lay.unit_base[u]))
            assert lay.param_offset[p] == expect
            cursor[u] = expect + numel[p]
        for i in range(n_units):
            assert cursor.get(i, int(lay.unit_base[i])) == lay.unit_base[i] + lay.unit_numel[i]
        # rank shards partition each unit exactly
        for i in range(n_units):
            covered = []
            for d in range(n):
                covered.extend(range(int(lay.unit_base[i] + d * lay.unit_shard[i]),
                                     int(lay.unit_base[i] + (d + 1) * lay.unit_shard[i])))
            assert covered == list(range(int(lay.unit_base[i]), int(lay.unit_base[i] + lay.unit_padded[i])))


def test_stage0_never_pads(oracle_lib):
    lay = oracle_lib.layout([1552, 7, 15], [0, 1, 2], 3, stage=0)
    assert list(lay.unit_padded) == [1552, 7, 15]
    assert list(lay.unit_shard) == [1552, 7, 15]


def test_rejects_decreasing_units(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.layout([4, 4], [1, 0], 2, stage=1)


@pytest.mark.parametrize("factory,total,n", [
    (si.toy_mlp, 34_192, 4),
    (si.lecture_mlp, 32_656, 4),
    (si.llama_1024, 73_417_728, 8),
    (si.llama_2048_units, 654_346_240, 8),
    (si.llama_2048_stage_buffer, 2_030_174_208, 2),
])
def test_workload_sizes(oracle_lib, factory, total, n):
    pl = factory()
    assert pl.total == total
    lay = oracle_lib.layout(pl.numel, pl.unit, n, stage=3)
    # none of the model workloads needs padding at its N
    assert lay.total_padded == total


def test_toy_mlp_units(oracle_lib):
    pl = si.toy_mlp()
    lay = oracle_lib.layout(pl.numel, pl.unit, 4, stage=1)
    assert list(lay.unit_numel) == [4224, 16512, 8256, 4160, 1040]


def test_llama_2048_units(oracle_lib):
    pl = si.llama_2048_units()
    lay = oracle_lib.layout(pl.numel, pl.unit, 8, stage=3)
    assert list(lay.unit_numel) == [83_886_080] + [60_821_504] * 8 + [83_888_128]
