"""Pins for the oracle's model-state ledger (not gpu): values printed on the pages."""

import json
import math
import os

import numpy as np

import synth_inputs as si
from conftest import GOLDEN

LEDGER = json.load(open(os.path.join(GOLDEN, "pages_ledger.json")))


def _round_half_up(x, decimals):
    q = 10.0 ** decimals
    return math.floor(x * q + 0.5) / q


def test_per_gpu_gb_printed(oracle_lib):
    for row in LEDGER["per_gpu_gb"]:
        psi, n = int(row["psi"]), row["n"]
        assert psi % n == 0  # these models need no padding at their N
        per_rank = oracle_lib.state_bytes([psi], n, row["stage"])
        assert np.all(per_rank == per_rank[0])
        gb = per_rank[0] / 1e9
        assert _round_half_up(gb, row["decimals"]) == row["printed"], (gb, row["cite"])


def test_bytes_per_param_n4(oracle_lib):
    row = LEDGER["bytes_per_param_n4"]
    psi = 4 * 1000
    for stage in range(4):
        b = oracle_lib.state_bytes([psi], row["n"], stage)[0] / psi
        assert b == row[f"stage{stage}"], row["cite"]


def _round_sig(x, sig):
    if x == 0:
        return 0
    return round(x, -int(math.floor(math.log10(abs(x)))) + (sig - 1))


def test_max_model_table2(oracle_lib):
    spec = LEDGER["max_model_32gb"]
    for row in spec["rows"]:
        # bytes per parameter at N_d data-parallel ways, from the ledger of a
        # model of N_d * 10^6 params (so no padding arises)
        psi = row["n"] * 1_000_000
        bpp = oracle_lib.state_bytes([psi], row["n"], row["stage"])[0] / psi
        max_params = 32e9 / bpp * row["mp"]
        assert _round_sig(max_params, row["sig"]) == row["printed_params"], (max_params, spec["cite"])


def test_zero3_peak_lecture_mlp(oracle_lib):
    z = LEDGER["zero3_lecture_mlp"]
    pl = si.lecture_mlp()
    lay = oracle_lib.layout(pl.numel, pl.unit, z["n"], stage=3)
    assert list(lay.unit_numel) == z["unit_numel"]
    assert int(lay.unit_numel.sum()) == z["psi"]
    steady = oracle_lib.state_bytes(lay.unit_padded, z["n"], 3)[0]
    assert steady == z["steady_bytes"], z["cite"]
    peak, where = oracle_lib.zero3_backward_peak(lay.unit_padded, z["n"])
    assert peak == z["peak_bytes"], z["cite"]
    assert where == z["peak_unit"], z["cite"]
    # the three parts of the worked answer
    shard = lay.unit_padded // z["n"]
    resident = 2 * shard.sum() + 12 * shard.sum()
    assert resident == z["resident_bytes"]
    assert 2 * shard[2:].sum() == z["reduced_grad_shards_at_peak"]
    assert 4 * lay.unit_padded[1] == z["full_unit_params_and_grads_at_peak"]
    assert 2 * lay.unit_padded[1] == z["p16_full_bytes"]


def test_ledger_formulas_random(oracle_lib):
    # 4P + 12P/N, 2P + 14P/N, 16P/N with P a multiple of N
    rng = np.random.default_rng(3)
    for _ in range(100):
        n = int(rng.integers(1, 65))
        p = n * int(rng.integers(1, 10_000))
        got = [oracle_lib.state_bytes([p], n, s)[0] for s in range(4)]
        assert got == [16 * p, 4 * p + 12 * p // n, 2 * p + 14 * p // n, 16 * p // n]
