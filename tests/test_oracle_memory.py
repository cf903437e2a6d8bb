"""Pins of the oracle's closed forms against the numbers the pages print.

Golden files under tests/golden/ carry the printed values and their sources.
"""
import os
from fractions import Fraction

import pytest

from oracle import memory as mem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_table1_every_cell():
    rows = _rows("table1_zero_dp_memory.txt")
    header, body = rows[0], rows[1:]
    models = {"7.5B": Fraction(75, 10) * 10**9, "128B": 128 * 10**9, "1T": 10**12}
    checked = 0
    for row in body:
        dp = int(row[0])
        for col, printed in zip(header[1:], row[1:]):
            model, stage = col.rsplit("_", 1)
            exact = mem.gb(mem.model_state_bytes(models[model], dp, int(stage)))
            assert mem.printed_matches(printed, exact), (model, dp, stage, printed, float(exact))
            checked += 1
    assert checked == 54


def test_table1_detects_wrong_formula():
    # A plausible slip -- K = 12 applied to the gradient share as well, or the
    # stage-2 grad share left unsharded -- must disagree with the table.
    exact_wrong = mem.gb(2 * Fraction(75, 10) * 10**9 + 12 * Fraction(75, 10) * 10**9 / 64)
    assert not mem.printed_matches("16.6", exact_wrong)
    wrong_stage1 = mem.gb(4 * Fraction(75, 10) * 10**9 + 14 * Fraction(75, 10) * 10**9 / 64)
    assert not mem.printed_matches("31.4", wrong_stage1)


def _size(tok):
    if tok.endswith("T"):
        return Fraction(tok[:-1]) * 1024 * 10**9
    return Fraction(tok[:-1]) * 10**9


def test_table2_max_model_size():
    rows = _rows("table2_max_model_size.txt")
    body = rows[1:]
    first = None
    for row in body:
        mp, gpus = int(row[0]), int(row[1])
        printed = [_size(t) for t in row[2:6]]
        exact = [mem.max_model_size(mp, gpus, st) for st in (0, 1, 2, 3)]
        if mp == 1:
            first = row[2:6]
            for tok, ex in zip(first, exact):
                assert mem.printed_matches(tok[:-1], ex / 10**9), (tok, float(ex))
        # every row is the MP = 1 row (as printed) scaled by MP, and within
        # 1% of the exact value at that row
        for st, (p, ex) in enumerate(zip(printed, exact)):
            assert p == mp * _size(first[st]), (mp, st)
            assert abs(p - ex) / ex < Fraction(1, 100), (mp, st, float(p), float(ex))


def test_worked_examples():
    n = 0
    with open(os.path.join(GOLDEN, "worked_examples.txt"), encoding="utf-8") as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            name, psi, dp, stage, printed, unit, _src = [x.strip() for x in ln.split("|")]
            psi, dp = Fraction(psi), int(dp)
            assert unit == "GB"
            if stage == "-":   # optimizer states alone: K * psi, 75% of 16 psi
                exact = mem.gb(mem.K_ADAM * psi)
                assert mem.K_ADAM * psi / mem.model_state_bytes(psi, 1, 0) == Fraction(3, 4)
            else:
                exact = mem.gb(mem.model_state_bytes(psi, dp, int(stage)))
            assert mem.printed_matches(printed, exact), (name, printed, float(exact))
            n += 1
    assert n == 9


def test_zero_adam_state_bytes():
    rows = dict(_rows("zero_adam_check.txt"))
    world, numel = int(rows["world"]), int(rows["numel"])
    # Linear(64,256) + Linear(256,10): weights and biases
    assert 64 * 256 + 256 + 256 * 10 + 10 == numel
    per_rank = mem.zero_adam_state_bytes(numel, world)
    full = mem.unsharded_adam_state_bytes(numel)
    assert per_rank == int(rows["state_bytes_rank"])      # pins ceil + padding (4803)
    assert full == int(rows["state_bytes_full"])
    assert round(full / per_rank) == int(rows["ratio"])
    # floor instead of ceil would give 3 * 4802 * 4
    assert 3 * (numel // world) * 4 != per_rank


def test_communication_volume():
    for n in (2, 4, 8, 64, 1024):
        psi = 10**9
        dp = mem.comm_elements_per_rank(psi, n, 0)
        assert dp == 2 * Fraction(n - 1, n) * psi
        assert mem.comm_elements_per_rank(psi, n, 1) == dp
        assert mem.comm_elements_per_rank(psi, n, 2) == dp
        assert mem.comm_elements_per_rank(psi, n, 3) == Fraction(3, 2) * dp


def test_constant_size_buffer_example():
    # ZeRO-R C_B: a 3B model's fp32 fused buffer reaches 12 GB
    assert mem.gb(mem.fused_fp32_buffer_bytes(3 * 10**9)) == 12


def test_stage_ordering_and_limits():
    for psi in (10**6, 7 * 10**9):
        for n in (1, 2, 8, 64):
            b = [mem.model_state_bytes(psi, n, s) for s in range(4)]
            if n == 1:
                assert b[0] == b[1] == b[2] == b[3] == 16 * psi
            else:
                assert b[0] > b[1] > b[2] > b[3]
    with pytest.raises(ValueError):
        mem.model_state_bytes(1, 1, 4)
