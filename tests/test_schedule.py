"""The decode kernels' work schedule on the host: the quota rule and the piece cursor of
decode_tc.cuh, compiled for the CPU by tests/schedule_harness.cu, walked for every SM pair
over many batch shapes. Every token is covered exactly once, every sequence's pieces take
slots 0, 1, ... in token order below the slot count the library reports
(mla_num_splits), the last piece marks the unused slots, and no pair exceeds its quota.
Batches of equal lengths take the split plan when it spares pairs a second piece."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import mla_latent_kv_69_b300 as mla
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PAIRS = 74   # SM pairs of a B300


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_harness")
    cmd = [nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(ROOT, "mla_latent_kv_69_b300", "csrc"), os.path.join(ROOT, "tests", "schedule_harness.cu"),
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _slots(B, lens):
    # what num_splits = 0 resolves to on a 148-SM part (the host query uses the device's
    # SM count when a GPU is present; on the CPU the library assumes 148)
    return mla.num_splits(B, int(max(lens)) if len(lens) else 0, 128)


def _run(harness, cases):
    text = "".join(f"{B} {S} {P} " + " ".join(str(int(x)) for x in lens) + "\n" for B, S, P, lens in cases)
    r = subprocess.run([harness], input=text, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = r.stdout.strip().splitlines()
    assert len(out) == len(cases)
    return [line.split() for line in out]


def test_workload_schedules_are_exact_and_balanced(harness):
    cases = []
    for name in W.WORKLOAD_ORDER:
        w = W.WORKLOADS[name]
        lens = W.seq_lens(w)
        cases.append((w.batch, _slots(w.batch, lens), PAIRS, lens))
    plans = {}
    for name, (B, S, P, lens), res in zip(W.WORKLOAD_ORDER, cases, _run(harness, cases)):
        assert res[0] == "ok", (B, res)
        max_tiles, ideal, split = int(res[1]), int(res[2]), int(res[4])
        T = int(np.sum((lens + 127) // 128))
        assert ideal == -(-T // P)
        if split == 0:
            # the slot count leaves the quota at the even share for these shapes
            assert max_tiles == ideal, (B, max_tiles, ideal)
        else:
            tiles = (lens + 127) // 128
            assert np.all(tiles == tiles[0])
            per = -(-int(tiles[0]) // split)
            assert max_tiles == -(-B * split // P) * per
            assert max_tiles <= ideal + 3   # cheaper than the tile plan's piece switch
        plans[name] = (split, max_tiles)
    # equal lengths are cut into whole pieces (no pair holds two), ragged batches share tiles
    assert plans["v2_b32_l4096"] == (2, 16)
    assert plans["long_b4_l128k"] == (18, 57)
    assert plans["paged_b64_l1k_32k"][0] == 0


def test_random_batches(harness):
    rng = np.random.default_rng(7)
    cases = []
    for _ in range(300):
        B = int(rng.choice([1, 2, 3, 5, 17, 64, 100, 300, 1000]))
        kind = rng.integers(0, 4)
        if kind == 0:
            lens = np.full(B, int(rng.integers(0, 40000)))
        elif kind == 1:
            lens = rng.integers(0, 3000, size=B)
        elif kind == 2:   # one long sequence among short ones
            lens = rng.integers(0, 200, size=B)
            lens[rng.integers(0, B)] = int(rng.integers(1, 200000))
        else:             # many empty sequences
            lens = np.where(rng.random(B) < 0.5, 0, rng.integers(1, 5000, size=B))
        P = int(rng.choice([1, 2, 7, 74]))
        S = _slots(B, lens) if rng.random() < 0.7 else int(rng.integers(1, 9))
        cases.append((B, S, P, lens.astype(np.int64)))
    for case, res in zip(cases, _run(harness, cases)):
        assert res[0] == "ok", (case[0], case[1], case[2], " ".join(res))
        tiles = (case[3] + 127) // 128
        if int(res[4]) > 0:   # the split plan only for equal, nonzero tile counts, within the slots
            assert np.all(tiles == tiles[0]) and tiles[0] > 0 and int(res[4]) <= case[1]


def test_slot_count_rule():
    assert mla.num_splits(1, 256, 16) == 2          # two tiles: one piece each at most
    assert mla.num_splits(4, 128, 128) == 1         # single-tile sequences never split
    assert mla.num_splits(32, 4096, 128) == 5       # ceil(74 / 32) + 2
    assert mla.num_splits(4, 131072, 128) == 21
    assert mla.num_splits(128, 8192, 128) == 3
    assert mla.num_splits(1, 10 ** 7, 128) == 76
    assert mla.num_splits(1, 0, 128) == 1
