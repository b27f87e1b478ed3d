"""The completion-signalling protocol run by host threads with C11 atomics
(`protocol_model.c`): producer threads play the thread blocks of every rank's
experts (several tiles per expert), consumer threads the destination ranks. The
orderings are those of the kernels: the count words stored at the start by the
rank's block 0, before its release; tile rows released into a per-expert tile
counter by acquire-release RMWs; the expert's completer increments the rank's
election counter with an acquire-release RMW; the elected producer releases the
rank flag of every destination ("ep_signal_completion", ep_ord_r with
has_rank_flag), or every count word is tagged with the epoch (per-expert mode).
Across many epochs and seeded interleavings every consumer that acquires a signal
sees all the rows and counts it covers, exactly one producer per (source,
destination) is elected, a producer that never signals makes the waits run out
instead of hanging, and two planted mistakes (a flag released by the first expert
instead of the last; the count words stored after block 0's release) are caught.
On an Arm host (weakly ordered) the fences are exercised as well as the logic."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def model(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path_factory.mktemp("pmodel") / "protocol_model"
    subprocess.run([cc, "-std=c11", "-O2", "-pthread", os.path.join(HERE, "protocol_model.c"),
                    "-o", str(exe)], check=True, capture_output=True)
    return str(exe)


def run(model, R, E, tiles, rows, epochs, mode, seed, fail=None):
    args = [model, *map(str, (R, E, tiles, rows, epochs, mode, seed))]
    if fail is not None:
        args += [str(fail[0]), str(fail[1])]
    out = subprocess.run(args, check=True, capture_output=True, text=True, timeout=120).stdout
    f = out.split()
    return {f[i]: int(f[i + 1]) for i in range(0, len(f), 2)}


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("R,E,tiles", [(4, 3, 2), (8, 2, 3), (2, 4, 1)])
def test_rank_flag_covers_every_row_and_count(model, R, E, tiles, seed):
    got = run(model, R, E, tiles, 48, 150, 0, seed)
    assert got["errors"] == 0 and got["timeouts"] == 0
    assert got["elections"] == R * R * 150  # one per (source, destination, epoch)


@pytest.mark.parametrize("seed", [1, 2])
def test_per_expert_words_cover_their_rows(model, seed):
    got = run(model, 4, 3, 2, 48, 150, 1, seed)
    assert got == {"epochs": 150, "errors": 0, "timeouts": 0, "elections": 0}


@pytest.mark.parametrize("mode", [0, 1])
def test_a_producer_that_never_signals_makes_the_waits_run_out(model, mode):
    R, E = 4, 3
    got = run(model, R, E, 2, 48, 1, mode, 5, fail=(2, 1))
    assert got["errors"] == 0
    assert got["timeouts"] == R  # every destination gives up on that rank (or that expert)
    if mode == 0:
        assert got["elections"] == (R - 1) * R  # the other ranks still publish


def test_the_checks_catch_a_flag_released_too_early(model):
    got = run(model, 4, 3, 2, 48, 150, 2, 9)
    assert got["errors"] > 0


def test_the_checks_catch_count_words_stored_after_the_release(model):
    got = sum(run(model, 4, 3, 2, 48, 150, 3, seed)["errors"] for seed in (9, 10, 11))
    assert got > 0
