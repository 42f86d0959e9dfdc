"""Host bookkeeping of programmatic dependent launch for the decode kernel
family (csrc/launch_order.h), on the CPU through a small driver built with g++.

The expected guards follow from the residency argument stated in the header:
when launch X starts, launch N-k can still run only if all blocks of
N-k+1..N and one block of N-k fit on the device at once; X's guard is the
number of new tokens per sequence those possibly-running launches append to
X's own (cache, layer)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "gqa_attention_preallocated_qa_gb300", "csrc")
GUARD_ALL = 1 << 30
CAP = 1 << 14


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("order") / "launch_order_driver")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "native", "launch_order_driver.cpp"),
                    "-o", exe, "-lpthread"], check=True)

    def run(lines):
        out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
        return [int(x) for x in out.stdout.split()]
    return run


def admit(layer, ctas, tmax=1, early=1, rmax=304, stream=1, cache=7):
    return f"admit {stream} {cache} {layer} {ctas} {tmax} {early} {rmax}"


def test_single_layer_loop_guard_is_bounded_by_residency(driver):
    # 256 blocks per step, 304 resident: N and N-1 can run (256 + 1 <= 304), N-2 cannot.
    assert driver([admit(0, 256)] * 6) == [0, 1, 2, 2, 2, 2]
    # 128 blocks: N, N-1, N-2 (128 + 128 + 1 <= 304; 384 + 1 > 304).
    assert driver([admit(0, 128)] * 6) == [0, 1, 2, 3, 3, 3]
    # Tiny launches: the depth grows with what fits.
    assert driver([admit(0, 10)] * 40)[-1] == 31  # 30 launches of 10 blocks + 1 <= 304


def test_layer_loop_has_no_guard(driver):
    lines = [admit(l, 128) for _ in range(3) for l in range(36)]
    assert driver(lines) == [0] * (3 * 36)
    # two layers alternating with small grids: same-layer launches two apart can still run
    lines = [admit(l % 2, 100) for l in range(8)]
    # the fifth launch (layer 0): launches 4, 3, 2 hold 300 blocks and 301 <= 304,
    # so launch 1 can still run as well; launches 1 and 3 append to layer 0
    assert driver(lines) == [0, 0, 1, 1, 2, 2, 2, 2]


def test_tokens_of_short_chunks_add_up(driver):
    lines = [admit(0, 10, tmax=3), admit(0, 10, tmax=8), admit(0, 10)]
    assert driver(lines) == [0, 3, 11]


def test_barrier_and_late_launch_end_the_walk(driver):
    lines = [admit(0, 10), admit(0, 10), "barrier 1", admit(0, 10)]
    assert driver(lines) == [0, 1, 0]
    # a launch that signals after its own wait (device positions) may still run,
    # nothing before it can
    lines = [admit(0, 10), admit(0, 10, early=0), admit(0, 10)]
    assert driver(lines) == [0, 1, 1]
    lines = [admit(0, 10), admit(0, 10), "clear", admit(0, 10)]
    assert driver(lines) == [0, 1, 0]


def test_streams_and_caches_are_separate(driver):
    # another stream: no ordering, no guard; another cache: blocks count, rows do not
    lines = [admit(0, 10, stream=1), admit(0, 10, stream=2), admit(0, 10, cache=9), admit(0, 10)]
    assert driver(lines) == [0, 0, 0, 1]
    # another cache's launches in between still take residency: with 100 blocks
    # of it resident the first launch can still run (100 + 1 <= 304), with 304
    # it cannot
    lines = [admit(0, 200), admit(0, 100, cache=9), admit(0, 10)]
    assert driver(lines) == [0, 0, 1]
    lines = [admit(0, 200), admit(0, 304, cache=9), admit(0, 10)]
    assert driver(lines) == [0, 0, 0]


def test_unknown_history_loads_everything_after_the_wait(driver):
    # more launches than the record keeps, none of them bounding the walk
    lines = [f"fill 1 7 1 {CAP + 5}", admit(0, 1, rmax=1 << 40)]
    assert driver(lines) == [GUARD_ALL]
    lines = [f"fill 1 7 1 {CAP + 5}", "barrier 1", admit(0, 1, rmax=1 << 40)]
    assert driver(lines) == [0]


def settled(layer, rmax=304, stream=1, cache=7):
    return f"settled {stream} {cache} {layer} {rmax}"


def inflight(layer, rmax=304, stream=1, cache=7):
    return f"inflight {stream} {cache} {layer} {rmax}"


def test_settled_layers_may_read_device_lengths_early(driver):
    # nothing recorded: settled; the layer's own launch possibly running: not
    assert driver([settled(0), admit(0, 100), settled(0), settled(1)]) == [1, 0, 0, 1]
    # a loop over layers: layer 0's previous launch is beyond the resident bound
    # once 304 blocks of later launches sit in between
    lines = [admit(l, 128) for l in range(4)] + [settled(0), settled(2), settled(3)]
    assert driver(lines) == [0, 0, 0, 0, 1, 0, 0]
    # a launch that signals only after its own wait may still run, nothing before it
    lines = [admit(0, 10), admit(1, 10, early=0), settled(0), settled(1)]
    assert driver(lines) == [0, 0, 1, 0]
    # a barrier settles everything; an unknown (truncated) history settles nothing
    assert driver([admit(0, 10), "barrier 1", settled(0)]) == [0, 1]
    assert driver([f"fill 1 7 1 {CAP + 5}", settled(0, rmax=1 << 40)]) == [0]


def test_in_flight_classifies_what_may_run_beside_the_next_launch(driver):
    lines = [inflight(0), admit(0, 100), inflight(0), inflight(1), "barrier 1", inflight(0),
             admit(1, 100, stream=2), inflight(0), inflight(0, stream=2)]
    assert driver(lines) == [0, 0, 2, 1, 0, 0, 0, 1]
