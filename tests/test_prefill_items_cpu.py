"""The prefill attention kernels' work items (csrc/k2_items.h), on the CPU
through a small driver built with g++.

Checked against what the items must be, not against the decoding itself:
every (sequence, query block, kv head, head group) of a launch is exactly one
item; items are numbered heaviest first (query block descending, then
sequence, kv head, head group); each worker gets its snake-order share; and an
item's rows, positions and key tiles follow from its query block, the
sequence's start and length and the attention window (row i sees keys
max(0, i + 1 - W) .. i, or 0 .. i without a window)."""
import os
import random
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "gqa_attention_preallocated_qa_gb300", "csrc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("items") / "k2_items_driver")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wno-unknown-pragmas", "-I", CSRC,
                    os.path.join(HERE, "native", "k2_items_driver.cpp"), "-o", exe], check=True)

    def run(cases):
        lines = []
        for c in cases:
            pad = lambda v: list(v) + [0] * (8 - len(v))
            lines.append(" ".join(map(str, [c["nseq"], c["Hkv"], c["G"], c["npairs"], c["hpi"], c["window"],
                                            *pad(c["len"]), *pad(c["start"]), *pad(c["cu"]), c["workers"]])))
        out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True,
                             check=True).stdout.split("\n")
        res, cur = [], []
        for ln in out:
            if ln == "end":
                res.append(cur)
                cur = []
            elif ln:
                cur.append(tuple(int(x) for x in ln.split()))
        return res
    return run


def case(lens, starts=None, Hkv=8, G=4, hpi=2, window=0, workers=152):
    starts = list(starts) if starts is not None else [0] * len(lens)
    cu = [sum(lens[:i]) for i in range(len(lens))]
    return {"nseq": len(lens), "len": list(lens), "start": starts, "cu": cu, "Hkv": Hkv, "G": G,
            "hpi": hpi, "npairs": (G + hpi - 1) // hpi, "window": window, "workers": workers}


def check(c, items):
    nseq, Hkv, G, hpi, npairs, W, P = c["nseq"], c["Hkv"], c["G"], c["hpi"], c["npairs"], c["window"], c["workers"]
    want = [(b, qb, kvh, pr) for b in range(nseq) for qb in range(-(-c["len"][b] // 128))
            for kvh in range(Hkv) for pr in range(npairs)]
    assert len(items) == len(want)
    by_idx = {}
    for (w, k, idx, b, kvh, qb, h0, L, qmin, j0, nkv, jmask, row0, same) in items:
        assert same == 1
        assert idx not in by_idx
        # the worker's snake-order share
        assert idx == k * P + (P - 1 - w if k & 1 else w)
        pr, r = divmod(h0 - kvh * G, hpi)
        assert r == 0 and 0 <= pr < npairs
        by_idx[idx] = (b, qb, kvh, pr)
        # rows, positions and key tiles from the definition
        assert L == c["len"][b] and qmin == c["start"][b] + 128 * qb and row0 == c["cu"][b] + 128 * qb
        rows = min(128, L - 128 * qb)
        assert rows >= 1
        first_row_lo = max(0, qmin + 1 - W) if W > 0 else 0     # the block's lowest visible key
        last_key = qmin + rows - 1                               # the block's highest visible key
        assert j0 == first_row_lo // 128 and j0 + nkv - 1 == last_key // 128
        # tiles below jmask hold no key past any row's position; tile jmask may
        assert jmask * 128 <= qmin < (jmask + 1) * 128
    assert sorted(by_idx) == list(range(len(want)))
    order = [by_idx[i] for i in range(len(want))]
    assert sorted(order) == sorted(want) and len(set(order)) == len(want)
    # heaviest first: query block descending, then sequence, kv head, head group
    assert order == sorted(want, key=lambda t: (-t[1], t[0], t[2], t[3]))


def test_benchmark_prefill_items(driver):
    cases = [case([2048] * 4), case([2048] * 4, G=4, hpi=4, workers=76),
             case([512, 1024, 1536, 2048], G=4, hpi=4, workers=76), case([512], hpi=1, workers=152)]
    for c, items in zip(cases, driver(cases)):
        check(c, items)


def test_ragged_chunks_windows_and_tails(driver):
    rng = random.Random(7)
    cases = []
    for _ in range(60):
        n = rng.randint(1, 8)
        lens = [rng.choice([0, 1, 127, 128, 129, rng.randint(1, 1500)]) for _ in range(n)]
        if not any(lens):
            lens[0] = 1
        starts = [rng.choice([0, 0, rng.randint(0, 3000)]) for _ in range(n)]
        G = rng.choice([1, 2, 4, 8])
        hpi = rng.choice([h for h in (1, 2, 4) if h <= G])
        cases.append(case(lens, starts, Hkv=rng.choice([1, 2, 8]), G=G, hpi=hpi,
                          window=rng.choice([0, 0, 1, 64, 200, 1024]), workers=rng.choice([1, 3, 76, 152])))
    for c, items in zip(cases, driver(cases)):
        check(c, items)


def test_a_mistaken_order_would_be_seen(driver):
    """The checks see a swapped pair of items: the property test is not vacuous."""
    c = case([300, 200], Hkv=2, G=2, hpi=1, workers=5)
    items = driver([c])[0]
    check(c, items)
    swapped = list(items)
    i, j = 0, 1
    a, b = swapped[i], swapped[j]
    swapped[i] = a[:3] + b[3:]
    swapped[j] = b[:3] + a[3:]
    with pytest.raises(AssertionError):
        check(c, swapped)
