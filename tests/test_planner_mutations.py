"""The planner's pins catch plausible mistakes.

Each case plants one slip in a private copy of the oracle's Python planner
(oracle/__init__.py, on the CPU, in a temporary directory) and runs the
planner pins (tests/test_planner.py: hand-counted plans, BERT-large bucket
counts, invariants) against that copy.  The pins must fail for every slip.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "oracle", "__init__.py")

MUTATIONS = {
    "tensors laid out in forward order":
        ("    for t in range(T - 1, -1, -1):\n        if numel[t] < 0:",
         "    for t in range(T):\n        if numel[t] < 0:"),
    "spans not padded to 8 elements":
        ("span = (numel[t] + PAD_ELEMS - 1) // PAD_ELEMS * PAD_ELEMS",
         "span = numel[t]"),
    "bucket closes only above the cap":
        ("if bucket_bytes > 0 and open_bytes >= bucket_bytes:",
         "if bucket_bytes > 0 and open_bytes > bucket_bytes:"),
    "cap counted in elements, not bytes":
        ("open_bytes += span * GRAD_BYTES", "open_bytes += span"),
    "cap 0 cuts every tensor":
        ("if bucket_bytes > 0 and open_bytes >= bucket_bytes:",
         "if bucket_bytes >= 0 and open_bytes >= bucket_bytes:"),
    "last open bucket dropped":
        ("    if cursor > open_begin:\n        buckets.append((open_begin, cursor))\n"
         "    return offsets, buckets, cursor",
         "    return offsets, buckets, cursor"),
    "ready after the highest layer, not the lowest":
        ("if lowest is None or layer_of[t] < lowest:",
         "if lowest is None or layer_of[t] > lowest:"),
    "open bucket's bytes not reset":
        ("            open_begin = cursor\n            open_bytes = 0",
         "            open_begin = cursor"),
    "shard ends rounded up instead of down":
        ("            stop_unit = (units * (q + 1)) // world",
         "            stop_unit = -((-units * (q + 1)) // world)"),
    "shard begins one unit late":
        ("            first_unit = (units * q) // world",
         "            first_unit = (units * q + world - 1) // world"),
    "ragged tail of a bucket dropped":
        ("            if q == world - 1:\n                hi = end",
         "            if q == world - 1:\n                hi = hi"),
    "shard state offsets not accumulated":
        ("            used[q] += hi - lo", "            used[q] = hi - lo"),
}


def _run_pins_on(mutated_source: str) -> subprocess.CompletedProcess:
    work = tempfile.mkdtemp(prefix="planner_mutant_")
    try:
        ign = shutil.ignore_patterns("*.so", "__pycache__", "_build")
        shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(work, "oracle"),
                        ignore=ign)
        with open(os.path.join(work, "oracle", "__init__.py"), "w") as f:
            f.write(mutated_source)
        shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(work, "tests"),
                        ignore=ign)
        pkg = "gradient_reduce_optimizer_gb300"
        os.makedirs(os.path.join(work, pkg))
        for name in ("__init__.py", "capi.py", "workloads.py"):
            shutil.copy(os.path.join(ROOT, pkg, name), os.path.join(work, pkg))
        shutil.copy(os.path.join(ROOT, "pytest.ini"), work)
        return subprocess.run(
            [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:warnings",
             "tests/test_planner.py"],
            cwd=work, capture_output=True, text=True, timeout=300)
    finally:
        shutil.rmtree(work, ignore_errors=True)


def test_every_planted_planner_slip_fails_a_pin():
    src = open(SOURCE).read()
    for name, (old, _) in MUTATIONS.items():
        assert src.count(old) == 1, f"mutation site not unique: {name}"
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = dict(zip(MUTATIONS, ex.map(
            lambda kv: _run_pins_on(src.replace(*kv)), MUTATIONS.values())))
    survivors = [n for n, r in results.items() if r.returncode == 0]
    assert not survivors, f"pins missed: {survivors}"
    broken = [n for n, r in results.items()
              if r.returncode != 1 or "failed" not in r.stdout]
    assert not broken, f"mutant did not run cleanly: {broken}"


def test_unmutated_planner_copy_passes():
    r = _run_pins_on(open(SOURCE).read())
    assert r.returncode == 0, r.stdout[-2000:]
