"""Reader for tests/golden/plan_small.txt (hand-counted bucket plans)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "plan_small.txt")


def load_cases(path: str = GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        elif key == "buckets":
            cur[key] = [tuple(int(x) for x in v.split(":")) for v in vals]
        elif key in ("bucket_bytes", "n_padded"):
            cur[key] = int(vals[0])
        else:
            cur[key] = [int(v) for v in vals]
    return cases
