"""Optional record of the errors the parity tests measure: when the environment
variable FATTN_PARITY_REPORT names a file, each call appends one JSON line
{"case": ..., "<output>": [max_abs, mean_abs], ...}.  The tests' pass/fail
decisions do not depend on it."""
import json
import os


def record(case, **errors):
    path = os.environ.get("FATTN_PARITY_REPORT")
    if not path:
        return
    line = {"case": case}
    for name, val in errors.items():
        line[name] = [float(v) for v in val] if isinstance(val, (tuple, list)) else float(val)
    with open(path, "a") as f:
        f.write(json.dumps(line) + "\n")
