"""Write the oracle's per-alpha errors for the full-size synthetic layers.

    python tests/golden/make_config_errs.py [name ...]

For each named workload (default: the three large ones) this draws the layer
with seed 0 from ``synthetic`` and runs the CPU oracle's whole alpha grid
(``oracle.awq_oracle.awq_search``: float64 statistics, powers, centring and
errors, float32 group quantizer), then stores every alpha's error, the kept
index and the oracle's wall time to ``config_errs_<name>.json`` beside this
script.  The GPU parity test compares the library's errors with these over
the whole grid.  It imports nothing but the oracle and the seeded input
generator, so no stored value comes from the CUDA path.

The values are float64 written with ``repr`` precision (JSON floats round
trip exactly).  The wall time is this host's, for the record only.
"""
from __future__ import annotations

import json
import os
import platform
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import awq_oracle as O  # noqa: E402
from synthetic import config_by_name, make_layer  # noqa: E402

LARGE = ["up-11008x4096-n512", "qkv-12288x4096-n2048", "down-8192x28672-n1024"]


def path_for(name: str) -> str:
    return os.path.join(HERE, "config_errs_%s.json" % name)


def write(name: str) -> dict:
    cfg = config_by_name(name)
    W, X = make_layer(cfg, seed=0)
    Wn, Xn = W.float().numpy(), X.double().numpy()
    del W, X
    t0 = time.perf_counter()
    res = O.awq_search(Wn, Xn, cfg.bits, cfg.group, cfg.grid, cfg.sym)
    wall = time.perf_counter() - t0
    rec = {
        "workload": name, "seed": 0, "bits": cfg.bits, "group": cfg.group, "sym": cfg.sym,
        "grid": cfg.grid, "errs": [float(e) for e in res.errs], "best": int(res.best),
        "oracle_wall_s": round(wall, 1), "oracle_host_cores": os.cpu_count(),
        "oracle_host": platform.processor() or platform.machine(),
    }
    with open(path_for(name), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


def main(argv):
    for name in (argv or LARGE):
        rec = write(name)
        print("%s: best %d, err %.6e, oracle %.1f s on %d cores"
              % (name, rec["best"], rec["errs"][rec["best"]], rec["oracle_wall_s"],
                 rec["oracle_host_cores"]), flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
