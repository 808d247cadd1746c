"""Write eps_configs.json: the search distance of each synthetic workload.

Calls only the oracle (fp64 brute force) and the seeded generators.  For
workload c, 1,000 query indices are drawn without replacement with
numpy.random.default_rng(1000 + c); eps is the oracle's picker result for the
workload's target mean neighbour count (self excluded), and the sampled mean
is re-counted with the float32 eps to confirm it equals the target (exactly
when a float32 lies between the two order statistics that bracket it).

    python tests/golden/make_eps.py [config ...]
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import datagen  # noqa: E402
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "eps_configs.json")
N_SAMPLE = 1000


def pick(cfg: int) -> dict:
    name, n, d, k = datagen.CONFIGS[cfg]
    x = datagen.generate(cfg)
    q = datagen.sample_queries(n, N_SAMPLE, seed=1000 + cfg)
    t0 = time.time()
    r = oracle.pick_eps(x, k, q)
    row_ptr, _, _, _ = oracle.rows(x, r["eps"], q, band=0.0)
    sampled_mean = (int(row_ptr[-1]) - q.size) / q.size
    r.update({"config": cfg, "workload": name, "n": n, "d": d, "sample_seed": 1000 + cfg,
              "sampled_mean_neighbours": sampled_mean, "seconds": round(time.time() - t0, 1)})
    # eps is a float32; when no float32 separates a and b the sampled mean
    # can miss K by a pair or two
    if abs(sampled_mean - k) > 0.01:
        raise SystemExit("config %d: sampled mean %r != %d" % (cfg, sampled_mean, k))
    return r


def main(argv):
    cfgs = [int(a) for a in argv] or sorted(datagen.CONFIGS)
    data = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            data = json.load(f)
    for c in cfgs:
        r = pick(c)
        print(json.dumps(r), flush=True)
        data[str(c)] = r
        with open(OUT, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
            f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:])
