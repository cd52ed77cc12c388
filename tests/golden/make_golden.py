"""Write tests/golden/tiny_oracle.json from the fp64 oracle alone.

The pages print no worked numerical example, so the stored values here are the oracle's own
output on the seeded tiny workload (1 layer, 1 KV head x 4 query heads, d = 64, n = 1024,
eta = 1/8, H = 4 + 64, eps = delta = 0.05, Philox seed 0).  They pin the oracle against silent
drift: tests/test_golden.py recomputes them and compares.  Only oracle/ and the input generator
are called.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
from verified_kv_cache_poissoncomp_gb300 import inputs as I  # noqa: E402


def _bits(mask):
    """A boolean mask as a hex string (bit i of the big-endian number = token i)."""
    return "%x" % int("".join("1" if b else "0" for b in reversed(list(mask))) or "0", 2)


def compute():
    w = I.tiny()
    pc = O.poissoncomp(w.tau[0, 0, 0], w.eta, w.n_sink, w.n_local, w.seed)
    K = O.bf16_to_f64(w.kv[0, 0, 0, :, 0, :])
    V = O.bf16_to_f64(w.kv[0, 0, 0, :, 1, :])
    queries = []
    for t in range(w.queries.shape[0]):
        qs = O.bf16_to_f64(w.queries[t, 0])
        u = O.attend_unit(qs, K, K, V, pc["r32"], pc["resident"], w.eps, w.delta)
        heads = []
        for hd in u["heads"]:
            c, e = hd["cert"], hd["est"]
            heads.append(dict(certified=c["certified"], k_star=c["k_star"],
                              eps_L=c["eps_L"], beta=c["beta"], D=c["D"],
                              F=_bits(c["F"]),
                              lse=e["lse"], o=[float(x) for x in e["o"][:8]]))
        fetch = [False] * w.n
        for i in u["fetch_ids"]:
            fetch[int(i)] = True
        queries.append(dict(heads=heads, fetch_ids=_bits(fetch)))
    return dict(c_exact=pc["c_exact"], c32=float(pc["c32"]), count=pc["count"],
                resident=_bits(pc["resident"]), queries=queries)


if __name__ == "__main__":
    out = os.path.join(HERE, "tiny_oracle.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=0)
    print(out)
