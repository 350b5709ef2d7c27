"""Write oracle_digest.json: SHA-256 digests of the oracle's outputs on fixed inputs.

Calls only the oracle (inputs are drawn here with numpy's PCG64). The digest turns any
change to the oracle's arithmetic into a visible test failure; regenerating it is a
deliberate act whose commit message names the passage, or the reading of it, that
justifies the change.

    python tests/golden/make_oracle_digest.py
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle as O  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_digest.json")


def _h(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def run():
    ora = O.default()
    rng = np.random.Generator(np.random.PCG64(20210204))
    n, W, C = 8192, 4, 512
    res = {}

    st = O.OracleState(n, W, C, x=rng.standard_normal(n) * 0.02, m=np.zeros(n),
                       v=rng.uniform(1e-8, 1e-4, n), wd=0.01,
                       mask=(rng.random(n) > 0.02).astype(np.uint8))
    outs = []
    for step in range(4):
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float16)
        o = ora.compressed_step(st, g)
        outs += [o["wbits"], o["wscale"], o["sbits"], o["sscale"]]
    res["compressed_f16_4steps"] = _h(st.x, st.m, st.ew, st.es, *outs)

    st = O.OracleState(n, W, C, x=rng.standard_normal(n) * 0.02, m=np.zeros(n), v=np.zeros(n))
    for step in range(3):
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
        ora.warmup_step(st, g, bias_correction=(step % 2 == 0))
    res["warmup_f32_3steps"] = _h(st.x, st.m, st.v)

    st = O.OracleState(n, W, C, x=rng.standard_normal(n) * 0.02, m=np.zeros(n), v=np.zeros(n))
    err = np.zeros((W, n), np.float32)
    outs = []
    for step in range(3):
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
        g_bf16 = (g.view(np.uint32) >> 16).astype(np.uint16)      # truncated to bfloat16
        o = ora.loco_step(st, g_bf16, err, beta=0.9, bits=4)
        outs += [o["codes"], o["scales"]]
    res["loco_bf16_3steps"] = _h(st.x, st.m, st.v, err, *outs)
    return res


if __name__ == "__main__":
    res = run()
    res["_about"] = ("SHA-256 of oracle outputs on fixed PCG64 inputs; written by "
                     "tests/golden/make_oracle_digest.py, which calls only the oracle")
    with open(OUT, "w") as f:
        json.dump(res, f, indent=1, sort_keys=True)
    print(json.dumps(res, indent=1))
