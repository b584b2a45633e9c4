"""Writes oracle_small.json: small fixed inputs and the fp64 oracle's outputs for them.

Calls nothing but ``oracle`` (and numpy's seeded generator for the inputs, which are
stored in the fixture as well).  Rerun it only together with a change of the oracle's
arithmetic; ``tests/test_golden.py`` checks the oracle against the stored values.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

# name, (NB, H, T, dk, dv), gated, with_h0, options, packed lengths (NB = 1) or None
CASES = [
    ("deltanet_T9_d3", (1, 1, 9, 3, 3), False, False, {}, None),
    ("gated_h0_T11_dk4_dv3", (2, 1, 11, 4, 3), True, True, {"scale": 0.75}, None),
    ("longhorn_raw_keys_T7_d3", (1, 2, 7, 3, 3), True, False, {"qk_l2norm": False, "longhorn": True}, None),
    ("packed_3_0_5_d2", (1, 2, 8, 2, 2), True, True, {}, [3, 0, 5]),
]


def case_inputs(i, shape, gated, with_h0, lengths):
    NB, H, T, dk, dv = shape
    rng = np.random.default_rng(1000 + i)
    x = {
        "q": rng.standard_normal((NB, H, T, dk)),
        "k": rng.standard_normal((NB, H, T, dk)),
        "v": rng.standard_normal((NB, H, T, dv)),
        "beta": 1.0 / (1.0 + np.exp(-rng.standard_normal((NB, H, T)))),
        "g": -np.log1p(np.exp(rng.standard_normal((NB, H, T)))) / 4 if gated else None,
    }
    n = len(lengths) if lengths else NB
    x["h0"] = 0.3 * rng.standard_normal((n, H, dk, dv)) if with_h0 else None
    x["do"] = rng.standard_normal((NB, H, T, dv))
    x["dhT"] = 0.1 * rng.standard_normal((n, H, dk, dv))
    x["cu_seqlens"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64) if lengths else None
    return x


def run_oracle(x, opts):
    o, hT = oracle.fwd(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], cu_seqlens=x["cu_seqlens"], **opts)
    gr = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], x["do"], x["dhT"],
                    cu_seqlens=x["cu_seqlens"], **opts)
    out = {"o": o, "hT": hT}
    out.update({"grad_" + n: a for n, a in gr.items() if a is not None})
    return out


def tolist(a):
    return None if a is None else np.asarray(a).tolist()


def main():
    cases = []
    for i, (name, shape, gated, with_h0, opts, lengths) in enumerate(CASES):
        x = case_inputs(i, shape, gated, with_h0, lengths)
        out = run_oracle(x, opts)
        cases.append({
            "name": name,
            "options": opts,
            "inputs": {k: tolist(v) for k, v in x.items()},
            "outputs": {k: tolist(v) for k, v in out.items()},
        })
    what = ("fp64 oracle outputs (forward o, h_T and every gradient of sum(o*do) + sum(h_T*dhT)) "
            "for small fixed inputs; written by tests/golden/make_golden.py, which calls only oracle/")
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        # one case per line
        f.write('{"what": ' + json.dumps(what) + ',\n "cases": [\n')
        f.write(",\n".join(json.dumps(c) for c in cases))
        f.write("\n]}\n")


if __name__ == "__main__":
    main()
