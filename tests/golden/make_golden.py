"""Write the oracle regression fixture for the tiny float32 workload.

The pages print no worked numeric example of the selective scan, so the
stored values here are not the pages': they are the fp64 oracle's outputs
on the seeded tiny workload (2 x 16 x 64, N = 16), written by this script,
which calls only ``oracle/`` and the input generator ``synth/``.  They guard
the oracle against unnoticed changes; the oracle itself is pinned by
tests/oracle_pins.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_f32_oracle.json")


def compute():
    cfg = synth.config(0)
    x = synth.make_inputs(cfg, with_dy=True)
    w = {k: synth.widen(v) for k, v in x.items()}
    out, h_last = oracle.scan_fwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                                  w["delta_bias"], True)
    g = oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                        w["delta_bias"], True, w["dy"])
    return {
        "out[::7]": out.ravel()[::7].tolist(),
        "h_last[::3]": h_last.ravel()[::3].tolist(),
        "dA": g["dA"].ravel().tolist(),
        "dD": g["dD"].tolist(),
        "ddelta_bias": g["ddelta_bias"].tolist(),
        "du[::11]": g["du"].ravel()[::11].tolist(),
        "ddelta[::11]": g["ddelta"].ravel()[::11].tolist(),
        "dz[::11]": g["dz"].ravel()[::11].tolist(),
        "dB[::11]": g["dB"].ravel()[::11].tolist(),
        "dC[::11]": g["dC"].ravel()[::11].tolist(),
    }


if __name__ == "__main__":
    data = compute()
    doc = {
        "what": "fp64 oracle outputs on the seeded tiny float32 workload (Bsz=2, Dch=16, L=64, N=16, "
                "seed 1000, softplus on, D/z/delta_bias present); slices are of the row-major "
                "flattened arrays",
        "source": "written by tests/golden/make_golden.py (calls only oracle/ and synth/); the pages "
                  "print no worked numeric example",
        "values": data,
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", OUT)
