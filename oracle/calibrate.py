"""Write the stored global scales of the synthetic full-size layer.

Test infrastructure only (see the package docstring). Run as
``python -m oracle.calibrate``; it calls nothing but this package and the
seeded input generators, and writes
``nvfp4_mixture_experts_route_gb300/calibration.json``.

The workloads set the global scales "from the absmax of a calibration draw";
the recipe is not on the pages, so this is the project's reading (open point
10): with x_cal a separate bf16 N(0, 1) draw of 8 tokens routed uniformly,

    a1_gscale = 448 * 6 / max |x_cal|
    a2_gscale = 448 * 6 / max |h_cal|

where h_cal = SiLU(gate) * up of the oracle on x_cal quantized with that
a1_gscale. 448 * 6 is the largest e4m3 scale times the largest e2m1 value,
so the calibration absmax lands on the largest representable product. Both
are rounded to fp32.
"""
from __future__ import annotations

import json
import sys

import numpy as np

from nvfp4_mixture_experts_route_gb300 import inputs

from .codecs import bf16_bits_to_f64
from .layer import expert_rows

RANGE = 448.0 * 6.0


def calibrate(w: inputs.Workload) -> dict[str, float]:
    layer = inputs.make_layer(w)
    cal = inputs.calibration_draw(w)
    a1 = float(np.float32(RANGE / np.max(np.abs(bf16_bits_to_f64(cal["x"])))))
    er = expert_rows(cal["x"], cal["topk_ids"], layer, a1, 1.0, mode="exact", return_intermediate=True)
    hmax = float(np.max(np.abs(er["h"].astype(np.float32))))
    a2 = float(np.float32(RANGE / hmax))
    return {"a1_gscale": a1, "a2_gscale": a2, "x_cal_absmax": float(np.max(np.abs(bf16_bits_to_f64(cal["x"])))),
            "h_cal_absmax": hmax}


def main() -> int:
    done: dict[str, dict] = {}
    for w in inputs.WORKLOADS.values():
        if w.unit_global_scales or w.layer_key in done:
            continue
        done[w.layer_key] = calibrate(w)
        print(w.layer_key, done[w.layer_key], file=sys.stderr)
    with open(inputs.CALIBRATION_FILE, "w") as f:
        json.dump(done, f, indent=1, sort_keys=True)
        f.write("\n")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
