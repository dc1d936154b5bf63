"""Write tests/golden/tiny_oracle.json from the oracle alone.

The pages print no loss values, so the stored numbers are the oracle's own
(pinned by path enumeration in test_oracle_pins.py) for the tiny seeded
workload; they guard the oracle and the input recipe against silent change.
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from transducer_loss_asr_gb300.workloads import make_inputs  # noqa: E402


def main():
    inp = make_inputs("tiny")
    w = inp["workload"]
    z = inp["logits"].float().numpy()
    r = oracle.tdt_loss(z, inp["labels"].numpy(), inp["logit_lens"].numpy(),
                        inp["label_lens"].numpy(), w.durations, w.blank, w.sigma, w.reduction)
    out = {
        "workload": "tiny",
        "source": "oracle/tdt_oracle.c via oracle.tdt_loss (float64)",
        "utt_loss": [float(x) for x in r.utt_loss],
        "grad_abs_sum": float(np.abs(r.grad).sum()),
        "grad_max": float(r.grad.max()),
        "grad_min": float(r.grad.min()),
        "logits_sum": float(z.astype(np.float64).sum()),
        "labels": inp["labels"].tolist(),
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
