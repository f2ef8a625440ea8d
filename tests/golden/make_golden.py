"""Write tests/golden/tiny_oracle.json: the oracle's results on the 'tiny' workload.

Calls only the oracle and the seeded input generator.  The stored values pin the
generator + oracle pair across machines (x86 and Arm hosts must reproduce the
same inputs bit for bit and the same float64 results); they are not taken from
the pages, which print no worked example.

Usage:  python tests/golden/make_golden.py
"""

import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from synth import make_workload, materialize  # noqa: E402


def tiny_record():
    b = materialize(make_workload("tiny"))
    w = b.w
    per, loss = oracle.opd_loss_fwd(b.draft_f64, b.target_f64, b.doff, w.clip_c, w.ce_weight)
    ver = oracle.verify_packed(b.target_f64, b.tokens, b.doff)
    grads = oracle.opd_loss_bwd(b.draft_f64, b.target_f64, b.doff, w.clip_c, w.ce_weight)
    return dict(
        workload="tiny",
        inputs_sha256=hashlib.sha256(b.draft.tobytes() + b.target.tobytes() + b.tokens.tobytes()).hexdigest(),
        doff=[int(x) for x in b.doff],
        loss=loss,
        kl=[per[d]["kl"] for d in range(w.num_draft_rows)],
        ce=[per[d]["ce"] for d in range(w.num_draft_rows)],
        lse_z=[per[d]["lse_z"] for d in range(w.num_draft_rows)],
        lse_t=[per[d]["lse_t"] for d in range(w.num_draft_rows)],
        S=[per[d]["S"] for d in range(w.num_draft_rows)],
        n_clipped=[per[d]["n_clipped"] for d in range(w.num_draft_rows)],
        accept_len=[ver[i]["accept_len"] for i in range(w.num_requests)],
        bonus_token=[ver[i]["bonus_token"] for i in range(w.num_requests)],
        accept_rate=[float(ver[i]["accept_rate"]) for i in range(w.num_requests)],
        grad_l1=[float(np.sum(np.abs(grads[d]))) for d in range(w.num_draft_rows)],
    )


if __name__ == "__main__":
    rec = tiny_record()
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(rec, f, indent=1)
    print("wrote tiny_oracle.json, loss", rec["loss"])
