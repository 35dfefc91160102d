"""Child process of the CTA-pair / single-SM comparison test.

The library reads MOE_TC_PAIR once per process, so each form of the
tensor-core GEMMs runs in its own process: this script runs the forward of
the 512-expert layer (activations saved, logits kept) on the first T tokens
of the seeded input for each T given and saves the results with torch.save.

    MOE_TC_PAIR=0 python tests/_forms_child.py OUT.pt T1 T2 ...
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402

import top_routed_grouped_gb300 as moe  # noqa: E402

from _util import full_weights, full_x, to_dev  # noqa: E402

KEYS = ("topk_ids", "logits", "topk_w", "shared_sig", "y", "y_routed", "y_shared")
SAVED = ("gu", "h", "gu_shared", "h_shared")


def run(T: int) -> dict:
    W = to_dev(full_weights())
    args = [W[n] for n in ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")]
    o = moe.forward(full_x(T).cuda(), *args, 10, save_for_backward=True, want_logits=True)
    out = {k: o[k].cpu() for k in KEYS}
    out.update({"saved_" + k: o["saved"][k].cpu() for k in SAVED})
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError("device status reports a failed check")
    return out


if __name__ == "__main__":
    path, Ts = sys.argv[1], [int(t) for t in sys.argv[2:]]
    torch.save({T: run(T) for T in Ts}, path)
