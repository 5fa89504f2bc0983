"""Write the CPU oracle's fixed-batch AdamW loss trajectories as golden files.

    python tests/golden/make_oracle_trajectories.py [workload ...]

Calls only ``oracle/`` (fed by ``synth``).  For each workload it runs the
number of steps the workload names on one fixed seeded batch (the llm.c test
overfits a single batch with Adam for ten iterations: page «千行C代码训完GPT-2»,
section «测试»), recording the loss of every forward, and stores the result as
``oracle_traj_<workload>.json`` beside this script.
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synth  # noqa: E402
from oracle import ref  # noqa: E402


def trajectory(w, steps=None):
    steps = steps or w.steps
    m = ref.RefModel(ref.config_from(w), w.B, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w, step=0)
    losses = []
    t0 = time.time()
    for t in range(1, steps + 1):
        losses.append(m.step(inp, tgt, t, lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                             weight_decay=w.weight_decay))
    m.close()
    return losses, time.time() - t0


def main(names):
    for name in names:
        w = synth.WORKLOADS[name]
        losses, secs = trajectory(w)
        out = {
            "workload": name,
            "source": "oracle/gpt2_ref.c (REAL=float) via tests/golden/make_oracle_trajectories.py",
            "init_seed": synth.INIT_SEED,
            "token_seed": synth.TOKEN_SEED,
            "batch": "synth.batch(w, step=0), fixed for every step",
            "adamw": {"lr": w.lr, "beta1": w.beta1, "beta2": w.beta2, "eps": w.eps, "weight_decay": w.weight_decay},
            "losses": losses,
            "oracle_seconds": round(secs, 1),
        }
        path = os.path.join(HERE, f"oracle_traj_{name}.json")
        with open(path, "w") as f:
            json.dump(out, f, indent=1)
        print(path, losses, f"{secs:.1f}s")


if __name__ == "__main__":
    main(sys.argv[1:] or ["tiny_L2_C64", "gpt2_124m_B4_T64_fp32"])
