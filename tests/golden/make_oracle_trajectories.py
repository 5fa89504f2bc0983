"""Write the CPU oracle's fixed-batch AdamW loss trajectories as golden files.

    python tests/golden/make_oracle_trajectories.py [workload ...]
    python tests/golden/make_oracle_trajectories.py --parity [workload ...]

Calls only ``oracle/`` (fed by ``synth``).  For each workload it runs the
number of steps the workload names on one fixed seeded batch (the llm.c test
overfits a single batch with Adam for ten iterations: page «千行C代码训完GPT-2»,
section «测试»), recording the loss of every forward, and stores the result as
``oracle_traj_<workload>.json`` beside this script.

``--parity`` covers the T = 1024 workloads (GPT-2 124M / 350M / 774M shapes),
whose full batches are too slow for the oracle to train on:

* ``oracle_traj_<workload>_B<b>.json``: the trajectory on the first ``b``
  sequences of the workload's batch (``PARITY_RUNS`` gives ``b`` and the step
  count), same architecture, same init, same AdamW settings;
* ``oracle_initloss_<workload>.json``: the loss of the initial model on the
  FULL batch.  Every sequence's forward is independent of the others, and the
  loss is the mean over all B*T positions, so it equals the mean of the B
  per-sequence losses; the oracle computes them one sequence at a time.
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

# (sub-batch B, AdamW steps) of the reduced-batch parity trajectories: B is
# set by the oracle's CPU time (one 124M step at B = 1, T = 1024 takes about
# 30 s on 8 cores; 350M about 3x that, 774M about 6x)
PARITY_RUNS = {
    "gpt2_124m_B16_T1024_bf16": (2, 20),
    "gpt2_350m_B8_T1024_bf16": (1, 10),
    "gpt2_774m_B4_T1024_bf16": (1, 10),
}


def trajectory(w, steps=None, B=None):
    steps = steps or w.steps
    B = B or w.B
    m = ref.RefModel(ref.config_from(w), B, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w, step=0)
    inp, tgt = inp[:B].copy(), tgt[:B].copy()
    losses = []
    t0 = time.time()
    for t in range(1, steps + 1):
        losses.append(m.step(inp, tgt, t, lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                             weight_decay=w.weight_decay))
        print(f"  {w.name} B={B} step {t}: {losses[-1]:.6f} ({time.time() - t0:.0f}s)", flush=True)
    m.close()
    return losses, time.time() - t0


def full_batch_initial_loss(w):
    """Per-sequence losses of the initial model on the workload's full batch."""
    m = ref.RefModel(ref.config_from(w), 1, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w, step=0)
    per_seq = []
    t0 = time.time()
    for b in range(w.B):
        per_seq.append(m.forward(inp[b:b + 1].copy(), tgt[b:b + 1].copy()))
        print(f"  {w.name} sequence {b}: {per_seq[-1]:.6f} ({time.time() - t0:.0f}s)", flush=True)
    m.close()
    return per_seq, time.time() - t0


def header(w):
    return {
        "workload": w.name,
        "source": "oracle/gpt2_ref.c (REAL=float) via tests/golden/make_oracle_trajectories.py",
        "init_seed": synth.INIT_SEED,
        "token_seed": synth.TOKEN_SEED,
        "adamw": {"lr": w.lr, "beta1": w.beta1, "beta2": w.beta2, "eps": w.eps, "weight_decay": w.weight_decay},
    }


def write(name, out):
    path = os.path.join(HERE, name)
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path, flush=True)


def main(argv):
    parity = "--parity" in argv
    names = [a for a in argv if not a.startswith("--")]
    if parity:
        for name in names or list(PARITY_RUNS):
            w = synth.WORKLOADS[name]
            per_seq, secs = full_batch_initial_loss(w)
            out = header(w)
            out.update({"batch": f"synth.batch(w, step=0): all {w.B} sequences, T={w.T}",
                        "per_sequence_losses": per_seq, "loss": float(np.mean(per_seq)),
                        "oracle_seconds": round(secs, 1)})
            write(f"oracle_initloss_{name}.json", out)
            B, steps = PARITY_RUNS[name]
            losses, secs = trajectory(w, steps=steps, B=B)
            out = header(w)
            out.update({"batch": f"the first {B} sequence(s) of synth.batch(w, step=0), fixed for every step",
                        "B": B, "T": w.T, "steps": steps, "losses": losses, "oracle_seconds": round(secs, 1)})
            write(f"oracle_traj_{name}_B{B}.json", out)
        return
    for name in names or ["tiny_L2_C64", "gpt2_124m_B4_T64_fp32"]:
        w = synth.WORKLOADS[name]
        losses, secs = trajectory(w)
        out = header(w)
        out.update({"batch": "synth.batch(w, step=0), fixed for every step", "losses": losses,
                    "oracle_seconds": round(secs, 1)})
        write(f"oracle_traj_{name}.json", out)


if __name__ == "__main__":
    main(sys.argv[1:])
