"""Op-level cases for profiling one kernel family in isolation (for example
under ncu): a linear-layer forward, or a causal attention backward (which runs
the attention forward first), on seeded normal inputs, through the C ABI; or
whole training steps of a named workload with fewer layers, which runs every
per-layer kernel at the workload's shapes while holding a few GB on the device.

    python -m gpt_train_step_02_b300.opcase matmul --N 16384 --IC 768 --OC 3072 --precision bf16
    python -m gpt_train_step_02_b300.opcase attention --B 16 --T 1024 --C 768 --NH 12 --precision bf16
    python -m gpt_train_step_02_b300.opcase step --workload gpt2_774m_B4_T1024_bf16 --layers 2

Each case runs --repeat times (default 3) on cuda:0, then synchronises.
"""
import argparse
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="case", required=True)
    mm = sub.add_parser("matmul", help="out = x W^T + b, x (N, IC), W (OC, IC)")
    mm.add_argument("--N", type=int, default=16384)
    mm.add_argument("--IC", type=int, default=768)
    mm.add_argument("--OC", type=int, default=3072)
    at = sub.add_parser("attention", help="attention backward of qkv (B, T, 3C) with NH heads")
    at.add_argument("--B", type=int, default=16)
    at.add_argument("--T", type=int, default=1024)
    at.add_argument("--C", type=int, default=768)
    at.add_argument("--NH", type=int, default=12)
    for p in (mm, at):
        p.add_argument("--precision", choices=["fp32", "bf16"], default="bf16")
    st = sub.add_parser("step", help="training steps (forward, zero_grad, backward, AdamW) of a workload")
    st.add_argument("--workload", default="gpt2_774m_B4_T1024_bf16")
    st.add_argument("--layers", type=int, default=0, help="layer count in place of the workload's (0: its own)")
    for p in (mm, at, st):
        p.add_argument("--repeat", type=int, default=3)
    args = ap.parse_args(argv)

    if args.case == "step":
        import dataclasses

        import torch

        import gpt_train_step_02_b300 as g
        import synth

        w = synth.WORKLOADS[args.workload]
        if args.layers:
            w = dataclasses.replace(w, name=f"{w.name}_L{args.layers}", num_layers=args.layers)
        m = g.GPT2(w, seed=synth.INIT_SEED)
        inp, tgt = synth.batch(w)
        for t in range(1, args.repeat + 1):
            m.train_step(inp, tgt, t, w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
        m.sync()
        m.close()
        torch.cuda.synchronize()
        print("ok", args.case, w.name)
        return 0

    import torch

    import gpt_train_step_02_b300 as g

    prec = g.GPT2_PREC_BF16 if args.precision == "bf16" else g.GPT2_PREC_FP32
    dev = "cuda"
    torch.manual_seed(0)
    if args.case == "matmul":
        x = torch.randn(args.N, args.IC, device=dev)
        W = torch.randn(args.OC, args.IC, device=dev) * 0.02
        b = torch.zeros(args.OC, device=dev)
        out = torch.empty(args.N, args.OC, device=dev)
        for _ in range(args.repeat):
            g.matmul_forward(out, x, W, b, precision=prec)
    else:
        qkv = torch.randn(args.B, args.T, 3 * args.C, device=dev)
        dy = torch.randn(args.B, args.T, args.C, device=dev)
        dqkv = torch.empty_like(qkv)
        for _ in range(args.repeat):
            g.attention_backward(dqkv, dy, qkv, args.NH, precision=prec)
    torch.cuda.synchronize()
    print("ok", args.case)
    return 0


if __name__ == "__main__":
    sys.exit(main())
