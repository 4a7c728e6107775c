"""A small, self-contained case of one kernel, for profilers.

  python profile_case.py --kernel prefill --tokens 8192
  python profile_case.py --kernel decode --batch 128
  python profile_case.py --kernel decode_multi --batch 256 --steps 4
  python profile_case.py --kernel state_copy --batch 256
  python profile_case.py --kernel decode_graph --batch 3 --steps 64
  python profile_case.py --kernel prefill_host --tokens 32768 --seg 5120
  python profile_case.py --kernel in_proj --tokens 32768 --hidden 2048
  python profile_case.py --kernel out_proj --tokens 32768 --hidden 2048

Builds seeded synthetic inputs (the same distributions as the benchmark),
runs the kernel ``--warmup`` times, then ``--iters`` times, and prints the
mean device time per call (CUDA events).  Sized by default so the inputs
exceed the 129 MB L2 while the whole case holds well under 1 GB of device
memory, which keeps an ncu capture short.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import gated_deltanet_linear_06_gb300 as gdn
    import gdn_inputs as gi

    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["prefill", "decode", "decode_multi", "state_copy", "decode_graph", "prefill_host",
                             "in_proj", "out_proj"], required=True)
    ap.add_argument("--tokens", type=int, default=8192, help="prefill: tokens of one sequence")
    ap.add_argument("--seqs", type=int, default=1, help="prefill: equal-length sequences")
    ap.add_argument("--batch", type=int, default=128, help="decode: sequences")
    ap.add_argument("--steps", type=int, default=4, help="decode_multi: tokens per sequence")
    ap.add_argument("--trace", action="store_true", help="decode_multi: also write the SSM trace")
    ap.add_argument("--seg", type=int, default=0, help="prefill_host: tokens per segment (0: default)")
    ap.add_argument("--hidden", type=int, default=2048, help="in_proj / out_proj: hidden size")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()

    dev = torch.device("cuda:0")
    sh = gi.LAYER
    dims = gdn.make_dims(h_k=sh.h_k, h_v=sh.h_v)
    stream = torch.cuda.current_stream(dev)
    if args.kernel == "prefill":
        N, T = args.seqs, args.seqs * args.tokens
        p = {k: v.to(dev) for k, v in gi.make_params(sh, 3).items()}
        x = {k: v.to(dev) for k, v in gi.make_tokens(sh, T, 3).items()}
        cu = gi.cu_seqlens([args.tokens] * N).to(dev)
        conv = torch.zeros(N, 3, sh.cc, device=dev)
        ssm = torch.zeros(N, sh.h_v, 128, 128, device=dev)
        out = torch.empty(T, sh.h_v, 128, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gdn.gdn_workspace_bytes(dims, N, T), dtype=torch.uint8, device=dev)

        def call():
            gdn.gdn_prefill(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                            p["conv_w"], p["norm_w"], cu, conv, ssm, out, ws, stream=stream)
        unit, per_call = "tokens", T
    elif args.kernel == "decode":
        B = args.batch
        p = {k: v.to(dev) for k, v in gi.make_params(sh, 4).items()}
        st = gi.make_states(sh, B, 4, ssm_std=0.1 ** 0.5, conv_std=1.0)
        conv, ssm = st["conv_state"].to(dev), st["ssm_state"].to(dev)
        x = {k: v.to(dev) for k, v in gi.make_tokens(sh, B, 4).items()}
        out = torch.empty(B, sh.h_v, 128, dtype=torch.bfloat16, device=dev)

        def call():
            gdn.gdn_decode_step(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                                p["conv_w"], p["norm_w"], None, B, conv, ssm, out, stream=stream)
        unit, per_call = "seq-steps", B
    elif args.kernel in ("in_proj", "out_proj"):
        T, H = args.tokens, args.hidden
        w = {k: v.to(dev) for k, v in gi.make_proj_weights(sh, H, 6).items()}
        if args.kernel == "in_proj":
            xh = gi.make_hidden(T, H, 6).to(dev)
            qkv = torch.empty(T, sh.cc, dtype=torch.bfloat16, device=dev)
            z = torch.empty(T, sh.h_v, 128, dtype=torch.bfloat16, device=dev)
            a = torch.empty(T, sh.h_v, dtype=torch.bfloat16, device=dev)
            b = torch.empty(T, sh.h_v, dtype=torch.bfloat16, device=dev)
            n_out = gdn.in_proj_features(dims)

            def call():
                gdn.gdn_in_proj(dims, H, xh, w["w_in"], qkv, z, a, b, stream=stream)
        else:
            o = gi.make_hidden(T, sh.cv, 6).to(dev).reshape(T, sh.h_v, 128)
            y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            n_out = H

            def call():
                gdn.gdn_out_proj(dims, H, o, w["w_out"], y, stream=stream)
        k_in = H if args.kernel == "in_proj" else sh.cv
        unit, per_call = "TFLOP", 2e-12 * T * n_out * k_in
    elif args.kernel == "prefill_host":
        # activations in pinned host memory, output back to it: the copies are
        # part of each call
        N, T = args.seqs, args.seqs * args.tokens
        p = {k: v.to(dev) for k, v in gi.make_params(sh, 3).items()}
        x = {k: v.pin_memory() for k, v in gi.make_tokens(sh, T, 3).items()}
        cu = gi.cu_seqlens([args.tokens] * N)
        conv = torch.zeros(N, 3, sh.cc, device=dev)
        ssm = torch.zeros(N, sh.h_v, 128, 128, device=dev)
        out = torch.empty(T, sh.h_v, 128, dtype=torch.bfloat16).pin_memory()
        ws = torch.empty(gdn.gdn_prefill_host_workspace_bytes(dims, N, T, args.seg),
                         dtype=torch.uint8, device=dev)

        def call():
            gdn.gdn_prefill_host(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                                 p["conv_w"], p["norm_w"], cu, conv, ssm, out, ws,
                                 seg_tokens=args.seg, stream=stream)
        unit, per_call = "tokens", T
    elif args.kernel == "decode_graph":
        B, S = args.batch, args.steps
        p = {k: v.to(dev) for k, v in gi.make_params(sh, 1).items()}
        st = gi.make_states(sh, B, 1, ssm_std=0.1 ** 0.5, conv_std=1.0)
        conv, ssm = st["conv_state"].to(dev), st["ssm_state"].to(dev)
        x = {k: v.to(dev) for k, v in gi.make_tokens(sh, S * B, 1).items()}
        out = torch.empty(S, B, sh.h_v, 128, dtype=torch.bfloat16, device=dev)
        graph = gdn.gdn_decode_graph_create(dims, S, x["qkv"], x["z"], x["a"], x["b"], p["A_log"],
                                            p["dt_bias"], p["conv_w"], p["norm_w"], None, B, conv,
                                            ssm, out)

        def call():
            graph.launch(stream=stream)
        unit, per_call = "seq-steps", B * S
    elif args.kernel == "state_copy":
        B = args.batch
        st = gi.make_states(sh, B, 5, ssm_std=0.1 ** 0.5, conv_std=1.0)
        conv, ssm = st["conv_state"].to(dev), st["ssm_state"].to(dev)
        bconv, bssm = torch.empty_like(conv), torch.empty_like(ssm)

        def call():
            gdn.gdn_state_copy(dims, conv, ssm, bconv, bssm, stream=stream)
        unit, per_call = "GB", 2e-9 * gdn.gdn_state_bytes(dims) * B
    else:
        B, K = args.batch, args.steps
        p = {k: v.to(dev) for k, v in gi.make_params(sh, 4).items()}
        st = gi.make_states(sh, B, 4, ssm_std=0.1 ** 0.5, conv_std=1.0)
        conv, ssm = st["conv_state"].to(dev), st["ssm_state"].to(dev)
        x = {k: v.to(dev) for k, v in gi.make_tokens(sh, B * K, 4).items()}
        out = torch.empty(B, K, sh.h_v, 128, dtype=torch.bfloat16, device=dev)
        trace = torch.empty(B, K, sh.h_v, 128, 128, device=dev) if args.trace else None

        def call():
            gdn.gdn_decode_multi(dims, x["qkv"], x["z"], x["a"], x["b"], p["A_log"], p["dt_bias"],
                                 p["conv_w"], p["norm_w"], None, B, conv, ssm, out, K,
                                 ssm_trace=trace, stream=stream)
        unit, per_call = "seq-steps", B * K

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.iters):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.iters
    print(f"{args.kernel}: {ms:.4f} ms per call, {per_call / (ms * 1e-3):.4g} {unit}/s")


if __name__ == "__main__":
    main()
