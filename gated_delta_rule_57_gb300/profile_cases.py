"""Run the hot path on one named workload, for profilers.

    python -m gated_delta_rule_57_gb300.profile_cases prefill [--B 8] [--calls 4]
    python -m gated_delta_rule_57_gb300.profile_cases decode  [--calls 4]
    python -m gated_delta_rule_57_gb300.profile_cases spec    [--calls 4]
    python -m gated_delta_rule_57_gb300.profile_cases long    [--T 65536] [--nseg 5|decay] [--calls 4]
    python -m gated_delta_rule_57_gb300.profile_cases t4k     [--nseg 4|decay|1] [--calls 4]

Draws the seeded synthetic inputs on the GPU, then makes `calls` back-to-back
calls of kda_chunk_fwd (prefill: B x 8192 tokens x 32 heads, d = 128, bf16)
or kda_decode_step (256 sequences x 32 heads, d = 128), or rounds of
kda_decode_multi (the same 256 x 32 states, 4 draft tokens: verify then
commit), or kda_chunk_fwd_segmented (long: one sequence of T tokens x 32 heads
split into nseg segments; three launches per call; --nseg decay plans the
split on the device from the decay probe: five launches; t4k: the same on
one sequence of 4096 tokens x 32 heads, half of them with g = -4.99). Under a profiler,
skip the first calls as warm-up (e.g. ncu -s 2 -c 1 -k regex:kda_).
"""
import argparse

import torch

from . import inputs, kda


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("which", choices=["prefill", "decode", "spec", "long", "t4k"])
    ap.add_argument("--B", type=int, default=8)
    ap.add_argument("--T", type=int, default=65536)
    ap.add_argument("--nseg", default="5", help="segment count, or 'decay'")
    ap.add_argument("--calls", type=int, default=4)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    if args.which == "prefill":
        w = inputs.PREFILL_B8_T8K
        x = inputs.prefill_inputs(w, dev, B=args.B)
        o = torch.empty_like(x["v"])
        hT = torch.empty(args.B, w.H, w.dk, w.dv, device=dev)
        for _ in range(args.calls):
            kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o=o, hT=hT)
    elif args.which == "decode":
        w = inputs.DECODE_N256
        x = inputs.decode_inputs(w, dev, steps=args.calls)
        for s in range(args.calls):
            kda.kda_decode_step(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], x["S"])
    elif args.which in ("long", "t4k"):
        # t4k: B=1, T=4096, H=32 with the stress heads (g = -4.99); --T is ignored
        w = inputs.PREFILL_T1M if args.which == "long" else inputs.PREFILL_T4K
        if args.which == "t4k":
            args.T = w.T
        x = inputs.prefill_inputs(w, dev, T=args.T)
        o = torch.empty_like(x["v"])
        hT = torch.empty(w.B, w.H, w.dk, w.dv, device=dev)
        nseg = 0 if args.nseg == "decay" else int(args.nseg)  # 0: planned on the device
        ws = torch.empty(kda.kda_chunk_fwd_segmented_workspace_size(
            w.B, args.T, w.H, w.dk, w.dv, nseg=nseg), dtype=torch.uint8, device=dev)
        for _ in range(args.calls):
            kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                        nseg=nseg, o=o, hT=hT, workspace=ws)
    else:
        w = inputs.DECODE_N256
        x = inputs.prefill_inputs(inputs.PrefillWorkload("draft", w.N, 4, w.H, w.dk, w.dv, w.io,
                                                         w.seed, h0_std=w.S_std), dev)
        for _ in range(args.calls):
            kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
            kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], commit=True,
                                 want_o=False)
    torch.cuda.synchronize()
    print(f"{args.which}: {args.calls} calls done")


if __name__ == "__main__":
    main()
