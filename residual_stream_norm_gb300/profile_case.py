"""Launch one kernel of the boundary path a few times on a small synthetic case (for ncu).

    python -m residual_stream_norm_gb300.profile_case --kernel moe --tokens 2048 --launches 3

Kernels: boundary, moe, allreduce (TP8 partials), qk_rope, qk_ssmax, gate, qk_rope_kv and
qk_ssmax_kv (FP8 KV cache), routing.  Inputs come from the seeded generators; the case is sized by --tokens (2048 tokens keep
every kernel's inputs above the 129 MB L2 for the MoE variant and a few hundred MB on the device
at most).
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import beam_inputs as bi  # noqa: E402
import residual_stream_norm_gb300 as rsn  # noqa: E402


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", required=True,
                    choices=["boundary", "moe", "allreduce", "qk_rope", "qk_ssmax", "gate", "qk_rope_kv",
                             "qk_ssmax_kv", "routing"])
    ap.add_argument("--tokens", type=int, default=2048)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args(argv)
    rsn.lib()
    dev = torch.device("cuda:0")
    T = args.tokens
    if args.kernel == "boundary":
        c = bi.prefill_boundary_case(T=T)
        h, x = c["h"].to(dev), c["x"].to(dev)
        wpo, wpr = c["w_post"].to(dev), c["w_pre"].to(dev)
        y = torch.empty_like(h)
        run = lambda i: rsn.beam_boundary_fwd(h, y, h, x, wpo[i % 104], wpr[i % 104], i % 104 + 1)
    elif args.kernel == "moe":
        c = bi.moe_case(T=T)
        h, e, w = c["h"].to(dev), c["e"].to(dev), c["topk_w"].to(dev)
        wpo, wpr = c["w_post"].to(dev), c["w_pre"].to(dev)
        y = torch.empty_like(h)
        run = lambda i: rsn.beam_moe_combine_boundary_fwd(h, y, h, e, w, wpo, wpr, 2 * (i % 52) + 2)
    elif args.kernel == "allreduce":
        c = bi.allreduce_case(T=T, P=bi.TP_RANKS)
        h, parts = c["h"].to(dev), c["parts"].to(dev)
        wpo, wpr = c["w_post"].to(dev), c["w_pre"].to(dev)
        y = torch.empty_like(h)
        run = lambda i: rsn.beam_allreduce_boundary_fwd(h, y, h, parts, wpo, wpr, i % 104 + 1)
    elif args.kernel in ("qk_rope", "qk_ssmax"):
        c = bi.attn_qk_case(T=T, pos_mode="uniform" if args.kernel == "qk_rope" else "contiguous")
        q, k = c["q"].to(dev), c["k"].to(dev)
        wq, wk, pos = c["wq"].to(dev), c["wk"].to(dev), c["pos"].to(dev)
        fn = rsn.beam_qk_norm_rope_fwd if args.kernel == "qk_rope" else rsn.beam_qk_norm_ssmax_fwd
        run = lambda i: fn(q, k, wq, wk, pos)
    elif args.kernel in ("qk_rope_kv", "qk_ssmax_kv"):
        rope = args.kernel == "qk_rope_kv"
        c = bi.attn_qk_case(T=T, pos_mode="uniform" if rope else "contiguous")
        kv = bi.kv_cache_case(T=T, pad_frac=0.0, oob_frac=0.0)
        q, k, v = c["q"].to(dev), c["k"].to(dev), kv["v"].to(dev)
        wq, wk, pos = c["wq"].to(dev), c["wk"].to(dev), c["pos"].to(dev)
        slots = kv["slot_mapping"].to(dev)
        kc = torch.zeros((kv["num_slots"], bi.N_KV_HEADS, bi.HEAD_DIM), dtype=torch.uint8,
                         device=dev)
        vc = torch.zeros_like(kc)
        fn = rsn.beam_qk_norm_rope_kv_fwd if rope else rsn.beam_qk_norm_ssmax_kv_fwd
        run = lambda i: fn(q, k, v, wq, wk, pos, slots, kc, vc, cache_dtype=rsn.CACHE_FP8_E4M3)
    elif args.kernel == "routing":
        c = bi.routing_case(T=T)
        logits, bias = c["logits"].to(dev), c["bias"].to(dev)
        ids = torch.empty((T, bi.TOP_K), dtype=torch.int32, device=dev)
        w = torch.empty((T, bi.TOP_K), dtype=torch.float32, device=dev)
        run = lambda i: rsn.beam_grouped_topk_fwd(ids, w, logits, bias)
    else:
        c = bi.gate_case(T=T)
        attn, gate, bias = c["attn"].to(dev), c["gate"].to(dev), c["bias"].to(dev)
        out = torch.empty_like(attn)
        run = lambda i: rsn.beam_attn_gate_fwd(out, attn, gate, bias, bi.N_Q_HEADS)
    torch.cuda.synchronize()
    for i in range(args.launches):
        run(i)
    torch.cuda.synchronize()
    print(f"{args.kernel}: {args.launches} launches on {T} tokens done")


if __name__ == "__main__":
    main()
