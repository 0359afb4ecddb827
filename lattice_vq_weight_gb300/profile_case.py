"""Small, fixed launch sequences of the liblq kernels for profiler captures.

    python -m lattice_vq_weight_gb300.profile_case quantize   # the 7 Llama-3-8B layer matrices
    python -m lattice_vq_weight_gb300.profile_case quantize --grouped   # the same in one grouped call
    python -m lattice_vq_weight_gb300.profile_case gemv --batch 1
    python -m lattice_vq_weight_gb300.profile_case gemv --batch 1 --gate-up   # one grouped call
    python -m lattice_vq_weight_gb300.profile_case gemm --M 256
    python -m lattice_vq_weight_gb300.profile_case kv --tokens 32768
    python -m lattice_vq_weight_gb300.profile_case rice --batch 1   # GEMV from the gate matrix's Rice stream

Each op runs `--reps` passes (default 2) after building inputs on the device;
the second pass is the one to capture (`ncu -s <launches of one pass>`).
Inputs: bf16 N(0, 0.02^2) weights of the Llama-3-8B layer shapes (gate-shaped
only with --gate-only), E8, tile 256, beta 0.25; activations N(0, 1) bf16;
GEMM on the 8192 x 28672 Llama-3-70B up-like shape with X of M rows.  With
--grouped the quantize is one lq_quantize_grouped call over the matrices.  With
--gate-up the GEMV is one grouped call over the gate and up matrices (as in
the benchmark's layer step).  kv: one layer of a Llama-3-8B KV cache (8 kv
heads, 32 query heads, head_dim 128, N(0, 1) K and V, E8, beta 0.25) and the
decode attention over --tokens cached tokens.  rice: the GEMV from the
Rice stream of a gate-shaped E8 matrix (14336 x 4096, tile 256).
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=("quantize", "gemv", "gemm", "kv", "rice"))
    ap.add_argument("--tokens", type=int, default=32768)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--M", type=int, default=256)
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--gate-only", action="store_true")
    ap.add_argument("--gate-up", action="store_true")
    ap.add_argument("--grouped", action="store_true")
    args = ap.parse_args(argv)

    import torch
    import lattice_vq_weight_gb300 as L
    from synthetic import LLAMA3_8B_LAYER

    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(0)
    if args.op == "kv":
        from synthetic import torch_gaussian_matrix
        K = torch_gaussian_matrix(args.tokens, 8 * 128, 1.0, 7000, device=dev)
        V = torch_gaussian_matrix(args.tokens, 8 * 128, 1.0, 7001, device=dev)
        kc, ks, kd = L.quantize(K, "e8", 128, 7100, 0.25)
        vc, vs, vd = L.quantize(V, "e8", 128, 7101, 0.25)
        q = torch.randn((32, 128), device=dev, generator=gen).to(torch.bfloat16)
        out = torch.empty((32, 128), dtype=torch.float32, device=dev)
        ws = torch.empty(L.lq_attention_workspace_size(args.tokens, 8, 32, 128), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            L.lq_attention_decode("e8", kc, ks, kd, vc, vs, vd, q, out, ws)
        torch.cuda.synchronize()
        print("ok")
        return
    if args.op == "rice":
        W = (torch.randn((14336, 4096), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        codes, scales, signs = L.quantize(W, "e8", 256, 1, 0.25)
        nb = L.lq_rice_stream_bound("e8", 14336, 4096, 256)
        words = torch.empty(nb // 4, dtype=torch.int32, device=dev)
        offs = torch.empty((14336, 16), dtype=torch.int32, device=dev)
        tot = torch.empty(1, dtype=torch.int64, device=dev)
        rws = torch.empty(L.lq_rice_workspace_size(14336, 4096, 256), dtype=torch.uint8, device=dev)
        L.lq_rice_encode("e8", codes, 256, words, offs, tot, rws)
        x = torch.randn((args.batch, 4096), device=dev, generator=gen).to(torch.bfloat16)
        y = torch.empty((args.batch, 14336), dtype=torch.float32, device=dev)
        ws = torch.empty(L.lq_gemv_workspace_size(args.batch, 4096, 256), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            L.lq_gemv_rice("e8", words, offs, scales, signs, 256, x, y, ws)
        torch.cuda.synchronize()
        print("ok")
        return
    if args.op == "gemm":
        N, K = 8192, 28672
        W = (torch.randn((N, K), device=dev, generator=gen) * 0.015).to(torch.bfloat16)
        codes, scales, signs = L.quantize(W, "e8", 256, 4000, 0.25)
        del W
        X = torch.randn((args.M, K), device=dev, generator=gen).to(torch.bfloat16)
        Y = torch.empty((args.M, N), dtype=torch.float32, device=dev)
        ws = torch.empty(L.lq_gemm_workspace_size(args.M, N, K), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            L.lq_gemm("e8", codes, scales, signs, 256, X, Y, ws)
        torch.cuda.synchronize()
        print("ok")
        return
    keep = ("gate",) if args.gate_only else ("gate", "up") if args.gate_up else None
    shapes = [s for s in LLAMA3_8B_LAYER if keep is None or s[0] in keep]
    mats = []
    for _, r, c in shapes:
        W = (torch.randn((r, c), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        codes = torch.empty((r, c), dtype=torch.int8, device=dev)
        scales = torch.empty((r, c // 256), dtype=torch.float32, device=dev)
        signs = torch.empty((c,), dtype=torch.int8, device=dev)
        L.lq_quantize("e8", W, 256, 1, 0.25, codes, scales, signs)
        x = torch.randn((args.batch, c), device=dev, generator=gen).to(torch.bfloat16)
        y = torch.empty((args.batch, r), dtype=torch.float32, device=dev)
        mats.append((W, codes, scales, signs, x, y))
    ws = torch.empty(max(L.lq_gemv_workspace_size(args.batch, c, 256) for _, _, c in shapes),
                     dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    if args.gate_up:
        ws = torch.empty(L.lq_gemv_grouped_workspace_size(2, args.batch, 4096, 256), dtype=torch.uint8,
                         device=dev)
    for _ in range(args.reps):
        if args.op == "quantize" and args.grouped:
            L.lq_quantize_grouped("e8", [m[0] for m in mats], 256, [1] * len(mats), 0.25, [m[1] for m in mats],
                                  [m[2] for m in mats], [m[3] for m in mats])
            continue
        if args.op == "gemv" and args.gate_up:
            L.lq_gemv_grouped("e8", [m[1] for m in mats], [m[2] for m in mats], [m[3] for m in mats], 256,
                              mats[0][4], [m[5] for m in mats], ws)
            continue
        for W, codes, scales, signs, x, y in mats:
            if args.op == "quantize":
                L.lq_quantize("e8", W, 256, 1, 0.25, codes, scales, signs)
            else:
                L.lq_gemv("e8", codes, scales, signs, 256, x, y, ws)
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
