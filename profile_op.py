"""Runs one operation of the library a few times on seeded synthetic inputs,
so that a profiler can capture it in isolation, e.g.

    ncu --set full --clock-control none -k regex:w4a16_skinny -s 2 -c 1 -o prof \\
        python profile_op.py w4a16 --T 4 --N 11008 --K 4096

Operations (sizes as flags):
  w4a16        qlin_w4a16_gemm, X [T][K] fp16, weights N x K (uint4 g128)
  w4a16_group  qlin_w4a16_gemm_grouped over --groups matrices of N x K each
  w4a16_decode qlin_w4a16_decode_run of a plan over --blocks decoder blocks (hidden K, intermediate N:
               q,k,v grouped; o; gate,up grouped; down), X [T][K] fp16; one launch per rep
  int8_quant   qlin_quant_act_int8, X [T][K] fp16, symmetric
  w8a8         qlin_w8a8_gemm, A [T][K] int8, B [N][K] int8, per-token / per-channel scales, bf16 out
  w8a8_f16b    qlin_w8a8_gemm_f16b, the same with B as exact fp16 codes
  w8a8_f16     qlin_w8a8_gemm_f16, the same with A and B as exact fp16 codes
  int8_quant_f16  qlin_quant_act_int8_f16, X [T][K] fp16, symmetric, codes written as fp16
  nvfp4_quant  qlin_quant_nvfp4, X [T][K] fp16 with S residual channels, MMA scale layout
  nvfp4_gemm   qlin_nvfp4_gemm, A [T][K] and B [N][K] NVFP4 (made by the quantizer), bf16 out
  mxfp8_quant / mxfp4_quant  qlin_quant_mx, X [T][K] fp16, MMA scale layout
  mxfp8_gemm / mxfp4_gemm    qlin_mx_gemm, A [T][K] and B [N][K] (made by the quantizer), bf16 out
  hadamard       qlin_hadamard, X [T][K] fp16, groups of --n (--kind 0 Sylvester, 1 regular), random signs
  w4a16_act_order  qlin_w4a16_gemm_act_order, X [T][K] fp16, act-order weights N x K (gather + GEMM)
  rmsnorm_nvfp4  qlin_rmsnorm_quant_nvfp4, X [T][K] fp16, gamma [K], S residual channels, MMA scale layout
  rmsnorm_int8   qlin_rmsnorm_quant, X [T][K] fp16, gamma [K], per-token int8
  fp8_quant    qlin_quant_fp8, X [T][K] fp16, per-row E4M3
  fp8_gemm     qlin_fp8_gemm, A [T][K] and B [N][K] E4M3 (made by the quantizer), bias, bf16 out

Every launch reads its own copy of the weights (--copies of them, rotated), so
that weight streams come from HBM as they do in a model; the launches run
back to back on one stream, then the device error word is checked.
"""

import argparse
import sys


def _setup(args, q, torch):
    g = torch.Generator(device="cuda")
    g.manual_seed(args.seed)
    T, N, K = args.T, args.N, args.K
    copies = max(1, args.copies)

    def randn(shape, dtype):
        return torch.randn(shape, device="cuda", generator=g).to(dtype)

    if args.op in ("w4a16", "w4a16_group"):
        nm = 1 if args.op == "w4a16" else args.groups
        mats = []
        for _ in range(copies):
            blk = []
            for _m in range(nm):
                wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
                sc = (torch.rand((N, K // 128), device="cuda", generator=g) * 0.015 + 0.005).half()
                zp = torch.randint(0, 256, (N, (K // 128 + 1) // 2), dtype=torch.uint8, device="cuda", generator=g)
                blk.append((wq, sc, zp))
            mats.append(blk)
        x = randn((T, K), torch.float16)
        ys = [torch.empty((T, N), dtype=torch.float16, device="cuda") for _ in range(nm)]

        def run(i):
            blk = mats[i % copies]
            if args.op == "w4a16":
                q.qlin_w4a16_gemm(x, *blk[0], ys[0])
            else:
                q.qlin_w4a16_gemm_grouped(x, [b[0] for b in blk], [b[1] for b in blk], [b[2] for b in blk], ys)
        return run

    if args.op == "w4a16_decode":
        def mat(n, k):
            wq = torch.randint(0, 256, (n, k // 2), dtype=torch.uint8, device="cuda", generator=g)
            sc = (torch.rand((n, k // 128), device="cuda", generator=g) * 0.015 + 0.005).half()
            zp = torch.randint(0, 256, (n, (k // 128 + 1) // 2), dtype=torch.uint8, device="cuda", generator=g)
            return wq, sc, zp
        act = lambda n: torch.zeros((T, n), dtype=torch.float16, device="cuda")  # noqa: E731
        x = randn((T, K), torch.float16)
        qkv, o, gate, up, down = [act(K) for _ in range(3)], act(K), act(N), act(N), act(K)
        steps = []
        for _ in range(args.blocks):
            m = {nm: mat(*shape) for nm, shape in (("q", (K, K)), ("k", (K, K)), ("v", (K, K)), ("o", (K, K)),
                                                   ("gate", (N, K)), ("up", (N, K)), ("down", (K, N)))}
            for names, xin, ys in ((("q", "k", "v"), x, qkv), (("o",), qkv[2], [o]), (("gate", "up"), o, [gate, up]),
                                   (("down",), up, [down])):
                steps.append((xin, [m[n][0] for n in names], [m[n][1] for n in names], [m[n][2] for n in names], ys))
        ws = torch.zeros(q.qlin_w4a16_decode_workspace_bytes(len(steps)), dtype=torch.uint8, device="cuda")
        plan = q.qlin_w4a16_decode_prepare(steps, ws)
        return lambda i: q.qlin_w4a16_decode_run(ws, *plan)

    if args.op == "int8_quant":
        xs = [randn((T, K), torch.float16) for _ in range(copies)]
        qa = torch.empty((T, K), dtype=torch.int8, device="cuda")
        sa = torch.empty(T, dtype=torch.float32, device="cuda")
        return lambda i: q.qlin_quant_act_int8(xs[i % copies], qa, sa)

    if args.op == "int8_quant_f16":
        xs = [randn((T, K), torch.float16) for _ in range(copies)]
        qa = torch.empty((T, K), dtype=torch.float16, device="cuda")
        sa = torch.empty(T, dtype=torch.float32, device="cuda")
        return lambda i: q.qlin_quant_act_int8_f16(xs[i % copies], qa, sa)

    if args.op in ("w8a8", "w8a8_f16b", "w8a8_f16"):
        a = torch.randint(-127, 128, (T, K), dtype=torch.int8, device="cuda", generator=g)
        sa = torch.rand(T, device="cuda", generator=g) * 0.01 + 0.001
        bs = [torch.randint(-127, 128, (N, K), dtype=torch.int8, device="cuda", generator=g) for _ in range(copies)]
        sb = torch.rand(N, device="cuda", generator=g) * 0.01 + 0.001
        out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        if args.op == "w8a8":
            return lambda i: q.qlin_w8a8_gemm(a, bs[i % copies], sa, sb, out)
        b16s = [torch.empty((N, K), dtype=torch.float16, device="cuda") for _ in range(copies)]
        for b, b16 in zip(bs, b16s):
            q.qlin_int8_to_f16(b, b16)
        if args.op == "w8a8_f16b":
            return lambda i: q.qlin_w8a8_gemm_f16b(a, b16s[i % copies], sa, sb, out)
        a16 = torch.empty((T, K), dtype=torch.float16, device="cuda")
        q.qlin_int8_to_f16(a, a16)
        return lambda i: q.qlin_w8a8_gemm_f16(a16, b16s[i % copies], sa, sb, out)

    if args.op in ("nvfp4_quant", "nvfp4_gemm"):
        S = args.S
        Kin = K if args.op == "nvfp4_quant" else K - S
        gx = torch.empty(1, dtype=torch.float32, device="cuda")
        perm = torch.randperm(Kin, generator=torch.Generator().manual_seed(args.seed)).to(torch.int32).cuda()

        def quantize(rows, x):
            qc = torch.empty((rows, (Kin + S) // 2), dtype=torch.uint8, device="cuda")
            sf = torch.empty(q.qlin_nvfp4_sf_bytes(rows, Kin + S, q.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
            gg = torch.empty(1, dtype=torch.float32, device="cuda")
            q.qlin_nvfp4_global_scale(x, gg)
            q.qlin_quant_nvfp4(x, gg, qc, sf, perm=perm, S=S, sf_layout=q.QLIN_SF_MMA)
            return qc, sf, gg

        if args.op == "nvfp4_quant":
            xs = [randn((T, Kin), torch.float16) for _ in range(copies)]
            q.qlin_nvfp4_global_scale(xs[0], gx)
            qc = torch.empty((T, (Kin + S) // 2), dtype=torch.uint8, device="cuda")
            sf = torch.empty(q.qlin_nvfp4_sf_bytes(T, Kin + S, q.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
            return lambda i: q.qlin_quant_nvfp4(xs[i % copies], gx, qc, sf, perm=perm, S=S,
                                                sf_layout=q.QLIN_SF_MMA)
        qa, sfa, ga = quantize(T, randn((T, Kin), torch.float16))
        ws = [quantize(N, randn((N, Kin), torch.float16) * 0.02) for _ in range(copies)]
        out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        return lambda i: q.qlin_nvfp4_gemm(qa, sfa, ws[i % copies][0], ws[i % copies][1], ga, ws[i % copies][2], out)

    if args.op in ("mxfp8_quant", "mxfp4_quant", "mxfp8_gemm", "mxfp4_gemm"):
        fmt = q.QLIN_MX_FP8_E4M3 if args.op.startswith("mxfp8") else q.QLIN_MX_FP4_E2M1
        cb = 1 if fmt == q.QLIN_MX_FP8_E4M3 else 2

        def mxq(rows, x):
            qc = torch.empty((rows, K // cb), dtype=torch.uint8, device="cuda")
            sf = torch.zeros(q.qlin_mx_sf_bytes(rows, K, q.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
            q.qlin_quant_mx(x, qc, sf, fmt=fmt, sf_layout=q.QLIN_SF_MMA)
            return qc, sf

        if args.op.endswith("quant"):
            xs = [randn((T, K), torch.float16) for _ in range(copies)]
            qc, sf = mxq(T, xs[0])
            return lambda i: q.qlin_quant_mx(xs[i % copies], qc, sf, fmt=fmt, sf_layout=q.QLIN_SF_MMA)
        qa, sfa = mxq(T, randn((T, K), torch.float16))
        ws = [mxq(N, randn((N, K), torch.float16) * 0.02) for _ in range(copies)]
        out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        return lambda i: q.qlin_mx_gemm(qa, sfa, ws[i % copies][0], ws[i % copies][1], out, fmt=fmt)

    if args.op == "hadamard":
        xs = [randn((T, K), torch.float16) for _ in range(copies)]
        ys = torch.empty_like(xs[0])
        signs = (torch.randint(0, 2, (K,), device="cuda", generator=g) * 2 - 1).to(torch.int8)
        return lambda i: q.qlin_hadamard(xs[i % copies], args.n, y=ys, kind=args.kind, signs=signs)

    if args.op == "w4a16_act_order":
        G = K // 128
        g_idx = torch.randperm(K, device="cuda", generator=g).to(torch.int32) // 128   # each group 128 columns
        x = randn((T, K), torch.float16)
        mats = []
        for _ in range(copies):
            wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
            perm = torch.empty(K, dtype=torch.int32, device="cuda")
            wq_sorted = torch.empty_like(wq)
            q.qlin_w4a16_act_order_prepare(g_idx, wq, perm, wq_sorted)
            sc = (torch.rand((N, G), device="cuda", generator=g) * 0.015 + 0.005).half()
            zp = torch.randint(0, 256, (N, (G + 1) // 2), dtype=torch.uint8, device="cuda", generator=g)
            mats.append((perm, wq_sorted, sc, zp))
        x_work = torch.empty_like(x)
        y = torch.empty((T, N), dtype=torch.float16, device="cuda")
        return lambda i: q.qlin_w4a16_gemm_act_order(x, *mats[i % copies], y, x_work=x_work)

    if args.op in ("rmsnorm_nvfp4", "rmsnorm_int8"):
        xs = [randn((T, K), torch.float16) for _ in range(copies)]
        gam = (torch.rand(K, device="cuda", generator=g) + 0.5).half()
        if args.op == "rmsnorm_int8":
            qc = torch.empty((T, K), dtype=torch.int8, device="cuda")
            sc = torch.empty(T, dtype=torch.float32, device="cuda")
            return lambda i: q.qlin_rmsnorm_quant(xs[i % copies], gam, 1e-6, qc, sc)
        S = args.S
        perm = torch.randperm(K, generator=torch.Generator().manual_seed(args.seed)).to(torch.int32).cuda()
        gx = torch.full((1,), 6.0 / 2688.0, dtype=torch.float32, device="cuda")
        qc = torch.empty((T, (K + S) // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty(q.qlin_nvfp4_sf_bytes(T, K + S, q.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
        return lambda i: q.qlin_rmsnorm_quant_nvfp4(xs[i % copies], gam, 1e-6, gx, qc, sf, perm=perm, S=S,
                                                    sf_layout=q.QLIN_SF_MMA)

    if args.op == "fp8_quant":
        xs = [randn((T, K), torch.float16) for _ in range(copies)]
        qc = torch.empty((T, K), dtype=torch.uint8, device="cuda")
        sc = torch.empty(T, dtype=torch.float32, device="cuda")
        return lambda i: q.qlin_quant_fp8(xs[i % copies], qc, sc)

    if args.op == "fp8_gemm":
        def quantize(rows, x):
            qc = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
            sc = torch.empty(rows, dtype=torch.float32, device="cuda")
            q.qlin_quant_fp8(x, qc, sc)
            return qc, sc

        qa, sa = quantize(T, randn((T, K), torch.float16))
        ws = [quantize(N, randn((N, K), torch.float16) * 0.02) for _ in range(copies)]
        bias = randn((N,), torch.float16)
        out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        return lambda i: q.qlin_fp8_gemm(qa, ws[i % copies][0], sa, ws[i % copies][1], out, bias=bias)

    raise ValueError(args.op)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("op", choices=["w4a16", "w4a16_group", "w4a16_decode", "int8_quant", "w8a8", "w8a8_f16b", "w8a8_f16", "int8_quant_f16",
                                   "nvfp4_quant", "nvfp4_gemm",
                                   "fp8_quant", "fp8_gemm", "rmsnorm_nvfp4", "rmsnorm_int8", "mxfp8_quant",
                                   "mxfp4_quant", "mxfp8_gemm", "mxfp4_gemm", "hadamard", "w4a16_act_order"])
    ap.add_argument("--n", type=int, default=256, help="Hadamard group size")
    ap.add_argument("--kind", type=int, default=0, help="Hadamard kind: 0 Sylvester, 1 regular")
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--S", type=int, default=128, help="NVFP4 residual channels (K includes them for nvfp4_gemm)")
    ap.add_argument("--groups", type=int, default=3, help="matrices per w4a16_group launch")
    ap.add_argument("--blocks", type=int, default=2, help="decoder blocks of a w4a16_decode plan")
    ap.add_argument("--copies", type=int, default=4, help="weight copies rotated over the launches")
    ap.add_argument("--reps", type=int, default=4, help="launches")
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)

    import torch
    import quantized_linear_layer_gb300 as q
    q.build()
    run = _setup(args, q, torch)
    for i in range(args.reps):
        run(i)
    torch.cuda.synchronize()
    err = q.qlin_get_device_error()
    if err != 0:
        print("device error word %#x" % err, file=sys.stderr)
        return 1
    print("%s: %d launches ok" % (args.op, args.reps))
    return 0


if __name__ == "__main__":
    sys.exit(main())
