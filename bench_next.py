"""Times the ranked follow-on operations (FP8 and MX GEMMs, the RMSNorm-fused
quantizers, the W4A16 prefill GEMM and act-order, the Hadamard rotation) on
seeded synthetic inputs and prints one JSON line per operation with its rate
against the roofline that bounds it:

    python bench_next.py [--only NAME ...]

Each operation is captured in a CUDA graph of 10 launches over rotating
inputs (weights rotate over three copies, so weight streams come from HBM),
replayed after three warm-up replays; the median of five timed replays with
CUDA events on the capturing stream is reported.  Peaks come from
MEASURED_PEAKS.json at the repository root (HBM GB/s and dense bf16 TFLOP/s;
fp8 at 2x and fp4 at 6x the bf16 rate, the nominal ratios).  These are not
the hot-path step of bench.py.
"""

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def _time(torch, fn, reps=10):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for _ in range(reps):
                fn()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(5):
            e0.record(s)
            graph.replay()
            e1.record(s)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
    return sorted(ts)[2] * 1e-3


def _rows(q, torch):
    """(name, workload, setup) where setup() returns (callable, units, bound)."""
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def randn(*shape, scale=1.0):
        return (torch.randn(shape, device=dev, generator=g) * scale).half()

    rows = []

    def fp8():
        T, N, K = 2048, 4096, 4096
        xs = [randn(T, K) for _ in range(2)]
        qa, sa = torch.empty((T, K), dtype=torch.uint8, device=dev), torch.empty(T, device=dev)
        ws = []
        for _ in range(3):
            qb, sb = torch.empty((N, K), dtype=torch.uint8, device=dev), torch.empty(N, device=dev)
            q.qlin_quant_fp8(randn(N, K, scale=0.02), qb, sb)
            ws.append((qb, sb))
        bias, out = randn(N), torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        it = [0]

        def run():
            it[0] += 1
            q.qlin_quant_fp8(xs[it[0] % 2], qa, sa)
            q.qlin_fp8_gemm(qa, ws[it[0] % 3][0], sa, ws[it[0] % 3][1], out, bias=bias)
        return run, 2.0 * T * N * K, "fp8"
    rows.append(("fp8_w8a8", "per-token E4M3 quantize + E4M3 GEMM + bias, T=2048 N=K=4096, bf16 out", fp8))

    def mx(fmt):
        def setup():
            T, N, K = 2048, 4096, 4096
            cb = 1 if fmt == q.QLIN_MX_FP8_E4M3 else 2

            def quant(x, rows_):
                c = torch.empty((rows_, K // cb), dtype=torch.uint8, device=dev)
                s = torch.zeros(q.qlin_mx_sf_bytes(rows_, K, q.QLIN_SF_MMA), dtype=torch.uint8, device=dev)
                q.qlin_quant_mx(x, c, s, fmt=fmt, sf_layout=q.QLIN_SF_MMA)
                return c, s
            xs = [randn(T, K) for _ in range(2)]
            qa, sfa = quant(xs[0], T)
            ws = [quant(randn(N, K, scale=0.02), N) for _ in range(3)]
            out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
            it = [0]

            def run():
                it[0] += 1
                q.qlin_quant_mx(xs[it[0] % 2], qa, sfa, fmt=fmt, sf_layout=q.QLIN_SF_MMA)
                q.qlin_mx_gemm(qa, sfa, ws[it[0] % 3][0], ws[it[0] % 3][1], out, fmt=fmt)
            return run, 2.0 * T * N * K, "fp8" if fmt == q.QLIN_MX_FP8_E4M3 else "fp4"
        return setup
    rows.append(("mxfp8", "MXFP8 quantize + block-scaled GEMM, T=2048 N=K=4096, bf16 out", mx(q.QLIN_MX_FP8_E4M3)))
    rows.append(("mxfp4", "MXFP4 quantize + block-scaled GEMM, T=2048 N=K=4096, bf16 out", mx(q.QLIN_MX_FP4_E2M1)))

    def rmsnorm(kind, dtype=torch.float16):
        def setup():
            T, K, S = 2048, 4096, 128
            xs = [randn(T, K).to(dtype) for _ in range(4)]
            gam = (torch.rand(K, device=dev, generator=g) + 0.5).to(dtype)
            it = [0]
            if kind == "nvfp4":
                perm = torch.randperm(K, device=dev, generator=g).to(torch.int32)
                gg = torch.full((1,), 6.0 / 2688.0, device=dev)
                qc = torch.empty((T, (K + S) // 2), dtype=torch.uint8, device=dev)
                sf = torch.empty(q.qlin_nvfp4_sf_bytes(T, K + S, q.QLIN_SF_MMA), dtype=torch.uint8, device=dev)

                def run():
                    it[0] += 1
                    q.qlin_rmsnorm_quant_nvfp4(xs[it[0] % 4], gam, 1e-6, gg, qc, sf, perm=perm, S=S,
                                               sf_layout=q.QLIN_SF_MMA)
                return run, T * K * 2 + T * (K + S) // 2 + T * (K + S) // 16, "hbm"
            fmt = q.QLIN_QFMT_INT8 if kind == "int8" else q.QLIN_QFMT_FP8_E4M3
            qc = torch.empty((T, K), dtype=torch.int8 if kind == "int8" else torch.uint8, device=dev)
            sc = torch.empty(T, device=dev)

            def run():
                it[0] += 1
                q.qlin_rmsnorm_quant(xs[it[0] % 4], gam, 1e-6, qc, sc, fmt=fmt)
            return run, T * K * 3 + T * 4, "hbm"
        return setup
    for kind in ("int8", "fp8", "nvfp4"):
        rows.append(("rmsnorm_" + kind, "RMSNorm fused with the %s quantizer, 2048 x 4096 fp16" % kind, rmsnorm(kind)))
    rows.append(("rmsnorm_int8_bf16", "RMSNorm fused with the int8 quantizer, 2048 x 4096 bf16", rmsnorm("int8", torch.bfloat16)))

    def w4(N, K, T, act_order=False):
        def setup():
            x = randn(T, K)
            G = K // 128
            mats = []
            for _ in range(3):
                wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=g)
                sc = (torch.rand((N, G), device=dev, generator=g) * 0.01 + 0.001).half()
                zp = torch.randint(0, 256, (N, (G + 1) // 2), dtype=torch.uint8, device=dev, generator=g)
                mats.append((wq, sc, zp))
            y = torch.empty((T, N), dtype=torch.float16, device=dev)
            perm = torch.randperm(K, device=dev, generator=g).to(torch.int32)
            xw = torch.empty_like(x)
            it = [0]

            def run():
                it[0] += 1
                wq, sc, zp = mats[it[0] % 3]
                if act_order:
                    q.qlin_w4a16_gemm_act_order(x, perm, wq, sc, zp, y, x_work=xw)
                else:
                    q.qlin_w4a16_gemm(x, wq, sc, zp, y)
            if T == 1:
                byts = N * K // 2 + N * G * 2 + N * ((G + 1) // 2) + 2 * K + 2 * N + (4 * K if act_order else 0)
                return run, byts, "hbm"
            return run, 2.0 * T * N * K, "bf16"
        return setup
    for T in (2048, 256, 65):
        for (N, K) in ((4096, 4096), (11008, 4096), (4096, 11008)):
            rows.append(("w4a16_prefill_t%d_%dx%d" % (T, N, K),
                         "W4A16 g128 prefill GEMM, T=%d, N=%d K=%d, fp16 out" % (T, N, K), w4(N, K, T)))
    rows.append(("w4a16_act_order_t1", "W4A16 act-order decode (gather + GEMV), T=1, N=K=4096", w4(4096, 4096, 1, True)))
    rows.append(("w4a16_act_order_t2048", "W4A16 act-order prefill (gather + GEMM), T=2048, N=K=4096",
                 w4(4096, 4096, 2048, True)))

    def had(kind, n):
        def setup():
            # 8192 x 8192 fp16 rows, three inputs in turn: 384 MB, larger than L2
            T, K = 8192, 8192
            xs = [randn(T, K) for _ in range(3)]
            y = torch.empty_like(xs[0])
            signs = (torch.randint(0, 2, (K,), device=dev, generator=g) * 2 - 1).to(torch.int8)
            it = [0]

            def run():
                it[0] += 1
                q.qlin_hadamard(xs[it[0] % 3], n, y=y, kind=kind, signs=signs)
            return run, 4 * T * K, "hbm"
        return setup
    for kind, name in ((q.QLIN_HADAMARD_SYLVESTER, "sylvester"), (q.QLIN_HADAMARD_REGULAR, "regular")):
        for n in ((256, 512, 1024, 2048, 4096) if name == "sylvester" else (64, 256)):
            rows.append(("hadamard_%s_%d" % (name, n), "online Hadamard (%s, groups of %d), 8192 x 8192 fp16" % (name, n),
                         had(kind, n)))
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--only", nargs="*", default=None, help="names of the operations to run")
    args = ap.parse_args(argv)
    import torch
    import quantized_linear_layer_gb300 as q
    q.build()
    hbm, bf16, source = _peaks()
    peak = {"hbm": (hbm, "GB/s", 1e9), "bf16": (bf16, "TFLOP/s", 1e12), "fp8": (2 * bf16, "TFLOP/s", 1e12),
            "fp4": (6 * bf16, "TFLOP/s", 1e12)}
    for name, workload, setup in _rows(q, torch):
        if args.only and name not in args.only:
            continue
        run, units, bound = setup()
        t = _time(torch, run)
        p, unit, scale = peak[bound]
        achieved = units / t / scale
        print(json.dumps({"row": name, "workload": workload, "us": round(t * 1e6, 2), "achieved": round(achieved, 1),
                          "unit": unit, "bound": "hbm" if bound == "hbm" else "tensor (%s)" % bound,
                          "peak": round(p, 1), "frac": round(achieved / p, 3), "peak_source": source}), flush=True)
        torch.cuda.empty_cache()
    err = q.qlin_get_device_error()
    if err:
        print("device error word %#x" % err, file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
