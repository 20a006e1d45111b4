"""Run by test_threads_gpu.py in a fresh process: the first GEMM calls of the process come
from several host threads at once, each on its own CUDA stream, so the library's one-time
per-device set-up (device probe, function attributes, co-resident cluster counts) and the
stream-K launch counter are reached concurrently.  The problems take different kernel forms
by the default choice (single CTA, narrow tiles, CTA pair, 224- and 512-column pairs, stream-K
with a workspace).  Integer-valued operands make every output unique, so each repetition's D must
equal the oracle's rounded result bit for bit.  Exits non-zero on any mismatch."""
import os
import sys
import threading

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from layout_algebra_gb300 import binding as G        # noqa: E402
from layout_algebra_gb300 import workloads as W      # noqa: E402
from oracle import gemm_ref as O                     # noqa: E402

DEV = torch.device("cuda", 0)
REPEAT = 4

# (problem, with a stream-K workspace, kernel form the default choice gives)
CASES = [
    (W.Problem("t_single", 128, 9792, 64, "f16", dist="int2", seed=701), False, 1),
    (W.Problem("t_narrow", 1024, 48, 256, "bf16", dist="int2", seed=702), False, 4),
    (W.Problem("t_pair224", 2560, 2816, 64, "f16", has_c=True, beta=1.0, dist="int2", c_dist="int2",
               seed=703), False, 5),
    (W.Problem("t_pair", 2560, 2816, 64, "bf16", majorB="MN", dist="int2", seed=704), False, 2),
    (W.Problem("t_pair512", 2560, 2048, 4096, "f16", majorB="MN", dist="int2", seed=707), False, 6),
    (W.Problem("t_sk_f16", 256, 512, 8192, "f16", dist="int2", seed=705), True, 4),
    (W.Problem("t_sk_bf16", 1280, 1536, 4096, "bf16", has_c=True, beta=1.0, dist="int2",
               c_dist="int2", seed=706), True, 1),
]


def expected(p, data):
    # the oracle reads the same logical operands stored K-major (contiguous k loop)
    pk = p.with_(majorA="K", majorB="K", lda=None, ldb=None)
    if pk != p:
        p, data = pk, W.make(pk)
    code = O.dtype_code(p.dtype)
    C = W.bits(data["C"]) if data["C"] is not None else None
    ref, _ = O.gemm(p.M, p.N, p.K, p.alpha, W.bits(data["A"]), data["lda"],
                    0 if p.majorA == "K" else 1, W.bits(data["B"]), data["ldb"],
                    0 if p.majorB == "K" else 1, p.beta, C, p.N, code)
    return O.round_to(code, ref).reshape(-1)


def main():
    for p, _, form in CASES:
        lda, ldb = W.leading_dims(p)
        got = G.plan(p.dtype, p.M, p.N, p.K, lda, p.majorA, ldb, p.majorB)["variant"]
        assert got == form, "%s: plan variant %d, expected %d" % (p.name, got, form)
    inputs = []
    for p, _, _ in CASES:
        data = W.make(p)
        dev = {k: data[k].to(DEV) if data[k] is not None else None for k in ("A", "B", "C")}
        inputs.append((data, dev))
    torch.cuda.synchronize()

    start = threading.Barrier(len(CASES))
    outs = [None] * len(CASES)
    errors = []

    def worker(i):
        try:
            p, use_ws, _ = CASES[i]
            data, dev = inputs[i]
            stream = torch.cuda.Stream(device=DEV)
            start.wait()
            with torch.cuda.stream(stream):
                ws = G.make_workspace(DEV) if use_ws else None
                Ds = [torch.empty(p.M * p.N, dtype=dev["A"].dtype, device=DEV) for _ in range(REPEAT)]
                for D in Ds:
                    G.gemm(dev["A"], dev["B"], p.M, p.N, p.K, lda=data["lda"], ldb=data["ldb"],
                           majorA=p.majorA, majorB=p.majorB, alpha=p.alpha, beta=p.beta,
                           C=dev["C"], D=D, stream=stream, workspace=ws)
            st, detail = G.last_device_status(stream)
            assert st == 0, "%s: device status %d detail %#x" % (p.name, st, detail)
            outs[i] = [W.bits(D.cpu()).reshape(-1) for D in Ds]
        except Exception as e:   # reported by the main thread
            errors.append("%s: %r" % (CASES[i][0].name, e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        print("\n".join(errors))
        return 1
    bad = 0
    for (p, _, _), (data, _), got in zip(CASES, inputs, outs):
        want = expected(p, data)
        for r, d in enumerate(got):
            if not np.array_equal(d, want):
                i = int(np.argmax(d != want))
                print("%s repetition %d: first mismatch at %d: %#06x vs %#06x" % (p.name, r, i, d[i], want[i]))
                bad += 1
    if bad:
        return 1
    print("ok: %d threads x %d calls" % (len(CASES), REPEAT))
    return 0


if __name__ == "__main__":
    sys.exit(main())
