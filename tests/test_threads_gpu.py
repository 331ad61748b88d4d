"""Two host threads making their first calls into the library at the same
time, in a fresh process (so no kernel attribute has been set yet).

The launchers that need more than 48 KB of dynamic shared memory raise that
limit once per (device, kernel) under a lock.  Both threads race through
those first launches -- the warp-specialised quantize kernels (groups along T
and along C), the warp-specialised dequantize / statistics kernel, the
cluster quantize kernel and the fused selection kernel -- each on its own
stream, and every result must still equal the CPU oracle bit for bit.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    sys.path.insert(0, sys.argv[1] + "/tests")
    import oracle as O
    from gpu_util import kq_of, to_host
    from kv_cache_quantization_kvq_gb300 import build
    build()
    from kv_cache_quantization_kvq_gb300 import binding as b
    from kv_cache_quantization_kvq_gb300 import workloads as W

    rng = np.random.default_rng(0)
    xk = W.to_bf16_bits(W.random_kv(rng, (4, 301, 128)))
    xl = W.to_bf16_bits(W.random_kv(rng, (2, 1100, 128)))
    hist = W.random_history(rng, 3, 5, 5000, planted=16)
    fmts = [
        (xk, O.QParams.asym(4, 0, 15, axis=O.ALONG_T, group=64, residual=13, scale_dtype=O.BF16, zero_dtype=O.BF16)),
        (xk, O.QParams.asym(4, 0, 15, axis=O.ALONG_C, group=64, residual=13, scale_dtype=O.BF16, zero_dtype=O.BF16)),
        (xl, O.QParams.sym(8, axis=O.ALONG_T, group=0)),
    ]
    want = [(O.quantize(x, O.BF16, q), O.dequantize(O.quantize(x, O.BF16, q), x.shape, q, O.BF16),
             O.error_stats(x, O.BF16, O.quantize(x, O.BF16, q), q)) for x, q in fmts]
    want_sel = O.h2o_select(hist, 300, 32)[0]
    torch.cuda.set_device(0)
    dev_in = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x, _ in fmts]
    hd = torch.from_numpy(hist).cuda()
    torch.cuda.synchronize()

    gate = threading.Barrier(2)
    errors = []

    def worker(tid):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                gate.wait()
                outs = []
                for xd, (x, q) in zip(dev_in, fmts):
                    kq = kq_of(b, q)
                    qt = b.quantize(xd, kq, stream=s)
                    xh = b.dequantize(qt, stream=s)
                    st = b.error_stats(xd, qt, stream=s)
                    outs.append((qt, xh, st))
                keep, _ = b.h2o_select(hd, 300, 32, stream=s)
            s.synchronize()
            for (qt, xh, st), (wq, wd, ws), (x, q) in zip(outs, want, fmts):
                assert np.array_equal(to_host(qt.codes), wq.codes), f"thread {tid}: codes"
                assert np.array_equal(to_host(xh).reshape(x.shape), wd), f"thread {tid}: dequantized values"
                np.testing.assert_allclose(st.cpu().numpy(), ws, rtol=1e-5)
            assert np.array_equal(keep.cpu().numpy(), want_sel), f"thread {tid}: keep set"
        except BaseException as e:
            errors.append(f"{type(e).__name__}: {e}")

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in ts), "a thread did not finish"
    assert not errors, errors
    assert b.kvq_wait_timeouts() == 0
    print("threads: ok")
""")


def test_two_threads_race_through_first_launches():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads: ok" in r.stdout
