"""Failure detection without a GPU fault: a pipeline wait of the GEMM or forward kernel runs out.

Every wait inside the kernels is bounded (BSQ_WAIT_LIMIT_MS / _US); on expiry the kernel
lets its copies in flight land, stops every role of both CTAs of the pair, frees its
tensor memory, returns, and records BSQ_DEVERR_TIMEOUT in the device error word.  Here
the test hook BSQ_TEST_DROP_ANNOUNCE=1 withholds the even CTA's operand-ready
announcements (a flag nothing sets), so the MMA thread's first wait runs out after a
50 ms limit.  The test checks that bsq_get_device_error reports BSQ_ERR_TIMEOUT, and that
the next calls in the same process, with the hook off, are correct and leave no error.
It covers the default kernel (linear dgrad), the short-tile kernel (grouped wgrad), the
fused backward launch and the forward kernel (packed X, and BF16 X with its own X
producer), and runs in a child process so that its environment settings touch no other
test.
"""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, {root!r})
    import numpy as np
    import torch
    from block_scaled_gemm_fp8_gb300 import bsq, synth
    from oracle import gemm as Gm
    from tests._util import assert_gemm, bf16_vals, oracle_deq

    W = synth.make_packed(synth.FMT_MXFP4, 1, 256, 512, 0.5, seed=1, device="cpu")
    X = synth.make_packed(synth.FMT_MXFP4, 1, 300, 512, 1.0, seed=2, device="cpu")
    G = synth.randn((300, 256), 1.0, 3, "cpu", torch.bfloat16)
    wd, xd, gd = W.to("cuda"), X.to("cuda"), G.cuda()
    offs = synth.offsets_from_counts([100, 0, 200])
    od = torch.from_numpy(offs).cuda()
    XB = synth.make_packed(synth.FMT_BF16, 1, 300, 512, 1.0, seed=4, device="cpu")
    xbd = XB.to("cuda")
    calls = {{
        "linear_dgrad": lambda: bsq.linear_dgrad(gd, wd),
        "grouped_wgrad": lambda: bsq.grouped_wgrad(gd, xd, od, 3),
        "linear_backward": lambda: bsq.linear_backward(gd, wd, xd),
        "linear_forward": lambda: bsq.linear_forward(xd, wd),
        "linear_forward_bf16_x": lambda: bsq.linear_forward(xbd, wd),
    }}
    g, w, x = bf16_vals(G), oracle_deq(W)[0], oracle_deq(X)[0]
    for name, call in calls.items():
        os.environ["BSQ_WAIT_LIMIT_MS"] = "50"
        os.environ["BSQ_TEST_DROP_ANNOUNCE"] = "1"
        call()
        st, code = bsq.get_device_error()
        assert st == bsq.BSQ_ERR_TIMEOUT and code == 1, (name, st, code)
        del os.environ["BSQ_WAIT_LIMIT_MS"], os.environ["BSQ_TEST_DROP_ANNOUNCE"]
        out = call()
        torch.cuda.synchronize()
        if name == "linear_dgrad":
            assert_gemm(bf16_vals(out), Gm.dgrad(g, w), g, w, 256, name)
        elif name == "grouped_wgrad":
            ref = Gm.grouped_wgrad(g, x, offs, 3)
            got = bf16_vals(out)
            for e in range(3):
                r0, r1 = Gm.expert_rows(offs, e)
                if r1 > r0:
                    assert_gemm(got[e], ref[e], g[r0:r1], x[r0:r1], r1 - r0, f"{{name}} e={{e}}")
                else:
                    assert (got[e] == 0).all()
        elif name == "linear_forward":
            assert_gemm(bf16_vals(out), Gm.forward(x, w), x, w, 512, name)
        elif name == "linear_forward_bf16_x":
            xb = oracle_deq(XB)[0]
            assert_gemm(bf16_vals(out), Gm.forward(xb, w), xb, w, 512, name)
        else:
            gx, gw = out
            assert_gemm(bf16_vals(gx), Gm.dgrad(g, w), g, w, 256, name + " dgrad")
            assert_gemm(bf16_vals(gw), Gm.wgrad(g, x), g, x, 300, name + " wgrad")
        st, code = bsq.get_device_error()
        assert st == bsq.BSQ_OK and code == 0, (name, "after recovery", st, code)
        print("ok", name)
""")


def test_wait_runs_out_then_next_call_is_correct():
    env = {k: v for k, v in os.environ.items() if not k.startswith("BSQ_")}
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 5, r.stdout
