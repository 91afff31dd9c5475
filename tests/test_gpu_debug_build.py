"""The debug build (python -m kda_linear_attention_gb300.build --debug,
selected with KDA_GB300_DEBUG=1): the same kernels with index checks on
their global-memory addressing, standing in for a memory checker.  On valid
inputs no check may fire and the results must keep parity with the oracle;
run in a child process so that the debug library is the one loaded."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import numpy as np, torch
import kda_inputs as ki, oracle
from oracle import layer as olayer
import kda_linear_attention_gb300 as kda
from kda_testlib import TOL_BF16, TOL_F32, assert_close, dev_tensor, prefill_on_gpu, decode_on_gpu
assert kda.library_path().endswith("libkda_gb300_debug.so"), kda.library_path()
kda.device_error(reset=True)
for dtype, chunk in (("bf16", 64), ("bf16", 32), ("f32", 16)):
    inp = ki.gen_prefill(901, [0, 1, 17, 64, 65, 200], H=3, dtype=dtype, chunk=chunk, with_s0=True)
    o, S = prefill_on_gpu(inp)               # asserts a clear error word
    o_ref, S_ref = oracle.prefill(inp)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_close(o, o_ref, tol, "debug prefill o %s/%d" % (dtype, chunk))
    assert_close(S, S_ref, tol, "debug prefill S %s/%d" % (dtype, chunk))
rng = np.random.Generator(np.random.PCG64(902))
S0 = ki.gen_decode_state(rng, 5, 4)
step = ki.gen_decode_step(rng, 5, 4, "bf16")
Sd = dev_tensor(S0)
od = decode_on_gpu(Sd, step)
o_ref, S_ref = oracle.decode(S0, step)
assert_close(od, o_ref, TOL_BF16, "debug decode o")
idx = np.array([3, -1, 0, 4, 1], dtype=np.int32)
d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
pool = dev_tensor(ki.gen_decode_state(rng, 6, 4))
kda.decode_step_pool(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, state_indices=dev_tensor(idx))
L = ki.gen_layer(903, [0, 3, 64, 130], H=2, with_conv0=True)
q, k, v, co = kda.conv_prologue(dev_tensor(L.xq), dev_tensor(L.xk), dev_tensor(L.xv), dev_tensor(L.conv_w),
                                dev_tensor(L.cu_seqlens), conv_in=dev_tensor(L.conv0).view(torch.bfloat16))
torch.cuda.synchronize()
err = kda.device_error(reset=True)
assert err == 0, "a debug index check fired on valid inputs: 0x%x" % err
print("debug build clean")
'''


def test_debug_build_is_clean_on_valid_inputs():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_linear_attention_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, KDA_GB300_DEBUG="1",
               PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build clean" in r.stdout
