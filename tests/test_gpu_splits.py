"""The decode kernel at every cluster shape: forced K-split counts, against the oracle.

LR_DECODE_SPLITS is read once per process, so each split count runs in a child
process.  S = 16 is a non-portable cluster size; S = 1 is the unsplit path.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import oracle, synth
import rank_decomposed_gb300 as lr
from lr_testutil import assert_parity, dev_bits, dev_factor, host_factor
d_in, d_out, r = 4096, 640, 192          # 64 k-blocks in the down projection, 3 in the up
f = dev_factor(21, 0, 1, d_in, d_out, r)
A, B = host_factor(21, 0, 1, d_in, d_out, r)
worst = 0.0
for M in (1, 37, 64, 200):
    x_bits = synth.bf16_normal(21, synth.make_tag(M, 9, synth.KIND_X), (M, d_in))
    ys = {{}}
    for ydt in (torch.float32, torch.bfloat16):
        y = torch.full((M, d_out), float("nan"), dtype=ydt, device="cuda")
        ws = torch.zeros(max(lr.linear_workspace_bytes(M, f), 256), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lr.linear_forward(dev_bits(x_bits), f, y, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ys[ydt] = y
    # parity on the fp32 output; a bf16 output is the RNE image of the fp32 one
    ref = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]
    got = ys[torch.float32].cpu().numpy().astype(np.float64)
    worst = max(worst, assert_parity(got, ref, "S={S} M=%d" % M))
    assert torch.equal(ys[torch.bfloat16], ys[torch.float32].to(torch.bfloat16)), "S={S} M=%d bf16" % M
print("ok", worst)
'''


@pytest.mark.parametrize("splits", [1, 2, 7, 11, 16])
def test_forced_split_counts(splits):
    env = dict(os.environ, LR_DECODE_SPLITS=str(splits))
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), S=splits)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
