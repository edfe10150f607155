"""The README's Python usage example runs as printed and does what its comments say."""
import os
import re

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example_runs():
    import torch

    import qkv_rope_kv_gb300 as Q

    Q.qkv_check_device_error()  # start from a clear device status word
    blocks = re.findall(r"```python\n(.*?)```", open(README).read(), re.S)
    assert len(blocks) == 1
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()
    kk = env["kv_k"].cpu().numpy().view(np.uint16)
    vv = env["kv_v"].cpu().numpy().view(np.uint16)
    written = {17, 18}
    for r in range(kk.shape[0]):
        assert (kk[r].any() and vv[r].any()) == (r in written), r
    # the replay at position 18 left v = biased projection, the same as the step at 17
    v = env["v"].cpu().numpy()
    assert np.array_equal(vv[17], vv[18])
    assert np.array_equal(vv[18], v.astype(np.float16).view(np.uint16))


def test_readme_prefill_matches_decode_steps():
    """The README's prefill writes cache rows 100..107 of its own cache only, and each token's
    q | k | v is the decode step's result for that token (the same bf16 values as f32) within
    the prefill gate."""
    import torch

    import qkv_rope_kv_gb300 as Q
    from gpu_helpers import PREFILL_RMS_FLOOR, assert_f32_close

    Q.qkv_check_device_error()
    blocks = re.findall(r"```python\n(.*?)```", open(README).read(), re.S)
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()
    pk = env["pk"].cpu().numpy().view(np.uint16)
    rows = {int(p) for p in env["positions"].cpu().numpy()}
    assert rows == set(range(100, 108))
    for r in range(pk.shape[0]):
        assert bool(pk[r].any()) == (r in rows), r
    plan, w, bias, nqt, nkt = env["plan"], env["w"], env["bias"], env["nqt"], env["nkt"]
    R = nqt + 2 * nkt
    for t in (0, 5):
        x = env["X"][t].float().contiguous()
        out = torch.empty(R, device="cuda")
        dk, dv = torch.zeros_like(env["kv_k"]), torch.zeros_like(env["kv_v"])
        pos = env["positions"][t:t + 1].contiguous()
        Q.qkv_decode_step(plan, x, w, bias, pos, out[:nqt], out[nqt:nqt + nkt], out[nqt + nkt:], dk, dv)
        torch.cuda.synchronize()
        assert_f32_close(env["Y"][t].cpu().numpy(), out.cpu().numpy().astype(np.float64),
                         "README prefill token %d" % t, floor=PREFILL_RMS_FLOOR)
