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
