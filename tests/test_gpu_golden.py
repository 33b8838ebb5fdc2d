"""The GPU activation quantizers against e4m3 codes worked out by hand (tests/golden/).

One 128-value group holds 448 (so its scale is amax/448 = 1 exactly and the code of each
value is the code of the value itself) and every hand-derived point that bfloat16 holds
exactly and that does not exceed 448."""

import numpy as np
import pytest
import torch

from golden_data import e4m3_points
from util import DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["g128", "tensor", "row"])
def test_quant_codes_equal_hand_derived(fge, mode):
    pts = [(v, c) for v, c, bf in e4m3_points() if bf and abs(v) <= 448.0]
    row = np.zeros(128, np.float32)
    codes = np.zeros(128, np.uint8)
    row[0], codes[0] = 448.0, 0x7E
    for i, (v, c) in enumerate(pts, start=1):
        row[i], codes[i] = v, c
    x = torch.from_numpy(row[None, :]).to(torch.bfloat16).to(DEV)
    assert np.array_equal(x.float().cpu().numpy()[0], row)   # the points are bf16-exact
    xq, xs = fge.fp8_quant_act(x, mode)
    torch.cuda.synchronize()
    assert float(xs.reshape(-1)[0].item()) == 1.0
    assert np.array_equal(xq.cpu().numpy()[0], codes)
