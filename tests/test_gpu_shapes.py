"""The forward on shapes other than the tiny and full ones, against the
oracle (every output).  Together they reach every supported extreme: the
smallest hidden size (256) and k = 1; I = 256 and I = 512 (the largest, which
changes FC1's units per token tile and FC2's stage count); 1024 experts with
k = 32; experts with several 128-row token tiles and a ragged last tile; H not
a multiple of 512; heavy tiles (256 pairs per expert) in units of two
output tiles, whose last units FC2 splits into single tiles (also with
I = 512)."""
import pytest
import torch

from oracle import cases
from nvfp4_routed_moe_gb300 import api
from gpu_util import Model, assert_close, out_bits

pytestmark = pytest.mark.gpu

SHAPES = [  # (H, I, E, k, T)
    (256, 128, 8, 1, 33),
    (768, 256, 40, 6, 50),
    (1024, 512, 64, 8, 40),
    (256, 128, 1024, 32, 20),
    (4096, 128, 16, 2, 300),
    (512, 128, 64, 4, 4096),
    (512, 512, 20, 4, 1300),
]


@pytest.mark.parametrize("H,I,E,k,T", SHAPES)
def test_shape_matches_oracle(H, I, E, k, T):
    inp = cases.prepare_small(11, T, H, I, E, k)
    m = Model(inp)
    out, ws = m.forward_inputs()
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert_close(out_bits(out), cases.run_oracle(inp), f"H={H} I={I} E={E} k={k} T={T}")
