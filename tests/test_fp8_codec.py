"""The e4m3 rounding the FP8 parity tests apply to the oracle's output, pinned
against hand-worked values of the OCP FP8 e4m3 format and against PyTorch's
own float8_e4m3fn conversion inside the finite range."""
import numpy as np
import torch

from tests._parity import round_e4m3, ulp_e4m3


def test_hand_worked_values():
    cases = {
        1.0: 1.0, 0.1: 0.1015625,       # 13 / 128
        448.0: 448.0, 500.0: 448.0,     # saturates to the largest finite value
        -1000.0: -448.0,
        2.0 ** -9: 2.0 ** -9,           # smallest subnormal
        2.0 ** -10: 0.0,                # half a step: tie to even (0)
        3 * 2.0 ** -10: 2.0 ** -8,      # 1.5 steps: tie to even (2 steps)
        1.0625: 1.0,                    # halfway 1.0 / 1.125: even mantissa 000
        1.1875: 1.25,                   # halfway 1.125 / 1.25: even mantissa 010
        240.0: 240.0, 250.0: 256.0,     # step 16 between 128 and 256, 32 above
    }
    for x, want in cases.items():
        assert round_e4m3(np.array([x]))[0] == want, (x, round_e4m3(np.array([x]))[0], want)
    assert ulp_e4m3(np.array([1.0]))[0] == 0.125
    assert ulp_e4m3(np.array([0.001]))[0] == 2.0 ** -9


def test_matches_torch_in_range():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(20000, generator=g, dtype=torch.float64) * 40).clamp(-440, 440)
    x = torch.cat([x, torch.randn(2000, generator=g, dtype=torch.float64) * 1e-2])
    ours = round_e4m3(x.numpy())
    theirs = x.to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # float64 -> float32 first can move a value across an e4m3 tie only if it
    # lies within a float32 step of it; none of these draws do.
    assert np.array_equal(ours, theirs)
