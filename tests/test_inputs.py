"""The seeded input generator's number formats against library conversions.

The generator rounds inputs to bf16 (both paths) and, for the estimator's
fp8 operands, to e4m3; these tests pin those roundings to torch's own
conversions (CPU), so that the oracle and the CUDA path see the intended
values.
"""
import numpy as np
import torch

from block_sparse_long_xattn_gb300.inputs import (
    E4M3_MAX, bf16_bits, e4m3_bits, round_to_bf16, round_to_e4m3)


def _samples():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s
                        for s in (1e-3, 0.05, 1.0, 8.0, 100.0)])
    # every e4m3 value and every midpoint between neighbouring values (ties)
    e4 = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).float()
    e4 = e4[torch.isfinite(e4)].numpy()
    pos = np.unique(e4[e4 >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    return np.concatenate([x, e4, mids, -mids, np.float32([0.0, -0.0, 2.0 ** -10])])


def test_bf16_rounding_matches_torch():
    x = _samples()
    ours = round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))
    np.testing.assert_array_equal(bf16_bits(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
                                  .numpy().view(np.uint16))


def test_e4m3_rounding_matches_torch():
    x = _samples()
    x = x[np.abs(x) <= E4M3_MAX]          # torch does not saturate
    ours = round_to_e4m3(x)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(ours, t.float().numpy())
    np.testing.assert_array_equal(e4m3_bits(ours), t.view(torch.uint8).numpy())


def test_e4m3_saturates():
    x = np.float32([449.0, 464.0, 470.0, 1e6, -500.0, -1e30])
    np.testing.assert_array_equal(round_to_e4m3(x), np.float32([448, 448, 448, 448, -448, -448]))
    np.testing.assert_array_equal(e4m3_bits(round_to_e4m3(x))[:2], np.uint8([0x7E, 0x7E]))
