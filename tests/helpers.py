"""Shared test helpers: device upload and the mask-parity rule."""
from __future__ import annotations

import numpy as np
import torch

# Parity bar (written here once, used by every GPU test):
O_TOL = {"bf16": 2e-2, "f32": 1e-4}   # max-abs error of O
LSE_TOL = 1e-3                         # max-abs error of LSE
MARGIN_TOL = 1e-4                      # near-threshold: cumulative mass within 1e-4 of tau
# Block sums are fp32 on the GPU: the per-cell probabilities carry a few ulp of
# relative error (~1e-6) and a block sum adds up to 128/S * 128/S of them, so
# |A_gpu - A| <= 1e-5 * T (T = 128/S, the row total) bounds it with room.
A_TOL_REL = 1e-5
# A cut between two blocks whose masses differ by less than twice the block-sum
# tolerance can fall either way: such rows are counted as ambiguous too.
GAP_TOL = 2 * A_TOL_REL


def to_dev(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.to(device).contiguous()


def check_mask(mask_gpu: np.ndarray, est, threshold: float, q_start_pos: int):
    """Compare a GPU mask with the oracle's estimate.

    Rows (b, h, qb) whose cumulative mass lies within MARGIN_TOL of the
    threshold, or whose cut separates blocks closer than GAP_TOL, are
    ambiguous: they must hold a valid selection (forced blocks, causal only,
    oracle mass >= tau*T - MARGIN_TOL*T, size within one of the oracle's)
    and are counted.  Every other row must match bit-exactly.
    Returns (n_rows, n_ambiguous).
    """
    m_o = est.mask
    m_g = mask_gpu.astype(bool)
    assert m_g.shape == m_o.shape
    B, Hq, nqb, nkb = m_o.shape
    cur = q_start_pos // 128
    amb = (est.margin <= MARGIN_TOL) | (est.gap <= GAP_TOL)
    n_amb = 0
    bad = []
    for b in range(B):
        for h in range(Hq):
            for qb in range(nqb):
                diag = cur + qb
                g = m_g[b, h, qb]
                if amb[b, h, qb]:
                    n_amb += 1
                    A = est.block_sums[b, h, qb]
                    T = A[:diag + 1].sum()
                    ok = g[0] and g[diag] and not g[diag + 1:].any()
                    ok = ok and A[g].sum() >= threshold * T - MARGIN_TOL * T - 1e-12
                    ok = ok and abs(int(g.sum()) - int(m_o[b, h, qb].sum())) <= 1
                    if not ok:
                        bad.append((b, h, qb, "invalid ambiguous row"))
                elif not np.array_equal(g, m_o[b, h, qb]):
                    diff = np.nonzero(g != m_o[b, h, qb])[0][:8].tolist()
                    bad.append((b, h, qb, f"differs at kb {diff}"))
    assert not bad, f"{len(bad)} mask rows differ, first: {bad[:5]}"
    return B * Hq * nqb, n_amb


def check_block_sums(A_gpu: np.ndarray, A_ref: np.ndarray, stride: int):
    T = 128 // stride
    err = np.abs(A_gpu.astype(np.float64) - A_ref).max()
    assert err <= A_TOL_REL * T, f"block sums max-abs error {err} > {A_TOL_REL * T}"
    return err
