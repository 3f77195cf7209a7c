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
# error actually measured on that row can fall either way (their order can
# flip); such rows must differ from the oracle only by swapping near-tied
# blocks at the cut.
TIE_SLACK_REL = 1e-7


def to_dev(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.to(device).contiguous()


def check_mask(mask_gpu: np.ndarray, est, threshold: float, q_start_pos: int,
               A_gpu: np.ndarray):
    """Compare a GPU mask with the oracle's estimate.

    Near-threshold rows (b, h, qb) -- some exclusive cumulative mass within
    MARGIN_TOL * T of threshold * T -- must hold a valid selection: the
    forced blocks, causal blocks only, oracle mass >= tau*T - MARGIN_TOL*T and
    a size within one of the oracle's.  Tie rows -- the last selected and the
    first unselected block closer than twice the row's measured block-sum
    error -- may differ from the oracle only in blocks whose mass is within
    that distance of the cut.  Every other row must match bit-exactly.
    Returns (n_rows, n_near_threshold, n_tie).
    """
    m_o = est.mask
    m_g = mask_gpu.astype(bool)
    assert m_g.shape == m_o.shape
    B, Hq, nqb, nkb = m_o.shape
    cur = q_start_pos // 128
    A = est.block_sums
    eps = np.abs(A_gpu.astype(np.float64) - A).max(axis=-1)       # [B, Hq, nqb]
    near = est.margin <= MARGIN_TOL
    n_near = n_tie = 0
    bad = []
    for b in range(B):
        for h in range(Hq):
            for qb in range(nqb):
                diag = cur + qb
                g, o = m_g[b, h, qb], m_o[b, h, qb]
                a = A[b, h, qb]
                T = a[:diag + 1].sum()
                if near[b, h, qb]:
                    n_near += 1
                    ok = g[0] and g[diag] and not g[diag + 1:].any()
                    ok = ok and a[g].sum() >= threshold * T - MARGIN_TOL * T - 1e-12
                    ok = ok and abs(int(g.sum()) - int(o.sum())) <= 1
                    if not ok:
                        bad.append((b, h, qb, "invalid near-threshold row"))
                    continue
                if np.array_equal(g, o):
                    continue
                tol = 2.0 * eps[b, h, qb] + TIE_SLACK_REL * T
                if est.gap[b, h, qb] * T <= tol:
                    # the cut value: mass of the oracle's smallest non-forced pick
                    picks = [kb for kb in np.nonzero(o)[0] if kb not in (0, diag)]
                    cut = a[picks].min() if picks else a[:diag + 1].max()
                    diff = np.nonzero(g != o)[0]
                    if np.all(np.abs(a[diff] - cut) <= tol) and g.sum() == o.sum():
                        n_tie += 1
                        continue
                diff = np.nonzero(g != o)[0][:8].tolist()
                bad.append((b, h, qb, f"differs at kb {diff}"))
    assert not bad, f"{len(bad)} mask rows differ, first: {bad[:5]}"
    return B * Hq * nqb, n_near, n_tie


def check_block_sums(A_gpu: np.ndarray, A_ref: np.ndarray, stride: int):
    T = 128 // stride
    err = np.abs(A_gpu.astype(np.float64) - A_ref).max()
    assert err <= A_TOL_REL * T, f"block sums max-abs error {err} > {A_TOL_REL * T}"
    return err
