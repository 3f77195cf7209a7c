"""GPU parity of every entry point against the fp64 oracle, at small sizes.

Sizes here let the oracle finish in seconds while still spanning several
128-token tiles, several key blocks per row, GQA groups, batch 2, every
supported stride, fp32 and bf16, q_start_pos = 0 and > 0, and the degenerate
cases (empty key range, a chunk of one block, threshold 1).
"""
import math

import numpy as np
import pytest
import torch

from block_sparse_long_xattn_gb300 import (
    bsx_bsa_prefill, bsx_bsa_prefill_split, bsx_chunk_prefill, bsx_chunk_step,
    bsx_cpu_block_mask, bsx_last_error, bsx_map_mask_to_cpu_blocks, bsx_merge_attn,
    bsx_quantize_e4m3, bsx_xattn_estimate)
from block_sparse_long_xattn_gb300.inputs import (
    e4m3_bits, make_workload, random_block_mask, round_to_bf16, round_to_e4m3)
from oracle import xattn_oracle as O
from tests.helpers import LSE_TOL, O_TOL, check_block_sums, check_mask, to_dev

pytestmark = pytest.mark.gpu


def _estimate(w, stride, tau):
    q, k = to_dev(w.q, w.dtype), to_dev(w.k, w.dtype)
    B, Lq, Hq, _ = w.q.shape
    nkb = w.k.shape[1] // 128
    A = torch.empty((B, Hq, Lq // 128, nkb), dtype=torch.float32, device="cuda")
    mask = bsx_xattn_estimate(q, k, w.q_start_pos, stride, tau, block_sums=A)
    torch.cuda.synchronize()
    return mask.cpu().numpy(), A.cpu().numpy()


ESTIMATE_CASES = [
    # (B, Hq, Hkv, d, Lk, P, stride, tau, dtype, alpha, n_hot)
    (1, 2, 1, 64, 1024, 0, 8, 0.9, "f32", 3.0, 0),     # the tiny single-chunk config
    (1, 4, 2, 128, 1024, 512, 8, 0.95, "bf16", 3.0, 2),
    (2, 4, 1, 64, 768, 256, 4, 0.9, "bf16", 2.0, 1),
    (1, 8, 2, 128, 2048, 1536, 16, 0.9, "bf16", 4.0, 3),
    (1, 2, 2, 128, 640, 0, 8, 0.8, "f32", 0.0, 0),
    (1, 4, 1, 128, 1152, 1024, 8, 0.99, "bf16", 3.0, 2),  # chunk of one block
    (1, 4, 2, 64, 896, 384, 16, 0.5, "bf16", 3.0, 1),
    (1, 2, 1, 64, 40960, 40704, 8, 0.9, "bf16", 3.0, 4),     # 320 key blocks per row
    (1, 1, 1, 64, 132096, 131968, 16, 0.9, "bf16", 3.0, 4),  # 1032: the CTA-per-row path
]


@pytest.mark.parametrize("case", ESTIMATE_CASES)
def test_estimate_mask_and_block_sums(case):
    B, Hq, Hkv, d, Lk, P, S, tau, dt, alpha, n_hot = case
    w = make_workload(seed=100 + Lk + P, B=B, Hq=Hq, Hkv=Hkv, d=d, Lk=Lk, q_start_pos=P,
                      alpha=alpha, n_hot=n_hot, dtype=dt)
    mask, A = _estimate(w, S, tau)
    est = O.xattn_estimate(w.q, w.k, P, S, tau)
    check_block_sums(A, est.block_sums, S)
    check_mask(mask, est, tau, P, A)
    assert bsx_last_error() == 0


def test_estimate_threshold_one_is_full_causal():
    w = make_workload(seed=5, B=1, Hq=4, Hkv=2, d=128, Lk=1024, q_start_pos=512,
                      alpha=3.0, n_hot=1, dtype="bf16")
    mask, _ = _estimate(w, 8, 1.0)
    cur = 512 // 128
    for qb in range(4):
        assert mask[:, :, qb, :cur + qb + 1].all()
        assert not mask[:, :, qb, cur + qb + 1:].any()


BSA_CASES = [
    # (B, Hq, Hkv, d, Lk, P, dtype, density)
    (1, 2, 1, 64, 1024, 0, "f32", 1.0),
    (1, 4, 2, 128, 1024, 512, "bf16", 0.5),
    (2, 4, 1, 64, 768, 256, "bf16", 0.3),
    (1, 8, 2, 128, 1536, 1024, "f32", 0.6),
    (1, 4, 4, 128, 512, 384, "bf16", 1.0),
    (1, 4, 1, 128, 8192, 7168, "bf16", 0.7),   # ~45 blocks per row: many pipeline phases
    (1, 2, 1, 64, 4096, 2048, "bf16", 0.9),
]


@pytest.mark.parametrize("case", BSA_CASES)
@pytest.mark.parametrize("cols", ["all", "hist", "curr"])
def test_bsa_prefill(case, cols):
    B, Hq, Hkv, d, Lk, P, dt, dens = case
    w = make_workload(seed=7 + Lk, B=B, Hq=Hq, Hkv=Hkv, d=d, Lk=Lk, q_start_pos=P,
                      alpha=3.0, n_hot=1, dtype=dt)
    Lq, nkb, cur = Lk - P, Lk // 128, P // 128
    mask = random_block_mask(17, B, Hq, Lq // 128, nkb, P, dens)
    kb0, kb1 = {"all": (0, nkb), "hist": (0, cur), "curr": (cur, nkb)}[cols]
    q, k, v = (to_dev(x, dt) for x in (w.q, w.k, w.v))
    o, lse = bsx_bsa_prefill(q, k, v, torch.from_numpy(mask).cuda(), P, kb0, kb1)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, mask, P, kb0, kb1)
    o_g = o.float().cpu().numpy()
    lse_g = lse.cpu().numpy()
    assert np.abs(o_g - o_ref).max() <= O_TOL[dt]
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_g), fin)
    if fin.any():
        assert np.abs(lse_g[fin] - lse_ref[fin]).max() <= LSE_TOL
    assert np.all(o_g[np.transpose(~fin, (0, 2, 1))] == 0.0)


def _pairing_mask(P, Lq, Hq, seed):
    """Rows of mixed lengths next to each other: head 0 has one long row (more
    than 128 selected blocks: many laps of the K/V ring) between two short
    ones; head 1 short rows that start at different blocks; head 2 long rows;
    head 3 short rows and one row holding only its diagonal block (an empty
    history part).  The tile count is odd."""
    rng = np.random.default_rng(seed)
    nqb, cur = Lq // 128, P // 128
    nkb = cur + nqb
    m = np.zeros((1, Hq, nqb, nkb), np.uint8)
    for h in range(Hq):
        for qb in range(nqb):
            diag = cur + qb
            if h == 2 or (h == 0 and qb == 1):
                m[0, h, qb, :diag + 1] = rng.random(diag + 1) < 0.95
            else:
                lo = {1: 3 + 7 * (qb & 1), 3: 10 - 7 * (qb & 1)}.get(h, 0)
                k = 2 if (h == 3 and qb == 2) else 30
                m[0, h, qb, lo + rng.choice(diag - lo, size=k, replace=False)] = 1
            m[0, h, qb, diag] = 1
    if Hq > 3:
        m[0, 3, 2, :cur + 2] = 0                  # only the diagonal block
    return m


def test_bsa_mixed_row_lengths():
    P, Lq, Hq = 20480, 384, 4
    Lk = P + Lq
    nkb, cur = Lk // 128, P // 128
    w = make_workload(seed=61, B=1, Hq=Hq, Hkv=2, d=128, Lk=Lk, q_start_pos=P,
                      alpha=2.0, n_hot=8, dtype="bf16")
    m = _pairing_mask(P, Lq, Hq, 5)
    assert (m.sum(axis=-1) > 128).any() and (m.sum(axis=-1) <= 128).any()
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    mask = torch.from_numpy(m).cuda()
    oh, lh, oc, lc = bsx_bsa_prefill_split(q, k, v, mask, P)
    oa, la = bsx_bsa_prefill(q, k, v, mask, P)
    torch.cuda.synchronize()
    for (o, lse), (kb0, kb1) in (((oh, lh), (0, cur)), ((oc, lc), (cur, nkb)),
                                 ((oa, la), (0, nkb))):
        o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, m, P, kb0, kb1)
        o_g, lse_g = o.float().cpu().numpy(), lse.cpu().numpy()
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse_g), fin)
        assert np.abs(o_g - o_ref).max() <= O_TOL["bf16"]
        assert np.abs(lse_g[fin] - lse_ref[fin]).max() <= LSE_TOL
    assert bsx_last_error() == 0


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_merge(dt, d):
    rng = np.random.default_rng(d)
    B, Lq, Hq = 2, 384, 4
    o1 = rng.standard_normal((B, Lq, Hq, d)).astype(np.float32)
    o2 = rng.standard_normal((B, Lq, Hq, d)).astype(np.float32)
    if dt == "bf16":
        o1 = to_dev(o1, dt).float().cpu().numpy()
        o2 = to_dev(o2, dt).float().cpu().numpy()
    l1 = (rng.standard_normal((B, Hq, Lq)) * 4).astype(np.float32)
    l2 = (rng.standard_normal((B, Hq, Lq)) * 4).astype(np.float32)
    l1[0, 0, :7] = -np.inf                   # one side empty
    l2[1, 1, 5:9] = -np.inf
    l1[1, 2, 0] = l2[1, 2, 0] = -np.inf      # both empty
    O1, L1 = to_dev(o1, dt), torch.from_numpy(l1).cuda()
    bsx_merge_attn(O1, L1, to_dev(o2, dt), torch.from_numpy(l2).cuda())
    torch.cuda.synchronize()
    o_ref, l_ref = O.merge_attn(o1, l1, o2, l2)
    assert np.abs(O1.float().cpu().numpy() - o_ref).max() <= O_TOL[dt]
    lg = L1.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5


@pytest.mark.parametrize("cpu_tokens,force", [(1024, False), (1024, True), (4096, False), (128, True)])
@pytest.mark.parametrize("Lq,offset", [(512, 0), (1024, 0), (1024, 1)])
def test_map(cpu_tokens, force, Lq, offset):
    """Lk/128 = 68 (byte loads), 72 (8-byte loads), 72 with a mask that starts
    one byte past an aligned address (byte loads)."""
    P = 8192
    mask = random_block_mask(3, 2, 4, Lq // 128, (P + Lq) // 128, P, 0.01)
    buf = torch.zeros(mask.size + offset, dtype=torch.uint8, device="cuda")
    dmask = buf[offset:].view(mask.shape)
    dmask.copy_(torch.from_numpy(mask))
    keep = bsx_map_mask_to_cpu_blocks(dmask, P, cpu_tokens, force)
    torch.cuda.synchronize()
    ref = O.map_mask_to_cpu_blocks(mask.astype(bool), P, cpu_tokens, force)
    np.testing.assert_array_equal(keep.cpu().numpy(), ref)


@pytest.mark.parametrize("P,Lq,d", [(1024, 512, 128), (0, 384, 128), (896, 256, 64)])
def test_bsa_split_equals_two_calls(P, Lq, d):
    """bsx_bsa_prefill_split gives, bit for bit, what bsx_bsa_prefill gives for
    the history and the current-chunk ranges, and both match the oracle."""
    w = make_workload(seed=31 + P + d, B=2, Hq=4, Hkv=2, d=d, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=2, dtype="bf16")
    nqb, nkb, cur = Lq // 128, (P + Lq) // 128, P // 128
    mask = random_block_mask(5 + P, 2, 4, nqb, nkb, P, 0.6)
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    dm = torch.from_numpy(mask).cuda()
    oh, lh, oc, lc = bsx_bsa_prefill_split(q, k, v, dm, P)
    oh2, lh2 = bsx_bsa_prefill(q, k, v, dm, P, 0, cur)
    oc2, lc2 = bsx_bsa_prefill(q, k, v, dm, P, cur, nkb)
    torch.cuda.synchronize()
    assert torch.equal(oh, oh2) and torch.equal(oc, oc2)
    assert torch.equal(lh, lh2) and torch.equal(lc, lc2)
    for (o_g, l_g), (kb0, kb1) in (((oc, lc), (cur, nkb)), ((oh, lh), (0, cur))):
        o_ref, l_ref = O.bsa_prefill(w.q, w.k, w.v, mask.astype(bool), P, kb0, kb1)
        fin = np.isfinite(l_ref)
        lg = l_g.cpu().numpy()
        assert np.array_equal(np.isfinite(lg), fin)
        if fin.any():
            assert np.abs(lg[fin] - l_ref[fin]).max() <= LSE_TOL
        assert np.abs(o_g.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]


def test_chunk_step_small():
    """Estimate -> BSA(history and current, one launch) -> merge -> map, small chunk."""
    P, S, tau = 768, 8, 0.9
    w = make_workload(seed=77, B=1, Hq=8, Hkv=2, d=128, Lk=P + 512, q_start_pos=P,
                      alpha=3.0, n_hot=2, dtype="bf16")
    est, o_ref, lse_ref, keep_ref = O.chunk_step(w.q, w.k, w.v, P, S, tau, 256)
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    # BSA runs on the oracle's mask so that near-threshold rows cannot differ
    A = torch.empty(est.block_sums.shape, dtype=torch.float32, device="cuda")
    mask_g = bsx_xattn_estimate(q, k, P, S, tau, block_sums=A)
    check_mask(mask_g.cpu().numpy(), est, tau, P, A.cpu().numpy())
    mask = torch.from_numpy(est.mask.astype(np.uint8)).cuda()
    cur, nkb = P // 128, (P + 512) // 128
    oh, lh, oc, lc = bsx_bsa_prefill_split(q, k, v, mask, P)
    bsx_merge_attn(oh, lh, oc, lc)
    keep = bsx_map_mask_to_cpu_blocks(mask, P, 256)
    torch.cuda.synchronize()
    assert np.abs(oh.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lh.cpu().numpy() - lse_ref).max() <= LSE_TOL
    np.testing.assert_array_equal(keep.cpu().numpy(), keep_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_bsa_running_max_grows_every_block(d):
    """Scores rise by ~8 (natural log) from each key block to the next, so the
    online softmax must rescale its accumulator at almost every block."""
    rng = np.random.default_rng(d)
    P, Lq, Hq = 1024, 256, 2
    Lk = P + Lq
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = (0.3 * rng.standard_normal((1, Lq, Hq, d)) + 4.0 * u).astype(np.float32)
    k = 0.3 * rng.standard_normal((1, Lk, 1, d))
    for kb in range(Lk // 128):
        k[0, kb * 128:(kb + 1) * 128, 0, :] += (2.0 * kb * math.sqrt(d)) * u  # logit +8 per block
    k = k.astype(np.float32)
    v = rng.standard_normal((1, Lk, 1, d)).astype(np.float32)
    qb_, kb_, vb_ = (to_dev(x, "bf16") for x in (q, k, v))
    q32, k32, v32 = (x.float().cpu().numpy() for x in (qb_, kb_, vb_))
    mask = np.ones((1, Hq, Lq // 128, Lk // 128), np.uint8)
    o, lse = bsx_bsa_prefill(qb_, kb_, vb_, torch.from_numpy(mask).cuda(), P)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.bsa_prefill(q32, k32, v32, mask, P, 0, Lk // 128)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL * max(1.0, np.abs(lse_ref).max() / 100)


FUSED_CASES = [
    # (B, Hq, Hkv, d, Lk, P, stride, tau, alpha, n_hot)
    (1, 8, 2, 128, 1280, 768, 8, 0.9, 3.0, 2),
    (2, 4, 1, 64, 768, 256, 4, 0.9, 2.0, 1),        # batch 2, d 64, stride 4
    (1, 4, 2, 128, 2048, 1536, 16, 0.9, 4.0, 3),    # stride 16
    (1, 2, 2, 128, 512, 0, 8, 0.8, 0.0, 0),         # whole-sequence prefill
    (1, 4, 1, 128, 1152, 1024, 8, 0.99, 3.0, 2),    # a chunk of one block
    (1, 4, 2, 128, 1024, 512, 8, 1.0, 3.0, 2),      # threshold 1: every causal block
    (1, 2, 1, 64, 40960, 40704, 8, 0.9, 3.0, 4),    # 320 key blocks: the 1024-key select
]


@pytest.mark.parametrize("case", FUSED_CASES)
def test_fused_chunk_prefill(case):
    """bsx_chunk_prefill as one kernel (estimate workers, in-kernel selection,
    attention CTAs waiting on row flags): the mask against the oracle's
    estimate (near-threshold rule; the tie rule with the stand-alone
    estimator's block sums, whose rounding the fused selection shares), and
    O / LSE against the oracle's attention over every key block on the
    kernel's own mask, every row."""
    B, Hq, Hkv, d, Lk, P, S, tau, alpha, n_hot = case
    w = make_workload(seed=91 + Lk + P, B=B, Hq=Hq, Hkv=Hkv, d=d, Lk=Lk, q_start_pos=P,
                      alpha=alpha, n_hot=n_hot, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    mask, o, lse = bsx_chunk_prefill(q, k, v, P, S, tau)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    _, A_g = _estimate(w, S, tau)
    est = O.xattn_estimate(w.q, w.k, P, S, tau)
    m_g = mask.cpu().numpy()
    check_mask(m_g, est, tau, P, A_g)
    if Lk > 8192:   # sampled rows: every query tile, both halves
        rows = np.array(sorted({r for t in range((Lk - P) // 128)
                                for r in (t * 128 + 3, t * 128 + 100)}))
        for h in range(Hq):
            o_r, l_r = O.bsa_rows(w.q, w.k, w.v, m_g, P, 0, Lk // 128, 0, h, rows)
            assert np.abs(o.float().cpu().numpy()[0, rows, h] - o_r).max() <= O_TOL["bf16"]
            assert np.abs(lse.cpu().numpy()[0, h, rows] - l_r).max() <= LSE_TOL
        return
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, m_g, P, 0, Lk // 128)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL


def test_fused_chunk_prefill_many_tiles_per_worker():
    """32 q-heads over an 8K context: more estimate tiles than SMs, so every
    worker takes several from the counter and the selection rows wait on
    tiles of other workers; the fused result equals the separate launches'
    (the same mask outside near-threshold rows, attention on it within the
    tolerance) and the oracle's on sampled rows of every query tile."""
    P, Lq, S, tau = 4096, 4096, 8, 0.9
    w = make_workload(seed=93, B=1, Hq=32, Hkv=8, d=128, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=8, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    mask, o, lse = bsx_chunk_prefill(q, k, v, P, S, tau)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    nkb = (P + Lq) // 128
    est = O.xattn_estimate(w.q, w.k, P, S, tau)
    _, A_g = _estimate(w, S, tau)
    m_g = mask.cpu().numpy()
    check_mask(m_g, est, tau, P, A_g)
    o2, lse2 = bsx_bsa_prefill(q, k, v, mask, P)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)   # the same attention code
    rows = np.array(sorted({t * 128 + (t * 41 + 7) % 128 for t in range(Lq // 128)}))
    for h in (0, 13, 31):
        o_r, l_r = O.bsa_rows(w.q, w.k, w.v, m_g, P, 0, nkb, 0, h, rows)
        assert np.abs(o.float().cpu().numpy()[0, rows, h] - o_r).max() <= O_TOL["bf16"]
        assert np.abs(lse.cpu().numpy()[0, h, rows] - l_r).max() <= LSE_TOL


CHUNK_STEP_CASES = [
    # (B, Hq, Hkv, d, Lk, P, stride, tau, cpu_block_tokens)
    (1, 8, 2, 128, 1280, 768, 8, 0.9, 256),
    (2, 4, 1, 64, 768, 256, 4, 0.9, 256),         # batch 2, d 64, stride 4
    (1, 4, 2, 128, 2048, 1536, 16, 0.9, 512),     # stride 16
    (1, 2, 2, 128, 512, 0, 8, 0.8, 128),          # no history: the current chunk alone
    (1, 4, 1, 128, 1152, 1024, 8, 0.99, 1024),    # a chunk of one block
    (1, 4, 2, 128, 1024, 512, 8, 1.0, 256),       # threshold 1
    (1, 2, 1, 64, 40960, 40704, 8, 0.9, 256),     # 320 key blocks: the 1024-key select
]


@pytest.mark.parametrize("case", CHUNK_STEP_CASES)
def test_chunk_step_one_kernel(case):
    """bsx_chunk_step as one kernel (estimate, selection with the CPU-block
    flags, attention on the history and on the current chunk, merged by the
    range that finishes second): the mask against the oracle's estimate; O,
    LSE and the flags bit-identical to the separate launches (split
    attention, merge, map) run on the kernel's own mask; O / LSE against the
    oracle's attention over every key block on that mask."""
    B, Hq, Hkv, d, Lk, P, S, tau, cpu = case
    w = make_workload(seed=97 + Lk + P, B=B, Hq=Hq, Hkv=Hkv, d=d, Lk=Lk, q_start_pos=P,
                      alpha=3.0, n_hot=2, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    mask, o, lse, keep = bsx_chunk_step(q, k, v, P, S, tau, cpu_block_tokens=cpu)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    _, A_g = _estimate(w, S, tau)
    est = O.xattn_estimate(w.q, w.k, P, S, tau)
    m_g = mask.cpu().numpy()
    check_mask(m_g, est, tau, P, A_g)
    nkb = Lk // 128
    oh, lh, oc, lc = bsx_bsa_prefill_split(q, k, v, mask, P)
    bsx_merge_attn(oh, lh, oc, lc)
    torch.cuda.synchronize()
    assert torch.equal(o, oh) and torch.equal(lse, lh)
    if P >= cpu:
        np.testing.assert_array_equal(keep.cpu().numpy(),
                                      bsx_map_mask_to_cpu_blocks(mask, P, cpu).cpu().numpy())
        np.testing.assert_array_equal(keep.cpu().numpy(), O.map_mask_to_cpu_blocks(m_g, P, cpu))
    else:
        assert keep is None
    if Lk > 8192:
        rows = np.array(sorted({r for t in range((Lk - P) // 128)
                                for r in (t * 128 + 3, t * 128 + 100)}))
        for h in range(Hq):
            o_r, l_r = O.bsa_rows(w.q, w.k, w.v, m_g, P, 0, nkb, 0, h, rows)
            assert np.abs(o.float().cpu().numpy()[0, rows, h] - o_r).max() <= O_TOL["bf16"]
            assert np.abs(lse.cpu().numpy()[0, h, rows] - l_r).max() <= LSE_TOL
        return
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, m_g, P, 0, nkb)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL


def test_offload_semantics_chunk_step():
    """The pages' offload attention: CPU blocks kept if any of their BSA blocks
    is selected (first and last forced), history dense over the kept CPU
    blocks, current chunk dense causal, merged by LSE."""
    P, S, tau, cpu = 1024, 8, 0.9, 256
    Lq = 512
    w = make_workload(seed=88, B=1, Hq=8, Hkv=2, d=128, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=2, dtype="bf16")
    est, keep_ref, o_ref, lse_ref = O.chunk_step_offload(w.q, w.k, w.v, P, S, tau, cpu)
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    mask_o = torch.from_numpy(est.mask.astype(np.uint8)).cuda()
    keep = bsx_map_mask_to_cpu_blocks(mask_o, P, cpu, True)
    om = bsx_cpu_block_mask(keep, Lq, P, 8, cpu)
    cur, nkb = P // 128, (P + Lq) // 128
    oh, lh = bsx_bsa_prefill(q, k, v, om, P, 0, cur)
    oc, lc = bsx_bsa_prefill(q, k, v, om, P, cur, nkb)
    bsx_merge_attn(oh, lh, oc, lc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(keep.cpu().numpy(), keep_ref)
    np.testing.assert_array_equal(om.cpu().numpy().astype(bool),
                                  O.offload_block_mask(keep_ref, 8, Lq, P, cpu))
    assert np.abs(oh.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lh.cpu().numpy() - lse_ref).max() <= LSE_TOL


@pytest.mark.parametrize("S,dt", [(8, "bf16"), (16, "bf16"), (8, "f32")])
def test_whole_sequence_prefill(S, dt):
    """GPU-only XAttention prefill of a whole sequence (q_start_pos 0): the
    estimate over all rows and one BSA launch over every key block."""
    Lk = 2048
    w = make_workload(seed=7 + S, B=1, Hq=4, Hkv=2, d=128 if dt == "bf16" else 64, Lk=Lk,
                      q_start_pos=0, alpha=3.0, n_hot=2, dtype=dt)
    q, k, v = (to_dev(x, dt) for x in (w.q, w.k, w.v))
    A = torch.empty((1, 4, Lk // 128, Lk // 128), dtype=torch.float32, device="cuda")
    mask = bsx_xattn_estimate(q, k, 0, S, 0.9, block_sums=A)
    est = O.xattn_estimate(w.q, w.k, 0, S, 0.9)
    check_block_sums(A.cpu().numpy(), est.block_sums, S)
    check_mask(mask.cpu().numpy(), est, 0.9, 0, A.cpu().numpy())
    m = torch.from_numpy(est.mask.astype(np.uint8)).cuda()
    o, lse = bsx_bsa_prefill(q, k, v, m, 0)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, est.mask, 0, 0, Lk // 128)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL[dt]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL


@pytest.mark.parametrize("n,offset", [(8192, 0), (1000, 0), (4096, 2)])
def test_quantize_e4m3_bit_exact(n, offset):
    """bf16 -> e4m3 bytes: nearest, ties to even, saturated; the 8-wide path
    (n % 8 == 0, aligned) and the one-value path (odd n, or an offset source)."""
    rng = np.random.default_rng(n + offset)
    x = np.concatenate([rng.standard_normal(n // 2).astype(np.float32) * 3,
                        rng.standard_normal(n - n // 2).astype(np.float32) * 200])
    x[:6] = [0.0, -0.0, 448.0, 464.0, -1e5, 2.0 ** -12]
    xb = round_to_bf16(x)
    buf = torch.from_numpy(np.concatenate([np.zeros(offset, np.float32), xb])).to(torch.bfloat16)
    src = buf.cuda()[offset:]
    out = bsx_quantize_e4m3(src)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.view(torch.uint8).cpu().numpy(),
                                  e4m3_bits(round_to_e4m3(xb)))


E4M3_CASES = [
    # (B, Hq, Hkv, Lk, P, stride, tau, alpha, n_hot), d = 128
    (1, 4, 2, 1024, 512, 8, 0.95, 3.0, 2),
    (2, 4, 1, 768, 256, 4, 0.9, 2.0, 1),
    (1, 8, 2, 2048, 1536, 16, 0.9, 4.0, 3),
    (1, 4, 2, 640, 0, 8, 0.8, 0.0, 0),
    (1, 2, 1, 40960, 40704, 8, 0.9, 3.0, 4),   # 320 key blocks per row
]


@pytest.mark.parametrize("case", E4M3_CASES)
def test_estimate_e4m3_operands(case):
    """The estimate on e4m3 Q and K (bsx_quantize_e4m3 of bf16 inputs) against
    the oracle's estimate of the same e4m3 values."""
    B, Hq, Hkv, Lk, P, S, tau, alpha, n_hot = case
    w = make_workload(seed=300 + Lk + P, B=B, Hq=Hq, Hkv=Hkv, d=128, Lk=Lk, q_start_pos=P,
                      alpha=alpha, n_hot=n_hot, dtype="bf16")
    est = O.xattn_estimate(round_to_e4m3(w.q), round_to_e4m3(w.k), P, S, tau)
    q8 = bsx_quantize_e4m3(to_dev(w.q, "bf16"))
    k8 = bsx_quantize_e4m3(to_dev(w.k, "bf16"))
    A = torch.empty(est.block_sums.shape, dtype=torch.float32, device="cuda")
    mask = bsx_xattn_estimate(q8, k8, P, S, tau, block_sums=A)
    torch.cuda.synchronize()
    A_g = A.cpu().numpy()
    check_block_sums(A_g, est.block_sums, S)
    check_mask(mask.cpu().numpy(), est, tau, P, A_g)
    assert bsx_last_error() == 0


HOST_STEP_CASES = [
    # (name, dtype, d, P, Lq, cpu, offload, force, e4m3, fused, two_streams)
    ("chunk", "bf16", 128, 768, 512, 256, False, False, False, False, True),
    ("one_stream", "bf16", 128, 768, 512, 256, False, True, False, False, False),
    ("offload", "bf16", 128, 1024, 512, 256, True, True, False, False, True),
    ("e4m3_estimate", "bf16", 128, 768, 512, 256, False, False, True, False, True),
    ("f32", "f32", 64, 512, 256, 256, False, False, False, False, True),
    ("first_chunk", "bf16", 128, 0, 384, 1024, False, False, False, False, True),
    ("fused", "bf16", 128, 768, 512, 256, False, False, False, True, True),
    ("whole_sequence", "bf16", 64, 0, 640, 1024, False, False, False, True, True),
]


@pytest.mark.parametrize("case", HOST_STEP_CASES, ids=[c[0] for c in HOST_STEP_CASES])
def test_chunk_step_host(case):
    """bsx_chunk_step_host (pinned host inputs -> host outputs, the uploads and
    read-back inside the call's stream work) equals the same step run through
    the device entry points bit for bit, and the oracle within the bar."""
    from block_sparse_long_xattn_gb300 import bsx_chunk_step_host, make_chunk_buffers
    _, dt, d, P, Lq, cpu, offload, force, e4m3, fused, two = case
    S, tau, Hq, Hkv = 8, 0.9, 8, 2
    w = make_workload(seed=500 + P + Lq + d, B=1, Hq=Hq, Hkv=Hkv, d=d, Lk=P + Lq,
                      q_start_pos=P, alpha=3.0, n_hot=2, dtype=dt)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    host = [torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(tdt).pin_memory()
            for x in (w.q, w.k, w.v)]
    bufs = make_chunk_buffers(host[0], host[1], P, S, cpu, offload=offload, e4m3_estimate=e4m3,
                              fused=fused)
    stream = torch.cuda.Stream()
    us, ds = (torch.cuda.Stream(), torch.cuda.Stream()) if two else (None, None)
    o_h, lse_h, keep_h = bsx_chunk_step_host(
        *host, P, S, tau, buffers=bufs, cpu_block_tokens=cpu, force_first_last=force,
        offload=offload, e4m3_estimate=e4m3, fused=fused, stream=stream, upload_stream=us,
        download_stream=ds)
    (ds or stream).synchronize()
    assert bsx_last_error() == 0

    # the same step through the device entry points.  A fused bf16 step
    # without the offload mask or e4m3 operands runs as one kernel
    # (bsx_chunk_prefill), whose selection may round a near-threshold row
    # differently from bsx_xattn_estimate's: then the attention after the
    # estimate takes the one kernel's mask and must match it bit for bit
    one_kernel = fused and dt == "bf16" and not (offload or e4m3)
    q, k, v = (x.cuda() for x in host)
    nkb, n_cpu = (P + Lq) // 128, P // cpu
    qe, ke = (bsx_quantize_e4m3(q), bsx_quantize_e4m3(k)) if e4m3 else (q, k)
    A = torch.empty((1, Hq, Lq // 128, nkb), dtype=torch.float32, device="cuda")
    mask = bsx_xattn_estimate(qe, ke, P, S, tau, block_sums=A)
    if one_kernel:
        mask = bufs["mask"].clone()
    keep = bsx_map_mask_to_cpu_blocks(mask, P, cpu, force) if n_cpu else None
    attn_mask = bsx_cpu_block_mask(keep, Lq, P, Hq, cpu) if offload else mask
    if fused:
        oh, lh = bsx_bsa_prefill(q, k, v, attn_mask, P, 0, nkb)
    else:
        oh, lh, oc, lc = bsx_bsa_prefill_split(q, k, v, attn_mask, P)
        bsx_merge_attn(oh, lh, oc, lc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bufs["mask"].cpu().numpy(), mask.cpu().numpy())
    assert torch.equal(o_h, oh.cpu()) and torch.equal(lse_h, lh.cpu())
    if n_cpu:
        np.testing.assert_array_equal(keep_h.numpy(), keep.cpu().numpy())
    else:
        assert keep_h is None

    # against the oracle
    qo, ko = (round_to_e4m3(w.q), round_to_e4m3(w.k)) if e4m3 else (w.q, w.k)
    est = O.xattn_estimate(qo, ko, P, S, tau)
    m_g = mask.cpu().numpy()
    check_mask(m_g, est, tau, P, A.cpu().numpy())
    if n_cpu:
        np.testing.assert_array_equal(keep_h.numpy(), O.map_mask_to_cpu_blocks(m_g, P, cpu, force))
    if offload:
        am = O.offload_block_mask(keep_h.numpy(), Hq, Lq, P, cpu)
        np.testing.assert_array_equal(attn_mask.cpu().numpy().astype(bool), am)
    else:
        am = m_g
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, am, P, 0, nkb)
    assert np.abs(o_h.float().numpy() - o_ref).max() <= O_TOL[dt]
    assert np.abs(lse_h.numpy() - lse_ref).max() <= LSE_TOL


def test_chunk_step_host_pipelined_buffer_sets():
    """Two buffer sets alternating on the same three streams (each step's
    uploads and read-back overlapping the other set's launches), four steps
    with different inputs: every step's host outputs equal the same step run
    alone."""
    from block_sparse_long_xattn_gb300 import bsx_chunk_step_host, make_chunk_buffers
    P, Lq, S, tau, cpu = 768, 512, 8, 0.9, 256
    ws = [make_workload(seed=900 + i, B=1, Hq=8, Hkv=2, d=128, Lk=P + Lq, q_start_pos=P,
                        alpha=3.0, n_hot=2, dtype="bf16") for i in range(4)]
    hosts = [[torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
              .pin_memory() for x in (w.q, w.k, w.v)] for w in ws]
    sets = [make_chunk_buffers(hosts[0][0], hosts[0][1], P, S, cpu) for _ in range(2)]
    st, us, ds = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    outs = [bsx_chunk_step_host(*hosts[i], P, S, tau, buffers=sets[i % 2], cpu_block_tokens=cpu,
                                stream=st, upload_stream=us, download_stream=ds)
            for i in range(4)]
    ds.synchronize()
    assert bsx_last_error() == 0
    for i in range(4):
        alone = make_chunk_buffers(hosts[i][0], hosts[i][1], P, S, cpu)
        o, lse, keep = bsx_chunk_step_host(*hosts[i], P, S, tau, buffers=alone,
                                           cpu_block_tokens=cpu)
        torch.cuda.synchronize()
        assert torch.equal(outs[i][0], o) and torch.equal(outs[i][1], lse)
        assert torch.equal(outs[i][2], keep)
    # different inputs gave different outputs (the sets were not mixed up)
    assert not torch.equal(outs[0][0], outs[1][0])


def test_bounded_wait_timeout_is_reported_and_the_context_survives():
    """Failure detection on the GPU without a fault: CTA 0's producer stops
    before K_2 (a phase nothing completes), its waits run out after their
    bound, the error word names the attention kernel and the wait that gave
    up, and the next launch on the same context is correct."""
    from block_sparse_long_xattn_gb300 import bsx_debug_drop_ring_item
    P, Lq = 1024, 256
    w = make_workload(seed=41, B=1, Hq=2, Hkv=1, d=128, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=1, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    nkb = (P + Lq) // 128
    mask_np = np.ones((1, 2, Lq // 128, nkb), np.uint8)   # CTA 0 has 10 key blocks
    mask = torch.from_numpy(mask_np).cuda()
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    bsx_debug_drop_ring_item(0, 3)
    bsx_bsa_prefill(q, k, v, mask, P)
    torch.cuda.synchronize()                  # the launch ends: no hang, no fault
    code = bsx_last_error()
    assert code & 0x80000000
    assert code & 0xFF == 1                   # the tcgen05 attention kernel
    assert (code >> 8) & 0xFF in (3, 5)       # the ring wait, or the S wait behind it
    o, lse = bsx_bsa_prefill(q, k, v, mask, P)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, mask_np, P, 0, nkb)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL


def test_fused_step_wait_timeout_is_reported_and_the_context_survives():
    """Failure detection in the fused chunk step without a fault: selection
    row 3 is never marked ready, so its attention CTA's bounded wait runs
    out; the error word names the fused step's row wait, that CTA writes
    o = 0 / lse = -inf, the other rows are correct, and the next fused step on
    the same context is correct everywhere."""
    from block_sparse_long_xattn_gb300 import bsx_debug_fused_skip_row
    P, Lq, S, tau = 512, 512, 8, 0.9
    w = make_workload(seed=45, B=1, Hq=2, Hkv=1, d=128, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=1, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    nqb, nkb = Lq // 128, (P + Lq) // 128
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    bsx_debug_fused_skip_row(3)               # b 0, h 0, qb 3
    mask, o, lse = bsx_chunk_prefill(q, k, v, P, S, tau)
    torch.cuda.synchronize()                  # the launch ends: no hang, no fault
    code = bsx_last_error()
    assert code & 0x80000000
    assert code & 0xFF == 3                   # the fused step's hand-over
    assert (code >> 8) & 0xFF == 1            # an attention CTA's wait for its row
    o_g, l_g = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o_g[0, 3 * 128:4 * 128, 0] == 0) and np.all(np.isneginf(l_g[0, 0, 384:512]))
    m_g = mask.cpu().numpy()
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, m_g, P, 0, nkb)
    keep = np.ones(o_g.shape[:3], bool)
    keep[0, 384:512, 0] = False
    assert np.abs(o_g - o_ref)[keep].max() <= O_TOL["bf16"]
    assert np.abs(l_g - lse_ref).transpose(0, 2, 1)[keep].max() <= LSE_TOL
    mask, o, lse = bsx_chunk_prefill(q, k, v, P, S, tau)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, mask.cpu().numpy(), P, 0, nkb)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL
    assert nqb == 4


def test_chunk_step_wait_timeout_is_reported_and_the_context_survives():
    """The one-kernel chunk step with selection row 2 never marked ready: the
    attention CTA of that query tile gives up after its bound and writes the
    empty result (o = 0, lse = -inf, the merge of two empty ranges); the
    error word names the fused step's row wait; every other row and the next
    step are correct."""
    from block_sparse_long_xattn_gb300 import bsx_debug_fused_skip_row
    P, Lq, S, tau, cpu = 512, 512, 8, 0.9, 256
    w = make_workload(seed=47, B=1, Hq=2, Hkv=1, d=128, Lk=P + Lq, q_start_pos=P,
                      alpha=3.0, n_hot=1, dtype="bf16")
    q, k, v = (to_dev(x, "bf16") for x in (w.q, w.k, w.v))
    nkb = (P + Lq) // 128
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    bsx_debug_fused_skip_row(2)               # b 0, h 0, qb 2
    mask, o, lse, _ = bsx_chunk_step(q, k, v, P, S, tau, cpu_block_tokens=cpu)
    torch.cuda.synchronize()
    code = bsx_last_error()
    assert code & 0x80000000 and code & 0xFF == 3 and (code >> 8) & 0xFF == 1
    o_g, l_g = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o_g[0, 256:384, 0] == 0) and np.all(np.isneginf(l_g[0, 0, 256:384]))
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, mask.cpu().numpy(), P, 0, nkb)
    keep_rows = np.ones(o_g.shape[:3], bool)
    keep_rows[0, 256:384, 0] = False
    assert np.abs(o_g - o_ref)[keep_rows].max() <= O_TOL["bf16"]
    assert np.abs(l_g - lse_ref).transpose(0, 2, 1)[keep_rows].max() <= LSE_TOL
    mask, o, lse, _ = bsx_chunk_step(q, k, v, P, S, tau, cpu_block_tokens=cpu)
    torch.cuda.synchronize()
    assert bsx_last_error() == 0
    o_ref, lse_ref = O.bsa_prefill(w.q, w.k, w.v, mask.cpu().numpy(), P, 0, nkb)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL
