"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in the oracle (on the CPU, by replacing one of its functions for the
duration of the test) and asserts that at least one pin from
tests/test_oracle_pins.py then fails.  The mistakes are the kind a restatement
of the pages could make: a stride reshape in the wrong direction, a dropped
factor of the softmax scale, a strict causal rule, a wrong GQA head mapping,
a selection that drops the crossing block or ignores the forced mass, a
selection margin that is always 0 or taken over inclusive sums, a gap not
divided by the row total, an
attention scale of 1/d (block-sparse or offload), a merge that weights by
LSE instead of exp(LSE), a CPU-block group shifted by one, an offload mask
without the diagonal block.
"""
import math

import numpy as np
import pytest

from oracle import xattn_oracle as O
from tests import test_oracle_pins as pins

BLOCK = 128
_offload_block_mask = O.offload_block_mask   # the unmutated functions
_select_row = O.select_row


def _q_forward(q_head, stride):
    return np.concatenate([q_head[t::stride, :] for t in range(stride)], axis=1)


def _k_reversed(k_head, stride):
    return np.concatenate([k_head[(stride - 1 - t)::stride, :] for t in range(stride)], axis=1)


def _scale_without_stride(d, stride):
    return 1.0 / math.sqrt(d)


def _strict_causal_rows(scores, row0, scale):
    R, C = scores.shape
    allowed = np.arange(C)[None, :] < (row0 + np.arange(R)[:, None])
    x = np.where(allowed, scores * scale, -np.inf)
    m = np.max(np.where(allowed, x, -1e300), axis=1, keepdims=True)
    e = np.where(allowed, np.exp(x - m), 0.0)
    s = e.sum(axis=1, keepdims=True)
    return e / np.where(s > 0, s, 1.0)


def _gqa_modulo_block_sums(q, k, q_start_pos, stride):
    B, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    out = np.zeros((B, Hq, Lq // BLOCK, Lk // BLOCK))
    for b in range(B):
        for h in range(Hq):
            s = O.antidiagonal_scores(q[b, :, h, :], k[b, :, h % Hkv, :], stride)
            p = O.causal_softmax_rows(s, q_start_pos // stride, O.estimator_scale(d, stride))
            out[b, h] = O.block_sums(p, BLOCK // stride)
    return out


def _select_dropping_crossing(a_row, forced, causal_end, threshold):
    rs = O.RowSelection(np.zeros(a_row.shape[0], bool), math.inf, math.inf, 0.0)
    vals = np.asarray(a_row, np.float64)[:causal_end]
    total = float(vals.sum())
    forced = sorted(set(f for f in forced if 0 <= f < causal_end))
    rs.selected[forced] = True
    if threshold >= 1.0:
        rs.selected[:causal_end] = True
        return rs
    c = float(sum(vals[f] for f in forced))
    for kb in sorted((kb for kb in range(causal_end) if kb not in forced),
                     key=lambda kb: (-vals[kb], kb)):
        if c + vals[kb] < threshold * total:   # inclusive sum: the crossing block is dropped
            rs.selected[kb] = True
            c += vals[kb]
        else:
            break
    rs.total = total
    return rs


def _select_ignoring_forced_mass(a_row, forced, causal_end, threshold):
    rs = O.RowSelection(np.zeros(a_row.shape[0], bool), math.inf, math.inf, 0.0)
    vals = np.asarray(a_row, np.float64)[:causal_end]
    total = float(vals.sum())
    forced = sorted(set(f for f in forced if 0 <= f < causal_end))
    rs.selected[forced] = True
    if threshold >= 1.0:
        rs.selected[:causal_end] = True
        return rs
    c = 0.0                                     # forced mass not counted
    for kb in sorted((kb for kb in range(causal_end) if kb not in forced),
                     key=lambda kb: (-vals[kb], kb)):
        if c < threshold * total:
            rs.selected[kb] = True
            c += vals[kb]
        else:
            break
    rs.total = total
    return rs


def _select_margin_zero(a_row, forced, causal_end, threshold):
    rs = _select_row(a_row, forced, causal_end, threshold)
    rs.margin = 0.0                             # every row would look near the threshold
    return rs


def _select_gap_not_normalised(a_row, forced, causal_end, threshold):
    rs = _select_row(a_row, forced, causal_end, threshold)
    rs.gap = rs.gap * rs.total                  # the raw mass difference, not / T
    return rs


def _select_margin_inclusive(a_row, forced, causal_end, threshold):
    rs = _select_row(a_row, forced, causal_end, threshold)
    vals = np.asarray(a_row, np.float64)[:causal_end]
    total = float(vals.sum())
    forced = sorted(set(f for f in forced if 0 <= f < causal_end))
    if threshold >= 1.0 or total <= 0:
        return rs
    c = float(sum(vals[f] for f in forced))
    margin = math.inf
    for kb in sorted((kb for kb in range(causal_end) if kb not in forced),
                     key=lambda kb: (-vals[kb], kb)):
        margin = min(margin, abs(c + vals[kb] - threshold * total) / total)  # inclusive sum
        if c >= threshold * total:
            break
        c += vals[kb]
    rs.margin = margin
    return rs


def _bsa_rows_variant(q, k, v, mask, q_start_pos, kb_begin, kb_end, b, h, rows, *,
                     power=0.5, strict=False, gqa_mod=False):
    """bsa_rows restated with one rule changed on request: the score divided
    by d**power (the oracle: 0.5), a strict token-causal rule, or kv-head
    h % Hkv instead of h // (Hq/Hkv)."""
    _, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    hk = h % Hkv if gqa_mod else h // (Hq // Hkv)
    rows = np.asarray(rows, np.int64)
    j = np.arange(Lk)
    causal = (j[None, :] < (q_start_pos + rows)[:, None]) if strict else \
        (j[None, :] <= (q_start_pos + rows)[:, None])
    allowed = ((j >= kb_begin * BLOCK) & (j < kb_end * BLOCK))[None, :] & \
        np.repeat(np.asarray(mask[b, h], bool)[rows // BLOCK], BLOCK, axis=1)[:, :Lk] & causal
    s = np.where(allowed, (np.asarray(q[b, rows, h, :], np.float64) @
                           np.asarray(k[b, :, hk, :], np.float64).T) / d ** power,
                 -np.inf)
    m = s.max(axis=1, keepdims=True)
    has = np.isfinite(m[:, 0])
    m = np.where(has[:, None], m, 0.0)
    e = np.where(allowed, np.exp(s - m), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((rows.shape[0], d))
    o[has] = (e[has] @ np.asarray(v[b, :, hk, :], np.float64)) / l[has, None]
    return o, np.where(has, m[:, 0] + np.log(np.where(has, l, 1.0)), -np.inf)


def _merge_by_lse(o1, lse1, o2, lse2):
    l1, l2 = np.asarray(lse1, np.float64), np.asarray(lse2, np.float64)
    w1 = np.where(np.isfinite(l1), l1, 0.0)
    w2 = np.where(np.isfinite(l2), l2, 0.0)
    den = np.where(w1 + w2 == 0, 1.0, w1 + w2)
    o = np.transpose(w1 / den, (0, 2, 1))[..., None] * o1 + \
        np.transpose(w2 / den, (0, 2, 1))[..., None] * o2
    return o, np.maximum(l1, l2)


def _map_shifted(mask, q_start_pos, cpu_block_tokens=1024, force_first_last=False):
    per = cpu_block_tokens // BLOCK
    n_cpu = q_start_pos // cpu_block_tokens
    keep = np.zeros((mask.shape[0], n_cpu), np.uint8)
    for b in range(mask.shape[0]):
        for c in range(n_cpu):
            keep[b, c] = 1 if mask[b, :, :, c * per + 1:(c + 1) * per + 1].any() else 0
        if force_first_last and n_cpu > 0:
            keep[b, 0] = keep[b, n_cpu - 1] = 1
    return keep


def _dense_attention_scale_1_over_d(qh, kh, vh, allowed):
    d = qh.shape[-1]
    s = np.where(allowed, (qh @ kh.T) / d, -np.inf)
    m = s.max(axis=1, keepdims=True)
    has = np.isfinite(m[:, 0])
    m = np.where(has[:, None], m, 0.0)
    e = np.where(allowed, np.exp(s - m), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((qh.shape[0], vh.shape[1]))
    o[has] = (e[has] @ vh) / l[has, None]
    return o, np.where(has, m[:, 0] + np.log(np.where(has, l, 1.0)), -np.inf)


def _offload_mask_strict_diagonal(keep, Hq, q_len, q_start_pos, cpu_block_tokens=1024):
    mask = _offload_block_mask(keep, Hq, q_len, q_start_pos, cpu_block_tokens)
    cur = q_start_pos // BLOCK
    for qb in range(q_len // BLOCK):
        mask[:, :, qb, cur + qb] = False           # the diagonal block dropped
    return mask


def _offload_pins():
    pins.test_offload_attention_all_kept_is_dense_causal()
    pins.test_offload_attention_equals_torch_on_kept_keys_and_bsa_with_its_mask()
    pins.test_offload_mask_small_example()


def _block_sum_pins():
    for S, P in ((8, 0), (8, 256), (4, 128), (16, 384)):
        pins.test_block_sums_match_torch_attention(S, P)
    pins.test_block_sums_row_invariant_and_causality()
    pins.test_block_sums_uniform_keys_closed_form()


def _selection_pins():
    pins.test_selection_worked_example()
    for seed in range(40):
        pins.test_selection_is_minimal_cover(seed)
    pins.test_selection_forced_mass_counts()


def _margin_gap_pins():
    pins.test_selection_margin_and_gap_worked_example()
    pins.test_selection_margin_and_gap_scaled_row_with_forced_block()
    pins.test_selection_margin_counts_the_forced_mass_alone()
    pins.test_selection_margin_and_gap_without_a_cut()
    for seed in range(30):
        pins.test_selection_margin_and_gap_brute_force(seed)


def _bsa_pins():
    for P, dens in ((0, 1.0), (0, 0.5), (384, 0.4), (256, 1.0)):
        pins.test_bsa_matches_torch_attention(P, dens)
    pins.test_bsa_empty_range_and_tau1_is_dense_causal()


MUTATIONS = {
    "query reshape taken forward": (
        "stride_reshape_q", _q_forward,
        lambda: (pins.test_reshape_positions_match_guide_example(),
                 pins.test_scores_equal_token_pair_loop(4, 3, 32, 48))),
    "softmax scale without the stride": ("estimator_scale", _scale_without_stride,
                                         _block_sum_pins),
    "strict reshaped causality": ("causal_softmax_rows", _strict_causal_rows, _block_sum_pins),
    "GQA head mapping h % Hkv": ("estimate_block_sums", _gqa_modulo_block_sums, _block_sum_pins),
    "crossing block dropped": ("select_row", _select_dropping_crossing, _selection_pins),
    "forced mass not counted": ("select_row", _select_ignoring_forced_mass, _selection_pins),
    "selection margin always 0": ("select_row", _select_margin_zero, _margin_gap_pins),
    "selection margin over inclusive sums": ("select_row", _select_margin_inclusive,
                                             _margin_gap_pins),
    "selection gap not divided by the row total": ("select_row", _select_gap_not_normalised,
                                                   _margin_gap_pins),
    "key reshape taken reversed": (
        "stride_reshape_k", _k_reversed,
        lambda: (pins.test_reshape_positions_match_guide_example(),
                 pins.test_scores_equal_token_pair_loop(4, 3, 32, 48))),
    "attention scale 1/d": (
        "bsa_rows", lambda *a: _bsa_rows_variant(*a, power=1.0), _bsa_pins),
    "strict token causality": (
        "bsa_rows", lambda *a: _bsa_rows_variant(*a, strict=True), _bsa_pins),
    "attention GQA head mapping h % Hkv": (
        "bsa_rows", lambda *a: _bsa_rows_variant(*a, gqa_mod=True), _bsa_pins),
    "merge weighted by LSE": ("merge_attn", _merge_by_lse,
                              lambda: (pins.test_merge_of_split_keys_equals_single_softmax(),
                                       pins.test_merge_identities())),
    "offload attention scale 1/d": ("_dense_attention", _dense_attention_scale_1_over_d,
                                    _offload_pins),
    "offload mask without the diagonal block": ("offload_block_mask",
                                                _offload_mask_strict_diagonal, _offload_pins),
    "CPU-block group shifted by one": (
        "map_mask_to_cpu_blocks", _map_shifted,
        lambda: (pins.test_map_golden_example(), pins.test_map_by_scatter(1024))),
}


def test_unmutated_bsa_rows_restatement_matches_the_oracle():
    """The restated attention used by the attention mutations agrees with the
    oracle with no rule changed, so each mutation changes only its rule."""
    from block_sparse_long_xattn_gb300.inputs import make_workload, random_block_mask
    w = make_workload(seed=2, B=1, Hq=4, Hkv=2, d=32, Lk=512, q_start_pos=256,
                      alpha=2.0, n_hot=1, dtype="f32")
    mask = random_block_mask(3, 1, 4, 2, 4, 256, 0.6)
    rows = np.arange(256)
    for h in range(4):
        o1, l1 = O.bsa_rows(w.q, w.k, w.v, mask, 256, 0, 4, 0, h, rows)
        o2, l2 = _bsa_rows_variant(w.q, w.k, w.v, mask, 256, 0, 4, 0, h, rows)
        np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_a_pin_catches_the_planted_mistake(name, monkeypatch):
    attr, fake, run_pins = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fake)
    with pytest.raises(AssertionError):
        run_pins()
