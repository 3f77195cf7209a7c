"""fp64 CPU oracle for the XAttention block-sparse chunked-prefill path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

Everything is computed in float64 with numpy.  Inputs are taken as exact
values (bf16 inputs are exactly representable in float64).  The only library
primitives used as steps are ``numpy.matmul``, ``numpy.exp``/``numpy.log``
and ``numpy.argsort``/``sorted``; there is no blocking, fusion or reordering
beyond what the cited definitions state.

Sources (nano-vllm pages):
  [guide]  nano-vllm compare page, docs/xattention_algorithm_guide.md
           ("XAttention 算法实现指南"): sections "算法流程", "Stride Reshape 详解",
           "Triton Kernels 详解", "块选择算法 (find_blocks_chunked)" with its
           "示例", "BSA (Block Sparse Attention)", "计算复杂度".
  [optim]  nano-vllm compare page, optimization guide, section
           "Online Softmax Merge - Triton Fused Kernel".
  [policy] nano-vllm nanovllm/kvcache/sparse/xattn_bsa.py @11a867f,
           XAttentionBSAPolicy.select_blocks (Steps 0-6) and
           compute_chunked_prefill.
  [plan]   nano-vllm task_plan.md @ad361c2, "核心设计理解" section 1
           (Block Size 关系) and section 3 (select_blocks 设计).

Layouts (token-major, as the C ABI takes them):
  q    [B, Lq, Hq, d]      k, v [B, Lk, Hkv, d]      Lk = q_start_pos + Lq
  mask [B, Hq, Lq/128, Lk/128] bool
  o    [B, Lq, Hq, d]      lse  [B, Hq, Lq] (natural log)

Readings of points the pages leave open, used by the oracle and the kernels alike:
  * the threshold-crossing block is kept (the worked example keeps it);
  * the forced sink/diagonal mass counts toward threshold * total;
  * ties in block mass break by ascending key-block index;
  * threshold >= 1 selects every causal block;
  * reshaped causality is J <= I in global reshaped indices;
  * softmax is the natural softmax of score / (sqrt(d) * stride);
  * BSA applies the mask on current-chunk columns too (token-causal AND mask).

Every function here is pinned by ``tests/test_oracle_pins.py``; no function is
"parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

BSA_BLOCK = 128  # [guide] "BSA (Block Sparse Attention)": block size fixed at 128


# --------------------------------------------------------------------------- #
# a1: stride reshape (inverse mode) and antidiagonal scores                    #
# --------------------------------------------------------------------------- #
def stride_reshape_k(k_head: np.ndarray, stride: int) -> np.ndarray:
    """K_r = concat over t of K[t::stride] along the feature axis.

    [guide] "Stride Reshape 详解 / Inverse 模式": keys are interleaved forward,
    so reshaped key row j is [K[j*S+0], K[j*S+1], ..., K[j*S+S-1]].
    k_head: [Lk, d] -> [Lk/S, S*d].
    """
    return np.concatenate([k_head[t::stride, :] for t in range(stride)], axis=1)


def stride_reshape_q(q_head: np.ndarray, stride: int) -> np.ndarray:
    """Q_r = concat over t of Q[(S-1-t)::S] along the feature axis.

    [guide] "Stride Reshape 详解 / Inverse 模式": queries are interleaved in
    reverse, so reshaped query row i is [Q[i*S+S-1], Q[i*S+S-2], ..., Q[i*S]].
    q_head: [Lq, d] -> [Lq/S, S*d].
    """
    return np.concatenate(
        [q_head[(stride - 1 - t)::stride, :] for t in range(stride)], axis=1)


def antidiagonal_scores(q_head: np.ndarray, k_head: np.ndarray,
                        stride: int) -> np.ndarray:
    """Raw estimator scores Q_r @ K_r^T (no scale, no mask).

    [guide] "算法流程" Phase 2a (flat_group_gemm_fuse_reshape computes
    Q_reshaped @ K_reshaped^T).  Returns [Lq/S, Lk/S] float64.
    """
    qr = stride_reshape_q(np.asarray(q_head, np.float64), stride)
    kr = stride_reshape_k(np.asarray(k_head, np.float64), stride)
    return qr @ kr.T


# --------------------------------------------------------------------------- #
# a2 + a3: causal row softmax and block sums                                   #
# --------------------------------------------------------------------------- #
def estimator_scale(d: int, stride: int) -> float:
    """Natural-log softmax scale 1/(sqrt(d)*S).

    [policy] select_blocks Step 0 uses log2(e)/sqrt(d)/stride/norm with exp2
    and norm = 1; exp2(x*log2 e) = exp(x), so the natural softmax of
    score/(sqrt(d)*S) is the same distribution.
    """
    return 1.0 / (math.sqrt(d) * stride)


def causal_softmax_rows(scores: np.ndarray, row0: int, scale: float) -> np.ndarray:
    """Row softmax of scale*scores over keys J <= I, I = row0 + i.

    [guide] "Triton Kernels 详解 / softmax_fuse_block_sum" (online softmax,
    here done exactly with max subtraction) and [policy] select_blocks Step 0
    (Q starts at reshaped index chunk_start in the global key sequence).
    Masked entries are exactly 0.  scores: [R, C] -> probabilities [R, C].
    """
    R, C = scores.shape
    rows = row0 + np.arange(R)[:, None]
    cols = np.arange(C)[None, :]
    allowed = cols <= rows
    x = np.where(allowed, scores * scale, -np.inf)
    m = x.max(axis=1, keepdims=True)
    e = np.where(allowed, np.exp(x - m), 0.0)
    return e / e.sum(axis=1, keepdims=True)


def block_sums(p: np.ndarray, rows_per_block: int) -> np.ndarray:
    """attn_sum[qb, kb] = sum of p over the (128/S) x (128/S) cell.

    [guide] "Triton Kernels 详解": the output attn_sum[b,h,qi,ki] is the sum of
    the normalised weights of Q block qi on K block ki.
    p: [R, C] -> [R/r, C/r].
    """
    R, C = p.shape
    r = rows_per_block
    return p.reshape(R // r, r, C // r, r).sum(axis=(1, 3))


def estimate_block_sums(q: np.ndarray, k: np.ndarray, q_start_pos: int,
                        stride: int) -> np.ndarray:
    """attn_sum A[B, Hq, Lq/128, Lk/128] for a Q chunk at q_start_pos.

    [policy] select_blocks Steps 0-4 (chunk_start = q_start_pos/S in reshaped
    space; the key sequence is all earlier keys plus the chunk).  GQA maps
    q-head h to kv-head h // (Hq/Hkv) ([policy] expand_kv_for_gqa uses
    repeat_interleave).
    """
    B, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    assert Lk == q_start_pos + Lq
    G = Hq // Hkv
    r = BSA_BLOCK // stride
    scale = estimator_scale(d, stride)
    out = np.zeros((B, Hq, Lq // BSA_BLOCK, Lk // BSA_BLOCK), np.float64)
    for b in range(B):
        for h in range(Hq):
            s = antidiagonal_scores(q[b, :, h, :], k[b, :, h // G, :], stride)
            p = causal_softmax_rows(s, q_start_pos // stride, scale)
            out[b, h] = block_sums(p, r)
    return out


# --------------------------------------------------------------------------- #
# a4: threshold block selection                                                #
# --------------------------------------------------------------------------- #
@dataclass
class RowSelection:
    selected: np.ndarray   # bool [nkb]
    margin: float          # min_k |c_k - tau*T| / T over candidates' exclusive sums
    gap: float             # A(last selected non-forced) - A(first unselected), / T
    total: float           # T


def select_row(a_row: np.ndarray, forced: list[int], causal_end: int,
               threshold: float) -> RowSelection:
    """Greedy threshold selection for one query block.

    [guide] "块选择算法 (find_blocks_chunked)": total = row sum, required =
    threshold * total; sink and diagonal blocks are always kept; the rest are
    taken in descending order of mass until the cumulative mass reaches
    required.  Readings: the crossing block is kept (the section's worked
    example selects 4 of 5 blocks), forced mass counts toward the target, ties
    break by ascending block index, threshold >= 1 keeps every causal block.
    Only blocks kb < causal_end are candidates.
    """
    nkb = a_row.shape[0]
    sel = np.zeros(nkb, bool)
    vals = np.asarray(a_row, np.float64)[:causal_end]
    total = float(vals.sum())
    forced = sorted(set(f for f in forced if 0 <= f < causal_end))
    for f in forced:
        sel[f] = True
    if threshold >= 1.0:
        sel[:causal_end] = True
        return RowSelection(sel, math.inf, math.inf, total)
    target = threshold * total
    others = [kb for kb in range(causal_end) if kb not in forced]
    others.sort(key=lambda kb: (-vals[kb], kb))
    c = float(sum(vals[f] for f in forced))
    margin = math.inf
    last_sel = None
    first_unsel = None
    for kb in others:
        if total > 0:
            margin = min(margin, abs(c - target) / total)
        if c < target:
            sel[kb] = True
            c += vals[kb]
            last_sel = kb
        else:
            first_unsel = kb
            break
    gap = math.inf
    if last_sel is not None and first_unsel is not None and total > 0:
        gap = (vals[last_sel] - vals[first_unsel]) / total
    return RowSelection(sel, margin, gap, total)


@dataclass
class EstimateResult:
    mask: np.ndarray       # bool [B, Hq, nqb, nkb]
    block_sums: np.ndarray  # float64 [B, Hq, nqb, nkb]
    margin: np.ndarray     # float64 [B, Hq, nqb]
    gap: np.ndarray        # float64 [B, Hq, nqb]


def select_blocks(A: np.ndarray, q_start_pos: int, threshold: float) -> EstimateResult:
    """find_blocks_chunked over every (b, h, qb) row of A, then the causal post-mask.

    [policy] select_blocks Step 4: current_index = q_start_pos/128; the sink
    block 0 and the diagonal block current_index + qb are forced ([guide]
    "块选择算法"); blocks above the diagonal of the current chunk are cleared.
    """
    B, Hq, nqb, nkb = A.shape
    cur = q_start_pos // BSA_BLOCK
    mask = np.zeros(A.shape, bool)
    margin = np.zeros((B, Hq, nqb))
    gap = np.zeros((B, Hq, nqb))
    for b in range(B):
        for h in range(Hq):
            for qb in range(nqb):
                diag = cur + qb
                rs = select_row(A[b, h, qb], [0, diag], diag + 1, threshold)
                mask[b, h, qb] = rs.selected
                margin[b, h, qb] = rs.margin
                gap[b, h, qb] = rs.gap
    # causal post-mask (select_row never selects kb > diag; restated here)
    for qb in range(nqb):
        mask[:, :, qb, cur + qb + 1:] = False
    return EstimateResult(mask, A, margin, gap)


def xattn_estimate(q: np.ndarray, k: np.ndarray, q_start_pos: int,
                   stride: int, threshold: float) -> EstimateResult:
    """Estimator + selection + causal post-mask for one chunk.

    [policy] select_blocks Steps 0-4: block sums over all Lk keys, then
    find_blocks_chunked and the causal post-mask.
    """
    return select_blocks(estimate_block_sums(q, k, q_start_pos, stride),
                         q_start_pos, threshold)


# --------------------------------------------------------------------------- #
# a5: block-sparse causal attention with LSE                                   #
# --------------------------------------------------------------------------- #
def bsa_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray,
             q_start_pos: int, kb_begin: int, kb_end: int, b: int, h: int,
             rows: np.ndarray):
    """Block-sparse causal attention for selected query rows of one (b, h).

    [guide] "BSA (Block Sparse Attention)": causal FlashAttention restricted
    to the selected 128x128 tiles; returns O and (flash-attn convention)
    the natural-log LSE.  Query row i (global position P+i) sees key j iff
    kb_begin*128 <= j < kb_end*128, j <= P+i and mask[b,h,i//128,j//128].
    Rows with no visible key get O = 0 and LSE = -inf.
    Returns o [len(rows), d] and lse [len(rows)], float64.
    """
    _, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    G = Hq // Hkv
    rows = np.asarray(rows, np.int64)
    j = np.arange(Lk)
    in_range = (j >= kb_begin * BSA_BLOCK) & (j < kb_end * BSA_BLOCK)
    kh = np.asarray(k[b, :, h // G, :], np.float64)
    vh = np.asarray(v[b, :, h // G, :], np.float64)
    qh = np.asarray(q[b, rows, h, :], np.float64)
    block_ok = np.asarray(mask[b, h], bool)[rows // BSA_BLOCK]       # [n, nkb]
    block_ok = np.repeat(block_ok, BSA_BLOCK, axis=1)[:, :Lk]         # [n, Lk]
    allowed = in_range[None, :] & block_ok & \
        (j[None, :] <= (q_start_pos + rows)[:, None])
    s = (qh @ kh.T) / math.sqrt(d)
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    has = np.isfinite(m[:, 0])
    m_safe = np.where(has[:, None], m, 0.0)
    e = np.where(allowed, np.exp(s - m_safe), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((rows.shape[0], d))
    o[has] = (e[has] @ vh) / l[has, None]
    lse = np.where(has, m_safe[:, 0] + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def bsa_prefill(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray,
                q_start_pos: int, kb_begin: int, kb_end: int):
    """bsa_rows over every (b, h, 128-row query block).

    Returns o [B, Lq, Hq, d] float64 and lse [B, Hq, Lq] float64.
    """
    B, Lq, Hq, d = q.shape
    o = np.zeros((B, Lq, Hq, d), np.float64)
    lse = np.full((B, Hq, Lq), -np.inf, np.float64)
    for b in range(B):
        for h in range(Hq):
            for qb in range(Lq // BSA_BLOCK):
                rows = np.arange(qb * BSA_BLOCK, (qb + 1) * BSA_BLOCK)
                o_r, lse_r = bsa_rows(q, k, v, mask, q_start_pos, kb_begin,
                                      kb_end, b, h, rows)
                o[b, rows, h, :] = o_r
                lse[b, h, rows] = lse_r
    return o, lse


# --------------------------------------------------------------------------- #
# a6: LSE merge of two partial attentions                                      #
# --------------------------------------------------------------------------- #
def merge_attn(o1: np.ndarray, lse1: np.ndarray, o2: np.ndarray,
               lse2: np.ndarray):
    """Combine two partial (O, LSE) pairs over disjoint key sets.

    [optim] "Online Softmax Merge": m = max(lse1, lse2),
    w_i = exp(lse_i - m), O = (w1*o1 + w2*o2)/(w1 + w2), LSE = m + log(w1 + w2).
    If both LSE are -inf the row had no keys: O = 0, LSE = -inf.
    o*: [B, Lq, Hq, d], lse*: [B, Hq, Lq].
    """
    l1 = np.asarray(lse1, np.float64)
    l2 = np.asarray(lse2, np.float64)
    m = np.maximum(l1, l2)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w1 = np.where(np.isfinite(l1), np.exp(l1 - m_safe), 0.0)
    w2 = np.where(np.isfinite(l2), np.exp(l2 - m_safe), 0.0)
    den = np.where(empty, 1.0, w1 + w2)
    # weights are [B, Hq, Lq]; outputs are [B, Lq, Hq, d]
    w1o = np.transpose(w1 / den, (0, 2, 1))[..., None]
    w2o = np.transpose(w2 / den, (0, 2, 1))[..., None]
    o = w1o * np.asarray(o1, np.float64) + w2o * np.asarray(o2, np.float64)
    lse = np.where(empty, -np.inf, m_safe + np.log(den))
    return o, lse


# --------------------------------------------------------------------------- #
# a7: BSA-block mask -> CPU-block keep flags                                   #
# --------------------------------------------------------------------------- #
def map_mask_to_cpu_blocks(mask: np.ndarray, q_start_pos: int,
                           cpu_block_tokens: int = 1024,
                           force_first_last: bool = False) -> np.ndarray:
    """keep[b, c] = OR over heads, q-blocks and the c-th group of BSA blocks.

    [plan] section 1 (one 1024-token CPU block = 8 BSA blocks) and section 3
    step 3 (a CPU block is kept if any of its BSA blocks is selected, OR over
    heads and q-blocks); [policy] select_blocks Step 6 aggregates the same way
    over the historical blocks c < q_start_pos / cpu_block_tokens and then
    always adds the first and last historical block (force_first_last).
    mask: [B, Hq, nqb, nkb] -> keep uint8 [B, q_start_pos // cpu_block_tokens].
    """
    B = mask.shape[0]
    per = cpu_block_tokens // BSA_BLOCK
    n_cpu = q_start_pos // cpu_block_tokens
    keep = np.zeros((B, n_cpu), np.uint8)
    for b in range(B):
        for c in range(n_cpu):
            keep[b, c] = 1 if mask[b, :, :, c * per:(c + 1) * per].any() else 0
        if force_first_last and n_cpu > 0:
            keep[b, 0] = 1
            keep[b, n_cpu - 1] = 1
    return keep


# --------------------------------------------------------------------------- #
# One chunk of chunked prefill (history + current, merged)                     #
# --------------------------------------------------------------------------- #
def chunk_step(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_start_pos: int,
               stride: int, threshold: float, cpu_block_tokens: int = 1024):
    """Estimate, select, attend to history and current chunk, merge, map.

    [policy] select_blocks then compute_chunked_prefill: history attention is
    computed over key blocks before the chunk, current-chunk attention is
    causal, and the two (O, LSE) pairs are merged by LSE.  Here both halves
    use the per-head BSA mask (history without token masking, since every
    history key precedes every query; current with token-causal masking).
    """
    est = xattn_estimate(q, k, q_start_pos, stride, threshold)
    cur = q_start_pos // BSA_BLOCK
    nkb = k.shape[1] // BSA_BLOCK
    o_h, lse_h = bsa_prefill(q, k, v, est.mask, q_start_pos, 0, cur)
    o_c, lse_c = bsa_prefill(q, k, v, est.mask, q_start_pos, cur, nkb)
    o, lse = merge_attn(o_h, lse_h, o_c, lse_c)
    keep = map_mask_to_cpu_blocks(est.mask, q_start_pos, cpu_block_tokens)
    return est, o, lse, keep


# --------------------------------------------------------------------------- #
# The pages' CPU-offload attention (history dense over selected CPU blocks)    #
# --------------------------------------------------------------------------- #
def _dense_attention(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray,
                     allowed: np.ndarray):
    """softmax(q k^T / sqrt(d)) v over the allowed (query, key) pairs, with
    the natural-log LSE; rows without an allowed key get O = 0, LSE = -inf."""
    d = qh.shape[-1]
    s = np.where(allowed, (qh @ kh.T) / math.sqrt(d), -np.inf)
    m = s.max(axis=1, keepdims=True)
    has = np.isfinite(m[:, 0])
    m_safe = np.where(has[:, None], m, 0.0)
    e = np.where(allowed, np.exp(s - m_safe), 0.0)
    l = e.sum(axis=1)
    o = np.zeros((qh.shape[0], vh.shape[1]))
    o[has] = (e[has] @ vh) / l[has, None]
    lse = np.where(has, m_safe[:, 0] + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def offload_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, keep: np.ndarray,
                      q_start_pos: int, cpu_block_tokens: int = 1024):
    """Attention as nano-vllm's offload path computes it.

    [policy] compute_chunked_prefill: for every selected CPU block, in order,
    flash_attn_with_lse(q, k_block, v_block, causal=False) merged into the
    running (O, LSE) with merge_attention_outputs; then the current chunk with
    causal=True, merged last.  keep: uint8 [B, q_start_pos/cpu_block_tokens].
    Returns o [B, Lq, Hq, d], lse [B, Hq, Lq].
    """
    B, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    G = Hq // Hkv
    o_all = np.zeros((B, Lq, Hq, d))
    lse_all = np.full((B, Hq, Lq), -np.inf)
    for b in range(B):
        blocks = [c for c in range(keep.shape[1]) if keep[b, c]]
        for h in range(Hq):
            qh = np.asarray(q[b, :, h, :], np.float64)
            kh = np.asarray(k[b, :, h // G, :], np.float64)
            vh = np.asarray(v[b, :, h // G, :], np.float64)
            o_acc = None
            lse_acc = None
            for c in blocks:
                keys = slice(c * cpu_block_tokens, (c + 1) * cpu_block_tokens)
                allowed = np.ones((Lq, cpu_block_tokens), bool)
                o_c, lse_c = _dense_attention(qh, kh[keys], vh[keys], allowed)
                if o_acc is None:
                    o_acc, lse_acc = o_c, lse_c
                else:
                    o_m, lse_m = merge_attn(o_acc[None, :, None, :], lse_acc[None, None, :],
                                            o_c[None, :, None, :], lse_c[None, None, :])
                    o_acc, lse_acc = o_m[0, :, 0, :], lse_m[0, 0]
            cur = slice(q_start_pos, Lk)
            rows = np.arange(Lq)[:, None]
            allowed = np.arange(Lq)[None, :] <= rows        # j - P <= i
            o_c, lse_c = _dense_attention(qh, kh[cur], vh[cur], allowed)
            if o_acc is not None:
                o_m, lse_m = merge_attn(o_acc[None, :, None, :], lse_acc[None, None, :],
                                        o_c[None, :, None, :], lse_c[None, None, :])
                o_c, lse_c = o_m[0, :, 0, :], lse_m[0, 0]
            o_all[b, :, h, :] = o_c
            lse_all[b, h] = lse_c
    return o_all, lse_all


def offload_block_mask(keep: np.ndarray, Hq: int, q_len: int, q_start_pos: int,
                       cpu_block_tokens: int = 1024) -> np.ndarray:
    """The 128-token block mask under which block-sparse attention equals
    offload_attention: history block kb visible iff its CPU block is kept
    (every head, every q-block); current-chunk block kb visible iff it is at
    or before the q-block's diagonal.  Returns bool [B, Hq, q_len/128, Lk/128].
    """
    B = keep.shape[0]
    nqb = q_len // BSA_BLOCK
    cur = q_start_pos // BSA_BLOCK
    nkb = cur + nqb
    per = cpu_block_tokens // BSA_BLOCK
    mask = np.zeros((B, Hq, nqb, nkb), bool)
    for b in range(B):
        for qb in range(nqb):
            for kb in range(nkb):
                if kb < cur:
                    mask[b, :, qb, kb] = bool(keep[b, kb // per])
                else:
                    mask[b, :, qb, kb] = kb <= cur + qb
    return mask


def chunk_step_offload(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_start_pos: int,
                       stride: int, threshold: float, cpu_block_tokens: int = 1024):
    """[policy] select_blocks (estimate, then CPU blocks kept if any of their
    BSA blocks is selected, first and last always added) followed by
    compute_chunked_prefill (offload_attention)."""
    est = xattn_estimate(q, k, q_start_pos, stride, threshold)
    keep = map_mask_to_cpu_blocks(est.mask, q_start_pos, cpu_block_tokens,
                                  force_first_last=True)
    o, lse = offload_attention(q, k, v, keep, q_start_pos, cpu_block_tokens)
    return est, keep, o, lse
