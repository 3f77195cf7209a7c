"""Host logic of bench.py that needs no GPU: the clock record of the timed
region (nvidia-smi samples filtered to the region's wall-clock window) and
the algorithmic flop counts behind the roofline figures."""
import datetime
import os
import tempfile

import bench


def _line(t, mhz, power, power_cap="Not Active", hw="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {mhz}, 2070, {power}, {hw}, Not Active, Not Active, {power_cap}\n"


def _sampler(lines):
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.writelines(lines)
    c.proc = object()  # a sampler that ran
    return c


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.2, 2070, 170.0),                      # before: idle
             _line(t0 + 0.02, 1900, 400.0),
             _line(t0 + 0.04, 1790, 800.0, power_cap="Active"),
             _line(t0 + 0.06, 1800, 900.0, power_cap="Active"),
             _line(t0 + 0.5, 300, 150.0, hw="Active")]           # after: idle, throttled
    c = _sampler(lines)
    c.mark(t0, t0 + 0.1)
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1800 and s["sm_mhz_min"] == 1790
    assert s["reasons"] == ["sw_power_cap"]       # hw_slowdown was outside the region
    assert s["power_w_max"] == 900.0


def test_clock_summary_without_samples_in_the_region_says_so():
    t0 = 1_800_000_000.0
    c = _sampler([_line(t0 - 1.0, 2070, 170.0)])
    c.mark(t0, t0 + 0.01)
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None
    assert s["reasons"] == ["no samples inside the timed region"]


def test_bsa_flops_counts_the_visible_pairs_of_the_selected_tiles():
    """The roofline's algorithmic flops: 4 * d per (query, key) pair that the
    attention computes, counted here pair by pair on small masks (key j is
    visible to query row i of the chunk iff j <= q_start_pos + i, and its
    block is selected and inside the key range)."""
    import numpy as np
    rng = np.random.default_rng(3)
    for B, Hq, P, Lq, d in ((1, 2, 256, 384, 128), (2, 1, 0, 256, 64)):
        nqb, nkb = Lq // 128, (P + Lq) // 128
        mask = (rng.random((B, Hq, nqb, nkb)) < 0.6).astype(np.uint8)
        for kb0, kb1 in ((0, nkb), (0, P // 128), (P // 128, nkb)):
            pairs = 0
            for b in range(B):
                for h in range(Hq):
                    for i in range(Lq):
                        for j in range(kb0 * 128, kb1 * 128):
                            if j <= P + i and mask[b, h, i // 128, j // 128]:
                                pairs += 1
            assert bench.bsa_flops(mask, P, kb0, kb1, d) == 4 * d * pairs


def test_estimate_flops_counts_the_causal_reshaped_pairs():
    """2 * d * S flops per reshaped (row I, key J) pair with J <= I and per
    q-head, rows I covering the chunk, counted pair by pair."""
    for q_len, P, S in ((256, 512, 8), (512, 0, 16), (128, 128, 4)):
        cfg = dict(B=2, Hq=3, d=64)
        pairs = sum(1 for I in range(P // S, (P + q_len) // S) for J in range((P + q_len) // S)
                    if J <= I)
        assert bench.estimate_flops(cfg, q_len, P, S) == 2.0 * 64 * S * pairs * 3 * 2


def test_mask_rows_vs_oracle_counts_near_and_differing_rows():
    """The bench's parity record for the oracle's sampled heads: rows whose
    margin is within 1e-4 count as near the threshold (exempt), any other
    row that differs from the oracle's mask is counted as differing."""
    from types import SimpleNamespace
    import numpy as np
    B, Hq, nqb, nkb = 1, 8, 3, 5
    gpu = np.zeros((B, Hq, nqb, nkb), np.uint8)
    ests, heads = [], [0, 4]
    for h in heads:
        m = np.zeros((B, 1, nqb, nkb), bool)
        m[0, 0, :, 0] = True
        margin = np.full((B, 1, nqb), 0.5)
        ests.append(SimpleNamespace(mask=m, margin=margin))
        gpu[0, h, :, 0] = 1
    # head 0, row 1: differs but is near the threshold; head 4, row 2: differs
    ests[0].margin[0, 0, 1] = 5e-5
    gpu[0, 0, 1, 3] = 1
    gpu[0, 4, 2, 2] = 1
    r = bench.mask_rows_vs_oracle(gpu, ests, heads)
    assert r["rows"] == 2 * nqb
    assert r["near_threshold"] == 1
    assert r["other_rows_differing"] == 1


def test_both_arms_print_the_same_config():
    """The GPU arm and the reference arm describe the workload with one dict,
    so a driver comparing the two lines sees the same configuration."""
    from types import SimpleNamespace
    for wl, step in (("llama8b-32k-chunk4096", "chunk"), ("llama8b-64k-chunked", "chunked"),
                     ("llama8b-128k-rho10", "chunk")):
        args = SimpleNamespace(workload=wl, step=step, seed=0, estimator="bf16")
        c = bench.config_dict(args, 1)
        assert c["workload"] == wl and c["parallelism"] == "replicas1"
        cfg = bench.CONFIGS[wl]
        assert c["stride"] == cfg["stride"] and c["threshold"] == cfg["threshold"]
        if step == "chunked":
            assert c["seq_len"] == cfg["Lk"] and c["chunks"] == cfg["Lk"] // cfg["chunk"]
        else:
            assert c["q_len"] + c["q_start_pos"] == c["Lk"] == cfg["Lk"]
