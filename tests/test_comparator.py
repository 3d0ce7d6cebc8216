"""The comparator that every parity test uses (tests/_parity.py), checked on the CPU: its fast
bf16 ulp equals the definition, and it accepts and rejects what the stated tolerance says."""
import numpy as np

from _parity import Parity, bf16_bits_to_f64, ulp_bf16, ulp_bf16_reference


def test_ulp_matches_definition():
    rng = np.random.default_rng(7)
    ref = rng.standard_normal(200000) * np.exp(rng.uniform(-40.0, 40.0, 200000))
    special = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 2.0 ** 127, 3.0e38, 1.0e-3, np.inf, -np.inf, np.nan,
                        2.0 ** -1015, 1e308])
    ref = np.concatenate([ref, special])
    assert np.array_equal(ulp_bf16(ref), ulp_bf16_reference(ref))
    assert ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7 and ulp_bf16(np.array([-3.0]))[0] == 2.0 ** -6


def test_bits_to_f64():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, 1e-40, np.inf], dtype=np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    expect = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(bf16_bits_to_f64(bits), expect)


def test_bf16_tolerance_edges():
    # one bf16 ulp away passes, two fail; below 0.125 the 1e-3 floor applies
    ref = np.array([1.0, 1.0, 0.01, 0.01])
    gpu = np.array([1.0 + 2.0 ** -7, 1.0 + 2.0 ** -6, 0.01 + 0.9e-3, 0.01 + 1.2e-3])
    bits = (gpu.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = bf16_bits_to_f64(bits)
    par = Parity("edges")
    par.bf16("out", bits[:1], ref[:1])
    assert par.t["out"].bad == 0
    par.bf16("out", bits[1:2], ref[1:2])
    assert par.t["out"].bad == 1
    # the floor cases compare the bf16-representable values actually produced
    par2 = Parity("floor")
    par2.bf16("out", bits[2:], ref[2:])
    assert par2.t["out"].bad == int((np.abs(got[2:] - ref[2:]) > 1e-3).sum())


def test_dp_tolerance_and_nan():
    par = Parity("dp")
    ref = np.array([1.0, 1.0, 0.0, np.nan])
    ref_abs = np.array([1.0, 1.0, 100.0, 1.0])
    gpu = np.array([1.0 + 0.9e-3, 1.0 + 1.1e-3, 0.9e-4, np.nan], dtype=np.float32)
    par.dp(gpu, ref, ref_abs)
    # 0.9e-3 relative passes; 1.1e-3 fails; 0.9e-4 against a cancelled row sum of 100 passes
    # through the 1e-6 * sum|g a| term; NaN on both sides passes
    assert par.t["dp"].bad == 1 and par.t["dp"].floor_rows == 1


def test_expert_groups_partition_every_expert_in_order():
    from _parity import expert_groups
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 400, size=97)
    counts[[0, 5, 96]] = 0                                   # empty experts at the ends and inside
    off = np.concatenate([[0], np.cumsum(counts)])
    groups = expert_groups(off, rows_per_group=1000)
    assert groups[0][0] == 0 and groups[-1][1] == len(counts)
    assert all(a[1] == b[0] and a[0] < a[1] for a, b in zip(groups, groups[1:]))
    for e0, e1 in groups[:-1]:                               # every run but the last is full
        assert off[e1] - off[e0] >= 1000
        assert off[e1 - 1] - off[e0] < 1000                  # and the shortest run that is


def test_expert_groups_parallel_merges_like_one_pass():
    """Tallies of runs of experts checked several at once equal one pass over all rows."""
    import torch

    from _parity import Parity, for_expert_groups_parallel
    rng = np.random.default_rng(4)
    counts = rng.integers(0, 50, size=40)
    off = np.concatenate([[0], np.cumsum(counts)])
    R = int(off[-1])
    ref = rng.standard_normal((R, 8))
    gpu = ref + rng.standard_normal((R, 8)) * 1e-4
    gpu[7, 3] += 1.0                                          # one element out of tolerance
    bits = torch.from_numpy(gpu).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    def check(part, e0, e1, nthreads):
        a, b = int(off[e0]), int(off[e1])
        part.bf16("dx", bits[a:b], ref[a:b], row0=a)
        return b - a

    whole = Parity("one pass")
    whole.bf16("dx", bits, ref)
    runs = Parity("runs")
    rows = for_expert_groups_parallel(runs, off, check, rows_per_group=100, workers=3)
    assert sum(rows) == R
    w, r = whole.t["dx"], runs.t["dx"]
    assert (r.n, r.bad, r.worst_ratio, r.worst_abs) == (w.n, w.bad, w.worst_ratio, w.worst_abs)
    assert r.bad == 1 and r.examples[0][:2] == (7, 3)
