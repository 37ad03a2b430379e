"""bench.py's FLOP accounting for fa_fwd_kv workloads (CPU only).

The kv pass counts 4 d FLOPs per visible (query, key) pair; the closed form
it uses is checked here against counting the pairs one by one, for both
causal alignments, no mask, padding to zero keys and more queries than keys.
"""
import itertools

import bench
import seeded_inputs


def brute_pairs(Nq, n, causal, off):
    return sum(1 for i in range(Nq) for j in range(n) if not causal or j <= i + off)


def test_visible_pairs_closed_form():
    for Nq, n, causal in itertools.product([1, 2, 5, 17, 40, 129], [0, 1, 3, 16, 50, 200],
                                           [None, "bottom_right", "upper_left"]):
        w = dict(B=1, Nq=Nq, Nk=max(n, 1), causal=causal)
        off = n - Nq if causal == "bottom_right" else 0
        assert bench.kv_visible_pairs(w, n, off) == brute_pairs(Nq, n, causal, off), \
            (Nq, n, causal)


def test_positions_follow_alignment_and_clamp():
    w = dict(B=3, Nq=10, Nk=100, causal="bottom_right")
    assert bench.kv_positions(w, [100, 7, 500]) == [(100, 90), (7, -3), (100, 90)]
    w["causal"] = "upper_left"
    assert bench.kv_positions(w, None) == [(100, 0)] * 3


def test_square_causal_matches_forward_convention():
    """Nq = Nk, upper-left: the exact count is the halved N^2 convention plus N/2."""
    N, d = 4096, 128
    w = dict(B=1, H=1, Nq=N, Nk=N, d=d, causal="upper_left")
    assert bench.step_flops_kv(w, None) == 4.0 * d * (N * N / 2 + N / 2)


def test_kv_workloads_are_well_formed():
    for w in seeded_inputs.KV_WORKLOADS:
        sl = seeded_inputs.make_seqlens(w["B"], w["Nk"], w["seed"]) if w["padded"] else None
        if sl is not None:
            assert sl.shape == (w["B"],) and int(sl.min()) >= 1 and int(sl.max()) <= w["Nk"]
        assert bench.step_flops_kv(w, sl) > 0
