"""Pins for the CPU oracle: each check fixes the oracle to something other
than itself (hand-worked values, exact rational arithmetic, closed forms,
invariants, brute-force metadata)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W
from conftest import GROUP_ROWS, TILE_ROWS, TC_MIN_QLEN

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _proj_from_golden(g):
    N, L = g["num_slots"], len(g["lane_d_out"])
    rank = np.array(g["rank"], dtype=np.int32)
    A = [[None] * L for _ in range(N)]
    B = [[None] * L for _ in range(N)]
    for key, v in g["A"].items():
        k, l = (int(s) for s in key.split(","))
        A[k][l] = W.bf16_bits(np.array(v, dtype=np.float32))
    for key, v in g["B"].items():
        k, l = (int(s) for s in key.split(","))
        B[k][l] = W.bf16_bits(np.array(v, dtype=np.float32))
    x = W.bf16_bits(np.array(g["x"], dtype=np.float32))
    return W.Projection("golden", g["d_in"], list(g["lane_d_out"]), rank,
                        np.array(g["scale"], dtype=np.float32), A, B, x,
                        np.array(g["y0"], dtype=np.float32), int(rank.max()))


def test_golden_handworked_delta(oracle_mod):
    with open(os.path.join(GOLDEN, "handworked_delta.json")) as f:
        g = json.load(f)
    proj = _proj_from_golden(g)
    T = int(sum(g["q_seq_lens"]))
    meta = oracle_mod.segments(g["adapter_ids"], g["q_seq_lens"], T, g["num_slots"],
                               g["metadata_tc_min_qlen"], g["metadata_tile_rows"],
                               g["metadata_group_rows"])
    assert meta["status"] == 0
    assert meta["slot"].tolist() == g["expected_slot"]
    assert meta["perm"].tolist() == g["expected_perm"]
    assert meta["seg_off"].tolist() == g["expected_seg_off"]
    assert meta["dec_work"].tolist() == g["expected_dec_work"]
    assert meta["tc_work"].tolist() == g["expected_tc_work"]
    assert meta["counts"].tolist() == g["expected_counts"]
    y, _ = oracle_mod.delta(proj, meta["slot"])
    assert np.array_equal(y, np.array(g["expected_y"], dtype=np.float64))


def _exact_delta_row(proj, t, k):
    """Exact rational delta of row t under slot k (Fractions; bf16/fp32 are dyadic)."""
    xf = W.bf16_bits_to_f32(proj.x[t])
    out = []
    for l, dout in enumerate(proj.lane_d_out):
        r = int(proj.rank[k, l])
        if k == 0 or r == 0:
            out += [Fraction(0)] * dout
            continue
        A = W.bf16_bits_to_f32(proj.A[k][l])
        B = W.bf16_bits_to_f32(proj.B[k][l])
        u = [sum(Fraction(float(A[i, j])) * Fraction(float(xf[j])) for j in range(proj.d_in))
             for i in range(r)]
        s = Fraction(float(proj.scale[k, l]))
        for o in range(dout):
            out.append(s * sum(Fraction(float(B[o, i])) * u[i] for i in range(r)))
    return out


def _abs_bound_row(proj, t, k):
    """sum of |terms| per output: a scale for the fp64 rounding error."""
    xf = np.abs(W.bf16_bits_to_f32(proj.x[t]).astype(np.float64))
    out = []
    for l, dout in enumerate(proj.lane_d_out):
        r = int(proj.rank[k, l])
        if k == 0 or r == 0:
            out.append(np.zeros(dout))
            continue
        A = np.abs(W.bf16_bits_to_f32(proj.A[k][l]).astype(np.float64))
        B = np.abs(W.bf16_bits_to_f32(proj.B[k][l]).astype(np.float64))
        out.append(abs(float(proj.scale[k, l])) * (B @ (A @ xf)))
    return np.concatenate(out)


def test_delta_against_exact_rationals(oracle_mod):
    # Several lanes, heterogeneous ranks, a rank-0 lane, base rows.
    rank = np.array([[0, 0], [3, 5], [4, 0], [1, 2]], dtype=np.int32)
    wl = W.custom_workload([1, 2, 1, 3, 1], [1, 2, 0, 3, 1], d_in=24, lane_d_out=[16, 8],
                           num_slots=4, max_rank=5, rank=rank, seed=3)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    _, dl = oracle_mod.delta(proj, slot)
    for t in range(wl.T):
        exact = _exact_delta_row(proj, t, int(slot[t]))
        bound = _abs_bound_row(proj, t, int(slot[t]))
        for c, e in enumerate(exact):
            assert abs(dl[t, c] - float(e)) <= 1e-14 * bound[c] + 1e-300, (t, c)


def test_y_is_y0_plus_delta_and_base_rows_untouched(oracle_mod):
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    y, dl = oracle_mod.delta(proj, slot)
    y0 = proj.y0.astype(np.float64)
    assert np.array_equal(y, y0 + dl)
    base = slot == 0
    assert base.any() and (~base).any()
    assert np.array_equal(y[base], y0[base])
    assert np.all(dl[base] == 0)
    assert np.all(np.abs(dl[~base]).max(axis=1) > 0)


def _rank1_projection(d_in, d_out, i, j, s, T, seed=0):
    rng = np.random.default_rng(seed)
    N = 2
    rank = np.array([[0], [1]], dtype=np.int32)
    A = [[None], [None]]
    B = [[None], [None]]
    a = np.zeros((1, d_in), dtype=np.float32)
    a[0, i] = 1.0
    b = np.zeros((d_out, 1), dtype=np.float32)
    b[j, 0] = 1.0
    A[1][0] = W.bf16_bits(a)
    B[1][0] = W.bf16_bits(b)
    x = W.bf16_bits(rng.standard_normal((T, d_in)).astype(np.float32))
    y0 = rng.standard_normal((T, d_out)).astype(np.float32)
    return W.Projection("rank1", d_in, [d_out], rank, np.array([[0], [s]], dtype=np.float32),
                        A, B, x, y0, 1)


@pytest.mark.parametrize("i,j,s", [(0, 0, 2.0), (5, 17, 0.75), (31, 2, -3.0)])
def test_rank1_unit_vectors_closed_form(oracle_mod, i, j, s):
    # A = e_i^T (1 x d_in), B = e_j (d_out x 1): delta[t] = s * x[t][i] at column j only.
    d_in, d_out, T = 32, 20, 6
    proj = _rank1_projection(d_in, d_out, i, j, s, T)
    slot = np.array([1, 0, 1, 1, 0, 1], dtype=np.int32)
    _, dl = oracle_mod.delta(proj, slot)
    xf = W.bf16_bits_to_f32(proj.x).astype(np.float64)
    expect = np.zeros((T, d_out))
    expect[slot == 1, j] = s * xf[slot == 1, i]
    assert np.array_equal(dl, expect)


def test_scale_zero_leaves_y_unchanged(oracle_mod):
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    y, dl = oracle_mod.delta(proj, wl.per_token_slot(), scale=np.zeros_like(proj.scale))
    assert np.array_equal(y, proj.y0.astype(np.float64))
    assert np.all(dl == 0)


def test_rank_zero_lane_is_not_written(oracle_mod):
    rank = np.array([[0, 0, 0], [4, 0, 4], [0, 4, 0]], dtype=np.int32)
    wl = W.custom_workload([1, 1, 1, 1], [1, 2, 1, 2], d_in=16, lane_d_out=[8, 8, 8],
                           num_slots=3, max_rank=4, rank=rank)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    _, dl = oracle_mod.delta(proj, slot)
    for t in range(4):
        k = slot[t]
        for l in range(3):
            seg = dl[t, 8 * l:8 * (l + 1)]
            if rank[k, l] == 0:
                assert np.all(seg == 0)
            else:
                assert np.any(seg != 0)


def test_association_independent_of_evaluation_order(oracle_mod):
    # (scale * B @ A) @ x evaluated with numpy float64 matches B @ (A @ x) to fp64 rounding.
    wl = W.custom_workload([3, 2, 4], [1, 2, 1], d_in=64, lane_d_out=[48, 16], num_slots=3,
                           max_rank=8, seed=11)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    _, dl = oracle_mod.delta(proj, slot)
    xf = W.bf16_bits_to_f32(proj.x).astype(np.float64)
    for t in range(wl.T):
        k = slot[t]
        ref = []
        for l, dout in enumerate(proj.lane_d_out):
            Wm = float(proj.scale[k, l]) * (W.bf16_bits_to_f32(proj.B[k][l]).astype(np.float64)
                                            @ W.bf16_bits_to_f32(proj.A[k][l]).astype(np.float64))
            ref.append(Wm @ xf[t])
        ref = np.concatenate(ref)
        assert np.allclose(dl[t], ref, rtol=1e-12, atol=1e-12)


def test_linearity_in_x(oracle_mod):
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    _, d1 = oracle_mod.delta(proj, slot)
    x2 = W.bf16_bits(2.0 * W.bf16_bits_to_f32(proj.x))
    _, d2 = oracle_mod.delta(proj, slot, x=x2)
    assert np.array_equal(d2, 2.0 * d1)


def test_rows_are_independent_of_batch_composition(oracle_mod):
    # The same row (same x, same slot) gives the same delta inside two different batches.
    wl = W.custom_workload([1] * 12, [1, 2, 0, 3, 1, 1, 2, 3, 0, 1, 2, 3], d_in=32,
                           lane_d_out=[24], num_slots=4, max_rank=6, seed=5)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    _, full = oracle_mod.delta(proj, slot)
    sub = np.array([7, 0, 11, 3], dtype=np.int64)
    _, part = oracle_mod.delta(proj, slot[sub], x=proj.x[sub], y0=proj.y0[sub])
    assert np.array_equal(part, full[sub])
    _, sel = oracle_mod.delta(proj, slot, rows=sub)
    assert np.array_equal(sel, full[sub])


def test_sequence_permutation_permutes_rows(oracle_mod):
    lens = [3, 1, 2, 1]
    ids = [1, 0, 2, 1]
    wl = W.custom_workload(lens, ids, d_in=16, lane_d_out=[8], num_slots=3, max_rank=4, seed=2)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    y, _ = oracle_mod.delta(proj, slot)
    starts = np.concatenate([[0], np.cumsum(lens)])
    order = [2, 0, 3, 1]
    rows = np.concatenate([np.arange(starts[s], starts[s + 1]) for s in order])
    meta = oracle_mod.segments([ids[s] for s in order], [lens[s] for s in order], sum(lens), 3,
                               TC_MIN_QLEN, TILE_ROWS, GROUP_ROWS)
    y2, _ = oracle_mod.delta(proj, meta["slot"], x=proj.x[rows], y0=proj.y0[rows])
    assert np.array_equal(y2, y[rows])


# ---------------------------------------------------------------- metadata pins

def _brute_metadata(ids, lens, T, N, tcq, tile, group):
    ids = np.asarray(ids, dtype=np.int64)
    lens = np.asarray(lens, dtype=np.int64)
    if (lens < 0).any() or lens.sum() != T:
        return {"status": -6}
    if ((ids < 0) | (ids >= N)).any():
        return {"status": -3}
    slot = np.repeat(ids, lens)
    seq = np.repeat(np.arange(len(ids)), lens)
    cls = (lens[seq] >= tcq).astype(np.int64)
    rows = [t for t in range(T) if slot[t] != 0]
    perm = sorted(rows, key=lambda t: (cls[t], slot[t], t))
    seg_off = []
    for c in range(2):
        for k in range(N + 1):
            seg_off.append(sum(1 for t in rows if (cls[t], slot[t]) < (c, k)))
    dec = []
    for k in range(N):
        mine = [p for p, t in enumerate(perm) if cls[t] == 0 and slot[t] == k]
        for b in range(0, len(mine), group):
            dec.append([k, mine[b], mine[min(b + group, len(mine)) - 1] + 1, 0])
    starts = np.concatenate([[0], np.cumsum(lens)])
    tcs = []
    seen = []
    for t in perm:
        if cls[t] == 1 and seq[t] not in seen:
            seen.append(seq[t])
    for s in seen:
        for b in range(starts[s], starts[s + 1], tile):
            tcs.append([ids[s], b, min(b + tile, starts[s + 1]), s])
    ndec = sum(1 for t in rows if cls[t] == 0)
    return {"status": 0, "slot": slot, "perm": perm, "seg_off": seg_off, "dec_work": dec,
            "tc_work": tcs, "counts": [len(rows), ndec, len(dec), len(tcs)]}


def _check_meta(oracle_mod, ids, lens, T, N, tcq=TC_MIN_QLEN, tile=TILE_ROWS, group=GROUP_ROWS):
    got = oracle_mod.segments(ids, lens, T, N, tcq, tile, group)
    exp = _brute_metadata(ids, lens, T, N, tcq, tile, group)
    assert got["status"] == exp["status"]
    if exp["status"] != 0:
        assert got["counts"].tolist() == [0, 0, 0, 0]
        return got
    assert got["slot"].tolist() == list(exp["slot"])
    assert got["perm"].tolist() == list(exp["perm"])
    assert got["seg_off"].tolist() == exp["seg_off"]
    assert got["dec_work"].tolist() == exp["dec_work"]
    assert got["tc_work"].tolist() == [list(map(int, w)) for w in exp["tc_work"]]
    assert got["counts"].tolist() == exp["counts"]
    return got


@pytest.mark.parametrize("seed", range(12))
def test_metadata_against_brute_force_random(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 40))
    N = int(rng.integers(1, 12))
    lens = rng.choice([0, 1, 1, 1, 2, 63, 64, 65, 127, 128, 129, 300], size=S)
    ids = rng.integers(0, N, size=S)
    _check_meta(oracle_mod, ids, lens, int(lens.sum()), N)


def test_metadata_closed_forms(oracle_mod):
    # All base: nothing active.
    g = _check_meta(oracle_mod, [0, 0, 0], [5, 1, 70], 76, 4)
    assert g["counts"].tolist() == [0, 0, 0, 0]
    # One adapter over all rows, all decode: one slot segment equal to rows 0..T-1.
    g = _check_meta(oracle_mod, [2] * 20, [1] * 20, 20, 4)
    assert g["perm"].tolist() == list(range(20))
    assert g["dec_work"].tolist() == [[2, 0, 8, 0], [2, 8, 16, 0], [2, 16, 20, 0]]
    # One long sequence: ragged tiles of 128.
    g = _check_meta(oracle_mod, [3], [300], 300, 4)
    assert g["tc_work"].tolist() == [[3, 0, 128, 0], [3, 128, 256, 0], [3, 256, 300, 0]]
    # Empty step.
    g = _check_meta(oracle_mod, [], [], 0, 4)
    assert g["counts"].tolist() == [0, 0, 0, 0]


def test_metadata_validation_status(oracle_mod):
    assert _check_meta(oracle_mod, [1, 5], [1, 1], 2, 4)["status"] == -3      # id >= N
    assert _check_meta(oracle_mod, [1, -1], [1, 1], 2, 4)["status"] == -3     # negative id
    assert _check_meta(oracle_mod, [1, 1], [1, -1], 0, 4)["status"] == -6     # negative length
    assert _check_meta(oracle_mod, [1, 1], [1, 1], 3, 4)["status"] == -6      # sum != T
    assert _check_meta(oracle_mod, [9, 1], [1, 1], 3, 4)["status"] == -6      # both: length wins


def test_workload_configs_metadata(oracle_mod):
    for name in W.CONFIG_NAMES:
        wl = W.make_workload(name, draw_xy=False)
        _check_meta(oracle_mod, wl.adapter_ids, wl.q_seq_lens, wl.T, wl.num_slots)


# ------------------------------------------------------------------ MoE layers

def test_moe_slot_follows_the_documented_rule():
    # adapter k (1..A) of expert e sits in slot 1 + e * A + (k - 1); adapter 0 is the base model
    import oracle
    assert oracle.moe_slot(0, 1, 8) == 1
    assert oracle.moe_slot(3, 2, 8) == 26
    assert oracle.moe_slot(127, 8, 8) == 1024
    assert oracle.moe_slot(5, 0, 8) == 0


def test_moe_runs_hand_example():
    # rows grouped by expert; a run is a maximal stretch of equal (expert, sequence, adapter)
    import oracle
    e = [0, 0, 0, 1, 1, 2, 2]
    s = [5, 5, 6, 5, 5, 6, 7]
    a = [1, 1, 2, 1, 1, 0, 0]
    ids, lens = oracle.moe_runs(e, a, s, 3, 8)
    assert ids.tolist() == [1, 2, 9, 0, 0]
    assert lens.tolist() == [2, 1, 2, 1, 1]
    # an expert id out of range gets slot 1 + E * A (outside the pool)
    ids, _ = oracle.moe_runs([0, 3], [1, 1], [0, 0], 3, 8)
    assert ids.tolist() == [1, 25]


def test_moe_delta_brute_force(oracle_mod):
    # the oracle's slot view of an MoE projection against the delta written out
    # per dispatched row: y0 + scale * B[e][a] @ (A[e][a] @ x)
    from adapter_gemv_lora_gb300 import workloads as W
    wl = W.moe_workload("t", [3, 1, 2], [1, 0, 2], num_experts=4, num_adapters=2, top_k=2, d_model=64,
                        d_expert=64, rank_per_adapter=[3, 5], seed=4)
    for mp in wl.projections:
        ids, lens = oracle_mod.moe_runs(wl.row_expert, wl.row_adapter, wl.row_seq, 4, 2)
        slot = np.repeat(ids, lens)
        _, d = oracle_mod.delta(oracle_mod.moe_projection(mp, 4, 2), slot)
        xf = W.bf16_bits_to_f32(mp.x).astype(np.float64)
        off = np.concatenate([[0], np.cumsum(mp.lane_d_out)])
        for r in range(wl.R):
            e, a = int(wl.row_expert[r]), int(wl.row_adapter[r])
            for l in range(mp.num_lanes):
                ref = np.zeros(mp.lane_d_out[l])
                if a > 0:
                    Af = W.bf16_bits_to_f32(mp.A[e][a][l]).astype(np.float64)
                    Bf = W.bf16_bits_to_f32(mp.B[e][a][l]).astype(np.float64)
                    ref = float(mp.scale[a, l]) * (Bf @ (Af @ xf[r]))
                np.testing.assert_allclose(d[r, off[l]:off[l + 1]], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ base projection
# The fused form writes x @ W^T + delta (the delta is added to the projection's
# fp32 partial sum: TensorFold PR #47, the paragraph on the delta).


def test_base_product_permutation_slice_is_a_gather(oracle_mod):
    # W[c][j] = 1 iff j == pi(c): the product picks x[t][pi(c)] exactly.
    rng = np.random.default_rng(5)
    d_in, D, T = 96, 64, 7
    pi = rng.permutation(d_in)[:D]
    w = np.zeros((D, d_in), dtype=np.float32)
    w[np.arange(D), pi] = 1.0
    x = W.bf16_bits(rng.standard_normal((T, d_in)).astype(np.float32))
    base, mag = oracle_mod.base_product(W.bf16_bits(w), x)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    assert np.array_equal(base, xf[:, pi])
    assert np.array_equal(mag, np.abs(xf[:, pi]))
    # reading W transposed (column c of W as the weights of output c) gathers
    # x[t][j] at the j whose pi(j) == c instead: a different matrix here
    wt_gather = np.zeros((T, D))
    for c in range(D):
        hit = np.nonzero(pi == c)[0]
        if hit.size:
            wt_gather[:, c] = xf[:, hit[0]]
    assert not np.array_equal(base, wt_gather)


def test_base_product_against_exact_rationals(oracle_mod):
    rng = np.random.default_rng(11)
    d_in, D, T = 40, 24, 5
    w = rng.standard_normal((D, d_in)).astype(np.float32)
    x = rng.standard_normal((T, d_in)).astype(np.float32)
    wb, xb = W.bf16_bits(w), W.bf16_bits(x)
    base, mag = oracle_mod.base_product(wb, xb, rows=[4, 0, 2])
    wf = W.bf16_bits_to_f32(wb)
    xf = W.bf16_bits_to_f32(xb)
    for q, t in enumerate([4, 0, 2]):
        for c in range(D):
            terms = [Fraction(float(wf[c, j])) * Fraction(float(xf[t, j])) for j in range(d_in)]
            exact = sum(terms)
            amag = sum(abs(v) for v in terms)
            assert abs(base[q, c] - float(exact)) <= 1e-14 * float(amag)
            assert abs(mag[q, c] - float(amag)) <= 1e-14 * float(amag)


def test_fused_projection_closed_form(oracle_mod):
    # W a permutation slice and a rank-1 adapter A = e_i, B = e_j with scale s:
    # y[t][c] = x[t][pi(c)] + s * x[t][i] * [c == j] for adapter rows, and
    # x[t][pi(c)] alone for base rows (y0 plays no part).
    d_in, d_out, T = 64, 64, 6
    i, j, s = 9, 40, -1.5
    proj = _rank1_projection(d_in, d_out, i, j, s, T, seed=2)
    pi = np.roll(np.arange(d_in), 7)[:d_out]
    w = np.zeros((d_out, d_in), dtype=np.float32)
    w[np.arange(d_out), pi] = 1.0
    slot = np.array([1, 0, 1, 1, 0, 1], dtype=np.int32)
    y, dl, _ = oracle_mod.fused_projection(proj, W.bf16_bits(w), slot)
    xf = W.bf16_bits_to_f32(proj.x).astype(np.float64)
    expect = xf[:, pi].copy()
    expect[slot == 1, j] += s * xf[slot == 1, i]
    assert np.array_equal(y, expect)
    assert np.all(dl[slot == 0] == 0)


def test_projection_weight_is_seeded_and_shaped():
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    w1 = W.projection_weight(proj)
    w2 = W.projection_weight(proj)
    assert w1.shape == (proj.D, proj.d_in) and w1.dtype == np.uint16
    assert np.array_equal(w1, w2)
    wf = W.bf16_bits_to_f32(w1)
    assert abs(float(wf.std()) * np.sqrt(proj.d_in) - 1.0) < 0.05
