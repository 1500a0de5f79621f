"""The delta on the GPU against the oracle, the closed forms and the
batch-invariance properties.  Tolerance on the delta: |gpu - oracle| <=
1e-3 + 1e-2 * |oracle| per element; untouched rows and invariances are
bit-exact."""
import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W
import lora_testlib as TL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from adapter_gemv_lora_gb300 import build
    build.build()


def _oracle_check(oracle_mod, wl, proj, rows=None, x=None, y0=None, what=""):
    x = proj.x if x is None else x
    y0 = proj.y0 if y0 is None else y0
    slot = wl.per_token_slot()
    y = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens, x=x, y0=y0)
    if rows is None:
        rows = np.arange(wl.T)
    _, dref = oracle_mod.delta(proj, slot, rows=rows, x=x, y0=y0)
    TL.assert_delta_close(y[rows], y0[rows], dref, what or wl.name)
    TL.assert_rows_untouched(y, y0, np.nonzero(slot == 0)[0])
    return y


def _mixed_workload(seed=0, lanes=(256, 128), ranks=(16, 32, 8, 24)):
    # decode rows, short and long prefill chunks (ragged tiles), base rows,
    # heterogeneous ranks including ranks that are not multiples of 16
    lens = [300, 1, 1, 64, 129, 5, 200, 63, 1, 1, 256, 2]
    ids = [1, 2, 0, 3, 4, 1, 2, 4, 3, 0, 0, 1]
    N, L = 5, len(lanes)
    rank = np.zeros((N, L), dtype=np.int32)
    for k in range(1, N):
        rank[k, :] = ranks[(k - 1) % len(ranks)]
    return W.custom_workload(lens, ids, d_in=512, lane_d_out=list(lanes), num_slots=N, max_rank=32,
                             rank=rank, seed=seed)


def test_mixed_small_full_oracle(oracle_mod):
    wl = _mixed_workload()
    _oracle_check(oracle_mod, wl, wl.projections[0], what="mixed")


def test_pool_reused_across_steps(oracle_mod):
    # one pool, several steps with different batches: the per-tile and
    # work-item counters the kernels keep in the pool's scratch must be back
    # at zero after every step, so each step matches the oracle and a repeated
    # step repeats its bits
    from adapter_gemv_lora_gb300 import lora_delta as LD  # noqa: F401
    base = _mixed_workload(seed=11)
    proj = base.projections[0]
    pool = TL.build_pool(proj, base.T)
    rng = np.random.default_rng(5)
    first = None
    for step in range(4):
        lens = rng.choice([1, 1, 2, 64, 70, 129, 300], size=int(rng.integers(3, 10)))
        lens = lens[np.cumsum(lens) <= base.T]  # the rows must fit the workload's x and y0
        ids = rng.integers(0, base.num_slots, size=len(lens))
        T = int(lens.sum())
        x, y0 = proj.x[:T], proj.y0[:T]
        slot = np.repeat(ids, lens)
        y = TL.run_gpu(proj, ids, lens, x=x, y0=y0, pool=pool)
        _, dref = oracle_mod.delta(proj, slot, rows=np.arange(T), x=x, y0=y0)
        TL.assert_delta_close(y, y0, dref, f"step {step}")
        if first is None:
            first = (ids, lens, y)
    ids, lens, y_first = first
    T = int(lens.sum())
    y_again = TL.run_gpu(proj, ids, lens, x=proj.x[:T], y0=proj.y0[:T], pool=pool)
    assert np.array_equal(y_again.view(np.uint32), y_first.view(np.uint32))


def test_graph_capture_matches_eager():
    # build + apply captured in a CUDA graph (the apply forks its decode
    # kernels onto the library's side stream and joins them back) replays to
    # the same bits as the eager calls
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _mixed_workload(seed=3)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, wl.T)
    seg = LD.LoraSegments(wl.S, wl.T, wl.num_slots, device="cuda")
    ids = torch.tensor(wl.adapter_ids, dtype=torch.int32, device="cuda")
    lens = torch.tensor(wl.q_seq_lens, dtype=torch.int32, device="cuda")
    x = TL.to_dev_u16(proj.x, "cuda")
    y0 = torch.from_numpy(proj.y0).cuda()
    y = y0.clone()

    def step():
        seg.build(ids, lens, num_tokens=wl.T)
        LD.apply(pool, seg, x, y)

    step()
    torch.cuda.synchronize()
    y_eager = y.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y.copy_(y0)
        with torch.cuda.graph(g):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        y.copy_(y0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_eager.view(torch.int32))
    assert seg.status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes_full_oracle(oracle_mod, seed):
    # random d_in, lane count and widths, rank bounds (including ranks that are
    # not multiples of 16 and zero lanes), slot counts and length mixes around
    # the path threshold and the tile size; every row against the oracle
    rng = np.random.default_rng(1000 + seed)
    d_in = int(rng.choice([64, 128, 640, 1024, 2112, 4096]))
    L = int(rng.integers(1, 5))
    lanes = [int(64 * rng.integers(1, 17)) for _ in range(L)]
    max_rank = int(rng.choice([1, 7, 16, 33, 64, 100, 128]))
    N = int(rng.integers(2, 13))
    S = int(rng.integers(1, 40))
    lens = rng.choice([0, 1, 1, 1, 2, 7, 63, 64, 65, 127, 128, 129, 300], size=S)
    while lens.sum() == 0:
        lens = rng.choice([1, 64, 129], size=S)
    ids = rng.integers(0, N, size=S)
    rank = rng.integers(0, max_rank + 1, size=(N, L)).astype(np.int32)
    rank[0] = 0
    rank[rng.random((N, L)) < 0.15] = 0
    wl = W.custom_workload(lens, ids, d_in=d_in, lane_d_out=lanes, num_slots=N, max_rank=max_rank, rank=rank,
                           seed=seed)
    _oracle_check(oracle_mod, wl, wl.projections[0], what=f"seed {seed}: d_in {d_in} lanes {lanes} R {max_rank}")


def test_one_graph_serves_any_adapter_mixture(oracle_mod):
    # captured once for a (num_seqs, num_tokens) shape, the step replays for
    # other adapter ids and other length splits of the same totals: the work
    # lists live in device memory and the grids are sized by capacity
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _mixed_workload(seed=6)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, wl.T)
    seg = LD.LoraSegments(wl.S, wl.T, wl.num_slots, device="cuda")
    ids = torch.tensor(wl.adapter_ids, dtype=torch.int32, device="cuda")
    lens = torch.tensor(wl.q_seq_lens, dtype=torch.int32, device="cuda")
    x = TL.to_dev_u16(proj.x, "cuda")
    y0 = torch.from_numpy(proj.y0).cuda()
    y = y0.clone()
    g = torch.cuda.CUDAGraph()
    s_ = torch.cuda.Stream()
    s_.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_):
        seg.build(ids, lens, num_tokens=wl.T)  # one eager step before capture
        LD.apply(pool, seg, x, y)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            seg.build(ids, lens, num_tokens=wl.T)
            LD.apply(pool, seg, x, y)
    torch.cuda.current_stream().wait_stream(s_)
    rng = np.random.default_rng(9)
    for mix in range(3):
        new_ids = rng.integers(0, wl.num_slots, size=wl.S).astype(np.int32)
        cut = np.sort(rng.choice(np.arange(1, wl.T), size=wl.S - 1, replace=False))
        new_lens = np.diff(np.concatenate([[0], cut, [wl.T]])).astype(np.int32)
        ids.copy_(torch.from_numpy(new_ids))
        lens.copy_(torch.from_numpy(new_lens))
        y.copy_(y0)
        g.replay()
        torch.cuda.synchronize()
        assert seg.status() == 0
        slot = np.repeat(new_ids, new_lens)
        _, dref = oracle_mod.delta(proj, slot)
        got = y.cpu().numpy()
        TL.assert_delta_close(got, proj.y0, dref, f"mixture {mix}")
        TL.assert_rows_untouched(got, proj.y0, np.nonzero(slot == 0)[0])


@pytest.mark.parametrize("shards", [2, 4])
def test_row_parallel_shards_sum_to_the_delta(oracle_mod, shards):
    # row-parallel layers (o_proj, down) under tensor parallelism cut A by
    # columns: rank p holds A[:, cols_p] and x[:, cols_p] and adds
    # scale * B @ (A_p @ x_p) into its partial sum, which the base's reduction
    # adds up.  Each shard is an ordinary pool of d_in / shards; summing the
    # shards' deltas on the host gives the full delta
    import torch
    base = _mixed_workload(seed=8, lanes=(256,))
    proj = base.projections[0]
    d_in = proj.d_in
    part = d_in // shards
    total = np.zeros_like(proj.y0, dtype=np.float64)
    for sh in range(shards):
        cols = slice(sh * part, (sh + 1) * part)
        wl_p = W.custom_workload(base.q_seq_lens, base.adapter_ids, d_in=part, lane_d_out=[256],
                                 num_slots=base.num_slots, max_rank=32, rank=proj.rank, seed=0)
        pp = wl_p.projections[0]
        for k in range(1, base.num_slots):
            if proj.rank[k, 0] > 0:
                pp.A[k][0] = np.ascontiguousarray(proj.A[k][0][:, cols])
                pp.B[k][0] = proj.B[k][0]
        pp.scale[:] = proj.scale
        zeros = np.zeros_like(proj.y0)
        y = TL.run_gpu(pp, base.adapter_ids, base.q_seq_lens, x=np.ascontiguousarray(proj.x[:, cols]), y0=zeros)
        total += y.astype(np.float64)
    _, dref = oracle_mod.delta(proj, base.per_token_slot())
    TL.assert_delta_close((proj.y0.astype(np.float64) + total).astype(np.float32), proj.y0, dref,
                          f"{shards} row-parallel shards")


def test_maximum_slot_count(oracle_mod):
    # a pool of LORA_MAX_SLOTS slots with adapters spread over the id range,
    # up to the last slot, on both paths
    N = 2048
    lens = [1, 70, 1, 1, 130, 2, 1, 64]
    ids = [2047, 1024, 1, 0, 2046, 3, 1500, 2047]
    rank = np.zeros((N, 1), dtype=np.int32)
    for k in set(ids) - {0}:
        rank[k, 0] = 4 + (k % 13)
    wl = W.custom_workload(lens, ids, d_in=128, lane_d_out=[64], num_slots=N, max_rank=16, rank=rank, seed=21)
    _oracle_check(oracle_mod, wl, wl.projections[0], what="2048 slots")


@pytest.mark.parametrize("d_in", [64, 192, 1088])
def test_k_block_counts(oracle_mod, d_in):
    # d_in of 1, 3 and 17 blocks of 64: the tensor shrink's two K ranges are
    # empty / uneven, and 1088 also spans two decode K chunks of 1024
    lens = [130, 1, 64, 3, 1, 77]
    ids = [1, 2, 2, 1, 0, 3]
    N = 4
    rank = np.array([[0], [16], [40], [7]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=d_in, lane_d_out=[192], num_slots=N, max_rank=48, rank=rank,
                           seed=d_in)
    _oracle_check(oracle_mod, wl, wl.projections[0], what=f"d_in={d_in}")


@pytest.mark.parametrize("lanes", [[256], [128, 64]])
def test_decode_rank_geometry(oracle_mod, lanes):
    # the decode shrink cuts a slot's rank rows into blocks of up to 32 and each
    # block into groups of 4 (their count rounded up to a power of two) and
    # deals the K blocks to 128 / groups splits: one slot per geometry, ranks
    # 1..128 with 4-row tails past a 32-row block, decode rows in groups of 1 to
    # 8 rows, and a ragged last K chunk (2112 = 2 x 1024 + 64); every row
    # against the oracle
    ranks = [1, 3, 4, 5, 8, 9, 12, 16, 17, 20, 31, 32, 33, 36, 48, 64, 65, 96, 100, 127, 128]
    N = len(ranks) + 1
    L = len(lanes)
    rank = np.zeros((N, L), dtype=np.int32)
    for k, r in enumerate(ranks, start=1):
        rank[k, :] = r
        if L > 1:
            rank[k, 1] = ranks[(k * 7) % len(ranks)]
    lens, ids = [], []
    for k in range(1, N):
        for _ in range(1 + (k * 3) % 8):  # 1..8 single-token rows of slot k
            lens.append(1)
            ids.append(k)
    lens += [1, 1, 5, 2]
    ids += [0, 3, 7, 0]
    wl = W.custom_workload(lens, ids, d_in=2112, lane_d_out=lanes, num_slots=N, max_rank=128, rank=rank, seed=77)
    _oracle_check(oracle_mod, wl, wl.projections[0], what=f"rank geometry, lanes {lanes}")


@pytest.mark.parametrize("name", ["tiny", "decode_oproj"])
def test_decode_configs_full(oracle_mod, name):
    wl = W.make_workload(name)
    _oracle_check(oracle_mod, wl, wl.projections[0])


def test_mlp_decode_full(oracle_mod):
    wl = W.make_workload("mlp_decode")
    for proj in wl.projections:
        _oracle_check(oracle_mod, wl, proj, what=proj.name)


@pytest.mark.parametrize("name", ["prefill_qkv", "cont_batch"])
def test_large_configs_full(oracle_mod, name):
    # every row of the step against the oracle (the oracle runs on all host cores)
    wl = W.make_workload(name)
    for proj in wl.projections:
        _oracle_check(oracle_mod, wl, proj, what=f"{name} {proj.name}")


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_config_batch_mix_invariance(name):
    # At each configuration's own shape: the kept sequences' rows keep their
    # bits when the batch around them changes (other sequences, another order,
    # foreign slots and lengths), the pool is padded to another max_rank and
    # every adapter sits under another slot label.
    wl = W.make_workload(name)
    rng = np.random.default_rng(sum(map(ord, name)))
    ids, lens, pieces = TL.remix_batch(wl, rng)
    N = wl.num_slots
    n2 = min(2 * N, 2048)
    labels = rng.permutation(np.arange(1, n2))[:N - 1]
    relabel = {k: int(labels[k - 1]) for k in range(1, N)}
    new_ids = np.array([relabel.get(int(k), 0) for k in ids], dtype=np.int32)
    starts = np.concatenate([[0], np.cumsum(wl.q_seq_lens)])
    for proj in wl.projections:
        y_full = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens)
        xs, ys = [], []
        for s, ln in zip(pieces, lens):
            if s is None:
                xs.append(W.bf16_bits(rng.standard_normal((ln, proj.d_in)).astype(np.float32)))
                ys.append(rng.standard_normal((ln, proj.D)).astype(np.float32))
            else:
                xs.append(proj.x[starts[s]:starts[s + 1]])
                ys.append(proj.y0[starts[s]:starts[s + 1]])
        x, y0 = np.concatenate(xs), np.concatenate(ys)
        pad = 128 if proj.max_rank < 128 else proj.max_rank
        pool = TL.build_pool(proj, x.shape[0], max_rank=pad, slot_map=relabel)
        y = TL.run_gpu(proj, new_ids, lens, x=x, y0=y0, pool=pool)
        at = 0
        for s, ln in zip(pieces, lens):
            if s is not None:
                a = np.ascontiguousarray(y[at:at + ln]).view(np.uint32)
                b = np.ascontiguousarray(y_full[starts[s]:starts[s + 1]]).view(np.uint32)
                assert np.array_equal(a, b), f"{name} {proj.name}: sequence {s} changed bits"
            at += ln


def test_fused_qkv_rank128(oracle_mod):
    # three lanes at rank up to 128: 384 rank columns of tensor memory per tile
    lens = [1, 200, 1, 3, 129, 64, 1, 2]
    ids = [1, 2, 0, 3, 4, 1, 4, 2]
    N = 5
    rank = np.array([[0, 0, 0], [128, 128, 128], [100, 64, 17], [1, 128, 33], [128, 0, 96]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=1024, lane_d_out=[512, 128, 128], num_slots=N, max_rank=128,
                           rank=rank, seed=31)
    _oracle_check(oracle_mod, wl, wl.projections[0], what="fused qkv rank 128")


def test_sentinels_in_base_rows_are_not_read_or_written(oracle_mod):
    wl = _mixed_workload(seed=3)
    proj = wl.projections[0]
    slot = wl.per_token_slot()
    x = proj.x.copy()
    y0 = proj.y0.copy()
    base = slot == 0
    x[base] = TL.SENTINEL_X_BITS
    y0.view(np.uint32)[base] = TL.SENTINEL_NAN_BITS
    y = _oracle_check(oracle_mod, wl, proj, rows=np.nonzero(~base)[0], x=x, y0=y0)
    assert np.all(y.view(np.uint32)[base] == TL.SENTINEL_NAN_BITS)


def test_rank_zero_lane_is_not_written():
    lens, ids = [1, 1, 200, 1], [1, 2, 1, 2]
    rank = np.array([[0, 0, 0], [16, 0, 16], [0, 16, 0]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=256, lane_d_out=[128, 64, 64], num_slots=3, max_rank=16, rank=rank)
    proj = wl.projections[0]
    y = TL.run_gpu(proj, ids, lens)
    slot = wl.per_token_slot()
    off = [0, 128, 192, 256]
    for t in range(wl.T):
        for l in range(3):
            a = y[t, off[l]:off[l + 1]].view(np.uint32)
            b = proj.y0[t, off[l]:off[l + 1]].view(np.uint32)
            assert np.array_equal(a, b) == (rank[slot[t], l] == 0)


def test_scale_zero_leaves_y_bit_identical():
    wl = _mixed_workload(seed=4)
    proj = wl.projections[0]
    proj.scale[:] = 0.0
    y = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens)
    assert np.array_equal(y.view(np.uint32), proj.y0.view(np.uint32))


@pytest.mark.parametrize("qlen", [1, 200])
def test_rank1_unit_vectors_closed_form(qlen):
    # A = e_i^T, B = e_j, scale 2 (a power of two): y[t][j] = fl(y0 + 2 * x[t][i]) exactly.
    d_in, d_out, i, j = 256, 128, 77, 5
    wl = W.custom_workload([qlen, qlen], [1, 0], d_in=d_in, lane_d_out=[d_out], num_slots=2, max_rank=16,
                           rank=np.array([[0], [1]]), alpha=np.array([[0.0], [2.0]]))
    proj = wl.projections[0]
    a = np.zeros((1, d_in), dtype=np.float32)
    a[0, i] = 1
    b = np.zeros((d_out, 1), dtype=np.float32)
    b[j, 0] = 1
    proj.A[1][0], proj.B[1][0] = W.bf16_bits(a), W.bf16_bits(b)
    y = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens)
    xf = W.bf16_bits_to_f32(proj.x)
    exp = proj.y0.copy()
    exp[:qlen, j] = proj.y0[:qlen, j] + np.float32(2.0) * xf[:qlen, i]
    assert np.array_equal(y.view(np.uint32), exp.view(np.uint32))


def test_linearity_doubling_x_doubles_y_from_zero():
    wl = _mixed_workload(seed=5)
    proj = wl.projections[0]
    y0 = np.zeros_like(proj.y0)
    y1 = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens, y0=y0)
    x2 = W.bf16_bits(2.0 * W.bf16_bits_to_f32(proj.x))
    y2 = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens, x=x2, y0=y0)
    assert np.array_equal(y2, 2.0 * y1)


def _seq_rows(lens):
    starts = np.concatenate([[0], np.cumsum(lens)])
    return [np.arange(starts[s], starts[s + 1]) for s in range(len(lens))]


def test_batch_composition_invariance():
    # The same sequences (x rows, slot, own length) inside different batches
    # give bit-identical rows.
    base = _mixed_workload(seed=6)
    proj = base.projections[0]
    lens, ids = list(base.q_seq_lens), list(base.adapter_ids)
    y_full = TL.run_gpu(proj, ids, lens)
    rows = _seq_rows(lens)
    rng = np.random.default_rng(0)
    for trial in range(3):
        keep = sorted(rng.choice(len(lens), size=6, replace=False).tolist())
        # add foreign sequences with other slots between them
        extra_lens = [1, 70, 1]
        extra_ids = [4, 3, 2]
        new_lens, new_ids, xs, ys, where = [], [], [], [], []
        rng2 = np.random.default_rng(trial)
        for n, s in enumerate(keep):
            if n == 1:
                for el, ei in zip(extra_lens, extra_ids):
                    new_lens.append(el)
                    new_ids.append(ei)
                    xs.append(W.bf16_bits(rng2.standard_normal((el, proj.d_in)).astype(np.float32)))
                    ys.append(rng2.standard_normal((el, proj.D)).astype(np.float32))
                    where.append(None)
            new_lens.append(lens[s])
            new_ids.append(ids[s])
            xs.append(proj.x[rows[s]])
            ys.append(proj.y0[rows[s]])
            where.append(s)
        x = np.concatenate(xs)
        y0 = np.concatenate(ys)
        y = TL.run_gpu(proj, new_ids, new_lens, x=x, y0=y0, pool=TL.build_pool(proj, x.shape[0]))
        for r, s in zip(_seq_rows(new_lens), where):
            if s is not None:
                assert np.array_equal(y[r].view(np.uint32), y_full[rows[s]].view(np.uint32)), (trial, s)


def test_padding_and_slot_relabel_invariance():
    wl = _mixed_workload(seed=7)
    proj = wl.projections[0]
    ids, lens = wl.adapter_ids, wl.q_seq_lens
    y_a = TL.run_gpu(proj, ids, lens)
    pool_b = TL.build_pool(proj, wl.T, max_rank=128)              # wider padding, same adapters
    y_b = TL.run_gpu(proj, ids, lens, pool=pool_b)
    assert np.array_equal(y_a.view(np.uint32), y_b.view(np.uint32))
    relabel = {1: 7, 2: 3, 3: 5, 4: 1}
    pool_c = TL.build_pool(proj, wl.T, slot_map=relabel)
    ids_c = np.array([relabel.get(int(k), 0) for k in ids], dtype=np.int32)
    y_c = TL.run_gpu(proj, ids_c, lens, pool=pool_c)
    assert np.array_equal(y_a.view(np.uint32), y_c.view(np.uint32))


def test_fused_lanes_equal_single_lane_pools(oracle_mod):
    wl = _mixed_workload(seed=8, lanes=(256, 128, 128))
    proj = wl.projections[0]
    y = TL.run_gpu(proj, wl.adapter_ids, wl.q_seq_lens)
    off = [0, 256, 384, 512]
    for l in range(3):
        single = W.Projection("lane", proj.d_in, [proj.lane_d_out[l]], proj.rank[:, l:l + 1].copy(),
                              proj.scale[:, l:l + 1].copy(),
                              [[proj.A[k][l]] for k in range(proj.rank.shape[0])],
                              [[proj.B[k][l]] for k in range(proj.rank.shape[0])],
                              proj.x, np.ascontiguousarray(proj.y0[:, off[l]:off[l + 1]]), proj.max_rank)
        ys = TL.run_gpu(single, wl.adapter_ids, wl.q_seq_lens)
        assert np.array_equal(ys.view(np.uint32), np.ascontiguousarray(y[:, off[l]:off[l + 1]]).view(np.uint32))


def test_empty_and_all_base_batches():
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _mixed_workload(seed=9)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, 1024)
    seg = LD.LoraSegments(16, 1024, pool.num_slots)
    x = torch.zeros((4, proj.d_in), dtype=torch.int16, device="cuda")
    y = torch.randn((4, proj.D), device="cuda")
    y_before = y.clone()
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    n0 = LD.lora_launch_count()
    seg.build(empty, empty, num_tokens=0)
    LD.apply(pool, seg, x, y)
    torch.cuda.synchronize()
    assert LD.lora_launch_count() == n0          # an empty step launches nothing
    assert seg.status() == 0
    seg.build(torch.zeros(2, dtype=torch.int32, device="cuda"),
              torch.tensor([3, 1], dtype=torch.int32, device="cuda"))
    LD.apply(pool, seg, x, y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y_before.view(torch.int32))
    # a pool with no loaded adapter launches nothing
    empty_pool = LD.LoraPool(pool.num_slots, 16, proj.d_in, proj.lane_d_out, 1024)
    seg.build(torch.tensor([1, 2], dtype=torch.int32, device="cuda"),
              torch.tensor([3, 1], dtype=torch.int32, device="cuda"))
    n1 = LD.lora_launch_count()
    LD.apply(empty_pool, seg, x, y)
    torch.cuda.synchronize()
    assert LD.lora_launch_count() == n1
    assert torch.equal(y.view(torch.int32), y_before.view(torch.int32))


def test_bad_metadata_makes_apply_a_noop():
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _mixed_workload(seed=10)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, 64)
    seg = LD.LoraSegments(8, 64, pool.num_slots)
    x = TL.to_dev_u16(proj.x[:4])
    y = torch.randn((4, proj.D), device="cuda")
    y_before = y.clone()
    seg.build(torch.tensor([1, 9], dtype=torch.int32, device="cuda"),
              torch.tensor([2, 2], dtype=torch.int32, device="cuda"))
    LD.apply(pool, seg, x, y)
    torch.cuda.synchronize()
    assert seg.status() == LD.LORA_ERR_SLOT
    assert torch.equal(y.view(torch.int32), y_before.view(torch.int32))
    seg.build(torch.tensor([1, 1], dtype=torch.int32, device="cuda"),
              torch.tensor([2, 3], dtype=torch.int32, device="cuda"), num_tokens=4)
    LD.apply(pool, seg, x, y)
    torch.cuda.synchronize()
    assert seg.status() == LD.LORA_ERR_META
    assert torch.equal(y.view(torch.int32), y_before.view(torch.int32))


def test_host_argument_checks():
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _mixed_workload(seed=11)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, 64)
    seg = TL.build_segments([1], [4], pool.num_slots, max_tokens=64)
    x = torch.zeros((4, proj.d_in), dtype=torch.int16, device="cuda")
    y = torch.zeros((4, proj.D), device="cuda")
    with pytest.raises(LD.LoraError):       # ldx below d_in
        LD.lora_apply_shrink_expand(pool.handle, seg.handle, x.data_ptr(), y.data_ptr(), 8, proj.D)
    with pytest.raises(LD.LoraError):       # misaligned y
        LD.lora_apply_shrink_expand(pool.handle, seg.handle, x.data_ptr(), y.data_ptr() + 4, proj.d_in, proj.D)
    with pytest.raises(LD.LoraError):       # slot 0 cannot be loaded
        LD.lora_pool_load(pool.handle, 0, 0, 4, 1.0, x.data_ptr(), x.data_ptr())
    with pytest.raises(LD.LoraError):       # rank above max_rank
        LD.lora_pool_load(pool.handle, 1, 0, 64, 1.0, x.data_ptr(), x.data_ptr())
