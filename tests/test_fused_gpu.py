"""The fused projection (y = x @ W^T + delta, one GEMM whose accumulator also
takes the expand) on the GPU against the oracle's fp64 base product and delta.

Tolerances, from the arithmetic:
  * base: an fp32 sum of d_in exact bf16 products, each addition off by at most
    one unit in the last place of the running sum, so
    |gpu - base| <= d_in * 2^-23 * sum_j |x_j W_cj|;
  * delta: the fused output minus the same rows' output with every row on the
    base model (computed by the same kernel) against the oracle's delta, within
    1e-3 + 1e-2 * |delta| plus two fp32 roundings of the outputs;
  * slot-0 rows, and every row under batch changes: bit-exact.
"""
import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W
import lora_testlib as TL

pytestmark = pytest.mark.gpu

MAC_BUDGET = 2e10  # base-product multiply-adds the oracle spends per projection


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from adapter_gemv_lora_gb300 import build
    build.build()


def run_fused(proj, ids, lens, Wb, x=None, pool=None, y_init=None, expect_status=0):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = TL.torch_mod()
    x = proj.x if x is None else x
    T = x.shape[0]
    if pool is None:
        pool = TL.build_pool(proj, max(T, 1))
    seg = TL.build_segments(ids, lens, pool.num_slots)
    xd = TL.to_dev_u16(x)
    wd = TL.to_dev_u16(Wb)
    if y_init is None:
        y_init = np.full((T, proj.D), np.nan, dtype=np.float32)
    yd = torch.from_numpy(np.ascontiguousarray(y_init)).cuda()
    LD.fused_projection(pool, seg, wd, xd, yd)
    torch.cuda.synchronize()
    st = seg.status()
    assert st == expect_status, f"device status {st}: {LD.lora_status_string(st)}"
    return yd.cpu().numpy()


def check_against_oracle(oracle_mod, proj, ids, lens, slot, Wb, pool=None, what=""):
    y_f = run_fused(proj, ids, lens, Wb, pool=pool)
    y_b = run_fused(proj, np.zeros_like(np.asarray(ids)), lens, Wb, pool=pool)
    T = proj.x.shape[0]
    # base product on every row, or on a seeded sample when that is too much work
    n_rows = int(min(T, max(16, MAC_BUDGET // (proj.D * proj.d_in))))
    rows = np.arange(T) if n_rows >= T else np.sort(np.random.default_rng(7).choice(T, n_rows, replace=False))
    base, mag = oracle_mod.base_product(Wb, proj.x, rows=rows)
    err = np.abs(y_b[rows].astype(np.float64) - base)
    bound = proj.d_in * 2.0 ** -23 * mag
    assert np.all(err <= bound), f"{what}: base product off by {float((err - bound).max()):.3g} over its bound"
    # the delta on every row
    _, dref = oracle_mod.delta(proj, slot)
    d_gpu = y_f.astype(np.float64) - y_b.astype(np.float64)
    tol = TL.ATOL + TL.RTOL * np.abs(dref) + 2.0 ** -22 * (np.abs(y_f) + np.abs(y_b))
    bad = np.abs(d_gpu - dref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} delta elements out of tolerance, first {np.argwhere(bad)[:3]}"
    # rows on the base model are exactly the base product
    b0 = np.nonzero(slot == 0)[0]
    assert np.array_equal(y_f[b0].view(np.uint32), y_b[b0].view(np.uint32)), f"{what}: a base row changed"
    return y_f


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_fused_configs_against_oracle(oracle_mod, name):
    wl = W.make_workload(name)
    slot = wl.per_token_slot()
    for i, proj in enumerate(wl.projections):
        Wb = W.projection_weight(proj, seed=1 + i)
        check_against_oracle(oracle_mod, proj, wl.adapter_ids, wl.q_seq_lens, slot, Wb, what=f"{name} {proj.name}")


def test_fused_ragged_tiles_and_lanes_inside_a_tile(oracle_mod):
    # 401 rows (a ragged last row tile), lanes of 192/128/64 columns (column
    # tiles of 256 hold parts of two lanes), rank-0 lanes, every path
    lens = [1, 200, 1, 3, 129, 64, 1, 2]
    ids = [1, 2, 0, 3, 4, 1, 4, 2]
    rank = np.array([[0, 0, 0], [40, 16, 3], [33, 0, 17], [1, 40, 0], [16, 8, 40]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=320, lane_d_out=[192, 128, 64], num_slots=5, max_rank=40,
                           rank=rank, seed=17)
    proj = wl.projections[0]
    check_against_oracle(oracle_mod, proj, ids, lens, wl.per_token_slot(), W.projection_weight(proj, seed=5),
                         what="ragged")


def test_fused_rank128_three_lanes(oracle_mod):
    lens = [1, 200, 1, 3, 129, 64, 1, 2]
    ids = [1, 2, 0, 3, 4, 1, 4, 2]
    rank = np.array([[0, 0, 0], [128, 128, 128], [100, 64, 17], [1, 128, 33], [128, 0, 96]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=1024, lane_d_out=[512, 128, 128], num_slots=5, max_rank=128,
                           rank=rank, seed=31)
    proj = wl.projections[0]
    check_against_oracle(oracle_mod, proj, ids, lens, wl.per_token_slot(), W.projection_weight(proj, seed=6),
                         what="rank 128")


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_fused_batch_mix_invariance(name):
    # the kept sequences' rows keep their bits when the batch around them
    # changes (row tiles of the GEMM then hold other rows and other slots), the
    # pool is padded to another max_rank and the adapters sit under other labels
    wl = W.make_workload(name, draw_xy=True)
    rng = np.random.default_rng(sum(map(ord, name)) + 1)
    ids, lens, pieces = TL.remix_batch(wl, rng)
    N = wl.num_slots
    n2 = min(2 * N, 2048)
    labels = rng.permutation(np.arange(1, n2))[:N - 1]
    relabel = {k: int(labels[k - 1]) for k in range(1, N)}
    new_ids = np.array([relabel.get(int(k), 0) for k in ids], dtype=np.int32)
    starts = np.concatenate([[0], np.cumsum(wl.q_seq_lens)])
    for i, proj in enumerate(wl.projections):
        Wb = W.projection_weight(proj, seed=1 + i)
        y_full = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, Wb)
        xs = []
        for s, ln in zip(pieces, lens):
            if s is None:
                xs.append(W.bf16_bits(rng.standard_normal((ln, proj.d_in)).astype(np.float32)))
            else:
                xs.append(proj.x[starts[s]:starts[s + 1]])
        x = np.concatenate(xs)
        pad = 128 if proj.max_rank < 128 else proj.max_rank
        pool = TL.build_pool(proj, x.shape[0], max_rank=pad, slot_map=relabel)
        y = run_fused(proj, new_ids, lens, Wb, x=x, pool=pool)
        at = 0
        for s, ln in zip(pieces, lens):
            if s is not None:
                a = np.ascontiguousarray(y[at:at + ln]).view(np.uint32)
                b = np.ascontiguousarray(y_full[starts[s]:starts[s + 1]]).view(np.uint32)
                assert np.array_equal(a, b), f"{name} {proj.name}: sequence {s} changed bits"
            at += ln


def test_fused_pair_and_single_cta_forms_agree():
    # a batch of long prompts runs in CTA pairs (tcgen05 pair MMA), a batch of
    # short sequences in single CTAs; the same rows (same x, same adapter, same
    # tensor-path shrink) must come out with the same bits in both
    lens = [600, 500, 330, 170]
    ids = [1, 2, 0, 3]
    rank = np.array([[0, 0], [16, 32], [48, 16], [32, 32]], dtype=np.int32)
    wl = W.custom_workload(lens, ids, d_in=512, lane_d_out=[256, 128], num_slots=4, max_rank=48, rank=rank,
                           seed=5)
    proj = wl.projections[0]
    Wb = W.projection_weight(proj)
    T = wl.T
    y_pair = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, Wb)  # T / S = 400 rows per sequence
    extra = 80  # single-row base sequences: T / S falls under 256
    rng = np.random.default_rng(9)
    x2 = np.concatenate([proj.x, W.bf16_bits(rng.standard_normal((extra, proj.d_in)).astype(np.float32))])
    ids2 = np.concatenate([wl.adapter_ids, np.zeros(extra, np.int32)]).astype(np.int32)
    lens2 = np.concatenate([wl.q_seq_lens, np.ones(extra, np.int32)]).astype(np.int32)
    assert x2.shape[0] < 256 * len(lens2) and T >= 256 * len(lens)
    pool = TL.build_pool(proj, x2.shape[0])
    y_single = run_fused(proj, ids2, lens2, Wb, x=x2, pool=pool)
    assert np.array_equal(y_single[:T].view(np.uint32), y_pair.view(np.uint32))


def test_fused_pool_without_adapters_is_the_base(oracle_mod):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    Wb = W.projection_weight(proj)
    empty = LD.LoraPool(wl.num_slots, proj.max_rank, proj.d_in, proj.lane_d_out, wl.T)
    y = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, Wb, pool=empty)
    y_b = run_fused(proj, np.zeros_like(wl.adapter_ids), wl.q_seq_lens, Wb)
    assert np.array_equal(y.view(np.uint32), y_b.view(np.uint32))
    base, mag = oracle_mod.base_product(Wb, proj.x)
    assert np.all(np.abs(y - base) <= proj.d_in * 2.0 ** -23 * mag)


def test_fused_writes_y_without_reading_it():
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    Wb = W.projection_weight(proj)
    y1 = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, Wb, y_init=np.zeros((wl.T, proj.D), np.float32))
    y2 = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, Wb,
                   y_init=np.random.default_rng(1).standard_normal((wl.T, proj.D)).astype(np.float32))
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_fused_routing_error_writes_nothing():
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    ids = wl.adapter_ids.copy()
    ids[1] = wl.num_slots  # out of range
    y0 = np.zeros((wl.T, proj.D), np.float32)
    y0.view(np.uint32)[:] = TL.SENTINEL_NAN_BITS
    y = run_fused(proj, ids, wl.q_seq_lens, W.projection_weight(proj), y_init=y0, expect_status=LD.LORA_ERR_SLOT)
    assert np.all(y.view(np.uint32) == TL.SENTINEL_NAN_BITS)


@pytest.mark.parametrize("qlen", [1, 200])
def test_fused_rank1_permutation_closed_form(qlen):
    # W a permutation slice, A = e_i^T, B = e_j, scale 2, x with exponents close
    # together: y[t][c] = x[t][pi(c)] + 2 * x[t][i] * [c == j] for adapter rows,
    # exactly (every sum is representable in fp32)
    d_in, d_out, i, j = 256, 128, 77, 5
    wl = W.custom_workload([qlen, qlen], [1, 0], d_in=d_in, lane_d_out=[d_out], num_slots=2, max_rank=16,
                           rank=np.array([[0], [1]]), alpha=np.array([[0.0], [2.0]]))
    proj = wl.projections[0]
    rng = np.random.default_rng(3)
    xv = rng.uniform(0.5, 2.0, size=(2 * qlen, d_in)) * rng.choice([-1.0, 1.0], size=(2 * qlen, d_in))
    proj.x = W.bf16_bits(xv.astype(np.float32))
    a = np.zeros((1, d_in), dtype=np.float32)
    a[0, i] = 1
    b = np.zeros((d_out, 1), dtype=np.float32)
    b[j, 0] = 1
    proj.A[1][0], proj.B[1][0] = W.bf16_bits(a), W.bf16_bits(b)
    pi = np.roll(np.arange(d_in), 11)[:d_out]
    w = np.zeros((d_out, d_in), dtype=np.float32)
    w[np.arange(d_out), pi] = 1.0
    y = run_fused(proj, wl.adapter_ids, wl.q_seq_lens, W.bf16_bits(w))
    xf = W.bf16_bits_to_f32(proj.x).astype(np.float64)
    exp = xf[:, pi].copy()
    exp[:qlen, j] += 2.0 * xf[:qlen, i]
    assert np.array_equal(y.astype(np.float64), exp)


def test_fused_stages_in_order_equal_the_call():
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = TL.torch_mod()
    lens = [1, 200, 1, 3, 129, 64, 1, 2]
    ids = [1, 2, 0, 3, 4, 1, 4, 2]
    wl = W.custom_workload(lens, ids, d_in=512, lane_d_out=[256, 128], num_slots=5, max_rank=32, seed=9)
    proj = wl.projections[0]
    Wb = W.projection_weight(proj)
    y_call = run_fused(proj, ids, lens, Wb)
    pool = TL.build_pool(proj, wl.T)
    seg = TL.build_segments(ids, lens, pool.num_slots)
    xd, wd = TL.to_dev_u16(proj.x), TL.to_dev_u16(Wb)
    yd = torch.full((wl.T, proj.D), float("nan"), device="cuda")
    for stage in (1, 2, 3):
        LD.fused_projection_stage(pool, seg, wd, xd, yd, stage)
    torch.cuda.synchronize()
    assert np.array_equal(yd.cpu().numpy().view(np.uint32), y_call.view(np.uint32))


def test_fused_host_checks():
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = TL.torch_mod()
    wl = W.make_workload("tiny")
    proj = wl.projections[0]
    pool = TL.build_pool(proj, wl.T)
    seg = TL.build_segments(wl.adapter_ids, wl.q_seq_lens, pool.num_slots)
    xd = TL.to_dev_u16(proj.x)
    yd = torch.zeros((wl.T, proj.D), device="cuda")
    wd = TL.to_dev_u16(W.projection_weight(proj))
    lib = LD.load_library()
    # null W, ldw below d_in, ldw not a multiple of 8
    assert lib.lora_apply_fused_projection(pool.handle, seg.handle, None, proj.d_in, xd.data_ptr(), yd.data_ptr(),
                                           proj.d_in, proj.D, None) == LD.LORA_ERR_ARG
    assert lib.lora_apply_fused_projection(pool.handle, seg.handle, wd.data_ptr(), proj.d_in - 8, xd.data_ptr(),
                                           yd.data_ptr(), proj.d_in, proj.D, None) == LD.LORA_ERR_ARG
    assert lib.lora_apply_fused_projection(pool.handle, seg.handle, wd.data_ptr(), proj.d_in + 4, xd.data_ptr(),
                                           yd.data_ptr(), proj.d_in, proj.D, None) == LD.LORA_ERR_ARG
    assert lib.lora_fused_projection_stage(pool.handle, seg.handle, wd.data_ptr(), proj.d_in, xd.data_ptr(),
                                           yd.data_ptr(), proj.d_in, proj.D, 4, None) == LD.LORA_ERR_ARG


def test_fused_one_graph_serves_any_adapter_mixture(oracle_mod):
    # build + fused projection captured once, replayed for other adapter ids
    # and other length splits of the same totals (decode and prompt rows)
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = TL.torch_mod()
    lens0 = [1, 200, 1, 3, 129, 64, 1, 2]
    ids0 = [1, 2, 0, 3, 4, 1, 4, 2]
    wl = W.custom_workload(lens0, ids0, d_in=512, lane_d_out=[256, 128], num_slots=5, max_rank=32, seed=12)
    proj = wl.projections[0]
    Wb = W.projection_weight(proj)
    pool = TL.build_pool(proj, wl.T)
    seg = LD.LoraSegments(wl.S, wl.T, wl.num_slots, device="cuda")
    ids = torch.tensor(wl.adapter_ids, dtype=torch.int32, device="cuda")
    lens = torch.tensor(wl.q_seq_lens, dtype=torch.int32, device="cuda")
    x = TL.to_dev_u16(proj.x)
    wd = TL.to_dev_u16(Wb)
    y = torch.zeros((wl.T, proj.D), device="cuda")
    g = torch.cuda.CUDAGraph()
    s_ = torch.cuda.Stream()
    s_.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_):
        seg.build(ids, lens, num_tokens=wl.T)  # one eager step before capture
        LD.fused_projection(pool, seg, wd, x, y)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            seg.build(ids, lens, num_tokens=wl.T)
            LD.fused_projection(pool, seg, wd, x, y)
    torch.cuda.current_stream().wait_stream(s_)
    rng = np.random.default_rng(21)
    base, mag = oracle_mod.base_product(Wb, proj.x)
    for mix in range(3):
        new_ids = rng.integers(0, wl.num_slots, size=wl.S).astype(np.int32)
        cut = np.sort(rng.choice(np.arange(1, wl.T), size=wl.S - 1, replace=False))
        new_lens = np.diff(np.concatenate([[0], cut, [wl.T]])).astype(np.int32)
        ids.copy_(torch.from_numpy(new_ids))
        lens.copy_(torch.from_numpy(new_lens))
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert seg.status() == 0
        slot = np.repeat(new_ids, new_lens)
        _, dref = oracle_mod.delta(proj, slot)
        got = y.cpu().numpy().astype(np.float64)
        err = np.abs(got - (base + dref))
        tol = TL.ATOL + TL.RTOL * np.abs(dref) + proj.d_in * 2.0 ** -23 * mag
        assert np.all(err <= tol), f"mixture {mix}: {int((err > tol).sum())} elements out of tolerance"
