"""MoE expert LoRA on the GPU: dispatched rows routed by lora_build_segments_moe
(runs of (expert, sequence, adapter) into the builder), the ordinary apply on
the dispatched rows, against the oracle.  Metadata bit-exact; the delta within
|gpu - oracle| <= 1e-3 + 1e-2 * |oracle|; base rows untouched."""
import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W
from conftest import GROUP_ROWS, TILE_ROWS, TC_MIN_QLEN
import lora_testlib as TL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from adapter_gemv_lora_gb300 import build
    build.build()


_WL = {}


def _workload(name):
    if name not in _WL:
        _WL[name] = W.make_moe_workload(name)
    return _WL[name]


def _segments(wl, rows=None, max_seqs=None):
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    e, a, s = wl.row_expert, wl.row_adapter, wl.row_seq
    if rows is not None:
        e, a, s = e[rows], a[rows], s[rows]
    n = int(e.shape[0])
    N = 1 + wl.num_experts * wl.num_adapters
    # the runs are at most the rows; 4096 sequences fit the builder's shared memory at 1025 slots
    seg = LD.LoraSegments(max_seqs or max(min(n, 4096), 1), max(n, 1), N)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).cuda()
    seg.build_moe(t(e), t(a), t(s), wl.num_experts, wl.num_adapters)
    return seg


def _pool(wl, mp, max_tokens):
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    N = 1 + wl.num_experts * wl.num_adapters
    pool = LD.LoraPool(N, mp.max_rank, mp.d_in, mp.lane_d_out, max_tokens)
    keep = []
    for ex in range(wl.num_experts):
        for ad in range(1, wl.num_adapters + 1):
            k = LD.lora_moe_slot(ex, ad, wl.num_adapters)
            for l in range(mp.num_lanes):
                if mp.rank[ad, l] > 0:
                    A = TL.to_dev_u16(mp.A[ex][ad][l])
                    B = TL.to_dev_u16(mp.B[ex][ad][l])
                    keep += [A, B]
                    pool.load(k, l, A, B, float(mp.scale[ad, l]))
    torch.cuda.synchronize()
    return pool


@pytest.mark.parametrize("name", W.MOE_CONFIG_NAMES)
def test_moe_metadata_matches_oracle(oracle_mod, name):
    wl = _workload(name)
    N = 1 + wl.num_experts * wl.num_adapters
    seg = _segments(wl)
    assert seg.status() == 0
    got = seg.read()
    ids, lens = oracle_mod.moe_runs(wl.row_expert, wl.row_adapter, wl.row_seq, wl.num_experts, wl.num_adapters)
    exp = oracle_mod.segments(ids, lens, wl.R, N, TC_MIN_QLEN, TILE_ROWS, GROUP_ROWS)
    assert exp["status"] == 0
    assert got["counts"].tolist() == exp["counts"].tolist()
    for key in ("slot", "perm", "seg_off", "dec_work", "tc_work"):
        assert np.array_equal(got[key], exp[key]), key


@pytest.mark.parametrize("name", W.MOE_CONFIG_NAMES)
def test_moe_delta_matches_oracle(oracle_mod, name):
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _workload(name)
    seg = _segments(wl)
    ids, lens = oracle_mod.moe_runs(wl.row_expert, wl.row_adapter, wl.row_seq, wl.num_experts, wl.num_adapters)
    slot = np.repeat(ids, lens)
    for mp in wl.projections:
        pool = _pool(wl, mp, wl.R)
        x = TL.to_dev_u16(mp.x)
        y = torch.from_numpy(mp.y0.copy()).cuda()
        LD.apply(pool, seg, x, y)
        torch.cuda.synchronize()
        assert seg.status() == 0
        got = y.cpu().numpy()
        _, dref = oracle_mod.delta(oracle_mod.moe_projection(mp, wl.num_experts, wl.num_adapters), slot)
        TL.assert_delta_close(got, mp.y0, dref, f"{name} {mp.name}")
        TL.assert_rows_untouched(got, mp.y0, np.nonzero(slot == 0)[0])


def test_moe_rows_keep_their_bits_without_the_other_sequences():
    # the dispatched rows of one prompt chunk give the same bits whether or not
    # another chunk's rows are routed in the same step (its runs, and so its
    # paths, depend on its own tokens only)
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _workload("moe_prefill")
    mp = wl.projections[1]
    pool = _pool(wl, mp, wl.R)
    rows = np.nonzero(wl.row_seq == 0)[0]
    outs = []
    for sel in (None, rows):
        seg = _segments(wl, rows=sel)
        x = TL.to_dev_u16(mp.x if sel is None else mp.x[sel])
        y0 = mp.y0 if sel is None else mp.y0[sel]
        y = torch.from_numpy(np.ascontiguousarray(y0)).cuda()
        LD.apply(pool, seg, x, y)
        torch.cuda.synchronize()
        assert seg.status() == 0
        outs.append(y.cpu().numpy())
    assert np.array_equal(np.ascontiguousarray(outs[0][rows]).view(np.uint32), outs[1].view(np.uint32))


def test_moe_bad_ids_and_capacity():
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    t = lambda v: torch.tensor(v, dtype=torch.int32, device="cuda")
    seg = LD.LoraSegments(4, 8, 1 + 3 * 2)
    # an expert id out of range: device status LORA_ERR_SLOT and no work
    seg.build_moe(t([0, 0, 3, 1]), t([1, 1, 1, 2]), t([0, 0, 0, 1]), 3, 2)
    assert seg.status() == LD.LORA_ERR_SLOT
    assert seg.read()["counts"].tolist() == [0, 0, 0, 0]
    # more runs (6) than max_seqs (4): LORA_ERR_META
    seg.build_moe(t([0, 1, 2, 0, 1, 2]), t([1] * 6), t([0] * 6), 3, 2)
    assert seg.status() == LD.LORA_ERR_META
    # host checks: slot count must be 1 + E * A
    with pytest.raises(LD.LoraError):
        seg.build_moe(t([0]), t([1]), t([0]), 2, 2)
