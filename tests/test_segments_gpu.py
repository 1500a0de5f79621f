"""Segment builder on the GPU against the oracle's metadata: bit-exact."""
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


def _compare(oracle_mod, ids, lens, N, T=None):
    T = int(np.asarray(lens, dtype=np.int64).sum()) if T is None else T
    exp = oracle_mod.segments(ids, lens, T, N, TC_MIN_QLEN, TILE_ROWS, GROUP_ROWS)
    seg = TL.build_segments(ids, lens, N, num_tokens=T, max_tokens=max(T, 1))
    st = seg.status()
    assert st == exp["status"]
    got = seg.read()
    assert got["counts"].tolist() == exp["counts"].tolist()
    if st != 0:
        return
    assert np.array_equal(got["slot"], exp["slot"])
    assert np.array_equal(got["perm"], exp["perm"])
    assert np.array_equal(got["seg_off"], exp["seg_off"])
    assert np.array_equal(got["dec_work"], exp["dec_work"])
    assert np.array_equal(got["tc_work"], exp["tc_work"])
    # each decode group's row list is its perm range, in order
    for w, (_, pb, pe, _) in enumerate(exp["dec_work"]):
        assert np.array_equal(got["dec_rows"][w, :pe - pb], exp["perm"][pb:pe]), f"group {w}"


@pytest.mark.parametrize("seed", range(10))
def test_random_batches(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(1, 3000))
    N = int(rng.integers(2, 70))
    lens = rng.choice([0, 1, 1, 1, 1, 2, 7, 63, 64, 65, 128, 129, 257, 1024], size=S)
    ids = rng.integers(0, N, size=S)
    _compare(oracle_mod, ids, lens, N)


def test_adversarial(oracle_mod):
    _compare(oracle_mod, [0] * 50, [1] * 50, 4)                      # all base
    _compare(oracle_mod, [3] * 40, [1] * 40, 4)                      # one adapter, decode
    _compare(oracle_mod, [1], [1], 2)                                # S = T = 1
    _compare(oracle_mod, [2], [333], 4)                              # one ragged prefill sequence
    _compare(oracle_mod, list(range(1, 65)) * 3, [1] * 192, 65)      # every slot
    _compare(oracle_mod, [5, 0, 5, 0], [64, 63, 65, 0], 8)           # threshold edges, a zero length
    _compare(oracle_mod, list(range(2048)), [1] * 2048, 2048)        # maximum slot count
    _compare(oracle_mod, [1] * 4000, [1] * 4000, 2)                  # many sequences, one slot


def test_workload_configs(oracle_mod):
    for name in W.CONFIG_NAMES:
        wl = W.make_workload(name, draw_xy=False)
        _compare(oracle_mod, wl.adapter_ids, wl.q_seq_lens, wl.num_slots)


def test_device_detected_errors(oracle_mod):
    _compare(oracle_mod, [1, 7], [1, 1], 4)          # slot id >= N
    _compare(oracle_mod, [1, -2], [1, 1], 4)         # negative slot id
    _compare(oracle_mod, [1, 1], [2, -1], 4, T=1)    # negative length
    _compare(oracle_mod, [1, 1], [2, 2], 4, T=3)     # lengths do not sum to T
    _compare(oracle_mod, [9, 1], [2, 2], 4, T=3)     # both: length error wins


def test_rebuild_reuses_workspace(oracle_mod):
    seg = TL.build_segments([1, 2, 0], [300, 1, 2], 4, max_seqs=64, max_tokens=4096)
    import torch
    for seed in range(3):
        rng = np.random.default_rng(seed)
        lens = rng.choice([1, 70, 200], size=20)
        ids = rng.integers(0, 4, size=20)
        seg.build(torch.tensor(ids, dtype=torch.int32, device="cuda"),
                  torch.tensor(lens, dtype=torch.int32, device="cuda"))
        got = seg.read()
        exp = oracle_mod.segments(ids, lens, int(lens.sum()), 4, TC_MIN_QLEN, TILE_ROWS, GROUP_ROWS)
        assert np.array_equal(got["perm"], exp["perm"])
        assert np.array_equal(got["tc_work"], exp["tc_work"])
        assert np.array_equal(got["dec_work"], exp["dec_work"])


@pytest.mark.parametrize("N", [65, 2048])
def test_many_sequences_beyond_shared_memory(oracle_mod, N):
    # 20000 sequences: the builder's per-sequence arrays live in the workspace
    rng = np.random.default_rng(N)
    S = 20000
    lens = rng.choice([0, 1, 1, 1, 2, 5, 64, 130], size=S)
    ids = rng.integers(0, N, size=S)
    _compare(oracle_mod, ids, lens, N)


def test_equal_and_unequal_lengths_inside_a_warp(oracle_mod):
    # warps whose same-slot sequences all have one length (ranks are counts)
    # next to warps where they differ (ranks are sums)
    ids = [1] * 32 + [2, 1] * 16 + [3] * 16 + [1] * 16
    lens = [1] * 32 + [1, 2] * 16 + [70] * 16 + [3, 1] * 8
    _compare(oracle_mod, ids, lens, 4)
