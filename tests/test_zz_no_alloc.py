"""lora_apply_shrink_expand_noalloc, the apply for callers that cannot allocate
device memory when they run (plugin hosts that pass only inputs and outputs,
serving loops with a frozen memory plan).  Its scratch is a fixed array inside
the library; its results must be bit-identical to the normal entry point's and match the
oracle.  This file is
collected last on purpose."""
import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W
import lora_testlib as TL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from adapter_gemv_lora_gb300 import build
    build.build()


def _case(seed):
    # decode rows, prefill chunks with ragged tiles, base rows, two lanes, mixed ranks
    lens = [1, 300, 1, 5, 130, 1, 64, 2]
    ids = [1, 2, 0, 3, 1, 2, 3, 0]
    rank = np.array([[0, 0], [16, 16], [8, 24], [32, 4]], dtype=np.int32)
    return W.custom_workload(lens, ids, d_in=2560, lane_d_out=[192, 128], num_slots=4, max_rank=32,
                             rank=rank, seed=seed)


def test_noalloc_matches_the_normal_entry_point_twice_in_a_row(oracle_mod):
    # Both entry points launch the same kernels on the same inputs and every
    # sum runs in a fixed order, so the two results must be bit-identical; the
    # no-alloc result is also checked against the oracle, on two calls in a row.
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    wl = _case(0)
    proj = wl.projections[0]
    pool = TL.build_pool(proj, wl.T)
    seg = TL.build_segments(wl.adapter_ids, wl.q_seq_lens, pool.num_slots)
    slot = wl.per_token_slot()
    rng = np.random.default_rng(1)
    for call in range(2):
        # a different x on each call, so a stale scratch from the first call would show
        x_np = proj.x if call == 0 else W.bf16_bits(rng.standard_normal(proj.x.shape).astype(np.float32))
        x = TL.to_dev_u16(x_np)
        y_ref = torch.from_numpy(proj.y0.copy()).cuda()
        y_na = torch.from_numpy(proj.y0.copy()).cuda()
        n0 = LD.lora_launch_count()
        LD.lora_apply_shrink_expand(pool.handle, seg.handle, x.data_ptr(), y_ref.data_ptr(),
                                    x.stride(0), y_ref.stride(0))
        n1 = LD.lora_launch_count()
        LD.lora_apply_shrink_expand_noalloc(pool.handle, seg.handle, x.data_ptr(), y_na.data_ptr(),
                                            x.stride(0), y_na.stride(0))
        assert LD.lora_launch_count() - n1 == n1 - n0 > 0  # the same kernels
        torch.cuda.synchronize()
        assert seg.status() == 0
        a, b = y_na.cpu().numpy(), y_ref.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"call {call}: bits differ"
        _, dref = oracle_mod.delta(proj, slot, x=x_np)
        TL.assert_delta_close(a, proj.y0, dref, f"call {call} vs oracle")
        TL.assert_rows_untouched(a, proj.y0, np.nonzero(slot == 0)[0])


def test_noalloc_rejects_a_step_beyond_its_scratch():
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    # one 70000-row prefill chunk at rank 128 needs at least
    # 3 partial rows x 70000 x 128 x 4 bytes = 103 MiB > the 64 MiB scratch
    T, d_in = 70000, 4096
    pool = LD.LoraPool(2, 128, d_in, [64], T)
    A = torch.zeros((128, d_in), dtype=torch.int16, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.int16, device="cuda")
    pool.load(1, 0, A, B, 1.0)
    seg = LD.LoraSegments(1, T, 2)
    seg.build(torch.tensor([1], dtype=torch.int32, device="cuda"),
              torch.tensor([T], dtype=torch.int32, device="cuda"), num_tokens=T)
    x = torch.zeros((T, d_in), dtype=torch.int16, device="cuda")
    y = torch.zeros((T, 64), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    n0 = LD.lora_launch_count()
    with pytest.raises(LD.LoraError) as err:
        LD.lora_apply_shrink_expand_noalloc(pool.handle, seg.handle, x.data_ptr(), y.data_ptr(), d_in, 64)
    assert err.value.status == LD.LORA_ERR_SHAPE
    assert LD.lora_launch_count() == n0
