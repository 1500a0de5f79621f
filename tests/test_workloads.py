"""The seeded input generator: shapes, laws and determinism of the workloads."""
import numpy as np
import pytest

from adapter_gemv_lora_gb300 import workloads as W


def test_bf16_rounding_ties_to_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -7], dtype=np.float32)
    bits = W.bf16_bits(vals)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even is 1 + 2^-6.
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]
    assert np.array_equal(W.bf16_bits_to_f32(bits), np.array([1, 1, 1 + 2 ** -6, -2.5, 1 + 2 ** -7],
                                                             dtype=np.float32))


def test_zipf_law():
    p = W.zipf_probs(32, 1.1)
    assert abs(p.sum() - 1) < 1e-12
    assert np.all(np.diff(p) < 0)
    assert abs(p[0] / p[1] - 2 ** 1.1) < 1e-12


def test_tiny_and_decode_shapes():
    wl = W.make_workload("tiny")
    assert wl.S == wl.T == 8 and wl.num_slots == 4
    p = wl.projections[0]
    assert p.d_in == 256 and p.lane_d_out == [256]
    assert np.all(p.rank[1:] == 8) and np.all(p.scale[1:] == 2.0)
    wl = W.make_workload("decode_oproj")
    assert wl.T == 256 and int((wl.adapter_ids == 0).sum()) == 51
    assert wl.adapter_ids.max() == 8 and wl.adapter_ids[wl.adapter_ids > 0].min() == 1


def test_prefill_qkv_shapes():
    wl = W.make_workload("prefill_qkv", draw_xy=False)
    assert wl.S == 16
    assert wl.q_seq_lens.min() >= 128 and wl.q_seq_lens.max() <= 2048
    p = wl.projections[0]
    assert p.lane_d_out == [4096, 1024, 1024] and p.d_in == 4096
    assert np.all(p.rank[1:] == 16)


def test_mlp_decode_shapes():
    wl = W.make_workload("mlp_decode", draw_xy=False)
    assert wl.T == 512 and int((wl.adapter_ids == 0).sum()) == 77
    gu, dn = wl.projections
    assert gu.lane_d_out == [14336, 14336] and gu.d_in == 4096
    assert dn.lane_d_out == [4096] and dn.d_in == 14336
    assert set(np.unique(gu.rank[1:])) <= {8, 16, 32, 64}
    assert np.array_equal(gu.rank[:, 0], dn.rank[:, 0])
    assert np.allclose(gu.scale[1:], 2.0)


def test_cont_batch_shapes():
    wl = W.make_workload("cont_batch", draw_xy=False)
    q = wl.q_seq_lens
    assert wl.S == 128 and wl.T == 16384
    assert int((q == 1).sum()) == 104
    chunks = q[q > 1]
    assert chunks.size == 24 and chunks.min() >= 128 and chunks.max() <= 1024
    p = wl.projections[0]
    assert set(np.unique(p.rank[1:])) <= {16, 32, 64, 128} and p.max_rank == 128


@pytest.mark.parametrize("name", ["tiny", "decode_oproj"])
def test_determinism(name):
    a = W.make_workload(name)
    b = W.make_workload(name)
    assert np.array_equal(a.adapter_ids, b.adapter_ids)
    pa, pb = a.projections[0], b.projections[0]
    assert np.array_equal(pa.x, pb.x) and np.array_equal(pa.y0, pb.y0)
    assert np.array_equal(pa.A[1][0], pb.A[1][0])
    c = W.make_workload(name, seed=1)
    assert not np.array_equal(pa.x, c.projections[0].x)
