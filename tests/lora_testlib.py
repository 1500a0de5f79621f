"""Shared helpers for the tests: run the CUDA path through the C ABI, run the
oracle, and compare them.  Inputs come only from the seeded workload module."""
from __future__ import annotations

import numpy as np

from adapter_gemv_lora_gb300 import workloads as W

# |gpu - oracle| <= ATOL + RTOL * |oracle| per element of the delta.
ATOL, RTOL = 1e-3, 1e-2

SENTINEL_NAN_BITS = np.uint32(0x7FC0DEAD)   # a quiet NaN with a payload
SENTINEL_X_BITS = np.uint16(0x7FD5)         # a bf16 quiet NaN with a payload


def torch_mod():
    import torch
    return torch


def to_dev_u16(a: np.ndarray, dev="cuda"):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def build_pool(proj: W.Projection, max_tokens: int, max_rank: int = None, slot_map=None, dev="cuda"):
    """A LoraPool holding every loaded (slot, lane) of `proj`.

    slot_map optionally relabels slots: factors of slot k go to slot_map[k]."""
    from adapter_gemv_lora_gb300 import lora_delta as LD
    N, L = proj.rank.shape
    R = proj.max_rank if max_rank is None else max_rank
    n_slots = N if slot_map is None else max(max(slot_map.values()) + 1, N)
    pool = LD.LoraPool(n_slots, R, proj.d_in, proj.lane_d_out, max_tokens, device=dev)
    keep = []
    for k in range(1, N):
        for l in range(L):
            r = int(proj.rank[k, l])
            if r > 0:
                A = to_dev_u16(proj.A[k][l], dev)
                B = to_dev_u16(proj.B[k][l], dev)
                keep += [A, B]
                kk = k if slot_map is None else slot_map[k]
                pool.load(kk, l, A, B, float(proj.scale[k, l]))
    torch_mod().cuda.synchronize()
    return pool


def build_segments(adapter_ids, q_seq_lens, num_slots: int, max_seqs=None, max_tokens=None, dev="cuda",
                   num_tokens=None):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = torch_mod()
    ids = torch.tensor(np.asarray(adapter_ids, dtype=np.int32), device=dev)
    lens = torch.tensor(np.asarray(q_seq_lens, dtype=np.int32), device=dev)
    S = int(ids.numel())
    T = int(np.asarray(q_seq_lens, dtype=np.int64).sum()) if num_tokens is None else num_tokens
    seg = LD.LoraSegments(max(S, 1) if max_seqs is None else max_seqs,
                          max(T, 1) if max_tokens is None else max_tokens, num_slots, device=dev)
    seg.build(ids, lens, num_tokens=T)
    return seg


def run_gpu(proj: W.Projection, adapter_ids, q_seq_lens, x=None, y0=None, pool=None, dev="cuda",
            num_slots=None):
    """y after one build + apply on the GPU (numpy float32 [T, D])."""
    from adapter_gemv_lora_gb300 import lora_delta as LD
    torch = torch_mod()
    x = proj.x if x is None else x
    y0 = proj.y0 if y0 is None else y0
    T = x.shape[0]
    if pool is None:
        pool = build_pool(proj, max(T, 1), dev=dev)
    N = pool.num_slots if num_slots is None else num_slots
    seg = build_segments(adapter_ids, q_seq_lens, N, dev=dev)
    xd = to_dev_u16(x, dev)
    yd = torch.from_numpy(np.ascontiguousarray(y0)).to(dev)
    LD.apply(pool, seg, xd, yd)
    torch.cuda.synchronize()
    st = seg.status()
    assert st == 0, f"device status {st}: {LD.lora_status_string(st)}"
    return yd.cpu().numpy()


def assert_delta_close(y_gpu: np.ndarray, y0: np.ndarray, delta_ref: np.ndarray, what: str = ""):
    d_gpu = y_gpu.astype(np.float64) - y0.astype(np.float64)
    err = np.abs(d_gpu - delta_ref)
    tol = ATOL + RTOL * np.abs(delta_ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first {idx.tolist()}: "
                             f"gpu {d_gpu[tuple(idx[0])]:.6g} ref {delta_ref[tuple(idx[0])]:.6g}")
    return float((err / tol).max()) if err.size else 0.0


def assert_rows_untouched(y_gpu: np.ndarray, y0: np.ndarray, rows):
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size:
        a = np.ascontiguousarray(y_gpu[rows]).view(np.uint32)
        b = np.ascontiguousarray(y0[rows]).view(np.uint32)
        assert np.array_equal(a, b), "rows that must not be written were changed"


def remix_batch(wl, rng):
    """A new batch around some of wl's sequences: about half of them, in a new
    order, with foreign sequences (other slots, lengths on both sides of the
    tensor-path threshold and of the tile size, base rows) between them.
    Returns (ids, lens, pieces) where pieces[i] is the source sequence of new
    sequence i, or None for a foreign one."""
    S, N = wl.S, wl.num_slots
    keep = rng.permutation(S)[:max(1, (S + 1) // 2)].tolist()
    n_foreign = max(3, S // 4)
    f_lens = rng.choice([1, 1, 1, 2, 5, 63, 64, 65, 127, 130, 300], size=n_foreign).tolist()
    f_ids = rng.integers(0, N, size=n_foreign).tolist()
    order = [("k", s) for s in keep] + [("f", i) for i in range(n_foreign)]
    order = [order[i] for i in rng.permutation(len(order))]
    ids, lens, pieces = [], [], []
    for kind, v in order:
        if kind == "k":
            ids.append(int(wl.adapter_ids[v]))
            lens.append(int(wl.q_seq_lens[v]))
            pieces.append(v)
        else:
            ids.append(int(f_ids[v]))
            lens.append(int(f_lens[v]))
            pieces.append(None)
    return np.array(ids, dtype=np.int32), np.array(lens, dtype=np.int32), pieces
