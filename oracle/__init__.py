"""CPU oracle for the mixed-adapter LoRA delta (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path never does.  The compiled part,
``lora_oracle.cpp``, is plain C++ with OpenMP and computes every value in
double precision; this module only builds it with g++ and marshals numpy
arrays into it.  See ``lora_oracle.cpp`` for what is computed and the passages
it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.cpp")
_LIB = os.path.join(_HERE, "liblora_oracle.so")
_lib = None

STATUS_OK, STATUS_SLOT, STATUS_META = 0, -3, -6


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_segments.argtypes = [ctypes.c_int] * 6 + [P] * 9
        lib.oracle_segments.restype = ctypes.c_int
        lib.oracle_delta.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P, P, P, P, P, P,
                                     P, i64, P, P, i64, P, i64, P, P, ctypes.c_int]
        lib.oracle_delta.restype = None
        lib.oracle_base_product.argtypes = [ctypes.c_int, ctypes.c_int, P, i64, P, i64, P, i64, P, P,
                                            ctypes.c_int]
        lib.oracle_base_product.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def segments(adapter_ids: Sequence[int], q_seq_lens: Sequence[int], T: int, N: int,
             tc_min_qlen: int, tile_rows: int, group_rows: int) -> Dict[str, np.ndarray]:
    """Routing metadata of one step (see ``oracle_segments`` in lora_oracle.cpp)."""
    lib = _load()
    ids = np.ascontiguousarray(adapter_ids, dtype=np.int32)
    q = np.ascontiguousarray(q_seq_lens, dtype=np.int32)
    S = int(ids.shape[0])
    slot = np.zeros(max(T, 1), dtype=np.int32)
    seq_start = np.zeros(S + 1, dtype=np.int32)
    perm = np.zeros(max(T, 1), dtype=np.int32)
    seg_off = np.zeros(2 * (N + 1), dtype=np.int32)
    cap = max(T, 1) + S + N + 1
    dec_work = np.zeros((cap, 4), dtype=np.int32)
    tc_work = np.zeros((cap, 4), dtype=np.int32)
    counts = np.zeros(4, dtype=np.int32)
    st = lib.oracle_segments(S, T, N, tc_min_qlen, tile_rows, group_rows, _ptr(ids), _ptr(q),
                             _ptr(slot), _ptr(seq_start), _ptr(perm), _ptr(seg_off),
                             _ptr(dec_work), _ptr(tc_work), _ptr(counts))
    n_act, n_dec_rows, nd, nt = (int(c) for c in counts)
    return {
        "status": int(st),
        "slot": slot[:T].copy() if st == 0 else None,
        "seq_start": seq_start if st == 0 else None,
        "perm": perm[:n_act].copy(),
        "seg_off": seg_off if st == 0 else None,
        "dec_work": dec_work[:nd].copy(),
        "tc_work": tc_work[:nt].copy(),
        "counts": counts.copy(),
        "n_active": n_act,
        "n_dec_rows": n_dec_rows,
    }


def flatten_factors(proj):
    """Pack a Projection's per-(slot, lane) A and B into flat arrays + offsets."""
    N, L = proj.rank.shape
    a_parts, b_parts = [], []
    a_off = np.zeros(N * L, dtype=np.int64)
    b_off = np.zeros(N * L, dtype=np.int64)
    ao = bo = 0
    for k in range(N):
        for l in range(L):
            r = int(proj.rank[k, l])
            a_off[k * L + l] = ao
            b_off[k * L + l] = bo
            if r > 0:
                a = np.ascontiguousarray(proj.A[k][l], dtype=np.uint16)
                b = np.ascontiguousarray(proj.B[k][l], dtype=np.uint16)
                assert a.shape == (r, proj.d_in) and b.shape == (proj.lane_d_out[l], r)
                a_parts.append(a.ravel())
                b_parts.append(b.ravel())
                ao += a.size
                bo += b.size
    A_flat = np.concatenate(a_parts) if a_parts else np.zeros(1, dtype=np.uint16)
    B_flat = np.concatenate(b_parts) if b_parts else np.zeros(1, dtype=np.uint16)
    return A_flat, a_off, B_flat, b_off


def delta(proj, slot: np.ndarray, rows: Optional[Sequence[int]] = None, num_threads: int = 0,
          x: Optional[np.ndarray] = None, y0: Optional[np.ndarray] = None,
          rank: Optional[np.ndarray] = None, scale: Optional[np.ndarray] = None, _flat=None):
    """(y_ref, delta) in float64 for the listed rows (all rows by default).

    ``proj`` is a workloads.Projection; x / y0 / rank / scale override its
    fields when given.  Returns arrays of shape [len(rows), D].
    """
    lib = _load()
    x = np.ascontiguousarray(proj.x if x is None else x, dtype=np.uint16)
    y0 = np.ascontiguousarray(proj.y0 if y0 is None else y0, dtype=np.float32)
    rank = np.ascontiguousarray(proj.rank if rank is None else rank, dtype=np.int32)
    scale = np.ascontiguousarray(proj.scale if scale is None else scale, dtype=np.float32)
    T = x.shape[0]
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    N, L = rank.shape
    d_out = np.ascontiguousarray(proj.lane_d_out, dtype=np.int32)
    D = int(d_out.sum())
    A_flat, a_off, B_flat, b_off = flatten_factors(proj) if _flat is None else _flat
    n = int(rows.shape[0])
    y_ref = np.zeros((max(n, 1), D), dtype=np.float64)
    dl = np.zeros((max(n, 1), D), dtype=np.float64)
    lib.oracle_delta(proj.d_in, L, _ptr(d_out), N, _ptr(rank), _ptr(scale),
                     _ptr(A_flat), _ptr(a_off), _ptr(B_flat), _ptr(b_off),
                     _ptr(x), x.shape[1], _ptr(slot), _ptr(y0), y0.shape[1],
                     _ptr(rows), n, _ptr(y_ref), _ptr(dl), int(num_threads))
    return y_ref[:n], dl[:n]


def base_product(W: np.ndarray, x: np.ndarray, rows: Optional[Sequence[int]] = None, num_threads: int = 0):
    """(base, abs_base) in float64 for the listed rows: base = x @ W^T over bf16
    values (W is [D][d_in] bf16 bits, x is [T][d_in] bf16 bits), abs_base the
    sum of the products' magnitudes.  Arrays of shape [len(rows), D]."""
    lib = _load()
    W = np.ascontiguousarray(W, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    D, d_in = W.shape
    assert x.shape[1] >= d_in
    if rows is None:
        rows = np.arange(x.shape[0], dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = int(rows.shape[0])
    base = np.zeros((max(n, 1), D), dtype=np.float64)
    mag = np.zeros((max(n, 1), D), dtype=np.float64)
    lib.oracle_base_product(d_in, D, _ptr(W), W.shape[1], _ptr(x), x.shape[1], _ptr(rows), n,
                            _ptr(base), _ptr(mag), int(num_threads))
    return base[:n], mag[:n]


def fused_projection(proj, W: np.ndarray, slot: np.ndarray, rows: Optional[Sequence[int]] = None,
                     num_threads: int = 0, _flat=None):
    """The projection with the delta in its output, float64, for the listed
    rows: (y, delta, abs_base) with y = x @ W^T + delta (slot-0 rows: the
    base product alone; y0 plays no part)."""
    base, mag = base_product(W, proj.x, rows, num_threads)
    _, dl = delta(proj, slot, rows, num_threads, _flat=_flat)
    return base + dl, dl, mag


# ------------------------------------------------------------------ MoE layers
#
# Expert LoRA of an MoE layer: each dispatched row (token, chosen expert) takes
# the delta of its expert's copy of its sequence's adapter.  The library's
# routing rule (its header, the MoE section): a maximal run of dispatched rows
# with the same (expert, sequence, adapter) is one sequence of the builder,
# whose slot is 1 + expert * A + (adapter - 1) (0 for the base model).  Written
# out here independently, as plain loops.

def moe_slot(expert: int, adapter: int, num_adapters: int) -> int:
    """Slot of an expert's copy of an adapter (0 for the base model)."""
    if adapter == 0:
        return 0
    return 1 + expert * num_adapters + (adapter - 1)


def moe_runs(row_expert, row_adapter, row_seq, num_experts: int, num_adapters: int):
    """(ids, lens) of the runs of equal (expert, sequence, adapter), in row
    order; an expert or adapter id out of range gives slot 1 + E * A (out of
    the pool's range)."""
    ids, lens = [], []
    prev = None
    n_slots = 1 + num_experts * num_adapters
    for e, a, s in zip(map(int, row_expert), map(int, row_adapter), map(int, row_seq)):
        key = (e, s, a)
        if key != prev:
            ok = 0 <= e < num_experts and 0 <= a <= num_adapters
            ids.append(moe_slot(e, a, num_adapters) if ok else n_slots)
            lens.append(0)
            prev = key
        lens[-1] += 1
    return np.asarray(ids, dtype=np.int32), np.asarray(lens, dtype=np.int32)


class _SlotProjection:
    """A projection view over slots 0..N-1 (the attributes delta() reads)."""

    def __init__(self, d_in, lane_d_out, rank, scale, A, B, x, y0, max_rank):
        self.d_in, self.lane_d_out = d_in, list(lane_d_out)
        self.rank, self.scale, self.A, self.B = rank, scale, A, B
        self.x, self.y0, self.max_rank = x, y0, max_rank

    @property
    def num_lanes(self):
        return len(self.lane_d_out)


def moe_projection(mproj, num_experts: int, num_adapters: int):
    """The expert projection as a projection over slots 1 + E * A (slot of
    (e, a) by moe_slot), for delta()."""
    N, L = 1 + num_experts * num_adapters, mproj.num_lanes
    rank = np.zeros((N, L), dtype=np.int32)
    scale = np.zeros((N, L), dtype=np.float32)
    A = [[None] * L for _ in range(N)]
    B = [[None] * L for _ in range(N)]
    for e in range(num_experts):
        for a in range(1, num_adapters + 1):
            k = moe_slot(e, a, num_adapters)
            for l in range(L):
                rank[k, l] = mproj.rank[a, l]
                scale[k, l] = mproj.scale[a, l]
                A[k][l], B[k][l] = mproj.A[e][a][l], mproj.B[e][a][l]
    return _SlotProjection(mproj.d_in, mproj.lane_d_out, rank, scale, A, B, mproj.x, mproj.y0, mproj.max_rank)
