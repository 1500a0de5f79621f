"""Python binding of liblora_delta.so (argument marshalling only).

The functions carry the C ABI's names and arguments (see include/lora_delta.h);
device pointers are plain integers (e.g. ``tensor.data_ptr()``) and streams are
``cudaStream_t`` integers (e.g. ``torch.cuda.current_stream().cuda_stream``).
Every computation runs in the library's CUDA kernels: this module has no
fallback and raises if the library cannot be loaded.

``LoraPool`` and ``LoraSegments`` are thin conveniences that allocate the
caller-owned device memory with PyTorch and forward to the C functions.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblora_delta.so")

LORA_OK, LORA_ERR_ARG, LORA_ERR_SHAPE, LORA_ERR_SLOT = 0, -1, -2, -3
LORA_ERR_RANK, LORA_ERR_CUDA, LORA_ERR_META, LORA_ERR_TIMEOUT = -4, -5, -6, -7
LORA_MAX_LANES, LORA_MAX_SLOTS = 4, 2048
LORA_DEC_GROUP_ROWS, LORA_TC_TILE_ROWS, LORA_TC_MIN_QLEN = 8, 128, 64

_lib = None


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {lora_status_string(status)} ({status})" if what else
                         f"{lora_status_string(status)} ({status})")


def load_library(path: str = LIB_PATH):
    """Load liblora_delta.so (raises OSError if it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: run `python -m adapter_gemv_lora_gb300.build` "
                      "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "lora_pool_bytes": (SZ, [I, I, I, I, P, I]),
        "lora_pool_create": (I, [P, P, SZ, I, I, I, I, P, I, P]),
        "lora_pool_load": (I, [P, I, I, I, ctypes.c_float, P, P, P]),
        "lora_pool_destroy": (I, [P]),
        "lora_segments_bytes": (SZ, [I, I, I]),
        "lora_segments_create": (I, [P, P, SZ, I, I, I]),
        "lora_build_segments": (I, [P, P, P, I, I, P]),
        "lora_build_segments_moe": (I, [P, P, P, P, I, I, I, P]),
        "lora_moe_slot": (I, [I, I, I]),
        "lora_segments_capacity": (I, [P, P, P]),
        "lora_segments_read": (I, [P, P, P, P, P, P, P, P]),
        "lora_segments_read_dec_rows": (I, [P, P, P]),
        "lora_get_status": (I, [P, P, P]),
        "lora_clear_status": (I, [P, P]),
        "lora_segments_destroy": (I, [P]),
        "lora_apply_shrink_expand": (I, [P, P, P, P, I64, I64, P]),
        "lora_apply_stage": (I, [P, P, P, P, I64, I64, I, P]),
        "lora_apply_shrink_expand_noalloc": (I, [P, P, P, P, I64, I64, P]),
        "lora_apply_fused_projection": (I, [P, P, P, I64, P, P, I64, I64, P]),
        "lora_fused_projection_stage": (I, [P, P, P, I64, P, P, I64, I64, I, P]),
        "lora_status_string": (ctypes.c_char_p, [I]),
        "lora_launch_count": (ctypes.c_uint64, []),
        "lora_last_error_string": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(st: int, what: str):
    if st != LORA_OK:
        detail = lora_last_error_string() if st == LORA_ERR_CUDA else ""
        raise LoraError(st, f"{what} [{detail}]" if detail else what)


def _arr(vals, ctype):
    return (ctype * len(vals))(*vals)


# ----------------------------------------------------------------- C functions

def lora_status_string(status: int) -> str:
    return load_library().lora_status_string(int(status)).decode()


def lora_last_error_string() -> str:
    return load_library().lora_last_error_string().decode()


def lora_launch_count() -> int:
    return int(load_library().lora_launch_count())


def lora_pool_bytes(num_slots: int, max_rank: int, d_in: int, lane_d_out: Sequence[int], max_tokens: int) -> int:
    lib = load_library()
    return int(lib.lora_pool_bytes(num_slots, max_rank, d_in, len(lane_d_out),
                                   _arr(list(lane_d_out), ctypes.c_int), max_tokens))


def lora_pool_create(dev_mem: int, nbytes: int, num_slots: int, max_rank: int, d_in: int,
                     lane_d_out: Sequence[int], max_tokens: int, stream: int = 0) -> int:
    lib = load_library()
    out = ctypes.c_void_p()
    st = lib.lora_pool_create(ctypes.byref(out), dev_mem, nbytes, num_slots, max_rank, d_in, len(lane_d_out),
                              _arr(list(lane_d_out), ctypes.c_int), max_tokens, stream)
    _check(st, "lora_pool_create")
    return out.value


def lora_pool_load(pool: int, slot: int, lane: int, rank: int, scale: float, A: int, B: int,
                   stream: int = 0) -> None:
    _check(load_library().lora_pool_load(pool, slot, lane, rank, float(scale), A, B, stream), "lora_pool_load")


def lora_pool_destroy(pool: int) -> None:
    _check(load_library().lora_pool_destroy(pool), "lora_pool_destroy")


def lora_segments_bytes(max_seqs: int, max_tokens: int, num_slots: int) -> int:
    return int(load_library().lora_segments_bytes(max_seqs, max_tokens, num_slots))


def lora_segments_create(dev_ws: int, nbytes: int, max_seqs: int, max_tokens: int, num_slots: int) -> int:
    out = ctypes.c_void_p()
    _check(load_library().lora_segments_create(ctypes.byref(out), dev_ws, nbytes, max_seqs, max_tokens, num_slots),
           "lora_segments_create")
    return out.value


def lora_build_segments(seg: int, adapter_ids: int, q_seq_lens: int, num_seqs: int, num_tokens: int,
                        stream: int = 0) -> None:
    _check(load_library().lora_build_segments(seg, adapter_ids, q_seq_lens, num_seqs, num_tokens, stream),
           "lora_build_segments")


def lora_moe_slot(expert: int, adapter: int, num_adapters: int) -> int:
    """Pool slot of adapter `adapter` (1..A; 0 = base) of expert `expert`."""
    return int(load_library().lora_moe_slot(expert, adapter, num_adapters))


def lora_build_segments_moe(seg: int, row_expert: int, row_adapter: int, row_seq: int, num_rows: int,
                            num_experts: int, num_adapters: int, stream: int = 0) -> None:
    _check(load_library().lora_build_segments_moe(seg, row_expert, row_adapter, row_seq, num_rows, num_experts,
                                                  num_adapters, stream), "lora_build_segments_moe")


def lora_segments_capacity(seg: int):
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(load_library().lora_segments_capacity(seg, ctypes.byref(a), ctypes.byref(b)), "lora_segments_capacity")
    return a.value, b.value


def lora_segments_read(seg: int, num_tokens: int, num_slots: int, stream: int = 0) -> dict:
    """Copy the last build's metadata to numpy arrays (synchronises the stream)."""
    dec_cap, tc_cap = lora_segments_capacity(seg)
    T = max(int(num_tokens), 1)
    slot = np.zeros(T, dtype=np.int32)
    perm = np.zeros(T, dtype=np.int32)
    seg_off = np.zeros(2 * (num_slots + 1), dtype=np.int32)
    counts = np.zeros(4, dtype=np.int32)
    dec = np.zeros((dec_cap, 4), dtype=np.int32)
    tc = np.zeros((tc_cap, 4), dtype=np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(load_library().lora_segments_read(seg, p(slot), p(perm), p(seg_off), p(counts), p(dec), p(tc), stream),
           "lora_segments_read")
    n_act, n_dec_rows, nd, nt = (int(c) for c in counts)
    return {"slot": slot[:num_tokens], "perm": perm[:n_act], "seg_off": seg_off, "counts": counts,
            "dec_work": dec[:nd], "tc_work": tc[:nt], "dec_rows": lora_segments_read_dec_rows(seg, stream)[:nd]}


def lora_segments_read_dec_rows(seg: int, stream: int = 0) -> np.ndarray:
    """The last build's decode-group row lists, [capacity][8] (rows past a group's count unspecified)."""
    dec_cap, _ = lora_segments_capacity(seg)
    rows = np.zeros((max(dec_cap, 1), 8), dtype=np.int32)
    _check(load_library().lora_segments_read_dec_rows(seg, rows.ctypes.data_as(ctypes.c_void_p), stream),
           "lora_segments_read_dec_rows")
    return rows


def lora_get_status(seg: int, stream: int = 0) -> int:
    v = ctypes.c_int32()
    _check(load_library().lora_get_status(seg, ctypes.byref(v), stream), "lora_get_status")
    return int(v.value)


def lora_clear_status(seg: int, stream: int = 0) -> None:
    _check(load_library().lora_clear_status(seg, stream), "lora_clear_status")


def lora_segments_destroy(seg: int) -> None:
    _check(load_library().lora_segments_destroy(seg), "lora_segments_destroy")


def lora_apply_shrink_expand(pool: int, seg: int, x: int, y: int, ldx: int, ldy: int, stream: int = 0) -> None:
    _check(load_library().lora_apply_shrink_expand(pool, seg, x, y, ldx, ldy, stream), "lora_apply_shrink_expand")


def lora_apply_shrink_expand_noalloc(pool: int, seg: int, x: int, y: int, ldx: int, ldy: int,
                                     stream: int = 0) -> None:
    """lora_apply_shrink_expand with the rank-space scratch in the library's
    fixed device array instead of the pool, for callers that cannot allocate."""
    _check(load_library().lora_apply_shrink_expand_noalloc(pool, seg, x, y, ldx, ldy, stream),
           "lora_apply_shrink_expand_noalloc")


def lora_apply_stage(pool: int, seg: int, x: int, y: int, ldx: int, ldy: int, stage: int, stream: int = 0) -> None:
    _check(load_library().lora_apply_stage(pool, seg, x, y, ldx, ldy, stage, stream), "lora_apply_stage")


def lora_apply_fused_projection(pool: int, seg: int, W: int, ldw: int, x: int, y: int, ldx: int, ldy: int,
                                stream: int = 0) -> None:
    _check(load_library().lora_apply_fused_projection(pool, seg, W, ldw, x, y, ldx, ldy, stream),
           "lora_apply_fused_projection")


def lora_fused_projection_stage(pool: int, seg: int, W: int, ldw: int, x: int, y: int, ldx: int, ldy: int,
                                stage: int, stream: int = 0) -> None:
    _check(load_library().lora_fused_projection_stage(pool, seg, W, ldw, x, y, ldx, ldy, stage, stream),
           "lora_fused_projection_stage")


# ------------------------------------------------------------ torch helpers

def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


class LoraPool:
    """A projection's adapter pool in a torch-owned device buffer."""

    def __init__(self, num_slots: int, max_rank: int, d_in: int, lane_d_out: Sequence[int], max_tokens: int,
                 device="cuda", stream=None):
        import torch
        self.num_slots, self.max_rank, self.d_in = num_slots, max_rank, d_in
        self.lane_d_out = list(lane_d_out)
        self.max_tokens = max_tokens
        self.nbytes = lora_pool_bytes(num_slots, max_rank, d_in, self.lane_d_out, max_tokens)
        if self.nbytes == 0:
            raise LoraError(LORA_ERR_SHAPE, "lora_pool_bytes")
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.handle = lora_pool_create(self.buffer.data_ptr(), self.nbytes, num_slots, max_rank, d_in,
                                       self.lane_d_out, max_tokens, _stream(stream))

    @property
    def D(self) -> int:
        return sum(self.lane_d_out)

    def load(self, slot: int, lane: int, A, B, scale: float, stream=None) -> None:
        """A: bf16/uint16/int16 device tensor [r, d_in]; B: [d_out, r]; None unloads."""
        if A is None:
            lora_pool_load(self.handle, slot, lane, 0, 0.0, 0, 0, _stream(stream))
            return
        assert A.is_cuda and B.is_cuda and A.is_contiguous() and B.is_contiguous()
        r = int(A.shape[0])
        assert tuple(A.shape) == (r, self.d_in) and tuple(B.shape) == (self.lane_d_out[lane], r)
        assert A.element_size() == 2 and B.element_size() == 2
        lora_pool_load(self.handle, slot, lane, r, scale, A.data_ptr(), B.data_ptr(), _stream(stream))

    def close(self):
        if getattr(self, "handle", None):
            lora_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LoraSegments:
    """Routing metadata workspace in a torch-owned device buffer."""

    def __init__(self, max_seqs: int, max_tokens: int, num_slots: int, device="cuda"):
        import torch
        self.max_seqs, self.max_tokens, self.num_slots = max_seqs, max_tokens, num_slots
        self.nbytes = lora_segments_bytes(max_seqs, max_tokens, num_slots)
        if self.nbytes == 0:
            raise LoraError(LORA_ERR_SHAPE, "lora_segments_bytes")
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.handle = lora_segments_create(self.buffer.data_ptr(), self.nbytes, max_seqs, max_tokens, num_slots)
        self.num_tokens = 0

    def build(self, adapter_ids, q_seq_lens, num_tokens: Optional[int] = None, stream=None) -> None:
        """adapter_ids, q_seq_lens: int32 device tensors [S] (num_tokens defaults to their host-known sum)."""
        import torch
        assert adapter_ids.dtype == torch.int32 and q_seq_lens.dtype == torch.int32
        assert adapter_ids.is_cuda and q_seq_lens.is_cuda
        S = int(adapter_ids.numel())
        T = int(q_seq_lens.sum().item()) if num_tokens is None else int(num_tokens)
        lora_build_segments(self.handle, adapter_ids.data_ptr(), q_seq_lens.data_ptr(), S, T, _stream(stream))
        self.num_tokens = T

    def build_moe(self, row_expert, row_adapter, row_seq, num_experts: int, num_adapters: int,
                  stream=None) -> None:
        """Dispatched MoE rows: int32 device tensors [num_rows] (expert, adapter, sequence of each row)."""
        import torch
        for t in (row_expert, row_adapter, row_seq):
            assert t.dtype == torch.int32 and t.is_cuda
        n = int(row_expert.numel())
        lora_build_segments_moe(self.handle, row_expert.data_ptr(), row_adapter.data_ptr(), row_seq.data_ptr(), n,
                                num_experts, num_adapters, _stream(stream))
        self.num_tokens = n

    def read(self, stream=None) -> dict:
        return lora_segments_read(self.handle, self.num_tokens, self.num_slots, _stream(stream))

    def status(self, stream=None) -> int:
        return lora_get_status(self.handle, _stream(stream))

    def clear_status(self, stream=None) -> None:
        lora_clear_status(self.handle, _stream(stream))

    def close(self):
        if getattr(self, "handle", None):
            lora_segments_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def apply(pool: LoraPool, seg: LoraSegments, x, y, stream=None) -> None:
    """y += delta for the rows of the last build.  x: bf16 [T, d_in], y: fp32 [T, D] (row-major views)."""
    assert x.is_cuda and y.is_cuda and x.element_size() == 2 and y.element_size() == 4
    assert x.stride(1) == 1 and y.stride(1) == 1
    lora_apply_shrink_expand(pool.handle, seg.handle, x.data_ptr(), y.data_ptr(), x.stride(0), y.stride(0),
                             _stream(stream))


def apply_stage(pool: LoraPool, seg: LoraSegments, x, y, stage: int, stream=None) -> None:
    """One kernel of apply(): 1 = decode path (fused shrink -> expand), 2 = tensor shrink, 3 = tensor expand."""
    lora_apply_stage(pool.handle, seg.handle, x.data_ptr(), y.data_ptr(), x.stride(0), y.stride(0), stage,
                     _stream(stream))


def fused_projection(pool: LoraPool, seg: LoraSegments, W, x, y, stream=None) -> None:
    """y = x @ W^T + delta for every row of the last build (y written, not read).
    W: bf16 [D, d_in], x: bf16 [T, d_in], y: fp32 [T, D] (row-major views)."""
    assert W.is_cuda and x.is_cuda and y.is_cuda
    assert W.element_size() == 2 and x.element_size() == 2 and y.element_size() == 4
    assert W.stride(1) == 1 and x.stride(1) == 1 and y.stride(1) == 1
    lora_apply_fused_projection(pool.handle, seg.handle, W.data_ptr(), W.stride(0), x.data_ptr(), y.data_ptr(),
                                x.stride(0), y.stride(0), _stream(stream))


def fused_projection_stage(pool: LoraPool, seg: LoraSegments, W, x, y, stage: int, stream=None) -> None:
    """One kernel of fused_projection(): 1 = decode shrink, 2 = tensor shrink (both in row mode), 3 = the GEMM."""
    lora_fused_projection_stage(pool.handle, seg.handle, W.data_ptr(), W.stride(0), x.data_ptr(), y.data_ptr(),
                                x.stride(0), y.stride(0), stage, _stream(stream))
