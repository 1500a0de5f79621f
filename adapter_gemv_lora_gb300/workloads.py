"""Seeded synthetic inputs for the mixed-adapter LoRA delta.

This module only draws numbers: routing metadata (per-sequence adapter slot
and query length), per-slot ranks and scales, bf16 factor bit patterns, bf16
activations and the fp32 base output.  It holds none of the delta's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it without sharing any of the method.

Workload shapes follow the pages' serving setting:
  * one adapter id per sequence, index-aligned with the query lengths, and a
    per-token slot obtained from them (xLLM PR #2014, "Wire-up",
    ModelInputParams::adapter_ids / adapter_ids_per_token);
  * slot 0 is the base model (tokenspeed PR #976, RequestSpec::lora_id, 0 =
    base);
  * r=16, lora_alpha=32 as in the xLLM validation paragraph, scale = alpha / r
    (PEFT convention; the pages give no other formula);
  * A is [r, d_in] and B is [d_out, r] (xLLM PR #2014, LoRAQKVParallelLinear:
    B.size(0) is the lane's output width).

Value laws: A ~ N(0, 1/d_in), B ~ N(0, 1/r), x ~ N(0, 1), y0 ~ N(0, 1), all
drawn in float32 with numpy's PCG64 and then rounded to bf16 (round to
nearest, ties to even) where the tensor is bf16.  Draw order: metadata, ranks,
then per projection A, B, x, y0.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "Projection",
    "Workload",
    "bf16_bits",
    "bf16_bits_to_f32",
    "zipf_probs",
    "make_workload",
    "custom_workload",
    "CONFIG_NAMES",
    "MoeProjection",
    "MoeWorkload",
    "MOE_CONFIG_NAMES",
    "make_moe_workload",
    "projection_weight",
]


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    bias = ((b >> 16) & 1) + 0x7FFF
    return ((b + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def zipf_probs(num: int, s: float = 1.1) -> np.ndarray:
    """Finite Zipf law over ranks 1..num: P(k) proportional to k**-s."""
    k = np.arange(1, num + 1, dtype=np.float64)
    w = k ** (-s)
    return w / w.sum()


@dataclass
class Projection:
    """One LoRA-edited projection: its lanes, factors and activations.

    A[k][l] is a uint16 bf16 array [rank[k][l], d_in] (None when the rank is 0),
    B[k][l] a uint16 bf16 array [lane_d_out[l], rank[k][l]].  x is [T, d_in]
    bf16 bits, y0 is [T, D] float32 with D = sum(lane_d_out).
    """

    name: str
    d_in: int
    lane_d_out: List[int]
    rank: np.ndarray          # int32 [N, L]
    scale: np.ndarray         # float32 [N, L]
    A: list                   # [N][L] -> uint16 [r, d_in] or None
    B: list                   # [N][L] -> uint16 [d_out_l, r] or None
    x: np.ndarray             # uint16 [T, d_in]
    y0: np.ndarray            # float32 [T, D]
    max_rank: int

    @property
    def num_lanes(self) -> int:
        return len(self.lane_d_out)

    @property
    def D(self) -> int:
        return int(sum(self.lane_d_out))

    @property
    def lane_offsets(self) -> List[int]:
        off, acc = [], 0
        for d in self.lane_d_out:
            off.append(acc)
            acc += d
        return off


@dataclass
class Workload:
    name: str
    adapter_ids: np.ndarray   # int32 [S]
    q_seq_lens: np.ndarray    # int32 [S]
    num_slots: int            # N, slot 0 included
    projections: List[Projection] = field(default_factory=list)

    @property
    def S(self) -> int:
        return int(self.adapter_ids.shape[0])

    @property
    def T(self) -> int:
        return int(self.q_seq_lens.sum())

    def per_token_slot(self) -> np.ndarray:
        """Token-level slot ids (np.repeat of the per-sequence ids)."""
        return np.repeat(self.adapter_ids, self.q_seq_lens).astype(np.int32)


def _draw_projection(rng, name, d_in, lane_d_out, rank, alpha, T, max_rank,
                     strength: float = 1.0, draw_xy: bool = True) -> Projection:
    N, L = rank.shape
    scale = np.zeros((N, L), dtype=np.float32)
    A = [[None] * L for _ in range(N)]
    B = [[None] * L for _ in range(N)]
    for k in range(1, N):
        for l in range(L):
            r = int(rank[k, l])
            if r > 0:
                scale[k, l] = np.float32(alpha[k, l] / r * strength)
    for k in range(1, N):
        for l in range(L):
            r = int(rank[k, l])
            if r > 0:
                A[k][l] = bf16_bits(rng.standard_normal((r, d_in), dtype=np.float32)
                                    * np.float32(1.0 / np.sqrt(d_in)))
    for k in range(1, N):
        for l in range(L):
            r = int(rank[k, l])
            if r > 0:
                B[k][l] = bf16_bits(rng.standard_normal((lane_d_out[l], r), dtype=np.float32)
                                    * np.float32(1.0 / np.sqrt(r)))
    D = int(sum(lane_d_out))
    if draw_xy:
        x = bf16_bits(rng.standard_normal((T, d_in), dtype=np.float32))
        y0 = rng.standard_normal((T, D), dtype=np.float32)
    else:
        x = np.zeros((T, d_in), dtype=np.uint16)
        y0 = np.zeros((T, D), dtype=np.float32)
    return Projection(name=name, d_in=d_in, lane_d_out=list(lane_d_out), rank=rank.astype(np.int32),
                      scale=scale, A=A, B=B, x=x, y0=y0, max_rank=max_rank)


def _base_rows_by_permutation(rng, S: int, n_base: int, n_slots: int, probs=None) -> np.ndarray:
    perm = rng.permutation(S)
    ids = np.zeros(S, dtype=np.int32)
    rest = perm[n_base:]
    if probs is None:
        ids[rest] = rng.integers(1, n_slots, size=rest.shape[0])
    else:
        ids[rest] = rng.choice(n_slots - 1, size=rest.shape[0], p=probs) + 1
    return ids


def _adjust_lengths(lengths: np.ndarray, target: int, lo: int, hi: int) -> np.ndarray:
    """Round-robin +-1 adjustment of chunk lengths toward a target sum, within [lo, hi]."""
    lengths = lengths.astype(np.int64).copy()
    i = 0
    n = lengths.shape[0]
    guard = 0
    while lengths.sum() != target:
        step = 1 if lengths.sum() < target else -1
        v = lengths[i] + step
        if lo <= v <= hi:
            lengths[i] = v
        i = (i + 1) % n
        guard += 1
        if guard > 100 * n * (hi - lo + 1):
            raise ValueError("length adjustment cannot reach the target")
    return lengths


CONFIG_NAMES = ["tiny", "decode_oproj", "prefill_qkv", "mlp_decode", "cont_batch"]


def make_workload(name: str, seed: int = 0, draw_xy: bool = True) -> Workload:
    """The five synthetic workloads, by name (or index 0..4).

    tiny          8 single-token rows, 256 -> 256, 4 slots of rank 8, alpha 16
    decode_oproj  256 single-token rows, o_proj 4096 -> 4096, 8 adapters r=16 a=32,
                  exactly 20 % (51) base rows, the rest uniform over slots 1..8
    prefill_qkv   16 sequences, lengths U{128..2048}, fused QKV 4096 -> q 4096 /
                  k 1024 / v 1024 (GQA, 32 q heads, 8 kv heads, head_dim 128),
                  rank 16 per lane, alpha 32, slot per sequence uniform {0..8}
    mlp_decode    512 single-token rows, gate_up 4096 -> 2x14336 then down
                  14336 -> 4096, 32 adapters, per-slot rank from {8,16,32,64}
                  padded to 64, alpha 2r, Zipf(1.1) popularity, 15 % (77) base rows
    cont_batch    128 sequences, 16384 rows: 104 decode rows plus 24 prefill
                  chunks of U{128..1024} tokens adjusted to sum to 16280,
                  7168 -> 7168, 64 adapters with ranks from {16,32,64,128}
                  (max 128), alpha 2r, Zipf(1.1), a sequence is base w.p. 0.25
    """
    if isinstance(name, int):
        name = CONFIG_NAMES[name]
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        S, N, R = 8, 4, 8
        q = np.ones(S, dtype=np.int32)
        ids = rng.integers(0, N, size=S).astype(np.int32)
        rank = np.zeros((N, 1), dtype=np.int32)
        rank[1:, 0] = 8
        alpha = np.full((N, 1), 16.0)
        wl = Workload(name, ids, q, N)
        wl.projections.append(_draw_projection(rng, "proj", 256, [256], rank, alpha, wl.T, R, draw_xy=draw_xy))
        return wl
    if name == "decode_oproj":
        S, N, R = 256, 9, 16
        q = np.ones(S, dtype=np.int32)
        ids = _base_rows_by_permutation(rng, S, 51, N)
        rank = np.zeros((N, 1), dtype=np.int32)
        rank[1:, 0] = 16
        alpha = np.full((N, 1), 32.0)
        wl = Workload(name, ids, q, N)
        wl.projections.append(_draw_projection(rng, "o_proj", 4096, [4096], rank, alpha, wl.T, R, draw_xy=draw_xy))
        return wl
    if name == "prefill_qkv":
        S, N, R = 16, 9, 16
        q = rng.integers(128, 2049, size=S).astype(np.int32)
        ids = rng.integers(0, N, size=S).astype(np.int32)
        rank = np.zeros((N, 3), dtype=np.int32)
        rank[1:, :] = 16
        alpha = np.full((N, 3), 32.0)
        wl = Workload(name, ids, q, N)
        wl.projections.append(_draw_projection(rng, "qkv_proj", 4096, [4096, 1024, 1024], rank, alpha,
                                               wl.T, R, draw_xy=draw_xy))
        return wl
    if name == "mlp_decode":
        S, N, R = 512, 33, 64
        q = np.ones(S, dtype=np.int32)
        ids = _base_rows_by_permutation(rng, S, 77, N, probs=zipf_probs(N - 1, 1.1))
        per_slot = np.zeros(N, dtype=np.int32)
        per_slot[1:] = rng.choice(np.array([8, 16, 32, 64]), size=N - 1)
        wl = Workload(name, ids, q, N)
        rank2 = np.repeat(per_slot[:, None], 2, axis=1)
        rank1 = per_slot[:, None].copy()
        wl.projections.append(_draw_projection(rng, "gate_up_proj", 4096, [14336, 14336], rank2,
                                               2.0 * rank2, wl.T, R, draw_xy=draw_xy))
        wl.projections.append(_draw_projection(rng, "down_proj", 14336, [4096], rank1,
                                               2.0 * rank1, wl.T, R, draw_xy=draw_xy))
        return wl
    if name == "cont_batch":
        S, N, R = 128, 65, 128
        n_dec, n_chunk = 104, 24
        chunk = rng.integers(128, 1025, size=n_chunk)
        chunk = _adjust_lengths(chunk, 16384 - n_dec, 128, 1024)
        lens = np.concatenate([np.ones(n_dec, dtype=np.int64), chunk])
        order = rng.permutation(S)
        q = lens[order].astype(np.int32)
        base = rng.random(S) < 0.25
        z = rng.choice(N - 1, size=S, p=zipf_probs(N - 1, 1.1)) + 1
        ids = np.where(base, 0, z).astype(np.int32)
        per_slot = np.zeros(N, dtype=np.int32)
        per_slot[1:] = rng.choice(np.array([16, 32, 64, 128]), size=N - 1)
        rank = per_slot[:, None].copy()
        wl = Workload(name, ids, q, N)
        wl.projections.append(_draw_projection(rng, "proj", 7168, [7168], rank, 2.0 * rank, wl.T, R,
                                               draw_xy=draw_xy))
        return wl
    raise KeyError(name)


def custom_workload(q_seq_lens: Sequence[int], adapter_ids: Sequence[int], d_in: int,
                    lane_d_out: Sequence[int], num_slots: int, max_rank: int,
                    rank: Optional[np.ndarray] = None, alpha: Optional[np.ndarray] = None,
                    seed: int = 0, strength: float = 1.0) -> Workload:
    """A workload with caller-chosen metadata and shapes (values drawn as above).

    rank defaults to max_rank for every adapter slot and lane; alpha to 2 * rank.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = np.asarray(q_seq_lens, dtype=np.int32)
    ids = np.asarray(adapter_ids, dtype=np.int32)
    L = len(lane_d_out)
    if rank is None:
        rank = np.zeros((num_slots, L), dtype=np.int32)
        rank[1:, :] = max_rank
    rank = np.asarray(rank, dtype=np.int32).reshape(num_slots, L)
    if alpha is None:
        alpha = 2.0 * rank
    wl = Workload("custom", ids, q, num_slots)
    wl.projections.append(_draw_projection(rng, "proj", d_in, list(lane_d_out), rank,
                                           np.asarray(alpha, dtype=np.float64).reshape(num_slots, L),
                                           int(q.sum()), max_rank, strength=strength))
    return wl


def projection_weight(proj, seed: int = 1) -> np.ndarray:
    """The base projection's weight for the fused form, as a linear layer
    stores it: bf16 bits [D][d_in] (output feature, input feature), the lanes
    stacked in lane order, drawn N(0, 1/d_in) from its own PCG64 stream (so the
    projection's other tensors stay as they were)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((proj.D, proj.d_in), dtype=np.float32) * np.float32(1.0 / np.sqrt(proj.d_in))
    return bf16_bits(w)


# ---------------------------------------------------------------- MoE layers
#
# Expert LoRA of an MoE layer (xLLM PR #2014 lists the fused MoE expert LoRA
# delta as the next step; its validation model is a 30B-A3B MoE with r=16,
# alpha=32).  Every expert has its own factors per adapter.  Tokens choose
# top_k distinct experts; the dispatched rows (one per (token, expert)) are
# grouped by expert, tokens in order inside an expert, as an MoE layer lays
# them out before its expert GEMMs.


@dataclass
class MoeProjection:
    """One expert projection: factors per (expert, adapter, lane) and the
    dispatched rows' activations and base outputs.

    A[e][a][l] uint16 bf16 [rank[a][l], d_in] (None for adapter 0 or rank 0),
    B[e][a][l] uint16 bf16 [lane_d_out[l], rank[a][l]]; rank and scale are per
    adapter (shared by the experts); x [R, d_in] bf16 bits, y0 [R, D] float32.
    """

    name: str
    d_in: int
    lane_d_out: List[int]
    rank: np.ndarray          # int32 [A + 1, L]
    scale: np.ndarray         # float32 [A + 1, L]
    A: list
    B: list
    x: np.ndarray
    y0: np.ndarray
    max_rank: int

    @property
    def num_lanes(self) -> int:
        return len(self.lane_d_out)

    @property
    def D(self) -> int:
        return int(sum(self.lane_d_out))


@dataclass
class MoeWorkload:
    name: str
    seq_lens: np.ndarray      # int32 [S] tokens per sequence
    seq_adapter: np.ndarray   # int32 [S] adapter of each sequence (0 = base)
    num_experts: int
    num_adapters: int         # adapters 1..A
    top_k: int
    row_token: np.ndarray     # int32 [R] token of each dispatched row
    row_expert: np.ndarray    # int32 [R]
    row_seq: np.ndarray       # int32 [R]
    row_adapter: np.ndarray   # int32 [R]
    projections: List[MoeProjection] = field(default_factory=list)

    @property
    def R(self) -> int:
        return int(self.row_expert.shape[0])

    @property
    def T(self) -> int:
        return int(self.seq_lens.sum())


MOE_CONFIG_NAMES = ["moe_decode", "moe_prefill"]


def _draw_moe_projection(rng, name, d_in, lane_d_out, E, A, rank, alpha, R, max_rank) -> MoeProjection:
    L = len(lane_d_out)
    scale = np.zeros((A + 1, L), dtype=np.float32)
    for a in range(1, A + 1):
        for l in range(L):
            if rank[a, l] > 0:
                scale[a, l] = np.float32(alpha[a, l] / rank[a, l])
    Af = [[[None] * L for _ in range(A + 1)] for _ in range(E)]
    Bf = [[[None] * L for _ in range(A + 1)] for _ in range(E)]
    for e in range(E):
        for a in range(1, A + 1):
            for l in range(L):
                r = int(rank[a, l])
                if r > 0:
                    Af[e][a][l] = bf16_bits(rng.standard_normal((r, d_in), dtype=np.float32)
                                            * np.float32(1.0 / np.sqrt(d_in)))
                    Bf[e][a][l] = bf16_bits(rng.standard_normal((lane_d_out[l], r), dtype=np.float32)
                                            * np.float32(1.0 / np.sqrt(r)))
    D = int(sum(lane_d_out))
    x = bf16_bits(rng.standard_normal((R, d_in), dtype=np.float32))
    y0 = rng.standard_normal((R, D), dtype=np.float32)
    return MoeProjection(name, d_in, list(lane_d_out), rank.astype(np.int32), scale, Af, Bf, x, y0, max_rank)


def moe_workload(name, seq_lens, seq_adapter, num_experts, num_adapters, top_k, d_model, d_expert,
                 rank_per_adapter, seed=0) -> MoeWorkload:
    """Routing (top_k distinct experts per token, uniform), the dispatch order
    (rows grouped by expert, tokens in order) and the expert projections
    gate_up (d_model -> 2 x d_expert) and down (d_expert -> d_model)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    seq_adapter = np.asarray(seq_adapter, dtype=np.int32)
    T = int(seq_lens.sum())
    tok_seq = np.repeat(np.arange(seq_lens.shape[0], dtype=np.int32), seq_lens)
    choice = np.stack([rng.choice(num_experts, size=top_k, replace=False) for _ in range(T)]).astype(np.int32)
    tok = np.repeat(np.arange(T, dtype=np.int32), top_k)
    exp = choice.reshape(-1)
    order = np.lexsort((tok, exp))  # by expert, then token
    row_token, row_expert = tok[order].astype(np.int32), exp[order].astype(np.int32)
    row_seq = tok_seq[row_token]
    row_adapter = seq_adapter[row_seq]
    wl = MoeWorkload(name, seq_lens, seq_adapter, num_experts, num_adapters, top_k, row_token, row_expert,
                     row_seq.astype(np.int32), row_adapter.astype(np.int32))
    R = wl.R
    rank = np.zeros((num_adapters + 1, 1), dtype=np.int32)
    rank[1:, 0] = np.asarray(rank_per_adapter, dtype=np.int32)
    rank2 = np.repeat(rank, 2, axis=1)
    wl.projections.append(_draw_moe_projection(rng, "experts.gate_up_proj", d_model, [d_expert, d_expert],
                                               num_experts, num_adapters, rank2, 2.0 * rank2, R,
                                               int(rank.max())))
    wl.projections.append(_draw_moe_projection(rng, "experts.down_proj", d_expert, [d_model], num_experts,
                                               num_adapters, rank, 2.0 * rank, R, int(rank.max())))
    return wl


def make_moe_workload(name: str, seed: int = 0) -> MoeWorkload:
    """Expert-LoRA workloads on a 30B-A3B-class MoE layer (128 experts, top 8,
    d_model 2048, expert width 768), 8 adapters of rank 16 (alpha 32):

    moe_decode   256 single-token sequences (2048 dispatched rows), 20 % (51)
                 base sequences by permutation, the rest uniform over 1..8
    moe_prefill  2 prompt chunks of 1024 tokens (16384 dispatched rows; a
                 chunk's tokens that chose one expert, about 64 rows, sit on
                 both sides of the tensor-path threshold), adapters 1 and 2
    """
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    E, A, k = 128, 8, 8
    if name == "moe_decode":
        S = 256
        lens = np.ones(S, dtype=np.int32)
        ids = _base_rows_by_permutation(rng, S, 51, A + 1)
    elif name == "moe_prefill":
        lens = np.array([1024, 1024], dtype=np.int32)
        ids = np.array([1, 2], dtype=np.int32)
    else:
        raise KeyError(name)
    return moe_workload(name, lens, ids, E, A, k, 2048, 768, [16] * A, seed=seed)
