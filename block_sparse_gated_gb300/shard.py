"""Head partition of one attention layer across ranks (one GPU per rank).

The gated prefill of a layer splits into independent pieces along the KV
heads: q-head h reads only KV head h // (Hq/Hkv), and its threshold row
T[h] is its own, so a rank that owns a contiguous range of KV heads, with
the query heads that read them and those heads' threshold rows, computes its
part of the layer with no data from any other rank (the way tensor
parallelism already shards attention heads).  No collective is needed inside
attention; only the timing is reduced across ranks.

Host logic only: no device code, no attention arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class HeadShard:
    """The part of a layer that one rank computes."""
    rank: int
    world: int
    kv_heads: range      # KV heads this rank owns
    q_heads: range       # query heads that read them (threshold rows too)

    @property
    def num_heads_kv(self) -> int:
        return len(self.kv_heads)

    @property
    def num_heads_q(self) -> int:
        return len(self.q_heads)


def head_shard(num_heads_q: int, num_heads_kv: int, rank: int, world: int) -> HeadShard:
    """Contiguous, balanced split of the KV heads over ``world`` ranks: the
    first ``Hkv % world`` ranks own one KV head more than the rest.  Every
    rank owns at least one KV head (``world <= Hkv``); a KV head is never
    split, so its K/V tiles are read by one rank only."""
    if num_heads_kv <= 0 or num_heads_q % num_heads_kv:
        raise ValueError("num_heads_q must be a positive multiple of num_heads_kv")
    if not 1 <= world <= num_heads_kv:
        raise ValueError(f"world size {world} must be between 1 and the {num_heads_kv} KV heads")
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside [0, {world})")
    g = num_heads_q // num_heads_kv
    base, extra = divmod(num_heads_kv, world)
    a = rank * base + min(rank, extra)
    b = a + base + (1 if rank < extra else 0)
    return HeadShard(rank, world, range(a, b), range(a * g, b * g))


def shard_tensors(shard: HeadShard, q, k, v, thresholds=None, head_dim_axis: int = -3):
    """Views of one rank's heads: q [..., Hq, L, d] -> its query heads,
    k, v [..., Hkv, L, d] -> its KV heads, thresholds [Hq, nT] (or
    [budgets, Hq, nT]) -> its query heads' rows.  ``head_dim_axis`` is the
    head axis of q, k and v (-3 for the [.., H, L, d] layouts)."""
    def cut(t, r):
        return t.narrow(head_dim_axis, r.start, len(r))

    qs, ks, vs = cut(q, shard.q_heads), cut(k, shard.kv_heads), cut(v, shard.kv_heads)
    ts = None
    if thresholds is not None:
        ts = thresholds.narrow(thresholds.dim() - 2, shard.q_heads.start, len(shard.q_heads))
    return qs, ks, vs, ts
