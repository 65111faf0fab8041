"""Head sharding of one tree's attention across ranks.

Tree attention has no exchange between kv-head groups: q head h reads only kv head
h // (Hq / Hkv), and the plan (order, positions, tile table) depends on the tree alone.  So
p ranks can split one tree by kv-head groups: each rank holds the plan (built from the same
parent / node_len arrays), its Hkv / p kv heads and the Hq / p q heads that read them, and
runs the ordinary single-GPU path on those heads.  Nothing crosses ranks in the forward or
the backward; a tensor-parallel QKV projection already produces each rank's heads as its own
contiguous [N, H / p, d] tensors, which is the layout the library takes.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class HeadShard:
    rank: int
    world: int
    q0: int          # first global q head of this rank
    q1: int          # one past its last
    kv0: int         # first global kv head
    kv1: int

    @property
    def Hq(self) -> int:
        return self.q1 - self.q0

    @property
    def Hkv(self) -> int:
        return self.kv1 - self.kv0


def kv_head_shard(Hq: int, Hkv: int, rank: int, world: int) -> HeadShard:
    """Rank `rank` of `world` takes kv heads [rank Hkv / world, (rank + 1) Hkv / world) and the q
    heads of their groups.  Requires Hq % Hkv == 0 and Hkv % world == 0 (every rank keeps
    whole groups, so the local GQA mapping h -> h // (Hq / Hkv) is the global one shifted)."""
    if Hq <= 0 or Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq = {Hq} must be a positive multiple of Hkv = {Hkv}")
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if Hkv % world != 0:
        raise ValueError(f"{Hkv} kv heads do not split evenly over {world} ranks")
    per = Hkv // world
    grp = Hq // Hkv
    return HeadShard(rank=rank, world=world, q0=rank * per * grp, q1=(rank + 1) * per * grp, kv0=rank * per,
                     kv1=(rank + 1) * per)
