"""Cross-rank checks for a data-parallel job that builds one owner map per rank.

DeepSpeed issue #8700, "Design points": the owner map needs no communication
to build, but it must come out identical on every rank, because it decides
which collective each bucket entry uses and every rank has to issue the same
sequence.  `check_owner_map` exchanges the map's 64-bit digest over
torch.distributed (any backend) before the first flush and raises on every
rank when a rank built its map from different metadata.
"""
from __future__ import annotations

from . import DpredError, OwnerMap


def check_owner_map(omap: OwnerMap, group=None, device: str = "cpu") -> int:
    """All ranks of `group` agree on the owner map, or DpredError(MISMATCH) is
    raised on all of them.  Returns the agreed digest.  `device` is where the
    exchange tensor lives ("cuda" for NCCL)."""
    import torch
    import torch.distributed as dist
    digest = omap.digest()
    ws = dist.get_world_size(group)
    mine = torch.tensor([digest & 0x7FFFFFFFFFFFFFFF, digest >> 63], dtype=torch.int64, device=device)
    everyone = [torch.empty_like(mine) for _ in range(ws)]
    dist.all_gather(everyone, mine, group=group)
    got = [int(t[0].item()) | (int(t[1].item()) << 63) for t in everyone]
    bad = [r for r, d in enumerate(got) if d != got[0]]
    if bad:
        raise DpredError(-4, f"owner map differs between ranks: rank(s) {bad} disagree with rank 0 "
                             f"(digests {[hex(d) for d in got]})")
    return got[0]
