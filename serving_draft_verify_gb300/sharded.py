"""Request-sharded prefix scheduling over several ranks.

Algorithm 1 (DeepSpec walkthrough, section 3.3 flowchart) sorts *all*
(request, position) pairs of the batch by survival, so when one logical batch
is split by request over G ranks (each rank drafting and verifying its own
requests), the scheduler needs one exchange: every rank contributes its
survivals a [B_r, gamma], all ranks gather the whole [B, gamma] in rank order,
run the same bit-exact scheduler on it, and keep the prefix lengths of their
own requests.  N and Theta_best are the batch's and identical on every rank.

This module is the host side of that exchange (argument marshalling and one
all-gather through torch.distributed: NCCL for CUDA tensors, gloo for CPU
ones); the scheduling itself is the caller's `schedule` callable, normally
the CUDA library's dspark_schedule_prefix.
"""
import torch
import torch.distributed as dist


def gather_survivals(a_local, group=None):
    """All-gather the per-rank survivals [B_r, gamma] (B_r may differ by rank).

    Returns (a_full [B, gamma] in rank order, offsets [G + 1] with rank r's
    requests at rows offsets[r] .. offsets[r + 1] - 1)."""
    world = dist.get_world_size(group)
    dev = a_local.device
    B_r, G = a_local.shape
    sizes = [torch.zeros(1, dtype=torch.int64, device=dev) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([B_r], dtype=torch.int64, device=dev), group=group)
    sizes = [int(x.item()) for x in sizes]
    width = max(sizes)
    padded = torch.zeros((width, G), dtype=a_local.dtype, device=dev)
    padded[:B_r] = a_local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    a_full = torch.cat([p[:n] for p, n in zip(parts, sizes)], dim=0).contiguous()
    offsets = [0]
    for n in sizes:
        offsets.append(offsets[-1] + n)
    return a_full, offsets


def schedule_sharded(a_local, sps, schedule, group=None):
    """This rank's l* after scheduling the whole batch.

    a_local [B_r, gamma] float32 survivals of this rank's requests; sps the
    batch's table [B (gamma + 1) + 1] (B = sum of B_r); schedule(a_full, sps)
    -> dict(ell [B], n_sched, theta).  Returns dict(ell [B_r] of this rank,
    n_sched, theta) with the batch's N and Theta_best."""
    a_full, offsets = gather_survivals(a_local, group)
    B, G = a_full.shape
    if sps.numel() != B * (G + 1) + 1:
        raise ValueError(f"sps has {sps.numel()} entries, the batch needs {B * (G + 1) + 1}")
    out = schedule(a_full, sps)
    r = dist.get_rank(group)
    return dict(ell=out["ell"][offsets[r]:offsets[r + 1]], n_sched=out["n_sched"], theta=out["theta"])
