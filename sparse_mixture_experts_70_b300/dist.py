"""Multi-process host logic: one process per GPU, torch.distributed for the few host exchanges.

The layer forward shards by tokens with no exchange on its data path: every rank runs the whole
layer on its own batch. Two things need the other ranks:
  * timing -- the slowest rank's time bounds the job (``max_over_ranks``), and the job's
    throughput is all ranks' tokens over that time (``job_tokens_per_s``);
  * the auxiliary value of a global batch split over ranks by tokens. With f_e = counts_e/(T k)
    and P_e = (1/T) sum_t p[t,e] over the WHOLE batch (lensaml.com "Mixture of Experts", Step 4),
    each rank contributes its routed counts and its per-expert sums of p; one all-reduce of
    2E + 1 numbers gives the global value (``global_aux``). The router z-loss of the whole batch
    likewise needs each rank's sum of squared log-sum-exp and its token count (``global_zloss``).
Everything here works with any backend (NCCL on GPUs, gloo on CPU for the tests).
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the launcher's environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str, device: torch.device | None = None) -> None:
    """Join the process group the launcher describes (MASTER_ADDR / MASTER_PORT env)."""
    if dist.is_initialized():
        return
    kw = {}
    if device is not None and device.type == "cuda":
        kw["device_id"] = device
    dist.init_process_group(backend, **kw)


def active() -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier() -> None:
    if active():
        dist.barrier()


def max_over_ranks(values: list[float], device: torch.device | str = "cpu") -> list[float]:
    """Element-wise maximum of `values` over all ranks (identity with one process)."""
    if not active():
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_slowest: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time per step."""
    return tokens_per_rank * world / (ms_slowest * 1e-3)


def global_aux(counts: torch.Tensor, psum: torch.Tensor, tokens: int, k: int) -> float:
    """E . sum_e f_e P_e of the batch formed by all ranks' tokens.

    counts [E] int: slots this rank routed to each expert; psum [E] float: this rank's per-expert
    sums of the router probability over its tokens (the column sums of psum_part); tokens: this
    rank's token count. Reduced in float64.
    """
    E = counts.numel()
    buf = torch.cat([counts.double().cpu().reshape(-1), psum.double().cpu().reshape(-1),
                     torch.tensor([float(tokens)], dtype=torch.float64)])
    if active():
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        buf = buf.to(dev)
        dist.all_reduce(buf, op=dist.ReduceOp.SUM)
        buf = buf.cpu()
    T = buf[2 * E].item()
    if T == 0:
        return 0.0
    f = buf[:E] / (T * k)
    P = buf[E:2 * E] / T
    return float(E * (f * P).sum().item())


def global_zloss(lse2_sum: float, tokens: int) -> float:
    """Router z-loss of the batch formed by all ranks' tokens: (sum of (log sum_e exp z)^2 over
    every rank's tokens) / (all tokens). lse2_sum is this rank's sum (column E of psum_part,
    summed over rows); one all-reduce of 2 numbers, in float64."""
    buf = torch.tensor([float(lse2_sum), float(tokens)], dtype=torch.float64)
    if active():
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        buf = buf.to(dev)
        dist.all_reduce(buf, op=dist.ReduceOp.SUM)
        buf = buf.cpu()
    return float(buf[0] / buf[1]) if buf[1] > 0 else 0.0


def shutdown() -> None:
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
