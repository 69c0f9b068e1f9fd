"""Expert parallelism: the E experts split over R ranks, tokens exchanged between them.

The pages place experts on separate GPUs and send tokens between them (arjunjaggi.com "Mixture of
Experts in LLMs", serving section; lensaml.com "Mixture of Experts", Step 6: experts spread across
devices). Rank r owns experts [r E/R, (r+1) E/R) and its own tokens. One forward on rank r:

  1. route its tokens over all E experts and dispatch them: rows grouped by expert, so the rows
     for owner q are the contiguous block [offsets[q E/R], offsets[(q+1) E/R]);
  2. exchange the per-expert row counts (all_to_all), then the rows themselves
     (all_to_all_single with those splits); received rows come grouped by source rank, and within
     a source by expert;
  3. regroup the received rows by local expert (a dispatch with k = 1 whose "expert choice" is
     each row's local expert), run the local experts' FFN, and put the outputs back in received
     order (a combine with k = 1 and gate 1: an exact copy);
  4. send the output rows back along the reverse splits and combine them with the gates in token
     order. The auxiliary value and the z-loss of the whole batch need every rank's counts,
     probability sums and squared log-sum-exp sums (dist.global_aux, dist.global_zloss); forward
     returns this rank's.

Only the exchange lives here; every compute step goes through a backend object:
  route(h) -> (topk_idx [T, k], gates [T, k], psum_part [rows, E + 1]: per-expert partial sums
               of p in columns 0..E-1, of the squared log-sum-exp in column E)
  dispatch(topk_idx, h) -> (counts [E], offsets [E+1], slot_of [T k], x_perm [T k, d])
  local_ffn(rows [n, d], local_expert [n], expert_lo, expert_hi) -> [n, d]
  combine(y_perm [T k, d], slot_of, gates) -> y [T, d]
LibmoeBackend runs them on the GPU through the C ABI (the regroup of step 3 with
moe_build_dispatch and moe_combine). The split sizes of an all_to_all must be known on the host,
so each forward copies the E counts to the host once. With NCCL the rows move between devices
directly; with gloo (a host transport) they are staged through host copies.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B
from . import dist as D


def expert_range(rank: int, world: int, E: int) -> tuple[int, int]:
    """Experts owned by `rank`: [lo, hi) with E split as evenly as possible, lower ranks first."""
    base, extra = divmod(E, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def send_splits(counts: torch.Tensor, world: int) -> list[int]:
    """Rows this rank sends to each owner rank (its routed rows per owner's expert block)."""
    E = counts.numel()
    c = counts.to("cpu", torch.int64)
    return [int(c[lo:hi].sum()) for lo, hi in (expert_range(q, world, E) for q in range(world))]


def exchange_counts(counts: torch.Tensor, world: int) -> torch.Tensor:
    """recv[s, e - lo]: rows source rank s sends this rank for its local expert e (int64, host).
    One all_to_all of each owner's block of the E counts."""
    E = counts.numel()
    rank = dist.get_rank() if D.active() else 0
    lo, hi = expert_range(rank, world, E)
    c = counts.to("cpu", torch.int64)
    if not D.active():
        return c[lo:hi].reshape(1, hi - lo).clone()
    # pad every owner's block to the largest block so one all_to_all_single moves them all
    width = max(h - l for l, h in (expert_range(q, world, E) for q in range(world)))
    send = torch.zeros(world, width, dtype=torch.int64)
    for q in range(world):
        l, h = expert_range(q, world, E)
        send[q, :h - l] = c[l:h]
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    recv = torch.empty_like(send, device=dev)
    dist.all_to_all_single(recv, send.to(dev))
    return recv.cpu()[:, :hi - lo]


def _all_to_all_rows(x: torch.Tensor, out: torch.Tensor, send: list[int],
                     recv: list[int]) -> torch.Tensor:
    """Rows of x go to the ranks in `send` split order; `out` receives `recv` rows per rank.
    NCCL moves device rows directly; gloo (host transport) moves host copies of them."""
    if not D.active():
        out.copy_(x)
    elif x.is_cuda and dist.get_backend() != "nccl":
        staged = torch.empty(out.shape, dtype=out.dtype)
        dist.all_to_all_single(staged, x.contiguous().cpu(), output_split_sizes=recv,
                               input_split_sizes=send)
        out.copy_(staged)
    else:
        dist.all_to_all_single(out, x.contiguous(), output_split_sizes=recv,
                               input_split_sizes=send)
    return out


def forward(backend, h: torch.Tensor, E: int, world: int) -> dict:
    """One expert-parallel forward of this rank's tokens h [T, d] (see the module text)."""
    rank = dist.get_rank() if D.active() else 0
    lo, hi = expert_range(rank, world, E)
    idx, gates, psum = backend.route(h)
    counts, offsets, slot_of, x_perm = backend.dispatch(idx, h)
    # rows kept per expert (fewer than the routed counts when a capacity drops slots)
    off = offsets.to("cpu", torch.int64)
    kept_counts = off[1:] - off[:-1]
    kept = int(off[-1])
    send = send_splits(kept_counts, world)
    recv_counts = exchange_counts(kept_counts, world)          # [world, hi - lo]
    recv = [int(v) for v in recv_counts.sum(1)]
    x_in = torch.empty((sum(recv), x_perm.shape[1]), dtype=x_perm.dtype, device=x_perm.device)
    _all_to_all_rows(x_perm[:kept], x_in, send, recv)
    # local expert of every received row: sources in rank order, experts ascending within each
    local = torch.repeat_interleave(
        torch.arange(hi - lo, dtype=torch.int32).repeat(world), recv_counts.reshape(-1))
    y_in = backend.local_ffn(x_in, local.to(x_in.device), lo, hi)
    y_perm = torch.empty_like(x_perm)  # rows past `kept` are never read (no slot points there)
    _all_to_all_rows(y_in, y_perm[:kept], recv, send)
    y = backend.combine(y_perm, slot_of, gates)
    part = psum.to("cpu", torch.float64).sum(0)
    return dict(y=y, idx=idx, gates=gates, counts=counts, psum=part[:E], lse2=float(part[E]),
                recv_counts=recv_counts)


class LibmoeBackend:
    """The compute steps on the GPU through libmoe's C ABI, for one rank's expert slice."""

    def __init__(self, cfg: B.moe_config_t, weights: dict, world: int):
        self.cfg = cfg
        self.w = weights
        self.world = world
        self.ws = B.workspace(cfg)
        self.dt = torch.bfloat16 if cfg.dtype == B.MOE_BF16 else torch.float32

    def route(self, h):
        c, dev = self.cfg, h.device
        idx = torch.empty((c.T, c.k), dtype=torch.int32, device=dev)
        gates = torch.empty((c.T, c.k), dtype=torch.float32, device=dev)
        psum = torch.empty((B.moe_router_partials(c), c.E + 1), dtype=torch.float32, device=dev)
        B.moe_router_topk(c, h, self.w["W_r"], self.w.get("b_r"), idx, gates, psum, self.ws,
                          sel_bias=self.w.get("sel_bias"))
        return idx, gates, psum

    def dispatch(self, idx, h):
        c, dev = self.cfg, h.device
        P = c.T * c.k
        counts = torch.empty(c.E, dtype=torch.int32, device=dev)
        offsets = torch.empty(c.E + 1, dtype=torch.int32, device=dev)
        sorted_token = torch.empty(P, dtype=torch.int32, device=dev)
        slot_of = torch.empty(P, dtype=torch.int32, device=dev)
        x_perm = torch.empty((P, c.d), dtype=self.dt, device=dev)
        B.moe_build_dispatch(c, idx, h, counts, offsets, sorted_token, slot_of, x_perm, self.ws)
        return counts, offsets, slot_of, x_perm

    def local_ffn(self, rows, local, lo, hi):
        c, n, dev = self.cfg, rows.shape[0], rows.device
        if n == 0:
            return rows.clone()
        El = hi - lo
        # regroup by local expert: a dispatch with k = 1 whose choice is the row's local expert
        lc = B.config(T=n, d=c.d, f=c.f, E=El, k=1, dtype=c.dtype, act=c.act, gate=c.gate,
                      has_bias=bool(c.has_bias))
        ws = B.workspace(lc)
        counts = torch.empty(El, dtype=torch.int32, device=dev)
        offsets = torch.empty(El + 1, dtype=torch.int32, device=dev)
        sorted_row = torch.empty(n, dtype=torch.int32, device=dev)
        slot_of = torch.empty(n, dtype=torch.int32, device=dev)
        grouped = torch.empty_like(rows)
        B.moe_build_dispatch(lc, local.reshape(n, 1).contiguous(), rows, counts, offsets,
                             sorted_row, slot_of, grouped, ws)
        sl = slice(lo, hi)
        w = self.w
        y_grouped = torch.empty_like(rows)
        B.moe_expert_ffn(lc, grouped, offsets, w["W1"][sl], None if w.get("b1") is None
                         else w["b1"][sl], None if w.get("W3") is None else w["W3"][sl],
                         w["W2"][sl], None if w.get("b2") is None else w["b2"][sl], y_grouped, ws)
        # back to received order: a combine with k = 1 and gate 1 copies each row exactly
        ones = torch.ones((n, 1), dtype=torch.float32, device=dev)
        out = torch.empty_like(rows)
        B.moe_combine(lc, y_grouped, slot_of, ones, out)
        return out

    def combine(self, y_perm, slot_of, gates):
        c = self.cfg
        y = torch.empty((c.T, c.d), dtype=self.dt, device=y_perm.device)
        B.moe_combine(c, y_perm, slot_of, gates, y)
        return y
