"""Sharded quantize-then-all-gather weight synchronization.

FP8-RL summary page, section 3.4.2 ("Dynamic Weight Synchronization Pipeline",
Phase 2): every RL step the trainer's updated BF16 weights, sharded across
ranks by FSDP, are gathered, quantized blockwise to E4M3 and handed to the
inference engine.  Gathering BF16 and then quantizing moves 2 bytes per
weight over the interconnect; here each rank first quantizes the rows it
owns (the library's multi-tensor kernel, one launch for all its shards) and
the ranks then all-gather the E4M3 codes and FP32 block scales, about half
the bytes.  Ownership is whole 128-row block bands
(``fp8rl_weight_shard_rows``), so no 128 x 128 block spans two ranks and the
gathered result equals the single-rank quantization of the whole tensor bit
for bit.

The exchange is ``torch.distributed.all_gather_into_tensor`` on one flat
buffer per dtype (codes of all tensors, then scales), each rank's piece padded
to the largest piece.  This module does no arithmetic of the method; it plans
shards, packs, and unpacks.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import binding


def plan(shapes: Sequence[Tuple[int, int]], world: int):
    """Per rank, per tensor: (row_begin, row_end) of its shard."""
    return [[binding.weight_shard_rows(n, world, r) for (n, _) in shapes] for r in range(world)]


def _piece_sizes(shapes, rows):
    """Bytes of codes and FP32 scales of one rank's shards (in tensor order)."""
    nq = sum((e - b) * k for (b, e), (_, k) in zip(rows, shapes))
    ns = sum(((e - b + 127) // 128) * ((k + 127) // 128) for (b, e), (_, k) in zip(rows, shapes))
    return nq, ns


def pack_piece(qs: Sequence[torch.Tensor], ss: Sequence[torch.Tensor], q_len: int, s_len: int,
               device) -> Tuple[torch.Tensor, torch.Tensor]:
    """One rank's codes and scales as flat buffers of q_len / s_len entries."""
    q = torch.zeros(q_len, dtype=torch.uint8, device=device)
    s = torch.zeros(s_len, dtype=torch.float32, device=device)
    oq = os_ = 0
    for qt, st in zip(qs, ss):
        q[oq:oq + qt.numel()] = qt.reshape(-1)
        s[os_:os_ + st.numel()] = st.reshape(-1)
        oq += qt.numel()
        os_ += st.numel()
    return q, s


def assemble(shapes: Sequence[Tuple[int, int]], plans, q_pieces: Sequence[torch.Tensor],
             s_pieces: Sequence[torch.Tensor]):
    """Full codes [n, k] and scales [ceil(n/128), ceil(k/128)] of every tensor
    from the ranks' flat pieces (rank order)."""
    device = q_pieces[0].device
    out_q = [torch.empty(n, k, dtype=torch.uint8, device=device) for (n, k) in shapes]
    out_s = [torch.empty((n + 127) // 128, (k + 127) // 128, dtype=torch.float32, device=device)
             for (n, k) in shapes]
    for r, rows in enumerate(plans):
        oq = os_ = 0
        for i, ((b, e), (n, k)) in enumerate(zip(rows, shapes)):
            cnt = (e - b) * k
            out_q[i][b:e] = q_pieces[r][oq:oq + cnt].view(e - b, k)
            oq += cnt
            kb = (k + 127) // 128
            nb = (e - b + 127) // 128
            out_s[i][b // 128:b // 128 + nb] = s_pieces[r][os_:os_ + nb * kb].view(nb, kb)
            os_ += nb * kb
    return out_q, out_s


def quantize_local(shards: Sequence[torch.Tensor]):
    """The library's multi-tensor re-quantization of this rank's shards."""
    live = [i for i, w in enumerate(shards) if w.shape[0] > 0]
    qs = [torch.empty(w.shape, dtype=torch.uint8, device=w.device) for w in shards]
    ss = [torch.empty((w.shape[0] + 127) // 128, (w.shape[1] + 127) // 128, dtype=torch.float32,
                      device=w.device) for w in shards]
    if live:
        binding.quantize_weights_blockwise_multi([shards[i] for i in live], [qs[i] for i in live],
                                                 [ss[i] for i in live])
    return qs, ss


def sync_weights(shards: Sequence[torch.Tensor], shapes: Sequence[Tuple[int, int]],
                 group=None, quantize: Optional[Callable] = None):
    """Quantize this rank's shards, all-gather codes and scales, return the full
    codes and scales of every tensor on every rank.

    shards  this rank's BF16 row shards, shards[i] = W_i[begin:end] with the
            rows of ``plan(shapes, world)[rank][i]`` (row-major, dense)
    shapes  (n, k) of every full tensor, the same on all ranks
    quantize  maps the list of shards to (codes, scales) lists; the library's
            kernel by default
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    plans = plan(shapes, world)
    for (b, e), w, (n, k) in zip(plans[rank], shards, shapes):
        if tuple(w.shape) != (e - b, k):
            raise ValueError("shard of shape %s does not match rows [%d, %d) of a [%d, %d] weight"
                             % (tuple(w.shape), b, e, n, k))
    qs, ss = (quantize or quantize_local)(list(shards))
    sizes = [_piece_sizes(shapes, plans[r]) for r in range(world)]
    q_len = max(1, max(s[0] for s in sizes))
    s_len = max(1, max(s[1] for s in sizes))
    dev = shards[0].device if shards else torch.device("cpu")
    q_local, s_local = pack_piece(qs, ss, q_len, s_len, dev)
    q_all = torch.empty(world * q_len, dtype=torch.uint8, device=dev)
    s_all = torch.empty(world * s_len, dtype=torch.float32, device=dev)
    dist.all_gather_into_tensor(q_all, q_local, group=group)
    dist.all_gather_into_tensor(s_all, s_local, group=group)
    q_pieces = [q_all[r * q_len:(r + 1) * q_len] for r in range(world)]
    s_pieces = [s_all[r * s_len:(r + 1) * s_len] for r in range(world)]
    return assemble(shapes, plans, q_pieces, s_pieces)


def gathered_bytes(shapes: Sequence[Tuple[int, int]], world: int) -> dict:
    """Bytes each rank receives: quantize-then-gather against gather-then-quantize."""
    plans = plan(shapes, world)
    sizes = [_piece_sizes(shapes, p) for p in plans]
    q_len = max(s[0] for s in sizes)
    s_len = max(s[1] for s in sizes)
    bf16 = sum(2 * n * k for n, k in shapes)
    return {"fp8_codes_and_scales": world * (q_len + 4 * s_len), "bf16": bf16}
