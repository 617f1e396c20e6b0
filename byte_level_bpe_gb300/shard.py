"""Request sharding: one call's segments encoded across several ranks.

Segments (requests) are independent ("Making Kimi K3 Tokenization 18x Faster
For Million Token Agentic Workloads", "Why Kimi K3 tokenization is
non-trivial": each typed segment is encoded on its own; "Where the speed
comes from": independent chunks go to separate workers; "tiktoken Deep Dive",
"Why the Rust core is fast": a batch encode fans its texts out). So a call's S
segments are cut into `world` contiguous ranges of about equal bytes, each
rank encodes its range with the one-GPU path (tk_encode_segments), and the
only exchange is one all-gather of an int64 id count per rank: its exclusive
scan is the position of the rank's ids in the call's output, so every rank
knows its slice [base, base + count) and its segments' global offsets.

This module holds host logic only (planning, the count exchange, offset
arithmetic); every id is produced by libtk's kernels on the rank's own GPU.
The exchange uses torch.distributed (NCCL between GPUs, gloo on CPU).
"""
import numpy as np

__all__ = ["plan", "exclusive_scan_counts", "encode_sharded", "gather_ids"]


def plan(seg_off, world):
    """Segment ranges of `world` ranks, cut at segment boundaries so that each
    holds about 1/world of the bytes: returns bounds[world + 1] with rank r
    taking segments bounds[r] .. bounds[r + 1] - 1 (a range may be empty)."""
    seg_off = np.asarray(seg_off, np.int64)
    S = len(seg_off) - 1
    n = int(seg_off[-1]) if S >= 0 else 0
    bounds = np.zeros(world + 1, np.int64)
    bounds[world] = S
    for r in range(1, world):
        target = (n * r) // world
        # the segment boundary nearest the byte target, never before the previous cut
        k = int(np.searchsorted(seg_off, target, side="left"))
        k = min(max(k, 0), S)
        if k > 0 and target - seg_off[k - 1] < seg_off[k] - target:
            k -= 1
        bounds[r] = max(k, bounds[r - 1])
    return bounds


def exclusive_scan_counts(count, group=None):
    """All-gathers one int64 per rank; returns (ids before this rank, total,
    every rank's count)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" \
        else torch.device("cpu")
    mine = torch.tensor([int(count)], dtype=torch.int64, device=dev)
    every = [torch.zeros(1, dtype=torch.int64, device=dev) for _ in range(world)]
    dist.all_gather(every, mine, group=group)
    counts = np.array([int(t.item()) for t in every], np.int64)
    return int(counts[:rank].sum()), int(counts.sum()), counts


def encode_sharded(tok, text, seg_off, allow, tiktoken_safe=True, group=None, encode_fn=None):
    """Encodes this rank's share of the call (text uint8[n], seg_off int64[S+1],
    allow uint8[S], on the host; every rank passes the whole call).

    Returns a dict: ids (this rank's ids, a device tensor from tok, or what
    encode_fn returned), offsets (int64[s1 - s0 + 1]: the global offsets of
    segments s0 .. s1, i.e. entries s0 .. s1 of the one-process call's
    offsets), base (the position of ids[0] in the call's output), total (ids
    of the whole call) and segments (s0, s1).

    encode_fn(text, seg_off, allow, tiktoken_safe) -> (ids, offsets) replaces
    the GPU encode (host stand-ins in tests); by default the share is copied to
    the rank's GPU and encoded there with tok.encode_device.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    seg_off = np.asarray(seg_off, np.int64)
    allow = np.asarray(allow, np.uint8)
    bounds = plan(seg_off, world)
    s0, s1 = int(bounds[rank]), int(bounds[rank + 1])
    b0, b1 = int(seg_off[s0]), int(seg_off[s1])
    l_text = np.ascontiguousarray(np.asarray(text, np.uint8)[b0:b1])
    l_off = np.ascontiguousarray(seg_off[s0:s1 + 1] - b0)
    l_allow = np.ascontiguousarray(allow[s0:s1]) if s1 > s0 else np.zeros(1, np.uint8)
    if encode_fn is None:
        import torch
        d_text = torch.from_numpy(l_text.copy()).to(tok.device)
        d_off = torch.from_numpy(l_off).to(tok.device)
        d_allow = torch.from_numpy(l_allow.copy()).to(tok.device)
        ids, offs = tok.encode_device(d_text, d_off, d_allow, tiktoken_safe)
        offs = offs.cpu().numpy()
    else:
        ids, offs = encode_fn(l_text, l_off, l_allow, tiktoken_safe)
        offs = np.asarray(offs, np.int64)
    count = int(offs[-1]) if len(offs) else 0
    base, total, _ = exclusive_scan_counts(count, group)
    return {"ids": ids, "offsets": offs + base, "base": base, "total": total, "segments": (s0, s1)}


def gather_ids(ids, group=None):
    """The whole call's ids on every rank (this rank's slice from
    encode_sharded in, the concatenation in rank order out, as a numpy array):
    an all-gather of the counts, then of the slices padded to the largest."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    nccl = dist.get_backend(group) == "nccl"
    dev = torch.device("cuda", torch.cuda.current_device()) if nccl else torch.device("cpu")
    t = ids if torch.is_tensor(ids) else torch.from_numpy(np.asarray(ids, np.int32))
    t = t.to(dev, dtype=torch.int32)
    _, _, counts = exclusive_scan_counts(t.numel(), group)
    m = int(max(counts.max(), 1))
    pad = torch.zeros(m, dtype=torch.int32, device=dev)
    pad[:t.numel()] = t
    parts = [torch.zeros(m, dtype=torch.int32, device=dev) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return np.concatenate([p[:int(c)].cpu().numpy() for p, c in zip(parts, counts)])
