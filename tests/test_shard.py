"""Request sharding across ranks (byte_level_bpe_gb300.shard): the plan, the
one-int64 count exchange and the offset arithmetic, on CPU with gloo ranks and
the oracle standing in for each rank's GPU encode. The concatenation of the
ranks' slices must equal the one-process encode, id for id, with the same
offsets."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _call(seed):
    """A small serving-like call: 40 requests with specials in some of them."""
    import workloads
    rng = np.random.default_rng(seed)
    table = workloads.full_table()
    segs = []
    for i in range(40):
        n = int(rng.integers(0, 3000))
        t = workloads.prose_text(table, n + 8, seed=seed * 100 + i)[:n].decode("utf-8", "ignore")
        if i % 7 == 3:
            t = "<|endoftext|>" + t
        segs.append((t.encode(), bool(i % 2)))
    text, off, allow = workloads.pack_segments(segs)
    return table, np.asarray(text, np.uint8), np.asarray(off, np.int64), np.asarray(allow, np.uint8)


def _rank_main(rank, world, port, out_dir, seed):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    import workloads
    from byte_level_bpe_gb300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    table, text, off, allow = _call(seed)
    enc = oracle.Encoding(table, workloads.SPECIALS)

    def host_encode(t, o, a, safe):
        return enc.encode_arrays(t, o, a, len(o) - 1, safe)

    r = shard.encode_sharded(None, text, off, allow, True, encode_fn=host_encode)
    every = shard.gather_ids(r["ids"])
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), ids=np.asarray(r["ids"]), offsets=r["offsets"],
             base=r["base"], total=r["total"], seg=np.asarray(r["segments"]), every=every)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_equals_one_process(tmp_path, world):
    import torch.multiprocessing as mp

    import oracle
    import workloads
    seed = 7
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), seed), nprocs=world, join=True)
    table, text, off, allow = _call(seed)
    exp_ids, exp_off = oracle.Encoding(table, workloads.SPECIALS).encode_arrays(text, off, allow,
                                                                               len(off) - 1, True)
    rs = [np.load(tmp_path / f"r{r}.npz") for r in range(world)]
    got = np.concatenate([r["ids"] for r in rs])
    assert np.array_equal(got, exp_ids)
    for r in rs:
        s0, s1 = r["seg"]
        assert np.array_equal(r["offsets"], exp_off[s0:s1 + 1])
        assert int(r["total"]) == len(exp_ids)
        assert np.array_equal(r["every"], exp_ids)
    assert [int(r["base"]) for r in rs] == [int(exp_off[r["seg"][0]]) for r in rs]
    assert rs[0]["seg"][0] == 0 and rs[-1]["seg"][1] == len(off) - 1


def test_plan_is_balanced_and_covers():
    sys.path.insert(0, ROOT)
    from byte_level_bpe_gb300 import shard
    rng = np.random.default_rng(3)
    for _ in range(200):
        S = int(rng.integers(0, 60))
        lens = rng.integers(0, 5000, size=S)
        off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        for world in (1, 2, 3, 8):
            b = shard.plan(off, world)
            assert b[0] == 0 and b[-1] == S and np.all(np.diff(b) >= 0)
            n = int(off[-1])
            biggest = int(lens.max()) if S else 0
            for r in range(world):
                got = int(off[b[r + 1]] - off[b[r]])
                assert got <= n / world + biggest + 1
