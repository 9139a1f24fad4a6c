"""Multi-process fills split by counter range (CPU, gloo, world size 2).

Each rank fills its own slice [offset, offset + length) of a global fill by
passing first_counter + offset (no data exchange on the path); the test
gathers the slices and checks that, in rank order, they are the
single-process fill.  The fills come from the CPU oracle: this covers the
host-side sharding arithmetic and the slice invariant it relies on."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from dropout_lowbias32_hash32_gb300.sharding import first_counter, shard


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, n_total, global_first, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    orc = oracle.default()
    off, length = shard(n_total, rank, world)
    c0 = first_counter(global_first, off)
    parts = {
        "u32": orc.fill_u32(3, c0, length),
        "normal_f64": orc.fill_normal_f64(7, c0, length),
        "below": orc.fill_u32_below(1, c0, (1 << 31) + 1, length),
    }
    gathered = [None] * world
    dist.all_gather_object(gathered, (rank, off, length, parts))
    if rank == 0:
        np.save(os.path.join(result_dir, "ok.npy"), np.array([1]))
        for name in parts:
            whole = np.concatenate([g[3][name] for g in sorted(gathered, key=lambda g: g[0])])
            np.save(os.path.join(result_dir, f"{name}.npy"), whole)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("n_total,global_first", [(10007, (1 << 32) - 5), (4, 0), (1, 3)])
def test_two_rank_counter_shards_concatenate_to_the_whole_fill(tmp_path, n_total, global_first):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), n_total, global_first, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    import oracle
    orc = oracle.default()
    assert np.array_equal(np.load(tmp_path / "u32.npy"), orc.fill_u32(3, global_first, n_total))
    assert np.array_equal(np.load(tmp_path / "normal_f64.npy").view(np.uint64),
                          orc.fill_normal_f64(7, global_first, n_total).view(np.uint64))
    assert np.array_equal(np.load(tmp_path / "below.npy"),
                          orc.fill_u32_below(1, global_first, (1 << 31) + 1, n_total))


def test_shard_covers_the_range_exactly():
    for n in (0, 1, 7, 1 << 20, (1 << 28) + 3):
        for world in (1, 2, 3, 8):
            spans = [shard(n, r, world) for r in range(world)]
            assert spans[0][0] == 0
            assert sum(length for _, length in spans) == n
            for (o1, l1), (o2, _) in zip(spans, spans[1:]):
                assert o1 + l1 == o2
    with pytest.raises(ValueError):
        shard(10, 2, 2)
    assert first_counter((1 << 32) - 5, 7) == 2
