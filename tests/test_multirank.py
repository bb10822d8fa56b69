"""The N>1 path on the CPU: two gloo ranks split the heads of one scan on
group boundaries, each computes its slice (with the oracle, standing in for
one GPU's ssd_scan_fwd), and the assembled result equals the unsplit one.
Also checks the max-over-ranks timing reduction the benchmark uses."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from state_space_model_chunked_gb300.sharding import batch_range, head_range, max_over_ranks


def test_head_ranges_cover_all_heads_on_group_boundaries():
    for H, G in [(80, 1), (24, 4), (32, 8), (6, 3)]:
        for world in (1, 2, 3, 4, 8):
            cuts = [head_range(H, G, world, r) for r in range(world)]
            assert cuts[0][0] == 0 and cuts[-1][1] == H
            for (a0, a1), (b0, b1) in zip(cuts, cuts[1:]):
                assert a1 == b0
            for a0, a1 in cuts:
                assert a0 % (H // G) == 0 and a1 % (H // G) == 0


def test_batch_ranges_partition():
    for batch in (1, 7, 16, 256):
        for world in (1, 2, 4, 8):
            cuts = [batch_range(batch, world, r) for r in range(world)]
            assert sum(b - a for a, b in cuts) == batch
            assert cuts[0][0] == 0 and cuts[-1][1] == batch


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, G = 8, 2
    inp = gen.scan_inputs(2, 96, H, 8, 16, G, "bf16", seed=123, random_init=True)
    h0, h1 = head_range(H, G, world, rank)
    g0, g1 = h0 // (H // G), h1 // (H // G)
    sl = slice(h0, h1)
    # this rank's slice: its heads and the groups they belong to
    y, fin = oracle.scan_seq(inp["x"][:, :, sl], inp["dt"][:, :, sl], inp["A"][sl],
                             inp["B"][:, :, g0:g1], inp["C"][:, :, g0:g1], inp["D"][sl],
                             inp["init"][:, sl], nthreads=1)
    np.save(os.path.join(out_dir, f"y{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"f{rank}.npy"), fin)
    worst = max_over_ranks(float(rank + 1) * 1.5, dist)
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([worst]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_scan(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.scan_inputs(2, 96, 8, 8, 16, 2, "bf16", seed=123, random_init=True)
    y_full, f_full = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"y{r}.npy") for r in range(world)]
    fs = [np.load(tmp_path / f"f{r}.npy") for r in range(world)]
    assert oracle.rel_l2(np.concatenate(ys, axis=2), y_full) < 1e-13
    assert oracle.rel_l2(np.concatenate(fs, axis=1), f_full) < 1e-13
    for r in range(world):
        assert float(np.load(tmp_path / f"t{r}.npy")[0]) == 3.0


def test_sequence_ranges_partition_and_balance():
    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import sequence_range
    for lengths in ([5, 0, 13, 1, 9], gen.packed_lengths(47, 64, 8192, seed=5), [100], [0, 0]):
        cu = np.concatenate([[0], np.cumsum(lengths)])
        T, longest = int(cu[-1]), max(lengths)
        for world in (1, 2, 3, 4, 8):
            parts = [sequence_range(cu, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == len(lengths)
            for (a0, a1, _), (b0, b1, _) in zip(parts, parts[1:]):
                assert a1 == b0
            for s0, s1, off in parts:
                assert off[0] == 0 and off[-1] == cu[s1] - cu[s0]
                assert off[-1] <= T / world + longest


def _varlen_worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import sequence_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = gen.varlen_inputs([30, 7, 0, 55, 12, 40], 4, 8, 16, 2, "bf16", seed=9,
                            random_init=True)
    s0, s1, off = sequence_range(inp["cu"], world, rank)
    t0, t1 = int(inp["cu"][s0]), int(inp["cu"][s1])
    y, fin = oracle.scan_varlen(inp["x"][t0:t1], inp["dt"][t0:t1], inp["A"], inp["B"][t0:t1],
                                inp["C"][t0:t1], off, inp["D"], inp["init"][s0:s1])
    np.save(os.path.join(out_dir, f"vy{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"vf{rank}.npy"), fin)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_a_packed_batch(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_varlen_worker, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    inp = gen.varlen_inputs([30, 7, 0, 55, 12, 40], 4, 8, 16, 2, "bf16", seed=9,
                            random_init=True)
    y_full, f_full = oracle.scan_varlen(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                        inp["cu"], inp["D"], inp["init"])
    ys = [np.load(tmp_path / f"vy{r}.npy") for r in range(world)]
    fs = [np.load(tmp_path / f"vf{r}.npy") for r in range(world)]
    assert ys[0].shape[0] > 0 and ys[1].shape[0] > 0
    np.testing.assert_array_equal(np.concatenate(ys, axis=0), y_full)
    np.testing.assert_array_equal(np.concatenate(fs, axis=0), f_full)
